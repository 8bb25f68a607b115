// F2/F3/F4: attention backward on sm_103a.
//
// Follows "FlashAttention and online softmax" (ML Systems lesson 4), section 3 "Backward pass:
// recompute instead of store": only O and lse are kept from the forward pass; every tile of P
// is rebuilt on chip as P = e^{S - lse} (no max and no sum needed), then
//   dV_j += P^T dO_i,  dP = dO_i V_j^T,  dS = P o (dP - D_i),  D_i = dO_i . O_i,
//   dQ_i += scale dS K_j,  dK_j += scale dS^T Q_i.
// The pages leave the loop order of the backward open; this file takes the plainest reading of
// the "+=" in steps 2 and 4: K_j and V_j stay on chip for a whole CTA (dK_j, dV_j accumulate in
// TMEM, written once), query tiles stream, and dQ is accumulated across key tiles in fp32.
//
//   F2  bwd_pre:   D = rowsum(dO o O) in fp32; zero the fp32 dQ accumulator.
//   F3  bwd_main:  one CTA per (128-key tile, head); 480 threads:
//         warp 0     TMA producer: K_j, V_j once; Q_i, dO_i per query tile through a 3-deep
//                    ring.  (lse_i and D_i are loaded by the dS warps themselves.)
//         warp 1     TMEM owner and MMA issuer: S^T = K Q^T, dP^T = V dO^T (keys on TMEM
//                    lanes), dV += P^T dO (P^T read from TMEM), dK += dS^T Q, and the dQ tile
//                    product, issued per step as dV_i, S/dP_{i+1}, dK_i, dQ_i.
//         warps 2-9  two warpgroups, thread = (key row, half of the query columns):
//                    P^T = 2^{S^T scale log2e - lse log2e} (masked), dS^T = P^T o (dP^T - D).
//                    P^T (bf16) goes back into TMEM over the S^T columns just read; dS^T
//                    (bf16) goes to shared memory, where the dK and dQ products read it.
//                    Epilogue: one group writes dV, the other dK (times scale), via TMA.
//         warps 10-13 drain the dQ tile from TMEM into the fp32 accumulator, overlapping the
//                    next tile's MMAs, through an fp32 box in shared memory and TMA
//                    reduce-adds (the L2 performs the adds): d = 128 a row-major box of its
//                    own, d = 64 the step's dS^T buffer (dead once the step's dK and dQ
//                    products are done), in the 128-byte-swizzled layout.
//         warp 14    helper: folds the waits that do not depend on the dS math (stage loaded,
//                    dS^T and dQ buffers free) into the hand-offs the MMA thread waits on.
//       TMEM (512 columns): dV, dK (d each), S^T, dP^T (BM each), two dQ tiles (64 each), so
//       the dQ drain of step i overlaps the dQ product of step i+1.
//       d = 128 uses 64-query steps and forms dQ^T = K^T dS^T (d on TMEM lanes);
//       d = 64 uses 128-query steps and forms dQ = dS K (queries on TMEM lanes).
//       S^T and dP^T are committed separately, so the dS warps exponentiate while dP^T runs.
//       Variants (template flags): VL -- packed variable-length batches; WIN -- a sliding
//       window (only the query tiles some row of the key tile sees); BS -- a block mask (only
//       the query blocks set with the key tile, found from a bit array of the mask column).
//       Short heads at d = 64 run on bwd_persistent_kernel64 (below): the same roles and
//       products, one CTA per SM walking (head, key tile) items.
//   F4  bwd_dq_convert: dq = bf16(scale * dQ_acc).
#include <algorithm>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {

template <int D>
struct BwdCfg {
  static constexpr int BN = 128;                    // keys per CTA
  static constexpr int BM = (D == 128) ? 64 : 128;  // queries per step
  static constexpr int KCH = D / 64;
  static constexpr int QCH = BM / 64;
  static constexpr int KV_TILE = BN * D * 2;
  static constexpr int KV_CHUNK = BN * 128;         // [128 rows x 64 cols] swizzled
  static constexpr int Q_TILE = BM * D * 2;
  static constexpr int Q_CHUNK = BM * 128;          // [BM rows x 64 cols] swizzled
  static constexpr int DS_TILE = BN * BM * 2;       // dS^T, [QCH][128][64]
  static constexpr int NST = 3;
  static constexpr int STAGE = 2 * Q_TILE;          // Q, dO (swizzled, 1 KB aligned)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_TILE;
  static constexpr int OFF_ST = 2 * KV_TILE;
  static constexpr int OFF_DS = OFF_ST + NST * STAGE;
  // d = 128: staging of one fp32 dQ tile [BM queries][d] for the TMA reduce-add into dQ_acc
  static constexpr int DQS_BYTES = (D == 128) ? BM * D * 4 : 0;
  static constexpr int OFF_DQS = OFF_DS + 2 * DS_TILE;      // dS^T double-buffered
  // one slot of HALF floats per dS warp, through which its lanes pass the step's -lse and then
  // -D to the whole warp (broadcast loads instead of shuffles)
  static constexpr int OFF_SLOT = OFF_DQS + DQS_BYTES;
  static constexpr int SLOT_BYTES = 8 * (BM / 2) * 4;
  static constexpr int OFF_BAR = OFF_SLOT + SLOT_BYTES;
  // kv_full, stage_full[NST], stage_empty[NST], st_full, dp_full, p_ready, ds_ready,
  // pds_free[2], dq_full[2], dq_free[2], mma_done, dqs_sync, dqs_done[2]
  static constexpr int NBAR = 1 + 2 * NST + 14;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;       // TMEM slot, abort flag, step count
  // block-sparse: one bit per query block, set where this CTA's key tile has work
  static constexpr int OFF_BSW = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = OFF_BSW + kBlockSparseMaxTiles / 8 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_DV = 0;
  static constexpr uint32_t T_DK = D;
  static constexpr uint32_t T_S = 2 * D;
  static constexpr uint32_t T_DP = 2 * D + BM;
  static constexpr uint32_t T_DQ = 2 * D + 2 * BM;  // two dQ tile buffers of 64 columns
  static constexpr int THREADS = 480;             // + warp 14, the MMA thread's helper
  static constexpr int DS_THREADS = 256;          // two dS warpgroups
  static constexpr int HALF = BM / 2;             // query columns per dS warpgroup
  static_assert(T_DQ + 128 <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
};

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  CUtensorMap tdq;                                  // fp32 dQ accumulator
  const float* lse;
  const float* delta;
  float* dq_acc;
  int n_q, n_kv, n_qtiles, n_kvtiles, causal;
  float scale, scale_log2;
  // Variable-length batches (packed token-major [total, H, d]; lse and D [H, total_q]; the dQ
  // accumulator in the packed row order (token * H + head)).
  int heads, total_q, total_k, max_q, max_k;
  const int* cu_q;
  const int* cu_k;
  uint16_t* dk;
  uint16_t* dv;
  // Visible keys of query i: i - win_left <= j <= i + win_right (kWinUnbounded: no bound).
  int win_left, win_right;
  // Block-sparse: 0/1 per (128-query block, 128-key block) pair, [n_qblocks][n_kvtiles] for
  // every head (bm_per_head = 0) or one such array per (b, h) plane.
  const uint8_t* block_mask;
  int bm_per_head, n_qblocks;
  unsigned long long* stats;                        // diagnostic counters (see fa_kernels.h)
  int n_items;                                      // persistent backward: B*H*n_kvtiles
};

template <int D, bool VL, bool WIN = false, bool BS = false>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1k(smem_raw);
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sDS = smem + C::OFF_DS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* stage_full = bars + 1;
  uint64_t* stage_empty = stage_full + C::NST;
  uint64_t* st_full = stage_empty + C::NST;
  uint64_t* dp_full = st_full + 1;       // dP^T of the step is in TMEM (committed after S^T)
  uint64_t* p_ready = dp_full + 1;       // P^T of the step is in TMEM (dV may start)
  uint64_t* ds_ready = p_ready + 1;      // dS^T of the step is in shared memory (dK, dQ may start)
  uint64_t* pds_free = ds_ready + 1;     // [2], one per dS^T buffer (d = 128)
  uint64_t* dq_full = pds_free + 2;      // [2], one per dQ TMEM buffer
  uint64_t* dq_free = dq_full + 2;       // [2]
  uint64_t* mma_done = dq_free + 2;
  uint64_t* dqs_sync = mma_done + 1;     // the four dQ warps around the staging buffer
  uint64_t* dqs_done = dqs_sync + 1;     // [2] d = 64: dQ staged in dS^T buffer b read by the TMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: key tile kt of head bh; causal key tiles with more query tiles run first,
  // across groups of kCausalGroup heads.  Under a block mask every head's key tile 0 runs
  // first, then every head's key tile 1, ...: a causal column shortens as kt grows and a
  // globally visible key block makes its column dense, so the long columns of all heads start
  // together (measured on a 16-head, 16K-token causal pattern with a global first block: 0.70
  // -> 0.50 ms against the head groups, whose last group's dense columns started late).
  int bh = blockIdx.x / p.n_kvtiles;                 // fixed length: (b, h) plane
  int kt = blockIdx.x % p.n_kvtiles;
  if (BS) {
    bh = blockIdx.x % (gridDim.x / p.n_kvtiles);
    kt = blockIdx.x / (gridDim.x / p.n_kvtiles);
  } else if (!VL && !WIN && p.causal) {
    causal_item(blockIdx.x, gridDim.x / p.n_kvtiles, p.n_kvtiles, &bh, &kt);
  }
  const int k0 = kt * C::BN;
  int n_q = p.n_q, n_kv = p.n_kv, q_beg = 0, k_beg = 0, head = 0;
  if (VL) {
    // item = (sequence, head, key tile) sized by the longest sequence; boundaries are checked
    const int seq = bh / p.heads;
    head = bh % p.heads;
    q_beg = p.cu_q[seq];
    n_q = p.cu_q[seq + 1] - q_beg;
    k_beg = p.cu_k[seq];
    n_kv = p.cu_k[seq + 1] - k_beg;
    if (q_beg < 0 || n_q < 0 || q_beg + n_q > p.total_q || n_q > p.max_q || k_beg < 0 ||
        n_kv < 0 || k_beg + n_kv > p.total_k || n_kv > p.max_k) {
      if (threadIdx.x == 0 && kt == 0) report_device_error(FA_DEV_BAD_CONFIG, 250);
      return;
    }
    if (k0 >= n_kv) return;                         // whole CTA, before any shared state
  }
  const int n_qtiles = (n_q + C::BM - 1) / C::BM;
  // Query tiles that see some key of [k0, k0 + BN): rows i with k0 - win_right <= i and
  // i <= k0 + BN - 1 + win_left; the others are skipped (never loaded).
  // Without a window only the causal start applies (WIN = false keeps that path lean).
  const int wr = min(p.win_right, kWinUnbounded - C::BN);
  const int wl = min(p.win_left, kWinUnbounded - C::BN);
  const int i_start = WIN ? max(0, k0 - wr) / C::BM : (p.causal ? (k0 / C::BM) : 0);
  const int i_end = WIN ? min(n_qtiles, (k0 + C::BN - 1 + wl) / C::BM + 1) : n_qtiles;
  int n = max(0, i_end - i_start);
  // Block-sparse: the steps are those of the query blocks whose block with this key tile is set
  // (with causal, on or below the diagonal), in order, 128 / BM steps each (fewer for a ragged
  // last block).  Warp 14 counts them before the roles start; each role that needs a step's
  // first query walks the mask column with its own cursor (step_q0, called once per step).
  const uint8_t* bs_col = nullptr;
  if constexpr (BS)
    bs_col = p.block_mask + static_cast<size_t>(p.bm_per_head ? bh : 0) * p.n_qblocks * p.n_kvtiles + kt;
  auto bs_set = [&](int qb) {
    return bs_col[static_cast<size_t>(qb) * p.n_kvtiles] != 0 && (!p.causal || qb >= kt);
  };
  auto bs_steps = [&](int qb) { return min(kBlockSize / C::BM, (n_q - qb * kBlockSize + C::BM - 1) / C::BM); };
  const uint32_t* s_bsw = reinterpret_cast<const uint32_t*>(smem + C::OFF_BSW);
  const int bs_words = (p.n_qblocks + 31) / 32;
  int bs_qb = -1, bs_sub = 0;
  auto step_q0 = [&](int i) -> int {
    if constexpr (BS) {
      if (bs_qb < 0 || ++bs_sub >= bs_steps(bs_qb)) {
        bs_sub = 0;                             // next set query block, from the bit words
        const int q = bs_qb + 1;
        int w = q >> 5;
        uint32_t word = (w < bs_words) ? (s_bsw[w] & (0xffffffffu << (q & 31))) : 0u;
        while (word == 0u && ++w < bs_words) word = s_bsw[w];
        bs_qb = (word != 0u) ? (w << 5) + __ffs(word) - 1 : p.n_qblocks;
      }
      return bs_qb * kBlockSize + bs_sub * C::BM;
    } else {
      return (i_start + i) * C::BM;
    }
  };
  if constexpr (BS) {
    if (warp == 14) {
      uint32_t* w_out = reinterpret_cast<uint32_t*>(smem + C::OFF_BSW);
      int cnt = 0;
      for (int base = 0; base < p.n_qblocks; base += 32) {
        const int qb = base + lane;
        const bool set = qb < p.n_qblocks && bs_set(qb);
        const uint32_t bal = __ballot_sync(0xffffffffu, set);
        if (lane == 0) w_out[base >> 5] = bal;
        cnt += __reduce_add_sync(0xffffffffu, set ? bs_steps(qb) : 0);
      }
      if (lane == 0) *reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8) = cnt;
    }
  }
  // TMA coordinates of local row ``row``: fixed length {x, row, (b,h)}; packed {x, h, beg+row}
  auto y1 = [&](int row) { return VL ? head : row; };
  auto y2 = [&](int beg, int row) { return VL ? beg + row : bh; };
  // packed-row index of local query q: fixed [B*H, N] order, packed token * H + head
  auto qrow = [&](int q) -> size_t {
    return VL ? static_cast<size_t>(q_beg + q) * p.heads + head : static_cast<size_t>(bh) * n_q + q;
  };

  auto stage_ptr = [&](int s) { return smem + C::OFF_ST + s * C::STAGE; };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&stage_full[s], 1);      // TMA bytes
      mbar_init(&stage_empty[s], 1);
    }
    // st_full: the MMA's commit + the helper, which folds in "stage i loaded" (lse, D) and
    // "dS^T buffer i & 1 free" (dK, dQ of step i-2 done) so the dS warps wait once per step
    mbar_init(st_full, 2);
    mbar_init(dp_full, 1);
    // the dS threads + the helper warp's lane 0 (which folds in the other conditions)
    mbar_init(p_ready, C::DS_THREADS + 1);
    mbar_init(ds_ready, C::DS_THREADS + 1);
    mbar_init(&pds_free[0], 1);
    mbar_init(&pds_free[1], 1);
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(&dq_full[b2], 1);
      mbar_init(&dq_free[b2], 128);
    }
    mbar_init(mma_done, 1);
    mbar_init(dqs_sync, 4);
    mbar_init(&dqs_done[0], 1);
    mbar_init(&dqs_done[1], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
    tma_prefetch_desc(&p.tdo);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  if constexpr (BS) n = *reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (n > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::KV_TILE);
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_3d(sK + c * C::KV_CHUNK, &p.tk, kv_full, c * 64, y1(k0), y2(k_beg, k0));
          tma_load_3d(sV + c * C::KV_CHUNK, &p.tv, kv_full, c * 64, y1(k0), y2(k_beg, k0));
        }
      }
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n; ++i) {
        const int s = i % C::NST;
        const uint32_t u = i / C::NST;
        if (u > 0 && !(ok = mbar_wait_warp(&stage_empty[s], (u - 1) & 1, abort_flag, 201))) break;
        uint8_t* st = stage_ptr(s);
        const int q0 = step_q0(i);
        if (lane == 0) {
          mbar_arrive_expect_tx(&stage_full[s], 2 * C::Q_TILE);
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(st + c * C::Q_CHUNK, &p.tq, &stage_full[s], c * 64, y1(q0), y2(q_beg, q0));
            tma_load_3d(st + C::Q_TILE + c * C::Q_CHUNK, &p.tdo, &stage_full[s], c * 64, y1(q0),
                        y2(q_beg, q0));
          }
        }
        issued = i + 1;
      }
      if (!ok && lane == 0) {
        mbar_wait(kv_full, 0, nullptr, 202);
        for (int i = max(0, issued - C::NST); i < issued; ++i)
          mbar_wait(&stage_full[i % C::NST], (i / C::NST) & 1, nullptr, 203);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // d = 64: the converged warp issues (umma_*_w); d = 128: one thread (measured: the
    // 4x32x4096x128 backward 2.49 ms against 2.52 ms with the warp, 4x16x2048x64 272 against
    // 279 us the other way)
    constexpr bool WI = D == 64;
    if ((WI || lane == 0) && n > 0) {
      const uint32_t id_s = idesc_bf16_f32(128, C::BM, 0, 0);     // K/V K-major, Q/dO K-major
      const uint32_t id_acc = idesc_bf16_f32(128, D, 0, 1);       // P^T (TMEM) / dS^T K-major, dO/Q MN-major
      const uint32_t id_dq = idesc_bf16_f32(128, 64, 1, 1);       // both MN-major
      // Descriptors are built once; every k-step adds a compile-time offset (desc_advance).
      const uint64_t dK_k = smem_desc_sw128(smem_u32(sK), 0, 1024);          // K as K-major A
      const uint64_t dV_k = smem_desc_sw128(smem_u32(sV), 0, 1024);          // V as K-major A
      const uint64_t dK_mn = smem_desc_sw128(smem_u32(sK), C::KV_CHUNK, 1024);  // K as MN-major
      const uint64_t dDS = smem_desc_sw128(smem_u32(sDS), 0, 1024);
      const uint64_t dDS_mn = smem_desc_sw128(smem_u32(sDS), C::KV_CHUNK, 1024);
      const uint64_t dST_k = smem_desc_sw128(smem_u32(stage_ptr(0)), 0, 1024);        // Q/dO K-major
      const uint64_t dST_mn = smem_desc_sw128(smem_u32(stage_ptr(0)), C::Q_CHUNK, 1024);  // MN-major
      auto issue_s_dp = [&](int i) {
        const uint32_t st = (i % C::NST) * C::STAGE;
        const uint64_t q_k = desc_advance(dST_k, st);
        const uint64_t do_k = desc_advance(dST_k, st + C::Q_TILE);
        // S^T first and committed on its own, so the dS warps exponentiate while dP^T runs
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t kv_off = (ks >> 2) * C::KV_CHUNK + (ks & 3) * 32;
          const uint32_t q_off = (ks >> 2) * C::Q_CHUNK + (ks & 3) * 32;
          umma_ss_by<WI>(tbase + C::T_S, desc_advance(dK_k, kv_off), desc_advance(q_k, q_off), id_s, ks > 0);
        }
        umma_commit_by<WI>(st_full);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t kv_off = (ks >> 2) * C::KV_CHUNK + (ks & 3) * 32;
          const uint32_t q_off = (ks >> 2) * C::Q_CHUNK + (ks & 3) * 32;
          umma_ss_by<WI>(tbase + C::T_DP, desc_advance(dV_k, kv_off), desc_advance(do_k, q_off), id_s, ks > 0);
        }
        umma_commit_by<WI>(dp_full);
      };
      bool ok = mbar_wait_by<WI>(kv_full, 0, abort_flag, 211) &&
                mbar_wait_by<WI>(&stage_full[0], 0, abort_flag, 212);
      if (ok) {
        tc_fence_after();
        issue_s_dp(0);
      }
      // Per step i: dV_i as soon as P^T_i is in TMEM (over the S^T columns), then S/dP of step
      // i+1 (they overwrite those columns, so they come after dV_i in issue order; the dS warps
      // have read S^T_i and dP^T_i before signalling P^T), then dK_i and dQ_i once dS^T_i is in
      // shared memory.  The tensor core thus runs dV_i and S/dP_{i+1} while the dS warps still
      // form dS_i, and dK_i/dQ_i while they start on step i+1.
      for (int i = 0; ok && i < n; ++i) {
        const int s = i % C::NST;
        if (!(ok = mbar_wait_by<WI>(p_ready, i & 1, abort_flag, 215))) break;
        tc_fence_after();
        const uint64_t q_mn = desc_advance(dST_mn, s * C::STAGE);
        const uint64_t do_mn = desc_advance(dST_mn, s * C::STAGE + C::Q_TILE);
#pragma unroll
        for (int ks = 0; ks < C::BM / 16; ++ks)       // dV += P^T dO
          umma_ts_by<WI>(tbase + C::T_DV, tbase + C::T_S + ks * 8 + ((16 * ks) / C::HALF) * (C::HALF / 2),
                  desc_advance(do_mn, ks * 2048), id_acc, (i > 0 || ks > 0) ? 1u : 0u);
        // stage i+1 is loaded: p_ready(i) includes the helper's check of it
        if (i + 1 < n) issue_s_dp(i + 1);
        if (!(ok = mbar_wait_by<WI>(ds_ready, i & 1, abort_flag, 218))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < C::BM / 16; ++ks) {     // dK += dS^T Q
          const uint32_t a_off = (ks >> 2) * C::KV_CHUNK + (ks & 3) * 32;
          umma_ss_by<WI>(tbase + C::T_DK, desc_advance(dDS, (i & 1) * C::DS_TILE + a_off), desc_advance(q_mn, ks * 2048), id_acc,
                  (i > 0 || ks > 0) ? 1u : 0u);
        }
        // dQ TMEM buffer of this step, drained: ds_ready(i) includes the helper's check of it
        const int qb = i & 1;
#pragma unroll
        for (int ks = 0; ks < C::BN / 16; ++ks) {
          // d = 128: dQ^T = K^T dS^T (A = K as MN-major, B = dS^T as MN-major)
          // d = 64:  dQ   = dS K     (A = dS^T as MN-major, B = K as MN-major)
          const uint64_t kd = desc_advance(dK_mn, ks * 2048);
          const uint64_t dd = desc_advance(dDS_mn, (i & 1) * C::DS_TILE + ks * 2048);
          if constexpr (D == 128) umma_ss_by<WI>(tbase + C::T_DQ + qb * 64, kd, dd, id_dq, ks > 0);
          else umma_ss_by<WI>(tbase + C::T_DQ + qb * 64, dd, kd, id_dq, ks > 0);
        }
        umma_commit_by<WI>(&dq_full[qb]);
        if constexpr (D == 128) umma_commit_by<WI>(&pds_free[i & 1]);   // d = 64: dqs_done (dQ warps)
        umma_commit_by<WI>(&stage_empty[s]);
      }
      umma_commit_by<WI>(mma_done);
      mbar_wait_by<WI>(mma_done, 0, nullptr, 217);
      if (ok && lane == 0 && p.stats != nullptr) atomicAdd(&p.stats[1], static_cast<unsigned long long>(n));
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------------ dS warpgroups
    const int sub = warp & 3;
    const int grp = (warp - 2) >> 2;               // which half of the query columns
    const int cb = grp * C::HALF;                  // first column of this group
    const int r = sub * 32 + lane;                 // key row within the tile
    const uint32_t t_lane = static_cast<uint32_t>(sub * 32) << 16;
    const int k_idx = k0 + r;
    const bool row_dead = k_idx >= n_kv;
    const float c2 = p.scale_log2;
    bool ok = true;
    // -lse (log2 units) and -D of query column q of the step: lane l loads column l from global
    // memory (L1/L2 hits: every dS warp of a group reads the same columns) and shuffles pass the
    // values round.  The loads are issued before the wait for S_i, which hides their latency.
    auto nlse_of = [&](int q) -> float {
      const size_t li = VL ? static_cast<size_t>(head) * p.total_q + q_beg + q : qrow(q);
      return (q < n_q) ? -__ldg(p.lse + li) * 1.4426950408889634f : -INFINITY;
    };
    auto nd_of = [&](int q) -> float {
      const size_t di = VL ? static_cast<size_t>(head) * p.total_q + q_beg + q : qrow(q);
      return (q < n_q) ? -__ldg(p.delta + di) : 0.f;
    };
    // a warp none of whose key rows is past the keys' end (only a ragged last key tile has some)
    bool warp_live = false;
    if constexpr (D == 128) warp_live = !__any_sync(0xffffffffu, row_dead);
    for (int i = 0; i < n; ++i) {
      const int q0 = step_q0(i);
      float lane_nd[C::HALF / 32], nl0[32];
      const float lane_nl = nlse_of(q0 + cb + lane);
      lane_nd[0] = nd_of(q0 + cb + lane);
      // st_full(i): S_i is done, stage i is loaded and dS^T buffer i & 1 is free (the last two
      // folded in by the helper); dp_full(i), waited for below: dP_i is done
      if (!(ok = mbar_wait_warp(st_full, i & 1, abort_flag, 221))) break;
      tc_fence_after();
      float* slot = reinterpret_cast<float*>(smem + C::OFF_SLOT) + (warp - 2) * C::HALF;
      slot[lane] = lane_nl;
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(slot + e);
        nl0[e] = v.x; nl0[e + 1] = v.y; nl0[e + 2] = v.z; nl0[e + 3] = v.w;
      }
      // a (key tile, query tile) pair that some pair of rows sees only in part
      const bool diag = WIN ? ((q0 < k0 + C::BN - 1 - wr) || (q0 + C::BM - 1 > k0 + wl))
                            : (p.causal && (q0 < k0 + C::BN - 1));
      // d = 128: nothing to mask in this step for this warp, so no per-element tests (measured:
      // -1.2% unmasked, -1.6% causal at 4x32x4096; at d = 64 the same form was 13-15% slower)
      const bool plain = D == 128 && !WIN && !diag && warp_live;
      const float2 c2v = make_float2(c2, c2);
      const int c_lo = k_idx - wr - q0, c_hi = k_idx + wl - q0;
      uint32_t pk_ds[C::HALF / 2];
      // P (exp) first; P^T goes back over S^T columns this thread has already read (its own
      // half, bf16 pairs): group g's query q sits at column g*HALF + (q - g*HALF)/2, where the
      // dV product reads it.  p_ready is signalled as soon as every thread has stored its P^T
      // and read its dP^T, so dV and the next S/dP products (which overwrite S^T and dP^T)
      // overlap the dS math below.
      // d = 64 (64 columns a thread) keeps P for the dS product as the bf16 pairs it stores for
      // the dV product: fp32 P would not fit the 128 registers a thread has with 15 warps (the
      // spills cost more than the rounding, which stays below dS's own bf16 rounding); d = 128
      // keeps fp32 P
      constexpr bool kPackedP = (D == 64);
      float pf[kPackedP ? 1 : C::HALF];
      uint32_t ppk[kPackedP ? C::HALF / 2 : 1];
      uint32_t dpu[C::HALF / 32][32];
#pragma unroll
      for (int c = 0; c < C::HALF / 32; ++c) {
        uint32_t rs[32];
        tmem_ld32(tbase + t_lane + C::T_S + cb + c * 32, rs);
        float nl[32];
        if (c == 0) {
#pragma unroll
          for (int e = 0; e < 32; ++e) nl[e] = nl0[e];
        } else {
          slot[c * 32 + lane] = nlse_of(q0 + cb + c * 32 + lane);
          lane_nd[c] = nd_of(q0 + cb + c * 32 + lane);
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 v = *reinterpret_cast<const float4*>(slot + c * 32 + e);
            nl[e] = v.x; nl[e + 1] = v.y; nl[e + 2] = v.z; nl[e + 3] = v.w;
          }
        }
        tmem_wait_ld();
        uint32_t pk_p[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = cb + c * 32 + e;
          const float2 x = ffma2(make_float2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2v,
                                 make_float2(nl[e], nl[e + 1]));
          float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
          if (!plain) {
            if constexpr (WIN) {
              // query q0 + col sees key k_idx iff c_lo <= col <= c_hi
              if (row_dead || (diag && (col < c_lo || col > c_hi))) p0 = 0.f;
              if (row_dead || (diag && (col + 1 < c_lo || col + 1 > c_hi))) p1 = 0.f;
            } else {
              if (row_dead || (diag && k_idx > q0 + col)) p0 = 0.f;
              if (row_dead || (diag && k_idx > q0 + col + 1)) p1 = 0.f;
            }
          }
          pk_p[e / 2] = pack_bf16x2(p0, p1);
          if constexpr (kPackedP) {
            ppk[c * 16 + e / 2] = pk_p[e / 2];
          } else {
            pf[c * 32 + e] = p0;
            pf[c * 32 + e + 1] = p1;
          }
        }
        tmem_st16(tbase + t_lane + C::T_S + cb + c * 16, pk_p);
      }
      if (!(ok = mbar_wait_warp(dp_full, i & 1, abort_flag, 224))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::HALF / 32; ++c) tmem_ld32(tbase + t_lane + C::T_DP + cb + c * 32, dpu[c]);
      tmem_wait_ld();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_ready);
      __syncwarp();                                // the slot now passes -D (-lse was read out)
#pragma unroll
      for (int c = 0; c < C::HALF / 32; ++c) slot[c * 32 + lane] = lane_nd[c];
      __syncwarp();
      // dS^T = P^T o (dP^T - D)
#pragma unroll
      for (int e = 0; e < C::HALF; e += 2) {
        const float2 dp = make_float2(__uint_as_float(dpu[e / 32][e % 32]), __uint_as_float(dpu[e / 32][e % 32 + 1]));
        const float2 nd = *reinterpret_cast<const float2*>(slot + e);
        float2 pp;
        if constexpr (kPackedP)
          pp = make_float2(__uint_as_float(ppk[e / 2] << 16), __uint_as_float(ppk[e / 2] & 0xffff0000u));
        else
          pp = make_float2(pf[e], pf[e + 1]);
        const float2 ds = fmul2(pp, fadd2(dp, nd));
        pk_ds[e / 2] = pack_bf16x2(ds.x, ds.y);
      }
      uint8_t* sDSi = sDS + (i & 1) * C::DS_TILE;
#pragma unroll
      for (int u = 0; u < C::HALF / 8; ++u) {
        const int c8 = cb / 8 + u;                   // 16-byte unit along the query axis
        const uint32_t off = (c8 >> 3) * C::KV_CHUNK + sw128_offset(r, (c8 & 7) * 8);
        *reinterpret_cast<uint4*>(sDSi + off) =
            make_uint4(pk_ds[4 * u], pk_ds[4 * u + 1], pk_ds[4 * u + 2], pk_ds[4 * u + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(ds_ready);
    }
    // ---------------------------------------------------------------- epilogue: dK, dV
    if (ok && n > 0) {
      ok = mbar_wait_warp(mma_done, 0, abort_flag, 223);
      tc_fence_after();
    }
    // A packed key tile that ends past its sequence is stored row by row (a TMA store of the
    // whole box would write into the next sequence's rows).
    const bool rowwise = VL && (k0 + C::BN > n_kv);
    if (ok) {
      {
        const int which = grp;                        // group 0 writes dV, group 1 dK
        uint8_t* dst = which ? sK : sV;               // operands are dead once mma_done fired
        uint16_t* grow = rowwise ? (which ? p.dk : p.dv) +
                                       (static_cast<size_t>(k_beg + k_idx) * p.heads + head) * D
                                 : nullptr;
        const uint32_t tcol = which ? C::T_DK : C::T_DV;
        const float mul = which ? p.scale : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          if (n > 0) {
            tmem_ld32(tbase + t_lane + tcol + c * 32, rr);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) rr[e] = 0u;
          }
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v4;
            v4.x = pack_bf16x2(__uint_as_float(rr[e + 0]) * mul, __uint_as_float(rr[e + 1]) * mul);
            v4.y = pack_bf16x2(__uint_as_float(rr[e + 2]) * mul, __uint_as_float(rr[e + 3]) * mul);
            v4.z = pack_bf16x2(__uint_as_float(rr[e + 4]) * mul, __uint_as_float(rr[e + 5]) * mul);
            v4.w = pack_bf16x2(__uint_as_float(rr[e + 6]) * mul, __uint_as_float(rr[e + 7]) * mul);
            const int col = c * 32 + e;
            if (rowwise) {
              if (!row_dead) *reinterpret_cast<uint4*>(grow + col) = v4;
            } else {
              *reinterpret_cast<uint4*>(dst + (col >> 6) * C::KV_CHUNK + sw128_offset(r, col & 63)) = v4;
            }
          }
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, C::DS_THREADS);
    if (ok && !rowwise && threadIdx.x == 64) {
      for (int c = 0; c < C::KCH; ++c) {
        tma_store_3d(&p.tdk, sK + c * C::KV_CHUNK, c * 64, y1(k0), y2(k_beg, k0));
        tma_store_3d(&p.tdv, sV + c * C::KV_CHUNK, c * 64, y1(k0), y2(k_beg, k0));
      }
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  } else if (warp == 14) {
    // ------------------------------------------------------------------ helper
    // Each wait of the MMA thread costs the tensor core a bubble (even a completed mbarrier wait
    // keeps the issuing thread ~150 cycles, and the queue ahead of it is short).  The MMA
    // thread therefore waits only on p_ready and ds_ready; this thread folds the other
    // conditions into them: stage i+1 loaded (needed by S/dP_{i+1}, issued after dV_i) and the
    // dQ TMEM buffer of step i drained (needed by dQ_i).  It arrives on phase i of each barrier
    // only after phase i-1 has completed, so its arrival cannot count for an earlier phase.
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; ok && i < n; ++i) {
        // st_full phase i: stage i loaded, dS^T buffer i & 1 free (dK, dQ of step i-2 done)
        if (!(ok = mbar_wait(&stage_full[i % C::NST], (i / C::NST) & 1, abort_flag, 244))) break;
        if (i >= 2 && !(ok = mbar_wait(D == 128 ? &pds_free[i & 1] : &dqs_done[i & 1], ((i >> 1) - 1) & 1,
                                       abort_flag, 245)))
          break;
        if (i > 0 && !(ok = mbar_wait(st_full, (i - 1) & 1, abort_flag, 246))) break;
        mbar_arrive(st_full);
        if (i + 1 < n &&
            !(ok = mbar_wait(&stage_full[(i + 1) % C::NST], ((i + 1) / C::NST) & 1, abort_flag, 240)))
          break;
        if (i > 0 && !(ok = mbar_wait(p_ready, (i - 1) & 1, abort_flag, 241))) break;
        mbar_arrive(p_ready);
        if (i >= 2 && !(ok = mbar_wait(&dq_free[i & 1], ((i >> 1) - 1) & 1, abort_flag, 242))) break;
        if (i > 0 && !(ok = mbar_wait(ds_ready, (i - 1) & 1, abort_flag, 243))) break;
        mbar_arrive(ds_ready);
      }
    }
  } else {
    // ------------------------------------------------------------------ dQ warpgroup
    const int sub = warp & 3;
    const int rr_ = sub * 32 + lane;               // TMEM lane: d (d=128) or query (d=64)
    const uint32_t t_lane = static_cast<uint32_t>(sub * 32) << 16;
    if constexpr (D == 128) {
      // lane = d, columns = queries.  Each step's tile goes TMEM -> registers (the TMEM buffer
      // is released at once) -> a row-major [BM][d] fp32 box in shared memory -> one TMA
      // reduce-add into dQ_acc, issued by one thread; the L2 performs the fp32 adds.
      float* stg = reinterpret_cast<float*>(smem + C::OFF_DQS);
      const bool leader = threadIdx.x == 320;
      uint32_t use = 0;                              // dqs_sync phases used so far
      for (int i = 0; i < n; ++i) {
        const int q0 = step_q0(i);
        const int qb = i & 1;
        if (!mbar_wait_warp(&dq_full[qb], (i >> 1) & 1, abort_flag, 231)) break;
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(tbase + t_lane + C::T_DQ + qb * 64, v[0]);
        tmem_ld32(tbase + t_lane + C::T_DQ + qb * 64 + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&dq_free[qb]);
        // the previous reduce must have finished reading the staging box
        if (leader && i > 0) bulk_wait_group_read0();
        if (!warps_sync(dqs_sync, use++ & 1, abort_flag, 232)) break;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) stg[(c * 32 + e) * D + rr_] = __uint_as_float(v[c][e]);
        fence_proxy_async_smem();
        if (!warps_sync(dqs_sync, use++ & 1, abort_flag, 233)) break;
        // rows past the sequence's end hold zeros (their P, hence dS, is 0): adding them to
        // whatever follows is harmless, and rows past the tensor are clipped
        if (leader) {
          tma_reduce_add_3d(&p.tdq, stg, 0, VL ? head : q0, VL ? q_beg + q0 : bh);
          bulk_commit_group();
        }
      }
      // the staging box must stay readable until the last reduce has read it; its adds into
      // the accumulator complete on their own (as a TMA store's writes do)
      if (leader) bulk_wait_group_read0();
    } else {
      // lane = query, columns = d.  The tile is staged in the step's dS^T buffer, free once the
      // step's dK and dQ products are done (dq_full) until the dS warps write step i+2 into it
      // (the helper holds them until the staging has been read: dqs_done), as fp32 rows in the
      // 128-byte-swizzled layout of two [128 x 32] TMA boxes (conflict-free 16-byte writes),
      // then added into dQ_acc by two TMA reduce-adds issued by one thread.
      const bool leader = threadIdx.x == 320;
      uint32_t use = 0;
      for (int i = 0; i < n; ++i) {
        const int q0 = step_q0(i);
        const int qb = i & 1;
        if (!mbar_wait_warp(&dq_full[qb], (i >> 1) & 1, abort_flag, 231)) break;
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(tbase + t_lane + C::T_DQ + qb * 64, v[0]);
        tmem_ld32(tbase + t_lane + C::T_DQ + qb * 64 + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&dq_free[qb]);
        uint8_t* stg = sDS + (i & 1) * C::DS_TILE;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(stg + h * (C::BM * 128) + rr_ * 128 + ((c ^ (rr_ & 7)) << 4)) =
                make_float4(__uint_as_float(v[h][4 * c]), __uint_as_float(v[h][4 * c + 1]),
                            __uint_as_float(v[h][4 * c + 2]), __uint_as_float(v[h][4 * c + 3]));
        fence_proxy_async_smem();
        if (!warps_sync(dqs_sync, use++ & 1, abort_flag, 234)) break;
        if (leader) {
          // rows past the sequence's end hold zeros (their P, hence dS, is 0); rows past the
          // tensor are clipped
          for (int h = 0; h < 2; ++h)
            tma_reduce_add_3d(&p.tdq, stg + h * (C::BM * 128), h * 32, VL ? head : q0, VL ? q_beg + q0 : bh);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&dqs_done[i & 1]);
        }
      }
      if (leader) bulk_wait_group_read0();
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------------
// F3 persistent variant for short heads at d = 64: one CTA per SM walks (head, key tile) items,
// rank-major (every head's first key tile, then every head's second, ...; with causal the
// longest first) in zig-zag rounds of the grid, and runs the roles of bwd_main_kernel across
// item boundaries.  Each mbarrier phase counts the CTA's steps (or items) from its start.  The
// producer streams the next item's Q/dO stages while the current item finishes; K is
// double-buffered by item and V reloaded as soon as the item's last dP product is done (it is
// brought into L2 beforehand); the next item's first S product follows the last dV product,
// its dP product the last dK/dQ products; and the dQ warpgroup, not the dS warps, reads dK/dV
// out of TMEM after the item's last product and stores them row by row while the dS warps go
// on with the next item.  Per (key tile, query step) the arithmetic, the products and their
// order are those of bwd_main_kernel, so dK and dV agree with it bit for bit.  This removes
// the per-CTA start (barriers, TMEM, first loads) and the dK/dV epilogue from every item but
// the CTA's first and last, which is most of a short key tile's time.
// ------------------------------------------------------------------------------------------
// Key tiles per head up to which the persistent backward runs (d = 64).  Measured on GB300 with
// the L2 flushed before each call: at 4 key tiles (512 tokens) it is 8-10% faster than one CTA
// per key tile; at 8 it wins for causal heads (a GPT-2-medium layer, whose causal key tiles
// average 4.5 steps: 0.136 -> 0.130 ms) and loses 2% for unmasked ones; at 16 it is up to 15%
// slower: its steps run slower than bwd_main_kernel's (also when launched with one CTA per
// item), which outweighs the per-CTA start and epilogue it saves once items are longer than a
// few steps.
constexpr int kPersistentBwdMaxKvTiles = 4;
inline bool use_persistent_bwd(int n_kvtiles, bool causal) {
  return n_kvtiles <= (causal ? 2 * kPersistentBwdMaxKvTiles : kPersistentBwdMaxKvTiles);
}

struct BwdP64 {
  using B = BwdCfg<64>;
  static constexpr int D = 64, BN = B::BN, BM = B::BM, NST = B::NST, HALF = B::HALF;
  static constexpr int OFF_K = 0;                       // K of the CTA's items 2j and 2j+1
  static constexpr int OFF_V = 2 * B::KV_TILE;
  static constexpr int OFF_ST = 3 * B::KV_TILE;         // Q, dO ring
  static constexpr int OFF_DS = OFF_ST + NST * B::STAGE;
  static constexpr int OFF_SLOT = OFF_DS + 2 * B::DS_TILE;   // -lse / -D slots (bwd_main_kernel)
  static constexpr int OFF_BAR = OFF_SLOT + 8 * HALF * 4;
  // k_full[2], k_free[2], v_full, v_free, stage_full[NST], stage_empty[NST], st_full, dp_full,
  // p_ready, ds_ready, dq_full[2], dq_free[2], acc_full, acc_free, mma_done, dqs_sync,
  // dqs_done[2]
  static constexpr int NBAR = 6 + 2 * NST + 4 + 4 + 3 + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // TMEM slot, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(OFF_ST % 1024 == 0 && OFF_DS % 1024 == 0, "operands on 1 KB boundaries");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
};

// One work item of the persistent backward: key tile kt of plane bh and its query steps.
struct BwdItem {
  int bh, kt, i_start, n;
};

__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int item) {
  BwdItem it;
  const int n_bh = p.n_items / p.n_kvtiles;
  it.bh = item % n_bh;
  it.kt = item / n_bh;
  it.i_start = p.causal ? it.kt * (BwdP64::BN / BwdP64::BM) : 0;
  it.n = max(0, p.n_qtiles - it.i_start);
  return it;
}

__global__ void __launch_bounds__(BwdCfg<64>::THREADS, 1)
bwd_persistent_kernel64(const __grid_constant__ BwdParams p) {
  using C = BwdP64;
  using B = BwdCfg<64>;
  constexpr int D = 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1k(smem_raw);
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sDS = smem + C::OFF_DS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bars;                 // [2] K of an item landed (one per K buffer)
  uint64_t* k_free = k_full + 2;           // [2] the item's last product reading K is done
  uint64_t* v_full = k_free + 2;
  uint64_t* v_free = v_full + 1;           // the item's last dP product is done
  uint64_t* stage_full = v_free + 1;
  uint64_t* stage_empty = stage_full + C::NST;
  uint64_t* st_full = stage_empty + C::NST;
  uint64_t* dp_full = st_full + 1;
  uint64_t* p_ready = dp_full + 1;
  uint64_t* ds_ready = p_ready + 1;
  uint64_t* dq_full = ds_ready + 1;        // [2]
  uint64_t* dq_free = dq_full + 2;         // [2]
  uint64_t* acc_full = dq_free + 2;        // dK, dV of the item complete in TMEM
  uint64_t* acc_free = acc_full + 1;       // ... and read out (the next item may overwrite)
  uint64_t* mma_done = acc_free + 1;
  uint64_t* dqs_sync = mma_done + 1;       // the four dQ warps around the staging
  uint64_t* dqs_done = dqs_sync + 1;       // [2] dQ staged in dS^T buffer b read by the TMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  // the CTA's next item with work, from its c-th on; c moves past it (n = 0: none left)
  auto next_work = [&](int& c) -> BwdItem {
    for (;; ++c) {
      const int item = pers_item(c, G);
      if (item >= p.n_items) return BwdItem{0, 0, 0, 0};
      const BwdItem it = bwd_item(p, item);
      if (it.n > 0) {
        ++c;
        return it;
      }
    }
  };
  auto stage_ptr = [&](int s) { return smem + C::OFF_ST + s * B::STAGE; };

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&k_free[b], 1);
      mbar_init(&dq_full[b], 1);
      mbar_init(&dq_free[b], 128);
    }
    mbar_init(v_full, 1);
    mbar_init(v_free, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&stage_full[s], 1);      // TMA bytes
      mbar_init(&stage_empty[s], 1);
    }
    mbar_init(st_full, 2);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, B::DS_THREADS + 1);
    mbar_init(ds_ready, B::DS_THREADS + 1);
    mbar_init(acc_full, 1);
    mbar_init(acc_free, 128);
    mbar_init(mma_done, 1);
    mbar_init(dqs_sync, 4);
    mbar_init(&dqs_done[0], 1);
    mbar_init(&dqs_done[1], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
    tma_prefetch_desc(&p.tdo);
  }
  if (warp == 1) tmem_alloc(tmem_slot, B::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    int g = 0, j = 0, issued = 0, n_kld[2] = {0, 0}, n_vld = 0;
    bool ok = true;
    for (int c = 0; ok;) {
      const BwdItem it = next_work(c);
      if (it.n == 0) break;
      const int kb = j & 1;
      const int k0 = it.kt * C::BN;
      // K of item j into buffer j & 1, free once item j - 2's last products are done
      if (j >= 2 && !(ok = mbar_wait_warp(&k_free[kb], ((j >> 1) - 1) & 1, abort_flag, 301))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&k_full[kb], B::KV_TILE);
        tma_load_3d(sK + kb * B::KV_TILE, &p.tk, &k_full[kb], 0, k0, it.bh);
        if (j > 0) tma_prefetch_l2_3d(&p.tv, 0, k0, it.bh);
      }
      ++n_kld[kb];
      for (int i = 0; i < it.n; ++i, ++g) {
        const int s = g % C::NST;
        const uint32_t u = g / C::NST;
        if (u > 0 && !(ok = mbar_wait_warp(&stage_empty[s], (u - 1) & 1, abort_flag, 303))) break;
        uint8_t* st = stage_ptr(s);
        const int q0 = (it.i_start + i) * C::BM;
        if (lane == 0) {
          mbar_arrive_expect_tx(&stage_full[s], 2 * B::Q_TILE);
          tma_load_3d(st, &p.tq, &stage_full[s], 0, q0, it.bh);
          tma_load_3d(st + B::Q_TILE, &p.tdo, &stage_full[s], 0, q0, it.bh);
        }
        issued = g + 1;
        if (i == 0) {
          // V of item j, once item j - 1's last dP product is done with the buffer
          if (j >= 1 && !(ok = mbar_wait_warp(v_free, (j - 1) & 1, abort_flag, 302))) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(v_full, B::KV_TILE);
            tma_load_3d(sV, &p.tv, v_full, 0, k0, it.bh);
          }
          ++n_vld;
        }
      }
      ++j;
    }
    if (!ok && lane == 0) {
      // loads still in flight land in this CTA's shared memory: let them finish first
      for (int b = 0; b < 2; ++b)
        if (n_kld[b] > 0) mbar_wait(&k_full[b], (n_kld[b] - 1) & 1, nullptr, 304);
      if (n_vld > 0) mbar_wait(v_full, (n_vld - 1) & 1, nullptr, 305);
      for (int g2 = max(0, issued - C::NST); g2 < issued; ++g2)
        mbar_wait(&stage_full[g2 % C::NST], (g2 / C::NST) & 1, nullptr, 306);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // one thread issues (measured: the GPT-2-medium layer backward 125 us, 135 us when the
    // converged warp issues)
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, C::BM, 0, 0);
      const uint32_t id_acc = idesc_bf16_f32(128, D, 0, 1);
      const uint32_t id_dq = idesc_bf16_f32(128, 64, 1, 1);
      const uint64_t dK_k = smem_desc_sw128(smem_u32(sK), 0, 1024);
      const uint64_t dV_k = smem_desc_sw128(smem_u32(sV), 0, 1024);
      const uint64_t dK_mn = smem_desc_sw128(smem_u32(sK), B::KV_CHUNK, 1024);
      const uint64_t dDS = smem_desc_sw128(smem_u32(sDS), 0, 1024);
      const uint64_t dDS_mn = smem_desc_sw128(smem_u32(sDS), B::KV_CHUNK, 1024);
      const uint64_t dST_k = smem_desc_sw128(smem_u32(stage_ptr(0)), 0, 1024);
      const uint64_t dST_mn = smem_desc_sw128(smem_u32(stage_ptr(0)), B::Q_CHUNK, 1024);
      auto issue_s = [&](int g, int kb) {
        const uint64_t q_k = desc_advance(dST_k, (g % C::NST) * B::STAGE);
        const uint64_t k_k = desc_advance(dK_k, kb * B::KV_TILE);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ss(tbase + B::T_S, desc_advance(k_k, ks * 32), desc_advance(q_k, ks * 32), id_s, ks > 0);
        umma_commit(st_full);
      };
      auto issue_dp = [&](int g, bool item_last) {
        const uint64_t do_k = desc_advance(dST_k, (g % C::NST) * B::STAGE + B::Q_TILE);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ss(tbase + B::T_DP, desc_advance(dV_k, ks * 32), desc_advance(do_k, ks * 32), id_s, ks > 0);
        umma_commit(dp_full);
        if (item_last) umma_commit(v_free);
      };
      int c = 0;
      BwdItem cur = next_work(c);
      bool ok = true;
      if (cur.n > 0) {
        ok = mbar_wait(&k_full[0], 0, abort_flag, 311) && mbar_wait(v_full, 0, abort_flag, 312) &&
             mbar_wait(&stage_full[0], 0, abort_flag, 313);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
          issue_dp(0, cur.n == 1);
        }
      }
      unsigned long long steps = 0;
      int g = 0;
      for (int j = 0; ok && cur.n > 0; ++j) {
        const BwdItem nxt = next_work(c);
        const int kb = j & 1;
        const uint64_t k_mn = desc_advance(dK_mn, kb * B::KV_TILE);
        for (int i = 0; i < cur.n; ++i, ++g) {
          const int s = g % C::NST;
          // p_ready(g) folds in: stage g+1 loaded, the next item's K (at its boundary), and
          // dK/dV of the previous item read out (at an item's first step)
          if (!(ok = mbar_wait(p_ready, g & 1, abort_flag, 315))) break;
          tc_fence_after();
          const uint64_t q_mn = desc_advance(dST_mn, s * B::STAGE);
          const uint64_t do_mn = desc_advance(dST_mn, s * B::STAGE + B::Q_TILE);
#pragma unroll
          for (int ks = 0; ks < C::BM / 16; ++ks)       // dV += P^T dO
            umma_ts(tbase + B::T_DV, tbase + B::T_S + ks * 8 + ((16 * ks) / C::HALF) * (C::HALF / 2),
                    desc_advance(do_mn, ks * 2048), id_acc, (i > 0 || ks > 0) ? 1u : 0u);
          if (i + 1 < cur.n) {
            issue_s(g + 1, kb);
            issue_dp(g + 1, i + 2 == cur.n);
          } else if (nxt.n > 0) {
            issue_s(g + 1, kb ^ 1);                     // dP of the next item after dK/dQ below
          }
          if (!(ok = mbar_wait(ds_ready, g & 1, abort_flag, 318))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < C::BM / 16; ++ks) {     // dK += dS^T Q
            const uint32_t a_off = (ks >> 2) * B::KV_CHUNK + (ks & 3) * 32;
            umma_ss(tbase + B::T_DK, desc_advance(dDS, (g & 1) * B::DS_TILE + a_off),
                    desc_advance(q_mn, ks * 2048), id_acc, (i > 0 || ks > 0) ? 1u : 0u);
          }
          const int qb = g & 1;
#pragma unroll
          for (int ks = 0; ks < C::BN / 16; ++ks)       // dQ = dS K
            umma_ss(tbase + B::T_DQ + qb * 64, desc_advance(dDS_mn, (g & 1) * B::DS_TILE + ks * 2048),
                    desc_advance(k_mn, ks * 2048), id_dq, ks > 0);
          umma_commit(&dq_full[qb]);
          umma_commit(&stage_empty[s]);
          ++steps;
          if (i + 1 == cur.n) {
            umma_commit(&k_free[kb]);
            umma_commit(acc_full);
            if (nxt.n > 0) {
              // the next item's V: reloaded once this item's last dP product was done
              if (!(ok = mbar_wait(v_full, (j + 1) & 1, abort_flag, 319))) break;
              tc_fence_after();
              issue_dp(g + 1, nxt.n == 1);
            }
          }
        }
        cur = nxt;
      }
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, nullptr, 317);
      if (ok && p.stats != nullptr) atomicAdd(&p.stats[1], steps);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------------ dS warpgroups
    // (the step of bwd_main_kernel without window or block mask)
    const int sub = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int cb = grp * C::HALF;
    const int r = sub * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(sub * 32) << 16;
    const float c2 = p.scale_log2;
    const float2 c2v = make_float2(c2, c2);
    bool ok = true;
    int g = 0;
    for (int c = 0; ok;) {
      const BwdItem it = next_work(c);
      if (it.n == 0) break;
      const int k0 = it.kt * C::BN;
      const int k_idx = k0 + r;
      const bool row_dead = k_idx >= p.n_kv;
      for (int i = 0; i < it.n; ++i, ++g) {
        const int q0 = (it.i_start + i) * C::BM;
        // -lse (log2 units) and -D of the step's query columns, loaded from global memory before
        // the wait for S (see bwd_main_kernel)
        auto nlse_of = [&](int q) -> float {
          return (q < p.n_q) ? -__ldg(p.lse + static_cast<size_t>(it.bh) * p.n_q + q) * 1.4426950408889634f
                             : -INFINITY;
        };
        auto nd_of = [&](int q) -> float {
          return (q < p.n_q) ? -__ldg(p.delta + static_cast<size_t>(it.bh) * p.n_q + q) : 0.f;
        };
        float lane_nd[C::HALF / 32], nl0[32];
        const float lane_nl = nlse_of(q0 + cb + lane);
        lane_nd[0] = nd_of(q0 + cb + lane);
        if (!(ok = mbar_wait_warp(st_full, g & 1, abort_flag, 321))) break;
        tc_fence_after();
        // -lse, then -D, pass to the whole warp through its slot (as in bwd_main_kernel)
        float* slot = reinterpret_cast<float*>(smem + C::OFF_SLOT) + (warp - 2) * C::HALF;
        slot[lane] = lane_nl;
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 v = *reinterpret_cast<const float4*>(slot + e);
          nl0[e] = v.x; nl0[e + 1] = v.y; nl0[e + 2] = v.z; nl0[e + 3] = v.w;
        }
        const bool diag = p.causal && (q0 < k0 + C::BN - 1);
        uint32_t pk_ds[C::HALF / 2];
        uint32_t ppk[C::HALF / 2];                   // P as bf16 pairs (see bwd_main_kernel)
        uint32_t dpu[C::HALF / 32][32];
#pragma unroll
        for (int cc = 0; cc < C::HALF / 32; ++cc) {
          uint32_t rs[32];
          tmem_ld32(tbase + t_lane + B::T_S + cb + cc * 32, rs);
          float nl[32];
          if (cc == 0) {
#pragma unroll
            for (int e = 0; e < 32; ++e) nl[e] = nl0[e];
          } else {
            slot[cc * 32 + lane] = nlse_of(q0 + cb + cc * 32 + lane);
            lane_nd[cc] = nd_of(q0 + cb + cc * 32 + lane);
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 v = *reinterpret_cast<const float4*>(slot + cc * 32 + e);
              nl[e] = v.x; nl[e + 1] = v.y; nl[e + 2] = v.z; nl[e + 3] = v.w;
            }
          }
          tmem_wait_ld();
          uint32_t pk_p[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = cb + cc * 32 + e;
            const float2 x = ffma2(make_float2(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2v,
                                   make_float2(nl[e], nl[e + 1]));
            float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
            if (row_dead || (diag && k_idx > q0 + col)) p0 = 0.f;
            if (row_dead || (diag && k_idx > q0 + col + 1)) p1 = 0.f;
            pk_p[e / 2] = pack_bf16x2(p0, p1);
            ppk[cc * 16 + e / 2] = pk_p[e / 2];
          }
          tmem_st16(tbase + t_lane + B::T_S + cb + cc * 16, pk_p);
        }
        if (!(ok = mbar_wait_warp(dp_full, g & 1, abort_flag, 324))) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < C::HALF / 32; ++cc) tmem_ld32(tbase + t_lane + B::T_DP + cb + cc * 32, dpu[cc]);
        tmem_wait_ld();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_ready);
        __syncwarp();                              // the slot now passes -D
#pragma unroll
        for (int cc = 0; cc < C::HALF / 32; ++cc) slot[cc * 32 + lane] = lane_nd[cc];
        __syncwarp();
#pragma unroll
        for (int e = 0; e < C::HALF; e += 2) {
          const float2 dp = make_float2(__uint_as_float(dpu[e / 32][e % 32]), __uint_as_float(dpu[e / 32][e % 32 + 1]));
          const float2 nd = *reinterpret_cast<const float2*>(slot + e);
          const float2 pp = make_float2(__uint_as_float(ppk[e / 2] << 16), __uint_as_float(ppk[e / 2] & 0xffff0000u));
          const float2 ds = fmul2(pp, fadd2(dp, nd));
          pk_ds[e / 2] = pack_bf16x2(ds.x, ds.y);
        }
        uint8_t* sDSi = sDS + (g & 1) * B::DS_TILE;
#pragma unroll
        for (int u = 0; u < C::HALF / 8; ++u) {
          const int c8 = cb / 8 + u;
          const uint32_t off = (c8 >> 3) * B::KV_CHUNK + sw128_offset(r, (c8 & 7) * 8);
          *reinterpret_cast<uint4*>(sDSi + off) =
              make_uint4(pk_ds[4 * u], pk_ds[4 * u + 1], pk_ds[4 * u + 2], pk_ds[4 * u + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(ds_ready);
      }
    }
  } else if (warp == 14) {
    // ------------------------------------------------------------------ helper
    // As in bwd_main_kernel, plus the item boundaries: p_ready of an item's last step also
    // waits for the next item's K (its first S product follows that step's dV), and p_ready of
    // an item's first step for the previous item's dK/dV to be read out of TMEM (that step's
    // dV and dK products start the accumulators afresh).
    if (lane == 0) {
      int c = 0, g = 0;
      BwdItem cur = next_work(c);
      bool ok = cur.n == 0 || mbar_wait(&k_full[0], 0, abort_flag, 340);
      for (int j = 0; ok && cur.n > 0; ++j) {
        const BwdItem nxt = next_work(c);
        for (int i = 0; i < cur.n; ++i, ++g) {
          const bool last = i + 1 == cur.n;
          const bool more = !last || nxt.n > 0;
          if (!(ok = mbar_wait(&stage_full[g % C::NST], (g / C::NST) & 1, abort_flag, 344))) break;
          if (g >= 2 && !(ok = mbar_wait(&dqs_done[g & 1], ((g >> 1) - 1) & 1, abort_flag, 345))) break;
          if (g > 0 && !(ok = mbar_wait(st_full, (g - 1) & 1, abort_flag, 346))) break;
          mbar_arrive(st_full);
          if (more && !(ok = mbar_wait(&stage_full[(g + 1) % C::NST], ((g + 1) / C::NST) & 1, abort_flag, 341)))
            break;
          if (last && nxt.n > 0 && !(ok = mbar_wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, abort_flag, 347)))
            break;
          if (i == 0 && j > 0 && !(ok = mbar_wait(acc_free, (j - 1) & 1, abort_flag, 348))) break;
          if (g > 0 && !(ok = mbar_wait(p_ready, (g - 1) & 1, abort_flag, 342))) break;
          mbar_arrive(p_ready);
          if (g >= 2 && !(ok = mbar_wait(&dq_free[g & 1], ((g >> 1) - 1) & 1, abort_flag, 343))) break;
          if (g > 0 && !(ok = mbar_wait(ds_ready, (g - 1) & 1, abort_flag, 349))) break;
          mbar_arrive(ds_ready);
        }
        cur = nxt;
      }
    }
  } else {
    // ------------------------------------------------------------------ dQ warpgroup
    // Per step: dQ (lane = query, columns = d) from TMEM into the fp32 accumulator, staged in the
    // step's dS^T buffer and added by two TMA reduce-adds (as in bwd_main_kernel at d = 64).
    // Per item, once its last products are done: first dK (times scale) and dV
    // (lane = key row) out of TMEM and the accumulators released (the next item's first dV
    // product waits for that), stored row by row as bf16 (zeros for a key tile no query sees);
    // then the last step's dQ.
    const int sub = warp & 3;
    const int rr_ = sub * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(sub * 32) << 16;
    const bool leader = threadIdx.x == 320;
    uint32_t use = 0;                                // dqs_sync phases used so far
    bool ok = true;
    int g = 0, j = 0;
    auto store_dk_dv = [&](const BwdItem& it) {
      const int k_idx = it.kt * C::BN + rr_;
      const bool live = k_idx < p.n_kv;
      const size_t row = (static_cast<size_t>(it.bh) * p.n_kv + (live ? k_idx : 0)) * D;
#pragma unroll
      for (int t = 0; t < 2; ++t) {                // dV, then dK (times scale)
        const float mul = t ? p.scale : 1.f;
        uint4* dst = reinterpret_cast<uint4*>((t ? p.dk : p.dv) + row);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t v[32];
          if (it.n > 0) {
            tmem_ld32(tbase + t_lane + (t ? B::T_DK : B::T_DV) + cc * 32, v);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            pk[e / 2] = pack_bf16x2(__uint_as_float(v[e]) * mul, __uint_as_float(v[e + 1]) * mul);
          if (live) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[cc * 4 + u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
      }
    };
    for (int c = 0; ok; ++c) {
      const int item = pers_item(c, G);
      if (item >= p.n_items) break;
      const BwdItem it = bwd_item(p, item);
      if (it.n == 0) store_dk_dv(it);
      for (int i = 0; i < it.n; ++i, ++g) {
        const int q0 = (it.i_start + i) * C::BM;
        const int qb = g & 1;
        if (i + 1 == it.n) {
          // acc_full(j) is committed after this step's dQ product: it covers dq_full too
          if (!(ok = mbar_wait_warp(acc_full, j & 1, abort_flag, 332))) break;
          tc_fence_after();
          store_dk_dv(it);
          tc_fence_before();
          mbar_arrive(acc_free);
          ++j;
        }
        if (!(ok = mbar_wait_warp(&dq_full[qb], (g >> 1) & 1, abort_flag, 331))) break;
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(tbase + t_lane + B::T_DQ + qb * 64, v[0]);
        tmem_ld32(tbase + t_lane + B::T_DQ + qb * 64 + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&dq_free[qb]);
        uint8_t* stg = sDS + (g & 1) * B::DS_TILE;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<float4*>(stg + h * (C::BM * 128) + rr_ * 128 + ((cc ^ (rr_ & 7)) << 4)) =
                make_float4(__uint_as_float(v[h][4 * cc]), __uint_as_float(v[h][4 * cc + 1]),
                            __uint_as_float(v[h][4 * cc + 2]), __uint_as_float(v[h][4 * cc + 3]));
        fence_proxy_async_smem();
        if (!(ok = warps_sync(dqs_sync, use++ & 1, abort_flag, 333))) break;
        if (leader) {
          for (int h = 0; h < 2; ++h) tma_reduce_add_3d(&p.tdq, stg + h * (C::BM * 128), h * 32, q0, it.bh);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&dqs_done[g & 1]);
        }
      }
    }
    if (leader) bulk_wait_group_read0();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, B::TMEM_COLS);
  }
}

// F2: D = rowsum(dO o O) (fp32) and zero the dQ accumulator.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                      const uint16_t* __restrict__ dO,
                                                      float* __restrict__ delta,
                                                      float4* __restrict__ dq_acc4,
                                                      long long rows, int vl_heads) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
  constexpr int TPR = D / 8;                        // threads per row, 8 bf16 each
  static_assert(D / 4 == 2 * TPR, "a thread clears two float4 of its row's accumulator");
  constexpr int RPW = 32 / TPR;                     // rows per warp and pass
  const int lane = threadIdx.x & 31;
  const int part = lane % TPR;
  const long long ngrp = nthr / TPR;
  // warp-uniform trip count so the shuffles below always see all 32 lanes
  for (long long r0 = (tid >> 5) * RPW; r0 < rows; r0 += ngrp) {
    const long long row = r0 + lane / TPR;
    const bool valid = row < rows;
    float s = 0.f;
    if (valid) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + part);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dO + row * D) + part);
      // the row's fp32 dQ accumulator is cleared beside the reads: one mixed read/write stream
      // instead of a write-only pass and then a read-only pass (4x32x4096x128: 93 against 107 us)
      float4* z = dq_acc4 + row * (D / 4) + part * 2;
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s = fmaf(__uint_as_float(aa[e] << 16), __uint_as_float(bb[e] << 16), s);
        s = fmaf(__uint_as_float(aa[e] & 0xffff0000u), __uint_as_float(bb[e] & 0xffff0000u), s);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    // packed variable-length rows (token * H + head) go head-major (head * total + token), the
    // order in which the main kernel's dS warps read a query tile's D (as they read lse)
    if (valid && part == 0) delta[vl_heads > 0 ? (row % vl_heads) * (rows / vl_heads) + row / vl_heads : row] = s;
  }
}

// F4: dq = bf16(scale * dQ_acc)
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                             uint2* __restrict__ dq, float scale,
                                                             long long n4) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long x = tid; x < n4; x += nthr) {
    const float4 v = acc[x];
    dq[x] = make_uint2(pack_bf16x2(v.x * scale, v.y * scale), pack_bf16x2(v.z * scale, v.w * scale));
  }
}

template <int D>
static cudaError_t launch_bwd_prep_d(const BwdArgs& a, cudaStream_t stream) {
  const uint64_t bh = static_cast<uint64_t>(a.B) * a.H;
  const long long rows = static_cast<long long>(bh) * a.n_q;
  if (rows == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long long>(152LL * 8, (rows * (D / 8) + 255) / 256));
  log_launch("bwd_pre_kernel<D>", static_cast<unsigned long long>(std::max(blocks, 1)), 256, static_cast<unsigned long long>(0));
  bwd_pre_kernel<D><<<std::max(blocks, 1), 256, 0, stream>>>(
      static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dO), a.delta,
      reinterpret_cast<float4*>(a.dq_acc), rows, a.cu_q != nullptr ? a.H : 0);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_bwd_main_d(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  if (a.n_kv == 0) return cudaSuccess;
  const uint64_t bh = static_cast<uint64_t>(a.B) * a.H;
  BwdParams p;
  const uint64_t nq = a.n_q > 0 ? a.n_q : 1;
  const void* qb = a.n_q > 0 ? a.q : a.k;
  const void* dob = a.n_q > 0 ? a.dO : a.k;
  if (!make_map_f32_3d(&p.tdq, a.dq_acc, D, nq, bh, D * 4, D * 4 * nq, D == 128 ? D : 32, C::BM, 1, D == 64) ||
      !make_map_bf16_3d(&p.tq, qb, D, nq, bh, 64, C::BM) ||
      !make_map_bf16_3d(&p.tdo, dob, D, nq, bh, 64, C::BM) ||
      !make_map_bf16_3d(&p.tk, a.k, D, a.n_kv, bh, 64, C::BN) ||
      !make_map_bf16_3d(&p.tv, a.v, D, a.n_kv, bh, 64, C::BN) ||
      !make_map_bf16_3d(&p.tdk, a.dk, D, a.n_kv, bh, 64, C::BN) ||
      !make_map_bf16_3d(&p.tdv, a.dv, D, a.n_kv, bh, 64, C::BN))
    return cudaErrorInvalidValue;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq_acc = a.dq_acc;
  p.n_q = a.n_q;
  p.n_kv = a.n_kv;
  p.n_qtiles = (a.n_q + C::BM - 1) / C::BM;
  p.n_kvtiles = (a.n_kv + C::BN - 1) / C::BN;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.heads = a.H;
  p.total_q = p.total_k = p.max_q = p.max_k = 0;
  p.cu_q = p.cu_k = nullptr;
  p.dk = static_cast<uint16_t*>(a.dk);
  p.dv = static_cast<uint16_t*>(a.dv);
  p.stats = debug_counters();
  attention_window(a.causal, a.windowed, a.win_left, a.win_right, &p.win_left, &p.win_right);
  p.block_mask = a.block_mask;
  p.bm_per_head = a.bm_per_head;
  p.n_qblocks = (a.n_q + kBlockSize - 1) / kBlockSize;
  p.n_items = 0;
  static int attr_done[64] = {0};   // one per instantiation of this launcher
  const uint64_t grid = static_cast<uint64_t>(p.n_kvtiles) * bh;
  if (a.block_mask != nullptr) {
    static int attr_bs[64] = {0};
    cudaError_t e = ensure_smem_attr(bwd_main_kernel<D, false, false, true>, C::SMEM_BYTES, attr_bs);
    if (e != cudaSuccess) return e;
    log_launch("bwd_main_kernel<D, false, false, true>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
    bwd_main_kernel<D, false, false, true><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
  }
  if constexpr (D == 64) {
    if (!a.windowed && use_persistent_bwd(p.n_kvtiles, a.causal != 0)) {
      static int attr_p[64] = {0};
      cudaError_t e = ensure_smem_attr(bwd_persistent_kernel64, BwdP64::SMEM_BYTES, attr_p);
      if (e != cudaSuccess) return e;
      int dev = 0, sms = 0;
      if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
      if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
      p.n_items = static_cast<int>(grid);
      const unsigned ctas = static_cast<unsigned>(std::min<uint64_t>(grid, static_cast<uint64_t>(std::max(sms, 1))));
      log_launch("bwd_persistent_kernel64", static_cast<unsigned long long>(ctas), C::THREADS, static_cast<unsigned long long>(BwdP64::SMEM_BYTES));
      bwd_persistent_kernel64<<<ctas, C::THREADS, BwdP64::SMEM_BYTES, stream>>>(p);
      return cudaGetLastError();
    }
  }
  if (a.windowed) {
    static int attr_win[64] = {0};
    cudaError_t e = ensure_smem_attr(bwd_main_kernel<D, false, true>, C::SMEM_BYTES, attr_win);
    if (e != cudaSuccess) return e;
    log_launch("bwd_main_kernel<D, false, true>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
    bwd_main_kernel<D, false, true><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
  }
  cudaError_t e = ensure_smem_attr(bwd_main_kernel<D, false>, C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  log_launch("bwd_main_kernel<D, false>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
  bwd_main_kernel<D, false><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

// Variable-length main kernel: packed [total, H, d] tensors, cu_seqlens boundaries.
template <int D>
static cudaError_t launch_bwd_main_varlen_d(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  if (a.total_k == 0 || a.max_seqlen_k == 0) return cudaSuccess;
  BwdParams p;
  const int tq = a.total_q > 0 ? a.total_q : 1;
  const void* qb = a.total_q > 0 ? a.q : a.k;
  const void* dob = a.total_q > 0 ? a.dO : a.k;
  if (!make_map_f32_3d(&p.tdq, a.dq_acc, D, a.H, tq, D * 4, static_cast<uint64_t>(D) * 4 * a.H,
                       D == 128 ? D : 32, 1, C::BM, D == 64) ||
      !make_map_bf16_tok(&p.tq, qb, D, a.H, tq, 64, C::BM) ||
      !make_map_bf16_tok(&p.tdo, dob, D, a.H, tq, 64, C::BM) ||
      !make_map_bf16_tok(&p.tk, a.k, D, a.H, a.total_k, 64, C::BN) ||
      !make_map_bf16_tok(&p.tv, a.v, D, a.H, a.total_k, 64, C::BN) ||
      !make_map_bf16_tok(&p.tdk, a.dk, D, a.H, a.total_k, 64, C::BN) ||
      !make_map_bf16_tok(&p.tdv, a.dv, D, a.H, a.total_k, 64, C::BN))
    return cudaErrorInvalidValue;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq_acc = a.dq_acc;
  p.n_q = p.n_kv = 0;
  p.n_qtiles = 0;
  p.n_kvtiles = (a.max_seqlen_k + C::BN - 1) / C::BN;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.heads = a.H;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.max_q = a.max_seqlen_q;
  p.max_k = a.max_seqlen_k;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.dk = static_cast<uint16_t*>(a.dk);
  p.dv = static_cast<uint16_t*>(a.dv);
  p.stats = debug_counters();
  attention_window(a.causal, false, 0, 0, &p.win_left, &p.win_right);
  p.block_mask = nullptr;
  p.bm_per_head = p.n_qblocks = 0;
  p.n_items = 0;
  static int attr_done[64] = {0};
  cudaError_t e = ensure_smem_attr(bwd_main_kernel<D, true>, C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const uint64_t grid = static_cast<uint64_t>(p.n_kvtiles) * a.n_seqs * a.H;
  log_launch("bwd_main_kernel<D, true>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
  bwd_main_kernel<D, true><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_bwd_finish_d(const BwdArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.n_q;
  if (rows == 0) return cudaSuccess;
  const long long n4 = rows * D / 4;
  const int blocks = static_cast<int>(std::min<long long>(152LL * 8, (n4 + 255) / 256));
  log_launch("bwd_dq_convert_kernel", static_cast<unsigned long long>(std::max(blocks, 1)), 256, static_cast<unsigned long long>(0));
  bwd_dq_convert_kernel<<<std::max(blocks, 1), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(a.dq_acc), static_cast<uint2*>(a.dq), a.scale, n4);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t s) {
  return a.d == 64 ? launch_bwd_prep_d<64>(a, s) : launch_bwd_prep_d<128>(a, s);
}
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t s) {
  if (a.cu_q) return a.d == 64 ? launch_bwd_main_varlen_d<64>(a, s) : launch_bwd_main_varlen_d<128>(a, s);
  return a.d == 64 ? launch_bwd_main_d<64>(a, s) : launch_bwd_main_d<128>(a, s);
}
cudaError_t launch_bwd_finish(const BwdArgs& a, cudaStream_t s) {
  return a.d == 64 ? launch_bwd_finish_d<64>(a, s) : launch_bwd_finish_d<128>(a, s);
}

}  // namespace fa

FA_DEFINE_STATUS_FETCH(status_fetch_bwd)
