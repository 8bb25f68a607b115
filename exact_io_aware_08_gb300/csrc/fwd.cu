// F1: attention forward on sm_103a.
//
// Follows "FlashAttention and online softmax" (ML Systems lesson 4), section 3 "The tiled
// forward pass" and "The online softmax theorem": a query tile stays on chip, 128-key tiles of
// K and V stream past it, and each row carries its state (m, l, o~) across tiles, dividing once
// at the end (the FlashAttention-2 form, "Keep o~ unnormalised").  Causal tiles above the
// diagonal are skipped and the diagonal tile is masked ("Causal masks").
//
// GB300 mapping.  One CTA (384 threads, one per SM) owns TWO 128-row query tiles of a head,
// which share every K/V tile loaded into shared memory:
//   warp 0      TMA producer: Q_0, Q_1 once, then K_j and V_j through NS-deep rings.
//   warp 1      TMEM owner and MMA issuer, the whole warp converged with one elected lane
//               issuing (tcgen05.mma kind::f16, fp32 in TMEM):
//                 S_t = Q_t K_j^T          A, B from shared memory (both K-major)
//                 O_t += P_t V_j           A = P_t from TMEM, B = V_j from shared memory
//               in the order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so the tensor core works
//               on one tile while the other tile's softmax runs.
//   warp 2      helper: folds "V_j loaded" and "K_{j+1} loaded" into the P hand-off (named barrier
//               BAR_P + t, mbarrier p_full[t] under a block mask), so
//               the MMA thread waits once per tile and key tile (each wait of the issuing thread
//               costs the tensor core a bubble).  Warp 3 is idle (warpgroup 0 gives up registers
//               with setmaxnreg).
//   warps 4-7   softmax of tile 0, warps 8-11 softmax of tile 1: thread = query row.  A thread
//               loads its S row from TMEM, updates (m, l) in the log2 domain (scale * log2 e
//               folded into one FMA), writes P as bf16 back over its S row in TMEM (P never
//               touches shared memory), and rescales its O row in TMEM when needed.  The
//               epilogue divides by l, stores O through TMA and writes lse = m + ln l.
// TMEM (512 columns): S_0, S_1 (128 each; P_t overwrites the first 64 columns of S_t),
// O_0, O_1 (d each).  An S_t product is issued after the PV_t product that reads P_t from the
// same columns; tcgen05.mma operations of one thread execute in issue order.
//
// Variants (template flags): VL -- packed variable-length batches (one work item per sequence,
// head and 256-row block); F8 -- e4m3 Q, K, V (tcgen05.mma kind::f8f6f4, K = 32 per
// instruction, P stored as e4m3 four per TMEM column over the first 32 columns of S_t); WIN --
// a sliding window (each query tile streams only the key tiles its rows can see); BS -- a block
// mask (the CTA streams the union of its two query tiles' set key blocks, each tile computes
// only its own).  Short heads (use_persistent) run on fwd_persistent_kernel (below), which
// walks several work items per CTA.
//
// Rescaling.  The online-softmax theorem holds for ANY reference value that l and o~ share:
// o~/l is unchanged when both are measured against a stale maximum.  So a row moves its
// reference m to the new running max only when the max grew by more than 2^8 (exp2 units);
// otherwise it keeps m, and its weights 2^{s - m} stay <= 256 (exact in fp32, no overflow).
// This skips most O corrections (a published FlashAttention-4 technique); the first tile
// always sets m.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {

template <int D, bool F8 = false>
struct FwdCfg {
  static_assert(!F8 || D == 128, "the fp8 forward is built for d = 128");
  static constexpr int EB = F8 ? 1 : 2;               // bytes per Q/K/V element
  static constexpr int BM = 128;                      // rows per query tile (2 tiles per CTA)
  static constexpr int BN = 128;                      // keys per K/V tile
  static constexpr int KCH = D * EB / 128;            // 128-byte chunks per Q/K/V row
  static constexpr int XCH = 128 / EB;                // elements per chunk (TMA x step)
  static constexpr int TILE = 128 * D * EB;           // bytes of one 128-row Q/K/V tile
  static constexpr int CHUNK = 128 * 128;             // bytes of one [128 rows x 128 B] chunk
  static constexpr int OCH = D / 64;                  // 64-column chunks of a bf16 O row
  static constexpr int OTILE = 128 * D * 2;           // bytes of one 128-row bf16 O tile
  static constexpr int NS = F8 ? 3 : ((D == 128) ? 2 : 4);   // K ring and V ring depth
  static constexpr int KS_S = D * EB / 32;            // 32-byte k-steps of S = Q K^T
  static constexpr int KS_PV = BN * EB / 32;          // 32-byte k-steps of O += P V
  static constexpr int PV_B_STEP = (32 / EB) * 128;   // V bytes per PV k-step (32/EB key rows)
  static constexpr int OFF_Q = 0;                     // Q_0, Q_1 (bf16: later O staging)
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  // O staging: the dead Q tiles when they are as large as O tiles (bf16), else its own space
  static constexpr int OFF_OST = F8 ? OFF_V + NS * TILE : OFF_Q;
  // d = 64: O_t carries 16 more columns, which the PV product fills against a block of ones
  // placed right after the V ring, so that they hold sum_j bf16(p_j), O's normaliser, formed
  // on the tensor core (and rescaled with O) instead of by the softmax threads.  d = 128 has no
  // TMEM left for them.
  static constexpr bool LB_MMA = D == 64 && !F8;
  static constexpr int DO = LB_MMA ? D + 16 : D;      // TMEM columns of O_t
  static constexpr int OFF_ONES = OFF_V + NS * TILE;  // [128 keys x 64 columns], LB_MMA only
  static constexpr int OFF_BAR = F8 ? OFF_OST + 2 * OTILE : OFF_ONES + (LB_MMA ? CHUNK : 0);
  // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full[2], o_done[2]
  static constexpr int NBAR = 1 + 4 * NS + 6;
  // TMEM slot, abort flag, block-sparse stream length and live counts of the two query tiles
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // block-sparse: the CTA's key-tile stream (int16 indices) and which query tile wants each
  static constexpr int OFF_BSL = OFF_MISC + 32;
  static constexpr int OFF_BSB = OFF_BSL + 2 * kBlockSparseMaxTiles;
  static constexpr int SMEM_BYTES = OFF_BSB + kBlockSparseMaxTiles + 1024;   // + 1 KB alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0;                  // S_t at columns [128 t, 128 t + 128)
  static constexpr uint32_t T_O = 256;                // O_t at columns [256 + DO t, ...)
  static_assert(T_O + 2 * DO <= TMEM_COLS, "TMEM budget");
  static constexpr int THREADS = 384;
  // setmaxnreg split: launched with 168 per thread (384 x 168 = 64512); warpgroup 0 (producer,
  // MMA) drops to 80, the two softmax warpgroups rise to 208: 128*80 + 2*128*208 = 63488.
  static constexpr uint32_t REG_CTRL = 80;
  static constexpr uint32_t REG_SOFTMAX = 208;
  // Weights are 2^{(s - m) c2 + P_BIAS} with m at most RESCALE_THRESHOLD (log2 units) below
  // the row's running max, so they stay <= 2^{P_BIAS + RESCALE_THRESHOLD} = 256: exact in fp32
  // for bf16; for e4m3 (largest finite 448) the bias lifts small weights out of the subnormal
  // range (e4m3 is normal down to 2^-6).
  static constexpr float RESCALE_THRESHOLD = F8 ? 4.f : 8.f;
  static constexpr float P_BIAS = F8 ? 4.f : 0.f;
  // The P hand-off of tile t as named barrier BAR_P + t (one generation per P V product: the
  // tile's 128 softmax threads arrive, the MMA and helper warps sync).  An mbarrier wait costs
  // the issuing warp ~150 cycles even when the phase is complete; the hardware barrier does
  // not.  Used by the fp8 forward (measured 0.59 -> 0.56 ms) and by the plain bf16 one (with
  // the products issued by the converged warp: 4x32x4096x128 724 -> 716 us, causal 423 -> 416
  // us; with one issuing thread it had been slower), the varlen one (2.54 -> 2.49 ms on 16
  // causal sequences of 512-8192 tokens) and the windowed one.  The block-sparse
  // instantiation, whose tiles skip steps, keeps the mbarrier, whose waits are bounded.
  static constexpr uint32_t BAR_P = 3;
  static constexpr uint32_t BAR_P_THREADS = 128 + 32 + 32;
};

// The normaliser block of a d = 64 forward: a [128 keys x 64 columns] bf16 tile, in the
// 128-byte-swizzled layout of a V tile, whose first 16 columns are 1 and the rest 0.  Written by
// the whole CTA before its first __syncthreads and made visible to the tensor core.
__device__ __forceinline__ void fill_ones_block(uint8_t* blk) {
  const uint4 ones = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int row = i >> 3, unit = i & 7;            // 16-byte unit (8 columns) of the row
    *reinterpret_cast<uint4*>(blk + sw128_offset(row, unit * 8)) = (unit < 2) ? ones : zero;
  }
  fence_proxy_async_smem();
}

// B operand of O_t += P_t [V_j | 1] at d = 64: V_j's 64 columns at v_addr + off, and the next
// 64-column chunk (of which the product reads 16) at the normaliser block ones_off bytes after
// v_addr: the chunk stride (leading byte offset) is whatever separates the two.
__device__ __forceinline__ uint64_t v_desc_ones(uint32_t v_addr, uint32_t off, uint32_t ones_off) {
  return smem_desc_sw128(v_addr + off, ones_off - off, 1024);
}

// Registers the setmaxnreg split of a forward configuration needs: warpgroup 0 at REG_CTRL,
// the two softmax warpgroups at REG_SOFTMAX.
template <typename Cfg>
constexpr int reg_split_need() {
  return 128 * static_cast<int>(Cfg::REG_CTRL) + 256 * static_cast<int>(Cfg::REG_SOFTMAX);
}

struct FwdParams {
  CUtensorMap tq, tk, tv, to;
  float* lse;
  int n_q, n_kv, n_qpairs, n_kvtiles, causal;
  float scale, scale_log2;
  // Variable-length batches: packed token-major [total, H, d] tensors, sequence s occupying
  // rows [cu_q[s], cu_q[s+1]) (queries) and [cu_k[s], cu_k[s+1]) (keys); lse is [H, total_q].
  int heads, total_q;
  const int* cu_q;
  const int* cu_k;
  uint16_t* o;                                        // for row-wise stores of a partial tile
  // FP8: scale = tau * s_q * s_k (the score scale of the raw code products); O is multiplied by
  // out_scale = s_v.  bf16: out_scale = 1.
  float out_scale;
  // Visible keys of query i: i - win_left <= j <= i + win_right (kWinUnbounded = no bound on
  // that side).  Causal is (kWinUnbounded, 0), no mask (kWinUnbounded, kWinUnbounded).
  int win_left, win_right;
  // Block-sparse: 0/1 per (128-query block, 128-key block) pair, [n_qblocks][n_kvtiles] for
  // every head (bm_per_head = 0) or one such array per (b, h) plane.
  const uint8_t* block_mask;
  int bm_per_head, n_qblocks;
  int n_items;                                        // persistent forward: B*H*n_qpairs
  unsigned long long* stats;                          // diagnostic counters (see fa_kernels.h)
};

template <int D, bool VL, bool F8 = false, bool WIN = false, bool BS = false>
__global__ void __launch_bounds__(FwdCfg<D, F8>::THREADS, 1)
fwd_kernel(const __grid_constant__ FwdParams p) {
  // the P hand-off by named barrier (FwdCfg::BAR_P), except under a block mask
  constexpr bool NAMED_P = F8 || !BS;
  using C = FwdCfg<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1k(smem_raw);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* v_full = k_empty + C::NS;
  uint64_t* v_empty = v_full + C::NS;
  uint64_t* s_full = v_empty + C::NS;      // [2]
  uint64_t* p_full = s_full + 2;           // [2]
  uint64_t* o_done = p_full + 2;           // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: query rows [256 c, 256 c + 256) of head bh.  Items of one head are adjacent so
  // the CTAs that run together share K/V in L2; causal items run longest-first across groups
  // of kCausalGroup heads.
  // Variable-length: item = (sequence, head, 256-row block), sized by the longest sequence;
  // blocks past a sequence's end exit at once.  Rows are then local to the sequence.
  // Under a block mask every head's rank-0 item runs first, then every head's rank 1, ...: the
  // work of an item is its rows' set blocks, so the heads' longest items start together instead
  // of the last head group's starting late (as in the block-sparse backward).
  int bh = blockIdx.x / p.n_qpairs;                   // fixed length: (b, h) plane
  int r = blockIdx.x % p.n_qpairs;
  if (BS) {
    bh = blockIdx.x % (gridDim.x / p.n_qpairs);
    r = blockIdx.x / (gridDim.x / p.n_qpairs);
  } else if (!VL && !WIN && p.causal) {
    causal_item(blockIdx.x, gridDim.x / p.n_qpairs, p.n_qpairs, &bh, &r);
  }
  int n_q = p.n_q, n_kv = p.n_kv, q_beg = 0, k_beg = 0, head = 0;
  if (VL) {
    const int seq = bh / p.heads;
    head = bh % p.heads;
    q_beg = p.cu_q[seq];
    n_q = p.cu_q[seq + 1] - q_beg;
    k_beg = p.cu_k[seq];
    n_kv = p.cu_k[seq + 1] - k_beg;
    // Boundaries come from the caller's device arrays: check them here, so bad ones become a
    // reported error instead of out-of-range rows (p.n_q = max_seqlen_q, p.n_kv = total_k).
    if (q_beg < 0 || n_q < 0 || q_beg + n_q > p.total_q || n_q > p.n_q || k_beg < 0 || n_kv < 0 ||
        k_beg + n_kv > p.n_kv) {
      if (threadIdx.x == 0 && r == 0) report_device_error(FA_DEV_BAD_CONFIG, 150);
      return;
    }
  }
  const int n_qpairs = (n_q + 2 * C::BM - 1) / (2 * C::BM);
  if (r >= n_qpairs) return;                          // whole CTA, before any shared state
  const int n_kvtiles = (n_kv + C::BN - 1) / C::BN;
  const int c = p.causal ? (n_qpairs - 1 - r) : r;
  // Key tiles of query tile t: [lo_t, lo_t + n_t[t]) -- every tile holding a key that some row
  // of the tile sees; tiles entirely outside every row's window are skipped, never loaded
  // ("Causal masks": the same skipping serves sliding windows).  The CTA streams the union
  // [j0, j0 + n_max) once (the two ranges overlap: both tiles see their diagonals), so tile t
  // starts at position off[t] of that stream.
  int q0[2], n_t[2], off[2], lo[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    q0[t] = c * 2 * C::BM + t * C::BM;
    if constexpr (WIN) {
      const int first_key = max(0, q0[t] - p.win_left);
      const int last_key = min(n_kv - 1, q0[t] + C::BM - 1 + min(p.win_right, kWinUnbounded - C::BM));
      lo[t] = first_key / C::BN;
      const int hi = (last_key < first_key) ? lo[t] : min(n_kvtiles, last_key / C::BN + 1);
      n_t[t] = (q0[t] >= n_q) ? 0 : hi - lo[t];
    } else {                                          // causal or no mask: from key tile 0
      lo[t] = 0;
      n_t[t] = (q0[t] >= n_q) ? 0 : (p.causal ? min(2 * c + t + 1, n_kvtiles) : n_kvtiles);
    }
  }
  const int j0 = WIN ? lo[0] : 0;
  int n_max = WIN ? ((n_t[1] > 0) ? lo[1] + n_t[1] - j0 : n_t[0]) : max(n_t[0], n_t[1]);
  off[0] = 0;
  off[1] = lo[1] - j0;
  // TMA coordinates of local row ``row``: fixed length {x, row, (b,h)}; packed {x, h, beg+row}
  auto y1 = [&](int row) { return VL ? head : row; };
  auto y2 = [&](int beg, int row) { return VL ? beg + row : bh; };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 129);         // the tile's 128 softmax threads + the helper
      mbar_init(&o_done[t], 1);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
    tma_prefetch_desc(&p.to);
  }
  if constexpr (C::LB_MMA) fill_ones_block(smem + C::OFF_ONES);
  // Block-sparse: the CTA streams the key tiles either query tile wants (the union of its two
  // mask rows, in order; with causal only tiles up to the diagonal), once.  Both tiles run
  // every streamed tile; a tile whose block is not set masks it whole (P = 0).
  int16_t* s_bsl = reinterpret_cast<int16_t*>(smem + C::OFF_BSL);
  uint8_t* s_bsb = smem + C::OFF_BSB;
  if constexpr (BS) {
    if (warp == 3) {
      const bool a0 = q0[0] < n_q, a1 = q0[1] < n_q;
      const int qb0 = q0[0] / C::BM, qb1 = a1 ? q0[1] / C::BM : qb0;
      const size_t plane = static_cast<size_t>(p.bm_per_head ? bh : 0) * p.n_qblocks;
      const uint8_t* r0 = p.block_mask + (plane + qb0) * n_kvtiles;
      const uint8_t* r1 = p.block_mask + (plane + qb1) * n_kvtiles;
      int cnt = 0, live0 = 0, live1 = 0;
      for (int base = 0; base < n_kvtiles; base += 32) {
        const int kt = base + lane;
        uint32_t b = 0;
        if (kt < n_kvtiles) {
          if (a0 && r0[kt] != 0 && (!p.causal || kt <= qb0)) b |= 1u;
          if (a1 && r1[kt] != 0 && (!p.causal || kt <= qb1)) b |= 2u;
        }
        live0 += __popc(__ballot_sync(0xffffffffu, (b & 1u) != 0u));
        live1 += __popc(__ballot_sync(0xffffffffu, (b & 2u) != 0u));
        const uint32_t bal = __ballot_sync(0xffffffffu, b != 0u);
        if (b != 0u) {
          const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
          s_bsl[pos] = static_cast<int16_t>(kt);
          s_bsb[pos] = static_cast<uint8_t>(b);
        }
        cnt += __popc(bal);
      }
      if (lane == 0) {
        volatile int* nb = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
        nb[0] = cnt;
        nb[1] = live0;                             // live blocks of each query tile
        nb[2] = live1;
      }
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // block-sparse: n_max stream positions; tile t runs only its n_t[t] live ones (a clear block
  // is neither computed nor waited for)
  auto live = [&](int t, int j) { return ((s_bsb[j] >> t) & 1u) != 0u; };
  if constexpr (BS) {
    const volatile int* nb = reinterpret_cast<const volatile int*>(smem + C::OFF_MISC + 8);
    n_max = nb[0];
    n_t[0] = nb[1];
    n_t[1] = nb[2];
  }
  if (warp < 4) {
  setmaxnreg_dec<C::REG_CTRL>();   // warpgroup 0: producer, MMA issuer, two idle warps
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && n_max > 0) {
      int issued = 0;
      // Q_t only for a tile with work: a tile without any (block-sparse: no set block) writes
      // its O = 0 through the staging area at once, which for bf16 is its Q buffer
      mbar_arrive_expect_tx(q_full, ((n_t[0] > 0) + (n_t[1] > 0)) * C::TILE);
      for (int t = 0; t < 2; ++t)
        if (n_t[t] > 0)
          for (int k = 0; k < C::KCH; ++k)
            tma_load_3d(sQ + t * C::TILE + k * C::CHUNK, &p.tq, q_full, k * C::XCH, y1(q0[t]), y2(q_beg, q0[t]));
      for (int j = 0; j < n_max; ++j) {               // stream position j = key tile j0 + j
        const int s = j % C::NS;
        const uint32_t u = j / C::NS;
        const int key = (BS ? s_bsl[j] : j0 + j) * C::BN;
        if (u > 0 && !mbar_wait(&k_empty[s], (u - 1) & 1, abort_flag, 101)) break;
        mbar_arrive_expect_tx(&k_full[s], C::TILE);
        for (int k = 0; k < C::KCH; ++k)
          tma_load_3d(sK + s * C::TILE + k * C::CHUNK, &p.tk, &k_full[s], k * C::XCH, y1(key), y2(k_beg, key));
        if (u > 0 && !mbar_wait(&v_empty[s], (u - 1) & 1, abort_flag, 102)) break;
        mbar_arrive_expect_tx(&v_full[s], C::TILE);
        for (int k = 0; k < C::KCH; ++k)
          tma_load_3d(sV + s * C::TILE + k * C::CHUNK, &p.tv, &v_full[s], k * C::XCH, y1(key), y2(k_beg, key));
        issued = j + 1;
      }
      if (*abort_flag) {
        // Drain: let every copy this thread started land before the CTA exits.
        mbar_wait(q_full, 0, nullptr, 103);
        for (int j = max(0, issued - C::NS); j < issued; ++j) {
          mbar_wait(&k_full[j % C::NS], (j / C::NS) & 1, nullptr, 104);
          mbar_wait(&v_full[j % C::NS], (j / C::NS) & 1, nullptr, 105);
        }
      }
    }
  } else if (NAMED_P && warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (named-barrier P hand-off)
    // The whole warp walks the loop (it takes part in the named-barrier hand-offs) and issues
    // (umma_*_w).  After a failed wait it keeps joining every hand-off, issuing nothing.
    if (n_max > 0) {
      const bool leader = lane == 0;
      // Q, K both K-major; P from TMEM, V MN-major
      const uint32_t idesc_s = F8 ? idesc_e4m3_f32(128, 128, 0, 0) : idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t idesc_o = F8 ? idesc_e4m3_f32(128, D, 0, 1) : idesc_bf16_f32(128, C::DO, 0, 1);
      // Descriptors are built once; each k-step adds a compile-time offset (desc_advance).
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 0, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 0, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), C::CHUNK, 1024);
      unsigned long long n_s = 0;                               // S products issued
      auto issue_s = [&](int t, int j) {                        // S_t = Q_t K_j^T
        ++n_s;
        const uint64_t a = desc_advance(dq0, t * C::TILE);
        const uint64_t b = desc_advance(dk0, (j % C::NS) * C::TILE);
        const uint32_t d_tmem = tbase + C::T_S + t * 128;
#pragma unroll
        for (int ks = 0; ks < C::KS_S; ++ks) {
          const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
          if constexpr (F8)
            umma_ss_f8_w(d_tmem, desc_advance(a, off), desc_advance(b, off), idesc_s, ks > 0);
          else
            umma_ss_w(d_tmem, desc_advance(a, off), desc_advance(b, off), idesc_s, ks > 0);
        }
        umma_commit_w(&s_full[t]);
      };
      auto issue_pv = [&](int t, int j, bool first) {           // O_t += P_t V_j
        const uint64_t b = C::LB_MMA ? v_desc_ones(smem_u32(sV), (j % C::NS) * C::TILE, C::NS * C::TILE)
                                     : desc_advance(dv0, (j % C::NS) * C::TILE);
        const uint32_t d_tmem = tbase + C::T_O + t * C::DO;
        const uint32_t a_tmem = tbase + C::T_S + t * 128;
#pragma unroll
        for (int ks = 0; ks < C::KS_PV; ++ks) {
          if constexpr (F8)
            umma_ts_f8_w(d_tmem, a_tmem + ks * 8, desc_advance(b, ks * C::PV_B_STEP), idesc_o,
                       (!first || ks > 0) ? 1u : 0u);
          else
            umma_ts_w(d_tmem, a_tmem + ks * 8, desc_advance(b, ks * C::PV_B_STEP), idesc_o,
                    (!first || ks > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait_warp(q_full, 0, abort_flag, 111) && mbar_wait_warp(&k_full[0], 0, abort_flag, 112);
      if (ok) {
        tc_fence_after();
        if (n_t[0] > 0) issue_s(0, 0);
        if (n_t[1] > 0 && (!WIN || off[1] == 0)) issue_s(1, 0);
        umma_commit_w(&k_empty[0]);
      }
      // stream position j; tile t is on its i-th key tile, i = j - off[t]
      for (int j = 0; j < n_max; ++j) {
        const int s = j % C::NS;
        // V_j and K_{j+1} are loaded: the helper checked them before joining the hand-off
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int i = WIN ? j - off[t] : j;       // without a window both tiles start at 0
          if ((!WIN || i >= 0) && i < n_t[t]) {
            __syncwarp();
            named_bar_sync(C::BAR_P + t, C::BAR_P_THREADS);
            if (ok) {
              tc_fence_after();
              issue_pv(t, j, i == 0);
              if (i + 1 == n_t[t]) umma_commit_w(&o_done[t]);
            }
          }
          if (ok && (!WIN || i + 1 >= 0) && i + 1 < n_t[t]) issue_s(t, j + 1);
        }
        if (ok) {
          umma_commit_w(&v_empty[s]);
          if (j + 1 < n_max) umma_commit_w(&k_empty[(j + 1) % C::NS]);
        }
      }
      if (leader && p.stats != nullptr) atomicAdd(&p.stats[0], n_s);
    }
  } else if (NAMED_P && warp == 2) {
    // ------------------------------------------------------------------ helper (named-barrier P hand-off)
    // Joins each P hand-off once V_j (and K_{j+1}, if an S(j+1) follows) is loaded, so the MMA
    // warp's single wait per hand-off also covers the loads.  The whole warp takes part; after
    // a failed wait it keeps joining every remaining hand-off.
    if (n_max > 0) {
      bool ok = true;
      for (int j = 0; j < n_max; ++j) {
        bool k_next = false;                         // does some tile need S(j+1)?
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int i = WIN ? j - off[t] : j;
          k_next |= (!WIN || i + 1 >= 0) && i + 1 < n_t[t];
        }
        if (ok) ok = mbar_wait_warp(&v_full[j % C::NS], (j / C::NS) & 1, abort_flag, 130);
        if (ok && k_next) ok = mbar_wait_warp(&k_full[(j + 1) % C::NS], ((j + 1) / C::NS) & 1, abort_flag, 131);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int i = WIN ? j - off[t] : j;
          if ((!WIN || i >= 0) && i < n_t[t]) {
            __syncwarp();
            named_bar_sync(C::BAR_P + t, C::BAR_P_THREADS);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (n_max > 0) {                               // the whole warp (umma_*_w)
      // Q, K both K-major; P from TMEM, V MN-major
      const uint32_t idesc_s = F8 ? idesc_e4m3_f32(128, 128, 0, 0) : idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t idesc_o = F8 ? idesc_e4m3_f32(128, D, 0, 1) : idesc_bf16_f32(128, C::DO, 0, 1);
      // Descriptors are built once; each k-step adds a compile-time offset (desc_advance).
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 0, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 0, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), C::CHUNK, 1024);
      unsigned long long n_s = 0;                               // S products issued
      auto issue_s = [&](int t, int j) {                        // S_t = Q_t K_j^T
        ++n_s;
        const uint64_t a = desc_advance(dq0, t * C::TILE);
        const uint64_t b = desc_advance(dk0, (j % C::NS) * C::TILE);
        const uint32_t d_tmem = tbase + C::T_S + t * 128;
#pragma unroll
        for (int ks = 0; ks < C::KS_S; ++ks) {
          const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
          if constexpr (F8)
            umma_ss_f8_w(d_tmem, desc_advance(a, off), desc_advance(b, off), idesc_s, ks > 0);
          else
            umma_ss_w(d_tmem, desc_advance(a, off), desc_advance(b, off), idesc_s, ks > 0);
        }
        umma_commit_w(&s_full[t]);
      };
      auto issue_pv = [&](int t, int j, bool first) {           // O_t += P_t V_j
        const uint64_t b = C::LB_MMA ? v_desc_ones(smem_u32(sV), (j % C::NS) * C::TILE, C::NS * C::TILE)
                                     : desc_advance(dv0, (j % C::NS) * C::TILE);
        const uint32_t d_tmem = tbase + C::T_O + t * C::DO;
        const uint32_t a_tmem = tbase + C::T_S + t * 128;
#pragma unroll
        for (int ks = 0; ks < C::KS_PV; ++ks) {
          if constexpr (F8)
            umma_ts_f8_w(d_tmem, a_tmem + ks * 8, desc_advance(b, ks * C::PV_B_STEP), idesc_o,
                       (!first || ks > 0) ? 1u : 0u);
          else
            umma_ts_w(d_tmem, a_tmem + ks * 8, desc_advance(b, ks * C::PV_B_STEP), idesc_o,
                    (!first || ks > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait_warp(q_full, 0, abort_flag, 111) && mbar_wait_warp(&k_full[0], 0, abort_flag, 112);
      if constexpr (BS) {
        // Only live (tile, block) pairs are computed; cnt[t] counts tile t's live steps.  An
        // S_t(j+1) of a tile that is clear at j waits for the other tile's hand-off at j, which
        // vouches for K_{j+1} (the helper checked it).
        int cnt[2] = {0, 0};
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (live(t, 0)) issue_s(t, 0);
          umma_commit_w(&k_empty[0]);
        }
        for (int j = 0; ok && j < n_max; ++j) {
          const int s = j % C::NS;
          const bool nxt = j + 1 < n_max;
          bool waited = false;
          int deferred = -1;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (live(t, j)) {
              if (!(ok = mbar_wait_warp(&p_full[t], cnt[t] & 1, abort_flag, 115 + t))) break;
              tc_fence_after();
              waited = true;
              issue_pv(t, j, cnt[t] == 0);
              if (++cnt[t] == n_t[t]) umma_commit_w(&o_done[t]);
            }
            if (nxt && live(t, j + 1)) {
              if (waited) issue_s(t, j + 1);
              else deferred = t;
            }
          }
          if (!ok) break;
          if (deferred >= 0) issue_s(deferred, j + 1);
          umma_commit_w(&v_empty[s]);
          if (nxt) umma_commit_w(&k_empty[(j + 1) % C::NS]);
        }
      }
      if (!BS && ok) {
        tc_fence_after();
        if (n_t[0] > 0) issue_s(0, 0);
        if (n_t[1] > 0 && (!WIN || off[1] == 0)) issue_s(1, 0);
        umma_commit_w(&k_empty[0]);
      }
      // stream position j; tile t is on its i-th key tile, i = j - off[t]
      for (int j = 0; !BS && ok && j < n_max; ++j) {
        const int s = j % C::NS;
        // V_j and K_{j+1} are loaded: the helper checked them before its p_full arrival
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int i = WIN ? j - off[t] : j;       // without a window both tiles start at 0
          if ((!WIN || i >= 0) && i < n_t[t]) {
            if (!(ok = mbar_wait_warp(&p_full[t], i & 1, abort_flag, 115 + t))) break;
            tc_fence_after();
            issue_pv(t, j, i == 0);
            if (i + 1 == n_t[t]) umma_commit_w(&o_done[t]);
          }
          if ((!WIN || i + 1 >= 0) && i + 1 < n_t[t]) issue_s(t, j + 1);
        }
        if (!ok) break;
        umma_commit_w(&v_empty[s]);
        if (j + 1 < n_max) umma_commit_w(&k_empty[(j + 1) % C::NS]);
      }
      if (lane == 0 && p.stats != nullptr) atomicAdd(&p.stats[0], n_s);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ helper
    if (lane == 0 && n_max > 0) {
      bool ok = true;
      int cnt[2] = {0, 0};                           // block-sparse: live steps per tile
      for (int j = 0; ok && j < n_max; ++j) {
        if (!(ok = mbar_wait(&v_full[j % C::NS], (j / C::NS) & 1, abort_flag, 130))) break;
        bool k_next = BS && j + 1 < n_max;           // does some tile need S(j+1)?
#pragma unroll
        for (int t = 0; t < 2 && !BS; ++t) {
          const int i = WIN ? j - off[t] : j;
          k_next |= (!WIN || i + 1 >= 0) && i + 1 < n_t[t];
        }
        if (k_next && !(ok = mbar_wait(&k_full[(j + 1) % C::NS], ((j + 1) / C::NS) & 1, abort_flag, 131)))
          break;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int i = BS ? cnt[t] : (WIN ? j - off[t] : j);
          if (BS ? live(t, j) : ((!WIN || i >= 0) && i < n_t[t])) {
            if constexpr (BS) ++cnt[t];
            // arrive on phase i only once phase i-1 is complete
            if (i > 0 && !(ok = mbar_wait(&p_full[t], (i - 1) & 1, abort_flag, 132 + t))) break;
            mbar_arrive(&p_full[t]);
          }
        }
      }
    }
  }
  } else {
  setmaxnreg_inc<C::REG_SOFTMAX>();   // warpgroups 1 and 2: softmax of query tiles 0 and 1
  {
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = (warp - 4) >> 2;            // query tile of this warpgroup
    const int sub = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = sub * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t t_s = tbase + t_lane + C::T_S + t * 128;
    const uint32_t t_o = tbase + t_lane + C::T_O + t * C::DO;
    const int q0t = q0[t];                    // this warpgroup's tile, hoisted out of the arrays
    const int lo_t = WIN ? lo[t] : 0;
    const int q_idx = q0t + row;
    const int n = n_t[t];
    // this row's visible keys [key_lo, key_hi) under a window
    const int key_lo = WIN ? max(0, q_idx - p.win_left) : 0;
    const int key_hi = WIN ? min(n_kv, q_idx + 1 + min(p.win_right, kWinUnbounded - C::BM)) : 0;
    const float c2 = p.scale_log2;
    float m = -INFINITY;                      // reference max (raw dot-product units)
    float l = 0.f;                            // sum of 2^{(s - m) c2} over keys seen (fp32)
    float lb = 0.f;                           // the same sum over the bf16-rounded weights
    bool ok = true;
    int handed = 0;                           // fp8: P hand-offs joined so far

    int pos = 0;                              // block-sparse: stream position of step j
    for (int j = 0; j < n; ++j) {
      int jp = j;
      if constexpr (BS) {                       // next stream position this tile's block is set at
        while (pos < n_max - 1 && !live(t, pos)) ++pos;
        jp = pos++;
      }
      if (!(ok = mbar_wait_warp(&s_full[t], j & 1, abort_flag, 121))) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t rr[32];
        tmem_ld32(t_s + k * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[k * 32 + i] = __uint_as_float(rr[i]);
      }
      tmem_wait_ld();

      const int k0 = (BS ? s_bsl[jp] : lo_t + j) * C::BN;
      // a tile that some row of the query tile sees only in part (window edge, causal
      // diagonal, ragged end of the keys) is masked element by element
      if constexpr (WIN) {
        if (k0 + C::BN > n_kv || k0 + C::BN - 1 > q0t + min(p.win_right, kWinUnbounded - C::BM) ||
            k0 < q0t + C::BM - 1 - p.win_left) {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k0 + k < key_lo || k0 + k >= key_hi) s[k] = -INFINITY;
        }
      } else if (k0 + C::BN > n_kv || (p.causal && k0 + C::BN - 1 > q0t)) {
        const int lim = p.causal ? min(q_idx + 1, n_kv) : n_kv;   // keys < lim visible
#pragma unroll
        for (int k = 0; k < 128; ++k)
          if (k0 + k >= lim) s[k] = -INFINITY;
      }
      // row max: four independent 3-input-max chains, then combined
      float mq[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        mq[g] = fmax3(s[32 * g], s[32 * g + 1], s[32 * g + 2]);
#pragma unroll
        for (int k = 3; k < 31; k += 2) mq[g] = fmax3(mq[g], s[32 * g + k], s[32 * g + k + 1]);
        mq[g] = fmaxf(mq[g], s[32 * g + 31]);
      }
      const float mx = fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]);
      const float cand = fmaxf(m, mx);
      // (under a window or a block mask a row may miss a whole tile: cand = -inf, nothing to
      // move; otherwise every row sees a key of its first tile)
      const bool move = (!(WIN || BS) || cand != -INFINITY) &&
                        ((m == -INFINITY) || ((cand - m) * c2 > C::RESCALE_THRESHOLD));
      if (__any_sync(0xffffffffu, move)) {
        const float alpha = move ? fast_exp2((m - cand) * c2) : 1.f;  // 0 when m = -inf
        if (move) {
          l *= alpha;
          lb *= alpha;
          m = cand;
        }
        if (j > 0) {
          // O_t is settled: PV_t(j-1) completed before S_t(j) (same issuing thread, in order).
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            uint32_t rr[32];
            tmem_ld32(t_o + k * 32, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 v = fmul2(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])),
                                     make_float2(alpha, alpha));
              rr[i] = __float_as_uint(v.x);
              rr[i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(t_o + k * 32, rr);
          }
          if constexpr (C::LB_MMA) {            // the normaliser columns move with O
            uint32_t rr[16];
            tmem_ld16(t_o + D, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tmem_st16(t_o + D, rr);
          }
        }
      }
      const float ms = (m == -INFINITY) ? 0.f : m * c2 - C::P_BIAS;
      const float2 c2v = make_float2(c2, c2), nms = make_float2(-ms, -ms);
      float2 rs[4], rb[4];                      // independent partial sums (ILP)
#pragma unroll
      for (int g = 0; g < 4; ++g) rs[g] = rb[g] = make_float2(0.f, 0.f);
      if constexpr (F8) {
        // P as e4m3, four weights per column, over the first 32 columns of S_t.  O is
        // normalised by the fp32 sum l: e4m3 rounding (relative 2^-4, to nearest) of each
        // weight perturbs O by a zero-mean sum, bounded by 2^-4 sum_j p_j |v_j| / l.
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 x0 = ffma2(make_float2(s[4 * k], s[4 * k + 1]), c2v, nms);
          const float2 x1 = ffma2(make_float2(s[4 * k + 2], s[4 * k + 3]), c2v, nms);
          const float2 e0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
          const float2 e1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
          pk[k] = pack_e4m3x4(e0.x, e0.y, e1.x, e1.y);
          rs[k & 3] = fadd2(rs[k & 3], fadd2(e0, e1));
        }
        tmem_st32(t_s, pk);
      } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {             // P over the first 64 columns of S_t, 2 halves
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 x = ffma2(make_float2(s[64 * h + 2 * k], s[64 * h + 2 * k + 1]), c2v, nms);
          const float p0 = fast_exp2(x.x);
          const float p1 = fast_exp2(x.y);
          pk[k] = pack_bf16x2(p0, p1);
          rs[k & 3] = fadd2(rs[k & 3], make_float2(p0, p1));
          // lb sums the bf16 weights the PV product uses, so O / lb is an exact weighted
          // average of V under those weights; lse keeps the fp32 sum (d = 64: the tensor core
          // forms lb in O's normaliser columns)
          if constexpr (!C::LB_MMA) rb[k & 3] = add_bf16x2_f32(rb[k & 3], pk[k]);
        }
        tmem_st32(t_s + h * 32, pk);
      }
      }
      const float2 rs01 = fadd2(fadd2(rs[0], rs[1]), fadd2(rs[2], rs[3]));
      const float2 rb01 = fadd2(fadd2(rb[0], rb[1]), fadd2(rb[2], rb[3]));
      l += rs01.x + rs01.y;
      lb += rb01.x + rb01.y;
      tmem_wait_st();
      tc_fence_before();
      if constexpr (NAMED_P) {
        __syncwarp();
        named_bar_arrive(C::BAR_P + t, C::BAR_P_THREADS);
        ++handed;
      } else {
        mbar_arrive(&p_full[t]);
      }
    }
    // named-barrier hand-off, after an abort: keep joining the remaining ones (blocking, so
    // these arrivals cannot run ahead of a generation the MMA and helper warps have not
    // completed)
    if constexpr (NAMED_P) {
      for (; handed < n; ++handed) {
        __syncwarp();
        named_bar_sync(C::BAR_P + t, C::BAR_P_THREADS);
      }
    }

    // ------------------------------------------------------------------ epilogue
    if (ok && n > 0) {
      ok = mbar_wait_warp(&o_done[t], 0, abort_flag, 123);
      tc_fence_after();
    }
    uint8_t* stage = smem + C::OFF_OST + t * C::OTILE;   // bf16: Q_t, dead once o_done[t] fired
    // A packed tile that ends past its sequence is stored row by row (a TMA store of the
    // whole box would write into the next sequence's rows).
    const bool rowwise = VL && (q0[t] + C::BM > n_q);
    uint16_t* orow = rowwise ? p.o + (static_cast<size_t>(q_beg + q_idx) * p.heads + head) * D : nullptr;
    if (ok && q0[t] < n_q) {
      if constexpr (C::LB_MMA) {               // the normaliser: O_t's column d
        uint32_t rl[16];
        if (n > 0) {
          tmem_ld16(t_o + D, rl);
          tmem_wait_ld();
          lb = __uint_as_float(rl[0]);
        }
      }
      const float inv_l = F8 ? ((l > 0.f) ? p.out_scale / l : 0.f) : ((lb > 0.f) ? 1.f / lb : 0.f);
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        uint32_t rr[32];
        if (n > 0) {
          tmem_ld32(t_o + k * 32, rr);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 v4;
          v4.x = pack_bf16x2(__uint_as_float(rr[i + 0]) * inv_l, __uint_as_float(rr[i + 1]) * inv_l);
          v4.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * inv_l, __uint_as_float(rr[i + 3]) * inv_l);
          v4.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * inv_l, __uint_as_float(rr[i + 5]) * inv_l);
          v4.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * inv_l, __uint_as_float(rr[i + 7]) * inv_l);
          const int col = k * 32 + i;
          if (rowwise) {
            if (q_idx < n_q) *reinterpret_cast<uint4*>(orow + col) = v4;
          } else {
            *reinterpret_cast<uint4*>(stage + (col >> 6) * C::CHUNK + sw128_offset(row, col & 63)) = v4;
          }
        }
      }
      if (q_idx < n_q) {
        const size_t li = VL ? static_cast<size_t>(head) * p.total_q + q_beg + q_idx
                                   : static_cast<size_t>(bh) * n_q + q_idx;
        // l carries the factor 2^P_BIAS of the weights
        p.lse[li] = (l > 0.f) ? fmaf(m, p.scale, logf(l) - C::P_BIAS * 0.6931471805599453f) : -INFINITY;
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + t, 128);
    if (ok && !rowwise && q0[t] < n_q && (threadIdx.x & 127) == 64) {
      for (int k = 0; k < C::OCH; ++k)
        tma_store_3d(&p.to, stage + k * C::CHUNK, k * 64, y1(q0[t]), y2(q_beg, q0[t]));
      bulk_commit_group();
      bulk_wait_group_read0();
    }
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
// Persistent forward (plain bf16: no window, block mask, varlen or fp8).  One CTA per SM walks
// the work items (the same items as one CTA per item, taken longest first in rounds of
// gridDim.x, zig-zag: pers_item), so that one item's tail overlaps the next one's
// start: the next item's Q is loaded as soon as the current item's last S products complete,
// its first S products follow the last PV products, and the softmax warps store the finished
// item's O (through a staging buffer the two tiles take in turn) while the tensor core works.
// Every mbarrier phase is counted across items.  Roles, TMEM and the online softmax are those
// of fwd_kernel.
// ------------------------------------------------------------------------------------------
// Heads short enough for the persistent forward: it pays when a work item is a few tiles long
// (measured on GB300: up to 16 key tiles for causal heads, whose items average half the head,
// and for d = 64; up to 8 for unmasked d = 128, where at 16 it was 3% slower; up to 32 for
// causal d = 64, where 4x32x4096x64 ran in 324 instead of 341 us, while at 32 key tiles causal
// d = 128 was 4% slower).
constexpr int kPersistentMaxKvTiles = 16;
__host__ __device__ constexpr bool use_persistent(int d, bool causal, int n_kvtiles) {
  return n_kvtiles <= ((causal && d == 64) ? 2 * kPersistentMaxKvTiles
                       : (causal || d == 64) ? kPersistentMaxKvTiles : kPersistentMaxKvTiles / 2);
}

template <int D>
struct FwdPCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int KCH = D * 2 / 128;             // 128-byte chunks per bf16 row
  static constexpr int TILE = 128 * D * 2;            // one 128-row Q/K/V tile (bf16)
  static constexpr int CHUNK = 128 * 128;
  static constexpr int OCH = D / 64;
  static constexpr int NS = (D == 128) ? 2 : 4;
  static constexpr int KS_S = D / 16, KS_PV = BN / 16;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  // d = 64: O's normaliser columns against a block of ones right after the V ring (as fwd_kernel)
  static constexpr bool LB_MMA = D == 64;
  static constexpr int DO = LB_MMA ? D + 16 : D;      // TMEM columns of O_t
  static constexpr int OFF_ONES = OFF_V + NS * TILE;
  static constexpr int OFF_OST = OFF_ONES + (LB_MMA ? CHUNK : 0);   // one O tile of staging
  static constexpr int OFF_BAR = OFF_OST + TILE;
  // q_full, q_empty, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full[2],
  // o_done[2], o_free[2], st_free
  static constexpr int NBAR = 2 + 4 * NS + 9;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512, T_S = 0, T_O = 256;
  static constexpr int THREADS = 384;
  // setmaxnreg split (launched with 168 per thread: 64512): 128 x 88 + 256 x 200 = 62464.  The
  // item loop keeps more state live than fwd_kernel's; at 80 / 208 the control warps spilled.
  static constexpr uint32_t REG_CTRL = 88, REG_SOFTMAX = 200;
  static constexpr float RESCALE_THRESHOLD = 8.f;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
};

// One work item of the fixed-length forward: query rows [256 c, 256 c + 256) of plane bh, and
// the key tiles each of its two query tiles streams.
struct FwdItem {
  int bh, q0[2], n_t[2], n_max;
};

__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int item) {
  FwdItem it;
  // rank-major: every head's longest item (causal), then every head's second, ...; the short
  // heads this kernel serves keep all their K/V in L2 at once
  const int n_bh = p.n_items / p.n_qpairs;
  const int bh = item % n_bh, r = item / n_bh;
  const int c = p.causal ? (p.n_qpairs - 1 - r) : r;
  it.bh = bh;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    it.q0[t] = c * 256 + t * 128;
    it.n_t[t] = (it.q0[t] >= p.n_q) ? 0 : (p.causal ? min(2 * c + t + 1, p.n_kvtiles) : p.n_kvtiles);
  }
  it.n_max = max(it.n_t[0], it.n_t[1]);
  return it;
}

template <int D>
__global__ void __launch_bounds__(FwdPCfg<D>::THREADS, 1)
fwd_persistent_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdPCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1k(smem_raw);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sO = smem + C::OFF_OST;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* v_full = k_empty + C::NS;
  uint64_t* v_empty = v_full + C::NS;
  uint64_t* s_full = v_empty + C::NS;      // [2]
  uint64_t* p_full = s_full + 2;           // [2]
  uint64_t* o_done = p_full + 2;           // [2]
  uint64_t* o_free = o_done + 2;           // [2]: the tile's O read out of TMEM by its epilogue
  uint64_t* st_free = o_free + 2;          // the O staging buffer is free again
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 129);         // the tile's 128 softmax threads + the helper
      mbar_init(&o_done[t], 1);
      mbar_init(&o_free[t], 128);
    }
    mbar_init(st_free, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
    tma_prefetch_desc(&p.to);
  }
  if constexpr (C::LB_MMA) fill_ones_block(smem + C::OFF_ONES);
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp < 4) {
  setmaxnreg_dec<C::REG_CTRL>();
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t P = 0, issued = 0;             // stream positions over all items
      int nq = 0;                             // Q loads issued
      bool ok = true;
      for (int k = 0; ok && pers_item(k, G) < p.n_items; ++k) {
        const FwdItem it = fwd_item(p, pers_item(k, G));
        if (k > 0 && !(ok = mbar_wait(q_empty, (k - 1) & 1, abort_flag, 141))) break;
        mbar_arrive_expect_tx(q_full, ((it.n_t[0] > 0) + (it.n_t[1] > 0)) * C::TILE);
        for (int t = 0; t < 2; ++t)
          if (it.n_t[t] > 0)
            for (int c = 0; c < C::KCH; ++c)
              tma_load_3d(sQ + t * C::TILE + c * C::CHUNK, &p.tq, q_full, c * 64, it.q0[t], it.bh);
        nq = k + 1;
        for (int j = 0; j < it.n_max; ++j, ++P) {
          const int s = P % C::NS;
          const uint32_t u = P / C::NS;
          const int key = j * C::BN;
          if (u > 0 && !(ok = mbar_wait(&k_empty[s], (u - 1) & 1, abort_flag, 142))) break;
          mbar_arrive_expect_tx(&k_full[s], C::TILE);
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(sK + s * C::TILE + c * C::CHUNK, &p.tk, &k_full[s], c * 64, key, it.bh);
          if (u > 0 && !(ok = mbar_wait(&v_empty[s], (u - 1) & 1, abort_flag, 143))) break;
          mbar_arrive_expect_tx(&v_full[s], C::TILE);
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(sV + s * C::TILE + c * C::CHUNK, &p.tv, &v_full[s], c * 64, key, it.bh);
          issued = P + 1;
        }
      }
      if (*abort_flag) {
        // let every copy this thread started land before the CTA exits
        if (nq > 0) mbar_wait(q_full, (nq - 1) & 1, nullptr, 144);
        for (uint32_t q = issued > C::NS ? issued - C::NS : 0; q < issued; ++q) {
          mbar_wait(&k_full[q % C::NS], (q / C::NS) & 1, nullptr, 145);
          mbar_wait(&v_full[q % C::NS], (q / C::NS) & 1, nullptr, 146);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    {                                              // the whole warp (umma_*_w)
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t idesc_o = idesc_bf16_f32(128, C::DO, 0, 1);
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 0, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 0, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), C::CHUNK, 1024);
      unsigned long long n_s = 0;                              // S products issued
      auto issue_s = [&](int t, uint32_t P) {                  // S_t = Q_t K^T (position P)
        ++n_s;
        const uint64_t a = desc_advance(dq0, t * C::TILE);
        const uint64_t b = desc_advance(dk0, (P % C::NS) * C::TILE);
#pragma unroll
        for (int ks = 0; ks < C::KS_S; ++ks) {
          const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
          umma_ss_w(tbase + C::T_S + t * 128, desc_advance(a, off), desc_advance(b, off), idesc_s, ks > 0);
        }
        umma_commit_w(&s_full[t]);
      };
      auto issue_pv = [&](int t, uint32_t P, bool first) {     // O_t += P_t V (position P)
        const uint64_t b = C::LB_MMA ? v_desc_ones(smem_u32(sV), (P % C::NS) * C::TILE, C::NS * C::TILE)
                                     : desc_advance(dv0, (P % C::NS) * C::TILE);
#pragma unroll
        for (int ks = 0; ks < C::KS_PV; ++ks)
          umma_ts_w(tbase + C::T_O + t * C::DO, tbase + C::T_S + t * 128 + ks * 8,
                  desc_advance(b, ks * 16 * 128), idesc_o, (!first || ks > 0) ? 1u : 0u);
      };
      uint32_t P = 0, cp[2] = {0, 0}, act[2] = {0, 0};
      bool ok = true;
      for (int k = 0; ok && pers_item(k, G) < p.n_items; ++k) {
        const FwdItem it = fwd_item(p, pers_item(k, G));
        if (!(ok = mbar_wait_warp(q_full, k & 1, abort_flag, 151) &&
                   mbar_wait_warp(&k_full[P % C::NS], (P / C::NS) & 1, abort_flag, 152)))
          break;
        tc_fence_after();
        // the S columns are free: the previous item's last PV products were issued before
        for (int t = 0; t < 2; ++t)
          if (it.n_t[t] > 0) issue_s(t, P);
        umma_commit_w(&k_empty[P % C::NS]);
        if (it.n_max == 1) umma_commit_w(q_empty);
        for (int j = 0; ok && j < it.n_max; ++j) {
          const uint32_t Pj = P + j;
          // V_j and K_{j+1} are loaded: the helper checked them before its p_full arrival
          for (int t = 0; t < 2; ++t) {
            if (j < it.n_t[t]) {
              if (!(ok = mbar_wait_warp(&p_full[t], cp[t] & 1, abort_flag, 153 + t))) break;
              ++cp[t];
              // O_t of this tile's previous item has been read out by its epilogue
              if (j == 0 && act[t] > 0 && !(ok = mbar_wait_warp(&o_free[t], (act[t] - 1) & 1, abort_flag, 155 + t)))
                break;
              tc_fence_after();
              issue_pv(t, Pj, j == 0);
              if (j + 1 == it.n_t[t]) umma_commit_w(&o_done[t]);
            }
            if (j + 1 < it.n_t[t]) issue_s(t, Pj + 1);
          }
          if (!ok) break;
          umma_commit_w(&v_empty[Pj % C::NS]);
          if (j + 1 < it.n_max) umma_commit_w(&k_empty[(Pj + 1) % C::NS]);
          if (j + 2 == it.n_max) umma_commit_w(q_empty);     // the item's last S products issued
        }
        for (int t = 0; t < 2; ++t) act[t] += it.n_t[t] > 0;
        P += it.n_max;
      }
      if (lane == 0 && p.stats != nullptr) atomicAdd(&p.stats[0], n_s);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ helper
    // Folds "V_j loaded" and "K_{j+1} loaded" into each P hand-off (the MMA thread waits once
    // per hand-off); arrives on phase i of a tile's p_full only once phase i-1 is complete.
    if (lane == 0) {
      uint32_t P = 0, ch[2] = {0, 0};
      bool ok = true;
      for (int k = 0; ok && pers_item(k, G) < p.n_items; ++k) {
        const FwdItem it = fwd_item(p, pers_item(k, G));
        for (int j = 0; ok && j < it.n_max; ++j) {
          const uint32_t Pj = P + j;
          if (!(ok = mbar_wait(&v_full[Pj % C::NS], (Pj / C::NS) & 1, abort_flag, 161))) break;
          if (j + 1 < it.n_max &&
              !(ok = mbar_wait(&k_full[(Pj + 1) % C::NS], ((Pj + 1) / C::NS) & 1, abort_flag, 162)))
            break;
          for (int t = 0; t < 2; ++t) {
            if (j < it.n_t[t]) {
              if (ch[t] > 0 && !(ok = mbar_wait(&p_full[t], (ch[t] - 1) & 1, abort_flag, 163 + t))) break;
              mbar_arrive(&p_full[t]);
              ++ch[t];
            }
          }
        }
        P += it.n_max;
      }
    }
  }
  } else {
  setmaxnreg_inc<C::REG_SOFTMAX>();
{
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = (warp - 4) >> 2;
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t t_s = tbase + t_lane + C::T_S + t * 128;
    const uint32_t t_o = tbase + t_lane + C::T_O + t * C::DO;
    const float c2 = p.scale_log2;
    const float2 c2v = make_float2(c2, c2);
    uint32_t cs = 0, act = 0, uses = 0;       // S hand-offs, items of this tile, staging uses
    bool ok = true;
    for (int k = 0; ok && pers_item(k, G) < p.n_items; ++k) {
      const FwdItem it = fwd_item(p, pers_item(k, G));
      // the staging buffer goes to the items' active tiles in order: tile 0, then tile 1
      const uint32_t my_use = uses + ((t == 1 && it.n_t[0] > 0) ? 1u : 0u);
      uses += (it.n_t[0] > 0) + (it.n_t[1] > 0);
      const int n = it.n_t[t];
      if (n == 0) continue;
      const int q0t = it.q0[t];
      const int q_idx = q0t + row;
      float m = -INFINITY, l = 0.f, lb = 0.f;
      for (int j = 0; j < n; ++j) {
        if (!(ok = mbar_wait_warp(&s_full[t], cs & 1, abort_flag, 171))) break;
        ++cs;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t rr[32];
          tmem_ld32(t_s + kk * 32, rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[kk * 32 + i] = __uint_as_float(rr[i]);
        }
        tmem_wait_ld();
        const int k0 = j * C::BN;
        if (k0 + C::BN > p.n_kv || (p.causal && k0 + C::BN - 1 > q0t)) {
          const int lim = p.causal ? min(q_idx + 1, p.n_kv) : p.n_kv;   // keys < lim visible
#pragma unroll
          for (int kk = 0; kk < 128; ++kk)
            if (k0 + kk >= lim) s[kk] = -INFINITY;
        }
        float mq[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          mq[g] = fmax3(s[32 * g], s[32 * g + 1], s[32 * g + 2]);
#pragma unroll
          for (int kk = 3; kk < 31; kk += 2) mq[g] = fmax3(mq[g], s[32 * g + kk], s[32 * g + kk + 1]);
          mq[g] = fmaxf(mq[g], s[32 * g + 31]);
        }
        const float cand = fmaxf(m, fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]));
        // every row sees a key of its first tile, so cand is finite from there on
        const bool move = (m == -INFINITY) || ((cand - m) * c2 > C::RESCALE_THRESHOLD);
        if (__any_sync(0xffffffffu, move)) {
          const float alpha = move ? fast_exp2((m - cand) * c2) : 1.f;
          if (move) {
            l *= alpha;
            lb *= alpha;
            m = cand;
          }
          if (j > 0) {                          // O_t settled: PV_t(j-1) preceded S_t(j)
#pragma unroll
            for (int kk = 0; kk < C::DO / 16; ++kk) {  // 16 columns at a time (s[] is live here)
              uint32_t rr[16];
              tmem_ld16(t_o + kk * 16, rr);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                const float2 v = fmul2(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])),
                                       make_float2(alpha, alpha));
                rr[i] = __float_as_uint(v.x);
                rr[i + 1] = __float_as_uint(v.y);
              }
              tmem_st16(t_o + kk * 16, rr);
            }
          }
        }
        const float2 nms = make_float2(-m * c2, -m * c2);
        float2 rs[4], rb[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) rs[g] = rb[g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {           // P (bf16) over the first 64 columns of S_t
          uint32_t pk[32];
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {
            const float2 x = ffma2(make_float2(s[64 * h + 2 * kk], s[64 * h + 2 * kk + 1]), c2v, nms);
            const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
            pk[kk] = pack_bf16x2(p0, p1);
            rs[kk & 3] = fadd2(rs[kk & 3], make_float2(p0, p1));
            // lb sums the bf16 weights the PV product uses (O / lb is their exact average);
            // d = 64: the tensor core forms it in O's normaliser columns
            if constexpr (!C::LB_MMA) rb[kk & 3] = add_bf16x2_f32(rb[kk & 3], pk[kk]);
          }
          tmem_st32(t_s + h * 32, pk);
        }
        const float2 rs01 = fadd2(fadd2(rs[0], rs[1]), fadd2(rs[2], rs[3]));
        const float2 rb01 = fadd2(fadd2(rb[0], rb[1]), fadd2(rb[2], rb[3]));
        l += rs01.x + rs01.y;
        lb += rb01.x + rb01.y;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      // ---------------------------------------------------------------- epilogue of the item
      // Every warp of the group reaches the group barrier below once per item, whatever its
      // waits returned (a named barrier cannot time out); the barrier ORs the failures, and the
      // whole group leaves together.
      if (ok) ok = mbar_wait_warp(&o_done[t], act & 1, abort_flag, 172);
      ++act;
      if (ok && my_use > 0) ok = mbar_wait_warp(st_free, (my_use - 1) & 1, abort_flag, 173);
      if (ok) {
        tc_fence_after();
        if constexpr (C::LB_MMA) {             // the normaliser: O_t's column d
          uint32_t rl[16];
          tmem_ld16(t_o + D, rl);
          tmem_wait_ld();
          lb = __uint_as_float(rl[0]);
        }
        const float inv_l = (lb > 0.f) ? 1.f / lb : 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
          uint32_t rr[32];
          tmem_ld32(t_o + kk * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v4;
            v4.x = pack_bf16x2(__uint_as_float(rr[i + 0]) * inv_l, __uint_as_float(rr[i + 1]) * inv_l);
            v4.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * inv_l, __uint_as_float(rr[i + 3]) * inv_l);
            v4.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * inv_l, __uint_as_float(rr[i + 5]) * inv_l);
            v4.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * inv_l, __uint_as_float(rr[i + 7]) * inv_l);
            const int col = kk * 32 + i;
            *reinterpret_cast<uint4*>(sO + (col >> 6) * C::CHUNK + sw128_offset(row, col & 63)) = v4;
          }
        }
        tc_fence_before();
        mbar_arrive(&o_free[t]);                // the next item's first PV may overwrite O_t
      }
      if (ok && q_idx < p.n_q)
        p.lse[static_cast<size_t>(it.bh) * p.n_q + q_idx] = (l > 0.f) ? fmaf(m, p.scale, logf(l)) : -INFINITY;
      fence_proxy_async_smem();
      if (named_bar_red_or(1 + t, 128, !ok)) {
        ok = false;
        break;
      }
      if ((threadIdx.x & 127) == 64) {
        for (int c = 0; c < C::OCH; ++c) tma_store_3d(&p.to, sO + c * C::CHUNK, c * 64, q0t, it.bh);
        bulk_commit_group();
        bulk_wait_group_read0();              // the staging buffer may be reused
        mbar_arrive(st_free);
      }
    }
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

template <int D>
static cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  FwdParams p;
  const uint64_t bh = static_cast<uint64_t>(a.B) * a.H;
  // With N_kv == 0 no key tile is ever loaded; the maps still need a non-zero extent.
  const uint64_t kv_rows = a.n_kv > 0 ? static_cast<uint64_t>(a.n_kv) : 1;
  const uint64_t kv_planes = a.n_kv > 0 ? bh : 1;
  if (!make_map_bf16_3d(&p.tq, a.q, D, a.n_q, bh, 64, 128) ||
      !make_map_bf16_3d(&p.tk, a.k, D, kv_rows, kv_planes, 64, 128) ||
      !make_map_bf16_3d(&p.tv, a.v, D, kv_rows, kv_planes, 64, 128) ||
      !make_map_bf16_3d(&p.to, a.o, D, a.n_q, bh, 64, 128))
    return cudaErrorInvalidValue;
  p.lse = a.lse;
  p.n_q = a.n_q;
  p.n_kv = a.n_kv;
  p.n_qpairs = (a.n_q + 2 * C::BM - 1) / (2 * C::BM);
  p.n_kvtiles = (a.n_kv + C::BN - 1) / C::BN;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.heads = a.H;
  p.total_q = 0;
  p.cu_q = p.cu_k = nullptr;
  p.o = static_cast<uint16_t*>(a.o);
  p.out_scale = 1.f;
  p.stats = debug_counters();
  attention_window(a.causal, a.windowed, a.win_left, a.win_right, &p.win_left, &p.win_right);
  p.block_mask = a.block_mask;
  p.bm_per_head = a.bm_per_head;
  p.n_qblocks = (a.n_q + kBlockSize - 1) / kBlockSize;
  static int attr_done[64] = {0};   // one per instantiation of this launcher
  const uint64_t grid = static_cast<uint64_t>(p.n_qpairs) * bh;
  if (a.block_mask != nullptr) {
    static int attr_bs[64] = {0};
    cudaError_t e = ensure_smem_attr(fwd_kernel<D, false, false, false, true>, C::SMEM_BYTES, attr_bs, C::THREADS, reg_split_need<C>());
    if (e != cudaSuccess) return e;
    log_launch("fwd_kernel<D, false, false, false, true>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
    fwd_kernel<D, false, false, false, true><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
  }
  if (!a.windowed && a.n_kv > 0 && use_persistent(D, a.causal != 0, p.n_kvtiles)) {
    // short items: the persistent kernel, one CTA per SM over the same items (measured: the
    // overlap at item boundaries pays when an item streams few key tiles; with long items the
    // one-CTA-per-item kernel runs its steps faster and wins)
    using PC = FwdPCfg<D>;
    static int attr_p[64] = {0};
    cudaError_t e = ensure_smem_attr(fwd_persistent_kernel<D>, PC::SMEM_BYTES, attr_p, PC::THREADS, reg_split_need<PC>());
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    p.n_items = static_cast<int>(grid);
    const unsigned ctas = static_cast<unsigned>(std::min<uint64_t>(grid, static_cast<uint64_t>(std::max(sms, 1))));
    log_launch("fwd_persistent_kernel<D>", static_cast<unsigned long long>(ctas), PC::THREADS, static_cast<unsigned long long>(PC::SMEM_BYTES));
    fwd_persistent_kernel<D><<<ctas, PC::THREADS, PC::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
  }
  if (a.windowed) {
    static int attr_win[64] = {0};
    cudaError_t e = ensure_smem_attr(fwd_kernel<D, false, false, true>, C::SMEM_BYTES, attr_win, C::THREADS, reg_split_need<C>());
    if (e != cudaSuccess) return e;
    log_launch("fwd_kernel<D, false, false, true>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
    fwd_kernel<D, false, false, true><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
  }
  cudaError_t e = ensure_smem_attr(fwd_kernel<D, false>, C::SMEM_BYTES, attr_done, C::THREADS, reg_split_need<C>());
  if (e != cudaSuccess) return e;
  log_launch("fwd_kernel<D, false>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
  fwd_kernel<D, false><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

// Variable-length forward: packed token-major [total, H, d] tensors and cu_seqlens.
template <int D>
static cudaError_t launch_fwd_varlen_d(const FwdVarlenArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  FwdParams p;
  // {d, H, total}: a {64, 1, 128} box is 128 consecutive tokens of one head
  auto make = [&](CUtensorMap* m, const void* base, int total) {
    const int rows = total > 0 ? total : 1;
    return make_map_bf16_tok(m, base, D, a.H, rows, 64, 128);
  };
  if (!make(&p.tq, a.q, a.total_q) || !make(&p.tk, a.k, a.total_k) || !make(&p.tv, a.v, a.total_k) ||
      !make(&p.to, a.o, a.total_q))
    return cudaErrorInvalidValue;
  p.lse = a.lse;
  p.n_q = a.max_seqlen_q;          // bound checked against every sequence in the kernel
  p.n_kv = a.total_k;
  p.n_qpairs = (a.max_seqlen_q + 2 * C::BM - 1) / (2 * C::BM);
  p.n_kvtiles = 0;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.heads = a.H;
  p.total_q = a.total_q;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.o = static_cast<uint16_t*>(a.o);
  p.out_scale = 1.f;
  p.stats = debug_counters();
  attention_window(a.causal, false, 0, 0, &p.win_left, &p.win_right);
  p.block_mask = nullptr;
  p.bm_per_head = p.n_qblocks = 0;
  static int attr_done[64] = {0};
  cudaError_t e = ensure_smem_attr(fwd_kernel<D, true>, C::SMEM_BYTES, attr_done, C::THREADS, reg_split_need<C>());
  if (e != cudaSuccess) return e;
  const uint64_t grid = static_cast<uint64_t>(p.n_qpairs) * a.n_seqs * a.H;
  if (grid == 0) return cudaSuccess;
  log_launch("fwd_kernel<D, true>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
  fwd_kernel<D, true><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

// FP8 forward (d = 128): e4m3 Q, K, V with one scale each; bf16 O, fp32 lse.
cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream) {
  constexpr int D = 128;
  using C = FwdCfg<D, true>;
  FwdParams p;
  const uint64_t bh = static_cast<uint64_t>(a.B) * a.H;
  const uint64_t kv_rows = a.n_kv > 0 ? static_cast<uint64_t>(a.n_kv) : 1;
  const uint64_t kv_planes = a.n_kv > 0 ? bh : 1;
  if (!make_map_u8_3d(&p.tq, a.q, D, a.n_q, bh, 128, 128) ||
      !make_map_u8_3d(&p.tk, a.k, D, kv_rows, kv_planes, 128, 128) ||
      !make_map_u8_3d(&p.tv, a.v, D, kv_rows, kv_planes, 128, 128) ||
      !make_map_bf16_3d(&p.to, a.o, D, a.n_q, bh, 64, 128))
    return cudaErrorInvalidValue;
  p.lse = a.lse;
  p.n_q = a.n_q;
  p.n_kv = a.n_kv;
  p.n_qpairs = (a.n_q + 2 * C::BM - 1) / (2 * C::BM);
  p.n_kvtiles = (a.n_kv + C::BN - 1) / C::BN;
  p.causal = a.causal;
  p.scale = a.scale * a.descale_q * a.descale_k;
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.heads = a.H;
  p.total_q = 0;
  p.cu_q = p.cu_k = nullptr;
  p.o = static_cast<uint16_t*>(a.o);
  p.out_scale = a.descale_v;
  p.stats = debug_counters();
  attention_window(a.causal, false, 0, 0, &p.win_left, &p.win_right);
  p.block_mask = nullptr;
  p.bm_per_head = p.n_qblocks = 0;
  static int attr_done[64] = {0};
  cudaError_t e = ensure_smem_attr(fwd_kernel<D, false, true>, C::SMEM_BYTES, attr_done, C::THREADS, reg_split_need<C>());
  if (e != cudaSuccess) return e;
  const uint64_t grid = static_cast<uint64_t>(p.n_qpairs) * bh;
  log_launch("fwd_kernel<D, false, true>", static_cast<unsigned long long>(static_cast<unsigned>(grid)), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
  fwd_kernel<D, false, true><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_varlen(const FwdVarlenArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_fwd_varlen_d<64>(a, stream);
  return launch_fwd_varlen_d<128>(a, stream);
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_fwd_d<64>(a, stream);
  return launch_fwd_d<128>(a, stream);
}

}  // namespace fa

FA_DEFINE_STATUS_FETCH(status_fetch_fwd)
