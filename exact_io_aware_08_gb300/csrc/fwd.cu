// F1: attention forward on sm_103a.
//
// Follows "FlashAttention and online softmax" (ML Systems lesson 4), section 3 "The tiled
// forward pass" and "The online softmax theorem": one CTA owns a tile of 128 query rows, keeps
// Q on chip, streams 128-key tiles of K and V, and carries the per-row state (m, l, o~) across
// tiles, dividing once at the end (the FlashAttention-2 form, "Keep o~ unnormalised").
// Causal tiles above the diagonal are skipped, the diagonal tile is masked ("Causal masks").
//
// GB300 mapping (one CTA per SM, 192 threads):
//   warp 0      TMA producer: Q once, then K_j / V_j into NST-deep shared-memory rings.
//   warp 1      TMEM owner and MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               score buffers, then O += P_j V_j into the TMEM output accumulator.
//   warps 2-5   softmax + correction: thread t owns query row t; it loads its S row from TMEM,
//               updates (m, l) in the log2 domain (scale * log2 e folded into one FMA), writes
//               P_j as bf16 into shared memory for the PV MMA, and rescales its O row in TMEM by
//               e^{m_old - m_new} when the max moved.  The epilogue divides by l, writes O
//               through a TMA store and lse = m + ln l.
// The MMA for S_{j+1} is issued before the PV of tile j, so the tensor core computes the next
// score tile while the softmax warps work on the current one.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int KCH = D / 64;                 // 64-column (128-byte) chunks per row
  static constexpr int TILE = 128 * D * 2;           // bytes of one 128-row bf16 tile
  static constexpr int CHUNK = 128 * 128;            // bytes of one [128 x 64] swizzled chunk
  static constexpr int NST = (D == 128) ? 2 : 4;     // K/V ring depth (one CTA per SM)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_P = OFF_V + NST * TILE;
  static constexpr int OFF_BAR = OFF_P + 2 * CHUNK;
  // q_full, k_full[NST], k_empty[NST], v_full[NST], v_empty[NST], s_full[2], s_free[2],
  // p_full, o_done, mma_done
  static constexpr int NBAR = 1 + 4 * NST + 4 + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + slack for 1 KB alignment
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0;      // two score buffers: columns [0,128) and [128,256)
  static constexpr uint32_t T_O = 256;    // output accumulator: columns [256, 256 + D)
  static constexpr int THREADS = 192;
};

struct FwdParams {
  CUtensorMap tq, tk, tv, to;
  float* lse;
  int n_q, n_kv, bh, n_qtiles, n_kvtiles, causal;
  float scale, scale_log2;
};

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1k(smem_raw);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::NST;
  uint64_t* v_full = k_empty + C::NST;
  uint64_t* v_empty = v_full + C::NST;
  uint64_t* s_full = v_empty + C::NST;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* mma_done = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: query tile qt of head bh.  Tiles of one head are adjacent so the CTAs that run
  // together share K/V in L2; causal runs the longer (later) tiles of each head first.
  const int bh = blockIdx.x / p.n_qtiles;
  const int r = blockIdx.x % p.n_qtiles;
  const int qt = p.causal ? (p.n_qtiles - 1 - r) : r;
  const int q0 = qt * C::BM;
  const int n_tiles = p.causal ? min(qt + 1, p.n_kvtiles) : p.n_kvtiles;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tq);
    tma_prefetch_desc(&p.tk);
    tma_prefetch_desc(&p.tv);
    tma_prefetch_desc(&p.to);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      int issued = 0;
      mbar_arrive_expect_tx(q_full, C::TILE);
      for (int c = 0; c < C::KCH; ++c) tma_load_3d(sQ + c * C::CHUNK, &p.tq, q_full, c * 64, q0, bh);
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % C::NST;
        const uint32_t n = j / C::NST;
        if (n > 0 && !mbar_wait(&k_empty[s], (n - 1) & 1, abort_flag, 101)) break;
        mbar_arrive_expect_tx(&k_full[s], C::TILE);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sK + s * C::TILE + c * C::CHUNK, &p.tk, &k_full[s], c * 64, j * C::BN, bh);
        if (n > 0 && !mbar_wait(&v_empty[s], (n - 1) & 1, abort_flag, 102)) break;
        mbar_arrive_expect_tx(&v_full[s], C::TILE);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sV + s * C::TILE + c * C::CHUNK, &p.tv, &v_full[s], c * 64, j * C::BN, bh);
        issued = j + 1;
      }
      if (*abort_flag) {
        // Drain: let every copy this thread started land before the CTA exits.
        mbar_wait(q_full, 0, nullptr, 103);
        for (int j = max(0, issued - C::NST); j < issued; ++j) {
          mbar_wait(&k_full[j % C::NST], (j / C::NST) & 1, nullptr, 104);
          mbar_wait(&v_full[j % C::NST], (j / C::NST) & 1, nullptr, 105);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
      const uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);    // P K-major, V MN-major
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t p_addr = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0, abort_flag, 111);
      auto issue_s = [&](int j) {
        const int s = j % C::NST;
        const uint32_t k_addr = smem_u32(sK + s * C::TILE);
        const uint32_t d_tmem = tbase + C::T_S + (j & 1) * 128;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
          umma_ss(d_tmem, smem_desc_sw128(q_addr + off, 0, 1024),
                  smem_desc_sw128(k_addr + off, 0, 1024), idesc_s, ks > 0);
        }
        umma_commit(&s_full[j & 1]);
        umma_commit(&k_empty[s]);
      };
      if (ok && (ok = mbar_wait(&k_full[0], 0, abort_flag, 112))) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          const int s1 = (j + 1) % C::NST;
          if (!(ok = mbar_wait(&k_full[s1], ((j + 1) / C::NST) & 1, abort_flag, 113))) break;
          if (j + 1 >= 2 &&
              !(ok = mbar_wait(&s_free[(j + 1) & 1], (((j + 1) >> 1) - 1) & 1, abort_flag, 114)))
            break;
          tc_fence_after();
          issue_s(j + 1);
        }
        const int s = j % C::NST;
        if (!(ok = mbar_wait(p_full, j & 1, abort_flag, 115))) break;
        if (!(ok = mbar_wait(&v_full[s], (j / C::NST) & 1, abort_flag, 116))) break;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sV + s * C::TILE);
#pragma unroll
        for (int ks = 0; ks < C::BN / 16; ++ks) {
          const uint32_t a_off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
          umma_ss(tbase + C::T_O, smem_desc_sw128(p_addr + a_off, 0, 1024),
                  smem_desc_sw128(v_addr + ks * 2048, C::CHUNK, 1024), idesc_o,
                  (j > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(o_done);
        umma_commit(&v_empty[s]);
      }
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, nullptr, 117);
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroup
    const int sub = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = sub * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(sub * 32) << 16;
    const int q_idx = q0 + row;
    const float c2 = p.scale_log2;
    float m = -INFINITY;                      // running max of the raw dot products
    float l = 0.f;                            // running sum, relative to m
    bool ok = true;

    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      if (!(ok = mbar_wait_warp(&s_full[b], (j >> 1) & 1, abort_flag, 121))) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tmem_ld32(tbase + t_lane + C::T_S + b * 128 + c * 32, rr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(rr[i]);
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);

      const int k0 = j * C::BN;
      if (k0 + C::BN > p.n_kv || (p.causal && j == qt)) {
        const int lim = p.causal ? min(q_idx + 1, p.n_kv) : p.n_kv;   // keys < lim visible
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (k0 + c >= lim) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx);
      const float ms = (m_new == -INFINITY) ? 0.f : m_new * c2;
      const float alpha = fast_exp2(m * c2 - ms);       // 0 on the first tile (m = -inf)
      float rs = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = fast_exp2(fmaf(s[2 * c], c2, -ms));
        const float p1 = fast_exp2(fmaf(s[2 * c + 1], c2, -ms));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      m = m_new;

      // PV_{j-1} must be finished before P_j overwrites the P buffer and O is rescaled.
      if (j > 0) {
        if (!(ok = mbar_wait_warp(o_done, (j - 1) & 1, abort_flag, 122))) break;
        tc_fence_after();
      }
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        uint4 v4 = make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        *reinterpret_cast<uint4*>(sP + (c8 >> 3) * C::CHUNK + sw128_offset(row, (c8 & 7) * 8)) = v4;
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          const uint32_t ta = tbase + t_lane + C::T_O + c * 32;
          tmem_ld32(ta, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
          tmem_st32(ta, rr);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }

    // ------------------------------------------------------------------ epilogue
    if (ok && n_tiles > 0) {
      ok = mbar_wait_warp(o_done, (n_tiles - 1) & 1, abort_flag, 123);
      tc_fence_after();
    }
    if (ok) {
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        if (n_tiles > 0) {
          tmem_ld32(tbase + t_lane + C::T_O + c * 32, rr);
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
          const int col = c * 32 + i;
          *reinterpret_cast<uint4*>(sQ + (col >> 6) * C::CHUNK + sw128_offset(row, col & 63)) = v4;
        }
      }
      if (q_idx < p.n_q)
        p.lse[static_cast<size_t>(bh) * p.n_q + q_idx] =
            (l > 0.f) ? fmaf(m, p.scale, logf(l)) : -INFINITY;
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && threadIdx.x == 64) {
      for (int c = 0; c < C::KCH; ++c) tma_store_3d(&p.to, sQ + c * C::CHUNK, c * 64, q0, bh);
      bulk_commit_group();
      bulk_wait_group_read0();
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
  p.bh = static_cast<int>(bh);
  p.n_qtiles = (a.n_q + C::BM - 1) / C::BM;
  p.n_kvtiles = (a.n_kv + C::BN - 1) / C::BN;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  static int attr_done[64] = {0};   // one per instantiation of this launcher
  cudaError_t e = ensure_smem_attr(fwd_kernel<D>, C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const uint64_t grid = static_cast<uint64_t>(p.n_qtiles) * bh;
  fwd_kernel<D><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_fwd_d<64>(a, stream);
  return launch_fwd_d<128>(a, stream);
}

}  // namespace fa

FA_DEFINE_STATUS_FETCH(status_fetch_fwd)
