// F5/F6: split-KV decode on sm_103a.
//
// Follows "FlashAttention and online softmax" (ML Systems lesson 4), section 3 "Split-KV for
// decoding (flash-decoding)": each (b, h) row's KV cache is cut into n_splits chunks, every
// chunk produces its online state (m, l, o~) ("The online softmax theorem"), and a second small
// kernel merges the states of a row ("Merging two partial results", computed stably with -inf
// guards).
//
// One query row against 128-wide keys is a matrix-vector product (about 1 FLOP per byte of
// K/V), so this path is HBM-bound and uses CUDA cores, not the tensor core.  GB300 mapping:
//   F5  persistent CTAs (2 per SM), 5 warps each.  Warp 4 streams 64-key sub-tiles of K and V
//       with TMA (128-byte swizzle, bank-conflict-free reads) through a 3-stage ring that runs
//       continuously across the CTA's work items.  Warps 0-3 each own 16 keys of a sub-tile:
//       lanes (key, half) form partial dot products with q (pre-scaled by scale * log2 e),
//       a shuffle joins the halves, and each warp keeps its own (m, l, o~) so no CTA-wide
//       barrier is needed per sub-tile; the four warp states merge once per chunk.
//   F6  one CTA per (b, h): lse-weighted merge of the n_splits partial states.
// Partial state layout: part[(bh * n_splits + split) * (d + 2) + {0..d-1, d, d+1}] =
// (o~[0..d-1], m2, l) with m2 = max_j S_j * log2 e (base-2 units) and l = sum_j 2^{S_j log2 e - m2}.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {

template <int D>
struct DecCfg {
  static constexpr int KEYS = kDecodeKeyStep;        // keys per sub-tile (64)
  static constexpr int KCH = D / 64;
  static constexpr int CHUNK = KEYS * 128;           // one [64 keys x 64 d] swizzled box
  static constexpr int SUB = KEYS * D * 2;           // K (or V) bytes of a sub-tile
  static constexpr int NST = 3;
  static constexpr int STAGE = 2 * SUB;
  static constexpr int CONS_WARPS = 4;
  static constexpr int THREADS = 32 * (CONS_WARPS + 1);
  static constexpr int UPL = D / 16;                 // 16-byte K units per lane (half a row)
  static constexpr int VPL = D / 32;                 // V elements per lane
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_MERGE = NST * STAGE;      // CONS_WARPS x (D + 2) floats
  static constexpr int OFF_BAR = OFF_MERGE + CONS_WARPS * (D + 2) * 4 + 64;
  static constexpr int SMEM_BYTES = OFF_BAR + (2 * NST + 2) * 8 + 16 + 1024;
};

struct DecParams {
  CUtensorMap tk, tv;
  const uint16_t* q;
  float* part;
  int n_kv, bh, n_splits, chunk, n_items;
  float scale_log2;
  // Paged KV cache: k/v cache [num_blocks, block_size, H, d]; logical key j of batch b lives in
  // block block_table[b * max_blocks + j / block_size] at row j % block_size; seqlens[b] keys.
  const int* block_table;
  const int* seqlens;
  int heads, block_size, max_blocks, num_blocks;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D, bool PG>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 2)
decode_split_kernel(const __grid_constant__ DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1k(smem_raw);
  float* merge = reinterpret_cast<float*>(smem + C::OFF_MERGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NST;
  uint64_t* mrg = empty + C::NST;           // [0]: warp states written, [1]: merge done
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + (2 * C::NST + 2) * 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::CONS_WARPS);
    }
    mbar_init(&mrg[0], C::CONS_WARPS);
    mbar_init(&mrg[1], C::CONS_WARPS);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();

  // Sub-tiles of item i: keys [split*chunk, min(split*chunk + chunk, n_kv)) in steps of 64.
  // Paged: the row's own length seqlens[b] (an out-of-range length is reported and treated as
  // empty).
  auto item_subtiles = [&](int item, int& key0, int& key_end) {
    const int split = item % p.n_splits;
    int n_kv = p.n_kv;
    if (PG) {
      // p.n_kv is the caller's max_seqlen_k (<= max_blocks * block_size, checked on the host),
      // which the chunks cover
      n_kv = p.seqlens[(item / p.n_splits) / p.heads];
      if (n_kv < 0 || n_kv > p.n_kv) {
        if (split == 0 && threadIdx.x == 0) report_device_error(FA_DEV_BAD_CONFIG, 350);
        n_kv = 0;
      }
    }
    key0 = split * p.chunk;
    key_end = min(key0 + p.chunk, n_kv);
    return key_end > key0 ? (key_end - key0 + C::KEYS - 1) / C::KEYS : 0;
  };

  if (warp == C::CONS_WARPS) {
    // -------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tk);
      tma_prefetch_desc(&p.tv);
      uint32_t g = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
        int key0, key_end;
        const int nsub = item_subtiles(item, key0, key_end);
        const int bh = item / p.n_splits;
        for (int t = 0; t < nsub; ++t, ++g) {
          const int s = g % C::NST;
          const uint32_t n = g / C::NST;
          if (n > 0 && !(ok = mbar_wait(&empty[s], (n - 1) & 1, abort_flag, 301))) break;
          uint8_t* st = smem + C::OFF_STAGE + s * C::STAGE;
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          const int kk = key0 + t * C::KEYS;
          int y1 = kk, y2 = bh;                     // contiguous cache: {x, key, (b,h)}
          if (PG) {
            // paged cache {x, h, block * block_size + row}; a 64-key sub-tile never crosses a
            // block (block_size and the chunk are multiples of 64)
            const int b = bh / p.heads;
            int phys = p.block_table[static_cast<size_t>(b) * p.max_blocks + kk / p.block_size];
            if (phys < 0 || phys >= p.num_blocks) {
              report_device_error(FA_DEV_BAD_CONFIG, 351);
              phys = 0;                             // stays in bounds; the result is reported invalid
            }
            y1 = bh % p.heads;
            y2 = phys * p.block_size + kk % p.block_size;
          }
#pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(st + c * C::CHUNK, &p.tk, &full[s], c * 64, y1, y2);
            tma_load_3d(st + C::SUB + c * C::CHUNK, &p.tv, &full[s], c * 64, y1, y2);
          }
        }
      }
      if (!ok) {
        // drain the copies already issued (at most NST outstanding)
        for (uint32_t x = (g > C::NST ? g - C::NST : 0); x < g; ++x)
          mbar_wait(&full[x % C::NST], (x / C::NST) & 1, nullptr, 302);
      }
    }
  } else {
    // -------------------------------------------------------------- consumers
    const int key_l = lane & 15;     // key within this warp's 16
    const int half = lane >> 4;      // which half of d this lane dots
    const int row = warp * 16 + key_l;
    uint32_t g = 0;
    uint32_t it = 0;                 // items processed by this CTA (merge barrier phase)
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, ++it) {
      int key0, key_end;
      const int nsub = item_subtiles(item, key0, key_end);
      const int bh = item / p.n_splits;
      // q for this lane's half of d, pre-scaled into the log2 domain
      float qf[C::UPL * 8];
      {
        const uint4* qp = reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(bh) * D) + half * C::UPL;
#pragma unroll
        for (int u = 0; u < C::UPL; ++u) {
          const uint4 w = __ldg(qp + u);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qf[u * 8 + 2 * e] = bf16lo(ww[e]) * p.scale_log2;
            qf[u * 8 + 2 * e + 1] = bf16hi(ww[e]) * p.scale_log2;
          }
        }
      }
      float m = -INFINITY, l = 0.f;
      float o[C::VPL];
#pragma unroll
      for (int i = 0; i < C::VPL; ++i) o[i] = 0.f;

      for (int t = 0; ok && t < nsub; ++t, ++g) {
        const int s = g % C::NST;
        if (!(ok = mbar_wait_warp(&full[s], (g / C::NST) & 1, abort_flag, 311))) break;
        const uint8_t* sk = smem + C::OFF_STAGE + s * C::STAGE;
        const uint8_t* sv = sk + C::SUB;
        // score of key `row`: this lane's half of the dot product
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < C::UPL; ++u) {
          const int ug = half * C::UPL + u;            // 16-byte unit along d
          const uint4 w = *reinterpret_cast<const uint4*>(
              sk + (ug >> 3) * C::CHUNK + row * 128 + (((ug & 7) ^ (row & 7)) << 4));
          acc = fmaf(qf[u * 8 + 0], bf16lo(w.x), acc);
          acc = fmaf(qf[u * 8 + 1], bf16hi(w.x), acc);
          acc = fmaf(qf[u * 8 + 2], bf16lo(w.y), acc);
          acc = fmaf(qf[u * 8 + 3], bf16hi(w.y), acc);
          acc = fmaf(qf[u * 8 + 4], bf16lo(w.z), acc);
          acc = fmaf(qf[u * 8 + 5], bf16hi(w.z), acc);
          acc = fmaf(qf[u * 8 + 6], bf16lo(w.w), acc);
          acc = fmaf(qf[u * 8 + 7], bf16hi(w.w), acc);
        }
        float sc = acc + __shfl_xor_sync(0xffffffffu, acc, 16);
        if (key0 + t * C::KEYS + row >= key_end) sc = -INFINITY;
        float mt = sc;
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        const float m_new = fmaxf(m, mt);
        if (m_new != -INFINITY) {
          const float alpha = fast_exp2(m - m_new);
          const float pv = fast_exp2(sc - m_new);
          float ps = pv;
#pragma unroll
          for (int off = 8; off >= 1; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
          l = l * alpha + ps;
#pragma unroll
          for (int i = 0; i < C::VPL; ++i) o[i] *= alpha;
          const int d0 = lane * C::VPL;
          const int unit = (d0 & 63) >> 3;
          const int boff = (d0 & 7) * 2;
          const uint8_t* vb = sv + (d0 >> 6) * C::CHUNK + boff;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float pk = __shfl_sync(0xffffffffu, pv, k);
            const int r = warp * 16 + k;
            // A paged block's rows past the sequence end are whatever the cache holds (possibly
            // not finite): skip them rather than add 0 * V.
            if (PG && key0 + t * C::KEYS + r >= key_end) break;
            const uint8_t* va = vb + r * 128 + ((unit ^ (r & 7)) << 4);
            if constexpr (C::VPL == 4) {
              const uint2 w = *reinterpret_cast<const uint2*>(va);
              o[0] = fmaf(pk, bf16lo(w.x), o[0]);
              o[1] = fmaf(pk, bf16hi(w.x), o[1]);
              o[2] = fmaf(pk, bf16lo(w.y), o[2]);
              o[3] = fmaf(pk, bf16hi(w.y), o[3]);
            } else {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(va);
              o[0] = fmaf(pk, bf16lo(w), o[0]);
              o[1] = fmaf(pk, bf16hi(w), o[1]);
            }
          }
          m = m_new;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (!ok) break;

      // merge the four warp states of this chunk and write the partial
      float* mw = merge + warp * (D + 2);
#pragma unroll
      for (int i = 0; i < C::VPL; ++i) mw[lane * C::VPL + i] = o[i];
      if (lane == 0) {
        mw[D] = m;
        mw[D + 1] = l;
      }
      if (!(ok = warps_sync(&mrg[0], it & 1, abort_flag, 312))) break;
      if (threadIdx.x < D) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::CONS_WARPS; ++w) M = fmaxf(M, merge[w * (D + 2) + D]);
        float acc_o = 0.f, acc_l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < C::CONS_WARPS; ++w) {
            const float mw_ = merge[w * (D + 2) + D];
            const float wt = (mw_ == -INFINITY) ? 0.f : fast_exp2(mw_ - M);
            acc_o = fmaf(wt, merge[w * (D + 2) + threadIdx.x], acc_o);
            acc_l = fmaf(wt, merge[w * (D + 2) + D + 1], acc_l);
          }
        }
        float* dst = p.part + static_cast<size_t>(item) * (D + 2);
        dst[threadIdx.x] = acc_o;
        if (threadIdx.x == 0) {
          dst[D] = M;
          dst[D + 1] = acc_l;
        }
      }
      if (!(ok = warps_sync(&mrg[1], it & 1, abort_flag, 313))) break;
    }
  }
  __syncwarp();
  __syncthreads();
}

// F6: one CTA of D threads per (b, h).
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const float* __restrict__ part,
                                                         uint16_t* __restrict__ o,
                                                         float* __restrict__ lse, int n_splits) {
  const int bh = blockIdx.x;
  const int t = threadIdx.x;
  const float* base = part + static_cast<size_t>(bh) * n_splits * (D + 2);
  float M = -INFINITY;
  for (int c = 0; c < n_splits; ++c) M = fmaxf(M, base[c * (D + 2) + D]);
  float acc_o = 0.f, acc_l = 0.f;
  if (M != -INFINITY) {
    for (int c = 0; c < n_splits; ++c) {
      const float mc = base[c * (D + 2) + D];
      if (mc == -INFINITY) continue;                 // empty chunk: weight 0
      const float wt = fast_exp2(mc - M);
      acc_o = fmaf(wt, base[c * (D + 2) + t], acc_o);
      acc_l = fmaf(wt, base[c * (D + 2) + D + 1], acc_l);
    }
  }
  const float out = (acc_l > 0.f) ? acc_o / acc_l : 0.f;
  const uint32_t packed = pack_bf16x2(out, 0.f);
  o[static_cast<size_t>(bh) * D + t] = static_cast<uint16_t>(packed & 0xffffu);
  if (t == 0) lse[bh] = (acc_l > 0.f) ? (M + log2f(acc_l)) * 0.6931471805599453f : -INFINITY;
}

static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  if (dev < 64) cached[dev] = n;
  return n;
}

template <int D>
static cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t stream) {
  using C = DecCfg<D>;
  const uint64_t bh = static_cast<uint64_t>(a.B) * a.H;
  DecParams p;
  const uint64_t rows = a.n_kv > 0 ? static_cast<uint64_t>(a.n_kv) : 1;
  if (!make_map_bf16_3d(&p.tk, a.k, D, rows, a.n_kv > 0 ? bh : 1, 64, C::KEYS) ||
      !make_map_bf16_3d(&p.tv, a.v, D, rows, a.n_kv > 0 ? bh : 1, 64, C::KEYS))
    return cudaErrorInvalidValue;
  p.q = static_cast<const uint16_t*>(a.q);
  p.part = a.part;
  p.n_kv = a.n_kv;
  p.bh = static_cast<int>(bh);
  p.n_splits = a.n_splits;
  p.chunk = a.chunk;
  p.n_items = static_cast<int>(bh) * a.n_splits;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  static int attr_done[64] = {0};   // one per instantiation of this launcher
  p.block_table = p.seqlens = nullptr;
  p.heads = a.H;
  p.block_size = p.max_blocks = p.num_blocks = 0;
  cudaError_t e = ensure_smem_attr(decode_split_kernel<D, false>, C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const int grid = min(p.n_items, 2 * sm_count());
  log_launch("decode_split_kernel<D, false>", static_cast<unsigned long long>(grid), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
  decode_split_kernel<D, false><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  log_launch("decode_merge_kernel<D>", static_cast<unsigned long long>(static_cast<unsigned>(bh)), D, static_cast<unsigned long long>(0));
  decode_merge_kernel<D><<<static_cast<unsigned>(bh), D, 0, stream>>>(
      a.part, static_cast<uint16_t*>(a.o), a.lse, a.n_splits);
  return cudaGetLastError();
}

// Paged KV cache decode: same split and merge kernels, cache rows found through the block table.
template <int D>
static cudaError_t launch_decode_paged_d(const DecodePagedArgs& a, cudaStream_t stream) {
  using C = DecCfg<D>;
  const uint64_t bh = static_cast<uint64_t>(a.B) * a.H;
  DecParams p;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.block_size;
  if (!make_map_bf16_tok(&p.tk, a.k_cache, D, a.H, rows, 64, C::KEYS) ||
      !make_map_bf16_tok(&p.tv, a.v_cache, D, a.H, rows, 64, C::KEYS))
    return cudaErrorInvalidValue;
  p.q = static_cast<const uint16_t*>(a.q);
  p.part = a.part;
  p.n_kv = a.max_seqlen;
  p.bh = static_cast<int>(bh);
  p.n_splits = a.n_splits;
  p.chunk = a.chunk;
  p.n_items = static_cast<int>(bh) * a.n_splits;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.block_table = a.block_table;
  p.seqlens = a.seqlens;
  p.heads = a.H;
  p.block_size = a.block_size;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  static int attr_done[64] = {0};
  cudaError_t e = ensure_smem_attr(decode_split_kernel<D, true>, C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const int grid = min(p.n_items, 2 * sm_count());
  log_launch("decode_split_kernel<D, true>", static_cast<unsigned long long>(grid), C::THREADS, static_cast<unsigned long long>(C::SMEM_BYTES));
  decode_split_kernel<D, true><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  log_launch("decode_merge_kernel<D>", static_cast<unsigned long long>(static_cast<unsigned>(bh)), D, static_cast<unsigned long long>(0));
  decode_merge_kernel<D><<<static_cast<unsigned>(bh), D, 0, stream>>>(
      a.part, static_cast<uint16_t*>(a.o), a.lse, a.n_splits);
  return cudaGetLastError();
}

cudaError_t launch_decode_paged(const DecodePagedArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_decode_paged_d<64>(a, stream);
  return launch_decode_paged_d<128>(a, stream);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_decode_d<64>(a, stream);
  return launch_decode_d<128>(a, stream);
}

// ------------------------------------------------------------------------------------------
// Fixed scratch for fa_decode_splitkv_noalloc: the per-chunk states live in this array instead
// of a caller workspace.  It is part of the library image, so every GPU that loads the library
// holds it until the process exits.  Host code must not pass the symbol itself to a kernel
// (on the host it names a stand-in, not device memory): decode_noalloc_scratch() looks up the
// device address once per device with that device current.
// ------------------------------------------------------------------------------------------
static __device__ __align__(256) float g_decode_scratch[kDecodeNoallocScratchBytes / sizeof(float)];

cudaError_t decode_noalloc_scratch(float** ptr) {
  static float* cached[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64) {
    float* c = __atomic_load_n(&cached[dev], __ATOMIC_ACQUIRE);
    if (c) {
      *ptr = c;
      return cudaSuccess;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess) return e;
  if (dev < 64) __atomic_store_n(&cached[dev], static_cast<float*>(p), __ATOMIC_RELEASE);
  *ptr = static_cast<float*>(p);
  return cudaSuccess;
}

}  // namespace fa

FA_DEFINE_STATUS_FETCH(status_fetch_decode)
