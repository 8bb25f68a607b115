// Internal launcher interface between the C ABI (api.cu) and the kernel translation units.
// Arguments arrive here already validated.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "host_tma.h"

namespace fa {

// Codes kernels record in their translation unit's device status word.
enum DevError : unsigned int {
  FA_DEV_TIMEOUT = 1u,       // a bounded mbarrier wait ran out
  FA_DEV_BAD_CONFIG = 2u,    // kernel found launch geometry it was not built for
};

// "No bound on this side" for attention windows: query i sees keys j with
// i - win_left <= j <= i + win_right.
constexpr int kWinUnbounded = 1 << 30;

// Diagnostic counters (device memory, set through fa_debug_counters; null = off): kernels add
// [0] the forward S products (query tile x key tile) they computed, [1] the backward
// (key tile, query step) pairs they visited.
unsigned long long* debug_counters();

// Host-side launch log: with the environment variable FA_LOG set to a non-empty value other
// than 0, every kernel launch is written to stderr (kernel, grid, block, dynamic shared memory).
void log_launch(const char* kernel, unsigned long long grid, unsigned threads, unsigned long long smem);

// Block-sparse attention: blocks are 128 queries x 128 keys, and a call covers at most this
// many key blocks (N_kv <= 131072), the length of the per-CTA stream list kept on chip.
constexpr int kBlockSize = 128;
constexpr int kBlockSparseMaxTiles = 1024;

// Causal work items differ in length (a query pair or key tile near the start of a head has
// the most partners).  The kernels map blockIdx so that items run longest-first across groups
// of this many heads: the CTAs that start last are short ones, while the heads in flight
// (about one group and a half) keep their K/V or Q/dO in L2.
constexpr int kCausalGroup = 8;

// (head, rank) of CTA ``block`` in a grid of n_bh heads x per_head items: rank 0 first across
// the heads of a group, then rank 1, ...  A bijection onto [0, n_bh) x [0, per_head).
__device__ __forceinline__ void causal_item(int block, int n_bh, int per_head, int* bh, int* rank) {
  const int per_group = kCausalGroup * per_head;
  const int g0 = (block / per_group) * kCausalGroup;
  const int g = min(kCausalGroup, n_bh - g0);          // heads in this (possibly last) group
  const int w = block - (g0 / kCausalGroup) * per_group;
  *rank = w / g;
  *bh = g0 + w % g;
}

// Item k of a persistent CTA: rounds of gridDim.x items, walked forward in even rounds and
// backward in odd ones, so that with items ordered longest first every CTA gets a similar total.
__device__ __forceinline__ int pers_item(int k, int G) {
  return k * G + ((k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
}

// Window of a call: an explicit window (win_left / win_right >= 0 or kWinUnbounded) when
// ``windowed``, else causal = (unbounded, 0) or no mask = (unbounded, unbounded).
inline void attention_window(int causal, bool windowed, int left, int right, int* wl, int* wr) {
  *wl = windowed ? left : kWinUnbounded;
  *wr = windowed ? right : (causal ? 0 : kWinUnbounded);
}

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, n_q, n_kv, d;
  float scale;
  int causal;
  float descale_q = 1.f, descale_k = 1.f, descale_v = 1.f;   // fp8 forward only
  bool windowed = false;                                     // sliding window (below)
  int win_left = kWinUnbounded, win_right = kWinUnbounded;
  const uint8_t* block_mask = nullptr;                       // block-sparse (device, below)
  int bm_per_head = 0;
};

struct FwdVarlenArgs {
  const void* q;     // [total_q, H, d]
  const void* k;     // [total_k, H, d]
  const void* v;
  void* o;           // [total_q, H, d]
  float* lse;        // [H, total_q]
  const int* cu_q;   // [n_seqs + 1], device
  const int* cu_k;
  int n_seqs, H, total_q, total_k, max_seqlen_q, max_seqlen_k, d;
  float scale;
  int causal;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;     // fp32 [B,H,N_q,d] workspace
  float* delta;      // fp32 [B,H,N_q]   workspace (D = rowsum(dO o O))
  int B, H, n_q, n_kv, d;
  float scale;
  int causal;
  // variable-length batches (cu_q != nullptr): packed [total, H, d] tensors; the prep and
  // finish steps then run over B = 1, n_q = total_q rows of the packed layout
  const int* cu_q = nullptr;
  const int* cu_k = nullptr;
  int n_seqs = 0, total_q = 0, total_k = 0, max_seqlen_q = 0, max_seqlen_k = 0;
  bool windowed = false;                                     // sliding window (as FwdArgs)
  int win_left = kWinUnbounded, win_right = kWinUnbounded;
  const uint8_t* block_mask = nullptr;                       // block-sparse (as FwdArgs)
  int bm_per_head = 0;
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  float* part;       // fp32 [B*H, n_splits, d + 2]: (o~[d], m, l) per chunk
  int B, H, n_kv, d;
  float scale;
  int n_splits;
  int chunk;         // keys per split (multiple of the kernel's key step)
};

struct DecodePagedArgs {
  const void* q;            // [B, H, d]
  const void* k_cache;      // [num_blocks, block_size, H, d]
  const void* v_cache;
  void* o;                  // [B, H, d]
  float* lse;               // [B, H]
  float* part;              // workspace, as for DecodeArgs
  const int* block_table;   // [B, max_blocks], device
  const int* seqlens;       // [B], device
  int B, H, d, num_blocks, block_size, max_blocks, max_seqlen;
  float scale;
  int n_splits, chunk;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream);   // d = 128 only
cudaError_t launch_fwd_varlen(const FwdVarlenArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t stream);    // F2
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream);    // F3
cudaError_t launch_bwd_finish(const BwdArgs& a, cudaStream_t stream);  // F4
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_paged(const DecodePagedArgs& a, cudaStream_t stream);

// Per-TU device status accessors (see fa_status.cuh).
cudaError_t status_fetch_fwd(cudaStream_t, unsigned int*, int*);
cudaError_t status_fetch_bwd(cudaStream_t, unsigned int*, int*);
cudaError_t status_fetch_decode(cudaStream_t, unsigned int*, int*);
cudaError_t status_fetch_selftest(cudaStream_t, unsigned int*, int*);

// Diagnostic kernel: a bounded wait that is never satisfied (selftest.cu).
cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

// Workspace layout of the backward pass.
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t bwd_dq_acc_bytes(int B, int H, int n_q, int d) {
  return align_up(static_cast<size_t>(B) * H * n_q * d * sizeof(float), 256);
}
inline size_t bwd_delta_bytes(int B, int H, int n_q) {
  return align_up(static_cast<size_t>(B) * H * n_q * sizeof(float), 256);
}

// Decode split policy: keys per chunk are a multiple of 64; n_splits <= 0 picks a count that
// gives every SM several CTAs when B*H alone does not.
constexpr int kDecodeKeyStep = 64;
constexpr int kDecodeMaxSplits = 1024;
inline int decode_auto_splits(int B, int H, int n_kv) {
  const long long bh = static_cast<long long>(B) * H;
  const long long want_ctas = 152LL * 8;
  long long s = (want_ctas + bh - 1) / bh;
  const long long max_by_len = (n_kv + 255) / 256;       // at least ~256 keys per chunk
  if (s > max_by_len) s = max_by_len;
  if (s < 1) s = 1;
  if (s > kDecodeMaxSplits) s = kDecodeMaxSplits;
  return static_cast<int>(s);
}
inline int decode_chunk(int n_kv, int n_splits) {
  int c = (n_kv + n_splits - 1) / n_splits;
  c = (c + kDecodeKeyStep - 1) / kDecodeKeyStep * kDecodeKeyStep;
  return c < kDecodeKeyStep ? kDecodeKeyStep : c;
}
inline size_t decode_part_bytes(int B, int H, int d, int n_splits) {
  return static_cast<size_t>(B) * H * n_splits * (d + 2) * sizeof(float);
}

// Size of the fixed device scratch behind fa_decode_splitkv_noalloc (decode.cu).
constexpr size_t kDecodeNoallocScratchBytes = size_t(8) << 20;
// Device address of that scratch on the current device (looked up once per device).
cudaError_t decode_noalloc_scratch(float** ptr);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device).  ``done`` is a
// per-kernel flag array owned by the caller (kernels of the same signature must not share one).
// A kernel that moves registers between warpgroups with setmaxnreg passes its thread count and
// the registers its split needs: setmaxnreg draws only on what the CTA was launched with
// (threads x registers per thread, the compiler's choice), and a split above that would wait
// forever, so the launch is refused (cudaErrorInvalidConfiguration) instead.
template <typename F>
cudaError_t ensure_smem_attr(F* func, int bytes, int (&done)[64], int threads = 0, int reg_need = 0) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && __atomic_load_n(&done[dev], __ATOMIC_ACQUIRE)) return cudaSuccess;
  if (reg_need > 0) {
    cudaFuncAttributes at;
    if ((e = cudaFuncGetAttributes(&at, func)) != cudaSuccess) return e;
    if (at.numRegs * threads < reg_need) return cudaErrorInvalidConfiguration;
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
  return e;
}

}  // namespace fa
