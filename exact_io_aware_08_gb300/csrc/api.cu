// C ABI of libfa (declared in include/fa.h): argument validation, workspace carving, dispatch
// to the kernel launchers, device-status collection.  Nothing here allocates memory or falls
// back to another implementation: an unsupported call returns an error before any launch.
#include <cmath>
#include <cstdlib>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/fa.h"
#include "fa_kernels.h"

namespace fa {
// Process-wide diagnostic counters (fa_debug_counters); read by the launchers.
unsigned long long* g_debug_counters = nullptr;
unsigned long long* debug_counters() { return g_debug_counters; }

void log_launch(const char* kernel, unsigned long long grid, unsigned threads, unsigned long long smem) {
  static const bool on = [] {
    const char* v = std::getenv("FA_LOG");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
  }();
  if (on) std::fprintf(stderr, "[fa] launch %s grid=%llu block=%u smem=%llu\n", kernel, grid, threads, smem);
}
}  // namespace fa

namespace {

thread_local char g_msg[512] = "no error";

fa_status_t fail(fa_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

fa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared shape checks.  Returns FA_OK or an error (message set).
fa_status_t check_shape(int B, int H, int n_q, int n_kv, int d, float scale) {
  if (B < 1 || H < 1) return fail(FA_ERR_INVALID_ARG, "B and H must be >= 1 (got B=%d H=%d)", B, H);
  if (n_q < 0 || n_kv < 0)
    return fail(FA_ERR_INVALID_ARG, "sequence lengths must be >= 0 (got N_q=%d N_kv=%d)", n_q, n_kv);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim d=%d not supported (64 or 128)", d);
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", static_cast<double>(scale));
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1LL << 30)) return fail(FA_ERR_UNSUPPORTED, "B*H=%lld too large", bh);
  const long long lim = (1LL << 31) / d;
  if (n_q >= lim || n_kv >= lim)
    return fail(FA_ERR_UNSUPPORTED, "sequence length too large for d=%d (limit %lld)", d, lim);
  // grid of (query tiles x heads) must fit in gridDim.x
  const long long tiles = (static_cast<long long>(n_q) + 127) / 128;
  if (tiles * bh >= (1LL << 31)) return fail(FA_ERR_UNSUPPORTED, "too many (tile, head) work items");
  return FA_OK;
}

// The decode kernels index their (b, h, chunk) work items with 32-bit ints.
fa_status_t check_decode_items(int B, int H, int n_splits) {
  const long long items = static_cast<long long>(B) * H * n_splits;
  if (items >= (1LL << 31))
    return fail(FA_ERR_UNSUPPORTED, "B*H*n_splits=%lld too large (limit 2^31 - 1)", items);
  return FA_OK;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status_t s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

const char* fa_last_error_message(void) { return g_msg; }

fa_status_t fa_fwd(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v, fa_bf16_t* o,
                   float* lse, int B, int H, int N_q, int N_kv, int d, float scale, int causal,
                   void* stream) {
  fa_status_t st = check_shape(B, H, N_q, N_kv, d, scale);
  if (st != FA_OK) return st;
  if (causal && N_q != N_kv)
    return fail(FA_ERR_UNSUPPORTED, "causal requires N_q == N_kv (got %d, %d)", N_q, N_kv);
  if (N_q == 0) return FA_OK;
  if (!q || !o || !lse || (N_kv > 0 && (!k || !v)))
    return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  fa::FwdArgs a{q, k ? k : q, v ? v : q, o, lse, B, H, N_q, N_kv, d, scale, causal ? 1 : 0};
  if (N_kv == 0) { a.k = q; a.v = q; }   // maps need a valid base; no key tile is read
  cudaError_t e = fa::launch_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd launch");
  return FA_OK;
}

fa_status_t fa_fwd_fp8(const fa_e4m3_t* q, const fa_e4m3_t* k, const fa_e4m3_t* v, fa_bf16_t* o,
                       float* lse, int B, int H, int N_q, int N_kv, int d, float scale,
                       float descale_q, float descale_k, float descale_v, int causal,
                       void* stream) {
  fa_status_t st = check_shape(B, H, N_q, N_kv, d, scale);
  if (st != FA_OK) return st;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "the fp8 forward supports d = 128 only (got %d)", d);
  for (float ds : {descale_q, descale_k, descale_v})
    if (!std::isfinite(ds) || !(ds > 0.f))
      return fail(FA_ERR_INVALID_ARG, "descale factors must be finite and > 0 (got %g)",
                  static_cast<double>(ds));
  if (!std::isfinite(scale * descale_q * descale_k) || !(scale * descale_q * descale_k > 0.f))
    return fail(FA_ERR_INVALID_ARG, "scale * descale_q * descale_k must be a finite positive float");
  if (causal && N_q != N_kv)
    return fail(FA_ERR_UNSUPPORTED, "causal requires N_q == N_kv (got %d, %d)", N_q, N_kv);
  if (N_q == 0) return FA_OK;
  if (!q || !o || !lse || (N_kv > 0 && (!k || !v)))
    return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  fa::FwdArgs a{q, k ? k : q, v ? v : q, o, lse, B, H, N_q, N_kv, d, scale, causal ? 1 : 0};
  if (N_kv == 0) { a.k = q; a.v = q; }
  a.descale_q = descale_q;
  a.descale_k = descale_k;
  a.descale_v = descale_v;
  cudaError_t e = fa::launch_fwd_fp8(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_fp8 launch");
  return FA_OK;
}

fa_status_t fa_fwd_varlen(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          fa_bf16_t* o, float* lse, const int* cu_seqlens_q,
                          const int* cu_seqlens_k, int n_seqs, int H, int total_q, int total_k,
                          int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                          void* stream) {
  if (n_seqs < 1) return fail(FA_ERR_INVALID_ARG, "n_seqs must be >= 1 (got %d)", n_seqs);
  if (total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(FA_ERR_INVALID_ARG, "totals and max sequence lengths must be >= 0");
  if (max_seqlen_q > total_q || max_seqlen_k > total_k)
    return fail(FA_ERR_INVALID_ARG, "max_seqlen exceeds the total token count");
  fa_status_t st = check_shape(1, H, max_seqlen_q, max_seqlen_k, d, scale);
  if (st != FA_OK) return st;
  const long long lim = (1LL << 31) / (static_cast<long long>(d) * H);
  if (total_q >= lim || total_k >= lim)
    return fail(FA_ERR_UNSUPPORTED, "total tokens too large for H=%d d=%d", H, d);
  const long long items = ((static_cast<long long>(max_seqlen_q) + 255) / 256) * n_seqs * H;
  if (items >= (1LL << 31)) return fail(FA_ERR_UNSUPPORTED, "too many (block, sequence, head) items");
  if (total_q == 0 || max_seqlen_q == 0) return FA_OK;
  if (!q || !o || !lse || !cu_seqlens_q || !cu_seqlens_k || (total_k > 0 && (!k || !v)))
    return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  fa::FwdVarlenArgs a{};
  a.q = q; a.k = total_k ? k : q; a.v = total_k ? v : q; a.o = o; a.lse = lse;
  a.cu_q = cu_seqlens_q; a.cu_k = cu_seqlens_k;
  a.n_seqs = n_seqs; a.H = H; a.total_q = total_q; a.total_k = total_k;
  a.max_seqlen_q = max_seqlen_q; a.max_seqlen_k = max_seqlen_k; a.d = d; a.scale = scale;
  a.causal = causal ? 1 : 0;
  cudaError_t e = fa::launch_fwd_varlen(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_varlen launch");
  return FA_OK;
}

size_t fa_bwd_workspace_size(int B, int H, int N_q, int N_kv, int d) {
  if (B < 1 || H < 1 || N_q < 0 || N_kv < 0 || (d != 64 && d != 128)) return 0;
  return fa::bwd_dq_acc_bytes(B, H, N_q, d) + fa::bwd_delta_bytes(B, H, N_q);
}

}  // extern "C"

namespace {

// Validation shared by fa_bwd and its three steps.  ``need`` selects which arrays must be
// present: bit i for argument i of {q, k, v, o, lse, dO, dq, dk, dv}.
fa_status_t check_bwd(const void* const (&ptrs)[9], unsigned need, const void* ws, size_t ws_bytes,
                      int B, int H, int N_q, int N_kv, int d, float scale, int causal,
                      fa::BwdArgs* a) {
  fa_status_t st = check_shape(B, H, N_q, N_kv, d, scale);
  if (st != FA_OK) return st;
  if (causal && N_q != N_kv)
    return fail(FA_ERR_UNSUPPORTED, "causal requires N_q == N_kv (got %d, %d)", N_q, N_kv);
  const bool rows_q[9] = {true, false, false, true, true, true, true, false, false};
  for (int i = 0; i < 9; ++i) {
    const bool nonempty = rows_q[i] ? N_q > 0 : N_kv > 0;
    if ((need >> i & 1u) && nonempty && !ptrs[i])
      return fail(FA_ERR_INVALID_ARG, "null pointer argument (#%d)", i);
    if (ptrs[i] && !aligned16(ptrs[i])) return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  }
  const size_t need_ws = fa_bwd_workspace_size(B, H, N_q, N_kv, d);
  if (!ws || ws_bytes < need_ws || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(FA_ERR_WORKSPACE, "workspace must be >= %zu bytes and 256-byte aligned (got %zu)",
                need_ws, ws_bytes);
  *a = fa::BwdArgs{};
  a->q = ptrs[0]; a->k = ptrs[1]; a->v = ptrs[2]; a->o = ptrs[3];
  a->lse = static_cast<const float*>(ptrs[4]); a->dO = ptrs[5];
  a->dq = const_cast<void*>(ptrs[6]); a->dk = const_cast<void*>(ptrs[7]);
  a->dv = const_cast<void*>(ptrs[8]);
  a->dq_acc = static_cast<float*>(const_cast<void*>(ws));
  a->delta = reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(ws)) +
                                      fa::bwd_dq_acc_bytes(B, H, N_q, d));
  a->B = B; a->H = H; a->n_q = N_q; a->n_kv = N_kv; a->d = d; a->scale = scale;
  a->causal = causal ? 1 : 0;
  return FA_OK;
}

constexpr unsigned kNeedAll = 0x1FFu;
constexpr unsigned kNeedPrep = (1u << 3) | (1u << 5);                                  // o, dO
constexpr unsigned kNeedMain = 1u | 2u | 4u | (1u << 4) | (1u << 5) | (1u << 7) | (1u << 8);
constexpr unsigned kNeedFinish = 1u << 6;                                              // dq

}  // namespace

extern "C" {

fa_status_t fa_bwd(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                   const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO, fa_bf16_t* dq,
                   fa_bf16_t* dk, fa_bf16_t* dv, void* ws, size_t ws_bytes, int B, int H,
                   int N_q, int N_kv, int d, float scale, int causal, void* stream) {
  fa::BwdArgs a;
  const void* const ptrs[9] = {q, k, v, o, lse, dO, dq, dk, dv};
  fa_status_t st = check_bwd(ptrs, kNeedAll, ws, ws_bytes, B, H, N_q, N_kv, d, scale, causal, &a);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_bwd_prep(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_main(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_finish(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_bwd launch");
  return FA_OK;
}

fa_status_t fa_fwd_window(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          fa_bf16_t* o, float* lse, int B, int H, int N, int d, float scale,
                          int window_left, int window_right, void* stream) {
  fa_status_t st = check_shape(B, H, N, N, d, scale);
  if (st != FA_OK) return st;
  if (N == 0) return FA_OK;
  if (!q || !k || !v || !o || !lse) return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  fa::FwdArgs a{q, k, v, o, lse, B, H, N, N, d, scale, 0};
  a.windowed = true;
  a.win_left = window_left < 0 ? fa::kWinUnbounded : std::min(window_left, fa::kWinUnbounded);
  a.win_right = window_right < 0 ? fa::kWinUnbounded : std::min(window_right, fa::kWinUnbounded);
  cudaError_t e = fa::launch_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_window launch");
  return FA_OK;
}

fa_status_t fa_bwd_window(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO,
                          fa_bf16_t* dq, fa_bf16_t* dk, fa_bf16_t* dv, void* ws, size_t ws_bytes,
                          int B, int H, int N, int d, float scale, int window_left,
                          int window_right, void* stream) {
  fa::BwdArgs a;
  const void* const ptrs[9] = {q, k, v, o, lse, dO, dq, dk, dv};
  fa_status_t st = check_bwd(ptrs, kNeedAll, ws, ws_bytes, B, H, N, N, d, scale, 0, &a);
  if (st != FA_OK) return st;
  a.windowed = true;
  a.win_left = window_left < 0 ? fa::kWinUnbounded : std::min(window_left, fa::kWinUnbounded);
  a.win_right = window_right < 0 ? fa::kWinUnbounded : std::min(window_right, fa::kWinUnbounded);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_bwd_prep(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_main(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_finish(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_bwd_window launch");
  return FA_OK;
}

// Block-sparse calls: the mask must exist (unless a side is empty) and cover at most
// kBlockSparseMaxTiles key blocks.
static fa_status_t check_block_mask(const unsigned char* block_mask, int mask_per_head, int N_q,
                                    int N_kv) {
  if (mask_per_head != 0 && mask_per_head != 1)
    return fail(FA_ERR_INVALID_ARG, "mask_per_head must be 0 or 1 (got %d)", mask_per_head);
  if (N_q > 0 && N_kv > 0 && !block_mask) return fail(FA_ERR_INVALID_ARG, "null block_mask");
  const int kb = (N_kv + fa::kBlockSize - 1) / fa::kBlockSize;
  if (kb > fa::kBlockSparseMaxTiles)
    return fail(FA_ERR_UNSUPPORTED, "block-sparse attention covers at most %d key blocks (N_kv <= %d; got %d)",
                fa::kBlockSparseMaxTiles, fa::kBlockSparseMaxTiles * fa::kBlockSize, N_kv);
  return FA_OK;
}

fa_status_t fa_fwd_block_sparse(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                                fa_bf16_t* o, float* lse, int B, int H, int N_q, int N_kv, int d,
                                float scale, int causal, const unsigned char* block_mask,
                                int mask_per_head, void* stream) {
  fa_status_t st = check_shape(B, H, N_q, N_kv, d, scale);
  if (st != FA_OK) return st;
  if (causal && N_q != N_kv)
    return fail(FA_ERR_UNSUPPORTED, "causal requires N_q == N_kv (got %d, %d)", N_q, N_kv);
  st = check_block_mask(block_mask, mask_per_head, N_q, N_kv);
  if (st != FA_OK) return st;
  if (N_q == 0) return FA_OK;
  if (!q || !o || !lse || (N_kv > 0 && (!k || !v)))
    return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  fa::FwdArgs a{q, k ? k : q, v ? v : q, o, lse, B, H, N_q, N_kv, d, scale, causal ? 1 : 0};
  if (N_kv == 0) {
    a.k = q;                             // no key at all: the plain kernel writes O = 0, lse = -inf
    a.v = q;
  } else {
    a.block_mask = reinterpret_cast<const uint8_t*>(block_mask);
    a.bm_per_head = mask_per_head;
  }
  cudaError_t e = fa::launch_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_block_sparse launch");
  return FA_OK;
}

fa_status_t fa_bwd_block_sparse(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                                const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO,
                                fa_bf16_t* dq, fa_bf16_t* dk, fa_bf16_t* dv, void* ws,
                                size_t ws_bytes, int B, int H, int N_q, int N_kv, int d,
                                float scale, int causal, const unsigned char* block_mask,
                                int mask_per_head, void* stream) {
  fa::BwdArgs a;
  const void* const ptrs[9] = {q, k, v, o, lse, dO, dq, dk, dv};
  fa_status_t st = check_bwd(ptrs, kNeedAll, ws, ws_bytes, B, H, N_q, N_kv, d, scale, causal, &a);
  if (st != FA_OK) return st;
  st = check_block_mask(block_mask, mask_per_head, N_q, N_kv);
  if (st != FA_OK) return st;
  a.block_mask = reinterpret_cast<const uint8_t*>(block_mask);
  a.bm_per_head = mask_per_head;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_bwd_prep(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_main(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_finish(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_bwd_block_sparse launch");
  return FA_OK;
}

fa_status_t fa_bwd_prep(const fa_bf16_t* o, const fa_bf16_t* dO, void* ws, size_t ws_bytes,
                        int B, int H, int N_q, int N_kv, int d, void* stream) {
  fa::BwdArgs a;
  const void* const ptrs[9] = {nullptr, nullptr, nullptr, o, nullptr, dO, nullptr, nullptr, nullptr};
  fa_status_t st = check_bwd(ptrs, kNeedPrep, ws, ws_bytes, B, H, N_q, N_kv, d, 1.f, 0, &a);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_bwd_prep(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "fa_bwd_prep launch");
}

fa_status_t fa_bwd_main(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                        const float* lse, const fa_bf16_t* dO, fa_bf16_t* dk, fa_bf16_t* dv,
                        void* ws, size_t ws_bytes, int B, int H, int N_q, int N_kv, int d,
                        float scale, int causal, void* stream) {
  fa::BwdArgs a;
  const void* const ptrs[9] = {q, k, v, nullptr, lse, dO, nullptr, dk, dv};
  fa_status_t st = check_bwd(ptrs, kNeedMain, ws, ws_bytes, B, H, N_q, N_kv, d, scale, causal, &a);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_bwd_main(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "fa_bwd_main launch");
}

fa_status_t fa_bwd_finish(fa_bf16_t* dq, const void* ws, size_t ws_bytes, int B, int H, int N_q,
                          int N_kv, int d, float scale, void* stream) {
  fa::BwdArgs a;
  const void* const ptrs[9] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr};
  fa_status_t st = check_bwd(ptrs, kNeedFinish, ws, ws_bytes, B, H, N_q, N_kv, d, scale, 0, &a);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_bwd_finish(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e, "fa_bwd_finish launch");
}

fa_status_t fa_bwd_varlen(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO,
                          fa_bf16_t* dq, fa_bf16_t* dk, fa_bf16_t* dv, void* ws, size_t ws_bytes,
                          const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H,
                          int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                          float scale, int causal, void* stream) {
  if (n_seqs < 1) return fail(FA_ERR_INVALID_ARG, "n_seqs must be >= 1 (got %d)", n_seqs);
  if (total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(FA_ERR_INVALID_ARG, "totals and max sequence lengths must be >= 0");
  if (max_seqlen_q > total_q || max_seqlen_k > total_k)
    return fail(FA_ERR_INVALID_ARG, "max_seqlen exceeds the total token count");
  if (!cu_seqlens_q || !cu_seqlens_k) return fail(FA_ERR_INVALID_ARG, "null cu_seqlens");
  const long long lim = (1LL << 31) / (static_cast<long long>(d > 0 ? d : 1) * (H > 0 ? H : 1));
  if (total_q >= lim || total_k >= lim)
    return fail(FA_ERR_UNSUPPORTED, "total tokens too large for H=%d d=%d", H, d);
  const long long items = ((static_cast<long long>(max_seqlen_k) + 127) / 128) * n_seqs * (H > 0 ? H : 1);
  if (items >= (1LL << 31)) return fail(FA_ERR_UNSUPPORTED, "too many (key tile, sequence, head) items");
  // the packed layout is one [1, H, total, d]-sized problem for the prep and finish steps
  fa::BwdArgs a;
  const void* const ptrs[9] = {q, k, v, o, lse, dO, dq, dk, dv};
  fa_status_t st = check_bwd(ptrs, kNeedAll, ws, ws_bytes, 1, H, total_q, total_k, d, scale, 0, &a);
  if (st != FA_OK) return st;
  if (total_q == 0 && total_k == 0) return FA_OK;
  a.causal = causal ? 1 : 0;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.n_seqs = n_seqs;
  a.total_q = total_q;
  a.total_k = total_k;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_bwd_prep(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_main(a, s);
  if (e == cudaSuccess) e = fa::launch_bwd_finish(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_bwd_varlen launch");
  return FA_OK;
}

size_t fa_decode_workspace_size(int B, int H, int N_kv, int d, int n_splits) {
  if (B < 1 || H < 1 || N_kv < 0 || (d != 64 && d != 128)) return 0;
  if (n_splits <= 0) n_splits = fa::decode_auto_splits(B, H, N_kv);
  if (n_splits > fa::kDecodeMaxSplits) return 0;
  if (static_cast<long long>(B) * H * n_splits >= (1LL << 31)) return 0;
  return fa::decode_part_bytes(B, H, d, n_splits);
}

fa_status_t fa_decode_splitkv(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                              fa_bf16_t* o, float* lse, int B, int H, int N_kv, int d,
                              float scale, int n_splits, void* ws, size_t ws_bytes,
                              void* stream) {
  fa_status_t st = check_shape(B, H, 1, N_kv, d, scale);
  if (st != FA_OK) return st;
  if (n_splits > fa::kDecodeMaxSplits)
    return fail(FA_ERR_UNSUPPORTED, "n_splits=%d exceeds %d", n_splits, fa::kDecodeMaxSplits);
  if (n_splits <= 0) n_splits = fa::decode_auto_splits(B, H, N_kv);
  if ((st = check_decode_items(B, H, n_splits)) != FA_OK) return st;
  if (!q || !o || !lse || (N_kv > 0 && (!k || !v)))
    return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  const size_t need_ws = fa::decode_part_bytes(B, H, d, n_splits);
  if (!ws || ws_bytes < need_ws || !aligned16(ws))
    return fail(FA_ERR_WORKSPACE, "workspace must be >= %zu bytes and 16-byte aligned (got %zu)",
                need_ws, ws_bytes);
  fa::DecodeArgs a{};
  a.q = q; a.k = N_kv ? k : q; a.v = N_kv ? v : q; a.o = o; a.lse = lse;
  a.part = static_cast<float*>(ws);
  a.B = B; a.H = H; a.n_kv = N_kv; a.d = d; a.scale = scale; a.n_splits = n_splits;
  a.chunk = fa::decode_chunk(N_kv, n_splits);
  cudaError_t e = fa::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv launch");
  return FA_OK;
}

fa_status_t fa_decode_splitkv_noalloc(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                                      fa_bf16_t* o, float* lse, int B, int H, int N_kv, int d,
                                      float scale, int n_splits, void* stream) {
  fa_status_t st = check_shape(B, H, 1, N_kv, d, scale);
  if (st != FA_OK) return st;
  if (n_splits > fa::kDecodeMaxSplits)
    return fail(FA_ERR_UNSUPPORTED, "n_splits=%d exceeds %d", n_splits, fa::kDecodeMaxSplits);
  if (n_splits <= 0) n_splits = fa::decode_auto_splits(B, H, N_kv);
  if ((st = check_decode_items(B, H, n_splits)) != FA_OK) return st;
  if (!q || !o || !lse || (N_kv > 0 && (!k || !v)))
    return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  const size_t need = fa::decode_part_bytes(B, H, d, n_splits);
  if (need > fa::kDecodeNoallocScratchBytes)
    return fail(FA_ERR_UNSUPPORTED,
                "fa_decode_splitkv_noalloc: B*H*n_splits*(d+2)*4 = %zu bytes exceeds the fixed "
                "scratch of %zu bytes; use fa_decode_splitkv with a workspace or fewer splits",
                need, fa::kDecodeNoallocScratchBytes);
  float* scratch = nullptr;
  cudaError_t e = fa::decode_noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_noalloc scratch lookup");
  fa::DecodeArgs a{};
  a.q = q; a.k = N_kv ? k : q; a.v = N_kv ? v : q; a.o = o; a.lse = lse;
  a.part = scratch;
  a.B = B; a.H = H; a.n_kv = N_kv; a.d = d; a.scale = scale; a.n_splits = n_splits;
  a.chunk = fa::decode_chunk(N_kv, n_splits);
  e = fa::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_noalloc launch");
  return FA_OK;
}

fa_status_t fa_decode_paged(const fa_bf16_t* q, const fa_bf16_t* k_cache,
                            const fa_bf16_t* v_cache, fa_bf16_t* o, float* lse,
                            const int* block_table, const int* seqlens_k, int B, int H,
                            int max_blocks_per_seq, int block_size, int num_blocks,
                            int max_seqlen_k, int d, float scale, int n_splits, void* ws,
                            size_t ws_bytes, void* stream) {
  fa_status_t st = check_shape(B, H, 1, max_seqlen_k, d, scale);
  if (st != FA_OK) return st;
  if (block_size < 64 || block_size % 64 != 0)
    return fail(FA_ERR_UNSUPPORTED, "block_size must be a positive multiple of 64 (got %d)",
                block_size);
  if (num_blocks < 1 || max_blocks_per_seq < 1)
    return fail(FA_ERR_INVALID_ARG, "num_blocks and max_blocks_per_seq must be >= 1 (got %d, %d)",
                num_blocks, max_blocks_per_seq);
  if (static_cast<long long>(num_blocks) * block_size >= (1LL << 31))
    return fail(FA_ERR_UNSUPPORTED, "num_blocks * block_size must be < 2^31");
  if (static_cast<long long>(max_seqlen_k) > static_cast<long long>(max_blocks_per_seq) * block_size)
    return fail(FA_ERR_INVALID_ARG, "max_seqlen_k=%d exceeds max_blocks_per_seq * block_size",
                max_seqlen_k);
  if (n_splits > fa::kDecodeMaxSplits)
    return fail(FA_ERR_UNSUPPORTED, "n_splits=%d exceeds %d", n_splits, fa::kDecodeMaxSplits);
  if (n_splits <= 0) n_splits = fa::decode_auto_splits(B, H, max_seqlen_k);
  if ((st = check_decode_items(B, H, n_splits)) != FA_OK) return st;
  if (!q || !k_cache || !v_cache || !o || !lse || !block_table || !seqlens_k)
    return fail(FA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      !aligned16(lse))
    return fail(FA_ERR_INVALID_ARG, "arrays must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(seqlens_k)) & 3u)
    return fail(FA_ERR_INVALID_ARG, "block_table and seqlens_k must be 4-byte aligned");
  const size_t need_ws = fa::decode_part_bytes(B, H, d, n_splits);
  if (!ws || ws_bytes < need_ws || !aligned16(ws))
    return fail(FA_ERR_WORKSPACE, "workspace must be >= %zu bytes and 16-byte aligned (got %zu)",
                need_ws, ws_bytes);
  fa::DecodePagedArgs a{};
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.o = o; a.lse = lse;
  a.part = static_cast<float*>(ws);
  a.block_table = block_table; a.seqlens = seqlens_k;
  a.B = B; a.H = H; a.d = d; a.num_blocks = num_blocks; a.block_size = block_size;
  a.max_blocks = max_blocks_per_seq; a.max_seqlen = max_seqlen_k;
  a.scale = scale; a.n_splits = n_splits;
  a.chunk = fa::decode_chunk(max_seqlen_k, n_splits);
  cudaError_t e = fa::launch_decode_paged(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_paged launch");
  return FA_OK;
}

fa_status_t fa_debug_counters(unsigned long long* device_counters) {
  fa::g_debug_counters = device_counters;
  return FA_OK;
}

fa_status_t fa_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 10u * 1000u * 1000u)
    return fail(FA_ERR_INVALID_ARG, "limit_us must be in [1, 10000000] (got %u)", limit_us);
  cudaError_t e = fa::launch_selftest_wait(static_cast<unsigned long long>(limit_us) * 1000ull,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_selftest_wait_timeout launch");
  return FA_OK;
}

fa_status_t fa_sync_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int code = 0, c = 0;
  int where = 0, w = 0;
  cudaError_t (*fetch[])(cudaStream_t, unsigned int*, int*) = {
      fa::status_fetch_fwd, fa::status_fetch_bwd, fa::status_fetch_decode,
      fa::status_fetch_selftest};
  for (auto f : fetch) {
    cudaError_t e = f(s, &c, &w);
    if (e != cudaSuccess) return cuda_fail(e, "fa_sync_status");
    if (c) { code |= c; where = w; }
  }
  if (code & fa::FA_DEV_TIMEOUT)
    return fail(FA_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out (site %d)", where);
  if (code & fa::FA_DEV_BAD_CONFIG)
    return fail(FA_ERR_INVALID_ARG,
                "a kernel found invalid sequence boundaries (cu_seqlens / max_seqlen) (site %d)",
                where);
  if (code) return fail(FA_ERR_CUDA, "device reported error code %u (site %d)", code, where);
  return FA_OK;
}

}  // extern "C"
