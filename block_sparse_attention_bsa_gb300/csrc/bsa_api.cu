// C ABI of libbsa: argument validation, workspace sizing, error reporting and
// the launch of the selector / forward / validation kernels.  Every function
// here follows the contract written in include/bsa.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <cmath>
#include <cstdint>
#include <string>

#include "bsa_internal.h"

namespace bsa {

namespace {
thread_local std::string g_last_error;
}

bsa_status set_error(bsa_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

void clear_error() { g_last_error.clear(); }

bsa_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return BSA_OK;
  return set_error(BSA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                     cudaGetErrorString(e) + ")");
}

int num_sms() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's cuTensorMapEncodeTiled, looked up once per process.
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}
}  // namespace

bsa_status encode_tensor_map(CUtensorMap* m, const void* base, int64_t rows, int64_t H, int D, int64_t ss,
                             int64_t sh, int box_rows, const char* name) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(BSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)H};
  cuuint64_t strides[2] = {(cuuint64_t)(ss * 2), (cuuint64_t)(sh * 2)};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(BSA_ERR_CUDA, std::string("cuTensorMapEncodeTiled failed for ") + name + " (CUresult " +
                                       std::to_string((int)r) + ")");
  return BSA_OK;
}

size_t select_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int d, int bq, int bk) {
  const size_t nQb = (size_t)cdiv64(Sq, bq), nKb = (size_t)cdiv64(Skv, bk);
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)B * Hq * nQb * d * sizeof(float)) + al((size_t)B * Hkv * nKb * d * sizeof(float));
}

namespace {

std::string s(int64_t v) { return std::to_string(v); }

bool supported_geometry(int bq, int bk) {
  return (bq == 64 || bq == 128 || bq == 256) && (bk == 64 || bk == 128);
}

bsa_status check_tensor(const bsa_tensor* t, const char* fn, const char* name) {
  if (!t) return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": " + name + " descriptor is NULL");
  if (!t->ptr) return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": " + name + "->ptr is NULL");
  if (t->B <= 0 || t->S <= 0 || t->H <= 0 || t->D <= 0)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": " + name + " has a non-positive dim [" +
                                              s(t->B) + "," + s(t->S) + "," + s(t->H) + "," + s(t->D) + "]");
  if (t->D != 64 && t->D != 128)
    return set_error(BSA_ERR_UNSUPPORTED, std::string(fn) + ": head dim " + s(t->D) + " of " + name +
                                              " is not supported (64 or 128)");
  if ((reinterpret_cast<uintptr_t>(t->ptr) & 15u) != 0)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": " + name + "->ptr is not 16-byte aligned");
  if ((t->stride_b % 8) || (t->stride_s % 8) || (t->stride_h % 8))
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": " + name +
                                              " strides must be multiples of 8 elements (16 bytes); got (" +
                                              s(t->stride_b) + "," + s(t->stride_s) + "," + s(t->stride_h) + ")");
  if (t->stride_b <= 0 || t->stride_s <= 0 || t->stride_h <= 0)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": " + name + " strides must be positive");
  return BSA_OK;
}

// Shared shape checks of select and forward.
bsa_status check_common(const char* fn, const bsa_tensor* q, const bsa_tensor* k, int32_t prefix_len,
                        const int32_t* seq_lens, int32_t bq, int32_t bk, int max_batch) {
  bsa_status st;
  if ((st = check_tensor(q, fn, "q")) != BSA_OK) return st;
  if ((st = check_tensor(k, fn, "k")) != BSA_OK) return st;
  if (q->B != k->B)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": batch of q (" + s(q->B) + ") != batch of k (" + s(k->B) + ")");
  if (q->D != k->D)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": head dim of q (" + s(q->D) + ") != head dim of k (" + s(k->D) + ")");
  if (q->H % k->H != 0)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": Hq (" + s(q->H) + ") is not a multiple of Hkv (" + s(k->H) + ")");
  if (q->H > kMaxHeads)
    return set_error(BSA_ERR_UNSUPPORTED, std::string(fn) + ": Hq " + s(q->H) + " above the limit " + s(kMaxHeads));
  if (q->B > max_batch)
    return set_error(BSA_ERR_UNSUPPORTED, std::string(fn) + ": batch " + s(q->B) + " above the limit " + s(max_batch));
  if (!supported_geometry(bq, bk))
    return set_error(BSA_ERR_UNSUPPORTED, std::string(fn) + ": block geometry (block_q=" + s(bq) + ", block_k=" +
                                              s(bk) + ") is not supported; block_q in {64,128,256}, block_k in {64,128}");
  if (prefix_len < 0)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": prefix_len " + s(prefix_len) + " is negative");
  if (q->S > INT32_MAX / 2 || k->S > INT32_MAX / 2)
    return set_error(BSA_ERR_UNSUPPORTED, std::string(fn) + ": sequence too long");
  for (int64_t b = 0; b < q->B; ++b) {
    const int64_t L = seq_lens ? seq_lens[b] : q->S;
    if (L < 0 || L > q->S)
      return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": seq_lens[" + s(b) + "] = " + s(L) +
                                                " outside [0, Sq=" + s(q->S) + "]");
    if ((int64_t)prefix_len + L > k->S)
      return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": prefix_len + seq_lens[" + s(b) + "] = " +
                                                s(prefix_len + L) + " exceeds Skv = " + s(k->S));
  }
  return BSA_OK;
}

bsa_status check_workspace(const char* fn, void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return BSA_OK;
  if (!ws) return set_error(BSA_ERR_WORKSPACE, std::string(fn) + ": workspace is NULL (needs " + s((int64_t)need) + " bytes)");
  if (ws_bytes < need)
    return set_error(BSA_ERR_WORKSPACE, std::string(fn) + ": workspace of " + s((int64_t)ws_bytes) +
                                            " bytes is smaller than the " + s((int64_t)need) + " bytes needed");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return set_error(BSA_ERR_WORKSPACE, std::string(fn) + ": workspace is not 256-byte aligned");
  return BSA_OK;
}

// One thread per row (b, h, qb): checks the list against the geometry.
struct ValidateParams {
  const int32_t* indices;
  const int32_t* counts;
  int B, Hq, nQb, nKb, block_q, block_k, prefix_len, require_prefix;
  int seq_lens[kMaxSelectBatch];
  int32_t* bad;
};

__global__ void validate_kernel(const __grid_constant__ ValidateParams p) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rows = (int64_t)p.B * p.Hq * p.nQb;
  if (row >= rows) return;
  const int qb = (int)(row % p.nQb);
  const int b = (int)(row / ((int64_t)p.Hq * p.nQb));
  const int L = p.seq_lens[b];
  const int valid_kv = p.prefix_len + L;
  const int nkv = (valid_kv + p.block_k - 1) / p.block_k;
  const int npb = min((p.prefix_len + p.block_k - 1) / p.block_k, nkv);
  const int c = p.counts[row];
  bool bad = false;
  if (qb * p.block_q >= L) {
    bad = c != 0;
  } else if (c < 0 || c > nkv) {
    bad = true;
  } else {
    const int32_t* r = p.indices + row * p.nKb;
    int prev = -1;
    for (int j = 0; j < c && !bad; ++j) {
      const int kb = r[j];
      if (kb < 0 || kb >= nkv || kb <= prev) bad = true;
      if (p.require_prefix && j < npb && kb != j) bad = true;
      prev = kb;
    }
    if (p.require_prefix && c < npb) bad = true;
  }
  if (bad) atomicAdd(p.bad, 1);
}

// BSA_DEBUG validation: malformed index-list rows that reached bsa_forward or
// bsa_backward, counted on the device and reported by bsa_device_status().
__device__ int g_debug_bad_rows = 0;

bool debug_validation() {
  const char* e = std::getenv("BSA_DEBUG");
  return e && *e && std::strcmp(e, "0") != 0;
}

// Enqueues validate_kernel (no prefix requirement) over the lists of every
// request, 64 requests per launch, counting malformed rows into
// g_debug_bad_rows.  Adds no synchronisation.
bsa_status debug_validate_lists(const int32_t* indices, const int32_t* counts, int B, int Hq, int Sq, int Skv,
                                int prefix_len, const int32_t* seq_lens, int block_q, int block_k,
                                cudaStream_t s) {
  int32_t* bad = nullptr;
  bsa_status st = cuda_check(cudaGetSymbolAddress(reinterpret_cast<void**>(&bad), g_debug_bad_rows),
                             "cudaGetSymbolAddress(BSA_DEBUG counter)");
  if (st != BSA_OK) return st;
  const int nQb = (int)cdiv64(Sq, block_q), nKb = (int)cdiv64(Skv, block_k);
  for (int b0 = 0; b0 < B; b0 += kMaxSelectBatch) {
    ValidateParams p{};
    const int Bn = B - b0 < kMaxSelectBatch ? B - b0 : kMaxSelectBatch;
    const int64_t first_row = (int64_t)b0 * Hq * nQb;
    p.indices = indices + first_row * nKb;
    p.counts = counts + first_row;
    p.B = Bn; p.Hq = Hq; p.nQb = nQb; p.nKb = nKb;
    p.block_q = block_q; p.block_k = block_k; p.prefix_len = prefix_len; p.require_prefix = 0;
    for (int i = 0; i < Bn; ++i) p.seq_lens[i] = seq_lens ? seq_lens[b0 + i] : Sq;
    p.bad = bad;
    const int64_t rows = (int64_t)Bn * Hq * nQb;
    validate_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "validate_kernel launch (BSA_DEBUG)")) != BSA_OK) return st;
  }
  return BSA_OK;
}

}  // namespace
}  // namespace bsa

using namespace bsa;

extern "C" {

int bsa_version(void) { return 100; }

const char* bsa_get_last_error(void) { return g_last_error.c_str(); }

size_t bsa_select_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int d, int block_q, int block_k) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || d <= 0 || block_q <= 0 || block_k <= 0) return 0;
  return select_workspace_bytes(B, Hq, Hkv, Sq, Skv, d, block_q, block_k);
}

}  // extern "C"

namespace bsa {
// Shared body of bsa_select, bsa_select_rope and bsa_select_noalloc (`rope`
// carries the tables and rotated outputs, or is NULL; `static_scratch`, when
// given, supplies the workspace after every argument has been checked).
bsa_status select_impl(const char* fn, const bsa_tensor* q, const bsa_tensor* k, int32_t prefix_len,
                       const int32_t* seq_lens, int32_t block_q, int32_t block_k, const float* keep_ratio,
                       int32_t n_keep, int32_t* indices, int32_t* counts, void* workspace, size_t ws_bytes,
                       bsa_stream_t stream, const SelectArgs* rope, StaticScratchFn static_scratch) {
  bsa_status st = check_common(fn, q, k, prefix_len, seq_lens, block_q, block_k, kMaxSelectBatch);
  if (st != BSA_OK) return st;
  if (!keep_ratio) return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": keep_ratio is NULL");
  if (n_keep != 1 && n_keep != q->H)
    return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": n_keep = " + std::to_string(n_keep) + " must be 1 or Hq = " +
                                              std::to_string(q->H));
  float keep[kMaxHeads];
  for (int h = 0; h < q->H; ++h) {
    const float r = keep_ratio[n_keep == 1 ? 0 : h];
    if (!(r >= 0.f && r <= 1.f))
      return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": keep_ratio[" + std::to_string(n_keep == 1 ? 0 : h) +
                                                "] = " + std::to_string(r) + " outside [0, 1]");
    keep[h] = r;
  }
  if (!indices) return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": indices is NULL");
  if (!counts) return set_error(BSA_ERR_INVALID_ARG, std::string(fn) + ": counts is NULL");
  const size_t need = select_workspace_bytes((int)q->B, (int)q->H, (int)k->H, (int)q->S, (int)k->S, (int)q->D,
                                             block_q, block_k);
  if (static_scratch) {
    if ((st = static_scratch(fn, need, &workspace, &ws_bytes)) != BSA_OK) return st;
  }
  if ((st = check_workspace(fn, workspace, ws_bytes, need)) != BSA_OK) return st;
  SelectArgs a{};
  a.q = q->ptr; a.q_sb = q->stride_b; a.q_ss = q->stride_s; a.q_sh = q->stride_h;
  a.k = k->ptr; a.k_sb = k->stride_b; a.k_ss = k->stride_s; a.k_sh = k->stride_h;
  a.B = (int)q->B; a.Hq = (int)q->H; a.Hkv = (int)k->H; a.Sq = (int)q->S; a.Skv = (int)k->S; a.d = (int)q->D;
  a.block_q = block_q; a.block_k = block_k; a.prefix_len = prefix_len;
  a.nQb = (int)cdiv64(q->S, block_q); a.nKb = (int)cdiv64(k->S, block_k);
  a.seq_lens = seq_lens; a.keep = keep;
  a.indices = indices; a.counts = counts;
  const size_t qbar_bytes = ((size_t)a.B * a.Hq * a.nQb * a.d * sizeof(float) + 255) & ~(size_t)255;
  if (rope) {
    a.rope = true;
    a.cos_q = rope->cos_q; a.sin_q = rope->sin_q; a.cos_k = rope->cos_k; a.sin_k = rope->sin_k;
    a.q_out = rope->q_out; a.k_out = rope->k_out;
  }
  a.qbar = static_cast<float*>(workspace);
  a.kbar = reinterpret_cast<float*>(static_cast<char*>(workspace) + qbar_bytes);
  return launch_select(a, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace bsa

extern "C" {

bsa_status bsa_select(const bsa_tensor* q, const bsa_tensor* k, int32_t prefix_len, const int32_t* seq_lens,
                      int32_t block_q, int32_t block_k, const float* keep_ratio, int32_t n_keep,
                      int32_t* indices, int32_t* counts, void* workspace, size_t ws_bytes,
                      bsa_stream_t stream) {
  clear_error();
  return select_impl("bsa_select", q, k, prefix_len, seq_lens, block_q, block_k, keep_ratio, n_keep, indices,
                     counts, workspace, ws_bytes, stream, nullptr, nullptr);
}

bsa_status bsa_select_rope(const bsa_tensor* q, const bsa_tensor* k, const float* cos_q, const float* sin_q,
                           const float* cos_k, const float* sin_k, int32_t prefix_len, const int32_t* seq_lens,
                           int32_t block_q, int32_t block_k, const float* keep_ratio, int32_t n_keep,
                           void* q_out, void* k_out, int32_t* indices, int32_t* counts, void* workspace,
                           size_t ws_bytes, bsa_stream_t stream) {
  clear_error();
  const void* ptrs[6] = {cos_q, sin_q, cos_k, sin_k, q_out, k_out};
  const char* names[6] = {"cos_q", "sin_q", "cos_k", "sin_k", "q_out", "k_out"};
  for (int i = 0; i < 6; ++i) {
    if (!ptrs[i]) return set_error(BSA_ERR_INVALID_ARG, std::string("bsa_select_rope: ") + names[i] + " is NULL");
    if (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u)
      return set_error(BSA_ERR_INVALID_ARG, std::string("bsa_select_rope: ") + names[i] + " is not 16-byte aligned");
  }
  SelectArgs r{};
  r.cos_q = cos_q; r.sin_q = sin_q; r.cos_k = cos_k; r.sin_k = sin_k; r.q_out = q_out; r.k_out = k_out;
  return select_impl("bsa_select_rope", q, k, prefix_len, seq_lens, block_q, block_k, keep_ratio, n_keep,
                     indices, counts, workspace, ws_bytes, stream, &r, nullptr);
}

size_t bsa_forward_workspace_size(int B, int Hq, int Sq, int Skv, int block_q, int block_k) {
  if (B <= 0 || Hq <= 0 || Sq <= 0 || Skv <= 0 || block_q <= 0 || block_k <= 0) return 0;
  return (size_t)cdiv64(B, kMaxFwdBatch) * forward_chunk_bytes(Hq) +
         merged_list_bytes(B, Hq, Sq, Skv, block_q, block_k);
}

bsa_status bsa_forward(const bsa_tensor* q, const bsa_tensor* k, const bsa_tensor* v, const int32_t* indices,
                       const int32_t* counts, int32_t prefix_len, const int32_t* seq_lens, int32_t block_q,
                       int32_t block_k, float softmax_scale, void* out, float* lse, void* workspace,
                       size_t ws_bytes, bsa_stream_t stream) {
  clear_error();
  const char* fn = "bsa_forward";
  bsa_status st = check_common(fn, q, k, prefix_len, seq_lens, block_q, block_k, 1 << 20);
  if (st != BSA_OK) return st;
  if ((st = check_tensor(v, fn, "v")) != BSA_OK) return st;
  if (v->B != k->B || v->S != k->S || v->H != k->H || v->D != k->D)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_forward: v shape differs from k shape");
  if (indices && !counts) return set_error(BSA_ERR_INVALID_ARG, "bsa_forward: counts is NULL but indices is not");
  if (!out) return set_error(BSA_ERR_INVALID_ARG, "bsa_forward: out is NULL");
  if (reinterpret_cast<uintptr_t>(out) & 15u)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_forward: out is not 16-byte aligned");
  if (!(std::isfinite(softmax_scale)))
    return set_error(BSA_ERR_INVALID_ARG, "bsa_forward: softmax_scale is not finite");
  if ((st = check_workspace(fn, workspace, ws_bytes, bsa_forward_workspace_size((int)q->B, (int)q->H, (int)q->S, (int)k->S, block_q, block_k))) != BSA_OK)
    return st;
  ForwardArgs a{};
  a.q = q->ptr; a.q_sb = q->stride_b; a.q_ss = q->stride_s; a.q_sh = q->stride_h;
  a.k = k->ptr; a.k_sb = k->stride_b; a.k_ss = k->stride_s; a.k_sh = k->stride_h;
  a.v = v->ptr; a.v_sb = v->stride_b; a.v_ss = v->stride_s; a.v_sh = v->stride_h;
  a.B = (int)q->B; a.Hq = (int)q->H; a.Hkv = (int)k->H; a.Sq = (int)q->S; a.Skv = (int)k->S; a.d = (int)q->D;
  a.block_q = block_q; a.block_k = block_k; a.prefix_len = prefix_len;
  a.nQb = (int)cdiv64(q->S, block_q); a.nKb = (int)cdiv64(k->S, block_k);
  a.seq_lens = seq_lens; a.indices = indices; a.counts = counts;
  a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)q->D);
  a.out = out; a.lse = lse; a.workspace = workspace;
  if (indices && debug_validation() &&
      (st = debug_validate_lists(indices, counts, a.B, a.Hq, a.Sq, a.Skv, prefix_len, seq_lens, block_q, block_k,
                                 reinterpret_cast<cudaStream_t>(stream))) != BSA_OK)
    return st;
  return launch_forward(a, reinterpret_cast<cudaStream_t>(stream));
}

bsa_status bsa_forward_causal(const bsa_tensor* q_und, const bsa_tensor* k, const bsa_tensor* v,
                              int32_t block_q, int32_t block_k, float softmax_scale, void* out, float* lse,
                              void* workspace, size_t ws_bytes, bsa_stream_t stream) {
  clear_error();
  const char* fn = "bsa_forward_causal";
  // The understanding stream: queries are q_und's rows, keys the first P rows of k/v.
  bsa_status st = check_common(fn, q_und, k, 0, nullptr, block_q, block_k, 1 << 20);
  if (st != BSA_OK) return st;
  if ((st = check_tensor(v, fn, "v")) != BSA_OK) return st;
  if (v->B != k->B || v->S != k->S || v->H != k->H || v->D != k->D)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_forward_causal: v shape differs from k shape");
  if (!out) return set_error(BSA_ERR_INVALID_ARG, "bsa_forward_causal: out is NULL");
  if (reinterpret_cast<uintptr_t>(out) & 15u)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_forward_causal: out is not 16-byte aligned");
  if (!(std::isfinite(softmax_scale)))
    return set_error(BSA_ERR_INVALID_ARG, "bsa_forward_causal: softmax_scale is not finite");
  if ((st = check_workspace(fn, workspace, ws_bytes,
                            bsa_forward_workspace_size((int)q_und->B, (int)q_und->H, (int)q_und->S, (int)k->S, block_q, block_k))) != BSA_OK)
    return st;
  ForwardArgs a{};
  a.q = q_und->ptr; a.q_sb = q_und->stride_b; a.q_ss = q_und->stride_s; a.q_sh = q_und->stride_h;
  a.k = k->ptr; a.k_sb = k->stride_b; a.k_ss = k->stride_s; a.k_sh = k->stride_h;
  a.v = v->ptr; a.v_sb = v->stride_b; a.v_ss = v->stride_s; a.v_sh = v->stride_h;
  a.B = (int)q_und->B; a.Hq = (int)q_und->H; a.Hkv = (int)k->H; a.Sq = (int)q_und->S; a.Skv = (int)k->S;
  a.d = (int)q_und->D;
  a.block_q = block_q; a.block_k = block_k;
  a.prefix_len = 0;                    // every understanding row is a query; keys are rows [0, P)
  a.nQb = (int)cdiv64(q_und->S, block_q); a.nKb = (int)cdiv64(k->S, block_k);
  a.seq_lens = nullptr;                // L_b = P for every request
  a.indices = nullptr; a.counts = nullptr;
  a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)q_und->D);
  a.out = out; a.lse = lse; a.workspace = workspace;
  a.causal = true;
  return launch_forward(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t bsa_backward_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int block_q, int block_k) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Sq <= 0 || Skv <= 0 || !supported_geometry(block_q, block_k)) return 0;
  return backward_workspace_bytes(B, Hq, Hkv, Sq, Skv, block_q, block_k);
}

bsa_status bsa_backward(const bsa_tensor* q, const bsa_tensor* k, const bsa_tensor* v, const bsa_tensor* out,
                        const bsa_tensor* dout, const float* lse, const int32_t* indices, const int32_t* counts,
                        int32_t prefix_len, const int32_t* seq_lens, int32_t block_q, int32_t block_k,
                        float softmax_scale, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                        bsa_stream_t stream) {
  clear_error();
  const char* fn = "bsa_backward";
  bsa_status st = check_common(fn, q, k, prefix_len, seq_lens, block_q, block_k, kMaxSelectBatch);
  if (st != BSA_OK) return st;
  if ((st = check_tensor(v, fn, "v")) != BSA_OK) return st;
  if ((st = check_tensor(out, fn, "out")) != BSA_OK) return st;
  if ((st = check_tensor(dout, fn, "dout")) != BSA_OK) return st;
  if (v->B != k->B || v->S != k->S || v->H != k->H || v->D != k->D)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_backward: v shape differs from k shape");
  for (const bsa_tensor* t : {out, dout})
    if (t->B != q->B || t->S != q->S || t->H != q->H || t->D != q->D)
      return set_error(BSA_ERR_INVALID_ARG, std::string("bsa_backward: ") + (t == out ? "out" : "dout") +
                                                " shape differs from q shape");
  if (!indices || !counts) return set_error(BSA_ERR_INVALID_ARG, "bsa_backward: indices and counts are required");
  if (!lse) return set_error(BSA_ERR_INVALID_ARG, "bsa_backward: lse is NULL");
  if (!dq || !dk || !dv) return set_error(BSA_ERR_INVALID_ARG, "bsa_backward: dq, dk and dv must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15u)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_backward: dq, dk and dv must be 16-byte aligned");
  if (!(std::isfinite(softmax_scale)))
    return set_error(BSA_ERR_INVALID_ARG, "bsa_backward: softmax_scale is not finite");
  if ((st = check_workspace(fn, workspace, ws_bytes,
                            backward_workspace_bytes((int)q->B, (int)q->H, (int)k->H, (int)q->S, (int)k->S, block_q,
                                                     block_k))) != BSA_OK)
    return st;
  BackwardArgs a{};
  a.q = q->ptr; a.q_sb = q->stride_b; a.q_ss = q->stride_s; a.q_sh = q->stride_h;
  a.k = k->ptr; a.k_sb = k->stride_b; a.k_ss = k->stride_s; a.k_sh = k->stride_h;
  a.v = v->ptr; a.v_sb = v->stride_b; a.v_ss = v->stride_s; a.v_sh = v->stride_h;
  a.o = out->ptr; a.o_sb = out->stride_b; a.o_ss = out->stride_s; a.o_sh = out->stride_h;
  a.dout = dout->ptr; a.d_sb = dout->stride_b; a.d_ss = dout->stride_s; a.d_sh = dout->stride_h;
  a.lse = lse;
  a.B = (int)q->B; a.Hq = (int)q->H; a.Hkv = (int)k->H; a.Sq = (int)q->S; a.Skv = (int)k->S; a.d = (int)q->D;
  a.block_q = block_q; a.block_k = block_k; a.prefix_len = prefix_len;
  a.seq_lens = seq_lens; a.indices = indices; a.counts = counts;
  a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)q->D);
  a.dq = dq; a.dk = dk; a.dv = dv; a.workspace = workspace;
  if (debug_validation() &&
      (st = debug_validate_lists(indices, counts, a.B, a.Hq, a.Sq, a.Skv, prefix_len, seq_lens, block_q, block_k,
                                 reinterpret_cast<cudaStream_t>(stream))) != BSA_OK)
    return st;
  return launch_backward(a, reinterpret_cast<cudaStream_t>(stream));
}

bsa_status bsa_validate_indices(const int32_t* indices, const int32_t* counts, int32_t B, int32_t Hq, int32_t Sq,
                                int32_t Skv, int32_t prefix_len, const int32_t* seq_lens, int32_t block_q,
                                int32_t block_k, int32_t require_prefix, int32_t* bad_rows, bsa_stream_t stream) {
  clear_error();
  if (!indices || !counts || !bad_rows)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_validate_indices: indices, counts and bad_rows must be non-NULL");
  if (B <= 0 || B > kMaxSelectBatch || Hq <= 0 || Sq <= 0 || Skv <= 0 || prefix_len < 0)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_validate_indices: bad sizes");
  if (!supported_geometry(block_q, block_k))
    return set_error(BSA_ERR_UNSUPPORTED, "bsa_validate_indices: unsupported block geometry");
  ValidateParams p{};
  p.indices = indices; p.counts = counts; p.B = B; p.Hq = Hq;
  p.nQb = (int)cdiv64(Sq, block_q); p.nKb = (int)cdiv64(Skv, block_k);
  p.block_q = block_q; p.block_k = block_k; p.prefix_len = prefix_len; p.require_prefix = require_prefix ? 1 : 0;
  for (int b = 0; b < B; ++b) {
    const int L = seq_lens ? seq_lens[b] : Sq;
    if (L < 0 || L > Sq || prefix_len + L > Skv)
      return set_error(BSA_ERR_INVALID_ARG, "bsa_validate_indices: seq_lens[" + std::to_string(b) + "] out of range");
    p.seq_lens[b] = L;
  }
  p.bad = bad_rows;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bsa_status st = cuda_check(cudaMemsetAsync(bad_rows, 0, sizeof(int32_t), s), "cudaMemsetAsync(bad_rows)");
  if (st != BSA_OK) return st;
  const int64_t rows = (int64_t)B * Hq * p.nQb;
  validate_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p);
  return cuda_check(cudaGetLastError(), "validate_kernel launch");
}

bsa_status bsa_device_status(bsa_stream_t stream) {
  clear_error();
  bsa_status st = cuda_check(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  if (st != BSA_OK) return st;
  // the forward kernels' and the backward kernels' error words (each read and cleared)
  const unsigned int ef = read_and_clear_fwd_error();
  const unsigned int eb = read_and_clear_bwd_error();
  if (ef == 0xFFFFFFFFu || eb == 0xFFFFFFFFu)
    return set_error(BSA_ERR_CUDA, "bsa_device_status: cannot read the device error word");
  int bad = 0;
  const int zero = 0;
  if ((st = cuda_check(cudaMemcpyFromSymbol(&bad, g_debug_bad_rows, sizeof(bad)), "read BSA_DEBUG counter")) !=
      BSA_OK)
    return st;
  if (bad != 0) {
    if ((st = cuda_check(cudaMemcpyToSymbol(g_debug_bad_rows, &zero, sizeof(zero)), "clear BSA_DEBUG counter")) !=
        BSA_OK)
      return st;
    return set_error(BSA_ERR_INVALID_INDICES,
                     std::to_string(bad) + " malformed index-list rows reached bsa_forward / bsa_backward "
                     "(BSA_DEBUG validation: indices in range of the request's real key blocks and strictly "
                     "ascending, count 0 for query blocks without real rows)" +
                         (((ef | eb) & 1u) ? "; a bounded device wait also gave up" : ""));
  }
  if ((ef | eb) & 1u)
    return set_error(BSA_ERR_TIMEOUT, std::string("a bounded device wait gave up in the ") +
                                          (ef & 1u ? (eb & 1u ? "forward and backward" : "forward") : "backward") +
                                          " kernels (the kernel aborted its tiles)");
  return BSA_OK;
}

bsa_status bsa_debug_wait_probe(int32_t family, uint64_t limit_ns, bsa_stream_t stream) {
  clear_error();
  if (family != 0 && family != 1)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_debug_wait_probe: family " + s(family) +
                                              " is not 0 (forward kernels) or 1 (backward kernels)");
  if (limit_ns < 1000000ull || limit_ns > 10000000000ull)
    return set_error(BSA_ERR_INVALID_ARG, "bsa_debug_wait_probe: limit_ns " + std::to_string(limit_ns) +
                                              " is outside [1 ms, 10 s]");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return family == 0 ? launch_fwd_wait_probe(limit_ns, st) : launch_bwd_wait_probe(limit_ns, st);
}

}  // extern "C"
