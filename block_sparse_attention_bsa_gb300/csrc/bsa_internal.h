// Host-side declarations shared by the translation units of libbsa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "../../include/bsa.h"

namespace bsa {

constexpr int kMaxSelectBatch = 64;   // batch elements per select launch
constexpr int kMaxHeads = 256;        // query heads (keep ratios in kernel params)
constexpr int kMaxFwdBatch = 8;       // batch elements per forward launch (tensor maps)

inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Records `msg` as this thread's last error and returns `st`.
bsa_status set_error(bsa_status st, const std::string& msg);
void clear_error();

// Checks a CUDA call; on failure records the call site and returns BSA_ERR_CUDA.
bsa_status cuda_check(cudaError_t e, const char* what);

// Number of SMs of the current device (cached per device).
int num_sms();

// TMA tensor map of a [rows, H, D] bf16 view (row stride ss, head stride sh,
// in elements): dims (D, rows, H), box (64, box_rows, 1), 128-byte swizzle;
// rows past `rows` read as zeros.  `name` labels the error message.
bsa_status encode_tensor_map(CUtensorMap* m, const void* base, int64_t rows, int64_t H, int D, int64_t ss,
                             int64_t sh, int box_rows, const char* name);

// ---- selector (bsa_select.cu) ----
struct SelectArgs {
  const void* q; int64_t q_sb, q_ss, q_sh;
  const void* k; int64_t k_sb, k_ss, k_sh;
  int B, Hq, Hkv, Sq, Skv, d, block_q, block_k, prefix_len;
  int nQb, nKb;
  const int32_t* seq_lens;   // host
  const float* keep;         // host, Hq values (expanded)
  int32_t* indices;
  int32_t* counts;
  float* qbar;               // workspace [B,Hq,nQb,d]
  float* kbar;               // workspace [B,Hkv,nKb,d]
  // rotary prologue (bsa_select_rope): tables [S, d] fp32, rotated outputs
  bool rope = false;
  const float* cos_q = nullptr; const float* sin_q = nullptr;
  const float* cos_k = nullptr; const float* sin_k = nullptr;
  void* q_out = nullptr; void* k_out = nullptr;
};
bsa_status launch_select(const SelectArgs& a, cudaStream_t stream);

// Supplies a selector workspace that the caller did not pass (the static
// scratch of bsa_select_noalloc): given the bytes needed, sets *ws and
// *ws_bytes or returns an error naming `fn`.
using StaticScratchFn = bsa_status (*)(const char* fn, size_t need, void** ws, size_t* ws_bytes);
// The selector entry points' common body (bsa_api.cu): checks every argument
// under the name `fn`, then launches.  `rope` is NULL for the plain selector;
// `static_scratch` is NULL when the caller passes the workspace.
bsa_status select_impl(const char* fn, const bsa_tensor* q, const bsa_tensor* k, int32_t prefix_len,
                       const int32_t* seq_lens, int32_t block_q, int32_t block_k, const float* keep_ratio,
                       int32_t n_keep, int32_t* indices, int32_t* counts, void* workspace, size_t ws_bytes,
                       bsa_stream_t stream, const SelectArgs* rope, StaticScratchFn static_scratch);

// ---- forward (bsa_fmha.cu) ----
struct ForwardArgs {
  const void* q; int64_t q_sb, q_ss, q_sh;
  const void* k; int64_t k_sb, k_ss, k_sh;
  const void* v; int64_t v_sb, v_ss, v_sh;
  int B, Hq, Hkv, Sq, Skv, d, block_q, block_k, prefix_len;
  int nQb, nKb;
  const int32_t* seq_lens;   // host, B values
  const int32_t* indices;    // NULL = dense
  const int32_t* counts;
  float scale;
  void* out;
  float* lse;
  void* workspace;           // forward_chunk_bytes(Hq) per chunk of kMaxFwdBatch requests
  bool causal;               // key position <= query row (dense pass over the prefix only)
  bool masked = false;       // internal: merged lists with membership bits
  int group_rows = 0;        // internal: rows per original query block of merged lists
  const int32_t* classes = nullptr;   // internal: merged lists' per-row class sizes
  int list_stride = 0;       // internal: entries per list row (0: nKb)
};
// Workspace bytes of the merged lists used when block_q < 256 (0 otherwise).
size_t merged_list_bytes(int B, int Hq, int Sq, int Skv, int block_q, int block_k);
// Workspace bytes per launch chunk: tile counter (256 B) + group order.
size_t forward_chunk_bytes(int Hq);
bsa_status launch_forward(const ForwardArgs& a, cudaStream_t stream);

// ---- backward (bsa_bwd.cu) ----
struct BackwardArgs {
  const void* q; int64_t q_sb, q_ss, q_sh;
  const void* k; int64_t k_sb, k_ss, k_sh;
  const void* v; int64_t v_sb, v_ss, v_sh;
  const void* o; int64_t o_sb, o_ss, o_sh;
  const void* dout; int64_t d_sb, d_ss, d_sh;
  const float* lse;          // [B, Hq, Sq]
  int B, Hq, Hkv, Sq, Skv, d, block_q, block_k, prefix_len;
  const int32_t* seq_lens;   // host, B values
  const int32_t* indices;
  const int32_t* counts;
  float scale;
  void* dq; void* dk; void* dv;
  void* workspace;
};
size_t backward_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int block_q, int block_k);
bsa_status launch_backward(const BackwardArgs& a, cudaStream_t stream);

// Device error word of the current device (0xFFFFFFFF if it cannot be read);
// cleared after reading.
// Each translation unit with device waits keeps its own device error word.
unsigned int read_and_clear_fwd_error();
unsigned int read_and_clear_bwd_error();
bsa_status launch_fwd_wait_probe(unsigned long long limit_ns, cudaStream_t stream);
bsa_status launch_bwd_wait_probe(unsigned long long limit_ns, cudaStream_t stream);

// ---- validation (bsa_api.cu) ----
size_t select_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int d, int bq, int bk);

}  // namespace bsa
