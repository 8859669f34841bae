/*
 * bsa.h -- C ABI of libbsa, selected-block (block-sparse) attention on GB300.
 *
 * The operations come from the vllm-omni pull request "[Core] Add shared
 * block-sparse attention adapters with FlashAttention-4" (Purpose): a
 * selector produces per-query-head key-block indices and counts, and an
 * attention adapter executes exactly that selection, keeping a protected KV
 * prefix, the native MHA/MQA/GQA head mapping and the block geometry, masking
 * single-document suffix padding, and never falling back to dense attention
 * or expanding K/V.  The attention semantics (generation queries attend
 * non-causally over cat(understanding, generation) keys; query head i reads
 * KV head i / (Hq/Hkv); padded keys are masked) are those of
 * cosmos_parallel.py (cosmos3_cp_attention, _repeat_kv_heads,
 * build_gen_key_mask).  The default softmax scale head_dim^-1/2 is the one
 * mstar PR 927 ("What the review checked") names.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor memory is device memory owned by the caller.  The library
 *    allocates nothing, never synchronises, and enqueues all work on the
 *    caller's stream (NULL = the legacy default stream).
 *  - Q: [B, Sq, Hq, d] bf16; K, V: [B, Skv, Hkv, d] bf16, described by
 *    bsa_tensor (element strides, innermost dim contiguous, base and every
 *    stride 16-byte aligned).  Key position t < prefix_len is the protected
 *    prefix; position prefix_len + i is generation token i.
 *  - seq_lens (HOST array of B int32, or NULL = every request has length Sq):
 *    request b has L_b real query rows [0, L_b) and real keys
 *    [0, prefix_len + L_b); everything after is suffix padding that is never
 *    read into a result.  Requires L_b <= Sq and prefix_len + L_b <= Skv.
 *  - Blocks: query block qb = rows [qb*block_q, (qb+1)*block_q); key block kb
 *    = key positions [kb*block_k, (kb+1)*block_k), tiling the concatenated
 *    sequence from position 0.  nQb = ceil(Sq/block_q), nKb = ceil(Skv/block_k).
 *    A key block holding any prefix position is a prefix block:
 *    npb = ceil(prefix_len/block_k).
 *  - Supported: d in {64, 128}; block_q in {64, 128, 256} with block_k in
 *    {64, 128} (all six pairs); Hq % Hkv == 0; Hq <= 256; bf16 only.  Batch:
 *    B <= 64 for the selector calls, bsa_backward and bsa_validate_indices;
 *    bsa_forward and bsa_forward_causal take larger batches (they launch 8
 *    requests at a time).  Anything else returns BSA_ERR_UNSUPPORTED (no
 *    fallback path exists).
 *  - Errors: every call validates its arguments on the host before launching
 *    and returns a status; bsa_get_last_error() gives a message naming the
 *    argument and value (thread-local, valid until the next call on the
 *    thread).  Launch failures return BSA_ERR_CUDA.  Device-side waits are
 *    bounded: a wait that gives up sets a device error word that
 *    bsa_device_status() reports as BSA_ERR_TIMEOUT.
 *  - Debug validation: when the environment variable BSA_DEBUG is set to a
 *    non-empty value other than "0" at the time of a bsa_forward (with
 *    lists) or bsa_backward call, the call first enqueues the checks of
 *    bsa_validate_indices (without the prefix requirement) on its lists;
 *    malformed rows are counted on the device and the next
 *    bsa_device_status() returns BSA_ERR_INVALID_INDICES.  No
 *    synchronisation is added.  Without it the kernels clamp out-of-range
 *    entries (they read zeros, fully masked) and never read out of bounds.
 */
#ifndef BSA_H_
#define BSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BSA_API __attribute__((visibility("default")))
#else
#define BSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bsa_status {
  BSA_OK = 0,
  BSA_ERR_INVALID_ARG = 1,      /* bad shape, pointer, stride or value */
  BSA_ERR_UNSUPPORTED = 2,      /* valid but not implemented (d, geometry, dtype) */
  BSA_ERR_WORKSPACE = 3,        /* workspace missing, misaligned or too small */
  BSA_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
  BSA_ERR_INVALID_INDICES = 5,  /* bsa_validate_indices found malformed rows */
  BSA_ERR_TIMEOUT = 6           /* a bounded device wait gave up */
} bsa_status;

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st* bsa_stream_t;

/* A 4-D bf16 tensor [B, S, H, D] in device memory.  Strides are in elements;
 * the D axis has stride 1.  ptr, stride_b, stride_s and stride_h must give
 * 16-byte aligned rows (stride_* * 2 bytes a multiple of 16). */
typedef struct bsa_tensor {
  const void* ptr;
  int64_t B, S, H, D;
  int64_t stride_b, stride_s, stride_h;
} bsa_tensor;

/* Library version as 10000*major + 100*minor + patch. */
BSA_API int bsa_version(void);

/* Message for the last failed call on this thread ("" if none). */
BSA_API const char* bsa_get_last_error(void);

/* ---------------------------------------------------------------- select ---
 * Workspace bytes bsa_select needs: fp32 block means of Q [B,Hq,nQb,d] and K
 * [B,Hkv,nKb,d], each 256-byte aligned. */
BSA_API size_t bsa_select_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                 int block_q, int block_k);

/* Selector: per (request b, query head h, query block qb) the list of key
 * blocks to attend (PR 8335, Purpose: "the selector produces per-query-head
 * block indices/counts").
 *
 * For each valid query block (qb < ceil(L_b/block_q)):
 *   qbar = mean of Q[b, rows, h, :] over the block's real rows, and for each
 *   key block kbar = mean of K[b, keys, h / (Hq/Hkv), :] over its real keys
 *   (fp32 sums); score(kb) = qbar . kbar (fp32) for the N_b non-prefix valid
 *   key blocks; k_h = min(N_b, ceil(r_h * N_b)) computed in double precision
 *   from the float keep ratio; the row lists the npb prefix blocks followed
 *   by the k_h best candidates under (score descending, block index
 *   ascending) -- ties go to the lower index -- all written ascending.
 *   counts = npb + k_h.  Query blocks with no real row get count 0.
 *
 * keep_ratio: HOST array of n_keep floats in [0,1]; n_keep is 1 (shared) or
 *   Hq (per query head).
 * indices: device int32 [B, Hq, nQb, nKb]; entries past a row's count are
 *   left untouched.  counts: device int32 [B, Hq, nQb].
 * workspace: device, >= bsa_select_workspace_size(...) bytes, 256-B aligned.
 * Returns BSA_OK once the kernels are enqueued. */
BSA_API bsa_status bsa_select(const bsa_tensor* q, const bsa_tensor* k, int32_t prefix_len,
                      const int32_t* seq_lens, int32_t block_q, int32_t block_k,
                      const float* keep_ratio, int32_t n_keep,
                      int32_t* indices, int32_t* counts,
                      void* workspace, size_t ws_bytes, bsa_stream_t stream);

/* ------------------------------------------------ select with RoPE fused ---
 * The rotary prologue of cosmos_parallel.py (_project_qkv_with_rope:
 * x' = x * cos + rotate_half(x) * sin per position, cos/sin shared by every
 * head) fused with the selector's block pooling: Q and K are read once,
 * rotated in fp32, written as bf16 to q_out / k_out (what bsa_forward then
 * reads), and the block means are taken of the written bf16 values, so the
 * result equals rotating first and calling bsa_select on q_out / k_out.
 * rotate_half pairs channel i with channel i + d/2: (x1, x2) -> (-x2, x1).
 *
 * cos_q, sin_q: device fp32 [Sq, d] (positions of the generation queries);
 * cos_k, sin_k: device fp32 [Skv, d] (understanding positions for key rows
 *   < prefix_len, then generation positions).  All 16-byte aligned.
 * q_out: device bf16 [B, Sq, Hq, d] contiguous; k_out: [B, Skv, Hkv, d]
 *   contiguous.  Every row is rotated (padding rows too); q_out may be q's
 *   own storage when q is contiguous (each element is read before it is
 *   written by the same thread), likewise k_out.
 * Everything else as bsa_select (same workspace size). */
BSA_API bsa_status bsa_select_rope(const bsa_tensor* q, const bsa_tensor* k,
                                   const float* cos_q, const float* sin_q,
                                   const float* cos_k, const float* sin_k,
                                   int32_t prefix_len, const int32_t* seq_lens,
                                   int32_t block_q, int32_t block_k,
                                   const float* keep_ratio, int32_t n_keep,
                                   void* q_out, void* k_out,
                                   int32_t* indices, int32_t* counts,
                                   void* workspace, size_t ws_bytes, bsa_stream_t stream);

/* ------------------------------------------------- select, no allocation ---
 * bsa_select for callers that cannot provide device scratch memory: for
 * example a plugin inside a serving runtime that owns every device
 * allocation and hands the plugin only its input and output buffers, or a
 * deployment whose device memory budget is fixed up front.  The pages have
 * no counterpart; this is a library convenience.
 *
 * Same contract and results as bsa_select, except that the block means live
 * in a buffer of BSA_NOALLOC_SCRATCH_BYTES that the library declares as a
 * static device array: every GPU that loads libbsa holds that much memory
 * until the process exits.  Nothing is allocated by this call (no
 * cudaMalloc, no allocating library routine).
 *  - A problem whose block means need more than BSA_NOALLOC_SCRATCH_BYTES
 *    (see bsa_select_workspace_size) returns BSA_ERR_UNSUPPORTED naming the
 *    size and the limit.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current).  The address belongs
 *    to the context it was looked up in: after a cudaDeviceReset the next
 *    call sees a new context (by its unique ID) and looks the address up
 *    again.
 *  - Arguments are checked under this entry point's name before the scratch
 *    is touched: invalid arguments return the same codes as bsa_select.
 *  - All calls share the one array and it keeps the last call's contents
 *    (every value a call reads is written by that call first).  Calls whose
 *    kernels overlap on the GPU -- on different streams, or from different
 *    host threads -- race on it; serialise them. */
#define BSA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
BSA_API bsa_status bsa_select_noalloc(const bsa_tensor* q, const bsa_tensor* k, int32_t prefix_len,
                                      const int32_t* seq_lens, int32_t block_q, int32_t block_k,
                                      const float* keep_ratio, int32_t n_keep,
                                      int32_t* indices, int32_t* counts, bsa_stream_t stream);

/* --------------------------------------------------------------- forward ---
 * Workspace bytes bsa_forward (and bsa_forward_causal) need: per launch chunk
 * of up to 8 requests, a work-tile counter and the order of the (request, KV
 * head) groups; with block_q of 64 or 128, also the merged key-block lists of
 * each 256-row super-block (int32 [B, Hq, ceil(Sq/256), nKb + 3], their
 * counts and two class sizes per row): those query blocks are attended 256
 * rows at a time over the union of their lists, each row masking the blocks
 * its own query block did not select, and each 128-row half of a super-block
 * skipping the key tiles only the other half's query blocks selected. */
BSA_API size_t bsa_forward_workspace_size(int B, int Hq, int Sq, int Skv, int block_q, int block_k);

/* Selected-block attention forward (PR 8335, Purpose: the adapter executes
 * the selection; cosmos_parallel.py cosmos3_cp_attention: non-causal
 * attention of generation queries over cat(und, gen) keys).
 *
 * For each request b, query head h and real query row i < L_b in block qb:
 *   keys = positions of the listed blocks indices[b,h,qb,0:count] that are
 *   < prefix_len + L_b, read from KV head h / (Hq/Hkv);
 *   z_j = (q_i . k_j) * softmax_scale;  out_i = sum_j softmax(z)_j v_j (bf16);
 *   lse_i = ln sum_j exp(z_j)  (fp32, natural log of the scaled logits).
 * Padded rows (i >= L_b) and rows with no key: out 0, lse -inf.
 *
 * indices/counts: device int32 as written by bsa_select, or indices == NULL
 *   for the dense pass (every valid key block; counts is then ignored and may
 *   be NULL).  A count above nKb is clamped to nKb; indices are not checked
 *   here (see bsa_validate_indices); an out-of-range index reads zeros.  Each
 *   list must be strictly ascending (as bsa_select writes it): with block_q
 *   below 256 the lists are merged and a repeated block is attended once.
 * softmax_scale <= 0 selects head_dim^-1/2.
 * out: device bf16 [B, Sq, Hq, d] contiguous.  lse: device fp32 [B, Hq, Sq]
 *   contiguous, or NULL.
 * workspace: device, >= bsa_forward_workspace_size(...) bytes, 256-B aligned.
 * Q, K, V may not alias out. */
BSA_API bsa_status bsa_forward(const bsa_tensor* q, const bsa_tensor* k, const bsa_tensor* v,
                       const int32_t* indices, const int32_t* counts,
                       int32_t prefix_len, const int32_t* seq_lens,
                       int32_t block_q, int32_t block_k, float softmax_scale,
                       void* out, float* lse,
                       void* workspace, size_t ws_bytes, bsa_stream_t stream);

/* ------------------------------------------ understanding stream, causal ---
 * Causal self-attention of the understanding (prefix) stream
 * (cosmos_parallel.py, cosmos3_cp_attention: the understanding pathway
 * self-attends causally over the whole understanding sequence), through the
 * same kernel as bsa_forward's dense pass.
 *
 * q_und: [B, P, Hq, d] bf16, P = q_und->S = the understanding length.
 * k, v: [B, Skv, Hkv, d] with Skv >= P; only rows [0, P) (the prefix) are
 *   read.  Row i of q_und attends key positions 0..i of KV head h/(Hq/Hkv):
 *   out_i = softmax((q_i . k_j) * scale)_j v_j over j <= i; lse_i = ln-sum-exp.
 * out: bf16 [B, P, Hq, d] contiguous; lse: fp32 [B, Hq, P] contiguous or NULL.
 * block_q/block_k: any supported geometry (the key blocks up to the one that
 *   holds a query block's last row are visited; the diagonal is masked per
 *   row).  workspace: bsa_forward_workspace_size(B, Hq, P, Skv, block_q, block_k) bytes. */
BSA_API bsa_status bsa_forward_causal(const bsa_tensor* q_und, const bsa_tensor* k, const bsa_tensor* v,
                                      int32_t block_q, int32_t block_k, float softmax_scale,
                                      void* out, float* lse, void* workspace, size_t ws_bytes,
                                      bsa_stream_t stream);

/* -------------------------------------------------------------- backward ---
 * Gradients of bsa_forward's output (the pages run inference only; this is
 * the plain derivative of the attention that PR 8335, Purpose, and
 * cosmos_parallel.py cosmos3_cp_attention define, over the same lists).
 * With z_ij = scale q_i.k_j over the keys row i attends, P = softmax(z),
 * D_i = sum_c dO_ic O_ic and dS_ij = P_ij (dO_i.v_j - D_i):
 *   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,
 *   dV_j = sum_i P_ij dO_i,
 * where dK_j/dV_j sum over every query head of j's KV group and every query
 * row whose list holds j's block.  P is recomputed from `lse`, so q, k, v,
 * indices, counts and lse must be the ones the forward used, and out its
 * output.  Results do not depend on scheduling: no atomics touch dQ/dK/dV.
 *
 * Supported: every geometry bsa_forward takes (head dim 64 or 128, block_q
 *   64, 128 or 256, block_k 64 or 128); indices/counts are required (dense
 *   lists come from bsa_select with keep_ratio 1).
 * q, k, v, out, dout: bf16 descriptors as in bsa_forward; out and dout have
 *   q's shape.  lse: device fp32 [B, Hq, Sq] contiguous from bsa_forward.
 * dq: device bf16 [B, Sq, Hq, d]; dk, dv: device bf16 [B, Skv, Hkv, d]; all
 *   contiguous and fully written (padded rows and keys no query reads get 0).
 * workspace: device, >= bsa_backward_workspace_size(...) bytes, 256-B
 *   aligned; it holds -lse and -D per 128-row query tile and the lists re-cut
 *   on 128 x 128 (query tile, key tile) pairs with their bitmaps: per query
 *   tile its key tiles, per key tile the query tiles, each with a mask of the
 *   selected 64-row / 64-key halves.
 * Gradient buffers may not alias any input. */
BSA_API size_t bsa_backward_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int block_q, int block_k);
BSA_API bsa_status bsa_backward(const bsa_tensor* q, const bsa_tensor* k, const bsa_tensor* v,
                                const bsa_tensor* out, const bsa_tensor* dout, const float* lse,
                                const int32_t* indices, const int32_t* counts,
                                int32_t prefix_len, const int32_t* seq_lens,
                                int32_t block_q, int32_t block_k, float softmax_scale,
                                void* dq, void* dk, void* dv,
                                void* workspace, size_t ws_bytes, bsa_stream_t stream);

/* ------------------------------------------------------------ validation ---
 * Debug check of index lists (PR 8335, Purpose: provider failures propagate
 * as errors).  Counts the rows (b, h, qb) whose list is malformed: count
 * outside [0, nKb_valid(b)], an index outside [0, nKb_valid(b)), indices not
 * strictly ascending, or (require_prefix != 0) a valid row whose first npb
 * entries are not 0..npb-1.  Rows of query blocks without real rows must have
 * count 0.  Writes the number of bad rows to *bad_rows (device int32),
 * asynchronously; the caller reads it after synchronising. */
BSA_API bsa_status bsa_validate_indices(const int32_t* indices, const int32_t* counts,
                                int32_t B, int32_t Hq, int32_t Sq, int32_t Skv,
                                int32_t prefix_len, const int32_t* seq_lens,
                                int32_t block_q, int32_t block_k, int32_t require_prefix,
                                int32_t* bad_rows, bsa_stream_t stream);

/* Synchronises `stream`, then reports and clears the device error words of
 * the current device: BSA_ERR_INVALID_INDICES if BSA_DEBUG validation found
 * malformed lists since the last call, BSA_ERR_TIMEOUT if a bounded wait in a
 * kernel gave up, BSA_ERR_CUDA if the stream reports an error, else BSA_OK. */
BSA_API bsa_status bsa_device_status(bsa_stream_t stream);

/* Diagnostics for the timeout path above.  Enqueues on `stream` one
 * single-thread kernel that waits, with the same bounded-wait code the
 * attention kernels use but a limit of `limit_ns`, for an mbarrier phase that
 * nothing completes: the wait gives up after limit_ns, records the timeout in
 * the device error word of the kernel family `family` (0 = selector-side and
 * forward kernels, 1 = backward kernels) and the kernel exits normally, so
 * the CUDA context stays usable.  The next bsa_device_status() returns
 * BSA_ERR_TIMEOUT.  No fault, trap or hang is involved.
 * Errors: BSA_ERR_INVALID_ARG for another family or a limit outside
 * [1 ms, 10 s]; BSA_ERR_CUDA if the launch fails. */
BSA_API bsa_status bsa_debug_wait_probe(int32_t family, uint64_t limit_ns, bsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H_ */
