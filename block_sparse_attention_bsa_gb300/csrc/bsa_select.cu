// Selector kernels: block mean pooling of Q and K, block scores, per-row
// top-k with the protected prefix forced in and the lowest-index tie rule,
// and compaction to ascending index lists.
//
// The selector's contract is the one of the vllm-omni pull request "[Core]
// Add shared block-sparse attention adapters with FlashAttention-4"
// (Purpose): per-query-head block indices and counts, protected KV prefix,
// suffix padding excluded, native GQA mapping (query head h scores against
// KV head h / G, as _repeat_kv_heads in cosmos_parallel.py pairs them).
#include <cuda_bf16.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "bsa_internal.h"

namespace bsa {
namespace {

// ------------------------------------------------------------- pooling ---
// One CTA per (block, batch element, 64 16-byte columns).  Thread column c
// covers 8 channels of one head; the 4 row groups of the CTA split the
// block's rows and are summed in shared memory.  HBM-bound: every element of
// Q and K is read exactly once with 16-byte loads.

constexpr int kPoolCols = 64;
constexpr int kPoolGroups = 4;

struct PoolParams {
  const __nv_bfloat16* x;
  int64_t sb, ss, sh;        // element strides
  int H, D, block, nb, cols; // cols = H * D / 8
  int valid[kMaxSelectBatch];
  float* out;                // [B, H, nb, D]
};

__global__ void __launch_bounds__(kPoolCols* kPoolGroups)
    pool_kernel(const __grid_constant__ PoolParams p) {
  const int blk = blockIdx.x;
  const int b = blockIdx.y;
  const int tc = threadIdx.x % kPoolCols;
  const int g = threadIdx.x / kPoolCols;
  const int c = blockIdx.z * kPoolCols + tc;
  const int r0 = blk * p.block;
  const int r1 = min(r0 + p.block, p.valid[b]);
  const int dc = p.D / 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  int h = 0, d0 = 0;
  if (c < p.cols) {
    h = c / dc;
    d0 = (c % dc) * 8;
    const __nv_bfloat16* base = p.x + (int64_t)b * p.sb + (int64_t)h * p.sh + d0;
#pragma unroll 4
    for (int r = r0 + g; r < r1; r += kPoolGroups) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)r * p.ss));
      const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(v2[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
      }
    }
  }
  __shared__ float red[kPoolGroups][kPoolCols][9];
#pragma unroll
  for (int i = 0; i < 8; ++i) red[g][tc][i] = acc[i];
  __syncthreads();
  if (g == 0 && c < p.cols) {
    const int n = max(r1 - r0, 0);
    const float inv = n > 0 ? 1.f / (float)n : 0.f;
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float s = red[0][tc][i];
#pragma unroll
      for (int gg = 1; gg < kPoolGroups; ++gg) s += red[gg][tc][i];
      m[i] = s * inv;
    }
    float* o = p.out + (((int64_t)b * p.H + h) * p.nb + blk) * p.D + d0;
    reinterpret_cast<float4*>(o)[0] = make_float4(m[0], m[1], m[2], m[3]);
    reinterpret_cast<float4*>(o)[1] = make_float4(m[4], m[5], m[6], m[7]);
  }
}

// ------------------------------------------------- rotary + pooling -------
// Fused prologue: x' = x * cos + rotate_half(x) * sin per row (tables [S, d]
// shared by every head and request), written back as bf16, and the block
// means of the written (rounded) values.  A thread owns channels
// [8j, 8j+8) and their partners [8j+d/2, 8j+d/2+8) of one head, so it holds
// both halves of every rotated pair; rows are summed in the same order as
// pool_kernel, so the means equal pooling the rotated tensor afterwards.

struct RopePoolParams {
  const __nv_bfloat16* x;
  int64_t sb, ss, sh;              // input strides (elements)
  __nv_bfloat16* y;                // output [B, S, H, D] contiguous
  const float* cos_t;              // [S, D]
  const float* sin_t;              // [S, D]
  int H, D, S, block, nb, cols;    // cols = H * D / 16
  int valid[kMaxSelectBatch];
  float* out;                      // means [B, H, nb, D]
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(v2[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&t);
  }
  return u;
}

__global__ void __launch_bounds__(kPoolCols* kPoolGroups)
    rope_pool_kernel(const __grid_constant__ RopePoolParams p) {
  const int blk = blockIdx.x;
  const int b = blockIdx.y;
  const int tc = threadIdx.x % kPoolCols;
  const int g = threadIdx.x / kPoolCols;
  const int c = blockIdx.z * kPoolCols + tc;
  const int r0 = blk * p.block;
  const int r_end = min(r0 + p.block, p.S);
  const int r_valid = min(r0 + p.block, p.valid[b]);
  const int jc = p.D / 16, half = p.D / 2;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  int h = 0, lo = 0;
  if (c < p.cols) {
    h = c / jc;
    lo = (c % jc) * 8;
    const __nv_bfloat16* xb = p.x + (int64_t)b * p.sb + (int64_t)h * p.sh;
    __nv_bfloat16* yb = p.y + (((int64_t)b * p.S) * p.H + h) * p.D;
    for (int r = r0 + g; r < r_end; r += kPoolGroups) {
      float xl[8], xh[8], cl[8], ch[8], sl[8], sh[8], yl[8], yh[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(xb + (int64_t)r * p.ss + lo)), xl);
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(xb + (int64_t)r * p.ss + lo + half)), xh);
      const float4* ct = reinterpret_cast<const float4*>(p.cos_t + (int64_t)r * p.D);
      const float4* st = reinterpret_cast<const float4*>(p.sin_t + (int64_t)r * p.D);
      *reinterpret_cast<float4*>(cl) = __ldg(ct + lo / 4);
      *reinterpret_cast<float4*>(cl + 4) = __ldg(ct + lo / 4 + 1);
      *reinterpret_cast<float4*>(ch) = __ldg(ct + (lo + half) / 4);
      *reinterpret_cast<float4*>(ch + 4) = __ldg(ct + (lo + half) / 4 + 1);
      *reinterpret_cast<float4*>(sl) = __ldg(st + lo / 4);
      *reinterpret_cast<float4*>(sl + 4) = __ldg(st + lo / 4 + 1);
      *reinterpret_cast<float4*>(sh) = __ldg(st + (lo + half) / 4);
      *reinterpret_cast<float4*>(sh + 4) = __ldg(st + (lo + half) / 4 + 1);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        yl[i] = fmaf(xl[i], cl[i], -xh[i] * sl[i]);   // first half: rotate_half gives -x2
        yh[i] = fmaf(xh[i], ch[i], xl[i] * sh[i]);    // second half: rotate_half gives x1
      }
      const uint4 ul = f32_to_bf16x8(yl), uh = f32_to_bf16x8(yh);
      __nv_bfloat16* yr = yb + (int64_t)r * p.H * p.D;
      *reinterpret_cast<uint4*>(yr + lo) = ul;
      *reinterpret_cast<uint4*>(yr + lo + half) = uh;
      if (r < r_valid) {
        float rl[8], rh[8];
        bf16x8_to_f32(ul, rl);
        bf16x8_to_f32(uh, rh);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[i] += rl[i];
          acc[8 + i] += rh[i];
        }
      }
    }
  }
  __shared__ float red[kPoolGroups][kPoolCols][17];
#pragma unroll
  for (int i = 0; i < 16; ++i) red[g][tc][i] = acc[i];
  __syncthreads();
  if (g == 0 && c < p.cols) {
    const int n = max(r_valid - r0, 0);
    const float inv = n > 0 ? 1.f / (float)n : 0.f;
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float s = red[0][tc][i];
#pragma unroll
      for (int gg = 1; gg < kPoolGroups; ++gg) s += red[gg][tc][i];
      m[i] = s * inv;
    }
    float* o = p.out + (((int64_t)b * p.H + h) * p.nb + blk) * p.D;
    reinterpret_cast<float4*>(o + lo)[0] = make_float4(m[0], m[1], m[2], m[3]);
    reinterpret_cast<float4*>(o + lo)[1] = make_float4(m[4], m[5], m[6], m[7]);
    reinterpret_cast<float4*>(o + lo + half)[0] = make_float4(m[8], m[9], m[10], m[11]);
    reinterpret_cast<float4*>(o + lo + half)[1] = make_float4(m[12], m[13], m[14], m[15]);
  }
}

// ---------------------------------------------------- score + top-k -------
// One CTA per (batch element, query head, kRows query blocks).
// Scores: every thread takes candidate key blocks in turn and computes their
// fp32 dot products with the kRows query-block means at once (the key-block
// mean streams from L2 as float4s; the query means sit transposed in shared
// memory and are read as broadcast float4s), so each key mean is read once
// per CTA and each multiply-add needs a fraction of a shared-memory load.
// Selection: one warp per row; the kh-th largest order-preserving score key
// is found by a radix select (4 passes of 8 bits over a per-warp 256-bin
// histogram), then one pass in ascending block order writes the blocks above
// it plus the lowest-index blocks equal to it.

constexpr int kRows = 16;
constexpr int kTopkThreads = 256;

struct TopkParams {
  const float* qbar;   // [B, Hq, nQb, D]
  const float* kbar;   // [B, Hkv, nKb, D]
  int Hq, Hkv, nQb, nKb, D, block_q, block_k, prefix_len;
  int seq_lens[kMaxSelectBatch];
  float keep[kMaxHeads];
  int32_t* indices;    // [B, Hq, nQb, nKb]
  int32_t* counts;     // [B, Hq, nQb]
};

// Monotone map float -> uint32 (larger float => larger key); -0 and +0 map to
// the same key because the score is canonicalised first.
__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// k = min(N, ceil(r * N)) in double precision (same expression as the host).
__device__ __forceinline__ int keep_count_dev(float r, int n) {
  if (n <= 0 || !(r > 0.f)) return 0;
  const double v = ceil((double)r * (double)n);
  return v >= (double)n ? n : (int)v;
}

__global__ void __launch_bounds__(kTopkThreads) score_topk_kernel(const __grid_constant__ TopkParams p) {
  extern __shared__ float sm[];
  const int D = p.D;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.z, h = blockIdx.y;
  const int qb0 = blockIdx.x * kRows;
  const int L = p.seq_lens[b];
  const int valid_kv = p.prefix_len + L;
  const int nkv = (valid_kv + p.block_k - 1) / p.block_k;
  const int npb = min((p.prefix_len + p.block_k - 1) / p.block_k, nkv);
  const int N = nkv - npb;
  const int kh = keep_count_dev(p.keep[h], N);
  const int nqv = (L + p.block_q - 1) / p.block_q;
  const int hk = h / (p.Hq / p.Hkv);
  const int rows_here = min(kRows, p.nQb - qb0);
  const int rows_valid = max(0, min(kRows, nqv - qb0));

  float* qT = sm;                                                    // [D][kRows]
  uint32_t* keys = reinterpret_cast<uint32_t*>(qT + D * kRows);      // [kRows][nKb]
  uint32_t* hist_all = keys + kRows * p.nKb;                         // [warps][256]

  if (rows_valid > 0 && kh > 0 && kh < N) {
    for (int i = threadIdx.x; i < D * kRows; i += blockDim.x) {
      const int e = i / kRows, r = i % kRows;
      qT[i] = (r < rows_valid) ? p.qbar[(((int64_t)b * p.Hq + h) * p.nQb + qb0 + r) * D + e] : 0.f;
    }
    __syncthreads();
    const float* kb_base = p.kbar + ((int64_t)b * p.Hkv + hk) * p.nKb * D;
    for (int c = threadIdx.x; c < N; c += blockDim.x) {
      const float4* krow = reinterpret_cast<const float4*>(kb_base + (int64_t)(npb + c) * D);
      float acc[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) acc[r] = 0.f;
#pragma unroll 4
      for (int e4 = 0; e4 < D / 4; ++e4) {
        const float4 kv = __ldg(krow + e4);
        const float ke[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4* qr = reinterpret_cast<const float4*>(qT + (e4 * 4 + u) * kRows);
#pragma unroll
          for (int r4 = 0; r4 < kRows / 4; ++r4) {
            const float4 q4 = qr[r4];
            acc[4 * r4 + 0] = fmaf(q4.x, ke[u], acc[4 * r4 + 0]);
            acc[4 * r4 + 1] = fmaf(q4.y, ke[u], acc[4 * r4 + 1]);
            acc[4 * r4 + 2] = fmaf(q4.z, ke[u], acc[4 * r4 + 2]);
            acc[4 * r4 + 3] = fmaf(q4.w, ke[u], acc[4 * r4 + 3]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r)
        if (r < rows_valid) keys[r * p.nKb + c] = order_key(acc[r] + 0.f);   // -0 -> +0
    }
    __syncthreads();
  }

  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int r = warp; r < rows_here; r += kTopkThreads / 32) {
    const int qb = qb0 + r;
    const int64_t row_id = ((int64_t)b * p.Hq + h) * p.nQb + qb;
    int32_t* out_idx = p.indices + row_id * p.nKb;
    if (qb >= nqv) {
      if (lane == 0) p.counts[row_id] = 0;
      continue;
    }
    for (int i = lane; i < npb; i += 32) out_idx[i] = i;
    if (lane == 0) p.counts[row_id] = npb + kh;
    if (kh == 0) continue;
    if (kh >= N) {
      for (int i = lane; i < N; i += 32) out_idx[npb + i] = npb + i;
      continue;
    }
    const uint32_t* my_keys = keys + r * p.nKb;
    // Threshold T = the kh-th largest key: most-significant-digit radix
    // select, 8 bits per pass, on a 256-bin histogram (one per warp) of the
    // keys whose higher digits equal those already chosen.  `remaining` is
    // T's rank among those keys.
    uint32_t* hist = hist_all + warp * 256;
    uint32_t T = 0, chosen = 0;
    uint32_t remaining = (uint32_t)kh;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = lane; i < 256; i += 32) hist[i] = 0u;
      __syncwarp();
      for (int i = lane; i < N; i += 32) {
        const uint32_t key = my_keys[i];
        if ((key & chosen) == T) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncwarp();
      // lane l holds digits 8 l .. 8 l + 7; `above` = keys with a larger digit
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[lane * 8 + j];
        tot += c[j];
      }
      uint32_t suf = tot;                 // keys with digit >= 8 lane (inclusive suffix scan)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      uint32_t above = suf - tot;
      int found = -1;
      uint32_t above_found = 0;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (found < 0 && above + c[j] >= remaining) {
          found = lane * 8 + j;
          above_found = above;
        }
        above += c[j];
      }
      // the digit is the largest one with (keys above it) < remaining <=
      // (keys at or above it): the highest lane that found one
      const uint32_t ball = __ballot_sync(0xffffffffu, found >= 0);
      const int src = 31 - __clz(ball);
      const int digit = __shfl_sync(0xffffffffu, found, src);
      remaining -= __shfl_sync(0xffffffffu, above_found, src);
      T |= (uint32_t)digit << shift;
      chosen |= 255u << shift;
      __syncwarp();
    }
    int c_gt = 0;
    for (int i = lane; i < N; i += 32) c_gt += (my_keys[i] > T) ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c_gt += __shfl_xor_sync(0xffffffffu, c_gt, o);
    const int need_eq = kh - c_gt;
    int written = 0, eq_seen = 0;
    for (int i0 = 0; i0 < N; i0 += 32) {
      const int i = i0 + lane;
      const uint32_t key = (i < N) ? my_keys[i] : 0u;
      const bool gt = (i < N) && key > T;
      const bool eq = (i < N) && key == T;
      const uint32_t eq_ball = __ballot_sync(0xffffffffu, eq);
      const int eq_rank = eq_seen + __popc(eq_ball & lt_mask);
      const bool sel = gt || (eq && eq_rank < need_eq);
      const uint32_t sel_ball = __ballot_sync(0xffffffffu, sel);
      if (sel) out_idx[npb + written + __popc(sel_ball & lt_mask)] = npb + i;
      written += __popc(sel_ball);
      eq_seen += __popc(eq_ball);
    }
  }
}

}  // namespace

static bsa_status launch_topk(const SelectArgs& a, cudaStream_t stream);

bsa_status launch_select(const SelectArgs& a, cudaStream_t stream) {
  bsa_status st;
  if (a.rope) {
    // RoPE on Q and K fused with their block means.
    for (int which = 0; which < 2; ++which) {
      RopePoolParams p{};
      const bool isq = which == 0;
      p.x = static_cast<const __nv_bfloat16*>(isq ? a.q : a.k);
      p.sb = isq ? a.q_sb : a.k_sb; p.ss = isq ? a.q_ss : a.k_ss; p.sh = isq ? a.q_sh : a.k_sh;
      p.y = static_cast<__nv_bfloat16*>(isq ? a.q_out : a.k_out);
      p.cos_t = isq ? a.cos_q : a.cos_k; p.sin_t = isq ? a.sin_q : a.sin_k;
      p.H = isq ? a.Hq : a.Hkv; p.D = a.d; p.S = isq ? a.Sq : a.Skv;
      p.block = isq ? a.block_q : a.block_k; p.nb = isq ? a.nQb : a.nKb; p.cols = p.H * a.d / 16;
      for (int b = 0; b < a.B; ++b) {
        const int L = a.seq_lens ? a.seq_lens[b] : a.Sq;
        p.valid[b] = isq ? L : a.prefix_len + L;
      }
      p.out = isq ? a.qbar : a.kbar;
      dim3 grid(p.nb, a.B, (p.cols + kPoolCols - 1) / kPoolCols);
      rope_pool_kernel<<<grid, kPoolCols * kPoolGroups, 0, stream>>>(p);
      if ((st = cuda_check(cudaGetLastError(), "rope_pool_kernel launch")) != BSA_OK) return st;
    }
    return launch_topk(a, stream);
  }
  // Pool Q over real query rows and K over real keys of every block.
  {
    PoolParams p{};
    p.x = static_cast<const __nv_bfloat16*>(a.q);
    p.sb = a.q_sb; p.ss = a.q_ss; p.sh = a.q_sh;
    p.H = a.Hq; p.D = a.d; p.block = a.block_q; p.nb = a.nQb; p.cols = a.Hq * a.d / 8;
    for (int b = 0; b < a.B; ++b) p.valid[b] = a.seq_lens ? a.seq_lens[b] : a.Sq;
    p.out = a.qbar;
    dim3 grid(a.nQb, a.B, (p.cols + kPoolCols - 1) / kPoolCols);
    pool_kernel<<<grid, kPoolCols * kPoolGroups, 0, stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "pool_kernel(Q) launch")) != BSA_OK) return st;
  }
  {
    PoolParams p{};
    p.x = static_cast<const __nv_bfloat16*>(a.k);
    p.sb = a.k_sb; p.ss = a.k_ss; p.sh = a.k_sh;
    p.H = a.Hkv; p.D = a.d; p.block = a.block_k; p.nb = a.nKb; p.cols = a.Hkv * a.d / 8;
    for (int b = 0; b < a.B; ++b) p.valid[b] = a.prefix_len + (a.seq_lens ? a.seq_lens[b] : a.Sq);
    p.out = a.kbar;
    dim3 grid(a.nKb, a.B, (p.cols + kPoolCols - 1) / kPoolCols);
    pool_kernel<<<grid, kPoolCols * kPoolGroups, 0, stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "pool_kernel(K) launch")) != BSA_OK) return st;
  }
  return launch_topk(a, stream);
}

static bsa_status launch_topk(const SelectArgs& a, cudaStream_t stream) {
  bsa_status st;
  {
    TopkParams p{};
    p.qbar = a.qbar; p.kbar = a.kbar;
    p.Hq = a.Hq; p.Hkv = a.Hkv; p.nQb = a.nQb; p.nKb = a.nKb; p.D = a.d;
    p.block_q = a.block_q; p.block_k = a.block_k; p.prefix_len = a.prefix_len;
    for (int b = 0; b < a.B; ++b) p.seq_lens[b] = a.seq_lens ? a.seq_lens[b] : a.Sq;
    for (int h = 0; h < a.Hq; ++h) p.keep[h] = a.keep[h];
    p.indices = a.indices; p.counts = a.counts;
    const size_t smem = sizeof(float) * (size_t)kRows * a.d + sizeof(uint32_t) * (size_t)kRows * a.nKb +
                        sizeof(uint32_t) * 256 * (kTopkThreads / 32);   // q means, keys, radix histograms
    if (smem > 227 * 1024)
      return set_error(BSA_ERR_UNSUPPORTED, "bsa_select: too many key blocks (nKb=" +
                                                std::to_string(a.nKb) + ") for one CTA's shared memory");
    // The kernel's shared-memory limit is raised once per device and size
    // (never lowered), so calls captured in a CUDA graph only launch.
    {
      static std::mutex mu;
      static int smem_set[64] = {};
      int dev = 0;
      cudaGetDevice(&dev);
      std::lock_guard<std::mutex> lock(mu);
      if (dev >= 64 || smem_set[dev] < (int)smem) {
        if ((st = cuda_check(cudaFuncSetAttribute(score_topk_kernel,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                             "cudaFuncSetAttribute(score_topk_kernel)")) != BSA_OK)
          return st;
        if (dev < 64) smem_set[dev] = (int)smem;
      }
    }
    dim3 grid((a.nQb + kRows - 1) / kRows, a.Hq, a.B);
    score_topk_kernel<<<grid, kTopkThreads, smem, stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "score_topk_kernel launch")) != BSA_OK) return st;
  }
  return BSA_OK;
}

}  // namespace bsa

// ------------------------------------------------------------------------
// bsa_select_noalloc: the selector with its block means in a static device
// array instead of caller workspace, for callers that cannot allocate device
// memory.  The array is the only scratch the selector needs; its size is the
// stated maximum and every device that loads the library keeps it for the
// life of the process.
namespace bsa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[BSA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up with cudaGetSymbolAddress
// the first time a device is used (the host-side symbol is only a stand-in,
// never a device address).  The unique ID of the context it was looked up in
// is kept with it: after cudaDeviceReset the module is loaded again in a new
// primary context, where the array may sit elsewhere, so a call made in a
// different context looks the address up again.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<F>(f);
  return nullptr;
}

// ID of the calling thread's current context; 0 when none is current yet.
bsa_status current_context_id(const char* fn, unsigned long long* id) {
  static std::once_flag once;
  static CtxGetCurrentFn get_ctx = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  if (!get_ctx || !get_id)
    return set_error(BSA_ERR_CUDA, std::string(fn) + ": cuCtxGetCurrent / cuCtxGetId are not available");
  CUcontext ctx = nullptr;
  *id = 0;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return set_error(BSA_ERR_CUDA, std::string(fn) + ": cuCtxGetCurrent failed");
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS)
    return set_error(BSA_ERR_CUDA, std::string(fn) + ": cuCtxGetId failed");
  return BSA_OK;
}

bsa_status noalloc_scratch(const char* fn, size_t need, void** ws, size_t* ws_bytes) {
  if (need > BSA_NOALLOC_SCRATCH_BYTES)
    return set_error(BSA_ERR_UNSUPPORTED, std::string(fn) + ": the block means need " + std::to_string(need) +
                                              " bytes, above the static scratch of " +
                                              std::to_string((size_t)BSA_NOALLOC_SCRATCH_BYTES) +
                                              " bytes; use bsa_select");
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static unsigned long long ctx_id[64] = {0};
  int dev = 0;
  bsa_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != BSA_OK) return st;
  if (dev < 0 || dev >= 64)
    return set_error(BSA_ERR_UNSUPPORTED, std::string(fn) + ": device ordinal " + std::to_string(dev) +
                                              " above the 64 devices it tracks");
  unsigned long long id = 0;
  if ((st = current_context_id(fn, &id)) != BSA_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || id == 0 || ctx_id[dev] != id) {
    void* p = nullptr;
    // also makes the device's primary context current if none was
    st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)");
    if (st != BSA_OK) return st;
    if ((st = current_context_id(fn, &id)) != BSA_OK) return st;
    addr[dev] = p;
    ctx_id[dev] = id;
  }
  *ws = addr[dev];
  *ws_bytes = BSA_NOALLOC_SCRATCH_BYTES;
  return BSA_OK;
}

}  // namespace
}  // namespace bsa

extern "C" bsa_status bsa_select_noalloc(const bsa_tensor* q, const bsa_tensor* k, int32_t prefix_len,
                                         const int32_t* seq_lens, int32_t block_q, int32_t block_k,
                                         const float* keep_ratio, int32_t n_keep, int32_t* indices,
                                         int32_t* counts, bsa_stream_t stream) {
  using namespace bsa;
  clear_error();
  return select_impl("bsa_select_noalloc", q, k, prefix_len, seq_lens, block_q, block_k, keep_ratio, n_keep,
                     indices, counts, nullptr, 0, stream, nullptr, noalloc_scratch);
}
