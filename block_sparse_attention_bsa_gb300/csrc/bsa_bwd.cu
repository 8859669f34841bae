// Backward pass of the selected-block attention (dQ, dK, dV) for sm_103a.
//
// The forward (vllm-omni PR 8335, Purpose: attend exactly the selector's
// per-query-head block lists; cosmos_parallel.py: non-causal attention over
// cat(und, gen) with padded keys masked) stores a natural-log LSE per row;
// the backward recomputes P = exp(scale q.k - lse) tile by tile:
//   D_i = sum_c dO_ic O_ic,   dS_ij = P_ij (dO_i.v_j - D_i),
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,
//   dV_j = sum_i P_ij dO_i,
// with dK/dV of a KV head summed over every query head of its group and
// every query block that listed the key's block.  No atomics touch the
// gradients, so results are deterministic:
//  * bwd_dq_kernel walks query tiles (128 rows) over their listed key blocks
//    and accumulates dQ in TMEM (S = Q K^T, dP = dO V^T, dQ += dS K);
//  * bwd_dkdv_kernel walks key blocks over the query tiles that listed them
//    (an inverse list built from bitmaps, ordered by query tile) and
//    accumulates dK and dV in TMEM (S^T = K Q^T, dP^T = V dO^T,
//    dV += P^T dO, dK += dS^T Q).
// Both use TMA tile loads, one MMA-issuing thread and one 128-thread
// warpgroup for the elementwise part; every wait is bounded.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {
namespace {

constexpr int kD = 128;                 // head dim
constexpr int kBKb = 128;               // key block
constexpr int kT = 128;                 // query tile rows
constexpr int kChunk = 128 * 128;       // 128 rows x 64 bf16 (one 128-byte column chunk)
constexpr int kTile = 2 * kChunk;       // 128 rows x 128 bf16 = 32 KB
constexpr int kThreads = 256;           // warp 0 TMA, warp 1 MMA, warps 4..7 elementwise
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  CUtensorMap tq[kMaxFwdBatch];
  CUtensorMap tk[kMaxFwdBatch];
  CUtensorMap tv[kMaxFwdBatch];
  CUtensorMap tdo[kMaxFwdBatch];
  int seq_lens[kMaxFwdBatch];
  int b0, Bn, Hq, Hkv, G, Sq, Skv, nQb, nKb, nQt, block_q, prefix_len, n_items;
  const int32_t* indices;     // [B, Hq, nQb, nKb]
  const int32_t* counts;      // [B, Hq, nQb]
  const float* lse;           // [B, Hq, Sq]
  const float* Dd;            // [B, Hq, Sq]
  const int32_t* inv_cnt;     // [B, Hkv, nKb]
  const int32_t* inv_list;    // [B, Hkv, nKb, G * nQb]: listing rows g * nQb + qb, ascending
  float scale, scale_log2;
  __nv_bfloat16* dq;          // [B, Sq, Hq, d]
  __nv_bfloat16* dk;          // [B, Skv, Hkv, d]
  __nv_bfloat16* dv;
};

struct Ring2 {
  uint32_t stage = 0, phase = 0;
  __device__ __forceinline__ void next() {
    if (++stage == 2) { stage = 0; phase ^= 1u; }
  }
};

// Descriptor helpers for the 128 x 128 bf16 tiles (two 128-byte swizzled
// column chunks of 16 KB): K-major use (rows are M or N, channels are K) and
// MN-major use (channels are N, rows are K).
__device__ __forceinline__ uint64_t kmaj(uint32_t tile, int kk) {
  return sdesc_sw128(tile + (kk / 4) * kChunk + (kk % 4) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmaj(uint32_t tile, int kk) {
  return sdesc_sw128(tile + kk * 16 * 128, kChunk, 1024);
}

// ---------------------------------------------------------------- dQ ---
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_s = smem;                    // Q tile
  uint8_t* do_s = smem + kTile;           // dO tile
  uint8_t* kv_s = smem + 2 * kTile;       // 2 stages of (K tile, V tile)
  uint64_t* bars = reinterpret_cast<uint64_t*>(kv_s + 2 * 2 * kTile);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* ds_full = bars + 3;
  uint64_t* dq_full = bars + 4;
  uint64_t* kv_full = bars + 5;           // [2]
  uint64_t* kv_empty = bars + 7;          // [2]
  uint64_t* mma_done = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_empty), 1);
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(ds_full), 128);
    mbar_init(smem_u32(dq_full), 1);
    mbar_init(smem_u32(mma_done), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(kv_full + i), 1);
      mbar_init(smem_u32(kv_empty + i), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;       // S cols [0,128), dP [128,256), dQ [256,384)

  // item -> (request, KV head, query tile, query head of the group)
  auto decode = [&](int t, int& bl, int& h, int& qt, int& qb, int& n, int& L) {
    const int g = t % p.G;
    int r = t / p.G;
    qt = r % p.nQt;
    r /= p.nQt;
    const int hk = r % p.Hkv;
    bl = r / p.Hkv;
    h = hk * p.G + g;
    qb = qt * kT / p.block_q;
    L = p.seq_lens[bl];
    n = 0;
    if (qt * kT < L) {
      const int c = p.counts[((int64_t)(p.b0 + bl) * p.Hq + h) * p.nQb + qb];
      n = c < 0 ? 0 : min(c, p.nKb);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA ---
    if (lane == 0) {
      Ring2 ring;
      uint32_t qi = 0;
      int q_armed = -1, kv_armed[2] = {-1, -1};     // parity of each barrier's last arming
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
        int bl, h, qt, qb, n, L;
        decode(t, bl, h, qt, qb, n, L);
        if (n == 0) continue;
        ok = mbar_wait(smem_u32(q_empty), (qi & 1u) ^ 1u, abort_flag);
        if (!ok) break;
        q_armed = (int)(qi & 1u);
        ++qi;
        mbar_arrive_expect_tx(smem_u32(q_full), 2 * kTile);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(smem_u32(q_s) + c * kChunk, &p.tq[bl], smem_u32(q_full), c * 64, qt * kT, h);
          tma_load_3d(smem_u32(do_s) + c * kChunk, &p.tdo[bl], smem_u32(q_full), c * 64, qt * kT, h);
        }
        const int32_t* lst = p.indices + (((int64_t)(p.b0 + bl) * p.Hq + h) * p.nQb + qb) * p.nKb;
        const int hk = h / p.G;
        for (int j = 0; j < n && ok; ++j) {
          int kb = __ldg(lst + j);
          if (kb < 0 || kb >= p.nKb) kb = p.nKb;
          ok = mbar_wait(smem_u32(kv_empty + ring.stage), ring.phase ^ 1u, abort_flag);
          if (!ok) break;
          const uint32_t fb = smem_u32(kv_full + ring.stage);
          const uint32_t base = smem_u32(kv_s) + ring.stage * 2 * kTile;
          mbar_arrive_expect_tx(fb, 2 * kTile);
          kv_armed[ring.stage] = (int)ring.phase;
          for (int c = 0; c < 2; ++c) {
            tma_load_3d(base + c * kChunk, &p.tk[bl], fb, c * 64, kb * kBKb, hk);
            tma_load_3d(base + kTile + c * kChunk, &p.tv[bl], fb, c * 64, kb * kBKb, hk);
          }
          ring.next();
        }
      }
      // let this thread's copies land before the CTA can exit
      if (q_armed >= 0) mbar_drain(smem_u32(q_full), (uint32_t)q_armed);
      for (int i = 0; i < 2; ++i)
        if (kv_armed[i] >= 0) mbar_drain(smem_u32(kv_full + i), (uint32_t)kv_armed[i]);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA ---
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_mn = idesc_bf16_f32(128, 128, true);
      Ring2 ring;
      uint32_t qi = 0, di = 0;
      bool ok = true;
      const uint32_t qa = smem_u32(q_s), da = smem_u32(do_s), kva = smem_u32(kv_s);
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
        int bl, h, qt, qb, n, L;
        decode(t, bl, h, qt, qb, n, L);
        if (n == 0) continue;
        ok = mbar_wait(smem_u32(q_full), qi & 1u, abort_flag);
        ++qi;
        if (!ok) break;
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t st = ring.stage;
          ok = mbar_wait(smem_u32(kv_full + st), ring.phase, abort_flag);
          ring.next();
          if (!ok) break;
          tc_fence_after();
          const uint32_t kt = kva + st * 2 * kTile, vt = kt + kTile;
          // S = Q K^T, dP = dO V^T
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) mma_ss(tmem, kmaj(qa, kk), kmaj(kt, kk), idesc_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) mma_ss(tmem + 128, kmaj(da, kk), kmaj(vt, kk), idesc_s, kk > 0);
          mma_commit(smem_u32(s_full));
          if (j == n - 1) mma_commit(smem_u32(q_empty));
          ok = mbar_wait(smem_u32(ds_full), di & 1u, abort_flag);
          ++di;
          if (!ok) break;
          tc_fence_after();
          // dQ += dS K  (dS bf16 in TMEM over S's first 64 columns; K as MN-major B)
#pragma unroll
          for (int kk = 0; kk < kBKb / 16; ++kk)
            mma_ts(tmem + 256, tmem + kk * 8, mnmaj(kt, kk), idesc_mn, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(kv_empty + st));
          if (j == n - 1) mma_commit(smem_u32(dq_full));
        }
      }
      mma_commit(smem_u32(mma_done));        // every MMA issued above has finished
      mbar_drain(smem_u32(mma_done), 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ----------------------------------------------------- elementwise ---
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(wq * 32) << 16;
    uint32_t si = 0, oi = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
      int bl, h, qt, qb, n, L;
      decode(t, bl, h, qt, qb, n, L);
      const int b = p.b0 + bl;
      const int row = qt * kT + r;
      const bool row_exists = row < p.Sq;
      const bool row_ok = row < L;
      __nv_bfloat16* drow = p.dq + (((int64_t)b * p.Sq + row) * p.Hq + h) * kD;
      if (n == 0) {
        if (row_exists) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < kD / 8; ++i) reinterpret_cast<uint4*>(drow)[i] = z;
        }
        continue;
      }
      const int64_t li = ((int64_t)b * p.Hq + h) * p.Sq + row;
      const float lse2 = row_ok ? __ldg(p.lse + li) * kLog2e : 0.f;
      const float Dr = row_ok ? __ldg(p.Dd + li) : 0.f;
      const int valid_kv = p.prefix_len + L;
      const int32_t* lst = p.indices + (((int64_t)b * p.Hq + h) * p.nQb + qb) * p.nKb;
      for (int j = 0; j < n; ++j) {
        int kb = __ldg(lst + j);
        if (kb < 0 || kb >= p.nKb) kb = p.nKb;
        const int kvalid = row_ok ? valid_kv - kb * kBKb : 0;
        ok = mbar_wait(smem_u32(s_full), si & 1u, abort_flag);
        ++si;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float s[64], dp[64];
          tmem_ld32f(tmem + lb + h2 * 64, s);
          tmem_ld32f(tmem + lb + h2 * 64 + 32, s + 32);
          tmem_ld32f(tmem + lb + 128 + h2 * 64, dp);
          tmem_ld32f(tmem + lb + 128 + h2 * 64 + 32, dp + 32);
          tmem_wait_ld();
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c0 = h2 * 64 + 2 * i;
            const float p0 = (c0 < kvalid) ? ex2_approx(fmaf(s[2 * i], p.scale_log2, -lse2)) : 0.f;
            const float p1 = (c0 + 1 < kvalid) ? ex2_approx(fmaf(s[2 * i + 1], p.scale_log2, -lse2)) : 0.f;
            pk[i] = pack_bf16x2(p0 * (dp[2 * i] - Dr), p1 * (dp[2 * i + 1] - Dr));
          }
          tmem_st32(tmem + lb + h2 * 32, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(ds_full));
      }
      if (!ok) break;
      ok = mbar_wait(smem_u32(dq_full), oi & 1u, abort_flag);
      ++oi;
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        float o[32];
        tmem_ld32f(tmem + lb + 256 + c * 32, o);
        tmem_wait_ld();
        if (row_exists) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = row_ok ? pack_bf16x2(o[2 * i] * p.scale, o[2 * i + 1] * p.scale) : 0u;
          uint4* dst = reinterpret_cast<uint4*>(drow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------- dK, dV ---
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* k_s = smem;                    // K tile of the key block
  uint8_t* v_s = smem + kTile;            // V tile
  uint8_t* qdo_s = smem + 2 * kTile;      // 2 stages of (Q tile, dO tile)
  float* rowv = reinterpret_cast<float*>(qdo_s + 2 * 2 * kTile);   // [2][2][128]: lse*log2e, D
  uint64_t* bars = reinterpret_cast<uint64_t*>(rowv + 2 * 2 * kT);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* p_full = bars + 3;
  uint64_t* acc_full = bars + 4;
  uint64_t* qdo_full = bars + 5;          // [2]
  uint64_t* qdo_empty = bars + 7;         // [2]
  uint64_t* row_ready = bars + 9;         // [2]: lse/D of a step staged in smem
  uint64_t* mma_done = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(kv_full), 1);
    mbar_init(smem_u32(kv_empty), 1);
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(p_full), 128);
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(mma_done), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(qdo_full + i), 1);
      mbar_init(smem_u32(qdo_empty + i), 1);
      mbar_init(smem_u32(row_ready + i), 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;       // S^T [0,128), dP^T [128,256), dV [256,384), dK [384,512)
  const int tiles_per_block = p.block_q / kT;

  // item -> (request, KV head, key block); steps = listed query blocks x tiles per block
  auto decode = [&](int t, int& bl, int& hk, int& kb, int& steps, const int32_t*& lst) {
    kb = t % p.nKb;
    const int r = t / p.nKb;
    hk = r % p.Hkv;
    bl = r / p.Hkv;
    const int64_t key = ((int64_t)(p.b0 + bl) * p.Hkv + hk) * p.nKb + kb;
    steps = p.inv_cnt[key] * tiles_per_block;
    lst = p.inv_list + key * p.G * p.nQb;
  };
  // step s of an item -> (query head, query tile)
  auto step_tile = [&](const int32_t* lst, int hk, int s, int& h, int& qt) {
    const int e = __ldg(lst + s / tiles_per_block);
    const int g = e / p.nQb, qb = e - g * p.nQb;
    h = hk * p.G + g;
    qt = qb * tiles_per_block + s % tiles_per_block;
  };

  if (warp == 0) {
    if (lane == 0) {
      Ring2 ring;
      uint32_t ki = 0;
      int kv_armed = -1, qdo_armed[2] = {-1, -1};   // parity of each barrier's last arming
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
        int bl, hk, kb, steps;
        const int32_t* lst;
        decode(t, bl, hk, kb, steps, lst);
        if (steps == 0) continue;
        ok = mbar_wait(smem_u32(kv_empty), (ki & 1u) ^ 1u, abort_flag);
        if (!ok) break;
        kv_armed = (int)(ki & 1u);
        ++ki;
        mbar_arrive_expect_tx(smem_u32(kv_full), 2 * kTile);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(smem_u32(k_s) + c * kChunk, &p.tk[bl], smem_u32(kv_full), c * 64, kb * kBKb, hk);
          tma_load_3d(smem_u32(v_s) + c * kChunk, &p.tv[bl], smem_u32(kv_full), c * 64, kb * kBKb, hk);
        }
        for (int s = 0; s < steps && ok; ++s) {
          int h, qt;
          step_tile(lst, hk, s, h, qt);
          ok = mbar_wait(smem_u32(qdo_empty + ring.stage), ring.phase ^ 1u, abort_flag);
          if (!ok) break;
          const uint32_t fb = smem_u32(qdo_full + ring.stage);
          const uint32_t base = smem_u32(qdo_s) + ring.stage * 2 * kTile;
          mbar_arrive_expect_tx(fb, 2 * kTile);
          qdo_armed[ring.stage] = (int)ring.phase;
          for (int c = 0; c < 2; ++c) {
            tma_load_3d(base + c * kChunk, &p.tq[bl], fb, c * 64, qt * kT, h);
            tma_load_3d(base + kTile + c * kChunk, &p.tdo[bl], fb, c * 64, qt * kT, h);
          }
          ring.next();
        }
      }
      // let this thread's copies land before the CTA can exit
      if (kv_armed >= 0) mbar_drain(smem_u32(kv_full), (uint32_t)kv_armed);
      for (int i = 0; i < 2; ++i)
        if (qdo_armed[i] >= 0) mbar_drain(smem_u32(qdo_full + i), (uint32_t)qdo_armed[i]);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_mn = idesc_bf16_f32(128, 128, true);
      Ring2 ring;
      uint32_t ki = 0, pi = 0;
      bool ok = true;
      const uint32_t ka = smem_u32(k_s), va = smem_u32(v_s), qda = smem_u32(qdo_s);
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
        int bl, hk, kb, steps;
        const int32_t* lst;
        decode(t, bl, hk, kb, steps, lst);
        if (steps == 0) continue;
        ok = mbar_wait(smem_u32(kv_full), ki & 1u, abort_flag);
        ++ki;
        if (!ok) break;
        for (int s = 0; s < steps && ok; ++s) {
          const uint32_t st = ring.stage;
          ok = mbar_wait(smem_u32(qdo_full + st), ring.phase, abort_flag);
          ring.next();
          if (!ok) break;
          tc_fence_after();
          const uint32_t qt_s = qda + st * 2 * kTile, dot_s = qt_s + kTile;
          // S^T = K Q^T, dP^T = V dO^T   (M = keys, N = query rows)
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) mma_ss(tmem, kmaj(ka, kk), kmaj(qt_s, kk), idesc_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) mma_ss(tmem + 128, kmaj(va, kk), kmaj(dot_s, kk), idesc_s, kk > 0);
          mma_commit(smem_u32(s_full));
          if (s == steps - 1) mma_commit(smem_u32(kv_empty));
          ok = mbar_wait(smem_u32(p_full), pi & 1u, abort_flag);
          ++pi;
          if (!ok) break;
          tc_fence_after();
          // dV += P^T dO, dK += dS^T Q   (A from TMEM, B = the row tiles as MN-major)
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + 256, tmem + kk * 8, mnmaj(dot_s, kk), idesc_mn, (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + 384, tmem + 128 + kk * 8, mnmaj(qt_s, kk), idesc_mn, (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(qdo_empty + st));
          if (s == steps - 1) mma_commit(smem_u32(acc_full));
        }
      }
      mma_commit(smem_u32(mma_done));        // every MMA issued above has finished
      mbar_drain(smem_u32(mma_done), 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(wq * 32) << 16;
    uint32_t si = 0, ai = 0, gstep = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
      int bl, hk, kb, steps;
      const int32_t* lst;
      decode(t, bl, hk, kb, steps, lst);
      const int b = p.b0 + bl;
      const int L = p.seq_lens[bl];
      const int key = kb * kBKb + r;
      const bool key_exists = key < p.Skv;
      const bool key_ok = key < p.prefix_len + L;
      __nv_bfloat16* dkrow = p.dk + (((int64_t)b * p.Skv + key) * p.Hkv + hk) * kD;
      __nv_bfloat16* dvrow = p.dv + (((int64_t)b * p.Skv + key) * p.Hkv + hk) * kD;
      if (steps == 0) {
        if (key_exists) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < kD / 8; ++i) {
            reinterpret_cast<uint4*>(dkrow)[i] = z;
            reinterpret_cast<uint4*>(dvrow)[i] = z;
          }
        }
        continue;
      }
      for (int s = 0; s < steps; ++s, ++gstep) {
        int h, qt;
        step_tile(lst, hk, s, h, qt);
        // per-column values of this query tile: lse (log2 units; +inf marks a
        // padded row so its P is 0) and D, double-buffered by step parity
        const uint32_t buf = gstep & 1u;
        float* lse_b = rowv + buf * 2 * kT;
        float* d_b = lse_b + kT;
        {
          const int row = qt * kT + r;
          const int64_t li = ((int64_t)b * p.Hq + h) * p.Sq + row;
          lse_b[r] = row < L ? __ldg(p.lse + li) * kLog2e : INFINITY;
          d_b[r] = row < L ? __ldg(p.Dd + li) : 0.f;
        }
        // the buffer is rewritten two steps later, after every thread has
        // arrived once more (so finished reading it)
        mbar_arrive(smem_u32(row_ready + buf));
        ok = mbar_wait(smem_u32(row_ready + buf), (gstep >> 1) & 1u, abort_flag);
        if (!ok) break;
        ok = mbar_wait(smem_u32(s_full), si & 1u, abort_flag);
        ++si;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float sv[64], dp[64];
          tmem_ld32f(tmem + lb + h2 * 64, sv);
          tmem_ld32f(tmem + lb + h2 * 64 + 32, sv + 32);
          tmem_ld32f(tmem + lb + 128 + h2 * 64, dp);
          tmem_ld32f(tmem + lb + 128 + h2 * 64 + 32, dp + 32);
          tmem_wait_ld();
          uint32_t pp[32], pd[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c0 = h2 * 64 + 2 * i;
            const float p0 = key_ok ? ex2_approx(fmaf(sv[2 * i], p.scale_log2, -lse_b[c0])) : 0.f;
            const float p1 = key_ok ? ex2_approx(fmaf(sv[2 * i + 1], p.scale_log2, -lse_b[c0 + 1])) : 0.f;
            pp[i] = pack_bf16x2(p0, p1);
            pd[i] = pack_bf16x2(p0 * (dp[2 * i] - d_b[c0]), p1 * (dp[2 * i + 1] - d_b[c0 + 1]));
          }
          tmem_st32(tmem + lb + h2 * 32, pp);
          tmem_st32(tmem + lb + 128 + h2 * 32, pd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(p_full));
      }
      if (!ok) break;
      ok = mbar_wait(smem_u32(acc_full), ai & 1u, abort_flag);
      ++ai;
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst_row = which == 0 ? dvrow : dkrow;
        const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          float o[32];
          tmem_ld32f(tmem + lb + 256 + which * 128 + c * 32, o);
          tmem_wait_ld();
          if (key_exists) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = key_ok ? pack_bf16x2(o[2 * i] * mul, o[2 * i + 1] * mul) : 0u;
            uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------- preprocessing ---
// D[b, h, i] = sum_c dO[b, i, h, c] * O[b, i, h, c] for real rows (0 for
// padding).  One warp per (b, row, h); 16-byte loads.
struct PrepParams {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  int64_t o_sb, o_ss, o_sh, d_sb, d_ss, d_sh;
  int B, Sq, Hq;
  int seq_lens[kMaxSelectBatch];
  float* Dd;
};

__global__ void bwd_prep_kernel(const __grid_constant__ PrepParams p) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int64_t total = (int64_t)p.B * p.Sq * p.Hq;
  if (w >= total) return;
  const int h = (int)(w % p.Hq);
  const int64_t rr = w / p.Hq;
  const int row = (int)(rr % p.Sq);
  const int b = (int)(rr / p.Sq);
  float acc = 0.f;
  if (row < p.seq_lens[b] && lane < kD / 4) {
    const __nv_bfloat16* op = p.o + b * p.o_sb + (int64_t)row * p.o_ss + (int64_t)h * p.o_sh + lane * 4;
    const __nv_bfloat16* dp = p.dout + b * p.d_sb + (int64_t)row * p.d_ss + (int64_t)h * p.d_sh + lane * 4;
    const uint2 a = *reinterpret_cast<const uint2*>(op);
    const uint2 c = *reinterpret_cast<const uint2*>(dp);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(c2[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) p.Dd[((int64_t)b * p.Hq + h) * p.Sq + row] = acc;
}

// ------------------------------------------------------ inverse lists ---
// Bitmaps: bit (g * nQb + qb, kb) of a KV head is set when query head
// hk * G + g listed block kb for query block qb (blocks with no real row are
// skipped).  One warp per list; OR is order-free, so the result is
// deterministic.
struct BitmapParams {
  const int32_t* indices;
  const int32_t* counts;
  uint32_t* bm;               // [B, Hkv, G * nQb, words]
  int B, Hq, Hkv, G, nQb, nKb, block_q, words;
  int seq_lens[kMaxSelectBatch];
};

__global__ void bwd_bitmap_kernel(const __grid_constant__ BitmapParams p) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int64_t rows = (int64_t)p.B * p.Hq * p.nQb;
  if (w >= rows) return;
  const int qb = (int)(w % p.nQb);
  const int64_t bh = w / p.nQb;
  const int h = (int)(bh % p.Hq), b = (int)(bh / p.Hq);
  if (qb * p.block_q >= p.seq_lens[b]) return;
  const int hk = h / p.G, g = h - hk * p.G;
  const int c = min(max(p.counts[w], 0), p.nKb);
  const int32_t* lst = p.indices + w * p.nKb;
  uint32_t* row = p.bm + ((((int64_t)b * p.Hkv + hk) * p.G + g) * p.nQb + qb) * p.words;
  for (int i = lane; i < c; i += 32) {
    const int kb = lst[i];
    if (kb >= 0 && kb < p.nKb) atomicOr(row + (kb >> 5), 1u << (kb & 31));
  }
}

// One warp per (b, hk, 32 key blocks): reads the bitmap 32 rows at a time
// (one row per lane), transposes each 32 x 32 bit square with ballots so that
// lane i holds the rows that listed key block 32 w + i, and appends them in
// ascending row order to that block's list.
struct InvParams {
  const uint32_t* bm;
  int32_t* inv_cnt;
  int32_t* inv_list;
  int n_groups, nrows, nKb, words;
};

__global__ void bwd_inverse_kernel(const __grid_constant__ InvParams p) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (wid >= (int64_t)p.n_groups * p.words) return;
  const int w = (int)(wid % p.words);
  const int64_t gi = wid / p.words;
  const uint32_t* bm = p.bm + gi * p.nrows * p.words;
  const int kb = w * 32 + lane;
  int32_t* out = p.inv_list + (gi * p.nKb + min(kb, p.nKb - 1)) * p.nrows;
  int cnt = 0;
  for (int r0 = 0; r0 < p.nrows; r0 += 32) {
    const int r = r0 + lane;
    const uint32_t word = r < p.nrows ? bm[(int64_t)r * p.words + w] : 0u;
    uint32_t mine = 0;
#pragma unroll
    for (int bit = 0; bit < 32; ++bit) {
      const uint32_t m = __ballot_sync(0xffffffffu, (word >> bit) & 1u);
      if (lane == bit) mine = m;
    }
    while (mine) {                      // bits exist only for kb < nKb
      out[cnt++] = r0 + __ffs(mine) - 1;
      mine &= mine - 1;
    }
  }
  if (kb < p.nKb) p.inv_cnt[gi * p.nKb + kb] = cnt;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bsa_status encode(CUtensorMap* m, const void* base, int64_t rows, int64_t H, int64_t ss, int64_t sh,
                  const char* name) {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return set_error(BSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    fn = reinterpret_cast<EncodeFn>(f);
  }
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)H};
  cuuint64_t strides[2] = {(cuuint64_t)(ss * 2), (cuuint64_t)(sh * 2)};
  cuuint32_t box[3] = {64u, 128u, 1u};
  cuuint32_t es[3] = {1u, 1u, 1u};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(BSA_ERR_CUDA, std::string("cuTensorMapEncodeTiled failed for ") + name);
  return BSA_OK;
}

constexpr int kDqSmem = 2 * kTile + 2 * 2 * kTile + 256 + 1024;   // tiles, barriers, alignment
constexpr int kDkvSmem = 2 * kTile + 2 * 2 * kTile + 2 * 2 * kT * 4 + 256 + 1024;

}  // namespace

size_t backward_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int block_q, int block_k) {
  const int64_t nQb = cdiv64(Sq, block_q), nKb = cdiv64(Skv, block_k), G = Hq / Hkv;
  const int64_t words = cdiv64(nKb, 32);
  auto al = [](int64_t x) { return (size_t)((x + 255) & ~(int64_t)255); };
  return al((int64_t)B * Hq * Sq * 4)                      // D
         + al((int64_t)B * Hkv * G * nQb * words * 4)      // bitmaps
         + al((int64_t)B * Hkv * nKb * 4)                  // inverse counts
         + al((int64_t)B * Hkv * nKb * G * nQb * 4);       // inverse lists
}

bsa_status launch_backward(const BackwardArgs& a, cudaStream_t stream) {
  bsa_status st;
  const int G = a.Hq / a.Hkv;
  const int nQb = (int)cdiv64(a.Sq, a.block_q), nKb = (int)cdiv64(a.Skv, a.block_k);
  const int words = (nKb + 31) / 32;
  auto al = [](int64_t x) { return (size_t)((x + 255) & ~(int64_t)255); };
  char* ws = static_cast<char*>(a.workspace);
  float* Dd = reinterpret_cast<float*>(ws);
  ws += al((int64_t)a.B * a.Hq * a.Sq * 4);
  uint32_t* bm = reinterpret_cast<uint32_t*>(ws);
  const size_t bm_bytes = al((int64_t)a.B * a.Hkv * G * nQb * words * 4);
  ws += bm_bytes;
  int32_t* inv_cnt = reinterpret_cast<int32_t*>(ws);
  ws += al((int64_t)a.B * a.Hkv * nKb * 4);
  int32_t* inv_list = reinterpret_cast<int32_t*>(ws);

  {  // D = rowsum(dO * O)
    PrepParams pp{};
    pp.o = static_cast<const __nv_bfloat16*>(a.o); pp.dout = static_cast<const __nv_bfloat16*>(a.dout);
    pp.o_sb = a.o_sb; pp.o_ss = a.o_ss; pp.o_sh = a.o_sh; pp.d_sb = a.d_sb; pp.d_ss = a.d_ss; pp.d_sh = a.d_sh;
    pp.B = a.B; pp.Sq = a.Sq; pp.Hq = a.Hq;
    for (int b = 0; b < a.B; ++b) pp.seq_lens[b] = a.seq_lens ? a.seq_lens[b] : a.Sq;
    pp.Dd = Dd;
    const int64_t warps = (int64_t)a.B * a.Sq * a.Hq;
    bwd_prep_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(pp);
    if ((st = cuda_check(cudaGetLastError(), "bwd_prep_kernel launch")) != BSA_OK) return st;
  }
  {  // inverse lists
    if ((st = cuda_check(cudaMemsetAsync(bm, 0, bm_bytes, stream), "cudaMemsetAsync(bitmaps)")) != BSA_OK) return st;
    BitmapParams bp{};
    bp.indices = a.indices; bp.counts = a.counts; bp.bm = bm;
    bp.B = a.B; bp.Hq = a.Hq; bp.Hkv = a.Hkv; bp.G = G; bp.nQb = nQb; bp.nKb = nKb; bp.block_q = a.block_q;
    bp.words = words;
    for (int b = 0; b < a.B; ++b) bp.seq_lens[b] = a.seq_lens ? a.seq_lens[b] : a.Sq;
    const int64_t rows = (int64_t)a.B * a.Hq * nQb;
    bwd_bitmap_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(bp);
    if ((st = cuda_check(cudaGetLastError(), "bwd_bitmap_kernel launch")) != BSA_OK) return st;
    InvParams ip{};
    ip.bm = bm; ip.inv_cnt = inv_cnt; ip.inv_list = inv_list;
    ip.n_groups = a.B * a.Hkv; ip.nrows = G * nQb; ip.nKb = nKb; ip.words = words;
    const int64_t warps = (int64_t)ip.n_groups * words;
    bwd_inverse_kernel<<<(unsigned)((warps * 32 + 127) / 128), 128, 0, stream>>>(ip);
    if ((st = cuda_check(cudaGetLastError(), "bwd_inverse_kernel launch")) != BSA_OK) return st;
  }
  static bool attr = false;
  if (!attr) {
    if ((st = cuda_check(cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem),
                         "cudaFuncSetAttribute(bwd_dq_kernel)")) != BSA_OK)
      return st;
    if ((st = cuda_check(cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDkvSmem),
                         "cudaFuncSetAttribute(bwd_dkdv_kernel)")) != BSA_OK)
      return st;
    attr = true;
  }
  const int sms = num_sms();
  for (int b0 = 0; b0 < a.B; b0 += kMaxFwdBatch) {
    const int Bn = std::min(kMaxFwdBatch, a.B - b0);
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    for (int i = 0; i < Bn; ++i) {
      const int b = b0 + i;
      const int L = a.seq_lens ? a.seq_lens[b] : a.Sq;
      p.seq_lens[i] = L;
      const char* qb = static_cast<const char*>(a.q) + (int64_t)b * a.q_sb * 2;
      const char* kb = static_cast<const char*>(a.k) + (int64_t)b * a.k_sb * 2;
      const char* vb = static_cast<const char*>(a.v) + (int64_t)b * a.v_sb * 2;
      const char* db = static_cast<const char*>(a.dout) + (int64_t)b * a.d_sb * 2;
      if ((st = encode(&p.tq[i], qb, L, a.Hq, a.q_ss, a.q_sh, "Q")) != BSA_OK) return st;
      if ((st = encode(&p.tdo[i], db, L, a.Hq, a.d_ss, a.d_sh, "dO")) != BSA_OK) return st;
      if ((st = encode(&p.tk[i], kb, a.prefix_len + L, a.Hkv, a.k_ss, a.k_sh, "K")) != BSA_OK) return st;
      if ((st = encode(&p.tv[i], vb, a.prefix_len + L, a.Hkv, a.v_ss, a.v_sh, "V")) != BSA_OK) return st;
    }
    p.b0 = b0; p.Bn = Bn; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.Sq = a.Sq; p.Skv = a.Skv;
    p.nQb = nQb; p.nKb = nKb; p.nQt = (int)cdiv64(a.Sq, kT); p.block_q = a.block_q; p.prefix_len = a.prefix_len;
    p.indices = a.indices; p.counts = a.counts; p.lse = a.lse; p.Dd = Dd;
    p.inv_cnt = inv_cnt; p.inv_list = inv_list;
    p.scale = a.scale; p.scale_log2 = a.scale * kLog2e;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.n_items = Bn * a.Hkv * p.nQt * G;
    bwd_dq_kernel<<<std::min(p.n_items, sms), kThreads, kDqSmem, stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "bwd_dq_kernel launch")) != BSA_OK) return st;
    p.n_items = Bn * a.Hkv * nKb;
    bwd_dkdv_kernel<<<std::min(p.n_items, sms), kThreads, kDkvSmem, stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "bwd_dkdv_kernel launch")) != BSA_OK) return st;
  }
  return BSA_OK;
}

}  // namespace bsa
