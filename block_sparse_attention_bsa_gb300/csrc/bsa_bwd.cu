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
// Every MMA is M128 x N128 (an N64 MMA costs as long as an N128 one).  Two
// elementwise warpgroups split each 128 x 128 score tile by columns and keep
// P in registers between the exponentials and dS, which frees the score
// columns early enough for the next tile's MMAs to overlap the elementwise
// work.  TMA tile loads, one MMA-issuing thread, every wait bounded.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {
namespace {

constexpr int kT = 128;                 // query tile rows
constexpr int kKT = 128;                // key tile
constexpr int kChunk = 128 * 128;       // 128 rows x 64 bf16 (one 128-byte column chunk)
constexpr int kRowStat = 2 * kT * 4;    // per query tile: -lse * log2(e) [128], -D [128]
constexpr int kEntryMask = (1 << 24) - 1;   // list entries: tile index | pair mask << 24

// A 128-row tile of Q, dO, K or V: D / 64 swizzled column chunks of 16 KB.
template <int D>
struct Tiles {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;
};
constexpr int kThreads = 384;           // warp 0 TMA, warp 1 MMA, warps 4..7 / 8..11 elementwise halves
constexpr float kLog2e = 1.4426950408889634f;

// The selector's lists (any block geometry) are re-expressed on 128 x 128
// (query tile, key tile) pairs.  A pair's mask has bit 2 i + j set when rows
// 64 i .. 64 i + 63 of the query tile belong to a query block that listed the
// key block holding keys 64 j .. 64 j + 63 of the key tile; with 256- or
// 128-row query blocks and 128-key blocks all four bits are equal.
struct BwdParams {
  CUtensorMap tq[kMaxFwdBatch];
  CUtensorMap tk[kMaxFwdBatch];
  CUtensorMap tv[kMaxFwdBatch];
  CUtensorMap tdo[kMaxFwdBatch];
  int seq_lens[kMaxFwdBatch];
  int b0, Bn, Hq, Hkv, G, Sq, Skv, nQt, nKt, prefix_len, n_items;
  const int32_t* dq_list;     // [B, Hq, nQt, nKt]: key tiles kt | mask << 24, ascending
  const int32_t* dq_cnt;      // [B, Hq, nQt]
  const float* rowstat;       // [B, Hq, nQt, 2, 128]: -lse * log2(e) (-inf on padded rows), -D
  int* counter;               // next dK/dV item (zeroed before the launch)
  const int32_t* inv_cnt;     // [B, Hkv, nKt]
  const int32_t* inv_list;    // [B, Hkv, nKt, G * nQt]: rows (g * nQt + qt) | mask << 24, ascending
  float scale, scale_log2;
  __nv_bfloat16* dq;          // [B, Sq, Hq, d]
  __nv_bfloat16* dk;          // [B, Skv, Hkv, d]
  __nv_bfloat16* dv;
};

template <int N>
struct RingN {
  uint32_t stage = 0, phase = 0;
  __device__ __forceinline__ void next() {
    if (++stage == N) { stage = 0; phase ^= 1u; }
  }
};
using Ring2 = RingN<2>;
constexpr int kKStages = 3;             // dQ kernel: K tiles are held until dQ += dS K
constexpr int kVStages = 2;             // V tiles only until dP = dO V^T

// Two-slot ring through which the producer hands the item ids it takes from
// the global counter to the other roles (-1 ends the loop).
struct ItemRing {
  Ring2 r;
  __device__ __forceinline__ int take(uint64_t* full, uint64_t* empty, volatile int* ids, volatile int* abort,
                                      bool& ok) {
    ok = mbar_wait(smem_u32(full + r.stage), r.phase, abort);
    const int t = ok ? ids[r.stage] : -1;
    if (ok) mbar_arrive(smem_u32(empty + r.stage));
    r.next();
    return t;
  }
};

// Descriptor helpers for the 128 x 128 bf16 tiles (two 128-byte swizzled
// column chunks of 16 KB): K-major use (rows are M or N, channels are K) and
// MN-major use (channels are N, rows are K, 16 rows per K step).
__device__ __forceinline__ uint64_t kmaj(uint32_t tile, int kk) {
  return sdesc_sw128(tile + (kk / 4) * kChunk + (kk % 4) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmaj(uint32_t tile, int kk) {
  return sdesc_sw128(tile + kk * 16 * 128, kChunk, 1024);
}

// 128 bf16 of a row written as zeros.
__device__ __forceinline__ void zero_row(__nv_bfloat16* row, int c0, int n) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int i = c0 / 8; i < (c0 + n) / 8; ++i) reinterpret_cast<uint4*>(row)[i] = z;
}

// 32 fp32 accumulator columns -> 32 bf16 at dst (times mul), or zeros.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float* o, float mul, bool keep) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = keep ? pack_bf16x2(o[2 * i] * mul, o[2 * i + 1] * mul) : 0u;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

// ---------------------------------------------------------------- dQ ---
// TMEM: S of key block j in buffer j % 2 at [0, 128) or [128, 256); dP in
// [256, 384), overwritten in place by dS (bf16, 32 columns per 64 keys);
// dQ accumulates in [384, 512).  The two elementwise warpgroups split the
// 128 keys of a block (group g: keys 64 g .. 64 g + 63) and keep P in
// registers between the exponentials and dS.  Issue order: S(j+1), dQ(j),
// dP(j+1), S(j+2), ...: block j+1's exponentials overlap dQ(j), dP(j+1)
// and S(j+2).  Entries whose mask excludes a (row half, key half) give P = 0
// there.  kFull: every mask is full (256/128-row query blocks, 128-key
// blocks), so the mask tests compile away.
template <int D, bool kFull>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using T = Tiles<D>;
  constexpr int kTile = T::kTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_s = smem;                    // Q tile
  uint8_t* do_s = smem + kTile;           // dO tile
  uint8_t* k_s = smem + 2 * kTile;        // kKStages K tiles
  uint8_t* v_s = k_s + kKStages * kTile;  // kVStages V tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(v_s + kVStages * kTile);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* s_full = bars + 2;            // [2] per S buffer
  uint64_t* dp_full = bars + 4;
  uint64_t* ds_full = bars + 5;
  uint64_t* dq_full = bars + 8;
  uint64_t* acc_empty = bars + 9;
  uint64_t* mma_done = bars + 10;
  uint64_t* k_full = bars + 11;           // [kKStages]
  uint64_t* k_empty = k_full + kKStages;  // [kKStages]
  uint64_t* v_full = k_empty + kKStages;  // [kVStages]
  uint64_t* v_empty = v_full + kVStages;  // [kVStages]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(v_empty + kVStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_empty), 1);
    mbar_init(smem_u32(dp_full), 1);
    mbar_init(smem_u32(ds_full), 256);
    mbar_init(smem_u32(dq_full), 1);
    mbar_init(smem_u32(acc_empty), 256);
    mbar_init(smem_u32(mma_done), 1);
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(s_full + i), 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(smem_u32(k_full + i), 1);
      mbar_init(smem_u32(k_empty + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(smem_u32(v_full + i), 1);
      mbar_init(smem_u32(v_empty + i), 1);
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
  const uint32_t tmem = *tmem_slot;

  // item -> (request, KV head, query tile, query head of the group) and its key-tile list
  auto decode = [&](int t, int& bl, int& h, int& qt, int& n, int& L, const int32_t*& lst) {
    const int g = t % p.G;
    int r = t / p.G;
    qt = r % p.nQt;
    r /= p.nQt;
    const int hk = r % p.Hkv;
    bl = r / p.Hkv;
    h = hk * p.G + g;
    L = p.seq_lens[bl];
    const int64_t row = ((int64_t)(p.b0 + bl) * p.Hq + h) * p.nQt + qt;
    lst = p.dq_list + row * p.nKt;
    n = qt * kT < L ? min(max(p.dq_cnt[row], 0), p.nKt) : 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA ---
    if (lane == 0) {
      RingN<kKStages> kr;
      RingN<kVStages> vr;
      uint32_t qi = 0;
      int q_armed = -1, k_armed[kKStages], v_armed[kVStages];     // parity of each barrier's last arming
      for (int i = 0; i < kKStages; ++i) k_armed[i] = -1;
      for (int i = 0; i < kVStages; ++i) v_armed[i] = -1;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
        int bl, h, qt, n, L;
        const int32_t* lst;
        decode(t, bl, h, qt, n, L, lst);
        if (n == 0) continue;
        ok = mbar_wait(smem_u32(q_empty), (qi & 1u) ^ 1u, abort_flag);
        if (!ok) break;
        q_armed = (int)(qi & 1u);
        ++qi;
        mbar_arrive_expect_tx(smem_u32(q_full), 2 * kTile);
        for (int c = 0; c < T::kChunks; ++c) {
          tma_load_3d(smem_u32(q_s) + c * kChunk, &p.tq[bl], smem_u32(q_full), c * 64, qt * kT, h);
          tma_load_3d(smem_u32(do_s) + c * kChunk, &p.tdo[bl], smem_u32(q_full), c * 64, qt * kT, h);
        }
        const int hk = h / p.G;
        for (int j = 0; j < n && ok; ++j) {
          int kb = __ldg(lst + j) & kEntryMask;       // key tile
          if (kb >= p.nKt) kb = p.nKt;
          ok = mbar_wait(smem_u32(k_empty + kr.stage), kr.phase ^ 1u, abort_flag);
          if (!ok) break;
          uint32_t fb = smem_u32(k_full + kr.stage);
          uint32_t base = smem_u32(k_s) + kr.stage * kTile;
          mbar_arrive_expect_tx(fb, kTile);
          k_armed[kr.stage] = (int)kr.phase;
          for (int c = 0; c < T::kChunks; ++c) tma_load_3d(base + c * kChunk, &p.tk[bl], fb, c * 64, kb * kKT, hk);
          kr.next();
          ok = mbar_wait(smem_u32(v_empty + vr.stage), vr.phase ^ 1u, abort_flag);
          if (!ok) break;
          fb = smem_u32(v_full + vr.stage);
          base = smem_u32(v_s) + vr.stage * kTile;
          mbar_arrive_expect_tx(fb, kTile);
          v_armed[vr.stage] = (int)vr.phase;
          for (int c = 0; c < T::kChunks; ++c) tma_load_3d(base + c * kChunk, &p.tv[bl], fb, c * 64, kb * kKT, hk);
          vr.next();
        }
      }
      // let this thread's copies land before the CTA can exit
      if (q_armed >= 0) mbar_drain(smem_u32(q_full), (uint32_t)q_armed);
      for (int i = 0; i < kKStages; ++i)
        if (k_armed[i] >= 0) mbar_drain(smem_u32(k_full + i), (uint32_t)k_armed[i]);
      for (int i = 0; i < kVStages; ++i)
        if (v_armed[i] >= 0) mbar_drain(smem_u32(v_full + i), (uint32_t)v_armed[i]);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA ---
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_mn = idesc_bf16_f32(128, D, true);
      RingN<kKStages> kr;
      RingN<kVStages> vr;
      uint32_t qi = 0, ai = 0, dsc = 0, jj = 0;
      bool ok = true;
      const uint32_t qa = smem_u32(q_s), da = smem_u32(do_s), ka = smem_u32(k_s), va = smem_u32(v_s);
      // S = Q K^T into S buffer `buf`; waits for the block's K tile, returns its stage
      auto issue_s = [&](uint32_t buf, uint32_t& kst) {
        kst = kr.stage;
        if (!mbar_wait(smem_u32(k_full + kst), kr.phase, abort_flag)) return false;
        kr.next();
        tc_fence_after();
        const uint32_t kt = ka + kst * kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + buf * 128, kmaj(qa, kk), kmaj(kt, kk), idesc_s, kk > 0);
        mma_commit(smem_u32(s_full + buf));
        return true;
      };
      // dP = dO V^T into [256, 384); waits for the block's V tile and frees it
      auto issue_dp = [&]() {
        const uint32_t vst = vr.stage;
        if (!mbar_wait(smem_u32(v_full + vst), vr.phase, abort_flag)) return false;
        vr.next();
        tc_fence_after();
        const uint32_t vt = va + vst * kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + 256, kmaj(da, kk), kmaj(vt, kk), idesc_s, kk > 0);
        mma_commit(smem_u32(dp_full));
        mma_commit(smem_u32(v_empty + vst));
        return true;
      };
      // dQ += dS K (dS bf16 of keys 64 g + .. at dP column 64 g; K as the MN-major B)
      auto issue_dq = [&](uint32_t kt, bool first) {
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk)
          mma_ts(tmem + 384, tmem + 256 + (kk / 4) * 64 + (kk % 4) * 8, mnmaj(kt, kk), idesc_mn,
                 (first && kk == 0) ? 0u : 1u);
      };
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
        int bl, h, qt, n, L;
        const int32_t* lst;
        decode(t, bl, h, qt, n, L, lst);
        if (n == 0) continue;
        ok = mbar_wait(smem_u32(acc_empty), (ai & 1u) ^ 1u, abort_flag);    // last epilogue read dQ
        ++ai;
        if (ok) ok = mbar_wait(smem_u32(q_full), qi & 1u, abort_flag);
        ++qi;
        if (!ok) break;
        // block 0's S and dP
        uint32_t kst = 0;
        if (!(ok = issue_s(jj & 1u, kst))) break;
        if (!(ok = issue_dp())) break;
        if (n == 1) mma_commit(smem_u32(q_empty));
        for (int j = 0; j < n && ok; ++j, ++jj) {
          // S(j+1) goes to the other buffer, whose S(j-1) the elementwise
          // groups finished with before dS(j-1) (waited for below, last block)
          uint32_t nkst = 0;
          if (j + 1 < n && !(ok = issue_s((jj + 1) & 1u, nkst))) break;
          ok = mbar_wait(smem_u32(ds_full), dsc & 1u, abort_flag);
          ++dsc;
          if (!ok) break;
          tc_fence_after();
          issue_dq(ka + kst * kTile, j == 0);
          mma_commit(smem_u32(k_empty + kst));
          if (j + 1 < n) {
            if (!(ok = issue_dp())) break;
            if (j + 2 == n) mma_commit(smem_u32(q_empty));
          }
          kst = nkst;
        }
        if (!ok) break;
        mma_commit(smem_u32(dq_full));
      }
      mma_commit(smem_u32(mma_done));        // every MMA issued above has finished
      mbar_drain(smem_u32(mma_done), 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ----------------------------------------------------- elementwise ---
    const int grp = (warp - 4) / 4;         // keys 64 grp .. 64 grp + 63 of each block
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    uint32_t oi = 0, jj = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x) {
      int bl, h, qt, n, L;
      const int32_t* lst;
      decode(t, bl, h, qt, n, L, lst);
      const int b = p.b0 + bl;
      const int row = qt * kT + r;
      const bool row_exists = row < p.Sq;
      const bool row_ok = row < L;
      __nv_bfloat16* drow = p.dq + (((int64_t)b * p.Sq + row) * p.Hq + h) * D;
      if (n == 0) {
        if (row_exists) zero_row(drow, grp * (D / 2), D / 2);
        continue;
      }
      const float* rs = p.rowstat + (((int64_t)b * p.Hq + h) * p.nQt + qt) * (2 * kT);
      const float nl = __ldg(rs + r);         // -lse log2(e); -inf on padded rows: P = 0
      const float nD = __ldg(rs + kT + r);
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nl2 = make_float2(nl, nl);
      const float2 nD2 = make_float2(nD, nD);
      const int valid_kv = p.prefix_len + L;
      const int qhalf = wq >> 1;              // rows 64 qhalf .. of the tile (warp-uniform)
      for (int j = 0; j < n; ++j, ++jj) {
        const uint32_t buf = jj & 1u;
        const int e = __ldg(lst + j);
        int kb = e & kEntryMask;
        if (kb >= p.nKt) kb = p.nKt;
        // this (row half, key half) pair selected?  keys of this group's half
        // below the end of the sequence (a tile holding the end only)
        const bool pair_ok = kFull || ((e >> (24 + qhalf * 2 + grp)) & 1);
        const int kvalid = valid_kv - kb * kKT - grp * 64;
        const bool all_valid = pair_ok && kvalid >= 64;
        ok = mbar_wait(smem_u32(s_full + buf), (jj >> 1) & 1u, abort_flag);
        if (!ok) break;
        tc_fence_after();
        if constexpr (!kFull) {
          if (!pair_ok) {
            // a pair no query block of these rows listed: P = 0, so dS = 0; it
            // is stored once this block's dP has landed (the MMA writes those
            // columns)
            ok = mbar_wait(smem_u32(dp_full), jj & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            uint32_t zk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zk[i] = 0u;
            tmem_st16(tl + 256 + grp * 64, zk);
            tmem_st16(tl + 256 + grp * 64 + 16, zk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(ds_full));
            continue;
          }
        }
        // P = 2^(S scale log2(e) - lse log2(e)), kept in registers
        float pr[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float s[32];
          tmem_ld32f(tl + buf * 128 + grp * 64 + c * 32, s);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), sc2, nl2);
            pr[c * 32 + 2 * i] = ex2_approx(x.x);
            pr[c * 32 + 2 * i + 1] = ex2_approx(x.y);
          }
        }
        if (!all_valid) {
#pragma unroll
          for (int i = 0; i < 64; ++i) pr[i] = (pair_ok && i < kvalid) ? pr[i] : 0.f;
        }
        // dS = P (dP - D), written over this group's dP columns
        ok = mbar_wait(smem_u32(dp_full), jj & 1u, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tb = tl + 256 + grp * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float dp[32];
          tmem_ld32f(tb + c * 32, dp);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 ds = __fmul2_rn(make_float2(pr[c * 32 + 2 * i], pr[c * 32 + 2 * i + 1]),
                                         __fadd2_rn(make_float2(dp[2 * i], dp[2 * i + 1]), nD2));
            pk[i] = pack_bf16x2(ds.x, ds.y);
          }
          tmem_st16(tb + c * 16, pk);
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
      for (int c = 0; c < D / 64; ++c) {         // group g writes columns g D / 2 ..
        float o[32];
        tmem_ld32f(tl + 384 + grp * (D / 2) + c * 32, o);
        tmem_wait_ld();
        if (row_exists) store_row32(drow + grp * (D / 2) + c * 32, o, p.scale, row_ok);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(acc_empty));
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
// TMEM: S^T in [0, 128) (P^T bf16 over it: query columns 64 g .. at column
// 64 g, 32 wide), dP^T in [128, 256) (dS^T bf16 the same way), dV in
// [256, 256 + D), dK in [256 + D, 256 + 2 D).  The two elementwise warpgroups split the
// 128 query rows of a step (group g: rows 64 g .. 64 g + 63) and keep P^T
// in registers between P^T and dS^T.  Issue order: S^T(s), dP^T(s), dV(s),
// S^T(s+1), dK(s), dP^T(s+1), ...
template <int D, bool kFull>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using T = Tiles<D>;
  constexpr int kTile = T::kTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kStage = 2 * kTile + kRowStat;   // Q tile, dO tile, lse/D of its rows
  uint8_t* k_s = smem;                    // K tile of the key block
  uint8_t* v_s = smem + kTile;            // V tile
  uint8_t* qdo_s = smem + 2 * kTile;      // 2 stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(qdo_s + 2 * kStage);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* dp_full = bars + 3;
  uint64_t* p_full = bars + 4;
  uint64_t* ds_full = bars + 5;
  uint64_t* acc_full = bars + 6;
  uint64_t* acc_empty = bars + 7;
  uint64_t* qdo_full = bars + 8;          // [2]
  uint64_t* qdo_empty = bars + 10;        // [2]
  uint64_t* mma_done = bars + 12;
  uint64_t* item_full = bars + 13;        // [2] item-id ring
  uint64_t* item_empty = bars + 15;       // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_ids = reinterpret_cast<volatile int*>(tmem_slot + 2);   // [2]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(kv_full), 1);
    mbar_init(smem_u32(kv_empty), 1);
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(dp_full), 1);
    mbar_init(smem_u32(p_full), 256);
    mbar_init(smem_u32(ds_full), 256);
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(acc_empty), 256);
    mbar_init(smem_u32(mma_done), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(qdo_full + i), 1);
      mbar_init(smem_u32(qdo_empty + i), 1);
      mbar_init(smem_u32(item_full + i), 1);
      mbar_init(smem_u32(item_empty + i), 1 + 256);    // MMA thread + elementwise threads
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
  const uint32_t tmem = *tmem_slot;

  // item -> (request, KV head, key tile); one step per query tile that listed it
  auto decode = [&](int t, int& bl, int& hk, int& kb, int& steps, const int32_t*& lst) {
    kb = t % p.nKt;
    const int r = t / p.nKt;
    hk = r % p.Hkv;
    bl = r / p.Hkv;
    const int64_t key = ((int64_t)(p.b0 + bl) * p.Hkv + hk) * p.nKt + kb;
    steps = min(max(p.inv_cnt[key], 0), p.G * p.nQt);
    lst = p.inv_list + key * p.G * p.nQt;
  };
  // step s of an item -> (query head, query tile)
  auto step_tile = [&](const int32_t* lst, int hk, int s, int& h, int& qt) {
    const int row = __ldg(lst + s) & kEntryMask;
    const int g = row / p.nQt;
    qt = row - g * p.nQt;
    h = hk * p.G + g;
  };

  if (warp == 0) {
    if (lane == 0) {
      Ring2 ring, items;
      uint32_t ki = 0;
      int kv_armed = -1, qdo_armed[2] = {-1, -1};   // parity of each barrier's last arming
      bool ok = true;
      while (ok) {
        // dynamic scheduling: the next item from the counter, published to the other roles
        int t = atomicAdd(p.counter, 1);
        if (t >= p.n_items) t = -1;
        ok = mbar_wait(smem_u32(item_empty + items.stage), items.phase ^ 1u, abort_flag);
        if (!ok) break;
        item_ids[items.stage] = t;
        mbar_arrive(smem_u32(item_full + items.stage));
        items.next();
        if (t < 0) break;
        int bl, hk, kb, steps;
        const int32_t* lst;
        decode(t, bl, hk, kb, steps, lst);
        if (steps == 0) continue;
        ok = mbar_wait(smem_u32(kv_empty), (ki & 1u) ^ 1u, abort_flag);
        if (!ok) break;
        kv_armed = (int)(ki & 1u);
        ++ki;
        mbar_arrive_expect_tx(smem_u32(kv_full), 2 * kTile);
        for (int c = 0; c < T::kChunks; ++c) {
          tma_load_3d(smem_u32(k_s) + c * kChunk, &p.tk[bl], smem_u32(kv_full), c * 64, kb * kKT, hk);
          tma_load_3d(smem_u32(v_s) + c * kChunk, &p.tv[bl], smem_u32(kv_full), c * 64, kb * kKT, hk);
        }
        for (int s = 0; s < steps && ok; ++s) {
          int h, qt;
          step_tile(lst, hk, s, h, qt);
          ok = mbar_wait(smem_u32(qdo_empty + ring.stage), ring.phase ^ 1u, abort_flag);
          if (!ok) break;
          const uint32_t fb = smem_u32(qdo_full + ring.stage);
          const uint32_t base = smem_u32(qdo_s) + ring.stage * kStage;
          mbar_arrive_expect_tx(fb, 2 * kTile + kRowStat);
          qdo_armed[ring.stage] = (int)ring.phase;
          for (int c = 0; c < T::kChunks; ++c) {
            tma_load_3d(base + c * kChunk, &p.tq[bl], fb, c * 64, qt * kT, h);
            tma_load_3d(base + kTile + c * kChunk, &p.tdo[bl], fb, c * 64, qt * kT, h);
          }
          bulk_load(base + 2 * kTile,
                    p.rowstat + (((int64_t)(p.b0 + bl) * p.Hq + h) * p.nQt + qt) * (2 * kT), kRowStat, fb);
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
      constexpr uint32_t idesc_mn = idesc_bf16_f32(128, D, true);
      Ring2 ring;
      uint32_t ki = 0, ai = 0, pc = 0, dc = 0;
      bool ok = true;
      const uint32_t ka = smem_u32(k_s), va = smem_u32(v_s), qda = smem_u32(qdo_s);
      auto issue_st = [&](uint32_t qs) {        // S^T = K Q^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem, kmaj(ka, kk), kmaj(qs, kk), idesc_s, kk > 0);
        mma_commit(smem_u32(s_full));
      };
      auto issue_dpt = [&](uint32_t qs) {       // dP^T = V dO^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + 128, kmaj(va, kk), kmaj(qs + kTile, kk), idesc_s, kk > 0);
        mma_commit(smem_u32(dp_full));
      };
      // dV += P^T dO, dK += dS^T Q  (A from TMEM, the row tiles as the MN-major B)
      auto issue_dv = [&](uint32_t qs, bool first) {
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + 256, tmem + (kk / 4) * 64 + (kk % 4) * 8, mnmaj(qs + kTile, kk), idesc_mn,
                 (first && kk == 0) ? 0u : 1u);
      };
      auto issue_dk = [&](uint32_t qs, bool first) {
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + 256 + D, tmem + 128 + (kk / 4) * 64 + (kk % 4) * 8, mnmaj(qs, kk), idesc_mn,
                 (first && kk == 0) ? 0u : 1u);
      };
      auto wait_stage = [&](uint32_t& qs, uint32_t& st) {
        st = ring.stage;
        const bool r = mbar_wait(smem_u32(qdo_full + st), ring.phase, abort_flag);
        ring.next();
        if (r) tc_fence_after();
        qs = qda + st * kStage;
        return r;
      };
      ItemRing items;
      while (ok) {
        const int t = items.take(item_full, item_empty, item_ids, abort_flag, ok);
        if (t < 0) break;
        int bl, hk, kb, steps;
        const int32_t* lst;
        decode(t, bl, hk, kb, steps, lst);
        if (steps == 0) continue;
        ok = mbar_wait(smem_u32(acc_empty), (ai & 1u) ^ 1u, abort_flag);    // last epilogue read dV/dK
        ++ai;
        if (ok) ok = mbar_wait(smem_u32(kv_full), ki & 1u, abort_flag);
        ++ki;
        if (!ok) break;
        uint32_t qs, st;
        if (!(ok = wait_stage(qs, st))) break;
        issue_st(qs);
        issue_dpt(qs);
        for (int s = 0; s < steps && ok; ++s) {
          ok = mbar_wait(smem_u32(p_full), pc & 1u, abort_flag);
          ++pc;
          if (!ok) break;
          tc_fence_after();
          issue_dv(qs, s == 0);
          uint32_t nqs = 0, nst = 0;
          if (s + 1 < steps) {
            if (!(ok = wait_stage(nqs, nst))) break;
            issue_st(nqs);
          }
          ok = mbar_wait(smem_u32(ds_full), dc & 1u, abort_flag);
          ++dc;
          if (!ok) break;
          tc_fence_after();
          issue_dk(qs, s == 0);
          mma_commit(smem_u32(qdo_empty + st));
          if (s + 1 < steps) issue_dpt(nqs);
          qs = nqs;
          st = nst;
        }
        if (!ok) break;
        mma_commit(smem_u32(kv_empty));
        mma_commit(smem_u32(acc_full));
      }
      mma_commit(smem_u32(mma_done));        // every MMA issued above has finished
      mbar_drain(smem_u32(mma_done), 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int grp = (warp - 4) / 4;         // query rows 64 grp .. 64 grp + 63 of each step
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    Ring2 ring;
    ItemRing items;
    uint32_t sc = 0, dc = 0, ai = 0;
    bool ok = true;
    while (ok) {
      const int t = items.take(item_full, item_empty, item_ids, abort_flag, ok);
      if (t < 0) break;
      int bl, hk, kb, steps;
      const int32_t* lst;
      decode(t, bl, hk, kb, steps, lst);
      const int b = p.b0 + bl;
      const int L = p.seq_lens[bl];
      const int key = kb * kKT + r;
      const bool key_exists = key < p.Skv;
      const bool key_ok = key < p.prefix_len + L;
      // keys past the end (zero-filled K/V rows) get P = 0; only the block
      // holding the end has any, so the warp-uniform test skips the multiply
      const bool warp_keys_ok = __all_sync(0xffffffffu, key_ok);
      const float2 km2 = make_float2(key_ok ? 1.f : 0.f, key_ok ? 1.f : 0.f);
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      // group 0 writes dV, group 1 dK
      __nv_bfloat16* grow = (grp == 0 ? p.dv : p.dk) + (((int64_t)b * p.Skv + key) * p.Hkv + hk) * D;
      if (steps == 0) {
        if (key_exists) zero_row(grow, 0, D);
        continue;
      }
      for (int s = 0; s < steps; ++s) {
        const uint32_t st = ring.stage;
        // the stage's lse/D must be visible to this thread: wait for its copy too
        ok = mbar_wait(smem_u32(qdo_full + st), ring.phase, abort_flag);
        ring.next();
        if (ok) ok = mbar_wait(smem_u32(s_full), sc & 1u, abort_flag);
        ++sc;
        if (!ok) break;
        tc_fence_after();
        // per query-row column: -lse log2(e) (-inf on padded rows) and -D
        const float* rs = reinterpret_cast<const float*>(qdo_s + st * kStage + 2 * kTile) + grp * 64;
        // this group's query-row half and this warp's key half selected as a pair?
        const bool pair_ok = kFull || ((__ldg(lst + s) >> (24 + grp * 2 + (wq >> 1))) & 1);
        if constexpr (!kFull) {
          if (!pair_ok) {
            // a pair this query block did not list: P^T = 0 and dS^T = 0 for
            // these keys and rows, stored without exponentials once the MMAs
            // have written the columns (S^T now, dP^T after its barrier)
            uint32_t zk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zk[i] = 0u;
            tmem_st16(tl + grp * 64, zk);
            tmem_st16(tl + grp * 64 + 16, zk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(p_full));
            ok = mbar_wait(smem_u32(dp_full), dc & 1u, abort_flag);
            ++dc;
            if (!ok) break;
            tc_fence_after();
            tmem_st16(tl + 128 + grp * 64, zk);
            tmem_st16(tl + 128 + grp * 64 + 16, zk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(ds_full));
            continue;
          }
        }
        const bool need_mask = !(warp_keys_ok && pair_ok);      // warp-uniform
        const float2 km = pair_ok ? km2 : make_float2(0.f, 0.f);
        // P^T = 2^(S^T scale log2(e) - lse log2(e)), kept in registers; bf16 over S^T
        float pr[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float sv[32];
          tmem_ld32f(tl + grp * 64 + c * 32, sv);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 l4 = *reinterpret_cast<const float4*>(rs + c * 32 + 4 * i);
            const float2 t0 = __ffma2_rn(make_float2(sv[4 * i], sv[4 * i + 1]), sc2, make_float2(l4.x, l4.y));
            const float2 t1 = __ffma2_rn(make_float2(sv[4 * i + 2], sv[4 * i + 3]), sc2, make_float2(l4.z, l4.w));
            float2 p0 = make_float2(ex2_approx(t0.x), ex2_approx(t0.y));
            float2 p1 = make_float2(ex2_approx(t1.x), ex2_approx(t1.y));
            if (need_mask) {
              p0 = __fmul2_rn(p0, km);
              p1 = __fmul2_rn(p1, km);
            }
            pr[c * 32 + 4 * i] = p0.x;
            pr[c * 32 + 4 * i + 1] = p0.y;
            pr[c * 32 + 4 * i + 2] = p1.x;
            pr[c * 32 + 4 * i + 3] = p1.y;
            pk[2 * i] = pack_bf16x2(p0.x, p0.y);
            pk[2 * i + 1] = pack_bf16x2(p1.x, p1.y);
          }
          tmem_st16(tl + grp * 64 + c * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(p_full));
        // dS^T = P^T (dP^T - D), bf16 over this group's dP^T columns
        ok = mbar_wait(smem_u32(dp_full), dc & 1u, abort_flag);
        ++dc;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float dp[32];
          tmem_ld32f(tl + 128 + grp * 64 + c * 32, dp);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 d4 = *reinterpret_cast<const float4*>(rs + kT + c * 32 + 4 * i);
            const float2 d0 = __fmul2_rn(make_float2(pr[c * 32 + 4 * i], pr[c * 32 + 4 * i + 1]),
                                         __fadd2_rn(make_float2(dp[4 * i], dp[4 * i + 1]), make_float2(d4.x, d4.y)));
            const float2 d1 = __fmul2_rn(make_float2(pr[c * 32 + 4 * i + 2], pr[c * 32 + 4 * i + 3]),
                                         __fadd2_rn(make_float2(dp[4 * i + 2], dp[4 * i + 3]), make_float2(d4.z, d4.w)));
            pk[2 * i] = pack_bf16x2(d0.x, d0.y);
            pk[2 * i + 1] = pack_bf16x2(d1.x, d1.y);
          }
          tmem_st16(tl + 128 + grp * 64 + c * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(ds_full));
      }
      if (!ok) break;
      ok = mbar_wait(smem_u32(acc_full), ai & 1u, abort_flag);
      ++ai;
      if (!ok) break;
      tc_fence_after();
      const float mul = grp == 0 ? 1.f : p.scale;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32f(tl + 256 + grp * D + c * 32, o);
        tmem_wait_ld();
        if (key_exists) store_row32(grow + c * 32, o, mul, key_ok);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(acc_empty));
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
// Per query tile (b, h, qt), 128 values of -lse * log2(e) (-inf on padded
// rows, so their P is 0) and 128 of -D, D = sum_c dO_c O_c (0 on padded
// rows), stored together so one bulk copy stages them.  One warp per
// (b, row, h) over every row of the tiles; each lane reads D / 32 elements.
struct PrepParams {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  int64_t o_sb, o_ss, o_sh, d_sb, d_ss, d_sh;
  int B, Sq, Hq, nQt;
  int seq_lens[kMaxSelectBatch];
  float* rowstat;
};

template <int D>
__global__ void bwd_prep_kernel(const __grid_constant__ PrepParams p) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int rows = p.nQt * kT;
  const int64_t total = (int64_t)p.B * rows * p.Hq;
  if (w >= total) return;
  const int h = (int)(w % p.Hq);
  const int64_t rr = w / p.Hq;
  const int row = (int)(rr % rows);
  const int b = (int)(rr / rows);
  const bool real = row < p.seq_lens[b];
  float acc = 0.f;
  if (real) {
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(
        p.o + b * p.o_sb + (int64_t)row * p.o_ss + (int64_t)h * p.o_sh + lane * (D / 32));
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(
        p.dout + b * p.d_sb + (int64_t)row * p.d_ss + (int64_t)h * p.d_sh + lane * (D / 32));
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
      const float2 x = __bfloat1622float2(o2[i]), y = __bfloat1622float2(d2[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    float* rs = p.rowstat + (((int64_t)b * p.Hq + h) * p.nQt + row / kT) * (2 * kT) + row % kT;
    rs[0] = real ? -p.lse[((int64_t)b * p.Hq + h) * p.Sq + row] * kLog2e : -INFINITY;
    rs[kT] = -acc;
  }
}

// ------------------------------------------------------- tile lists ---
// Four bitmap planes, one per mask bit 2 i + j: row (b, hk, g, qt), bit kt.
// One warp per selector list (b, h, qb) sets, for every listed key block,
// the bits of the (query tile, row half) x (key tile, key half) pairs the
// two blocks cover.  OR is order-free, so the result is deterministic.
struct BitmapParams {
  const int32_t* indices;
  const int32_t* counts;
  uint32_t* planes;           // 4 x [B, Hkv, G, nQt, words]
  int64_t plane_words;
  int B, Hq, Hkv, G, nQb, nKb, nQt, nKt, block_q, block_k, words;
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
  const int L = p.seq_lens[b];
  if (qb * p.block_q >= L) return;
  const int hk = h / p.G, g = h - hk * p.G;
  // query tiles and row halves of this query block (tiles past the last real row skipped)
  int qt0, nqt, ibits;
  if (p.block_q == 64) {
    qt0 = qb >> 1; nqt = 1; ibits = 1 << (qb & 1);
  } else {
    qt0 = qb * p.block_q / kT; nqt = p.block_q / kT; ibits = 3;
  }
  const int c = min(max(p.counts[w], 0), p.nKb);
  const int32_t* lst = p.indices + w * p.nKb;
  const int64_t row0 = (((int64_t)b * p.Hkv + hk) * p.G + g) * p.nQt;
  for (int i = lane; i < c; i += 32) {
    const int kb = lst[i];
    if (kb < 0 || kb >= p.nKb) continue;
    const int kt = p.block_k == 64 ? kb >> 1 : kb;
    const int jbits = p.block_k == 64 ? 1 << (kb & 1) : 3;
    for (int q = 0; q < nqt; ++q) {
      const int qt = qt0 + q;
      if (qt * kT >= L) break;
      for (int ii = 0; ii < 2; ++ii) {
        if (!((ibits >> ii) & 1)) continue;
        for (int jj = 0; jj < 2; ++jj) {
          if (!((jbits >> jj) & 1)) continue;
          uint32_t* pl = p.planes + (ii * 2 + jj) * p.plane_words;
          atomicOr(pl + (row0 + qt) * p.words + (kt >> 5), 1u << (kt & 31));
        }
      }
    }
  }
}

// One warp per (b, h, qt): the ascending key tiles of its four plane rows,
// each with its mask (the dQ kernel's lists).
struct TileListParams {
  const uint32_t* planes;
  int64_t plane_words;
  int32_t* dq_list;
  int32_t* dq_cnt;
  int n_rows, nKt, words;
};

__global__ void bwd_tilelist_kernel(const __grid_constant__ TileListParams p) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;   // (b, hk, g, qt) = (b, h, qt)
  const int lane = threadIdx.x % 32;
  if (row >= p.n_rows) return;
  int32_t* out = p.dq_list + row * p.nKt;
  int running = 0;
  for (int w0 = 0; w0 < p.words; w0 += 32) {
    const int w = w0 + lane;
    uint32_t m[4] = {0u, 0u, 0u, 0u};
    if (w < p.words)
      for (int i = 0; i < 4; ++i) m[i] = p.planes[i * p.plane_words + row * p.words + w];
    uint32_t u = m[0] | m[1] | m[2] | m[3];
    const int cnt = __popc(u);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int pos = running + incl - cnt;
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      int mask = 0;
      for (int i = 0; i < 4; ++i) mask |= (int)((m[i] >> bit) & 1u) << i;
      out[pos++] = (w * 32 + bit) | (mask << 24);
    }
    running += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) p.dq_cnt[row] = running;
}

// One warp per (b, hk, 32 key tiles): reads the plane rows 32 at a time (one
// row per lane), transposes each 32 x 32 bit square with ballots so that lane
// i holds the rows that selected key tile 32 w + i, and appends them in
// ascending row order with their masks (the dK/dV kernel's lists).
struct InvParams {
  const uint32_t* planes;
  int64_t plane_words;
  int32_t* inv_cnt;
  int32_t* inv_list;
  int n_groups, nrows, nKt, words;
};

__global__ void bwd_inverse_kernel(const __grid_constant__ InvParams p) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (wid >= (int64_t)p.n_groups * p.words) return;
  const int w = (int)(wid % p.words);
  const int64_t gi = wid / p.words;
  const int64_t base = gi * p.nrows * p.words;
  const int kt = w * 32 + lane;
  int32_t* out = p.inv_list + (gi * p.nKt + min(kt, p.nKt - 1)) * p.nrows;
  int cnt = 0;
  for (int r0 = 0; r0 < p.nrows; r0 += 32) {
    const int r = r0 + lane;
    uint32_t word[4];
    for (int i = 0; i < 4; ++i)
      word[i] = r < p.nrows ? p.planes[i * p.plane_words + base + (int64_t)r * p.words + w] : 0u;
    uint32_t mine[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int bit = 0; bit < 32; ++bit) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t m = __ballot_sync(0xffffffffu, (word[i] >> bit) & 1u);
        if (lane == bit) mine[i] = m;
      }
    }
    uint32_t u = mine[0] | mine[1] | mine[2] | mine[3];
    while (u) {                          // bits exist only for kt < nKt
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      int mask = 0;
      for (int i = 0; i < 4; ++i) mask |= (int)((mine[i] >> bit) & 1u) << i;
      out[cnt++] = (r0 + bit) | (mask << 24);
    }
  }
  if (kt < p.nKt) p.inv_cnt[gi * p.nKt + kt] = cnt;
}

template <int D>
constexpr int dq_smem() { return (2 + kKStages + kVStages) * Tiles<D>::kTile + 256 + 1024; }
template <int D>
constexpr int dkdv_smem() { return 2 * Tiles<D>::kTile + 2 * (2 * Tiles<D>::kTile + kRowStat) + 256 + 1024; }
static_assert(dq_smem<128>() <= 232448 && dkdv_smem<128>() <= 232448, "shared memory above the per-block limit");

// Workspace layout (each part rounded up to 256 bytes).
struct BwdWorkspace {
  float* rowstat;
  int* counters;              // 256 bytes, zeroed together with the planes that follow
  uint32_t* planes;
  size_t planes_bytes;
  int64_t plane_words;
  int32_t* dq_list;
  int32_t* dq_cnt;
  int32_t* inv_cnt;
  int32_t* inv_list;
  size_t total;
};

// With base == nullptr only the sizes are computed (pointers stay null).
BwdWorkspace carve(void* base, int B, int Hq, int Hkv, int Sq, int Skv) {
  const int64_t nQt = cdiv64(Sq, kT), nKt = cdiv64(Skv, kKT), G = Hq / Hkv, words = cdiv64(nKt, 32);
  auto al = [](int64_t x) { return (size_t)((x + 255) & ~(int64_t)255); };
  char* c = static_cast<char*>(base);
  size_t off = 0;
  auto at = [&](size_t o) -> void* { return c ? static_cast<void*>(c + o) : nullptr; };
  BwdWorkspace w{};
  w.rowstat = static_cast<float*>(at(off));
  off += al((int64_t)B * Hq * nQt * kRowStat);
  w.counters = static_cast<int*>(at(off));
  off += 256;
  w.plane_words = (int64_t)B * Hkv * G * nQt * words;
  w.planes = static_cast<uint32_t*>(at(off));
  w.planes_bytes = al(4 * w.plane_words * 4);
  off += w.planes_bytes;
  w.dq_list = static_cast<int32_t*>(at(off));
  off += al((int64_t)B * Hq * nQt * nKt * 4);
  w.dq_cnt = static_cast<int32_t*>(at(off));
  off += al((int64_t)B * Hq * nQt * 4);
  w.inv_cnt = static_cast<int32_t*>(at(off));
  off += al((int64_t)B * Hkv * nKt * 4);
  w.inv_list = static_cast<int32_t*>(at(off));
  off += al((int64_t)B * Hkv * nKt * G * nQt * 4);
  w.total = off;
  return w;
}

template <int D, bool kFull>
bsa_status launch_tiles(const BackwardArgs& a, const BwdWorkspace& w, cudaStream_t stream) {
  bsa_status st;
  static std::atomic<bool> attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr[dev].load(std::memory_order_acquire)) {
    if ((st = cuda_check(cudaFuncSetAttribute(bwd_dq_kernel<D, kFull>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              dq_smem<D>()),
                         "cudaFuncSetAttribute(bwd_dq_kernel)")) != BSA_OK)
      return st;
    if ((st = cuda_check(cudaFuncSetAttribute(bwd_dkdv_kernel<D, kFull>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              dkdv_smem<D>()),
                         "cudaFuncSetAttribute(bwd_dkdv_kernel)")) != BSA_OK)
      return st;
    attr[dev].store(true, std::memory_order_release);
  }
  const int G = a.Hq / a.Hkv;
  const int nQt = (int)cdiv64(a.Sq, kT), nKt = (int)cdiv64(a.Skv, kKT);
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
      if ((st = encode_tensor_map(&p.tq[i], qb, L, a.Hq, D, a.q_ss, a.q_sh, 128, "Q")) != BSA_OK) return st;
      if ((st = encode_tensor_map(&p.tdo[i], db, L, a.Hq, D, a.d_ss, a.d_sh, 128, "dO")) != BSA_OK) return st;
      if ((st = encode_tensor_map(&p.tk[i], kb, a.prefix_len + L, a.Hkv, D, a.k_ss, a.k_sh, 128, "K")) != BSA_OK) return st;
      if ((st = encode_tensor_map(&p.tv[i], vb, a.prefix_len + L, a.Hkv, D, a.v_ss, a.v_sh, 128, "V")) != BSA_OK) return st;
    }
    p.b0 = b0; p.Bn = Bn; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.Sq = a.Sq; p.Skv = a.Skv;
    p.nQt = nQt; p.nKt = nKt; p.prefix_len = a.prefix_len;
    p.dq_list = w.dq_list; p.dq_cnt = w.dq_cnt; p.rowstat = w.rowstat;
    p.inv_cnt = w.inv_cnt; p.inv_list = w.inv_list;
    p.scale = a.scale; p.scale_log2 = a.scale * kLog2e;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.n_items = Bn * a.Hkv * nQt * G;
    bwd_dq_kernel<D, kFull><<<std::min(p.n_items, sms), kThreads, dq_smem<D>(), stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "bwd_dq_kernel launch")) != BSA_OK) return st;
    p.n_items = Bn * a.Hkv * nKt;
    p.counter = w.counters + b0 / kMaxFwdBatch;
    bwd_dkdv_kernel<D, kFull><<<std::min(p.n_items, sms), kThreads, dkdv_smem<D>(), stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "bwd_dkdv_kernel launch")) != BSA_OK) return st;
  }
  return BSA_OK;
}

}  // namespace

size_t backward_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int block_q, int block_k) {
  (void)block_q;
  (void)block_k;
  return carve(nullptr, B, Hq, Hkv, Sq, Skv).total;
}

bsa_status launch_backward(const BackwardArgs& a, cudaStream_t stream) {
  bsa_status st;
  const int G = a.Hq / a.Hkv;
  const int nQb = (int)cdiv64(a.Sq, a.block_q), nKb = (int)cdiv64(a.Skv, a.block_k);
  const int nQt = (int)cdiv64(a.Sq, kT), nKt = (int)cdiv64(a.Skv, kKT);
  const int words = (nKt + 31) / 32;
  const BwdWorkspace w = carve(a.workspace, a.B, a.Hq, a.Hkv, a.Sq, a.Skv);

  {  // -lse * log2(e) and -D per query tile
    PrepParams pp{};
    pp.o = static_cast<const __nv_bfloat16*>(a.o); pp.dout = static_cast<const __nv_bfloat16*>(a.dout);
    pp.lse = a.lse;
    pp.o_sb = a.o_sb; pp.o_ss = a.o_ss; pp.o_sh = a.o_sh; pp.d_sb = a.d_sb; pp.d_ss = a.d_ss; pp.d_sh = a.d_sh;
    pp.B = a.B; pp.Sq = a.Sq; pp.Hq = a.Hq; pp.nQt = nQt;
    for (int b = 0; b < a.B; ++b) pp.seq_lens[b] = a.seq_lens ? a.seq_lens[b] : a.Sq;
    pp.rowstat = w.rowstat;
    const int64_t warps = (int64_t)a.B * nQt * kT * a.Hq;
    const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
    if (a.d == 128) bwd_prep_kernel<128><<<grid, 256, 0, stream>>>(pp);
    else bwd_prep_kernel<64><<<grid, 256, 0, stream>>>(pp);
    if ((st = cuda_check(cudaGetLastError(), "bwd_prep_kernel launch")) != BSA_OK) return st;
  }
  {  // tile lists for dQ and inverse tile lists for dK/dV
    if ((st = cuda_check(cudaMemsetAsync(w.counters, 0, 256 + w.planes_bytes, stream), "cudaMemsetAsync(bitmaps)")) !=
        BSA_OK)
      return st;
    BitmapParams bp{};
    bp.indices = a.indices; bp.counts = a.counts; bp.planes = w.planes; bp.plane_words = w.plane_words;
    bp.B = a.B; bp.Hq = a.Hq; bp.Hkv = a.Hkv; bp.G = G; bp.nQb = nQb; bp.nKb = nKb; bp.nQt = nQt; bp.nKt = nKt;
    bp.block_q = a.block_q; bp.block_k = a.block_k; bp.words = words;
    for (int b = 0; b < a.B; ++b) bp.seq_lens[b] = a.seq_lens ? a.seq_lens[b] : a.Sq;
    const int64_t rows = (int64_t)a.B * a.Hq * nQb;
    bwd_bitmap_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(bp);
    if ((st = cuda_check(cudaGetLastError(), "bwd_bitmap_kernel launch")) != BSA_OK) return st;
    TileListParams tp{};
    tp.planes = w.planes; tp.plane_words = w.plane_words; tp.dq_list = w.dq_list; tp.dq_cnt = w.dq_cnt;
    tp.n_rows = a.B * a.Hq * nQt; tp.nKt = nKt; tp.words = words;
    bwd_tilelist_kernel<<<(unsigned)(((int64_t)tp.n_rows * 32 + 255) / 256), 256, 0, stream>>>(tp);
    if ((st = cuda_check(cudaGetLastError(), "bwd_tilelist_kernel launch")) != BSA_OK) return st;
    InvParams ip{};
    ip.planes = w.planes; ip.plane_words = w.plane_words; ip.inv_cnt = w.inv_cnt; ip.inv_list = w.inv_list;
    ip.n_groups = a.B * a.Hkv; ip.nrows = G * nQt; ip.nKt = nKt; ip.words = words;
    const int64_t warps = (int64_t)ip.n_groups * words;
    bwd_inverse_kernel<<<(unsigned)((warps * 32 + 127) / 128), 128, 0, stream>>>(ip);
    if ((st = cuda_check(cudaGetLastError(), "bwd_inverse_kernel launch")) != BSA_OK) return st;
  }
  const bool full = a.block_q >= kT && a.block_k == kKT;     // every pair mask full
  if (a.d == 128) return full ? launch_tiles<128, true>(a, w, stream) : launch_tiles<128, false>(a, w, stream);
  return full ? launch_tiles<64, true>(a, w, stream) : launch_tiles<64, false>(a, w, stream);
}

unsigned int read_and_clear_bwd_error() { return take_error_word(); }

bsa_status launch_bwd_wait_probe(unsigned long long limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cuda_check(cudaGetLastError(), "wait_probe_kernel launch (backward)");
}

}  // namespace bsa
