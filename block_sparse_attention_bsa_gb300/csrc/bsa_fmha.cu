// Selected-block attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes is fixed by the vllm-omni pull request "[Core] Add shared
// block-sparse attention adapters with FlashAttention-4" (Purpose: execute
// exactly the selector's per-query-head block lists, native GQA mapping,
// protected prefix, suffix padding masked, no dense fallback) and by
// cosmos_parallel.py (cosmos3_cp_attention: non-causal attention of
// generation queries over cat(und, gen); build_gen_key_mask: padded keys
// never contribute).  The FA4 kernel the pages run is prior art; these are
// fresh designs for GB300.  Two kernels share the work-tile scheduler and the
// softmax/epilogue arithmetic:
//
//  * fmha_fwd_pair_kernel (head dim 128): a cluster of two CTAs on the two
//    SMs of a TPC attends one 256-row query block, 128 rows per CTA, with
//    M = 256 MMAs (cta_group::2) issued by two threads of the even CTA (one
//    for S = Q K^T, one for O += P V).  See the comment above the kernel.
//  * fmha_fwd_kernel (head dim 64, and 64-key blocks at head dim 128): one
//    persistent CTA per SM and 256-row query block, the two 128-row halves
//    ping-ponged by one MMA thread; over merged lists (64/128-row query
//    blocks) each half walks only the key tiles its own query blocks selected.
//
// Common to both:
//  * Persistent CTAs walk work tiles (b, query block, head) in (request, KV
//    head) groups, GQA siblings innermost, so the running CTAs share one KV
//    head's K/V in L2.
//  * Warp 0 is the TMA producer: Q once per work tile, then K and V tiles of
//    the listed blocks, gathered by index (row = index * block_k), into
//    shared-memory rings (one of K/V stages in the pair kernel, a K ring and a
//    V ring in the single-CTA kernel).  Per-request tensor maps bound the rows
//    at prefix + L_b, so padded keys/values load as zeros.
//  * Softmax warps: thread r owns query row r (TMEM lane r): tcgen05.ld of
//    its S row, key mask, online softmax in the log2 domain with a lazy
//    rescale (O is rescaled in TMEM only when the running max grows by more
//    than 2^8), P (bf16) back to TMEM over S, and the epilogue (O / l to
//    bf16, LSE = ln-sum-exp of the scaled logits).
//  * Every mbarrier wait is bounded (see mbar_wait); a CTA that gives up
//    raises the device error word, leaves its loops and frees its TMEM.
#include <cuda_bf16.h>

#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

namespace {

struct FmhaParams {   // CUtensorMap members make it 128-byte aligned
  CUtensorMap tq[kMaxFwdBatch];
  CUtensorMap tk[kMaxFwdBatch];
  CUtensorMap tv[kMaxFwdBatch];
  int seq_lens[kMaxFwdBatch];
  int b0;           // first request of this launch
  int Bn;           // requests in this launch
  int Hq, Hkv, G, Sq, nQb, nKb, block_q, prefix_len, n_tiles;
  int causal;              // 1: query row i sees key positions 0..i only (dense pass)
  int group_rows;          // merged lists: rows per original query block (64 or 128)
  int masked;              // 1: list entries are kb | membership << 24 (merged lists)
  int list_stride;         // entries per list row (nKb, or the merged lists' row length)
  const int32_t* indices;  // NULL = dense pass
  const int32_t* counts;
  const int32_t* classes;  // merged lists: per row, steps only half 0 / only half 1 attends
  int* counter;            // next work tile (zeroed by the schedule kernel)
  const int* group_order;  // (request, KV head) groups, heaviest first
  float scale_log2;        // softmax scale * log2(e)
  __nv_bfloat16* out;      // [B, Sq, Hq, D]
  float* lse;              // [B, Hq, Sq] or NULL
};

template <int D, int BK, int NH>
struct Cfg {
  static constexpr int kChunks = D / 64;                  // 128-byte chunks per row
  static constexpr int kQHalfBytes = 128 * 128 * kChunks; // 128 rows x D bf16
  static constexpr int kQBytes = NH * kQHalfBytes;
  static constexpr int kTileBytes = BK * 128 * kChunks;   // one K or V tile
  static constexpr int kBarBytes = 512;
  static constexpr int kAlignSlack = 1024;
  static constexpr int kSmemMax = 232448;                 // 227 KB per CTA
  // K and V tiles live in two rings: K of a step is needed when its S MMA is
  // issued, V one softmax step later, so V gets the deeper ring.
  static constexpr int kTilesFit = (kSmemMax - kQBytes - kBarBytes - kAlignSlack) / kTileBytes;
  static constexpr int kKStages = kTilesFit / 2 > 8 ? 8 : kTilesFit / 2;
  static constexpr int kVStages = kTilesFit - kKStages > 8 ? 8 : kTilesFit - kKStages;
  static constexpr int kSmemBytes = kQBytes + (kKStages + kVStages) * kTileBytes + kBarBytes + kAlignSlack;
  static constexpr int kThreads = 128 + 128 * NH;
  static constexpr uint32_t kTmemCols = NH == 2 ? 512 : 256;
  static constexpr uint32_t kOCol = NH * 128;             // O_h at kOCol + 128 h
  static_assert(kKStages >= 2 && kVStages >= 2, "not enough shared memory for the K/V rings");
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BK == 64 || BK == 128, "key block");
};

// Merged-list entries: key block in the low 24 bits, one membership bit per
// original query block of the 256-row super-block from bit 24.
constexpr int kEntryBlockMask = (1 << 24) - 1;
constexpr int kEntryGroupShift = 24;

struct TileInfo {
  int bl, b, qb, h, hk, L, valid_kv;
  int n;          // list entries (key blocks of the lists' geometry)
  int steps;      // key tiles the kernel walks: n, or ceil(n / 2) when 64-key blocks are paired
  int nb, c0, c1; // steps both halves attend, only half 0, only half 1 (nb = steps unless merged)
  const int32_t* idx;
};

// Work tile t -> (request, KV head, query block, query head of the group).
// Tiles are grouped by (request, KV head); groups come in the order the
// schedule kernel wrote (most selected work first), and inside a group the
// GQA siblings are innermost, then neighbouring query blocks.  The CTAs
// running at any moment therefore share one KV head's K/V (<= 90 MB at
// 720p), which stays resident in the 126 MB L2.
__device__ __forceinline__ TileInfo decode_tile(const FmhaParams& p, int t, int KB, int BK) {
  TileInfo ti;
  const int per_group = p.G * p.nQb;
  const int gi = t / per_group;
  const int grp = p.group_order ? p.group_order[gi] : gi;
  const int w = t - gi * per_group;
  const int g = w % p.G;
  ti.qb = w / p.G;
  ti.hk = grp % p.Hkv;
  ti.bl = grp / p.Hkv;
  ti.h = ti.hk * p.G + g;
  ti.b = p.b0 + ti.bl;
  ti.L = p.seq_lens[ti.bl];
  ti.valid_kv = p.prefix_len + ti.L;
  const int64_t row = ((int64_t)ti.b * p.Hq + ti.h) * p.nQb + ti.qb;
  if (ti.qb * p.block_q >= ti.L) {
    ti.n = 0;
  } else if (p.indices == nullptr) {
    // dense pass; a causal pass stops at the block holding the block's last row
    const int kv_end = p.causal ? min(ti.valid_kv, min((ti.qb + 1) * p.block_q, ti.L)) : ti.valid_kv;
    ti.n = (kv_end + KB - 1) / KB;
  } else {
    const int c = p.counts[row];
    ti.n = c < 0 ? 0 : (c > p.list_stride ? p.list_stride : c);
  }
  ti.idx = p.indices ? p.indices + row * p.list_stride : nullptr;
  ti.steps = KB < BK ? (ti.n + 1) / 2 : ti.n;
  ti.c0 = ti.c1 = 0;
  if (p.classes && ti.steps > 0) {
    ti.c0 = min(max(p.classes[2 * row], 0), ti.steps);
    ti.c1 = min(max(p.classes[2 * row + 1], 0), ti.steps - ti.c0);
  }
  ti.nb = ti.steps - ti.c0 - ti.c1;
  return ti;
}

// K/V stage order of step k of half hh.  Merged lists come in three classes
// (see merge_lists_kernel): the key tiles both halves attend (positions
// 0 .. nb-1), then the tiles only one half attends, one for half 0 and one for
// half 1 in turn while both classes last, then the rest of the longer class.
// Other lists have nb = steps: step k is position k for both halves.
__device__ __forceinline__ int step_pos(const TileInfo& ti, int hh, int k) {
  if (k < ti.nb) return k;
  k -= ti.nb;
  const int m = min(ti.c0, ti.c1);
  return k < m ? ti.nb + 2 * k + hh : ti.nb + m + k;
}

// Max of v[LO .. LO + N) in four independent chains of three-input max.
template <int LO, int N, int M>
__device__ __forceinline__ float row_max(const float (&v)[M]) {
  static_assert(LO + N <= M && N % 8 == 0, "row range");
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int c = LO; c < LO + N; c += 8) {
    m0 = max3f(m0, v[c], v[c + 1]);
    m1 = max3f(m1, v[c + 2], v[c + 3]);
    m2 = max3f(m2, v[c + 4], v[c + 5]);
    m3 = max3f(m3, v[c + 6], v[c + 7]);
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

struct Ring {
  uint32_t stage = 0, phase = 0;
  template <int S>
  __device__ __forceinline__ void next() {
    if (++stage == S) { stage = 0; phase ^= 1u; }
  }
};

// Consumer side of the tile-id ring: waits for the next published id, reads
// it, releases the slot.  Returns -1 at the end of the work (or on abort).
struct TileRing {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == 2) { slot = 0; phase ^= 1u; }
  }
  __device__ __forceinline__ int take(uint64_t* full, uint64_t* empty, volatile int* ids,
                                      volatile int* abort, bool& ok) {
    ok = mbar_wait(smem_u32(full + slot), phase, abort);
    const int t = ok ? ids[slot] : -1;
    if (ok) mbar_arrive(smem_u32(empty + slot));
    next();
    return t;
  }
};

// BK is the key tile of the MMAs (128); KB the key block of the lists.  With
// KB = 64 two consecutive list entries fill one 128-key tile (rows 0..63 and
// 64..127 of the K/V stage), so the S MMA stays 128 wide (a 64-wide MMA
// costs as long as a 128-wide one) and each half is masked on its own.
template <int D, int BK, int NH, int KB = BK>
__global__ void __launch_bounds__(Cfg<D, BK, NH>::kThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ FmhaParams p) {
  static_assert(KB == BK || (KB == 64 && BK == 128), "key block pairing");
  static_assert(NH == 2, "two 128-row halves per work tile");
  using C = Cfg<D, BK, NH>;
  constexpr int kK = C::kKStages, kV = C::kVStages;
  // Rings of equal depth (head dim 64) act as one ring: a step's K and V
  // slots are released together after its last P V, one commit per step.
  // With a shallower K ring (head dim 128) K is released after its last S,
  // so that the next tiles' K can land while P V still reads V.
  constexpr bool kJointRelease = kK == kV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_smem = smem;
  uint8_t* k_smem = smem + C::kQBytes;
  uint8_t* v_smem = k_smem + kK * C::kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(v_smem + kV * C::kTileBytes);
  // barrier slots
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* s_full = bars + 2;            // [2]
  uint64_t* p_full = bars + 4;            // [2]
  uint64_t* o_full = bars + 6;            // [2]
  uint64_t* tile_full = bars + 8;         // [2] tile-id ring
  uint64_t* tile_empty = bars + 10;       // [2]
  uint64_t* kv_full = bars + 12;          // [kK] K tile and V tile of one step landed
  uint64_t* k_empty = kv_full + kK;       // [kK]
  uint64_t* v_empty = k_empty + kK;       // [kV]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(v_empty + kV);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tile_ids = reinterpret_cast<volatile int*>(tmem_slot + 2);   // [2]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(s_full + i), 1);
      mbar_init(smem_u32(p_full + i), 128);
      mbar_init(smem_u32(o_full + i), 1);
    }
    for (int i = 0; i < kK; ++i) {
      mbar_init(smem_u32(kv_full + i), 1);
      mbar_init(smem_u32(k_empty + i), 1);
    }
    for (int i = 0; i < kV; ++i) mbar_init(smem_u32(v_empty + i), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(tile_full + i), 1);
      mbar_init(smem_u32(tile_empty + i), 1 + 128 * NH);   // MMA thread + softmax threads
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.Bn; ++i) {
      tma_prefetch_desc(&p.tq[i]);
      tma_prefetch_desc(&p.tk[i]);
      tma_prefetch_desc(&p.tv[i]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ---
    // Key tiles in step order into the K ring and the V ring.  A step's K
    // and V tiles complete on one barrier (kv_full, indexed like the K
    // ring); the two rings' slots are released on their own barriers.
    Ring kr, vr;
    uint32_t qi = 0;
    const uint32_t q_base = smem_u32(q_smem);
    const uint32_t k_base = smem_u32(k_smem);
    const uint32_t v_base = smem_u32(v_smem);
    const uint64_t q_policy = l2_policy_evict_first();   // Q is read once
    bool ok = true;
    TileRing tr;
    while (ok) {
      // Dynamic scheduling: take the next tile and publish its id to the
      // MMA and softmax roles through the two-slot tile ring.
      int t = -1;
      if (lane == 0) {
        t = atomicAdd(p.counter, 1);
        if (t >= p.n_tiles) t = -1;
        ok = mbar_wait(smem_u32(tile_empty + tr.slot), tr.phase ^ 1u, abort_flag);
        if (ok) {
          tile_ids[tr.slot] = t;
          mbar_arrive(smem_u32(tile_full + tr.slot));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      t = __shfl_sync(0xffffffffu, t, 0);
      tr.next();
      if (!ok || t < 0) break;
      const TileInfo ti = decode_tile(p, t, KB, BK);
      if (ti.n == 0) continue;
      if (lane == 0) {
        ok = mbar_wait(smem_u32(q_empty), (qi & 1u) ^ 1u, abort_flag);
        if (ok) {
          mbar_arrive_expect_tx(smem_u32(q_full), C::kQBytes);
          for (int hh = 0; hh < NH; ++hh)
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d_hint(q_base + (hh * C::kChunks + c) * 16384, &p.tq[ti.bl], smem_u32(q_full),
                               c * 64, ti.qb * p.block_q + hh * 128, ti.h, q_policy);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++qi;
      for (int j0 = 0; j0 < ti.n && ok; j0 += 32) {
        int my_kb = ti.idx ? (j0 + lane < ti.n ? __ldg(ti.idx + j0 + lane) : 0) : j0 + lane;
        if (p.masked) my_kb &= kEntryBlockMask;
        const int m = min(32, ti.n - j0);
        for (int jj = 0; jj < m && ok; jj += BK / KB) {
          int kb = __shfl_sync(0xffffffffu, my_kb, jj);
          if (kb < 0 || kb >= p.nKb) kb = p.nKb;   // out of range: rows past the end read zeros
          // paired 64-key blocks: the second entry of the pair (past the end
          // of the list, the block past the end: zeros, fully masked)
          int kb1 = p.nKb;
          if constexpr (KB < BK) {
            const int t1 = __shfl_sync(0xffffffffu, my_kb, (jj + 1) & 31);
            if (jj + 1 < m && t1 >= 0 && t1 < p.nKb) kb1 = t1;
          }
          if (lane == 0) {
            ok = (kJointRelease || mbar_wait(smem_u32(k_empty + kr.stage), kr.phase ^ 1u, abort_flag)) &&
                 mbar_wait(smem_u32(v_empty + vr.stage), vr.phase ^ 1u, abort_flag);
            const uint32_t fb = smem_u32(kv_full + kr.stage);
            if (ok) mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
            for (int which = 0; which < 2 && ok; ++which) {
              const CUtensorMap* tm = which == 0 ? &p.tk[ti.bl] : &p.tv[ti.bl];
              const uint32_t base = which == 0 ? k_base + kr.stage * C::kTileBytes : v_base + vr.stage * C::kTileBytes;
              for (int c = 0; c < C::kChunks; ++c) {
                const uint32_t dst = base + c * (BK * 128);
                if constexpr (KB == BK) {
                  tma_load_3d(dst, tm, fb, c * 64, kb * BK, ti.hk);
                } else {            // rows 0..63 from the first block, 64..127 from the second
                  tma_load_3d(dst, tm, fb, c * 64, kb * KB, ti.hk);
                  tma_load_3d(dst + KB * 128, tm, fb, c * 64, kb1 * KB, ti.hk);
                }
              }
            }
            kr.next<kK>();
            vr.next<kV>();
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, BK, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, true);
      const uint32_t q_base = smem_u32(q_smem);
      Ring kc, vc;         // K and V ring cursors: the next tile to be used
      uint32_t qi = 0;
      uint32_t pph0 = 0u, pph1 = 0u;
      bool ok = true;
      // Shared-memory descriptors are computed once: a descriptor's start
      // address field is (address >> 4) in its low 14 bits, so moving the
      // operand by `off` bytes is a plain add of off >> 4 (shared addresses
      // stay below 2^18, so the field never carries).  Each MMA then costs one
      // 64-bit add; the issuing thread shares its SM sub-partition with two
      // busy softmax warps, and its issue rate bounds the tensor pipe.
      uint64_t qdesc[NH];
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) qdesc[hh] = sdesc_sw128(q_base + hh * C::kChunks * 16384, 16, 1024);
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(k_smem), 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(v_smem), BK * 128, 1024);
      // issue_s / issue_pv take the byte offset of the K or V tile in its ring.
      auto issue_s = [&](int hh, uint32_t tile_off) {
        const uint32_t d_t = tmem + hh * 128;
        const uint64_t bs = kdesc0 + (uint64_t)(tile_off >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          constexpr int kQChunk = 16384 >> 4, kKChunk = (BK * 128) >> 4;
          const uint64_t a = qdesc[hh] + (uint64_t)((kk / 4) * kQChunk + (kk % 4) * 2);
          const uint64_t b = bs + (uint64_t)((kk / 4) * kKChunk + (kk % 4) * 2);
          if (kk == 0) mma_ss_acc<0>(d_t, a, b, idesc_s);
          else mma_ss_acc<1>(d_t, a, b, idesc_s);
        }
      };
      auto issue_pv = [&](int hh, uint32_t tile_off, bool acc) {
        const uint32_t d_t = tmem + C::kOCol + hh * 128;
        const uint64_t bs = vdesc0 + (uint64_t)(tile_off >> 4);
        const uint32_t a_t = tmem + hh * 128;
        if (acc) mma_ts_acc<1>(d_t, a_t, bs, idesc_o);
        else mma_ts_acc<0>(d_t, a_t, bs, idesc_o);
#pragma unroll
        for (int kk = 1; kk < BK / 16; ++kk)
          mma_ts_acc<1>(d_t, a_t + kk * 8, bs + (uint64_t)(kk * ((16 * 128) >> 4)), idesc_o);
      };
      TileRing tr;
      while (ok) {
        const int t = tr.take(tile_full, tile_empty, tile_ids, abort_flag, ok);
        if (t < 0) break;
        const TileInfo ti = decode_tile(p, t, KB, BK);
        if (ti.steps == 0) continue;
        ok = mbar_wait(smem_u32(q_full), qi & 1u, abort_flag);
        ++qi;
        if (!ok) break;
        // Each half walks its own steps (step_pos): its first nb steps are
        // the key tiles both halves attend, used by half 0 first, so half 1's
        // S and P V are their last uses and release the K and V slots.  While
        // both halves have steps left they alternate, so the tensor pipe runs
        // one half's MMAs while the other half's softmax works; the rest of
        // the longer half-only class runs alone.  S and P V are issued in
        // ring order (a shared tile by both halves in a row), so each ring
        // has one cursor.  The half is a compile-time constant in each body
        // (H0 / H1): its TMEM columns, barriers and descriptors stay in
        // registers.
        const int nb = ti.nb, nh0 = nb + ti.c0, nh1 = nb + ti.c1;
        int s_left = nh0 + nh1;
        auto start_s = [&](auto H, int k) -> bool {     // S of the half's step k
          constexpr int hh = decltype(H)::value;
          const bool last = hh == 1 || k >= nb;          // last use of the K tile
          if (hh == 0 || k >= nb) {           // the step's K and V tiles have landed
            if (!mbar_wait(smem_u32(kv_full + kc.stage), kc.phase, abort_flag)) return false;
            tc_fence_after();
          }
          issue_s(hh, kc.stage * C::kTileBytes);
          mma_commit(smem_u32(s_full + hh));
          if (last) {
            if (!kJointRelease) mma_commit(smem_u32(k_empty + kc.stage));
            kc.template next<kK>();
          }
          if (--s_left == 0) mma_commit(smem_u32(q_empty));
          return true;
        };
        auto step = [&](auto H, int& k, uint32_t& ph, int nh) -> bool {   // P V of step k, S of k + 1
          constexpr int hh = decltype(H)::value;
          const bool last = hh == 1 || k >= nb;          // last use of the V tile
          if (!mbar_wait(smem_u32(p_full + hh), ph & 1u, abort_flag)) return false;
          ++ph;
          tc_fence_after();                      // V landed with K, waited for before this step's S
          issue_pv(hh, vc.stage * C::kTileBytes, k > 0);
          if (last) {
            mma_commit(smem_u32(v_empty + vc.stage));
            vc.template next<kV>();
          }
          if (++k < nh) return start_s(H, k);
          mma_commit(smem_u32(o_full + hh));
          return true;
        };
        const std::integral_constant<int, 0> H0;
        const std::integral_constant<int, 1> H1;
        int k0 = 0, k1 = 0;
        if (nh0 > 0) ok = start_s(H0, 0);
        if (ok && nh1 > 0) ok = start_s(H1, 0);
        while (ok && (k0 < nh0 || k1 < nh1)) {
          if (k0 < nh0) ok = step(H0, k0, pph0, nh0);
          if (ok && k1 < nh1) ok = step(H1, k1, pph1, nh1);
        }
      }
    }
    __syncwarp();
  }
  } else {
    // --------------------------------------------------- softmax + epilogue ---
    const int hh = (warp - 4) / 4;
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_t = tmem + lane_base + hh * 128;
    const uint32_t o_t = tmem + lane_base + C::kOCol + hh * 128;
    uint32_t sph = 0, oph = 0;
    bool ok = true;
    TileRing tr;
    while (ok) {
      const int t = tr.take(tile_full, tile_empty, tile_ids, abort_flag, ok);
      if (t < 0) break;
      const TileInfo ti = decode_tile(p, t, KB, BK);
      const int row_in_blk = hh * 128 + r;
      const int row = ti.qb * p.block_q + row_in_blk;
      const bool row_exists = row_in_blk < p.block_q && row < p.Sq;
      const bool row_ok = row_exists && row < ti.L;
      __nv_bfloat16* orow = p.out + (((int64_t)ti.b * p.Sq + row) * p.Hq + ti.h) * D;
      float* lrow = p.lse ? p.lse + ((int64_t)ti.b * p.Hq + ti.h) * p.Sq + row : nullptr;
      const int nsteps = ti.nb + (hh == 0 ? ti.c0 : ti.c1);   // this half's key tiles
      if (nsteps == 0) {
        if (row_exists) {
          uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) reinterpret_cast<uint4*>(orow)[i] = z;
          if (lrow) *lrow = -INFINITY;
        }
        continue;
      }
      float m_ref = -INFINITY;
      float l = 0.f;
      // list entry e -> key block this row attends (the block past the end,
      // i.e. fully masked, when out of range or not selected by the row's
      // own query block in a merged list)
      auto entry_block = [&](int e) {
        if (e >= ti.n) return p.nKb;
        const int entry = ti.idx ? __ldg(ti.idx + e) : e;
        int kb = (ti.idx && p.masked) ? (entry & kEntryBlockMask) : entry;
        if (kb < 0 || kb >= p.nKb) kb = p.nKb;     // same clamp as the producer: fully masked
        // merged lists: a key block that this row's own query block did not
        // select is masked whole (it contributes exact zeros)
        if (p.masked && !((entry >> (kEntryGroupShift + row_in_blk / p.group_rows)) & 1)) kb = p.nKb;
        return kb;
      };
      for (int kk = 0; kk < nsteps; ++kk) {
        const int j = step_pos(ti, hh, kk);
        const int kb = entry_block(KB < BK ? 2 * j : j);
        const int kb1 = KB < BK ? entry_block(2 * j + 1) : 0;    // second 64-key half of the tile
        // keys of this block this row may see: the real keys, and in a causal
        // pass only positions <= the row
        const int kv_end = p.causal ? min(ti.valid_kv, row + 1) : ti.valid_kv;
        // Paired 64-key blocks: a half that this row cannot see at all (a block
        // its own query block did not select in a merged list, or one past the
        // end) takes no part in the max and is not exponentiated; its P is
        // stored as zeros.
        // The test is uniform over a warp except in a causal pass.
        int kvalid0 = BK, kvalid1 = BK;
        bool skip0 = false, skip1 = false;
        if constexpr (KB < BK) {
          kvalid0 = kv_end - kb * KB;
          kvalid1 = kv_end - kb1 * KB;
          skip0 = kvalid0 <= 0;
          skip1 = kvalid1 <= 0;
        }
        ok = mbar_wait(smem_u32(s_full + hh), sph & 1u, abort_flag);
        ++sph;
        if (!ok) break;
        tc_fence_after();
        float s[BK];
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) tmem_ld32f(s_t + c * 32, s + c * 32);
        tmem_wait_ld();
        float mx;
        if constexpr (KB == BK) {
          const int kvalid = kv_end - kb * BK;
          if (kvalid < BK) {
#pragma unroll
            for (int c = 0; c < BK; ++c)
              if (c >= kvalid) s[c] = -INFINITY;
          }
          mx = row_max<0, BK>(s);
        } else {
          if ((!skip0 && kvalid0 < KB) || (!skip1 && kvalid1 < KB)) {
#pragma unroll
            for (int c = 0; c < KB; ++c) {
              if (c >= kvalid0) s[c] = -INFINITY;
              if (c >= kvalid1) s[KB + c] = -INFINITY;
            }
          }
          const float mx_lo = skip0 ? -INFINITY : row_max<0, KB>(s);
          const float mx_hi = skip1 ? -INFINITY : row_max<KB, KB>(s);
          mx = fmaxf(mx_lo, mx_hi);
        }
        const float m_new = fmaxf(m_ref, mx * p.scale_log2);
        const bool grow = m_new > m_ref + 8.0f;
        const bool rescale_o = grow && m_ref != -INFINITY;
        const float alpha = rescale_o ? ex2_approx(m_ref - m_new) : 1.f;
        if (grow) m_ref = m_new;
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        // p = 2^(s * scale * log2 e - m): packed FFMA2 for the argument, MUFU
        // ex2 per element, packed FADD2 row sums in two chains; P is packed to
        // bf16 pairs as soon as it is computed and stored over the first BK/2
        // columns of S_h 64 keys at a time, so the fp32 values do not stay live.
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m_use, -m_use);
        float2 ls0 = make_float2(0.f, 0.f), ls1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < BK / 64; ++cc) {
          uint32_t pk[32];
          if constexpr (KB < BK) {           // a skipped 64-key half: P = 0
            if (cc == 0 ? skip0 : skip1) {
#pragma unroll
              for (int i = 0; i < 32; ++i) pk[i] = 0u;
              tmem_st32(s_t + cc * 32, pk);
              continue;
            }
          }
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float2 a = __ffma2_rn(make_float2(s[cc * 64 + c], s[cc * 64 + c + 1]), sc2, nm2);
            const float2 b = __ffma2_rn(make_float2(s[cc * 64 + c + 2], s[cc * 64 + c + 3]), sc2, nm2);
            const float2 e0 = make_float2(ex2_approx(a.x), ex2_approx(a.y));
            const float2 e1 = make_float2(ex2_approx(b.x), ex2_approx(b.y));
            ls0 = __fadd2_rn(ls0, e0);
            ls1 = __fadd2_rn(ls1, e1);
            pk[c / 2] = pack_bf16x2(e0.x, e0.y);
            pk[c / 2 + 1] = pack_bf16x2(e1.x, e1.y);
          }
          tmem_st32(s_t + cc * 32, pk);
        }
        const float lsum = (ls0.x + ls0.y) + (ls1.x + ls1.y);
        l = l * alpha + lsum;
        // Lazy rescale of O (rare): after P is out of registers, before PV is issued.
        if (__any_sync(0xffffffffu, rescale_o)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32f(o_t + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32f(o_t + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(p_full + hh));
      }
      if (!ok) break;
      ok = mbar_wait(smem_u32(o_full + hh), oph & 1u, abort_flag);
      ++oph;
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32f(o_t + c * 32, o);
        tmem_wait_ld();
        if (row_exists) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = row_ok ? pack_bf16x2(o[2 * i] * inv_l, o[2 * i + 1] * inv_l) : 0u;
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (row_exists && lrow)
        *lrow = (row_ok && l > 0.f) ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------ CTA pairs ---
// The same attention for head dim 128, with one 256-row query block per
// cluster of two CTAs (the two SMs of a TPC).  CTA rank r owns query rows
// r*128 .. r*128+127 of the block, so both CTAs attend the block's one list.
// One thread of the even CTA issues M = 256 tcgen05 MMAs (cta_group::2) for
// both: S = Q K^T into each CTA's TMEM (128 lanes x 128 keys), O += P V with
// P read from each CTA's TMEM.  B operands are split across the pair: for S
// each CTA holds 64 of the tile's 128 keys (all 128 dims), for P V all 128
// keys and 64 of the 128 value dims.  Per SM, an S MMA therefore reads 6 KB
// of shared memory instead of 8 KB, and every key block costs 16 MMA
// instructions for 256 rows instead of 32.  TMEM per CTA: two S buffers
// (S of step j+1 is computed while the softmax works on step j) and O.
//
// Synchronisation across the pair (barriers at the same offsets in both
// CTAs): the even CTA's producer takes work tiles from the global counter
// and writes each id into both CTAs' tile rings (remote store, then a
// cluster-scope release arrive; consumers acquire at cluster scope); each
// CTA's producer loads its own halves with completion counted on the even
// CTA's full barriers (TMA .cta_group::2); the MMA thread's commits are
// multicast to both CTAs (S ready, a P V finished, stage and Q buffer free);
// each softmax warp arrives once per step on the even CTA's P barrier.  The
// per-step hand-offs carry TMEM or TMA data only, ordered by the tcgen05 and
// transaction-count rules, so they use CTA-scope waits and a relaxed remote
// arrive (a cluster-scope release costs ~1,000 cycles per step).
constexpr int kPairSBufs = 3;   // S buffers of the CTA-pair kernel

template <int NS>
struct PairCfg {
  static constexpr int D = 128;
  static constexpr int kQBytes = 128 * 128 * 2;     // 128 rows x 128 dims: two 64-dim chunks of 16 KB
  static constexpr int kQBufs = 2;
  static constexpr int kKBytes = 64 * 128 * 2;      // 64 keys x 128 dims: two chunks of 8 KB
  static constexpr int kVBytes = 128 * 64 * 2;      // 128 keys x 64 dims: one chunk
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kAlignSlack = 1024;
  static constexpr int kSmemMax = 232448;
  static constexpr int kStagesFit = (kSmemMax - kQBufs * kQBytes - kBarBytes - kAlignSlack) / kStageBytes;
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kSmemBytes = kQBufs * kQBytes + kStages * kStageBytes + kBarBytes + kAlignSlack;
  static constexpr int kThreads = 256;              // warp 0 TMA, warp 1 S MMAs + TMEM, warp 2 P V MMAs, warps 4..7 softmax
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 128 * NS;       // S buffers at 0, 128, ..., O after them
  static constexpr int kTileEmptyCount = 11;        // 2 MMA threads + 4 softmax warps + peer producer + 4 peer warps
  static constexpr int kPFullCount = 8;             // 4 softmax warps per CTA
  static_assert(kStages >= 3, "not enough shared memory for a K/V ring");
  static_assert(NS >= 2 && 128 * NS + 128 <= 512, "TMEM columns");
  static constexpr int kNumBars = 9 + 3 * NS + 2 * kStages;
  static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier block");
};

template <int KB, int NS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<NS>::kThreads, 1)
    fmha_fwd_pair_kernel(const __grid_constant__ FmhaParams p) {
  static_assert(KB == 128 || KB == 64, "key block");
  using C = PairCfg<NS>;
  constexpr int BK = 128;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_smem = smem;
  uint8_t* kv_smem = smem + C::kQBufs * C::kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(kv_smem + S * C::kStageBytes);
  uint64_t* q_full = bars + 0;             // [2] even CTA: both halves of a Q buffer landed
  uint64_t* q_empty = bars + 2;            // [2] both: the tile's last S MMA finished
  uint64_t* mma_done = bars + 4;           // both: the MMA threads' last commits (exit)
  uint64_t* tile_full = bars + 5;          // [2] both: tile id published
  uint64_t* tile_empty = bars + 7;         // [2] even CTA: every consumer of both CTAs read the id
  uint64_t* s_full = bars + 9;             // [NS] both: S buffer b holds this step's scores
  uint64_t* p_full = bars + 9 + NS;        // [NS] even CTA: P of S buffer b written by both CTAs
  uint64_t* pv_done = bars + 9 + 2 * NS;   // [NS] both: the P V reading S buffer b finished
  uint64_t* kv_full = bars + 9 + 3 * NS;   // [S] even CTA: both halves of a K/V stage landed
  uint64_t* kv_empty = kv_full + S;        // [S] both: the stage's P V finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tile_ids = reinterpret_cast<volatile int*>(tmem_slot + 2);   // [2]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(q_full + i), 1);
      mbar_init(smem_u32(q_empty + i), 1);
      mbar_init(smem_u32(tile_full + i), 1);
      mbar_init(smem_u32(tile_empty + i), C::kTileEmptyCount);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(s_full + i), 1);
      mbar_init(smem_u32(p_full + i), C::kPFullCount);
      mbar_init(smem_u32(pv_done + i), 1);
    }
    mbar_init(smem_u32(mma_done), 2);
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(kv_full + i), 1);
      mbar_init(smem_u32(kv_empty + i), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.Bn; ++i) {
      tma_prefetch_desc(&p.tq[i]);
      tma_prefetch_desc(&p.tk[i]);
      tma_prefetch_desc(&p.tv[i]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();   // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // shared::cluster addresses in the even CTA (or in the peer)
  auto at_leader = [&](const void* x) { return cluster_addr(smem_u32(x), 0u); };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ---
    Ring ring;
    uint32_t qi = 0;
    const uint32_t q_base = smem_u32(q_smem);
    const uint32_t kv_base = smem_u32(kv_smem);
    const uint64_t q_policy = l2_policy_evict_first();
    bool ok = true;
    TileRing tr;
    while (ok) {
      int t = -1;
      if (lane == 0) {
        if (leader) {
          // take the next tile and publish its id in both CTAs' rings
          t = atomicAdd(p.counter, 1);
          if (t >= p.n_tiles) t = -1;
          ok = mbar_wait_cl(smem_u32(tile_empty + tr.slot), tr.phase ^ 1u, abort_flag);
          if (ok) {
            tile_ids[tr.slot] = t;
            st_cluster_u32(cluster_addr(smem_u32(const_cast<int*>(tile_ids + tr.slot)), 1u), (uint32_t)t);
            mbar_arrive(smem_u32(tile_full + tr.slot));
            mbar_arrive_remote(cluster_addr(smem_u32(tile_full + tr.slot), 1u));
          }
        } else {
          ok = mbar_wait_cl(smem_u32(tile_full + tr.slot), tr.phase, abort_flag);
          t = ok ? tile_ids[tr.slot] : -1;
          if (ok) mbar_arrive_remote(at_leader(tile_empty + tr.slot));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      t = __shfl_sync(0xffffffffu, t, 0);
      tr.next();
      if (!ok || t < 0) break;
      const TileInfo ti = decode_tile(p, t, KB, BK);
      if (ti.n == 0) continue;
      if (lane == 0) {
        const uint32_t qs = qi & 1u;
        ok = mbar_wait(smem_u32(q_empty + qs), ((qi >> 1) & 1u) ^ 1u, abort_flag);
        if (ok) {
          if (leader) mbar_arrive_expect_tx(smem_u32(q_full + qs), 2 * C::kQBytes);
          const uint32_t fb = at_leader(q_full + qs);
          for (int c = 0; c < 2; ++c)
            tma_load_3d_pair_hint(q_base + qs * C::kQBytes + c * 16384, &p.tq[ti.bl], fb, c * 64,
                                  ti.qb * p.block_q + (int)rank * 128, ti.h, q_policy);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++qi;
      for (int j0 = 0; j0 < ti.n && ok; j0 += 32) {
        int my_kb = ti.idx ? (j0 + lane < ti.n ? __ldg(ti.idx + j0 + lane) : 0) : j0 + lane;
        if (p.masked) my_kb &= kEntryBlockMask;
        const int m = min(32, ti.n - j0);
        for (int jj = 0; jj < m && ok; jj += BK / KB) {
          int kb = __shfl_sync(0xffffffffu, my_kb, jj);
          if (kb < 0 || kb >= p.nKb) kb = p.nKb;   // out of range: rows past the end read zeros
          int kb1 = p.nKb;                          // second 64-key block of the tile
          if constexpr (KB < BK) {
            const int t1 = __shfl_sync(0xffffffffu, my_kb, (jj + 1) & 31);
            if (jj + 1 < m && t1 >= 0 && t1 < p.nKb) kb1 = t1;
          }
          if (lane == 0) {
            ok = mbar_wait(smem_u32(kv_empty + ring.stage), ring.phase ^ 1u, abort_flag);
            if (ok) {
              if (leader) mbar_arrive_expect_tx(smem_u32(kv_full + ring.stage), 2 * C::kStageBytes);
              const uint32_t fb = at_leader(kv_full + ring.stage);
              const uint32_t kd = kv_base + ring.stage * C::kStageBytes;
              const uint32_t vd = kd + C::kKBytes;
              // K: this CTA's 64 keys of the tile, all 128 dims (two chunks)
              const int krow = KB == BK ? kb * BK + (int)rank * 64 : (rank == 0 ? kb : kb1) * KB;
              for (int c = 0; c < 2; ++c) tma_load_3d_pair(kd + c * 8192, &p.tk[ti.bl], fb, c * 64, krow, ti.hk);
              // V: all 128 keys of the tile, this CTA's 64 dims
              if constexpr (KB == BK) {
                tma_load_3d_pair(vd, &p.tv[ti.bl], fb, (int)rank * 64, kb * BK, ti.hk);
              } else {
                tma_load_3d_pair(vd, &p.tv[ti.bl], fb, (int)rank * 64, kb * KB, ti.hk);
                tma_load_3d_pair(vd + KB * 128, &p.tv[ti.bl], fb, (int)rank * 64, kb1 * KB, ti.hk);
              }
              ring.next<S>();
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
    }
    __syncwarp();
    // On an abort, copies of this CTA may still be in flight: give them time
    // to land (they complete in microseconds) before the CTA can exit.
    if (*abort_flag && lane == 0) {
      const unsigned long long t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 20000000ull) {
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ----------------------------------------------------- MMA issuers ---
    // Two threads of the even CTA issue the pair's MMAs: warp 1 the S MMAs,
    // warp 2 the P V MMAs.  Each one's barrier waits and commits overlap the
    // other's MMAs, so the tensor pipe is fed while one of them waits.  They
    // follow the same step, buffer and K/V stage rotation; their
    // dependencies go through barriers: S into buffer b waits for the P V
    // that last read b (pv_done[b]); P V (j) waits for P (j), which implies
    // S (j), and so K/V (j), complete.
    if (leader && lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(256, BK, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(256, C::D, true);
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(q_smem), 16, 1024);
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(kv_smem), 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(kv_smem) + C::kKBytes, 16, 1024);
      constexpr uint16_t kBoth = 3;
      const bool s_role = warp == 1;
      Ring ring;
      uint32_t qi = 0;
      uint32_t b = 0;                   // S buffer of the next step (steps rotate over the NS buffers)
      // Per-buffer phase bits packed in registers: bit b of ph = parity of
      // the next phase to wait for (p_full[b] for the P V thread; pv_done[b]
      // for the S thread); bit b of used = buffer b has held an S before.
      uint32_t ph = 0u, used = 0u;
      bool ok = true;
      TileRing tr;
      while (ok) {
        ok = mbar_wait_cl(smem_u32(tile_full + tr.slot), tr.phase, abort_flag);
        const int t = ok ? tile_ids[tr.slot] : -1;
        if (ok) mbar_arrive(smem_u32(tile_empty + tr.slot));
        tr.next();
        if (t < 0) break;
        const TileInfo ti = decode_tile(p, t, KB, BK);
        const int n = ti.steps;
        if (n == 0) continue;
        if (s_role) {
          const uint32_t qs = qi & 1u;
          ok = mbar_wait(smem_u32(q_full + qs), (qi >> 1) & 1u, abort_flag);
          ++qi;
          if (!ok) break;
          const uint64_t a0 = qdesc0 + (uint64_t)((qs * C::kQBytes) >> 4);
          for (int j = 0; j < n && ok; ++j) {
            const uint32_t st = ring.stage;
            ok = mbar_wait(smem_u32(kv_full + st), ring.phase, abort_flag);
            ring.next<S>();
            if (ok && ((used >> b) & 1u)) {
              ok = mbar_wait(smem_u32(pv_done + b), (ph >> b) & 1u, abort_flag);
              ph ^= 1u << b;
            }
            if (!ok) break;
            used |= 1u << b;
            tc_fence_after();
            // S_b = Q K_st^T (K = 128 dims in 8 steps of 16)
            const uint32_t d_t = tmem + b * 128;
            const uint64_t b0 = kdesc0 + (uint64_t)((st * C::kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < C::D / 16; ++kk) {
              const uint64_t a = a0 + (uint64_t)((kk / 4) * (16384 >> 4) + (kk % 4) * 2);
              const uint64_t bb = b0 + (uint64_t)((kk / 4) * (8192 >> 4) + (kk % 4) * 2);
              if (kk == 0) mma2_ss_acc<0>(d_t, a, bb, idesc_s);
              else mma2_ss_acc<1>(d_t, a, bb, idesc_s);
            }
            mma2_commit_mc(smem_u32(s_full + b), kBoth);
            if (j + 1 == n) mma2_commit_mc(smem_u32(q_empty + qs), kBoth);
            b = b + 1 == (uint32_t)NS ? 0u : b + 1;
          }
        } else {
          for (int j = 0; j < n && ok; ++j) {
            const uint32_t st = ring.stage;
            ring.next<S>();
            ok = mbar_wait(smem_u32(p_full + b), (ph >> b) & 1u, abort_flag);
            ph ^= 1u << b;
            if (!ok) break;
            tc_fence_after();
            // O += P_b V_st (K = 128 keys in 8 steps of 16; P bf16 packed in S_b)
            const uint32_t d_t = tmem + C::kOCol;
            const uint32_t a_t = tmem + b * 128;
            const uint64_t bs = vdesc0 + (uint64_t)((st * C::kStageBytes) >> 4);
            if (j > 0) mma2_ts_acc<1>(d_t, a_t, bs, idesc_o);
            else mma2_ts_acc<0>(d_t, a_t, bs, idesc_o);
#pragma unroll
            for (int kk = 1; kk < BK / 16; ++kk)
              mma2_ts_acc<1>(d_t, a_t + kk * 8, bs + (uint64_t)(kk * ((16 * 128) >> 4)), idesc_o);
            mma2_commit_mc(smem_u32(pv_done + b), kBoth);
            mma2_commit_mc(smem_u32(kv_empty + st), kBoth);
            b = b + 1 == (uint32_t)NS ? 0u : b + 1;
          }
        }
      }
      // every MMA issued has finished before either CTA frees its TMEM
      mma2_commit_mc(smem_u32(mma_done), kBoth);
    }
    __syncwarp();
    if (warp == 1 && lane == 0) mbar_drain_cl(smem_u32(mma_done), 0u, kWaitTimeoutNs);
    __syncwarp();
  } else if (warp >= 4) {
    // --------------------------------------------------- softmax + epilogue ---
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t o_t = tmem + lane_base + C::kOCol;
    const uint32_t p_full_cl0 = at_leader(p_full);   // p_full + b at p_full_cl0 + 8 b
    const uint32_t tile_empty_cl[2] = {at_leader(tile_empty), at_leader(tile_empty + 1)};
    uint32_t b = 0;                   // S buffer of the next step
    // Bit b of sph: phase of s_full[b] to wait for next.  Bit b of pvph:
    // parity of the phase of pv_done[b] that the next P V on buffer b will
    // complete (it flips when this thread hands a P of buffer b over).  Waiting for the
    // P V of the previous step, on buffer bp, is unambiguous whenever it is
    // needed: the one before it on bp finished before S(this step) was
    // computed, and the one after it needs a P this thread has not made.
    // bit b of sph / pvph (packed in registers, not runtime-indexed arrays)
    uint32_t sph = 0u, pvph = 0u;
    bool ok = true;
    TileRing tr;
    while (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait_cl(smem_u32(tile_full + tr.slot), tr.phase, abort_flag));
      const int t = ok ? tile_ids[tr.slot] : -1;
      __syncwarp();
      if (ok && lane == 0) {
        if (leader) mbar_arrive(smem_u32(tile_empty + tr.slot));
        else mbar_arrive_remote(tile_empty_cl[tr.slot]);
      }
      tr.next();
      if (t < 0) break;
      const TileInfo ti = decode_tile(p, t, KB, BK);
      const int row_in_blk = (int)rank * 128 + r;
      const int row = ti.qb * p.block_q + row_in_blk;
      const bool row_exists = row_in_blk < p.block_q && row < p.Sq;
      const bool row_ok = row_exists && row < ti.L;
      __nv_bfloat16* orow = p.out + (((int64_t)ti.b * p.Sq + row) * p.Hq + ti.h) * C::D;
      float* lrow = p.lse ? p.lse + ((int64_t)ti.b * p.Hq + ti.h) * p.Sq + row : nullptr;
      if (ti.n == 0) {
        if (row_exists) {
          uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < C::D / 8; ++i) reinterpret_cast<uint4*>(orow)[i] = z;
          if (lrow) *lrow = -INFINITY;
        }
        continue;
      }
      float m_ref = -INFINITY;
      float l = 0.f;
      auto entry_block = [&](int e) {
        if (e >= ti.n) return p.nKb;
        const int entry = ti.idx ? __ldg(ti.idx + e) : e;
        int kb = (ti.idx && p.masked) ? (entry & kEntryBlockMask) : entry;
        if (kb < 0 || kb >= p.nKb) kb = p.nKb;
        if (p.masked && !((entry >> (kEntryGroupShift + row_in_blk / p.group_rows)) & 1)) kb = p.nKb;
        return kb;
      };
      for (int j = 0; j < ti.steps; ++j, b = b + 1 == (uint32_t)NS ? 0u : b + 1) {
        const uint32_t s_t = tmem + lane_base + b * 128;
        const int kb = entry_block(KB < BK ? 2 * j : j);
        const int kb1 = KB < BK ? entry_block(2 * j + 1) : 0;
        const int kv_end = p.causal ? min(ti.valid_kv, row + 1) : ti.valid_kv;
        int kvalid0 = BK, kvalid1 = BK;
        bool skip0 = false, skip1 = false;
        if constexpr (KB < BK) {
          kvalid0 = kv_end - kb * KB;
          kvalid1 = kv_end - kb1 * KB;
          skip0 = kvalid0 <= 0;
          skip1 = kvalid1 <= 0;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(s_full + b), (sph >> b) & 1u, abort_flag));
        sph ^= 1u << b;
        if (!ok) break;
        tc_fence_after();
        float sv[BK];
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) tmem_ld32f(s_t + c * 32, sv + c * 32);
        tmem_wait_ld();
        float mx;
        if constexpr (KB == BK) {
          const int kvalid = kv_end - kb * BK;
          if (kvalid < BK) {
#pragma unroll
            for (int c = 0; c < BK; ++c)
              if (c >= kvalid) sv[c] = -INFINITY;
          }
          mx = row_max<0, BK>(sv);
        } else {
          if ((!skip0 && kvalid0 < KB) || (!skip1 && kvalid1 < KB)) {
#pragma unroll
            for (int c = 0; c < KB; ++c) {
              if (c >= kvalid0) sv[c] = -INFINITY;
              if (c >= kvalid1) sv[KB + c] = -INFINITY;
            }
          }
          const float mx_lo = skip0 ? -INFINITY : row_max<0, KB>(sv);
          const float mx_hi = skip1 ? -INFINITY : row_max<KB, KB>(sv);
          mx = fmaxf(mx_lo, mx_hi);
        }
        const float m_new = fmaxf(m_ref, mx * p.scale_log2);
        const bool grow = m_new > m_ref + 8.0f;
        const bool rescale_o = grow && m_ref != -INFINITY;
        const float alpha = rescale_o ? ex2_approx(m_ref - m_new) : 1.f;
        if (grow) m_ref = m_new;
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m_use, -m_use);
        float2 ls0 = make_float2(0.f, 0.f), ls1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < BK / 64; ++cc) {
          uint32_t pk[32];
          if constexpr (KB < BK) {
            if (cc == 0 ? skip0 : skip1) {
#pragma unroll
              for (int i = 0; i < 32; ++i) pk[i] = 0u;
              tmem_st32(s_t + cc * 32, pk);
              continue;
            }
          }
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float2 a = __ffma2_rn(make_float2(sv[cc * 64 + c], sv[cc * 64 + c + 1]), sc2, nm2);
            const float2 bq = __ffma2_rn(make_float2(sv[cc * 64 + c + 2], sv[cc * 64 + c + 3]), sc2, nm2);
            const float2 e0 = make_float2(ex2_approx(a.x), ex2_approx(a.y));
            const float2 e1 = make_float2(ex2_approx(bq.x), ex2_approx(bq.y));
            ls0 = __fadd2_rn(ls0, e0);
            ls1 = __fadd2_rn(ls1, e1);
            pk[c / 2] = pack_bf16x2(e0.x, e0.y);
            pk[c / 2 + 1] = pack_bf16x2(e1.x, e1.y);
            // each 32 keys of P go to TMEM as soon as they are packed
            if (c == 28) tmem_st16(s_t + cc * 32, pk);
          }
          tmem_st16(s_t + cc * 32 + 16, pk + 16);
        }
        const float lsum = (ls0.x + ls0.y) + (ls1.x + ls1.y);
        l = l * alpha + lsum;
        // O is rescaled (rare) only after the P V of the previous step finished.
        if (__any_sync(0xffffffffu, rescale_o)) {
          const uint32_t bp = b == 0 ? (uint32_t)NS - 1 : b - 1;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(pv_done + bp), ((pvph >> bp) & 1u) ^ 1u, abort_flag));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < C::D / 32; ++c) {
            float o[32];
            tmem_ld32f(o_t + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32f(o_t + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(smem_u32(p_full + b));
          else mbar_arrive_remote_relaxed(p_full_cl0 + 8u * b);
        }
        pvph ^= 1u << b;
      }
      if (!ok) break;
      {  // the tile's last P V (on the buffer before b)
        const uint32_t bl = b == 0 ? (uint32_t)NS - 1 : b - 1;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(pv_done + bl), ((pvph >> bl) & 1u) ^ 1u, abort_flag));
      }
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < C::D / 32; ++c) {
        float o[32];
        tmem_ld32f(o_t + c * 32, o);
        tmem_wait_ld();
        if (row_exists) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = row_ok ? pack_bf16x2(o[2 * i] * inv_l, o[2 * i + 1] * inv_l) : 0u;
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (row_exists && lrow)
        *lrow = (row_ok && l > 0.f) ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
    }
  }
  tc_fence_before();
  cluster_sync_all();   // no arrival, store or MMA of either CTA targets the other after this
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------- scheduling ---
// One CTA: total selected work of every (request, KV head) group (query rows
// x listed blocks, summed over the group's query heads and query blocks),
// groups ranked heaviest first (ties: lower group first), and the tile
// counter reset for the forward launch that follows on the same stream.
struct ScheduleParams {
  const int32_t* counts;   // NULL = dense pass
  int causal;
  int b0, Bn, Hq, Hkv, G, nQb, nKb, block_q, block_k, prefix_len;
  int seq_lens[kMaxFwdBatch];
  int* counter;
  int* order;
};

constexpr int kMaxGroups = kMaxFwdBatch * kMaxHeads;

__global__ void __launch_bounds__(1024) schedule_kernel(const __grid_constant__ ScheduleParams p) {
  __shared__ unsigned long long cost[kMaxGroups];
  const int ng = p.Bn * p.Hkv;
  for (int i = threadIdx.x; i < ng; i += blockDim.x) cost[i] = 0ull;
  __syncthreads();
  // Warps split the groups' tiles (query blocks fastest, so count reads are
  // coalesced); each warp reduces its slice and adds it with one atomic.
  const int per_group = p.G * p.nQb;
  const int nwarps = blockDim.x / 32;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wpg = max(1, nwarps / ng);            // warps per group
  for (int task = warp; task < ng * wpg; task += nwarps) {
    const int gi = task / wpg, part = task - gi * wpg;
    const int bl = gi / p.Hkv, hk = gi - bl * p.Hkv;
    const int L = p.seq_lens[bl];
    unsigned long long c = 0;
    for (int w = part * 32 + lane; w < per_group; w += 32 * wpg) {
      const int g = w / p.nQb, qb = w - g * p.nQb;
      const int rows = min(p.block_q, L - qb * p.block_q);
      if (rows <= 0) continue;
      const int kv_end = p.causal ? min(p.prefix_len + L, min((qb + 1) * p.block_q, L)) : p.prefix_len + L;
      int n = (kv_end + p.block_k - 1) / p.block_k;
      if (p.counts) {
        n = p.counts[((int64_t)(p.b0 + bl) * p.Hq + hk * p.G + g) * p.nQb + qb];
        n = n < 0 ? 0 : min(n, p.nKb);
      }
      c += (unsigned long long)rows * (unsigned long long)n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0 && c) atomicAdd(&cost[gi], c);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ng; i += blockDim.x) {
    int rank = 0;
    for (int j = 0; j < ng; ++j) rank += (cost[j] > cost[i]) || (cost[j] == cost[i] && j < i);
    p.order[rank] = i;
  }
  if (threadIdx.x == 0) *p.counter = 0;
}

// ------------------------------------------------------------- host side ---

template <int D, int BK, int NH, int KB = BK>
bsa_status launch_t(const ForwardArgs& a, cudaStream_t stream) {
  using C = Cfg<D, BK, NH>;
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  bsa_status st;
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    if ((st = cuda_check(cudaFuncSetAttribute(fmha_fwd_kernel<D, BK, NH, KB>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              C::kSmemBytes),
                         "cudaFuncSetAttribute(fmha_fwd_kernel)")) != BSA_OK)
      return st;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int sms = num_sms();
  for (int b0 = 0; b0 < a.B; b0 += kMaxFwdBatch) {
    const int Bn = std::min(kMaxFwdBatch, a.B - b0);
    FmhaParams p;
    std::memset(&p, 0, sizeof(p));
    for (int i = 0; i < Bn; ++i) {
      const int b = b0 + i;
      const int L = a.seq_lens ? a.seq_lens[b] : a.Sq;
      p.seq_lens[i] = L;
      const char* qb = static_cast<const char*>(a.q) + (int64_t)b * a.q_sb * 2;
      const char* kb = static_cast<const char*>(a.k) + (int64_t)b * a.k_sb * 2;
      const char* vb = static_cast<const char*>(a.v) + (int64_t)b * a.v_sb * 2;
      if ((st = encode_tensor_map(&p.tq[i], qb, L, a.Hq, D, a.q_ss, a.q_sh, 128, "Q")) != BSA_OK) return st;
      if ((st = encode_tensor_map(&p.tk[i], kb, a.prefix_len + L, a.Hkv, D, a.k_ss, a.k_sh, KB, "K")) != BSA_OK)
        return st;
      if ((st = encode_tensor_map(&p.tv[i], vb, a.prefix_len + L, a.Hkv, D, a.v_ss, a.v_sh, KB, "V")) != BSA_OK)
        return st;
    }
    p.b0 = b0;
    p.Bn = Bn;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.Sq = a.Sq;
    p.nQb = a.nQb;
    p.nKb = a.nKb;
    p.block_q = a.block_q;
    p.prefix_len = a.prefix_len;
    p.n_tiles = Bn * a.nQb * a.Hq;
    p.indices = a.indices;
    p.counts = a.counts;
    p.classes = a.classes;
    p.list_stride = a.list_stride > 0 ? a.list_stride : a.nKb;
    p.causal = a.causal ? 1 : 0;
    p.masked = a.masked ? 1 : 0;
    p.group_rows = a.group_rows > 0 ? a.group_rows : a.block_q;
    char* cws = static_cast<char*>(a.workspace) + (size_t)(b0 / kMaxFwdBatch) * forward_chunk_bytes(a.Hq);
    p.counter = reinterpret_cast<int*>(cws);
    p.group_order = reinterpret_cast<const int*>(cws + 256);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    const int grid = std::min(p.n_tiles, sms);
    if (grid <= 0) continue;
    ScheduleParams sp{};
    sp.counts = a.indices ? a.counts : nullptr;
    sp.causal = a.causal ? 1 : 0;
    sp.b0 = b0; sp.Bn = Bn; sp.Hq = a.Hq; sp.Hkv = a.Hkv; sp.G = a.Hq / a.Hkv;
    sp.nQb = a.nQb; sp.nKb = a.nKb; sp.block_q = a.block_q; sp.block_k = KB; sp.prefix_len = a.prefix_len;
    for (int i = 0; i < Bn; ++i) sp.seq_lens[i] = p.seq_lens[i];
    sp.counter = p.counter;
    sp.order = const_cast<int*>(p.group_order);
    schedule_kernel<<<1, 1024, 0, stream>>>(sp);
    if ((st = cuda_check(cudaGetLastError(), "schedule_kernel launch")) != BSA_OK) return st;
    fmha_fwd_kernel<D, BK, NH, KB><<<grid, C::kThreads, C::kSmemBytes, stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "fmha_fwd_kernel launch")) != BSA_OK) return st;
  }
  return BSA_OK;
}

// CTA-pair launch: the same per-chunk parameters, tensor maps whose K box is
// 64 rows (each CTA loads half of a key tile) and a grid of as many 2-CTA
// clusters as can be resident at once.
template <int KB, int NS>
bsa_status launch_pair(const ForwardArgs& a, cudaStream_t stream) {
  using C = PairCfg<NS>;
  static std::atomic<int> clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  bsa_status st;
  int max_clusters = dev < 64 ? clusters[dev].load(std::memory_order_acquire) : 0;
  if (max_clusters <= 0) {
    if ((st = cuda_check(cudaFuncSetAttribute(fmha_fwd_pair_kernel<KB, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              C::kSmemBytes),
                         "cudaFuncSetAttribute(fmha_fwd_pair_kernel)")) != BSA_OK)
      return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)(num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if ((st = cuda_check(cudaOccupancyMaxActiveClusters(&max_clusters, fmha_fwd_pair_kernel<KB, NS>, &cfg),
                         "cudaOccupancyMaxActiveClusters(fmha_fwd_pair_kernel)")) != BSA_OK)
      return st;
    if (max_clusters <= 0) return set_error(BSA_ERR_UNSUPPORTED, "bsa_forward: no CTA pair fits on this device");
    if (dev < 64) clusters[dev].store(max_clusters, std::memory_order_release);
  }
  for (int b0 = 0; b0 < a.B; b0 += kMaxFwdBatch) {
    const int Bn = std::min(kMaxFwdBatch, a.B - b0);
    FmhaParams p;
    std::memset(&p, 0, sizeof(p));
    for (int i = 0; i < Bn; ++i) {
      const int b = b0 + i;
      const int L = a.seq_lens ? a.seq_lens[b] : a.Sq;
      p.seq_lens[i] = L;
      const char* qb = static_cast<const char*>(a.q) + (int64_t)b * a.q_sb * 2;
      const char* kb = static_cast<const char*>(a.k) + (int64_t)b * a.k_sb * 2;
      const char* vb = static_cast<const char*>(a.v) + (int64_t)b * a.v_sb * 2;
      if ((st = encode_tensor_map(&p.tq[i], qb, L, a.Hq, 128, a.q_ss, a.q_sh, 128, "Q")) != BSA_OK) return st;
      if ((st = encode_tensor_map(&p.tk[i], kb, a.prefix_len + L, a.Hkv, 128, a.k_ss, a.k_sh, 64, "K")) != BSA_OK)
        return st;
      if ((st = encode_tensor_map(&p.tv[i], vb, a.prefix_len + L, a.Hkv, 128, a.v_ss, a.v_sh, KB, "V")) != BSA_OK)
        return st;
    }
    p.b0 = b0;
    p.Bn = Bn;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.Sq = a.Sq;
    p.nQb = a.nQb;
    p.nKb = a.nKb;
    p.block_q = a.block_q;
    p.prefix_len = a.prefix_len;
    p.n_tiles = Bn * a.nQb * a.Hq;
    p.indices = a.indices;
    p.counts = a.counts;
    p.classes = a.classes;
    p.list_stride = a.list_stride > 0 ? a.list_stride : a.nKb;
    p.causal = a.causal ? 1 : 0;
    p.masked = a.masked ? 1 : 0;
    p.group_rows = a.group_rows > 0 ? a.group_rows : a.block_q;
    char* cws = static_cast<char*>(a.workspace) + (size_t)(b0 / kMaxFwdBatch) * forward_chunk_bytes(a.Hq);
    p.counter = reinterpret_cast<int*>(cws);
    p.group_order = reinterpret_cast<const int*>(cws + 256);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    const int n_clusters = std::min(p.n_tiles, max_clusters);
    if (n_clusters <= 0) continue;
    ScheduleParams sp{};
    sp.counts = a.indices ? a.counts : nullptr;
    sp.causal = a.causal ? 1 : 0;
    sp.b0 = b0; sp.Bn = Bn; sp.Hq = a.Hq; sp.Hkv = a.Hkv; sp.G = a.Hq / a.Hkv;
    sp.nQb = a.nQb; sp.nKb = a.nKb; sp.block_q = a.block_q; sp.block_k = KB; sp.prefix_len = a.prefix_len;
    for (int i = 0; i < Bn; ++i) sp.seq_lens[i] = p.seq_lens[i];
    sp.counter = p.counter;
    sp.order = const_cast<int*>(p.group_order);
    schedule_kernel<<<1, 1024, 0, stream>>>(sp);
    if ((st = cuda_check(cudaGetLastError(), "schedule_kernel launch")) != BSA_OK) return st;
    fmha_fwd_pair_kernel<KB, NS><<<2 * n_clusters, C::kThreads, C::kSmemBytes, stream>>>(p);
    if ((st = cuda_check(cudaGetLastError(), "fmha_fwd_pair_kernel launch")) != BSA_OK) return st;
  }
  return BSA_OK;
}

}  // namespace

size_t forward_chunk_bytes(int Hq) {
  return 256 + (((size_t)4 * kMaxFwdBatch * Hq + 255) & ~(size_t)255);
}

unsigned int read_and_clear_fwd_error() { return take_error_word(); }

bsa_status launch_fwd_wait_probe(unsigned long long limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cuda_check(cudaGetLastError(), "wait_probe_kernel launch (forward)");
}

// ------------------------------------------------------ merged lists ---
// For query blocks of 64 or 128 rows, the 256/block_q query blocks of each
// 256-row super-block are attended together: one warp ORs their key-block
// lists into bitmaps and writes the union with one membership bit per query
// block (kb | bits << 24).  The forward then runs its 256-row, two-half
// ping-pong path over the union and masks, per row, the key blocks the row's
// own query block did not select -- the same result as attending each query
// block's list alone, with K/V tiles reused by both 128-row halves where both
// attend them.
//
// The union is written in steps of per_step entries (one key tile of the
// forward: two 64-key blocks, or one 128-key block), in three classes, each
// in ascending key order: the blocks both halves' query blocks selected, then
// the blocks only half 0's or only half 1's selected, one step of each in
// turn while both last, then the rest of the longer class.  A class whose
// size is not a multiple of per_step ends with a padding entry (the block
// past the end, no membership bit), so no step mixes classes and a half
// skips every step of the other half's class (step_pos in the forward walks
// the same order).  Per row: count = entries including padding, classes =
// (steps of the half-0-only class, steps of the half-1-only class).
struct MergeParams {
  const int32_t* indices;   // [B, Hq, nQb, nKb]
  const int32_t* counts;    // [B, Hq, nQb]
  int32_t* uindices;        // [B, Hq, nSb, stride]
  int32_t* ucounts;         // [B, Hq, nSb]
  int32_t* uclasses;        // [B, Hq, nSb, 2]
  int Hq, nQb, nKb, nSb, ratio, words, per_step, stride;
};

// Row length of a merged list: the union (at most nKb blocks) plus one
// padding entry per class.
inline int merged_stride(int nKb) { return nKb + 3; }

__global__ void __launch_bounds__(32) merge_lists_kernel(const __grid_constant__ MergeParams p) {
  extern __shared__ uint32_t bm[];   // [ratio][words]
  const int lane = threadIdx.x;
  const int sb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  for (int i = lane; i < p.ratio * p.words; i += 32) bm[i] = 0u;
  __syncwarp();
  for (int g = 0; g < p.ratio; ++g) {
    const int qb = sb * p.ratio + g;
    if (qb >= p.nQb) break;
    const int64_t row = ((int64_t)b * p.Hq + h) * p.nQb + qb;
    const int c = min(max(p.counts[row], 0), p.nKb);
    const int32_t* lst = p.indices + row * p.nKb;
    for (int i = lane; i < c; i += 32) {
      const int kb = lst[i];
      if (kb >= 0 && kb < p.nKb) atomicOr(&bm[g * p.words + (kb >> 5)], 1u << (kb & 31));
    }
  }
  __syncwarp();
  const int gh = p.ratio / 2;   // query blocks per 128-row half
  // the three classes of word w: both halves, half 0 only, half 1 only
  auto classes_of = [&](int w, uint32_t (&cl)[3]) {
    uint32_t h0 = 0u, h1 = 0u;
    if (w < p.words)
      for (int g = 0; g < p.ratio; ++g) (g < gh ? h0 : h1) |= bm[g * p.words + w];
    cl[0] = h0 & h1;
    cl[1] = h0 & ~h1;
    cl[2] = h1 & ~h0;
  };
  int nc[3] = {0, 0, 0};
  for (int w = lane; w < p.words; w += 32) {
    uint32_t cl[3];
    classes_of(w, cl);
    for (int c = 0; c < 3; ++c) nc[c] += __popc(cl[c]);
  }
  for (int c = 0; c < 3; ++c)
    for (int o = 16; o > 0; o >>= 1) nc[c] += __shfl_xor_sync(0xffffffffu, nc[c], o);
  const int S = p.per_step;
  const int st[3] = {(nc[0] + S - 1) / S, (nc[1] + S - 1) / S, (nc[2] + S - 1) / S};
  const int m = min(st[1], st[2]);
  // entry e of class c -> its place in the merged row
  auto out_pos = [&](int c, int e) {
    if (c == 0) return e;
    const int k = e / S;
    const int step = st[0] + (k < m ? 2 * k + (c - 1) : m + k);
    return step * S + e % S;
  };
  const int64_t srow = ((int64_t)b * p.Hq + h) * p.nSb + sb;
  int32_t* out = p.uindices + srow * p.stride;
  int running[3] = {0, 0, 0};
  for (int w0 = 0; w0 < p.words; w0 += 32) {
    const int w = w0 + lane;
    uint32_t cl[3];
    classes_of(w, cl);
    for (int c = 0; c < 3; ++c) {
      uint32_t u = cl[c];
      const int cnt = __popc(u);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int e = running[c] + incl - cnt;
      while (u) {
        const int bit = __ffs(u) - 1;
        u &= u - 1;
        int mask = 0;
        for (int g = 0; g < p.ratio; ++g) mask |= (int)((bm[g * p.words + w] >> bit) & 1u) << g;
        out[out_pos(c, e++)] = (w * 32 + bit) | (mask << kEntryGroupShift);
      }
      running[c] += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (lane == 0) {
    for (int c = 0; c < 3; ++c)
      for (int e = nc[c]; e < st[c] * S; ++e) out[out_pos(c, e)] = p.nKb;   // padding
    p.ucounts[srow] = S * (st[0] + st[1] + st[2]);
    p.uclasses[2 * srow] = st[1];
    p.uclasses[2 * srow + 1] = st[2];
  }
}

size_t merged_list_bytes(int B, int Hq, int Sq, int Skv, int block_q, int block_k) {
  if (block_q >= 256) return 0;
  const size_t rows = (size_t)B * Hq * (size_t)cdiv64(Sq, 256);
  const size_t stride = (size_t)merged_stride((int)cdiv64(Skv, block_k));
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al(rows * stride * 4) + al(rows * 4) + al(rows * 8);
}

bsa_status launch_forward(const ForwardArgs& a_in, cudaStream_t stream) {
  ForwardArgs a = a_in;
  if (a.block_q < 256) {
    // 64- and 128-row query blocks run as 256-row super-blocks (see above).
    const int ratio = 256 / a.block_q;
    const int nSb = (int)cdiv64(a.Sq, 256);
    if (a.indices) {
      char* mws = static_cast<char*>(a.workspace) + forward_chunk_bytes(a.Hq) * (size_t)cdiv64(a.B, kMaxFwdBatch);
      auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
      const size_t rows = (size_t)a.B * a.Hq * nSb;
      const int stride = merged_stride(a.nKb);
      MergeParams mp{};
      mp.indices = a.indices; mp.counts = a.counts;
      mp.uindices = reinterpret_cast<int32_t*>(mws);
      mp.ucounts = reinterpret_cast<int32_t*>(mws + al(rows * stride * 4));
      mp.uclasses = reinterpret_cast<int32_t*>(mws + al(rows * stride * 4) + al(rows * 4));
      mp.Hq = a.Hq; mp.nQb = a.nQb; mp.nKb = a.nKb; mp.nSb = nSb; mp.ratio = ratio;
      mp.words = (a.nKb + 31) / 32;
      mp.per_step = a.block_k == 64 ? 2 : 1;   // 64-key blocks: two per 128-key tile
      mp.stride = stride;
      merge_lists_kernel<<<dim3(nSb, a.Hq, a.B), 32, sizeof(uint32_t) * ratio * mp.words, stream>>>(mp);
      bsa_status st = cuda_check(cudaGetLastError(), "merge_lists_kernel launch");
      if (st != BSA_OK) return st;
      a.indices = mp.uindices;
      a.counts = mp.ucounts;
      a.classes = mp.uclasses;
      a.list_stride = stride;
      a.masked = true;
    }
    a.group_rows = a.block_q;
    a.block_q = 256;
    a.nQb = nSb;
  }
  // head dim 128 with 128-key blocks: CTA pairs (M = 256 MMAs).  64-key
  // blocks (two list entries per 128-key tile) run faster on the single-CTA
  // kernel, which skips a row's unselected 64-key halves (measured at 480p:
  // 9.0 ms against 10.1 ms); so does head dim 64.
  if (a.d == 128 && a.block_k == 128) return launch_pair<128, kPairSBufs>(a, stream);
  if (a.d == 128 && a.block_k == 64) return launch_t<128, 128, 2, 64>(a, stream);   // paired 64-key blocks
  if (a.d == 64 && a.block_k == 128) return launch_t<64, 128, 2>(a, stream);
  if (a.d == 64 && a.block_k == 64) return launch_t<64, 128, 2, 64>(a, stream);
  return set_error(BSA_ERR_UNSUPPORTED, "bsa_forward: unsupported (d, block_k)");
}

}  // namespace bsa
