// Single-token paged decode attention for sm_103a.
//
// What is computed ("PagedAttention — how vLLM stopped wasting 80% of your GPU
// memory", section "The PagedAttention kernel: computing attention over
// scattered blocks"): for sequence s and query head h of KV group g,
//   out[s,h] = softmax_p(scale * q[s,h] . K[slot(p), g]) . V[slot(p), g],  p < ctx[s],
// with slot(p) = block_table[s][p / 16] * 16 + p % 16 ("What is paged
// attention?", section "How it works").
//
// How it is scheduled.  The work of one launch is the flat list of steps
// (s, g, j) — sequence s, KV head g, logical block j < ceil(ctx[s]/16) — in
// that order.  It is cut into equal runs, one per worker warp, so every warp
// streams the same number of 16-token K/V tiles whatever the length mix.  A
// warp walks its run with its own pipeline:
//   * lane 0 issues TMA tiled loads of the step's K and V tiles (the
//     [16, head_dim] rows of one block and one KV head are contiguous in the
//     [num_blocks, num_kv_heads, 16, head_dim] layout of "PagedAttention: How
//     vLLM Borrowed Virtual Memory...", section "The Custom CUDA Kernel"; for
//     16-bit caches one 4-D box per tile lands it as two 8-row groups of
//     swizzle atoms) into a ring of shared-memory stages, with the G query rows
//     of the group bulk-copied alongside the first tile of each (s, g);
//   * the block-table entries of the run are prefetched 32 at a time into shared
//     memory with cp.async, a window ahead of the loads that need them;
//   * the stage of a step is refilled as soon as its arithmetic is done (moving
//     the tile to registers first and refilling at once measured slower: it only
//     adds requests to an already saturated memory system);
//   * the warp keeps an fp32 online-softmax state (running max and sum, rescaled
//     accumulator) per query head of the group.
// A (s, g) whose steps lie in one run is finished by that warp.  One cut by run
// boundaries leaves one partial state per piece; each piece's warp takes a ticket
// when its run ends, and the warp holding the last ticket merges the pieces in
// logical order with a log-sum-exp ("two-pass reduction ... numerically stable
// merge", "PagedAttention: How vLLM Borrowed Virtual Memory...", section "The
// Custom CUDA Kernel") — no warp ever waits for another.  Cut points depend only
// on the context lengths and the warp count, and the merge order is fixed, so
// results never depend on physical block ids or on which warp merges.
//
// fp16/bf16: every query head of the group reuses each gathered tile; scores are
// S^T[16 tokens x 8 heads] = K[16 x D] Q^T on the tensor cores (m16n8k16, fp32
// accumulate), P^T is re-laid out in registers with movmatrix, and
// O^T[D x 8] += V^T P^T on the tensor cores.  fp32: CUDA-core FMA.
//
// Block sizes 8 and 32 (16-bit caches) keep the 16-token steps: a step reads half
// of a 32-token block or two 8-token blocks, and the block-id windows hold two ids
// per step, so the schedule, the cut points and the results are those of block
// size 16.  fp8 (E4M3) and int8 caches: the same schedule and merges with 4 KB
// stages of codes (V tiles stored transposed), more warps per CTA, the codes widened
// exactly to f16 pairs by integer operations and scaled per KV head around the same
// tensor-core contractions.
//
// The kernel is launched with programmatic stream serialisation: its prologue
// (schedule, block-table prefetch) overlaps the tail of the preceding cache write
// (pkv_kv_write, or the decode step's write of each new token), and
// griddepcontrol.wait orders every K/V read after that write.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "decode_layout.h"
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

// Build-time tuning knobs (defaults are the measured best on GB300).
#ifndef PKV_WARPS_PER_CTA
#define PKV_WARPS_PER_CTA 4
#endif
// 8-bit (fp8 or int8) stages are half the size (and hold no query rows): more warps
// fit, and hide each other's latency; at head_dim 256 the register budget allows fewer.
#ifndef PKV_WARPS_PER_CTA_FP8
#define PKV_WARPS_PER_CTA_FP8 16
#endif
#ifndef PKV_WARPS_PER_CTA_FP8_WIDE
#define PKV_WARPS_PER_CTA_FP8_WIDE 8
#endif
#ifndef PKV_MAX_STAGES
#define PKV_MAX_STAGES 8
#endif
#ifndef PKV_MAX_STAGES_FP8
#define PKV_MAX_STAGES_FP8 12
#endif
// Start-up cost of a (sequence, KV head) unit in quarter steps, for group sizes
// below 4 and from 4 up (query copy, finalise, output write).
#ifndef PKV_UNIT_COST_SMALL_G
#define PKV_UNIT_COST_SMALL_G 2
#endif
#ifndef PKV_UNIT_COST_LARGE_G
#define PKV_UNIT_COST_LARGE_G 4
#endif

constexpr int kTok = 16;                 // tokens per cache block (kernel requirement)
constexpr int kSwizzleRow = 128;         // bytes per swizzled shared-memory row
constexpr int kSubTile = kTok * kSwizzleRow;  // one swizzled [16 x 128 B] sub-tile
constexpr int kWarps = PKV_WARPS_PER_CTA;     // worker warps per CTA (16/32-bit caches)
constexpr int kWarpsFp8 = PKV_WARPS_PER_CTA_FP8;  // the same for the fp8 cache, head_dim 128
constexpr int kWarpsFp8Wide = PKV_WARPS_PER_CTA_FP8_WIDE;  // ... and head_dim 256

__host__ __device__ constexpr int fp8_warps_per_cta(int D) {
  return D <= 128 ? kWarpsFp8 : kWarpsFp8Wide;
}
constexpr int kMaxStages = PKV_MAX_STAGES;    // per-warp pipeline depth limit
constexpr int kMaxStagesFp8 = PKV_MAX_STAGES_FP8;  // the same for 4 KB fp8 stages
constexpr int kMaxSeqs = 2048;
constexpr int kMaxGroup = 8;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait before giving up
constexpr int kStatusBytes = 256;        // head of the workspace: status word + padding

struct DecodeArgs {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_ml;    // [2 * total_warps, G, 2]  (max in log2 units, sum)
  float* part_o;     // [2 * total_warps, G, D]  (unnormalised accumulator)
  int32_t* tickets;  // [total_warps], zero between launches
  int32_t* status;
  const float* k_scale;  // fp8 cache: per-KV-head scales (else NULL)
  const float* v_scale;
  int32_t S, Hq, Hkv, G, MAXB, NB;
  int32_t block_size;  // 8, 16 or 32 tokens per cache block (steps are 16 tokens)
  int32_t total_warps;
  int32_t stages;    // per-warp pipeline depth
  int32_t q_bytes;   // G * D * elt
  int32_t q_stride;  // per-stage q slot
  int32_t unit_cost; // start-up cost of a unit, in quarter steps
  float scale_log2;  // scale * log2(e)
};

// Cache element tags of the 8-bit caches, fp8 (E4M3) and int8 codes with
// per-KV-head scales; q and out stay 16-bit there.
struct E4M3 {};
struct I8 {};
template <typename C>
struct CacheBytes {
  static constexpr int value = sizeof(C);
};
template <>
struct CacheBytes<E4M3> {
  static constexpr int value = 1;
};
template <>
struct CacheBytes<I8> {
  static constexpr int value = 1;
};

template <typename C, int D>
struct Shape {
  static constexpr bool kQ8 = std::is_same<C, E4M3>::value || std::is_same<C, I8>::value;
  static constexpr int kElt = CacheBytes<C>::value;
  static constexpr int kWarpsPerCta = kQ8 ? fp8_warps_per_cta(D) : kWarps;
  static constexpr bool kQRegs = kQ8;  // 8-bit: q rows straight to registers, no stage slot
  static constexpr int kTileBytes = kTok * D * kElt;
  static constexpr int kSub = D * kElt / kSwizzleRow;     // sub-tiles per tile
  static constexpr int kBoxCols = kSwizzleRow / kElt;      // elements per sub-tile row
  static constexpr int kStageBytes = 2 * kTileBytes;       // K and V tile
  // 8-bit: K in kSub boxes of [16 rows x 128 B]; V (stored [D x 16 B]) in one box.
  // 16-bit: tiles stored as groups of 8 tokens (one swizzle atom per 128 B of row,
  // side by side), so that one 4-D box moves a whole step, or a whole 8-token block.
  // fp32: kSub boxes of [16 rows x 128 B].
  static constexpr bool kGrouped = !kQ8 && kElt == 2;
  static_assert(kSub * kSwizzleRow == D * kElt, "head_dim * elt must be a multiple of 128 B");
};


// ---------------------------------------------------------------------------------
// Schedule, built by every CTA from the context lengths:
//   pre[s]  = sum_{s' < s} nb(s') * Hkv            flat step index of (s, 0, 0)
//   prew[s] = sum_{s' < s} Hkv * (4 nb(s') + c)    its cost in quarter steps
// with nb = ceil(ctx / 16) and c the unit start-up cost (0 for empty sequences).
// Warp w owns the steps whose cost position lies in [w R, (w+1) R): equal cost,
// not equal step count, so warps holding many short contexts get fewer steps.
// ---------------------------------------------------------------------------------
__device__ void build_schedule(const int32_t* __restrict__ context_lens, int S, int MAXB,
                               int block_size, int Hkv,
                               int unit_cost, int32_t* ctx_s, int32_t* pre, int32_t* prew,
                               int32_t* scratch, int32_t* status) {
  const int limit = MAXB * block_size;
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    int c = context_lens[s];
    if (c < 0 || c > limit) {
      if (blockIdx.x == 0) atomicOr(status, PKV_DEV_BAD_CONTEXT_LEN);
      c = c < 0 ? 0 : limit;
    }
    ctx_s[s] = c;
  }
  __syncthreads();
  const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = T >> 5;
  const int chunk = (S + T - 1) / T;
  const int b0 = min(S, tid * chunk), b1 = min(S, b0 + chunk);
  auto steps_of = [&](int s) { return ((ctx_s[s] + kTok - 1) / kTok) * Hkv; };
  auto cost_of = [&](int s) {
    const int nb = (ctx_s[s] + kTok - 1) / kTok;
    return nb > 0 ? Hkv * (4 * nb + unit_cost) : 0;
  };
  int local = 0, localw = 0;
  for (int s = b0; s < b1; ++s) {
    local += steps_of(s);
    localw += cost_of(s);
  }
  int x = local, xw = localw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    const int yw = __shfl_up_sync(0xffffffffu, xw, o);
    if (lane >= o) {
      x += y;
      xw += yw;
    }
  }
  if (lane == 31) {
    scratch[wid] = x;
    scratch[32 + wid] = xw;
  }
  __syncthreads();
  if (wid == 0) {
    int v = lane < nw ? scratch[lane] : 0;
    int vw = lane < nw ? scratch[32 + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      const int yw = __shfl_up_sync(0xffffffffu, vw, o);
      if (lane >= o) {
        v += y;
        vw += yw;
      }
    }
    if (lane < nw) {
      scratch[lane] = v;
      scratch[32 + lane] = vw;
    }
  }
  __syncthreads();
  int run = x - local + (wid > 0 ? scratch[wid - 1] : 0);
  int runw = xw - localw + (wid > 0 ? scratch[32 + wid - 1] : 0);
  for (int s = b0; s < b1; ++s) {
    pre[s] = run;
    prew[s] = runw;
    run += steps_of(s);
    runw += cost_of(s);
  }
  if (tid == T - 1) {
    pre[S] = run;
    prew[S] = runw;
  }
  __syncthreads();
}

// Position of flat step f in (sequence, KV head, logical block) coordinates.
struct Cursor {
  int s, g, j, nb;
};

__device__ __forceinline__ int seq_of_step(const int32_t* pre, int S, int f) {
  int lo = 0, hi = S;  // pre[lo] <= f < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= f) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ Cursor cursor_at(const int32_t* pre, int S, int Hkv, int f) {
  Cursor c;
  c.s = seq_of_step(pre, S, f);
  const int r = f - pre[c.s];
  c.nb = (pre[c.s + 1] - pre[c.s]) / Hkv;
  c.g = r / c.nb;
  c.j = r - c.g * c.nb;
  return c;
}

// Flat index of the first step whose cost position is >= P (total steps if none).
// Step j of unit g of sequence s sits at prew[s] + g (4 nb + c) + c + 4 j.
__device__ __forceinline__ int flat_at_cost(const int32_t* pre, const int32_t* prew, int S, int Hkv,
                                            int unit_cost, uint32_t P) {
  if (P >= static_cast<uint32_t>(prew[S])) return pre[S];
  int lo = 0, hi = S;  // prew[lo] <= P < prew[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<uint32_t>(prew[mid]) <= P) lo = mid; else hi = mid;
  }
  const int nb = (pre[lo + 1] - pre[lo]) / Hkv;
  const int us = 4 * nb + unit_cost;
  const int r = static_cast<int>(P - static_cast<uint32_t>(prew[lo]));
  int g = r / us;
  const int r2 = r - g * us;
  int j = r2 <= unit_cost ? 0 : (r2 - unit_cost + 3) / 4;
  if (j >= nb) {  // past this unit's last step: the next unit's first
    j = 0;
    ++g;
  }
  return pre[lo] + g * nb + j;
}

// Warp owning step j of unit (s, g) for runs of R quarter steps.
__device__ __forceinline__ int owner_of(const int32_t* pre, const int32_t* prew, int Hkv,
                                        int unit_cost, int s, int g, int j, int64_t R) {
  const int nb = (pre[s + 1] - pre[s]) / Hkv;
  const int64_t pos = prew[s] + static_cast<int64_t>(g) * (4 * nb + unit_cost) + unit_cost + 4 * j;
  return static_cast<int>(pos / R);
}

__device__ __forceinline__ void advance(Cursor& c, const int32_t* pre, int S, int Hkv) {
  if (++c.j < c.nb) return;
  c.j = 0;
  if (++c.g < Hkv) return;
  c.g = 0;
  do {
    ++c.s;
  } while (c.s < S && pre[c.s + 1] == pre[c.s]);
  if (c.s < S) c.nb = (pre[c.s + 1] - pre[c.s]) / Hkv;
}

// ---------------------------------------------------------------------------------
// Per-warp compute on one staged K/V tile.
// Tile layout in shared memory (8-bit and fp32 caches): kSub sub-tiles of
// [16 rows x 128 B]; the 16-byte chunk c of row r sits at chunk position
// c ^ (r & 7) (the TMA 128-byte swizzle).
// ---------------------------------------------------------------------------------
// Grouped tiles (16-bit caches) are instead two groups of 8 rows, each group kSub
// swizzle atoms [8 rows x 128 B] side by side (atom c holding chunks 8c..8c+7 of
// its rows).
template <int kSub, bool kGrouped = false>
__device__ __forceinline__ uint32_t tile_offset(int row, int chunk16) {
  if constexpr (kGrouped) {
    return (row >> 3) * (kSub * 8 * kSwizzleRow) + (chunk16 >> 3) * (8 * kSwizzleRow) +
           (row & 7) * kSwizzleRow + (((chunk16 & 7) ^ (row & 7)) << 4);
  } else {
    return (chunk16 >> 3) * kSubTile + row * kSwizzleRow + (((chunk16 & 7) ^ (row & 7)) << 4);
  }
}

template <typename T, int D>
struct MmaState {
  static constexpr int KS = D / 16;
  static constexpr int kSub = D * static_cast<int>(sizeof(T)) / kSwizzleRow;
  static __device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int chunk16) {
    return tile + tile_offset<kSub, true>(row, chunk16);
  }
  float o[KS][4];   // O^T[d = mt*16 + gid (+8)][h = 2*tig (+1)]
  uint32_t qb[KS][2];
  float m0, m1, l0, l1;  // heads 2*tig and 2*tig+1 (log2 units for m)

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  __device__ __forceinline__ void load_q(const uint8_t* qs, int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const T* row = reinterpret_cast<const T*>(qs) + gid * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (gid < G) {
        qb[ks][0] = *reinterpret_cast<const uint32_t*>(row + ks * 16 + 2 * tig);
        qb[ks][1] = *reinterpret_cast<const uint32_t*>(row + ks * 16 + 2 * tig + 8);
      } else {
        qb[ks][0] = qb[ks][1] = 0u;
      }
    }
  }

  // K as the A operand of S^T = K Q^T: ldmatrix matrices
  // {tok 0-7, d lo}, {tok 8-15, d lo}, {tok 0-7, d hi}, {tok 8-15, d hi} per k-step.
  static __device__ __forceinline__ void load_k(uint32_t ktile, int ks, int lane,
                                                uint32_t (&a)[4]) {
    const int mi = lane >> 3, r = lane & 7;
    ptx::ldsm_x4(swz(ktile, r + (mi & 1) * 8, ks * 2 + (mi >> 1)), a);
  }
  // V^T as the A operand of O^T += V^T P^T: transposing ldmatrix of matrices
  // {tok 0-7, d lo}, {tok 0-7, d hi}, {tok 8-15, d lo}, {tok 8-15, d hi} per m-tile.
  static __device__ __forceinline__ void load_v(uint32_t vtile, int mt, int lane,
                                                uint32_t (&a)[4]) {
    const int mi = lane >> 3, r = lane & 7;
    ptx::ldsm_x4_trans(swz(vtile, r + (mi >> 1) * 8, mt * 2 + (mi & 1)), a);
  }

  __device__ __forceinline__ void scores(const uint32_t (&kf)[KS][4], int valid,
                                         float scale_log2, int lane, float (&x)[4]) {
    const int gid = lane >> 2;
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (ks & 1) ptx::mma_16816<T>(c1, kf[ks], qb[ks][0], qb[ks][1]);
      else ptx::mma_16816<T>(c0, kf[ks], qb[ks][0], qb[ks][1]);
    }
    // x[0]: (tok gid, head 2tig)  x[1]: (gid, 2tig+1)  x[2]: (gid+8, 2tig)  x[3]: (gid+8, 2tig+1)
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = (c0[i] + c1[i]) * scale_log2;
    if (valid < kTok) {
      if (gid >= valid) x[0] = x[1] = -INFINITY;
      if (gid + 8 >= valid) x[2] = x[3] = -INFINITY;
    }
  }

  // Online-softmax update; returns P^T as the B operand [16 tokens x 8 heads].
  __device__ __forceinline__ void softmax(const float (&x)[4], uint32_t& pb0, uint32_t& pb1) {
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    const float p0 = exp2f(x[0] - mn0), p1 = exp2f(x[1] - mn1);
    const float p2 = exp2f(x[2] - mn0), p3 = exp2f(x[3] - mn1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    m0 = mn0;
    m1 = mn1;
    {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    // transpose the (tokens x heads) halves in registers
    pb0 = ptx::movmatrix_trans(ptx::pack2<T>(p0, p1));
    pb1 = ptx::movmatrix_trans(ptx::pack2<T>(p2, p3));
  }

  // Rows past the context may hold anything, NaN included: zero their V lanes.
  static __device__ __forceinline__ void mask_v(uint32_t (&a)[4], int valid, int lane) {
    const int tig = lane & 3;
    const uint32_t mlo =
        (2 * tig < valid ? 0x0000ffffu : 0u) | (2 * tig + 1 < valid ? 0xffff0000u : 0u);
    const uint32_t mhi =
        (2 * tig + 8 < valid ? 0x0000ffffu : 0u) | (2 * tig + 9 < valid ? 0xffff0000u : 0u);
    a[0] &= mlo;
    a[1] &= mlo;
    a[2] &= mhi;
    a[3] &= mhi;
  }

  // Whole step reading the tile from shared memory as it goes.
  __device__ __forceinline__ void step_smem(uint32_t ktile, uint32_t vtile, int valid,
                                            float scale_log2, int lane) {
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      load_k(ktile, ks, lane, a);
      if (ks & 1) ptx::mma_16816<T>(c1, a, qb[ks][0], qb[ks][1]);
      else ptx::mma_16816<T>(c0, a, qb[ks][0], qb[ks][1]);
    }
    const int gid = lane >> 2;
    float x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = (c0[i] + c1[i]) * scale_log2;
    if (valid < kTok) {
      if (gid >= valid) x[0] = x[1] = -INFINITY;
      if (gid + 8 >= valid) x[2] = x[3] = -INFINITY;
    }
    uint32_t pb0, pb1;
    softmax(x, pb0, pb1);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a[4];
      load_v(vtile, mt, lane, a);
      if (valid < kTok) mask_v(a, valid, lane);
      ptx::mma_16816<T>(o[mt], a, pb0, pb1);
    }
  }

  __device__ __forceinline__ void reduce_sums() {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }

  // Normalised rows of the G heads into out[s, g*G + h, :].
  __device__ __forceinline__ void write_out(T* out_rows, int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const uint32_t lo = ptx::movmatrix_trans(ptx::pack2<T>(o[mt][0] * i0, o[mt][1] * i1));
      const uint32_t hi = ptx::movmatrix_trans(ptx::pack2<T>(o[mt][2] * i0, o[mt][3] * i1));
      if (gid < G) {
        T* row = out_rows + gid * D + mt * 16 + 2 * tig;
        *reinterpret_cast<uint32_t*>(row) = lo;
        *reinterpret_cast<uint32_t*>(row + 8) = hi;
      }
    }
  }

  __device__ __forceinline__ void write_partial(float* po, float* pml, int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      if (h0 < G) {
        po[h0 * D + mt * 16 + gid] = o[mt][0];
        po[h0 * D + mt * 16 + gid + 8] = o[mt][2];
      }
      if (h1 < G) {
        po[h1 * D + mt * 16 + gid] = o[mt][1];
        po[h1 * D + mt * 16 + gid + 8] = o[mt][3];
      }
    }
    if (gid == 0) {
      if (h0 < G) { pml[h0 * 2] = m0; pml[h0 * 2 + 1] = l0; }
      if (h1 < G) { pml[h1 * 2] = m1; pml[h1 * 2 + 1] = l1; }
    }
  }
};

// 8-bit tiles (fp8 E4M3 or int8 codes).  K: [16 tokens x D bytes] in 128-byte
// swizzled sub-tiles.
// V: stored transposed, [D x 16 bytes] unswizzled, each 16-byte row holding the
// 16 tokens in the order 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15.  Operand
// fragments come from ldmatrix on bytes: a lane's 32-bit word holds 4 consecutive
// bytes of one row, widened exactly to two f16 pairs with integer operations (see
// widen), and the contractions run on the f16 tensor cores with fp32 accumulation
// (an int8 code, |c| <= 127, and an E4M3 value times 2^-8 are both exact in f16):
//   scores: the MMA's k index maps to head_dim as k = 2i, 2i+1 -> d = 4i, 4i+1
//     and k = 2i+8, 2i+9 -> d = 4i+2, 4i+3 (within each 16-wide step); q is loaded
//     in the same order, so the dot products are unchanged;
//   P.V:    a V word holds tokens 2i, 2i+1, 2i+8, 2i+9 of one head_dim row, the
//     token order in which P^T comes out of movmatrix, so P needs no reshuffle.
// q (f16 or bf16) is converted to f16; k_scale folds into the score scale and
// v_scale multiplies the accumulator when it is written.
template <typename T, typename C, int D>
struct Q8State {
  static constexpr bool kInt8 = std::is_same<C, I8>::value;
  static constexpr int KS = D / 16;
  static constexpr int kSub = D / kSwizzleRow;
  float o[KS][4];   // O^T[d = mt*16 + gid (+8)][h = 2*tig (+1)]
  uint32_t qb[KS][2];
  float m0, m1, l0, l1;
  float sl2, vs;    // score scale (log2 units, k_scale folded in), v_scale

  // int8: bytes 0-1 (widen) or 2-3 (widen_hi) of w as an exact f16 pair.  With the
  // sign bit flipped a code c reads as c + 128 in [0, 255]; under the exponent
  // byte 0x64 that is the f16 1024 + c + 128 (the f16 step is 1 on [1024, 2048)),
  // and subtracting 1152 leaves c exactly.
  static __device__ __forceinline__ uint32_t widen_i8(uint32_t w, uint32_t sel) {
    const uint32_t b = __byte_perm(w ^ 0x80808080u, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(b), "r"(0x64806480u));
    return r;
  }
  // fp8: bytes 0-1 (widen) or 2-3 (widen_hi) of w as an f16 pair holding
  // value * 2^-8: the E4M3 exponent and mantissa bits shifted left by 7 are exactly
  // the f16 bits of value * 2^-8 (subnormals included) once the sign sits in bit 15.
  // The byte permute puts each code in the low byte of its f16 and, in its sign
  // mode, the code's sign bit replicated over the high byte; after the shift by 7
  // bits 7-13 hold exponent and mantissa, bit 15 the sign, and the mask clears the
  // rest (three integer operations per f16 pair).
  static __device__ __forceinline__ uint32_t spread(uint32_t w, uint32_t sel) {
    uint32_t x;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(x) : "r"(w), "r"(sel));
    return (x << 7) & 0xbf80bf80u;
  }
  static __device__ __forceinline__ uint32_t widen(uint32_t w) {
    if constexpr (kInt8) return widen_i8(w, 0x4140);
    return spread(w, 0x9180u);
  }
  static __device__ __forceinline__ uint32_t widen_hi(uint32_t w) {
    if constexpr (kInt8) return widen_i8(w, 0x4342);
    return spread(w, 0xb3a2u);
  }
  static constexpr float kWidenScale = kInt8 ? 1.f : 256.f;

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  __device__ __forceinline__ void set_scales(float k_scale, float v_scale, float scale_log2) {
    sl2 = scale_log2 * (k_scale * kWidenScale);
    vs = v_scale * kWidenScale;
  }

  // The G query rows of the unit, read from global memory (8 bytes per lane and
  // step: head gid, elements 16 ks + 4 tig .. + 3) and converted to f16.
  __device__ __forceinline__ void load_q_rows(const T* rows, int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const T* row = rows + gid * D + 4 * tig;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (gid < G) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + ks * 16));
        const T* p = reinterpret_cast<const T*>(&u);
        qb[ks][0] = ptx::pack2<__half>(ptx::to_float(p[0]), ptx::to_float(p[1]));
        qb[ks][1] = ptx::pack2<__half>(ptx::to_float(p[2]), ptx::to_float(p[3]));
      } else {
        qb[ks][0] = qb[ks][1] = 0u;
      }
    }
  }

  __device__ __forceinline__ void step_smem(uint32_t ktile, uint32_t vtile, int valid,
                                            float /*scale_log2*/, int lane) {
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, r = lane & 7;
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    // ldmatrix of K: matrices {tok 0-7, chunk 2p}, {tok 8-15, 2p}, {0-7, 2p+1}, {8-15, 2p+1}
    const int krow = r + (mi & 1) * 8;
#pragma unroll
    for (int p = 0; p < KS / 2; ++p) {
      uint32_t w[4], a[4];
      ptx::ldsm_x4(ktile + tile_offset<kSub>(krow, 2 * p + (mi >> 1)), w);
      a[0] = widen(w[0]);
      a[1] = widen(w[1]);
      a[2] = widen_hi(w[0]);
      a[3] = widen_hi(w[1]);
      ptx::mma_16816<__half>(c0, a, qb[2 * p][0], qb[2 * p][1]);
      a[0] = widen(w[2]);
      a[1] = widen(w[3]);
      a[2] = widen_hi(w[2]);
      a[3] = widen_hi(w[3]);
      ptx::mma_16816<__half>(c1, a, qb[2 * p + 1][0], qb[2 * p + 1][1]);
    }
    float x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = (c0[i] + c1[i]) * sl2;
    if (valid < kTok) {
      if (gid >= valid) x[0] = x[1] = -INFINITY;
      if (gid + 8 >= valid) x[2] = x[3] = -INFINITY;
    }
    // online softmax, P^T as the f16 B operand
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = ptx::ex2(m0 - mn0), al1 = ptx::ex2(m1 - mn1);
    const float p0 = ptx::ex2(x[0] - mn0), p1 = ptx::ex2(x[1] - mn1);
    const float p2 = ptx::ex2(x[2] - mn0), p3 = ptx::ex2(x[3] - mn1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    m0 = mn0;
    m1 = mn1;
    // once the running maxima settle, whole steps leave them unchanged (al == 1)
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    const uint32_t pb0 = ptx::movmatrix_trans(ptx::pack2<__half>(p0, p1));
    const uint32_t pb1 = ptx::movmatrix_trans(ptx::pack2<__half>(p2, p3));
    // masks of the V lanes: a word's f16 pairs hold tokens (2 tig, 2 tig + 1) and
    // (2 tig + 8, 2 tig + 9); rows past the context may hold anything, NaN included
    const bool partial = valid < kTok;
    const uint32_t mlo =
        (2 * tig < valid ? 0x0000ffffu : 0u) | (2 * tig + 1 < valid ? 0xffff0000u : 0u);
    const uint32_t mhi =
        (2 * tig + 8 < valid ? 0x0000ffffu : 0u) | (2 * tig + 9 < valid ? 0xffff0000u : 0u);
    // ldmatrix of V^T: matrix j holds head_dim rows 32p + 8j .. 32p + 8j + 7
#pragma unroll
    for (int p = 0; p < KS / 2; ++p) {
      uint32_t w[4], a[4];
      ptx::ldsm_x4(vtile + (32 * p + 8 * mi + r) * 16, w);
      a[0] = widen(w[0]);
      a[1] = widen(w[1]);
      a[2] = widen_hi(w[0]);
      a[3] = widen_hi(w[1]);
      if (partial) {
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
      }
      ptx::mma_16816<__half>(o[2 * p], a, pb0, pb1);
      a[0] = widen(w[2]);
      a[1] = widen(w[3]);
      a[2] = widen_hi(w[2]);
      a[3] = widen_hi(w[3]);
      if (partial) {
        a[0] &= mlo;
        a[1] &= mlo;
        a[2] &= mhi;
        a[3] &= mhi;
      }
      ptx::mma_16816<__half>(o[2 * p + 1], a, pb0, pb1);
    }
  }

  __device__ __forceinline__ void reduce_sums() {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }

  __device__ __forceinline__ void write_out(T* out_rows, int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const float i0 = vs / l0, i1 = vs / l1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const uint32_t lo = ptx::movmatrix_trans(ptx::pack2<T>(o[mt][0] * i0, o[mt][1] * i1));
      const uint32_t hi = ptx::movmatrix_trans(ptx::pack2<T>(o[mt][2] * i0, o[mt][3] * i1));
      if (gid < G) {
        T* row = out_rows + gid * D + mt * 16 + 2 * tig;
        *reinterpret_cast<uint32_t*>(row) = lo;
        *reinterpret_cast<uint32_t*>(row + 8) = hi;
      }
    }
  }

  __device__ __forceinline__ void write_partial(float* po, float* pml, int G, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      if (h0 < G) {
        po[h0 * D + mt * 16 + gid] = o[mt][0] * vs;
        po[h0 * D + mt * 16 + gid + 8] = o[mt][2] * vs;
      }
      if (h1 < G) {
        po[h1 * D + mt * 16 + gid] = o[mt][1] * vs;
        po[h1 * D + mt * 16 + gid + 8] = o[mt][3] * vs;
      }
    }
    if (gid == 0) {
      if (h0 < G) { pml[h0 * 2] = m0; pml[h0 * 2 + 1] = l0; }
      if (h1 < G) { pml[h1 * 2] = m1; pml[h1 * 2 + 1] = l1; }
    }
  }
};

template <int D>
struct FmaState {
  static constexpr int E = D / 32;  // elements of a row per lane: d = lane + 32 * e
  static constexpr int kSub = D * 4 / kSwizzleRow;
  float qv[kMaxGroup][E];
  float acc[kMaxGroup][E];
  float m[kMaxGroup], l[kMaxGroup];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
    }
  }

  __device__ __forceinline__ void load_q(const uint8_t* qs, int G, int lane) {
    const float* q = reinterpret_cast<const float*>(qs);
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h)
#pragma unroll
      for (int e = 0; e < E; ++e) qv[h][e] = h < G ? q[h * D + lane + 32 * e] : 0.f;
  }

  static __device__ __forceinline__ float at(const uint8_t* tile, int t, int d) {
    const int chunk = d >> 2;  // 16-byte chunk of the 128-byte row
    return *reinterpret_cast<const float*>(tile + tile_offset<kSub>(t, chunk) +
                                           (d & 3) * 4);
  }

  __device__ __forceinline__ void step(const uint8_t* kt, const uint8_t* vt, int valid,
                                       float scale_log2, int G, int lane) {
    float kv[kTok][E];
#pragma unroll
    for (int t = 0; t < kTok; ++t)
#pragma unroll
      for (int e = 0; e < E; ++e) kv[t][e] = at(kt, t, lane + 32 * e);
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h >= G) break;
      float sc[kTok];
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) part = fmaf(qv[h][e], kv[t][e], part);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        sc[t] = t < valid ? part * scale_log2 : -INFINITY;
        mx = fmaxf(mx, sc[t]);
      }
      const float mn = fmaxf(m[h], mx);
      const float al = exp2f(m[h] - mn);
      float ps = 0.f;
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        sc[t] = exp2f(sc[t] - mn);
        ps += sc[t];
      }
      l[h] = l[h] * al + ps;
      m[h] = mn;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        float a = acc[h][e] * al;
#pragma unroll
        for (int t = 0; t < kTok; ++t)
          if (t < valid) a = fmaf(sc[t], at(vt, t, lane + 32 * e), a);
        acc[h][e] = a;
      }
    }
  }

  __device__ __forceinline__ void reduce_sums() {}

  __device__ __forceinline__ void write_out(float* out_rows, int G, int lane) {
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h >= G) break;
      const float inv = 1.f / l[h];
#pragma unroll
      for (int e = 0; e < E; ++e) out_rows[h * D + lane + 32 * e] = acc[h][e] * inv;
    }
  }

  __device__ __forceinline__ void write_partial(float* po, float* pml, int G, int lane) {
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h >= G) break;
#pragma unroll
      for (int e = 0; e < E; ++e) po[h * D + lane + 32 * e] = acc[h][e];
      if (lane == 0) {
        pml[h * 2] = m[h];
        pml[h * 2 + 1] = l[h];
      }
    }
  }
};

// Partial-state slot of warp w's piece of a cut (s, g): 2w+1 if the (s, g) starts
// inside w's run (w is its first warp), else 2w.
__device__ __forceinline__ int64_t piece_slot(int w, int first_warp) {
  return w == first_warp ? 2 * static_cast<int64_t>(w) + 1 : 2 * static_cast<int64_t>(w);
}

// Log-sum-exp merge of the pieces of (s, g) held by warps w0..w1, in that order:
// M = max_i m_i;  out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
// The warp's lanes split the G heads and, within a head, the head_dim; the lanes
// of one head share the max over pieces, and piece loads are issued two at a
// time so the merge costs a few L2 round trips, not one per value.
template <typename T, int D, int G>
__device__ void merge_pieces_g(const DecodeArgs& a, int s, int g, int w0, int w1, int lane) {
  constexpr int LPH = 32 / G;          // lanes per head
  constexpr int E = D / LPH;           // contiguous elements of the row per lane
  const int h = lane / LPH, sub = lane % LPH;
  float M = -INFINITY;
  for (int w = w0 + sub; w <= w1; w += LPH)
    M = fmaxf(M, __ldcg(a.part_ml + (piece_slot(w, w0) * G + h) * 2));
#pragma unroll
  for (int off = 1; off < LPH; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float lsum = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 2
  for (int w = w0; w <= w1; ++w) {
    const int64_t slot = piece_slot(w, w0);
    const float* ml = a.part_ml + (slot * G + h) * 2;
    const float* po = a.part_o + (slot * G + h) * D + sub * E;
    const float wt = exp2f(__ldcg(ml) - M);
    lsum = fmaf(wt, __ldcg(ml + 1), lsum);
    if constexpr (E % 4 == 0) {
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(po + e));
        acc[e] = fmaf(wt, v.x, acc[e]);
        acc[e + 1] = fmaf(wt, v.y, acc[e + 1]);
        acc[e + 2] = fmaf(wt, v.z, acc[e + 2]);
        acc[e + 3] = fmaf(wt, v.w, acc[e + 3]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(wt, __ldcg(po + e), acc[e]);
    }
  }
  const float inv = 1.f / lsum;
  T* const row = reinterpret_cast<T*>(a.out) + (static_cast<int64_t>(s) * a.Hq + g * G + h) * D +
                 sub * E;
#pragma unroll
  for (int e = 0; e < E; ++e) row[e] = ptx::from_float<T>(acc[e] * inv);
}

template <typename T, int D>
__device__ void merge_pieces(const DecodeArgs& a, int s, int g, int w0, int w1, int lane) {
  switch (a.G) {
    case 1: merge_pieces_g<T, D, 1>(a, s, g, w0, w1, lane); break;
    case 2: merge_pieces_g<T, D, 2>(a, s, g, w0, w1, lane); break;
    case 4: merge_pieces_g<T, D, 4>(a, s, g, w0, w1, lane); break;
    default: merge_pieces_g<T, D, 8>(a, s, g, w0, w1, lane); break;
  }
}

// A cut (s, g) whose piece this warp finished: merged by the last piece to finish.
struct CutUnit {
  int s, g, w0, w1;
};

// The merge of up to two cuts of two pieces each (the common case at the end of a
// run), with every load of both issued before any is used: one L2 round trip
// instead of two per cut.  Same operations in the same order as merge_pieces_g, so
// the same bits.
template <typename T, int D, int G>
__device__ void merge_pairs_g(const DecodeArgs& a, const CutUnit* u, int n, int lane) {
  constexpr int LPH = 32 / G;
  constexpr int E = D / LPH;
  constexpr int KU = E <= 16 ? 2 : 1;  // cuts in flight at once (register budget)
  const int h = lane / LPH, sub = lane % LPH;
  for (int k0 = 0; k0 < n; k0 += KU) {
    float m[KU][2], l[KU][2], o[KU][2][E];
#pragma unroll
    for (int k = 0; k < KU; ++k) {
      if (k0 + k < n) {
        const CutUnit& c = u[k0 + k];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const int64_t slot = piece_slot(c.w0 + p, c.w0);
          const float* ml = a.part_ml + (slot * G + h) * 2;
          const float* po = a.part_o + (slot * G + h) * D + sub * E;
          m[k][p] = __ldcg(ml);
          l[k][p] = __ldcg(ml + 1);
          if constexpr (E % 4 == 0) {
#pragma unroll
            for (int e = 0; e < E; e += 4) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(po + e));
              o[k][p][e] = v.x;
              o[k][p][e + 1] = v.y;
              o[k][p][e + 2] = v.z;
              o[k][p][e + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) o[k][p][e] = __ldcg(po + e);
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < KU; ++k) {
      if (k0 + k < n) {
        const CutUnit& c = u[k0 + k];
        const float M = fmaxf(m[k][0], m[k][1]);
        float lsum = 0.f;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const float wt = exp2f(m[k][p] - M);
          lsum = fmaf(wt, l[k][p], lsum);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(wt, o[k][p][e], acc[e]);
        }
        const float inv = 1.f / lsum;
        T* const row = reinterpret_cast<T*>(a.out) +
                       (static_cast<int64_t>(c.s) * a.Hq + c.g * G + h) * D + sub * E;
#pragma unroll
        for (int e = 0; e < E; ++e) row[e] = ptx::from_float<T>(acc[e] * inv);
      }
    }
  }
}

template <typename T, int D>
__device__ void merge_pairs(const DecodeArgs& a, const CutUnit* u, int n, int lane) {
  switch (a.G) {
    case 1: merge_pairs_g<T, D, 1>(a, u, n, lane); break;
    case 2: merge_pairs_g<T, D, 2>(a, u, n, lane); break;
    case 4: merge_pairs_g<T, D, 4>(a, u, n, lane); break;
    default: merge_pairs_g<T, D, 8>(a, u, n, lane); break;
  }
}

// ---------------------------------------------------------------------------------
// The decode kernel: one persistent pass of every worker warp over its run.
// ---------------------------------------------------------------------------------
// kBlk: 16 for caches of 16-token blocks; 0 for 8- or 32-token blocks (the size
// then comes from the arguments).
template <typename T, typename C, int D, int kBlk>
__global__ void __launch_bounds__(Shape<C, D>::kWarpsPerCta * 32, 1)
    decode_attention_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using Sh = Shape<C, D>;
  static_assert(Sh::kGrouped || kBlk == kTok, "8- and 32-token blocks need a 16-bit cache");
  constexpr int kIdStride = kBlk == kTok ? 1 : 2;  // block ids per step in the id windows
  const int NS = a.stages;
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
    // The block tables are read a window at a time once the schedule is known:
    // start pulling this CTA's slice of them into L2 now (16-byte aligned interior).
    {
      const uintptr_t t0 = reinterpret_cast<uintptr_t>(a.block_tables);
      const uintptr_t t1 = t0 + static_cast<uintptr_t>(a.S) * a.MAXB * sizeof(int32_t);
      const uintptr_t lo = (t0 + 15) & ~uintptr_t(15), hi = t1 & ~uintptr_t(15);
      if (hi > lo) {
        const uintptr_t slice = ((hi - lo) / gridDim.x + 16) & ~uintptr_t(15);
        const uintptr_t b0 = lo + slice * blockIdx.x;
        if (b0 < hi) {
          const uintptr_t b1 = b0 + slice < hi ? b0 + slice : hi;
          ptx::prefetch_l2(reinterpret_cast<const void*>(b0), static_cast<uint32_t>(b1 - b0));
        }
      }
    }
  }
  // Words 1..3 of the status area record the layout (warps, group, head_dim) of the
  // last launch; a workspace reused under another layout holds stale tickets, which
  // is reported rather than silently mis-merged.  Read now, checked once the
  // schedule is built, so the loads overlap it.
  int32_t sig_w = 0, sig_g = 0, sig_d = 0;
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    sig_w = __ldcg(a.status + 1);
    sig_g = __ldcg(a.status + 2);
    sig_d = __ldcg(a.status + 3);
  }
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base_s = (raw + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (base_s - raw);
  const SmemLayout L = smem_layout(Sh::kStageBytes, NS, a.q_stride, a.S, Sh::kWarpsPerCta);
  int32_t* const ctx_s = reinterpret_cast<int32_t*>(base + L.ctx);
  int32_t* const pre = reinterpret_cast<int32_t*>(base + L.pre);
  int32_t* const prew = reinterpret_cast<int32_t*>(base + L.prew);
  build_schedule(a.context_lens, a.S, a.MAXB, a.block_size, a.Hkv, a.unit_cost, ctx_s, pre, prew,
                 reinterpret_cast<int32_t*>(base + L.scratch), a.status);
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    if (sig_w != 0 && (sig_w != a.total_warps || sig_g != a.G || sig_d != D))
      atomicOr(a.status, PKV_DEV_WORKSPACE_MISMATCH);
    a.status[1] = a.total_warps;
    a.status[2] = a.G;
    a.status[3] = D;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * Sh::kWarpsPerCta + warp;
  const int S = a.S, Hkv = a.Hkv, MAXB = a.MAXB;
  const int total = pre[S];
  const int W = a.total_warps;
  const int UC = a.unit_cost;
  // Runs of R quarter steps; R is at least the widest gap between consecutive
  // step positions (4 + UC), so every warp between the first and the last owner
  // of a unit holds a piece of it.
  // (cost positions stay below 2^31, checked on the host: 32-bit arithmetic holds)
  const uint32_t R = max((static_cast<uint32_t>(prew[S]) + static_cast<uint32_t>(W) - 1u) /
                             static_cast<uint32_t>(W),
                         static_cast<uint32_t>(4 + UC));
  const int64_t R64 = R;
  T* const out = reinterpret_cast<T*>(a.out);

  // Rows of empty contexts are zero.
  if (gw < W) {
    for (int s = gw; s < S; s += W) {
      if (pre[s + 1] != pre[s]) continue;
      T* const rows = out + static_cast<int64_t>(s) * a.Hq * D;
      for (int i = lane; i < a.Hq * D; i += 32) rows[i] = ptx::from_float<T>(0.f);
    }
  }
  // the run's bounds, searched by the two half-warps at once
  int fb = total;
  if (gw < W) {
    const uint32_t P = static_cast<uint32_t>(gw + (lane >= 16 ? 1 : 0)) * R;
    fb = flat_at_cost(pre, prew, S, Hkv, UC, P);
  }
  const int f0 = __shfl_sync(0xffffffffu, fb, 0);
  const int f1 = __shfl_sync(0xffffffffu, fb, 16);
  const int nsteps = f1 - f0;
  if (nsteps <= 0) return;

  const uint32_t tiles = base_s + L.tiles + warp * NS * Sh::kStageBytes;
  const uint32_t qslot_s = base_s + L.q + warp * NS * a.q_stride;
  const uint8_t* const qslot = base + L.q + warp * NS * a.q_stride;
  const uint32_t bars = base_s + L.bars + warp * NS * 8;
  const int32_t* const ids = reinterpret_cast<const int32_t*>(base + L.ids) + warp * 64 * kIdStride;
  const uint32_t ids_s = base_s + L.ids + warp * 64 * kIdStride * 4;
  const int Bsz = kBlk ? kBlk : a.block_size;

  if (lane == 0) {
    for (int st = 0; st < NS; ++st) ptx::mbar_init(bars + 8 * st, 1);
    ptx::fence_barrier_init();
  }
  __syncwarp();

  // Block-table prefetch: window k holds, for local steps [32k, 32k + 32), the
  // block ids each 16-token step reads: table[s][j] (block size 16), table[s][j/2]
  // (32), or table[s][2j] and table[s][2j+1] (8; the second only if the context
  // reaches it).
  // (copies of one lane's entry of window k, for the step at cursor c)
  auto put_window = [&](int k, const Cursor& c) {
    const int32_t* row = a.block_tables + static_cast<int64_t>(c.s) * MAXB;
    const uint32_t slot = ids_s + (((k & 1) * 32 + lane) * kIdStride) * 4;
    if (kBlk == kTok || Bsz == 16) {
      ptx::cp_async_4(slot, row + c.j);
    } else if (Bsz == 32) {
      ptx::cp_async_4(slot, row + (c.j >> 1));
    } else {
      ptx::cp_async_4(slot, row + 2 * c.j);
      if (2 * c.j + 1 < (ctx_s[c.s] + 7) / 8) ptx::cp_async_4(slot + 4, row + 2 * c.j + 1);
    }
  };
  auto load_window = [&](int k) {
    const int m = 32 * k + lane;
    if (m < nsteps) put_window(k, cursor_at(pre, S, Hkv, f0 + m));
    ptx::cp_async_commit();
  };
  // The cursors of the run's first 32 steps, one a lane (clamped to the run's last
  // step): the first table window and the ring fill below both start from them.
  const Cursor lc = cursor_at(pre, S, Hkv, min(f0 + lane, total - 1));
  if (lane < nsteps) put_window(0, lc);
  ptx::cp_async_commit();
  load_window(1);
  ptx::cp_async_wait<1>();
  __syncwarp();

  // Every K/V read below comes after the preceding grid (the cache write of the
  // new tokens) has completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const uint64_t policy = ptx::policy_evict_first();
  const int32_t rows_total = a.NB * Hkv * Bsz;
  const char* const qbase = reinterpret_cast<const char*>(a.q);

  // Copies of step (s, g, j) into stage `stage` (executed by one lane): the K and V
  // rows of the step's 16 tokens, and the group's query rows when need_q.
  auto issue_copies = [&](int stage, int s, int g, int j, int id0, int id1, bool need_q) {
    // block size 8: the step's second block exists unless the context ends in the first
    const bool second = kBlk != kTok && Bsz == 8 && j * kTok + 8 < ctx_s[s];
    const uint32_t bar = bars + 8 * stage;
    const uint32_t kt = tiles + stage * Sh::kStageBytes;
    const uint32_t vt = kt + Sh::kTileBytes;
    auto row_of = [&](int id, int within) -> int32_t {
      if (static_cast<uint32_t>(id) < static_cast<uint32_t>(a.NB))
        return (id * Hkv + g) * Bsz + within;
      atomicOr(a.status, PKV_DEV_BAD_BLOCK_ID);
      return rows_total;  // a box wholly past the end: the TMA unit fills it with zeros
    };
    const int32_t extra = need_q ? a.q_bytes : 0;
    if constexpr (Sh::kGrouped) {
      // 8-row groups of the cache: a 16-token step is one box of two groups, an
      // 8-token block one box of one group (the step's second block in group 1)
      if (kBlk != kTok && Bsz == 8) {
        ptx::mbar_arrive_expect_tx(bar, (second ? Sh::kStageBytes : Sh::kStageBytes / 2) +
                                            extra);
        const int32_t g0 = row_of(id0, 0) >> 3;
        ptx::tma_load_4d(kt, &kmap, 0, 0, 0, g0, bar, policy);
        ptx::tma_load_4d(vt, &vmap, 0, 0, 0, g0, bar, policy);
        if (second) {
          const int32_t g1 = row_of(id1, 0) >> 3;
          ptx::tma_load_4d(kt + Sh::kTileBytes / 2, &kmap, 0, 0, 0, g1, bar, policy);
          ptx::tma_load_4d(vt + Sh::kTileBytes / 2, &vmap, 0, 0, 0, g1, bar, policy);
        }
      } else {
        ptx::mbar_arrive_expect_tx(bar, Sh::kStageBytes + extra);
        const int32_t g = row_of(id0, (kBlk != kTok && Bsz == 32) ? (j & 1) * kTok : 0) >> 3;
        ptx::tma_load_4d(kt, &kmap, 0, 0, 0, g, bar, policy);
        ptx::tma_load_4d(vt, &vmap, 0, 0, 0, g, bar, policy);
      }
    } else {
      // 8-bit and fp32 caches (16-token blocks only): kSub boxes of [16 rows x 128 B]
      // for K; V likewise, or one box of the transposed 8-bit tile
      ptx::mbar_arrive_expect_tx(bar, Sh::kStageBytes + extra);
      const int32_t y = row_of(id0, 0);
#pragma unroll
      for (int c = 0; c < Sh::kSub; ++c)
        ptx::tma_load_2d(kt + c * kSubTile, &kmap, c * Sh::kBoxCols, y, bar, policy);
      if constexpr (Sh::kQ8) {
        ptx::tma_load_2d(vt, &vmap, 0, (y / kTok) * (D / 8), bar, policy);
      } else {
#pragma unroll
        for (int c = 0; c < Sh::kSub; ++c)
          ptx::tma_load_2d(vt + c * kSubTile, &vmap, c * Sh::kBoxCols, y, bar, policy);
      }
    }
    if (need_q) {
      const char* src = qbase + (static_cast<int64_t>(s) * a.Hq + g * a.G) * D * sizeof(T);
      ptx::bulk_load(qslot_s + stage * a.q_stride, src, a.q_bytes, bar);
    }
  };

  Cursor pc{0, 0, 0, 1};
  int p_stage = 0;
  auto issue = [&](int m) {  // warp-uniform; lane 0 issues the copies of local step m
    if ((m & 31) == 0 && m > 0) {
      load_window((m >> 5) + 1);
      ptx::cp_async_wait<1>();
      __syncwarp();
    }
    if (lane == 0) {
      const int w = (((m >> 5) & 1) * 32 + (m & 31)) * kIdStride;
      issue_copies(p_stage, pc.s, pc.g, pc.j, ids[w], kIdStride == 2 ? ids[w + 1] : -1,
                   !Sh::kQRegs && ((m == 0) || (pc.j == 0)));
    }
    if (++p_stage == NS) p_stage = 0;
    advance(pc, pre, S, Hkv);
  };

  // Fill the ring: lanes 0..NS-1 issue the first NS steps at once, one step each;
  // lane NS finds the step after them, where the producer continues.
  const int prologue = nsteps < NS ? nsteps : NS;
  if (lane < prologue) {
    issue_copies(lane, lc.s, lc.g, lc.j, ids[kIdStride * lane],
                 kIdStride == 2 ? ids[kIdStride * lane + 1] : -1,
                 !Sh::kQRegs && ((lane == 0) || (lc.j == 0)));
  }
  __syncwarp();
  p_stage = prologue == NS ? 0 : prologue;
  pc.s = __shfl_sync(0xffffffffu, lc.s, prologue);
  pc.g = __shfl_sync(0xffffffffu, lc.g, prologue);
  pc.j = __shfl_sync(0xffffffffu, lc.j, prologue);
  pc.nb = __shfl_sync(0xffffffffu, lc.nb, prologue);

  using State = typename std::conditional<
      Sh::kQ8, Q8State<T, C, D>,
      typename std::conditional<sizeof(T) == 2, MmaState<T, D>, FmaState<D>>::type>::type;
  State st_;
  // The consumer starts at lane 0's cursor.  (The 16-bit instantiations search for
  // it again: with the broadcast the compiler allocates their streaming loop
  // differently, which measured 4% slower.)
  Cursor cc;
  if constexpr (Sh::kQ8) {
    cc.s = __shfl_sync(0xffffffffu, lc.s, 0);
    cc.g = __shfl_sync(0xffffffffu, lc.g, 0);
    cc.j = __shfl_sync(0xffffffffu, lc.j, 0);
    cc.nb = __shfl_sync(0xffffffffu, lc.nb, 0);
  } else {
    cc = cursor_at(pre, S, Hkv, f0);
  }
  int first_j = cc.j;
  CutUnit cut[2];
  int ncut = 0;
  int c_stage = 0;
  uint32_t parity = 0;

  for (int n = 0; n < nsteps; ++n) {
    const uint32_t bar = bars + 8 * c_stage;
    const bool ok = ptx::mbar_wait(bar, parity, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) atomicOr(a.status, PKV_DEV_WAIT_TIMEOUT);
      // give the copies already issued a bounded chance to land, then leave
      int st = c_stage;
      uint32_t ph = parity;
      for (int k = n; k < min(nsteps, n + NS); ++k) {
        ptx::mbar_wait(bars + 8 * st, ph, kWaitLimitNs / 8);
        if (++st == NS) { st = 0; ph ^= 1u; }
      }
      ptx::cp_async_wait<0>();
      return;
    }
    if (n == 0 || cc.j == 0) {
      if constexpr (Sh::kQ8) {
        st_.load_q_rows(reinterpret_cast<const T*>(a.q) +
                            (static_cast<int64_t>(cc.s) * a.Hq + cc.g * a.G) * D,
                        a.G, lane);
      } else {
        st_.load_q(qslot + c_stage * a.q_stride, a.G, lane);
      }
      st_.reset();
      if constexpr (Sh::kQ8) st_.set_scales(a.k_scale[cc.g], a.v_scale[cc.g], a.scale_log2);
      first_j = cc.j;
    }
    const int valid = (cc.j == cc.nb - 1) ? ctx_s[cc.s] - cc.j * kTok : kTok;
    const uint32_t kt = tiles + c_stage * Sh::kStageBytes;
    if constexpr (sizeof(T) == 2) {
      st_.step_smem(kt, kt + Sh::kTileBytes, valid, a.scale_log2, lane);
    } else {
      const uint8_t* ktp = base + (kt - base_s);
      st_.step(ktp, ktp + Sh::kTileBytes, valid, a.scale_log2, a.G, lane);
    }
    // the stage is refilled once its arithmetic is done
    __syncwarp();
    if (n + NS < nsteps) issue(n + NS);
    if (++c_stage == NS) { c_stage = 0; parity ^= 1u; }
    const bool unit_end = (cc.j == cc.nb - 1);
    if (unit_end || n == nsteps - 1) {
      st_.reduce_sums();
      if (unit_end && first_j == 0) {
        st_.write_out(out + (static_cast<int64_t>(cc.s) * a.Hq + cc.g * a.G) * D, a.G, lane);
      } else {
        const int slot = 2 * gw + (first_j == 0 ? 1 : 0);
        st_.write_partial(a.part_o + static_cast<int64_t>(slot) * a.G * D,
                          a.part_ml + static_cast<int64_t>(slot) * a.G * 2, a.G, lane);
        cut[ncut++] = CutUnit{cc.s, cc.g, owner_of(pre, prew, Hkv, UC, cc.s, cc.g, 0, R64),
                              owner_of(pre, prew, Hkv, UC, cc.s, cc.g, cc.nb - 1, R64)};
      }
    }
    advance(cc, pre, S, Hkv);
  }
  ptx::cp_async_wait<0>();

  // Tickets of the cut (s, g) this warp took part in; the last piece merges.
  if (ncut > 0) {
    __threadfence();
    __syncwarp();
    int t0 = 0, t1 = 0;
    if (lane == 0) {
      t0 = atomicAdd(a.tickets + cut[0].w0, 1);
      if (ncut > 1) t1 = atomicAdd(a.tickets + cut[1].w0, 1);
    }
    t0 = __shfl_sync(0xffffffffu, t0, 0);
    t1 = __shfl_sync(0xffffffffu, t1, 0);
    // the cuts this warp finished last; those of two pieces are merged together
    CutUnit mine[2], pairs[2];
    int nmine = 0, npairs = 0;
    for (int i = 0; i < ncut; ++i) {
      if ((i == 0 ? t0 : t1) == cut[i].w1 - cut[i].w0) {
        mine[nmine++] = cut[i];
        if (cut[i].w1 == cut[i].w0 + 1) pairs[npairs++] = cut[i];
      }
    }
    if (nmine > 0) {
      __threadfence();
      if (npairs > 0) merge_pairs<T, D>(a, pairs, npairs, lane);
      for (int i = 0; i < nmine; ++i) {
        const CutUnit& u = mine[i];
        if (u.w1 != u.w0 + 1) merge_pieces<T, D>(a, u.s, u.g, u.w0, u.w1, lane);
        if (lane == 0) a.tickets[u.w0] = 0;  // ready for the next launch
      }
    }
  }
}

// ---------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------
namespace {

struct HostArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int32_t MAXB;
  const int32_t* context_lens;
  int32_t S, Hq, Hkv, D, block_size, NB;
  float scale;
  void* out;
  void* workspace;
  size_t workspace_bytes;
  int32_t num_warps;
  int32_t dtype;  // of q and out (and of the caches unless 8-bit)
  cudaStream_t stream;
  int32_t codes = 0;  // 8-bit caches with per-KV-head scales: PKV_FP8_E4M3 or PKV_INT8
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
};

bool supported_head_dim(int32_t dtype, int32_t D) {
  if (dtype == PKV_F32) return D == 32 || D == 64 || D == 128;
  if (dtype == PKV_FP8_E4M3 || dtype == PKV_INT8) return D == 128 || D == 256;
  return D == 64 || D == 128 || D == 256;
}

// Opt-in shared memory per block of the current device (cached per device).
int device_smem_optin(int* bytes) {
  static std::once_flag flags[64];
  static int values[64];
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::call_once(flags[dev], [&] {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      v = 0;
    values[dev] = v;
  });
  if (values[dev] <= 0) return fail(PKV_ERR_CUDA, "could not query shared memory of device %d", dev);
  *bytes = values[dev];
  return PKV_OK;
}

template <typename T, typename C, int D, int kBlk>
int ensure_smem_attr() {
  // Raise the dynamic shared-memory limit once per device for this instantiation.
  static std::once_flag flags[64];
  static int results[64];
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int optin = 0;
  int rc = device_smem_optin(&optin);
  if (rc != PKV_OK) return rc;
  std::call_once(flags[dev], [&] {
    results[dev] = cudaFuncSetAttribute(decode_attention_kernel<T, C, D, kBlk>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  });
  if (results[dev] != cudaSuccess)
    return cuda_fail(static_cast<cudaError_t>(results[dev]), "cudaFuncSetAttribute");
  return PKV_OK;
}

// One CTA per SM (the kernel sizes its pipeline to fill the SM's shared memory),
// so the default warp count is SMs x warps per CTA.  dtype PKV_FP8_E4M3 or PKV_INT8
// stands for attention over that 8-bit cache.
int default_warps(int32_t dtype, int32_t D) {
  if (!supported_head_dim(dtype, D))
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d unsupported for dtype %d", D, dtype);
  int sms = 0, dev = 0;
  int rc = device_sm_count(&sms, &dev);
  if (rc != PKV_OK) return rc;
  const bool q8 = dtype == PKV_FP8_E4M3 || dtype == PKV_INT8;
  return sms * (q8 ? fp8_warps_per_cta(D) : kWarps);
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WorkspaceLayout {
  size_t tickets, ml, o, total;
};

WorkspaceLayout workspace_layout(int32_t G, int32_t D, int32_t W) {
  WorkspaceLayout L;
  L.tickets = kStatusBytes;
  L.ml = L.tickets + round256(static_cast<size_t>(W) * sizeof(int32_t));
  L.o = L.ml + round256(static_cast<size_t>(2) * W * G * 2 * sizeof(float));
  L.total = L.o + static_cast<size_t>(2) * W * G * D * sizeof(float);
  return L;
}

size_t workspace_bytes_for(int32_t G, int32_t D, int32_t W) {
  return workspace_layout(G, D, W).total;
}

int validate(const HostArgs& h, int* warps_out) {
  PKV_REQUIRE(element_bytes(h.dtype) != 0, PKV_ERR_DTYPE, "unknown dtype %d", h.dtype);
  if (h.codes != 0) {
    PKV_REQUIRE(h.dtype == PKV_F16 || h.dtype == PKV_BF16, PKV_ERR_DTYPE,
                "q dtype %d: attention over an 8-bit cache takes f16 or bf16 q", h.dtype);
    PKV_REQUIRE(h.D == 128 || h.D == 256, PKV_ERR_UNSUPPORTED,
                "head_dim %d unsupported for an 8-bit cache (128 or 256)", h.D);
    PKV_REQUIRE(h.S == 0 || (h.k_scale && h.v_scale), PKV_ERR_INVALID_ARG,
                "NULL k_scale / v_scale");
    PKV_REQUIRE(static_cast<int64_t>(h.NB) * h.Hkv * h.D < (int64_t(1) << 31),
                PKV_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * head_dim >= 2^31");
  } else {
    PKV_REQUIRE(h.dtype != PKV_FP8_E4M3 && h.dtype != PKV_INT8, PKV_ERR_DTYPE,
                "8-bit caches are read by pkv_decode_attention_fp8 / _int8");
  }
  PKV_REQUIRE(h.S >= 0 && h.S <= kMaxSeqs, PKV_ERR_UNSUPPORTED,
              "num_seqs %d outside [0, %d]", h.S, kMaxSeqs);
  PKV_REQUIRE(h.Hq > 0 && h.Hkv > 0 && h.Hq % h.Hkv == 0, PKV_ERR_INVALID_ARG,
              "num_q_heads %d must be a positive multiple of num_kv_heads %d", h.Hq, h.Hkv);
  const int G = h.Hq / h.Hkv;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, PKV_ERR_UNSUPPORTED,
              "query heads per KV head %d not in {1,2,4,8}", G);
  PKV_REQUIRE(supported_head_dim(h.dtype, h.D), PKV_ERR_UNSUPPORTED,
              "head_dim %d unsupported for dtype %d", h.D, h.dtype);
  PKV_REQUIRE(h.block_size == 8 || h.block_size == 16 || h.block_size == 32,
              PKV_ERR_UNSUPPORTED, "block_size %d not in {8, 16, 32}", h.block_size);
  PKV_REQUIRE(h.block_size == kTok || (h.codes == 0 && h.dtype != PKV_F32),
              PKV_ERR_UNSUPPORTED, "block_size %d needs an f16 or bf16 cache", h.block_size);
  PKV_REQUIRE(h.MAXB > 0, PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
  PKV_REQUIRE(static_cast<int64_t>(h.S) * h.MAXB * h.Hkv < (int64_t(1) << 31),
              PKV_ERR_UNSUPPORTED, "num_seqs * max_blocks_per_seq * num_kv_heads >= 2^31");
  PKV_REQUIRE(h.num_warps >= 0, PKV_ERR_INVALID_ARG, "negative num_warps");
  int W = h.num_warps;
  if (W == 0) {
    W = default_warps(h.codes != 0 ? h.codes : h.dtype, h.D);
    if (W < 0) return W;
  }
  *warps_out = W;
  PKV_REQUIRE(h.workspace != nullptr && aligned(h.workspace, 256), PKV_ERR_INVALID_ARG,
              "workspace must be non-NULL and 256-byte aligned");
  PKV_REQUIRE(h.workspace_bytes >= workspace_bytes_for(G, h.D, W), PKV_ERR_INVALID_ARG,
              "workspace of %zu bytes < %zu needed", h.workspace_bytes,
              workspace_bytes_for(G, h.D, W));
  PKV_REQUIRE(h.NB > 0, PKV_ERR_INVALID_ARG, "num_blocks must be positive");
  PKV_REQUIRE(static_cast<int64_t>(h.NB) * h.Hkv * h.block_size * 4 < (int64_t(1) << 31),
              PKV_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * block_size * 4 >= 2^31");
  PKV_REQUIRE(static_cast<int64_t>(h.S) * h.MAXB * h.Hkv * 4 +
                      static_cast<int64_t>(h.S) * h.Hkv * 8 < (int64_t(1) << 31),
              PKV_ERR_UNSUPPORTED, "schedule cost exceeds 2^31 quarter steps");
  PKV_REQUIRE(h.S == 0 || (h.q && h.k_cache && h.v_cache && h.block_tables && h.context_lens &&
                           h.out),
              PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(aligned(h.q, 16) && aligned(h.k_cache, 16) && aligned(h.v_cache, 16) &&
                  aligned(h.out, 16) && aligned(h.block_tables, 4),
              PKV_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned");

  return PKV_OK;
}

DecodeArgs device_args(const HostArgs& h, int W) {
  DecodeArgs a{};
  const int G = h.Hq / h.Hkv;
  const int elt = element_bytes(h.dtype);
  char* ws = static_cast<char*>(h.workspace);
  const WorkspaceLayout WL = workspace_layout(G, h.D, W);
  a.q = h.q;
  a.out = h.out;
  a.block_tables = h.block_tables;
  a.context_lens = h.context_lens;
  a.status = reinterpret_cast<int32_t*>(ws);
  a.tickets = reinterpret_cast<int32_t*>(ws + WL.tickets);
  a.part_ml = reinterpret_cast<float*>(ws + WL.ml);
  a.part_o = reinterpret_cast<float*>(ws + WL.o);
  a.S = h.S;
  a.Hq = h.Hq;
  a.Hkv = h.Hkv;
  a.G = G;
  a.MAXB = h.MAXB;
  a.NB = h.NB;
  a.block_size = h.block_size;
  a.total_warps = W;
  a.q_bytes = G * h.D * elt;
  a.q_stride = (a.q_bytes + 127) & ~127;
  a.unit_cost = G >= 4 ? PKV_UNIT_COST_LARGE_G : PKV_UNIT_COST_SMALL_G;
  a.scale_log2 = h.scale * 1.4426950408889634f;
  a.k_scale = h.k_scale;
  a.v_scale = h.v_scale;
  return a;
}

template <typename T, typename C, int D, int kBlk>
int launch_decode(const HostArgs& h, int W) {
  using Sh = Shape<C, D>;
  int rc = ensure_smem_attr<T, C, D, kBlk>();
  if (rc != PKV_OK) return rc;
  int optin = 0;
  rc = device_smem_optin(&optin);
  if (rc != PKV_OK) return rc;
  DecodeArgs a = device_args(h, W);
  if constexpr (Sh::kQRegs) a.q_stride = 0;  // q rows are read straight into registers
  // Deepest pipeline that fits the SM's shared memory.
  const uint32_t fixed =
      smem_layout(Sh::kStageBytes, 0, a.q_stride, h.S, Sh::kWarpsPerCta).total;
  const uint32_t per_stage = Sh::kWarpsPerCta * (Sh::kStageBytes + a.q_stride + 8);
  int stages = optin > static_cast<int>(fixed) ? static_cast<int>((optin - fixed) / per_stage) : 0;
  const int max_stages = Sh::kQ8 ? kMaxStagesFp8 : kMaxStages;
  stages = stages > max_stages ? max_stages : stages;
  PKV_REQUIRE(stages >= 2, PKV_ERR_UNSUPPORTED, "pipeline does not fit in shared memory");
  a.stages = stages;
  const SmemLayout L =
      smem_layout(Sh::kStageBytes, stages, a.q_stride, h.S, Sh::kWarpsPerCta);
  // an access past its boundary faults the launch: refuse the launch instead
  PKV_REQUIRE(smem_layout_aligned(L, Sh::kStageBytes, a.q_stride), PKV_ERR_UNSUPPORTED,
              "shared-memory layout misaligned (%d sequences)", h.S);
  CUtensorMap kmap, vmap;
  const int64_t rows = static_cast<int64_t>(h.NB) * h.Hkv * h.block_size;
  if constexpr (Sh::kQ8) {
    // K: [rows, D] bytes, boxes of 16 rows x 128 B, swizzled.  V: each transposed
    // [D x 16 B] tile is 16 D contiguous bytes, viewed as D/8 rows of 128 B so that
    // one unswizzled box of D/8 rows moves it (the bytes land in the same order).
    rc = encode_map_2d(&kmap, h.k_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, D,
                       Sh::kBoxCols, kTok, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != PKV_OK) return rc;
    rc = encode_map_2d(&vmap, h.v_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                       static_cast<int64_t>(h.NB) * h.Hkv * (D / 8), kSwizzleRow, kSwizzleRow,
                       D / 8, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != PKV_OK) return rc;
  } else if constexpr (Sh::kGrouped) {
    // [rows, D] viewed as (column in a 128-byte chunk, row in an 8-row group, chunk,
    // group); a box is two groups (a 16-token step) or one (an 8-token block)
    const CUtensorMapDataType ty =
        h.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int64_t dims[4] = {Sh::kBoxCols, 8, Sh::kSub, rows / 8};
    const int64_t strides[3] = {static_cast<int64_t>(D) * 2, kSwizzleRow,
                                8 * static_cast<int64_t>(D) * 2};
    const int32_t box[4] = {Sh::kBoxCols, 8, Sh::kSub, h.block_size == 8 ? 1 : 2};
    rc = encode_map_4d(&kmap, h.k_cache, ty, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != PKV_OK) return rc;
    rc = encode_map_4d(&vmap, h.v_cache, ty, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != PKV_OK) return rc;
  } else {
    // fp32: [rows, D], boxes of 16 rows x 128 B
    rc = encode_cache_map(&kmap, h.k_cache, h.dtype, rows, D, Sh::kBoxCols, kTok);
    if (rc != PKV_OK) return rc;
    rc = encode_cache_map(&vmap, h.v_cache, h.dtype, rows, D, Sh::kBoxCols, kTok);
    if (rc != PKV_OK) return rc;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((W + Sh::kWarpsPerCta - 1) / Sh::kWarpsPerCta);
  cfg.blockDim = dim3(Sh::kWarpsPerCta * 32);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = h.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  PKV_CUDA(cudaLaunchKernelEx(&cfg, decode_attention_kernel<T, C, D, kBlk>, kmap, vmap, a));
  return PKV_OK;
}

int dispatch(const HostArgs& h, int W) {
  if (h.codes != 0) {
#define PKV_CASE8(CT, DT, TT, DD) \
  if (h.dtype == DT && h.D == DD) return launch_decode<TT, CT, DD, kTok>(h, W);
    if (h.codes == PKV_FP8_E4M3) {
      PKV_CASE8(E4M3, PKV_BF16, __nv_bfloat16, 128)
      PKV_CASE8(E4M3, PKV_BF16, __nv_bfloat16, 256)
      PKV_CASE8(E4M3, PKV_F16, __half, 128)
      PKV_CASE8(E4M3, PKV_F16, __half, 256)
    } else {
      PKV_CASE8(I8, PKV_BF16, __nv_bfloat16, 128)
      PKV_CASE8(I8, PKV_BF16, __nv_bfloat16, 256)
      PKV_CASE8(I8, PKV_F16, __half, 128)
      PKV_CASE8(I8, PKV_F16, __half, 256)
    }
#undef PKV_CASE8
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d unsupported for an 8-bit cache", h.D);
  }
  if (h.block_size != kTok) {
#define PKV_CASEB(DT, TT, DD) \
  if (h.dtype == DT && h.D == DD) return launch_decode<TT, TT, DD, 0>(h, W);
    PKV_CASEB(PKV_BF16, __nv_bfloat16, 64)
    PKV_CASEB(PKV_BF16, __nv_bfloat16, 128)
    PKV_CASEB(PKV_BF16, __nv_bfloat16, 256)
    PKV_CASEB(PKV_F16, __half, 64)
    PKV_CASEB(PKV_F16, __half, 128)
    PKV_CASEB(PKV_F16, __half, 256)
#undef PKV_CASEB
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d needs an f16 or bf16 cache", h.block_size);
  }
#define PKV_CASE(DT, TT, DD) \
  if (h.dtype == DT && h.D == DD) return launch_decode<TT, TT, DD, kTok>(h, W);
  PKV_CASE(PKV_BF16, __nv_bfloat16, 64)
  PKV_CASE(PKV_BF16, __nv_bfloat16, 128)
  PKV_CASE(PKV_BF16, __nv_bfloat16, 256)
  PKV_CASE(PKV_F16, __half, 64)
  PKV_CASE(PKV_F16, __half, 128)
  PKV_CASE(PKV_F16, __half, 256)
  PKV_CASE(PKV_F32, float, 32)
  PKV_CASE(PKV_F32, float, 64)
  PKV_CASE(PKV_F32, float, 128)
#undef PKV_CASE
  return fail(PKV_ERR_UNSUPPORTED, "head_dim %d unsupported for dtype %d", h.D, h.dtype);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_decode_default_warps(int32_t head_dim, int32_t dtype, int32_t* num_warps) {
  PKV_REQUIRE(num_warps != nullptr, PKV_ERR_INVALID_ARG, "num_warps is NULL");
  PKV_REQUIRE(element_bytes(dtype) != 0, PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  const int W = default_warps(dtype, head_dim);
  if (W < 0) return W;
  *num_warps = W;
  return ok();
}

int pkv_decode_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t dtype, int32_t num_warps, size_t* bytes) {
  PKV_REQUIRE(bytes != nullptr, PKV_ERR_INVALID_ARG, "bytes is NULL");
  PKV_REQUIRE(element_bytes(dtype) != 0, PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  PKV_REQUIRE(num_q_heads > 0 && num_kv_heads > 0 && num_q_heads % num_kv_heads == 0,
              PKV_ERR_INVALID_ARG, "bad head counts %d / %d", num_q_heads, num_kv_heads);
  PKV_REQUIRE(supported_head_dim(dtype, head_dim), PKV_ERR_UNSUPPORTED,
              "head_dim %d unsupported for dtype %d", head_dim, dtype);
  PKV_REQUIRE(num_warps >= 0, PKV_ERR_INVALID_ARG, "negative num_warps");
  int W = num_warps;
  if (W == 0) {
    W = default_warps(dtype, head_dim);
    if (W < 0) return W;
  }
  *bytes = workspace_bytes_for(num_q_heads / num_kv_heads, head_dim, W);
  return ok();
}

namespace {
HostArgs host_args(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                   const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                   float scale, void* out, void* workspace, size_t workspace_bytes,
                   int32_t num_warps, int32_t dtype, void* stream) {
  HostArgs h;
  h.q = q;
  h.k_cache = k_cache;
  h.v_cache = v_cache;
  h.block_tables = block_tables;
  h.MAXB = max_blocks_per_seq;
  h.context_lens = context_lens;
  h.S = num_seqs;
  h.Hq = num_q_heads;
  h.Hkv = num_kv_heads;
  h.D = head_dim;
  h.block_size = block_size;
  h.NB = num_blocks;
  h.scale = scale;
  h.out = out;
  h.workspace = workspace;
  h.workspace_bytes = workspace_bytes;
  h.num_warps = num_warps;
  h.dtype = dtype;
  h.stream = static_cast<cudaStream_t>(stream);
  return h;
}

int decode_entry(const HostArgs& h) {
  int W = 0;
  int rc = validate(h, &W);
  if (rc != PKV_OK) return rc;
  if (h.S == 0) return ok();
  rc = dispatch(h, W);
  return rc == PKV_OK ? ok() : rc;
}
}  // namespace

int pkv_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, float scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream) {
  return decode_entry(host_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                block_size, num_blocks, scale, out, workspace, workspace_bytes,
                                num_warps, dtype, stream));
}

int pkv_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int32_t num_blocks, float scale, void* out, void* workspace,
                    size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream) {
  // Validate the attention arguments first, so that a refused call writes nothing.
  const HostArgs h = host_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                               context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, num_blocks, scale, out, workspace, workspace_bytes,
                               num_warps, dtype, stream);
  int W = 0;
  int rc = validate(h, &W);
  if (rc != PKV_OK) return rc;
  if (num_seqs == 0) return ok();
  rc = launch_decode_append(k_new, v_new, block_tables, max_blocks_per_seq, context_lens,
                            num_seqs, k_cache, v_cache, num_blocks, num_kv_heads, block_size,
                            head_dim, dtype, stream);
  if (rc != PKV_OK) return rc;
  rc = dispatch(h, W);
  return rc == PKV_OK ? ok() : rc;
}

namespace {
int decode_q8_entry(int32_t codes, const void* q, const void* k_cache, const void* v_cache,
                    const float* k_scale, const float* v_scale, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t num_blocks, float scale, void* out,
                    void* workspace, size_t workspace_bytes, int32_t num_warps, int32_t dtype,
                    void* stream) {
  HostArgs h = host_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         scale, out, workspace, workspace_bytes, num_warps, dtype, stream);
  h.codes = codes;
  h.k_scale = k_scale;
  h.v_scale = v_scale;
  return decode_entry(h);
}

int decode_step_q8_entry(int32_t codes, const void* q, const void* k_new, const void* v_new,
                         void* k_cache, void* v_cache, const float* k_scale,
                         const float* v_scale, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                         void* out, void* workspace, size_t workspace_bytes, int32_t num_warps,
                         int32_t dtype, void* stream) {
  HostArgs h = host_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         scale, out, workspace, workspace_bytes, num_warps, dtype, stream);
  h.codes = codes;
  h.k_scale = k_scale;
  h.v_scale = v_scale;
  int W = 0;
  int rc = validate(h, &W);
  if (rc != PKV_OK) return rc;
  if (num_seqs == 0) return ok();
  rc = launch_kv_write_q8(k_new, v_new, nullptr, block_tables, max_blocks_per_seq, context_lens,
                          num_seqs, k_cache, v_cache, k_scale, v_scale, num_blocks, num_kv_heads,
                          head_dim, dtype, codes, stream);
  if (rc != PKV_OK) return rc;
  rc = dispatch(h, W);
  return rc == PKV_OK ? ok() : rc;
}
}  // namespace

int pkv_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks, float scale, void* out, void* workspace,
                             size_t workspace_bytes, int32_t num_warps, int32_t dtype,
                             void* stream) {
  return decode_q8_entry(PKV_FP8_E4M3, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                         max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, scale, out, workspace,
                         workspace_bytes, num_warps, dtype, stream);
}

int pkv_decode_attention_int8(const void* q, const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks, float scale, void* out, void* workspace,
                              size_t workspace_bytes, int32_t num_warps, int32_t dtype,
                              void* stream) {
  return decode_q8_entry(PKV_INT8, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                         max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, scale, out, workspace,
                         workspace_bytes, num_warps, dtype, stream);
}

int pkv_decode_step_fp8(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const float* k_scale, const float* v_scale,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t num_blocks, float scale, void* out, void* workspace,
                        size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream) {
  return decode_step_q8_entry(PKV_FP8_E4M3, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                              block_tables, max_blocks_per_seq, context_lens, num_seqs,
                              num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                              out, workspace, workspace_bytes, num_warps, dtype, stream);
}

int pkv_decode_step_int8(const void* q, const void* k_new, const void* v_new, void* k_cache,
                         void* v_cache, const float* k_scale, const float* v_scale,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, float scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream) {
  return decode_step_q8_entry(PKV_INT8, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                              block_tables, max_blocks_per_seq, context_lens, num_seqs,
                              num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                              out, workspace, workspace_bytes, num_warps, dtype, stream);
}

int pkv_decode_status(void* workspace, int32_t* status, void* stream) {
  PKV_REQUIRE(workspace && status, PKV_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  PKV_CUDA(cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s));
  PKV_CUDA(cudaMemsetAsync(workspace, 0, sizeof(v), s));
  PKV_CUDA(cudaStreamSynchronize(s));
  *status = v;
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory: the partial states
// live in a fixed array of the library's device image instead of a caller
// workspace.  The host only ever passes the array's device address, resolved per
// device with cudaGetSymbolAddress; the array's name in host code is a host-side
// stand-in and is never handed to a kernel.
// ---------------------------------------------------------------------------------
namespace pkv {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch for the current device, resolved with that
// device current and remembered once it succeeds (a failed lookup is retried on
// the next call rather than remembered).
int static_scratch_address(void** ptr) {
  static std::mutex mu;
  static void* addrs[64];
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (addrs[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no sticky error behind for the caller's next call
      return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                       "cudaGetSymbolAddress(static scratch)");
    }
    addrs[dev] = p;
  }
  *ptr = addrs[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_decode_attention_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float scale, void* out, int32_t num_warps, int32_t dtype, void* stream) {
  PKV_REQUIRE(element_bytes(dtype) != 0, PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  PKV_REQUIRE(num_q_heads > 0 && num_kv_heads > 0 && num_q_heads % num_kv_heads == 0,
              PKV_ERR_INVALID_ARG, "bad head counts %d / %d", num_q_heads, num_kv_heads);
  PKV_REQUIRE(supported_head_dim(dtype, head_dim), PKV_ERR_UNSUPPORTED,
              "head_dim %d unsupported for dtype %d", head_dim, dtype);
  PKV_REQUIRE(num_warps >= 0, PKV_ERR_INVALID_ARG, "negative num_warps");
  int W = num_warps;
  if (W == 0) {
    W = default_warps(dtype, head_dim);
    if (W < 0) return W;
  }
  const size_t need = workspace_bytes_for(num_q_heads / num_kv_heads, head_dim, W);
  PKV_REQUIRE(need <= PKV_STATIC_SCRATCH_BYTES, PKV_ERR_UNSUPPORTED,
              "this launch needs %zu bytes of scratch but the static scratch holds %u bytes; "
              "pass a smaller num_warps or use pkv_decode_attention with a workspace",
              need, PKV_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  int rc = static_scratch_address(&scratch);
  if (rc != PKV_OK) return rc;
  // Every argument is checked before anything is queued, so a refused call leaves
  // the shared array (and everything else) untouched.
  const HostArgs h = host_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                               context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, num_blocks, scale, out, scratch,
                               PKV_STATIC_SCRATCH_BYTES, W, dtype, stream);
  int W_checked = 0;
  rc = validate(h, &W_checked);
  if (rc != PKV_OK) return rc;
  if (num_seqs == 0) return ok();
  // The status word and the merge tickets are the parts of the scratch that must
  // start at zero; the partial states are always written before they are read.
  PKV_CUDA(cudaMemsetAsync(scratch, 0, workspace_layout(num_q_heads / num_kv_heads, head_dim, W).ml,
                           static_cast<cudaStream_t>(stream)));
  rc = dispatch(h, W_checked);
  return rc == PKV_OK ? ok() : rc;
}
