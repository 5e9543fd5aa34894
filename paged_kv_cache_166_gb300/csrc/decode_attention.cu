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
//     vLLM Borrowed Virtual Memory...", section "The Custom CUDA Kernel") into a
//     ring of shared-memory stages, with the G query rows of the group
//     bulk-copied alongside the first tile of each (s, g);
//   * the block-table entries of the run are prefetched 32 at a time into shared
//     memory with cp.async, a window ahead of the loads that need them;
//   * the warp keeps an fp32 online-softmax state (running max and sum, rescaled
//     accumulator) per query head of the group.
// A (s, g) whose steps lie in one run is finished by that warp; one cut by run
// boundaries leaves one partial state per piece, and the reduce kernel merges the
// pieces in logical order with a log-sum-exp ("two-pass reduction ... numerically
// stable merge", "PagedAttention: How vLLM Borrowed Virtual Memory...", section
// "The Custom CUDA Kernel").  Cut points depend only on the context lengths and
// the warp count, so results never depend on physical block ids.
//
// fp16/bf16: every query head of the group reuses each gathered tile; scores are
// S^T[16 tokens x 8 heads] = K[16 x D] Q^T on the tensor cores (m16n8k16, fp32
// accumulate), P^T is re-laid out in registers with movmatrix, and
// O^T[D x 8] += V^T P^T on the tensor cores.  fp32: CUDA-core FMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {

constexpr int kTok = 16;                 // tokens per cache block (kernel requirement)
constexpr int kSwizzleRow = 128;         // bytes per swizzled shared-memory row
constexpr int kSubTile = kTok * kSwizzleRow;  // one swizzled [16 x 128 B] sub-tile
constexpr int kWarps = 4;                // worker warps per CTA
constexpr int kMaxSeqs = 2048;
constexpr int kMaxGroup = 8;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait before giving up
constexpr int kStatusBytes = 256;        // head of the workspace: status word + padding

struct DecodeArgs {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_ml;  // [2 * total_warps, G, 2]  (max in log2 units, sum)
  float* part_o;   // [2 * total_warps, G, D]  (unnormalised accumulator)
  int32_t* status;
  int32_t S, Hq, Hkv, G, MAXB, NB;
  int32_t total_warps;
  int32_t q_bytes;   // G * D * elt
  int32_t q_stride;  // per-stage q slot
  float scale_log2;  // scale * log2(e)
};

template <typename T, int D>
struct Shape {
  static constexpr int kElt = sizeof(T);
  static constexpr int kTileBytes = kTok * D * kElt;
  static constexpr int kSub = D * kElt / kSwizzleRow;     // sub-tiles per tile
  static constexpr int kBoxCols = kSwizzleRow / kElt;      // elements per sub-tile row
  static constexpr int kStages = 16384 / kTileBytes;       // 32 KB of K+V stages per warp
  static constexpr int kStageBytes = 2 * kTileBytes;
  static_assert(kSub * kSwizzleRow == D * kElt, "head_dim * elt must be a multiple of 128 B");
  static_assert(kStages >= 2, "pipeline needs two stages");
};

struct SmemLayout {
  uint32_t tiles, q, bars, ids, ctx, pre, scratch, total;
};

__host__ __device__ inline SmemLayout smem_layout(int tile_bytes, int stages, int q_stride,
                                                  int S) {
  SmemLayout L;
  uint32_t off = 0;
  L.tiles = off;
  off += kWarps * stages * 2 * tile_bytes;
  L.q = off;
  off += kWarps * stages * q_stride;
  off = (off + 15u) & ~15u;
  L.bars = off;
  off += kWarps * stages * 8;
  L.ids = off;
  off += kWarps * 64 * 4;
  L.ctx = off;
  off += S * 4;
  L.pre = off;
  off += (S + 1) * 4;
  off = (off + 15u) & ~15u;
  L.scratch = off;
  off += 32 * 4;
  L.total = off + 1024;  // slack for aligning the tiles to 1024 B
  return L;
}

__host__ __device__ inline SmemLayout reduce_smem_layout(int S) {
  SmemLayout L{};
  uint32_t off = 0;
  L.ctx = off;
  off += S * 4;
  L.pre = off;
  off += (S + 1) * 4;
  off = (off + 15u) & ~15u;
  L.scratch = off;
  off += 32 * 4;
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------------
// Schedule: per-sequence step counts and their prefix sums, built by every CTA.
// pre[s] = sum_{s' < s} ceil(ctx[s'] / 16) * Hkv;  pre[S] = total steps.
// ---------------------------------------------------------------------------------
__device__ void build_schedule(const int32_t* __restrict__ context_lens, int S, int MAXB, int Hkv,
                               int32_t* ctx_s, int32_t* pre, int32_t* scratch,
                               int32_t* status) {
  const int limit = MAXB * kTok;
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    int c = context_lens[s];
    if (c < 0 || c > limit) {
      if (status != nullptr && blockIdx.x == 0) atomicOr(status, PKV_DEV_BAD_CONTEXT_LEN);
      c = c < 0 ? 0 : limit;
    }
    ctx_s[s] = c;
  }
  __syncthreads();
  const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = T >> 5;
  const int chunk = (S + T - 1) / T;
  const int b0 = min(S, tid * chunk), b1 = min(S, b0 + chunk);
  int local = 0;
  for (int s = b0; s < b1; ++s) local += ((ctx_s[s] + kTok - 1) / kTok) * Hkv;
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int v = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane < nw) scratch[lane] = v;
  }
  __syncthreads();
  int run = x - local + (wid > 0 ? scratch[wid - 1] : 0);
  for (int s = b0; s < b1; ++s) {
    pre[s] = run;
    run += ((ctx_s[s] + kTok - 1) / kTok) * Hkv;
  }
  if (tid == T - 1) pre[S] = run;
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
// Tile layout in shared memory: kSub sub-tiles of [16 rows x 128 B]; the 16-byte
// chunk c of row r sits at chunk position c ^ (r & 7) (the TMA 128-byte swizzle).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int chunk16) {
  return tile + (chunk16 >> 3) * kSubTile + row * kSwizzleRow +
         (((chunk16 & 7) ^ (row & 7)) << 4);
}

template <typename T, int D>
struct MmaState {
  static constexpr int KS = D / 16;
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

  __device__ __forceinline__ void step(uint32_t ktile, uint32_t vtile, int valid,
                                       float scale_log2, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const int mi = lane >> 3, r = lane & 7;
    // S^T = K Q^T : A = K rows (tokens) x d, ldmatrix matrices
    // {tok 0-7, d lo}, {tok 8-15, d lo}, {tok 0-7, d hi}, {tok 8-15, d hi}.
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    const int tok_a = r + (mi & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      ptx::ldsm_x4(swz(ktile, tok_a, ks * 2 + (mi >> 1)), a);
      if (ks & 1) ptx::mma_16816<T>(c1, a, qb[ks][0], qb[ks][1]);
      else ptx::mma_16816<T>(c0, a, qb[ks][0], qb[ks][1]);
    }
    // c[0]: (tok gid, head 2tig)  c[1]: (gid, 2tig+1)  c[2]: (gid+8, 2tig)  c[3]: (gid+8, 2tig+1)
    float x0 = (c0[0] + c1[0]) * scale_log2, x1 = (c0[1] + c1[1]) * scale_log2;
    float x2 = (c0[2] + c1[2]) * scale_log2, x3 = (c0[3] + c1[3]) * scale_log2;
    if (valid < kTok) {
      if (gid >= valid) x0 = x1 = -INFINITY;
      if (gid + 8 >= valid) x2 = x3 = -INFINITY;
    }
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
    const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }
    // P^T as the B operand [16 tokens x 8 heads]: transpose the (tokens x heads)
    // accumulator halves in registers.
    const uint32_t pb0 = ptx::movmatrix_trans(ptx::pack2<T>(p0, p1));
    const uint32_t pb1 = ptx::movmatrix_trans(ptx::pack2<T>(p2, p3));
    // O^T += V^T P^T : A = V^T (d x tokens) via transposing ldmatrix of matrices
    // {tok 0-7, d lo}, {tok 0-7, d hi}, {tok 8-15, d lo}, {tok 8-15, d hi}.
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (valid < kTok) {  // rows past the context may hold anything, NaN included
      mlo = (2 * tig < valid ? 0x0000ffffu : 0u) | (2 * tig + 1 < valid ? 0xffff0000u : 0u);
      mhi = (2 * tig + 8 < valid ? 0x0000ffffu : 0u) | (2 * tig + 9 < valid ? 0xffff0000u : 0u);
    }
    const int tok_v = r + (mi >> 1) * 8;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a[4];
      ptx::ldsm_x4_trans(swz(vtile, tok_v, mt * 2 + (mi & 1)), a);
      a[0] &= mlo;
      a[1] &= mlo;
      a[2] &= mhi;
      a[3] &= mhi;
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

template <int D>
struct FmaState {
  static constexpr int E = D / 32;  // elements of a row per lane: d = lane + 32 * e
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
    const int chunk = d >> 2;  // 16-byte chunk of the 128-byte sub-tile row
    const uint8_t* p = tile + (chunk >> 3) * kSubTile + t * kSwizzleRow +
                       (((chunk & 7) ^ (t & 7)) << 4) + (d & 3) * 4;
    return *reinterpret_cast<const float*>(p);
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

// ---------------------------------------------------------------------------------
// Partition kernel: every warp streams its run of steps.
// ---------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32, 1)
    decode_partition_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using Sh = Shape<T, D>;
  constexpr int NS = Sh::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base_s = (raw + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (base_s - raw);
  const SmemLayout L = smem_layout(Sh::kTileBytes, NS, a.q_stride, a.S);
  int32_t* const ctx_s = reinterpret_cast<int32_t*>(base + L.ctx);
  int32_t* const pre = reinterpret_cast<int32_t*>(base + L.pre);
  build_schedule(a.context_lens, a.S, a.MAXB, a.Hkv, ctx_s, pre,
                 reinterpret_cast<int32_t*>(base + L.scratch), a.status);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kWarps + warp;
  const int total = pre[a.S];
  const int W = a.total_warps;
  const int run_len = (total + W - 1) / W;
  const int f0 = gw < W ? min(total, gw * run_len) : total;
  const int f1 = min(total, f0 + run_len);
  const int nsteps = f1 - f0;
  if (nsteps <= 0) return;

  const uint32_t tiles = base_s + L.tiles + warp * NS * Sh::kStageBytes;
  const uint32_t qslot_s = base_s + L.q + warp * NS * a.q_stride;
  const uint8_t* const qslot = base + L.q + warp * NS * a.q_stride;
  const uint32_t bars = base_s + L.bars + warp * NS * 8;
  const int32_t* const ids = reinterpret_cast<const int32_t*>(base + L.ids) + warp * 64;
  const uint32_t ids_s = base_s + L.ids + warp * 64 * 4;
  const int S = a.S, Hkv = a.Hkv, MAXB = a.MAXB;

  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < NS; ++st) ptx::mbar_init(bars + 8 * st, 1);
    ptx::fence_barrier_init();
  }
  __syncwarp();

  // Block-table prefetch: window k holds the ids of local steps [32k, 32k + 32).
  auto load_window = [&](int k) {
    const int m = 32 * k + lane;
    if (m < nsteps) {
      const Cursor c = cursor_at(pre, S, Hkv, f0 + m);
      ptx::cp_async_4(ids_s + ((k & 1) * 32 + lane) * 4,
                      a.block_tables + static_cast<int64_t>(c.s) * MAXB + c.j);
    }
    ptx::cp_async_commit();
  };
  load_window(0);
  load_window(1);
  ptx::cp_async_wait<1>();
  __syncwarp();

  const uint64_t policy = ptx::policy_evict_first();
  const int32_t rows_total = a.NB * Hkv * kTok;
  const char* const qbase = reinterpret_cast<const char*>(a.q);

  Cursor pc = cursor_at(pre, S, Hkv, f0);
  auto issue = [&](int m) {  // warp-uniform; lane 0 issues the copies of local step m
    if ((m & 31) == 0 && m > 0) {
      load_window((m >> 5) + 1);
      ptx::cp_async_wait<1>();
      __syncwarp();
    }
    if (lane == 0) {
      const int st = m % NS;
      const int id = ids[((m >> 5) & 1) * 32 + (m & 31)];
      const bool need_q = (m == 0) || (pc.j == 0);
      const uint32_t bar = bars + 8 * st;
      ptx::mbar_arrive_expect_tx(bar, Sh::kStageBytes + (need_q ? a.q_bytes : 0));
      int32_t y;
      if (static_cast<uint32_t>(id) < static_cast<uint32_t>(a.NB)) {
        y = (id * Hkv + pc.g) * kTok;
      } else {
        atomicOr(a.status, PKV_DEV_BAD_BLOCK_ID);
        y = rows_total;  // a box wholly past the end: the TMA unit fills it with zeros
      }
      const uint32_t kt = tiles + st * Sh::kStageBytes;
      const uint32_t vt = kt + Sh::kTileBytes;
#pragma unroll
      for (int c = 0; c < Sh::kSub; ++c)
        ptx::tma_load_2d(kt + c * kSubTile, &kmap, c * Sh::kBoxCols, y, bar, policy);
#pragma unroll
      for (int c = 0; c < Sh::kSub; ++c)
        ptx::tma_load_2d(vt + c * kSubTile, &vmap, c * Sh::kBoxCols, y, bar, policy);
      if (need_q) {
        const char* src =
            qbase + (static_cast<int64_t>(pc.s) * a.Hq + pc.g * a.G) * D * Sh::kElt;
        ptx::bulk_load(qslot_s + st * a.q_stride, src, a.q_bytes, bar);
      }
    }
    advance(pc, pre, S, Hkv);
  };

  const int prologue = nsteps < NS ? nsteps : NS;
  for (int m = 0; m < prologue; ++m) issue(m);

  using State = typename std::conditional<sizeof(T) == 2, MmaState<T, D>, FmaState<D>>::type;
  State st_;
  Cursor cc = cursor_at(pre, S, Hkv, f0);
  int first_j = cc.j;
  T* const out = reinterpret_cast<T*>(a.out);

  for (int n = 0; n < nsteps; ++n) {
    const int st = n % NS;
    const uint32_t parity = (n / NS) & 1;
    const bool ok = ptx::mbar_wait(bars + 8 * st, parity, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) atomicOr(a.status, PKV_DEV_WAIT_TIMEOUT);
      const int last = min(nsteps, n + NS);
      for (int k = n; k < last; ++k)
        ptx::mbar_wait(bars + 8 * (k % NS), (k / NS) & 1, kWaitLimitNs / 8);
      ptx::cp_async_wait<0>();
      return;
    }
    if (n == 0 || cc.j == 0) {
      st_.load_q(qslot + st * a.q_stride, a.G, lane);
      st_.reset();
      first_j = cc.j;
    }
    const int valid = (cc.j == cc.nb - 1) ? ctx_s[cc.s] - cc.j * kTok : kTok;
    const uint32_t kt = tiles + st * Sh::kStageBytes;
    if constexpr (sizeof(T) == 2) {
      st_.step(kt, kt + Sh::kTileBytes, valid, a.scale_log2, lane);
    } else {
      const uint8_t* ktp = base + (kt - base_s);
      st_.step(ktp, ktp + Sh::kTileBytes, valid, a.scale_log2, a.G, lane);
    }
    const bool unit_end = (cc.j == cc.nb - 1);
    if (unit_end || n == nsteps - 1) {
      st_.reduce_sums();
      if (unit_end && first_j == 0) {
        st_.write_out(out + (static_cast<int64_t>(cc.s) * a.Hq + cc.g * a.G) * D, a.G, lane);
      } else {
        const int slot = 2 * gw + (first_j == 0 ? 1 : 0);
        st_.write_partial(a.part_o + static_cast<int64_t>(slot) * a.G * D,
                          a.part_ml + static_cast<int64_t>(slot) * a.G * 2, a.G, lane);
      }
    }
    advance(cc, pre, S, Hkv);
    __syncwarp();
    if (n + NS < nsteps) issue(n + NS);
  }
  ptx::cp_async_wait<0>();
}

// ---------------------------------------------------------------------------------
// Reduce kernel: merges the pieces of every cut (s, g) in logical order and
// writes zero rows for empty contexts.  Warp w merges the (s, g) that starts in
// its run and continues past it; the pieces come from warps w, w+1, ..., w_last,
// stored at slot 2w+1 for w and slot 2w' for the later warps.
// ---------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
    decode_reduce_kernel(const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const SmemLayout L = reduce_smem_layout(a.S);
  int32_t* const ctx_s = reinterpret_cast<int32_t*>(smem_raw + L.ctx);
  int32_t* const pre = reinterpret_cast<int32_t*>(smem_raw + L.pre);
  build_schedule(a.context_lens, a.S, a.MAXB, a.Hkv, ctx_s, pre,
                 reinterpret_cast<int32_t*>(smem_raw + L.scratch), nullptr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kWarps + warp;
  const int W = a.total_warps;
  if (gw >= W) return;
  const int total = pre[a.S];
  const int run_len = (total + W - 1) / W;
  T* const out = reinterpret_cast<T*>(a.out);
  const int f0 = min(total, gw * run_len);
  const int f1 = min(total, f0 + run_len);
  if (f1 > f0) {
    const Cursor c = cursor_at(pre, a.S, a.Hkv, f1 - 1);
    const int u0 = pre[c.s] + c.g * c.nb;
    const int u1 = u0 + c.nb;
    if (u0 >= f0 && u1 > f1) {
      const int w_last = (u1 - 1) / run_len;
      T* const rows = out + (static_cast<int64_t>(c.s) * a.Hq + c.g * a.G) * D;
      for (int h = 0; h < a.G; ++h) {
        float M = -INFINITY;
        for (int w = gw; w <= w_last; ++w) {
          const int slot = w == gw ? 2 * w + 1 : 2 * w;
          M = fmaxf(M, a.part_ml[(static_cast<int64_t>(slot) * a.G + h) * 2]);
        }
        float lsum = 0.f;
        float acc[D / 32];
#pragma unroll
        for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
        for (int w = gw; w <= w_last; ++w) {
          const int64_t slot = w == gw ? 2 * w + 1 : 2 * w;
          const float* ml = a.part_ml + (slot * a.G + h) * 2;
          const float wt = exp2f(ml[0] - M);
          lsum += wt * ml[1];
          const float* po = a.part_o + (slot * a.G + h) * D;
#pragma unroll
          for (int e = 0; e < D / 32; ++e) acc[e] = fmaf(wt, po[lane + 32 * e], acc[e]);
        }
        const float inv = 1.f / lsum;
#pragma unroll
        for (int e = 0; e < D / 32; ++e)
          rows[h * D + lane + 32 * e] = ptx::from_float<T>(acc[e] * inv);
      }
    }
  }
  for (int s = gw; s < a.S; s += W) {
    if (pre[s + 1] != pre[s]) continue;
    T* const rows = out + static_cast<int64_t>(s) * a.Hq * D;
    for (int i = lane; i < a.Hq * D; i += 32) rows[i] = ptx::from_float<T>(0.f);
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
  int32_t dtype;
  cudaStream_t stream;
};

bool supported_head_dim(int32_t dtype, int32_t D) {
  if (dtype == PKV_F32) return D == 32 || D == 64 || D == 128;
  return D == 64 || D == 128 || D == 256;
}

template <typename T, int D>
int max_partition_smem() {
  using Sh = Shape<T, D>;
  return static_cast<int>(
      smem_layout(Sh::kTileBytes, Sh::kStages, kMaxGroup * D * Sh::kElt, kMaxSeqs).total);
}

template <typename T, int D>
int ensure_smem_attr() {
  // Raise the dynamic shared-memory limit once per device for this instantiation.
  static std::once_flag flags[64];
  static int results[64];
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::call_once(flags[dev], [&] {
    results[dev] = cudaFuncSetAttribute(decode_partition_kernel<T, D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        max_partition_smem<T, D>());
  });
  if (results[dev] != cudaSuccess)
    return cuda_fail(static_cast<cudaError_t>(results[dev]), "cudaFuncSetAttribute");
  return PKV_OK;
}

template <typename T, int D>
int default_warps_for() {
  // One full wave of the partition kernel: SMs x resident CTAs x warps per CTA,
  // computed once per device at the largest shared-memory footprint the kernel
  // can request, so the count never depends on the batch.
  static std::once_flag flags[64];
  static int results[64];
  int sms = 0, dev = 0;
  int rc = device_sm_count(&sms, &dev);
  if (rc != PKV_OK) return rc;
  rc = ensure_smem_attr<T, D>();
  if (rc != PKV_OK) return rc;
  std::call_once(flags[dev], [&] {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_partition_kernel<T, D>,
                                                      kWarps * 32,
                                                      max_partition_smem<T, D>()) != cudaSuccess)
      per_sm = 0;
    results[dev] = per_sm;
  });
  if (results[dev] < 1) return fail(PKV_ERR_UNSUPPORTED, "partition kernel does not fit on an SM");
  return sms * results[dev] * kWarps;
}

int default_warps(int32_t dtype, int32_t D) {
#define PKV_CASE(DT, TT, DD) \
  if (dtype == DT && D == DD) return default_warps_for<TT, DD>();
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
  return fail(PKV_ERR_UNSUPPORTED, "head_dim %d unsupported for dtype %d", D, dtype);
}

size_t workspace_bytes_for(int32_t G, int32_t D, int32_t W) {
  const size_t ml = static_cast<size_t>(2) * W * G * 2 * sizeof(float);
  const size_t po = static_cast<size_t>(2) * W * G * D * sizeof(float);
  const size_t ml_al = (ml + 255) & ~static_cast<size_t>(255);
  return kStatusBytes + ml_al + po;
}

int validate(const HostArgs& h, bool need_kernels_inputs, int* warps_out) {
  PKV_REQUIRE(element_bytes(h.dtype) != 0, PKV_ERR_DTYPE, "unknown dtype %d", h.dtype);
  PKV_REQUIRE(h.S >= 0 && h.S <= kMaxSeqs, PKV_ERR_UNSUPPORTED,
              "num_seqs %d outside [0, %d]", h.S, kMaxSeqs);
  PKV_REQUIRE(h.Hq > 0 && h.Hkv > 0 && h.Hq % h.Hkv == 0, PKV_ERR_INVALID_ARG,
              "num_q_heads %d must be a positive multiple of num_kv_heads %d", h.Hq, h.Hkv);
  const int G = h.Hq / h.Hkv;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, PKV_ERR_UNSUPPORTED,
              "query heads per KV head %d not in {1,2,4,8}", G);
  PKV_REQUIRE(supported_head_dim(h.dtype, h.D), PKV_ERR_UNSUPPORTED,
              "head_dim %d unsupported for dtype %d", h.D, h.dtype);
  PKV_REQUIRE(h.block_size == kTok, PKV_ERR_UNSUPPORTED, "block_size %d (kernels use 16)",
              h.block_size);
  PKV_REQUIRE(h.MAXB > 0, PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
  PKV_REQUIRE(static_cast<int64_t>(h.S) * h.MAXB * h.Hkv < (int64_t(1) << 31),
              PKV_ERR_UNSUPPORTED, "num_seqs * max_blocks_per_seq * num_kv_heads >= 2^31");
  PKV_REQUIRE(h.num_warps >= 0, PKV_ERR_INVALID_ARG, "negative num_warps");
  int W = h.num_warps;
  if (W == 0) {
    W = default_warps(h.dtype, h.D);
    if (W < 0) return W;
  }
  *warps_out = W;
  PKV_REQUIRE(h.workspace != nullptr && aligned(h.workspace, 256), PKV_ERR_INVALID_ARG,
              "workspace must be non-NULL and 256-byte aligned");
  PKV_REQUIRE(h.workspace_bytes >= workspace_bytes_for(G, h.D, W), PKV_ERR_INVALID_ARG,
              "workspace of %zu bytes < %zu needed", h.workspace_bytes,
              workspace_bytes_for(G, h.D, W));
  PKV_REQUIRE(h.S == 0 || (h.context_lens && h.out), PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(aligned(h.out, 16), PKV_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (need_kernels_inputs) {
    PKV_REQUIRE(h.NB > 0, PKV_ERR_INVALID_ARG, "num_blocks must be positive");
    PKV_REQUIRE(static_cast<int64_t>(h.NB) * h.Hkv * kTok < (int64_t(1) << 31),
                PKV_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * 16 >= 2^31");
    PKV_REQUIRE(h.S == 0 || (h.q && h.k_cache && h.v_cache && h.block_tables),
                PKV_ERR_INVALID_ARG, "NULL pointer");
    PKV_REQUIRE(aligned(h.q, 16) && aligned(h.k_cache, 16) && aligned(h.v_cache, 16) &&
                    aligned(h.block_tables, 4),
                PKV_ERR_INVALID_ARG, "q and caches must be 16-byte aligned");
  }
  return PKV_OK;
}

DecodeArgs device_args(const HostArgs& h, int W) {
  DecodeArgs a{};
  const int G = h.Hq / h.Hkv;
  const int elt = element_bytes(h.dtype);
  char* ws = static_cast<char*>(h.workspace);
  const size_t ml = static_cast<size_t>(2) * W * G * 2 * sizeof(float);
  const size_t ml_al = (ml + 255) & ~static_cast<size_t>(255);
  a.q = h.q;
  a.out = h.out;
  a.block_tables = h.block_tables;
  a.context_lens = h.context_lens;
  a.status = reinterpret_cast<int32_t*>(ws);
  a.part_ml = reinterpret_cast<float*>(ws + kStatusBytes);
  a.part_o = reinterpret_cast<float*>(ws + kStatusBytes + ml_al);
  a.S = h.S;
  a.Hq = h.Hq;
  a.Hkv = h.Hkv;
  a.G = G;
  a.MAXB = h.MAXB;
  a.NB = h.NB;
  a.total_warps = W;
  a.q_bytes = G * h.D * elt;
  a.q_stride = (a.q_bytes + 127) & ~127;
  a.scale_log2 = h.scale * 1.4426950408889634f;
  return a;
}

template <typename T, int D>
int launch_partition(const HostArgs& h, int W) {
  using Sh = Shape<T, D>;
  int rc = ensure_smem_attr<T, D>();
  if (rc != PKV_OK) return rc;
  const DecodeArgs a = device_args(h, W);
  CUtensorMap kmap, vmap;
  const int64_t rows = static_cast<int64_t>(h.NB) * h.Hkv * kTok;
  rc = encode_cache_map(&kmap, h.k_cache, h.dtype, rows, D, Sh::kBoxCols);
  if (rc != PKV_OK) return rc;
  rc = encode_cache_map(&vmap, h.v_cache, h.dtype, rows, D, Sh::kBoxCols);
  if (rc != PKV_OK) return rc;
  const SmemLayout L = smem_layout(Sh::kTileBytes, Sh::kStages, a.q_stride, h.S);
  const int grid = (W + kWarps - 1) / kWarps;
  decode_partition_kernel<T, D><<<grid, kWarps * 32, L.total, h.stream>>>(kmap, vmap, a);
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

template <typename T, int D>
int launch_reduce(const HostArgs& h, int W) {
  const DecodeArgs a = device_args(h, W);
  const SmemLayout L = reduce_smem_layout(h.S);
  const int grid = (W + kWarps - 1) / kWarps;
  decode_reduce_kernel<T, D><<<grid, kWarps * 32, L.total, h.stream>>>(a);
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

template <bool kPartition>
int dispatch(const HostArgs& h, int W) {
#define PKV_CASE(DT, TT, DD)                                                     \
  if (h.dtype == DT && h.D == DD)                                                \
    return kPartition ? launch_partition<TT, DD>(h, W) : launch_reduce<TT, DD>(h, W);
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

HostArgs make_args(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, int32_t MAXB, const int32_t* context_lens,
                   int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t block_size, int32_t NB,
                   float scale, void* out, void* workspace, size_t workspace_bytes,
                   int32_t num_warps, int32_t dtype, void* stream) {
  HostArgs h;
  h.q = q;
  h.k_cache = k_cache;
  h.v_cache = v_cache;
  h.block_tables = block_tables;
  h.MAXB = MAXB;
  h.context_lens = context_lens;
  h.S = S;
  h.Hq = Hq;
  h.Hkv = Hkv;
  h.D = D;
  h.block_size = block_size;
  h.NB = NB;
  h.scale = scale;
  h.out = out;
  h.workspace = workspace;
  h.workspace_bytes = workspace_bytes;
  h.num_warps = num_warps;
  h.dtype = dtype;
  h.stream = static_cast<cudaStream_t>(stream);
  return h;
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

int pkv_decode_attention_partition(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks, float scale, void* out,
                                   void* workspace, size_t workspace_bytes, int32_t num_warps,
                                   int32_t dtype, void* stream) {
  const HostArgs h = make_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                               context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, num_blocks, scale, out, workspace, workspace_bytes,
                               num_warps, dtype, stream);
  int W = 0;
  int rc = validate(h, true, &W);
  if (rc != PKV_OK) return rc;
  if (h.S == 0) return ok();
  rc = dispatch<true>(h, W);
  return rc == PKV_OK ? ok() : rc;
}

int pkv_decode_attention_reduce(const int32_t* context_lens, int32_t max_blocks_per_seq,
                                int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, void* out, void* workspace,
                                size_t workspace_bytes, int32_t num_warps, int32_t dtype,
                                void* stream) {
  const HostArgs h = make_args(nullptr, nullptr, nullptr, nullptr, max_blocks_per_seq,
                               context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, 1, 1.f, out, workspace, workspace_bytes, num_warps,
                               dtype, stream);
  int W = 0;
  int rc = validate(h, false, &W);
  if (rc != PKV_OK) return rc;
  if (h.S == 0) return ok();
  rc = dispatch<false>(h, W);
  return rc == PKV_OK ? ok() : rc;
}

int pkv_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, float scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream) {
  const HostArgs h = make_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                               context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, num_blocks, scale, out, workspace, workspace_bytes,
                               num_warps, dtype, stream);
  int W = 0;
  int rc = validate(h, true, &W);
  if (rc != PKV_OK) return rc;
  if (h.S == 0) return ok();
  rc = dispatch<true>(h, W);
  if (rc != PKV_OK) return rc;
  rc = dispatch<false>(h, W);
  return rc == PKV_OK ? ok() : rc;
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

// Device address of g_static_scratch for the current device, resolved once per
// device with that device current.
int static_scratch_address(void** ptr) {
  static std::once_flag flags[64];
  static void* addrs[64];
  static cudaError_t errs[64];
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::call_once(flags[dev], [&] {
    void* p = nullptr;
    errs[dev] = cudaGetSymbolAddress(&p, g_static_scratch);
    addrs[dev] = p;
  });
  if (errs[dev] != cudaSuccess) return cuda_fail(errs[dev], "cudaGetSymbolAddress(static scratch)");
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
  // The status word is the only part of the scratch that must start at zero.
  if (num_seqs > 0)
    PKV_CUDA(cudaMemsetAsync(scratch, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)));
  return pkv_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                              num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              num_blocks, scale, out, scratch, PKV_STATIC_SCRATCH_BYTES, W, dtype,
                              stream);
}
