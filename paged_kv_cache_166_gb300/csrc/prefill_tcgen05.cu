// Paged (chunked) prefill attention on the 5th-generation tensor cores (sm_103a).
//
// What is computed is pkv_prefill_attention's definition ("PagedAttention: How
// vLLM Borrowed Virtual Memory to Unlock GPU Serving at Scale", section "Walking
// Through the Lifecycle", Prefill): query row q0 + i of sequence s sits at
// position p = t - c + i and, for query head h of KV group g = h / G, attends to
// every position j <= p read through the block table.
//
// How.  A unit is a tile of 128 rows of one (sequence, KV head) — row R is query
// R / G, head g*G + R % G — against the keys 0 .. p_max of its last row, taken
// in KV tiles of 128 keys (16, 8 or 4 cache blocks of 8, 16 or 32 tokens).  Per
// KV tile j:
//   S_j = Q K_j^T    tcgen05 MMA, M = 128 rows, N = 128 keys, K = head_dim:
//                    Q and K_j K-major in 128-byte-swizzled shared memory,
//                    S_j in tensor memory (two buffers).  A K or V tile is 16
//                    groups of 8 keys; each group holds one 1024-byte swizzle
//                    atom (8 rows x 128 B) per 64-column chunk of head_dim, side
//                    by side, so that a cache block (BS / 8 groups, every chunk)
//                    arrives as one 4-D TMA box whose axes are reordered on the
//                    way in (column, row, chunk, group);
//   softmax          two threads per row (its tensor-memory lane), one per half
//                    of the keys: causal mask (keys past the row score -inf),
//                    the row max (three-input max) agreed through shared memory,
//                    P_j = exp2(S_j - m) (base 2; the exponents of a key pair
//                    formed by one packed f32x2 FMA, rounded to f16 and raised
//                    by one f16x2 ex2) in the input type (f16: that pair as it
//                    is; bf16: widened and rounded) and stored into tensor memory
//                    (two buffers; row r in lane r, keys 2c and 2c + 1 packed in
//                    column c), the row sum in fp32 (f16 halves added by
//                    mixed-precision adds, or packed f32x2 adds);
//   O += P_j V_j     tcgen05 MMA with A = P_j read from tensor memory, N =
//                    head_dim, K = 128 keys: V_j MN-major in shared memory (rows
//                    of keys, head_dim contiguous), O accumulating in tensor
//                    memory over the unit's KV tiles.
// Keeping P out of shared memory leaves the shared-memory bandwidth to the
// operand reads of the MMAs and the TMA writes of K and V, which bound the kernel.
// The reference m of a row is its running max, moved only when the max grows by
// more than 2^8: then the row's threads scale their halves of O (tensor memory)
// and the sum by exp2(m_old - m_new) between two P.V products.  In between P may
// exceed 1 (by at most 2^8), which the output's final division absorbs: the
// result is softmax(S) V whatever the reference.
// Warp roles (12 warps): 11 = TMA producer of the query tiles (a 3-D map of q; two
// buffers, so the next unit's tile is in place before the current one ends);
// 0 = TMA producer of the K blocks of each KV tile and 10 of the V blocks
// (through the block table); 1 = MMA issuer (the whole warp, one elected lane
// issuing) and owner of the tensor memory; 2..9 = softmax and epilogue (row
// 32 * (warp % 4) + lane, key and head_dim half (warp - 2) / 4).  K and V have rings of their own: a K stage is
// free again once S_j is computed, a V stage once P_j V_j is.  Hand-offs are
// mbarriers: TMA transaction bytes, tcgen05 commits and thread arrivals.  The MMA
// issuer runs one stream over all KV tiles of the CTA, S_{j+1} ahead of P_j V_j,
// across unit boundaries too, so the tensor cores work on S while row threads
// process the tile before.
// One CTA per SM, persistent: the units of all sequences, in order, are cut into
// contiguous runs of equal cost (KV tiles + 1 per unit), one per CTA.  Every
// wait is bounded; a wait that runs out sets PKV_DEV_WAIT_TIMEOUT and the CTA
// drains its copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "prefill_common.cuh"
#include "ptx.cuh"

namespace pkv {
namespace {

// 32-byte global store (address 32-byte aligned), evict-first in L2, not kept in L1.
__device__ __forceinline__ void st_global_v8_hint(void* ptr, const uint32_t (&v)[8],
                                                  uint64_t policy) {
  asm volatile(
      "st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;"
      ::"l"(ptr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
        "r"(v[7]), "l"(policy)
      : "memory");
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (a0, a1) * s + (c, c), two lanes of one packed fp32 instruction.
__device__ __forceinline__ void fma2(float a0, float a1, float s, float c, float& d0, float& d1) {
  uint64_t a, b, e, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(b) : "f"(s));
  asm("mov.b64 %0, {%1, %1};" : "=l"(e) : "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(e));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}
// (s0, s1) += (x0, x1), one packed fp32 instruction.
__device__ __forceinline__ void add2(float& s0, float& s1, float x0, float x1) {
  uint64_t a, b, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(x0), "f"(x1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(d));
}
// s + each half of an f16 pair, each half widened exactly (mixed-precision adds).
__device__ __forceinline__ void add_f16x2(float& s0, float& s1, uint32_t x) {
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.f16 %0, l, %0;\n\t"
      "add.rn.f32.f16 %1, h, %1;\n\t}"
      : "+f"(s0), "+f"(s1) : "r"(x));
}

constexpr int kTcRows = 128;          // rows of a unit = tensor-memory lanes = MMA M
constexpr int kTcKeys = 128;          // keys of a KV tile = N of S = K of P.V
constexpr int kTcRowWarps = 8;        // softmax warps 2 .. 9
constexpr int kTcVWarp = 2 + kTcRowWarps;  // V producer
constexpr int kTcQWarp = 3 + kTcRowWarps;  // query-tile producer
constexpr int kTcWarps = 4 + kTcRowWarps;
constexpr int kTcHalfKeys = kTcKeys / 2;
// A warp may read and write only the tensor-memory lanes of its own quarter
// (warp % 4).  Row warp w (2 .. 9) serves lanes 32 (w % 4) .. + 31 and half
// (w - 2) / 4 of the keys, so each quarter has exactly one warp per half.
static_assert(kTcRowWarps == 8 && kTcRows == 4 * 32,
              "two row warps per tensor-memory lane quarter, one per half of the keys");
constexpr float kTcRescale = 8.f;     // log2 of the growth of the row max that moves m
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcChunk = 128 * 128;   // one [128 rows x 128 B] swizzled column chunk

// mbarriers (8 bytes each), then the tensor-memory base and the CTA's schedule
enum {
  kBarKFull = 0,     // [4] K stage landed (TMA bytes)
  kBarKEmpty = 4,    // [4] K stage consumed (commit after S_j)
  kBarVFull = 8,     // [4] V stage landed
  kBarVEmpty = 12,   // [4] V stage consumed (commit after P_j V_j)
  kBarQFull = 16,    // [2] query tile landed
  kBarQEmpty = 18,   // [2] query tile consumed (commit after the unit's last S_j)
  kBarSFull = 20,    // [2] S_j in tensor memory (commit)
  kBarSEmpty = 22,   // [2] S_j read by the row warps
  kBarPFull = 24,    // [2] P_j in tensor memory (row warps)
  kBarPvDone = 26,   // [2] P_j V_j done: P_j's buffer free (commit)
  kBarOEmpty = 28,   // the unit's O read out by the row warps
  kBarDrain = 29,    // every MMA of the CTA done (final commit)
  kNumBars = 30
};
constexpr uint32_t kSlotOff = 8 * kNumBars;          // tensor-memory base address
constexpr uint32_t kSchedOff = kSlotOff + 8;         // TcSched (8-byte aligned)
constexpr uint32_t kDeadOff = kSchedOff + 32;        // [4] give-up bits of the row-warp pairs
constexpr uint32_t kBarArea = 512;

template <typename T, int D>
struct TcShape {
  static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  static constexpr int kChunks = D * 2 / 128;         // 128-byte column chunks of a row
  static constexpr int kTile = kTcRows * D * 2;       // Q, K or V tile
  static constexpr uint32_t kGroup = kChunks * 1024;  // 8 keys of a K or V tile, every chunk
  static constexpr int kKStages = D == 128 ? 2 : 3;   // K ring (freed as soon as S_j is done)
  static constexpr int kVStages = D == 128 ? 3 : 4;   // V ring
  static constexpr uint32_t kQOff = 0;                // two query tiles
  static constexpr uint32_t kKOff = 2 * kTile;
  static constexpr uint32_t kVOff = kKOff + kKStages * kTile;
  static constexpr uint32_t kBarOff = kVOff + kVStages * kTile;
  static constexpr uint32_t kXchOff = kBarOff + kBarArea;  // [2 halves][128 rows] floats
  static constexpr uint32_t kBytes = kXchOff + 2 * kTcRows * 4 + 1024;  // + alignment slack
  static_assert(kDeadOff + 16 <= kBarArea, "barrier area");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSCol = 0;                // S[b]: columns 128 b ..
  static constexpr uint32_t kOCol = 2 * kTcKeys;      // O: columns 256 .. 256 + D - 1
  static constexpr uint32_t kPCol = 384;              // P[b]: columns 384 + 64 b .. (packed pairs)
  static constexpr uint32_t kIdQK = ptx::idesc_f16(kTcRows, kTcKeys, kBf16, false);
  static constexpr uint32_t kIdPV = ptx::idesc_f16(kTcRows, D, kBf16, true);
  static constexpr int kHalfD = D / 2;                // O columns of a row thread
  static_assert(kOCol + D <= kPCol && kPCol + 2 * kTcKeys / 2 <= kTmemCols, "tensor memory");
  static_assert(kChunks * 64 == D, "head_dim 64 or 128");
};

struct TcSched {
  int32_t s, g, tile, pad;
  long long P;   // cost before the unit (s, g, tile)
  long long hi;  // the CTA's units are those with P < hi
};

// log2 of the group size (G is 1, 2, 4 or 8, checked on the host): rows R of a unit
// are query R >> gshift, head R & (G - 1).
__device__ __forceinline__ int tc_gshift(const PrefillArgs& a) { return __ffs(a.G) - 1; }

__device__ __forceinline__ int tc_tiles(const PrefillArgs& a, int c) {
  return (c * a.G + kTcRows - 1) / kTcRows;
}

// KV tiles a unit reads: keys 0 .. p of its last row.
__device__ __forceinline__ int tc_kv_tiles(const PrefillArgs& a, int t, int c, int tile) {
  const int last_row = min((tile + 1) * kTcRows, c * a.G) - 1;
  return (t - c + (last_row >> tc_gshift(a))) / kTcKeys + 1;
}

// Cost of a sequence: every unit's KV tiles + 1, for every KV head.
__device__ __forceinline__ long long tc_seq_cost(const PrefillArgs& a, int s, bool report) {
  int t, c, q0;
  pf_seq(a, s, t, c, q0, report);
  long long cost = 0;
  const int nt = tc_tiles(a, c);
  for (int tile = 0; tile < nt; ++tile) cost += tc_kv_tiles(a, t, c, tile) + 1;
  return cost * a.Hkv;
}

// Next unit after u (which has nkt KV tiles, its sequence chunk length c); u.s == S
// past the last.
__device__ __forceinline__ void tc_advance(const PrefillArgs& a, TcSched& u, int nkt, int c) {
  int t, q0;
  u.P += nkt + 1;
  if (++u.tile < tc_tiles(a, c)) return;
  u.tile = 0;
  if (++u.g < a.Hkv) return;
  u.g = 0;
  for (++u.s; u.s < a.S; ++u.s) {
    pf_seq(a, u.s, t, c, q0, false);
    if (c > 0) break;
  }
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using Sh = TcShape<T, D>;
  constexpr int NK = Sh::kKStages, NV = Sh::kVStages;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base_s = (raw + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (base_s - raw);
  const uint32_t bars = base_s + Sh::kBarOff;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t* const slot = reinterpret_cast<uint32_t*>(base + Sh::kBarOff + kSlotOff);
  TcSched* const sched = reinterpret_cast<TcSched*>(base + Sh::kBarOff + kSchedOff);

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
    for (int st = 0; st < 4; ++st) {
      ptx::mbar_init(bar(kBarKFull + st), 1);
      ptx::mbar_init(bar(kBarKEmpty + st), 1);
      ptx::mbar_init(bar(kBarVFull + st), 1);
      ptx::mbar_init(bar(kBarVEmpty + st), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bar(kBarQFull + b), 1);
      ptx::mbar_init(bar(kBarQEmpty + b), 1);
      ptx::mbar_init(bar(kBarSFull + b), 1);
      ptx::mbar_init(bar(kBarSEmpty + b), kTcRowWarps);
      ptx::mbar_init(bar(kBarPFull + b), kTcRowWarps);
      ptx::mbar_init(bar(kBarPvDone + b), 1);
    }
    ptx::mbar_init(bar(kBarOEmpty), kTcRowWarps);
    ptx::mbar_init(bar(kBarDrain), 1);
    ptx::fence_barrier_init();
    for (int i = 0; i < 4; ++i) reinterpret_cast<int*>(base + Sh::kBarOff + kDeadOff)[i] = 0;
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(slot), Sh::kTmemCols);
    ptx::tmem_relinquish();
  }

  // ---- schedule: per-sequence cost prefix (in the P area, free until the first
  // softmax), then this CTA's first unit and cost bound --------------------------
  {
    long long* const cpre = reinterpret_cast<long long*>(base + Sh::kKOff);  // free until the first load
    long long* const wsum = cpre + a.S + 1;
    const int nth = blockDim.x, tid = threadIdx.x;
    const int per = (a.S + nth - 1) / nth;
    const int b0 = min(a.S, tid * per), b1 = min(a.S, b0 + per);
    long long local = 0;
    for (int s = b0; s < b1; ++s) local += tc_seq_cost(a, s, blockIdx.x == 0);
    long long x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    long long run = x - local;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int s = b0; s < b1; ++s) {
      cpre[s] = run;
      run += tc_seq_cost(a, s, false);
    }
    if (tid == nth - 1) cpre[a.S] = run;
    __syncthreads();
    if (tid == 0) {
      const long long C = cpre[a.S];
      const long long lo = C * blockIdx.x / gridDim.x;
      TcSched u{a.S, 0, 0, 0, lo, C * (blockIdx.x + 1) / gridDim.x};
      if (lo < C) {
        int l = 0, h = a.S;  // largest s with cpre[s] <= lo
        while (h - l > 1) {
          const int mid = (l + h) >> 1;
          if (cpre[mid] <= lo) l = mid; else h = mid;
        }
        int t, c, q0;
        pf_seq(a, l, t, c, q0, false);
        const long long cost_g = (cpre[l + 1] - cpre[l]) / a.Hkv;
        const int g = static_cast<int>((lo - cpre[l]) / cost_g);
        long long P = cpre[l] + g * cost_g;
        int tile = 0;
        const int nt = tc_tiles(a, c);
        while (tile < nt && P < lo) P += tc_kv_tiles(a, t, c, tile++) + 1;
        u.s = l;
        u.g = g;
        u.tile = tile;
        u.P = P;
        if (tile == nt) {  // lo fell inside the last unit of (l, g): start at the next one
          u.tile = nt - 1;
          u.P = P - (tc_kv_tiles(a, t, c, nt - 1) + 1);
          tc_advance(a, u, tc_kv_tiles(a, t, c, nt - 1), c);
        }
      }
      *sched = u;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *slot;
  const TcSched start = *sched;

  if (warp == kTcQWarp) {
    // ---- TMA producer of the query tiles (two buffers, one per unit in flight) -----
    uint32_t un = 0;
    bool alive = true;
    const uint64_t qpolicy = ptx::policy_evict_first();  // each query tile is read once
    TcSched u = start;
    while (alive && u.s < a.S && u.P < start.hi) {
      int t, c, q0;
      pf_seq(a, u.s, t, c, q0, false);
      const int qb = static_cast<int>(un & 1u);
      bool ok = true;
      if (lane == 0) {
        ok = ptx::mbar_wait(bar(kBarQEmpty + qb), ((un >> 1) & 1u) ^ 1u, kPfWaitNs);
        if (ok) {
          ptx::mbar_arrive_expect_tx(bar(kBarQFull + qb), Sh::kTile);
#pragma unroll
          for (int cc = 0; cc < Sh::kChunks; ++cc)
            ptx::tma_load_3d(base_s + Sh::kQOff + qb * Sh::kTile + cc * kTcChunk, &qmap, cc * 64,
                             u.g * a.G, q0 + u.tile * (kTcRows >> tc_gshift(a)), bar(kBarQFull + qb),
                             qpolicy);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) { alive = false; break; }
      ++un;
      tc_advance(a, u, tc_kv_tiles(a, t, c, u.tile), c);
    }
    if (lane == 0) {
      if (!alive) pf_flag(a, PKV_DEV_WAIT_TIMEOUT);
      for (uint32_t k = un > 2u ? un - 2u : 0u; k < un; ++k)  // copies in flight land first
        ptx::mbar_wait(bar(kBarQFull + (k & 1u)), (k >> 1) & 1u, kPfWaitNs / 8);
    }
  } else if (warp == 0 || warp == kTcVWarp) {
    // ---- TMA producers: warp 0 K, warp 10 V --------------------------------------
    const bool is_k = warp == 0;
    // later units of (s, g) read K/V again: keep them in L2 ahead of the q and out streams
    const uint64_t policy = ptx::policy_evict_last();
    const int32_t groups_total = a.NB * a.Hkv * (BS / 8);  // 8-row groups of the cache
    constexpr int nblk = kTcKeys / BS;  // cache blocks (TMA boxes) of a KV tile
    const CUtensorMap* const map = is_k ? &kmap : &vmap;
    const int full0 = is_k ? kBarKFull : kBarVFull, empty0 = is_k ? kBarKEmpty : kBarVEmpty;
    const uint32_t ring = base_s + (is_k ? Sh::kKOff : Sh::kVOff);
    const uint32_t NS = is_k ? NK : NV;
    uint32_t it = 0;
    bool alive = true;
    TcSched u = start;
    while (alive && u.s < a.S && u.P < start.hi) {
      int t, c, q0;
      pf_seq(a, u.s, t, c, q0, false);
      const int nkt = tc_kv_tiles(a, t, c, u.tile);
      bool ok = true;
      for (int j = 0; j < nkt; ++j, ++it) {
        const uint32_t st = it % NS;
        const int bi = nblk * j + (lane & (nblk - 1));
        int32_t y = groups_total;  // a box wholly past the end: zero-filled
        if (lane < nblk && bi * BS < t) {
          const int id = __ldg(a.block_tables + static_cast<int64_t>(u.s) * a.MAXB + bi);
          if (static_cast<uint32_t>(id) < static_cast<uint32_t>(a.NB))
            y = (id * a.Hkv + u.g) * (BS / 8);
          else if (is_k)
            pf_flag(a, PKV_DEV_BAD_BLOCK_ID);
        }
        if (lane == 0) {
          ok = ptx::mbar_wait(bar(empty0 + st), ((it / NS) & 1u) ^ 1u, kPfWaitNs);
          if (ok) ptx::mbar_arrive_expect_tx(bar(full0 + st), Sh::kTile);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) { alive = false; break; }
        __syncwarp();
        if (lane < nblk)  // block `lane`: key groups lane * BS / 8 ..
          ptx::tma_load_4d(ring + st * Sh::kTile + lane * (BS / 8) * Sh::kGroup, map, 0, 0, 0, y,
                           bar(full0 + st), policy);
      }
      if (!alive) break;
      tc_advance(a, u, nkt, c);
    }
    if (lane == 0) {
      if (!alive) pf_flag(a, PKV_DEV_WAIT_TIMEOUT);
      // let the copies in flight land before the CTA can leave
      for (uint32_t k = it > NS ? it - NS : 0; k < it; ++k)
        ptx::mbar_wait(bar(full0 + k % NS), (k / NS) & 1u, kPfWaitNs / 8);
    }
  } else if (warp == 1) {
    // ---- MMA issuer (lane 0): one stream over the CTA's KV tiles, S of a tile
    // issued before P.V of the one before, across unit boundaries too ------------------
    uint32_t it = 0, un = 0;
    bool alive = true;
    // every lane polls (the warp stays converged for the elected MMA issue); the
    // vote keeps a time-out seen by one lane a time-out for all
    auto wait1 = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(b, parity, kPfWaitNs)) != 0;
    };
    // O (+)= P_x V_x for KV tile j (context t) of unit n; before a unit's first
    // product, O must have been read out for the unit before
    auto pv = [&](uint32_t x, int j, int t, uint32_t n) {
      const int b = static_cast<int>(x & 1u);
      const uint32_t st = x % NV;
      if (j == 0 && !wait1(bar(kBarOEmpty), (n & 1u) ^ 1u)) return false;
      if (!wait1(bar(kBarPFull + b), (x >> 1) & 1u)) return false;
      if (!wait1(bar(kBarVFull + st), (x / NV) & 1u)) return false;
      ptx::tc_fence_after();
      const uint32_t vt = base_s + Sh::kVOff + st * Sh::kTile;
      // keys past the context inside its last cache block may hold anything (NaN
      // included) and P is 0 there: zero those V rows so that 0 * V stays 0
      constexpr int nblk = kTcKeys / BS;
      const int last = (t - 1) / BS;
      if ((t % BS) != 0 && last / nblk == j) {
        const int r0 = (last % nblk) * BS + t % BS;
        const int n16 = (BS - t % BS) * 8 * Sh::kChunks;  // 16-byte units
        for (int i = lane; i < n16; i += 32) {
          const int row = r0 + i / (8 * Sh::kChunks), rem = i % (8 * Sh::kChunks);
          ptx::st_shared_v4(vt + (row >> 3) * Sh::kGroup + (rem / 8) * 1024 + (row & 7) * 128 +
                                (rem % 8) * 16,
                            0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
      }
      // the whole warp issues (one elected lane), so the operands stay uniform
      const uint32_t pt = tmem + Sh::kPCol + b * (kTcKeys / 2);
#pragma unroll
      for (int ks = 0; ks < kTcKeys / 16; ++ks)  // 16 keys = 8 packed columns of P
        ptx::umma_f16_ta_elect(tmem + Sh::kOCol, pt + ks * 8,
                               ptx::smem_desc_sw128(vt + ks * 2 * Sh::kGroup, 1024, Sh::kGroup),
                               Sh::kIdPV,
                               j > 0 || ks > 0);
      ptx::umma_commit_elect(bar(kBarPvDone + b));
      ptx::umma_commit_elect(bar(kBarVEmpty + st));
      __syncwarp();
      return true;
    };
    bool pending = false;  // a P.V product not issued yet: tile px, index pj of unit pn
    uint32_t px = 0, pn = 0;
    int pj = 0, pt = 0;
    TcSched u = start;
    while (alive && u.s < a.S && u.P < start.hi) {
      int t, c, q0;
      pf_seq(a, u.s, t, c, q0, false);
      const int nkt = tc_kv_tiles(a, t, c, u.tile);
      const int qb = static_cast<int>(un & 1u);
      if (!wait1(bar(kBarQFull + qb), (un >> 1) & 1u)) { alive = false; break; }
      const uint32_t n = un++;
      ptx::tc_fence_after();
      for (int j = 0; j < nkt; ++j, ++it) {
        const uint32_t st = it % NK;
        const int b = static_cast<int>(it & 1u);
        if (!wait1(bar(kBarKFull + st), (it / NK) & 1u) ||
            !wait1(bar(kBarSEmpty + b), ((it >> 1) & 1u) ^ 1u)) {
          alive = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t qa = base_s + Sh::kQOff + qb * Sh::kTile;
        const uint32_t kb = base_s + Sh::kKOff + st * Sh::kTile;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t kin = (ks & 3) * 32;  // 16 columns inside a 128-byte chunk
          ptx::umma_f16_elect(tmem + Sh::kSCol + b * kTcKeys,
                              ptx::smem_desc_sw128(qa + (ks >> 2) * kTcChunk + kin, 16, 1024),
                              ptx::smem_desc_sw128(kb + (ks >> 2) * 1024 + kin, 16, Sh::kGroup),
                              Sh::kIdQK, ks > 0);
        }
        ptx::umma_commit_elect(bar(kBarSFull + b));
        ptx::umma_commit_elect(bar(kBarKEmpty + st));
        if (j == nkt - 1) ptx::umma_commit_elect(bar(kBarQEmpty + qb));
        __syncwarp();
        if (pending && !pv(px, pj, pt, pn)) { alive = false; break; }
        pending = true;
        px = it;
        pj = j;
        pt = t;
        pn = n;
      }
      if (!alive) break;
      tc_advance(a, u, nkt, c);
    }
    if (alive && pending && !pv(px, pj, pt, pn)) alive = false;
    if (lane == 0) {
      if (!alive) pf_flag(a, PKV_DEV_WAIT_TIMEOUT);
      ptx::umma_commit(bar(kBarDrain));  // lands once every MMA issued above is done
      ptx::mbar_wait(bar(kBarDrain), 0, kPfWaitNs);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + kTcRowWarps) {
    // ---- row threads: softmax, rescaling, output -----------------------------------
    // The two warps of a lane quarter meet at every exchange (named barrier); a
    // warp whose wait ran out skips ahead to the next exchange and flags itself
    // there, and both leave together, so neither is left waiting at the barrier.
    constexpr int HD = Sh::kHalfD;
    const int q4 = warp & 3, h = (warp - 2) >> 2;
    const int r = 32 * q4 + lane;  // tile row = tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    // this thread's keys 64 h .. 64 h + 63 of row r: 32 packed columns of P
    const uint32_t pcol = tmem + lane_off + Sh::kPCol + h * (kTcHalfKeys / 2);
    float* const xch = reinterpret_cast<float*>(base + Sh::kXchOff);
    volatile int* const dead_bits = reinterpret_cast<volatile int*>(base + Sh::kBarOff + kDeadOff);
    const uint32_t pair_bar = 1 + q4;
    bool dead = false;       // this warp gave up a wait
    bool pair_dead = false;  // either warp of the pair did
    // the other half's value of x for this row
    auto exchange = [&](float x) {
      ptx::named_bar_sync(pair_bar, 64);  // the previous exchange has been read
      if (dead && lane == 0) dead_bits[q4] = dead_bits[q4] | (1 << h);
      xch[h * kTcRows + r] = x;
      ptx::named_bar_sync(pair_bar, 64);
      pair_dead = dead_bits[q4] != 0;
      return xch[(1 - h) * kTcRows + r];
    };
    T* const og = reinterpret_cast<T*>(a.out);
    const uint64_t opolicy = ptx::policy_evict_first();  // the output is not read here
    uint32_t it = 0;
    auto wait_all = [&](uint32_t b, uint32_t parity) {
      if (dead) return;
      dead = !__all_sync(0xffffffffu, ptx::mbar_wait(b, parity, kPfWaitNs));
    };
    const uint32_t oa = tmem + lane_off + Sh::kOCol + h * HD;  // this thread's half of O
    // A unit's output is written after the first tile of the next unit (its last
    // P.V is done by then), so that the tensor cores are not left waiting on it.
    bool pend = false, pend_valid = false;
    T* pend_row = nullptr;
    float pend_l = 0.f;
    uint32_t pend_x = 0;  // the unit's last KV tile
    auto epilogue = [&]() {
      pend = false;
      const float lt = pend_l + exchange(pend_l);
      if (pair_dead) return;
      wait_all(bar(kBarPvDone + (pend_x & 1u)), (pend_x >> 1) & 1u);
      if (dead) return;
      ptx::tc_fence_after();
      const float inv = 1.f / lt;
      // 32-byte stores when the output allows them (it need only be 16-byte aligned)
      const bool wide = (reinterpret_cast<uintptr_t>(pend_row) & 31u) == 0;
#pragma unroll
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t w[32];
        ptx::tmem_ld32(oa + c0, w);
        if (pend_valid) {
#pragma unroll
          for (int d = 0; d < 32; d += 16) {
            uint32_t pk8[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float x0, x1;
              fma2(__uint_as_float(w[d + e]), __uint_as_float(w[d + e + 1]), inv, 0.f, x0, x1);
              pk8[e / 2] = ptx::pack2<T>(x0, x1);
            }
            if (wide) {
              st_global_v8_hint(pend_row + c0 + d, pk8, opolicy);
            } else {
              ptx::st_global_v4_hint(pend_row + c0 + d, make_uint4(pk8[0], pk8[1], pk8[2], pk8[3]),
                                     opolicy);
              ptx::st_global_v4_hint(pend_row + c0 + d + 8,
                                     make_uint4(pk8[4], pk8[5], pk8[6], pk8[7]), opolicy);
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarOEmpty));
    };
    TcSched u = start;
    while (!pair_dead && u.s < a.S && u.P < start.hi) {
      int t, c, q0;
      pf_seq(a, u.s, t, c, q0, false);
      const int nkt = tc_kv_tiles(a, t, c, u.tile);
      const int R = u.tile * kTcRows + r;
      const bool valid = R < c * a.G;
      const int p = valid ? t - c + (R >> tc_gshift(a)) : t - 1;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkt; ++j, ++it) {
        const int b = static_cast<int>(it & 1u);
        wait_all(bar(kBarSFull + b), (it >> 1) & 1u);
        uint32_t v[kTcHalfKeys];
        const int lim = p - kTcKeys * j - kTcHalfKeys * h;  // keys 0 .. lim of the half visible
        const bool full = lim >= kTcHalfKeys - 1;
        float mx = -INFINITY;
        if (!dead) {
          ptx::tc_fence_after();
          const uint32_t sa = tmem + lane_off + Sh::kSCol + b * kTcKeys + h * kTcHalfKeys;
          ptx::tmem_ld32_nowait(sa, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          ptx::tmem_ld32_nowait(sa + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          ptx::tmem_wait_ld();
          // keys past the row's position score -inf: they drop out of the max, and
          // their 2^(s - m) is 0 (m is finite: key 0 of tile 0 is visible to every row)
          if (!full) {
#pragma unroll
            for (int i = 0; i < kTcHalfKeys; ++i)
              if (i > lim) v[i] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int i = 0; i < kTcHalfKeys; i += 2)
            mx = fmax3(mx, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        }
        mx = fmaxf(mx, exchange(mx));
        if (pair_dead) break;
        const float mt = mx * a.scale_log2;  // the row's max over this tile, log2 units
        // P_j's buffer is free once O_{j-2}'s product is done
        wait_all(bar(kBarPvDone + b), ((it >> 1) & 1u) ^ 1u);
        if (j == 0) {
          m = mt;
        } else {
          // move the reference of the rows whose max grew by more than 2^8: O and l
          // scaled by exp2(m - mt), once P_{j-1} V_{j-1} has landed in O.  The
          // tensor-memory accesses are warp-wide, so the whole warp takes the branch
          // and the other rows scale by exactly 1.
          const bool move = mt > m + kTcRescale;
          if (__any_sync(0xffffffffu, move)) {
            const float al = move ? ptx::ex2(m - mt) : 1.f;
            wait_all(bar(kBarPvDone + (b ^ 1)), ((it - 1) >> 1) & 1u);
            if (!dead) {
              ptx::tc_fence_after();
#pragma unroll
              for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t w[32];
                ptx::tmem_ld32(oa + c0, w);
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * al);
                ptx::tmem_st32(oa + c0, w);
              }
            }
            if (move) {
              l *= al;
              m = mt;
            }
          }
        }
        if (dead) continue;  // on to the next exchange
        float s0 = 0.f, s1 = 0.f;
        uint32_t pk[kTcHalfKeys / 2];
#pragma unroll
        for (int k = 0; k < kTcHalfKeys / 2; ++k) {  // keys 2k, 2k + 1 of the half
          // exponents rounded to an f16 pair, two 2^x per ex2 instruction
          float y0, y1;
          fma2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]), a.scale_log2, -m, y0, y1);
          const uint32_t e = ptx::ex2_f16x2(ptx::f16x2_of(y0, y1));
          if constexpr (std::is_same<T, __half>::value) {
            pk[k] = e;  // P is the f16 pair itself
            add_f16x2(s0, s1, e);
          } else {
            float x0, x1;
            ptx::f32_of_f16x2(e, x0, x1);
            pk[k] = ptx::pack2<T>(x0, x1);
            add2(s0, s1, x0, x1);
          }
        }
        ptx::tmem_st32(pcol + b * (kTcKeys / 2), pk);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(bar(kBarSEmpty + b));
          ptx::mbar_arrive(bar(kBarPFull + b));
        }
        l += s0 + s1;
        if (j == 0 && pend) {  // the previous unit's output
          epilogue();
          if (pair_dead) break;
        }
      }
      if (pair_dead) break;
      pend = true;
      pend_valid = valid;
      pend_row = og + (static_cast<int64_t>(q0 + (R >> tc_gshift(a))) * a.Hq + u.g * a.G +
                        (R & (a.G - 1))) * D + h * HD;
      pend_l = l;
      pend_x = it - 1;
      tc_advance(a, u, nkt, c);
    }
    if (pend && !pair_dead) epilogue();
    if (pair_dead && lane == 0) pf_flag(a, PKV_DEV_WAIT_TIMEOUT);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, Sh::kTmemCols);
}

int tc_smem_optin(int* bytes) {
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

template <typename T, int D, int BS>
int launch_tc(const PrefillArgs& a, const void* k_cache, const void* v_cache, int32_t dtype,
              cudaStream_t stream) {
  using Sh = TcShape<T, D>;
  static std::once_flag flags[64];
  static int results[64];
  int dev = 0, optin = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int rc = tc_smem_optin(&optin);
  if (rc != PKV_OK) return rc;
  PKV_REQUIRE(static_cast<int>(Sh::kBytes) <= optin, PKV_ERR_UNSUPPORTED,
              "prefill needs %u bytes of shared memory, the device offers %d", Sh::kBytes, optin);
  // the schedule's cost prefix lives in the P area
  PKV_REQUIRE(static_cast<int64_t>(a.S + 1 + kTcWarps) * 8 <= Sh::kKStages * Sh::kTile,
              PKV_ERR_UNSUPPORTED,
              "too many sequences");
  std::call_once(flags[dev], [&] {
    results[dev] = cudaFuncSetAttribute(prefill_tc_kernel<T, D, BS>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kBytes);
  });
  if (results[dev] != cudaSuccess)
    return cuda_fail(static_cast<cudaError_t>(results[dev]), "cudaFuncSetAttribute");
  CUtensorMap qmap, kmap, vmap;
  // q [T, Hq, D]: boxes of 64 head_dim elements (128 B) x G heads x 128 / G queries,
  // landing as the 128 swizzled rows (query, head) of one column chunk
  const CUtensorMapDataType ty =
      dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int64_t qdims[3] = {D, a.Hq, a.T};
  const int64_t qstrides[2] = {static_cast<int64_t>(D) * 2, static_cast<int64_t>(a.Hq) * D * 2};
  const int32_t qbox[3] = {64, a.G, kTcRows / a.G};
  rc = encode_map_3d(&qmap, a.q, ty, 2, qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != PKV_OK) return rc;
  // K and V [rows, D] viewed as (column in chunk, row in group, chunk, 8-row group):
  // one box = one cache block of one KV head, landing chunk-major within each group
  const int64_t kvdims[4] = {64, 8, Sh::kChunks, static_cast<int64_t>(a.NB) * a.Hkv * (BS / 8)};
  const int64_t kvstrides[3] = {static_cast<int64_t>(D) * 2, 128, 8 * static_cast<int64_t>(D) * 2};
  const int32_t kvbox[4] = {64, 8, Sh::kChunks, BS / 8};
  rc = encode_map_4d(&kmap, k_cache, ty, kvdims, kvstrides, kvbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != PKV_OK) return rc;
  rc = encode_map_4d(&vmap, v_cache, ty, kvdims, kvstrides, kvbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != PKV_OK) return rc;
  int sms = 0;
  rc = device_sm_count(&sms, &dev);
  if (rc != PKV_OK) return rc;
  prefill_tc_kernel<T, D, BS><<<sms, kTcThreads, Sh::kBytes, stream>>>(qmap, kmap, vmap, a);
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

// One kernel per block size, so that the producers' box arithmetic is constant.
template <typename T, int D>
int launch_tc_bs(const PrefillArgs& a, const void* k_cache, const void* v_cache, int32_t dtype,
                 cudaStream_t stream) {
  switch (a.bs) {
    case 8: return launch_tc<T, D, 8>(a, k_cache, v_cache, dtype, stream);
    case 16: return launch_tc<T, D, 16>(a, k_cache, v_cache, dtype, stream);
    case 32: return launch_tc<T, D, 32>(a, k_cache, v_cache, dtype, stream);
    default: return fail(PKV_ERR_UNSUPPORTED, "block_size %d not in {8, 16, 32}", a.bs);
  }
}

}  // namespace

int launch_prefill_tc(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                      int32_t dtype, int32_t head_dim, cudaStream_t stream) {
  if (dtype == PKV_BF16)
    return head_dim == 64 ? launch_tc_bs<__nv_bfloat16, 64>(a, k_cache, v_cache, dtype, stream)
                          : launch_tc_bs<__nv_bfloat16, 128>(a, k_cache, v_cache, dtype, stream);
  return head_dim == 64 ? launch_tc_bs<__half, 64>(a, k_cache, v_cache, dtype, stream)
                        : launch_tc_bs<__half, 128>(a, k_cache, v_cache, dtype, stream);
}

}  // namespace pkv
