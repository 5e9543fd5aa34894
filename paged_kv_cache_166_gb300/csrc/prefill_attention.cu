// Paged (chunked) prefill attention for sm_103a.
//
// What is computed ("PagedAttention: How vLLM Borrowed Virtual Memory to Unlock GPU
// Serving at Scale", section "Walking Through the Lifecycle", Prefill; chunked
// prefill in section "RadixAttention ..."): sequence s has t = context_lens[s]
// cached tokens, its new chunk of c = query_start[s+1] - query_start[s] queries
// being the last c positions; query row query_start[s] + i sits at position
// p = t - c + i and, for query head h of KV group g = h / G, attends to every
// position j <= p read through the block table:
//   out[row, h] = softmax_j(scale * q[row, h] . K[slot(j), g]) . V[slot(j), g].
//
// Two kernels compute it.  The default runs on the 5th-generation tensor cores
// (tcgen05, tensor memory; prefill_tcgen05.cu).  The one below, kept as the
// measured warp-level alternative (build with PKV_PREFILL_TCGEN05=0), uses
// mma.sync:  a tile is 64 rows of one (sequence, KV head): row R is query R / G and
// head g*G + R % G, so the G heads of a query share every K/V tile.  A CTA has
// four consumer warps (16 rows each: scores and P.V on the tensor cores, m16n8k16
// with fp32 accumulation, online softmax in fp32, base 2) and one producer warp
// that streams the tile's 16-token K/V blocks, in logical order through the block
// table, with TMA (128-byte swizzle) into a ring of shared-memory stages.  Stage
// hand-off uses mbarriers: "full" completes on the TMA transaction bytes, "empty"
// on one arrival per consumer warp.  Tiles are taken round-robin by the CTAs of a
// persistent grid; every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "prefill_common.cuh"
#include "ptx.cuh"

#ifndef PKV_PREFILL_TCGEN05
#define PKV_PREFILL_TCGEN05 1
#endif

namespace pkv {
namespace {

constexpr int kPfRows = 64;                // rows of a tile
constexpr int kPfConsumers = 4;            // consumer warps (16 rows each)
constexpr int kPfThreads = (kPfConsumers + 1) * 32;
constexpr int kPfStages = 4;
constexpr int kPfCtasPerSm = 2;

template <typename T, int D>
struct PfShape {
  static constexpr int kTileBytes = kPfTok * D * static_cast<int>(sizeof(T));  // K or V tile
  static constexpr int kSub = D * static_cast<int>(sizeof(T)) / 128;          // 128-B sub-tiles
  static constexpr int kBoxCols = 128 / static_cast<int>(sizeof(T));
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kKS = D / 16;        // 16-wide k steps of q . k
  static constexpr int kDT = D / 8;         // 8-wide output tiles
};

struct PfSmem {
  uint32_t tiles, full, empty, upre, scratch, total;
};

__host__ __device__ inline PfSmem pf_smem(int stage_bytes, int S) {
  PfSmem L;
  uint32_t off = 0;
  L.tiles = off;
  off += kPfStages * stage_bytes;
  L.full = off;
  off += kPfStages * 8;
  L.empty = off;
  off += kPfStages * 8;
  L.upre = off;
  off += (S + 1) * 4;
  off = (off + 15u) & ~15u;
  L.scratch = off;
  off += 8 * 4;
  L.total = off + 1024;  // slack to align the tiles to 1024 B
  return L;
}

__device__ __forceinline__ int pf_tiles(const PrefillArgs& a, int c) {
  return (c * a.G + kPfRows - 1) / kPfRows;
}

// Key blocks a tile reads: up to the position of its last row.
__device__ __forceinline__ int pf_blocks(const PrefillArgs& a, int t, int c, int tile) {
  const int last_row = min((tile + 1) * kPfRows, c * a.G) - 1;
  const int p_max = t - c + last_row / a.G;
  return p_max / kPfTok + 1;
}

template <typename T, int D>
__global__ void __launch_bounds__(kPfThreads, kPfCtasPerSm)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using Sh = PfShape<T, D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base_s = (raw + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (base_s - raw);
  const PfSmem L = pf_smem(Sh::kStageBytes, a.S);
  int32_t* const upre = reinterpret_cast<int32_t*>(base + L.upre);
  int32_t* const scratch = reinterpret_cast<int32_t*>(base + L.scratch);
  const uint32_t tiles = base_s + L.tiles;
  const uint32_t full = base_s + L.full;
  const uint32_t empty = base_s + L.empty;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
    for (int st = 0; st < kPfStages; ++st) {
      ptx::mbar_init(full + 8 * st, 1);
      ptx::mbar_init(empty + 8 * st, kPfConsumers);
    }
    ptx::fence_barrier_init();
  }
  // Units (sequence, KV head, tile) in order; upre[s] = units before sequence s.
  {
    const int S = a.S, nthreads = blockDim.x, tid = threadIdx.x;
    const int chunk = (S + nthreads - 1) / nthreads;
    const int b0 = min(S, tid * chunk), b1 = min(S, b0 + chunk);
    int local = 0;
    for (int s = b0; s < b1; ++s) {
      int t, c, q0;
      pf_seq(a, s, t, c, q0, blockIdx.x == 0);
      local += a.Hkv * pf_tiles(a, c);
    }
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += scratch[w];
    int run = before + x - local;
    for (int s = b0; s < b1; ++s) {
      upre[s] = run;
      int t, c, q0;
      pf_seq(a, s, t, c, q0, false);
      run += a.Hkv * pf_tiles(a, c);
    }
    if (tid == nthreads - 1) upre[S] = run;
    __syncthreads();
  }
  const int total = upre[a.S];

  // Unit u -> sequence, KV head, tile.
  auto unit = [&](int u, int& s, int& g, int& tile, int& t, int& c, int& q0) {
    int lo = 0, hi = a.S;  // upre[lo] <= u < upre[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (upre[mid] <= u) lo = mid; else hi = mid;
    }
    s = lo;
    pf_seq(a, s, t, c, q0, false);
    const int nt = pf_tiles(a, c);
    const int r = u - upre[s];
    g = r / nt;
    tile = r - g * nt;
  };

  if (warp == kPfConsumers) {
    // ---- producer warp: K/V blocks of every unit of this CTA, in order ----------
    // (the other query tiles of the same sequence and KV head read them again)
    const uint64_t policy = ptx::policy_evict_normal();
    const int32_t rows_total = a.NB * a.Hkv * kPfTok;
    uint32_t k = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      int s, g, tile, t, c, q0;
      unit(u, s, g, tile, t, c, q0);
      const int nkb = pf_blocks(a, t, c, tile);
      int ids = 0;
      for (int j = 0; j < nkb; ++j, ++k) {
        if ((j & 31) == 0)  // block ids 32 at a time, one per lane
          ids = j + lane < nkb ? __ldg(a.block_tables + static_cast<int64_t>(s) * a.MAXB + j + lane) : 0;
        const int id = __shfl_sync(0xffffffffu, ids, j & 31);
        const int st = k % kPfStages;
        const uint32_t parity = ((k / kPfStages) & 1u) ^ 1u;
        bool ok = true;
        if (lane == 0) ok = ptx::mbar_wait(empty + 8 * st, parity, kPfWaitNs);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) pf_flag(a, PKV_DEV_WAIT_TIMEOUT);
          return;
        }
        if (lane == 0) {
          int32_t y;
          if (static_cast<uint32_t>(id) < static_cast<uint32_t>(a.NB)) {
            y = (id * a.Hkv + g) * kPfTok;
          } else {
            pf_flag(a, PKV_DEV_BAD_BLOCK_ID);
            y = rows_total;  // a box wholly past the end: filled with zeros
          }
          const uint32_t bar = full + 8 * st;
          ptx::mbar_arrive_expect_tx(bar, Sh::kStageBytes);
          const uint32_t kt = tiles + st * Sh::kStageBytes;
          const uint32_t vt = kt + Sh::kTileBytes;
#pragma unroll
          for (int cc = 0; cc < Sh::kSub; ++cc)
            ptx::tma_load_2d(kt + cc * 2048, &kmap, cc * Sh::kBoxCols, y, bar, policy);
#pragma unroll
          for (int cc = 0; cc < Sh::kSub; ++cc)
            ptx::tma_load_2d(vt + cc * 2048, &vmap, cc * Sh::kBoxCols, y, bar, policy);
        }
      }
    }
    return;
  }

  // ---- consumer warps -------------------------------------------------------------
  const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, r8 = lane & 7;
  const T* const qg = reinterpret_cast<const T*>(a.q);
  T* const og = reinterpret_cast<T*>(a.out);
  uint32_t k = 0;
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    int s, g, tile, t, c, q0;
    unit(u, s, g, tile, t, c, q0);
    const int nkb = pf_blocks(a, t, c, tile);
    const int rows = c * a.G;
    const int R0 = tile * kPfRows + warp * 16;
    const int Ra = R0 + gid, Rb = R0 + gid + 8;  // this thread's two rows
    const bool va = Ra < rows, vb = Rb < rows;
    const int pa = va ? t - c + Ra / a.G : t - 1;
    const int pb = vb ? t - c + Rb / a.G : t - 1;
    const bool any_rows = R0 < rows;
    const int p_lo = t - c + R0 / a.G;                                  // first row's position
    const int p_hi = t - c + (min(R0 + 16, rows) - 1) / a.G;            // last valid row's

    // q fragments (A operand, rows x head_dim), straight from global memory
    uint32_t qf[Sh::kKS][4];
    {
      const T* rowa = qg + (static_cast<int64_t>(q0 + Ra / a.G) * a.Hq + g * a.G + Ra % a.G) * D;
      const T* rowb = qg + (static_cast<int64_t>(q0 + Rb / a.G) * a.Hq + g * a.G + Rb % a.G) * D;
#pragma unroll
      for (int ks = 0; ks < Sh::kKS; ++ks) {
        const int d = ks * 16 + 2 * tig;
        qf[ks][0] = va ? __ldg(reinterpret_cast<const uint32_t*>(rowa + d)) : 0u;
        qf[ks][1] = vb ? __ldg(reinterpret_cast<const uint32_t*>(rowb + d)) : 0u;
        qf[ks][2] = va ? __ldg(reinterpret_cast<const uint32_t*>(rowa + d + 8)) : 0u;
        qf[ks][3] = vb ? __ldg(reinterpret_cast<const uint32_t*>(rowb + d + 8)) : 0u;
      }
    }
    float o[Sh::kDT][4];
#pragma unroll
    for (int i = 0; i < Sh::kDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;

    for (int j = 0; j < nkb; ++j, ++k) {
      const int st = k % kPfStages;
      const uint32_t parity = (k / kPfStages) & 1u;
      const bool ok = ptx::mbar_wait(full + 8 * st, parity, kPfWaitNs);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) pf_flag(a, PKV_DEV_WAIT_TIMEOUT);
        return;
      }
      const int key0 = j * kPfTok;
      if (any_rows && key0 <= p_hi) {
        const uint32_t kt = tiles + st * Sh::kStageBytes;
        const uint32_t vt = kt + Sh::kTileBytes;
        // S = Q K^T: B fragments from K rows (keys) via ldmatrix; two 8-key tiles
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = r8 + 8 * (mi >> 1);
#pragma unroll
        for (int ks = 0; ks < Sh::kKS; ++ks) {
          uint32_t b[4];
          ptx::ldsm_x4(kt + (((2 * ks + (mi & 1)) >> 3) * 2048) + krow * 128 +
                           ((((2 * ks + (mi & 1)) & 7) ^ (krow & 7)) << 4),
                       b);
          ptx::mma_16816<T>(sc[0], qf[ks], b[0], b[1]);
          ptx::mma_16816<T>(sc[1], qf[ks], b[2], b[3]);
        }
        // scale, causal mask (key > row position), online softmax per row
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) x[nt][e] = sc[nt][e] * a.scale_log2;
        if (key0 + kPfTok - 1 > p_lo) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int kk = key0 + 8 * nt + 2 * tig;
            if (kk > pa) x[nt][0] = -INFINITY;
            if (kk + 1 > pa) x[nt][1] = -INFINITY;
            if (kk > pb) x[nt][2] = -INFINITY;
            if (kk + 1 > pb) x[nt][3] = -INFINITY;
          }
        }
        float mxa = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mxb = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
          mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
          mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
        }
        const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
        const float ala = exp2f(ma - na), alb = exp2f(mb - nb);
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pr[nt][0] = exp2f(x[nt][0] - na);
          pr[nt][1] = exp2f(x[nt][1] - na);
          pr[nt][2] = exp2f(x[nt][2] - nb);
          pr[nt][3] = exp2f(x[nt][3] - nb);
        }
        la = la * ala + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
        lb = lb * alb + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
        ma = na;
        mb = nb;
#pragma unroll
        for (int i = 0; i < Sh::kDT; ++i) {
          o[i][0] *= ala;
          o[i][1] *= ala;
          o[i][2] *= alb;
          o[i][3] *= alb;
        }
        // P as the A operand (rows x 16 keys)
        uint32_t pf[4];
        pf[0] = ptx::pack2<T>(pr[0][0], pr[0][1]);
        pf[1] = ptx::pack2<T>(pr[0][2], pr[0][3]);
        pf[2] = ptx::pack2<T>(pr[1][0], pr[1][1]);
        pf[3] = ptx::pack2<T>(pr[1][2], pr[1][3]);
        // V as the B operand (16 keys x 8 head_dim) via transposing ldmatrix; keys past
        // the context (last block) may hold anything, NaN included: zero their lanes
        const int valid = t - key0;
        const uint32_t mlo = (2 * tig < valid ? 0x0000ffffu : 0u) | (2 * tig + 1 < valid ? 0xffff0000u : 0u);
        const uint32_t mhi = (2 * tig + 8 < valid ? 0x0000ffffu : 0u) | (2 * tig + 9 < valid ? 0xffff0000u : 0u);
        const int vrow = r8 + 8 * (mi & 1);
#pragma unroll
        for (int p = 0; p < Sh::kDT / 2; ++p) {
          uint32_t b[4];
          const int ch = 2 * p + (mi >> 1);
          ptx::ldsm_x4_trans(vt + ((ch >> 3) * 2048) + vrow * 128 + (((ch & 7) ^ (vrow & 7)) << 4), b);
          if (valid < kPfTok) {
            b[0] &= mlo;
            b[1] &= mhi;
            b[2] &= mlo;
            b[3] &= mhi;
          }
          ptx::mma_16816<T>(o[2 * p], pf, b[0], b[1]);
          ptx::mma_16816<T>(o[2 * p + 1], pf, b[2], b[3]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty + 8 * st);
    }
    if (!any_rows) continue;
    // normalise and write this thread's two rows
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, off);
      lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    const float ia = 1.f / la, ib = 1.f / lb;
    T* const outa = og + (static_cast<int64_t>(q0 + Ra / a.G) * a.Hq + g * a.G + Ra % a.G) * D;
    T* const outb = og + (static_cast<int64_t>(q0 + Rb / a.G) * a.Hq + g * a.G + Rb % a.G) * D;
#pragma unroll
    for (int i = 0; i < Sh::kDT; ++i) {
      const int d = 8 * i + 2 * tig;
      if (va) *reinterpret_cast<uint32_t*>(outa + d) = ptx::pack2<T>(o[i][0] * ia, o[i][1] * ia);
      if (vb) *reinterpret_cast<uint32_t*>(outb + d) = ptx::pack2<T>(o[i][2] * ib, o[i][3] * ib);
    }
  }
}

// ---------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------
int pf_smem_optin(int* bytes) {
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

template <typename T, int D>
int launch_prefill(const PrefillArgs& a, const void* k_cache, const void* v_cache, int dtype,
                   cudaStream_t stream) {
  using Sh = PfShape<T, D>;
  const PfSmem L = pf_smem(Sh::kStageBytes, a.S);
  static std::once_flag flags[64];
  static int results[64];
  int dev = 0, optin = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int rc = pf_smem_optin(&optin);
  if (rc != PKV_OK) return rc;
  PKV_REQUIRE(static_cast<int>(L.total) <= optin, PKV_ERR_UNSUPPORTED,
              "prefill needs %u bytes of shared memory", L.total);
  std::call_once(flags[dev], [&] {
    results[dev] = cudaFuncSetAttribute(prefill_attention_kernel<T, D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  });
  if (results[dev] != cudaSuccess)
    return cuda_fail(static_cast<cudaError_t>(results[dev]), "cudaFuncSetAttribute");
  CUtensorMap kmap, vmap;
  const int64_t rows = static_cast<int64_t>(a.NB) * a.Hkv * kPfTok;
  rc = encode_cache_map(&kmap, k_cache, dtype, rows, D, Sh::kBoxCols, kPfTok);
  if (rc != PKV_OK) return rc;
  rc = encode_cache_map(&vmap, v_cache, dtype, rows, D, Sh::kBoxCols, kPfTok);
  if (rc != PKV_OK) return rc;
  int sms = 0;
  rc = device_sm_count(&sms, &dev);
  if (rc != PKV_OK) return rc;
  prefill_attention_kernel<T, D><<<sms * kPfCtasPerSm, kPfThreads, L.total, stream>>>(kmap, vmap, a);
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, const int32_t* query_start,
                                     int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                                     int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                     float scale, void* out, int32_t* status, int32_t dtype,
                                     void* stream) {
  PKV_REQUIRE(dtype == PKV_F16 || dtype == PKV_BF16, PKV_ERR_DTYPE,
              "prefill takes f16 or bf16 (dtype %d)", dtype);
  PKV_REQUIRE(num_seqs >= 0 && num_seqs <= kPfMaxSeqs, PKV_ERR_UNSUPPORTED,
              "num_seqs %d outside [0, %d]", num_seqs, kPfMaxSeqs);
  PKV_REQUIRE(num_q_heads > 0 && num_kv_heads > 0 && num_q_heads % num_kv_heads == 0,
              PKV_ERR_INVALID_ARG, "num_q_heads %d must be a positive multiple of num_kv_heads %d",
              num_q_heads, num_kv_heads);
  const int G = num_q_heads / num_kv_heads;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, PKV_ERR_UNSUPPORTED,
              "query heads per KV head %d not in {1,2,4,8}", G);
  PKV_REQUIRE(head_dim == 64 || head_dim == 128, PKV_ERR_UNSUPPORTED,
              "prefill head_dim %d not in {64, 128}", head_dim);
  if (PKV_PREFILL_TCGEN05)
    PKV_REQUIRE(block_size == 8 || block_size == 16 || block_size == 32, PKV_ERR_UNSUPPORTED,
                "block_size %d not in {8, 16, 32}", block_size);
  else
    PKV_REQUIRE(block_size == kPfTok, PKV_ERR_UNSUPPORTED, "block_size %d (kernel uses 16)",
                block_size);
  PKV_REQUIRE(max_blocks_per_seq > 0 && num_blocks > 0, PKV_ERR_INVALID_ARG, "bad sizes");
  PKV_REQUIRE(static_cast<int64_t>(max_blocks_per_seq) * block_size < (int64_t(1) << 31),
              PKV_ERR_UNSUPPORTED, "max_blocks_per_seq * block_size >= 2^31");
  PKV_REQUIRE(static_cast<int64_t>(num_blocks) * num_kv_heads * block_size * 4 < (int64_t(1) << 31),
              PKV_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * block_size * 4 >= 2^31");
  PKV_REQUIRE(static_cast<int64_t>(num_seqs) * max_blocks_per_seq < (int64_t(1) << 31),
              PKV_ERR_UNSUPPORTED, "num_seqs * max_blocks_per_seq >= 2^31");
  PKV_REQUIRE(num_tokens >= 0, PKV_ERR_INVALID_ARG, "negative num_tokens");
  PKV_REQUIRE(static_cast<int64_t>(num_tokens) * num_q_heads * head_dim < (int64_t(1) << 40),
              PKV_ERR_UNSUPPORTED, "q too large");
  if (num_seqs == 0 || num_tokens == 0) return ok();
  PKV_REQUIRE(q && k_cache && v_cache && block_tables && context_lens && query_start && out,
              PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(aligned(q, 16) && aligned(k_cache, 16) && aligned(v_cache, 16) && aligned(out, 16),
              PKV_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned");
  PrefillArgs a{};
  a.q = q;
  a.out = out;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.query_start = query_start;
  a.status = status;
  a.S = num_seqs;
  a.T = num_tokens;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.G = G;
  a.MAXB = max_blocks_per_seq;
  a.NB = num_blocks;
  a.bs = block_size;
  a.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc;
  if (PKV_PREFILL_TCGEN05) {
    rc = launch_prefill_tc(a, k_cache, v_cache, dtype, head_dim, st);
  } else if (dtype == PKV_BF16) {
    rc = head_dim == 64 ? launch_prefill<__nv_bfloat16, 64>(a, k_cache, v_cache, dtype, st)
                        : launch_prefill<__nv_bfloat16, 128>(a, k_cache, v_cache, dtype, st);
  } else {
    rc = head_dim == 64 ? launch_prefill<__half, 64>(a, k_cache, v_cache, dtype, st)
                        : launch_prefill<__half, 128>(a, k_cache, v_cache, dtype, st);
  }
  return rc == PKV_OK ? ok() : rc;
}
