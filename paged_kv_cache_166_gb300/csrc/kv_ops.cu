// Cache write (scatter of new tokens into their slots) and whole-block copy for
// copy-on-write.  Both are pure data movement in 16-byte vectors: each thread
// moves one 16-byte piece of one row, so a warp covers contiguous bytes of a
// [head_dim] row on both sides.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace pkv {
namespace {

// For token t, KV head h, vector c of the row:
//   cache[slot / B, h, slot % B, c] = src[t, h, c]   (slot = slot_mapping[t] >= 0).
// The cache-write step of "PagedAttention and vLLM: Virtual Memory for the KV
// Cache", section "L2 — Mechanism" (allocation lifecycle), with the slot formula of
// "What is paged attention?", section "How it works".
__global__ void kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                const int32_t* __restrict__ slots, int64_t total_vecs,
                                int32_t Hkv, int32_t B, int32_t row_vecs, int64_t num_slots,
                                uint4* __restrict__ kc, uint4* __restrict__ vc) {
  // Let a decode-attention launch queued behind this write start its prologue now;
  // it orders its cache reads after this grid with griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_vecs;
       i += stride) {
    // The rows are loaded before the slot is known (i < total_vecs keeps them in
    // bounds), so the row and slot loads are in flight together: one memory round
    // trip before the stores instead of two.
    const uint4 kr = __ldg(k + i), vr = __ldg(v + i);
    const int64_t th = i / row_vecs;
    const int32_t c = static_cast<int32_t>(i - th * row_vecs);
    const int64_t t = th / Hkv;
    const int32_t h = static_cast<int32_t>(th - t * Hkv);
    const int32_t slot = __ldg(slots + t);
    if (slot < 0 || slot >= num_slots) continue;
    const int64_t dst = ((static_cast<int64_t>(slot / B) * Hkv + h) * B + slot % B) * row_vecs + c;
    kc[dst] = kr;
    vc[dst] = vr;
  }
}

// For pair p: block dst = pairs[2p+1] becomes a copy of block src = pairs[2p]
// ("allocates a new physical block, copies the content", "PagedAttention: How
// vLLM Borrowed Virtual Memory...", section "Copy-on-Write for Beam Search and
// Parallel Sampling").
__global__ void copy_blocks_kernel(uint4* __restrict__ kc, uint4* __restrict__ vc,
                                   const int32_t* __restrict__ pairs, int32_t n, int32_t NB,
                                   int64_t block_vecs) {
  const int64_t total = static_cast<int64_t>(n) * block_vecs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t p = i / block_vecs;
    const int64_t c = i - p * block_vecs;
    const int32_t src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
    if (src < 0 || src >= NB || dst < 0 || dst >= NB) continue;
    kc[dst * block_vecs + c] = kc[src * block_vecs + c];
    vc[dst * block_vecs + c] = vc[src * block_vecs + c];
  }
}

// The same copies in every layer's caches at once: a block id indexes the same
// block in each layer's tensors, so a copy-on-write pair applies to all of them.
// Work item i is vector c of pair p in layer l, layer outermost, so consecutive
// threads move consecutive bytes of one block.
struct LayerCaches {
  uint4* k[kMaxCopyLayers];
  uint4* v[kMaxCopyLayers];
};

__global__ void copy_blocks_layers_kernel(const __grid_constant__ LayerCaches caches, int32_t L,
                                          const int32_t* __restrict__ pairs, int32_t n,
                                          int32_t NB, int64_t block_vecs) {
  const int64_t per_layer = static_cast<int64_t>(n) * block_vecs;
  const int64_t total = per_layer * L;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int32_t l = static_cast<int32_t>(i / per_layer);
    const int64_t r = i - l * per_layer;
    const int64_t p = r / block_vecs;
    const int64_t c = r - p * block_vecs;
    const int32_t src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
    if (src < 0 || src >= NB || dst < 0 || dst >= NB) continue;
    uint4* const kc = caches.k[l];
    uint4* const vc = caches.v[l];
    kc[dst * block_vecs + c] = kc[src * block_vecs + c];
    vc[dst * block_vecs + c] = vc[src * block_vecs + c];
  }
}

// Decode-step cache write: sequence s's new token is its position t - 1, t = ctx[s];
// its slot comes from the block table, slot = table[s][(t-1) / B] * B + (t-1) % B
// ("What is paged attention?", section "How it works"), and its rows of every KV
// head are copied there.  Sequences with t <= 0 or t > max_blocks * B, and slots
// outside the pool, write nothing.
__global__ void decode_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                     const int32_t* __restrict__ tables, int32_t MAXB,
                                     const int32_t* __restrict__ ctx, int64_t total_vecs,
                                     int32_t Hkv, int32_t B, int32_t row_vecs, int32_t NB,
                                     uint4* __restrict__ kc, uint4* __restrict__ vc) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_vecs;
       i += stride) {
    const int64_t th = i / row_vecs;
    const int32_t c = static_cast<int32_t>(i - th * row_vecs);
    const int64_t s = th / Hkv;
    const int32_t h = static_cast<int32_t>(th - s * Hkv);
    // the rows do not depend on the slot: their loads go out with the slot lookups
    const uint4 kv = __ldg(k + i), vv = __ldg(v + i);
    const int32_t t = __ldg(ctx + s);
    if (t <= 0 || t > MAXB * B) continue;
    const int32_t b = __ldg(tables + s * MAXB + (t - 1) / B);
    if (b < 0 || b >= NB) continue;
    const int64_t dst = ((static_cast<int64_t>(b) * Hkv + h) * B + (t - 1) % B) * row_vecs + c;
    kc[dst] = kv;
    vc[dst] = vv;
  }
}

// ---- 8-bit (fp8 E4M3 or int8) quantising cache write --------------------------------
// Byte of token t (0..15) inside a 16-byte head_dim row of an 8-bit V tile: the
// tokens are stored in the order 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15.
__device__ __forceinline__ int fp8_v_pos(int t) {
  return t < 8 ? 4 * (t >> 1) + (t & 1) : 4 * ((t - 8) >> 1) + 2 + (t & 1);
}

// The bytes of 16 consecutive input elements (16-byte aligned source), loaded as
// they are: widened to fp32 by widen16 once they are needed.
template <typename Tin>
struct Raw16 {
  uint4 u[sizeof(Tin)];
};
template <typename Tin>
__device__ __forceinline__ Raw16<Tin> load_raw16(const Tin* p) {
  Raw16<Tin> r;
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(Tin)); ++i)
    r.u[i] = __ldg(reinterpret_cast<const uint4*>(p) + i);
  return r;
}
__device__ __forceinline__ void widen16(const Raw16<float>& r, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[4 * i] = __uint_as_float(r.u[i].x);
    x[4 * i + 1] = __uint_as_float(r.u[i].y);
    x[4 * i + 2] = __uint_as_float(r.u[i].z);
    x[4 * i + 3] = __uint_as_float(r.u[i].w);
  }
}
__device__ __forceinline__ void widen16(const Raw16<__half>& r, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w[4] = {r.u[i].x, r.u[i].y, r.u[i].z, r.u[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
      x[8 * i + 2 * j] = f.x;
      x[8 * i + 2 * j + 1] = f.y;
    }
  }
}
__device__ __forceinline__ void widen16(const Raw16<__nv_bfloat16>& r, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w[4] = {r.u[i].x, r.u[i].y, r.u[i].z, r.u[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
      x[8 * i + 2 * j] = f.x;
      x[8 * i + 2 * j + 1] = f.y;
    }
  }
}

// E4M3 codes of x[i] / scale, i < 16: the quotient a correctly rounded fp32
// division, then round to nearest even with saturation to +-448 (the hardware
// conversion); byte i of the result is element i.
__device__ __forceinline__ uint4 quantize16(const float (&x)[16], float scale) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 q = make_float2(__fdiv_rn(x[2 * j], scale), __fdiv_rn(x[2 * j + 1], scale));
    const uint32_t pair = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
    w[j >> 1] |= (pair & 0xffffu) << (16 * (j & 1));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// int8 codes of x[i] / scale, i < 16: the quotient a correctly rounded fp32
// division, rounded to the nearest integer with ties to even, clamped to
// [-127, 127]; NaN gives 0.  Byte i of the result is element i.
__device__ __forceinline__ uint4 quantize16_int8(const float (&x)[16], float scale) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float q = __fdiv_rn(x[j], scale);
    int c = __float2int_rn(q);           // saturates at the int range for +-inf
    c = q != q ? 0 : (c < -127 ? -127 : (c > 127 ? 127 : c));
    w[j >> 2] |= (static_cast<uint32_t>(c) & 0xffu) << (8 * (j & 3));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool kInt8>
__device__ __forceinline__ uint4 quantize16_as(const float (&x)[16], float scale) {
  if constexpr (kInt8) return quantize16_int8(x, scale);
  return quantize16(x, scale);
}

// Token i (or sequence i's new token, when slots is NULL: position ctx[i] - 1 of
// its block table) for KV head h, elements [16 c, 16 c + 16) of the row, with Q
// the E4M3 or the int8 quantisation:
//   K8[slot / 16, h, slot % 16, 16c + e]       = Q(k[i, h, 16c + e] / k_scale[h])
//   V8[slot / 16, h, 16c + e, V_POS[slot % 16]] = Q(v[i, h, 16c + e] / v_scale[h])
template <typename Tin, bool kInt8>
__global__ void kv_write_q8_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v,
                                    const int32_t* __restrict__ slots,
                                    const int32_t* __restrict__ tables, int32_t MAXB,
                                    const int32_t* __restrict__ ctx, int64_t total, int32_t Hkv,
                                    int32_t D, int32_t NB, const float* __restrict__ ks,
                                    const float* __restrict__ vs, uint8_t* __restrict__ kc,
                                    uint8_t* __restrict__ vc) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int groups = D / 16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t th = i / groups;
    const int32_t c = static_cast<int32_t>(i - th * groups);
    const int64_t t = th / Hkv;
    const int32_t h = static_cast<int32_t>(th - t * Hkv);
    // The rows and scales do not depend on the slot, and th * D + 16 * c = 16 i lies
    // inside the [total * 16] inputs: their loads go out with the slot lookup's.
    const Raw16<Tin> rk = load_raw16(k + th * D + 16 * c), rv = load_raw16(v + th * D + 16 * c);
    const float sk = __ldg(ks + h), sv = __ldg(vs + h);
    int32_t slot;
    if (slots != nullptr) {
      slot = __ldg(slots + t);
      if (slot < 0 || slot >= NB * 16) continue;
    } else {
      const int32_t n = __ldg(ctx + t);
      if (n <= 0 || n > MAXB * 16) continue;
      const int32_t b = __ldg(tables + t * MAXB + (n - 1) / 16);
      if (b < 0 || b >= NB) continue;
      slot = b * 16 + (n - 1) % 16;
    }
    const int64_t tile = static_cast<int64_t>(slot / 16) * Hkv + h;
    const int32_t off = slot % 16;
    float x[16];
    widen16(rk, x);
    *reinterpret_cast<uint4*>(kc + (tile * 16 + off) * D + 16 * c) = quantize16_as<kInt8>(x, sk);
    widen16(rv, x);
    const uint4 q = quantize16_as<kInt8>(x, sv);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint8_t* const col = vc + (tile * D + 16 * c) * 16 + fp8_v_pos(off);
#pragma unroll
    for (int e = 0; e < 16; ++e) col[e * 16] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
  }
}

// Preemption by swapping ("PagedAttention — how vLLM stopped wasting 80% of your
// GPU memory", section "Preemption: what happens when memory runs out anyway"):
// out: host block i = cache block ids[i];  in: cache block ids[i] = host block i,
// for K and V, whole blocks, 16-byte vectors.  Host buffers are page-locked host
// memory the kernel reads or writes directly (over the CPU-GPU link).  Ids
// outside [0, NB) are skipped.
__global__ void swap_blocks_kernel(const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                                   uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                                   const int32_t* __restrict__ ids, int32_t n, int32_t NB,
                                   int64_t block_vecs, bool to_host) {
  const int64_t total = static_cast<int64_t>(n) * block_vecs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t p = i / block_vecs;
    const int64_t c = i - p * block_vecs;
    const int32_t b = __ldg(ids + p);
    if (b < 0 || b >= NB) continue;
    const int64_t cache_at = static_cast<int64_t>(b) * block_vecs + c;
    const int64_t host_at = p * block_vecs + c;
    if (to_host) {
      dst_k[host_at] = __ldcs(src_k + cache_at);
      dst_v[host_at] = __ldcs(src_v + cache_at);
    } else {
      dst_k[cache_at] = __ldcs(src_k + host_at);
      dst_v[cache_at] = __ldcs(src_v + host_at);
    }
  }
}

int grid_for(int64_t work, int threads) {
  int sms = 0, dev = 0;
  if (device_sm_count(&sms, &dev) != PKV_OK) sms = 132;
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

int launch_kv_write_q8(const void* k, const void* v, const int32_t* slot_mapping,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t num_tokens, void* k_cache,
                       void* v_cache, const float* k_scale, const float* v_scale,
                       int32_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                       int32_t dtype, int32_t codes, void* stream) {
  PKV_REQUIRE(dtype == PKV_F32 || dtype == PKV_F16 || dtype == PKV_BF16, PKV_ERR_DTYPE,
              "input dtype %d is not f32, f16 or bf16", dtype);
  PKV_REQUIRE(codes == PKV_FP8_E4M3 || codes == PKV_INT8, PKV_ERR_DTYPE,
              "cache code %d is not PKV_FP8_E4M3 or PKV_INT8", codes);
  PKV_REQUIRE(num_tokens >= 0 && num_blocks > 0 && num_kv_heads > 0 && head_dim > 0 &&
                  head_dim % 16 == 0,
              PKV_ERR_INVALID_ARG, "bad sizes (head_dim must be a positive multiple of 16)");
  PKV_REQUIRE(static_cast<int64_t>(num_blocks) * 16 < (int64_t(1) << 31), PKV_ERR_INVALID_ARG,
              "num_blocks * 16 must be < 2^31");
  if (num_tokens == 0) return PKV_OK;
  PKV_REQUIRE(k && v && k_cache && v_cache && k_scale && v_scale, PKV_ERR_INVALID_ARG,
              "NULL pointer");
  PKV_REQUIRE(slot_mapping || (block_tables && context_lens), PKV_ERR_INVALID_ARG,
              "NULL slot mapping / block tables");
  PKV_REQUIRE(aligned(k, 16) && aligned(v, 16) && aligned(k_cache, 16) && aligned(v_cache, 16),
              PKV_ERR_INVALID_ARG, "k, v and caches must be 16-byte aligned");
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim / 16);
  const int threads = 256;
  const dim3 grid(grid_for(total, threads));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
#define PKV_Q8_WRITE(TT, I8)                                                                \
  kv_write_q8_kernel<TT, I8><<<grid, threads, 0, st>>>(                                     \
      static_cast<const TT*>(k), static_cast<const TT*>(v), slot_mapping, block_tables,     \
      max_blocks_per_seq, context_lens, total, num_kv_heads, head_dim, num_blocks, k_scale, \
      v_scale, kc, vc)
  const bool i8 = codes == PKV_INT8;
  if (dtype == PKV_F32) {
    if (i8) PKV_Q8_WRITE(float, true); else PKV_Q8_WRITE(float, false);
  } else if (dtype == PKV_F16) {
    if (i8) PKV_Q8_WRITE(__half, true); else PKV_Q8_WRITE(__half, false);
  } else {
    if (i8) PKV_Q8_WRITE(__nv_bfloat16, true); else PKV_Q8_WRITE(__nv_bfloat16, false);
  }
#undef PKV_Q8_WRITE
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

// Device address of a page-locked (or managed) host buffer, or an error if the
// device cannot address it.
int host_buffer_device_ptr(const void* host, void** dev_ptr) {
  cudaPointerAttributes attr{};
  PKV_CUDA(cudaPointerGetAttributes(&attr, host));
  PKV_REQUIRE(attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeManaged,
              PKV_ERR_INVALID_ARG,
              "host buffer %p is not page-locked or managed memory (type %d)", host,
              static_cast<int>(attr.type));
  PKV_REQUIRE(attr.devicePointer != nullptr, PKV_ERR_INVALID_ARG,
              "host buffer %p is not mapped into the device address space", host);
  *dev_ptr = attr.devicePointer;
  return PKV_OK;
}

// Swapping of every layer's caches in one launch: host buffer of layer l holds its
// n blocks at [l * n, (l + 1) * n) (layer-major), so layer l's block i of the id
// list is host block l * n + i.  Layer outermost, as in the multi-layer copy.
__global__ void swap_blocks_layers_kernel(const __grid_constant__ LayerCaches caches, int32_t L,
                                          uint4* __restrict__ host_k, uint4* __restrict__ host_v,
                                          const int32_t* __restrict__ ids, int32_t n, int32_t NB,
                                          int64_t block_vecs, bool to_host) {
  const int64_t per_layer = static_cast<int64_t>(n) * block_vecs;
  const int64_t total = per_layer * L;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int32_t l = static_cast<int32_t>(i / per_layer);
    const int64_t r = i - l * per_layer;
    const int64_t p = r / block_vecs;
    const int64_t c = r - p * block_vecs;
    const int32_t b = __ldg(ids + p);
    if (b < 0 || b >= NB) continue;
    const int64_t cache_at = static_cast<int64_t>(b) * block_vecs + c;
    uint4* const kc = caches.k[l];
    uint4* const vc = caches.v[l];
    if (to_host) {
      host_k[i] = __ldcs(kc + cache_at);
      host_v[i] = __ldcs(vc + cache_at);
    } else {
      kc[cache_at] = __ldcs(host_k + i);
      vc[cache_at] = __ldcs(host_v + i);
    }
  }
}

int launch_swap_layers(const void* const* k_caches, const void* const* v_caches, int32_t L,
                       void* host_k, void* host_v, const int32_t* ids, int32_t n, int32_t NB,
                       int64_t block_bytes, bool to_host, void* stream) {
  PKV_REQUIRE(L >= 1 && L <= kMaxCopyLayers, PKV_ERR_UNSUPPORTED, "num_layers %d outside [1, %d]",
              L, kMaxCopyLayers);
  PKV_REQUIRE(n >= 0 && NB > 0 && block_bytes > 0 && block_bytes % 16 == 0, PKV_ERR_INVALID_ARG,
              "bad sizes (block_bytes must be a positive multiple of 16)");
  PKV_REQUIRE(k_caches && v_caches, PKV_ERR_INVALID_ARG, "NULL cache list");
  LayerCaches caches{};
  for (int l = 0; l < L; ++l) {
    PKV_REQUIRE(k_caches[l] && v_caches[l], PKV_ERR_INVALID_ARG, "NULL cache of layer %d", l);
    PKV_REQUIRE(aligned(k_caches[l], 16) && aligned(v_caches[l], 16), PKV_ERR_INVALID_ARG,
                "caches of layer %d must be 16-byte aligned", l);
    caches.k[l] = static_cast<uint4*>(const_cast<void*>(k_caches[l]));
    caches.v[l] = static_cast<uint4*>(const_cast<void*>(v_caches[l]));
  }
  if (n == 0) return PKV_OK;
  PKV_REQUIRE(host_k && host_v && ids, PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(aligned(host_k, 16) && aligned(host_v, 16), PKV_ERR_INVALID_ARG,
              "host buffers must be 16-byte aligned");
  void *dk = nullptr, *dv = nullptr;
  int rc = host_buffer_device_ptr(host_k, &dk);
  if (rc != PKV_OK) return rc;
  rc = host_buffer_device_ptr(host_v, &dv);
  if (rc != PKV_OK) return rc;
  const int64_t block_vecs = block_bytes / 16;
  const int threads = 256;
  swap_blocks_layers_kernel<<<grid_for(static_cast<int64_t>(L) * n * block_vecs, threads), threads,
                              0, static_cast<cudaStream_t>(stream)>>>(
      caches, L, static_cast<uint4*>(dk), static_cast<uint4*>(dv), ids, n, NB, block_vecs,
      to_host);
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

int launch_swap(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                const int32_t* ids, int32_t n, int32_t NB, int64_t block_bytes, bool to_host,
                void* stream) {
  PKV_REQUIRE(n >= 0 && NB > 0 && block_bytes > 0 && block_bytes % 16 == 0, PKV_ERR_INVALID_ARG,
              "bad sizes (block_bytes must be a positive multiple of 16)");
  if (n == 0) return PKV_OK;
  PKV_REQUIRE(src_k && src_v && dst_k && dst_v && ids, PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(aligned(src_k, 16) && aligned(src_v, 16) && aligned(dst_k, 16) && aligned(dst_v, 16),
              PKV_ERR_INVALID_ARG, "caches and host buffers must be 16-byte aligned");
  const void* hk = to_host ? dst_k : src_k;
  const void* hv = to_host ? dst_v : src_v;
  void *dk = nullptr, *dv = nullptr;
  int rc = host_buffer_device_ptr(hk, &dk);
  if (rc != PKV_OK) return rc;
  rc = host_buffer_device_ptr(hv, &dv);
  if (rc != PKV_OK) return rc;
  const int64_t block_vecs = block_bytes / 16;
  const int threads = 256;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (to_host) {
    swap_blocks_kernel<<<grid_for(n * block_vecs, threads), threads, 0, st>>>(
        static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v),
        static_cast<uint4*>(dk), static_cast<uint4*>(dv), ids, n, NB, block_vecs, true);
  } else {
    swap_blocks_kernel<<<grid_for(n * block_vecs, threads), threads, 0, st>>>(
        static_cast<const uint4*>(dk), static_cast<const uint4*>(dv), static_cast<uint4*>(dst_k),
        static_cast<uint4*>(dst_v), ids, n, NB, block_vecs, false);
  }
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

int launch_decode_append(const void* k_new, const void* v_new, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                         void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                         int32_t block_size, int32_t head_dim, int32_t dtype, void* stream) {
  const int elt = element_bytes(dtype);
  PKV_REQUIRE(elt != 0, PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  PKV_REQUIRE(k_new && v_new, PKV_ERR_INVALID_ARG, "NULL k_new / v_new");
  PKV_REQUIRE(aligned(k_new, 16) && aligned(v_new, 16), PKV_ERR_INVALID_ARG,
              "k_new and v_new must be 16-byte aligned");
  PKV_REQUIRE((static_cast<int64_t>(head_dim) * elt) % 16 == 0, PKV_ERR_INVALID_ARG,
              "head_dim * element size must be a multiple of 16 bytes");
  const int32_t row_vecs = static_cast<int32_t>(static_cast<int64_t>(head_dim) * elt / 16);
  const int64_t total = static_cast<int64_t>(num_seqs) * num_kv_heads * row_vecs;
  const int threads = 256;
  decode_append_kernel<<<grid_for(total, threads), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables,
      max_blocks_per_seq, context_lens, total, num_kv_heads, block_size, row_vecs, num_blocks,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache));
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_kv_write(const void* k, const void* v, const int32_t* slot_mapping, int32_t num_tokens,
                 void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                 int32_t block_size, int32_t head_dim, int32_t dtype, void* stream) {
  const int elt = element_bytes(dtype);
  PKV_REQUIRE(elt != 0, PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  PKV_REQUIRE(dtype != PKV_FP8_E4M3 && dtype != PKV_INT8, PKV_ERR_DTYPE,
              "8-bit caches are written by pkv_kv_write_fp8 / _int8 (quantising, V tiles "
              "transposed)");
  PKV_REQUIRE(num_tokens >= 0 && num_blocks > 0 && num_kv_heads > 0 && block_size > 0 &&
                  head_dim > 0,
              PKV_ERR_INVALID_ARG, "sizes must be positive (num_tokens >= 0)");
  PKV_REQUIRE((static_cast<int64_t>(head_dim) * elt) % 16 == 0, PKV_ERR_INVALID_ARG,
              "head_dim * element size must be a multiple of 16 bytes");
  PKV_REQUIRE(static_cast<int64_t>(num_blocks) * block_size < (int64_t(1) << 31),
              PKV_ERR_INVALID_ARG, "num_blocks * block_size must be < 2^31");
  if (num_tokens == 0) return ok();
  PKV_REQUIRE(k && v && slot_mapping && k_cache && v_cache, PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(aligned(k, 16) && aligned(v, 16) && aligned(k_cache, 16) && aligned(v_cache, 16),
              PKV_ERR_INVALID_ARG, "k, v and caches must be 16-byte aligned");
  const int32_t row_vecs = static_cast<int32_t>(static_cast<int64_t>(head_dim) * elt / 16);
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * row_vecs;
  const int threads = 256;
  kv_write_kernel<<<grid_for(total, threads), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, total,
      num_kv_heads, block_size, row_vecs, static_cast<int64_t>(num_blocks) * block_size,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache));
  PKV_CUDA(cudaGetLastError());
  return ok();
}

namespace {
int kv_write_q8_entry(int32_t codes, const void* k, const void* v, const int32_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache, const float* k_scale,
                      const float* v_scale, int32_t num_blocks, int32_t num_kv_heads,
                      int32_t block_size, int32_t head_dim, int32_t dtype, void* stream) {
  PKV_REQUIRE(block_size == 16, PKV_ERR_UNSUPPORTED, "8-bit caches use block_size 16, not %d",
              block_size);
  PKV_REQUIRE(num_tokens == 0 || slot_mapping, PKV_ERR_INVALID_ARG, "NULL slot_mapping");
  const int rc = launch_kv_write_q8(k, v, slot_mapping, nullptr, 0, nullptr, num_tokens, k_cache,
                                    v_cache, k_scale, v_scale, num_blocks, num_kv_heads,
                                    head_dim, dtype, codes, stream);
  return rc == PKV_OK ? ok() : rc;
}
}  // namespace

int pkv_kv_write_fp8(const void* k, const void* v, const int32_t* slot_mapping,
                     int32_t num_tokens, void* k_cache, void* v_cache, const float* k_scale,
                     const float* v_scale, int32_t num_blocks, int32_t num_kv_heads,
                     int32_t block_size, int32_t head_dim, int32_t dtype, void* stream) {
  return kv_write_q8_entry(PKV_FP8_E4M3, k, v, slot_mapping, num_tokens, k_cache, v_cache,
                           k_scale, v_scale, num_blocks, num_kv_heads, block_size, head_dim,
                           dtype, stream);
}

int pkv_kv_write_int8(const void* k, const void* v, const int32_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache, const float* k_scale,
                      const float* v_scale, int32_t num_blocks, int32_t num_kv_heads,
                      int32_t block_size, int32_t head_dim, int32_t dtype, void* stream) {
  return kv_write_q8_entry(PKV_INT8, k, v, slot_mapping, num_tokens, k_cache, v_cache, k_scale,
                           v_scale, num_blocks, num_kv_heads, block_size, head_dim, dtype,
                           stream);
}

int pkv_swap_out_blocks(const void* k_cache, const void* v_cache, const int32_t* block_ids,
                        int32_t num_ids, int32_t num_blocks, int64_t block_bytes, void* host_k,
                        void* host_v, void* stream) {
  const int rc = launch_swap(k_cache, v_cache, host_k, host_v, block_ids, num_ids, num_blocks,
                             block_bytes, true, stream);
  return rc == PKV_OK ? ok() : rc;
}

int pkv_swap_out_blocks_layers(const void* const* k_caches, const void* const* v_caches,
                               int32_t num_layers, const int32_t* block_ids, int32_t num_ids,
                               int32_t num_blocks, int64_t block_bytes, void* host_k,
                               void* host_v, void* stream) {
  const int rc = launch_swap_layers(k_caches, v_caches, num_layers, host_k, host_v, block_ids,
                                    num_ids, num_blocks, block_bytes, true, stream);
  return rc == PKV_OK ? ok() : rc;
}

int pkv_swap_in_blocks_layers(const void* host_k, const void* host_v, const int32_t* block_ids,
                              int32_t num_ids, int32_t num_blocks, int64_t block_bytes,
                              void* const* k_caches, void* const* v_caches, int32_t num_layers,
                              void* stream) {
  const int rc = launch_swap_layers(const_cast<const void* const*>(k_caches),
                                    const_cast<const void* const*>(v_caches), num_layers,
                                    const_cast<void*>(host_k), const_cast<void*>(host_v),
                                    block_ids, num_ids, num_blocks, block_bytes, false, stream);
  return rc == PKV_OK ? ok() : rc;
}

int pkv_swap_in_blocks(const void* host_k, const void* host_v, const int32_t* block_ids,
                       int32_t num_ids, int32_t num_blocks, int64_t block_bytes, void* k_cache,
                       void* v_cache, void* stream) {
  const int rc = launch_swap(host_k, host_v, k_cache, v_cache, block_ids, num_ids, num_blocks,
                             block_bytes, false, stream);
  return rc == PKV_OK ? ok() : rc;
}

int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst_pairs, int32_t num_pairs,
                    int32_t num_blocks, int64_t block_elems, int32_t dtype, void* stream) {
  const int elt = element_bytes(dtype);
  PKV_REQUIRE(elt != 0, PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  PKV_REQUIRE(num_pairs >= 0 && num_blocks > 0 && block_elems > 0, PKV_ERR_INVALID_ARG,
              "bad sizes");
  PKV_REQUIRE((block_elems * elt) % 16 == 0, PKV_ERR_INVALID_ARG,
              "block_elems * element size must be a multiple of 16 bytes");
  if (num_pairs == 0) return ok();
  PKV_REQUIRE(k_cache && v_cache && src_dst_pairs, PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(aligned(k_cache, 16) && aligned(v_cache, 16), PKV_ERR_INVALID_ARG,
              "caches must be 16-byte aligned");
  const int64_t block_vecs = block_elems * elt / 16;
  const int threads = 256;
  copy_blocks_kernel<<<grid_for(num_pairs * block_vecs, threads), threads, 0,
                       static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src_dst_pairs, num_pairs,
      num_blocks, block_vecs);
  PKV_CUDA(cudaGetLastError());
  return ok();
}

int pkv_copy_blocks_layers(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                           const int32_t* src_dst_pairs, int32_t num_pairs, int32_t num_blocks,
                           int64_t block_elems, int32_t dtype, void* stream) {
  const int elt = element_bytes(dtype);
  PKV_REQUIRE(elt != 0, PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  PKV_REQUIRE(num_layers >= 1 && num_layers <= kMaxCopyLayers, PKV_ERR_UNSUPPORTED,
              "num_layers %d outside [1, %d]", num_layers, kMaxCopyLayers);
  PKV_REQUIRE(num_pairs >= 0 && num_blocks > 0 && block_elems > 0, PKV_ERR_INVALID_ARG,
              "bad sizes");
  PKV_REQUIRE((block_elems * elt) % 16 == 0, PKV_ERR_INVALID_ARG,
              "block_elems * element size must be a multiple of 16 bytes");
  PKV_REQUIRE(k_caches && v_caches, PKV_ERR_INVALID_ARG, "NULL cache list");
  LayerCaches caches{};
  for (int l = 0; l < num_layers; ++l) {
    PKV_REQUIRE(k_caches[l] && v_caches[l], PKV_ERR_INVALID_ARG, "NULL cache of layer %d", l);
    PKV_REQUIRE(aligned(k_caches[l], 16) && aligned(v_caches[l], 16), PKV_ERR_INVALID_ARG,
                "caches of layer %d must be 16-byte aligned", l);
    caches.k[l] = static_cast<uint4*>(k_caches[l]);
    caches.v[l] = static_cast<uint4*>(v_caches[l]);
  }
  if (num_pairs == 0) return ok();
  PKV_REQUIRE(src_dst_pairs, PKV_ERR_INVALID_ARG, "NULL pointer");
  const int64_t block_vecs = block_elems * elt / 16;
  const int threads = 256;
  const int64_t work = static_cast<int64_t>(num_layers) * num_pairs * block_vecs;
  copy_blocks_layers_kernel<<<grid_for(work, threads), threads, 0,
                              static_cast<cudaStream_t>(stream)>>>(
      caches, num_layers, src_dst_pairs, num_pairs, num_blocks, block_vecs);
  PKV_CUDA(cudaGetLastError());
  return ok();
}

}  // extern "C"
