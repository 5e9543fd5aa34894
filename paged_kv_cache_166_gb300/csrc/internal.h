// Host-side helpers shared by the library's CUDA translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv.h"
#include "status.h"

namespace pkv {

inline int element_bytes(int32_t dtype) {
  switch (dtype) {
    case PKV_F32: return 4;
    case PKV_F16: return 2;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
    case PKV_INT8: return 1;
    default: return 0;
  }
}

// Records a failed CUDA call and returns PKV_ERR_CUDA.
int cuda_fail(cudaError_t e, const char* what);

#define PKV_CUDA(call)                                      \
  do {                                                      \
    cudaError_t e_ = (call);                                \
    if (e_ != cudaSuccess) return ::pkv::cuda_fail(e_, #call); \
  } while (0)

// Layers one pkv_copy_blocks_layers launch takes (their cache pointers travel as
// kernel parameters: 2 x 128 x 8 bytes).
constexpr int kMaxCopyLayers = 128;

// Number of SMs of the current device (cached per device).
int device_sm_count(int* sms, int* device);

// Encodes a 2-D TMA map over a cache viewed as [rows, cols] (rows contiguous,
// cols elements each), boxes of [box_rows x box_cols elements], 128-byte swizzle.
int encode_cache_map(CUtensorMap* map, const void* base, int32_t dtype, int64_t rows,
                     int32_t cols, int32_t box_cols, int32_t box_rows);

// The same for any element type and swizzle mode.
int encode_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType type, int elt_bytes,
                  int64_t rows, int32_t cols, int32_t box_cols, int32_t box_rows,
                  CUtensorMapSwizzle swizzle);

// A 3-D map: dims innermost first, byte strides of dims 1 and 2, box innermost first.
int encode_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType type, int elt_bytes,
                  const int64_t dims[3], const int64_t strides[2], const int32_t box[3],
                  CUtensorMapSwizzle swizzle);

// A 4-D map, laid out as the 3-D one.  The byte strides need not increase with the
// dimension: a box then lands in shared memory in the order of the map's dims,
// which is how a caller reorders the axes of a tile on the way in.
int encode_map_4d(CUtensorMap* map, const void* base, CUtensorMapDataType type,
                  const int64_t dims[4], const int64_t strides[3], const int32_t box[4],
                  CUtensorMapSwizzle swizzle);

// Launches the 8-bit quantising cache write (kv_ops.cu); codes is PKV_FP8_E4M3
// or PKV_INT8.  With slot_mapping set, token i goes to slot_mapping[i]; with it
// NULL, sequence i's token goes to slot(t - 1) of its block table,
// t = context_lens[i] (the decode-step append).
int launch_kv_write_q8(const void* k, const void* v, const int32_t* slot_mapping,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t num_tokens, void* k_cache,
                       void* v_cache, const float* k_scale, const float* v_scale,
                       int32_t num_blocks, int32_t num_kv_heads, int32_t head_dim,
                       int32_t dtype, int32_t codes, void* stream);

// Launches the decode-step cache write: for every sequence s with t = ctx[s] > 0,
// the rows k_new[s], v_new[s] go to slot(t - 1) of its block table (kv_ops.cu).
int launch_decode_append(const void* k_new, const void* v_new, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                         void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                         int32_t block_size, int32_t head_dim, int32_t dtype, void* stream);

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace pkv
