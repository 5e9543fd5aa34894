// Library-wide host plumbing: error messages, version, device queries and the
// TMA tensor-map encoder (reached through the runtime's driver entry point, so
// the library links no driver stub and loads on machines without a GPU).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {
thread_local char g_message[512] = {0};

// One thread waits on an mbarrier that nothing completes, through the bounded wait
// every kernel of the library uses (ptx::mbar_wait); once it gives up it records
// PKV_DEV_WAIT_TIMEOUT and the time it waited, then completes the barrier's phase
// itself and waits again, which must succeed at once.
__global__ void wait_timeout_selftest_kernel(int32_t* status, int64_t* report,
                                             uint64_t limit_ns) {
  __shared__ alignas(8) uint64_t bar_word;
  if (threadIdx.x != 0) return;
  const uint32_t bar = ptx::smem_addr(&bar_word);
  ptx::mbar_init(bar, 1);
  ptx::fence_barrier_init();
  const uint64_t t0 = ptx::globaltimer_ns();
  const bool landed = ptx::mbar_wait(bar, 0, limit_ns);
  report[0] = static_cast<int64_t>(ptx::globaltimer_ns() - t0);
  if (!landed) atomicOr(status, PKV_DEV_WAIT_TIMEOUT);
  ptx::mbar_arrive(bar);
  report[1] = ptx::mbar_wait(bar, 0, limit_ns) ? 1 : 0;
}
}  // namespace

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_message, sizeof(g_message), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_message[0] = 0;
  return PKV_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s failed: %s (%s)", what, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

int device_sm_count(int* sms, int* device) {
  static std::once_flag flags[64];
  static int counts[64];
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::call_once(flags[dev], [&] {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
    counts[dev] = n;
  });
  if (counts[dev] <= 0) return fail(PKV_ERR_CUDA, "could not query the SM count of device %d", dev);
  *sms = counts[dev];
  *device = dev;
  return PKV_OK;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag flag;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(flag, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

int encode_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType type, int elt_bytes,
                  int64_t rows, int32_t cols, int32_t box_cols, int32_t box_rows,
                  CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elt_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PKV_OK;
}

int encode_cache_map(CUtensorMap* map, const void* base, int32_t dtype, int64_t rows,
                     int32_t cols, int32_t box_cols, int32_t box_rows) {
  CUtensorMapDataType dt;
  switch (dtype) {
    case PKV_F32: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; break;
    case PKV_F16: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; break;
    case PKV_BF16: dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; break;
    case PKV_FP8_E4M3:
    case PKV_INT8: dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;
    default: return fail(PKV_ERR_DTYPE, "unknown dtype %d", dtype);
  }
  return encode_map_2d(map, base, dt, element_bytes(dtype), rows, cols, box_cols, box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

int encode_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType type, int elt_bytes,
                  const int64_t dims[3], const int64_t strides[2], const int32_t box[3],
                  CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  (void)elt_bytes;
  const cuuint64_t d[3] = {static_cast<cuuint64_t>(dims[0]), static_cast<cuuint64_t>(dims[1]),
                           static_cast<cuuint64_t>(dims[2])};
  const cuuint64_t st[2] = {static_cast<cuuint64_t>(strides[0]),
                            static_cast<cuuint64_t>(strides[1])};
  const cuuint32_t bx[3] = {static_cast<cuuint32_t>(box[0]), static_cast<cuuint32_t>(box[1]),
                            static_cast<cuuint32_t>(box[2])};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, type, 3, const_cast<void*>(base), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
  return PKV_OK;
}

int encode_map_4d(CUtensorMap* map, const void* base, CUtensorMapDataType type,
                  const int64_t dims[4], const int64_t strides[3], const int32_t box[4],
                  CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t d[4], st[3];
  cuuint32_t bx[4];
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  for (int i = 0; i < 4; ++i) {
    d[i] = static_cast<cuuint64_t>(dims[i]);
    bx[i] = static_cast<cuuint32_t>(box[i]);
    if (i < 3) st[i] = static_cast<cuuint64_t>(strides[i]);
  }
  CUresult r = fn(map, type, 4, const_cast<void*>(base), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (4-D) failed (%d)", (int)r);
  return PKV_OK;
}

}  // namespace pkv

extern "C" {

const char* pkv_last_error_string(void) { return pkv::g_message; }

int pkv_version(void) { return 100; }

int pkv_wait_timeout_selftest(int32_t* status, int64_t* report, int32_t limit_us, void* stream) {
  PKV_REQUIRE(status != nullptr && report != nullptr, PKV_ERR_INVALID_ARG,
              "status and report must be device pointers");
  PKV_REQUIRE(limit_us >= 1 && limit_us <= 1000000, PKV_ERR_INVALID_ARG,
              "limit_us %d outside [1, 1000000]", limit_us);
  PKV_REQUIRE(pkv::aligned(report, 8) && pkv::aligned(status, 4), PKV_ERR_INVALID_ARG,
              "report must be 8-byte and status 4-byte aligned");
  pkv::wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, report, static_cast<uint64_t>(limit_us) * 1000u);
  PKV_CUDA(cudaGetLastError());
  return pkv::ok();
}

}  // extern "C"
