// Definitions shared by the paged prefill entry point (prefill_attention.cu) and
// its kernel (prefill_tcgen05.cu): the launch arguments, the per-sequence length
// checks and the device status word.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "pkv.h"

namespace pkv {

constexpr int kPfMaxSeqs = 2048;
constexpr uint64_t kPfWaitNs = 1000000000ull;  // 1 s per wait before giving up

struct PrefillArgs {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  int32_t* status;  // device status word, may be NULL
  int32_t S, T, Hq, Hkv, G, MAXB, NB;  // T: rows of q and out
  int32_t bs;                          // tokens per cache block
  float scale_log2;
};

__device__ __forceinline__ void pf_flag(const PrefillArgs& a, int bits) {
  if (a.status) atomicOr(a.status, bits);
}

// Context t, chunk length c and first query row q0 of sequence s, clamped to
// 0 <= c <= t <= MAXB * bs and 0 <= q0, q0 + c <= T (a clamp is reported once,
// by the caller that passes report).
__device__ __forceinline__ void pf_seq(const PrefillArgs& a, int s, int& t, int& c, int& q0,
                                       bool report) {
  t = __ldg(a.context_lens + s);
  q0 = __ldg(a.query_start + s);
  c = __ldg(a.query_start + s + 1) - q0;
  const int limit = a.MAXB * a.bs;
  if (t < 0 || t > limit || c < 0 || c > t || q0 < 0 || q0 > a.T || c > a.T - q0) {
    if (report) pf_flag(a, PKV_DEV_BAD_CONTEXT_LEN);
    t = t < 0 ? 0 : (t > limit ? limit : t);
    q0 = q0 < 0 ? 0 : (q0 > a.T ? a.T : q0);
    c = c < 0 ? 0 : c;
    c = c > t ? t : c;
    c = c > a.T - q0 ? a.T - q0 : c;
  }
}

// Launches the tensor-core (tcgen05) prefill kernel (prefill_tcgen05.cu).
int launch_prefill_tc(const PrefillArgs& a, const void* k_cache, const void* v_cache,
                      int32_t dtype, int32_t head_dim, cudaStream_t stream);

}  // namespace pkv
