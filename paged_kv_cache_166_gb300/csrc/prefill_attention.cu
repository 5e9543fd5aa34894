// Paged (chunked) prefill attention for sm_103a: the entry point.
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
// The kernel runs on the 5th-generation tensor cores (tcgen05 MMAs with
// tensor-memory accumulators, TMA-fed K/V rings; prefill_tcgen05.cu).  This file
// checks the arguments and launches it.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "prefill_common.cuh"

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
  PKV_REQUIRE(block_size == 8 || block_size == 16 || block_size == 32, PKV_ERR_UNSUPPORTED,
              "block_size %d not in {8, 16, 32}", block_size);
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
  const int rc = launch_prefill_tc(a, k_cache, v_cache, dtype, head_dim,
                                   static_cast<cudaStream_t>(stream));
  return rc == PKV_OK ? ok() : rc;
}
