/*
 * pkv.h — C ABI of the GB300 paged KV-cache decode library (libpkv.so).
 *
 * The library implements the data-parallel hot path of PagedAttention:
 *   - the cache write that scatters each new token's K and V into its slot,
 *   - single-token decode attention read through per-sequence block tables,
 *     split over the context and merged with a log-sum-exp reduce, alone or as
 *     one decode step together with the write of each sequence's new token,
 *   - the whole-block copy that copy-on-write needs (one layer, or every layer
 *     in one launch),
 *   - a host-side block manager (O(1) free list, per-block refcounts, fork,
 *     append with copy-on-write, free, swap out and in),
 * and beyond it: fp8 (E4M3) and int8 caches (quantising write, decode over the
 * codes), swapping of blocks to and from page-locked host memory, and causal
 * prefill attention over the paged cache on the 5th-generation tensor cores.
 *
 * Conventions (all entry points):
 *   - Every function returns an int status: PKV_OK (0) or a negative PKV_ERR_*.
 *     No C++ exception crosses the ABI.  pkv_last_error_string() returns a
 *     thread-local message describing the last failure in the calling thread.
 *   - Device pointers are plain CUDA device addresses owned by the caller; the
 *     library never allocates or frees device memory.  Host pointers are
 *     caller-owned host memory.  Block-manager handles are owned by the library
 *     and released with pkv_allocator_destroy.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device calls
 *     only enqueue work on it and return; results are ready once the stream is
 *     synchronised.  A status of PKV_ERR_CUDA means a launch or API call failed.
 *   - Cache layout (per layer, K and V as two separate tensors):
 *       [num_blocks, num_kv_heads, block_size, head_dim], row-major, contiguous,
 *     the layout "PagedAttention: How vLLM Borrowed Virtual Memory to Unlock GPU
 *     Serving at Scale" gives in section "The Custom CUDA Kernel".  One physical
 *     block id indexes the same block in every layer's tensors.
 *   - Slot of logical position p of a sequence with block table bt:
 *       slot(p) = bt[p / block_size] * block_size + p % block_size
 *     ("What is paged attention?", section "How it works").  Token slot s lives at
 *     cache[s / block_size, :, s % block_size, :].
 *   - dtype codes: PKV_F32, PKV_F16, PKV_BF16; q, out, k, v and the caches share
 *     one dtype, except on the 8-bit cache entry points (sections "fp8 KV cache"
 *     and "int8 KV cache").  Index tensors are int32.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = -1,  /* bad pointer, size, shape, alignment or id */
  PKV_ERR_DTYPE = -2,        /* unknown dtype code */
  PKV_ERR_OUT_OF_BLOCKS = -3,/* block manager cannot serve the request; state unchanged */
  PKV_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed (see message) */
  PKV_ERR_UNSUPPORTED = -5,  /* valid request outside what the kernels implement */
  PKV_ERR_DEVICE = -6        /* a kernel reported a device-side error (see pkv_decode_status) */
};

enum pkv_dtype {
  PKV_F32 = 0,
  PKV_F16 = 1,
  PKV_BF16 = 2,
  PKV_FP8_E4M3 = 3, /* 8-bit quantised cache elements; only where an entry point says so */
  PKV_INT8 = 4      /* the same, as int8 codes */
};

/* Device-side status bits recorded by the decode kernels in the workspace. */
enum pkv_device_status {
  PKV_DEV_BAD_CONTEXT_LEN = 1, /* a context length was < 0 or > max_blocks_per_seq * block_size; clamped */
  PKV_DEV_BAD_BLOCK_ID = 2,    /* a block-table entry was outside [0, num_blocks); read as zeros */
  PKV_DEV_WAIT_TIMEOUT = 4,    /* a copy into shared memory did not complete within ~1 s; unit skipped */
  PKV_DEV_WORKSPACE_MISMATCH = 8 /* the workspace was last used with another (num_warps, group, head_dim) */
};

/* Message of the last failure in this thread ("" if none).  Never NULL. */
const char* pkv_last_error_string(void);

/* Library version, encoded as major*10000 + minor*100 + patch. */
int pkv_version(void);

/*
 * pkv_wait_timeout_selftest — exercises on the current device the bounded wait that
 * every kernel of the library uses on its mbarriers (TMA copies, tensor-core commits,
 * hand-offs between warps), without a fault: one thread waits on an mbarrier that
 * nothing completes, gives up after limit_us microseconds, ORs PKV_DEV_WAIT_TIMEOUT
 * into *status and writes the nanoseconds it waited to report[0]; it then completes
 * the barrier's phase itself and waits again, writing 1 to report[1] if that wait
 * succeeded.  A healthy device ends with the bit set, report[0] >= limit_us * 1000 and
 * report[1] == 1, and stays usable afterwards.
 * status   device int32 word, 4-byte aligned (bits are ORed in, never cleared).
 * report   device int64 [2], 8-byte aligned.
 * limit_us 1 .. 1,000,000.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA.
 */
int pkv_wait_timeout_selftest(int32_t* status, int64_t* report, int32_t limit_us, void* stream);

/* ------------------------------------------------------------------------- */
/* Cache write                                                                */
/* ------------------------------------------------------------------------- */

/*
 * pkv_kv_write — scatter new tokens' K and V into their cache slots.
 *
 * Follows the decode step "write the new token's K,V into the last block"
 * ("PagedAttention and vLLM: Virtual Memory for the KV Cache", section
 * "L2 — Mechanism", allocation lifecycle) with the slot formula above:
 *   for i < num_tokens, h < num_kv_heads with s = slot_mapping[i] >= 0:
 *     k_cache[s / block_size, h, s % block_size, :] = k[i, h, :]   (bit copy)
 *     v_cache[s / block_size, h, s % block_size, :] = v[i, h, :]
 *
 * k, v          device, [num_tokens, num_kv_heads, head_dim], contiguous.
 * slot_mapping  device int32 [num_tokens].  A negative slot marks a padding
 *               token and writes nothing.  Slots >= num_blocks*block_size are
 *               skipped.  Two tokens with the same slot: the result is one of
 *               the two rows (unspecified which).
 * k_cache, v_cache  device caches in the layout above, updated in place.
 * Requirements: head_dim * element size a multiple of 16 bytes; all pointers
 * 16-byte aligned; num_blocks*block_size < 2^31.  num_tokens == 0 is a no-op.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_DTYPE, PKV_ERR_CUDA.
 */
int pkv_kv_write(const void* k, const void* v, const int32_t* slot_mapping, int32_t num_tokens,
                 void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                 int32_t block_size, int32_t head_dim, int32_t dtype, void* stream);

/* ------------------------------------------------------------------------- */
/* Decode attention                                                           */
/* ------------------------------------------------------------------------- */

/*
 * pkv_decode_workspace_size — bytes of device workspace pkv_decode_attention needs.
 *
 * The workspace holds a status word, one merge ticket per worker warp and the
 * per-piece softmax partial states of contexts that are split across warps.  Its
 * size depends only on the head shape, the dtype and the number of worker warps
 * the launch uses (num_warps; 0 = the default for the current device), never on
 * the context lengths or the batch.  A workspace belongs to one layout, i.e. one
 * (num_q_heads / num_kv_heads, head_dim, num_warps): zero-fill it before its first
 * use and before using it under another layout (a launch that finds another
 * layout's leftovers sets PKV_DEV_WORKSPACE_MISMATCH and its output is not to be
 * trusted).  Every launch leaves the merge tickets at zero again; the status
 * word is sticky (kernels only set bits in it; pkv_decode_status reads and
 * clears it).  After a launch that reported PKV_DEV_WAIT_TIMEOUT, zero-fill the
 * workspace again before reuse.
 * One workspace must not be used by two launches that may run concurrently.
 */
/* dtype PKV_FP8_E4M3 (PKV_INT8) sizes the workspace of pkv_decode_attention_fp8
 * and pkv_decode_step_fp8 (_int8), whose default warp count differs. */
int pkv_decode_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t dtype, int32_t num_warps, size_t* bytes);

/*
 * pkv_decode_attention — single-token decode attention over a block-paged cache.
 *
 * For every sequence s < num_seqs and query head h < num_q_heads, with
 * G = num_q_heads / num_kv_heads, g = h / G and t = context_lens[s]:
 *   out[s, h, :] = sum_{p<t} w_p * V[slot(p), g, :] / sum_{p<t} w_p,
 *   w_p = exp(scale * q[s, h, :] . K[slot(p), g, :] - max_p(...)),
 * i.e. softmax(q K^T * scale) V over the sequence's t cached positions read
 * through its block table — the same attention a contiguous cache gives
 * ("PagedAttention — how vLLM stopped wasting 80% of your GPU memory", section
 * "The PagedAttention kernel: computing attention over scattered blocks").
 * t counts the token being decoded, whose K/V must already be in the cache
 * (write with pkv_kv_write first).  t == 0 yields a zero row.
 *
 * One kernel launch.  Work is split into equal runs of (sequence, KV head,
 * block) steps over all worker warps; a context cut by a run boundary is
 * finished as several partial softmax states, which the last warp to finish a
 * piece merges in fixed order with a log-sum-exp ("two-pass reduction ...
 * numerically stable merge", "PagedAttention: How vLLM Borrowed Virtual
 * Memory...", section "The Custom CUDA Kernel").  Results depend only on the
 * values, context lengths and num_warps — never on which physical blocks hold
 * the data — and are bit-identical between runs.  The launch uses programmatic
 * stream serialisation, so its prologue overlaps a pkv_kv_write queued just
 * before it on the same stream; every cache read still follows that write.
 *
 * q             device [num_seqs, num_q_heads, head_dim], contiguous.
 * k_cache, v_cache  device caches [num_blocks, num_kv_heads, block_size, head_dim].
 * block_tables  device int32 [num_seqs, max_blocks_per_seq]; entries past
 *               ceil(t / block_size) are never read.
 * context_lens  device int32 [num_seqs].
 * scale         softmax scale (typically 1/sqrt(head_dim)).
 * out           device [num_seqs, num_q_heads, head_dim], written in full.
 * workspace     device, >= pkv_decode_workspace_size(...) bytes, 256-byte aligned,
 *               zero-filled before first use.
 * num_warps     worker warps (0 = device default); pass the same value given to
 *               pkv_decode_workspace_size.
 * Supported: block_size 8, 16 or 32 (the kernels work in 16-token steps: half a
 * 32-token block, or two 8-token blocks; results do not depend on the block
 * size); dtype F16/BF16 with head_dim 64, 128 or 256, or F32 with head_dim 32,
 * 64 or 128; G in {1, 2, 4, 8}; num_seqs <= 2048;
 * num_blocks*num_kv_heads*block_size*4 < 2^31; num_seqs*max_blocks_per_seq*num_kv_heads < 2^31.
 * Invalid device data (a context length outside [0, max_blocks_per_seq *
 * block_size], a block id outside [0, num_blocks)) never faults: it is clamped or read as zeros
 * and recorded in the workspace status word (see pkv_decode_status).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_DTYPE, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
int pkv_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, float scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream);

/*
 * pkv_decode_step — one decode step: the cache write of each sequence's new token,
 * then pkv_decode_attention, from one call.
 *
 * Same arguments as pkv_decode_attention plus k_new, v_new (device [num_seqs,
 * num_kv_heads, head_dim], contiguous, 16-byte aligned).  For every sequence s with
 * t = context_lens[s] > 0 the new token is position t - 1 ("each decode step ->
 * write the new token's K,V into the last block", "PagedAttention and vLLM: Virtual
 * Memory for the KV Cache", section "L2 — Mechanism"): its K and V rows are written
 * to slot(t - 1) of the caches, the slot read from block_tables, exactly as
 * pkv_kv_write with that slot would; the attention of the step covers the new
 * token.  Two launches chained with programmatic dependent launch: the write, then
 * the attention, whose prologue (schedule, table prefetch) overlaps the write.
 * Output and caches are bit-identical to pkv_kv_write followed by
 * pkv_decode_attention with the same num_warps.  Sequences with t <= 0 or
 * t > max_blocks_per_seq * block_size, and slots outside the pool, write nothing.
 * Arguments are validated before anything is written; k_new and v_new must be
 * non-NULL and 16-byte aligned.
 * Errors: as pkv_decode_attention.
 */
int pkv_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int32_t num_blocks, float scale, void* out, void* workspace,
                    size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream);

/*
 * pkv_decode_status — read and clear the device status word of a workspace.
 * Synchronises `stream`, copies the word to *status (PKV_DEV_* bits, 0 = clean)
 * and zeroes it on the device.
 */
int pkv_decode_status(void* workspace, int32_t* status, void* stream);

/* Number of worker warps the default launch uses on the current device. */
/* (dtype PKV_FP8_E4M3 or PKV_INT8: the default of attention over that cache.) */
int pkv_decode_default_warps(int32_t head_dim, int32_t dtype, int32_t* num_warps);

/*
 * pkv_decode_attention_static_scratch — pkv_decode_attention for callers that
 * cannot allocate device memory.  (The pages have no counterpart: this is a
 * deployment variant of the same computation.)
 *
 * Some callers cannot hand the library a workspace: serving engines that give
 * every byte of HBM to the KV block pool at start-up and forbid allocations
 * afterwards, plugins running inside a host framework that owns all device
 * memory, and latency-critical decode loops where cudaMalloc's implicit device
 * synchronisation is not acceptable.  This entry point takes the same arguments
 * as pkv_decode_attention minus the workspace, and keeps the split-context
 * partial states in a fixed scratch array of PKV_STATIC_SCRATCH_BYTES that is
 * part of the library's device image: every GPU that loads the library holds
 * that memory until the process exits.  The call itself allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library routine).
 *
 * The first call on a device resolves the array's device address for that
 * device (cudaGetSymbolAddress) and sets the kernels' shared-memory limit; make
 * that first call before any stream capture.  The scratch status word is
 * cleared at the start of each call; device-side status bits are not reported
 * by this entry point (use pkv_decode_attention with a workspace and
 * pkv_decode_status to read them).
 *
 * All calls on a device share the one array, which keeps the last call's
 * contents.  Calls that may overlap on the GPU (on different streams, or from
 * different host threads without ordering) race on it and give wrong results:
 * order them on one stream.  A request whose partial states need more than
 * PKV_STATIC_SCRATCH_BYTES (pkv_decode_workspace_size with the same head shape,
 * dtype and num_warps) is rejected with PKV_ERR_UNSUPPORTED; a smaller num_warps
 * needs less scratch.  Every argument is checked before any work is enqueued, so
 * a refused call (oversized, or anything pkv_decode_attention would refuse) writes
 * nothing, the shared array included.  If the array's address cannot be resolved
 * the call fails with PKV_ERR_CUDA and the next call tries again.
 */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)
int pkv_decode_attention_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                        float scale, void* out, int32_t num_warps, int32_t dtype,
                                        void* stream);

/* ------------------------------------------------------------------------- */
/* Paged prefill attention                                                    */
/* ------------------------------------------------------------------------- */

/*
 * pkv_prefill_attention — causal attention of a chunk of new prompt tokens per
 * sequence over the paged cache (prefill, or chunked prefill: "PagedAttention: How
 * vLLM Borrowed Virtual Memory...", section "Walking Through the Lifecycle",
 * Prefill, and section "RadixAttention ..." on chunked prefill).
 *
 * Sequence s has t = context_lens[s] tokens in the cache — its chunk included,
 * written before this call (pkv_kv_write) — and c = query_start[s+1] -
 * query_start[s] queries, the last c positions: query row query_start[s] + i is
 * at position p = t - c + i and, for query head h of KV group g = h / G, attends
 * to every position j <= p:
 *   out[row, h] = softmax_j(scale * q[row, h] . K[slot(j), g]) . V[slot(j), g].
 * A whole-prompt prefill is c = t.
 *
 * q, out        device [num_tokens, num_q_heads, head_dim], f16 or bf16,
 *               contiguous; num_tokens >= query_start[num_seqs] (a chunk reaching
 *               past num_tokens is clamped and reported); only rows of the chunks
 *               are written.
 * block_tables, context_lens, caches: as pkv_decode_attention.
 * query_start   device int32 [num_seqs + 1], non-decreasing, query_start[0] = 0.
 * status        device int32 word or NULL: PKV_DEV_* bits are ORed into it
 *               (lengths out of range are clamped, bad block ids read as zeros,
 *               a wait that timed out abandons the launch).
 * Supported: block_size 8, 16 or 32 (a 128-key tile is read as 16, 8 or 4
 * blocks), head_dim 64 or 128, G in {1, 2, 4, 8}, num_seqs <= 2048,
 * max_blocks_per_seq * block_size < 2^31.  Computed on the 5th-generation tensor cores (tcgen05 MMAs
 * with tensor-memory accumulators; bf16/f16 inputs, probabilities rounded to the
 * input type for P.V, fp32 accumulation and softmax); results depend only on the
 * values and lengths.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_DTYPE, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
int pkv_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, const int32_t* query_start,
                          int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, float scale, void* out, int32_t* status,
                          int32_t dtype, void* stream);

/* ------------------------------------------------------------------------- */
/* fp8 KV cache                                                               */
/* ------------------------------------------------------------------------- */

/*
 * A quantised KV cache stores K and V in 8 bits instead of 16, halving the bytes
 * per cached token; the pages call it orthogonal to paging and composable with
 * it ("PagedAttention — how vLLM stopped wasting 80% of your GPU memory", FAQ
 * "How does this relate to quantization?").  They fix no format; this library
 * uses:
 *   - elements: fp8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 *     subnormals, no infinity, largest finite 448, S.1111.111 is NaN);
 *   - scales: one fp32 scale per KV head for K (k_scale[num_kv_heads]) and one
 *     for V (v_scale[...]), both device arrays; an element reads back as
 *     code * scale;
 *   - quantisation on write: code = E4M3(x / scale), x widened to fp32, the
 *     quotient a correctly rounded fp32 division, then rounded to the nearest
 *     E4M3 value with ties to an even code and saturated to +-448 (NaN stays NaN);
 *   - layouts (block_size 16):
 *       k_cache [num_blocks, num_kv_heads, 16, head_dim] uint8 (as above);
 *       v_cache [num_blocks, num_kv_heads, head_dim, 16] uint8: each (block, KV
 *       head) tile transposed, and within each 16-byte head_dim row token t of
 *       the block at byte V_POS[t], the byte order being the tokens
 *       0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15 (byte j holds the j-th of these).
 *   pkv_copy_blocks copies fp8 blocks with dtype PKV_FP8_E4M3 and
 *   block_elems = num_kv_heads * 16 * head_dim.  pkv_swap_out_blocks and
 *   pkv_swap_in_blocks move 8-bit blocks like any others (block_bytes =
 *   num_kv_heads * 16 * head_dim).
 */

/*
 * pkv_kv_write_fp8 — quantise new tokens' K and V and scatter them into the fp8
 * caches: for i < num_tokens, h < num_kv_heads with s = slot_mapping[i] >= 0,
 *   k_cache[s / 16, h, s % 16, :]          = E4M3(k[i, h, :] / k_scale[h])
 *   v_cache[s / 16, h, :, V_POS[s % 16]]   = E4M3(v[i, h, :] / v_scale[h])
 * k, v          device [num_tokens, num_kv_heads, head_dim] in `dtype`
 *               (PKV_F32, PKV_F16 or PKV_BF16), contiguous, 16-byte aligned.
 * slot_mapping, num_blocks, block_size (must be 16): as pkv_kv_write.
 * k_scale, v_scale  device float [num_kv_heads], positive and finite.
 * Requirements: head_dim a multiple of 16; caches 16-byte aligned.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_DTYPE, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
int pkv_kv_write_fp8(const void* k, const void* v, const int32_t* slot_mapping,
                     int32_t num_tokens, void* k_cache, void* v_cache, const float* k_scale,
                     const float* v_scale, int32_t num_blocks, int32_t num_kv_heads,
                     int32_t block_size, int32_t head_dim, int32_t dtype, void* stream);

/*
 * pkv_decode_attention_fp8 — pkv_decode_attention over fp8 caches: the same
 * attention with K[slot, g, :] = code * k_scale[g] and V likewise, computed as
 *   scores = (scale * k_scale[g]) * q . code_k,  out = v_scale[g] * softmax . code_v.
 * q and out are `dtype` (PKV_F16 or PKV_BF16); the cache codes are widened
 * exactly to f16 for the tensor-core contractions, q is converted to f16 (exact
 * for values of magnitude in [2^-14, 65504]; |q| must stay below 65504), and
 * scores, softmax and accumulation are fp32.  The workspace, num_warps,
 * determinism, status reporting and the programmatic-launch chaining are those
 * of pkv_decode_attention; size the workspace with pkv_decode_workspace_size
 * for dtype PKV_FP8_E4M3 and the same head shape and num_warps (by default one
 * CTA per SM of 16 worker warps at head_dim 128 and 8 at head_dim 256: the 4 KB
 * 8-bit stages leave room for more warps than the 16-bit caches' 8 KB ones).
 * Supported: block_size 16, head_dim 128 or 256, G in {1, 2, 4, 8}.
 * Errors: as pkv_decode_attention.
 */
int pkv_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks, float scale, void* out, void* workspace,
                             size_t workspace_bytes, int32_t num_warps, int32_t dtype,
                             void* stream);

/*
 * pkv_decode_step_fp8 — one decode step over fp8 caches: each sequence's new
 * token (k_new, v_new [num_seqs, num_kv_heads, head_dim] in `dtype`, position
 * t - 1 for t = context_lens[s] > 0, slot from its block table) is quantised
 * into the caches exactly as pkv_kv_write_fp8 would, then
 * pkv_decode_attention_fp8 runs; the two launches are chained with programmatic
 * dependent launch.  Output and caches are bit-identical to pkv_kv_write_fp8
 * followed by pkv_decode_attention_fp8.
 * Errors: as pkv_decode_attention_fp8.
 */
int pkv_decode_step_fp8(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const float* k_scale, const float* v_scale,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t num_blocks, float scale, void* out, void* workspace,
                        size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream);

/* ------------------------------------------------------------------------- */
/* int8 KV cache                                                              */
/* ------------------------------------------------------------------------- */

/*
 * The pages name int8 beside fp8 as the narrower element of a quantised KV cache
 * ("PagedAttention — how vLLM stopped wasting 80% of your GPU memory", FAQ "How
 * does this relate to quantization?") and fix no format; this library uses
 * symmetric codes:
 *   - elements: int8 codes c in [-127, 127] (-128 is never written); an element
 *     reads back as c * scale;
 *   - scales: one fp32 scale per KV head for K and one for V (device arrays
 *     k_scale[num_kv_heads], v_scale[...]), as for the fp8 cache;
 *   - quantisation on write: c = clamp(round(x / scale), -127, 127), x widened
 *     to fp32, the quotient a correctly rounded fp32 division rounded to the
 *     nearest integer with ties to even; +-infinity saturates, NaN gives 0;
 *   - layouts: those of the fp8 cache (block_size 16, K [num_blocks,
 *     num_kv_heads, 16, head_dim], V tiles transposed with the same byte order).
 *   pkv_copy_blocks copies int8 blocks with dtype PKV_INT8.
 * The three entry points take the arguments of their fp8 counterparts, with the
 * same requirements, errors and guarantees; only the element format differs.
 */

/* pkv_kv_write_int8 — pkv_kv_write_fp8 with int8 codes:
 *   k_cache[s / 16, h, s % 16, :]        = clamp(round(k[i, h, :] / k_scale[h]))
 *   v_cache[s / 16, h, :, V_POS[s % 16]] = clamp(round(v[i, h, :] / v_scale[h])) */
int pkv_kv_write_int8(const void* k, const void* v, const int32_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache, const float* k_scale,
                      const float* v_scale, int32_t num_blocks, int32_t num_kv_heads,
                      int32_t block_size, int32_t head_dim, int32_t dtype, void* stream);

/* pkv_decode_attention_int8 — decode attention over int8 caches:
 *   scores = (scale * k_scale[g]) * q . c_k,  out = v_scale[g] * softmax . c_v,
 * the codes widened exactly to f16 for the tensor-core contractions, q converted
 * to f16, fp32 scores, softmax and accumulation.  Workspace sized for dtype
 * PKV_INT8.  Supported: block_size 16, head_dim 128 or 256, G in {1, 2, 4, 8}. */
int pkv_decode_attention_int8(const void* q, const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks, float scale, void* out, void* workspace,
                              size_t workspace_bytes, int32_t num_warps, int32_t dtype,
                              void* stream);

/* pkv_decode_step_int8 — the new tokens quantised into the int8 caches as
 * pkv_kv_write_int8 would, then pkv_decode_attention_int8, chained with
 * programmatic dependent launch; bit-identical to the two calls in sequence. */
int pkv_decode_step_int8(const void* q, const void* k_new, const void* v_new, void* k_cache,
                         void* v_cache, const float* k_scale, const float* v_scale,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, float scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t num_warps, int32_t dtype, void* stream);

/* ------------------------------------------------------------------------- */
/* Copy-on-write block copy                                                   */
/* ------------------------------------------------------------------------- */

/*
 * pkv_copy_blocks — copy whole physical blocks, K and V, for copy-on-write.
 *
 * For each pair i < num_pairs: block src = pairs[2i] is copied onto block
 * dst = pairs[2i+1] in both caches (all KV heads and slots: block_elems =
 * num_kv_heads*block_size*head_dim elements each).  This is the data copy of
 * "allocates a new physical block, copies the content" ("PagedAttention: How
 * vLLM Borrowed Virtual Memory...", section "Copy-on-Write for Beam Search and
 * Parallel Sampling").  Pairs with an id outside [0, num_blocks) are skipped.
 * A dst that is also some pair's src, or two pairs with one dst: unspecified.
 * src_dst_pairs is device int32 [num_pairs, 2].  block_elems * element size
 * must be a multiple of 16 bytes and both caches 16-byte aligned.  dtype may
 * be PKV_FP8_E4M3 or PKV_INT8 for 8-bit caches (one byte per element).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_DTYPE, PKV_ERR_CUDA.
 */
int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst_pairs, int32_t num_pairs,
                    int32_t num_blocks, int64_t block_elems, int32_t dtype, void* stream);

/*
 * pkv_copy_blocks_layers — pkv_copy_blocks for the caches of num_layers layers
 * in one launch.  A physical block id names the same block in every layer's
 * tensors (section "Copy-on-Write for Beam Search and Parallel Sampling": the
 * copy is of the block's content, which spans all layers), so each pair is
 * copied in every layer.
 *
 * k_caches, v_caches  HOST arrays of num_layers device pointers, layer l's K and
 *               V cache; every layer's caches have the same shape and dtype
 *               (num_blocks blocks of block_elems elements), each 16-byte aligned.
 * The other arguments, the skipping of out-of-range pairs and the unspecified
 * cases are those of pkv_copy_blocks.  1 <= num_layers <= 128.  The arrays are
 * read before the call returns.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_DTYPE, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
int pkv_copy_blocks_layers(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                           const int32_t* src_dst_pairs, int32_t num_pairs, int32_t num_blocks,
                           int64_t block_elems, int32_t dtype, void* stream);

/* ------------------------------------------------------------------------- */
/* Swapping blocks to host memory                                             */
/* ------------------------------------------------------------------------- */

/*
 * pkv_swap_out_blocks — copy whole blocks, K and V, to host memory: host block i
 * (bytes [i*block_bytes, (i+1)*block_bytes) of host_k and of host_v) becomes a
 * copy of cache block block_ids[i], for i < num_ids.  pkv_swap_in_blocks — the
 * reverse: cache block block_ids[i] becomes host block i.  These are the data
 * copies of preemption by swapping (see pkv_seq_swap_out / pkv_seq_swap_in).
 * The kernel reads or writes the host buffers directly over the CPU-GPU link.
 * block_ids    device int32 [num_ids]; ids outside [0, num_blocks) are skipped.
 * block_bytes  bytes of one block of one cache (num_kv_heads * block_size *
 *              head_dim * element size), a multiple of 16.
 * host_k, host_v  page-locked (or managed) host memory of at least
 *              num_ids * block_bytes bytes each, 16-byte aligned; other host
 *              memory is refused with PKV_ERR_INVALID_ARG before any work is
 *              queued.  The caller keeps the buffers alive until the stream has
 *              passed the copy.
 * k_cache, v_cache  device caches, 16-byte aligned (any element type and layout:
 *              blocks are moved as bytes).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA.
 */
int pkv_swap_out_blocks(const void* k_cache, const void* v_cache, const int32_t* block_ids,
                        int32_t num_ids, int32_t num_blocks, int64_t block_bytes, void* host_k,
                        void* host_v, void* stream);
int pkv_swap_in_blocks(const void* host_k, const void* host_v, const int32_t* block_ids,
                       int32_t num_ids, int32_t num_blocks, int64_t block_bytes, void* k_cache,
                       void* v_cache, void* stream);

/*
 * pkv_swap_out_blocks_layers / pkv_swap_in_blocks_layers — the same copies for
 * the caches of num_layers layers in one launch (a block id names the same block
 * in every layer's tensors, so preempting a sequence moves its blocks in all of
 * them).  host_k and host_v hold the layers one after another: layer l's copy of
 * block_ids[i] is host block l * num_ids + i (bytes [(l * num_ids + i) *
 * block_bytes, ... + block_bytes)), so each buffer needs num_layers * num_ids *
 * block_bytes bytes.  k_caches, v_caches: HOST arrays of num_layers device
 * pointers, every layer's caches of one shape, each 16-byte aligned; read before
 * the call returns.  1 <= num_layers <= 128.  Everything else as
 * pkv_swap_out_blocks / pkv_swap_in_blocks.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 */
int pkv_swap_out_blocks_layers(const void* const* k_caches, const void* const* v_caches,
                               int32_t num_layers, const int32_t* block_ids, int32_t num_ids,
                               int32_t num_blocks, int64_t block_bytes, void* host_k,
                               void* host_v, void* stream);
int pkv_swap_in_blocks_layers(const void* host_k, const void* host_v, const int32_t* block_ids,
                              int32_t num_ids, int32_t num_blocks, int64_t block_bytes,
                              void* const* k_caches, void* const* v_caches, int32_t num_layers,
                              void* stream);

/* ------------------------------------------------------------------------- */
/* Host block manager                                                         */
/* ------------------------------------------------------------------------- */
/*
 * The block manager of "PagedAttention: How vLLM Borrowed Virtual Memory...",
 * sections "The OS-Inspired Insight" and "Walking Through the Lifecycle", and
 * "What is paged attention?", section "How it works":
 *   - a fixed pool of num_blocks blocks; allocation pops the free list, freeing
 *     pushes it, both O(1).  The free list is a stack whose first pops return
 *     pop_order[0], pop_order[1], ... (ascending ids when pop_order is NULL);
 *   - a refcount per block counts the table entries that point at it; a block
 *     returns to the free list when its count reaches 0;
 *   - fork copies a table and increments every block in it;
 *   - appending position p: if p % block_size == 0 a new block is pushed on the
 *     table (never a copy); otherwise, if the last block is shared (refcount > 1),
 *     the writer gets a fresh block, the (old, new) copy-on-write pair is
 *     reported, the old block is decremented and the new one replaces it;
 *     the slot is table[p / block_size] * block_size + p % block_size;
 *   - freeing a sequence decrements its table in reverse order.
 * Sequence ids are 0, 1, 2, ... in creation order and never reused.
 * Every failing call leaves the state unchanged, including one whose host memory
 * allocation fails (PKV_ERR_INVALID_ARG, "host memory exhausted": every call makes
 * its room before it changes anything).  A handle is not thread-safe.
 */
typedef struct pkv_allocator pkv_allocator_t;

int pkv_allocator_create(int32_t num_blocks, int32_t block_size, const int32_t* pop_order,
                         pkv_allocator_t** out);
int pkv_allocator_destroy(pkv_allocator_t* a);

int pkv_block_alloc(pkv_allocator_t* a, int32_t* block_id);   /* PKV_ERR_OUT_OF_BLOCKS if empty */
int pkv_block_incref(pkv_allocator_t* a, int32_t block_id);   /* block must be allocated */
int pkv_block_decref(pkv_allocator_t* a, int32_t block_id);   /* block must be allocated */
int pkv_block_refcount(pkv_allocator_t* a, int32_t block_id, int32_t* refcount);
int pkv_num_free_blocks(pkv_allocator_t* a, int32_t* num_free);

int pkv_seq_create(pkv_allocator_t* a, int32_t* seq);
int pkv_seq_fork(pkv_allocator_t* a, int32_t parent, int32_t* child);
int pkv_seq_free(pkv_allocator_t* a, int32_t seq);

/*
 * Preemption by swapping ("PagedAttention — how vLLM stopped wasting 80% of
 * your GPU memory", section "Preemption: what happens when memory runs out
 * anyway": copy the preempted sequence's blocks out to CPU RAM, and back into
 * freshly allocated GPU blocks when it resumes; all or nothing per sequence).
 *
 * pkv_seq_swap_out — writes the sequence's table (physical ids in logical order,
 * *n of them; ids_out must hold them all) and gives every block back in reverse
 * table order, as pkv_seq_free does; the sequence keeps its length and is
 * swapped out: append, fork, blocks_needed, export and swap_out refuse it until
 * pkv_seq_swap_in.  Copy the blocks' contents to host memory with
 * pkv_swap_out_blocks before any of the returned ids is reused.
 * pkv_seq_swap_in — gives a swapped-out sequence ceil(length / block_size)
 * freshly allocated blocks, written to ids_out in logical order (PKV_ERR_OUT_OF_BLOCKS
 * with the state unchanged if the pool cannot supply them all); restore their
 * contents with pkv_swap_in_blocks.
 */
int pkv_seq_swap_out(pkv_allocator_t* a, int32_t seq, int32_t* ids_out, int32_t capacity,
                     int32_t* n);
int pkv_seq_swap_in(pkv_allocator_t* a, int32_t seq, int32_t* ids_out, int32_t capacity,
                    int32_t* n);

/* Blocks an append of n_tokens would take from the free list (CoW copy included). */
int pkv_seq_blocks_needed(pkv_allocator_t* a, int32_t seq, int32_t n_tokens, int32_t* needed);

/*
 * Append n_tokens positions to seq, all or nothing.  slots_out (host int32
 * [n_tokens], may be NULL when n_tokens == 0) receives each position's slot.
 * cow_pair_out (host int32 [2]) receives the copy-on-write (src, dst) pair and
 * *n_cow is set to 0 or 1 (only the first appended position can need a copy).
 * PKV_ERR_OUT_OF_BLOCKS if the pool cannot serve every block the append needs.
 */
int pkv_seq_append(pkv_allocator_t* a, int32_t seq, int32_t n_tokens, int32_t* slots_out,
                   int32_t* cow_pair_out, int32_t* n_cow);

/*
 * pkv_seq_append_one_each — one decode step's bookkeeping in one call: appends one
 * position to each of the k distinct sequences seqs[0..k-1], in that order, with the
 * result pkv_seq_append(a, seqs[i], 1, ...) would give called for each in turn
 * ("PagedAttention: How vLLM Borrowed Virtual Memory...", section "Walking Through
 * the Lifecycle", Decode: each sequence's new token goes into its last block, a new
 * block when the last one is full; section "Copy-on-Write for Beam Search and
 * Parallel Sampling": a write into a shared block moves the writer onto a copy, and
 * a later writer that finds itself the last holder writes in place).
 * seqs          host int32 [k], resident sequence ids, no id twice.
 * slots_out     host int32 [k]: the slot of each new position.
 * cow_pairs_out host int32 [2 k]: the (src, dst) pairs of the copies needed, in
 *               list order, *n_cow of them.
 * All or nothing: PKV_ERR_OUT_OF_BLOCKS (state unchanged) if the pool cannot serve
 * every block the k appends take; PKV_ERR_INVALID_ARG for a bad, swapped-out or
 * repeated id.  k = 0 is a no-op.
 */
int pkv_seq_append_one_each(pkv_allocator_t* a, const int32_t* seqs, int32_t k,
                            int32_t* slots_out, int32_t* cow_pairs_out, int32_t* n_cow);

int pkv_seq_len(pkv_allocator_t* a, int32_t seq, int32_t* len);
/* Copies up to `capacity` ids of seq's table to ids_out; *n = table length. */
int pkv_seq_table(pkv_allocator_t* a, int32_t seq, int32_t* ids_out, int32_t capacity, int32_t* n);

/*
 * Export the tables of `num` sequences as a row-major host int32
 * [num, max_blocks] array (entries past a table's end are 0) and their lengths
 * into ctx_out [num].  PKV_ERR_INVALID_ARG if a table is longer than max_blocks.
 */
int pkv_export_tables(pkv_allocator_t* a, const int32_t* seqs, int32_t num, int32_t max_blocks,
                      int32_t* tables_out, int32_t* ctx_out);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
