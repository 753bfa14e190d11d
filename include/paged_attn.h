/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) paged-KV GQA/MQA attention
 * library (libpaged_attn.so).
 *
 * What is computed.  Attention of query heads over a paged KV cache, for
 * grouped-query (G = num_heads / num_kv_heads query heads share one KV head)
 * and multi-query (one KV head) models:
 *
 *   out[t, h, :] = sum_j softmax_j(scale * q[t, h, :] . K[j, h / G, :]) V[j, h / G, :]
 *
 * over the keys j that query token t may see.  This is exactly multi-head
 * attention after each KV head is expanded to its G query heads, as in vLLM
 * issue #1880 "[Performance] Use optimized kernels for MQA/GQA" (item 1); the
 * kernels reach it without expanding, reading each KV head's cache blocks
 * once for all G query heads and doing the grouped dot products on tensor
 * cores (same issue, opening paragraph and item 2).  The mixed batch of
 * chunked prefill and decode follows vLLM PR #14431 "[Kernel][V1] Further
 * optimizations to ROCm (Triton) Backend to better handle GQA" (opening post,
 * review thread on chunked_prefill_paged_decode).
 *
 * Data layout (all row-major, contiguous, element type fp16 or bf16):
 *   q           [T, Hq, D]          (decode: T = num_seqs, one token each)
 *   k_cache     [NB, Hkv, bs, D]    physical block, KV head, slot, dim
 *   v_cache     [NB, Hkv, bs, D]
 *   block_tables[B, max_blocks_per_seq] int32 physical block ids; entries
 *               past a sequence's last block are not read (pad with -1)
 *   context_lens[B] int32: tokens of each sequence in the cache, INCLUDING
 *               this step's query tokens (written by reshape_and_cache first)
 *   cu_query_lens[B + 1] int32: prefix sums of the query-token counts
 *   out         [T, Hq, D], same element type as q
 * Causal alignment: query token i of a sequence with qlen query tokens and
 * ctx context tokens sits at position ctx - qlen + i and sees keys 0 .. that
 * position.  A sequence with ctx = 0 gets a zero output row.
 *
 * Ownership and execution.  Every pointer argument is device memory owned
 * by the caller (except where a function says "host").  Calls only enqueue
 * work on `stream`; they never synchronise, never allocate device memory and
 * never create streams.  Scratch space comes from the caller's `workspace`
 * (size from the matching *_workspace_bytes function, 256-byte aligned).
 * Two calls that share a workspace must not run concurrently.
 * Stream capture: every kernel reads lengths, tables and offsets from device
 * memory when it runs, so a step captured in a CUDA graph replays correctly
 * for any batch of the captured shapes (the scalar arguments are baked into
 * the graph).  Make the first call on a device outside any capture.
 *
 * Errors.  Arguments are validated on the host first; a negative pa_status
 * is returned and nothing is enqueued.  A failed launch returns
 * PA_ERR_CUDA.  Data errors found on the device (a block id or a slot out of
 * range, a pipeline wait that timed out) skip the faulty access and set bits
 * in a status word inside the workspace, read with pa_read_device_status().
 * The library never aborts, exits or traps.
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_NULL = -1,       /* a required pointer is NULL */
    PA_ERR_SHAPE = -2,      /* inconsistent or out-of-range sizes */
    PA_ERR_DTYPE = -3,      /* element type is neither PA_F16 nor PA_BF16 */
    PA_ERR_HEADDIM = -4,    /* head_dim not 64 or 128 */
    PA_ERR_BLOCKSIZE = -5,  /* block_size not a multiple of 16 in [16, 256] */
    PA_ERR_WORKSPACE = -6,  /* workspace NULL, too small or misaligned */
    PA_ERR_CUDA = -7,       /* a CUDA runtime call or launch failed */
    PA_ERR_ALIGN = -8,      /* a tensor pointer is not 16-byte aligned */
    PA_ERR_DEVICE = -9      /* the current device is not sm_100-family */
} pa_status;

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

/* Bits of the device status word (pa_read_device_status). */
#define PA_DEV_BAD_BLOCK_ID 0x1u  /* a block-table entry outside [0, NB) */
#define PA_DEV_BAD_SLOT 0x2u      /* a slot_mapping entry outside [-1, NB*bs) */
#define PA_DEV_WAIT_TIMEOUT 0x4u  /* a pipeline wait ran out of time */
#define PA_DEV_BAD_LENGTHS 0x8u   /* a sequence with ctx < 0, ctx > mbs * bs
                                     or qlen > ctx: skipped.  A query range
                                     outside [0, total_query_tokens) or with
                                     qlen < 0 (cu_query_lens not
                                     non-decreasing within the token count):
                                     the whole call does no work, since the
                                     other ranges may overlap */

/* Human-readable name of a pa_status value (static string). */
PA_API const char* pa_status_string(int status);

/*
 * reshape_and_cache -- write this step's new K/V rows into the paged cache.
 *
 *   k_cache[s / bs, h, s % bs, :] = k[t, h, :]   (same for v)
 *   for every token t with s = slot_mapping[t] >= 0; slot -1 skips a token.
 *
 * Source: the cache-write step that precedes paged attention in the
 * attention layer of the pages' serving system (vLLM issue #1880, item 2:
 * the decode kernel reads K/V from the paged cache); layout as above.
 *   k, v          [num_tokens, num_kv_heads, head_dim]
 *   slot_mapping  [num_tokens] int64
 * Every other byte of the caches is left unchanged.  Two tokens mapped to
 * the same slot is invalid input (which one lands is unspecified).  A slot
 * outside [-1, num_blocks * block_size) is skipped and flags
 * PA_DEV_BAD_SLOT in `status_word` (a device int32, may be NULL).
 */
PA_API int reshape_and_cache(const void* k, const void* v, void* k_cache,
                      void* v_cache, const int64_t* slot_mapping,
                      int num_tokens, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, int dtype,
                      uint32_t* status_word, pa_stream_t stream);

/*
 * Workspace size in bytes for paged_attn_decode with these sizes.
 * num_splits: 0 = automatic (equal shares of the batch's key tiles up to
 * 2048 sequences, else splits of 256 tokens, at most 64 per sequence),
 * else the fixed number of KV splits per sequence (1..64).
 */
PA_API size_t paged_attn_workspace_bytes(int num_seqs, int num_heads,
                                  int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int block_size,
                                  int num_splits);

/*
 * paged_attn_decode -- one query token per sequence.
 *
 *   q [num_seqs, num_heads, head_dim]; out [num_seqs, num_heads, head_dim]
 *
 * num_splits = 0 (up to 2048 sequences): the batch's 16-key tiles, over
 * all (sequence, KV head) units, are shared out in equal contiguous ranges
 * over the warp groups of a persistent grid; a unit cut between groups
 * gives one partial output and log-sum-exp per piece, merged by a
 * log-sum-exp combine kernel.  Larger batches take 256-token splits, at
 * most 64.
 * num_splits = S > 0: split s of a sequence with nb blocks covers blocks
 * [s * c, (s + 1) * c), c = ceil(nb / S), and a combine kernel merges the
 * splits.  Sequences with no keys get zero output rows.  scale (> 0)
 * multiplies q . k before the softmax (base e).
 */
PA_API int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, float scale, int num_seqs,
                      int num_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, int dtype,
                      int num_splits, void* out, void* workspace,
                      size_t workspace_bytes, pa_stream_t stream);

/* Workspace size in bytes for paged_attn_chunked_prefill. */
PA_API size_t paged_attn_chunked_prefill_workspace_bytes(
    int num_seqs, int total_query_tokens, int num_heads, int num_kv_heads,
    int head_dim, int max_blocks_per_seq, int block_size, int num_splits);

/*
 * paged_attn_chunked_prefill -- a batch mixing query chunks (qlen > 1,
 * causal within the chunk, after a cached prefix) with decode rows
 * (qlen = 1), in the cu_query_lens layout.
 *
 *   q [total_query_tokens, num_heads, head_dim]; out same shape.
 *   total_query_tokens = cu_query_lens[num_seqs] and max_query_len are the
 *   host-known bounds the launch is sized by (no device sync); rows of
 *   sequences with qlen = 1 follow the decode path (with KV splits as in
 *   paged_attn_decode), the rest the prefill path.
 *
 *   Scheduling, all on `stream` and on the device (no host sync): a
 *   work-list kernel sorts the rows into the two paths and, from their key
 *   counts, sizes the decode path's share of the SMs; the prefill kernel
 *   and the decode kernel then run side by side, the decode kernel taking
 *   that share at once and each SM the prefill kernel frees later.  The
 *   call's kernels finish, and its outputs are written, before work queued
 *   after it on `stream` starts.
 */
PA_API int paged_attn_chunked_prefill(const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               int max_blocks_per_seq,
                               const int32_t* cu_query_lens,
                               const int32_t* context_lens,
                               int total_query_tokens, int max_query_len,
                               float scale, int num_seqs, int num_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, int dtype, int num_splits,
                               void* out, void* workspace,
                               size_t workspace_bytes, pa_stream_t stream);

/*
 * paged_attn_cross_attention -- attention of decoder query rows over a
 * static, already written encoder K/V cache (vLLM PR #7448, "[Core]
 * More-efficient cross-attention parallel QKV computation", opening post:
 * Q comes from the decoder, K and V from the encoder output, and during
 * decode the encoder sequence is static, so no new K/V are written).
 *
 * Same arguments, layouts, ownership and errors as
 * paged_attn_chunked_prefill, with two differences: context_lens[b] is the
 * number of encoder tokens of sequence b in the cache, and there is no
 * causal mask -- every query row of sequence b attends to all
 * context_lens[b] keys, whatever its position among the sequence's rows, so
 * a sequence may carry more query rows than keys.  Sequences with one query
 * row take the decode path (with KV splits), the others the tensor-core
 * path; a sequence without encoder tokens gives zero rows.  The workspace
 * size is paged_attn_chunked_prefill_workspace_bytes.
 */
PA_API int paged_attn_cross_attention(const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* cu_query_lens,
                               const int32_t* context_lens, int total_query_tokens,
                               int max_query_len, float scale, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, int dtype,
                               int num_splits, void* out, void* workspace,
                               size_t workspace_bytes, pa_stream_t stream);

/* Workspace size in bytes for gqa_varlen_prefill. */
PA_API size_t gqa_varlen_prefill_workspace_bytes(int num_seqs, int total_query_tokens,
                                                 int num_heads, int num_kv_heads,
                                                 int head_dim);

/*
 * gqa_varlen_prefill -- prompt attention over the new tokens' own keys and
 * values, before any cache write, without expanding K/V per query head
 * (vLLM issue #1880, "[Performance] Use optimized kernels for MQA/GQA",
 * item 1: the prefill path broadcasts K/V [T, Hkv, D] to [T, Hq, D] and
 * runs a multi-head kernel; here each KV head's rows are read once for its
 * G query heads).
 *
 *   q [total_query_tokens, num_heads, head_dim]; k, v
 *   [total_key_tokens, num_kv_heads, head_dim], contiguous (device).
 *   Sequence b owns query rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key
 *   rows [cu_seqlens_k[b], cu_seqlens_k[b+1]) (int32, device, num_seqs + 1
 *   entries, starting at 0); its key count must be at least its query count.
 *   Causal, bottom-right: with klen keys and qlen rows, row t sees keys
 *   0 .. klen - qlen + t; cu_seqlens_q == cu_seqlens_k is plain causal
 *   self-attention over each prompt.  max_seqlen_q bounds the chunk length.
 *   out has q's shape.  Errors as for the paged entry points; a sequence
 *   with fewer keys than query rows is skipped and flagged
 *   PA_DEV_BAD_LENGTHS in the workspace status word.
 */
PA_API int gqa_varlen_prefill(const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                              int total_query_tokens, int total_key_tokens,
                              int max_seqlen_q, float scale, int num_seqs, int num_heads,
                              int num_kv_heads, int head_dim, int dtype, void* out,
                              void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Read (and clear, if `clear` != 0) the device status word kept in a
 * workspace after the work queued on `stream` so far has finished.  This
 * call synchronises `stream`.  *flags receives PA_DEV_* bits (host pointer).
 */
PA_API int pa_read_device_status(const void* workspace, int clear, uint32_t* flags,
                          pa_stream_t stream);

/*
 * paged_attn_decode_noalloc -- paged_attn_decode without a caller workspace.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot obtain device scratch memory at all (a runtime whose allocator
 * has already reserved nearly all of HBM for its KV-cache pool and forbids
 * further allocations, a plugin host that passes kernels only their input
 * and output tensors, a C program with no device-memory manager).  It runs
 * the same kernels as paged_attn_decode, with the workspace taken from a
 * 32 MiB array that the library holds in device memory on every GPU that
 * loads it, until the process exits.  Arguments and results are those of
 * paged_attn_decode; q, caches, tables and out are still the caller's.
 *
 * Limits and rules:
 *  - a problem whose paged_attn_workspace_bytes() exceeds 32 MiB returns
 *    PA_ERR_WORKSPACE (pass a smaller num_splits, or split the batch);
 *  - every call made outside a stream capture looks up the array's device
 *    address (cudaGetSymbolAddress) with the current device, so a context
 *    that was reset and created again is followed; a call inside a capture
 *    reuses the address of the device's latest uncaptured call, so make the
 *    first call on each device before any stream capture (a first call
 *    inside a capture returns PA_ERR_CUDA);
 *  - all calls share the one array and each call's work-list kernel
 *    rewrites what the next kernels read, so nothing needs clearing, but
 *    calls that overlap on the GPU (other streams, other host threads) race
 *    on it and must be serialised by the caller;
 *  - device status bits of these calls land in the shared array and are not
 *    readable through pa_read_device_status.
 * It never calls cudaMalloc, cudaFree or any allocating routine.
 */
PA_API int paged_attn_decode_noalloc(const void* q, const void* k_cache,
                                     const void* v_cache,
                                     const int32_t* block_tables,
                                     int max_blocks_per_seq,
                                     const int32_t* context_lens, float scale,
                                     int num_seqs, int num_heads,
                                     int num_kv_heads, int head_dim,
                                     int block_size, int num_blocks, int dtype,
                                     int num_splits, void* out,
                                     pa_stream_t stream);

/*
 * Measurement hook.  The next attention call made on this thread records
 * `start_event` on its stream just before its first attention kernel
 * (prefill or decode) and `stop_event` just after its last one, so the
 * work-list build and the split combine fall outside the interval.  The
 * events are cudaEvent_t values passed as void*; the hook is consumed by
 * that one call.  Passing NULLs clears it.
 */
PA_API void pa_profile_next_call(void* start_event, void* stop_event);

/*
 * Caps the number of CTAs (one per SM) of the persistent attention kernels
 * of the next attention call made on this host thread (decode, chunked
 * prefill, cross-attention or varlen prefill), so that two calls on two
 * streams can run side by side on disjoint SMs; max_ctas <= 0 clears it.
 * The cap is consumed by that call; a mixed call splits its capped SMs
 * between its two paths as above.  The pages define no such call: it
 * exists to compare one mixed-batch call with a prefill call and a
 * concurrent decode call, the two-kernel arrangement of vLLM PR #14431's
 * op (review thread on chunked_prefill_paged_decode.py).
 */
PA_API void pa_limit_next_call_ctas(int max_ctas);

/*
 * Limit, in nanoseconds, of each pipeline wait of the decode kernels (of
 * paged_attn_decode and of the decode rows of the chunked and
 * cross-attention calls) enqueued after this call, process-wide; 0 restores
 * the default of 2 s.  A wait that runs out sets PA_DEV_WAIT_TIMEOUT in the
 * call's status word; the kernel then stops issuing work, waits (with the
 * fixed 2 s limit) for the copies it still has in flight, and returns, so
 * the device stays usable and the next call runs normally; the outputs of
 * the call that timed out are undefined.  The pages define no such call: it
 * exists so the timeout path can be exercised (a limit of a few
 * nanoseconds makes waits give up before the first copies land).
 */
PA_API void pa_set_pipeline_wait_limit(uint64_t limit_ns);

/* Library version and the number of kernels the last call enqueued. */
PA_API int pa_version(void);
PA_API int pa_last_launch_count(void);

/*
 * The CUDA runtime error (a cudaError_t value) behind the most recent
 * PA_ERR_CUDA that a launch, function-attribute or stream call on the
 * calling thread produced, and its text; 0 and "no error" until one has
 * occurred.  Kept per host thread; a later successful call does not clear
 * it.  The pages define no such call: it only explains PA_ERR_CUDA.
 */
PA_API int pa_last_cuda_error(void);
PA_API const char* pa_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H */
