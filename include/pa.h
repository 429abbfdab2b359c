/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-attention library.
 *
 * The library computes attention for decode and chunked-prefill queries over a KV cache stored
 * in fixed-size physical blocks reached through a per-sequence block table, with grouped-query
 * heads and prefix blocks that may be aliased across sequences:
 *   - "Local_LLM_03_vLLM_Architecture", paged-KV slide: fixed-size blocks (16 tokens by
 *     default), a per-sequence block table from logical positions to physical blocks, and an
 *     attention kernel that gathers K/V from the scattered blocks; block-size slide: the block
 *     size is a knob; KV-sizing slide: GQA-8; chunked-prefill slide: prefills cut into chunks
 *     and interleaved with decodes.
 *   - "vLLM: LLM Inference That Doesn't Waste Your GPU", sections "KV cache, in one picture"
 *     (every processed token's K/V is stored once and reused), "Continuous batching" (prefill and
 *     decode mixed in one step) and "PagedAttention: virtual memory for KV".
 *   - "Scaling inference with vLLM": requests with the same start share physical pages.
 *
 * Conventions (the pages fix none of them):
 *   - Every pointer in a pa_tensor is a DEVICE pointer of the current CUDA device.  The library
 *     owns no buffer and allocates no device memory; the caller owns everything, including
 *     the attention workspace.
 *   - Strides are in elements.  The innermost dimension must be contiguous (stride 1).
 *   - fp16 is IEEE binary16; bf16 is bfloat16 (the upper half of an IEEE binary32).  A call
 *     works in one 16-bit type: k, v, q, out and the pools all fp16 or all bf16 (FP8 pools take
 *     fp16 tokens, q and out).  Accumulation is fp32; outputs are rounded to nearest-even.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream), like a
 *     kernel launch.  Nothing synchronises except pa_get_device_error.
 *   - Host-checkable errors are returned synchronously and nothing is launched.  Device-data
 *     errors (a slot or block id outside the pool, query_len > seq_len, a sequence longer than
 *     the hint) make the affected work item skip its memory accesses, set a bit in a device
 *     error word (the device's, or the stream's own: pa_set_stream_error_word) and leave its
 *     output rows unwritten; pa_get_device_error reports them.
 *   - Every wait inside a kernel gives up after two seconds (pa_set_wait_limit) and reports
 *     PA_ERR_TIMEOUT.
 *   - Thread-safety: functions may be called from several host threads; pa_last_error is
 *     per thread.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_VERSION 3
#define PA_PARTITION_TOKENS 512 /* keys per split-context partition */
#define PA_MAX_DIMS 5

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* bad pointer, dtype, rank, shape, stride or alignment */
  PA_ERR_UNSUPPORTED = 2, /* well-formed but not built: head_dim, block_size, group size */
  PA_ERR_CUDA = 3,        /* CUDA runtime error; pa_last_error() has the message */
  PA_ERR_TIMEOUT = 4,     /* device: a bounded wait gave up (reported by pa_get_device_error) */
  PA_ERR_OUT_OF_RANGE = 5,/* device: slot or block id outside the pool; access skipped */
  PA_ERR_WORKSPACE = 6,   /* workspace missing, misaligned or smaller than required */
  PA_ERR_DESCRIPTOR = 7,  /* device: query_len > seq_len, short block table, or hint exceeded */
  PA_ERR_NO_BLOCKS = 8    /* host block manager: too few free or evictable blocks */
} pa_status;

typedef enum pa_dtype {
  PA_F16 = 0,
  PA_I32 = 1,
  PA_I64 = 2,
  PA_F8E4M3 = 3, /* one byte: 1 sign, 4 exponent (bias 7), 3 mantissa bits; 0x7F/0xFF NaN, max 448 */
  PA_BF16 = 4    /* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits */
} pa_dtype;

typedef struct pa_tensor {
  void* data;                 /* device pointer, 16-byte aligned for fp16 / bf16 tensors */
  int32_t dtype;              /* pa_dtype */
  int32_t ndim;
  int64_t shape[PA_MAX_DIMS];
  int64_t stride[PA_MAX_DIMS];/* in elements */
} pa_tensor;

/* Host-side facts about the batch the scheduler already knows.  Upper bounds are fine; a
 * sequence that exceeds them is skipped on the device and reported as PA_ERR_DESCRIPTOR. */
typedef struct pa_batch_hint {
  int32_t max_query_len;    /* max over sequences of query_start_loc[s+1] - query_start_loc[s] */
  int32_t max_seq_len;      /* max over sequences of seq_lens[s] */
  int32_t num_prefill_seqs; /* count of sequences with more than one query row; 0 = not known,
                               then the prefill launch covers every sequence.  A batch with more
                               such sequences than this skips the extra ones and reports
                               PA_ERR_DESCRIPTOR.  When it equals the number of sequences (and
                               max_query_len > 1) the decode launches are skipped; a one-row
                               sequence in such a batch is then reported the same way. */
  int32_t shared_prefix_tokens; /* 0, or a multiple of 512 (and of the block size) smaller than
                               every sequence's seq_len: the first shared_prefix_tokens keys of
                               every sequence are the same physical blocks (the block tables
                               agree there), so they are attended once for all query rows (p1:
                               requests that start alike share pages; p2 prefix-caching slide)
                               and merged with each sequence's own keys by the log-sum-exp rule.
                               Decode rows only (else PA_ERR_UNSUPPORTED); a
                               sequence whose table differs there, or with no key past the
                               prefix, is reported as PA_ERR_DESCRIPTOR. */
} pa_batch_hint;

/*
 * pa_reshape_and_cache -- write this step's new K/V tokens into their cache slots.
 * ("vLLM: LLM Inference That Doesn't Waste Your GPU", "KV cache, in one picture": the K/V of every
 * processed token is stored once; "Local_LLM_03_vLLM_Architecture", paged-KV slide: the store is a
 * set of fixed-size blocks.)
 *
 *   k, v          fp16 or bf16 [T_new, Hkv, d]; token stride free (multiple of 8), head stride d.
 *   k_cache,
 *   v_cache       [NB, Hkv, bs, d] of the same type as k and v, contiguous ("HND" per block: one (block, kv head) is a
 *                 contiguous bs x d tile).  Written in place.
 *   slot_mapping  int64 [T_new]; token t goes to block slot/bs, offset slot%bs.  slot < 0 means
 *                 "padding, skip".  A slot >= NB*bs is skipped and reported on the device.
 * For every t with slot >= 0 and every kv head h: k_cache[slot/bs][h][slot%bs][:] = k[t][h][:]
 * (bit-exact copy), same for v.  Two tokens with the same slot race (the last writer is
 * unspecified), as the pages give no order between them.
 * Supported: d in {64, 128}, bs in {16, 32}.
 */
int pa_reshape_and_cache(const pa_tensor* k, const pa_tensor* v, const pa_tensor* k_cache,
                         const pa_tensor* v_cache, const pa_tensor* slot_mapping, void* stream);

/*
 * pa_attention_workspace_size -- bytes of scratch pa_attention needs for a batch.
 * Split-context partials: for T query rows, Hq heads and P = ceil(max_seq_len / 512)
 * partitions, fp32 o[T][Hq][P][d] plus fp32 m[T][Hq][P] and l[T][Hq][P].  0 when P <= 1.
 */
size_t pa_attention_workspace_size(int64_t num_tokens, int64_t num_q_heads, int64_t head_dim,
                                   int32_t max_seq_len);

/*
 * pa_attention -- paged attention for one mixed continuous-batching step.
 * ("Local_LLM_03_vLLM_Architecture", paged-KV slide: the kernel gathers K/V from scattered
 * physical blocks through the block table; chunked-prefill slide; "vLLM: LLM Inference That
 * Doesn't Waste Your GPU", "Continuous batching": prefill and decode in the same step.)
 *
 *   q                fp16 or bf16 [T, Hq, d]; token stride free (multiple of 8), head stride d.
 *   k_cache, v_cache [NB, Hkv, bs, d] of q's type, contiguous, already holding this step's tokens
 *                    (call pa_reshape_and_cache first, on the same stream).
 *   block_tables     int32 [N, MB]; row stride free.  Entry j of row s = physical block of
 *                    logical positions j*bs .. j*bs+bs-1 of sequence s.  Entries past
 *                    ceil(seq_lens[s]/bs) are never read.  Aliasing (the same block id in
 *                    several rows) is allowed and is how shared prefixes are expressed.
 *   seq_lens         int32 [N]; keys of sequence s after this step's tokens were written.
 *   query_start_loc  int32 [N+1]; query_start_loc[0] = 0, non-decreasing, [N] = T.  Sequence s
 *                    owns rows query_start_loc[s] .. query_start_loc[s+1]-1.  One row is a
 *                    decode step, several a prefill chunk; any mix and order in one call.
 *   scale            multiplies q.k before the softmax (typically 1/sqrt(d)).
 *   out              [T, Hq, d] of q's type, contiguous.
 *   hint             required; see pa_batch_hint.
 *   workspace        device scratch of at least pa_attention_workspace_size(T, Hq, d,
 *                    hint->max_seq_len) bytes, 256-byte aligned (NULL allowed when that is 0).
 *                    Owned by the caller; must not be shared by calls in flight at once.
 * Row i of sequence s sits at absolute position seq_lens[s] - q_len + i and attends to keys
 * 0 .. seq_lens[s] - q_len + i (bottom-right causal; q_len = 1 attends to all keys).  Query
 * head h reads kv head h / (Hq / Hkv).  out = softmax(scale * q K^T) V per row and head.
 * Rows with q_len = 1 and more than 512 keys are computed in 512-key partitions merged with
 * the log-sum-exp rule; so are verify rows (every sequence with at most a few rows: q_len x G
 * <= 8, or <= 32 over an FP8 cache), each with its own causal limit.  Longer chunks run on the
 * tensor-core prefill kernels, beside the decode work when the call has both; the
 * shared-prefix pass (hint->shared_prefix_tokens) runs beside the decode kernel too.  Both use
 * a side stream of the library's (one per device and host thread, created by the first such
 * call), forked from and joined back into `stream` with events, so a capture of the call into a
 * CUDA graph records the fork and the join.
 * Supported: d in {64, 128}, bs in {16, 32}, Hq / Hkv in 1..16.
 */
int pa_attention(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                 const pa_tensor* block_tables, const pa_tensor* seq_lens,
                 const pa_tensor* query_start_loc, float scale, const pa_tensor* out,
                 const pa_batch_hint* hint, void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * FP8 KV cache ("Local_LLM_03_vLLM_Architecture", KV-sizing slide: the cache's bytes per token
 * decide how many sequences fit and how fast decode reads them; the pages quantise weights
 * only, so storing K/V in 8 bits is this library's extension).  The pools are PA_F8E4M3
 * [NB, Hkv, bs, d] with one scale per tensor: a stored code c of K stands for
 * k_scale * value(c), of V for v_scale * value(c).  Both scales must be finite and > 0.
 */
typedef struct pa_kv_scales {
  float k_scale;
  float v_scale;
} pa_kv_scales;

/*
 * pa_reshape_and_cache_fp8 -- pa_reshape_and_cache into an FP8 cache: each new value x (fp16)
 * is stored as the E4M3 code of x * (1 / scale), the reciprocal and the product in float32,
 * rounded to nearest even; magnitudes from 448 up (and infinities) saturate to +-448, NaN
 * stays NaN.  Arguments and errors as pa_reshape_and_cache, with k_cache / v_cache PA_F8E4M3.
 */
int pa_reshape_and_cache_fp8(const pa_tensor* k, const pa_tensor* v, const pa_tensor* k_cache,
                             const pa_tensor* v_cache, const pa_tensor* slot_mapping,
                             const pa_kv_scales* scales, void* stream);

/*
 * pa_attention_fp8 -- pa_attention over an FP8 cache (q and out stay fp16).  Every E4M3 value
 * is exact in fp16, so the kernels widen the codes to fp16 (decode: into MMA operands in
 * registers; prefill: tile by tile in shared memory) and run the fp16 arithmetic with the score
 * scale multiplied by k_scale and the output by v_scale.  Any mix of decode, verify and prefill
 * rows, and the shared-prefix pass, as for pa_attention.  Workspace as for pa_attention.
 */
int pa_attention_fp8(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                     const pa_tensor* block_tables, const pa_tensor* seq_lens,
                     const pa_tensor* query_start_loc, float scale, const pa_tensor* out,
                     const pa_batch_hint* hint, const pa_kv_scales* scales, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * pa_attention_static_scratch -- pa_attention without a caller-provided workspace, for callers
 * that cannot allocate device memory (no paper counterpart: the pages describe no such call).
 *
 * Some callers may not call cudaMalloc at all: plugins inside a host program whose own pool
 * owns all device memory, or code on a serving path where allocating is not allowed because
 * cudaMalloc may block or synchronise and cudaFree synchronises the device.  This call takes the
 * same arguments as pa_attention minus the workspace and uses a fixed 32 MiB array in the
 * library's device memory for the split-context partials instead.  It allocates nothing.
 *   - Every GPU that loads the library holds the 32 MiB until the process exits.
 *   - A batch needing more than 32 MiB of scratch (pa_attention_workspace_size(T, Hq, d,
 *     hint->max_seq_len) > 32 MiB) is rejected with PA_ERR_WORKSPACE and a message; nothing runs.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current) and caches it; make that first call before any stream capture.
 *     The cached address belongs to the device's primary context as it was then: after
 *     cudaDeviceReset (or any teardown of that context) this entry point must not be called
 *     again in the same process.
 *   - All calls on a device share the array, which keeps the last call's contents; nothing in it
 *     needs to start at zero.  Calls that overlap on the GPU race on it: order them.
 * Results are those of pa_attention on the same inputs.
 */
int pa_attention_static_scratch(const pa_tensor* q, const pa_tensor* k_cache,
                                const pa_tensor* v_cache, const pa_tensor* block_tables,
                                const pa_tensor* seq_lens, const pa_tensor* query_start_loc,
                                float scale, const pa_tensor* out, const pa_batch_hint* hint,
                                void* stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char* pa_last_error(void);

/*
 * pa_get_device_error -- synchronise `stream`, then read and clear the error word that calls on
 * `stream` report into: the word registered for it with pa_set_stream_error_word, else the
 * current device's own word (shared by every unregistered stream of the device).  Returns PA_OK,
 * PA_ERR_TIMEOUT, PA_ERR_OUT_OF_RANGE or PA_ERR_DESCRIPTOR (most severe first); *bits (may be
 * NULL) receives the raw word: 1 timeout, 2 slot out of range, 4 block id out of range,
 * 8 descriptor, 16 hint exceeded.
 */
int pa_get_device_error(void* stream, uint32_t* bits);

/*
 * pa_set_stream_error_word -- let later calls on `stream` (a cudaStream_t; NULL is the legacy
 * default stream) report their device errors into `device_word` instead of the device's shared
 * word, so that a caller serving several streams reads each stream's errors apart.  The word is
 * a caller-owned, 4-byte aligned device uint32 that the caller zeroes first; the library only
 * ORs bits into it and pa_get_device_error(stream, ...) clears it.  NULL turns the stream back
 * to the device's word.  The word must stay allocated while calls registered to it can run.  At
 * most 64 streams hold a word of their own at a time (PA_ERR_INVALID_ARG beyond, and for a
 * misaligned word).  Any host thread may register; the registration is process-wide.
 */
int pa_set_stream_error_word(void* stream, uint32_t* device_word);

/*
 * pa_copy_blocks -- copy whole physical blocks of the pool: K and V of every kv head of block
 * pairs[i][0] are copied to block pairs[i][1] ("Local_LLM_03_vLLM_Architecture", prefix-caching
 * slide: shared blocks; a sequence that appends into a partial block it shares gets its own
 * copy first, the copy-on-write the host block manager asks for).
 *   k_cache, v_cache  [NB, Hkv, bs, d], contiguous, fp16, bf16 or PA_F8E4M3 (both the same).
 *   pairs             int32 [n, 2] contiguous device array (src, dst).  Destinations must be
 *                     distinct and never a source of the same call.
 * A pair with an id outside the pool is skipped and reported as PA_ERR_OUT_OF_RANGE by
 * pa_get_device_error.  n = 0 is a no-op.
 */
int pa_copy_blocks(const pa_tensor* k_cache, const pa_tensor* v_cache, const pa_tensor* pairs,
                   void* stream);

/*
 * pa_set_timing_events -- measurement hook.  When both are non-NULL (cudaEvent_t handles),
 * every later pa_attention call on this host thread records `start` on its stream just before
 * launching the selected kernel and `stop` just after it, so a caller can time that kernel with
 * CUDA events inside a longer step: `kernel` is PA_TIMED_DECODE (the decode-partition kernel,
 * launched by every call with rows), PA_TIMED_PREFILL (the chunked-prefill kernel, launched
 * when hint->max_query_len > 1) or PA_TIMED_SHARED_PREFIX (the shared-prefix pass, launched
 * when hint->shared_prefix_tokens > 0).  No work is skipped or reordered.  Pass NULL, NULL to turn
 * the selected hook off.  Returns PA_OK, or PA_ERR_INVALID_ARG for an unknown `kernel`.
 */
#define PA_TIMED_DECODE 0
#define PA_TIMED_PREFILL 1
#define PA_TIMED_SHARED_PREFIX 2
int pa_set_timing_events(int kernel, void* start, void* stop);

/*
 * pa_set_wait_limit -- how long every bounded wait inside the kernels of later pa_attention and
 * pa_attention_fp8 calls on this host thread may last before it gives up: the waiting work item
 * then lets its own copies in flight land, leaves its output rows unwritten and sets the
 * timeout bit that pa_get_device_error reports as PA_ERR_TIMEOUT (the CUDA context stays
 * usable).  A legitimate wait lasts microseconds; the default is 2 s.  Returns PA_OK, or
 * PA_ERR_INVALID_ARG (limit unchanged) outside [PA_WAIT_LIMIT_MIN_NS, PA_WAIT_LIMIT_MAX_NS].
 */
#define PA_WAIT_LIMIT_DEFAULT_NS 2000000000ull
#define PA_WAIT_LIMIT_MIN_NS 1000ull
#define PA_WAIT_LIMIT_MAX_NS 10000000000ull
int pa_set_wait_limit(uint64_t limit_ns);

/* PA_VERSION of the built library. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
