/*
 * pkv.h -- C ABI of the paged-KV grouped-query attention library for GB300 (sm_103a).
 *
 * Two operations make up one attention layer's step of a continuous-batching, paged-KV
 * serving engine:
 *
 *   pkv_kv_append        fused RoPE + KV-cache write of the step's new tokens
 *                        ("mini_engine" README, "Next: fused kernels": fused RoPE, fused QKV
 *                        split and KV-cache write; "09 -- Mini Inference Engine (The
 *                        Capstone)", "Week 4 -- Paged KV cache": pool of fixed-size
 *                        blocks; "Design decisions you'll face": 16 tokens per block for
 *                        a first engine, the block size a tunable to measure later).
 *   pkv_paged_attention  grouped-query attention of every new token over its sequence's
 *                        paged context, decode tokens and causal prefill chunks mixed in one
 *                        call ("mini_engine" README, "What it does": GQA, paged KV cache,
 *                        chunked prefill; "09 -- ...", "Week 3 -- Continuous batching":
 *                        mixed prefill/decode batches with varying lengths; "Week 4":
 *                        attention that gathers through the block table).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named *_dev are CUDA device pointers; the library never dereferences them on
 *    the host.  All tensors are owned by the caller; the library allocates no device memory
 *    (scratch space comes from the caller's workspace), never synchronises, and enqueues its
 *    kernels asynchronously on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *    default stream).  Every call works on the device that is current on the calling thread.
 *  - bf16 tensors hold IEEE bfloat16 values.  The last dimension (head_dim) is contiguous;
 *    other strides are in ELEMENTS.  Every row of head_dim elements must start on a 16-byte
 *    boundary (base pointers 16-byte aligned, strides multiples of 8 elements).
 *  - KV pool layout (per layer): k_cache and v_cache are each a contiguous bf16 tensor
 *    [num_blocks][block_size][num_kv_heads][head_dim].  block_size is a power of two from 8
 *    to 128 (16 is the usual choice).  Slot s denotes row (s % block_size) of physical
 *    block (s / block_size), i.e. row s of the pool viewed as
 *    [num_blocks * block_size][num_kv_heads][head_dim].  num_blocks < 2^31 (int32 ids).
 *  - q head h attends with kv head h / (num_q_heads / num_kv_heads).
 *  - RoPE is the rotate-half form: pair (i, i + d/2) turns by pos * theta^(-2i/d).
 *  - Return value: PKV_OK, or a PKV_ERR_* code.  On a host-side validation error nothing is
 *    launched.  No C++ exception crosses this boundary.
 *  - Data-dependent index errors (a slot or block id outside the pool, a context longer than
 *    its block-table row, a malformed query_start_loc) are detected on the device: the
 *    offending access is skipped (or redirected to block 0), the affected output is
 *    unspecified, and a bit is or-ed into a per-device error word that
 *    pkv_get_device_error() reads.  Kernels never trap.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes returned by every entry point ---- */
#define PKV_OK 0
#define PKV_ERR_NULL 1        /* a required pointer is NULL                                   */
#define PKV_ERR_SHAPE 2       /* a size is negative or sizes disagree                          */
#define PKV_ERR_STRIDE 3      /* a stride is not allowed (overlapping rows, non-contiguous pool) */
#define PKV_ERR_ALIGN 4       /* a pointer or stride breaks the 16-byte row alignment           */
#define PKV_ERR_UNSUPPORTED 5 /* head_dim / block_size / head counts outside the compiled set   */
#define PKV_ERR_WORKSPACE 6   /* workspace NULL, misaligned (256 B) or smaller than required    */
#define PKV_ERR_CUDA 7        /* a CUDA runtime call or kernel launch failed                    */

/* ---- device-side error bits (pkv_get_device_error) ---- */
#define PKV_DEVERR_SLOT_RANGE 0x1u  /* kv_append: slot >= num_blocks*block_size; write skipped    */
#define PKV_DEVERR_BLOCK_RANGE 0x2u /* attention: block id outside [0, num_blocks); read block 0  */
#define PKV_DEVERR_SPAN 0x4u        /* attention: query_start_loc not monotone, past num_tokens,
                                       or context shorter than the span; sequence skipped        */
#define PKV_DEVERR_CONTEXT 0x8u     /* context > max_blocks_per_seq*block_size; seq/token skipped */
#define PKV_DEVERR_TIMEOUT 0x10u    /* a bounded wait inside a kernel ran out; output unspecified */

/* Block sizes: the default, and the supported range (powers of two). */
#define PKV_BLOCK_SIZE 16
#define PKV_MIN_BLOCK_SIZE 8
#define PKV_MAX_BLOCK_SIZE 128

/* Human-readable name of a status code (static string, never NULL). */
PKV_API const char* pkv_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
PKV_API int pkv_version(void);

/*
 * pkv_kv_append -- fused RoPE and KV-cache append for the step's new tokens.
 *
 * For each new token t in [0, num_tokens):
 *   q[t, h, :]   <- bf16(rope(q[t, h, :], positions[t]))            for every q head (in place)
 *   if slot_mapping[t] >= 0, with s = slot_mapping[t]:
 *     k_cache[s/bs, s%bs, h, :] <- bf16(rope(k[t, h, :], positions[t]))   for every kv head
 *     v_cache[s/bs, s%bs, h, :] <- v[t, h, :]                              (bit copy)
 *   (bs = block_size)
 * Rotation: the angle pos * f_i is reduced modulo one turn exactly in 64-bit fixed point
 * (pkv_rope_turn_table), then to a quarter turn and an fp32 remainder in [-pi/4, pi/4];
 * sincosf and the pairwise rotation run in fp32; rounding to bf16 nearest-even.  Before that
 * rounding a rotated value is within 2.7e-7 (|x_i| + |x_{i+d/2}|) of the exact rotation of
 * the bf16 inputs (positions below 2^31).
 * A negative slot marks padding and writes nothing.  A slot >= num_blocks*bs is skipped
 * and sets PKV_DEVERR_SLOT_RANGE.  Duplicate slots in one call give an unspecified row.
 *
 *   q_dev          bf16 [num_tokens][num_q_heads][head_dim], strides (q_stride_token,
 *                  q_stride_head); rotated in place.  May alias a packed QKV buffer.
 *   k_dev, v_dev   bf16 [num_tokens][num_kv_heads][head_dim] with their own strides; read only.
 *   positions_dev  int64 [num_tokens]: absolute position of each token (>= 0).
 *   slot_mapping_dev int64 [num_tokens]: destination slot, or < 0 to skip.
 *   k_cache_dev, v_cache_dev  bf16 pools (layout above) of num_blocks blocks.
 *   head_dim       64 or 128.   block_size  8, 16, 32, 64 or 128.
 *   rope_theta     RoPE base, finite and > 0 (any value above 1e-280), e.g. 1e6 for Qwen3;
 *                  else PKV_ERR_SHAPE.
 * num_tokens == 0 is a no-op returning PKV_OK.
 */
PKV_API int pkv_kv_append(void* q_dev, int64_t q_stride_token, int64_t q_stride_head,
                  const void* k_dev, int64_t k_stride_token, int64_t k_stride_head,
                  const void* v_dev, int64_t v_stride_token, int64_t v_stride_head,
                  const int64_t* positions_dev, const int64_t* slot_mapping_dev,
                  void* k_cache_dev, void* v_cache_dev,
                  int64_t num_tokens, int64_t num_q_heads, int64_t num_kv_heads,
                  int64_t head_dim, int64_t num_blocks, int64_t block_size,
                  double rope_theta, void* stream);

/*
 * pkv_kv_append_paged -- pkv_kv_append with each token's position and slot derived on the
 * device from the scheduler's tables instead of passed in ("mini-vllm" README, "Milestones",
 * 7: GPU-side slot derivation).  Token t belongs to the sequence b whose span
 * [query_start_loc[b], query_start_loc[b+1]) contains it; it sits at position
 * pos = context_lens[b] - span_b + (t - query_start_loc[b]) and is written to slot
 * block_tables[b][pos / bs] * bs + pos % bs.  Tokens outside every span are only rotated
 * (q) and write nothing.  Inconsistent tables set PKV_DEVERR_SPAN / _CONTEXT / _BLOCK_RANGE
 * and skip the token's K/V write.  Table arguments as in pkv_paged_attention; the others as in
 * pkv_kv_append.  positions_out / slot_mapping_out (int64 [num_tokens], may be NULL) receive
 * the derived values (-1 slot for skipped tokens).
 */
PKV_API int pkv_kv_append_paged(void* q_dev, int64_t q_stride_token, int64_t q_stride_head,
                                const void* k_dev, int64_t k_stride_token, int64_t k_stride_head,
                                const void* v_dev, int64_t v_stride_token, int64_t v_stride_head,
                                const int32_t* block_tables_dev, int64_t block_tables_stride,
                                int64_t max_blocks_per_seq,
                                const int32_t* context_lens_dev, const int32_t* query_start_loc_dev,
                                int64_t num_seqs, void* k_cache_dev, void* v_cache_dev,
                                int64_t num_tokens, int64_t num_q_heads, int64_t num_kv_heads,
                                int64_t head_dim, int64_t num_blocks, int64_t block_size,
                                double rope_theta, int64_t* positions_out_dev,
                                int64_t* slot_mapping_out_dev, void* stream);

/*
 * pkv_rope_turn_table -- the rotation frequencies pkv_kv_append uses, computed on the host (no
 * GPU, no CUDA call): out[i], i < head_dim / 2, is f_i / (2 pi) modulo 1 as a 0.64 fixed-point
 * fraction of a turn, f_i = rope_theta^(-2i / head_dim) evaluated with the C library's pow in
 * fp64, i.e. round(frac(f_i / (2 pi)) * 2^64) mod 2^64, within one unit.  A token at position
 * p turns pair i by 2 pi ((p * out[i]) mod 2^64) / 2^64 radians.  ("mini_engine" README, "What
 * it does": RoPE.)  out holds head_dim / 2 values, owned by the caller.  Returns PKV_ERR_NULL
 * for a NULL out, PKV_ERR_UNSUPPORTED for head_dim outside {64, 128}, PKV_ERR_SHAPE for a
 * theta pkv_kv_append refuses.
 */
PKV_API int pkv_rope_turn_table(double rope_theta, int64_t head_dim, uint64_t* out);

/*
 * pkv_paged_attention_workspace_size -- bytes of device workspace pkv_paged_attention needs
 * for these sizes on the current device (the split-K partials and the work plan).
 * Returns 0 if the sizes are invalid.  The result depends on the device's SM count and on
 * pkv_set_decode_ctas(); call it on the device that will run the attention.
 */
PKV_API size_t pkv_paged_attention_workspace_size(int64_t num_tokens, int64_t num_seqs,
                                          int64_t num_q_heads, int64_t num_kv_heads,
                                          int64_t head_dim, int64_t max_blocks_per_seq);

/*
 * pkv_paged_attention -- grouped-query attention over a ragged batch of paged sequences.
 *
 * Sequence b owns query rows [query_start_loc[b], query_start_loc[b+1]) (its span, n rows)
 * and context_lens[b] keys (ctx, counting the span's own tokens, which kv_append has already
 * written).  Its keys live in physical blocks block_tables[b, 0 .. ceil(ctx/bs)-1]
 * (bs = block_size).
 * Row r of the span is the token at position ctx - n + r; for every q head h:
 *     out[row, h, :] = softmax_j(scale * q[row, h, :] . K[j, h/G, :]) V[j, h/G, :],
 *     j over keys 0 .. ctx - n + r           (G = num_q_heads / num_kv_heads)
 * A span of one row is a decode step and sees the whole context; longer spans are causal
 * chunked-prefill spans.  Accumulation is fp32; out is rounded to bf16 nearest-even.
 * Rows of out outside every span are not written.  Spans may be empty.
 *
 *   q_dev            bf16 [num_tokens][num_q_heads][head_dim] (already rotated), strides as given.
 *   k_cache_dev, v_cache_dev  the pool (layout above), num_blocks blocks of block_size
 *                    tokens (8, 16, 32, 64 or 128).
 *   block_tables_dev int32 [num_seqs][block_tables_stride]; only the first
 *                    ceil(ctx/bs) <= max_blocks_per_seq entries of row b are read.
 *   context_lens_dev int32 [num_seqs].
 *   query_start_loc_dev int32 [num_seqs + 1], non-decreasing, [0] = 0, [num_seqs] <= num_tokens.
 *   out_dev          bf16 [num_tokens][num_q_heads][head_dim], strides as given; must not
 *                    overlap q.
 *   scale            softmax scale (typically 1/sqrt(head_dim)).
 *   workspace_dev    >= pkv_paged_attention_workspace_size(...) bytes, 256-byte aligned,
 *                    owned by the caller, used as scratch; its contents need no
 *                    initialisation and are clobbered.  Calls that share a workspace
 *                    must be stream-ordered.
 * Supported: head_dim in {64, 128}; num_kv_heads in {1, 2, 4, 8};
 *            num_q_heads / num_kv_heads in [1, 8].
 * Ordering: all work is ordered after earlier work on `stream`, and later work on `stream`
 * is ordered after all of it.  With prefill spans (num_tokens > num_seqs) the prefill tiles
 * may run on a second stream, forked from `stream` after the planner and joined back into it
 * before the call returns (pkv_set_overlap): the caller's own (pkv_paged_attention_ex) or the
 * library's, one per device, shared by all callers.  The library's second stream is used
 * only when no CUDA graph capture holds it, or when the capture holding it is the one this
 * call is captured into; otherwise the call runs its kernels in the serial order on `stream`
 * (same results up to fp32 rounding of the decode rows).  So a capture of `stream` and
 * eager calls on other streams can be open at the same time.  With num_tokens <= num_seqs
 * no prefill kernel is launched: the rows of a longer span (which then needs empty spans
 * beside it) are computed by the decode path, each row over its own causal context.
 */
PKV_API int pkv_paged_attention(const void* q_dev, int64_t q_stride_token, int64_t q_stride_head,
                        const void* k_cache_dev, const void* v_cache_dev,
                        int64_t num_blocks, int64_t block_size,
                        const int32_t* block_tables_dev, int64_t block_tables_stride,
                        int64_t max_blocks_per_seq,
                        const int32_t* context_lens_dev, const int32_t* query_start_loc_dev,
                        int64_t num_seqs,
                        void* out_dev, int64_t out_stride_token, int64_t out_stride_head,
                        int64_t num_tokens, int64_t num_q_heads, int64_t num_kv_heads,
                        int64_t head_dim, float scale,
                        void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * pkv_attention_options -- per-call settings of pkv_paged_attention_ex.  Zero-initialise,
 * set struct_size = sizeof(pkv_attention_options), then set what the call needs; a zero field
 * keeps the process default (the pkv_set_* functions below).
 *   decode_kernel   0 default, 1 CUDA cores, 2 tensor cores (as pkv_set_decode_kernel)
 *   prefill_kernel  0 default, 1 mma.sync tiles, 2 tcgen05 tiles (as pkv_set_prefill_kernel)
 *   overlap         0 default, 1 prefill tiles beside the decode when possible, 2 serial order
 *   decode_ctas     0 default, else the decode grid of this call (1 .. 65536); the workspace
 *                   must then hold pkv_paged_attention_workspace_size_ex(..., decode_ctas)
 *   flags           0, or PKV_ATTN_PLAN_EARLY: the planner reads query_start_loc and
 *                   context_lens, and does all its arithmetic, while the work enqueued just
 *                   before this call may still be running, and writes the workspace only once
 *                   that work has finished; a decode step then hides the planner behind its
 *                   pkv_kv_append.  Set it only when that work neither writes these two arrays
 *                   nor lets later work start before their writer has finished: the step's
 *                   pkv_kv_append qualifies (it waits for all earlier work before it lets later
 *                   work start).  Batches of more than 1024 sequences ignore the flag.
 *                   PKV_ATTN_STREAM_EARLY (implies PKV_ATTN_PLAN_EARLY): besides, the planner
 *                   writes the workspace as soon as the plan is known, and the tensor-core
 *                   decode starts copying the pages that hold no key of this step's new tokens
 *                   while that work may still be running; it reads q, and every page that may
 *                   hold a new token's key, only once that work has finished.  Set it only when
 *                   that work also writes nothing this call reads except q and the new tokens'
 *                   slots of k_cache and v_cache (positions context - span .. context - 1 of each
 *                   sequence), and starts later work only after all work before it has finished
 *                   (so no kernel of an earlier call still reads the workspace): the step's
 *                   pkv_kv_append qualifies.  Batches of more than 1024 sequences ignore it.
 *                   The decode then learns that the plan is ready through a word the planner
 *                   publishes, about one round trip to L2 later than through the planner's end:
 *                   on a small, latency-bound batch that costs more than it hides (GB300: about
 *                   +1 us for 32 sequences of up to 1152 keys, -2 us for 256 of up to 2048).
 *   side_stream, fork_event, join_event
 *                   all NULL: the library's own second stream for the prefill beside the
 *                   decode; else a caller-owned stream (cudaStream_t) and two caller-created
 *                   events (cudaEvent_t, timing disabled) that order it after the planner and
 *                   back into `stream` -- independent callers on different streams then never
 *                   share, or serialise on, a stream of the library's.  The caller must not
 *                   use them for anything else until the call's work has completed.
 * Invalid values (unknown flag bits included) give PKV_ERR_SHAPE; one or two of the three
 * handles given give PKV_ERR_NULL.
 */
#define PKV_ATTN_PLAN_EARLY 1
#define PKV_ATTN_STREAM_EARLY 2
typedef struct pkv_attention_options {
  uint32_t struct_size;
  int32_t decode_kernel;
  int32_t prefill_kernel;
  int32_t overlap;
  int32_t decode_ctas;
  int32_t flags;  /* PKV_ATTN_* bits */
  void* side_stream;
  void* fork_event;
  void* join_event;
} pkv_attention_options;

/* pkv_paged_attention with per-call settings (NULL options: the same as pkv_paged_attention). */
PKV_API int pkv_paged_attention_ex(const void* q_dev, int64_t q_stride_token, int64_t q_stride_head,
                                   const void* k_cache_dev, const void* v_cache_dev,
                                   int64_t num_blocks, int64_t block_size,
                                   const int32_t* block_tables_dev, int64_t block_tables_stride,
                                   int64_t max_blocks_per_seq,
                                   const int32_t* context_lens_dev, const int32_t* query_start_loc_dev,
                                   int64_t num_seqs,
                                   void* out_dev, int64_t out_stride_token, int64_t out_stride_head,
                                   int64_t num_tokens, int64_t num_q_heads, int64_t num_kv_heads,
                                   int64_t head_dim, float scale,
                                   void* workspace_dev, size_t workspace_bytes, void* stream,
                                   const pkv_attention_options* options);

/* Workspace bytes for a call with options.decode_ctas = decode_ctas (0: the process default,
 * as pkv_paged_attention_workspace_size).  Returns 0 for invalid sizes. */
PKV_API size_t pkv_paged_attention_workspace_size_ex(int64_t num_tokens, int64_t num_seqs,
                                                     int64_t num_q_heads, int64_t num_kv_heads,
                                                     int64_t head_dim, int64_t max_blocks_per_seq,
                                                     int32_t decode_ctas);

/*
 * pkv_paged_attention_noalloc -- pkv_paged_attention for callers that cannot allocate
 * device memory.  It has no counterpart in the pages; it is a deployment convenience.
 *
 * Some callers may not call cudaMalloc: code that receives its device buffers from a host
 * framework that owns all device memory, and serving loops that keep cudaMalloc / cudaFree
 * out of the step because those calls can block, synchronise the device, or fail mid-step
 * when memory is tight.  This entry point takes the same arguments as pkv_paged_attention
 * except the workspace: its scratch is a fixed array of PKV_NOALLOC_SCRATCH_BYTES (16 MiB)
 * inside the library.  The caller still passes (and owns) every input and the output.
 *
 *  - Every GPU that loads the library holds the 16 MiB array until the process exits.
 *  - The first call on a device (with that device current) looks up the array's device
 *    address once; make that first call before any stream capture.
 *  - Sizes whose scratch would exceed PKV_NOALLOC_SCRATCH_BYTES (see
 *    pkv_paged_attention_workspace_size) are refused with PKV_ERR_WORKSPACE and nothing is
 *    launched.  Other errors are those of pkv_paged_attention.
 *  - All calls on a device share the one array, and it keeps the last call's contents
 *    (nothing in it needs to start at zero).  Calls whose kernels overlap on the GPU (other
 *    streams, other host threads without ordering) race on it: order them on one stream.
 *  - No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
PKV_API int pkv_paged_attention_noalloc(const void* q_dev, int64_t q_stride_token, int64_t q_stride_head,
                                        const void* k_cache_dev, const void* v_cache_dev,
                                        int64_t num_blocks, int64_t block_size,
                                        const int32_t* block_tables_dev, int64_t block_tables_stride,
                                        int64_t max_blocks_per_seq,
                                        const int32_t* context_lens_dev, const int32_t* query_start_loc_dev,
                                        int64_t num_seqs,
                                        void* out_dev, int64_t out_stride_token, int64_t out_stride_head,
                                        int64_t num_tokens, int64_t num_q_heads, int64_t num_kv_heads,
                                        int64_t head_dim, float scale, void* stream);

/*
 * The pkv_set_* settings below are process-wide defaults for calls without options (every
 * thread and stream of the process sees a change at once); they are meant for tests and
 * tuning.  Per-call settings: pkv_paged_attention_ex.
 *
 * pkv_set_decode_ctas -- override the number of CTAs the decode split-K kernel uses
 * (0 = automatic: one per SM; at most 65536).  Changes the
 * split points, hence rounding, never the result beyond fp32 rounding.  Returns PKV_OK,
 * or PKV_ERR_SHAPE for a negative value.
 */
PKV_API int pkv_set_decode_ctas(int32_t ctas);

/*
 * pkv_set_overlap -- 1 (default): a batch with prefill spans runs its prefill tiles on a
 * second stream at the same time as the decode, the SMs split between the two by the
 * planner (the decode is bound by HBM bandwidth and reaches it without every SM); 0: the
 * prefill tiles and then the decode run on the caller's stream, each over all SMs.  Only
 * the tcgen05 prefill tiles with the default decode grid (pkv_set_decode_ctas(0)) use the
 * split.  Prefill rows are bit-identical either way; decode rows may differ by fp32
 * rounding (other split points).  Process-wide.  Returns PKV_ERR_SHAPE for another value.
 */
PKV_API int pkv_set_overlap(int on);

/*
 * pkv_set_decode_kernel -- choose the arithmetic of the decode split-K kernel for later calls:
 * 0 automatic (currently the tensor cores for every group size, the faster of the two on GB300),
 * 1 CUDA cores (per-lane fp32 FMA, warp-shuffle reductions),
 * 2 tensor cores (bf16 mma.sync with the GQA group as the N dimension).
 * Both compute the same result up to fp32 rounding.  Process-wide; for tests and tuning.
 * Returns PKV_ERR_SHAPE for another value.
 */
PKV_API int pkv_set_decode_kernel(int kind);

/*
 * pkv_set_prefill_kernel -- choose the arithmetic of the prefill-chunk tiles for later calls:
 * 0 automatic (currently 2), 1 bf16 mma.sync tiles of 64 query rows of one q head, 2 tcgen05
 * tiles of 128 rows stacking the G q heads of a kv head (floor(128 / G) positions x G heads;
 * TMEM accumulators, TMA-staged operands; falls back to 1 when q's strides do not admit a TMA
 * tensor map).  Both compute the same result up to fp32 rounding.
 * Process-wide; for tests and tuning.  Returns PKV_ERR_SHAPE for another value.
 */
PKV_API int pkv_set_prefill_kernel(int kind);

/*
 * pkv_set_kernel_events -- instrumentation: from now on, every launch of kernel `which`
 * records `start_event` on its stream just before the launch and `stop_event` just after
 * (both cudaEvent_t passed as void*, created by the caller).  NULL events (or which = 0)
 * switch recording off for that kernel.  Process-wide; meant for benchmarks that time one
 * kernel inside a call.  Returns PKV_ERR_SHAPE for an unknown `which`.
 *   which: 1 kv_append, 2 planner, 3 prefill tiles, 4 decode split-K (which also runs the
 *   split merge of sequences cut by its CTA ranges).
 */
#define PKV_KERNEL_APPEND 1
#define PKV_KERNEL_PLAN 2
#define PKV_KERNEL_PREFILL 3
#define PKV_KERNEL_DECODE 4
PKV_API int pkv_set_kernel_events(int which, void* start_event, void* stop_event);

/*
 * pkv_set_fault_injection -- TEST ONLY: makes later pkv_paged_attention calls exercise the
 * bounded waits inside the kernels (failure detection without a GPU fault).  kind 0 (default)
 * turns it off.  PKV_FAULT_DECODE_NO_COPIES: the tensor-core decode kernel's producer warp
 * issues no copy and no barrier arrival, so every consumer wait of a CTA with work runs out
 * after about 2^31 SM clocks (about one second), sets PKV_DEVERR_TIMEOUT in the error word
 * and the CTA finishes without further waits; nothing is left in flight and the context
 * stays usable.  The decode rows of such a call are unspecified.
 * PKV_FAULT_PLAN_NO_READY: with PKV_ATTN_STREAM_EARLY the planner never publishes its ready
 * word, so every decode CTA's bounded poll of it runs out (2^24 SM clocks, about 8 ms) and the
 * CTA falls back to waiting for the planner's end: the call is slower but its rows are
 * correct and no error is reported.  Process-wide.  Returns PKV_ERR_SHAPE for another kind.
 */
#define PKV_FAULT_DECODE_NO_COPIES 1
#define PKV_FAULT_PLAN_NO_READY 2
PKV_API int pkv_set_fault_injection(int kind);

/*
 * pkv_copy -- copy `bytes` from `src` to `dst` with a kernel on `stream` (no function of the
 * pages: plumbing for staging a step's inputs).  Either buffer may be device memory or pinned
 * host memory the device can address under unified addressing (e.g. from cudaHostAlloc); on
 * a Grace-Blackwell part the SMs reach pinned host memory over NVLink-C2C.  Ordered on
 * `stream` like any kernel.  Both pointers and `bytes` must be multiples of 16 (else
 * PKV_ERR_ALIGN); NULL pointers give PKV_ERR_NULL; bytes == 0 is a no-op.  The buffers must
 * not overlap.
 */
PKV_API int pkv_copy(void* dst, const void* src, size_t bytes, void* stream);

/*
 * pkv_get_device_error -- read the current device's error word (PKV_DEVERR_* bits or-ed
 * together since the last clear) into *bits, after synchronising `stream`.  If clear != 0
 * the word is reset to zero.  This call blocks the host; the others never do.
 */
PKV_API int pkv_get_device_error(uint32_t* bits, int clear, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
