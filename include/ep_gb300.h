/*
 * ep_gb300.h -- C ABI of the single-GPU MoE expert-parallel layout /
 * dispatch / combine library (libep_gb300.so, sm_103a).
 *
 * The operations are the ones of the EPHandle / dispatch / combine API of
 * "DeepEP overall architecture analysis" (ElasticBuffer class diagram:
 * dispatch(x, topk_idx, ...) -> (recv_x, handle), combine(x, handle, ...);
 * EPHandle class listing; "Dispatch data flow" and "Combine data flow"
 * figures), with the configuration fields of EpCfg from "MORI JIT v2" §3.2
 * and that page's conventions for a C boundary (§6: every entry point catches
 * everything, returns a negative code on error and leaves the message in a
 * last-error string; §3.5: a configuration that cannot be served is rejected
 * when the handle is built, never turned into wrong numbers).
 *
 * All "ranks" are logical: rank r owns experts [r*Epr, (r+1)*Epr) and one
 * contiguous slice of the receive buffer, all in the memory of the current
 * GPU.  No call transfers data between GPUs.
 *
 * Conventions for every entry point:
 *   - Pointers documented "device" must point to memory of the current CUDA
 *     device; the library never dereferences them on the host.
 *   - The caller owns every buffer it passes (inputs and outputs).  The
 *     handle owns its routing metadata (allocated by ep_handle_create, freed
 *     by ep_handle_free).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream).  No
 *     entry point synchronises the device: ep_handle_create waits for its
 *     own clearing memset only, ep_handle_status and ep_handle_free for the
 *     handle's last stream only.  The layout,
 *     dispatch and combine calls allocate nothing and can be enqueued while a
 *     stream is being captured into a CUDA graph.
 *   - Return value 0 on success, else one of the negative EP_E* codes, with
 *     a message available from ep_last_error() on the calling thread.
 *   - One handle holds one routing (its fields, and the barrier state of the
 *     single-launch layout): the caller orders the work it enqueues on one
 *     handle (one stream, or events between streams), as it would for any
 *     buffer two kernels write.  Different handles are independent and may
 *     run at the same time on different streams.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stdint.h>

#ifdef __cplusplus
#define EP_NOEXCEPT noexcept
extern "C" {
#else
#define EP_NOEXCEPT
#endif

/* Same object as cudaStream_t; declared here so that this header needs no CUDA header. */
typedef struct CUstream_st *ep_stream_t;

/* Transport dtype of the dispatched rows; numbering as EpDType in
 * "MORI JIT v2" §3.7 (Bf16 = 0, Fp32 = 1, Fp8 = 2, Fp4x2 = 3).
 *   EP_BF16, EP_FP32  rows of H bf16 / fp32 values, moved as bytes;
 *   EP_FP4X2          rows of H packed e2m1 values (H/2 bytes, two per byte),
 *                     moved as bytes (the payload arrives already packed);
 *   EP_FP8_E4M3       bf16 rows cast on the way to OCP e4m3, one fp32 scale
 *                     per 128 channels.
 * Combine always reduces bf16 expert outputs, whatever was dispatched. */
typedef enum {
    EP_BF16 = 0,
    EP_FP32 = 1,
    EP_FP8_E4M3 = 2,
    EP_FP4X2 = 3
} ep_dtype_t;

/* Configuration ("MORI JIT v2" §3.2 EpCfg; expert_alignment from the EPHandle
 * listing).  Valid ranges (checked by ep_handle_create):
 *   1 <= world_size <= 64, 1 <= max_tok_per_rank, world_size*max_tok_per_rank <= 2^24,
 *   1 <= num_expert_per_rank, world_size*num_expert_per_rank <= 2048,
 *   1 <= num_expert_per_token <= 16, 1 <= expert_alignment <= 4096,
 *   hidden_dim >= 8, hidden_dim % 8 == 0 (rows are whole 16-byte units), hidden_dim <= 32768;
 *   for EP_FP8_E4M3 also hidden_dim % 128 == 0, for EP_FP4X2 hidden_dim % 32 == 0;
 *   the receive capacity (ep_recv_capacity) must fit in int32. */
typedef struct {
    int32_t world_size;           /* W: logical ranks */
    int32_t hidden_dim;           /* H: channels per token row */
    int32_t max_tok_per_rank;     /* T: tokens per logical rank; N <= W*T */
    int32_t num_expert_per_rank;  /* Epr; E = W*Epr experts */
    int32_t num_expert_per_token; /* K: top-k */
    int32_t expert_alignment;     /* A: each expert's receive segment is padded to a multiple of A */
    int32_t dispatch_dtype;       /* ep_dtype_t */
    int32_t use_weights;          /* 1: combine weights rows by topk_weights; 0: plain sum */
    int32_t no_expand;            /* 0: expand layout (EPHandle do_expand = true): one receive
                                   *    row per (token, expert), grouped by expert, padded to A;
                                   * 1: non-expand layout (do_expand = false): one receive row per
                                   *    (token, destination rank), grouped by rank, no padding;
                                   *    requires use_weights = 0 (the rank's experts apply the
                                   *    weights; combine sums the rank rows) */
} ep_cfg_t;

enum {
    EP_OK = 0,
    EP_EINVAL = -1,        /* invalid argument or configuration */
    EP_EUNSUPPORTED = -2,  /* a valid request this library does not serve */
    EP_ECUDA = -3,         /* a CUDA runtime call failed (message has the CUDA error) */
    EP_ENOMEM = -4         /* device allocation failed */
};

/* Opaque handle: the configuration, the routing metadata of the last
 * ep_layout call, and the kernels chosen for this configuration. */
typedef struct ep_handle *ep_handle_t;

/* Receive-buffer rows needed for any routing of up to W*T tokens:
 * expand layout Rcap = W*T*K + E*(A-1) (every (token, k) gets a row; each
 * expert segment adds at most A-1 padding rows); non-expand layout
 * Rcap = W*T*min(K, W) (a token reaches at most min(K, W) ranks).  Returns a
 * negative EP_E* code for an invalid configuration. */
int64_t ep_recv_capacity(const ep_cfg_t *cfg) EP_NOEXCEPT;

/* Validate cfg, pick the compiled kernel variants for it and allocate the
 * handle's device metadata on the current device (sized for W*T tokens), with
 * the stream-ordered allocator (cudaMallocAsync) on a private non-blocking
 * stream, then clear it on that stream and wait for that stream alone: work
 * running on the caller's streams is neither waited for nor disturbed.
 * *out receives the handle.  Errors: EP_EINVAL (bad cfg or NULL;
 * no_expand = 1 with use_weights = 1), EP_EUNSUPPORTED, EP_ENOMEM, EP_ECUDA. */
int ep_handle_create(const ep_cfg_t *cfg, ep_handle_t *out) EP_NOEXCEPT;

/* A handle that uses the routing of another handle's ep_layout instead of
 * computing its own, e.g. an FP8 dispatch fed by the layout that already
 * serves a bf16 dispatch of the same tokens (one layout per routing, as the
 * router produces one topk_idx per step).  cfg must equal layout_src's cfg in
 * world_size, max_tok_per_rank, num_expert_per_rank, num_expert_per_token,
 * expert_alignment and no_expand; hidden_dim, dispatch_dtype and use_weights
 * may differ.  The new handle allocates no metadata: ep_dispatch /
 * ep_combine on it read layout_src's routing as of layout_src's last
 * ep_layout (order the calls on one stream, or with events), ep_handle_get
 * returns layout_src's fields, ep_handle_status reads and clears layout_src's
 * error word, and ep_layout on it returns EP_EINVAL.  layout_src must stay
 * alive until the new handle is freed; sharing a shared handle shares its
 * layout_src.  Errors: EP_EINVAL (NULL, bad or mismatched cfg, another
 * device), EP_EUNSUPPORTED, EP_ECUDA. */
int ep_handle_create_shared(const ep_cfg_t *cfg, ep_handle_t layout_src, ep_handle_t *out) EP_NOEXCEPT;

/* Layout.  topk_idx: device int64 [num_tokens, K] row-major, token t of
 * logical rank t / T.  Entries equal to -1 are masked (no receive row); any
 * other value outside [0, E) is skipped and sets the value 1 (bit 0) in the
 * device error word (see ep_handle_status).  Computes on the device, into the handle:
 *   num_unaligned_recv_tokens_per_expert [E]   entries routed to each expert
 *   num_tokens_per_rank [W]                    tokens with >= 1 expert on rank r
 *   psum_num_recv_tokens_per_expert [E+1]      exclusive prefix sum of the
 *                                              counts padded to a multiple of A
 *   psum_num_recv_tokens_per_rank [W+1]        the same sum at each rank's first expert
 *   num_recv_tokens [1]                        R = psum_expert[E]
 *   dst_slot [num_tokens, K]                   receive row of each (t, k), -1 if skipped;
 *                                              rows of one expert follow the flat order t*K+k
 *   recv_src_metadata [Rcap, K+2]              for each received row:
 *                                              {t / T, t mod T, dst_slot[t][0..K-1]};
 *                                              -1 in every row that receives nothing
 *   send_slot [num_tokens, K]                  the rows dispatch writes token t to and
 *                                              combine reads it from (expand: dst_slot)
 * (EPHandle listing of "DeepEP overall architecture analysis").
 * Non-expand layout (cfg.no_expand = 1; the EPHandle's do_expand = false): the
 * counts and psum_num_recv_tokens_per_expert are as above (the receiving
 * experts' token counts), and
 *   psum_num_recv_tokens_per_rank [W+1]        exclusive prefix sum of num_tokens_per_rank
 *   num_recv_tokens [1]                        R = psum_rank[W], one row per (token, rank)
 *   rows                                       rank r owns [psum_rank[r], psum_rank[r+1]),
 *                                              its tokens once each, ascending
 *   dst_slot [num_tokens, K]                   the row of t on the rank of topk_idx[t][k]
 *                                              (entries on one rank share it), -1 if skipped
 *   send_slot [num_tokens, K]                  t's distinct rows, ascending, then -1
 *   recv_src_metadata [Rcap, K+2]              {t / T, t mod T, dst_slot[t][0..K-1]} per row
 * 0 <= num_tokens <= W*T, else EP_EINVAL.  The number of tokens is kept in the
 * handle for the following ep_dispatch / ep_combine calls.
 * Mid-size batches run as one cooperative launch whose CTAs meet at a grid
 * barrier; each wait there is bounded (EP_GB300_WAIT_NS when the handle was
 * created, default 1 s) and a CTA that gives up records the value 2 (bit 1)
 * in the device error word and leaves its part of the outputs unwritten.  A
 * cooperative launch that cannot be resident at once fails with EP_ECUDA. */
int ep_layout(ep_handle_t h, const int64_t *topk_idx, int32_t num_tokens, ep_stream_t stream) EP_NOEXCEPT;

/* Dispatch ("Dispatch data flow": token data + scale factors to the receive
 * buffer).  x: device [N, row] row-major, 16-byte aligned.
 * EP_BF16 / EP_FP32 / EP_FP4X2: x holds bf16 / fp32 / packed-e2m1 rows and
 *              recv_x [Rcap, row] receives recv_x[dst_slot[t][k]] = x[t], bit-exact.
 * EP_FP8_E4M3: x bf16 [N, H]; recv_x device uint8 (e4m3) [Rcap, H], recv_scales device fp32
 *              [Rcap, H/128]; per token and 128-channel group g:
 *              s = amax|x[t, g]| / 448 (fp32), q = e4m3_rn_satfinite(x / s),
 *              s = 0 and q = 0 when amax = 0; written to every row dst_slot[t][k].
 * Non-expand layout: x[t] is written once to each row send_slot[t][j] >= 0.
 * recv_scales must be non-NULL for EP_FP8_E4M3 and NULL otherwise.  Rows
 * that receive no token are not written.  Uses the routing of the last
 * ep_layout call on this handle (same stream, or ordered after it).
 * Buffers must be 16-byte aligned, else EP_EINVAL. */
int ep_dispatch(ep_handle_t h, const void *x, void *recv_x, float *recv_scales,
                ep_stream_t stream) EP_NOEXCEPT;

/* Dispatch that also forwards the routing with each received row (the copy
 * epilogue of the "Dispatch data flow" fills recv_topk_idx and
 * recv_topk_weights).  Same as ep_dispatch, and for every received (t, k):
 *   recv_topk_weights[dst_slot[t][k]] = topk_weights[t][k]   (fp32 [Rcap])
 *   recv_topk_idx[dst_slot[t][k]]     = topk_idx[t][k]       (int32 [Rcap], global expert id)
 * Non-expand layout: every received row s of token t gets K entries,
 *   recv_topk_idx[s][k]     = topk_idx[t][k] if (t, k) is carried by s (dst_slot[t][k] == s), else -1
 *   recv_topk_weights[s][k] = topk_weights[t][k] if so, else 0.0f   (both [Rcap, K])
 * Either output may be NULL (then it is not written); topk_weights (device
 * fp32 [N, K]) is required when recv_topk_weights is given.  Rows that
 * receive nothing are not written. */
int ep_dispatch_fwd(ep_handle_t h, const void *x, void *recv_x, float *recv_scales,
                    const float *topk_weights, float *recv_topk_weights, int32_t *recv_topk_idx,
                    ep_stream_t stream) EP_NOEXCEPT;

/* Combine ("Combine data flow": reduce weighted by topk_weights back to token
 * order).  y: device bf16 [Rcap, H] expert outputs, in the receive layout;
 * topk_weights: device fp32 [N, K] (ignored, may be NULL, when use_weights is
 * 0); out: device bf16 [N, H].  For every token t and channel c:
 *   acc = +0.0f; for k = 0..K-1 with dst_slot[t][k] >= 0:
 *       acc = fmaf(w[t][k], y[dst_slot[t][k]][c], acc)     (acc += y without weights)
 *   out[t][c] = bf16 round-to-nearest-even(acc).
 * Non-expand layout: acc = +0.0f; acc = acc + y[send_slot[t][j]][c] for the
 * token's rows in ascending order (ascending rank); no weights.
 * Padding rows of y are never read.  Buffers must be 16-byte aligned.  With
 * EP_GB300_COMBINE_TMA=1 set when the handle was created, the rows are staged
 * in shared memory by TMA bulk copies (same result; a wait on those copies is
 * bounded and reports device error value 2 when it gives up). */
int ep_combine(ep_handle_t h, const void *y, const float *topk_weights, void *out,
               ep_stream_t stream) EP_NOEXCEPT;

/* Layout without any device allocation.  The pages have no counterpart to
 * this call; it exists for callers that cannot call cudaMalloc, for example
 * code whose device memory is entirely owned by another framework's pool
 * allocator, a serving loop that must not allocate after start-up, or a
 * caller that is handed buffers but has no allocator of its own.
 * ep_handle_create allocates the layout's outputs and scratch; this call
 * writes the same outputs as ep_layout (same definitions, same bytes) into
 * buffers the caller passes, and keeps its scratch in a fixed 1 MiB array
 * compiled into the library (held by every GPU that loads the library until
 * the process exits).  Batches of up to 2048 tokens run the single-launch
 * cluster layout, which needs no scratch at all.
 *   cfg                       as for ep_handle_create (dispatch_dtype,
 *                             hidden_dim and use_weights are checked but unused;
 *                             no_expand = 1 returns EP_EUNSUPPORTED)
 *   topk_idx                  device int64 [num_tokens, K], 8-byte aligned
 *   num_unaligned_per_expert  device int32 [E]
 *   num_tokens_per_rank       device int32 [W]
 *   psum_per_expert           device int32 [E+1]
 *   psum_per_rank             device int32 [W+1]
 *   num_recv                  device int32 [1]
 *   dst_slot                  device int32 [num_tokens, K]
 *   recv_src_metadata         device int32 [Rcap, K+2] (8-byte aligned when K is even)
 *   device_error              device int32 [1]; cleared, then error bits as in
 *                             ep_handle_status (value 1 (bit 0): an id outside [-1, E) was skipped)
 * Size limit: 3*(E+W)*ceil(num_tokens/128) + (E+W) int32 of scratch must fit
 * in 262144 (for example 32768 tokens over 256 experts and 8 ranks need
 * 203016); larger requests return EP_EINVAL with the sizes in the message.
 * The first call on a device, with that device current, looks up the
 * scratch array's address and sets the layout kernels' shared-memory limit
 * on that device; make that first call before any stream capture.  That
 * set-up is kept only when it succeeds (a failed one is tried again by the
 * next call) and belongs to the device's current CUDA context: after
 * cudaDeviceReset the next call repeats it.  Every
 * call shares the scratch array: calls that may run at the same time on the
 * GPU (unordered streams) overwrite each other's scratch and give wrong
 * results, so order them (one stream, or events).  Allocates nothing. */
int ep_layout_noalloc(const ep_cfg_t *cfg, const int64_t *topk_idx, int32_t num_tokens,
                      int32_t *num_unaligned_per_expert, int32_t *num_tokens_per_rank,
                      int32_t *psum_per_expert, int32_t *psum_per_rank, int32_t *num_recv,
                      int32_t *dst_slot, int32_t *recv_src_metadata, int32_t *device_error,
                      ep_stream_t stream) EP_NOEXCEPT;

/* Combine with a bias and a choice of output ("Combine data flow": reduce
 * weighted by topk_weights, "+ bias", write back).  As ep_combine, and then
 *   acc += bias[t][c]            (bias: device bf16 [N, H], or NULL; one fp32 add)
 *   out[t][c] = acc              (out_dtype EP_FP32: out device fp32 [N, H])
 *   out[t][c] = bf16_rn(acc)     (out_dtype EP_BF16: out device bf16 [N, H])
 * Other out_dtype values return EP_EINVAL. */
int ep_combine_ex(ep_handle_t h, const void *y, const float *topk_weights, const void *bias,
                  void *out, int32_t out_dtype, ep_stream_t stream) EP_NOEXCEPT;

/* Release the handle and its device memory.  Waits for the stream of the
 * handle's last layout / dispatch / combine call (which must still exist),
 * then frees the metadata in stream order on the handle's private stream.
 * Work on other streams that uses the handle must be complete, or ordered
 * before that last call, when this is called.  NULL is ignored. */
void ep_handle_free(ep_handle_t h) EP_NOEXCEPT;

/* Fields of the handle, for ep_handle_get. */
enum {
    EP_FIELD_NUM_UNALIGNED_PER_EXPERT = 0, /* int32 [E] */
    EP_FIELD_NUM_TOKENS_PER_RANK = 1,      /* int32 [W] */
    EP_FIELD_PSUM_PER_EXPERT = 2,          /* int32 [E+1] */
    EP_FIELD_PSUM_PER_RANK = 3,            /* int32 [W+1] */
    EP_FIELD_DST_SLOT = 4,                 /* int32 [N, K] (N of the last layout) */
    EP_FIELD_RECV_SRC_METADATA = 5,        /* int32 [Rcap, K+2] */
    EP_FIELD_NUM_RECV = 6,                 /* int32 [1] */
    EP_FIELD_DEVICE_ERROR = 7,             /* int32 [1], sticky error bits */
    EP_FIELD_TOPK_IDX = 8,                 /* int32 [N, K] copy of topk_idx (-1 where skipped) */
    EP_FIELD_SEND_SLOT = 9                 /* int32 [N, K] rows of each token (expand: dst_slot) */
};

/* Device pointer and element count of one handle field (the handle keeps
 * ownership; valid until ep_handle_free).  EP_EINVAL for an unknown field. */
int ep_handle_get(ep_handle_t h, int32_t field, void **dev_ptr, int64_t *numel) EP_NOEXCEPT;

/* Read and clear the sticky device error word, in order on the stream of
 * the handle's last layout / dispatch / combine call, and wait for that
 * stream only.  Values: 1 (bit 0) = a topk id outside [-1, E) was skipped;
 * 2 (bit 1) = a kernel gave up a bounded wait (the layout's grid barrier, the
 * TMA dispatch's or TMA combine's copies).  Returns EP_ECUDA if the
 * copy or the synchronisation fails. */
int ep_handle_status(ep_handle_t h, int32_t *device_error) EP_NOEXCEPT;

/* Name of the kernel variant chosen for a step (0 = layout, 1 = dispatch,
 * 2 = combine) written to buf (NUL-terminated, truncated to len).  A name
 * carries the compile-time shape, e.g. "ep_dispatch_bf16_h7168_k8", or
 * "..._generic" when no specialisation for the shape was compiled.  For the
 * layout it names what the last ep_layout ran: "ep_layout_cluster_k8" for
 * the single-launch thread-block-cluster kernel that serves batches of up to
 * 2048 tokens (unless EP_GB300_LAYOUT_CLUSTER=0 when the handle was created),
 * "ep_layout_fused_k8" for the single-launch cooperative kernel that serves
 * batches of up to a few hundred ranges of 128-256 tokens (unless
 * EP_GB300_LAYOUT_FUSED=0), "ep_layout_k8" for the three launches (count,
 * spine, slots). */
int ep_handle_variant(ep_handle_t h, int32_t step, char *buf, int32_t len) EP_NOEXCEPT;

/* Run-time specialisation ("MORI JIT v2" §1-§3.4, §6 precompile; the JIT
 * flow of "DeepEP overall architecture analysis").  A configuration whose
 * (hidden, top-k) has no compiled variant gets one at ep_handle_create: the
 * kernel bodies are rendered into source text for that shape, compiled with
 * NVRTC for the device, and kept in an on-disk cache keyed by SHA-256 of the
 * entry name, compiler version, flags, kernel-body headers and source text
 * (directory $EP_GB300_JIT_CACHE, default ~/.cache/ep_gb300/jit; entries
 * published by an atomic rename, so concurrent processes agree).  Such a
 * kernel serves 32-byte-aligned buffers (combine: without bias, bf16 output);
 * the compiled generic variant serves the rest, and everything when NVRTC is
 * missing or EP_GB300_JIT=0.  ep_handle_variant reports which ran.
 * ep_jit_precompile fills the cache for cfg without a GPU, for architecture
 * `arch` (NULL or "" = "sm_103a"), and writes one line per step to report
 * ("<name> compiled-in|generic|compiled <dir>|cached <dir>").  Returns the
 * number of kernels it compiled (0 when all were cached or compiled in), or
 * EP_EINVAL, EP_EUNSUPPORTED (no NVRTC), EP_ECUDA (compile or file error, with
 * the compiler log in ep_last_error()). */
int ep_jit_precompile(const ep_cfg_t *cfg, const char *arch, char *report, int32_t len) EP_NOEXCEPT;

/* Message of the last failed call on this thread ("" if none). */
const char *ep_last_error(void) EP_NOEXCEPT;

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
