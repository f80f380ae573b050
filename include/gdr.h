/*
 * gdr.h -- C ABI of the GB300 channelwise gated delta rule forward library.
 *
 * The operation (page "Reorder channelwise gated delta rule chunked hot loops
 * for autovectorization", pytorch/executorch PR #21021): each value head keeps
 * a float32 state S[dk][dv] (row i = key channel, column j = value channel).
 * Every token t, in order,
 *     decays the rows of S by exp(g_t[i])            (per key channel),
 *     predicts  vhat = S^T k_t                      (from the decayed state),
 *     updates   S += beta_t * k_t (v_t - vhat)^T    (rank-one delta correction),
 *     outputs   o_t = S^T q_t                       (from the updated state).
 * There is no 1/sqrt(dk) query scale: fold one into q if wanted.
 *
 * Routing (same page, second commit summary): T == 1 runs the single-token
 * decode kernel, which streams the state once; T > 1 runs the chunkwise
 * WY/UT prefill (per-channel log-decay prefix sums, causal query/key terms,
 * the beta-folded unit-lower triangular transform, WY pseudo-keys and
 * pseudo-values, inter-chunk state carry, ragged last chunk).
 *
 * Grouped heads (trymirai/uzu PR #576, review thread on the per-value-head
 * gram): HK key/query heads serve HV value heads, G = HV / HK; value head hv
 * reads key/query head hv / G (contiguous groups).
 *
 * Memory and layouts.  Every pointer is DEVICE memory owned by the caller,
 * 16-byte aligned (beta: 4-byte aligned), densely packed row-major with the
 * last index fastest:
 *     q, k   [B][T][HK][dk]   dtype qkv_dtype
 *     v      [B][T][HV][dv]   dtype qkv_dtype
 *     g      [B][T][HV][dk]   float32, natural-log decay (<= 0 expected, not checked)
 *     beta   [B][T][HV]       float32, used as given (no sigmoid applied)
 *     h0     [B][HV][dk][dv]  float32 initial state, or NULL for zeros
 *     out    [B][T][HV][dv]   dtype qkv_dtype (rounded to nearest even for bf16)
 *     ht     [B][HV][dk][dv]  float32 final state, or NULL to skip storing it
 * ht == h0 (the same pointer) updates the state in place.  Any other overlap
 * between an output (out, ht) and any other argument is rejected.
 *
 * Supported shapes: B >= 0, T >= 0, HK >= 1, HV % HK == 0, dk and dv in
 * {32, 64, 128}, chunk in {16, 32, 64} (the prefill chunk length; the result
 * does not depend on it beyond rounding).  B == 0 does nothing.  T == 0
 * writes ht = h0 (or zeros) and nothing else.
 *
 * Streams and errors.  All work is enqueued on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and the calls return without waiting for it.
 * Argument errors are detected before anything is enqueued and leave every
 * output untouched.  GDR_ERR_CUDA means a CUDA runtime call or launch failed;
 * gdr_last_cuda_error() gives the cudaError_t code.  No call allocates device
 * memory except gdr_forward, which owns a per-device workspace (see there).
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>

#if defined(__GNUC__)
#define GDR_API __attribute__((visibility("default")))
#else
#define GDR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdr_status {
    GDR_OK = 0,
    GDR_ERR_NULL = 1,        /* a required pointer is NULL */
    GDR_ERR_SHAPE = 2,       /* negative size, HV % HK != 0, or a size that overflows */
    GDR_ERR_UNSUPPORTED = 3, /* dk, dv, chunk or dtype outside the supported set */
    GDR_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned (beta: 4-byte) */
    GDR_ERR_WORKSPACE = 5,   /* caller workspace NULL or smaller than gdr_workspace_bytes */
    GDR_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
    GDR_ERR_TIMEOUT = 7,     /* a kernel gave up on a bounded wait (see gdr_device_check) */
    GDR_ERR_ALIAS = 8        /* an output overlaps another argument (other than ht == h0) */
} gdr_status;

typedef enum gdr_dtype {
    GDR_F32 = 0,  /* q, k, v, out are float32 */
    GDR_BF16 = 1  /* q, k, v, out are bfloat16; g, beta, h0, ht stay float32 */
} gdr_dtype;

/* Flags for gdr_forward_ex and the other entries that take them (0 in normal
 * calls; the first two are for tests and diagnosis). */
#define GDR_FLAG_FORCE_CHUNKED 1u /* run the chunked prefill even when T == 1 */
/* the chunked prefill on CUDA cores throughout (chunk prep and state scan),
 * even where the fused tensor-core kernel or the tensor-core state scan applies */
#define GDR_FLAG_FORCE_GENERIC 2u
/*
 * Scalar gate: g holds one log-decay per token and value head, [B][T][HV]
 * float32 (varlen: [total][HV]), applied to every key channel -- the gated
 * delta rule with a per-head decay, the case the review thread of "Support
 * TreeUpdateSolve kernel" (trymirai/uzu PR #576) discusses for a per-key-head
 * gram.  Accepted by gdr_forward_ex, gdr_workspace_bytes, gdr_forward_varlen,
 * gdr_varlen_workspace_bytes, gdr_forward_tree and gdr_tree_workspace_bytes
 * (trees of up to 64 tokens with a scalar gate run as one CUDA-core chunk,
 * longer ones on the blocked solve).
 */
#define GDR_FLAG_SCALAR_GATE 4u
/*
 * Segmented state scan (gdr_forward, gdr_forward_ex, gdr_workspace_bytes; the
 * tensor-core prefill, and the chunked prefill's state scan on the tensor
 * cores when dk = dv = 128).  The chunk-to-chunk state carry is serial, one
 * CTA per (batch, value head) walking its chunks in order, so a small batch
 * x heads leaves most SMs idle.  The route then cuts the sequence into P
 * segments of whole chunks.  Over a segment the recurrence is an affine map
 * of the state, S_end = M S_start + c (M [dk][dk] from k, g and beta alone),
 * which is how the chunk carry of the second commit summary of "Reorder
 * channelwise gated delta rule chunked hot loops for autovectorization"
 * (pytorch/executorch PR #21021) composes.  Segment 0 runs from h0 at the
 * same time as the runs that give the middle segments' maps; the maps are
 * chained to every segment's start state; the other segments then run from
 * those starts.  The walk is two segments long instead of P.
 *
 * Chosen automatically when it pays: P is the largest value with
 * B * HV * (2P - 3) CTAs fitting on the device's SMs at once and segments
 * of at least 8 chunks; P >= 3 is needed.  The route needs workspace
 * (gdr_workspace_bytes reports it): its tables, which are copied in from
 * host memory like those of gdr_forward_varlen (pass GDR_FLAG_NO_SEGMENTS
 * when capturing into a CUDA graph), and 2P - 3 f32 states per (batch,
 * value head).  Results agree with the unsegmented route to within the
 * tolerance of the route, not bit for bit (the states of later segments
 * are reached through the maps).
 *
 * On the chunked prefill (f32 q/k/v, or a chunk other than 64) every chunk's
 * records are built at once as before and only the state scan is cut: its
 * runs are scan CTAs over those records (the map runs read the values as
 * zero), segments are whole chunks of the call's chunk length, and the
 * launches are the prep, the first scan wave, the combine and the second
 * scan wave (and, with h0, one copy of it into the first segments' states).  GDR_FLAG_FORCE_GENERIC (the CUDA-core scan) and
 * dk or dv other than 128 never segment.
 *
 * GDR_FLAG_NO_SEGMENTS: never segment.
 * GDR_FLAG_SEGMENTS(n): segment into at most n pieces (2 <= n <= 255;
 * fewer when the sequence has fewer chunks), whatever the device; for tests.
 */
#define GDR_FLAG_NO_SEGMENTS 8u
#define GDR_FLAG_SEGMENTS(n) ((((unsigned)(n)) & 0xffu) << 8)
/* gdr_forward_tree: take the blocked solve (the route of trees past 64
 * tokens) at any T. */
#define GDR_FLAG_TREE_BLOCKED 0x10000u
/* gdr_forward_tree, blocked solve, scalar gate: build the gram once per value
 * head (the fused form) instead of once per key head and share it across the
 * key head's value heads (the default); for comparing the two. */
#define GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD 0x20000u

/*
 * Bytes of device workspace gdr_forward_ex needs for this call (0 when the
 * chosen route needs none).  Returns 0 for arguments gdr_forward_ex would
 * reject.  Same shape arguments and flags as gdr_forward_ex.
 * Passage: none in the pages; it sizes the scratch of the routes of
 * gdr_forward_ex (the CUDA-core chunked prefill keeps per-chunk records, the
 * segmented scan its tables and segment states).
 */
GDR_API size_t gdr_workspace_bytes(int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                   int qkv_dtype, unsigned flags);

/*
 * The forward pass with a caller-owned workspace.  `workspace` is device
 * memory of at least gdr_workspace_bytes(...) bytes (may be NULL when that is
 * 0), 256-byte aligned, not overlapping any other argument, and must not be
 * used by anything else until the enqueued work is done.  Allocates nothing.
 * Passage: "Reorder channelwise gated delta rule chunked hot loops for
 * autovectorization" (pytorch/executorch PR #21021), first commit summary
 * (the two-pass token recurrence that T == 1 runs) and second commit summary
 * (the routing by length and the chunkwise WY/UT form that T > 1 runs).
 */
GDR_API gdr_status gdr_forward_ex(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const float *h0, void *out, float *ht,
                                  int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                  void *stream, int qkv_dtype, void *workspace,
                                  size_t workspace_bytes, unsigned flags);

/*
 * The forward pass with the library's own workspace.  The library keeps one
 * workspace per device and grows it with cudaMalloc when a call needs more
 * (cudaMalloc synchronises the device, so a growing call is not
 * asynchronous).  Calls that share the library workspace must be ordered:
 * issue them on one stream per device, or use gdr_forward_ex.
 * gdr_forward takes no flags, so a tensor-core prefill with a small batch x
 * heads may take the segmented state scan (GDR_FLAG_NO_SEGMENTS below).  On
 * that route the call copies its tables from pageable host memory, so it
 * cannot be captured in a CUDA graph; whether it is taken depends on the
 * device's SM count; and its results agree with the single walk within the
 * route's tolerance, not bit for bit.  gdr_forward_ex with
 * GDR_FLAG_NO_SEGMENTS is the deterministic, capturable alternative.
 * Passage: as gdr_forward_ex; the argument list is that of the method's
 * description (q, k, v, g, beta, h0, out, ht, B, T, HK, HV, dk, dv, chunk,
 * stream) plus the q/k/v dtype.
 */
GDR_API gdr_status gdr_forward(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, const float *h0, void *out, float *ht,
                               int B, int T, int HK, int HV, int dk, int dv, int chunk,
                               void *stream, int qkv_dtype);

/*
 * Passage: none in the pages (memory management of gdr_forward).
 * Registers a caller-owned device workspace for gdr_forward on the current
 * device: from now on gdr_forward uses it instead of allocating, and a call
 * that needs more than `bytes` returns GDR_ERR_WORKSPACE (size it with
 * gdr_workspace_bytes for the largest call).  `dev_ptr` must be 256-byte
 * aligned (GDR_ERR_ALIGN) and non-NULL when bytes > 0 (GDR_ERR_NULL); it
 * stays the caller's, must outlive the work enqueued with it, and must not
 * be used by anything else meanwhile.  dev_ptr = NULL (or bytes = 0) goes back
 * to the library's own workspace.  The library's buffer, if one was
 * allocated, is kept.  gdr_forward_ex and the other entries take their
 * workspace per call and ignore this.
 */
GDR_API gdr_status gdr_set_workspace(void *dev_ptr, size_t bytes);

/*
 * Size in bytes of the fixed device scratch array behind
 * gdr_forward_chunked_noalloc (64 MiB, held on every device that loads the
 * library until the process exits).
 */
#define GDR_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * The chunked CUDA-core prefill (the same kernels and results as
 * gdr_forward_ex with GDR_FLAG_FORCE_CHUNKED | GDR_FLAG_FORCE_GENERIC) with
 * its workspace taken from a fixed array inside the library instead of being
 * allocated or passed in.  Nothing in the pages corresponds to it: it exists
 * for callers that cannot allocate device memory -- a runtime whose memory
 * planner owns every device byte and gives operators only their inputs and
 * outputs, a serving loop that must never pay cudaMalloc's device-wide
 * synchronisation, or a plugin whose host process lets only its own caching
 * allocator own device memory.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Arguments, layouts and errors are those of gdr_forward (T == 1 is run
 * through the chunked path too).  A problem whose workspace
 * (gdr_workspace_bytes with those two flags) exceeds
 * GDR_NOALLOC_SCRATCH_BYTES is rejected with GDR_ERR_WORKSPACE before
 * anything is enqueued.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current) and caches
 * it; make that first call before any stream capture.  All calls on a device
 * share the one array and it keeps the last call's contents (each call writes
 * every scratch word it reads, so nothing needs clearing): calls whose work
 * can overlap on the GPU -- different streams, or different host threads --
 * race on it and must be serialised by the caller.
 */
GDR_API gdr_status gdr_forward_chunked_noalloc(const void *q, const void *k, const void *v,
                                               const float *g, const float *beta,
                                               const float *h0, void *out, float *ht, int B,
                                               int T, int HK, int HV, int dk, int dv, int chunk,
                                               void *stream, int qkv_dtype);

/*
 * The forward pass on HOST buffers.  Arguments and layouts are those of
 * gdr_forward, except that q, k, v, g, beta, h0, out and ht are host memory
 * (page-locked for the copies to run asynchronously; pageable memory works
 * but each copy then waits for the host).  Nothing in the pages corresponds
 * to it: it is the input/output path of a caller whose tensors live on the
 * host.  Each batch element is streamed in segments of whole chunks (2048
 * tokens when T > 4096, else the whole sequence), each segment resuming from
 * the state the previous one left in a device state buffer, through two
 * device slots in `staging` (device memory of gdr_host_staging_bytes(...)
 * bytes, 256-byte aligned): while one segment computes on `stream`, the next
 * is copied in and the previous one copied out on two library-owned streams,
 * so the copies in both directions overlap the compute.  Ordered after
 * earlier work on `stream`; later work on `stream` starts after the last
 * copy out.  Up to T = 4096 the results equal those of gdr_forward on the
 * same values bit for bit; beyond, they differ by the rounding of the state
 * handed from segment to segment.  Calls from several host threads are
 * serialised while they enqueue.  Errors as gdr_forward_ex
 * (GDR_ERR_WORKSPACE for a short staging buffer); a failure after the first
 * copy leaves the outputs partly written, and the call makes `stream` wait
 * for the copies already queued on the library's streams before it returns
 * the error, so the host buffers may be reused once `stream` has completed.
 */
GDR_API size_t gdr_host_staging_bytes(int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                      int qkv_dtype);
GDR_API gdr_status gdr_forward_host(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *h0, void *out, float *ht,
                                    int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                    void *stream, int qkv_dtype, void *staging,
                                    size_t staging_bytes);

/*
 * Packed variable-length batches.  The same page's second commit summary
 * treats every sequence of a batch independently, routes a sequence of one
 * token to the single-token recurrence and runs a ragged last chunk through
 * the chunkwise path; this entry runs N such sequences of different lengths
 * stored back to back, with one launch per route for the whole batch.
 *
 *   cu_seqlens  HOST int32 [N + 1]: cu_seqlens[0] == 0, non-decreasing;
 *               sequence n is token rows cu_seqlens[n] .. cu_seqlens[n+1]-1.
 *               Read during the call only.
 *   q, k        [total][HK][dk]   (total = cu_seqlens[N]), dtype qkv_dtype
 *   v, out      [total][HV][dv]   dtype qkv_dtype
 *   g           [total][HV][dk]   float32
 *   beta        [total][HV]       float32
 *   h0, ht      [N][HV][dk][dv]   float32, slot n = sequence n; NULL as in
 *               gdr_forward (ht == h0 updates in place)
 *
 * Sequence n starts from h0[n] (zeros if NULL) and leaves its final state in
 * ht[n]; a zero-length sequence copies h0[n] (or zeros) to ht[n].  Each
 * sequence takes the route gdr_forward_ex would give it as a B = 1 call
 * with the same flags: length 1 the single-token kernel, longer ones the
 * tensor-core prefill (bf16, dk = dv = 128, chunk 64) or else the chunked
 * prefill (chunk prep, then the state scan on the tensor cores unless
 * GDR_FLAG_FORCE_GENERIC); the outputs equal those of N such calls with
 * GDR_FLAG_NO_SEGMENTS bit for bit, except on the sequences cut below.
 * Long prefill sequences may take the segmented state scan (see
 * GDR_FLAG_SEGMENTS), those of the tensor-core prefill and those of the
 * chunked prefill's tensor-core scan each chosen among their own kind:
 * automatically the largest P >= 3 for which HV CTAs per whole-walking
 * sequence plus HV (2P - 3) per cut one fit on the device's SMs at once,
 * cutting the sequences of at least 8P chunks that spread over exactly P
 * segments; GDR_FLAG_SEGMENTS(n) cuts every prefill sequence that spreads
 * over exactly n; GDR_FLAG_NO_SEGMENTS none.
 * A cut sequence agrees with the unsegmented result within the route's
 * tolerance, not bit for bit.
 * Enqueued on `stream`: one host-to-device copy of the batch's tables (from
 * pageable host memory: the call returns once the bytes have been taken, so
 * it cannot be captured in a CUDA graph), one copy or memset per zero-length
 * sequence, then at most four kernel launches, plus those of the segmented
 * scan (a second table copy, an initialisation, two prefill waves, the
 * combine and one state copy per cut sequence) when sequences are cut.
 *
 * `workspace`: device memory of at least gdr_varlen_workspace_bytes(...)
 * bytes, 256-byte aligned, untouched by anything else until the stream has
 * passed this call.  Allocates nothing.  Errors: GDR_ERR_SHAPE for a
 * cu_seqlens that breaks the rules above; the rest as gdr_forward_ex.
 */
GDR_API size_t gdr_varlen_workspace_bytes(const int *cu_seqlens, int N, int HK, int HV, int dk,
                                          int dv, int chunk, int qkv_dtype, unsigned flags);
GDR_API gdr_status gdr_forward_varlen(const void *q, const void *k, const void *v, const float *g,
                                      const float *beta, const float *h0, void *out, float *ht,
                                      const int *cu_seqlens, int N, int HK, int HV, int dk, int dv,
                                      int chunk, void *stream, int qkv_dtype, void *workspace,
                                      size_t workspace_bytes, unsigned flags);

/*
 * Tree verification (page "Support TreeUpdateSolve kernel", trymirai/uzu PR
 * #576): each batch element's T tokens are a tree of draft tokens, and each
 * token sees the state reached by running the recurrence along its own root
 * path -- its ancestors from the root down, then itself -- starting from
 * h0[b] (zeros if NULL).  out[b][t] is that run's output for token t.
 *
 *   parent  HOST int32 [B][T]: parent[b][t] in [-1, t-1] (parents precede
 *           their children; -1: the token follows h0 directly).  Read during
 *           the call only.
 *   q, k, v, g, beta, h0, out: layouts as in gdr_forward, T <= 512.
 *
 * There is no final-state output: a tree has one state per leaf.  To commit
 * an accepted path, run gdr_forward (or gdr_forward_varlen) on its tokens
 * from the same h0.  A tree is one unit-lower system over its tokens: path
 * prefix sums of g, and the ancestor relation in place of the causal order.
 * Routes: T <= 64 with bf16 q/k/v and dk = dv = 128 runs as one chunk of the
 * tensor-core prefill kernel (one launch); other T <= 64 calls, or any with
 * GDR_FLAG_FORCE_GENERIC, as one chunk of the CUDA-core kernels (two
 * launches, float32 throughout); T > 64, or any call with
 * GDR_FLAG_TREE_BLOCKED, on the blocked solve (four launches: ancestor
 * masks, path sums of g, the ancestor-masked grams of every 16 x 16 block
 * pair in parallel, then one CTA per tree, value head and dv part
 * substituting through the blocks in order; bf16 mma.sync, bf16 pairs
 * hi + lo for f32 q/k/v).  With a scalar gate the gram is built once per key
 * head and shared by its value heads (GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD:
 * once per value head).
 * `workspace`: device memory of gdr_tree_workspace_bytes(...) bytes (same
 * flags), 256-byte aligned, untouched until the stream has passed the call.
 * Also enqueues one host-to-device copy of the parents (pageable: the call
 * returns once they have been taken).  Errors: GDR_ERR_UNSUPPORTED for
 * T > 512, GDR_ERR_SHAPE for a parent outside [-1, t-1], the rest as
 * gdr_forward_ex.  B == 0 or T == 0 does nothing.
 */
GDR_API size_t gdr_tree_workspace_bytes(int B, int T, int HK, int HV, int dk, int dv,
                                        int qkv_dtype, unsigned flags);
GDR_API gdr_status gdr_forward_tree(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *h0, void *out,
                                    const int *parent, int B, int T, int HK, int HV, int dk,
                                    int dv, void *stream, int qkv_dtype, void *workspace,
                                    size_t workspace_bytes, unsigned flags);

/*
 * Passage: none in the pages (error reporting of the bounded waits).
 * Waits for `stream`, then reads and clears the library's device error word
 * on the current device.  Returns GDR_ERR_TIMEOUT if a kernel gave up on a
 * bounded wait since the last check, GDR_ERR_CUDA if the stream reported an
 * error, else GDR_OK.
 */
GDR_API gdr_status gdr_device_check(void *stream);

/*
 * Passage: none in the pages (measurement support).
 * Launch tracing.  While enabled (process-wide), every kernel launch made by
 * this library is bracketed by two CUDA events recorded on the launching
 * stream.  gdr_trace_read waits for the recorded events, writes per kernel
 * kind its name, launch count and summed event-to-event milliseconds into
 * the caller's arrays (each of max_kernels entries; any may be NULL),
 * forgets the records, and returns the number of kernel kinds written, or
 * -1 if a CUDA event query failed.  Tracing adds two event records per launch.
 */
GDR_API gdr_status gdr_trace_enable(int on);
GDR_API int gdr_trace_read(int max_kernels, const char **names, int *launches, double *total_ms);

/* Human-readable name of a gdr_status value (static string, never NULL).
 * Passage: none in the pages. */
GDR_API const char *gdr_status_string(int status);

/* cudaError_t code of the last CUDA failure seen by this thread (0 if none).
 * Passage: none in the pages. */
GDR_API int gdr_last_cuda_error(void);

/* Library version string, e.g. "0.1.0" (static string).  Passage: none in the pages. */
GDR_API const char *gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
