/*
 * palimpsa.h — C ABI of the GB300 (sm_103a) Palimpsa dual-state recurrence.
 *
 * The operation is the metaplastic linear attention of Bonnet, Lohoff,
 * Finkbeiner, Shiqerukaj and Neftci, "Learning to Remember, Learn, and Forget
 * in Attention-Based Models" (ICML 2026). Per head it keeps a memory mean
 * mu and an elementwise precision ("importance") I, both d_v x d_k, and for
 * every token t:
 *
 *   alpha_t = exp(-A * d_t)                                   (slide 5; paper Sec. 2.2)
 *   I_t     = alpha_t I_{t-1} + (1 - alpha_t) I_prior + beta_t (x) k_t^2
 *   mu_t    = alpha_t (I_{t-1} / I_t) (.) mu_{t-1}
 *             + (1 / I_t) (.) [(beta_t (.) v_t) (x) k_t]       (slide 7; paper Eq. 5)
 *   y_t     = mu_t q_t                                         (slide 4; paper Eq. 2)
 *
 * Squares, divisions and (.) are elementwise; (x) is an outer product with the
 * value index i as the row and the key index j as the column. The read y_t
 * uses the state after token t's write. The chunked entry point evaluates the
 * same recurrence through the natural parameters M = I (.) mu and I (slide 9;
 * paper App. A.12); the step entry point is the recurrent inference update of
 * one token (slide 22; paper App. A.13, Fig. 7).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: every array argument is a DEVICE pointer owned by the caller;
 *   nothing is copied, retained or freed. All arrays are dense row-major.
 *   The library's own working memory is described under "Scratch memory"
 *   near the end of this header.
 * - Alignment: every array pointer must be 16-byte aligned, except d_t, A and
 *   I_prior (4-byte aligned). Misaligned pointers give PALIMPSA_ERR_ALIGN.
 * - Sizes: 1 <= B, H; d_k in {64, 128}; d_v a multiple of 8 in [8, 256].
 * - Input dtype: q, k, v, beta are PALIMPSA_F32 (float) or PALIMPSA_BF16
 *   (__nv_bfloat16, upcast exactly to fp32). d_t, A, I_prior, the state and
 *   y are always fp32. All arithmetic is fp32.
 * - Streams: work is enqueued on `cuda_stream` (a cudaStream_t, NULL = the
 *   legacy default stream) on the CURRENT device; the call returns without
 *   synchronising. Argument checks run on the host before anything is
 *   enqueued: when a call returns an error nothing was launched and no output
 *   was written.
 * - Domain: A > 0, I_prior > 0, d_t >= 0, beta >= 0 and I0 > 0 (all finite)
 *   are preconditions. They are tested on the device: by the forward and step
 *   kernels as they read the inputs, and, for palimpsa_backward (and its
 *   checkpointed and packed forms), palimpsa_segment_summary and
 *   palimpsa_state_combine, by a short separate pass over the inputs enqueued
 *   before their kernels. A violation
 *   leaves that call's outputs unspecified and latches PALIMPSA_ERR_DOMAIN into
 *   the device status word (palimpsa_get_device_status).
 * - Errors are returned as status codes; nothing aborts and no C++ exception
 *   crosses this interface. A CUDA launch failure returns PALIMPSA_ERR_CUDA.
 * - Thread safety: calls may be made from several host threads; the debug
 *   setters below are process-wide.
 */
#ifndef PALIMPSA_H
#define PALIMPSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PALIMPSA_ABI_VERSION 1

typedef enum {
  PALIMPSA_F32 = 0,  /* float                                 */
  PALIMPSA_BF16 = 1  /* bfloat16 (1-8-7), upcast exactly to fp32 */
} palimpsa_dtype;

typedef enum {
  PALIMPSA_OK = 0,
  PALIMPSA_ERR_NULL = 1,        /* a required pointer is NULL                         */
  PALIMPSA_ERR_SHAPE = 2,       /* a size is out of range or overflows                */
  PALIMPSA_ERR_ALIGN = 3,       /* a pointer is not aligned as required               */
  PALIMPSA_ERR_DTYPE = 4,       /* unknown palimpsa_dtype                             */
  PALIMPSA_ERR_DOMAIN = 5,      /* (device status) an input broke a precondition      */
  PALIMPSA_ERR_UNSUPPORTED = 6, /* d_k, d_v or chunk not supported by this build      */
  PALIMPSA_ERR_CUDA = 7,        /* a CUDA runtime call failed                         */
  PALIMPSA_ERR_TIMEOUT = 8,     /* (device status) a bounded device wait gave up      */
  PALIMPSA_ERR_SCRATCH_LIMIT = 9 /* palimpsa_forward_chunked_noalloc: its fixed scratch
                                    buffer is too small for this call                 */
} palimpsa_status;

/*
 * palimpsa_forward_chunked — the recurrence over T tokens for B x H heads.
 *
 * Defined by slide 7 / paper Eq. (5) (state update), slide 4 / Eq. (2)
 * (readout) and slide 9 / App. A.12 (chunked scan of the natural parameters:
 * chunks of `chunk` tokens are staged on chip, the state is carried from one
 * chunk to the next). The result does not depend on `chunk`.
 *
 * When B*H heads are too few to fill the GPU, the sequence is cut into
 * segments whose summaries are scanned first (the affine carry of slide 9);
 * that path takes temporary device memory (2 * d_v * d_k + 1 floats per head
 * and segment boundary, plus 2 * d_v * d_k floats per head for a copy of the
 * initial state, so that mu_T / I_T may alias mu0 / I0 even when time is split)
 * in stream order on `cuda_stream`, from a memory pool
 * the library creates per device and that keeps what it has reserved (at most
 * the largest scratch one call needed) until the process exits. An allocation
 * failure returns PALIMPSA_ERR_CUDA. Results match the unsplit scan up to
 * fp32 rounding.
 *
 *   q, k     [B, H, T, d_k]  in_dtype
 *   v, beta  [B, H, T, d_v]  in_dtype, beta >= 0 (per value channel)
 *   d_t      [B, H, T]       fp32, >= 0
 *   A        [H]             fp32, > 0   (alpha = exp(-A d_t))
 *   I_prior  [H]             fp32, > 0   (prior precision, one per head)
 *   mu0, I0  [B, H, d_v, d_k] fp32 initial state, or NULL: mu0 = NULL means
 *            mu0 = 0; I0 = NULL means I0 = I_prior. I0 > 0.
 *   y        [B, H, T, d_v]  fp32 output, y[b,h,t,i] = sum_j mu_t[i,j] q_t[j]
 *   mu_T, I_T [B, H, d_v, d_k] fp32 final state. mu_T may be the same pointer
 *            as mu0 and I_T the same as I0 (in-place update); any other
 *            overlap between inputs and outputs is undefined.
 *   T >= 0. T = 0 copies the initial state to (mu_T, I_T); q, k, v, beta,
 *            d_t and y are then not read and may be NULL.
 *   chunk    0 (library default) or one of {16, 32, 64, 128} tokens. The
 *            result does not depend on it: it only sets the staging
 *            granularity, and the kernels stage at most 32 tokens at a
 *            time, so 64 and 128 are staged as 32-token chunks.
 */
palimpsa_status palimpsa_forward_chunked(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    float* y, float* mu_T, float* I_T,
    int B, int H, int T, int d_k, int d_v, int chunk,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_forward_plan — the launch plan palimpsa_forward_chunked (and the
 * fused, varlen and no-allocation variants) would use for these sizes on the
 * current device, computed by the same planner; nothing is launched or
 * allocated. Outputs (host pointers, all required):
 *   segments      time segments per sequence (1 = no time split)
 *   segment_len   tokens per segment (a multiple of the staging chunk)
 *   launches      kernel launches of one forward call: 1, or 3 with a time
 *                 split (summaries, carry, recurrence)
 *   scratch_bytes temporary device memory the call takes from the pool
 * For a packed batch pass N as B and max_seqlen as T. Honours
 * palimpsa_set_forward_segments. Errors as for palimpsa_forward_chunked;
 * PALIMPSA_ERR_CUDA when the device cannot be queried.
 */
palimpsa_status palimpsa_forward_plan(
    int B, int H, int T, int d_k, int d_v, int chunk, palimpsa_dtype in_dtype,
    int* segments, int* segment_len, int* launches, size_t* scratch_bytes);

/*
 * palimpsa_forward_chunked_noalloc — palimpsa_forward_chunked for callers that
 * must not allocate device memory. (The paper has no counterpart: this is a
 * deployment variant of the same computation.)
 *
 * Who needs it: code that runs where a CUDA allocation is not allowed or not
 * safe — a serving process that reserves all device memory at start-up and
 * forbids allocations while requests are in flight (an allocation there can
 * fail with out-of-memory or stall behind a device-wide synchronisation), a
 * plugin inside a host framework that owns the device heap and does not let
 * guests call the CUDA allocator, or a latency-critical loop that cannot pay
 * for an allocator call. palimpsa_forward_chunked takes its time-split
 * scratch from the stream-ordered allocator; this entry point instead uses a
 * fixed 16 MiB array compiled into the library (every GPU that loads the
 * library holds it until the process exits). It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Arguments, layouts, results and errors are those of
 * palimpsa_forward_chunked, plus one error: when the launch plan needs more
 * than 16 MiB of scratch it returns PALIMPSA_ERR_SCRATCH_LIMIT and launches
 * nothing. The plan needs about 8 * d_v * d_k bytes per head and segment
 * (64 KiB at d_v = 64, d_k = 128, so about 255 head-segments fit; the exact
 * figure is the scratch_bytes of palimpsa_forward_plan);
 * palimpsa_set_forward_segments(1) makes any call fit (one segment needs no
 * scratch), smaller segment counts make larger calls fit.
 *
 * Sharing: all calls on a device use the same array, which keeps the last
 * call's contents; nothing in it has to start at zero, because every scratch
 * element a call reads was written earlier in that same call. Calls that
 * overlap on the GPU (issued on different streams, or from several threads
 * without ordering) race on the array and corrupt each other's results:
 * order them on one stream.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 */
palimpsa_status palimpsa_forward_chunked_noalloc(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    float* y, float* mu_T, float* I_T,
    int B, int H, int T, int d_k, int d_v, int chunk,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_forward_varlen — palimpsa_forward_chunked over a packed batch of N
 * independent sequences of different lengths (each with its own initial and
 * final state), without padding. Each sequence runs the recurrence from its
 * own initial state (slide 7 / Eq. (5), carried along the sequence as in
 * slide 9), exactly as if it were the only one.
 *
 * Layout: the dense layout with B = 1 and the sequences concatenated along T.
 *   q, k      [H, total_T, d_k] in_dtype
 *   v, beta   [H, total_T, d_v] in_dtype, beta >= 0
 *   d_t       [H, total_T]      fp32, >= 0
 *   y         [H, total_T, d_v] fp32; rows of tokens outside every sequence
 *             are not written
 *   cu_seqlens [N + 1] int32 in DEVICE memory: sequence n is tokens
 *             [cu_seqlens[n], cu_seqlens[n+1]) of every head; the offsets must
 *             be non-decreasing, within [0, total_T], and no sequence longer
 *             than max_seqlen (empty sequences are allowed and pass their state
 *             through)
 *   max_seqlen the longest sequence's length (host value, used to plan the
 *             launch; a tighter value is faster, a smaller one is an error)
 *   mu0, I0   [N, H, d_v, d_k] fp32 or NULL (defaults as for the forward)
 *   mu_T, I_T [N, H, d_v, d_k] fp32
 *   A, I_prior, d_k, d_v, chunk, in_dtype, cuda_stream as for the forward.
 *
 * The offsets live on the device, so the host cannot check them: every CTA
 * checks its own sequence's offsets before it reads anything, and a sequence
 * whose offsets break the rules above is skipped (its outputs are left as
 * they were) and latches PALIMPSA_ERR_DOMAIN in the device status. Long
 * sequences are cut into segments as in palimpsa_forward_chunked, planned
 * from max_seqlen, with scratch as for the forward (per sequence and head).
 */
palimpsa_status palimpsa_forward_varlen(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    float* y, float* mu_T, float* I_T,
    const int* cu_seqlens, int N, int H, int total_T, int max_seqlen,
    int d_k, int d_v, int chunk, palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * Time-sharded sequences (one exchange). Both natural-parameter recurrences are
 * affine in the state with the shared scalar decay alpha (slide 9 / App.
 * A.12), so a stretch of tokens acts on the state as
 *     (M, Ibar) -> Gamma (M, Ibar) + (dM, dIbar),   M = I (.) mu, Ibar = I - I_prior,
 * with Gamma the product of its alphas and (dM, dIbar) the state it produces
 * from zero. When the T tokens of each sequence are split into R consecutive
 * shards (one per GPU), shard r: (1) computes its summary with
 * palimpsa_segment_summary, (2) gathers the summaries of all shards (the one
 * exchange), (3) folds the summaries of shards 0 .. r-1 into the initial state
 * with palimpsa_state_combine, and (4) runs palimpsa_forward_chunked on its
 * own tokens from that state. The result equals the unsharded forward up to
 * fp32 rounding.
 *
 * palimpsa_segment_summary — the summary of each head's T tokens.
 *   q, k, v, beta, d_t, A, I_prior, B, H, T, d_k, d_v, chunk, in_dtype as for
 *   palimpsa_forward_chunked (T = 0 gives Gamma = 1 and a zero summary).
 *   summary  [B, H, 2, d_v, d_k] fp32 out: [..., 0, :, :] = dM, [..., 1, :, :] = dIbar
 *   gamma    [B, H] fp32 out
 * Long ranges are cut into segments as in the forward (scratch from the same
 * pool: 2 * d_v * d_k + 1 floats per head and segment, when split).
 */
palimpsa_status palimpsa_segment_summary(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    float* summary, float* gamma,
    int B, int H, int T, int d_k, int d_v, int chunk,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_state_combine — the state after R stretches, in order, from an
 * initial state:
 *   summaries [R, B, H, 2, d_v, d_k] fp32 (as written by palimpsa_segment_summary)
 *   gammas    [R, B, H] fp32
 *   I_prior   [H] fp32; mu0, I0 [B, H, d_v, d_k] fp32 or NULL (defaults as for
 *             the forward)
 *   mu_out, I_out [B, H, d_v, d_k] fp32: the state as (mu, I), ready to pass as
 *             mu0 / I0 to palimpsa_forward_chunked. They may alias mu0 / I0.
 * R = 0 copies the initial state. Summaries and gammas may be NULL when R = 0.
 */
palimpsa_status palimpsa_state_combine(
    const float* summaries, const float* gammas, int R,
    const float* I_prior, const float* mu0, const float* I0,
    float* mu_out, float* I_out,
    int B, int H, int d_k, int d_v, void* cuda_stream);

/*
 * palimpsa_forward_varlen_fused — palimpsa_forward_varlen with the prologue
 * of palimpsa_forward_fused: raw q, k, v (or v*), beta_raw, d_raw in the packed
 * layout, b_scale [H] or NULL, flags (palimpsa_fuse_flags). Everything else as
 * for palimpsa_forward_varlen.
 */
palimpsa_status palimpsa_forward_varlen_fused(
    const void* q, const void* k, const void* v, const void* beta_raw,
    const float* d_raw, const float* A, const float* I_prior,
    const float* b_scale, const float* mu0, const float* I0,
    float* y, float* mu_T, float* I_T,
    const int* cu_seqlens, int N, int H, int total_T, int max_seqlen,
    int d_k, int d_v, int chunk, unsigned int flags,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_step — one recurrent (decode) token for B x H heads, in place.
 *
 * The recurrent inference update of slide 22 / paper App. A.13 (Fig. 7):
 * Eq. (5) and the readout for a single token, the state read from and written
 * back to HBM.
 *
 *   q, k     [B, H, d_k]     in_dtype
 *   v, beta  [B, H, d_v]     in_dtype, beta >= 0
 *   d_t      [B, H]          fp32, >= 0
 *   A        [H]             fp32, > 0
 *   I_prior  [H]             fp32, > 0
 *   mu, I    [B, H, d_v, d_k] fp32 state, updated in place (I > 0)
 *   y        [B, H, d_v]     fp32 output (must not overlap the state)
 *
 * Launch: the step goes out with programmatic dependent launch. It may start
 * while the kernel before it in the stream finishes, and waits for that kernel
 * before its first read. It lets the next kernel in the stream start early, so
 * a kernel launched after it with the programmatic-serialization attribute
 * must wait (cudaGridDependencySynchronize / griddepcontrol.wait) before it
 * reads y or the state; kernels launched normally, copies and events are
 * ordered as usual.
 */
palimpsa_status palimpsa_step(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    float* mu, float* I, float* y,
    int B, int H, int d_k, int d_v,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_step_sequence — S decode tokens in order, as S palimpsa_step
 * launches enqueued by one call (arguments validated once). Token s reads
 * q[s], k[s], v[s], beta[s], d_t[s] and writes y[s]; the state (mu, I) is
 * updated in place after every token, exactly as S palimpsa_step calls would.
 *
 *   q, k     [S, B, H, d_k]  in_dtype
 *   v, beta  [S, B, H, d_v]  in_dtype
 *   d_t      [S, B, H]       fp32 (each token's slice must stay 4-byte aligned)
 *   y        [S, B, H, d_v]  fp32
 *   other arguments as for palimpsa_step; S >= 0.
 */
palimpsa_status palimpsa_step_sequence(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    float* mu, float* I, float* y,
    int S, int B, int H, int d_k, int d_v,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * Options of the fused entry points (bit flags; combine with |).
 *   PALIMPSA_FUSE_QK_NORM  divide q_t and k_t by their L2 norm over d_k
 *                          (x / max(||x||_2, 1e-12)), as the Palimpsa-D block
 *                          does (slide 10);
 *   PALIMPSA_FUSE_V_STAR   v holds v* = beta (.) v, the kernel input of slide 11:
 *                          the content write is v*_i k_j, and beta (activated)
 *                          enters only the precision.
 */
typedef enum {
  PALIMPSA_FUSE_QK_NORM = 1,
  PALIMPSA_FUSE_V_STAR = 2
} palimpsa_fuse_flags;

/*
 * palimpsa_forward_fused — palimpsa_forward_chunked with the layer's prologue
 * applied in the kernels as each chunk is staged, so that raw projections go
 * in without extra passes over HBM:
 *
 *   d_t  = softplus(d_raw)                        (so d_t >= 0, slide 5)
 *   beta = b_scale[h] * sigmoid(beta_raw)         (so beta >= 0; per-head
 *                                                  b_scale, slide 11)
 *   q, k L2-normalised per token                  (PALIMPSA_FUSE_QK_NORM)
 *   write v* as given instead of beta (.) v       (PALIMPSA_FUSE_V_STAR)
 *
 * The pages do not print the two activations; they are the ones that map any
 * real input into the recurrence's domain, as in the workload recipes.
 *
 *   q, k      [B, H, T, d_k] in_dtype (raw)
 *   v         [B, H, T, d_v] in_dtype: v, or v* with PALIMPSA_FUSE_V_STAR
 *   beta_raw  [B, H, T, d_v] in_dtype (pre-activation)
 *   d_raw     [B, H, T]      fp32 (pre-activation)
 *   b_scale   [H] fp32 >= 0, or NULL for 1
 *   flags     palimpsa_fuse_flags; unknown bits give PALIMPSA_ERR_UNSUPPORTED
 *   all other arguments, the time split and the errors are those of
 *   palimpsa_forward_chunked. A negative or non-finite b_scale, or a
 *   non-finite raw gate, latches PALIMPSA_ERR_DOMAIN in the device status.
 */
palimpsa_status palimpsa_forward_fused(
    const void* q, const void* k, const void* v, const void* beta_raw,
    const float* d_raw, const float* A, const float* I_prior,
    const float* b_scale, const float* mu0, const float* I0,
    float* y, float* mu_T, float* I_T,
    int B, int H, int T, int d_k, int d_v, int chunk, unsigned int flags,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_step_fused — palimpsa_step with the same prologue on the token's
 * raw inputs: q, k [B,H,d_k], v and beta_raw [B,H,d_v] in in_dtype, d_raw [B,H]
 * fp32, b_scale [H] or NULL, flags as for palimpsa_forward_fused. State, y and
 * errors as for palimpsa_step.
 */
palimpsa_status palimpsa_step_fused(
    const void* q, const void* k, const void* v, const void* beta_raw,
    const float* d_raw, const float* A, const float* I_prior,
    const float* b_scale, float* mu, float* I, float* y,
    int B, int H, int d_k, int d_v, unsigned int flags,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_step_sequence_fused — palimpsa_step_fused for S tokens in order,
 * enqueued by one call as palimpsa_step_sequence does for palimpsa_step: the
 * inputs carry a leading token index (q, k [S, B, H, d_k]; v, beta_raw
 * [S, B, H, d_v]; d_raw [S, B, H]) and y is [S, B, H, d_v]. Arguments are
 * validated once; other arguments and errors as for palimpsa_step_fused.
 */
palimpsa_status palimpsa_step_sequence_fused(
    const void* q, const void* k, const void* v, const void* beta_raw,
    const float* d_raw, const float* A, const float* I_prior,
    const float* b_scale, float* mu, float* I, float* y,
    int S, int B, int H, int d_k, int d_v, unsigned int flags,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_forward_without_meta — the "without Meta" comparator: the same
 * recurrence with the importance frozen at its prior (I_t = I_prior), i.e. the
 * Mamba2 limit of Eq. (5) (slide 11; slide 10 names Mamba2 as Palimpsa-M's
 * "without Meta" model):
 *
 *   mu_t = alpha_t mu_{t-1} + ((beta_t (.) v_t) / I_prior) (x) k_t,   y_t = mu_t q_t.
 *
 * It exists to measure what metaplasticity costs on this GPU (slide 22 compares
 * Palimpsa's kernel with a Simple GLA kernel of this scalar-decay form).
 * Arguments and conventions are those of palimpsa_forward_chunked without the
 * precision state: mu0 [B,H,d_v,d_k] or NULL (= 0), y [B,H,T,d_v],
 * mu_T [B,H,d_v,d_k] (may alias mu0). Few long sequences are cut into time
 * segments exactly as palimpsa_forward_chunked plans them (its state
 * m = I_prior mu follows Palimpsa's M recurrence, so the same summaries and
 * carry apply), with the same scratch from the library's pool.
 */
palimpsa_status palimpsa_forward_without_meta(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, float* y, float* mu_T,
    int B, int H, int T, int d_k, int d_v, int chunk,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * palimpsa_backward — gradients of a scalar loss L through
 * palimpsa_forward_chunked (the same recurrence: slide 7 / Eq. (5), slide 4 /
 * Eq. (2); the pages train the projections and gates that feed it by
 * backpropagating through it, slide 4 and slide 9).
 *
 *   inputs   q, k, v, beta, d_t, A, I_prior, mu0, I0 exactly as given to the
 *            forward (mu0 / I0 may be NULL for the defaults);
 *            dy [B,H,T,d_v] fp32 = dL/dy; dmu_T, dI_T [B,H,d_v,d_k] fp32 =
 *            dL/dmu_T, dL/dI_T, or NULL for zero.
 *   outputs  (fp32, whatever in_dtype is) dq, dk [B,H,T,d_k]; dv, dbeta
 *            [B,H,T,d_v]; dd_t [B,H,T]; dA, dI_prior [H] (summed over the
 *            batch); dmu0, dI0 [B,H,d_v,d_k] or NULL when not wanted. When I0
 *            is NULL the initial precision is I_prior itself and its gradient
 *            is included in dI_prior.
 *
 * The forward states are recomputed, never stored by the forward: one sweep
 * keeps a checkpoint every 32 tokens in stream-ordered scratch from the
 * library's pool (B * H * ceil(T / 32) * 8 * d_v * d_k bytes). All states used
 * come from forward-direction steps. dq, dk, dd_t, dA and dI_prior are
 * accumulated with fp32 atomics (the library zeroes them first), so their last
 * bits may differ between runs; everything else is deterministic.
 */
palimpsa_status palimpsa_backward(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    const float* dy, const float* dmu_T, const float* dI_T,
    float* dq, float* dk, float* dv, float* dbeta, float* dd_t,
    float* dA, float* dI_prior, float* dmu0, float* dI0,
    int B, int H, int T, int d_k, int d_v,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * Training pair. palimpsa_forward_checkpointed is palimpsa_forward_chunked that
 * also writes the state of every head before tokens 0, 32, 64, ... into
 * `ckpt`. palimpsa_backward_checkpointed is palimpsa_backward reading those
 * states instead of recomputing them with a forward sweep of its own, which
 * saves about a sixth of the backward's work and all of its scratch memory.
 *
 *   ckpt  fp32 [B, H, ceil(T / 32), d_v, 2, d_k], palimpsa_checkpoint_bytes()
 *         bytes, 16-byte aligned: for checkpoint c and value row i, the natural
 *         parameter M_i = I_i (.) mu_i over the d_k keys, then I_i.
 *
 * The forward writes ckpt in addition to its usual outputs (other arguments
 * and errors as for palimpsa_forward_chunked). The backward's other arguments
 * and errors are those of palimpsa_backward; its ckpt must come from a forward
 * call on the same inputs (q, k, v, beta, d_t, A, I_prior, mu0, I0), which the
 * library cannot check.
 */
size_t palimpsa_checkpoint_bytes(int B, int H, int T, int d_k, int d_v);

palimpsa_status palimpsa_forward_checkpointed(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    float* y, float* mu_T, float* I_T, float* ckpt,
    int B, int H, int T, int d_k, int d_v, int chunk,
    palimpsa_dtype in_dtype, void* cuda_stream);

palimpsa_status palimpsa_backward_checkpointed(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    const float* dy, const float* dmu_T, const float* dI_T,
    float* dq, float* dk, float* dv, float* dbeta, float* dd_t,
    float* dA, float* dI_prior, float* dmu0, float* dI0,
    const float* ckpt,
    int B, int H, int T, int d_k, int d_v,
    palimpsa_dtype in_dtype, void* cuda_stream);

/*
 * Packed training pair: palimpsa_forward_varlen_checkpointed and
 * palimpsa_backward_varlen are the training pair above over the packed batch of
 * palimpsa_forward_varlen (N sequences of different lengths, one state each;
 * the gradient of each sequence is that of the recurrence run on it alone, and
 * dA, dI_prior sum over all sequences).
 *
 *   per-token arrays (q, k, v, beta, d_t, dy and the gradients dq, dk, dv,
 *             dbeta, dd_t) in the layout of palimpsa_forward_varlen:
 *             [H, total_T, ...]; gradient rows of tokens outside every
 *             sequence are zero (dq, dk, dd_t) or not written (dv, dbeta)
 *   per-sequence states mu0, I0, dmu_T, dI_T, dmu0, dI0: [N, H, d_v, d_k]
 *   cu_seqlens, N, H, total_T, max_seqlen as for palimpsa_forward_varlen
 *   ckpt      fp32 [H, total_T / 32 + N, d_v, 2, d_k] (integer division),
 *             palimpsa_checkpoint_bytes_varlen(N, H, total_T, d_k, d_v)
 *             bytes, 16-byte aligned; memory grows with the tokens, not with
 *             N x max_seqlen. Head h of sequence n (which starts at token s0)
 *             keeps its state before its token 32 c in slot
 *             s0 / 32 + n + c of head h, as (M_i, I_i) per value row i like
 *             the dense checkpoints; sequences never share a slot, and slots
 *             that no sequence owns are not written. For the backward, ckpt
 *             may be NULL: it then recomputes the states with a forward sweep
 *             into scratch of that size from the library's pool.
 *
 * Offsets that break the rules of palimpsa_forward_varlen are reported as
 * there: the CTAs of that sequence touch nothing else and latch
 * PALIMPSA_ERR_DOMAIN (its dmu0 / dI0 are then not written). Other errors as
 * for palimpsa_backward.
 */
size_t palimpsa_checkpoint_bytes_varlen(int N, int H, int total_T, int d_k, int d_v);

palimpsa_status palimpsa_forward_varlen_checkpointed(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    float* y, float* mu_T, float* I_T, float* ckpt,
    const int* cu_seqlens, int N, int H, int total_T, int max_seqlen,
    int d_k, int d_v, int chunk, palimpsa_dtype in_dtype, void* cuda_stream);

palimpsa_status palimpsa_backward_varlen(
    const void* q, const void* k, const void* v, const void* beta,
    const float* d_t, const float* A, const float* I_prior,
    const float* mu0, const float* I0,
    const float* dy, const float* dmu_T, const float* dI_T,
    float* dq, float* dk, float* dv, float* dbeta, float* dd_t,
    float* dA, float* dI_prior, float* dmu0, float* dI0,
    const float* ckpt,
    const int* cu_seqlens, int N, int H, int total_T, int max_seqlen,
    int d_k, int d_v, palimpsa_dtype in_dtype, void* cuda_stream);

/* Static English text for a status code (never NULL). */
const char* palimpsa_status_string(palimpsa_status s);

/*
 * palimpsa_get_device_status — synchronises `cuda_stream`, then reads and
 * clears the current device's status word, which kernels latch when a
 * bounded wait gives up (PALIMPSA_ERR_TIMEOUT) or an input breaks a
 * precondition (PALIMPSA_ERR_DOMAIN). Returns PALIMPSA_OK when nothing was
 * latched, the latched code (TIMEOUT before DOMAIN) otherwise, or
 * PALIMPSA_ERR_CUDA when the synchronisation itself fails.
 */
palimpsa_status palimpsa_get_device_status(void* cuda_stream);

/* PALIMPSA_ABI_VERSION of the loaded library. */
int palimpsa_abi_version(void);

/*
 * Failure-detection controls (process-wide; for tests).
 * palimpsa_set_wait_timeout_ns sets how long a kernel waits for a staged copy
 * before it records PALIMPSA_ERR_TIMEOUT and returns (default 2e9 ns).
 * palimpsa_debug_withhold_first_copy(1) makes the next chunked launches skip
 * issuing their first staged copy, so that their wait can never be satisfied
 * and must run out; 0 restores normal operation. Neither changes results
 * otherwise.
 */
void palimpsa_set_wait_timeout_ns(uint64_t ns);
void palimpsa_debug_withhold_first_copy(int on);

/*
 * palimpsa_set_forward_segments — process-wide override of the number of
 * time segments palimpsa_forward_chunked cuts each sequence into (0 = the
 * library chooses from the problem size and the GPU; S > 0 = S segments, as
 * far as whole chunks allow). For tests and tuning; results change only by
 * fp32 rounding.
 */
void palimpsa_set_forward_segments(int segments);

/*
 * palimpsa_set_step_l2_keep_bytes — process-wide tuning of the decode step
 * (palimpsa_step, palimpsa_step_sequence, palimpsa_step_fused). The step
 * streams the whole state through HBM. Consecutive launches walk it in
 * opposite orders, and each launch stores the last `bytes` of its walk with
 * an evict-last L2 policy instead of streaming them, so the next launch starts
 * on rows that are still in L2. 0 turns this off: every launch then walks in
 * the same order and streams everything. Default 96 MiB. Results are the same
 * bits either way; only the DRAM traffic changes.
 */
void palimpsa_set_step_l2_keep_bytes(long long bytes);

/*
 * Scratch memory. The time-split forward and the backward need device scratch
 * for the length of one call (the segment states of the time split, the
 * backward's 32-token state checkpoints). The library takes it in stream order
 * from a memory pool of its own, one per device, created on the first call
 * that needs scratch; it is freed in stream order when the call's work ends.
 * Freed pages stay mapped for the next call, up to a retention bound, so that
 * repeated calls do not pay to map fresh pages; at each synchronisation of the
 * stream, an event or the device, the pool gives back to the driver whatever
 * it holds above that bound. No other memory is kept between calls.
 *
 * palimpsa_set_scratch_retention — sets the retention bound, in bytes, of
 *   every device's pool, existing and future (process-wide). Default 512 MiB:
 *   well above the forward's time-split scratch at the layer sizes this
 *   library is tuned on (64 to 132 MiB; the split is planned to fill a few
 *   waves of CTAs, each of which carries 64 KiB of state at d_v = 64,
 *   d_k = 128), so the forward keeps its pages, while a large backward's
 *   scratch above the bound is given back. 0 keeps nothing mapped between
 *   synchronisations. Returns PALIMPSA_ERR_CUDA if a pool refuses the bound.
 * palimpsa_release_scratch — gives all freed scratch of the CURRENT device's
 *   pool back to the driver now. It first synchronises the device (so that no
 *   work in flight still uses the scratch), then trims the pool to zero. OK
 *   when the library has no pool on this device; PALIMPSA_ERR_CUDA when the
 *   synchronisation or the trim fails.
 * palimpsa_scratch_reserved_bytes — the bytes the CURRENT device's pool holds
 *   mapped (in use or kept), 0 without a pool. PALIMPSA_ERR_NULL for a NULL
 *   `bytes`.
 * These calls have no counterpart on the pages; they manage this library's
 * own working memory.
 */
palimpsa_status palimpsa_set_scratch_retention(unsigned long long bytes);
palimpsa_status palimpsa_release_scratch(void);
palimpsa_status palimpsa_scratch_reserved_bytes(size_t* bytes);

/*
 * palimpsa_probe_issue_rate — measures how many instructions of one kind an SM
 * of the current device completes per clock: the denominator of the roofline
 * the ALU-bound kernels are reported against. The chunked forward and the
 * backward spend one SFU reciprocal per element-token on the readout's M / I
 * (slide 9; paper App. A.12), so their bound is PALIMPSA_PROBE_RCP's rate x
 * SMs x clock. The probe runs one CTA per SM (32 warps, 8 independent chains
 * of the instruction per thread), times it with the SM cycle counter and
 * returns the median over SMs in *per_clk_per_sm. It is synchronous on
 * `cuda_stream` (about a millisecond) and allocates a few bytes of device
 * memory for the cycle counts.
 *   op  PALIMPSA_PROBE_RCP (rcp.approx.ftz.f32), PALIMPSA_PROBE_EX2
 *       (ex2.approx.ftz.f32), PALIMPSA_PROBE_FFMA (fma.rn.f32),
 *       PALIMPSA_PROBE_RSQ (rsqrt.approx.ftz.f32) or PALIMPSA_PROBE_LG2
 *       (lg2.approx.ftz.f32).
 * Errors: PALIMPSA_ERR_NULL, PALIMPSA_ERR_UNSUPPORTED (unknown op),
 * PALIMPSA_ERR_CUDA. This call has no counterpart on the pages.
 */
typedef enum {
  PALIMPSA_PROBE_RCP = 0,
  PALIMPSA_PROBE_EX2 = 1,
  PALIMPSA_PROBE_FFMA = 2,
  PALIMPSA_PROBE_RSQ = 3,
  PALIMPSA_PROBE_LG2 = 4
} palimpsa_probe_op;
palimpsa_status palimpsa_probe_issue_rate(int op, double* per_clk_per_sm, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* PALIMPSA_H */
