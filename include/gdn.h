/*
 * gdn.h -- C ABI of libgdn, the Gated-DeltaNet token mixer for GB300 (sm_103a).
 *
 * The operation is the SSM block of "qwen35moe -- Forward-Pass Design
 * (Pantheon port)". These calls cover its section "SSM block -- Gated-Delta-Net"
 * from the already-projected streams up to, but not including, the ssm_out
 * projection:
 *   causal conv1d (k=4, with conv_state) + SiLU over the 8192-channel q|k|v
 *   stream; split into q[16x128], k[16x128], v[32x128]; L2-normalise q and k
 *   per head; GQA repeat 16 -> 32 with V-head vh reading K-head vh % 16
 *   (watch-list item on the interleaved repeat); decay g = -exp(A_log) *
 *   softplus(alpha + dt_bias) and beta = sigmoid(beta) (section "Decay gate");
 *   the per-token delta-rule recurrence (a)-(d) with read-after-write and one
 *   1/sqrt(128) scale (section "Per-token recurrence"); and
 *   gated = RMSNorm(y, ssm_norm) * silu(z) (section "Output path").
 *
 * Fixed dimensions (section "Config (mini)"): 32 V-heads, 16 K-heads, head dim
 * 128 for keys and values, conv width 4, 8192 conv channels, d_inner 4096.
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is caller-owned DEVICE memory, dense, row-major, and
 *    16-byte aligned. The library never allocates, frees or keeps a pointer
 *    after a call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Every call only enqueues work on that stream and returns; no call
 *    synchronises, except gdn_device_error, which says so.
 *  - Activations (qkv, z, alpha, beta, conv_state) all use one dtype `act`;
 *    `out_dt` is the dtype of `out`. Parameters and the SSM state are fp32.
 *  - The SSM state of one (sequence, V-head) is the page's S[i][j] (i = key
 *    index, j = value index) stored TRANSPOSED: ssm_state[..][j][i], with the
 *    key index contiguous, 128 x 128 fp32 = 64 KiB.
 *  - conv_state[n] holds the last 3 raw (pre-conv) inputs of sequence n,
 *    oldest row first, [3][8192] in the activation dtype.
 *  - Invalid arguments return a status and enqueue nothing. Nothing throws,
 *    aborts or traps. GDN_ERR_CUDA means a launch was rejected by the runtime;
 *    gdn_last_error() then describes it.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 1

#define GDN_NUM_V_HEADS 32
#define GDN_NUM_K_HEADS 16
#define GDN_HEAD_DIM 128
#define GDN_CONV_K 4
#define GDN_CONV_CHANNELS 8192
#define GDN_D_INNER 4096
#define GDN_DECODE_MAX_T 8   /* tokens per sequence of gdn_decode_multi, at most */
#define GDN_HIDDEN 2048      /* n_embd: the model width (in_proj input, ssm_out output) */
#define GDN_IN_PROJ_ROWS 12352   /* stacked input-projection weight rows: 8192 + 4096 + 32 + 32 */
/* The full-attention layers (section "Full-attention block"): GQA with 16
 * query heads and 2 KV heads of head_dim 256; query head h reads KV head h / 8. */
#define GDN_ATTN_Q_HEADS 16
#define GDN_ATTN_KV_HEADS 2
#define GDN_ATTN_HEAD_DIM 256

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, bad enum     */
    GDN_ERR_UNSUPPORTED = 2,   /* well-formed request the library does not serve  */
    GDN_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required      */
    GDN_ERR_CUDA = 4,          /* the CUDA runtime rejected a launch              */
    GDN_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up              */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Per-layer parameters: device pointers to fp32 tensors, plus two epsilons.
 * Page tensor names in brackets. */
typedef struct {
    const float *conv_w;   /* [8192][4] (ssm_conv1d.weight); tap 3 multiplies the
                              current token, taps 0..2 the conv_state rows
                              oldest-first. The page lists no conv bias.       */
    const float *A_log;    /* [32]; the decay uses -exp(A_log) (ssm_a)          */
    const float *dt_bias;  /* [32] (ssm_dt.bias)                                */
    const float *norm_w;   /* [128] (ssm_norm.weight), shared by all V-heads and
                              applied as w, not 1 + w. NULL: the gated norm is
                              left out and `out` receives the mixer's raw
                              output y = scale * S^T q per head (z is not
                              read), for gdn_gated_out_proj to apply the norm
                              inside the output projection.                    */
    float norm_eps;        /* RMSNorm epsilon: y * (mean(y^2) + eps)^-1/2       */
    float l2_eps;          /* L2 epsilon: x * (sum(x^2) + eps)^-1/2             */
} gdn_params;

/*
 * gdn_conv_step -- the conv part alone, for one token of B sequences.
 * Section "Causal conv1d": qkv_out[b][c] = SiLU(sum_m conv_w[c][m] * win[m])
 * where win = (conv_state[b][0..2][c], qkv_in[b][c]); then conv_state[b]
 * shifts by one token (row 0 drops out, qkv_in[b] becomes row 2).
 *   conv_w      [8192][4] fp32
 *   qkv_in      [B][8192] act          qkv_out [B][8192] act (may not alias qkv_in)
 *   conv_state  [B][3][8192] act, updated in place
 * B == 0 is a no-op. Errors: GDN_ERR_INVALID_ARG.
 */
gdn_status gdn_conv_step(const float *conv_w, const void *qkv_in, void *qkv_out,
                         void *conv_state, int B, gdn_dtype act, void *stream);

/*
 * gdn_decode_step -- one token for each of B independent sequences, the whole
 * mixer fused: conv -> split -> L2 -> GQA -> gates -> recurrence -> gated norm.
 * Each (sequence, V-head) state is read once and written once.
 *   p           layer parameters
 *   qkv         [B][8192] act          z          [B][4096] act
 *   alpha, beta [B][32] act (raw logits; the gates are computed inside)
 *   conv_state  [B][3][8192] act, updated in place
 *   ssm_state   [B][32][128 j][128 i] fp32, updated in place
 *   out         [B][4096] out_dt, head-major (out[b][vh*128 + j])
 * 1 <= B <= 65535 (B == 0 is a no-op). Errors: GDN_ERR_INVALID_ARG, GDN_ERR_CUDA.
 */
gdn_status gdn_decode_step(const gdn_params *p, const void *qkv, const void *z,
                           const void *alpha, const void *beta, void *conv_state,
                           float *ssm_state, void *out, int B, gdn_dtype act,
                           gdn_dtype out_dt, void *stream);

/*
 * gdn_decode_multi -- T consecutive tokens (1 <= T <= GDN_DECODE_MAX_T) for each
 * of B independent sequences, for example a speculative step's draft tokens. It
 * is the same mixer as gdn_decode_step, applied to the T tokens in order: the
 * conv window is the conv_state followed by the T inputs, and the recurrence
 * (a)-(d) of section "Per-token recurrence" runs token after token with
 * read-after-write. The result equals T successive gdn_decode_step calls up to
 * rounding order. Each state is read once and written once for all T tokens.
 *   p           layer parameters
 *   qkv         [B][T][8192] act          z          [B][T][4096] act
 *   alpha, beta [B][T][32] act (raw logits)
 *   conv_state  [B][3][8192] act, updated in place (it ends with the last three
 *               raw inputs of the window)
 *   ssm_state   [B][32][128 j][128 i] fp32, updated in place
 *   out         [B][T][4096] out_dt
 * 1 <= B <= 65535 (B == 0 is a no-op). Errors: GDN_ERR_INVALID_ARG (also for T
 * out of range), GDN_ERR_CUDA. A bounded device wait that gives up is reported
 * afterwards by gdn_device_error.
 */
gdn_status gdn_decode_multi(const gdn_params *p, const void *qkv, const void *z,
                            const void *alpha, const void *beta, void *conv_state,
                            float *ssm_state, void *out, int B, int T, gdn_dtype act,
                            gdn_dtype out_dt, void *stream);

/*
 * gdn_prefill -- N packed sequences of total length T_total, each run through
 * the whole mixer token by token in order, with state carried in and out.
 *   cu_seqlens      DEVICE int32 [N+1]: cu[0] = 0, cu[n] <= cu[n+1], cu[N] =
 *                   T_total; sequence n owns rows [cu[n], cu[n+1]). Empty
 *                   sequences are allowed (their states pass through).
 *   qkv [T_total][8192], z [T_total][4096], alpha/beta [T_total][32]   act
 *   conv_state_in   [N][3][8192] act, or NULL for all-zero initial conv state
 *   conv_state_out  [N][3][8192] act, or NULL to skip; may alias conv_state_in
 *   ssm_state_in    [N][32][128][128] fp32 (transposed as above), or NULL = 0
 *   ssm_state_out   [N][32][128][128] fp32, or NULL to skip; may alias the input
 *   out             [T_total][4096] out_dt
 *   chunk_size      0 = library choice; 1 = exact per-token scan (fp32 math,
 *                   any act); 64 = chunked WY/UT form on tensor cores (act must
 *                   be GDN_BF16). The chunked form is an exact re-association
 *                   of the same recurrence; the two differ only by rounding.
 *                   Library choice: GDN_F32 -> 1, GDN_BF16 -> 64.
 *   workspace       DEVICE scratch, 256-byte aligned; contents need no
 *                   initialisation and are clobbered. Calls that share a
 *                   workspace must be ordered on one stream. Size:
 *                   - chunk_size 1: at least gdn_prefill_workspace_size(...).
 *                   - chunk_size 64: the packed tokens run in windows sized
 *                     to the workspace given, with the state carried from
 *                     window to window, so the scratch does not grow with the
 *                     prompt. gdn_prefill_workspace_size(...) is the size for
 *                     one window of up to 4096 tokens (the same for any
 *                     T_total >= 4096); any size down to
 *                     gdn_prefill_workspace_size(N, 64, act, 64) (one 64-token
 *                     window) is accepted, and a larger one gives longer
 *                     windows.
 * chunk_size 64 runs each window's prep, state chains and gated norm as one
 * cooperative kernel of one CTA per SM, which occupies the whole device while it
 * runs. Where such a grid cannot be resident (e.g. a share of the SMs), or with
 * GDN_PREFILL_SPLIT=1 in the environment when the library first runs a prefill,
 * the same work runs as separate kernels with the same results.
 * 0 <= N <= 65535, 0 <= T_total <= 2^24. cu_seqlens is read on the device only;
 * a cu_seqlens that breaks the rules above gives unspecified results for the
 * offending sequences but never touches memory outside the stated extents.
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE,
 * GDN_ERR_CUDA. A bounded device wait that gives up is reported afterwards by
 * gdn_device_error.
 */
gdn_status gdn_prefill(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                       const void *beta, const int32_t *cu_seqlens, int N, int T_total,
                       const void *conv_state_in, void *conv_state_out,
                       const float *ssm_state_in, float *ssm_state_out, void *out,
                       gdn_dtype act, gdn_dtype out_dt, int chunk_size, void *workspace,
                       size_t ws_bytes, void *stream);

/*
 * gdn_prefill_static -- gdn_prefill for callers that cannot allocate device
 * memory. It takes the same arguments minus the workspace. The paper has no
 * counterpart to this call: it exists only for how the library is used.
 *
 * Who needs it: code that runs where allocation is not allowed or not
 * possible. Examples are a plugin inside a framework that owns every device
 * allocation and hands it only input and output buffers, or a serving loop
 * that forbids allocation after start-up. Such a caller has no workspace to
 * pass.
 *
 * Scratch: a file-scope device array of GDN_STATIC_SCRATCH_BYTES (64 MiB) in
 * libgdn. Every GPU that loads the library holds it until the process exits.
 * The chunked form (bf16) runs in windows that fit the array, about 1,600
 * tokens each for one sequence, so a prompt of any length fits; only a call
 * with so many sequences that one 64-token window does not fit is refused.
 * The exact scan needs room for all of its tokens: up to about 1,300 tokens
 * per call. A call that does not fit returns GDN_ERR_WORKSPACE without
 * launching anything, after the same argument checks as gdn_prefill.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it for the life
 * of the process, so the device's primary context must not be reset
 * (cudaDeviceReset) afterwards. Make that first call before any stream
 * capture on the device.
 *
 * Sharing: every call on a device uses the same scratch, and the scratch keeps
 * the previous call's contents (the kernels need none of it cleared). Calls
 * that overlap on the GPU (different streams, or another host thread) race on
 * it. Order them on one stream.
 *
 * Allocation: none. No cudaMalloc, no cudaFree, no library allocator.
 * Errors: as gdn_prefill, plus GDN_ERR_WORKSPACE for the size limit, and
 * GDN_ERR_CUDA if the set-up lookup fails.
 */
#define GDN_STATIC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_prefill_static(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                              const void *beta, const int32_t *cu_seqlens, int N, int T_total,
                              const void *conv_state_in, void *conv_state_out,
                              const float *ssm_state_in, float *ssm_state_out, void *out,
                              gdn_dtype act, gdn_dtype out_dt, int chunk_size, void *stream);

/* Bytes of the fixed scratch gdn_prefill_static uses (GDN_STATIC_SCRATCH_BYTES
 * of the built library). Pure host arithmetic. */
size_t gdn_static_scratch_bytes(void);

/*
 * gdn_in_proj -- the four input projections of section "SSM block --
 * Gated-Delta-Net", from the normed hidden state: attn_qkv -> qkv [8192],
 * attn_gate -> z [4096], ssm_alpha -> alpha [32], ssm_beta -> beta [32]. They
 * run as one tensor-core GEMM (bf16 operands, fp32 accumulation) over the four
 * weights stacked by rows; the epilogue writes each column range to its own
 * array, laid out as gdn_prefill and gdn_decode_step take them.
 *   h      [M][2048] bf16, row-major: attn_norm'd hidden states
 *   w_in   [12352][2048] bf16, row-major: attn_qkv.weight (rows 0..8191),
 *          attn_gate.weight (8192..12287), ssm_alpha.weight (12288..12319),
 *          ssm_beta.weight (12320..12351)
 *   qkv [M][8192], z [M][4096], alpha [M][32], beta [M][32] in dtype act
 * 0 <= M <= 2^24 (M == 0 is a no-op). Errors: GDN_ERR_INVALID_ARG, GDN_ERR_CUDA
 * (also when the driver's tensor-map encoder is unavailable).
 */
gdn_status gdn_in_proj(const void *h, const void *w_in, void *qkv, void *z, void *alpha, void *beta, int M,
                       gdn_dtype act, void *stream);

/*
 * gdn_in_proj_conv -- the input projections of gdn_in_proj with the causal
 * conv1d, SiLU and the q/k L2 norms ("Projections", "Causal conv1d" and the
 * split of section "SSM block -- Gated-Delta-Net") applied in the GEMM's
 * epilogue, so the raw q|k|v stream is never written. Over packed sequences
 * (cu_seqlens as for gdn_prefill):
 *   qkv = h w_qkv^T (fp32, not stored)
 *   xhat[m][c] = SiLU(sum_k conv_w[c][k] win_k[c]), win = the three inputs
 *       before m in its sequence (conv_state_in rows before the sequence's
 *       start, zeros without it) and qkv[m]; then each q and k head of 128
 *       channels divided by sqrt(sum of squares + l2_eps)
 *   z, alpha, beta = the other projections, rounded to bf16
 *   conv_state_out[n] = the raw inputs at the sequence's last three positions
 *       (rows of conv_state_in for positions before its start), bf16
 *   p          conv_w and l2_eps are read (the other fields are not)
 *   h          [M][2048] bf16;  w_in [12352][2048] bf16 (as gdn_in_proj)
 *   cu_seqlens device int32 [N+1], 0 = cu[0] <= ... <= cu[N] = M
 *   conv_state_in, conv_state_out  [N][3][8192] bf16, each may be NULL; they
 *              must not overlap
 *   xhat       [M][8192] fp16: the input gdn_prefill_xhat takes
 *   z [M][4096], alpha [M][32], beta [M][32] bf16
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_CUDA.
 */
gdn_status gdn_in_proj_conv(const gdn_params *p, const void *h, const void *w_in, const int32_t *cu_seqlens, int N,
                            int M, const void *conv_state_in, void *conv_state_out, void *xhat, void *z,
                            void *alpha, void *beta, void *stream);

/*
 * gdn_prefill_xhat -- gdn_prefill (chunked tensor-core form, bf16) starting
 * from the activations gdn_in_proj_conv writes: xhat replaces qkv and its
 * conv, and conv_state is not touched (gdn_in_proj_conv has advanced it).
 * Arguments, workspace (gdn_prefill_workspace_size(N, T_total, GDN_BF16, 64)
 * or any size down to one 64-token window) and errors as gdn_prefill.
 */
gdn_status gdn_prefill_xhat(const gdn_params *p, const void *xhat, const void *z, const void *alpha,
                            const void *beta, const int32_t *cu_seqlens, int N, int T_total,
                            const float *ssm_state_in, float *ssm_state_out, void *out, gdn_dtype out_dt,
                            void *workspace, size_t ws_bytes, void *stream);

/*
 * gdn_out_proj -- the projection right after the mixer, section "Output path":
 * cur = ssm_out . gated, 4096 -> GDN_HIDDEN (2048). It computes
 *   y[m][n] = sum_k x[m][k] * w[n][k]
 * with bf16 operands and fp32 accumulation on the tensor cores.
 *   x   [M][4096] bf16: the gated output of gdn_decode_step / gdn_prefill
 *       (out_dt = GDN_BF16), row-major
 *   w   [2048][4096] bf16: the layer's ssm_out.weight, row-major (one row per
 *       output feature)
 *   y   [M][2048] out_dt
 * 0 <= M <= 2^24 (M == 0 is a no-op). x and w must be 16-byte aligned (their row
 * stride, 8192 bytes, is fixed). Errors: GDN_ERR_INVALID_ARG, GDN_ERR_CUDA (also
 * when the driver's tensor-map encoder is unavailable). A bounded device wait
 * that gives up is reported afterwards by gdn_device_error.
 */
gdn_status gdn_out_proj(const void *x, const void *w, void *y, int M, gdn_dtype out_dt, void *stream);

/*
 * gdn_gated_out_proj -- the end of section "Output path" in one tensor-core
 * GEMM: the gated RMSNorm . silu(z) of the mixer's raw output y, then
 * cur = ssm_out . gated, 4096 -> GDN_HIDDEN (2048):
 *   gated[m][h*128 + j] = y[m][h*128 + j] * r * norm_w[j] * silu(z[m][h*128 + j]),
 *       r = (mean_j y[m][h*128 + j]^2 + norm_eps)^-1/2   (per row m and head h)
 *   out[m][n] = sum_k gated[m][k] * w[n][k]
 * The gated rows are formed inside the GEMM, as bf16 tensor-core operands
 * (fp32 accumulation), and never written to memory.
 *   norm_w [128] fp32 (ssm_norm.weight, applied as w)
 *   y      [M][4096] act: the mixer's output with the norm left out, i.e.
 *          gdn_decode_step / gdn_prefill called with params->norm_w == NULL
 *   z      [M][4096] act
 *   w      [2048][4096] bf16: ssm_out.weight, row-major
 *   out    [M][2048] out_dt
 * 0 <= M <= 2^24 (M == 0 is a no-op). All pointers 16-byte aligned. Errors:
 * GDN_ERR_INVALID_ARG, GDN_ERR_CUDA (also when the driver's tensor-map encoder
 * is unavailable). A bounded device wait that gives up is reported afterwards
 * by gdn_device_error.
 */
gdn_status gdn_gated_out_proj(const float *norm_w, float norm_eps, const void *y, const void *z, const void *w,
                              void *out, int M, gdn_dtype act, gdn_dtype out_dt, void *stream);

/*
 * gdn_attn_decode -- decode attention of the full-attention layers, steps 5-6
 * of section "Full-attention block" (the other layer type of the same model):
 * for every sequence b and query head h, with g = h / 8 (GQA: 8 query heads
 * share one KV head) and L = ctx_len[b],
 *   o   = sum_{p < L} softmax_p(k[b][g][p] . q[b][h] / sqrt(256)) v[b][g][p]
 *   out = o * sigmoid(z[b][h])            (elementwise over the 256 dims)
 *   q        [B][16][256] bf16: the new token's queries after their RMSNorm
 *            and partial RoPE (steps 2-4)
 *   k_cache, v_cache [B][2][Lmax][256] bf16: the KV cache, keys after their
 *            RMSNorm and RoPE, the new token's row already appended
 *   ctx_len  [B] int32 (device): cached positions of each sequence, clamped to
 *            [0, Lmax]; rows at or past ctx_len are never used, whatever they
 *            hold; ctx_len 0 gives out = 0
 *   z        [B][16][256] bf16: the output gate (second half of each head of
 *            the joint Q+gate projection)
 *   out      [B][16][256] out_dt
 *   workspace: device scratch of gdn_attn_decode_workspace_size(B, Lmax)
 *            bytes, 16-byte aligned, owned by the caller; contents on entry
 *            and exit are unspecified
 * The softmax weights enter the value product rounded to bf16 (fp32
 * accumulation), as the kernel's tensor cores take them.
 * 1 <= B <= 65535 (B == 0 is a no-op), 1 <= Lmax, B * 2 * Lmax <= 2^30.
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_WORKSPACE, GDN_ERR_CUDA (also when the
 * driver's tensor-map encoder is unavailable). A bounded device wait that gives
 * up is reported afterwards by gdn_device_error.
 */
gdn_status gdn_attn_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *ctx_len,
                           const void *z, void *out, int B, int Lmax, void *workspace, size_t workspace_bytes,
                           gdn_dtype out_dt, void *stream);

/* Bytes of workspace gdn_attn_decode needs for (B, Lmax); 0 if they are out of
 * range. Pure host arithmetic. */
size_t gdn_attn_decode_workspace_size(int B, int Lmax);

/* Bytes of workspace gdn_prefill needs for these sizes (0 if the arguments are
 * invalid; never 0 for valid ones). Pure host arithmetic. */
size_t gdn_prefill_workspace_size(int N, int T_total, gdn_dtype act, int chunk_size);

/* Device-side waits (on TMA copies and tensor-core completions) are bounded:
 * a wait that gives up leaves its kernel early, leaves that call's outputs
 * unspecified, and records GDN_ERR_TIMEOUT in a library-wide error word of the
 * current device. This call synchronises `stream`, then reads and clears that
 * word: GDN_OK, or GDN_ERR_TIMEOUT if any kernel of this library on the
 * current device gave up since the word was last cleared. */
gdn_status gdn_device_error(void *stream);

/* The same query under the name and argument list that the mixer's boundary
 * is specified with: `workspace` is accepted for that signature and not read
 * (the error word is per device, not per workspace, so a timeout in any call
 * is seen whichever workspace is named; NULL is fine). Same result and
 * synchronisation as gdn_device_error(stream). */
gdn_status gdn_get_device_error(void *workspace, void *stream);

/* Diagnostic of the failure path above: enqueues one small kernel that waits
 * on an mbarrier nothing ever completes, through the library's bounded wait.
 * After the limit (2 s) the kernel records GDN_ERR_TIMEOUT and returns
 * normally, so the next gdn_device_error on this stream reports
 * GDN_ERR_TIMEOUT (and clears it) and the context stays usable. Errors:
 * GDN_ERR_CUDA. */
gdn_status gdn_selftest_wait_timeout(void *stream);

/* Human-readable name of a status (static storage). */
const char *gdn_status_string(gdn_status s);

/* Text of the last GDN_ERR_CUDA / GDN_ERR_INVALID_ARG seen by the calling host
 * thread (thread-local, static storage; "" if none). */
const char *gdn_last_error(void);

/* GDN_ABI_VERSION of the built library. */
int gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
