/*
 * gdn.h -- C ABI of libgdn, the Gated DeltaNet token mixer on one GB300 GPU.
 *
 * The mixer is the linear-attention layer of the Qwen3.5 / Qwen3.8 hybrid
 * decoders.  Per sequence b, per value head h, per token t it computes
 *
 *   1. u = silu(causal depthwise conv, width 4) on the q|k|v channels
 *        page "Qwen3.8-27B" (docs.theformalera.com), node gdn.conv:
 *        y[t,c] = silu( sum_{j<4} w[c,j] * x[t+j-3, c] ); tokens before the
 *        first come from the carried conv window.
 *   2. q^ = q / sqrt(sum q^2 + eps_l2) * q_scale,  k^ = k / sqrt(sum k^2 + eps_l2)
 *        page "How Qwen3.5 works" (azmle112.github.io), section 9.4; value
 *        head h reads key head h / (Hv / Hk) (integer division).
 *   3. S_t = e^{g_t} S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T,
 *      o_t = S_t q^_t
 *        node gdn.core of the same spec (S is Dv x Dk, "value rows");
 *        "How Qwen3.5 works" section 9.6 gives the decay -> predict ->
 *        correct -> read order, section 9.11 the chunked form used by
 *        gdn_prefill.
 *   4. y_t = norm_w * o_t / sqrt(mean(o_t^2) + eps_norm) * silu(z_t), per head
 *        node gdn.norm; "How Qwen3.5 works" section 9.9.
 *
 * Layouts (row-major, innermost last; C = 2*Hk*Dk + Hv*Dv conv channels,
 * ordered q (Hk heads) | k (Hk heads) | v (Hv heads)):
 *   qkv_pre [B][T][C]       z, o [B][T][Hv*Dv]      g, beta [B][T][Hv] (fp32)
 *   conv_w  [C][4]          norm_w [Dv]             S [B][Hv][Dv][Dk] (fp32)
 *   conv window [B][3][C]   raw (pre-conv) rows of the three previous tokens,
 *                           oldest first
 * "io" tensors (qkv_pre, z, o, conv windows, conv_w, norm_w) all have the
 * dtype shape->io_dtype; g, beta and the state are always fp32.
 *
 * Ownership and execution: every pointer is a device pointer owned by the
 * caller; the library allocates no memory, keeps no state between calls
 * (apart from a per-device error word, see gdn_device_status), and enqueues
 * its kernels on `stream` (a cudaStream_t; NULL = the legacy default stream)
 * without synchronising.  Calls on different streams do not share buffers.
 *
 * Errors: arguments are checked on the host before anything is launched; a
 * non-zero status means nothing was enqueued, except GDN_ERR_CUDA from the
 * launch itself.  Values are not checked: g must be <= 0 (finite, or -inf
 * for a reset) and beta in [0, 1]; other values give unspecified results
 * but stay within the buffers.
 *
 * Numeric domain of the bf16-io prefill (the chunked tensor-core kernels).
 * The products run on the tensor cores with fp16 operands and fp32
 * accumulation; the state itself stays fp32.
 *   - g below -80 acts as -80: a decay of e^-80 (about 1.8e-35) stands in for
 *     any smaller one, the reset g = -inf included.  Decode and the fp32-io
 *     kernels use e^g as given (e^-inf = 0).
 *   - Overflow: the fp16 copy of the state that multiplies W and q^, the
 *     chunk's Delta = U - W S (and Delta scaled by decay ratios <= 1) and W
 *     are converted without a range clamp, so |S|, |Delta| and |W| must stay
 *     below 65504; entries beyond it become inf.  Inputs (v, S0, the inverse
 *     T) are saturated to +-65504 instead.  Normalised q^ and k^ are <= 1.
 *   - Underflow: entries below 6.1e-5 in magnitude are fp16 subnormals
 *     (absolute spacing 6.0e-8), so where the state's entries are of order
 *     1e-4 and smaller, the products S W^T and S q^ carry them with fewer
 *     significant bits (the fp32 state and its update keep full precision).
 *   Tested against the fp64 oracle within the tolerances: qkv_pre scaled by
 *   1e-3 and by 30, initial states of rms 1e-4 and 10, g = -inf anywhere in
 *   a chunk, g down to -1e4, runs of beta = 0 and beta = 1.
 */
#ifndef GDN_H
#define GDN_H

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 4

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,       /* null pointer, B < 1, T < 1, bad dtype or eps */
  GDN_ERR_UNSUPPORTED_SHAPE = 2, /* Dk or Dv != 128, Hv % Hk != 0, too large */
  GDN_ERR_ALIGNMENT = 3,         /* a pointer not 16-byte aligned */
  GDN_ERR_ALIAS = 4,             /* two buffers overlap where that is forbidden */
  GDN_ERR_CUDA = 5,              /* a CUDA runtime call failed */
  GDN_ERR_TIMEOUT = 6,           /* a device-side wait gave up (see gdn_device_status) */
  GDN_ERR_NO_DEVICE = 7,         /* the current device is not an sm_103 GPU */
  GDN_ERR_BOUNDS = 8             /* a device bounds check failed (GDN_CHECKS builds only) */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef struct {
  int B;          /* sequences */
  int T;          /* tokens per sequence in this call (decode: 1) */
  int Hk, Hv;     /* key heads, value heads; Hv % Hk == 0 */
  int Dk, Dv;     /* head widths; the GPU kernels take 128 only */
  int io_dtype;   /* gdn_dtype of the io tensors */
  float eps_l2;   /* epsilon inside the q/k L2 root (1e-6 in the models) */
  float eps_norm; /* epsilon of the gated RMSNorm (1e-6 in the models) */
  float q_scale;  /* query scale after normalising; 0 means 1/sqrt(Dk) */
} gdn_shape;

/* GDN_ABI_VERSION of the loaded library. */
int gdn_abi_version(void);

/* A static, human-readable name for a status code. */
const char *gdn_status_str(int status);

/*
 * Prefill: run T tokens of B sequences through the mixer, carrying the state.
 *
 *   qkv_pre, z, g, beta      this call's tokens, layouts above
 *   conv_w, norm_w           layer weights
 *   S0     [B][Hv][Dv][Dk]   incoming state, or NULL for zeros
 *   conv0  [B][3][C]         incoming conv window, or NULL for zeros
 *   o      [B][T][Hv*Dv]     out: the mixer output (after the gated norm)
 *   S_T    [B][Hv][Dv][Dk]   out: final state; may be exactly S0 (in place),
 *                            must not otherwise overlap any buffer
 *   conv_T [B][3][C]         out: the last three raw rows of conv0 ++ qkv_pre;
 *                            must not overlap conv0 or qkv_pre
 *   o must not overlap any input.  All pointers 16-byte aligned.
 *
 * The chunked form ("How Qwen3.5 works" section 9.11, chunk 64) is used:
 * it is the same recurrence reorganised, so results match the token loop up
 * to rounding.  Continuing a prefill from (S_T, conv_T) equals one longer
 * prefill; a decode step is a prefill of one token.
 */
gdn_status gdn_prefill(const gdn_shape *shape, const void *qkv_pre, const void *z,
                       const float *g, const float *beta, const void *conv_w,
                       const void *norm_w, const float *S0, const void *conv0, void *o,
                       float *S_T, void *conv_T, void *stream);

/*
 * Decode: one new token for each of B sequences ("How Qwen3.5 works"
 * section 13.3: each linear layer updates its conv window and does one
 * recurrent step on the cached state).  shape->T must be 1.
 *
 *   qkv_pre [B][C], z [B][Hv*Dv], g and beta [B][Hv]    the new token
 *   S       [B][Hv][Dv][Dk]   the cached state, updated in place
 *   conv_in [B][3][C]         the cached window
 *   conv_out[B][3][C]         out: the new window; must not overlap conv_in
 *                             (callers ping-pong two buffers)
 *   o       [B][Hv*Dv]        out: the mixer output for the token
 */
gdn_status gdn_decode_step(const gdn_shape *shape, const void *qkv_pre, const void *z,
                           const float *g, const float *beta, const void *conv_w,
                           const void *norm_w, float *S, const void *conv_in, void *conv_out,
                           void *o, void *stream);

/*
 * Raw gate projections ("How Qwen3.5 works" section 9.5): per token and
 * value head the library forms, in fp32,
 *   beta = sigmoid(b),   g = -exp(A_log[h]) * softplus(a + dt_bias[h]).
 *   a, b            [tokens][Hv], io dtype (the outputs of the a and b
 *                   projections, same token order as z)
 *   A_log, dt_bias  [Hv] fp32 layer parameters
 */
typedef struct {
  const void *a, *b;
  const float *A_log, *dt_bias;
} gdn_raw_gates;

/*
 * Arguments of gdn_prefill_ex.  Exactly one gate source: (g, beta) or
 * raw_gates.  "tokens" is B*T for fixed-length sequences and T for packed
 * ones (below).
 *   qkv_pre [tokens][C]   z, o [tokens][Hv*Dv]   g, beta [tokens][Hv]
 *   S0, S_T, conv0, conv_T per sequence, as for gdn_prefill
 *   cu_seqlens  device int32 [B+1] or NULL.  When given, the B sequences are
 *               packed back to back ("varlen"): sequence s owns tokens
 *               cu_seqlens[s] .. cu_seqlens[s+1]-1 and shape->T is the total
 *               token count.  Each sequence starts from its own S0[s] and
 *               conv0[s] (or zeros); nothing flows between sequences.  A
 *               sequence of length 0 copies its incoming state and window.
 *               The offsets are read on the device: offsets that decrease
 *               or leave [0, T] make the kernel skip that sequence (its
 *               outputs stay untouched) and record GDN_ERR_INVALID_ARG for
 *               gdn_device_status.
 *   S_snap      [tokens][Hv][Dv][Dk] fp32 or NULL: the state after every
 *               token (for rollback; costs one state write per token).
 *   workspace   device scratch, 256-byte aligned, overlapping no other
 *               argument, or NULL; workspace_bytes says how large it is.
 *               Owned by the caller; its contents are undefined after the
 *               call and it must not be shared by calls that may run
 *               concurrently.  The chunked prefill takes the fastest form
 *               the workspace holds:
 *                 >= gdn_prefill_workspace_bytes(), and B * Hv (sequences x
 *                    value heads) below twice the GPU's SM count: the
 *                    chunk-parallel form (with more units the staged form
 *                    below already fills every SM, and moves fewer bytes).
 *                    q^ and k^ are formed once per key head (first kernel);
 *                    everything of a chunk that does not depend on the
 *                    carried state (the inverse T, U, W, the decayed
 *                    Q K^T) is formed for every chunk at once (second
 *                    kernel); a third kernel walks the chunks of each
 *                    (sequence, value head) with the state in TMEM, doing
 *                    only the state-dependent products, the state update
 *                    and the gated norm ("How Qwen3.5 works" section 9.11
 *                    separates exactly these two parts).
 *                 >= gdn_prefill_staged_bytes(): q^ and k^ once per key head
 *                    into the workspace, then one kernel per (sequence,
 *                    value head) for the rest.
 *                 smaller: GDN_ERR_INVALID_ARG.
 *               NULL: one kernel per (sequence, value head) does everything.
 *               All forms compute the same chunked recurrence; they differ
 *               in rounding order only.
 * bf16 io without snapshots (fixed length or packed) runs the chunked
 * tensor-core kernels; fp32 io and snapshots run the token-serial kernel,
 * which ignores the workspace.
 */
typedef struct {
  const void *qkv_pre, *z;
  const float *g, *beta;
  const gdn_raw_gates *raw_gates;
  const void *conv_w, *norm_w;
  const float *S0;
  const void *conv0;
  void *o;
  float *S_T;
  void *conv_T;
  const int *cu_seqlens;
  float *S_snap;
  void *workspace;
  size_t workspace_bytes;
} gdn_prefill_io;

/* Bytes of workspace of the chunk-parallel prefill for this shape (packed:
 * the call passes cu_seqlens, so the token rows are shape->T, else B*T):
 * the staged q^ and k^ (gdn_prefill_staged_bytes, rounded up to 256) plus
 * 57,860 bytes per (chunk slot, value head) -- U^T fp32 and -W^T fp16
 * [128][64], M fp16 [64][64], two fp32 vectors of 64 and a ready flag (the
 * two parts may run in one launch) -- where the chunk
 * slots are B * ceil(T/64) for fixed-length sequences and T/64 + B + 2 for
 * packed ones.  Where the work items would exceed 2^24 it returns the staged
 * size.  0 when the shape is invalid or the call would not run the chunked
 * kernels (fp32 io). */
size_t gdn_prefill_workspace_bytes(const gdn_shape *shape, int packed);

/* Bytes of workspace of the staged form alone: the q^ and k^ of every token
 * row and key head, 3 fp16 values per element (q^, and k^ as a hi/lo
 * pair).  0 as above. */
size_t gdn_prefill_staged_bytes(const gdn_shape *shape, int packed);

/* Prefill with the options above; aliasing and alignment rules as for
 * gdn_prefill (raw gates, cu_seqlens and S_snap count as inputs / outputs). */
gdn_status gdn_prefill_ex(const gdn_shape *shape, const gdn_prefill_io *io, void *stream);

/*
 * gdn_prefill_ex with no caller workspace and no allocation: the call runs
 * in a device scratch array that the library owns, one per device,
 * GDN_STATIC_SCRATCH_BYTES large, as gdn_prefill_ex would with a workspace
 * of that size (the chunk-parallel form where it fits, else the staged
 * form).  The pages have no counterpart; this is a serving convenience of
 * the library.
 *   io->workspace must be NULL (GDN_ERR_INVALID_ARG otherwise).
 *   A call whose staged need (gdn_prefill_staged_bytes) exceeds the scratch
 *   returns GDN_ERR_UNSUPPORTED_SHAPE before any launch.
 *   Nothing in the scratch has to start at zero: every byte a kernel reads
 *   there is written first by an earlier kernel of the same call.
 *   The scratch is shared by every call on the device: calls that overlap in
 *   time (different streams, or unordered host threads) race on it and give
 *   undefined results.  Issue them on one stream, or order them.
 *   The array is device memory of the library's own module; with lazy
 *   module loading (the CUDA default) it is allocated at the first call.
 */
#define GDN_STATIC_SCRATCH_BYTES (512ull << 20)
gdn_status gdn_prefill_static(const gdn_shape *shape, const gdn_prefill_io *io, void *stream);

/*
 * Arguments of gdn_decode_ex: shape->T >= 1 new tokens for each of B
 * sequences from the cached state, e.g. the draft tokens of speculative
 * decoding being verified ("How Qwen3.5 works" section 13).
 *   qkv_pre [B][T][C]   z, o [B][T][Hv*Dv]   g, beta [B][T][Hv] (or raw_gates)
 *   S        [B][Hv][Dv][Dk]     the cached state, updated in place (final state)
 *   S_snap   [B][T][Hv][Dv][Dk]  or NULL: the state after each token, so that a
 *                                caller who accepts only the first m tokens can
 *                                restore snapshot m-1
 *   conv_in, conv_out [B][3][C]  cached window in; window after the T tokens out
 *                                (must not overlap)
 * T <= 16 runs the decode kernel of gdn_decode_step (the state streamed once
 * through registers for all T tokens); longer runs use the token-serial
 * prefill kernel with the state in place.
 */
typedef struct {
  const void *qkv_pre, *z;
  const float *g, *beta;
  const gdn_raw_gates *raw_gates;
  const void *conv_w, *norm_w;
  float *S;
  float *S_snap;
  const void *conv_in;
  void *conv_out;
  void *o;
} gdn_decode_io;

gdn_status gdn_decode_ex(const gdn_shape *shape, const gdn_decode_io *io, void *stream);

/*
 * The projections around the mixer, nodes gdn.in_proj (K=5120 -> N=16480)
 * and gdn.out_proj (K=6144 -> N=5120) of the page "Qwen3.8-27B":
 *   y[t, n] = sum_k x[t, k] w[n, k],   t < M, n < N, k < K
 * bf16 inputs, fp32 accumulation on the tensor cores, bf16 outputs.  The
 * pages give the formula; the column routing is this library's: columns
 * [col_begin, col_end) of y are written to ptr[t * ld + (n - col_begin)],
 * so the in_proj output can land directly in the mixer's qkv_pre, z, b and a
 * buffers (columns 0-10239, 10240-16383, 16384-16431, 16432-16479 at the 27B
 * shape).
 *   x   [M][ldx] bf16, ldx >= K       w [N][ldw] bf16 (nn.Linear layout), ldw >= K
 *   ldx, ldw multiples of 8 (16-byte rows); x, w 16-byte aligned
 *   out[0 .. n_out-1], 1 <= n_out <= 4: disjoint column ranges inside [0, N),
 *   ld >= col_end - col_begin; output rows must not overlap x, w or each other
 * Columns not covered by any range are computed and dropped.
 */
typedef struct {
  int col_begin, col_end;
  void *ptr;
  long long ld;
} gdn_linear_out;

gdn_status gdn_linear(int M, int N, int K, const void *x, long long ldx, const void *w, long long ldw,
                      int n_out, const gdn_linear_out *out, void *stream);

/*
 * Synchronise `stream` and report device-side failures recorded since the
 * last reset: GDN_ERR_TIMEOUT if a kernel's bounded wait gave up (the kernel
 * then returned early and its outputs are incomplete), GDN_ERR_BOUNDS if a
 * store failed its bounds check (only in a library built with GDN_CHECKS,
 * where every thread-issued global store of the prefill and decode kernels
 * is checked against its buffer and skipped when outside it),
 * GDN_ERR_INVALID_ARG if a kernel met packed-sequence offsets it could not
 * use, GDN_ERR_CUDA if the synchronisation itself failed, GDN_OK otherwise.  reset != 0 clears the
 * record afterwards.  The record is one word per device, shared by all
 * streams.
 */
gdn_status gdn_device_status(void *stream, int reset);

/*
 * Failure-detection self-test; the pages have no counterpart (they describe
 * no kernels).  Enqueues one CTA that takes the same steps as a prefill
 * kernel whose awaited work never completes: it allocates TMEM, waits on an
 * mbarrier that nothing arrives on with the bounded wait the prefill kernel
 * uses, here limited to `wait_us` microseconds (1 .. 1000000), records the
 * timeout in the device error word, frees its TMEM and returns.  Afterwards
 * gdn_device_status reports GDN_ERR_TIMEOUT and the context stays usable.
 * Nothing is allocated and no caller buffer is touched.
 * Errors: GDN_ERR_INVALID_ARG for wait_us out of range, GDN_ERR_NO_DEVICE,
 * GDN_ERR_CUDA from the launch.
 */
gdn_status gdn_selftest_wait_timeout(int wait_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
