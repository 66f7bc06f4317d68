/*
 * yoco.h -- C ABI of libyoco, the GB300 (sm_103a) token-mixing path of YOCO
 * ("You Only Cache Once: Decoder-Decoder Architectures for Language Models",
 * arXiv:2405.05254v2).
 *
 * Two parts of the model are covered:
 *   - gated retention (gRet), the self-decoder's token mixer
 *     (paper Section 3.1, Eqs. 4-6; Appendix F);
 *   - the cross-decoder's causal grouped-query softmax attention against the
 *     ONE shared K^/V^ cache projected once from the self-decoder output
 *     (paper Section 2.2, Eqs. 2-3).
 * Prefill runs the chunkwise gRet form and fills the shared cache, then runs
 * the cross layers only for the last prompt token; generation runs the
 * recurrent gRet form and appends one cache slot per token before the cross
 * layers read it (paper Section 2.3, Fig. 3).
 *
 * Conventions common to every call:
 *   - Every tensor argument is a DEVICE pointer to caller-owned memory, dense
 *     row-major with the last index fastest.  The library allocates nothing
 *     on the device and never frees caller memory.  Its only state is
 *     process-wide bookkeeping: the per-thread error text, a launch counter,
 *     each device's SM count (queried once), the test hooks below, and the
 *     no-workspace decode's built-in scratch array (see
 *     yoco_cross_attn_decode_noalloc).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work on it and return without synchronising.
 *   - Arguments are validated on the host before anything is enqueued; on
 *     any error nothing is launched and nothing is written.
 *   - Status YOCO_ERR_CUDA means a launch failed; yoco_last_error() has the
 *     CUDA error text.  It is per thread.
 *   - bf16 tensors hold raw bfloat16 bit patterns (uint16 per element).
 *   - Gate logits and gRet states are always fp32.
 */
#ifndef YOCO_H
#define YOCO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define YOCO_VERSION 100 /* 1.0.0 */

#if defined(__GNUC__)
#define YOCO_API __attribute__((visibility("default")))
#else
#define YOCO_API
#endif

typedef enum {
    YOCO_OK = 0,
    YOCO_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad position       */
    YOCO_ERR_UNSUPPORTED = 2, /* head size / dtype / ratio the kernels lack  */
    YOCO_ERR_CAPACITY = 3,    /* append would pass the cache capacity        */
    YOCO_ERR_CUDA = 4,        /* a kernel launch or CUDA call failed         */
    YOCO_ERR_TIMEOUT = 5,     /* a bounded on-device wait gave up            */
    YOCO_ERR_WORKSPACE = 6    /* workspace missing, too small or misaligned  */
} yoco_status;

typedef enum { YOCO_F32 = 0, YOCO_BF16 = 1 } yoco_dtype;

/*
 * The shared K^/V^ cache (paper Section 2.2: projected once from the
 * self-decoder output, reused by every cross-decoder layer).  One cache per
 * batch of B sequences that all have the same length.
 *   k, v      [B, Hkv, capacity, d] of `dtype` (caller-owned device memory)
 *   len_dev   device int32[2]; [0] = current length, [1] = an internal
 *             counter that must be 0 before the first append (zero both).
 *             Appends update [0] on the device, so a captured CUDA graph
 *             sees the new length on replay.
 *   len_host  host copy of the length; appends advance it, attention calls
 *             read it.  The caller keeps it equal to len_dev[0].
 *   Attention calls may start loading k and v while the kernel before them
 *   on the stream is still finishing (programmatic dependent launch).  An
 *   append never lets a following kernel start early, so appends are always
 *   complete; a caller that writes k or v with a kernel of its own must not
 *   have that kernel release its dependents early either.
 *   rope_base 0: no rotary encoding.  > 1: rotary position encoding (paper
 *             Section 3.1, Q (.) Theta / K (.) conj(Theta); the shared K^ is
 *             rotated once when projected, each cross layer rotates its Q):
 *             appends turn channel pair (2i, 2i+1) of K^ at slot p by
 *             p * rope_base^(-2i/d) before rounding, and attention calls turn
 *             each query row's pairs by its position the same way.  V is never
 *             rotated.
 */
typedef struct {
    void *k;
    void *v;
    int32_t *len_dev;
    int64_t len_host;
    int32_t B;
    int32_t Hkv;
    int32_t d;
    int64_t capacity;
    yoco_dtype dtype;
    float rope_base;
} yoco_kv_cache;

/* ------------------------------------------------------------------ gRet */

/*
 * Chunkwise gated-retention prefill (paper Section 3.1, Eq. 6 with
 * consistent indices; Appendix F ChunkwiseRetention), per head:
 *     gamma_n = sigmoid(logit_n)^(1/tau), taken as exp(logsigmoid(logit)/tau)
 *     S_n = gamma_n S_{n-1} + k_n^T v_n,    o_n = q_n S_n
 * evaluated chunk by chunk (intra-chunk decay-masked Q K^T V plus the carried
 * state).  No 1/sqrt(d) scale and no group norm are applied: o is the raw
 * retention output.
 *   q, k         [B, N, H, dk]  in_dt        v  [B, N, H, dv] in_dt
 *   gate_logits  [B, N, H]      fp32         o  [B, N, H, dv] out_dt
 *   state        [B, H, dk, dv] fp32, in: the state before token 0 (zero it
 *                for a fresh sequence), out: the state after token N-1.
 *   chunk        0, 64 or 128 (anything else: YOCO_ERR_UNSUPPORTED); the
 *                result depends on it only through rounding.  0 and 128 run
 *                the tensor-core kernel (128-token chunks) when in_dt is bf16
 *                and dk = dv = 128, else the CUDA-core kernel (64-token
 *                chunks, fp32 arithmetic); 64 always runs the CUDA-core kernel.
 *                With bf16 and d = 128 the tensor-core kernel leaves out state
 *                contributions whose decay weight is below e^-40 (~4e-18).
 *   workspace    device scratch of at least yoco_gret_prefill_workspace_size
 *                bytes, 256-byte aligned (may be NULL when that size is 0).
 * Supported: dk = dv in {64, 128}; in_dt = out_dt; N >= 0 (N = 0 leaves
 * state unchanged); gate logits may be +-inf.
 * Calls that share `workspace` must be ordered on one stream.
 */
YOCO_API yoco_status yoco_gret_prefill_chunkwise(const void *q, const void *k, const void *v,
                                        const float *gate_logits, float tau, void *o,
                                        float *state, int B, int N, int H, int dk, int dv,
                                        int chunk, yoco_dtype in_dt, yoco_dtype out_dt,
                                        void *workspace, size_t ws_bytes, void *stream);

YOCO_API size_t yoco_gret_prefill_workspace_size(int B, int N, int H, int dk, int dv, int chunk,
                                        yoco_dtype in_dt);

/*
 * One recurrent gated-retention step (paper Section 3.1, Eq. 5; Appendix F
 * RecurrentRetention without its group norm), per head:
 *     S <- gamma S + k^T v,   o = q S
 *   q, k [B, H, dk], v [B, H, dv]  in_dt;  gate_logits [B, H] fp32;
 *   state [B, H, dk, dv] fp32 updated in place;  o [B, H, dv] out_dt.
 * Supported: dk = dv in {64, 128}.
 */
YOCO_API yoco_status yoco_gret_decode_step(const void *q, const void *k, const void *v,
                                  const float *gate_logits, float tau, float *state, void *o,
                                  int B, int H, int dk, int dv, yoco_dtype in_dt,
                                  yoco_dtype out_dt, void *stream);

/* ------------------------------------------------------------- shared KV */

/*
 * Shared K^/V^ projection and append (paper Section 2.2, Eq. 2):
 *     K^ = RMSNorm(M) W_K,   V^ = RMSNorm(M) W_V
 *     RMSNorm(m) = m * g / sqrt(mean(m^2) + eps)
 * for T new tokens of each of the B sequences, written to cache slots
 * [len, len + T) of every kv head, after which the length is len + T.
 *   M      [B, T, dm]       cache dtype
 *   rms_w  [dm] gain g      cache dtype, or NULL for ones
 *   Wk, Wv [dm, Hkv * d]    cache dtype; column h*d + c feeds head h, lane c
 * All four pointers 16-byte aligned.
 * Exactly slots [len, len + T) change; every other cache byte is untouched.
 * The weights (Wk, Wv, rms_w) may be read while the kernel before the call on
 * the stream is still finishing (programmatic dependent launch); a caller that
 * writes them with a kernel of its own just before the append must not let that
 * kernel release its dependents early.  M is read only after it has finished.
 * Returns YOCO_ERR_CAPACITY (nothing written) if len + T > capacity.
 *   workspace  >= yoco_shared_kv_workspace_size bytes, 256-byte aligned.
 */
YOCO_API yoco_status yoco_shared_kv_project_append(const void *M, const void *rms_w, float eps,
                                          const void *Wk, const void *Wv, int T, int dm,
                                          yoco_kv_cache *cache, void *workspace,
                                          size_t ws_bytes, void *stream);

YOCO_API size_t yoco_shared_kv_workspace_size(int B, int T, int dm, const yoco_kv_cache *cache);

/* ------------------------------------------------------- cross attention */

/*
 * Cross-decoder attention, prefill form (paper Section 2.2, Eq. 3): causal
 * grouped-query softmax attention of T query rows at positions p0 .. p0+T-1
 * against the shared cache; row t reads slots 0 .. p0 + t.
 *     o = sum_m softmax_m(scale * q . k_m) v_m
 * Query head h reads kv head h / (Hq / Hkv).
 *   Q, O [B, T, Hq, d] cache dtype.   Requires p0 >= 0, p0 + T <= len.
 * With early exit (paper Section 2.3, Fig. 3) a prefill calls this with
 * T = 1 at p0 = len - 1.
 */
YOCO_API yoco_status yoco_cross_attn_prefill(const void *Q, int Hq, int T, int64_t p0,
                                    const yoco_kv_cache *cache, float scale, void *O,
                                    void *workspace, size_t ws_bytes, void *stream);

/*
 * Cross-decoder attention for the newest token of each sequence (position
 * len - 1, so it reads every slot including its own, which the preceding
 * append wrote).  Split-KV: num_splits slices of the cache are reduced in
 * parallel and merged by log-sum-exp; 0 = automatic, at most 4096 (more
 * returns YOCO_ERR_UNSUPPORTED).
 *   Q, O [B, Hq, d] cache dtype.   Requires len >= 1.
 */
YOCO_API yoco_status yoco_cross_attn_decode(const void *Q, int Hq, const yoco_kv_cache *cache,
                                   float scale, int num_splits, void *O, void *workspace,
                                   size_t ws_bytes, void *stream);

/*
 * Cross-attention decode without a workspace, for callers that cannot
 * allocate device memory when they decode (a runtime that forbids allocation
 * after start-up, a serving loop with a fixed memory budget, a plugin handed
 * only its input and output buffers).  The paper has no counterpart: this is
 * a deployment variant of yoco_cross_attn_decode with the same arguments and
 * result, minus the workspace.
 *   - Its scratch is a 4 MiB array built into the library's device code.  The
 *     CUDA runtime creates it on every GPU that loads libyoco; it stays there
 *     until the process exits.  The call itself allocates nothing.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress on the current device); make that first call
 *     before capturing any stream on that device.
 *   - num_splits = 0 picks the usual split count, lowered until the partial
 *     results fit in 4 MiB.  An explicit num_splits whose partials
 *     (B * Hq * num_splits * (d + 2) * 4 bytes) do not fit, or above 4096,
 *     returns YOCO_ERR_UNSUPPORTED and launches nothing.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (every partial read is first written by the same call, so
 *     nothing needs clearing).  Calls that overlap on the GPU, e.g. on two
 *     streams at once, race on it: order them on one stream.
 *   - The array's first 256 bytes are the status word a workspace would hold
 *     (see yoco_workspace_status): read it with
 *     yoco_cross_attn_decode_noalloc_status.
 */
YOCO_API yoco_status yoco_cross_attn_decode_noalloc(const void *Q, int Hq, const yoco_kv_cache *cache,
                                                    float scale, int num_splits, void *O, void *stream);

/*
 * Status word of the no-workspace decode's built-in scratch on the current
 * device, as yoco_workspace_status reports it for a workspace: waits for
 * `stream`, returns YOCO_OK or YOCO_ERR_TIMEOUT (a bounded on-device wait of an
 * earlier no-workspace call gave up; detail in yoco_last_error()), and with
 * clear != 0 resets the word.  Allocates nothing.
 */
YOCO_API yoco_status yoco_cross_attn_decode_noalloc_status(int clear, void *stream);

/* Workspace bytes for a prefill (T rows) or decode (T = 1) attention call. */
YOCO_API size_t yoco_cross_attn_workspace_size(int B, int Hq, int T, const yoco_kv_cache *cache,
                                      int num_splits);

/* ------------------------------------- gated retention output (Eq. 7) */

/*
 * Output of multi-head gated retention (paper Section 3.1, Eq. 7):
 *     z = swish(gate) (.) GroupNorm_h(o),   swish(x) = x sigmoid(x),
 * GroupNorm with one group per head: each token's head vector is centred and
 * divided by sqrt(variance over its d channels + eps), then multiplied by
 * gn_weight and shifted by gn_bias per channel (fp32 [H * d]; NULL = 1 / 0).
 * o, gate, z [B, N, H, d] of dtype dt (gate = X W_G, computed by the caller);
 * N = 1 serves a decode step.  z may be o.  d in {64, 128}; eps > 0.
 */
YOCO_API yoco_status yoco_gret_group_norm_gate(const void *o, const void *gate, const float *gn_weight,
                                               const float *gn_bias, float eps, void *z, int B, int N, int H, int d,
                                               yoco_dtype dt, void *stream);

/*
 * One recurrent step (as yoco_gret_decode_step) followed by Eq. 7's output for
 * that token, fused: z = swish(gate) (.) GroupNorm_h(o) with o the step's
 * fp32 output, never rounded or stored.  GroupNorm as in
 * yoco_gret_group_norm_gate (one group per head, biased variance over the dv
 * channels, eps > 0, gn_weight / gn_bias fp32 [H * dv] or NULL), except that
 * the variance is formed as E[o^2] - E[o]^2 in fp32.
 *   q, k [B, H, dk], v, gate, z [B, H, dv] of dtype dt; gate_logits [B, H]
 *   fp32; state [B, H, dk, dv] fp32 in/out.  dk = dv in {64, 128}.
 * The dv/32 CTAs of each head run as one thread-block cluster.
 */
YOCO_API yoco_status yoco_gret_decode_step_gn_gate(const void *q, const void *k, const void *v,
                                                   const float *gate_logits, float tau, float *state,
                                                   const void *gate, const float *gn_weight, const float *gn_bias,
                                                   float eps, void *z, int B, int H, int dk, int dv, yoco_dtype dt,
                                                   void *stream);

/*
 * Chunkwise gated-retention prefill with the paper's Eq. 7 output for every
 * token, fused (Section 3.1 Eq. 7; Appendix F ChunkwiseRetention applies the
 * group norm to the chunk output):
 *     z = swish(gate) (.) GroupNorm_h(o),   o = yoco_gret_prefill_chunkwise's output
 * GroupNorm as in yoco_gret_group_norm_gate: one group per head, biased
 * variance over the head's d channels, eps > 0, gn_weight / gn_bias fp32
 * [H * d] or NULL (1 / 0).  With bf16 and d = 128 (the tensor-core kernel) o is
 * never rounded or stored: each output row is normalised (moments of its fp32
 * values) and gated as it leaves tensor memory.  Otherwise the CUDA-core kernel
 * writes o into z and Eq. 7 is applied to z in place (two launches).
 *   q, k, v, gate, z [B, N, H, d] of dtype dt (gate = X W_G, the caller's);
 *   gate_logits [B, N, H] fp32; state as in yoco_gret_prefill_chunkwise.
 *   workspace: yoco_gret_prefill_workspace_size(B, N, H, d, d, 0, dt) bytes.
 * Supported: dk = dv in {64, 128}.
 */
YOCO_API yoco_status yoco_gret_prefill_chunkwise_gn_gate(const void *q, const void *k, const void *v,
                                                         const float *gate_logits, float tau, const void *gate,
                                                         const float *gn_weight, const float *gn_bias, float eps,
                                                         void *z, float *state, int B, int N, int H, int dk, int dv,
                                                         yoco_dtype dt, void *workspace, size_t ws_bytes,
                                                         void *stream);

/* ------------------------- gated-retention input projections in one GEMM */

/*
 * The gated-retention layer's input projections (paper Section 3.1:
 * Q = (X W_Q) (.) Theta, K = (X W_K) (.) conj(Theta), V = X W_V,
 * gamma = sigmoid(X W_gamma)^(1/tau)) as one GEMM that reads X once:
 *     [q | k | v | gate_logits] = X [W_Q | W_K | W_V | W_gamma]
 *   X [B, N, dm] bf16 (the layer's normalised input);
 *   W [dm, 3 H d + H] bf16, columns W_Q | W_K | W_V | W_gamma;
 *   q, k, v [B, N, H, d] bf16 token-major, as yoco_gret_prefill_chunkwise reads them;
 *   gate_logits [B, N, H] fp32 = X W_gamma (the chunk and recurrent kernels apply
 *   logsigmoid / tau).
 * rope_base > 1 turns q and k by position pos0 + n (channel pairs (2i, 2i+1),
 * base^(-2i/d)); 0 leaves them.  bf16 on the tensor cores; d in {64, 128};
 * dm and H multiples of 8.  workspace: yoco_gret_qkvg_workspace_size bytes.
 */
YOCO_API yoco_status yoco_gret_qkvg_project(const void *X, const void *W, int B, int N, int dm, int H, int d,
                                            int64_t pos0, float rope_base, void *q, void *k, void *v,
                                            float *gate_logits, void *workspace, size_t ws_bytes, void *stream);
YOCO_API size_t yoco_gret_qkvg_workspace_size(int B, int N, int H, int d, float rope_base);

/* ----------------------------------------------- rotary position encoding */

/*
 * Rotary position encoding in place (paper Section 3.1: Q (.) Theta,
 * K (.) conj(Theta), Theta_n = e^{i n theta}), for the q and k a self-decoder
 * layer (gated retention or sliding-window attention) mixes: channel pair
 * (2i, 2i+1) of row n turns by (pos0 + n) * base^(-2i/d).  The shared K^ and
 * the cross layers' queries are rotated inside the append and attention calls
 * instead (yoco_kv_cache.rope_base).
 *   x [B, N, H, d] token-major, dtype dt; d in {64, 128}; base > 1; pos0 >= 0.
 */
YOCO_API yoco_status yoco_rope_apply(void *x, int B, int N, int H, int d, int64_t pos0, float base, yoco_dtype dt,
                                     void *stream);

/* ------------------------------------------- sliding-window self-decoder */

/*
 * The pages' second self-decoder choice (paper Section 3.2, Eq. 8): each query
 * attends to the C most recent keys of its own layer, itself included,
 *     head = softmax(scale * Q K^T + B) V,  B_nm = 0 for n - C < m <= n, else -inf,
 * so the layer's cache is a ring of C tokens whatever the sequence length.
 * (Eq. 8 prints no scale; `scale` is the caller's, 1 / sqrt(d) in practice.)
 *
 * Ring cache, caller-owned: token at position p lives in slot p % window of
 *   k, v [B, Hkv, window, d] (dtype).  `pos` is the number of tokens seen, i.e.
 *   the next token's position; prefill and decode advance it on the host.
 */
typedef struct {
    void *k, *v;
    int B, Hkv, d;
    int window;   /* C */
    int64_t pos;  /* tokens seen */
    yoco_dtype dtype;
} yoco_swa_ring;

/*
 * Prefill of a new sequence (ring->pos must be 0): q [B, N, Hq, d], k, v
 * [B, N, Hkv, d] token-major as the projections write them; o [B, N, Hq, d].
 * Writes the last min(N, window) tokens' k, v into the ring and sets
 * ring->pos = N.  bf16 with d = 128 (tensor cores), else YOCO_ERR_UNSUPPORTED.
 * workspace: >= 256 bytes, 256-byte aligned (status word).
 */
YOCO_API yoco_status yoco_swa_prefill(const void *q, const void *k, const void *v, int Hq, int N, float scale,
                                      void *o, yoco_swa_ring *ring, void *workspace, size_t ws_bytes,
                                      void *stream);

/*
 * One generated token: q [B, Hq, d], k, v [B, Hkv, d] (the token's own), o
 * [B, Hq, d].  Writes k, v into slot ring->pos % window, attends over the
 * min(ring->pos + 1, window) filled slots, then increments ring->pos.
 * bf16 or f32, d in {64, 128}.  workspace: >= yoco_swa_workspace_size bytes.
 */
YOCO_API yoco_status yoco_swa_decode(const void *q, const void *k, const void *v, int Hq, float scale, void *o,
                                     yoco_swa_ring *ring, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes for yoco_swa_decode (also enough for yoco_swa_prefill). */
YOCO_API size_t yoco_swa_workspace_size(int B, int Hq, const yoco_swa_ring *ring);

/* ------------------------------------------------------------ utilities */

YOCO_API const char *yoco_status_string(yoco_status s);
YOCO_API const char *yoco_last_error(void);
YOCO_API int yoco_version(void);

/*
 * Status word of a workspace.  Kernels that wait on on-device signals give up
 * after a bounded time instead of hanging; they then record the failure in
 * the first bytes of the workspace they were given.  This call waits for
 * `stream`, reads that word and returns YOCO_OK or YOCO_ERR_TIMEOUT (the
 * detail is in yoco_last_error()); with clear != 0 it also resets the word.
 * A freshly allocated workspace needs no initialisation.
 */
YOCO_API yoco_status yoco_workspace_status(void *workspace, int clear, void *stream);

/*
 * Failure-path self-test: enqueues one kernel that waits on an on-device
 * barrier nothing ever completes, using the same bounded wait as the
 * tensor-core kernels; after limit_ns (<= 10 s) it gives up and records the
 * timeout in `workspace` (>= 256 bytes, 256-byte aligned).  A following
 * yoco_workspace_status returns YOCO_ERR_TIMEOUT and the CUDA context stays
 * usable.  Not part of the method; it exists so tests can exercise the
 * timeout path without faulting or hanging a GPU.
 */
YOCO_API yoco_status yoco_selftest_wait_timeout(void *workspace, uint64_t limit_ns, void *stream);

/*
 * Self-test for a shared device: enqueues `ctas` (<= 4 x the SM count) CTAs that
 * each claim 200 KB of shared memory, so that nothing needing much shared memory
 * fits beside them on their SM, and sleep for `ns` (<= 1 s) of wall time.  They
 * touch no global memory.  Tests run libyoco's calls on another stream meanwhile
 * to check that they make progress with part of the SMs taken.  Not part of the
 * method.
 */
YOCO_API yoco_status yoco_selftest_occupy_sms(int ctas, uint64_t ns, void *stream);

/* Number of kernels this process has enqueued through libyoco so far
 * (monotonic, all threads).  A diagnostic for counting launches per step. */
YOCO_API uint64_t yoco_launch_count(void);

/*
 * Test hooks: process-wide switches that let tests reach failure and ordering
 * paths that ordinary inputs cannot force.  Not part of the method; all are 0
 * (off) at load.  Returns YOCO_ERR_INVALID_ARG for an unknown hook or a value
 * out of range.
 *   YOCO_HOOK_FAIL_NEXT_CALLS     the next `value` (<= 1e6) calls that would
 *       launch a kernel instead return YOCO_ERR_CUDA ("unspecified launch
 *       failure" in yoco_last_error()) after their argument checks and before
 *       enqueuing anything, so nothing is written: a stand-in for a failed
 *       launch that faults no GPU.
 *   YOCO_HOOK_GRET_SEG0_DELAY_NS  with the tensor-core gRet prefill split into
 *       segments, segment 0 of every head takes the caller's initial state
 *       `value` ns (<= 1e9) late, so the last segment finishes first and its
 *       final state goes through the hand-off's parked path.  Results are
 *       unchanged; only timing moves.
 *   YOCO_HOOK_GRET_SEGMENTS  the tensor-core gRet prefill cuts each head into
 *       `value` (<= 4096, at most one per chunk) segments instead of about one
 *       CTA per SM; 0 restores the default.  Set it before querying the
 *       workspace size.  Results are unchanged up to rounding; for measuring
 *       the sequence-parallel split.
 */
/*
 * Index checks of a debug build.  Built with YOCO_DEBUG_CHECKS (build.py with
 * debug=True writes _build_debug/libyoco.so), every kernel checks the global
 * indices it forms from runtime values before using them; a failed check skips
 * the access and records 0x59434F00 | site, never a trap.  This call waits for
 * the device, stores the first recorded word (0: every check passed) in *word
 * and with clear != 0 resets it.  A release build returns YOCO_ERR_UNSUPPORTED.
 */
YOCO_API yoco_status yoco_debug_checks(int clear, uint32_t *word);

#define YOCO_HOOK_FAIL_NEXT_CALLS 1
#define YOCO_HOOK_GRET_SEG0_DELAY_NS 2
#define YOCO_HOOK_GRET_SEGMENTS 3
YOCO_API yoco_status yoco_test_hook(int hook, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* YOCO_H */
