/*
 * fgm.h - C ABI of the GB300 batch-1 fine-grained MoE verify-step library.
 *
 * The library runs the memory-bound decode/verify step of speculative
 * decoding on a Gemma-4-26B-A4B-shaped mixture of experts: hidden width 2816,
 * 128 routed experts of FFN width 704 plus one always-on shared expert,
 * top-8 routing, FP8-E4M3 expert weights with one fp32 scale per output row,
 * and a tied 262,144-word bf16 lm_head (or its E4M3 copy with one fp32 scale
 * per row, fgm_lm_head_argmax_fp8). One call processes M = gamma + 1
 * tokens (the real token and gamma drafted ones) in a single pass over the
 * weights ("llm-decoding", us-homepage.pages.dev, §"Lever 2: fewer passes
 * (native MTP)": the full model verifies the drafted tokens in one pass).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, unless an
 *    entry point says otherwise. The library never frees them and keeps no
 *    reference after the call returns.
 *  - Row-major layouts; bf16 is passed as raw 16-bit patterns (uint16_t).
 *  - Weight pointers and activation pointers must be 16-byte aligned.
 *  - `ws` is caller-allocated device scratch of at least
 *    fgm_workspace_bytes(M, V) bytes, 256-byte aligned; the library uses it
 *    only during the call (calls that share a workspace must not overlap).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on that stream except where stated.
 *  - Return value: FGM_OK (0) or a negative FGM_ERR_* code; arguments are
 *    validated on the host before anything is launched, so an error return
 *    means nothing was enqueued, except FGM_ERR_CUDA from a failed launch.
 *    fgm_last_error() gives a message for the calling thread.
 *  - Kernels never trap. Anomalies they detect (non-finite router logits,
 *    a timed-out wait) set bits of a status word in the workspace, read
 *    with fgm_read_status().
 */
#ifndef FGM_H
#define FGM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Model shape ("llm-decoding", §"The exact architecture"). */
#define FGM_HIDDEN 2816     /* hidden width */
#define FGM_FFN 704         /* expert FFN width */
#define FGM_EXPERTS 128     /* routed experts */
#define FGM_SHARED 1        /* always-on shared experts, stored after the routed ones */
#define FGM_TOPK 8          /* routed experts per token */
#define FGM_MAX_M 8         /* tokens per call: 1 real + up to 7 drafted */
#define FGM_MAX_LAYERS 48   /* layers per stack call */
#define FGM_RMS_EPS 1e-6f   /* RMSNorm epsilon of the stack */

enum {
    FGM_OK = 0,
    FGM_ERR_INVALID_ARG = -1, /* null/misaligned pointer, M or V out of range */
    FGM_ERR_WORKSPACE = -2,   /* workspace missing, misaligned or too small */
    FGM_ERR_CUDA = -3,        /* a CUDA runtime call failed; see fgm_last_error() */
    FGM_ERR_DEVICE = -4,      /* the current device is not a supported GPU (sm_103) */
};

/* Execution paths (fgm_select_path). */
enum {
    FGM_PATH_FUSED = 0,  /* default: one persistent cooperative kernel per call; weight rows stream
                            through a TMA-bulk shared-memory ring into FP8/bf16 mma.sync tiles, and
                            at M <= 5 the down products (routed experts and the shared expert or
                            the dense MLP's parts) run on tcgen05.mma (TMA tensor copies,
                            tensor-memory accumulators) */
    FGM_PATH_STAGED = 1, /* one launch per stage with fp32 CUDA-core arithmetic (comparison path) */
    FGM_PATH_FUSED_TC = 2, /* as FGM_PATH_FUSED, with the FP8 lm_head on tcgen05.mma as well */
    FGM_PATH_FUSED_MMA = 3, /* as FGM_PATH_FUSED, with the down products on mma.sync at every M
                               (comparison path) */
};

/* Status bits written by kernels into the workspace (fgm_read_status). */
enum {
    FGM_STATUS_NONFINITE_LOGITS = 1, /* a router or lm_head logit was NaN; treated as -inf */
    FGM_STATUS_WAIT_TIMEOUT = 2,     /* a grid-wide wait gave up; outputs are invalid */
};

/* One MoE layer's weights (all device pointers).
 *  router_w  bf16 [128][2816]         router logits l = router_w . x + router_b
 *  router_b  fp32 [128] or NULL       additive logit bias
 *  gate_q    E4M3 [129][704][2816]    expert e's gate rows (e = 128: shared)
 *  gate_s    fp32 [129][704]          per-row scales: W = e4m3(q) * s
 *  up_q      E4M3 [129][704][2816]
 *  up_s      fp32 [129][704]
 *  down_q    E4M3 [129][2816][704]
 *  down_s    fp32 [129][2816]
 * Weights follow "llm-decoding" §"Where the 7.36 GB goes" (gate, up and down
 * of 2816x704 per expert) and §"Lever 1" (8-bit weights, dequantised at
 * higher precision). */
typedef struct fgm_layer {
    const uint16_t *router_w;
    const float *router_b;
    const uint8_t *gate_q;
    const float *gate_s;
    const uint8_t *up_q;
    const float *up_s;
    const uint8_t *down_q;
    const float *down_s;
} fgm_layer;

/* An always-on dense (shared) gated-GELU MLP of width W, E4M3 weights with
 * one fp32 scale per output row (the experts' format):
 *   mlp(x) = s_d (Q_d (gelu_tanh(s_g (Q_g x)) * s_u (Q_u x))). */
typedef struct fgm_mlp {
    const uint8_t *gate_q;  /* E4M3 [W][2816], 16-byte aligned */
    const float *gate_s;    /* [W] */
    const uint8_t *up_q;    /* E4M3 [W][2816] */
    const float *up_s;      /* [W] */
    const uint8_t *down_q;  /* E4M3 [2816][W] (row stride W bytes) */
    const float *down_s;    /* [2816] */
    int width;              /* W: a multiple of 704, at most 2112 */
} fgm_mlp;

/* Bytes of scratch an M-token call needs; V is the vocabulary size for the
 * lm_head entry points (0 if unused). Never fails; 0 for M out of range. */
size_t fgm_workspace_bytes(int M, int64_t V);

/* Zeroes a workspace (status word and wait counters included). Call once
 * after allocating it, before its first use by any other entry point. */
int fgm_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* One MoE FFN layer (no norm, no residual) on M tokens:
 *   y_t = sum_{i<8} w_{t,i} * expert_{id_{t,i}}(x_t) + expert_128(x_t),
 *   expert_e(x) = s_d (Q_d (gelu_tanh(s_g (Q_g x)) * s_u (Q_u x))),
 * with ids/w from the router: softmax over the 128 biased logits, top-8
 * (ties to the lower index), renormalised to sum to 1. Accumulation is fp32.
 * Source: "llm-decoding" §"The exact architecture" (top 8 of 128 + one shared).
 *  x         bf16 [M][2816] input
 *  y         bf16 [M][2816] output (may not alias x)
 *  topk_ids  int32 [M][8] or NULL: chosen expert ids, descending weight
 *  topk_w    fp32 [M][8] or NULL: their renormalised weights */
int fgm_moe_layer_fwd(const fgm_layer *layer, const uint16_t *x, uint16_t *y, int M,
                      int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream);

/* fgm_moe_layer_fwd without a caller workspace, for callers that may not
 * allocate device memory while they run: a serving loop whose memory pool is
 * already handed out to weights and caches, a host framework that owns every
 * allocation and forbids them inside its per-step hook, or latency-critical
 * code where a cudaMalloc/cudaFree could stall on a device-wide
 * synchronisation. The operation is the same as fgm_moe_layer_fwd (same
 * arguments, same results); the pages describe no such variant, it is an
 * interface convenience only.
 *  - Scratch: a fixed device array inside the library (4 MiB, enough for
 *    M <= FGM_MAX_M = 8 tokens), reserved when the library's CUDA module is
 *    loaded. The call allocates nothing; M outside [1, 8] returns
 *    FGM_ERR_INVALID_ARG with a message naming the limit.
 *  - Set-up: the first call on each device, with that device current, looks
 *    up the array's device address (the CUDA runtime may load the module
 *    then). Make that first call before any stream capture begins. The
 *    address is kept for the life of the process: after cudaDeviceReset (or
 *    any other teardown of the device's primary context) in the same process
 *    it is stale, so do not call this entry point again in that process.
 *    The per-device set-up of every other entry point (the device check and
 *    kernel attributes) has the same lifetime.
 *  - Each call clears the array's status word and barrier counters on
 *    `stream` before it launches.
 *  - One array per device serves every caller on it: calls on that device
 *    whose GPU work overlaps (other streams, other threads) race on the
 *    scratch and give wrong results. Order them on one stream, or use
 *    fgm_moe_layer_fwd with one workspace per stream.
 *  - The status word cannot be read back (it lives in the library's array);
 *    use fgm_moe_layer_fwd when the status must be checked. */
int fgm_moe_layer_fwd_noalloc(const fgm_layer *layer, const uint16_t *x, uint16_t *y, int M,
                              int32_t *topk_ids, float *topk_w, void *stream);

/* fgm_moe_layer_fwd with an always-on dense MLP of width W in place of the
 * shared expert (the layer's expert 128 is not read):
 *   y_t = sum_{i<8} w_{t,i} * expert_{id_{t,i}}(x_t) + mlp(x_t).
 * A GeGLU MLP splits exactly into W/704 column blocks of width 704 whose
 * outputs add up (each down row keeps its full-width scale), so the kernels
 * run it as W/704 always-on parts of weight 1 next to the routed experts.
 * Source: "llm-decoding" §"Where the 7.36 GB goes" (an always-on dense MLP of
 * 2816 x 2112 per layer). On the fused paths a 2112-wide MLP runs in the
 * persistent kernel, its three parts taking the shared expert's place in the
 * always-on schedule; other widths, and the staged path, use the per-stage
 * kernels.
 *  dense   HOST pointer to the MLP's device weights (see fgm_mlp)
 *  other arguments as fgm_moe_layer_fwd */
int fgm_moe_layer_dense_fwd(const fgm_layer *layer, const fgm_mlp *dense, const uint16_t *x, uint16_t *y, int M,
                            int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream);

/* n_layers stacked layers (attention omitted), each
 *   h <- h + moe_layer(RMSNorm(h)),  RMSNorm(h) = h / sqrt(mean(h^2) + 1e-6),
 * starting from h = x; the residual stream stays fp32 inside the call.
 *  layers     HOST array of n_layers fgm_layer (1 <= n_layers <= 48)
 *  x          bf16 [M][2816] input hidden states
 *  y          bf16 [M][2816] output: the final residual stream h (no norm)
 *  ids_trace  int32 [n_layers][M][8] or NULL: routing of every layer */
int fgm_moe_stack_fwd(const fgm_layer *layers, int n_layers, const uint16_t *x, uint16_t *y,
                      int M, int32_t *ids_trace, void *ws, size_t ws_bytes, void *stream);

/* The stack with an always-on dense MLP in every layer in place of the
 * shared expert (layer l: h <- h + moe_layer_dense(RMSNorm(h)) with MLP
 * mlps[l], as fgm_moe_layer_dense_fwd): the model whose byte list has a
 * 2816 x 2112 dense MLP per layer ("llm-decoding" §"Where the 7.36 GB goes").
 * When every MLP is 2112 wide the fused paths run it in the persistent
 * kernel (the MLP's three parts as its always-on slots); otherwise, and on
 * the staged path, the per-stage kernels.
 *  mlps   HOST array of n_layers fgm_mlp (device weights)
 *  other arguments as fgm_moe_stack_fwd */
int fgm_moe_stack_dense_fwd(const fgm_layer *layers, const fgm_mlp *mlps, int n_layers, const uint16_t *x,
                            uint16_t *y, int M, int32_t *ids_trace, void *ws, size_t ws_bytes, void *stream);

/* Tied lm_head fused with argmax: z_{t,v} = sum_j emb[v][j] * h[t][j]
 * (fp32 accumulation), argmax over v with ties to the lower index.
 * Source: "llm-decoding" §"The exact architecture" (262,144-word tied
 * lm_head) and §"Where the 7.36 GB goes" (read once per step).
 *  emb       bf16 [V][2816], 1 <= V < 2^31
 *  h         bf16 [M][2816] final hidden states
 *  argmax    int32 [M] output
 *  maxlogit  fp32 [M] or NULL: the winning logit */
int fgm_lm_head_argmax(const uint16_t *emb, int64_t V, const uint16_t *h, int M, int32_t *argmax,
                       float *maxlogit, void *ws, size_t ws_bytes, void *stream);

/* FP8 lm_head fused with argmax: the tied embedding stored as E4M3 codes with
 * one fp32 scale per row (the expert weights' format),
 *   z_{t,v} = emb_s[v] * sum_j e4m3(emb_q[v][j]) * h[t][j]
 * (fp32 accumulation), argmax over v with ties to the lower index. Half the
 * bytes of fgm_lm_head_argmax. Source: "llm-decoding" §"Lever 1: fewer bytes
 * (FP8 weights)" (every weight stored in 8 bits) and §"First principles:
 * compute-bound or memory-bound?" (the BF16 lm_head is a fifth of the bytes).
 *  emb_q     uint8 [V][2816] E4M3 codes (16-byte aligned), 1 <= V < 2^31
 *  emb_s     fp32 [V] row scales (4-byte aligned)
 *  h         bf16 [M][2816] final hidden states (16-byte aligned)
 *  argmax    int32 [M] output
 *  maxlogit  fp32 [M] or NULL: the winning logit
 * A row holding the NaN code gives NaN logits, which never win; if every
 * logit of a token is NaN its argmax is 0 and FGM_STATUS_NONFINITE_LOGITS is
 * raised. One launch: its CTAs count themselves done in the workspace (a
 * word fgm_workspace_init zeroes and the call leaves at zero), and the last
 * one reduces the per-CTA partials. */
int fgm_lm_head_argmax_fp8(const uint8_t *emb_q, const float *emb_s, int64_t V, const uint16_t *h, int M,
                           int32_t *argmax, float *maxlogit, void *ws, size_t ws_bytes, void *stream);

/* Greedy acceptance of gamma = M - 1 drafted tokens: a = largest j <= gamma
 * with draft[0..j-1] == target[0..j-1]; out = {a, target[a]} (the accepted
 * count and the token emitted after the accepted drafts). Source:
 * "llm-decoding" §"Lever 2" (keep the tokens the model would have produced)
 * and §"What we learned" (identical output to ordinary decoding).
 *  target  int32 [M] argmax tokens at the M positions (device)
 *  draft   int32 [M-1] drafted tokens d_1..d_gamma (device; unused if M == 1)
 *  out     int32 [2] (device) */
int fgm_spec_verify(const int32_t *target, const int32_t *draft, int M, int32_t *out,
                    void *stream);

/* One full verify step: the n_layers stack from x, a final unit RMSNorm
 * rounded to bf16, the lm_head argmax, and greedy acceptance of the drafts.
 *  layers   HOST array of n_layers fgm_layer
 *  emb      bf16 [V][2816]
 *  x        bf16 [M][2816]
 *  draft    int32 [M-1] (device; may be NULL when M == 1)
 *  argmax   int32 [M] output (device) or NULL
 *  out      int32 [2] output {accepted, next} (device) */
int fgm_verify_step(const fgm_layer *layers, int n_layers, const uint16_t *emb, int64_t V,
                    const uint16_t *x, const int32_t *draft, int M, int32_t *argmax, int32_t *out,
                    void *ws, size_t ws_bytes, void *stream);

/* fgm_verify_step on the stack with a dense MLP per layer (see
 * fgm_moe_stack_dense_fwd); mlps is a HOST array of n_layers fgm_mlp. */
int fgm_verify_step_dense(const fgm_layer *layers, const fgm_mlp *mlps, int n_layers, const uint16_t *emb,
                          int64_t V, const uint16_t *x, const int32_t *draft, int M, int32_t *argmax, int32_t *out,
                          void *ws, size_t ws_bytes, void *stream);

/* fgm_verify_step with the FP8 lm_head of fgm_lm_head_argmax_fp8 in place of
 * the bf16 one (same stack, final norm and acceptance). Two launches: the
 * stack, then the FP8 lm_head, which applies the final norm to the fp32
 * residual stream itself and ends with the acceptance.
 *  emb_q    uint8 [V][2816] E4M3 codes;  emb_s  fp32 [V] row scales
 *  other arguments as fgm_verify_step */
int fgm_verify_step_fp8_head(const fgm_layer *layers, int n_layers, const uint8_t *emb_q, const float *emb_s,
                             int64_t V, const uint16_t *x, const int32_t *draft, int M, int32_t *argmax,
                             int32_t *out, void *ws, size_t ws_bytes, void *stream);

/* fgm_verify_step with HOST input and output buffers: copies x_host
 * (bf16 [M][2816]) and draft_host (int32 [M-1]) into the workspace, runs the
 * step, copies {accepted, next} into out_host (int32 [2]) and synchronises
 * the stream before returning. Host buffers should be pinned for speed. */
int fgm_verify_step_host(const fgm_layer *layers, int n_layers, const uint16_t *emb, int64_t V,
                         const uint16_t *x_host, const int32_t *draft_host, int M,
                         int32_t *out_host, void *ws, size_t ws_bytes, void *stream);

/* Speculative sampling verify at temperature T > 0, on the tied lm_head
 * logits z_{t,v} = sum_j emb[v][j] * h[t][j] (fp32 accumulation) of M
 * positions and gamma = M - 1 drafted tokens. With p_t = softmax(z_t / T):
 * for t = 0 .. M-2 draft d_t is accepted while u_acc[t] < p_t(d_t); at the
 * first rejected position t the emitted token is the inverse-CDF sample, in
 * vocabulary order, of p_t with d_t removed (renormalised) at u_next[t]; if
 * every draft is accepted, position M-1 emits the sample of p_{M-1} at
 * u_next[M-1]. out = {accepted drafts, emitted token}. The drafter proposes
 * tokens only (its proposal is one-hot), so the emitted sequence has the
 * distribution of ordinary sampling from p. Source: "llm-decoding" §"What we
 * learned, and where this goes" (a kept token passes the full model's
 * distribution, a rejected one falls back to a real model step, the output
 * distribution is unchanged). Decisions within fp32 rounding of a boundary
 * (|u_acc[t] - p_t(d_t)|, or u_next at a partial sum of the CDF) may go
 * either way. As T -> 0 this is greedy acceptance (fgm_lm_head_argmax +
 * fgm_spec_verify).
 *  emb     bf16 [V][2816], 1 <= V < 2^31 (16-byte aligned)
 *  h       bf16 [M][2816] final hidden states (16-byte aligned)
 *  T       temperature: finite, > 0, and 1/T finite
 *  draft   int32 [M-1] (device; may be NULL when M == 1); a draft outside
 *          [0, V) has probability 0 (rejected, nothing removed)
 *  u_acc   fp32 [M-1] uniforms in [0, 1) (device; may be NULL when M == 1)
 *  u_next  fp32 [M] uniforms in [0, 1) (device)
 *  z       fp32 [M][V] output: the logits (device, 4-byte aligned, caller-owned)
 *  argmax  int32 [M] output or NULL: the greedy argmax of every position
 *  out     int32 [2] output (device)
 * Runs on the persistent kernel whatever fgm_select_path chose; its last CTA
 * takes the decisions. */
int fgm_lm_head_sample(const uint16_t *emb, int64_t V, const uint16_t *h, int M, float T, const int32_t *draft,
                       const float *u_acc, const float *u_next, float *z, int32_t *argmax, int32_t *out,
                       void *ws, size_t ws_bytes, void *stream);

/* One full verify step with speculative sampling at temperature T: the
 * n_layers stack from x, the final unit RMSNorm rounded to bf16, then
 * fgm_lm_head_sample on those rows. One launch of the persistent kernel.
 *  layers  HOST array of n_layers fgm_layer;  x  bf16 [M][2816]
 *  other arguments as fgm_lm_head_sample */
int fgm_verify_step_sample(const fgm_layer *layers, int n_layers, const uint16_t *emb, int64_t V,
                           const uint16_t *x, const int32_t *draft, int M, float T, const float *u_acc,
                           const float *u_next, float *z, int32_t *argmax, int32_t *out, void *ws,
                           size_t ws_bytes, void *stream);

/* Selects the execution path of subsequent calls in this process; returns the
 * previous one. An unknown value leaves the path unchanged. Both paths compute
 * the same step; they differ in kernel design only. */
int fgm_select_path(int path);

/* Upper bound, in ns of GPU time, on every wait inside the persistent kernel
 * (grid barriers, ring slots). When a wait runs out the kernel raises
 * FGM_STATUS_WAIT_TIMEOUT, skips its remaining work and exits; its outputs are
 * then invalid. Default 2 s; ns < 0 only queries. Returns the previous value. */
long long fgm_set_wait_limit_ns(long long ns);

/* Profiling aid: when buf (DEVICE, n int64 entries) is non-NULL, each later
 * persistent-kernel launch records %globaltimer stamps (ns). Per CTA at the
 * phase boundaries of layer l: entry [(l * 12 + k) * G + cta] with k = 0 layer
 * start, 1 norm/router partials ready, 2 after their reduction, 3 activation
 * terms ready, 4 shared gate/up done, 5 after barrier 1, 10 top-k done,
 * 11 expert list done, 6 routing known, 7 routed gate/up done, 8 start of
 * the down rows, 9 down done; then [(L*12) * G + cta] after the last layer
 * and [(L*12 + 1) * G + cta] at the end (G = CTAs, one
 * per SM). Then, for CTA G/2 only, [L][48][8] SM clock64 values per ring stage
 * of each layer: producer issue, data landed (consumer wait over), products
 * done, slot released, last exchange of the stage posted, consumer wait
 * begun, unused, and (stage 0 only) the layer start. A buffer
 * shorter than (L*12 + 2) * G + L*48*8 entries disables recording. NULL stops. */
int fgm_set_phase_trace(long long *buf, size_t n);

/* Test hook for failure detection: the next persistent-kernel launch adds one
 * grid barrier that can never complete, so its bounded wait must run out,
 * raise FGM_STATUS_WAIT_TIMEOUT and let the kernel exit (outputs invalid). */
int fgm_debug_stall_next_launch(void);

/* The same at the start of the given layer of the next persistent-kernel
 * launch (layers before it run normally, their down-tile counters and
 * activation markers left as an interrupted call leaves them). */
int fgm_debug_stall_next_launch_at(int layer);

/* Reads the status word of a workspace (synchronises the stream) and, if
 * `clear`, resets it. */
int fgm_read_status(void *ws, size_t ws_bytes, int clear, int32_t *status, void *stream);

/* After FGM_STATUS_WAIT_TIMEOUT: where the first wait gave up, as 4 int32
 * (HOST report): {site, block, warp, index}; site 1 = ring slot free
 * (producer), 2 = routing known (producer), 3 = ring data landed, 6 = grid
 * barrier (warp = counter value, index = target), 7 = activation rows of an
 * expert written (index = its slot); the tcgen05 down phase: 8 =
 * accumulator read, 10 = accumulator full, 11 = activation rows written
 * (index = slot), 12 = second home slot's operand built (9 is no longer
 * reported). When every CTA stops at a grid barrier, the first report may
 * come from the barrier (6) or from a producer waiting for the routing that
 * the barrier holds back (2). Synchronises the stream. */
int fgm_read_wait_report(void *ws, size_t ws_bytes, int32_t *report, void *stream);

/* Message describing the last error returned on the calling thread. */
const char *fgm_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int fgm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FGM_H */
