/*
 * qbmoe — Stable LatentMoE forward with Quantile Balancing on one GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  "Device" pointers are CUDA device
 * (or managed) memory on the current device; "host" pointers are ordinary
 * host memory.  Every call that takes a stream is asynchronous and
 * stream-ordered on it (NULL = the legacy default stream); nothing here
 * synchronises the host except qbmoe_status and the functions documented as
 * synchronous.
 *
 * Errors.  Every call checks its arguments, encodes every tensor map and
 * sets up the device (kernel attributes, once per device) before its first
 * launch; a negative code from any of those steps means nothing was
 * launched and no output was touched.  Only QBMOE_ECUDA can also come from a
 * launch itself (the CUDA runtime refusing a launch or a copy); then the
 * launches that preceded it in the same call stay enqueued and the call's
 * outputs may be partly written.  Failures inside kernels are reported
 * later, by qbmoe_status.
 *
 * Sources, by page title and section:
 *   [K3-width]  "Kimi K3 模型结构（5）：宽度维度，Stable LatentMoE" (xhh.club),
 *               its 延伸解读 (extended reading) sections and its Q&A.
 *   [K3-explainer]  "KIMI K3" LatentMoE explainer (dimsnsums.com),
 *               "Why does the router need three moves?".
 */
#ifndef QBMOE_H
#define QBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Compatible with cudaStream_t. */
typedef struct CUstream_st* qbmoe_stream_t;

typedef enum {
    QBMOE_OK = 0,
    QBMOE_EINVAL = -1,     /* bad size, null or misaligned pointer, unsupported option */
    QBMOE_ENOMEM = -2,     /* device allocation failed (qbmoe_create, qbmoe_pack_weights) */
    QBMOE_ECUDA = -3,      /* a CUDA runtime/driver call or a launch failed */
    QBMOE_EARCH = -4,      /* current device is not compute capability 10.3 */
    QBMOE_EWORKSPACE = -5, /* caller workspace too small / ctx built for fewer tokens */
    QBMOE_ETIMEOUT = -6,   /* a kernel's bounded wait expired (reported by qbmoe_status) */
    QBMOE_EDEVICE = -7     /* a kernel's own check failed (reported by qbmoe_status) */
} qbmoe_status_t;

/* Storage types. */
enum { QBMOE_F32 = 0, QBMOE_BF16 = 1 };
/* Routed-expert weight formats. */
enum { QBMOE_W_F32 = 0, QBMOE_W_BF16 = 1, QBMOE_W_MXFP4 = 2 };
/* QB sweep forms: every expert from the same biases (the default, one
 * exchange of per-expert quantiles per sweep), or cyclic coordinate descent
 * (each expert's step sees the latest biases; moe_route_qb_gs). */
enum { QBMOE_QB_JACOBI = 0, QBMOE_QB_GAUSS_SEIDEL = 1 };

/* Limits of this build. */
#define QBMOE_MAX_EXPERTS 1024
#define QBMOE_MAX_TOPK 32

/*
 * Scores.  s = sigmoid(logit) is an exactly specified fp32 result: clamp the
 * logit to [-80, 80], y = -x, j = rint(y*0x1.715476p+0),
 * r = (y - j*0x1.62e4p-1) - j*0x1.7f7d1cp-20, p = degree-7 Taylor series of
 * e^r in Horner form (coefficients 1/5040, 1/720, 1/120, 1/24, 1/6 rounded to
 * fp32, then 1/2, 1, 1), e = p*2^j, s = 1/(1+e); every step one IEEE fp32
 * operation, no fused multiply-add.  ([K3-width] Q&A on routing: sigmoid
 * router on the full-width input.)
 */

/*
 * ---------------------------------------------------------------------------
 * moe_route_qb — router scores, Quantile Balancing, biased top-k.
 *
 * [K3-width] Q&A on Quantile Balancing: each expert's bias is the (1 - k/n)
 * quantile over tokens of its margin, minus a common offset, so that every
 * expert admits its target load T*k/n; 延伸解读 "QB vs DeepSeek-V3": one
 * exact coordinate-descent step on the balanced-assignment dual.  Q&A on
 * routing: top-k on score + bias, mixture weights = raw scores renormalised
 * over the chosen k, bias frozen at inference (qb_sweeps = 0).
 *
 * Per sweep (Jacobi: every expert from the same bias b):
 *   v = fl(s + b); per token the experts ranked by (v desc, index asc);
 *   tau[t][j] = the (k+1)-th ranked v if j is in the token's top k, else the
 *   k-th; m[t][j] = fl(s - tau) (-0 -> +0);
 *   r_j = floor(T*k/n) + (j < T*k mod n);  M = m[.][j] sorted descending;
 *   q_j = fl(fl(M_r + M_{r+1}) * 0.5)  (r=0: fl(M_1 + 1); r>=T: fl(M_T - 1));
 *   b'_j = -q_j;  c = fl(S / n), S = pairwise tree sum of b' padded with +0
 *   to 2^ceil(log2 n); b = fl(b' - c).
 * Final: idx[t] = top k of fl(s + b) in rank order; w[t][i] =
 * fl(s[idx_i] / sum), sum accumulated in rank order in fp32;
 * loads[j] = number of routes to j.
 *
 * T >= 1, 2 <= n <= QBMOE_MAX_EXPERTS, 1 <= k < n, k <= QBMOE_MAX_TOPK,
 * qb_sweeps >= 0.
 * logits   [T, n] fp32 device, row-major, pre-sigmoid.
 * bias_in  [n] fp32 device (NULL = zeros).  bias_out [n] fp32 device; may
 *          equal bias_in.
 * scores   [T, n] fp32 device out.  topk_idx [T, k] int32, topk_w [T, k]
 *          fp32, loads [n] int32 device out.
 * workspace: device, >= qbmoe_route_workspace_bytes(T, n, k) bytes, 256-byte
 *          aligned; owned by the caller; contents are scratch.
 * All device pointers 16-byte aligned.  Results are bit-reproducible.
 * Returns QBMOE_OK after enqueueing, or a negative code (see Errors above).
 */
size_t qbmoe_route_workspace_bytes(int T, int n, int k);
int moe_route_qb(int T, int n, int k, int qb_sweeps,
                 const float* logits, const float* bias_in, float* bias_out,
                 float* scores, int32_t* topk_idx, float* topk_w, int32_t* loads,
                 void* workspace, size_t workspace_bytes, qbmoe_stream_t stream);

/*
 * moe_route_qb_gs — Quantile Balancing by cyclic coordinate descent.
 *
 * [K3-width] 延伸解读 "QB vs DeepSeek-V3": QB solves the balanced-assignment
 * dual by coordinate descent, jumping to the exact coordinate minimiser.
 * This is the literal cyclic form: within a sweep the experts are updated in
 * order j = 0..n-1, each step computing expert j's margins under the latest
 * biases (tau[t][j] = k-th best fl(s + b) among the other experts) and
 * setting b_j = -midpoint of its r_j-th and (r_j+1)-th largest margins, as in
 * moe_route_qb; after the sweep the common offset is subtracted.  Repeated
 * sweeps never raise the dual; once every expert's load equals its target
 * the assignment is optimal for the balanced problem.
 *
 * max_sweeps >= 0 sweeps are run; with stop_when_balanced != 0 the sweeps
 * stop (on the device) after the first sweep whose loads equal the targets.
 * sweeps_done: device int32 or NULL, receives the number of sweeps run.
 * Other arguments as moe_route_qb; workspace >= qbmoe_route_gs_workspace_bytes.
 * Cost: about 2n + 5 kernel launches per sweep (a quality mode for balancing,
 * not the layer's hot path, which uses the one-pass Jacobi sweep).
 */
size_t qbmoe_route_gs_workspace_bytes(int T, int n, int k);
int moe_route_qb_gs(int T, int n, int k, int max_sweeps, int stop_when_balanced,
                    const float* logits, const float* bias_in, float* bias_out,
                    float* scores, int32_t* topk_idx, float* topk_w, int32_t* loads,
                    int32_t* sweeps_done, void* workspace, size_t workspace_bytes,
                    qbmoe_stream_t stream);

/*
 * moe_route_signsgd — DeepSeek-V3's fixed-step sign rule, the comparator of
 * Quantile Balancing.
 *
 * [K3-width] 延伸解读 "QB vs DeepSeek-V3": DeepSeek-V3 moves each expert's
 * bias by a fixed, hand-tuned step along a sign; that rule is SignSGD on the
 * same dual that QB minimises exactly.  From b = bias_in (NULL = zeros),
 * `steps` times: loads under the biased top-k of b, then
 *   b_j = fl(b_j - gamma) if load_j > r_j;  fl(b_j + gamma) if load_j < r_j;
 *   unchanged if load_j = r_j  (r_j as in moe_route_qb, no common offset).
 * Then the final routing on b as in moe_route_qb; bias_out = b.
 * steps >= 0, 0 < gamma < inf; other arguments as moe_route_qb, workspace
 * >= qbmoe_route_signsgd_workspace_bytes(T, n, k).  Bit-reproducible.
 */
size_t qbmoe_route_signsgd_workspace_bytes(int T, int n, int k);
int moe_route_signsgd(int T, int n, int k, int steps, float gamma,
                      const float* logits, const float* bias_in, float* bias_out,
                      float* scores, int32_t* topk_idx, float* topk_w, int32_t* loads,
                      void* workspace, size_t workspace_bytes, qbmoe_stream_t stream);

/*
 * Token-sharded Quantile Balancing with a histogram exchange.
 *
 * [K3-width] Q&A on Quantile Balancing: the quantiles are formed from
 * histogram estimates so that the communication stays cheap.  A batch of
 * T_total tokens is split into shards (on one or several devices); no shard
 * sees another's margins.  Each expert's coordinate step needs the r_j-th
 * and (r_j+1)-th largest margin over the whole batch (moe_route_qb).  Four
 * passes each exchange, per expert and per tracked rank, the 256-bin
 * histogram of one 8-bit digit of the margins' order keys among the keys
 * that match the digits fixed so far (n * 2 * 256 int32 per pass, against
 * T_total * n margins), and refine the estimate until both order
 * statistics are exact.  The bias is then bit-identical to moe_route_qb's
 * one-sweep bias of the whole batch, and each shard routes its tokens with
 * moe_route_qb(qb_sweeps = 0, bias_in = that bias).
 *
 * Per sweep:
 *   moe_qb_hist_init(T_total, n, k, state, hist)          targets, zeroed hist
 *   moe_qb_shard_margins(shard)                          each local shard
 *   for pass = 0..3:
 *     moe_qb_shard_hist(shard, pass, state, ws, hist)    each local shard ADDS
 *                                                        its counts into hist
 *     (the caller sums hist over devices: an all-reduce)
 *     moe_qb_hist_advance(n, pass, hist, state)          fixes the digit and
 *                                                        zeroes hist
 *   moe_qb_hist_bias(n, state, bias)                      b' and common offset
 *
 * state: device, qbmoe_qb_hist_state_bytes(n), caller-owned, one per device
 * (every device holds the same state after each advance).  hist: device
 * int32 [n][2][256] (qbmoe_qb_hist_bytes(n)).  Shard workspace: device,
 * qbmoe_qb_shard_workspace_bytes(T_shard, n, k), 256-byte aligned; holds the
 * shard's margins [n, T_shard] from moe_qb_shard_margins until its last
 * moe_qb_shard_hist.  moe_qb_shard_margins: logits [T_shard, n] fp32 in,
 * scores [T_shard, n] fp32 out, bias_in [n] or NULL (zeros) - the bias the
 * sweep starts from, the same on every shard.  T_total * k < 2^31.
 */
size_t qbmoe_qb_hist_state_bytes(int n);
size_t qbmoe_qb_hist_bytes(int n);
size_t qbmoe_qb_shard_workspace_bytes(int T_shard, int n, int k);
int moe_qb_hist_init(int T_total, int n, int k, void* state, int32_t* hist, qbmoe_stream_t stream);
int moe_qb_shard_margins(int T_shard, int n, int k, const float* logits, const float* bias_in, float* scores,
                         void* workspace, size_t workspace_bytes, qbmoe_stream_t stream);
int moe_qb_shard_hist(int T_shard, int n, int pass, const void* state, const void* workspace, int32_t* hist,
                      qbmoe_stream_t stream);
int moe_qb_hist_advance(int n, int pass, int32_t* hist, void* state, qbmoe_stream_t stream);
int moe_qb_hist_bias(int n, const void* state, float* bias_out, qbmoe_stream_t stream);

/*
 * moe_route_qb_noalloc — moe_route_qb for callers that cannot allocate.
 *
 * The pages have no counterpart: this is a deployment variant of the router
 * above with identical results, for callers that cannot hand it a workspace
 * because they may not allocate device memory where they route (a serving
 * path whose device memory is planned up front and may not grow, or a
 * plug-in that only receives its inputs and outputs from a host program
 * that owns all memory).  Arguments are those
 * of moe_route_qb without the workspace.  The scratch lives in one fixed
 * device array of qbmoe_route_noalloc_max_bytes() bytes (32 MiB) that every
 * GPU which loads the library keeps until the process exits; sizes whose
 * scratch (qbmoe_route_workspace_bytes(T, n, k)) exceeds it are refused with
 * QBMOE_EWORKSPACE before anything is launched.  The call makes no cudaMalloc
 * or cudaFree and calls no allocating library routine.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress) and sets the library's kernel attributes
 * there; make that first call before any stream capture.  All calls share
 * the one array, so calls that may overlap on the GPU (different streams, or
 * different host threads on one device) race and must be serialised by the
 * caller.  Nothing needs to start at zero: every
 * scratch region is written before it is read.
 */
size_t qbmoe_route_noalloc_max_bytes(void);
int moe_route_qb_noalloc(int T, int n, int k, int qb_sweeps,
                         const float* logits, const float* bias_in, float* bias_out,
                         float* scores, int32_t* topk_idx, float* topk_w, int32_t* loads,
                         qbmoe_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * Layer context.
 */
typedef struct {
    int d;              /* model width */
    int latent;         /* latent width ([K3-width] 延伸解读: 7168 -> 3584) */
    int n_experts;      /* routed experts */
    int top_k;          /* experts per token */
    int expert_inter;   /* routed expert GLU intermediate */
    int shared_inter;   /* merged shared-expert intermediate; 0 = no shared expert */
    float situ_beta1;   /* gate softcap, 4 on the pages */
    float situ_beta2;   /* up softcap, 25 on the pages */
    float rms_eps;      /* RMSNorm epsilon */
    int act_dtype;      /* QBMOE_F32 | QBMOE_BF16: activations and dense weights */
    int expert_wfmt;    /* QBMOE_W_F32 | QBMOE_W_BF16 | QBMOE_W_MXFP4 */
    int qb_sweeps;      /* 0 = frozen bias (inference); 1 = one QB step */
    int qb_mode;        /* QBMOE_QB_JACOBI (default) | QBMOE_QB_GAUSS_SEIDEL */
} qbmoe_config;

/*
 * Weights: device pointers in canonical K-major layouts ("[rows, K]", K
 * contiguous), typed by act_dtype unless stated.  The caller owns them and
 * must keep them alive and unchanged while the context uses them (the
 * context keeps pointers, not copies).
 *   w_router [n, d]; router_offset [n] fp32 or NULL (per-expert logit offset)
 *   w_down [latent, d]
 *   w_gate, w_up [n, m, latent]; w_out [n, latent, m]    (expert_wfmt)
 *     MXFP4: values packed two per byte (element 2i in the low nibble) as
 *     [rows, K/2] u8 with 32-byte aligned bases, scales E8M0 [rows, K/32]
 *     u8 in s_gate/s_up/s_out (tensor-core path: K a multiple of 512).
 *   rms_gamma [latent] fp32
 *   w_proj_up [d, latent]
 *   w_shared_gate, w_shared_up [m_s, d]; w_shared_out [d, m_s]  (m_s > 0)
 */
typedef struct {
    const void* w_router;
    const float* router_offset;
    const void* w_down;
    const void* w_gate;
    const void* w_up;
    const void* w_out;
    const uint8_t* s_gate;
    const uint8_t* s_up;
    const uint8_t* s_out;
    const float* rms_gamma;
    const void* w_proj_up;
    const void* w_shared_gate;
    const void* w_shared_up;
    const void* w_shared_out;
} qbmoe_weights;

typedef struct qbmoe_ctx qbmoe_ctx;

/* Validate cfg, allocate the context's device workspace for up to max_tokens
 * tokens on the current device (synchronous).  *out = NULL on failure. */
int qbmoe_create(qbmoe_ctx** out, const qbmoe_config* cfg, int max_tokens);
/* Bytes of device workspace qbmoe_create allocates for these sizes. */
size_t qbmoe_layer_workspace_bytes(const qbmoe_config* cfg, int max_tokens);
/* Record the weight pointers (host call, no device work, no copies). */
int qbmoe_set_weights(qbmoe_ctx* ctx, const qbmoe_weights* w);
/* Copy the weights into device memory the context owns, then use the
 * copies (as qbmoe_set_weights on them).  w holds device pointers in the
 * layouts above; the caller may free or change its tensors once the call
 * returns.  Synchronous: enqueues the copies and a check of every MXFP4
 * scale byte on `stream`, then waits for them.  A scale byte of 0xFF (E8M0
 * NaN, not a weight scale) gives QBMOE_EINVAL and leaves the context's
 * weights as they were.  Allocates one buffer (cudaMalloc; QBMOE_ENOMEM on
 * failure); a later call replaces it, qbmoe_destroy frees it.  Nothing else
 * in the forward path allocates. */
int qbmoe_pack_weights(qbmoe_ctx* ctx, const qbmoe_weights* w, qbmoe_stream_t stream);
/* Free the context's workspace (synchronous). NULL is a no-op. */
int qbmoe_destroy(qbmoe_ctx* ctx);

/*
 * moe_latent_forward — one Stable LatentMoE layer forward for T tokens.
 *
 *   scores = sigmoid(x W_r^T + o) (or of logits_in when given)   [K3-width] Q&A routing
 *   b, idx, w, loads as moe_route_qb
 *   h   = round(x W_down^T)                                       [K3-width] 延伸解读 latent
 *   act = round(SiTU-GLU(h W_g[e]^T, h W_u[e]^T)) per route       [K3-width] Q&A SiTU-GLU
 *         SiTU-GLU(g, u) = a*sigmoid(a)*b, a = b1*tanh(g/b1), b = b2*tanh(u/b2)
 *   e   = round(act W_o[e]^T)
 *   z   = round(RMSNorm(sum_i w_i e_i) * gamma)                   [K3-width] Q&A RMSNorm
 *   out = round(z W_proj_up^T + act_s W_shared_out^T),
 *         act_s = round(SiTU-GLU(x W_shared_gate^T, x W_shared_up^T))   Q&A shared expert
 * ("round" = to act_dtype; accumulation is fp32.  With bf16 activations the
 * tensor-core SiTU epilogues use the hardware tanh approximation, relative
 * error about 2^-11, below the bf16 rounding.  MXFP4 experts run on the
 * block-scaled MMA: each block of 32 bf16 activations along K gets an E8M0
 * scale 2^e, e = floor(log2 max|a|) - 7, and each scaled value c = a 2^-e
 * (|c| < 256) enters as e4m3(c) + e4m3(16 (c - e4m3(c))) / 16, which is
 * exact for 2^-6 <= |c| < 256; nothing saturates.)
 *
 * x [T, d] act_dtype device; out [T, d] act_dtype device.
 * logits_in: NULL, or [T, n] fp32 device router logits used instead of the
 *   router GEMM (x W_r^T + o is then not computed).
 * bias_in [n] fp32 device or NULL (zeros); bias_out [n] fp32 device (may
 *   alias bias_in) or NULL.
 * scores_opt [T, n] fp32, idx_opt [T, k] int32, w_opt [T, k] fp32,
 *   loads_opt [n] int32: device outputs, each NULL if not wanted.
 * 1 <= T <= max_tokens.  No allocation, no host synchronisation.
 * With qb_mode = QBMOE_QB_GAUSS_SEIDEL the qb_sweeps sweeps are cyclic, as
 * moe_route_qb_gs (about 2n launches per sweep).
 */
int moe_latent_forward(qbmoe_ctx* ctx, int T, const void* x, const float* logits_in,
                       const float* bias_in, float* bias_out, void* out,
                       float* scores_opt, int32_t* idx_opt, float* w_opt, int32_t* loads_opt,
                       qbmoe_stream_t stream);

/*
 * Synchronise `stream`, then return and clear the context's device status
 * word: QBMOE_OK, QBMOE_ETIMEOUT (a bounded wait expired; the kernel
 * returned early and its outputs are undefined) or QBMOE_EDEVICE.
 * ctx may be NULL (then only the stream's CUDA error state is checked).
 */
int qbmoe_status(qbmoe_ctx* ctx, qbmoe_stream_t stream);

/*
 * Stage timing.  qbmoe_set_timing(ctx, slots) (synchronous) keeps CUDA events
 * around each stage of the next `slots` forwards (a ring; 0 = off, at most
 * 4096) on the forward's stream, without synchronising.  qbmoe_stage_times
 * (synchronous) writes each stage's mean milliseconds over the recorded
 * forwards still in the ring into ms[0..max-1] and the stages' names (static
 * strings) into names (may be NULL); returns the number of stages, 0 if none.
 */
int qbmoe_set_timing(qbmoe_ctx* ctx, int slots);
int qbmoe_stage_times(qbmoe_ctx* ctx, float* ms, const char** names, int max);

/* Number of kernels the last moe_latent_forward / moe_route_qb call launched. */
int qbmoe_last_launch_count(qbmoe_ctx* ctx);
int qbmoe_route_last_launch_count(void);

/* Test hook: cap on bounded device waits, in polls of at most 20 us each
 * (<= 0 restores the default of 2^17).  Applies to launches made after the
 * call. */
int qbmoe_set_wait_limit(qbmoe_ctx* ctx, long long iterations);

/* Test hook: while enabled, the tensor-core GEMM kernels withhold their first
 * accumulator hand-off, so the epilogue's bounded wait expires and the next
 * qbmoe_status reports QBMOE_ETIMEOUT (outputs undefined).  The kernels then
 * drain their own copies and MMAs, free TMEM and return; the context stays
 * usable.  No effect when the layer runs on CUDA cores. */
int qbmoe_debug_stall(qbmoe_ctx* ctx, int enable);

/* 1 when the context's bf16 GEMMs run on the tcgen05 tensor-core kernels, 0
 * when they run on the CUDA-core kernels (fp32 layers, shapes the tensor-core
 * tiling does not cover, or QBMOE_DISABLE_TC=1 in the environment at
 * qbmoe_create). */
int qbmoe_uses_tensor_cores(qbmoe_ctx* ctx);

/*
 * Tensor-core rate probe (synchronous; a measurement hook, not part of the
 * layer).  Runs one CTA per SM that issues 4 * iters back-to-back MMAs of
 * the given kind on fixed shared-memory tiles (M = 128, N = 256; no TMA, no
 * epilogue) between two CUDA events on the legacy default stream.  Kinds:
 * QBMOE_PROBE_BF16 (kind::f16, bf16 x bf16, K = 16 per MMA) and
 * QBMOE_PROBE_MXF4F8 (kind::mxf8f6f4 block-scaled, E2M1 x E4M3 with E8M0
 * scales, K = 32 per MMA: the MXFP4 expert GEMMs' instruction).  Writes the
 * elapsed milliseconds and the flops issued (2 * M * N * K per MMA).
 * Allocates a 4-byte status word (cudaMalloc) for its bounded wait.
 */
enum { QBMOE_PROBE_BF16 = 0, QBMOE_PROBE_MXF4F8 = 1 };
int qbmoe_mma_probe(int kind, int iters, float* ms_out, double* flops_out);

const char* qbmoe_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* QBMOE_H */
