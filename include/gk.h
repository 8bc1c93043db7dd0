/*
 * gk.h — C ABI of libgk: the forward, reverse-mode backward, AdamW update and KV-cache decode
 * of a GPT-2-style decoder step, as hand-written CUDA kernels for one GB300 (sm_103a).
 *
 * Sources cited below (page title, then section):
 *   [LM1] arabroot.io, "Build a language model in C# from scratch (1): the Autograd engine".
 *   [LM4] arabroot.io, "Build a language model in C# from scratch (4): running GPT-2 weights".
 *
 * Conventions shared by every entry point
 *   - Tensors are row-major. A Linear weight is stored [in, out] ([LM4] "Loading weights into
 *     our classes": the Conv1D layout, no transpose). `ld*` arguments are row strides in
 *     elements (>= the row length), so padded rows (e.g. a vocabulary of 50257 stored with a
 *     stride of 50304) are allowed.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; libgk never frees it.
 *     Host pointers are named as such (`gk_param` arrays, `gk_gpt_cfg`, `gk_sample_cfg`).
 *   - Every call is asynchronous on the context's CUDA stream, allocates nothing on the device
 *     (context and KV-cache creation excepted) and never synchronises, so the calls can be
 *     captured in a CUDA graph. Errors found on the host are returned at once; errors found by
 *     a kernel (a token id outside the vocabulary, a bounded wait that gave up) set the
 *     context's device error word and are returned by the next gk_sync.
 *   - Backward calls ADD into parameter-gradient buffers ([LM1] "Why += and not =": a tensor
 *     used twice receives the sum; the caller zeroes them, like ZeroGrad). Activation
 *     gradients take an `accumulate` flag.
 *   - dtype arguments take GK_F32 or GK_BF16 (bfloat16 stored as uint16_t bits); some outputs
 *     also take GK_BF16X2, a float32 value kept as two bfloat16 planes: hi = bf16(v) at the
 *     pointer, lo = bf16(v - hi) at pointer + rows * ld elements (about 16 significant bits).
 */
#ifndef GK_H
#define GK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int gk_status;
enum {
    GK_OK = 0,
    GK_ERR_ARG = 1,         /* null pointer, bad size, bad enum value */
    GK_ERR_ALIGN = 2,       /* pointer or stride misses the kernel's alignment rule */
    GK_ERR_UNSUPPORTED = 3, /* valid request this build has no kernel for */
    GK_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    GK_ERR_TIMEOUT = 5,     /* a kernel's bounded wait expired (read back by gk_sync) */
    GK_ERR_OVERFLOW = 6,    /* KV cache full */
    GK_ERR_INDEX = 7,       /* a token id outside [0, V) (read back by gk_sync) */
    GK_ERR_WORKSPACE = 8,   /* the context's workspace is smaller than the call needs */
    GK_ERR_IO = 9,          /* a file could not be opened, read, written or renamed */
    GK_ERR_FORMAT = 10      /* a malformed file, or a dtype this build does not read */
};

enum { GK_F32 = 0, GK_BF16 = 1, GK_BF16X2 = 2 };
/* Arithmetic of the products with float32 operands (the faithful mode):
 *   GK_MATH_3XTF32 (default): each operand x is split into TF32 parts hi = tf32(x) and
 *     lo = tf32(x - hi) (about 22 significant bits together), and the product is
 *     A_hi B_hi + A_hi B_lo + A_lo B_hi on the tensor cores (kind::tf32, float32 accumulation in
 *     tensor memory); the planes are written K-major into the context's workspace, in blocks
 *     of the output (and of K for plain sums) when the whole does not fit, so it needs at
 *     least 8 * Kc * (128 + 256) bytes for some K slice Kc (GK_ERR_WORKSPACE otherwise).
 *     Products with a bf16 result keep the FMA kernel.
 *   GK_MATH_FP32: float32 FMA on the CUDA cores (exact float32 products, float32 sums). */
enum { GK_MATH_FP32 = 0, GK_MATH_3XTF32 = 1 };
enum { GK_ACT_NONE = 0, GK_ACT_GELU = 1 };

typedef struct gk_ctx gk_ctx;

/* ------------------------------------------------------------------------------ context */

/* Create a context bound to `cuda_stream` (a cudaStream_t; NULL = the legacy default
 * stream) on the current device. It allocates a device error word and `workspace_bytes`
 * of device scratch used by the calls that need scratch (each says how much). Returns
 * GK_ERR_CUDA if an allocation fails. Not thread-safe: one context per host thread. */
gk_status gk_ctx_create(gk_ctx** out, void* cuda_stream, size_t workspace_bytes);
void gk_ctx_destroy(gk_ctx* ctx);
/* Rebind the stream (e.g. to the stream a graph capture runs on). */
gk_status gk_ctx_set_stream(gk_ctx* ctx, void* cuda_stream);
/* GK_MATH_3XTF32 (default) or GK_MATH_FP32 for the float32 products of later calls. */
gk_status gk_set_math(gk_ctx* ctx, int math);
/* Wait for the stream, then read and clear the device error word: returns the first kernel
 * error recorded since the last gk_sync (GK_ERR_INDEX, GK_ERR_TIMEOUT, ...), else GK_OK. */
gk_status gk_sync(gk_ctx* ctx);
/* Human-readable text of the last host-side error of this context (static storage). */
const char* gk_last_error(gk_ctx* ctx);
/* Number of kernel launches this context has issued since creation. */
int64_t gk_launch_count(gk_ctx* ctx);

/* Self-test of the bounded-wait failure path (no counterpart on the pages: it checks this
 * library's own failure detection). One CTA allocates tensor memory, waits on an mbarrier
 * with the same bounded wait the tensor-core kernels use, limit `limit_ns` (0 < limit <= 1 s),
 * then frees the tensor memory and exits. With arrive = 0 no thread arrives: the wait expires,
 * GK_ERR_TIMEOUT is recorded in the device error word (returned by the next gk_sync) and the
 * context stays usable. With arrive != 0 one thread arrives first and nothing is recorded.
 * elapsed_ns (device int64, may be NULL) receives the time the wait took. */
gk_status gk_selftest_wait_timeout(gk_ctx* ctx, int64_t limit_ns, int arrive, long long* elapsed_ns);

/* -------------------------------------------------------------------------- embedding */

/* x[b*T + t, :] = wte[ids[b*T + t], :] + wpe[t, :].  [LM1] "Ops..." op table (Embedding);
 * [LM4] "Generation with a KV cache" (the token row plus the position row).
 * ids int32 [B*T]; wte [V, C]; wpe [>= T, C]; x [B*T, C] (all float32, contiguous).
 * An id outside [0, V) writes zeros for its row and records GK_ERR_INDEX. */
gk_status gk_embedding_fwd(gk_ctx* ctx, const int32_t* ids, const float* wte, const float* wpe,
                           float* x, int B, int T, int C, int V);

/* dwte[ids[r], :] += dx[r, :] and dwpe[r % T, :] += dx[r, :] for r = 0 .. B*T-1.
 * Exact and deterministic: every gradient element receives its rows' float32 additions in
 * ascending r, so the result is bit-identical to that sequential loop.
 * [LM1] "Ops..." (Embedding backward scatter-adds); "Why += and not =". */
gk_status gk_embedding_bwd(gk_ctx* ctx, const int32_t* ids, const float* dx, float* dwte,
                           float* dwpe, int B, int T, int C, int V);

/* -------------------------------------------------------------------------- layernorm */

/* Per row: y = (x - mean) * rstd * gamma + beta, rstd = 1/sqrt(var + eps), var biased.
 * [LM1] op table (LayerNorm); eps 1e-5 in GPT-2. x float32 [rows, C] contiguous; y is
 * `y_dtype` [rows, C] (GK_BF16X2: two planes of rows * C); mean and rstd float32 [rows] (saved
 * for backward, may be NULL). x_copy (float32 [rows, C], may be NULL, must not overlap x)
 * receives a copy of x: the residual stream's next buffer, which a projection then adds into
 * in place (x_next = x + f(y), "residual reuse" of the GPT-2 block), while x stays as the
 * saved input of this LayerNorm. */
gk_status gk_layernorm_fwd(gk_ctx* ctx, const float* x, const float* gamma, const float* beta,
                           void* y, int y_dtype, float* mean, float* rstd, int64_t rows, int C,
                           float eps, float* x_copy);

/* Backward of gk_layernorm_fwd for upstream dy (float32 [rows, C]):
 *   dx (=, or += if accumulate_dx) rstd * (dy*gamma - mean(dy*gamma) - xhat*mean(dy*gamma*xhat));
 *   dgamma += sum_rows dy*xhat;  dbeta += sum_rows dy   (deterministic order);
 *   dx_colsum += sum_rows dx, the column sums of the dx this call leaves (after accumulating):
 *   when dx is also the output gradient of a layer with a bias (the projection feeding the
 *   residual stream), this is that bias's gradient (the MatMul/bias backward rule), produced
 *   here so the rows are read once.
 * dx_bf16, if not NULL, receives a bfloat16 copy of the resulting dx. dgamma, dbeta and
 * dx_colsum may be NULL. Workspace: np * C * P * 4 bytes (np = 3 with dx_colsum, else 2, and
 * none without dgamma, dbeta and dx_colsum), with P <= 1216 partial slots for C <= 1024
 * (fewer for wide rows), and for C > 1024 P = ceil(rows / 32) plus 8 * rows bytes of row
 * statistics. */
gk_status gk_layernorm_bwd(gk_ctx* ctx, const float* x, const float* gamma, const float* mean,
                           const float* rstd, const float* dy, float* dx, int accumulate_dx,
                           uint16_t* dx_bf16, float* dgamma, float* dbeta, float* dx_colsum,
                           int64_t rows, int C);

/* LayerNorm backward that allocates nothing (no counterpart on the pages: it serves callers
 * that cannot allocate device memory). Same arguments, layout and results as
 * gk_layernorm_bwd without dx_colsum, but it takes a CUDA stream (cudaStream_t, NULL = legacy default) instead
 * of a context, and its dgamma/dbeta partial sums live in a fixed 4 MiB array compiled into
 * the library rather than in a workspace.
 *   Who needs it: code that cannot call cudaMalloc, e.g. a host framework that owns all device
 *   memory through its own pool, a loop that must never block in the allocator, or a plugin
 *   whose process fixed its memory budget before loading it.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before any stream
 *   capture. The array stays allocated on every GPU that loads the library until exit.
 *   Limits: C <= 524288 (one partial slot of 2*C floats must fit); larger C returns
 *   GK_ERR_WORKSPACE. Nothing in the array needs to start at zero: each call writes every
 *   partial slot before reading it, and the array keeps the last call's contents.
 *   Concurrency: all calls share the one array per device, so calls whose kernels overlap on
 *   the GPU (other streams, other host threads) race on it; serialise them. The per-device
 *   address lookup itself is safe to race from several host threads. The cached address
 *   assumes the device is not reset (cudaDeviceReset) while the library stays loaded.
 * Returns GK_ERR_ARG for null pointers or sizes <= 0, GK_ERR_CUDA if a CUDA call fails. A
 * CUDA error already pending from the caller's earlier work (cudaPeekAtLastError) makes the
 * call return GK_ERR_CUDA before it launches anything, and that error is left pending for the
 * caller; otherwise GK_ERR_CUDA is the status of this call's own launches. */
gk_status gk_layernorm_bwd_noalloc(void* cuda_stream, const float* x, const float* gamma,
                                   const float* mean, const float* rstd, const float* dy, float* dx,
                                   int accumulate_dx, uint16_t* dx_bf16, float* dgamma, float* dbeta,
                                   int64_t rows, int C);

/* ------------------------------------------------------------------------------ GELU */

/* y = 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))) elementwise on float32 [n].
 * [LM4] "Common mistakes": GPT-2 uses the tanh form ("gelu_new"), not the erf form. */
gk_status gk_gelu_fwd(gk_ctx* ctx, const float* x, float* y, int64_t n);
/* dx = dy * gelu'(x) (dx may alias dy). */
gk_status gk_gelu_bwd(gk_ctx* ctx, const float* x, const float* dy, float* dx, int64_t n);

/* ---------------------------------------------------------------------------- matmul */

/* Y = act(X W + bias + residual) with X [N, K]; W [K, M] (transW = 0, MatMul) or W [M, K]
 * (transW = 1, MatMulT: the tied LM head). [LM1] "Ops...", MatMul listing and op table.
 *   dtype      GK_F32 (fp32 arithmetic per gk_set_math) or GK_BF16 (bf16 operands, fp32
 *              accumulation on the tensor cores); X and W both have this type.
 *   bias       float32 [M] or NULL.  residual  float32 [N, M] (stride ldr) or NULL; it may
 *              alias Y when y_dtype is GK_F32 (in-place x += ...).
 *   act        GK_ACT_GELU stores the pre-activation in `preact` (y_dtype, bf16 for
 *              GK_BF16X2; stride ldp) and gelu(pre) in Y.
 *   X_lo, W_lo optional low bf16 planes (same layout) of bf16 X and W: the product becomes
 *              X_hi W_hi + X_hi W_lo + X_lo W_hi, i.e. split-bf16 operands of about 16
 *              significant bits on the bf16 tensor cores.
 *   y_dtype    GK_F32, GK_BF16 or GK_BF16X2 (Y's low plane at Y + N * ldy).
 * bf16 operands need 16-byte aligned base pointers and strides that are multiples of 8. */
gk_status gk_matmul_fwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W,
                        int64_t ldw, int transW, const float* bias, const float* residual,
                        int64_t ldr, void* Y, int64_t ldy, int y_dtype, int64_t N, int64_t K,
                        int64_t M, int act, void* preact, int64_t ldp, const void* X_lo,
                        const void* W_lo);

/* Backward of Y = X W (transW = 0) or X W^T (transW = 1) for upstream dY [N, M]:
 *   dX  = dY W^T (transW = 0) or dY W (transW = 1); written (=), or added (+=) if
 *         accumulate_dX (float32 dX only). If preact_X is given (X was gelu(preact_X)),
 *         the product is (dY W^T) * gelu'(preact_X), the GELU backward fused in, and that
 *         is what is written or added. dX may be NULL.
 *   dW += X^T dY ([K, M]) or dY^T X ([M, K]); float32; may be NULL.
 *   dbias += sum over rows of dY; float32 [M]; may be NULL.
 * [LM1] "Ops...", MatMul backward rule (dx = g w^T, dw = x^T g, both accumulating).
 * dtype is the type of X, W and dY. Workspace for dbias: 128 * M * 4 bytes. */
gk_status gk_matmul_bwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W,
                        int64_t ldw, int transW, const void* dY, int64_t lddy, void* dX,
                        int64_t lddx, int dx_dtype, int accumulate_dX, const void* preact_X,
                        int64_t ldp, float* dW, int64_t lddw, float* dbias, int64_t N,
                        int64_t K, int64_t M);

/* ------------------------------------------------------------------------- attention */

/* Causal multi-head self-attention of the fused projection qkv [B*T, 3C] (q, k, v in column
 * blocks [0,C), [C,2C), [2C,3C); head h uses columns h*hs .. h*hs+hs-1 of each block):
 * y[:, h] = softmax(q_h k_h^T / sqrt(hs), keys j <= query i) v_h, written to y [B*T, C];
 * lse [B, H, T] float32 receives the log-sum-exp of each scaled score row (for backward).
 * [LM1] op table (BatchMatMulT, CausalSoftmax, BatchMatMul, SplitHeads, MergeHeads);
 * [LM4] "The 12 tensors we do not use" (the causal mask by arithmetic, visible = i + 1).
 * dtype (GK_F32 / GK_BF16) is the type of qkv and y; scores and softmax are float32.
 * hs must be a multiple of 4 and at most 128. */
gk_status gk_attn_fwd(gk_ctx* ctx, int dtype, const void* qkv, void* y, float* lse, int B,
                      int T, int H, int hs);

/* dqkv [B*T, 3C] (written, same dtype) of gk_attn_fwd for upstream dy [B*T, C]: with
 * P recomputed from q, k and lse, dv = P^T dy, dP = dy v^T, dS = P (dP - rowsum(dy * y)),
 * dq = dS k / sqrt(hs), dk = dS^T q / sqrt(hs). Deterministic (no atomics).
 * Workspace: B * H * T * 4 bytes. */
gk_status gk_attn_bwd(gk_ctx* ctx, int dtype, const void* qkv, const void* y, const float* lse,
                      const void* dy, void* dqkv, int B, int T, int H, int hs);

/* ------------------------------------------------------------- softmax cross-entropy */

/* loss (device float32 scalar, written) = mean over rows of (logsumexp(row) - row[target]);
 * lse [rows] float32 receives each row's log-sum-exp. logits float32 [rows, V], stride ldl.
 * [LM1] "Ops...", SoftmaxCrossEntropy listing. A target outside [0, V) records
 * GK_ERR_INDEX. Workspace: rows * 4 bytes. */
gk_status gk_softmax_ce_fwd(gk_ctx* ctx, const float* logits, int64_t ldl, const int32_t* targets,
                            float* loss, float* lse, int64_t rows, int V);

/* dlogits = (dloss / rows) (softmax(row) - onehot(target)), dloss a device float32 scalar
 * (NULL = 1). dlogits has dl_dtype and stride lddl; columns V .. lddl-1 are written as 0.
 * dlogits may alias logits when both are float32 with the same stride (in place).
 * [LM1] "Ops...", SoftmaxCrossEntropy backward (probs minus one at the target). */
gk_status gk_softmax_ce_bwd(gk_ctx* ctx, const float* logits, int64_t ldl, const int32_t* targets,
                            const float* lse, const float* dloss, void* dlogits, int64_t lddl,
                            int dl_dtype, int64_t rows, int V);

/* LM head fused with softmax cross-entropy: the tied projection logits = X W^T ([LM4]
 * "... running GPT-2 weights", the output head reuses wte) and the loss of [LM1]
 * "Ops...", SoftmaxCrossEntropy, without a [N, V] logits tensor.
 *   X  bf16 [N, C] (row stride ldx), W bf16 [V, C] (row stride ldw; row v = vocabulary
 *   entry v), targets int32 [N] in [0, V).
 * gk_lmhead_ce_fwd: *loss = mean_r (lse_r - logit[r, targets[r]]) (float32 device scalar),
 *   lse [N] = per-row natural log-sum-exp of the logits (saved for backward). Logits come
 *   from bf16 operands with float32 accumulation. A target outside [0, V) contributes 0 and
 *   records GK_ERR_INDEX (read back by gk_sync). Workspace: N * (8 * ceil(V / 256) * 2 + 8)
 *   bytes (rounded up), e.g. 52 MB at N = 16384, V = 50257.
 * gk_lmhead_ce_bwd: with g = *dloss (1 if dloss is NULL) and
 *   dlogits = (g / N) (softmax(logits) - onehot(targets)):
 *   dX (=, or += if accumulate_dX) dlogits W (float32 [N, C], stride lddx; may be NULL);
 *   dW += dlogits^T X (float32 [V, C], stride lddw; may be NULL).
 *   The logits are recomputed per vocabulary chunk and turned into bf16 dlogits in the
 *   caller's scratch (bf16, scratch_elems elements, device memory the caller owns); the
 *   chunk is the largest multiple of 256 columns with N * chunk <= scratch_elems, at least
 *   256 (else GK_ERR_WORKSPACE).
 * Both need 16-byte aligned operands with row strides a multiple of 8 elements
 * (GK_ERR_ALIGN otherwise) and dtype GK_BF16 (GK_ERR_UNSUPPORTED otherwise). */
gk_status gk_lmhead_ce_fwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W,
                           int64_t ldw, const int32_t* targets, float* loss, float* lse, int64_t N,
                           int64_t C, int64_t V);
gk_status gk_lmhead_ce_bwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W,
                           int64_t ldw, const int32_t* targets, const float* lse,
                           const float* dloss, float* dX, int64_t lddx, int accumulate_dX,
                           float* dW, int64_t lddw, void* scratch, int64_t scratch_elems,
                           int64_t N, int64_t C, int64_t V);

/* Round float32 [n] to bfloat16 [n] (round to nearest even): the bf16 operand copy of a
 * float32 tensor, e.g. the weights before the first step (AdamW refreshes it afterwards).
 * y_lo, if not NULL, receives the low plane bf16(x - y) of the split-bf16 form. */
gk_status gk_to_bf16(gk_ctx* ctx, const float* x, uint16_t* y, uint16_t* y_lo, int64_t n);

/* ---------------------------------------------------------------------------- AdamW */

/* One parameter block for gk_adamw_step (a host struct holding device pointers). */
typedef struct {
    float* p;          /* parameters, updated in place */
    float* g;          /* gradient (zeroed after use if the call's zero_grad is set) */
    float* m;          /* first moment */
    float* v;          /* second moment */
    int64_t n;         /* number of elements */
    int decay;         /* 1: apply weight decay (tensors with >= 2 dims), 0: not */
    uint16_t* p_bf16;  /* optional bfloat16 copy of the updated p, or NULL */
    uint16_t* p_bf16_lo; /* optional low plane bf16(p - p_bf16) (needs p_bf16), or NULL */
} gk_param;

/* AdamW at step `step` (>= 1) over n_params blocks (host array):
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;  mhat = m/(1-b1^step);  vhat = v/(1-b2^step);
 *   p -= lr (mhat / (sqrt(vhat) + eps) + wd_k p),  wd_k = wd if decay else 0.
 * [LM1] "The optimizer: from gradient to step", AdamW listing (Loshchilov & Hutter): decay
 * applies to matrices only, and uses p before the update. zero_grad = 1 also sets g = 0
 * (the ZeroGrad of the next step, fused). */
gk_status gk_adamw_step(gk_ctx* ctx, const gk_param* params, int n_params, float lr, float beta1,
                        float beta2, float eps, float wd, int step, int zero_grad);

/* ------------------------------------------------------------------ flat GPT-2 layout */

/* Model sizes: vocabulary, context (positions), width, heads, layers. */
typedef struct { int V, T, C, H, L; } gk_gpt_cfg;

enum {
    GK_T_WTE = 0, GK_T_WPE, GK_T_LN1_W, GK_T_LN1_B, GK_T_ATTN_W, GK_T_ATTN_B, GK_T_ATTNPROJ_W,
    GK_T_ATTNPROJ_B, GK_T_LN2_W, GK_T_LN2_B, GK_T_FC_W, GK_T_FC_B, GK_T_MLPPROJ_W,
    GK_T_MLPPROJ_B, GK_T_LNF_W, GK_T_LNF_B, GK_T_COUNT
};

/* Parameters of a whole model live in ONE float32 buffer: first every tensor with >= 2 dims
 * (wte, wpe, then per layer c_attn.w [C,3C], attn.c_proj.w [C,C], mlp.c_fc.w [C,4C],
 * mlp.c_proj.w [4C,C]), then every vector (per layer ln_1.w, ln_1.b, c_attn.b, attn.c_proj.b,
 * ln_2.w, ln_2.b, c_fc.b, mlp.c_proj.b; then ln_f.w, ln_f.b). So AdamW's decay boundary is
 * one index. Gradients, moments and the bf16 copy use the same layout.
 * Returns the element offset of tensor `which` of layer `layer` (ignored for wte, wpe and
 * ln_f), or -1 for a bad argument. */
int64_t gk_gpt_offset(const gk_gpt_cfg* cfg, int which, int layer);
/* Total elements, V*C + T*C + L*(12 C^2 + 13 C) + 2 C. */
int64_t gk_gpt_numel(const gk_gpt_cfg* cfg);
/* Elements of the leading block of tensors with >= 2 dims (the decayed block). */
int64_t gk_gpt_n_decay(const gk_gpt_cfg* cfg);

/* ------------------------------------------------------------------- KV-cache decode */

typedef struct gk_kv gk_kv;

/* Sampling settings: top_k <= 0 or >= V keeps every logit; top_k == 1 or temperature <= 0
 * is greedy (lowest index among the largest). Selection s of a cache draws
 * u = Philox4x32-10(key = seed, counter = (counter + s, batch row, 0, 0)) word 0 >> 8, times
 * 2^-24, and takes the first kept index whose running float64 sum of exp((l - max)/T)
 * exceeds u times the total. [LM4] "Temperature and top-k". */
typedef struct { int top_k; float temperature; uint64_t seed; uint64_t counter; } gk_sample_cfg;

/* Allocate a float32 cache [L][2][B][H][Tmax][hs] plus the decode activations for B rows and
 * prompts up to Tmax tokens. [LM4] "Generation with a KV cache" (one key and value row per
 * layer per position). Owned by libgk; free with gk_kv_destroy. */
gk_status gk_kv_create(gk_ctx* ctx, gk_kv** out, const gk_gpt_cfg* cfg, int B, int Tmax);
void gk_kv_destroy(gk_kv* kv);
/* Device pointer to the cache (layout above) and its current length (host mirror). */
float* gk_kv_data(gk_kv* kv);
int gk_kv_length(gk_kv* kv);

/* Forget the cache contents and run a [B, Tp] prompt (ids int32, device) through one causal
 * forward, writing every layer's keys and values and the logits of each row's LAST position
 * to last_logits [B, V] (float32, stride V). Float32 weights in the flat layout. */
gk_status gk_prefill(gk_ctx* ctx, const float* params, gk_kv* kv, const int32_t* ids, int Tp,
                     float* last_logits);

/* One token per row (tokens int32 [B], device) at position = the cache length: every layer
 * appends its key and value and attends over all cached positions (no mask: the cache holds
 * only the past), then ln_f and the tied head write logits [B, V]; if `next` is not NULL a
 * selection (greedy if s is NULL) writes next [B]. The cache length advances by one.
 * [LM4] "Generation with a KV cache" (Attention.Step, Gpt.Step). GK_ERR_OVERFLOW if full. */
gk_status gk_decode_step(gk_ctx* ctx, const float* params, gk_kv* kv, const int32_t* tokens,
                         float* logits, int32_t* next, const gk_sample_cfg* s);

/* n_steps decode steps in a row, each one gk_decode_step(ctx, params, kv, tokens, logits,
 * next, s) followed by copying next into tokens (skipped when they are the same buffer), so
 * every step feeds the token just selected: [LM4] "Generation with a KV cache"
 * (GenerateCached's loop). tokens and next are device int32 [B]; logits [B, V] holds the
 * last step's logits. The first call for a given (params, tokens, logits, next, s values,
 * stream) records one step as a CUDA graph kept with the cache; later calls replay it, one
 * graph launch per step (on the legacy default stream, which cannot be captured, the steps
 * are launched one by one). Results are those of the step-by-step calls. GK_ERR_OVERFLOW
 * (nothing run) if the cache length plus n_steps exceeds Tmax; GK_ERR_ARG for null
 * pointers or n_steps < 0. */
gk_status gk_decode_run(gk_ctx* ctx, const float* params, gk_kv* kv, int32_t* tokens,
                        float* logits, int32_t* next, const gk_sample_cfg* s, int n_steps);

/* Uncached generation, [LM4] "Generation with a KV cache" (Generate: the whole sequence runs
 * through the model again for every new token, the baseline the cached loop is measured
 * against). ids: device int32 [B, Tp + n_new], row stride Tp + n_new, holding the prompt in
 * its first Tp columns. For i = 0 .. n_new-1 the prefix ids[:, :Tp+i] goes through one causal
 * forward (as gk_prefill; the cache serves as scratch and is overwritten every step) and
 * selection i (as gk_sample, the cache's selection count set to i, so the draws are those of
 * gk_prefill + gk_sample + gk_decode_run) is written to ids[:, Tp+i]. logits [B, V] holds the
 * last step's logits. GK_ERR_OVERFLOW (nothing run) if Tp + n_new - 1 exceeds the cache;
 * GK_ERR_ARG for null pointers, Tp < 1 or n_new < 0. */
gk_status gk_generate_uncached(gk_ctx* ctx, const float* params, gk_kv* kv, int32_t* ids, int Tp,
                               int n_new, float* logits, const gk_sample_cfg* s);

/* Select next [B] from logits [B, V] (stride ld) as gk_sample_cfg describes; the selection
 * index s is the cache's selection count, which this advances by one. */
gk_status gk_sample(gk_ctx* ctx, gk_kv* kv, const float* logits, int64_t ld, int32_t* next,
                    const gk_sample_cfg* s);

/* ---- Generic ops of the autograd engine and plain SGD ([LM1] "Build a language model in C#
 * from scratch (1)": Ops, the op table (Add with broadcast, Scale, Sum, Tanh), "Why += and not =",
 * The optimizer; [AD] "Chain rule and automatic differentiation", Steps 1-5: the tanh neuron).
 * All tensors are float32 device buffers of n elements, row-major. Backward calls take
 * `accumulate`: 0 writes the gradient, 1 adds it to the buffer (the pages' += rule; zeroing
 * before a backward pass is the caller's job). Elementwise outputs may alias an input of the
 * same index. n == 0 is a no-op. GK_ERR_ARG for null pointers or n < 0. */

/* y = a + b, b broadcast over the leading dimensions: b has m elements and m divides n (m == n
 * is the plain sum, m = the row width is the bias added to every row). GK_ERR_ARG if m does not
 * divide n. */
gk_status gk_add_fwd(gk_ctx* ctx, const float* a, const float* b, float* y, int64_t n, int64_t m);
/* da (+)= g; db (+)= g summed over the rows of g viewed as [n / m, m] (the broadcast's
 * gradient; in double, fixed order). Either output may be NULL. Needs (chunks x m) doubles of
 * workspace for m < n (GK_ERR_WORKSPACE if the context's workspace is smaller than m doubles). */
gk_status gk_add_bwd(gk_ctx* ctx, const float* g, float* da, float* db, int64_t n, int64_t m, int accumulate);
/* y = a * b elementwise. */
gk_status gk_mul_fwd(gk_ctx* ctx, const float* a, const float* b, float* y, int64_t n);
/* da (+)= g * b, db (+)= g * a (either may be NULL). */
gk_status gk_mul_bwd(gk_ctx* ctx, const float* g, const float* a, const float* b, float* da, float* db,
                     int64_t n, int accumulate);
/* y = s * a, s a host scalar. */
gk_status gk_scale_fwd(gk_ctx* ctx, const float* a, float s, float* y, int64_t n);
/* da (+)= s * g. */
gk_status gk_scale_bwd(gk_ctx* ctx, const float* g, float s, float* da, int64_t n, int accumulate);
/* y[0] = sum of a in a fixed order (aligned groups of four added in float32, the groups and the
 * partial sums in double; n == 0 gives 0). Needs up to 8 KB of workspace. */
gk_status gk_sum_fwd(gk_ctx* ctx, const float* a, float* y, int64_t n);
/* da (+)= g[0] for every element (g: one float32 on the device). */
gk_status gk_sum_bwd(gk_ctx* ctx, const float* g, float* da, int64_t n, int accumulate);
/* y = tanh(x). */
gk_status gk_tanh_fwd(gk_ctx* ctx, const float* x, float* y, int64_t n);
/* dx (+)= g * (1 - y^2), y the forward's output. */
gk_status gk_tanh_bwd(gk_ctx* ctx, const float* y, const float* g, float* dx, int64_t n, int accumulate);
/* Plain SGD step ([LM1] The optimizer, Sgd): p -= lr * g. */
gk_status gk_sgd_step(gk_ctx* ctx, float* p, const float* g, int64_t n, float lr);

/* ---- safetensors files of float32 tensors ([LM4] "Build a language model in C# from scratch
 * (4): running GPT-2 weights", "The safetensors format"): an 8-byte little-endian header length
 * N, N bytes of JSON giving each tensor's dtype, shape and data_offsets [begin, end) (byte
 * offsets from the end of the header) and an optional "__metadata__" object of strings, then
 * the raw little-endian bytes. Host code; no context. A failing call returns its status and
 * leaves a message for gk_st_last_error (per host thread). */
typedef struct gk_st gk_st;
/* Open and check a file: the header must parse, every entry must have a dtype string, a shape
 * of non-negative integers and data_offsets inside the file (GK_ERR_FORMAT otherwise; GK_ERR_IO
 * if it cannot be opened or read). Close with gk_st_close. */
gk_status gk_st_open(const char* path, gk_st** out);
void gk_st_close(gk_st* st);
/* Tensors in header order (metadata excluded): count, name, dtype, rank and shape (owned by st);
 * NULL / -1 for a bad index. gk_st_find gives a name's index or -1. */
int gk_st_count(const gk_st* st);
const char* gk_st_name(const gk_st* st, int i);
const char* gk_st_dtype(const gk_st* st, int i);
int gk_st_ndim(const gk_st* st, int i);
const int64_t* gk_st_shape(const gk_st* st, int i);
int gk_st_find(const gk_st* st, const char* name);
/* A "__metadata__" value, or NULL. */
const char* gk_st_metadata(const gk_st* st, const char* key);
/* Read tensor i (n = its element count, else GK_ERR_ARG) into dst, a host buffer or, with
 * dst_on_device, a device buffer (staged through host memory, synchronous). GK_ERR_FORMAT for
 * a dtype other than F32 or data_offsets that do not span 4 bytes per element. */
gk_status gk_st_read_f32(const gk_st* st, int i, float* dst, int64_t n, int dst_on_device);
/* Write n float32 tensors (names unique, not "__metadata__"; ndims[t] extents each, taken in
 * order from shapes; data[t] host or, with data_on_device, device pointers) and n_meta metadata
 * strings. Tensors are laid out back to back in the order given, the JSON padded with spaces to
 * a multiple of 8 bytes; the file is written as path + ".tmp" and renamed over path. */
gk_status gk_st_write_f32(const char* path, int n, const char* const* names, const int* ndims,
                          const int64_t* shapes, const float* const* data, int data_on_device,
                          int n_meta, const char* const* meta_keys, const char* const* meta_values);
/* The message of the last failing gk_st_* call on this host thread ("" if none). */
const char* gk_st_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* GK_H */
