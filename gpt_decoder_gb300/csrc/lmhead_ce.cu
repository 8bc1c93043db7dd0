// LM head fused with softmax cross-entropy, without a materialised [rows, V] logits tensor.
// [LM1] = "Build a language model in C# from scratch (1)", SoftmaxCrossEntropy listing and
// backward rule (loss = mean over rows of LSE - logit[target]; dlogits = (g / rows) *
// (softmax - one-hot)); [LM4] = "... (4): running GPT-2 weights", the tied head
// logits = ln_f(x) wte^T.
//
// Forward: one tensor-core GEMM over the whole vocabulary whose epilogue keeps, per row and
// 128-column half tile, an online (max, sum of exponentials) pair and picks out the target's
// logit (the logits themselves are never stored); a row kernel combines the pairs into the
// row's log-sum-exp and loss, and a fixed-order sum gives the mean.
// Backward: the vocabulary is walked in chunks that fit the caller's scratch. Per chunk the
// logits are recomputed by a GEMM whose epilogue writes bf16 dlogits directly, and two GEMMs
// consume them: dX (+)= dlogits_chunk wte_chunk and dwte_chunk += dlogits_chunk^T X.
#include <math.h>

#include <algorithm>

#include "gemm.cuh"

namespace gk {
namespace {

constexpr int BN_TILE = 256;  // the tensor-core GEMM's column tile (two 128-column halves)

// Row r: M = max_j m_j, S = sum_j s_j 2^(m_j - M) over the row's partial pairs (log2 units),
// lse = (M + log2 S) ln 2, loss_r = lse - logit[target]. One warp per row; lane l takes pairs
// l, l + 32, ...; the warp reductions run in a fixed order.
__global__ void ce_combine_kernel(const float2* __restrict__ part, int P, const float* __restrict__ tgt_logit,
                                  const int32_t* __restrict__ targets, int64_t V, float* __restrict__ lse,
                                  float* __restrict__ row_loss, int64_t rows, int* err) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float2* pr = part + row * P;
    float m = -INFINITY;
    for (int j = lane; j < P; j += 32) m = fmaxf(m, pr[j].x);
    m = warp_max(m);
    float s = 0.f;
    for (int j = lane; j < P; j += 32) {
        const float2 q = pr[j];
        if (q.y > 0.f) s += q.y * exp2f(q.x - m);
    }
    s = warp_sum(s);
    if (lane == 0) {
        const float l = (m + log2f(s)) * 0.6931471805599453f;
        lse[row] = l;
        const int32_t t = targets[row];
        if (t < 0 || t >= V) {
            report(err, GK_ERR_INDEX);
            row_loss[row] = 0.f;
        } else {
            row_loss[row] = l - tgt_logit[row];
        }
    }
}

// *loss = mean of row_loss (fixed partition, double-float accumulation).
__global__ void ce_mean_kernel(const float* __restrict__ row_loss, int64_t rows, float* loss) {
    block_mean_fixed(row_loss, rows, loss);
}

bool ok_operand(const void* p, int64_t ld, int64_t inner) { return p && aligned16(p) && ld >= inner && ld % 8 == 0; }

}  // namespace
}  // namespace gk

using namespace gk;

extern "C" {

gk_status gk_lmhead_ce_fwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W, int64_t ldw,
                           const int32_t* targets, float* loss, float* lse, int64_t N, int64_t C, int64_t V) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, X && W && targets && loss && lse && N > 0 && C > 0 && V > 0 && ldx >= C && ldw >= C, GK_ERR_ARG,
               "gk_lmhead_ce_fwd: bad argument");
    GK_REQUIRE(ctx, dtype == GK_BF16, GK_ERR_UNSUPPORTED, "gk_lmhead_ce_fwd: bf16 operands only");
    GK_REQUIRE(ctx, ok_operand(X, ldx, C) && ok_operand(W, ldw, C), GK_ERR_ALIGN,
               "gk_lmhead_ce_fwd: operands need 16-byte aligned rows");
    GK_REQUIRE(ctx, N < (1ll << 31) && V < (1ll << 31), GK_ERR_UNSUPPORTED, "gk_lmhead_ce_fwd: too large");
    const int P = (int)(2 * cdiv(V, BN_TILE));
    const size_t part_bytes = ((size_t)N * P * sizeof(float2) + 255) & ~size_t(255);
    const size_t need = part_bytes + 2 * (((size_t)N * sizeof(float) + 255) & ~size_t(255));
    char* ws = (char*)workspace(ctx, need);
    GK_REQUIRE(ctx, ws, GK_ERR_WORKSPACE, "gk_lmhead_ce_fwd: needs %zu workspace bytes", need);
    float2* part = (float2*)ws;
    float* tgt_logit = (float*)(ws + part_bytes);
    float* row_loss = (float*)(ws + part_bytes + (((size_t)N * sizeof(float) + 255) & ~size_t(255)));
    Gemm g;
    g.M = N; g.N = V; g.K = C;
    g.A = X; g.lda = ldx; g.a_kmajor = true;
    g.B = W; g.ldb = ldw; g.b_kmajor = true;  // logits = X W^T, W rows are vocabulary entries
    g.ab_dtype = GK_BF16;
    g.c_dtype = GK_BF16;
    g.ce_mode = CE_LSE;
    g.ce_tgt = targets;
    g.ce_part = part;
    g.ce_nparts = P;
    g.ce_tgt_logit = tgt_logit;
    GK_TRY(gemm_tc(ctx, g));
    ce_combine_kernel<<<(unsigned)cdiv(N * 32, 256), 256, 0, ctx->stream>>>(part, P, tgt_logit, targets, V, lse,
                                                                             row_loss, N, ctx->d_err);
    GK_TRY(launched(ctx, "ce_combine"));
    ce_mean_kernel<<<1, 1024, 0, ctx->stream>>>(row_loss, N, loss);
    return launched(ctx, "ce_mean");
}

gk_status gk_lmhead_ce_bwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W, int64_t ldw,
                           const int32_t* targets, const float* lse, const float* dloss, float* dX, int64_t lddx,
                           int accumulate_dX, float* dW, int64_t lddw, void* scratch, int64_t scratch_elems,
                           int64_t N, int64_t C, int64_t V) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, X && W && targets && lse && scratch && N > 0 && C > 0 && V > 0 && ldx >= C && ldw >= C,
               GK_ERR_ARG, "gk_lmhead_ce_bwd: bad argument");
    GK_REQUIRE(ctx, (!dX || lddx >= C) && (!dW || lddw >= C), GK_ERR_ARG, "gk_lmhead_ce_bwd: stride too small");
    GK_REQUIRE(ctx, dtype == GK_BF16, GK_ERR_UNSUPPORTED, "gk_lmhead_ce_bwd: bf16 operands only");
    GK_REQUIRE(ctx, ok_operand(X, ldx, C) && ok_operand(W, ldw, C) && aligned16(scratch), GK_ERR_ALIGN,
               "gk_lmhead_ce_bwd: operands need 16-byte aligned rows");
    GK_REQUIRE(ctx, N < (1ll << 31) && V < (1ll << 31), GK_ERR_UNSUPPORTED, "gk_lmhead_ce_bwd: too large");
    // vocabulary chunk: a multiple of the column tile whose [N, chunk] bf16 dlogits fit the scratch
    int64_t chunk = std::min<int64_t>(cdiv(V, BN_TILE) * BN_TILE, (scratch_elems / N) / BN_TILE * BN_TILE);
    GK_REQUIRE(ctx, chunk >= BN_TILE, GK_ERR_WORKSPACE,
               "gk_lmhead_ce_bwd: scratch holds %lld elements, needs at least %lld", (long long)scratch_elems,
               (long long)(N * BN_TILE));
    const __nv_bfloat16* Wb = static_cast<const __nv_bfloat16*>(W);
    for (int64_t v0 = 0; v0 < V; v0 += chunk) {
        const int64_t vc = std::min(chunk, V - v0), ldd = cdiv(vc, 8) * 8;
        // dlogits of the chunk, from recomputed logits
        Gemm g;
        g.M = N; g.N = vc; g.K = C;
        g.A = X; g.lda = ldx; g.a_kmajor = true;
        g.B = Wb + v0 * ldw; g.ldb = ldw; g.b_kmajor = true;
        g.ab_dtype = GK_BF16;
        g.C = scratch; g.ldc = ldd; g.c_dtype = GK_BF16;
        g.ce_mode = CE_DLOGITS;
        g.ce_tgt = targets;
        g.ce_col0 = v0;
        g.ce_lse = lse;
        g.ce_dloss = dloss;
        g.ce_scale = 1.f / (float)N;
        GK_TRY(gemm_tc(ctx, g));
        if (dX) {  // dX (+)= dlogits_chunk W_chunk
            Gemm d;
            d.M = N; d.N = C; d.K = vc;
            d.A = scratch; d.lda = ldd; d.a_kmajor = true;
            d.B = Wb + v0 * ldw; d.ldb = ldw; d.b_kmajor = false;
            d.ab_dtype = GK_BF16;
            d.C = dX; d.ldc = lddx; d.c_dtype = GK_F32;
            d.accumulate = accumulate_dX || v0 > 0;
            GK_TRY(gemm(ctx, d));
        }
        if (dW) {  // dW_chunk += dlogits_chunk^T X
            Gemm d;
            d.M = vc; d.N = C; d.K = N;
            d.A = scratch; d.lda = ldd; d.a_kmajor = false;
            d.B = X; d.ldb = ldx; d.b_kmajor = false;
            d.ab_dtype = GK_BF16;
            d.C = dW + v0 * lddw; d.ldc = lddw; d.c_dtype = GK_F32;
            d.accumulate = true;
            GK_TRY(gemm(ctx, d));
        }
    }
    return GK_OK;
}

}  // extern "C"
