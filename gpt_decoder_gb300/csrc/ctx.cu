// Context lifetime, error reporting and the flat GPT-2 parameter layout.
#include <stdarg.h>
#include <string.h>

#include "common.cuh"

namespace gk {

gk_status fail(gk_ctx* ctx, gk_status code, const char* fmt, ...) {
    if (ctx) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(ctx->msg, sizeof(ctx->msg), fmt, ap);
        va_end(ap);
    }
    return code;
}

gk_status launched(gk_ctx* ctx, const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ctx, GK_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    ctx->launches++;
    return GK_OK;
}

}  // namespace gk

using namespace gk;

extern "C" {

gk_status gk_ctx_create(gk_ctx** out, void* cuda_stream, size_t workspace_bytes) {
    if (!out) return GK_ERR_ARG;
    *out = nullptr;
    gk_ctx* ctx = new gk_ctx();
    ctx->stream = static_cast<cudaStream_t>(cuda_stream);
    if (cudaGetDevice(&ctx->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
        delete ctx;
        return GK_ERR_CUDA;
    }
    if (cudaMalloc(&ctx->d_err, 4 * sizeof(int)) != cudaSuccess) {
        delete ctx;
        return GK_ERR_CUDA;
    }
    cudaMemset(ctx->d_err, 0, 4 * sizeof(int));
    if (workspace_bytes) {
        if (cudaMalloc(&ctx->ws, workspace_bytes) != cudaSuccess) {
            cudaFree(ctx->d_err);
            delete ctx;
            return GK_ERR_CUDA;
        }
        ctx->ws_bytes = workspace_bytes;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        gk_ctx_destroy(ctx);
        return GK_ERR_CUDA;
    }
    *out = ctx;
    return GK_OK;
}

void gk_ctx_destroy(gk_ctx* ctx) {
    if (!ctx) return;
    if (ctx->d_err) cudaFree(ctx->d_err);
    if (ctx->ws) cudaFree(ctx->ws);
    delete ctx;
}

gk_status gk_ctx_set_stream(gk_ctx* ctx, void* cuda_stream) {
    if (!ctx) return GK_ERR_ARG;
    ctx->stream = static_cast<cudaStream_t>(cuda_stream);
    return GK_OK;
}

gk_status gk_set_math(gk_ctx* ctx, int math) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, math == GK_MATH_FP32 || math == GK_MATH_3XTF32, GK_ERR_ARG, "gk_set_math: unknown mode %d", math);
    ctx->math = math;
    return GK_OK;
}

gk_status gk_sync(gk_ctx* ctx) {
    if (!ctx) return GK_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return fail(ctx, GK_ERR_CUDA, "gk_sync: %s", cudaGetErrorString(e));
    int err = 0;
    e = cudaMemcpy(&err, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(ctx, GK_ERR_CUDA, "gk_sync: %s", cudaGetErrorString(e));
    if (err) {
        cudaMemset(ctx->d_err, 0, sizeof(int));
        return fail(ctx, err, "kernel reported error %d", err);
    }
    return GK_OK;
}

const char* gk_last_error(gk_ctx* ctx) { return ctx ? ctx->msg : "no context"; }

int64_t gk_launch_count(gk_ctx* ctx) { return ctx ? ctx->launches : -1; }

// ------------------------------------------------------------------- flat layout
int64_t gk_gpt_numel(const gk_gpt_cfg* c) {
    if (!c || c->V <= 0 || c->T <= 0 || c->C <= 0 || c->L <= 0) return -1;
    int64_t C = c->C;
    return (int64_t)c->V * C + (int64_t)c->T * C + (int64_t)c->L * (12 * C * C + 13 * C) + 2 * C;
}

int64_t gk_gpt_n_decay(const gk_gpt_cfg* c) {
    if (!c || c->V <= 0 || c->T <= 0 || c->C <= 0 || c->L <= 0) return -1;
    int64_t C = c->C;
    return (int64_t)c->V * C + (int64_t)c->T * C + (int64_t)c->L * 12 * C * C;
}

int64_t gk_gpt_offset(const gk_gpt_cfg* c, int which, int layer) {
    if (!c || c->V <= 0 || c->T <= 0 || c->C <= 0 || c->L <= 0 || which < 0 || which >= GK_T_COUNT) return -1;
    int64_t C = c->C;
    int64_t VC = (int64_t)c->V * C, TC = (int64_t)c->T * C;
    if (which == GK_T_WTE) return 0;
    if (which == GK_T_WPE) return VC;
    int64_t nd = gk_gpt_n_decay(c);
    if (which == GK_T_LNF_W) return nd + (int64_t)c->L * 13 * C;
    if (which == GK_T_LNF_B) return nd + (int64_t)c->L * 13 * C + C;
    if (layer < 0 || layer >= c->L) return -1;
    int64_t mats = VC + TC + (int64_t)layer * 12 * C * C;
    int64_t vecs = nd + (int64_t)layer * 13 * C;
    switch (which) {
        case GK_T_ATTN_W: return mats;
        case GK_T_ATTNPROJ_W: return mats + 3 * C * C;
        case GK_T_FC_W: return mats + 4 * C * C;
        case GK_T_MLPPROJ_W: return mats + 8 * C * C;
        case GK_T_LN1_W: return vecs;
        case GK_T_LN1_B: return vecs + C;
        case GK_T_ATTN_B: return vecs + 2 * C;
        case GK_T_ATTNPROJ_B: return vecs + 5 * C;
        case GK_T_LN2_W: return vecs + 6 * C;
        case GK_T_LN2_B: return vecs + 7 * C;
        case GK_T_FC_B: return vecs + 8 * C;
        case GK_T_MLPPROJ_B: return vecs + 12 * C;
        default: return -1;
    }
}

}  // extern "C"
