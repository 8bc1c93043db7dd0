// Causal multi-head self-attention, forward and backward, without materialising the
// T x T score matrix (online softmax over key tiles; the backward recomputes P from the
// saved log-sum-exp). [LM1] = "Build a language model in C# from scratch (1)", op table
// (BatchMatMulT, CausalSoftmax, BatchMatMul, SplitHeads, MergeHeads); [LM4] = "... (4):
// running GPT-2 weights", "The 12 tensors we do not use" (mask by arithmetic, visible =
// i + 1) and "Generation with a KV cache" (scale 1/sqrt(head size)).
//
// Each query (forward, dq) or key (dk, dv) row is owned by a group of 4 consecutive lanes;
// each lane holds hs/4 of the row's dimensions in registers, and dot products are finished
// with two xor-shuffles inside the group. Key / query tiles are staged in shared memory as
// float32. Scores, softmax and accumulation are float32.
#include <math.h>

#include "gemm.cuh"

using namespace gk;

namespace {

constexpr int G = 4;        // lanes per row
constexpr int ROWS = 32;    // rows (queries or keys) per block -> 128 threads
constexpr int TILE = 32;    // rows of the other side staged per shared-memory tile

template <int D>
__device__ __forceinline__ float group_dot(const float* a, const float* b) {
    float s = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) s = fmaf(a[d], b[d], s);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    return s;
}

// Stage rows [r0, r0 + TILE) of one head's column block `col0` of a [B*T, ld] tensor.
template <typename T, int HS>
__device__ __forceinline__ void stage(float (*S)[HS + 1], const T* __restrict__ base, int64_t ld, int64_t rowbase,
                                      int r0, int T_, int col0) {
    for (int e = threadIdx.x; e < TILE * HS; e += blockDim.x) {
        int r = e / HS, d = e % HS;
        int t = r0 + r;
        S[r][d] = t < T_ ? load_as_f32(base + (rowbase + t) * ld + col0 + d) : 0.f;
    }
}

template <typename T, int HS>
__global__ void __launch_bounds__(ROWS* G) attn_fwd_kernel(const T* __restrict__ qkv, T* __restrict__ y,
                                                            float* __restrict__ lse, int Bn, int T_, int H) {
    constexpr int D = HS / G;
    __shared__ float Ks[TILE][HS + 1];
    __shared__ float Vs[TILE][HS + 1];
    const int C = H * HS;
    const int64_t ld = 3 * (int64_t)C;
    int bh = blockIdx.y, b = bh / H, h = bh % H;
    int64_t rowbase = (int64_t)b * T_;
    int qi = blockIdx.x * ROWS + threadIdx.x / G;
    int g = threadIdx.x % G;
    bool valid = qi < T_;
    const float scale = rsqrtf((float)HS);
    float q[D], o[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        q[d] = valid ? load_as_f32(qkv + (rowbase + qi) * ld + h * HS + g * D + d) : 0.f;
        o[d] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    int last = min(T_ - 1, blockIdx.x * ROWS + ROWS - 1);
    for (int j0 = 0; j0 <= last; j0 += TILE) {
        __syncthreads();
        stage<T, HS>(Ks, qkv, ld, rowbase, j0, T_, C + h * HS);
        stage<T, HS>(Vs, qkv, ld, rowbase, j0, T_, 2 * C + h * HS);
        __syncthreads();
        float s[TILE];
        float mt = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < TILE; ++jj) {
            float v = group_dot<D>(q, &Ks[jj][g * D]) * scale;
            s[jj] = (j0 + jj <= qi) ? v : -INFINITY;
            mt = fmaxf(mt, s[jj]);
        }
        if (mt == -INFINITY) continue;  // no visible key in this tile for this row
        float mn = fmaxf(m, mt);
        float corr = expf(m - mn);  // exp(-inf) = 0 on the first visible tile
        l *= corr;
#pragma unroll
        for (int d = 0; d < D; ++d) o[d] *= corr;
#pragma unroll
        for (int jj = 0; jj < TILE; ++jj) {
            float p = expf(s[jj] - mn);
            l += p;
#pragma unroll
            for (int d = 0; d < D; ++d) o[d] = fmaf(p, Vs[jj][g * D + d], o[d]);
        }
        m = mn;
    }
    if (!valid) return;
    float inv = 1.f / l;
#pragma unroll
    for (int d = 0; d < D; ++d) store_from_f32(y + (rowbase + qi) * C + h * HS + g * D + d, o[d] * inv);
    if (g == 0) lse[(int64_t)bh * T_ + qi] = m + logf(l);
}

// Dvec[b, h, i] = sum_d dy[i, h*hs + d] * y[i, h*hs + d]  (rowsum(dP * P) of the softmax bwd)
template <typename T>
__global__ void attn_dvec_kernel(const T* __restrict__ y, const T* __restrict__ dy, float* __restrict__ dvec,
                                 int64_t rows, int T_, int H, int hs) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * H) return;
    int64_t r = i / H;
    int h = (int)(i % H);
    int64_t C = (int64_t)H * hs;
    float s = 0.f;
    for (int d = 0; d < hs; ++d) s += load_as_f32(dy + r * C + h * hs + d) * load_as_f32(y + r * C + h * hs + d);
    int64_t b = r / T_, t = r % T_;
    dvec[(b * H + h) * T_ + t] = s;
}

// dk and dv for a tile of keys, looping over every query tile at or after the keys.
template <typename T, int HS>
__global__ void __launch_bounds__(ROWS* G) attn_bwd_dkdv_kernel(const T* __restrict__ qkv, const T* __restrict__ dy,
                                                                 const float* __restrict__ lse,
                                                                 const float* __restrict__ dvec, T* __restrict__ dqkv,
                                                                 int T_, int H) {
    constexpr int D = HS / G;
    __shared__ float Qs[TILE][HS + 1];
    __shared__ float Os[TILE][HS + 1];
    __shared__ float Ls[TILE], Ds[TILE];
    const int C = H * HS;
    const int64_t ld = 3 * (int64_t)C;
    int bh = blockIdx.y, b = bh / H, h = bh % H;
    int64_t rowbase = (int64_t)b * T_;
    int kj = blockIdx.x * ROWS + threadIdx.x / G;
    int g = threadIdx.x % G;
    bool valid = kj < T_;
    const float scale = rsqrtf((float)HS);
    float k[D], v[D], dk[D], dv[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        k[d] = valid ? load_as_f32(qkv + (rowbase + kj) * ld + C + h * HS + g * D + d) : 0.f;
        v[d] = valid ? load_as_f32(qkv + (rowbase + kj) * ld + 2 * C + h * HS + g * D + d) : 0.f;
        dk[d] = dv[d] = 0.f;
    }
    int first = (blockIdx.x * ROWS / TILE) * TILE;
    for (int i0 = first; i0 < T_; i0 += TILE) {
        __syncthreads();
        stage<T, HS>(Qs, qkv, ld, rowbase, i0, T_, h * HS);
        stage<T, HS>(Os, dy, C, rowbase, i0, T_, h * HS);
        for (int e = threadIdx.x; e < TILE; e += blockDim.x) {
            int t = i0 + e;
            Ls[e] = t < T_ ? lse[(int64_t)bh * T_ + t] : 0.f;
            Ds[e] = t < T_ ? dvec[(int64_t)bh * T_ + t] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int ii = 0; ii < TILE; ++ii) {
            int qi = i0 + ii;
            float s = group_dot<D>(k, &Qs[ii][g * D]) * scale;
            float dp = group_dot<D>(v, &Os[ii][g * D]);
            bool vis = valid && qi < T_ && qi >= kj;
            float p = vis ? expf(s - Ls[ii]) : 0.f;
            float ds = p * (dp - Ds[ii]) * scale;
#pragma unroll
            for (int d = 0; d < D; ++d) {
                dv[d] = fmaf(p, Os[ii][g * D + d], dv[d]);
                dk[d] = fmaf(ds, Qs[ii][g * D + d], dk[d]);
            }
        }
    }
    if (!valid) return;
#pragma unroll
    for (int d = 0; d < D; ++d) {
        store_from_f32(dqkv + (rowbase + kj) * ld + C + h * HS + g * D + d, dk[d]);
        store_from_f32(dqkv + (rowbase + kj) * ld + 2 * C + h * HS + g * D + d, dv[d]);
    }
}

// dq for a tile of queries, looping over the key tiles up to the queries.
template <typename T, int HS>
__global__ void __launch_bounds__(ROWS* G) attn_bwd_dq_kernel(const T* __restrict__ qkv, const T* __restrict__ dy,
                                                               const float* __restrict__ lse,
                                                               const float* __restrict__ dvec, T* __restrict__ dqkv,
                                                               int T_, int H) {
    constexpr int D = HS / G;
    __shared__ float Ks[TILE][HS + 1];
    __shared__ float Vs[TILE][HS + 1];
    const int C = H * HS;
    const int64_t ld = 3 * (int64_t)C;
    int bh = blockIdx.y, b = bh / H, h = bh % H;
    int64_t rowbase = (int64_t)b * T_;
    int qi = blockIdx.x * ROWS + threadIdx.x / G;
    int g = threadIdx.x % G;
    bool valid = qi < T_;
    const float scale = rsqrtf((float)HS);
    float q[D], o[D], dq[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        q[d] = valid ? load_as_f32(qkv + (rowbase + qi) * ld + h * HS + g * D + d) : 0.f;
        o[d] = valid ? load_as_f32(dy + (rowbase + qi) * C + h * HS + g * D + d) : 0.f;
        dq[d] = 0.f;
    }
    float L = valid ? lse[(int64_t)bh * T_ + qi] : 0.f;
    float Dq = valid ? dvec[(int64_t)bh * T_ + qi] : 0.f;
    int last = min(T_ - 1, blockIdx.x * ROWS + ROWS - 1);
    for (int j0 = 0; j0 <= last; j0 += TILE) {
        __syncthreads();
        stage<T, HS>(Ks, qkv, ld, rowbase, j0, T_, C + h * HS);
        stage<T, HS>(Vs, qkv, ld, rowbase, j0, T_, 2 * C + h * HS);
        __syncthreads();
#pragma unroll 4
        for (int jj = 0; jj < TILE; ++jj) {
            float s = group_dot<D>(q, &Ks[jj][g * D]) * scale;
            float dp = group_dot<D>(o, &Vs[jj][g * D]);
            bool vis = valid && (j0 + jj) <= qi;
            float p = vis ? expf(s - L) : 0.f;
            float ds = p * (dp - Dq) * scale;
#pragma unroll
            for (int d = 0; d < D; ++d) dq[d] = fmaf(ds, Ks[jj][g * D + d], dq[d]);
        }
    }
    if (!valid) return;
#pragma unroll
    for (int d = 0; d < D; ++d) store_from_f32(dqkv + (rowbase + qi) * ld + h * HS + g * D + d, dq[d]);
}

template <typename T, int HS>
gk_status fwd_typed(gk_ctx* ctx, const void* qkv, void* y, float* lse, int B, int T_, int H) {
    dim3 grid((unsigned)cdiv(T_, ROWS), (unsigned)(B * H));
    attn_fwd_kernel<T, HS><<<grid, ROWS * G, 0, ctx->stream>>>((const T*)qkv, (T*)y, lse, B, T_, H);
    return launched(ctx, "attn_fwd");
}

template <typename T, int HS>
gk_status bwd_typed(gk_ctx* ctx, const void* qkv, const void* y, const float* lse, const void* dy, void* dqkv,
                    float* dvec, int B, int T_, int H) {
    int64_t rows = (int64_t)B * T_;
    attn_dvec_kernel<T><<<(unsigned)cdiv(rows * H, 256), 256, 0, ctx->stream>>>((const T*)y, (const T*)dy, dvec, rows,
                                                                              T_, H, HS);
    GK_TRY(launched(ctx, "attn_dvec"));
    dim3 grid((unsigned)cdiv(T_, ROWS), (unsigned)(B * H));
    attn_bwd_dkdv_kernel<T, HS><<<grid, ROWS * G, 0, ctx->stream>>>((const T*)qkv, (const T*)dy, lse, dvec, (T*)dqkv,
                                                                   T_, H);
    GK_TRY(launched(ctx, "attn_bwd_dkdv"));
    attn_bwd_dq_kernel<T, HS><<<grid, ROWS * G, 0, ctx->stream>>>((const T*)qkv, (const T*)dy, lse, dvec, (T*)dqkv,
                                                                 T_, H);
    return launched(ctx, "attn_bwd_dq");
}

#define GK_HS_SWITCH(hs, FN, T, ...)                   \
    switch (hs) {                                      \
        case 8: return FN<T, 8>(__VA_ARGS__);          \
        case 16: return FN<T, 16>(__VA_ARGS__);        \
        case 24: return FN<T, 24>(__VA_ARGS__);        \
        case 32: return FN<T, 32>(__VA_ARGS__);        \
        case 48: return FN<T, 48>(__VA_ARGS__);        \
        case 64: return FN<T, 64>(__VA_ARGS__);        \
        case 96: return FN<T, 96>(__VA_ARGS__);        \
        case 128: return FN<T, 128>(__VA_ARGS__);      \
        default: break;                                \
    }

}  // namespace

extern "C" {

gk_status gk_attn_fwd(gk_ctx* ctx, int dtype, const void* qkv, void* y, float* lse, int B, int T, int H, int hs) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, qkv && y && lse && B > 0 && T > 0 && H > 0 && hs > 0, GK_ERR_ARG, "gk_attn_fwd: bad argument");
    GK_REQUIRE(ctx, dtype == GK_F32 || dtype == GK_BF16, GK_ERR_ARG, "gk_attn_fwd: bad dtype");
    GK_REQUIRE(ctx, (int64_t)B * H < 65536, GK_ERR_UNSUPPORTED, "gk_attn_fwd: B*H too large");
    if (dtype == GK_F32) {
        if (ctx->math == GK_MATH_3XTF32) {
            gk_status s = attn_fwd_3xtf32(ctx, static_cast<const float*>(qkv), static_cast<float*>(y), lse, B, T, H, hs);
            if (s != GK_ERR_UNSUPPORTED) return s;
        }
        GK_HS_SWITCH(hs, fwd_typed, float, ctx, qkv, y, lse, B, T, H)
    } else {
        gk_status s = attn_fwd_tc(ctx, qkv, y, lse, B, T, H, hs);
        if (s != GK_ERR_UNSUPPORTED) return s;
        GK_HS_SWITCH(hs, fwd_typed, __nv_bfloat16, ctx, qkv, y, lse, B, T, H)
    }
    return fail(ctx, GK_ERR_UNSUPPORTED, "gk_attn_fwd: head size %d not built (8,16,24,32,48,64,96,128)", hs);
}

gk_status gk_attn_bwd(gk_ctx* ctx, int dtype, const void* qkv, const void* y, const float* lse, const void* dy,
                      void* dqkv, int B, int T, int H, int hs) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, qkv && y && lse && dy && dqkv && B > 0 && T > 0 && H > 0 && hs > 0, GK_ERR_ARG,
               "gk_attn_bwd: bad argument");
    GK_REQUIRE(ctx, dtype == GK_F32 || dtype == GK_BF16, GK_ERR_ARG, "gk_attn_bwd: bad dtype");
    GK_REQUIRE(ctx, (int64_t)B * H < 65536, GK_ERR_UNSUPPORTED, "gk_attn_bwd: B*H too large");
    if (dtype == GK_BF16) {
        gk_status s = attn_bwd_tc(ctx, qkv, y, lse, dy, dqkv, B, T, H, hs);
        if (s != GK_ERR_UNSUPPORTED) return s;
    } else if (ctx->math == GK_MATH_3XTF32) {
        gk_status s = attn_bwd_3xtf32(ctx, static_cast<const float*>(qkv), static_cast<const float*>(y), lse,
                                      static_cast<const float*>(dy), static_cast<float*>(dqkv), B, T, H, hs);
        if (s != GK_ERR_UNSUPPORTED) return s;
    }
    float* dvec = (float*)workspace(ctx, (size_t)B * H * T * sizeof(float));
    GK_REQUIRE(ctx, dvec, GK_ERR_WORKSPACE, "gk_attn_bwd: needs %lld workspace bytes", (long long)B * H * T * 4);
    if (dtype == GK_F32) {
        GK_HS_SWITCH(hs, bwd_typed, float, ctx, qkv, y, lse, dy, dqkv, dvec, B, T, H)
    } else {
        GK_HS_SWITCH(hs, bwd_typed, __nv_bfloat16, ctx, qkv, y, lse, dy, dqkv, dvec, B, T, H)
    }
    return fail(ctx, GK_ERR_UNSUPPORTED, "gk_attn_bwd: head size %d not built", hs);
}

}  // extern "C"
