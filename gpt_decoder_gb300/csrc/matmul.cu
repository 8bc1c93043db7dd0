// MatMul / MatMulT entry points ([LM1] = "Build a language model in C# from scratch (1):
// the Autograd engine", Ops: MatMul listing, backward rule, op table) mapped onto the
// internal GEMM, plus the deterministic column sum used for bias gradients.
#include <algorithm>

#include "gemm.cuh"

namespace gk {
namespace {

constexpr int COLSUM_VEC = 8;    // columns per thread (one 16-byte bf16 load, two float4 loads)
constexpr int COLSUM_WARPS = 8;  // warps per block, each on its own rows of the same 256 columns

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]) {
    if constexpr (sizeof(T) == 2) {
        uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __low2float(h[k]);
            v[2 * k + 1] = __high2float(h[k]);
        }
    } else {
        float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// partial[s][c] for column block blockIdx.x (256 columns: 8 per lane) and split s = blockIdx.y:
// warp w of the block sums rows s*8 + w + k*S*8 (k = 0, 1, ...) with four running sums
// (k mod 4), the four are added, then the 8 warp sums in warp order: a fixed summation order.
template <typename T>
__global__ void __launch_bounds__(COLSUM_WARPS * 32)
    colsum_partial_kernel(const T* __restrict__ src, int64_t ld, int64_t rows, int64_t cols, int vec,
                          float* __restrict__ partial) {
    __shared__ float red[COLSUM_WARPS][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t c0 = (int64_t)blockIdx.x * 256 + lane * COLSUM_VEC;
    const int64_t stride = (int64_t)gridDim.y * COLSUM_WARPS;
    float acc[4][COLSUM_VEC];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int k = 0; k < COLSUM_VEC; ++k) acc[u][k] = 0.f;
    int64_t r = (int64_t)blockIdx.y * COLSUM_WARPS + warp;
    if (vec && c0 + COLSUM_VEC <= cols) {
        for (; r + 3 * stride < rows; r += 4 * stride) {
            float v[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) load8<T>(src + (r + u * stride) * ld + c0, v[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[u][k] += v[u][k];
        }
        for (; r < rows; r += stride) {
            float v[8];
            load8<T>(src + r * ld + c0, v);
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[0][k] += v[k];
        }
    } else if (c0 < cols) {
        for (; r < rows; r += stride)
            for (int k = 0; k < COLSUM_VEC && c0 + k < cols; ++k) acc[0][k] += load_as_f32(src + r * ld + c0 + k);
    }
#pragma unroll
    for (int k = 0; k < COLSUM_VEC; ++k)
        red[warp][lane * COLSUM_VEC + k] = (acc[0][k] + acc[1][k]) + (acc[2][k] + acc[3][k]);
    __syncthreads();
    const int64_t c = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (c < cols) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < COLSUM_WARPS; ++w) t += red[w][threadIdx.x];
        partial[(int64_t)blockIdx.y * cols + c] = t;
    }
}

// dst[c] += sum_s partial[s][c]: 32 warps per 32 columns, warp w sums slots w, w + 32, ...
// (four independent running sums, so four loads are in flight), then the warp sums are added
// in warp order (fixed order, deterministic).
constexpr int COLSUM_RED_WARPS = 32;
__global__ void __launch_bounds__(COLSUM_RED_WARPS * 32)
    colsum_reduce_kernel(const float* __restrict__ partial, int splits, int64_t cols, float* dst) {
    __shared__ float red[COLSUM_RED_WARPS][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t c = (int64_t)blockIdx.x * 32 + lane;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < cols) {
        int s = warp;
        for (; s + 3 * COLSUM_RED_WARPS < splits; s += 4 * COLSUM_RED_WARPS)
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] += partial[(int64_t)(s + u * COLSUM_RED_WARPS) * cols + c];
        for (; s < splits; s += COLSUM_RED_WARPS) a[0] += partial[(int64_t)s * cols + c];
    }
    red[warp][lane] = (a[0] + a[1]) + (a[2] + a[3]);
    __syncthreads();
    if (warp == 0 && c < cols) {
        float t = 0.f;
        for (int w = 0; w < COLSUM_RED_WARPS; ++w) t += red[w][lane];
        dst[c] += t;
    }
}

// Resident blocks of colsum_partial_kernel<T> per SM (the grid is sized to one full wave).
template <typename T>
int colsum_blocks_per_sm() {
    static int n = 0;
    if (n == 0) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, colsum_partial_kernel<T>, COLSUM_WARPS * 32, 0) !=
                cudaSuccess || b < 1)
            b = 1;
        n = b;
    }
    return n;
}

}  // namespace

gk_status colsum_add(gk_ctx* ctx, const void* src, int64_t ld, int dtype, int64_t rows, int64_t cols, float* dst) {
    // one full wave of resident blocks (a second, partial wave would leave most SMs idle
    // while it drains)
    const int64_t col_blocks = cdiv(cols, 256);
    const int64_t resident =
        (int64_t)ctx->num_sms * (dtype == GK_F32 ? colsum_blocks_per_sm<float>() : colsum_blocks_per_sm<__nv_bfloat16>());
    int splits = (int)std::max<int64_t>(1, std::min<int64_t>({resident / col_blocks, cdiv(rows, COLSUM_WARPS), 1024}));
    float* partial = (float*)workspace(ctx, (size_t)splits * cols * sizeof(float));
    GK_REQUIRE(ctx, partial, GK_ERR_WORKSPACE, "bias gradient needs %lld workspace bytes",
               (long long)splits * cols * 4);
    GK_REQUIRE(ctx, col_blocks < (1ll << 31), GK_ERR_UNSUPPORTED, "bias gradient: too many columns");
    int esize = dtype == GK_F32 ? 4 : 2;
    int vec = aligned16(src) && ((ld * esize) % 16 == 0);
    dim3 grid((unsigned)col_blocks, (unsigned)splits);
    if (dtype == GK_F32)
        colsum_partial_kernel<float><<<grid, COLSUM_WARPS * 32, 0, ctx->stream>>>((const float*)src, ld, rows, cols,
                                                                                vec, partial);
    else
        colsum_partial_kernel<__nv_bfloat16><<<grid, COLSUM_WARPS * 32, 0, ctx->stream>>>(
            (const __nv_bfloat16*)src, ld, rows, cols, vec, partial);
    GK_TRY(launched(ctx, "colsum_partial"));
    colsum_reduce_kernel<<<(unsigned)cdiv(cols, 32), COLSUM_RED_WARPS * 32, 0, ctx->stream>>>(partial, splits, cols,
                                                                                             dst);
    return launched(ctx, "colsum_reduce");
}

gk_status gemm(gk_ctx* ctx, const Gemm& g) {
    if (g.M == 0 || g.N == 0) return GK_OK;
    if (g.ab_dtype == GK_BF16) {
        gk_status s = gemm_tc(ctx, g);
        if (s != GK_ERR_UNSUPPORTED) return s;
    }
    if (g.ab_dtype == GK_F32 && ctx->math == GK_MATH_3XTF32) {
        // float32 products with float32 results; other output types (a bf16 result of float32
        // operands) keep the float32 FMA kernel
        gk_status s = gemm_3xtf32(ctx, g);
        if (s != GK_ERR_UNSUPPORTED) return s;
    }
    return gemm_simt(ctx, g);
}

}  // namespace gk

using namespace gk;

static bool dtype_ok(int d) { return d == GK_F32 || d == GK_BF16; }
static bool out_dtype_ok(int d) { return d == GK_F32 || d == GK_BF16 || d == GK_BF16X2; }

extern "C" {

gk_status gk_matmul_fwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W, int64_t ldw, int transW,
                        const float* bias, const float* residual, int64_t ldr, void* Y, int64_t ldy, int y_dtype,
                        int64_t N, int64_t K, int64_t M, int act, void* preact, int64_t ldp, const void* X_lo,
                        const void* W_lo) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, X && W && Y && N >= 0 && K >= 0 && M >= 0, GK_ERR_ARG, "gk_matmul_fwd: bad argument");
    GK_REQUIRE(ctx, dtype_ok(dtype) && out_dtype_ok(y_dtype), GK_ERR_ARG, "gk_matmul_fwd: bad dtype");
    GK_REQUIRE(ctx, (!X_lo && !W_lo) || dtype == GK_BF16, GK_ERR_ARG, "gk_matmul_fwd: low planes need bf16 operands");
    GK_REQUIRE(ctx, ldx >= K && ldy >= M && ldw >= (transW ? K : M), GK_ERR_ARG, "gk_matmul_fwd: stride too small");
    GK_REQUIRE(ctx, !residual || ldr >= M, GK_ERR_ARG, "gk_matmul_fwd: residual stride too small");
    GK_REQUIRE(ctx, act == GK_ACT_NONE || (act == GK_ACT_GELU && preact && ldp >= M), GK_ERR_ARG,
               "gk_matmul_fwd: GELU needs a preact buffer");
    GK_REQUIRE(ctx, !(residual && (const void*)residual == Y) || y_dtype == GK_F32, GK_ERR_ARG,
               "gk_matmul_fwd: in-place residual needs float32 Y");
    if (N == 0 || M == 0) return GK_OK;
    Gemm g;
    g.M = N; g.N = M; g.K = K;
    g.A = X; g.lda = ldx; g.a_kmajor = true;
    g.B = W; g.ldb = ldw; g.b_kmajor = transW != 0;
    g.ab_dtype = dtype;
    g.C = Y; g.ldc = ldy; g.c_dtype = y_dtype == GK_BF16X2 ? GK_BF16 : y_dtype;
    if (y_dtype == GK_BF16X2) g.c_plane = N * ldy;
    g.bias = bias; g.residual = residual; g.ldr = ldr;
    if (residual && (const void*)residual == Y && ldr == ldy && act == GK_ACT_NONE) {
        // in place, Y += X W + bias: an accumulation, which the tensor-core epilogue does by TMA
        // reduce-add (no read of the residual through the SM) with the same sum
        g.residual = nullptr;
        g.accumulate = true;
    }
    g.A_lo = X_lo; g.B_lo = W_lo;
    if (act == GK_ACT_GELU) {
        g.epi = EPI_GELU; g.aux = preact; g.ldaux = ldp; g.aux_dtype = g.c_dtype;
    }
    if (K == 0) {
        // no products: the result is the epilogue of zero (still a kernel, for uniformity)
        return gemm_simt(ctx, g);
    }
    return gemm(ctx, g);
}

gk_status gk_matmul_bwd(gk_ctx* ctx, int dtype, const void* X, int64_t ldx, const void* W, int64_t ldw, int transW,
                        const void* dY, int64_t lddy, void* dX, int64_t lddx, int dx_dtype, int accumulate_dX,
                        const void* preact_X, int64_t ldp, float* dW, int64_t lddw, float* dbias, int64_t N,
                        int64_t K, int64_t M) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, dY && N >= 0 && K >= 0 && M >= 0 && lddy >= M, GK_ERR_ARG, "gk_matmul_bwd: bad argument");
    GK_REQUIRE(ctx, dtype_ok(dtype), GK_ERR_ARG, "gk_matmul_bwd: bad dtype");
    if (dX && N > 0 && K > 0) {
        GK_REQUIRE(ctx, W && dtype_ok(dx_dtype) && lddx >= K && ldw >= (transW ? K : M), GK_ERR_ARG,
                   "gk_matmul_bwd: bad dX arguments");
        GK_REQUIRE(ctx, !accumulate_dX || dx_dtype == GK_F32, GK_ERR_ARG, "gk_matmul_bwd: accumulate needs float32 dX");
        GK_REQUIRE(ctx, !preact_X || ldp >= K, GK_ERR_ARG, "gk_matmul_bwd: preact stride too small");
        Gemm g;
        g.M = N; g.N = K; g.K = M;
        g.A = dY; g.lda = lddy; g.a_kmajor = true;
        g.B = W; g.ldb = ldw; g.b_kmajor = transW == 0;
        g.ab_dtype = dtype;
        g.C = dX; g.ldc = lddx; g.c_dtype = dx_dtype;
        g.accumulate = accumulate_dX != 0;
        if (preact_X) {
            g.epi = EPI_DGELU; g.aux = const_cast<void*>(preact_X); g.ldaux = ldp; g.aux_dtype = dtype;
        }
        GK_TRY(M == 0 ? gemm_simt(ctx, g) : gemm(ctx, g));
    }
    if (dW && N > 0 && K > 0 && M > 0) {
        GK_REQUIRE(ctx, X && ldx >= K && lddw >= (transW ? K : M), GK_ERR_ARG, "gk_matmul_bwd: bad dW arguments");
        Gemm g;
        if (!transW) {
            g.M = K; g.N = M; g.K = N;
            g.A = X; g.lda = ldx; g.a_kmajor = false;
            g.B = dY; g.ldb = lddy; g.b_kmajor = false;
        } else {
            g.M = M; g.N = K; g.K = N;
            g.A = dY; g.lda = lddy; g.a_kmajor = false;
            g.B = X; g.ldb = ldx; g.b_kmajor = false;
        }
        g.ab_dtype = dtype;
        g.C = dW; g.ldc = lddw; g.c_dtype = GK_F32;
        g.accumulate = true;
        GK_TRY(gemm(ctx, g));
    }
    if (dbias && N > 0) GK_TRY(colsum_add(ctx, dY, lddy, dtype, N, M, dbias));
    return GK_OK;
}

}  // extern "C"
