// CUDA-core GEMM: 128x128 output tile per 256-thread block, 8x8 outputs per thread, K
// staged 8 at a time through double-buffered shared memory. Float32 FMA accumulation over
// float32 or bfloat16 operands of either majorness. This is the float32 ("faithful")
// arithmetic of the decoder step's MatMul / MatMulT ([LM1] = "Build a language model in C#
// from scratch (1)", Ops: MatMul listing and op table) and the fallback for shapes the
// tensor-core kernel does not take.
#include "gemm.cuh"

namespace gk {
namespace {

constexpr int BM = 128, BN = 128, BK = 8, THREADS = 256;
constexpr int PAD = 4;

template <typename T, bool KMAJOR>
__device__ __forceinline__ void load_tile(const T* __restrict__ P, const T* __restrict__ Plo, int64_t ld, int64_t rows,
                                          int64_t K, int64_t row0, int64_t k0, float (*S)[BM + PAD]) {
    int t = threadIdx.x;
    if (KMAJOR) {
        // element (r, k) at P[r*ld + k]: thread loads 4 consecutive k of one row
        int r = t >> 1, kk = (t & 1) * 4;
        int64_t gr = row0 + r;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int64_t gk = k0 + kk + i;
            float v = 0.f;
            if (gr < rows && gk < K) {
                v = load_as_f32(P + gr * ld + gk);
                if (Plo) v += load_as_f32(Plo + gr * ld + gk);
            }
            S[kk + i][r] = v;
        }
    } else {
        // element (r, k) at P[k*ld + r]: thread loads 4 consecutive r of one k
        int kk = t >> 5, r = (t & 31) * 4;
        int64_t gk = k0 + kk;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int64_t gr = row0 + r + i;
            float v = 0.f;
            if (gr < rows && gk < K) {
                v = load_as_f32(P + gk * ld + gr);
                if (Plo) v += load_as_f32(Plo + gk * ld + gr);
            }
            S[kk][r + i] = v;
        }
    }
}

template <typename TC>
__device__ __forceinline__ void epilogue_store(const Gemm& g, int64_t m, int64_t n, float v) {
    if (m >= g.M || n >= g.N) return;
    TC* C = static_cast<TC*>(g.C);
    int64_t ci = m * g.ldc + n;
    if (g.bias) v += g.bias[n];
    if (g.residual) v += g.residual[m * g.ldr + n];
    if (g.epi == EPI_GELU) {
        if (g.aux_dtype == GK_F32)
            static_cast<float*>(g.aux)[m * g.ldaux + n] = v;
        else
            static_cast<__nv_bfloat16*>(g.aux)[m * g.ldaux + n] = __float2bfloat16_rn(v);
        v = gelu_tanh(v);
    } else if (g.epi == EPI_DGELU) {
        float pre = g.aux_dtype == GK_F32 ? static_cast<const float*>(g.aux)[m * g.ldaux + n]
                                          : __bfloat162float(static_cast<const __nv_bfloat16*>(g.aux)[m * g.ldaux + n]);
        v *= gelu_tanh_grad(pre);
    }
    if (g.accumulate) v += load_as_f32(C + ci);
    store_from_f32(C + ci, v);
    if (g.c_plane) {
        __nv_bfloat16* Cb = reinterpret_cast<__nv_bfloat16*>(C);
        Cb[ci + g.c_plane] = __float2bfloat16_rn(v - __bfloat162float(Cb[ci]));
    }
}

template <typename TA, bool AK, bool BKM, typename TC>
__global__ void __launch_bounds__(THREADS) gemm_simt_kernel(const Gemm g) {
    __shared__ float As[2][BK][BM + PAD];
    __shared__ float Bs[2][BK][BN + PAD];
    const TA* A = static_cast<const TA*>(g.A);
    const TA* B = static_cast<const TA*>(g.B);
    const TA* Alo = static_cast<const TA*>(g.A_lo);
    const TA* Blo = static_cast<const TA*>(g.B_lo);
    int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    int64_t ktiles = (g.K + BK - 1) / BK;
    load_tile<TA, AK>(A, Alo, g.lda, g.M, g.K, m0, 0, As[0]);
    load_tile<TA, BKM>(B, Blo, g.ldb, g.N, g.K, n0, 0, Bs[0]);
    __syncthreads();
    for (int64_t kt = 0; kt < ktiles; ++kt) {
        int cur = kt & 1;
        if (kt + 1 < ktiles) {
            load_tile<TA, AK>(A, Alo, g.lda, g.M, g.K, m0, (kt + 1) * BK, As[cur ^ 1]);
            load_tile<TA, BKM>(B, Blo, g.ldb, g.N, g.K, n0, (kt + 1) * BK, Bs[cur ^ 1]);
        }
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[8], b[8];
            float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
            float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
            float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][k][tx * 4]);
            float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][k][64 + tx * 4]);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int64_t n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            epilogue_store<TC>(g, m, n, acc[i][j]);
        }
    }
}

template <typename TA, typename TC>
gk_status launch_typed(gk_ctx* ctx, const Gemm& g) {
    dim3 grid((unsigned)cdiv(g.N, BN), (unsigned)cdiv(g.M, BM));
    if (g.a_kmajor && g.b_kmajor)
        gemm_simt_kernel<TA, true, true, TC><<<grid, THREADS, 0, ctx->stream>>>(g);
    else if (g.a_kmajor && !g.b_kmajor)
        gemm_simt_kernel<TA, true, false, TC><<<grid, THREADS, 0, ctx->stream>>>(g);
    else if (!g.a_kmajor && g.b_kmajor)
        gemm_simt_kernel<TA, false, true, TC><<<grid, THREADS, 0, ctx->stream>>>(g);
    else
        gemm_simt_kernel<TA, false, false, TC><<<grid, THREADS, 0, ctx->stream>>>(g);
    return launched(ctx, "gemm_simt");
}

}  // namespace

gk_status gemm_simt(gk_ctx* ctx, const Gemm& g) {
    GK_REQUIRE(ctx, cdiv(g.M, BM) < 65536, GK_ERR_UNSUPPORTED, "gemm_simt: M=%lld too large", (long long)g.M);
    if (g.ab_dtype == GK_F32) {
        return g.c_dtype == GK_F32 ? launch_typed<float, float>(ctx, g) : launch_typed<float, __nv_bfloat16>(ctx, g);
    }
    return g.c_dtype == GK_F32 ? launch_typed<__nv_bfloat16, float>(ctx, g)
                               : launch_typed<__nv_bfloat16, __nv_bfloat16>(ctx, g);
}

}  // namespace gk
