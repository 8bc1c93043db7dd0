// Float32 products on the tensor cores in 3xTF32 (the faithful mode's MatMul / MatMulT:
// [LM1] = "Build a language model in C# from scratch (1): the Autograd engine", Ops: MatMul
// listing, backward rule and op table).
//
// A TF32 value keeps 10 of float32's 23 explicit mantissa bits. Every float32 x is written as
// x = hi + lo with hi = tf32(x) (round to nearest, ties away) and lo = tf32(x - hi); x - hi is
// exact in float32, and lo keeps the next 11 significant bits, so hi + lo carries about 22 bits.
// The product A B is then A_hi B_hi + A_hi B_lo + A_lo B_hi, three kind::tf32 tensor-core
// products accumulated in float32 in tensor memory; the dropped A_lo B_lo term is about 2^-22
// of the product (the published 3xTF32 scheme of Ootomo and Yokota, 2022).
//
// The hi / lo planes are written here, K-major, into the context's workspace (an operand stored
// MN-major is transposed on the way, through a shared-memory tile), so the tensor-core kernel
// always reads K-major TF32 tiles. When the planes of the whole product do not fit, the output
// is cut into column blocks and row blocks, and (for epilogues that are plain sums) K into
// slices whose partial products are added into C; the bias and residual go with the first slice.
#include <algorithm>

#include "gemm.cuh"

namespace gk {
namespace {

// K-major source: plane element (r, k) = src[(row0 + r) * ld + k0 + k], k < kc. Each thread
// takes four consecutive k of one row (16-byte accesses when `vec`).
__global__ void tf32_split_rows_kernel(const float* __restrict__ src, int64_t ld, int64_t row0, int64_t k0, int64_t R,
                                       int64_t kc, float* __restrict__ hi, float* __restrict__ lo, int64_t ldp,
                                       int vec) {
    const int64_t q4 = (kc + 3) / 4;
    const int64_t total = R * q4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / q4, k = (i - r * q4) * 4;
        const float* s = src + (row0 + r) * ld + k0 + k;
        float v[4];
        if (vec && k + 3 < kc) {
            const float4 f = *reinterpret_cast<const float4*>(s);
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = k + j < kc ? s[j] : 0.f;
        }
        float h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) tf32_split(v[j], h[j], l[j]);
        *reinterpret_cast<float4*>(hi + r * ldp + k) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(lo + r * ldp + k) = make_float4(l[0], l[1], l[2], l[3]);
    }
}

// MN-major source: plane element (r, k) = src[(k0 + k) * ld + row0 + r]. A 32 x 32 tile per
// block (32 x 8 threads) is read along r and written along k.
__global__ void __launch_bounds__(256) tf32_split_cols_kernel(const float* __restrict__ src, int64_t ld, int64_t row0,
                                                             int64_t k0, int64_t R, int64_t kc, float* __restrict__ hi,
                                                             float* __restrict__ lo, int64_t ldp) {
    __shared__ float t[32][33];
    const int64_t r0 = (int64_t)blockIdx.x * 32, kb = (int64_t)blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t k = kb + ty + 8 * j, r = r0 + tx;
        t[ty + 8 * j][tx] = (k < kc && r < R) ? src[(k0 + k) * ld + row0 + r] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t r = r0 + ty + 8 * j, k = kb + tx;
        if (r < R && k < kc) {
            float h, l;
            tf32_split(t[tx][ty + 8 * j], h, l);
            hi[r * ldp + k] = h;
            lo[r * ldp + k] = l;
        }
    }
}

inline int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// Workspace bytes for planes of an Mc x Kc block of A and an Nc x Kc block of B.
inline size_t plane_bytes(int64_t rows, int64_t kc) { return (size_t)round_up(rows * round_up(kc, 4) * 4, 256); }
inline size_t chunk_bytes(int64_t mc, int64_t nc, int64_t kc) { return 2 * plane_bytes(mc, kc) + 2 * plane_bytes(nc, kc); }

}  // namespace

gk_status split_planes(gk_ctx* ctx, const float* src, int64_t ld, bool kmajor, int64_t row0, int64_t k0, int64_t R,
                       int64_t kc, float* hi, float* lo, int64_t ldp) {
    if (kmajor) {
        const int vec = aligned16(src) && ld % 4 == 0 && k0 % 4 == 0;
        const int64_t work = R * ((kc + 3) / 4);
        const unsigned blocks = (unsigned)std::min<int64_t>(cdiv(work, 256), (int64_t)ctx->num_sms * 16);
        tf32_split_rows_kernel<<<blocks, 256, 0, ctx->stream>>>(src, ld, row0, k0, R, kc, hi, lo, ldp, vec);
        return launched(ctx, "tf32_split_rows");
    }
    GK_REQUIRE(ctx, cdiv(kc, 32) <= 65535, GK_ERR_UNSUPPORTED, "3xTF32: K slice too long");
    dim3 grid((unsigned)cdiv(R, 32), (unsigned)cdiv(kc, 32));
    tf32_split_cols_kernel<<<grid, dim3(32, 8), 0, ctx->stream>>>(src, ld, row0, k0, R, kc, hi, lo, ldp);
    return launched(ctx, "tf32_split_cols");
}

gk_status gemm_3xtf32(gk_ctx* ctx, const Gemm& g) {
    if (g.ab_dtype != GK_F32 || g.tf32 || g.A_lo || g.B_lo || g.ce_mode != CE_NONE || g.c_dtype != GK_F32 ||
        g.c_plane || g.M <= 0 || g.N <= 0 || g.K <= 0)
        return GK_ERR_UNSUPPORTED;
    // K may be cut into slices added into C only when the epilogue is a plain sum (the bias
    // and residual then ride on the first slice)
    const bool k_slices = g.epi == EPI_NONE;
    int64_t Mc = g.M, Nc = g.N, Kc = g.K;
    while (chunk_bytes(Mc, Nc, Kc) > ctx->ws_bytes) {
        const int64_t a = Mc * Kc, b = Nc * Kc;
        if (k_slices && Kc > 512 && Kc >= std::max(Mc, Nc))
            Kc = round_up(cdiv(Kc, 2), 32);
        else if (a >= b && Mc > 128)
            Mc = round_up(cdiv(Mc, 2), 128);
        else if (Nc > 256)
            Nc = round_up(cdiv(Nc, 2), 256);
        else if (Mc > 128)
            Mc = round_up(cdiv(Mc, 2), 128);
        else if (k_slices && Kc > 32)
            Kc = round_up(cdiv(Kc, 2), 32);
        else
            return fail(ctx, GK_ERR_WORKSPACE, "3xTF32 product %lldx%lldx%lld: the workspace (%zu bytes) cannot hold "
                        "its smallest operand block", (long long)g.M, (long long)g.N, (long long)g.K, ctx->ws_bytes);
    }
    char* ws = static_cast<char*>(ctx->ws);
    float* a_hi = reinterpret_cast<float*>(ws);
    float* a_lo = reinterpret_cast<float*>(ws + plane_bytes(Mc, Kc));
    float* b_hi = reinterpret_cast<float*>(ws + 2 * plane_bytes(Mc, Kc));
    float* b_lo = reinterpret_cast<float*>(ws + 2 * plane_bytes(Mc, Kc) + plane_bytes(Nc, Kc));
    const float* A = static_cast<const float*>(g.A);
    const float* B = static_cast<const float*>(g.B);
    const size_t aux_esz = g.aux_dtype == GK_F32 ? 4 : 2;
    // B's planes are written once when one block of B covers the whole product
    const bool b_once = Nc == g.N && Kc == g.K;
    if (b_once) GK_TRY(split_planes(ctx, B, g.ldb, g.b_kmajor, 0, 0, g.N, g.K, b_hi, b_lo, round_up(g.K, 4)));
    for (int64_t m0 = 0; m0 < g.M; m0 += Mc) {
        const int64_t mc = std::min(Mc, g.M - m0);
        for (int64_t k0 = 0; k0 < g.K; k0 += Kc) {
            const int64_t kc = std::min(Kc, g.K - k0), ldp = round_up(kc, 4);
            GK_TRY(split_planes(ctx, A, g.lda, g.a_kmajor, m0, k0, mc, kc, a_hi, a_lo, ldp));
            for (int64_t n0 = 0; n0 < g.N; n0 += Nc) {
                const int64_t nc = std::min(Nc, g.N - n0);
                if (!b_once) GK_TRY(split_planes(ctx, B, g.ldb, g.b_kmajor, n0, k0, nc, kc, b_hi, b_lo, ldp));
                Gemm c = g;
                c.M = mc; c.N = nc; c.K = kc;
                c.A = a_hi; c.A_lo = a_lo; c.lda = ldp; c.a_kmajor = true;
                c.B = b_hi; c.B_lo = b_lo; c.ldb = ldp; c.b_kmajor = true;
                c.tf32 = true;
                c.C = static_cast<float*>(g.C) + m0 * g.ldc + n0;
                c.bias = (k0 == 0 && g.bias) ? g.bias + n0 : nullptr;
                c.residual = (k0 == 0 && g.residual) ? g.residual + m0 * g.ldr + n0 : nullptr;
                c.aux = g.aux ? static_cast<char*>(g.aux) + (m0 * g.ldaux + n0) * aux_esz : nullptr;
                c.accumulate = g.accumulate || k0 > 0;
                GK_TRY(gemm_tc(ctx, c));
            }
        }
    }
    return GK_OK;
}

}  // namespace gk
