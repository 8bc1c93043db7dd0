// Causal attention of the faithful mode on the tensor cores: its contractions as batched 3xTF32
// products. [LM1] = "Build a language model in C# from scratch (1): the Autograd engine", op
// table: BatchMatMulT (S = Q K^T), CausalSoftmax, BatchMatMul (Y = P V), with their backward
// rules; scale 1/sqrt(hs), masked probabilities exactly 0.
//
// Each (batch row b, head h) is one product of a batch (z = b H + h), so every head's Q K^T,
// P V and the backward's dY V^T, P^T dY, dS K and dS^T Q run as one launch each: the operands
// are TF32 hi / lo planes (value = hi + lo), the scores S are materialised ([T, T] per head,
// float32), and the softmax and its backward are row kernels between the products.
//   forward:  S = Q K^T;  P = softmax(s S) over j <= i (lse saved);  Y = P V
//   backward: S again;  dP = dY V^T;  D_i = sum_d dY_id Y_id;  dS = s P (dP - D);
//             dV = P^T dY;  dQ = dS K;  dK = dS^T Q
// The full square of S is computed (the masked half is discarded by the row kernels). The
// heads are processed in groups whose buffers fit the context's workspace.
#include <math.h>

#include <algorithm>

#include "gemm.cuh"

namespace gk {
namespace {

// Planes of the rows of a [R, K] region, K-major: plane[(zl * R + r) * ldp + k] = split(src_z[r *
// ld + k]) (`kmajor`), or = split(src_z[k * ld + r]) (transposed); src_z = src + (zg / zh) * sb +
// (zg % zh) * sh + zl * sl with zg = z0 + zl. 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) split_batched_kernel(const float* __restrict__ src, int64_t ld, int64_t sb,
                                                            int64_t sh, int64_t sl, int zh, int z0, int R, int K,
                                                            int kmajor, float* __restrict__ hi, float* __restrict__ lo,
                                                            int64_t ldp) {
    __shared__ float t[32][33];
    const int zl = blockIdx.z, zg = z0 + zl;
    const float* s = src + (int64_t)(zg / zh) * sb + (int64_t)(zg % zh) * sh + (int64_t)zl * sl;
    const int r0 = blockIdx.x * 32, k0 = blockIdx.y * 32, tx = threadIdx.x, ty = threadIdx.y;
    float* ph = hi + (int64_t)zl * R * ldp;
    float* pl = lo + (int64_t)zl * R * ldp;
    if (kmajor) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = r0 + ty + 8 * j, k = k0 + tx;
            if (r < R && k < K) {
                float h, l;
                tf32_split(s[(int64_t)r * ld + k], h, l);
                ph[(int64_t)r * ldp + k] = h;
                pl[(int64_t)r * ldp + k] = l;
            }
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int k = k0 + ty + 8 * j, r = r0 + tx;
        t[ty + 8 * j][tx] = (k < K && r < R) ? s[(int64_t)k * ld + r] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = r0 + ty + 8 * j, k = k0 + tx;
        if (r < R && k < K) {
            float h, l;
            tf32_split(t[tx][ty + 8 * j], h, l);
            ph[(int64_t)r * ldp + k] = h;
            pl[(int64_t)r * ldp + k] = l;
        }
    }
}

constexpr int SM_MAXT = 2048;  // widest score row the forward row kernel holds in registers (T / 128 float4 per lane)

// Forward row kernel, one warp per row (zl, i) of the scores S [nz * T, T]: m = max over j <= i
// of s S_ij, lse_i = m + log sum exp(s S_ij - m), P_ij = exp(s S_ij - lse_i) (0 for j > i),
// written as TF32 planes; lse goes to lse[zg * T + i].
__global__ void __launch_bounds__(256) attn_softmax_fwd_kernel(const float* __restrict__ S, int T, int nz, int z0,
                                                               float scale, float* __restrict__ p_hi,
                                                               float* __restrict__ p_lo, float* __restrict__ lse) {
    const int lane = threadIdx.x & 31;
    const int64_t rr = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (rr >= (int64_t)nz * T) return;
    const int zl = (int)(rr / T), i = (int)(rr % T);
    const float* sr = S + rr * T;
    float4 v[SM_MAXT / 128];
#pragma unroll
    for (int u = 0; u < SM_MAXT / 128; ++u) {
        const int j = 4 * (lane + 32 * u);
        v[u] = (j < T && j <= i) ? *reinterpret_cast<const float4*>(sr + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = -INFINITY;
#pragma unroll
    for (int u = 0; u < SM_MAXT / 128; ++u) {
        const int j = 4 * (lane + 32 * u);
        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (j + k <= i && j + k < T) m = fmaxf(m, scale * e[k]);
    }
    m = warp_max(m);
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < SM_MAXT / 128; ++u) {
        const int j = 4 * (lane + 32 * u);
        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (j + k <= i && j + k < T) sum += expf(scale * e[k] - m);
    }
    sum = warp_sum(sum);
    const float L = m + logf(sum);
    if (lane == 0) lse[(int64_t)(z0 + zl) * T + i] = L;
#pragma unroll
    for (int u = 0; u < SM_MAXT / 128; ++u) {
        const int j = 4 * (lane + 32 * u);
        if (j >= T) break;
        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        float h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) tf32_split(j + k <= i ? expf(scale * e[k] - L) : 0.f, h[k], l[k]);
        *reinterpret_cast<float4*>(p_hi + rr * T + j) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(p_lo + rr * T + j) = make_float4(l[0], l[1], l[2], l[3]);
    }
}

// D[zg * T + i] = sum_d dY[b T + i, h hs + d] * Y[b T + i, h hs + d] for every (b, h, i): one warp
// per (row, head).
__global__ void attn_dvec_kernel(const float* __restrict__ y, const float* __restrict__ dy, int B, int T, int H, int hs,
                                 float* __restrict__ D) {
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // (b T + i) * H + h
    if (w >= (int64_t)B * T * H) return;
    const int64_t row = w / H;
    const int h = (int)(w % H), C = H * hs;
    float s = 0.f;
    for (int d = lane; d < hs; d += 32) s += y[row * C + h * hs + d] * dy[row * C + h * hs + d];
    s = warp_sum(s);
    const int b = (int)(row / T), i = (int)(row % T);
    if (lane == 0) D[((int64_t)b * H + h) * T + i] = s;
}

// Backward row kernel, one warp per row (zl, i): P_ij = exp(s S_ij - lse_i) and dS_ij = s P_ij
// (dP_ij - D_i) for j <= i (both 0 above the diagonal). P overwrites S and dS overwrites dP (both
// float32, for the transposed planes), and dS is also written as TF32 planes (row-major).
__global__ void __launch_bounds__(256) attn_softmax_bwd_kernel(float* __restrict__ S, float* __restrict__ dP, int T,
                                                               int nz, int z0, float scale,
                                                               const float* __restrict__ lse,
                                                               const float* __restrict__ D, float* __restrict__ ds_hi,
                                                               float* __restrict__ ds_lo) {
    const int lane = threadIdx.x & 31;
    const int64_t rr = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (rr >= (int64_t)nz * T) return;
    const int zl = (int)(rr / T), i = (int)(rr % T);
    const float L = lse[(int64_t)(z0 + zl) * T + i], Di = D[(int64_t)(z0 + zl) * T + i];
    float* sr = S + rr * T;
    float* dr = dP + rr * T;
    for (int j = 4 * lane; j < T; j += 128) {
        const float4 sv = *reinterpret_cast<const float4*>(sr + j);
        const float4 dv = *reinterpret_cast<const float4*>(dr + j);
        const float se[4] = {sv.x, sv.y, sv.z, sv.w}, de[4] = {dv.x, dv.y, dv.z, dv.w};
        float pe[4], ge[4], h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            pe[k] = j + k <= i ? expf(scale * se[k] - L) : 0.f;
            ge[k] = scale * pe[k] * (de[k] - Di);
            tf32_split(ge[k], h[k], l[k]);
        }
        *reinterpret_cast<float4*>(sr + j) = make_float4(pe[0], pe[1], pe[2], pe[3]);
        *reinterpret_cast<float4*>(dr + j) = make_float4(ge[0], ge[1], ge[2], ge[3]);
        *reinterpret_cast<float4*>(ds_hi + rr * T + j) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(ds_lo + rr * T + j) = make_float4(l[0], l[1], l[2], l[3]);
    }
}

struct Planes {
    float *hi, *lo;
};

// Carve `bytes` (256-aligned) off the workspace cursor.
float* carve(char*& cur, size_t bytes) {
    float* p = reinterpret_cast<float*>(cur);
    cur += (bytes + 255) & ~size_t(255);
    return p;
}

// Batched product C_z = A_z B_z^T over TF32 planes (both K-major), nz products of [M x K] x [K x N].
// The shifts of each operand follow the Gemm::zo convention; ext are the buffers' extents.
struct BatchOp {
    Planes a, b;
    float* c;
    int64_t lda, ldb, ldc;
    int64_t a_ext[2], b_ext[2], c_ext[2];
    int zo[3][2][3];
};

gk_status batched_product(gk_ctx* ctx, const BatchOp& op, int M, int N, int K, int nz, int zh, int z0) {
    Gemm g;
    g.M = M; g.N = N; g.K = K;
    g.A = op.a.hi; g.A_lo = op.a.lo; g.lda = op.lda; g.a_kmajor = true;
    g.B = op.b.hi; g.B_lo = op.b.lo; g.ldb = op.ldb; g.b_kmajor = true;
    g.ab_dtype = GK_F32;
    g.tf32 = true;
    g.C = op.c; g.ldc = op.ldc; g.c_dtype = GK_F32;
    g.nz = nz; g.zh = zh; g.z0 = z0;
    for (int o = 0; o < 3; ++o)
        for (int c = 0; c < 2; ++c)
            for (int t = 0; t < 3; ++t) g.zo[o][c][t] = op.zo[o][c][t];
    for (int c = 0; c < 2; ++c) {
        g.a_ext[c] = op.a_ext[c];
        g.b_ext[c] = op.b_ext[c];
        g.c_ext[c] = op.c_ext[c];
    }
    gk_status s = gemm_tc(ctx, g);
    if (s == GK_ERR_UNSUPPORTED) return fail(ctx, s, "3xTF32 attention: the batched product was refused");
    return s;
}

// zo entry helpers: shift per head, per batch row, per local product
void set_shift(int (&zo)[3][2][3], int o, int c, int per_h, int per_b, int per_local) {
    zo[o][c][0] = per_h;
    zo[o][c][1] = per_b;
    zo[o][c][2] = per_local;
}

gk_status split_batch(gk_ctx* ctx, const float* src, int64_t ld, int64_t sb, int64_t sh, int64_t sl, int zh, int z0,
                      int nz, int R, int K, bool kmajor, Planes dst, int64_t ldp) {
    dim3 grid((unsigned)cdiv(R, 32), (unsigned)cdiv(K, 32), (unsigned)nz);
    split_batched_kernel<<<grid, dim3(32, 8), 0, ctx->stream>>>(src, ld, sb, sh, sl, zh, z0, R, K, kmajor ? 1 : 0,
                                                                dst.hi, dst.lo, ldp);
    return launched(ctx, "tf32_split_batched");
}

bool shape_ok(int T, int hs) { return T % 128 == 0 && T <= SM_MAXT && hs % 32 == 0 && hs <= 256; }

}  // namespace

gk_status attn_fwd_3xtf32(gk_ctx* ctx, const float* qkv, float* y, float* lse, int B, int T, int H, int hs) {
    if (!shape_ok(T, hs)) return GK_ERR_UNSUPPORTED;
    const int C = H * hs, Z = B * H;
    const int64_t N = (int64_t)B * T;
    // workspace: the qkv planes, then per head S, P planes and V^T planes
    const size_t fixed = 2 * ((size_t)N * 3 * C * 4 + 255);
    const size_t per_z = ((size_t)T * T * 4 + 255) * 3 + 2 * ((size_t)hs * T * 4 + 255);
    if (ctx->ws_bytes < fixed + per_z) return GK_ERR_UNSUPPORTED;  // the float32 kernels run instead
    const int zc = (int)std::min<size_t>(Z, (ctx->ws_bytes - fixed) / per_z);
    char* cur = static_cast<char*>(ctx->ws);
    Planes q{carve(cur, (size_t)N * 3 * C * 4), carve(cur, (size_t)N * 3 * C * 4)};
    float* S = carve(cur, (size_t)zc * T * T * 4);
    Planes p{carve(cur, (size_t)zc * T * T * 4), carve(cur, (size_t)zc * T * T * 4)};
    Planes vt{carve(cur, (size_t)zc * hs * T * 4), carve(cur, (size_t)zc * hs * T * 4)};
    GK_TRY(split_planes(ctx, qkv, 3 * C, true, 0, 0, N, 3 * C, q.hi, q.lo, 3 * C));
    const float scale = 1.f / sqrtf((float)hs);
    for (int z0 = 0; z0 < Z; z0 += zc) {
        const int nz = std::min(zc, Z - z0);
        // S_z = Q_z K_z^T: Q at columns h hs, K at C + h hs, rows b T of the qkv planes
        BatchOp s{};
        s.a = q;
        s.b = Planes{q.hi + C, q.lo + C};
        s.c = S;
        s.lda = s.ldb = 3 * C;
        s.ldc = T;
        s.a_ext[0] = 3 * C; s.a_ext[1] = N;
        s.b_ext[0] = 2 * C; s.b_ext[1] = N;
        s.c_ext[0] = T; s.c_ext[1] = (int64_t)nz * T;
        set_shift(s.zo, 0, 0, hs, 0, 0);
        set_shift(s.zo, 0, 1, 0, T, 0);
        set_shift(s.zo, 1, 0, hs, 0, 0);
        set_shift(s.zo, 1, 1, 0, T, 0);
        set_shift(s.zo, 2, 1, 0, 0, T);
        GK_TRY(batched_product(ctx, s, T, T, hs, nz, H, z0));
        attn_softmax_fwd_kernel<<<(unsigned)cdiv((int64_t)nz * T, 8), 256, 0, ctx->stream>>>(S, T, nz, z0, scale, p.hi,
                                                                                           p.lo, lse);
        GK_TRY(launched(ctx, "attn_softmax_tf32"));
        // V_z^T planes [hs, T]
        GK_TRY(split_batch(ctx, qkv + 2 * C, 3 * C, (int64_t)T * 3 * C, hs, 0, H, z0, nz, hs, T, false, vt, T));
        // Y_z = P_z V_z into y at columns h hs, rows b T
        BatchOp o{};
        o.a = p;
        o.b = vt;
        o.c = y;
        o.lda = o.ldb = T;
        o.ldc = C;
        o.a_ext[0] = T; o.a_ext[1] = (int64_t)nz * T;
        o.b_ext[0] = T; o.b_ext[1] = (int64_t)nz * hs;
        o.c_ext[0] = C; o.c_ext[1] = N;
        set_shift(o.zo, 0, 1, 0, 0, T);
        set_shift(o.zo, 1, 1, 0, 0, hs);
        set_shift(o.zo, 2, 0, hs, 0, 0);
        set_shift(o.zo, 2, 1, 0, T, 0);
        GK_TRY(batched_product(ctx, o, T, hs, T, nz, H, z0));
    }
    return GK_OK;
}

gk_status attn_bwd_3xtf32(gk_ctx* ctx, const float* qkv, const float* y, const float* lse, const float* dy, float* dqkv,
                          int B, int T, int H, int hs) {
    if (!shape_ok(T, hs)) return GK_ERR_UNSUPPORTED;
    const int C = H * hs, Z = B * H;
    const int64_t N = (int64_t)B * T;
    // workspace: qkv and dY planes and D, then per head S/P, dP/dS, the dS, P^T and dS^T planes,
    // and the K^T, Q^T and dY^T planes
    const size_t fixed = 2 * ((size_t)N * 3 * C * 4 + 255) + 2 * ((size_t)N * C * 4 + 255) + ((size_t)Z * T * 4 + 255);
    const size_t tt = (size_t)T * T * 4 + 255, ht = (size_t)hs * T * 4 + 255;
    const size_t per_z = 2 * tt + 6 * tt + 6 * ht;
    if (ctx->ws_bytes < fixed + per_z) return GK_ERR_UNSUPPORTED;  // the float32 kernels run instead
    const int zc = (int)std::min<size_t>(Z, (ctx->ws_bytes - fixed) / per_z);
    char* cur = static_cast<char*>(ctx->ws);
    Planes q{carve(cur, (size_t)N * 3 * C * 4), carve(cur, (size_t)N * 3 * C * 4)};
    Planes g{carve(cur, (size_t)N * C * 4), carve(cur, (size_t)N * C * 4)};
    float* D = carve(cur, (size_t)Z * T * 4);
    float* S = carve(cur, (size_t)zc * T * T * 4);
    float* dP = carve(cur, (size_t)zc * T * T * 4);
    Planes ds{carve(cur, (size_t)zc * T * T * 4), carve(cur, (size_t)zc * T * T * 4)};
    Planes pt{carve(cur, (size_t)zc * T * T * 4), carve(cur, (size_t)zc * T * T * 4)};
    Planes dst{carve(cur, (size_t)zc * T * T * 4), carve(cur, (size_t)zc * T * T * 4)};
    Planes kt{carve(cur, (size_t)zc * hs * T * 4), carve(cur, (size_t)zc * hs * T * 4)};
    Planes qt{carve(cur, (size_t)zc * hs * T * 4), carve(cur, (size_t)zc * hs * T * 4)};
    Planes gt{carve(cur, (size_t)zc * hs * T * 4), carve(cur, (size_t)zc * hs * T * 4)};
    GK_TRY(split_planes(ctx, qkv, 3 * C, true, 0, 0, N, 3 * C, q.hi, q.lo, 3 * C));
    GK_TRY(split_planes(ctx, dy, C, true, 0, 0, N, C, g.hi, g.lo, C));
    attn_dvec_kernel<<<(unsigned)cdiv(N * H, 8), 256, 0, ctx->stream>>>(y, dy, B, T, H, hs, D);
    GK_TRY(launched(ctx, "attn_dvec_tf32"));
    const float scale = 1.f / sqrtf((float)hs);
    for (int z0 = 0; z0 < Z; z0 += zc) {
        const int nz = std::min(zc, Z - z0);
        // S again, and dP = dY V^T
        BatchOp s{};
        s.a = q;
        s.b = Planes{q.hi + C, q.lo + C};
        s.c = S;
        s.lda = s.ldb = 3 * C;
        s.ldc = T;
        s.a_ext[0] = 3 * C; s.a_ext[1] = N;
        s.b_ext[0] = 2 * C; s.b_ext[1] = N;
        s.c_ext[0] = T; s.c_ext[1] = (int64_t)nz * T;
        set_shift(s.zo, 0, 0, hs, 0, 0);
        set_shift(s.zo, 0, 1, 0, T, 0);
        set_shift(s.zo, 1, 0, hs, 0, 0);
        set_shift(s.zo, 1, 1, 0, T, 0);
        set_shift(s.zo, 2, 1, 0, 0, T);
        GK_TRY(batched_product(ctx, s, T, T, hs, nz, H, z0));
        BatchOp dp = s;
        dp.a = g;
        dp.b = Planes{q.hi + 2 * C, q.lo + 2 * C};
        dp.c = dP;
        dp.lda = C;
        dp.a_ext[0] = C;
        dp.b_ext[0] = C;
        GK_TRY(batched_product(ctx, dp, T, T, hs, nz, H, z0));
        // P (into S), dS (into dP) and the dS planes
        attn_softmax_bwd_kernel<<<(unsigned)cdiv((int64_t)nz * T, 8), 256, 0, ctx->stream>>>(S, dP, T, nz, z0, scale,
                                                                                           lse, D, ds.hi, ds.lo);
        GK_TRY(launched(ctx, "attn_softmax_bwd_tf32"));
        // transposed planes: P^T, dS^T [T, T] per head; K^T, Q^T, dY^T [hs, T] per head
        GK_TRY(split_batch(ctx, S, T, 0, 0, (int64_t)T * T, H, z0, nz, T, T, false, pt, T));
        GK_TRY(split_batch(ctx, dP, T, 0, 0, (int64_t)T * T, H, z0, nz, T, T, false, dst, T));
        GK_TRY(split_batch(ctx, qkv + C, 3 * C, (int64_t)T * 3 * C, hs, 0, H, z0, nz, hs, T, false, kt, T));
        GK_TRY(split_batch(ctx, qkv, 3 * C, (int64_t)T * 3 * C, hs, 0, H, z0, nz, hs, T, false, qt, T));
        GK_TRY(split_batch(ctx, dy, C, (int64_t)T * C, hs, 0, H, z0, nz, hs, T, false, gt, T));
        // dV = P^T dY, dQ = dS K, dK = dS^T Q: [T x hs] products into dqkv
        BatchOp o{};
        o.lda = o.ldb = T;
        o.ldc = 3 * C;
        o.a_ext[0] = T; o.a_ext[1] = (int64_t)nz * T;
        o.b_ext[0] = T; o.b_ext[1] = (int64_t)nz * hs;
        o.c_ext[0] = 3 * C; o.c_ext[1] = N;
        set_shift(o.zo, 0, 1, 0, 0, T);
        set_shift(o.zo, 1, 1, 0, 0, hs);
        set_shift(o.zo, 2, 0, hs, 0, 0);
        set_shift(o.zo, 2, 1, 0, T, 0);
        o.a = pt; o.b = gt; o.c = dqkv + 2 * C;
        o.c_ext[0] = C;
        GK_TRY(batched_product(ctx, o, T, hs, T, nz, H, z0));
        o.a = ds; o.b = kt; o.c = dqkv;
        GK_TRY(batched_product(ctx, o, T, hs, T, nz, H, z0));
        o.a = dst; o.b = qt; o.c = dqkv + C;
        GK_TRY(batched_product(ctx, o, T, hs, T, nz, H, z0));
    }
    return GK_OK;
}

}  // namespace gk
