// Generic tensor ops of the autograd engine and plain SGD, float32, HBM-bound elementwise
// kernels. [LM1] = "Build a language model in C# from scratch (1)": Ops (Mul and its backward
// rule), the op table (Add with broadcast, Scale, Sum, Tanh), "Why += and not =", Gradient
// Check, The optimizer (SGD); [AD] = "Chain rule and automatic differentiation", Steps 1-5
// (the tanh neuron and its derivative 1 - tanh^2).
//
// Elementwise outputs may alias an input of the same index (y == a, da == g).
// Every backward entry point takes `accumulate`: 0 writes the gradient, 1 adds it to what the
// buffer holds (the pages' += rule, with ZeroGrad the caller's job). Reductions (Sum, the
// broadcast bias gradient) run in a fixed order in double, so results do not depend on timing.
#include <algorithm>

#include "common.cuh"

namespace gk {
namespace {

constexpr int EW_THREADS = 256;

// Grid of a grid-stride elementwise kernel: enough blocks to fill the SMs several times over.
// float4 path: every operand (null ones aside) 16-byte aligned
bool al(const void* p) { return !p || aligned16(p); }
template <typename... Ps>
bool vec4(const Ps*... ps) {
    return (al(ps) && ...);
}

unsigned ew_blocks(const gk_ctx* ctx, int64_t n) {
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(cdiv(n, EW_THREADS), (int64_t)ctx->num_sms * 16));
}

// Elementwise kernels walk float4 groups when every operand is 16-byte aligned (`vec`), then
// the scalar tail; element i of every operand sits at the same index.
template <typename V, typename S>
__device__ __forceinline__ void ew_loops(int64_t n, bool vec, V vbody, S sbody) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t n4 = vec ? n / 4 : 0;
    for (int64_t j = tid; j < n4; j += stride) vbody(j);
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) sbody(i);
}

__device__ __forceinline__ float4 f4(const float* p, int64_t j) { return reinterpret_cast<const float4*>(p)[j]; }
__device__ __forceinline__ void st4(float* p, int64_t j, float4 v) { reinterpret_cast<float4*>(p)[j] = v; }

// y = a + b[i % m] (vec needs m % 4 == 0)
__global__ void add_fwd_kernel(const float* a, const float* b, float* y, int64_t n, int64_t m, bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        const float4 x = f4(a, j), c = f4(b, (4 * j) % m / 4);
        st4(y, j, make_float4(x.x + c.x, x.y + c.y, x.z + c.z, x.w + c.w));
    }, [&](int64_t i) { y[i] = a[i] + b[m == n ? i : i % m]; });
}

// dst (+)= src
__global__ void copy_acc_kernel(const float* src, float* dst, int64_t n, int acc, bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        float4 v = f4(src, j);
        if (acc) {
            const float4 d = f4(dst, j);
            v = make_float4(d.x + v.x, d.y + v.y, d.z + v.z, d.w + v.w);
        }
        st4(dst, j, v);
    }, [&](int64_t i) { dst[i] = acc ? dst[i] + src[i] : src[i]; });
}

// part[p, c] = sum of g[r, c] over the rows r of chunk p ([R, m] row-major), in row order, in
// double-float (the float32 pipe; float64 is a slow one on this GPU)
__global__ void colsum_chunks_kernel(const float* __restrict__ g, int64_t R, int64_t m, int64_t rows_per,
                                     double* __restrict__ part) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= m) return;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per, r1 = min(R, r0 + rows_per);
    float2 s = make_float2(0.f, 0.f);
    for (int64_t r = r0; r < r1; ++r) s = df_add(s, make_float2(g[r * m + c], 0.f));
    part[(int64_t)blockIdx.y * m + c] = (double)s.x + (double)s.y;
}

// db[c] (+)= sum over chunks p in order of part[p, c]
__global__ void colsum_finish_kernel(const double* __restrict__ part, int64_t P, int64_t m, float* __restrict__ db,
                                     int acc) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= m) return;
    double s = 0.0;
    for (int64_t p = 0; p < P; ++p) s += part[p * m + c];
    db[c] = acc ? db[c] + (float)s : (float)s;
}

__global__ void mul_fwd_kernel(const float* a, const float* b, float* y, int64_t n, bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        const float4 x = f4(a, j), z = f4(b, j);
        st4(y, j, make_float4(x.x * z.x, x.y * z.y, x.z * z.z, x.w * z.w));
    }, [&](int64_t i) { y[i] = a[i] * b[i]; });
}

// da (+)= g * b, db (+)= g * a (either may be null)
__global__ void mul_bwd_kernel(const float* g, const float* a, const float* b, float* da, float* db, int64_t n, int acc,
                               bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        const float4 gv = f4(g, j);
        if (da) {
            const float4 bv = f4(b, j);
            float4 v = make_float4(gv.x * bv.x, gv.y * bv.y, gv.z * bv.z, gv.w * bv.w);
            if (acc) {
                const float4 o = f4(da, j);
                v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
            }
            st4(da, j, v);
        }
        if (db) {
            const float4 av = f4(a, j);
            float4 v = make_float4(gv.x * av.x, gv.y * av.y, gv.z * av.z, gv.w * av.w);
            if (acc) {
                const float4 o = f4(db, j);
                v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
            }
            st4(db, j, v);
        }
    }, [&](int64_t i) {
        const float gi = g[i];
        if (da) da[i] = acc ? da[i] + gi * b[i] : gi * b[i];
        if (db) db[i] = acc ? db[i] + gi * a[i] : gi * a[i];
    });
}

// y = s * a (forward), or da (+)= s * g (backward: the same map with accumulation)
__global__ void scale_kernel(const float* a, float s, float* y, int64_t n, int acc, bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        const float4 x = f4(a, j);
        float4 v = make_float4(s * x.x, s * x.y, s * x.z, s * x.w);
        if (acc) {
            const float4 o = f4(y, j);
            v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
        }
        st4(y, j, v);
    }, [&](int64_t i) { y[i] = acc ? y[i] + s * a[i] : s * a[i]; });
}

// Compensated (Kahan) float32 addition: s + c carries the running sum to about one ulp of the
// sum, whatever the number of terms (Kahan 1965).
__device__ __forceinline__ void kahan_add(float& s, float& c, float v) {
    const float y = v - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
}

// part[block] = sum of this block's grid-stride elements, in a fixed order: each aligned float4
// group is added in float ((x + y) + (z + w)); a thread's k-th group goes to its compensated
// float32 chain k % SC (SC independent chains, so SC loads are in flight per round trip), the
// tail to the first; the chains, then the lanes of a warp (xor tree) are combined in double-float,
// the warps in double. Double arithmetic is a slow pipe on this GPU: a per-thread double tree
// over every block ended each wave with microseconds of float64 work.
constexpr int SC = 4;
__global__ void sum_partial_kernel(const float* __restrict__ a, int64_t n, double* __restrict__ part, bool vec) {
    __shared__ double red[EW_THREADS / 32];
    float s4[SC], c4[SC];
#pragma unroll
    for (int k = 0; k < SC; ++k) s4[k] = c4[k] = 0.f;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t n4 = vec ? n / 4 : 0;
    int64_t j = tid;
    for (; j + (SC - 1) * stride < n4; j += SC * stride) {
        float4 v[SC];
#pragma unroll
        for (int k = 0; k < SC; ++k) v[k] = f4(a, j + k * stride);
#pragma unroll
        for (int k = 0; k < SC; ++k) kahan_add(s4[k], c4[k], (v[k].x + v[k].y) + (v[k].z + v[k].w));
    }
#pragma unroll
    for (int k = 0; k < SC - 1; ++k) {  // fewer than SC groups left
        if (j < n4) {
            const float4 v = f4(a, j);
            kahan_add(s4[k], c4[k], (v.x + v.y) + (v.z + v.w));
            j += stride;
        }
    }
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) kahan_add(s4[0], c4[0], a[i]);
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < SC; ++k) s = df_add(s, make_float2(s4[k], -c4[k]));
    for (int o = 16; o > 0; o >>= 1)
        s = df_add(s, make_float2(__shfl_xor_sync(0xffffffffu, s.x, o), __shfl_xor_sync(0xffffffffu, s.y, o)));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = (double)s.x + (double)s.y;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < EW_THREADS / 32; ++w) t += red[w];
        part[blockIdx.x] = t;
    }
}

// y[0] = sum of part[0 .. P): thread t adds part[t], part[t + 256], ... in index order, then
// the 256 thread sums are combined in a fixed tree (lane xor-tree, then warps in order). The
// order depends only on P, so the result is deterministic; one thread walking all P partials
// would wait out P / 4 dependent L2 round trips.
constexpr int SUM_FINISH_THREADS = 256;
__global__ void __launch_bounds__(SUM_FINISH_THREADS) sum_finish_kernel(const double* __restrict__ part, int P,
                                                                      float* __restrict__ y) {
    __shared__ double red[SUM_FINISH_THREADS / 32];
    double t = 0.0;
    for (int p = threadIdx.x; p < P; p += SUM_FINISH_THREADS) t += part[p];
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < SUM_FINISH_THREADS / 32; ++w) s += red[w];
        *y = (float)s;
    }
}

// da (+)= g[0] for every element
__global__ void sum_bwd_kernel(const float* g, float* da, int64_t n, int acc, bool vec) {
    const float gv = *g;
    ew_loops(n, vec, [&](int64_t j) {
        float4 v = make_float4(gv, gv, gv, gv);
        if (acc) {
            const float4 o = f4(da, j);
            v = make_float4(o.x + gv, o.y + gv, o.z + gv, o.w + gv);
        }
        st4(da, j, v);
    }, [&](int64_t i) { da[i] = acc ? da[i] + gv : gv; });
}

__global__ void tanh_fwd_kernel(const float* x, float* y, int64_t n, bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        const float4 v = f4(x, j);
        st4(y, j, make_float4(tanhf(v.x), tanhf(v.y), tanhf(v.z), tanhf(v.w)));
    }, [&](int64_t i) { y[i] = tanhf(x[i]); });
}

// dx (+)= g (1 - y^2), y = tanh(x) saved by the forward
__global__ void tanh_bwd_kernel(const float* y, const float* g, float* dx, int64_t n, int acc, bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        const float4 yv = f4(y, j), gv = f4(g, j);
        float4 v = make_float4(gv.x * (1.f - yv.x * yv.x), gv.y * (1.f - yv.y * yv.y), gv.z * (1.f - yv.z * yv.z),
                               gv.w * (1.f - yv.w * yv.w));
        if (acc) {
            const float4 o = f4(dx, j);
            v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
        }
        st4(dx, j, v);
    }, [&](int64_t i) {
        const float yi = y[i];
        const float v = g[i] * (1.f - yi * yi);
        dx[i] = acc ? dx[i] + v : v;
    });
}

// p -= lr * g
__global__ void sgd_kernel(float* p, const float* g, int64_t n, float lr, bool vec) {
    ew_loops(n, vec, [&](int64_t j) {
        const float4 pv = f4(p, j), gv = f4(g, j);
        st4(p, j, make_float4(pv.x - lr * gv.x, pv.y - lr * gv.y, pv.z - lr * gv.z, pv.w - lr * gv.w));
    }, [&](int64_t i) { p[i] -= lr * g[i]; });
}

}  // namespace
}  // namespace gk

using namespace gk;

extern "C" {

gk_status gk_add_fwd(gk_ctx* ctx, const float* a, const float* b, float* y, int64_t n, int64_t m) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0 && m >= 1 && (n == 0 || n % m == 0), GK_ERR_ARG,
               "gk_add_fwd: b's %lld elements do not tile a's %lld", (long long)m, (long long)n);
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, a && b && y, GK_ERR_ARG, "gk_add_fwd: null pointer");
    add_fwd_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(a, b, y, n, m, vec4(a, b, y) && (m == n || m % 4 == 0));
    return launched(ctx, "add_fwd");
}

gk_status gk_add_bwd(gk_ctx* ctx, const float* g, float* da, float* db, int64_t n, int64_t m, int accumulate) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0 && m >= 1 && (n == 0 || n % m == 0), GK_ERR_ARG,
               "gk_add_bwd: b's %lld elements do not tile a's %lld", (long long)m, (long long)n);
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, g, GK_ERR_ARG, "gk_add_bwd: null gradient");
    if (da) {
        copy_acc_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(g, da, n, accumulate != 0, vec4(g, da));
        GK_TRY(launched(ctx, "add_bwd_a"));
    }
    if (!db) return GK_OK;
    if (m == n) {
        copy_acc_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(g, db, n, accumulate != 0, vec4(g, db));
        return launched(ctx, "add_bwd_b");
    }
    // db = column sums of g viewed as [R, m]: row chunks in parallel, then the chunks in order
    const int64_t R = n / m;
    int64_t P = std::min<int64_t>(R, std::max<int64_t>(1, cdiv((int64_t)ctx->num_sms * 2048, m)));
    P = std::min<int64_t>(P, std::max<int64_t>(1, (int64_t)(ctx->ws_bytes / ((size_t)m * sizeof(double)))));
    const int64_t rows_per = cdiv(R, P);
    P = cdiv(R, rows_per);
    double* part = static_cast<double*>(workspace(ctx, (size_t)P * m * sizeof(double)));
    GK_REQUIRE(ctx, part && P <= 65535, GK_ERR_WORKSPACE, "gk_add_bwd: needs %zu workspace bytes",
               (size_t)P * m * sizeof(double));
    colsum_chunks_kernel<<<dim3((unsigned)cdiv(m, EW_THREADS), (unsigned)P), EW_THREADS, 0, ctx->stream>>>(
        g, R, m, rows_per, part);
    GK_TRY(launched(ctx, "add_bwd_colsum"));
    colsum_finish_kernel<<<(unsigned)cdiv(m, EW_THREADS), EW_THREADS, 0, ctx->stream>>>(part, P, m, db,
                                                                                        accumulate != 0);
    return launched(ctx, "add_bwd_finish");
}

gk_status gk_mul_fwd(gk_ctx* ctx, const float* a, const float* b, float* y, int64_t n) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_mul_fwd: negative size");
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, a && b && y, GK_ERR_ARG, "gk_mul_fwd: null pointer");
    mul_fwd_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(a, b, y, n, vec4(a, b, y));
    return launched(ctx, "mul_fwd");
}

gk_status gk_mul_bwd(gk_ctx* ctx, const float* g, const float* a, const float* b, float* da, float* db, int64_t n,
                     int accumulate) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_mul_bwd: negative size");
    if (n == 0 || (!da && !db)) return GK_OK;
    GK_REQUIRE(ctx, g && (!da || b) && (!db || a), GK_ERR_ARG, "gk_mul_bwd: null pointer");
    mul_bwd_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(g, a, b, da, db, n, accumulate != 0,
                                                                     vec4(g, da ? b : nullptr, db ? a : nullptr, da, db));
    return launched(ctx, "mul_bwd");
}

gk_status gk_scale_fwd(gk_ctx* ctx, const float* a, float s, float* y, int64_t n) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_scale_fwd: negative size");
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, a && y, GK_ERR_ARG, "gk_scale_fwd: null pointer");
    scale_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(a, s, y, n, 0, vec4(a, y));
    return launched(ctx, "scale_fwd");
}

gk_status gk_scale_bwd(gk_ctx* ctx, const float* g, float s, float* da, int64_t n, int accumulate) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_scale_bwd: negative size");
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, g && da, GK_ERR_ARG, "gk_scale_bwd: null pointer");
    scale_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(g, s, da, n, accumulate != 0, vec4(g, da));
    return launched(ctx, "scale_bwd");
}

gk_status gk_sum_fwd(gk_ctx* ctx, const float* a, float* y, int64_t n) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0 && y && (n == 0 || a), GK_ERR_ARG, "gk_sum_fwd: bad argument");
    // one full wave of resident blocks (64 bytes of loads in flight per thread), each thread at
    // least 32 elements
    static int per_sm = 0;
    if (per_sm == 0) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, sum_partial_kernel, EW_THREADS, 0) != cudaSuccess || b < 1)
            b = 1;
        per_sm = b;
    }
    const int P = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(n, EW_THREADS * 32), (int64_t)per_sm * ctx->num_sms));
    double* part = static_cast<double*>(workspace(ctx, (size_t)P * sizeof(double)));
    GK_REQUIRE(ctx, part, GK_ERR_WORKSPACE, "gk_sum_fwd: needs %zu workspace bytes", (size_t)P * sizeof(double));
    sum_partial_kernel<<<P, EW_THREADS, 0, ctx->stream>>>(a, n, part, vec4(a));
    GK_TRY(launched(ctx, "sum_partial"));
    sum_finish_kernel<<<1, SUM_FINISH_THREADS, 0, ctx->stream>>>(part, P, y);
    return launched(ctx, "sum_finish");
}

gk_status gk_sum_bwd(gk_ctx* ctx, const float* g, float* da, int64_t n, int accumulate) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_sum_bwd: negative size");
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, g && da, GK_ERR_ARG, "gk_sum_bwd: null pointer");
    sum_bwd_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(g, da, n, accumulate != 0, vec4(da));
    return launched(ctx, "sum_bwd");
}

gk_status gk_tanh_fwd(gk_ctx* ctx, const float* x, float* y, int64_t n) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_tanh_fwd: negative size");
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, x && y, GK_ERR_ARG, "gk_tanh_fwd: null pointer");
    tanh_fwd_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(x, y, n, vec4(x, y));
    return launched(ctx, "tanh_fwd");
}

gk_status gk_tanh_bwd(gk_ctx* ctx, const float* y, const float* g, float* dx, int64_t n, int accumulate) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_tanh_bwd: negative size");
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, y && g && dx, GK_ERR_ARG, "gk_tanh_bwd: null pointer");
    tanh_bwd_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(y, g, dx, n, accumulate != 0, vec4(y, g, dx));
    return launched(ctx, "tanh_bwd");
}

gk_status gk_sgd_step(gk_ctx* ctx, float* p, const float* g, int64_t n, float lr) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, n >= 0, GK_ERR_ARG, "gk_sgd_step: negative size");
    if (n == 0) return GK_OK;
    GK_REQUIRE(ctx, p && g, GK_ERR_ARG, "gk_sgd_step: null pointer");
    sgd_kernel<<<ew_blocks(ctx, n), EW_THREADS, 0, ctx->stream>>>(p, g, n, lr, vec4(p, g));
    return launched(ctx, "sgd");
}

}  // extern "C"
