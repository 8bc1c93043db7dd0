// Shared definitions of libgk's CUDA sources: the context, argument checks, launch
// bookkeeping and small device helpers (bf16 conversion, warp reductions).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/gk.h"

struct gk_ctx {
    cudaStream_t stream = nullptr;
    int device = 0;
    int num_sms = 0;
    int* d_err = nullptr;      // device error word: first kernel-side error code
    void* ws = nullptr;        // device workspace
    size_t ws_bytes = 0;
    int math = GK_MATH_3XTF32;
    int64_t launches = 0;
    char msg[512] = {0};
};

namespace gk {

gk_status fail(gk_ctx* ctx, gk_status code, const char* fmt, ...);
// Check the launch that was just issued and count it.
gk_status launched(gk_ctx* ctx, const char* what);

#define GK_REQUIRE(ctx, cond, code, ...)                 \
    do {                                                 \
        if (!(cond)) return ::gk::fail((ctx), (code), __VA_ARGS__); \
    } while (0)

#define GK_TRY(expr)                      \
    do {                                  \
        gk_status _s = (expr);            \
        if (_s != GK_OK) return _s;       \
    } while (0)

__host__ __device__ inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace of at least `bytes`, or nullptr (the caller returns GK_ERR_WORKSPACE).
inline void* workspace(gk_ctx* ctx, size_t bytes) { return bytes <= ctx->ws_bytes ? ctx->ws : nullptr; }

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float load_as_f32(const float* p) { return *p; }
__device__ __forceinline__ float load_as_f32(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void store_from_f32(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_from_f32(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Double-float arithmetic: (hi, lo) stands for the unevaluated sum hi + lo of two float32
// values, about 48 significant bits (Knuth's TwoSum gives the exact error of a float addition).
// Float64 runs on a slow pipe on this GPU; these run on the float32 one.
__device__ __forceinline__ float2 df_add(float2 x, float2 y) {
    const float s = x.x + y.x, bp = s - x.x;
    const float e = ((x.x - (s - bp)) + (y.x - bp)) + (x.y + y.y);
    const float hi = s + e;
    return make_float2(hi, e - (hi - s));
}

// *out = (sum of v[0 .. n)) / n by one block in a fixed order: thread t adds v[t], v[t + blockDim],
// ... in double-float, a lane xor tree in double-float, then the warps in order in double.
__device__ __forceinline__ void block_mean_fixed(const float* __restrict__ v, int64_t n, float* out) {
    __shared__ double red[32];
    float2 s = make_float2(0.f, 0.f);
    for (int64_t r = threadIdx.x; r < n; r += blockDim.x) s = df_add(s, make_float2(v[r], 0.f));
    for (int o = 16; o > 0; o >>= 1)
        s = df_add(s, make_float2(__shfl_xor_sync(0xffffffffu, s.x, o), __shfl_xor_sync(0xffffffffu, s.y, o)));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = (double)s.x + (double)s.y;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        *out = (float)(t / (double)n);
    }
}

// Record the first kernel-side error of a launch in the context's error word.
__device__ __forceinline__ void report(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Tanh-form GELU and its derivative (float32). The constants are those of the published
// approximation: sqrt(2/pi) and 0.044715.
__device__ __forceinline__ float gelu_tanh(float x) {
    const float k = 0.7978845608028654f;
    float u = k * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(u));
}
__device__ __forceinline__ float gelu_tanh_grad(float x) {
    const float k = 0.7978845608028654f;
    float u = k * (x + 0.044715f * x * x * x);
    float t = tanhf(u);
    float du = k * (1.0f + 3.0f * 0.044715f * x * x);
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * du;
}

}  // namespace gk
