// KV-cache decoding: prefill, one-token decode steps and token selection.
// [LM4] = arabroot.io, "Build a language model in C# from scratch (4): running GPT-2
// weights": "Generation with a KV cache" (Attention.Step, KvCache, Gpt.Step,
// GenerateCached) and "Temperature and top-k" (SampleNext).
//
// Decode is bound by reading the weights once per step, so the per-token matrix products are
// split-K GEMV kernels that stream each weight row once and reuse it for every batch row.
// The cache position and the selection count live on the device, so a decode step is a
// fixed sequence of launches that can be captured once in a CUDA graph and replayed.
#include <math.h>

#include <algorithm>

#include "gemm.cuh"

struct gk_kv {
    gk_gpt_cfg cfg{};
    int B = 0, Tmax = 0;
    float* cache = nullptr;  // [L][2][B][H][Tmax][hs]
    int* state = nullptr;    // device: [0] cache length, [1] selections made
    int length = 0;          // host mirror of state[0]
    // activations (prefill uses B*Tmax rows, decode B rows)
    float *x = nullptr, *ln = nullptr, *qkv = nullptr, *y = nullptr, *pre = nullptr, *h = nullptr;
    float *mean = nullptr, *rstd = nullptr, *lse = nullptr, *last = nullptr;
    float* partial = nullptr;  // split-K partial sums
    size_t partial_floats = 0;
    float* attn_part = nullptr;  // decode attention partials [B*H][chunks][hs + 2]
    // gk_decode_run: one captured decode step (instantiated graph) and what it was captured for
    cudaGraphExec_t graph = nullptr;
    int64_t graph_launches = 0;
    const void* graph_key[6] = {};
    gk_sample_cfg graph_s{};
    bool graph_has_s = false;
};

using namespace gk;

namespace {

constexpr int GEMV_THREADS = 256;  // 8 warps; a warp covers 128 columns (float4 per lane)
constexpr int GEMV_COLS = 128;
constexpr int KCHUNK = 64;         // keys per decode-attention block

// partial[s][b][n] = sum over k in slice s of X[b, k] W[k, n], for n in this block's columns.
template <int NB>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_partial_kernel(const float* __restrict__ X, int64_t ldx,
                                                                    const float* __restrict__ W, int64_t ldw, int B,
                                                                    int K, int M, int kslice,
                                                                    float* __restrict__ partial) {
    extern __shared__ float sm[];  // Xs[NB][kslice] then red[8][NB][128]
    float* Xs = sm;
    float* red = sm + NB * kslice;
    int s = blockIdx.y;
    int k0 = s * kslice, k1 = min(K, k0 + kslice);
    int n = blockIdx.x * GEMV_COLS + (threadIdx.x & 31) * 4;
    int warp = threadIdx.x >> 5;
    for (int e = threadIdx.x; e < NB * kslice; e += GEMV_THREADS) {
        int b = e / kslice, k = k0 + e % kslice;
        Xs[e] = (b < B && k < k1) ? X[(int64_t)b * ldx + k] : 0.f;
    }
    __syncthreads();
    float acc[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0.f;
    if (n < M) {
        for (int k = k0 + warp; k < k1; k += 8) {
            float4 w = *reinterpret_cast<const float4*>(W + (int64_t)k * ldw + n);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float xv = Xs[b * kslice + (k - k0)];
                acc[b][0] = fmaf(xv, w.x, acc[b][0]);
                acc[b][1] = fmaf(xv, w.y, acc[b][1]);
                acc[b][2] = fmaf(xv, w.z, acc[b][2]);
                acc[b][3] = fmaf(xv, w.w, acc[b][3]);
            }
        }
    }
    int col = (threadIdx.x & 31) * 4;
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int j = 0; j < 4; ++j) red[(warp * NB + b) * GEMV_COLS + col + j] = acc[b][j];
    __syncthreads();
    for (int e = threadIdx.x; e < NB * GEMV_COLS; e += GEMV_THREADS) {
        int b = e / GEMV_COLS, c = e % GEMV_COLS;
        int nn = blockIdx.x * GEMV_COLS + c;
        if (b >= B || nn >= M) continue;
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[(w * NB + b) * GEMV_COLS + c];
        partial[((int64_t)s * B + b) * M + nn] = t;
    }
}

// Y[b, n] = act(sum_s partial[s][b][n] + bias[n] + residual[b, n]) (slices in order).
__global__ void gemv_finish_kernel(const float* __restrict__ partial, int S, int B, int M, const float* bias,
                                   const float* residual, float* Y, int64_t ldy, int act, float* preact) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * M) return;
    int b = (int)(i / M), n = (int)(i % M);
    float t = 0.f;
    for (int s = 0; s < S; ++s) t += partial[((int64_t)s * B + b) * M + n];
    if (bias) t += bias[n];
    if (residual) t += residual[(int64_t)b * ldy + n];
    if (act == GK_ACT_GELU) {
        if (preact) preact[(int64_t)b * M + n] = t;
        t = gelu_tanh(t);
    }
    Y[(int64_t)b * ldy + n] = t;
}

// logits[b, v] = sum_c X[b, c] wte[v, c]: one warp per vocabulary row (MatMulT head).
template <int NB>
__global__ void lm_head_kernel(const float* __restrict__ X, const float* __restrict__ wte, int B, int C, int V,
                               float* __restrict__ logits, int64_t ldl) {
    extern __shared__ float xs[];  // [NB][C]
    for (int e = threadIdx.x; e < NB * C; e += blockDim.x) xs[e] = (e / C) < B ? X[e] : 0.f;
    __syncthreads();
    int lane = threadIdx.x & 31;
    int warps = blockDim.x >> 5;
    for (int v = blockIdx.x * warps + (threadIdx.x >> 5); v < V; v += gridDim.x * warps) {
        const float* row = wte + (int64_t)v * C;
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = 0.f;
        for (int c = lane * 4; c < C; c += 128) {
            float4 w = *reinterpret_cast<const float4*>(row + c);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float* xb = xs + b * C + c;
                acc[b] = fmaf(w.x, xb[0], fmaf(w.y, xb[1], fmaf(w.z, xb[2], fmaf(w.w, xb[3], acc[b]))));
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
        if (lane < NB && lane < B) {
            float r = 0.f;
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b == lane) r = acc[b];
            logits[(int64_t)lane * ldl + v] = r;
        }
    }
}

// x[b, :] = wte[tokens[b], :] + wpe[pos, :] with pos the device cache length.
__global__ void embed_step_kernel(const int32_t* __restrict__ tokens, const float* __restrict__ wte,
                                  const float* __restrict__ wpe, float* __restrict__ x, int B, int C, int V,
                                  int Tmax, const int* __restrict__ state, int* err) {
    int b = blockIdx.x;
    int pos = state[0];
    int id = tokens[b];
    bool ok = id >= 0 && id < V && pos < Tmax;
    if (!ok && threadIdx.x == 0) report(err, pos >= Tmax ? GK_ERR_OVERFLOW : GK_ERR_INDEX);
    for (int c = threadIdx.x; c < C; c += blockDim.x)
        x[(int64_t)b * C + c] = ok ? wte[(int64_t)id * C + c] + wpe[(int64_t)pos * C + c] : 0.f;
}

__device__ __forceinline__ int64_t cache_index(int l, int kv, int b, int h, int t, int B, int H, int Tmax, int hs) {
    return ((((int64_t)(l * 2 + kv) * B + b) * H + h) * Tmax + t) * hs;
}

// Append this step's key and value rows (columns [C, 2C) and [2C, 3C) of qkv) at pos.
__global__ void kv_append_kernel(const float* __restrict__ qkv, float* __restrict__ cache, int l, int B, int H, int hs,
                                 int Tmax, const int* __restrict__ state) {
    int pos = state[0];
    if (pos >= Tmax) return;
    int C = H * hs;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * C) return;
    int b = (int)(i / C), c = (int)(i % C), h = c / hs, d = c % hs;
    cache[cache_index(l, 0, b, h, pos, B, H, Tmax, hs) + d] = qkv[(int64_t)b * 3 * C + C + c];
    cache[cache_index(l, 1, b, h, pos, B, H, Tmax, hs) + d] = qkv[(int64_t)b * 3 * C + 2 * C + c];
}

// Prefill: keys and values of positions 0 .. Tp-1 from qkv [B*Tp, 3C].
__global__ void kv_write_prefill_kernel(const float* __restrict__ qkv, float* __restrict__ cache, int l, int B,
                                        int Tp, int H, int hs, int Tmax) {
    int C = H * hs;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * Tp * C) return;
    int64_t r = i / C;
    int c = (int)(i % C), h = c / hs, d = c % hs;
    int b = (int)(r / Tp), t = (int)(r % Tp);
    cache[cache_index(l, 0, b, h, t, B, H, Tmax, hs) + d] = qkv[r * 3 * C + C + c];
    cache[cache_index(l, 1, b, h, t, B, H, Tmax, hs) + d] = qkv[r * 3 * C + 2 * C + c];
}

// Decode attention, split over key chunks of KCHUNK (flash-decoding): block (chunk, b*H+h)
// writes (max, sum, unnormalised output[hs]) of its chunk; no mask (the cache holds the past).
__global__ void __launch_bounds__(128) decode_attn_partial_kernel(const float* __restrict__ qkv,
                                                                  const float* __restrict__ cache, int l, int B,
                                                                  int H, int hs, int Tmax,
                                                                  const int* __restrict__ state,
                                                                  float* __restrict__ part, int nchunks) {
    __shared__ float q[128];
    __shared__ float p[KCHUNK];
    __shared__ float red[4];
    __shared__ float ored[2][128];
    int chunk = blockIdx.x, bh = blockIdx.y, b = bh / H, h = bh % H;
    int n = min(state[0] + 1, Tmax);  // keys 0 .. pos (the current one was appended)
    int j0 = chunk * KCHUNK;
    float* out = part + ((int64_t)bh * nchunks + chunk) * (hs + 2);
    if (j0 >= n) {
        if (threadIdx.x == 0) {
            out[0] = -INFINITY;
            out[1] = 0.f;
        }
        return;
    }
    int C = H * hs;
    for (int d = threadIdx.x; d < hs; d += blockDim.x) q[d] = qkv[(int64_t)b * 3 * C + h * hs + d];
    __syncthreads();
    const float scale = rsqrtf((float)hs);
    const float* K = cache + cache_index(l, 0, b, h, 0, B, H, Tmax, hs);
    const float* Vc = cache + cache_index(l, 1, b, h, 0, B, H, Tmax, hs);
    // two threads per key: each takes half of the dimensions
    int kk = threadIdx.x >> 1, half = threadIdx.x & 1;
    int j = j0 + kk;
    float s = 0.f;
    if (j < n) {
        const float* kr = K + (int64_t)j * hs;
        int d0 = half * (hs / 2), d1 = d0 + hs / 2;
        for (int d = d0; d < d1; ++d) s = fmaf(q[d], kr[d], s);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s = (j < n) ? s * scale : -INFINITY;
    float m = warp_max(s);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    float e = (j < n) ? expf(s - m) : 0.f;
    if (half == 0) p[kk] = e;
    __syncthreads();
    if (threadIdx.x == 0) {
        float l_ = 0.f;
        for (int t = 0; t < KCHUNK; ++t) l_ += p[t];
        out[0] = m;
        out[1] = l_;
    }
    // output: thread (d, g) sums keys g, g+2, ... of the chunk for dimension d
    int g = threadIdx.x / 64, d = threadIdx.x % 64;
    for (int dd = d; dd < hs; dd += 64) {
        float o = 0.f;
        for (int t = g; t < KCHUNK && j0 + t < n; t += 2) o = fmaf(p[t], Vc[(int64_t)(j0 + t) * hs + dd], o);
        ored[g][dd] = o;
    }
    __syncthreads();
    for (int dd = threadIdx.x; dd < hs; dd += blockDim.x) out[2 + dd] = ored[0][dd] + ored[1][dd];
}

__global__ void decode_attn_combine_kernel(const float* __restrict__ part, int nchunks, int H, int hs,
                                           float* __restrict__ y) {
    int bh = blockIdx.x, b = bh / H, h = bh % H;
    const float* pp = part + (int64_t)bh * nchunks * (hs + 2);
    float M = -INFINITY;
    for (int c = 0; c < nchunks; ++c) M = fmaxf(M, pp[c * (hs + 2)]);
    float L = 0.f;
    for (int c = 0; c < nchunks; ++c) {
        float mc = pp[c * (hs + 2)];
        if (mc != -INFINITY) L += pp[c * (hs + 2) + 1] * expf(mc - M);
    }
    for (int d = threadIdx.x; d < hs; d += blockDim.x) {
        float o = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            float mc = pp[c * (hs + 2)];
            if (mc != -INFINITY) o += pp[c * (hs + 2) + 2 + d] * expf(mc - M);
        }
        y[(int64_t)b * H * hs + h * hs + d] = o / L;
    }
}

__global__ void gather_last_kernel(const float* __restrict__ x, int B, int Tp, int C, float* __restrict__ last) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * C) return;
    int b = (int)(i / C), c = (int)(i % C);
    last[i] = x[((int64_t)b * Tp + Tp - 1) * C + c];
}

__global__ void copy_ids_kernel(const int32_t* __restrict__ src, int32_t* __restrict__ dst, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = src[i];
}

__global__ void set_state_kernel(int* state, int length, int selections) {
    state[0] = length;
    state[1] = selections;
}

__global__ void advance_kernel(int* state, int dlen, int dsel) {
    state[0] += dlen;
    state[1] += dsel;
}

// ---------------------------------------------------------------- token selection
// Philox4x32-10 (Salmon, Moraes, Dror & Shaw, SC'11): 10 rounds of two 32x32 -> 64-bit
// products with the published multipliers, key bumped by the published Weyl constants.
__device__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

// Ordered-integer image of a float: larger float <-> larger unsigned.
__device__ __forceinline__ uint32_t ord_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int SEL_THREADS = 1024;

// One block per batch row. Greedy: lowest index of the maximum. Top-k: the k-th largest
// value by a 4-pass radix select on ordered keys, keep l >= it (ties kept), weights
// exp((l - max)/T) in float64, running sum over ascending indices (contiguous segments per
// thread, combined in thread order), first index whose running sum exceeds u * total.
__global__ void __launch_bounds__(SEL_THREADS) select_kernel(const float* __restrict__ logits, int64_t ld, int V,
                                                             int top_k, float temperature, uint64_t seed,
                                                             uint64_t counter, const int* __restrict__ state,
                                                             int32_t* __restrict__ next) {
    __shared__ unsigned hist[256];
    __shared__ float fred[32];
    __shared__ int ired[32];
    __shared__ double dscan[SEL_THREADS];
    __shared__ uint32_t prefix_s, want_s;
    __shared__ int pick_s;
    int b = blockIdx.x;
    const float* x = logits + (int64_t)b * ld;
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // maximum and its lowest index
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = threadIdx.x; i < V; i += SEL_THREADS) {
        float v = x[i];
        if (v > best || (v == best && i < bi)) {
            best = v;
            bi = i;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, best, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) {
            best = ov;
            bi = oi;
        }
    }
    if (lane == 0) {
        fred[warp] = best;
        ired[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float bv = fred[0];
        int bx = ired[0];
        for (int w = 1; w < SEL_THREADS / 32; ++w)
            if (fred[w] > bv || (fred[w] == bv && ired[w] < bx)) {
                bv = fred[w];
                bx = ired[w];
            }
        fred[0] = bv;
        ired[0] = bx;
    }
    __syncthreads();
    float mx = fred[0];
    if (top_k == 1 || temperature <= 0.f) {
        if (threadIdx.x == 0) next[b] = ired[0];
        return;
    }
    // threshold: the k-th largest value (or keep everything)
    float kth = -INFINITY;
    if (top_k > 0 && top_k < V) {
        if (threadIdx.x == 0) {
            prefix_s = 0;
            want_s = (uint32_t)top_k;
        }
        for (int pass = 0; pass < 4; ++pass) {
            int shift = 24 - 8 * pass;
            for (int i = threadIdx.x; i < 256; i += SEL_THREADS) hist[i] = 0;
            __syncthreads();
            uint32_t pre = prefix_s;
            uint32_t mask_hi = pass == 0 ? 0u : (0xFFFFFFFFu << (32 - 8 * pass));
            for (int i = threadIdx.x; i < V; i += SEL_THREADS) {
                uint32_t k = ord_key(x[i]);
                if ((k & mask_hi) == pre) atomicAdd(&hist[(k >> shift) & 0xFF], 1u);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                uint32_t want = want_s, cum = 0;
                int d = 255;
                for (; d > 0; --d) {
                    if (cum + hist[d] >= want) break;
                    cum += hist[d];
                }
                want_s = want - cum;
                prefix_s = pre | ((uint32_t)d << shift);
            }
            __syncthreads();
        }
        kth = key_float(prefix_s);
    }
    // float64 weights over contiguous index segments, running sums in index order
    int seg = (V + SEL_THREADS - 1) / SEL_THREADS;
    int i0 = threadIdx.x * seg, i1 = min(V, i0 + seg);
    double inv_t = 1.0 / (double)temperature;
    double local = 0.0;
    for (int i = i0; i < i1; ++i) {
        float v = x[i];
        if (v >= kth) local += exp(((double)v - (double)mx) * inv_t);
    }
    dscan[threadIdx.x] = local;
    __syncthreads();
    if (threadIdx.x == 0) {
        double run = 0.0;
        for (int t = 0; t < SEL_THREADS; ++t) {
            double s = dscan[t];
            dscan[t] = run;  // exclusive prefix
            run += s;
        }
        uint32_t w0 = philox_word0((uint32_t)(counter + (uint64_t)state[1]), (uint32_t)b, 0u, 0u, (uint32_t)seed,
                                   (uint32_t)(seed >> 32));
        double u = (double)(w0 >> 8) * (1.0 / 16777216.0);
        double target = u * run;
        pick_s = -1;
        // the segment where the running sum first exceeds the target
        int t = SEL_THREADS - 1;
        while (t > 0 && dscan[t] > target) --t;
        fred[1] = 0.f;
        ired[1] = t;
        dscan[0] = target;  // reuse slot 0 for the target (segment 0's prefix is 0)
        ired[2] = 0;
    }
    __syncthreads();
    if ((int)threadIdx.x == ired[1]) {
        double target = dscan[0];
        double run = threadIdx.x == 0 ? 0.0 : dscan[threadIdx.x];
        int last_kept = -1, chosen = -1;
        for (int i = i0; i < i1; ++i) {
            float v = x[i];
            if (!(v >= kth)) continue;
            last_kept = i;
            run += exp(((double)v - (double)mx) * inv_t);
            if (run > target) {
                chosen = i;
                break;
            }
        }
        pick_s = chosen >= 0 ? chosen : last_kept;
    }
    __syncthreads();
    if (threadIdx.x == 0) next[b] = pick_s >= 0 ? pick_s : ired[0];
}

int gemv_nb(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16; }

gk_status gemv(gk_ctx* ctx, gk_kv* kv, const float* X, int64_t ldx, const float* W, int64_t ldw, int K, int M,
               const float* bias, const float* residual, float* Y, int act, float* preact) {
    int B = kv->B;
    int colblocks = (int)cdiv(M, GEMV_COLS);
    int S = (int)std::max<int64_t>(1, std::min<int64_t>(K / 8, cdiv(2 * ctx->num_sms, colblocks)));
    int kslice = (int)cdiv(K, S);
    S = (int)cdiv(K, kslice);
    GK_REQUIRE(ctx, (size_t)S * B * M <= kv->partial_floats, GK_ERR_WORKSPACE, "decode gemv: partial buffer too small");
    int nb = gemv_nb(B);
    size_t smem = ((size_t)nb * kslice + 8 * (size_t)nb * GEMV_COLS) * sizeof(float);
    dim3 grid(colblocks, S);
#define GEMV_CASE(NBV)                                                                                       \
    case NBV:                                                                                                \
        cudaFuncSetAttribute(gemv_partial_kernel<NBV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        gemv_partial_kernel<NBV><<<grid, GEMV_THREADS, smem, ctx->stream>>>(X, ldx, W, ldw, B, K, M, kslice,   \
                                                                            kv->partial);                    \
        break;
    switch (nb) {
        GEMV_CASE(1) GEMV_CASE(2) GEMV_CASE(4) GEMV_CASE(8) GEMV_CASE(16)
    }
#undef GEMV_CASE
    GK_TRY(launched(ctx, "gemv_partial"));
    gemv_finish_kernel<<<(unsigned)cdiv((int64_t)B * M, 256), 256, 0, ctx->stream>>>(kv->partial, S, B, M, bias,
                                                                                   residual, Y, M, act, preact);
    return launched(ctx, "gemv_finish");
}

gk_status lm_head(gk_ctx* ctx, gk_kv* kv, const float* X, const float* wte, float* logits, int64_t ldl) {
    int B = kv->B, C = kv->cfg.C, V = kv->cfg.V;
    int nb = gemv_nb(B);
    size_t smem = (size_t)nb * C * sizeof(float);
    int blocks = ctx->num_sms * 4;
#define LM_CASE(NBV)                                                                                         \
    case NBV:                                                                                                \
        cudaFuncSetAttribute(lm_head_kernel<NBV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
        lm_head_kernel<NBV><<<blocks, 256, smem, ctx->stream>>>(X, wte, B, C, V, logits, ldl);                 \
        break;
    switch (nb) {
        LM_CASE(1) LM_CASE(2) LM_CASE(4) LM_CASE(8) LM_CASE(16)
    }
#undef LM_CASE
    return launched(ctx, "lm_head");
}

struct W {
    const float* p;
    gk_gpt_cfg c;
    const float* t(int which, int layer = 0) const { return p + gk_gpt_offset(&c, which, layer); }
};

void drop_graph(gk_kv* kv) {
    if (kv->graph) cudaGraphExecDestroy(kv->graph);
    kv->graph = nullptr;
    kv->graph_launches = 0;
}

gk_status check_kv_args(gk_ctx* ctx, const float* params, gk_kv* kv) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, params && kv, GK_ERR_ARG, "decode: null params or cache");
    GK_REQUIRE(ctx, aligned16(params), GK_ERR_ALIGN, "decode: params must be 16-byte aligned");
    return GK_OK;
}

}  // namespace

extern "C" {

gk_status gk_kv_create(gk_ctx* ctx, gk_kv** out, const gk_gpt_cfg* cfg, int B, int Tmax) {
    if (!ctx || !out || !cfg) return GK_ERR_ARG;
    *out = nullptr;
    GK_REQUIRE(ctx, gk_gpt_numel(cfg) > 0 && cfg->H > 0 && cfg->C % cfg->H == 0, GK_ERR_ARG, "gk_kv_create: bad cfg");
    GK_REQUIRE(ctx, B >= 1 && B <= 16, GK_ERR_UNSUPPORTED, "gk_kv_create: batch %d outside 1..16", B);
    GK_REQUIRE(ctx, Tmax >= 1 && Tmax <= cfg->T, GK_ERR_ARG, "gk_kv_create: Tmax %d outside 1..T", Tmax);
    int hs = cfg->C / cfg->H;
    GK_REQUIRE(ctx, hs <= 128 && cfg->C % 4 == 0, GK_ERR_UNSUPPORTED, "gk_kv_create: head size / width unsupported");
    gk_kv* kv = new gk_kv();
    kv->cfg = *cfg;
    kv->B = B;
    kv->Tmax = Tmax;
    int64_t C = cfg->C, rows = (int64_t)B * Tmax;
    int nchunks = (int)cdiv(Tmax, KCHUNK);
    kv->partial_floats = (size_t)2 * ctx->num_sms * 16 * 4 * C + (size_t)64 * 16 * 4 * C;
    struct A {
        float** p;
        size_t n;
    } allocs[] = {{&kv->cache, (size_t)cfg->L * 2 * rows * C},
                  {&kv->x, (size_t)rows * C},
                  {&kv->ln, (size_t)rows * C},
                  {&kv->qkv, (size_t)rows * 3 * C},
                  {&kv->y, (size_t)rows * C},
                  {&kv->pre, (size_t)rows * 4 * C},
                  {&kv->h, (size_t)rows * 4 * C},
                  {&kv->mean, (size_t)rows},
                  {&kv->rstd, (size_t)rows},
                  {&kv->lse, (size_t)rows * cfg->H},
                  {&kv->last, (size_t)B * C},
                  {&kv->partial, kv->partial_floats},
                  {&kv->attn_part, (size_t)B * cfg->H * nchunks * (hs + 2)}};
    for (auto& a : allocs) {
        if (cudaMalloc(a.p, a.n * sizeof(float)) != cudaSuccess) {
            gk_kv_destroy(kv);
            return fail(ctx, GK_ERR_CUDA, "gk_kv_create: out of device memory");
        }
    }
    if (cudaMalloc(&kv->state, 2 * sizeof(int)) != cudaSuccess || cudaMemset(kv->state, 0, 2 * sizeof(int)) != cudaSuccess ||
        cudaMemset(kv->cache, 0, (size_t)cfg->L * 2 * rows * C * sizeof(float)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        gk_kv_destroy(kv);
        return fail(ctx, GK_ERR_CUDA, "gk_kv_create: device setup failed");
    }
    *out = kv;
    return GK_OK;
}

void gk_kv_destroy(gk_kv* kv) {
    if (!kv) return;
    drop_graph(kv);
    float* ptrs[] = {kv->cache, kv->x, kv->ln, kv->qkv, kv->y, kv->pre, kv->h, kv->mean, kv->rstd, kv->lse, kv->last,
                     kv->partial, kv->attn_part};
    for (float* p : ptrs)
        if (p) cudaFree(p);
    if (kv->state) cudaFree(kv->state);
    delete kv;
}

float* gk_kv_data(gk_kv* kv) { return kv ? kv->cache : nullptr; }
int gk_kv_length(gk_kv* kv) { return kv ? kv->length : -1; }

gk_status gk_prefill(gk_ctx* ctx, const float* params, gk_kv* kv, const int32_t* ids, int Tp, float* last_logits) {
    GK_TRY(check_kv_args(ctx, params, kv));
    GK_REQUIRE(ctx, ids && last_logits && Tp >= 1, GK_ERR_ARG, "gk_prefill: bad argument");
    GK_REQUIRE(ctx, Tp <= kv->Tmax, GK_ERR_OVERFLOW, "gk_prefill: prompt of %d exceeds the cache (%d)", Tp, kv->Tmax);
    const gk_gpt_cfg& c = kv->cfg;
    W w{params, c};
    int B = kv->B, C = c.C, H = c.H, hs = C / H;
    int64_t N = (int64_t)B * Tp;
    GK_TRY(gk_embedding_fwd(ctx, ids, w.t(GK_T_WTE), w.t(GK_T_WPE), kv->x, B, Tp, C, c.V));
    for (int l = 0; l < c.L; ++l) {
        GK_TRY(gk_layernorm_fwd(ctx, kv->x, w.t(GK_T_LN1_W, l), w.t(GK_T_LN1_B, l), kv->ln, GK_F32, nullptr, nullptr, N,
                                C, 1e-5f));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->ln, C, w.t(GK_T_ATTN_W, l), 3 * C, 0, w.t(GK_T_ATTN_B, l), nullptr, 0,
                             kv->qkv, 3 * C, GK_F32, N, C, 3 * C, GK_ACT_NONE, nullptr, 0, nullptr, nullptr));
        kv_write_prefill_kernel<<<(unsigned)cdiv(N * C, 256), 256, 0, ctx->stream>>>(kv->qkv, kv->cache, l, B, Tp, H,
                                                                                    hs, kv->Tmax);
        GK_TRY(launched(ctx, "kv_write_prefill"));
        GK_TRY(gk_attn_fwd(ctx, GK_F32, kv->qkv, kv->y, kv->lse, B, Tp, H, hs));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->y, C, w.t(GK_T_ATTNPROJ_W, l), C, 0, w.t(GK_T_ATTNPROJ_B, l), kv->x, C,
                             kv->x, C, GK_F32, N, C, C, GK_ACT_NONE, nullptr, 0, nullptr, nullptr));
        GK_TRY(gk_layernorm_fwd(ctx, kv->x, w.t(GK_T_LN2_W, l), w.t(GK_T_LN2_B, l), kv->ln, GK_F32, nullptr, nullptr, N,
                                C, 1e-5f));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->ln, C, w.t(GK_T_FC_W, l), 4 * C, 0, w.t(GK_T_FC_B, l), nullptr, 0, kv->h,
                             4 * C, GK_F32, N, C, 4 * C, GK_ACT_GELU, kv->pre, 4 * C, nullptr, nullptr));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->h, 4 * C, w.t(GK_T_MLPPROJ_W, l), C, 0, w.t(GK_T_MLPPROJ_B, l), kv->x, C,
                             kv->x, C, GK_F32, N, 4 * C, C, GK_ACT_NONE, nullptr, 0, nullptr, nullptr));
    }
    gather_last_kernel<<<(unsigned)cdiv((int64_t)B * C, 256), 256, 0, ctx->stream>>>(kv->x, B, Tp, C, kv->last);
    GK_TRY(launched(ctx, "gather_last"));
    GK_TRY(gk_layernorm_fwd(ctx, kv->last, w.t(GK_T_LNF_W), w.t(GK_T_LNF_B), kv->ln, GK_F32, nullptr, nullptr, B, C,
                            1e-5f));
    GK_TRY(lm_head(ctx, kv, kv->ln, w.t(GK_T_WTE), last_logits, c.V));
    set_state_kernel<<<1, 1, 0, ctx->stream>>>(kv->state, Tp, 0);
    GK_TRY(launched(ctx, "set_state"));
    kv->length = Tp;
    return GK_OK;
}

}  // extern "C"

namespace {

// The launches of one decode step (arguments checked by the caller); the host mirror of the
// cache length is left to the caller.
gk_status decode_step_launches(gk_ctx* ctx, const float* params, gk_kv* kv, const int32_t* tokens, float* logits,
                               int32_t* next, const gk_sample_cfg* s) {
    const gk_gpt_cfg& c = kv->cfg;
    W w{params, c};
    int B = kv->B, C = c.C, H = c.H, hs = C / H;
    int nchunks = (int)cdiv(kv->Tmax, KCHUNK);
    embed_step_kernel<<<B, 256, 0, ctx->stream>>>(tokens, w.t(GK_T_WTE), w.t(GK_T_WPE), kv->x, B, C, c.V, kv->Tmax,
                                                  kv->state, ctx->d_err);
    GK_TRY(launched(ctx, "embed_step"));
    for (int l = 0; l < c.L; ++l) {
        GK_TRY(gk_layernorm_fwd(ctx, kv->x, w.t(GK_T_LN1_W, l), w.t(GK_T_LN1_B, l), kv->ln, GK_F32, nullptr, nullptr, B,
                                C, 1e-5f));
        GK_TRY(gemv(ctx, kv, kv->ln, C, w.t(GK_T_ATTN_W, l), 3 * C, C, 3 * C, w.t(GK_T_ATTN_B, l), nullptr, kv->qkv,
                    GK_ACT_NONE, nullptr));
        kv_append_kernel<<<(unsigned)cdiv((int64_t)B * C, 256), 256, 0, ctx->stream>>>(kv->qkv, kv->cache, l, B, H, hs,
                                                                                      kv->Tmax, kv->state);
        GK_TRY(launched(ctx, "kv_append"));
        decode_attn_partial_kernel<<<dim3(nchunks, B * H), 128, 0, ctx->stream>>>(kv->qkv, kv->cache, l, B, H, hs,
                                                                                  kv->Tmax, kv->state, kv->attn_part,
                                                                                  nchunks);
        GK_TRY(launched(ctx, "decode_attn_partial"));
        decode_attn_combine_kernel<<<B * H, 64, 0, ctx->stream>>>(kv->attn_part, nchunks, H, hs, kv->y);
        GK_TRY(launched(ctx, "decode_attn_combine"));
        GK_TRY(gemv(ctx, kv, kv->y, C, w.t(GK_T_ATTNPROJ_W, l), C, C, C, w.t(GK_T_ATTNPROJ_B, l), kv->x, kv->x,
                    GK_ACT_NONE, nullptr));
        GK_TRY(gk_layernorm_fwd(ctx, kv->x, w.t(GK_T_LN2_W, l), w.t(GK_T_LN2_B, l), kv->ln, GK_F32, nullptr, nullptr, B,
                                C, 1e-5f));
        GK_TRY(gemv(ctx, kv, kv->ln, C, w.t(GK_T_FC_W, l), 4 * C, C, 4 * C, w.t(GK_T_FC_B, l), nullptr, kv->h,
                    GK_ACT_GELU, kv->pre));
        GK_TRY(gemv(ctx, kv, kv->h, 4 * C, w.t(GK_T_MLPPROJ_W, l), C, 4 * C, C, w.t(GK_T_MLPPROJ_B, l), kv->x, kv->x,
                    GK_ACT_NONE, nullptr));
    }
    GK_TRY(gk_layernorm_fwd(ctx, kv->x, w.t(GK_T_LNF_W), w.t(GK_T_LNF_B), kv->ln, GK_F32, nullptr, nullptr, B, C, 1e-5f));
    GK_TRY(lm_head(ctx, kv, kv->ln, w.t(GK_T_WTE), logits, c.V));
    int dsel = 0;
    if (next) {
        int top_k = s ? s->top_k : 1;
        float temp = s ? s->temperature : 0.f;
        select_kernel<<<B, SEL_THREADS, 0, ctx->stream>>>(logits, c.V, c.V, top_k, temp, s ? s->seed : 0,
                                                          s ? s->counter : 0, kv->state, next);
        GK_TRY(launched(ctx, "select"));
        dsel = 1;
    }
    advance_kernel<<<1, 1, 0, ctx->stream>>>(kv->state, 1, dsel);
    return launched(ctx, "advance");
}

}  // namespace

extern "C" {

gk_status gk_decode_step(gk_ctx* ctx, const float* params, gk_kv* kv, const int32_t* tokens, float* logits,
                         int32_t* next, const gk_sample_cfg* s) {
    GK_TRY(check_kv_args(ctx, params, kv));
    GK_REQUIRE(ctx, tokens && logits, GK_ERR_ARG, "gk_decode_step: bad argument");
    GK_REQUIRE(ctx, kv->length < kv->Tmax, GK_ERR_OVERFLOW, "gk_decode_step: cache full (%d)", kv->Tmax);
    GK_TRY(decode_step_launches(ctx, params, kv, tokens, logits, next, s));
    kv->length += 1;
    return GK_OK;
}

gk_status gk_decode_run(gk_ctx* ctx, const float* params, gk_kv* kv, int32_t* tokens, float* logits, int32_t* next,
                        const gk_sample_cfg* s, int n_steps) {
    GK_TRY(check_kv_args(ctx, params, kv));
    GK_REQUIRE(ctx, tokens && logits && next && n_steps >= 0, GK_ERR_ARG, "gk_decode_run: bad argument");
    GK_REQUIRE(ctx, (int64_t)kv->length + n_steps <= kv->Tmax, GK_ERR_OVERFLOW,
               "gk_decode_run: %d steps from length %d overflow the cache (%d)", n_steps, kv->length, kv->Tmax);
    if (n_steps == 0) return GK_OK;
    auto step = [&]() -> gk_status {
        GK_TRY(decode_step_launches(ctx, params, kv, tokens, logits, next, s));
        if (next != tokens) {
            copy_ids_kernel<<<1, 32 * (int)cdiv(kv->B, 32), 0, ctx->stream>>>(next, tokens, kv->B);
            GK_TRY(launched(ctx, "copy_ids"));
        }
        return GK_OK;
    };
    if (!ctx->stream) {  // the legacy default stream cannot be captured: plain launches
        for (int i = 0; i < n_steps; ++i) {
            GK_TRY(step());
            kv->length += 1;
        }
        return GK_OK;
    }
    const void* key[6] = {params, tokens, logits, next, ctx->stream, ctx};
    const bool same_s = (s != nullptr) == kv->graph_has_s &&
                        (!s || (s->top_k == kv->graph_s.top_k && s->temperature == kv->graph_s.temperature &&
                                s->seed == kv->graph_s.seed && s->counter == kv->graph_s.counter));
    if (!kv->graph || !same_s || !std::equal(key, key + 6, kv->graph_key)) {
        drop_graph(kv);
        const int64_t l0 = ctx->launches;
        if (cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeRelaxed) != cudaSuccess)
            return fail(ctx, GK_ERR_CUDA, "gk_decode_run: stream capture failed to start");
        gk_status st = step();
        cudaGraph_t g = nullptr;
        cudaError_t e = cudaStreamEndCapture(ctx->stream, &g);
        const int64_t per_step = ctx->launches - l0;
        ctx->launches = l0;  // captured, not run
        if (st != GK_OK) {
            if (g) cudaGraphDestroy(g);
            return st;
        }
        if (e != cudaSuccess || !g) return fail(ctx, GK_ERR_CUDA, "gk_decode_run: capture failed: %s", cudaGetErrorString(e));
        e = cudaGraphInstantiate(&kv->graph, g, 0);
        cudaGraphDestroy(g);
        if (e != cudaSuccess) {
            kv->graph = nullptr;
            return fail(ctx, GK_ERR_CUDA, "gk_decode_run: graph instantiation failed: %s", cudaGetErrorString(e));
        }
        kv->graph_launches = per_step;
        std::copy(key, key + 6, kv->graph_key);
        kv->graph_has_s = s != nullptr;
        if (s) kv->graph_s = *s;
    }
    for (int i = 0; i < n_steps; ++i) {
        cudaError_t e = cudaGraphLaunch(kv->graph, ctx->stream);
        if (e != cudaSuccess) return fail(ctx, GK_ERR_CUDA, "gk_decode_run: graph launch failed: %s", cudaGetErrorString(e));
        ctx->launches += kv->graph_launches;
        kv->length += 1;
    }
    return GK_OK;
}

gk_status gk_sample(gk_ctx* ctx, gk_kv* kv, const float* logits, int64_t ld, int32_t* next, const gk_sample_cfg* s) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, kv && logits && next && ld >= kv->cfg.V, GK_ERR_ARG, "gk_sample: bad argument");
    int top_k = s ? s->top_k : 1;
    float temp = s ? s->temperature : 0.f;
    select_kernel<<<kv->B, SEL_THREADS, 0, ctx->stream>>>(logits, ld, kv->cfg.V, top_k, temp, s ? s->seed : 0,
                                                          s ? s->counter : 0, kv->state, next);
    GK_TRY(launched(ctx, "select"));
    advance_kernel<<<1, 1, 0, ctx->stream>>>(kv->state, 0, 1);
    return launched(ctx, "advance");
}

}  // extern "C"
