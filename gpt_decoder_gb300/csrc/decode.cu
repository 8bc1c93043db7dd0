// KV-cache decoding: prefill, one-token decode steps and token selection.
// [LM4] = arabroot.io, "Build a language model in C# from scratch (4): running GPT-2
// weights": "Generation with a KV cache" (Attention.Step, KvCache, Gpt.Step,
// GenerateCached) and "Temperature and top-k" (SampleNext).
//
// Decode is bound by reading the weights once per step, so the per-token matrix products are
// split-K GEMV kernels that stream each weight row once and reuse it for every batch row.
// A step is five launches per layer: the GEMVs apply the preceding LayerNorm to their input
// rows themselves, and the last block of each column block adds the split-K slices (fixed
// order) with bias, residual, GELU and the key/value append; the attention's last chunk block
// combines the chunks. The cache position and the selection count live on the device, so a
// decode step is a fixed sequence of launches that can be captured once in a CUDA graph.
#include <math.h>

#include <algorithm>

#include "gemm.cuh"

#include "decode.cuh"

using namespace gk;

namespace {

constexpr int GEMV_THREADS = 256;  // 8 warps; a warp covers 128 columns (float4 per lane)
constexpr int GEMV_COLS = 128;
constexpr int KCHUNK = 64;         // keys per decode-attention block
constexpr int GEMV_PF = 8;         // weight rows per warp loaded before the previous kernel ends

// Programmatic dependent launch: a decode kernel lets the next one start as soon as all its
// blocks are running (trigger), and waits for its predecessor's completion and memory before
// touching anything a previous kernel wrote (wait). Only the weights, which nothing in a
// decode step writes, are read before the wait. Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with the blocks grouped in clusters of cluster_y blocks along y (the K slices of one
// column block of a GEMV).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                               int cluster_y, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 1;
    at[1].val.clusterDim.y = (unsigned)cluster_y;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Cluster helpers: every thread of every block of the cluster arrives, then waits (release /
// acquire at cluster scope); the shared::cluster address of `p` (this block's shared memory) in
// block `rank` of the cluster; a float32 load from such an address.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ int64_t cache_index(int l, int kv, int b, int h, int t, int B, int H, int Tmax, int hs) {
    return ((((int64_t)(l * 2 + kv) * B + b) * H + h) * Tmax + t) * hs;
}

// Mean and rstd (biased variance, eps 1e-5) of rows b < B of X (K columns), one warp per
// row, into st[2 * b], st[2 * b + 1]; the LayerNorm of [LM1]'s op table applied by the
// kernels that consume its output.
__device__ __forceinline__ void row_stats(const float* __restrict__ X, int64_t ldx, int B, int K, float* st) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (K % 128 == 0 && K <= 1024 && ldx % 4 == 0 && (reinterpret_cast<uintptr_t>(X) & 15) == 0) {
        // the whole row in registers (K / 128 float4 per lane, all requested at once): the
        // mean, then the variance of the deviations from it
        for (int b = warp; b < B; b += nw) {
            const float4* xr = reinterpret_cast<const float4*>(X + (int64_t)b * ldx);
            const int n4 = K / 128;
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = i < n4 ? xr[lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
            const float mu = warp_sum(s) / K;
            float q = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < n4) {
                    const float a = v[i].x - mu, c = v[i].y - mu, d = v[i].z - mu, e = v[i].w - mu;
                    q += (a * a + c * c) + (d * d + e * e);
                }
            const float var = warp_sum(q) / K;
            if (lane == 0) {
                st[2 * b] = mu;
                st[2 * b + 1] = rsqrtf(var + 1e-5f);
            }
        }
        return;
    }
    for (int b = warp; b < B; b += nw) {
        // one pass over the row, shifted by its first element so that E[d^2] - E[d]^2 does
        // not cancel when the mean is large against the spread
        const float* xr = X + (int64_t)b * ldx;
        const float sh = xr[0];
        float s = 0.f, q = 0.f;
        int k = lane;
        for (; k + 224 < K; k += 256) {  // eight loads in flight per lane
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = xr[k + 32 * u];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float d = v[u] - sh;
                s += d;
                q = fmaf(d, d, q);
            }
        }
        for (; k < K; k += 32) {
            const float d = xr[k] - sh;
            s += d;
            q = fmaf(d, d, q);
        }
        const float md = warp_sum(s) / K;
        const float v = fmaxf(warp_sum(q) / K - md * md, 0.f);
        if (lane == 0) {
            st[2 * b] = sh + md;
            st[2 * b + 1] = rsqrtf(v + 1e-5f);
        }
    }
}

struct GemvArgs {
    const float* X;
    int64_t ldx;
    const float* ln_g;  // not null: the rows of X go through LayerNorm(ln_g, ln_b) first
    const float* ln_b;
    const float* W;
    int64_t ldw;
    int B, K, M, kslice;
    float* partial;
    int* tickets;
    const float* bias;
    const float* residual;
    float* Y;
    int64_t ldy;
    int act;
    float* preact;
    // not null: columns [C, 3C) of Y (keys, values) are also appended to the cache at the
    // device position state[0]
    float* cache;
    int layer, H, hs, Tmax;
    const int* state;
};

// The non-cluster finish of gemv_kernel: the block's sums to partial[s], then the last block of
// the column block (atomic ticket) adds the slices in slice order and applies the epilogue.
template <int NB>
__device__ __forceinline__ void gemv_finish_by_ticket(const GemvArgs& a, const float* red, int s) {
    __shared__ int last;
    for (int e = threadIdx.x; e < NB * GEMV_COLS; e += GEMV_THREADS) {
        const int b = e / GEMV_COLS, c = e % GEMV_COLS;
        const int nn = blockIdx.x * GEMV_COLS + c;
        if (b >= a.B || nn >= a.M) continue;
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[(w * NB + b) * GEMV_COLS + c];
        a.partial[((int64_t)s * a.B + b) * a.M + nn] = t;
    }
    // the last slice of this column block to arrive finishes it
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(&a.tickets[blockIdx.x], 1) == (int)gridDim.y - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    const int pos = a.cache ? a.state[0] : 0;
    const int C = a.H * a.hs;
    // this thread's outputs e = threadIdx.x + 256 i (row e / 128, column e % 128 of the block);
    // each adds the slices in slice order, the loads of all its outputs for SL slices (64 loads
    // at the wide batches) in flight together
    constexpr int EPT = NB >= 2 ? NB / 2 : 1;
    constexpr int SL = EPT >= 4 ? 8 : 16;
    const int S = (int)gridDim.y;
    const int64_t step = (int64_t)a.B * a.M;
    float tsum[EPT];
    int src[EPT];  // offset of the output in a slice's partial sums (B x M < 2^31); -1 past the end
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
        const int e = threadIdx.x + GEMV_THREADS * i, b = e / GEMV_COLS, nn = blockIdx.x * GEMV_COLS + e % GEMV_COLS;
        src[i] = (e < NB * GEMV_COLS && b < a.B && nn < a.M) ? b * a.M + nn : -1;
        tsum[i] = 0.f;
    }
    for (int q = 0; q < S; q += SL) {
        float v[EPT][SL];
#pragma unroll
        for (int i = 0; i < EPT; ++i)
#pragma unroll
            for (int u = 0; u < SL; ++u)
                v[i][u] = (src[i] >= 0 && q + u < S) ? __ldcg(a.partial + (q + u) * step + src[i]) : 0.f;
#pragma unroll
        for (int i = 0; i < EPT; ++i)
#pragma unroll
            for (int u = 0; u < SL; ++u)
                if (q + u < S) tsum[i] += v[i][u];
    }
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
        if (src[i] < 0) continue;
        const int e = threadIdx.x + GEMV_THREADS * i, b = e / GEMV_COLS, nn = blockIdx.x * GEMV_COLS + e % GEMV_COLS;
        float t = tsum[i];
        if (a.bias) t += a.bias[nn];
        if (a.residual) t += a.residual[(int64_t)b * a.ldy + nn];
        if (a.act == GK_ACT_GELU) {
            if (a.preact) a.preact[(int64_t)b * a.M + nn] = t;
            t = gelu_tanh(t);
        }
        a.Y[(int64_t)b * a.ldy + nn] = t;
        if (a.cache && nn >= C && pos < a.Tmax) {
            const int which = nn / C - 1, c = nn % C;
            a.cache[cache_index(a.layer, which, b, c / a.hs, pos, a.B, a.H, a.Tmax, a.hs) + c % a.hs] = t;
        }
    }
    if (threadIdx.x == 0) a.tickets[blockIdx.x] = 0;  // ready for the next launch
}

// Split-K GEMV: block (column block, slice s) forms the sums over k in slice s of
// X'[b, k] W[k, n] (X' = X or its LayerNorm) for the block's 128 columns and every row b. CL: the
// slices of a column block form one cluster; each keeps its sums in its shared memory, and after
// a cluster barrier block s adds the S slices' sums of its share of the outputs (in slice order,
// read from the other blocks' shared memory) and applies bias, residual, GELU and the key/value
// append. Otherwise the sums go to partial[s][b][n] and the last block of a column block to
// finish (atomic ticket) adds the slices in slice order and applies the epilogue. No block
// waits on another outside its cluster.
// Offset of the reduction area after the staged rows: rounded up to four floats, so that
// its float4 stores are aligned.
__host__ __device__ __forceinline__ int gemv_red_offset(int nb, int kslice) { return (nb * kslice + 3) & ~3; }

// Two blocks per SM (at most 128 registers a thread): a launch of up to 2 x SMs blocks then
// runs in one wave.
template <int NB, bool CL>
__global__ void __launch_bounds__(GEMV_THREADS, 2) gemv_kernel(const GemvArgs a) {
    // Xs[NB][kslice], red[8][NB][128], st[2 * NB] (padded to four floats), fin[NB][128] (CL)
    extern __shared__ __align__(16) float sm[];
    float* Xs = sm;
    float* red = sm + gemv_red_offset(NB, a.kslice);
    float* st = red + 8 * NB * GEMV_COLS;
    float* fin = st + ((2 * NB + 3) & ~3);
    const int s = blockIdx.y;
    const int k0 = s * a.kslice, k1 = min(a.K, k0 + a.kslice);
    const int n = blockIdx.x * GEMV_COLS + (threadIdx.x & 31) * 4;
    const int warp = threadIdx.x >> 5;
    pdl_trigger();
    // this warp's first weight rows (k0 + warp + 8 i) while the previous kernel finishes
    float4 wpre[GEMV_PF];
#pragma unroll
    for (int i = 0; i < GEMV_PF; ++i) {
        const int k = k0 + warp + 8 * i;
        wpre[i] = (n < a.M && k < k1) ? *reinterpret_cast<const float4*>(a.W + (int64_t)k * a.ldw + n)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    if (a.ln_g) {
        row_stats(a.X, a.ldx, a.B, a.K, st);
        __syncthreads();
    }
    for (int e = threadIdx.x; e < NB * a.kslice; e += GEMV_THREADS) {
        const int b = e / a.kslice, k = k0 + e % a.kslice;
        float v = 0.f;
        if (b < a.B && k < k1) {
            v = a.X[(int64_t)b * a.ldx + k];
            if (a.ln_g) v = (v - st[2 * b]) * st[2 * b + 1] * a.ln_g[k] + a.ln_b[k];
        }
        Xs[e] = v;
    }
    __syncthreads();
    float acc[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0.f;
    if (n < a.M) {
#pragma unroll
        for (int i = 0; i < GEMV_PF; ++i) {
            const int kk = warp + 8 * i;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float xv = k0 + kk < k1 ? Xs[b * a.kslice + kk] : 0.f;
                acc[b][0] = fmaf(xv, wpre[i].x, acc[b][0]);
                acc[b][1] = fmaf(xv, wpre[i].y, acc[b][1]);
                acc[b][2] = fmaf(xv, wpre[i].z, acc[b][2]);
                acc[b][3] = fmaf(xv, wpre[i].w, acc[b][3]);
            }
        }
        // the remaining rows, eight in flight per warp (rows k, k + 8, ..., k + 56 below k1; the
        // row is the same for the whole warp)
        for (int k = k0 + warp + 8 * GEMV_PF; k < k1; k += 64) {
            float4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                w[u] = k + 8 * u < k1 ? *reinterpret_cast<const float4*>(a.W + (int64_t)(k + 8 * u) * a.ldw + n)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k + 8 * u >= k1) break;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float xv = Xs[b * a.kslice + (k + 8 * u - k0)];
                    acc[b][0] = fmaf(xv, w[u].x, acc[b][0]);
                    acc[b][1] = fmaf(xv, w[u].y, acc[b][1]);
                    acc[b][2] = fmaf(xv, w[u].z, acc[b][2]);
                    acc[b][3] = fmaf(xv, w[u].w, acc[b][3]);
                }
            }
        }
    }
    const int col = (threadIdx.x & 31) * 4;
#pragma unroll
    for (int b = 0; b < NB; ++b)
        *reinterpret_cast<float4*>(red + (warp * NB + b) * GEMV_COLS + col) =
            make_float4(acc[b][0], acc[b][1], acc[b][2], acc[b][3]);
    __syncthreads();
    if constexpr (CL) {
        for (int e = threadIdx.x; e < NB * GEMV_COLS; e += GEMV_THREADS) {
            const int b = e / GEMV_COLS, c = e % GEMV_COLS;
            float t = 0.f;
            for (int w = 0; w < 8; ++w) t += red[(w * NB + b) * GEMV_COLS + c];
            fin[e] = t;
        }
        cluster_barrier();  // every slice's sums are in its block's shared memory
        const int S = (int)gridDim.y;  // the cluster: the column block's S slices, rank = slice
        const int per = (NB * GEMV_COLS + S - 1) / S;
        const int e_end = min(NB * GEMV_COLS, (s + 1) * per);
        const int pos = a.cache ? a.state[0] : 0;
        const int C = a.H * a.hs;
        for (int e = s * per + (int)threadIdx.x; e < e_end; e += GEMV_THREADS) {
            const int b = e / GEMV_COLS, nn = blockIdx.x * GEMV_COLS + e % GEMV_COLS;
            const bool valid = b < a.B && nn < a.M;
            // the epilogue's operands requested with the slices' sums
            const float bias = (valid && a.bias) ? a.bias[nn] : 0.f;
            const float res = (valid && a.residual) ? a.residual[(int64_t)b * a.ldy + nn] : 0.f;
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = u < S ? ld_cluster_f32(cluster_addr(fin + e, (uint32_t)u)) : 0.f;
            float t = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (u < S) t += v[u];
            if (!valid) continue;
            if (a.bias) t += bias;
            if (a.residual) t += res;
            if (a.act == GK_ACT_GELU) {
                if (a.preact) a.preact[(int64_t)b * a.M + nn] = t;
                t = gelu_tanh(t);
            }
            a.Y[(int64_t)b * a.ldy + nn] = t;
            if (a.cache && nn >= C && pos < a.Tmax) {
                const int which = nn / C - 1, c = nn % C;
                a.cache[cache_index(a.layer, which, b, c / a.hs, pos, a.B, a.H, a.Tmax, a.hs) + c % a.hs] = t;
            }
        }
        cluster_barrier();  // no block leaves while another may still read its shared memory
    } else {
        gemv_finish_by_ticket<NB>(a, red, s);
    }
}


// Sum of v[i] over the 32 lanes for every i < N (N = 32 or 64), spread over the lanes: after
// the call, lane l holds the sums of i = (N / 32) l + k in v[k], k < N / 32. Level o pairs the
// lanes that differ in bit o (16 first, as warp_sum does, so each sum is the same as warp_sum's);
// the lane keeps the half of its values that its bit selects and adds its partner's partial of
// that half, so a level costs N / 2^(level+1) shuffles instead of N.
template <int N>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N], int lane) {
    static_assert(N == 32 || N == 64, "32 or 64 values");
#pragma unroll
    for (int lv = 0; lv < 5; ++lv) {
        const int o = 16 >> lv, half = (N >> lv) / 2;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float lo = v[i], hi = v[i + half];
            const float send = up ? lo : hi;
            const float keep = up ? hi : lo;
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
}

// logits[b, v] = sum_c X[b, c] wte[v, c]: one warp per vocabulary row (MatMulT head).
// With ln_g, the rows of X go through LayerNorm(ln_g, ln_b) first (ln_f fused in).
template <int NB>
__global__ void __launch_bounds__(256, 2) lm_head_kernel(const float* __restrict__ X, const float* __restrict__ ln_g,
                               const float* __restrict__ ln_b, const float* __restrict__ wte, int B, int C, int V,
                               float* __restrict__ logits, int64_t ldl) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ float xs[];  // [NB][C], then row statistics [2 NB]
    float* st = xs + NB * C;
    if (ln_g) {
        row_stats(X, C, B, C, st);
        __syncthreads();
    }
    for (int e = threadIdx.x; e < NB * C; e += blockDim.x) {
        const int b = e / C, c = e % C;
        float v = b < B ? X[e] : 0.f;
        if (ln_g && b < B) v = (v - st[2 * b]) * st[2 * b + 1] * ln_g[c] + ln_b[c];
        xs[e] = v;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    // two vocabulary rows per warp and pass; every weight load of a 768-column tile (six float4
    // a lane and row) is issued before the first use, so a pass waits for memory once per tile
    constexpr int RH = 2, CT = 6;
    for (int v0 = (blockIdx.x * warps + (threadIdx.x >> 5)) * RH; v0 < V; v0 += gridDim.x * warps * RH) {
        float acc[RH][NB];
#pragma unroll
        for (int r = 0; r < RH; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
        for (int cb = 0; cb < C; cb += 128 * CT) {
            float4 w[RH][CT];
#pragma unroll
            for (int r = 0; r < RH; ++r)
#pragma unroll
                for (int i = 0; i < CT; ++i) {
                    const int c = cb + i * 128 + lane * 4;
                    w[r][i] = (v0 + r < V && c < C) ? *reinterpret_cast<const float4*>(wte + (int64_t)(v0 + r) * C + c)
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int i = 0; i < CT; ++i) {
                const int c = cb + i * 128 + lane * 4;
                if (c >= C) break;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float4 xb = *reinterpret_cast<const float4*>(xs + b * C + c);
#pragma unroll
                    for (int r = 0; r < RH; ++r)
                        acc[r][b] = fmaf(w[r][i].x, xb.x,
                                         fmaf(w[r][i].y, xb.y, fmaf(w[r][i].z, xb.z, fmaf(w[r][i].w, xb.w, acc[r][b]))));
                }
            }
        }
        if constexpr (RH * NB == 32 || RH * NB == 64) {
            // the RH NB sums spread over the lanes: value i = r NB + b, lane l holds
            // i = (RH NB / 32) l + k
            constexpr int N = RH * NB, PER = N / 32;
            float f[N];
#pragma unroll
            for (int r = 0; r < RH; ++r)
#pragma unroll
                for (int b = 0; b < NB; ++b) f[r * NB + b] = acc[r][b];
            warp_reduce_scatter<N>(f, lane);
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int i = PER * lane + k, r = i / NB, b = i % NB;
                if (b < B && v0 + r < V) logits[(int64_t)b * ldl + v0 + r] = f[k];
            }
        } else {
#pragma unroll
            for (int r = 0; r < RH; ++r)
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[r][b] = warp_sum(acc[r][b]);
#pragma unroll
            for (int r = 0; r < RH; ++r) {
                if (lane < NB && lane < B && v0 + r < V) {
                    float o = 0.f;
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        if (b == lane) o = acc[r][b];
                    logits[(int64_t)lane * ldl + v0 + r] = o;
                }
            }
        }
    }
}

// x[b, :] = wte[tokens[b], :] + wpe[pos, :] with pos the device cache length.
__global__ void embed_step_kernel(const int32_t* __restrict__ tokens, const float* __restrict__ wte,
                                  const float* __restrict__ wpe, float* __restrict__ x, int B, int C, int V,
                                  int Tmax, const int* __restrict__ state, int* err) {
    pdl_trigger();
    pdl_wait();
    int b = blockIdx.x;
    int pos = state[0];
    int id = tokens[b];
    bool ok = id >= 0 && id < V && pos < Tmax;
    if (!ok && threadIdx.x == 0) report(err, pos >= Tmax ? GK_ERR_OVERFLOW : GK_ERR_INDEX);
    for (int c = threadIdx.x; c < C; c += blockDim.x)
        x[(int64_t)b * C + c] = ok ? wte[(int64_t)id * C + c] + wpe[(int64_t)pos * C + c] : 0.f;
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
// of two warps writes (max, sum, unnormalised output[hs]) of its chunk (no mask: the cache
// holds the past). Scores: lane = key, the key's row read as float4s; output: lane = head
// dimension(s), the warp's 32 keys taken in turn (coalesced rows of V). For hs <= 64 every
// load of the chunk (the lane's key row and its two value dimensions of the warp's 32 keys) is
// issued before the first use, so the chunk costs one round trip to memory. The last chunk of
// (b, h) to arrive (atomic ticket) combines the chunks in chunk order into y, sixteen chunks'
// partials in flight at a time; no block waits on another.
__global__ void __launch_bounds__(64) decode_attn_kernel(const float* __restrict__ qkv,
                                                         const float* __restrict__ cache, int l, int B, int H, int hs,
                                                         int Tmax, const int* __restrict__ state,
                                                         float* __restrict__ part, int nchunks, int* tickets,
                                                         float* __restrict__ y) {
    pdl_trigger();
    pdl_wait();
    __shared__ __align__(16) float q[128];
    __shared__ float red[2][2];
    __shared__ float ored[2][128];
    __shared__ int last;
    const int chunk = blockIdx.x, bh = blockIdx.y, b = bh / H, h = bh % H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = min(state[0] + 1, Tmax);  // keys 0 .. pos (the current one was appended)
    const int j0 = chunk * KCHUNK;
    float* out = part + ((int64_t)bh * nchunks + chunk) * (hs + 2);
    const int C = H * hs;
    if (j0 >= n) {
        if (threadIdx.x == 0) {
            out[0] = -INFINITY;
            out[1] = 0.f;
        }
    } else {
        const float* K = cache + cache_index(l, 0, b, h, 0, B, H, Tmax, hs);
        const float* Vc = cache + cache_index(l, 1, b, h, 0, B, H, Tmax, hs);
        const int jw = j0 + warp * 32;  // this warp's first key
        const int j = jw + lane;
        const int nk = max(0, min(32, n - jw));  // keys of this warp
        float sc = -INFINITY;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        if (hs <= 64) {
            float4 kr[16];
            float v0[32], v1[32];
            const float* kp = K + (int64_t)(j < n ? j : 0) * hs;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                kr[u] = (j < n && 4 * u < hs) ? *reinterpret_cast<const float4*>(kp + 4 * u)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                v0[t] = (t < nk && lane < hs) ? Vc[(int64_t)(jw + t) * hs + lane] : 0.f;
                v1[t] = (t < nk && lane + 32 < hs) ? Vc[(int64_t)(jw + t) * hs + lane + 32] : 0.f;
            }
            for (int d = threadIdx.x; d < hs; d += blockDim.x) q[d] = qkv[(int64_t)b * 3 * C + h * hs + d];
            __syncthreads();
            if (j < n) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int u = 0; u < 16; u += 2) {
                    if (4 * u < hs) {
                        const float4 q4 = *reinterpret_cast<const float4*>(q + 4 * u);
                        a0 = fmaf(q4.x, kr[u].x, fmaf(q4.y, kr[u].y, fmaf(q4.z, kr[u].z, fmaf(q4.w, kr[u].w, a0))));
                    }
                    if (4 * u + 4 < hs) {
                        const float4 q5 = *reinterpret_cast<const float4*>(q + 4 * u + 4);
                        a1 = fmaf(q5.x, kr[u + 1].x,
                                  fmaf(q5.y, kr[u + 1].y, fmaf(q5.z, kr[u + 1].z, fmaf(q5.w, kr[u + 1].w, a1))));
                    }
                }
                sc = (a0 + a1) * rsqrtf((float)hs);
            }
            float m = warp_max(sc);
            if (lane == 0) red[0][warp] = m;
            __syncthreads();
            m = fmaxf(red[0][0], red[0][1]);
            const float p = j < n ? expf(sc - m) : 0.f;
            const float ls = warp_sum(p);
            if (lane == 0) red[1][warp] = ls;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float pt = __shfl_sync(0xffffffffu, p, t);
                o[0] = fmaf(t < nk ? pt : 0.f, v0[t], o[0]);
                o[1] = fmaf(t < nk ? pt : 0.f, v1[t], o[1]);
            }
            if (threadIdx.x == 0) out[0] = m;
        } else {
            for (int d = threadIdx.x; d < hs; d += blockDim.x) q[d] = qkv[(int64_t)b * 3 * C + h * hs + d];
            __syncthreads();
            if (j < n) {
                const float* kr = K + (int64_t)j * hs;
                float a0 = 0.f, a1 = 0.f;
                for (int d = 0; d < hs; d += 8) {
                    const float4 k4 = *reinterpret_cast<const float4*>(kr + d);
                    const float4 q4 = *reinterpret_cast<const float4*>(q + d);
                    a0 = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, fmaf(q4.w, k4.w, a0))));
                    if (d + 4 < hs) {
                        const float4 k5 = *reinterpret_cast<const float4*>(kr + d + 4);
                        const float4 q5 = *reinterpret_cast<const float4*>(q + d + 4);
                        a1 = fmaf(q5.x, k5.x, fmaf(q5.y, k5.y, fmaf(q5.z, k5.z, fmaf(q5.w, k5.w, a1))));
                    }
                }
                sc = (a0 + a1) * rsqrtf((float)hs);
            }
            float m = warp_max(sc);
            if (lane == 0) red[0][warp] = m;
            __syncthreads();
            m = fmaxf(red[0][0], red[0][1]);
            const float p = j < n ? expf(sc - m) : 0.f;
            const float ls = warp_sum(p);
            if (lane == 0) red[1][warp] = ls;
            // eight keys' rows of V in flight at a time
            for (int t0 = 0; t0 < nk; t0 += 8) {
                float vv[8][4];
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        vv[u][i] = (t0 + u < nk && lane + 32 * i < hs) ? Vc[(int64_t)(jw + t0 + u) * hs + lane + 32 * i] : 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float pt = __shfl_sync(0xffffffffu, p, (t0 + u) & 31);
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = fmaf(t0 + u < nk ? pt : 0.f, vv[u][i], o[i]);
                }
            }
            if (threadIdx.x == 0) out[0] = m;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (lane + 32 * i < hs) ored[warp][lane + 32 * i] = o[i];
        __syncthreads();
        for (int d = threadIdx.x; d < hs; d += blockDim.x) out[2 + d] = ored[0][d] + ored[1][d];
        if (threadIdx.x == 0) out[1] = red[1][0] + red[1][1];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(&tickets[bh], 1) == nchunks - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    // every thread: the chunks' maxima and sums (the same for all), and its output dimensions
    // d = threadIdx.x, + 64; sixteen chunks' loads in flight at a time. One pass when
    // nchunks <= 16 (the global maximum first); beyond that the running maximum rescales.
    const float* pp = part + (int64_t)bh * nchunks * (hs + 2);
    const int d0 = threadIdx.x, d1 = threadIdx.x + 64;
    float M = -INFINITY, L = 0.f, od0 = 0.f, od1 = 0.f;
    for (int c0 = 0; c0 < nchunks; c0 += 16) {
        float mc[16], lc[16], p0[16], p1[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int c = c0 + u;
            const bool in = c < nchunks;
            mc[u] = in ? __ldcg(pp + (int64_t)c * (hs + 2)) : -INFINITY;
            lc[u] = in ? __ldcg(pp + (int64_t)c * (hs + 2) + 1) : 0.f;
            p0[u] = (in && d0 < hs) ? __ldcg(pp + (int64_t)c * (hs + 2) + 2 + d0) : 0.f;
            p1[u] = (in && d1 < hs) ? __ldcg(pp + (int64_t)c * (hs + 2) + 2 + d1) : 0.f;
        }
        float Mb = M;
#pragma unroll
        for (int u = 0; u < 16; ++u) Mb = fmaxf(Mb, mc[u]);
        if (Mb > M && M != -INFINITY) {
            const float r = expf(M - Mb);
            L *= r;
            od0 *= r;
            od1 *= r;
        }
        M = Mb;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (mc[u] != -INFINITY) {
                const float e = expf(mc[u] - M);
                L += lc[u] * e;
                od0 += p0[u] * e;
                od1 += p1[u] * e;
            }
        }
    }
    if (d0 < hs) y[(int64_t)b * C + h * hs + d0] = od0 / L;
    if (d1 < hs) y[(int64_t)b * C + h * hs + d1] = od1 / L;
    if (threadIdx.x == 0) tickets[bh] = 0;  // ready for the next launch
}

__global__ void gather_last_kernel(const float* __restrict__ x, int B, int Tp, int C, float* __restrict__ last) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * C) return;
    int b = (int)(i / C), c = (int)(i % C);
    last[i] = x[((int64_t)b * Tp + Tp - 1) * C + c];
}

__global__ void copy_ids_kernel(const int32_t* __restrict__ src, int32_t* __restrict__ dst, int n) {
    pdl_trigger();
    pdl_wait();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = src[i];
}

// out [B, t] = the first t columns of ids [B, stride]
__global__ void gather_prefix_kernel(const int32_t* __restrict__ ids, int64_t stride, int B, int t,
                                     int32_t* __restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * t) return;
    out[i] = ids[(i / t) * stride + i % t];
}

// ids[b, pos] = next[b]
__global__ void put_column_kernel(const int32_t* __restrict__ next, int B, int32_t* __restrict__ ids, int64_t stride,
                                  int pos) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) ids[(int64_t)b * stride + pos] = next[b];
}

__global__ void set_state_kernel(int* state, int length, int selections) {
    state[0] = length;
    state[1] = selections;
}

__global__ void advance_kernel(int* state, int dlen, int dsel) {
    pdl_trigger();
    pdl_wait();
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
// value by a 4-pass radix select on ordered keys (each pass's bin found by a parallel scan of
// the 256 counts), keep l >= it (ties kept), weights exp((l - max)/T) in float64, running sum
// over ascending indices, first index whose running sum exceeds u * total. The running sum is
// taken per warp range: warp w owns indices [w R, (w + 1) R) (lanes on consecutive indices),
// the warps' totals locate the range where u * total falls, and that warp walks its range in
// index order, 32 indices at a time by a warp scan.
__global__ void __launch_bounds__(SEL_THREADS) select_kernel(const float* __restrict__ logits, int64_t ld, int V,
                                                             int top_k, float temperature, uint64_t seed,
                                                             uint64_t counter, const int* __restrict__ state,
                                                             int32_t* __restrict__ next) {
    pdl_trigger();
    pdl_wait();
    __shared__ unsigned hist[256];
    __shared__ unsigned wtot[8];
    __shared__ float fred[32];
    __shared__ int ired[32];
    __shared__ double dscan[33];
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
            // warp-aggregated counts: the lanes of a warp that fall in the same bin add once
            // (logits crowd into a few bins of each byte, so per-lane atomics would serialise)
            for (int i0 = warp * 32; i0 < V; i0 += SEL_THREADS) {
                const int i = i0 + lane;
                const uint32_t k = i < V ? ord_key(x[i]) : 0u;
                const bool in = i < V && (k & mask_hi) == pre;
                const unsigned act = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const uint32_t bin = (k >> shift) & 0xFF;
                    const unsigned same = __match_any_sync(act, bin);
                    if ((unsigned)lane == (unsigned)(__ffs(same) - 1)) atomicAdd(&hist[bin], (unsigned)__popc(same));
                }
            }
            __syncthreads();
            // the bin of the want-th largest key: thread t < 256 takes bin 255 - t, and P(t), the
            // count of bins 255 - t .. 255 (inclusive scan over t), first reaches want at
            // t* = #{t : P(t) < want}; the keys above that bin number P(t*) - count(t*)
            const uint32_t want = want_s;
            uint32_t pt = 0, h = 0;
            if (threadIdx.x < 256) {
                h = hist[255 - threadIdx.x];
                pt = h;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t nb = __shfl_up_sync(0xffffffffu, pt, o);
                    if (lane >= o) pt += nb;
                }
                if (lane == 31) wtot[warp] = pt;
            }
            __syncthreads();
            if (threadIdx.x < 256)
                for (int w = 0; w < warp; ++w) pt += wtot[w];
            const int ts = min(__syncthreads_count(threadIdx.x < 256 && pt < want), 255);
            if ((int)threadIdx.x == ts) {
                want_s = want - (pt - h);
                prefix_s = pre | ((uint32_t)(255 - ts) << shift);
            }
            __syncthreads();
        }
        kth = key_float(prefix_s);
    }
    // float64 weights of the kept logits, summed per warp range (lanes on consecutive indices)
    const int R = ((V + 31) / 32 + 31) / 32 * 32;  // V / 32 rounded up to a multiple of 32
    const int r0 = warp * R, r1 = min(V, r0 + R);
    const double inv_t = 1.0 / (double)temperature;
    double local = 0.0;
    for (int i = r0 + lane; i < r1; i += 32) {
        const float v = x[i];
        if (v >= kth) local += exp(((double)v - (double)mx) * inv_t);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if (lane == 0) dscan[warp] = local;
    if (threadIdx.x == 0) pick_s = -1;
    __syncthreads();
    if (threadIdx.x == 0) {
        double run = 0.0;
        for (int t = 0; t < SEL_THREADS / 32; ++t) {
            const double sw = dscan[t];
            dscan[t] = run;  // exclusive prefix
            run += sw;
        }
        uint32_t w0 = philox_word0((uint32_t)(counter + (uint64_t)state[1]), (uint32_t)b, 0u, 0u, (uint32_t)seed,
                                   (uint32_t)(seed >> 32));
        double u = (double)(w0 >> 8) * (1.0 / 16777216.0);
        double target = u * run;
        // the last range whose prefix does not exceed the target
        int t = SEL_THREADS / 32 - 1;
        while (t > 0 && dscan[t] > target) --t;
        ired[1] = t;
        dscan[32] = target;
    }
    __syncthreads();
    if (warp == ired[1]) {
        // this range in index order: the first kept index whose running sum exceeds the target
        // (the last kept one if rounding leaves the sum at or below it)
        const double target = dscan[32];
        double run = dscan[warp];
        int last_kept = -1, chosen = -1;
        for (int i0 = r0; i0 < r1 && chosen < 0; i0 += 32) {
            const int i = i0 + lane;
            const float v = i < r1 ? x[i] : -INFINITY;
            const bool kept = i < r1 && v >= kth;
            const unsigned kb = __ballot_sync(0xffffffffu, kept);
            if (!kb) continue;
            double sc = kept ? exp(((double)v - (double)mx) * inv_t) : 0.0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double nb = __shfl_up_sync(0xffffffffu, sc, o);
                if (lane >= o) sc += nb;
            }
            const unsigned over = __ballot_sync(0xffffffffu, kept && run + sc > target);
            if (over) {
                chosen = i0 + __ffs(over) - 1;
            } else {
                last_kept = i0 + 31 - __clz(kb);
                run += __shfl_sync(0xffffffffu, sc, 31);
            }
        }
        if (lane == 0) pick_s = chosen >= 0 ? chosen : last_kept;
    }
    __syncthreads();
    if (threadIdx.x == 0) next[b] = pick_s >= 0 ? pick_s : ired[0];
}

int gemv_nb(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16; }

// Whether every cluster of the grid (clusters of cs GEMV blocks, NB rows, smem bytes each) can
// be resident at once on this GPU: one wave.
template <int NB>
bool gemv_cluster_fits_nb(dim3 grid, size_t smem, int cs) {
    auto k = gemv_kernel<NB, true>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return false;
    if (cs > 8 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return false;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(GEMV_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = (unsigned)cs;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    return cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess &&
           (int64_t)n * cs >= (int64_t)grid.x * grid.y;
}
// An error already pending from the caller's code is left in place (and the plain GEMV runs);
// an error that the queries themselves raise is cleared.
bool gemv_cluster_fits(int nb, dim3 grid, size_t smem, int cs) {
    if (cudaPeekAtLastError() != cudaSuccess) return false;
    bool ok = false;
    switch (nb) {
        case 1: ok = gemv_cluster_fits_nb<1>(grid, smem, cs); break;
        case 2: ok = gemv_cluster_fits_nb<2>(grid, smem, cs); break;
        case 4: ok = gemv_cluster_fits_nb<4>(grid, smem, cs); break;
        case 8: ok = gemv_cluster_fits_nb<8>(grid, smem, cs); break;
        default: ok = gemv_cluster_fits_nb<16>(grid, smem, cs); break;
    }
    cudaGetLastError();
    return ok;
}

// Y [B, M] = act(LN?(X) W + bias + residual), one launch (see gemv_kernel); append_layer >= 0
// also appends the key/value columns to that layer of the cache.
gk_status gemv(gk_ctx* ctx, gk_kv* kv, const float* X, int64_t ldx, const float* ln_g, const float* ln_b,
               const float* W, int64_t ldw, int K, int M, const float* bias, const float* residual, float* Y, int act,
               float* preact, int append_layer = -1) {
    int B = kv->B;
    int colblocks = (int)cdiv(M, GEMV_COLS);
    GK_REQUIRE(ctx, colblocks <= 1024, GK_ERR_UNSUPPORTED, "decode gemv: %d columns", M);
    int nb = gemv_nb(B);
    // Clusters: the K slices of a column block as one cluster of S blocks (a power of two up to
    // 16), the most whose grid fits one wave at two blocks per SM, with at least 8 rows per slice
    // and every cluster resident at once (a grid whose clusters cannot all be placed runs in
    // waves, each a full latency chain).
    int S = 0;
    for (int cs = 16; cs >= 2 && !S; cs >>= 1) {
        if ((int64_t)colblocks * cs > 2 * ctx->num_sms || K / cs < 8) continue;
        const int ks = (int)cdiv(K, cs);
        if (cdiv(K, ks) != cs) continue;  // every slice non-empty
        const size_t sm = ((size_t)gemv_red_offset(nb, ks) + 8 * (size_t)nb * GEMV_COLS + ((2 * nb + 3) & ~3) +
                           (size_t)nb * GEMV_COLS) * sizeof(float);
        if (gemv_cluster_fits(nb, dim3(colblocks, cs), sm, cs)) S = cs;
    }
    const bool cl = S > 0;
    if (!cl) {
        // K slices: enough blocks for two per SM; at wide batches (more arithmetic per weight
        // row, and every slice adds B x 128 partial sums for the finishing block to read) each
        // slice keeps at least 64 rows (128 for long K)
        const int min_rows = B >= 4 ? (K >= 2048 ? 128 : 64) : 8;
        S = (int)std::max<int64_t>(1, std::min<int64_t>(K / min_rows, cdiv(2 * ctx->num_sms, colblocks)));
    }
    int kslice = (int)cdiv(K, S);
    S = (int)cdiv(K, kslice);
    GK_REQUIRE(ctx, cl || (size_t)S * B * M <= kv->partial_floats, GK_ERR_WORKSPACE,
               "decode gemv: partial buffer too small");
    size_t smem = ((size_t)gemv_red_offset(nb, kslice) + 8 * (size_t)nb * GEMV_COLS + ((2 * nb + 3) & ~3) +
                   (cl ? (size_t)nb * GEMV_COLS : 0)) * sizeof(float);
    GemvArgs a;
    a.X = X; a.ldx = ldx; a.ln_g = ln_g; a.ln_b = ln_b; a.W = W; a.ldw = ldw;
    a.B = B; a.K = K; a.M = M; a.kslice = kslice;
    a.partial = kv->partial; a.tickets = kv->tickets;
    a.bias = bias; a.residual = residual; a.Y = Y; a.ldy = M; a.act = act; a.preact = preact;
    a.cache = append_layer >= 0 ? kv->cache : nullptr;
    a.layer = append_layer; a.H = kv->cfg.H; a.hs = kv->cfg.C / kv->cfg.H; a.Tmax = kv->Tmax; a.state = kv->state;
    dim3 grid(colblocks, S);
    cudaError_t e = cudaSuccess;
#define GEMV_CASE(NBV)                                                                                       \
    case NBV:                                                                                                \
        if (cl) {                                                                                            \
            cudaFuncSetAttribute(gemv_kernel<NBV, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
            e = launch_pdl_cluster(gemv_kernel<NBV, true>, grid, dim3(GEMV_THREADS), smem, ctx->stream, S, a); \
        } else {                                                                                             \
            cudaFuncSetAttribute(gemv_kernel<NBV, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
            e = launch_pdl(gemv_kernel<NBV, false>, grid, dim3(GEMV_THREADS), smem, ctx->stream, a);      \
        }                                                                                                    \
        break;
    switch (nb) {
        GEMV_CASE(1) GEMV_CASE(2) GEMV_CASE(4) GEMV_CASE(8) GEMV_CASE(16)
    }
#undef GEMV_CASE
    if (e != cudaSuccess) return fail(ctx, GK_ERR_CUDA, "decode gemv launch failed: %s", cudaGetErrorString(e));
    return launched(ctx, "gemv");
}

gk_status lm_head(gk_ctx* ctx, gk_kv* kv, const float* X, const float* ln_g, const float* ln_b, const float* wte,
                  float* logits, int64_t ldl) {
    int B = kv->B, C = kv->cfg.C, V = kv->cfg.V;
    int nb = gemv_nb(B);
    size_t smem = ((size_t)nb * C + 2 * (size_t)nb) * sizeof(float);
    int blocks = ctx->num_sms * 2;  // one wave at two blocks per SM
#define LM_CASE(NBV)                                                                                         \
    case NBV:                                                                                                \
        cudaFuncSetAttribute(lm_head_kernel<NBV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
        launch_pdl(lm_head_kernel<NBV>, dim3(blocks), dim3(256), smem, ctx->stream, X, ln_g, ln_b, wte, B, C, V, \
                   logits, ldl);                                                                             \
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
    GK_REQUIRE(ctx, hs <= 128 && hs % 4 == 0 && cfg->C % 4 == 0, GK_ERR_UNSUPPORTED,
               "gk_kv_create: head size / width unsupported");
    GK_REQUIRE(ctx, (int64_t)B * cfg->H <= 1024, GK_ERR_UNSUPPORTED, "gk_kv_create: batch x heads above 1024");
    gk_kv* kv = new gk_kv();
    kv->cfg = *cfg;
    kv->B = B;
    kv->Tmax = Tmax;
    int64_t C = cfg->C, rows = (int64_t)B * Tmax;
    // attention partial slots: chunks of 32 keys (the persistent step's) cover the 64-key chunks
    // of the per-layer path too
    int nchunks = (int)cdiv(Tmax, 32);
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
        cudaMalloc(&kv->ids, ((size_t)rows + B) * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&kv->tickets, 2048 * sizeof(int)) != cudaSuccess ||
        cudaMemset(kv->tickets, 0, 2048 * sizeof(int)) != cudaSuccess ||
        cudaMalloc(&kv->bar, 64 * sizeof(unsigned)) != cudaSuccess ||
        cudaMemset(kv->bar, 0, 64 * sizeof(unsigned)) != cudaSuccess ||
        cudaMemset(kv->cache, 0, (size_t)cfg->L * 2 * rows * C * sizeof(float)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        gk_kv_destroy(kv);
        return fail(ctx, GK_ERR_CUDA, "gk_kv_create: device setup failed");
    }
    mega_setup(ctx, kv);
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
    if (kv->tickets) cudaFree(kv->tickets);
    if (kv->bar) cudaFree(kv->bar);
    if (kv->ids) cudaFree(kv->ids);
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
                                C, 1e-5f, nullptr));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->ln, C, w.t(GK_T_ATTN_W, l), 3 * C, 0, w.t(GK_T_ATTN_B, l), nullptr, 0,
                             kv->qkv, 3 * C, GK_F32, N, C, 3 * C, GK_ACT_NONE, nullptr, 0, nullptr, nullptr));
        kv_write_prefill_kernel<<<(unsigned)cdiv(N * C, 256), 256, 0, ctx->stream>>>(kv->qkv, kv->cache, l, B, Tp, H,
                                                                                    hs, kv->Tmax);
        GK_TRY(launched(ctx, "kv_write_prefill"));
        GK_TRY(gk_attn_fwd(ctx, GK_F32, kv->qkv, kv->y, kv->lse, B, Tp, H, hs));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->y, C, w.t(GK_T_ATTNPROJ_W, l), C, 0, w.t(GK_T_ATTNPROJ_B, l), kv->x, C,
                             kv->x, C, GK_F32, N, C, C, GK_ACT_NONE, nullptr, 0, nullptr, nullptr));
        GK_TRY(gk_layernorm_fwd(ctx, kv->x, w.t(GK_T_LN2_W, l), w.t(GK_T_LN2_B, l), kv->ln, GK_F32, nullptr, nullptr, N,
                                C, 1e-5f, nullptr));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->ln, C, w.t(GK_T_FC_W, l), 4 * C, 0, w.t(GK_T_FC_B, l), nullptr, 0, kv->h,
                             4 * C, GK_F32, N, C, 4 * C, GK_ACT_GELU, kv->pre, 4 * C, nullptr, nullptr));
        GK_TRY(gk_matmul_fwd(ctx, GK_F32, kv->h, 4 * C, w.t(GK_T_MLPPROJ_W, l), C, 0, w.t(GK_T_MLPPROJ_B, l), kv->x, C,
                             kv->x, C, GK_F32, N, 4 * C, C, GK_ACT_NONE, nullptr, 0, nullptr, nullptr));
    }
    gather_last_kernel<<<(unsigned)cdiv((int64_t)B * C, 256), 256, 0, ctx->stream>>>(kv->x, B, Tp, C, kv->last);
    GK_TRY(launched(ctx, "gather_last"));
    GK_TRY(gk_layernorm_fwd(ctx, kv->last, w.t(GK_T_LNF_W), w.t(GK_T_LNF_B), kv->ln, GK_F32, nullptr, nullptr, B, C,
                            1e-5f, nullptr));
    GK_TRY(lm_head(ctx, kv, kv->ln, nullptr, nullptr, w.t(GK_T_WTE), last_logits, c.V));
    set_state_kernel<<<1, 1, 0, ctx->stream>>>(kv->state, Tp, 0);
    GK_TRY(launched(ctx, "set_state"));
    kv->length = Tp;
    return GK_OK;
}

}  // extern "C"

namespace {

// Selection of the next tokens (if `next`) and the device cache position's advance; `pdl`:
// launched as programmatic dependents of the kernel before them (the per-layer path).
gk_status select_and_advance(gk_ctx* ctx, gk_kv* kv, const float* logits, int32_t* next, const gk_sample_cfg* s,
                             bool pdl) {
    const int V = kv->cfg.V;
    int dsel = 0;
    if (next) {
        int top_k = s ? s->top_k : 1;
        float temp = s ? s->temperature : 0.f;
        const uint64_t seed = s ? s->seed : 0, counter = s ? s->counter : 0;
        if (pdl)
            launch_pdl(select_kernel, dim3(kv->B), dim3(SEL_THREADS), 0, ctx->stream, logits, (int64_t)V, V, top_k,
                       temp, seed, counter, (const int*)kv->state, next);
        else
            select_kernel<<<kv->B, SEL_THREADS, 0, ctx->stream>>>(logits, (int64_t)V, V, top_k, temp, seed, counter,
                                                                  kv->state, next);
        GK_TRY(launched(ctx, "select"));
        dsel = 1;
    }
    if (pdl)
        launch_pdl(advance_kernel, dim3(1), dim3(1), 0, ctx->stream, kv->state, 1, dsel);
    else
        advance_kernel<<<1, 1, 0, ctx->stream>>>(kv->state, 1, dsel);
    return launched(ctx, "advance");
}

// The launches of one decode step (arguments checked by the caller); the host mirror of the
// cache length is left to the caller.
gk_status decode_step_launches(gk_ctx* ctx, const float* params, gk_kv* kv, const int32_t* tokens, float* logits,
                               int32_t* next, const gk_sample_cfg* s) {
    const gk_gpt_cfg& c = kv->cfg;
    W w{params, c};
    int B = kv->B, C = c.C, H = c.H, hs = C / H;
    int nchunks = (int)cdiv(kv->Tmax, KCHUNK);
    if (kv->mega) {
        // the whole step (embedding, layers, ln_f and head) in one persistent kernel
        GK_TRY(mega_step(ctx, kv, params, tokens, logits));
        return select_and_advance(ctx, kv, logits, next, s, false);
    }
    launch_pdl(embed_step_kernel, dim3(B), dim3(256), 0, ctx->stream, tokens, w.t(GK_T_WTE), w.t(GK_T_WPE), kv->x, B,
               C, c.V, kv->Tmax, (const int*)kv->state, ctx->d_err);
    GK_TRY(launched(ctx, "embed_step"));
    // per layer: LN1 + QKV (+ key/value append), attention, projection + residual,
    // LN2 + MLP up + GELU, MLP down + residual: five launches
    for (int l = 0; l < c.L; ++l) {
        GK_TRY(gemv(ctx, kv, kv->x, C, w.t(GK_T_LN1_W, l), w.t(GK_T_LN1_B, l), w.t(GK_T_ATTN_W, l), 3 * C, C, 3 * C,
                    w.t(GK_T_ATTN_B, l), nullptr, kv->qkv, GK_ACT_NONE, nullptr, l));
        launch_pdl(decode_attn_kernel, dim3(nchunks, B * H), dim3(64), 0, ctx->stream, (const float*)kv->qkv,
                   (const float*)kv->cache, l, B, H, hs, kv->Tmax, (const int*)kv->state, kv->attn_part, nchunks,
                   kv->tickets + 1024, kv->y);
        GK_TRY(launched(ctx, "decode_attn"));
        GK_TRY(gemv(ctx, kv, kv->y, C, nullptr, nullptr, w.t(GK_T_ATTNPROJ_W, l), C, C, C, w.t(GK_T_ATTNPROJ_B, l),
                    kv->x, kv->x, GK_ACT_NONE, nullptr));
        GK_TRY(gemv(ctx, kv, kv->x, C, w.t(GK_T_LN2_W, l), w.t(GK_T_LN2_B, l), w.t(GK_T_FC_W, l), 4 * C, C, 4 * C,
                    w.t(GK_T_FC_B, l), nullptr, kv->h, GK_ACT_GELU, kv->pre));
        GK_TRY(gemv(ctx, kv, kv->h, 4 * C, nullptr, nullptr, w.t(GK_T_MLPPROJ_W, l), C, 4 * C, C,
                    w.t(GK_T_MLPPROJ_B, l), kv->x, kv->x, GK_ACT_NONE, nullptr));
    }
    GK_TRY(lm_head(ctx, kv, kv->x, w.t(GK_T_LNF_W), w.t(GK_T_LNF_B), w.t(GK_T_WTE), logits, c.V));
    return select_and_advance(ctx, kv, logits, next, s, true);
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
            launch_pdl(copy_ids_kernel, dim3(1), dim3(32 * (int)cdiv(kv->B, 32)), 0, ctx->stream, (const int32_t*)next,
                       tokens, kv->B);
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

gk_status gk_generate_uncached(gk_ctx* ctx, const float* params, gk_kv* kv, int32_t* ids, int Tp, int n_new,
                               float* logits, const gk_sample_cfg* s) {
    GK_TRY(check_kv_args(ctx, params, kv));
    GK_REQUIRE(ctx, ids && logits && Tp >= 1 && n_new >= 0, GK_ERR_ARG, "gk_generate_uncached: bad argument");
    GK_REQUIRE(ctx, (int64_t)Tp + n_new - 1 <= kv->Tmax, GK_ERR_OVERFLOW,
               "gk_generate_uncached: %d + %d tokens exceed the cache (%d)", Tp, n_new, kv->Tmax);
    const int B = kv->B;
    const int64_t stride = (int64_t)Tp + n_new;
    int32_t* next = kv->ids + (int64_t)B * kv->Tmax;
    for (int i = 0; i < n_new; ++i) {
        const int t = Tp + i;
        gather_prefix_kernel<<<(unsigned)cdiv((int64_t)B * t, 256), 256, 0, ctx->stream>>>(ids, stride, B, t, kv->ids);
        GK_TRY(launched(ctx, "gather_prefix"));
        GK_TRY(gk_prefill(ctx, params, kv, kv->ids, t, logits));
        // selection i, as in the cached loop (the prompt's selection, then one per step)
        set_state_kernel<<<1, 1, 0, ctx->stream>>>(kv->state, t, i);
        GK_TRY(launched(ctx, "set_state"));
        GK_TRY(gk_sample(ctx, kv, logits, kv->cfg.V, next, s));
        put_column_kernel<<<1, 32 * (unsigned)cdiv(B, 32), 0, ctx->stream>>>(next, B, ids, stride, t);
        GK_TRY(launched(ctx, "put_column"));
    }
    return GK_OK;
}

}  // extern "C"
