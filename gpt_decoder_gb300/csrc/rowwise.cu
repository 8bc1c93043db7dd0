// Row-wise and elementwise kernels of the decoder step: embedding, LayerNorm, GELU,
// softmax cross-entropy, AdamW. These are HBM-bound: each reads and writes its tensors
// once with coalesced (where alignment allows, 128-bit) accesses and reduces rows with warp
// shuffles. Sources: [LM1] = "Build a language model in C# from scratch (1): the Autograd
// engine", [LM4] = "... (4): running GPT-2 weights" (arabroot.io).
#include <math.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"

using namespace gk;

namespace {

// ------------------------------------------------------------------------ embedding
// x[r, :] = wte[ids[r], :] + wpe[r % T, :]   ([LM1] op table, Embedding; [LM4] Gpt.Step)
__global__ void embedding_fwd_kernel(const int32_t* __restrict__ ids, const float* __restrict__ wte,
                                     const float* __restrict__ wpe, float* __restrict__ x, int64_t N, int T,
                                     int C, int V, int* err) {
    int64_t r = blockIdx.x;
    if (r >= N) return;
    int id = ids[r];
    bool ok = id >= 0 && id < V;
    if (!ok && threadIdx.x == 0) report(err, GK_ERR_INDEX);
    const float* te = wte + (int64_t)(ok ? id : 0) * C;
    const float* pe = wpe + (int64_t)(r % T) * C;
    float* xr = x + r * C;
    if ((C & 3) == 0) {
        for (int c = threadIdx.x * 4; c < C; c += blockDim.x * 4) {
            float4 a = *reinterpret_cast<const float4*>(te + c);
            float4 b = *reinterpret_cast<const float4*>(pe + c);
            float4 o = ok ? make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w) : make_float4(0, 0, 0, 0);
            *reinterpret_cast<float4*>(xr + c) = o;
        }
    } else {
        for (int c = threadIdx.x; c < C; c += blockDim.x) xr[c] = ok ? te[c] + pe[c] : 0.0f;
    }
}

// dwte[id, :] += dx[r, :] for every row r with ids[r] == id, rows in ascending order.
// Block b owns the token range [b*span, (b+1)*span). It scans all ids in chunks of
// blockDim rows, compacts the matching rows of each chunk into shared memory in ascending
// order (warp ballots + a prefix over warps), then its threads add those rows column by
// column. Each (id, column) element is owned by one thread, which performs its additions
// in ascending r: bit-identical to the sequential definition.
constexpr int EMB_BWD_THREADS = 256;
__global__ void __launch_bounds__(EMB_BWD_THREADS) embedding_bwd_wte_kernel(
        const int32_t* __restrict__ ids, const float* __restrict__ dx, float* __restrict__ dwte,
        int64_t N, int C, int V, int span, int* err) {
    __shared__ int rows[EMB_BWD_THREADS];
    __shared__ int warp_cnt[EMB_BWD_THREADS / 32];
    __shared__ int total;
    int lo = blockIdx.x * span, hi = min(V, lo + span);
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t base = 0; base < N; base += EMB_BWD_THREADS) {
        int64_t r = base + threadIdx.x;
        int id = r < N ? ids[r] : -1;
        if (blockIdx.x == 0 && r < N && (id < 0 || id >= V)) report(err, GK_ERR_INDEX);
        bool mine = id >= lo && id < hi;
        unsigned ball = __ballot_sync(0xffffffffu, mine);
        if (lane == 0) warp_cnt[warp] = __popc(ball);
        __syncthreads();
        if (threadIdx.x == 0) {
            int s = 0;
            for (int w = 0; w < EMB_BWD_THREADS / 32; ++w) {
                int c = warp_cnt[w];
                warp_cnt[w] = s;
                s += c;
            }
            total = s;
        }
        __syncthreads();
        if (mine) rows[warp_cnt[warp] + __popc(ball & ((1u << lane) - 1u))] = (int)r;
        __syncthreads();
        int n = total;
        for (int i = 0; i < n; ++i) {
            int rr = rows[i];
            float* dst = dwte + (int64_t)ids[rr] * C;
            const float* src = dx + (int64_t)rr * C;
            for (int c = threadIdx.x; c < C; c += EMB_BWD_THREADS) dst[c] += src[c];
        }
        __syncthreads();
    }
}

// dwpe[t, c] += dx[b*T + t, c] for b ascending: one thread per (t, c).
__global__ void embedding_bwd_wpe_kernel(const float* __restrict__ dx, float* __restrict__ dwpe, int B, int T,
                                         int C) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * C) return;
    int64_t t = i / C, c = i % C;
    float acc = dwpe[i];
    for (int b = 0; b < B; ++b) acc += dx[((int64_t)b * T + t) * C + c];
    dwpe[i] = acc;
}

// ------------------------------------------------------------------------ layernorm
// One warp per row for C <= 1024 with C % 128 == 0 rows held in registers (VPT float4 per
// lane); two-pass mean / variance in registers, so x is read once.
template <int VPT, typename TY>
__global__ void layernorm_fwd_warp_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                          const float* __restrict__ beta, TY* __restrict__ y, float* mean_out,
                                          float* rstd_out, int64_t rows, int C, float eps, int64_t lo_plane,
                                          float* __restrict__ x_copy) {
    int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* xr = x + row * C;
    float4 v[VPT];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        v[i] = *reinterpret_cast<const float4*>(xr + (i * 32 + lane) * 4);
        s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
    float mu = warp_sum(s) / C;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        float a = v[i].x - mu, b = v[i].y - mu, c = v[i].z - mu, d = v[i].w - mu;
        q += (a * a + b * b) + (c * c + d * d);
    }
    float rs = rsqrtf(warp_sum(q) / C + eps);
    if (lane == 0) {
        if (mean_out) mean_out[row] = mu;
        if (rstd_out) rstd_out[row] = rs;
    }
    TY* yr = y + row * C;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        int c = (i * 32 + lane) * 4;
        if (x_copy) *reinterpret_cast<float4*>(x_copy + row * C + c) = v[i];
        float4 g = *reinterpret_cast<const float4*>(gamma + c);
        float4 b = *reinterpret_cast<const float4*>(beta + c);
        float o[4] = {(v[i].x - mu) * rs * g.x + b.x, (v[i].y - mu) * rs * g.y + b.y,
                      (v[i].z - mu) * rs * g.z + b.z, (v[i].w - mu) * rs * g.w + b.w};
        if constexpr (sizeof(TY) == 4) {
            *reinterpret_cast<float4*>(yr + c) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
            // four bf16 in one 8-byte store; the low plane holds what the rounding dropped
            __nv_bfloat162 h0 = __floats2bfloat162_rn(o[0], o[1]), h1 = __floats2bfloat162_rn(o[2], o[3]);
            uint2 hw;
            hw.x = *reinterpret_cast<uint32_t*>(&h0);
            hw.y = *reinterpret_cast<uint32_t*>(&h1);
            *reinterpret_cast<uint2*>(yr + c) = hw;
            if (lo_plane) {
                __nv_bfloat162 l0 = __floats2bfloat162_rn(o[0] - __low2float(h0), o[1] - __high2float(h0));
                __nv_bfloat162 l1 = __floats2bfloat162_rn(o[2] - __low2float(h1), o[3] - __high2float(h1));
                uint2 lw;
                lw.x = *reinterpret_cast<uint32_t*>(&l0);
                lw.y = *reinterpret_cast<uint32_t*>(&l1);
                *reinterpret_cast<uint2*>(yr + c + lo_plane) = lw;
            }
        }
    }
}

// Block-wide sum of one float (any block size that is a multiple of 32, up to 1024).
__device__ float block_sum(float v, float* red) {
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < nw ? red[lane] : 0.f;
    return warp_sum(t);
}

// Block-wide sums of two floats (blocks of 256 threads).
__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    a = warp_sum(a);
    b = warp_sum(b);
    __syncthreads();
    if (lane == 0) red[warp] = make_float2(a, b);
    __syncthreads();
    float2 t = lane < nw ? red[lane] : make_float2(0.f, 0.f);
    return make_float2(warp_sum(t.x), warp_sum(t.y));
}

// General LayerNorm forward (any C): one 256-thread block per row, several rows in flight per
// SM. Pass 1 sums x - s and (x - s)^2 with s the row's first element (so the variance does not
// cancel when the mean is large against the spread); pass 2 re-reads the row, which is still
// in L2, and writes y (and the copy of x): DRAM sees about one read and one write per element.
template <typename TY>
__global__ void __launch_bounds__(256) layernorm_fwd_rows_kernel(const float* __restrict__ x,
                                                                 const float* __restrict__ gamma,
                                                                 const float* __restrict__ beta, TY* __restrict__ y,
                                                                 float* mean_out, float* rstd_out, int64_t rows, int C,
                                                                 float eps, int64_t lo_plane, float* __restrict__ x_copy,
                                                                 int vec) {
    __shared__ float2 red[8];
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * C;
        const float sh = xr[0];
        float s = 0.f, q = 0.f;
        if (vec) {
#pragma unroll 4
            for (int c = threadIdx.x * 4; c < C; c += 1024) {
                const float4 v = *reinterpret_cast<const float4*>(xr + c);
                const float a = v.x - sh, b = v.y - sh, d = v.z - sh, e = v.w - sh;
                s += (a + b) + (d + e);
                q += (a * a + b * b) + (d * d + e * e);
            }
        } else {
            for (int c = threadIdx.x; c < C; c += 256) {
                const float a = xr[c] - sh;
                s += a;
                q = fmaf(a, a, q);
            }
        }
        const float2 t = block_sum2(s, q, red);
        const float md = t.x / C;
        const float mu = sh + md, rs = rsqrtf(fmaxf(t.y / C - md * md, 0.f) + eps);
        if (threadIdx.x == 0) {
            if (mean_out) mean_out[row] = mu;
            if (rstd_out) rstd_out[row] = rs;
        }
        TY* yr = y + row * C;
        for (int c = threadIdx.x; c < C; c += 256) {
            const float a = xr[c];
            if (x_copy) x_copy[row * C + c] = a;
            const float o = (a - mu) * rs * gamma[c] + beta[c];
            store_from_f32(yr + c, o);
            if (lo_plane) store_from_f32(yr + c + lo_plane, o - to_f32(yr[c]));
        }
    }
}

// A row of n floats at p, cut at 16-byte boundaries: `head` leading floats before the first
// boundary, `nb` aligned float4 pieces, `tail` trailing floats (rows of any width and offset,
// the buffers' bases 16-byte aligned). Thread t < head + tail holds edge element edge_index(t).
struct RowCut {
    int head, nb, tail;
    __device__ RowCut(const float* p, int n) {
        head = (int)(((16u - ((uint32_t)(uintptr_t)p & 15u)) & 15u) >> 2);
        if (head > n) head = n;
        nb = (n - head) / 4;
        tail = n - head - 4 * nb;
    }
    __device__ int edge_index(int t) const { return t < head ? t : t < head + tail ? head + 4 * nb + (t - head) : -1; }
};

// Wide rows (C <= LNR_MAXC) held in registers: one 512-thread block per row, every piece of
// the row requested at once (about 200 KB in flight per SM at C = 50257), the mean and then
// the variance of the deviations from registers, and y written from them: DRAM sees one read
// and one write per element. x, y and x_copy must have 16-byte aligned bases.
constexpr int LNR_THREADS = 512, LNR_V4 = 25, LNR_MAXC = LNR_THREADS * 4 * LNR_V4;
template <typename TY>
__global__ void __launch_bounds__(LNR_THREADS, 1) layernorm_fwd_reg_kernel(const float* __restrict__ x,
                                                                           const float* __restrict__ gamma,
                                                                           const float* __restrict__ beta,
                                                                           TY* __restrict__ y, float* mean_out,
                                                                           float* rstd_out, int64_t rows, int C,
                                                                           float eps, int64_t lo_plane,
                                                                           float* __restrict__ x_copy) {
    __shared__ float2 red[LNR_THREADS / 32];
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * C;
        const RowCut cut(xr, C);
        const float4* xb = reinterpret_cast<const float4*>(xr + cut.head);
        float4 v[LNR_V4];
#pragma unroll
        for (int i = 0; i < LNR_V4; ++i) {
            const int q = threadIdx.x + i * LNR_THREADS;
            v[i] = q < cut.nb ? xb[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const int ei = cut.edge_index(threadIdx.x);
        const float ev = ei >= 0 ? xr[ei] : 0.f;
        float s = ev;
#pragma unroll
        for (int i = 0; i < LNR_V4; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
        const float mu = block_sum2(s, 0.f, red).x / C;
        float q2 = ei >= 0 ? (ev - mu) * (ev - mu) : 0.f;
#pragma unroll
        for (int i = 0; i < LNR_V4; ++i) {
            if (threadIdx.x + i * LNR_THREADS < cut.nb) {
                const float a = v[i].x - mu, b = v[i].y - mu, d = v[i].z - mu, e = v[i].w - mu;
                q2 += (a * a + b * b) + (d * d + e * e);
            }
        }
        const float rs = rsqrtf(block_sum2(q2, 0.f, red).x / C + eps);
        if (threadIdx.x == 0) {
            if (mean_out) mean_out[row] = mu;
            if (rstd_out) rstd_out[row] = rs;
        }
        TY* yr = y + row * C;
        if (ei >= 0) {
            if (x_copy) x_copy[row * C + ei] = ev;
            const float o = (ev - mu) * rs * gamma[ei] + beta[ei];
            store_from_f32(yr + ei, o);
            if (lo_plane) store_from_f32(yr + ei + lo_plane, o - to_f32(yr[ei]));
        }
#pragma unroll
        for (int i = 0; i < LNR_V4; ++i) {
            const int q = threadIdx.x + i * LNR_THREADS;
            if (q >= cut.nb) break;
            const int c = cut.head + 4 * q;
            if (x_copy) *reinterpret_cast<float4*>(x_copy + row * C + c) = v[i];
            const float o[4] = {(v[i].x - mu) * rs * gamma[c] + beta[c], (v[i].y - mu) * rs * gamma[c + 1] + beta[c + 1],
                                (v[i].z - mu) * rs * gamma[c + 2] + beta[c + 2],
                                (v[i].w - mu) * rs * gamma[c + 3] + beta[c + 3]};
            if constexpr (sizeof(TY) == 4) {
                *reinterpret_cast<float4*>(yr + c) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    store_from_f32(yr + c + k, o[k]);
                    if (lo_plane) store_from_f32(yr + c + k + lo_plane, o[k] - to_f32(yr[c + k]));
                }
            }
        }
    }
}

// LayerNorm backward, one warp per row (C % 128 == 0, C <= 1024). All of a row's global
// reads (x, dy and, when accumulating, dx) are issued before its two reductions, so a row
// costs one memory round trip. Each block also keeps per-column partial sums of dy*xhat, dy
// and (np == 3) of the resulting dx over its rows and writes them to the workspace
// (partials [gridDim.x][np][C]); a second kernel adds them in block order.
template <int VPT>
__global__ void layernorm_bwd_warp_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                          const float* __restrict__ mean, const float* __restrict__ rstd,
                                          const float* __restrict__ dy, float* __restrict__ dx, int accumulate,
                                          __nv_bfloat16* __restrict__ dx_bf16, float* __restrict__ partial, int np,
                                          int64_t rows, int C) {
    extern __shared__ float sp[];  // [nwarps][np][C] when partials are kept
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float4 pg[VPT], pb[VPT], pd[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) pg[i] = pb[i] = pd[i] = make_float4(0, 0, 0, 0);
    float4 gm[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) gm[i] = *reinterpret_cast<const float4*>(gamma + (i * 32 + lane) * 4);
    for (int64_t row = (int64_t)blockIdx.x * nw + warp; row < rows; row += (int64_t)gridDim.x * nw) {
        const float* xr = x + row * C;
        const float* gr = dy + row * C;
        float* dr = dx + row * C;
        float mu = mean[row], rs = rstd[row];
        float4 a[VPT], g[VPT], p[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            int c = (i * 32 + lane) * 4;
            a[i] = *reinterpret_cast<const float4*>(xr + c);
            g[i] = *reinterpret_cast<const float4*>(gr + c);
            p[i] = accumulate ? *reinterpret_cast<const float4*>(dr + c) : make_float4(0, 0, 0, 0);
        }
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            a[i] = make_float4((a[i].x - mu) * rs, (a[i].y - mu) * rs, (a[i].z - mu) * rs, (a[i].w - mu) * rs);
            float h0 = g[i].x * gm[i].x, h1 = g[i].y * gm[i].y, h2 = g[i].z * gm[i].z, h3 = g[i].w * gm[i].w;
            s1 += (h0 + h1) + (h2 + h3);
            s2 += (h0 * a[i].x + h1 * a[i].y) + (h2 * a[i].z + h3 * a[i].w);
            pg[i].x += g[i].x * a[i].x; pg[i].y += g[i].y * a[i].y;
            pg[i].z += g[i].z * a[i].z; pg[i].w += g[i].w * a[i].w;
            pb[i].x += g[i].x; pb[i].y += g[i].y; pb[i].z += g[i].z; pb[i].w += g[i].w;
        }
        float m1 = warp_sum(s1) / C, m2 = warp_sum(s2) / C;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            int c = (i * 32 + lane) * 4;
            float4 o;
            o.x = rs * (g[i].x * gm[i].x - m1 - a[i].x * m2) + p[i].x;
            o.y = rs * (g[i].y * gm[i].y - m1 - a[i].y * m2) + p[i].y;
            o.z = rs * (g[i].z * gm[i].z - m1 - a[i].z * m2) + p[i].z;
            o.w = rs * (g[i].w * gm[i].w - m1 - a[i].w * m2) + p[i].w;
            *reinterpret_cast<float4*>(dr + c) = o;
            pd[i].x += o.x; pd[i].y += o.y; pd[i].z += o.z; pd[i].w += o.w;
            if (dx_bf16) {
                __nv_bfloat162 lo2 = __floats2bfloat162_rn(o.x, o.y), hi2 = __floats2bfloat162_rn(o.z, o.w);
                uint2 packed;
                packed.x = *reinterpret_cast<uint32_t*>(&lo2);
                packed.y = *reinterpret_cast<uint32_t*>(&hi2);
                *reinterpret_cast<uint2*>(dx_bf16 + row * C + c) = packed;
            }
        }
    }
    if (!partial) return;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        int c = (i * 32 + lane) * 4;
        *reinterpret_cast<float4*>(sp + (warp * np + 0) * C + c) = pg[i];
        *reinterpret_cast<float4*>(sp + (warp * np + 1) * C + c) = pb[i];
        if (np == 3) *reinterpret_cast<float4*>(sp + (warp * np + 2) * C + c) = pd[i];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < np * C; c += blockDim.x) {
        int which = c / C, col = c % C;
        float acc = 0.f;
        for (int w = 0; w < nw; ++w) acc += sp[(w * np + which) * C + col];
        partial[((int64_t)blockIdx.x * np + which) * C + col] = acc;
    }
}

// General LayerNorm backward: one block per row (row stats through a block reduction).
// Per-column partials of dy*xhat, dy (and dx when np == 3) go to partial[slot][np][C] rows
// accumulated by a fixed set of rows per slot (rows r with r % nparts == slot, handled in
// ascending order by one block each), keeping the sum order fixed.
__global__ void layernorm_bwd_block_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                           const float* __restrict__ mean, const float* __restrict__ rstd,
                                           const float* __restrict__ dy, float* __restrict__ dx, int accumulate,
                                           __nv_bfloat16* __restrict__ dx_bf16, float* __restrict__ partial,
                                           int np, int64_t rows, int C) {
    __shared__ float red[32];
    int nparts = gridDim.x;
    for (int64_t row = blockIdx.x; row < rows; row += nparts) {
        const float* xr = x + row * C;
        const float* gr = dy + row * C;
        float mu = mean[row], rs = rstd[row];
        float s1 = 0.f, s2 = 0.f;
        for (int c = threadIdx.x; c < C; c += blockDim.x) {
            float xh = (xr[c] - mu) * rs, h = gr[c] * gamma[c];
            s1 += h;
            s2 += h * xh;
        }
        float m1 = block_sum(s1, red) / C;
        float m2 = block_sum(s2, red) / C;
        float* dr = dx + row * C;
        for (int c = threadIdx.x; c < C; c += blockDim.x) {
            float xh = (xr[c] - mu) * rs, g = gr[c];
            float o = rs * (g * gamma[c] - m1 - xh * m2);
            if (accumulate) o += dr[c];
            dr[c] = o;
            if (dx_bf16) dx_bf16[row * C + c] = __float2bfloat16_rn(o);
            if (partial) {
                float* pp = partial + (int64_t)blockIdx.x * np * C;
                if (row == blockIdx.x) {
                    pp[c] = g * xh;
                    pp[C + c] = g;
                    if (np == 3) pp[2 * C + c] = o;
                } else {
                    pp[c] += g * xh;
                    pp[C + c] += g;
                    if (np == 3) pp[2 * C + c] += o;
                }
            }
        }
    }
}

// Wide-row LayerNorm backward, pass 1: per row, m1 = mean(dy * gamma) and m2 =
// mean(dy * gamma * xhat) into stats[2 row], stats[2 row + 1]; one 256-thread block per row.
__global__ void __launch_bounds__(256) layernorm_bwd_stats_kernel(const float* __restrict__ x,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ mean,
                                                                  const float* __restrict__ rstd,
                                                                  const float* __restrict__ dy, float* __restrict__ stats,
                                                                  int64_t rows, int C, int vec) {
    __shared__ float2 red[8];
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * C;
        const float* gr = dy + row * C;
        const float mu = mean[row], rs = rstd[row];
        float s1 = 0.f, s2 = 0.f;
        if (vec) {
            for (int c = threadIdx.x * 4; c < C; c += 1024) {
                const float4 xv = *reinterpret_cast<const float4*>(xr + c);
                const float4 gv = *reinterpret_cast<const float4*>(gr + c);
                const float4 w = *reinterpret_cast<const float4*>(gamma + c);
                const float h0 = gv.x * w.x, h1 = gv.y * w.y, h2 = gv.z * w.z, h3 = gv.w * w.w;
                s1 += (h0 + h1) + (h2 + h3);
                s2 += (h0 * ((xv.x - mu) * rs) + h1 * ((xv.y - mu) * rs)) +
                      (h2 * ((xv.z - mu) * rs) + h3 * ((xv.w - mu) * rs));
            }
        } else {
            for (int c = threadIdx.x; c < C; c += 256) {
                const float h = gr[c] * gamma[c];
                s1 += h;
                s2 += h * ((xr[c] - mu) * rs);
            }
        }
        const float2 t = block_sum2(s1, s2, red);
        if (threadIdx.x == 0) {
            stats[2 * row] = t.x / C;
            stats[2 * row + 1] = t.y / C;
        }
    }
}

// Wide-row LayerNorm backward, pass 2: a block takes 256 columns (one per thread) of LNB_ROWS
// consecutive rows, writes dx (and its bf16 copy), and leaves the column partials of dy * xhat,
// dy (and, np == 3, dx) over its rows in partial[row block][np][C] (rows in ascending order:
// a fixed summation order).
constexpr int LNB_ROWS = 32;
__global__ void __launch_bounds__(256) layernorm_bwd_cols_kernel(const float* __restrict__ x,
                                                                 const float* __restrict__ gamma,
                                                                 const float* __restrict__ mean,
                                                                 const float* __restrict__ rstd,
                                                                 const float* __restrict__ dy,
                                                                 const float* __restrict__ stats, float* __restrict__ dx,
                                                                 int accumulate, __nv_bfloat16* __restrict__ dx_bf16,
                                                                 float* __restrict__ partial, int np, int64_t rows,
                                                                 int C) {
    const int64_t c = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.y * LNB_ROWS, r1 = std::min<int64_t>(rows, r0 + LNB_ROWS);
    if (c >= C) return;
    const float w = gamma[c];
    float pg = 0.f, pb = 0.f, pd = 0.f;
    for (int64_t r = r0; r < r1; ++r) {
        const int64_t i = r * C + c;
        const float mu = mean[r], rs = rstd[r], m1 = stats[2 * r], m2 = stats[2 * r + 1];
        const float xh = (x[i] - mu) * rs, g = dy[i];
        float o = rs * (g * w - m1 - xh * m2);
        if (accumulate) o += dx[i];
        dx[i] = o;
        if (dx_bf16) dx_bf16[i] = __float2bfloat16_rn(o);
        pg += g * xh;
        pb += g;
        pd += o;
    }
    if (partial) {
        float* pp = partial + (int64_t)blockIdx.y * np * C;
        pp[c] = pg;
        pp[C + c] = pb;
        if (np == 3) pp[2 * C + c] = pd;
    }
}

// out_k[c] += sum_p partial[p][k][c] for k < np (out_0 = dgamma, out_1 = dbeta, out_2 = the
// column sums of dx; a null output is skipped). Block (x, k) takes 32 columns of array k:
// warp w sums slots w, w + 32, ... with four independent running sums (slot order fixed),
// then the 32 warp sums are added in warp order: a fixed summation order. With 32 warps a
// warp has few slots, so the reduction is a few load round trips long.
constexpr int RP_WARPS = 32;
__global__ void __launch_bounds__(RP_WARPS * 32) reduce_partials_kernel(const float* __restrict__ partial, int nparts,
                                                                       int np, int C, float* out0, float* out1,
                                                                       float* out2) {
    __shared__ float red[RP_WARPS][32];
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int k = blockIdx.y, c = blockIdx.x * 32 + lane;
    float* out = k == 0 ? out0 : k == 1 ? out1 : out2;
    if (!out) return;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (c < C) {
        const float* src = partial + (int64_t)k * C + c;
        const int64_t step = (int64_t)np * C;
        int p = warp;
        for (; p + 3 * RP_WARPS < nparts; p += 4 * RP_WARPS) {
            a0 += src[p * step];
            a1 += src[(p + RP_WARPS) * step];
            a2 += src[(p + 2 * RP_WARPS) * step];
            a3 += src[(p + 3 * RP_WARPS) * step];
        }
        for (; p < nparts; p += RP_WARPS) a0 += src[p * step];
    }
    red[warp][lane] = (a0 + a1) + (a2 + a3);
    __syncthreads();
    if (warp == 0 && c < C) {
        float t = 0.f;
        for (int w = 0; w < RP_WARPS; ++w) t += red[w][lane];
        out[c] += t;
    }
}

// ----------------------------------------------------------------------------- GELU
__global__ void gelu_fwd_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        y[i] = gelu_tanh(x[i]);
}
__global__ void gelu_bwd_kernel(const float* __restrict__ x, const float* dy, float* dx, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dx[i] = dy[i] * gelu_tanh_grad(x[i]);
}
__global__ void gelu_fwd_vec_kernel(const float4* __restrict__ x, float4* __restrict__ y, int64_t n4) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = x[i];
        y[i] = make_float4(gelu_tanh(a.x), gelu_tanh(a.y), gelu_tanh(a.z), gelu_tanh(a.w));
    }
}
__global__ void gelu_bwd_vec_kernel(const float4* __restrict__ x, const float4* dy, float4* dx, int64_t n4) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = x[i], g = dy[i];
        dx[i] = make_float4(g.x * gelu_tanh_grad(a.x), g.y * gelu_tanh_grad(a.y), g.z * gelu_tanh_grad(a.z),
                            g.w * gelu_tanh_grad(a.w));
    }
}

// ------------------------------------------------------------- softmax cross-entropy
// One block per row: running (max, sum of exp(x - max)) per thread, merged across the
// block; LSE = max + log(sum). Each thread first takes a vector of values, subtracts its
// own running max once per vector, so about one exp per element.
struct MaxSum {
    float m, s;
};
__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b) {
    float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.f};
    return {m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}
__device__ __forceinline__ MaxSum ms_add4(MaxSum a, float4 v) {
    float vm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    float m = fmaxf(a.m, vm);
    float s = (a.m == -INFINITY ? 0.f : a.s * expf(a.m - m)) + expf(v.x - m) + expf(v.y - m) + expf(v.z - m) +
              expf(v.w - m);
    return {m, s};
}
__device__ __forceinline__ MaxSum ms_add1(MaxSum a, float v) {
    float m = fmaxf(a.m, v);
    return {m, (a.m == -INFINITY ? 0.f : a.s * expf(a.m - m)) + expf(v - m)};
}

constexpr int CE_THREADS = 512;
__global__ void __launch_bounds__(CE_THREADS) softmax_ce_fwd_kernel(const float* __restrict__ logits, int64_t ldl,
                                                                    const int32_t* __restrict__ targets,
                                                                    float* __restrict__ lse_out,
                                                                    float* __restrict__ row_loss, int V, int* err) {
    __shared__ MaxSum red[CE_THREADS / 32];
    int64_t row = blockIdx.x;
    const float* xr = logits + row * ldl;
    MaxSum acc = {-INFINITY, 0.f};
    bool vec = ((ldl & 3) == 0) && aligned16(logits);
    int V4 = vec ? V / 4 : 0;
    for (int i = threadIdx.x; i < V4; i += CE_THREADS) acc = ms_add4(acc, reinterpret_cast<const float4*>(xr)[i]);
    for (int c = V4 * 4 + threadIdx.x; c < V; c += CE_THREADS) acc = ms_add1(acc, xr[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum b = {__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.s, o)};
        acc = ms_merge(acc, b);
    }
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        MaxSum t = red[0];
        for (int w = 1; w < CE_THREADS / 32; ++w) t = ms_merge(t, red[w]);
        float lse = t.m + logf(t.s);
        lse_out[row] = lse;
        int tg = targets[row];
        if (tg < 0 || tg >= V) {
            report(err, GK_ERR_INDEX);
            tg = 0;
        }
        row_loss[row] = lse - xr[tg];
    }
}

// The same per row for narrow rows (V <= 4096, float4-aligned): one warp per row, eight rows
// per block, each lane an online (max, sum) over its float4 pieces, merged across the warp.
__global__ void __launch_bounds__(256) softmax_ce_fwd_warp_kernel(const float* __restrict__ logits, int64_t ldl,
                                                                  const int32_t* __restrict__ targets,
                                                                  float* __restrict__ lse_out,
                                                                  float* __restrict__ row_loss, int64_t rows, int V,
                                                                  int* err) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float* xr = logits + row * ldl;
    MaxSum acc = {-INFINITY, 0.f};
    const int V4 = V / 4;
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // every piece of the row requested before the first use
        const int q = lane + 32 * i;
        v[i] = q < V4 ? reinterpret_cast<const float4*>(xr)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (lane + 32 * i < V4) acc = ms_add4(acc, v[i]);
    for (int c = V4 * 4 + lane; c < V; c += 32) acc = ms_add1(acc, xr[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum b = {__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.s, o)};
        acc = ms_merge(acc, b);
    }
    if (lane == 0) {
        const float lse = acc.m + logf(acc.s);
        lse_out[row] = lse;
        int tg = targets[row];
        if (tg < 0 || tg >= V) {
            report(err, GK_ERR_INDEX);
            tg = 0;
        }
        row_loss[row] = lse - xr[tg];
    }
}

// Wide rows streamed once: one 256-thread block per row (several blocks per SM, so the loads
// of one row overlap the reductions of others). Each thread keeps a running maximum m and a
// sum s of exp(x - m) over its elements, eight float4 pieces at a time (s is rescaled by
// exp(m_old - m_new) when a piece raises the maximum); the threads' (m, s) pairs are combined
// in a fixed tree (lanes, then warps in order), lse = m + log(s). Same result as the two-pass
// form up to float32 rounding; DRAM sees one read per element.
constexpr int CES_THREADS = 256, CES_U = 8;
__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;  // both empty
    s = s * expf(m - M) + s2 * expf(m2 - M);
    m = M;
}
__global__ void __launch_bounds__(CES_THREADS) softmax_ce_fwd_stream_kernel(const float* __restrict__ logits,
                                                                          int64_t ldl,
                                                                          const int32_t* __restrict__ targets,
                                                                          float* __restrict__ lse_out,
                                                                          float* __restrict__ row_loss, int64_t rows,
                                                                          int V, int* err) {
    __shared__ float2 red[CES_THREADS / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = logits + row * ldl;
        const RowCut cut(xr, V);
        const float4* xb = reinterpret_cast<const float4*>(xr + cut.head);
        const int ei = cut.edge_index(threadIdx.x);
        float m = ei >= 0 ? xr[ei] : -INFINITY;
        float s = ei >= 0 ? 1.f : 0.f;
        for (int q0 = threadIdx.x; q0 < cut.nb; q0 += CES_U * CES_THREADS) {
            float4 v[CES_U];
#pragma unroll
            for (int u = 0; u < CES_U; ++u) {
                const int q = q0 + u * CES_THREADS;
                v[u] = q < cut.nb ? xb[q] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            float cm = m;
#pragma unroll
            for (int u = 0; u < CES_U; ++u) cm = fmaxf(cm, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
            if (cm == -INFINITY) continue;  // nothing in this piece yet
            s *= expf(m - cm);  // 0 while s = 0 and m = -inf: exp(-inf) = 0
            m = cm;
            float t = 0.f;
#pragma unroll
            for (int u = 0; u < CES_U; ++u)
                t += (expf(v[u].x - m) + expf(v[u].y - m)) + (expf(v[u].z - m) + expf(v[u].w - m));
            s += t;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
            lse_combine(m, s, m2, s2);
        }
        __syncthreads();  // the previous row's reads of red are done
        if (lane == 0) red[warp] = make_float2(m, s);
        __syncthreads();
        if (threadIdx.x == 0) {
            float M = red[0].x, S = red[0].y;
            for (int w = 1; w < CES_THREADS / 32; ++w) lse_combine(M, S, red[w].x, red[w].y);
            const float lse = M + logf(S);
            lse_out[row] = lse;
            int tg = targets[row];
            if (tg < 0 || tg >= V) {
                report(err, GK_ERR_INDEX);
                tg = 0;
            }
            row_loss[row] = lse - xr[tg];
        }
    }
}

// Resident blocks of softmax_ce_fwd_stream_kernel per SM.
int ce_stream_blocks_per_sm() {
    static int n = 0;
    if (n == 0) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, softmax_ce_fwd_stream_kernel, CES_THREADS, 0) !=
                cudaSuccess || b < 1)
            b = 1;
        n = b;
    }
    return n;
}

// loss = (sum over rows, in a fixed order, in double-float) / rows; one block.
__global__ void mean_rows_kernel(const float* __restrict__ row_loss, int64_t rows, float* loss) {
    block_mean_fixed(row_loss, rows, loss);
}

template <typename TD>
__global__ void softmax_ce_bwd_kernel(const float* __restrict__ logits, int64_t ldl,
                                      const int32_t* __restrict__ targets, const float* __restrict__ lse,
                                      const float* __restrict__ dloss, TD* __restrict__ dl, int64_t lddl,
                                      int64_t rows, int V) {
    int64_t row = blockIdx.y;
    float scale = (dloss ? *dloss : 1.0f) / (float)rows;
    float L = lse[row];
    int tg = targets[row];
    const float* xr = logits + row * ldl;
    TD* dr = dl + row * lddl;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < lddl; c += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        if (c < V) v = scale * (expf(xr[c] - L) - (c == tg ? 1.f : 0.f));
        store_from_f32(dr + c, v);
    }
}

// float32 logits and float32 dlogits, aligned rows: 4 columns per thread.
constexpr int CEB_U = 4;
// float32 dlogits, aligned rows: the float4 pieces of every row (lddl / 4 per row) in one
// grid-stride sweep, CEB_U pieces per thread and pass loaded before any store (dl may alias the
// logits: each thread writes only what it has read).
__global__ void softmax_ce_bwd_vec_kernel(const float* __restrict__ logits, int64_t ldl,
                                          const int32_t* __restrict__ targets, const float* __restrict__ lse,
                                          const float* __restrict__ dloss, float* dl, int64_t lddl, int64_t rows,
                                          int V) {
    const float scale = (dloss ? *dloss : 1.0f) / (float)rows;
    const int64_t q4 = lddl / 4, total = rows * q4;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e0 < total; e0 += CEB_U * step) {
        float4 a[CEB_U];
#pragma unroll
        for (int u = 0; u < CEB_U; ++u) {
            const int64_t e = e0 + u * step;
            a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < total) {
                const int64_t row = e / q4, c = (e - row * q4) * 4;
                const float* xr = logits + row * ldl;
                if (c + 3 < V) {
                    a[u] = *reinterpret_cast<const float4*>(xr + c);
                } else if (c < V) {
                    float t[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int k = 0; k < 4; ++k)
                        if (c + k < V) t[k] = xr[c + k];
                    a[u] = make_float4(t[0], t[1], t[2], t[3]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < CEB_U; ++u) {
            const int64_t e = e0 + u * step;
            if (e >= total) break;
            const int64_t row = e / q4, c = (e - row * q4) * 4;
            const float L = lse[row];
            const int tg = targets[row];
            float t[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) t[k] = c + k < V ? scale * expf(t[k] - L) : 0.f;
            if (tg >= c && tg < c + 4) t[tg - c] -= scale;
            *reinterpret_cast<float4*>(dl + row * lddl + c) = make_float4(t[0], t[1], t[2], t[3]);
        }
    }
}

// float32 dlogits for rows of any width and offset (16-byte aligned bases, (ldl - lddl) % 4 ==
// 0 so that a row of the logits and of dlogits start at the same offset): block (x, row) takes
// float4 pieces of the row's aligned body, CEB_U per thread loaded before any store; block 0
// also the row's leading and trailing floats.
__global__ void softmax_ce_bwd_cut_kernel(const float* __restrict__ logits, int64_t ldl,
                                          const int32_t* __restrict__ targets, const float* __restrict__ lse,
                                          const float* __restrict__ dloss, float* dl, int64_t lddl, int64_t rows,
                                          int V) {
    const int64_t row = blockIdx.y;
    const float scale = (dloss ? *dloss : 1.0f) / (float)rows;
    const float L = lse[row];
    const int tg = targets[row];
    const float* xr = logits + row * ldl;
    float* dr = dl + row * lddl;
    const RowCut cut(xr, V);
    const int step = gridDim.x * blockDim.x;
    for (int q0 = blockIdx.x * blockDim.x + threadIdx.x; q0 < cut.nb; q0 += CEB_U * step) {
        float4 a[CEB_U];
#pragma unroll
        for (int u = 0; u < CEB_U; ++u) {
            const int q = q0 + u * step;
            a[u] = q < cut.nb ? reinterpret_cast<const float4*>(xr + cut.head)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < CEB_U; ++u) {
            const int q = q0 + u * step;
            if (q >= cut.nb) break;
            const int c = cut.head + 4 * q;
            float t[4] = {scale * expf(a[u].x - L), scale * expf(a[u].y - L), scale * expf(a[u].z - L),
                          scale * expf(a[u].w - L)};
            if (tg >= c && tg < c + 4) t[tg - c] -= scale;
            *reinterpret_cast<float4*>(dr + c) = make_float4(t[0], t[1], t[2], t[3]);
        }
    }
    if (blockIdx.x == 0) {
        const int ei = cut.edge_index(threadIdx.x);
        if (ei >= 0) dr[ei] = scale * (expf(xr[ei] - L) - (ei == tg ? 1.f : 0.f));
        // padding columns [V, lddl) of dlogits
        for (int64_t c = V + threadIdx.x; c < lddl; c += blockDim.x) dr[c] = 0.f;
    }
}

// bfloat16 dlogits, aligned rows: 8 columns per thread (16-byte stores).
__global__ void softmax_ce_bwd_bf16_kernel(const float* __restrict__ logits, int64_t ldl,
                                           const int32_t* __restrict__ targets, const float* __restrict__ lse,
                                           const float* __restrict__ dloss, __nv_bfloat16* dl, int64_t lddl,
                                           int64_t rows, int V) {
    int64_t row = blockIdx.y;
    float scale = (dloss ? *dloss : 1.0f) / (float)rows;
    float L = lse[row];
    int tg = targets[row];
    const float* xr = logits + row * ldl;
    __nv_bfloat16* dr = dl + row * lddl;
    for (int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; c < lddl;
         c += (int64_t)gridDim.x * blockDim.x * 8) {
        float t[8];
        if (c + 7 < V) {
            float4 a = *reinterpret_cast<const float4*>(xr + c);
            float4 b = *reinterpret_cast<const float4*>(xr + c + 4);
            t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w; t[4] = b.x; t[5] = b.y; t[6] = b.z; t[7] = b.w;
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = scale * expf(t[k] - L);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = (c + k < V) ? scale * expf(xr[c + k] - L) : 0.f;
        }
        if (tg >= c && tg < c + 8) t[tg - c] -= scale;
        uint4 packed;
        uint32_t* pw = reinterpret_cast<uint32_t*>(&packed);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(t[2 * k], t[2 * k + 1]);
            pw[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(dr + c) = packed;
    }
}

// ---------------------------------------------------------------------------- AdamW
// [LM1] "The optimizer", AdamW: float32 arithmetic as on the page.
__global__ void adamw_kernel(float* __restrict__ p, float* __restrict__ g, float* __restrict__ m,
                             float* __restrict__ v, __nv_bfloat16* __restrict__ pb, __nv_bfloat16* __restrict__ pbl,
                             int64_t n, float lr, float b1,
                             float b2, float eps, float wd, float inv_bc1, float inv_bc2, int zero_grad) {
    int64_t n4 = n / 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 pp = reinterpret_cast<float4*>(p)[i], gg = reinterpret_cast<float4*>(g)[i];
        float4 mm = reinterpret_cast<float4*>(m)[i], vv = reinterpret_cast<float4*>(v)[i];
        float* pe = &pp.x; float* ge = &gg.x; float* me = &mm.x; float* ve = &vv.x;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            me[k] = b1 * me[k] + (1.f - b1) * ge[k];
            ve[k] = b2 * ve[k] + (1.f - b2) * ge[k] * ge[k];
            float mhat = me[k] * inv_bc1, vhat = ve[k] * inv_bc2;
            pe[k] -= lr * (mhat / (sqrtf(vhat) + eps) + wd * pe[k]);
        }
        reinterpret_cast<float4*>(p)[i] = pp;
        reinterpret_cast<float4*>(m)[i] = mm;
        reinterpret_cast<float4*>(v)[i] = vv;
        if (zero_grad) reinterpret_cast<float4*>(g)[i] = make_float4(0, 0, 0, 0);
        if (pb) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y), hi = __floats2bfloat162_rn(pp.z, pp.w);
            uint2 packed;
            packed.x = *reinterpret_cast<uint32_t*>(&lo);
            packed.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(pb)[i] = packed;
            if (pbl) {
                __nv_bfloat162 l0 = __floats2bfloat162_rn(pp.x - __low2float(lo), pp.y - __high2float(lo));
                __nv_bfloat162 l1 = __floats2bfloat162_rn(pp.z - __low2float(hi), pp.w - __high2float(hi));
                uint2 pl;
                pl.x = *reinterpret_cast<uint32_t*>(&l0);
                pl.y = *reinterpret_cast<uint32_t*>(&l1);
                reinterpret_cast<uint2*>(pbl)[i] = pl;
            }
        }
    }
    // tail
    for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float gg = g[i];
        float mm = b1 * m[i] + (1.f - b1) * gg;
        float vv = b2 * v[i] + (1.f - b2) * gg * gg;
        m[i] = mm;
        v[i] = vv;
        float pp = p[i];
        pp -= lr * ((mm * inv_bc1) / (sqrtf(vv * inv_bc2) + eps) + wd * pp);
        p[i] = pp;
        if (zero_grad) g[i] = 0.f;
        if (pb) {
            __nv_bfloat16 hb = __float2bfloat16_rn(pp);
            pb[i] = hb;
            if (pbl) pbl[i] = __float2bfloat16_rn(pp - __bfloat162float(hb));
        }
    }
}

__global__ void to_bf16_kernel(const float* __restrict__ x, __nv_bfloat16* __restrict__ y,
                               __nv_bfloat16* __restrict__ lo, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        __nv_bfloat16 h = __float2bfloat16_rn(x[i]);
        y[i] = h;
        if (lo) lo[i] = __float2bfloat16_rn(x[i] - __bfloat162float(h));
    }
}

int grid_for(gk_ctx* ctx, int64_t work, int threads, int per_sm = 8) {
    int64_t b = cdiv(work, threads);
    int64_t cap = (int64_t)ctx->num_sms * per_sm;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

extern "C" {

gk_status gk_embedding_fwd(gk_ctx* ctx, const int32_t* ids, const float* wte, const float* wpe, float* x, int B,
                           int T, int C, int V) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, ids && wte && wpe && x && B > 0 && T > 0 && C > 0 && V > 0, GK_ERR_ARG, "gk_embedding_fwd: bad argument");
    GK_REQUIRE(ctx, (C & 3) != 0 || (aligned16(wte) && aligned16(wpe) && aligned16(x)), GK_ERR_ALIGN,
               "gk_embedding_fwd: float32 tables must be 16-byte aligned");
    int64_t N = (int64_t)B * T;
    int threads = C >= 512 ? 256 : 128;
    embedding_fwd_kernel<<<(unsigned)N, threads, 0, ctx->stream>>>(ids, wte, wpe, x, N, T, C, V, ctx->d_err);
    return launched(ctx, "embedding_fwd");
}

gk_status gk_embedding_bwd(gk_ctx* ctx, const int32_t* ids, const float* dx, float* dwte, float* dwpe, int B,
                           int T, int C, int V) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, ids && dx && B > 0 && T > 0 && C > 0 && V > 0, GK_ERR_ARG, "gk_embedding_bwd: bad argument");
    int64_t N = (int64_t)B * T;
    if (dwte) {
        int blocks = ctx->num_sms * 4;
        if (blocks > V) blocks = V;
        int span = (int)cdiv(V, blocks);
        blocks = (int)cdiv(V, span);
        embedding_bwd_wte_kernel<<<blocks, EMB_BWD_THREADS, 0, ctx->stream>>>(ids, dx, dwte, N, C, V, span, ctx->d_err);
        GK_TRY(launched(ctx, "embedding_bwd_wte"));
    }
    if (dwpe) {
        int64_t n = (int64_t)T * C;
        embedding_bwd_wpe_kernel<<<(unsigned)cdiv(n, 256), 256, 0, ctx->stream>>>(dx, dwpe, B, T, C);
        GK_TRY(launched(ctx, "embedding_bwd_wpe"));
    }
    return GK_OK;
}

gk_status gk_layernorm_fwd(gk_ctx* ctx, const float* x, const float* gamma, const float* beta, void* y, int y_dtype,
                           float* mean, float* rstd, int64_t rows, int C, float eps, float* x_copy) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, x && gamma && beta && y && rows > 0 && C > 0, GK_ERR_ARG, "gk_layernorm_fwd: bad argument");
    GK_REQUIRE(ctx, y_dtype == GK_F32 || y_dtype == GK_BF16 || y_dtype == GK_BF16X2, GK_ERR_ARG,
               "gk_layernorm_fwd: bad dtype");
    int64_t lo_plane = y_dtype == GK_BF16X2 ? rows * C : 0;
    if (y_dtype == GK_BF16X2) y_dtype = GK_BF16;
    GK_REQUIRE(ctx, !x_copy || (x_copy + rows * C <= x || x + rows * C <= x_copy), GK_ERR_ARG,
               "gk_layernorm_fwd: x_copy overlaps x");
    bool warp_path = (C % 128 == 0) && C <= 1024 && aligned16(x) && aligned16(gamma) && aligned16(beta) &&
                     (!x_copy || aligned16(x_copy)) &&
                     (y_dtype == GK_F32 ? aligned16(y) : ((uintptr_t)y & 7) == 0);
    if (warp_path) {
        int wpb = 4;
        unsigned grid = (unsigned)cdiv(rows, wpb);
        int vpt = C / 128;
#define LN_FWD_CASE(V)                                                                                          \
    case V:                                                                                                     \
        if (y_dtype == GK_F32)                                                                                  \
            layernorm_fwd_warp_kernel<V, float><<<grid, wpb * 32, 0, ctx->stream>>>(x, gamma, beta, (float*)y,  \
                                                                                   mean, rstd, rows, C, eps, lo_plane, \
                                                                                   x_copy);                          \
        else                                                                                                    \
            layernorm_fwd_warp_kernel<V, __nv_bfloat16><<<grid, wpb * 32, 0, ctx->stream>>>(                    \
                x, gamma, beta, (__nv_bfloat16*)y, mean, rstd, rows, C, eps, lo_plane, x_copy);                    \
        break;
        switch (vpt) {
            LN_FWD_CASE(1) LN_FWD_CASE(2) LN_FWD_CASE(3) LN_FWD_CASE(4)
            LN_FWD_CASE(5) LN_FWD_CASE(6) LN_FWD_CASE(7) LN_FWD_CASE(8)
        }
#undef LN_FWD_CASE
        return launched(ctx, "layernorm_fwd");
    }
    const int vec = (C % 4 == 0) && aligned16(x);
    if (C > 4096 && C <= LNR_MAXC && aligned16(x) && (!x_copy || aligned16(x_copy)) && aligned16(y)) {
        // wide rows held in registers: one read and one write of each element
        const unsigned g = (unsigned)std::min<int64_t>(rows, (int64_t)ctx->num_sms * 2);
        if (y_dtype == GK_F32)
            layernorm_fwd_reg_kernel<float><<<g, LNR_THREADS, 0, ctx->stream>>>(x, gamma, beta, (float*)y, mean, rstd,
                                                                               rows, C, eps, 0, x_copy);
        else
            layernorm_fwd_reg_kernel<__nv_bfloat16><<<g, LNR_THREADS, 0, ctx->stream>>>(
                x, gamma, beta, (__nv_bfloat16*)y, mean, rstd, rows, C, eps, lo_plane, x_copy);
        return launched(ctx, "layernorm_fwd");
    }
    const unsigned grid = (unsigned)std::min<int64_t>(rows, (int64_t)ctx->num_sms * 8);
    if (y_dtype == GK_F32)
        layernorm_fwd_rows_kernel<float><<<grid, 256, 0, ctx->stream>>>(x, gamma, beta, (float*)y, mean, rstd, rows, C,
                                                                       eps, 0, x_copy, vec);
    else
        layernorm_fwd_rows_kernel<__nv_bfloat16><<<grid, 256, 0, ctx->stream>>>(
            x, gamma, beta, (__nv_bfloat16*)y, mean, rstd, rows, C, eps, lo_plane, x_copy, vec);
    return launched(ctx, "layernorm_fwd");
}

gk_status gk_layernorm_bwd(gk_ctx* ctx, const float* x, const float* gamma, const float* mean, const float* rstd,
                           const float* dy, float* dx, int accumulate_dx, uint16_t* dx_bf16, float* dgamma,
                           float* dbeta, float* dx_colsum, int64_t rows, int C) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, x && gamma && mean && rstd && dy && dx && rows > 0 && C > 0, GK_ERR_ARG,
               "gk_layernorm_bwd: bad argument");
    const bool want_partials = dgamma || dbeta || dx_colsum;
    const int np = dx_colsum ? 3 : 2;  // partial arrays: dy*xhat, dy (, dx)
    bool warp_path = (C % 128 == 0) && C <= 1024 && aligned16(x) && aligned16(dy) && aligned16(dx) &&
                     aligned16(gamma) && (!dx_bf16 || ((uintptr_t)dx_bf16 & 7) == 0);
    // rows wider than 1024: a statistics pass, then a pass over column strips of 32 rows (the
    // one-block-per-row kernel cannot keep enough bytes in flight at those widths)
    const bool wide = !warp_path && C > 1024;
    int nparts;
    if (warp_path) {
        int wpb = 8;
        nparts = (int)std::min<int64_t>(cdiv(rows, wpb), (int64_t)ctx->num_sms * 2);
    } else if (wide) {
        nparts = (int)cdiv(rows, LNB_ROWS);  // row blocks of the column kernel
    } else {
        // one block per row slot; bound the partial buffer (np x C floats per slot)
        int64_t cap = std::max<int64_t>(8, std::min<int64_t>(1216, (int64_t)(16 << 20) / ((int64_t)np * C * 4)));
        nparts = (int)std::min<int64_t>(rows, cap);
    }
    // workspace: the partial sums, then (wide rows) the per-row statistics
    const size_t part_bytes = want_partials ? (((size_t)nparts * np * C * sizeof(float) + 255) & ~size_t(255)) : 0;
    const size_t stat_bytes = wide ? (size_t)rows * 2 * sizeof(float) : 0;
    char* ws = (char*)workspace(ctx, part_bytes + stat_bytes);
    GK_REQUIRE(ctx, ws || part_bytes + stat_bytes == 0, GK_ERR_WORKSPACE, "gk_layernorm_bwd: needs %zu workspace bytes",
               part_bytes + stat_bytes);
    float* partial = want_partials ? (float*)ws : nullptr;
    if (warp_path) {
        int wpb = 8;
        int vpt = C / 128;
        size_t smem = want_partials ? (size_t)wpb * np * C * sizeof(float) : 0;
#define LN_BWD_CASE(V)                                                                                       \
    case V:                                                                                                  \
        cudaFuncSetAttribute(layernorm_bwd_warp_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                             (int)smem);                                                                     \
        layernorm_bwd_warp_kernel<V><<<nparts, wpb * 32, smem, ctx->stream>>>(                               \
            x, gamma, mean, rstd, dy, dx, accumulate_dx, (__nv_bfloat16*)dx_bf16, partial, np, rows, C);     \
        break;
        switch (vpt) {
            LN_BWD_CASE(1) LN_BWD_CASE(2) LN_BWD_CASE(3) LN_BWD_CASE(4)
            LN_BWD_CASE(5) LN_BWD_CASE(6) LN_BWD_CASE(7) LN_BWD_CASE(8)
        }
#undef LN_BWD_CASE
    } else if (!wide) {
        layernorm_bwd_block_kernel<<<nparts, 512, 0, ctx->stream>>>(x, gamma, mean, rstd, dy, dx, accumulate_dx,
                                                                   (__nv_bfloat16*)dx_bf16, partial, np, rows, C);
    } else {
        GK_REQUIRE(ctx, cdiv(rows, LNB_ROWS) <= 65535, GK_ERR_UNSUPPORTED, "gk_layernorm_bwd: too many rows");
        float* stats = (float*)(ws + part_bytes);
        const int vec = (C % 4 == 0) && aligned16(x) && aligned16(dy) && aligned16(gamma);
        layernorm_bwd_stats_kernel<<<(unsigned)std::min<int64_t>(rows, (int64_t)ctx->num_sms * 8), 256, 0,
                                     ctx->stream>>>(x, gamma, mean, rstd, dy, stats, rows, C, vec);
        GK_TRY(launched(ctx, "layernorm_bwd_stats"));
        layernorm_bwd_cols_kernel<<<dim3((unsigned)cdiv(C, 256), (unsigned)nparts), 256, 0, ctx->stream>>>(
            x, gamma, mean, rstd, dy, stats, dx, accumulate_dx, (__nv_bfloat16*)dx_bf16, partial, np, rows, C);
    }
    GK_TRY(launched(ctx, "layernorm_bwd"));
    if (want_partials) {
        reduce_partials_kernel<<<dim3((unsigned)cdiv(C, 32), (unsigned)np), RP_WARPS * 32, 0, ctx->stream>>>(
            partial, nparts, np, C, dgamma, dbeta, dx_colsum);
        GK_TRY(launched(ctx, "layernorm_bwd_reduce"));
    }
    return GK_OK;
}

gk_status gk_gelu_fwd(gk_ctx* ctx, const float* x, float* y, int64_t n) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, x && y && n >= 0, GK_ERR_ARG, "gk_gelu_fwd: bad argument");
    if (n == 0) return GK_OK;
    if ((n & 3) == 0 && aligned16(x) && aligned16(y))
        gelu_fwd_vec_kernel<<<grid_for(ctx, n / 4, 256), 256, 0, ctx->stream>>>((const float4*)x, (float4*)y, n / 4);
    else
        gelu_fwd_kernel<<<grid_for(ctx, n, 256), 256, 0, ctx->stream>>>(x, y, n);
    return launched(ctx, "gelu_fwd");
}

gk_status gk_gelu_bwd(gk_ctx* ctx, const float* x, const float* dy, float* dx, int64_t n) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, x && dy && dx && n >= 0, GK_ERR_ARG, "gk_gelu_bwd: bad argument");
    if (n == 0) return GK_OK;
    if ((n & 3) == 0 && aligned16(x) && aligned16(dy) && aligned16(dx))
        gelu_bwd_vec_kernel<<<grid_for(ctx, n / 4, 256), 256, 0, ctx->stream>>>((const float4*)x, (const float4*)dy,
                                                                               (float4*)dx, n / 4);
    else
        gelu_bwd_kernel<<<grid_for(ctx, n, 256), 256, 0, ctx->stream>>>(x, dy, dx, n);
    return launched(ctx, "gelu_bwd");
}

gk_status gk_softmax_ce_fwd(gk_ctx* ctx, const float* logits, int64_t ldl, const int32_t* targets, float* loss,
                            float* lse, int64_t rows, int V) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, logits && targets && loss && lse && rows > 0 && V > 0 && ldl >= V, GK_ERR_ARG,
               "gk_softmax_ce_fwd: bad argument");
    GK_REQUIRE(ctx, rows < (1ll << 31), GK_ERR_UNSUPPORTED, "gk_softmax_ce_fwd: too many rows");
    float* row_loss = (float*)workspace(ctx, (size_t)rows * sizeof(float));
    GK_REQUIRE(ctx, row_loss, GK_ERR_WORKSPACE, "gk_softmax_ce_fwd: needs %lld workspace bytes", (long long)rows * 4);
    const bool al = (ldl & 3) == 0 && aligned16(logits);
    if (V <= 4096 && al)
        softmax_ce_fwd_warp_kernel<<<(unsigned)cdiv(rows, 8), 256, 0, ctx->stream>>>(logits, ldl, targets, lse, row_loss,
                                                                                    rows, V, ctx->d_err);
    else if (aligned16(logits))
        softmax_ce_fwd_stream_kernel<<<(unsigned)std::min<int64_t>(rows, (int64_t)ctx->num_sms * ce_stream_blocks_per_sm()),
                                       CES_THREADS, 0, ctx->stream>>>(logits, ldl, targets, lse, row_loss, rows, V,
                                                                      ctx->d_err);
    else
        softmax_ce_fwd_kernel<<<(unsigned)rows, CE_THREADS, 0, ctx->stream>>>(logits, ldl, targets, lse, row_loss, V,
                                                                             ctx->d_err);
    GK_TRY(launched(ctx, "softmax_ce_fwd"));
    mean_rows_kernel<<<1, 1024, 0, ctx->stream>>>(row_loss, rows, loss);
    return launched(ctx, "softmax_ce_mean");
}

gk_status gk_softmax_ce_bwd(gk_ctx* ctx, const float* logits, int64_t ldl, const int32_t* targets, const float* lse,
                            const float* dloss, void* dlogits, int64_t lddl, int dl_dtype, int64_t rows, int V) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, logits && targets && lse && dlogits && rows > 0 && V > 0 && ldl >= V && lddl >= V, GK_ERR_ARG,
               "gk_softmax_ce_bwd: bad argument");
    GK_REQUIRE(ctx, dl_dtype == GK_F32 || dl_dtype == GK_BF16, GK_ERR_ARG, "gk_softmax_ce_bwd: bad dtype");
    GK_REQUIRE(ctx, rows < 65536 * 4096ll, GK_ERR_UNSUPPORTED, "gk_softmax_ce_bwd: too many rows");
    bool alias = (const void*)logits == dlogits;
    GK_REQUIRE(ctx, !alias || (dl_dtype == GK_F32 && lddl == ldl), GK_ERR_ARG,
               "gk_softmax_ce_bwd: in-place needs float32 and equal strides");
    int threads = 256;
    if (dl_dtype == GK_F32 && (ldl & 3) == 0 && (lddl & 3) == 0 && aligned16(logits) && aligned16(dlogits)) {
        const unsigned grid = (unsigned)std::min<int64_t>(cdiv(rows * (lddl / 4), (int64_t)threads * CEB_U),
                                                          (int64_t)ctx->num_sms * 8);
        softmax_ce_bwd_vec_kernel<<<grid, threads, 0, ctx->stream>>>(logits, ldl, targets, lse, dloss, (float*)dlogits,
                                                                    lddl, rows, V);
    } else if (dl_dtype == GK_F32 && aligned16(logits) && aligned16(dlogits) && ((ldl - lddl) & 3) == 0 &&
               rows <= 65535) {
        dim3 grid((unsigned)std::max<int64_t>(1, std::min<int64_t>(cdiv(V / 4, threads * CEB_U), 64)), (unsigned)rows);
        softmax_ce_bwd_cut_kernel<<<grid, threads, 0, ctx->stream>>>(logits, ldl, targets, lse, dloss, (float*)dlogits,
                                                                    lddl, rows, V);
    } else if (dl_dtype == GK_BF16 && (ldl & 7) == 0 && (lddl & 7) == 0 && aligned16(logits) && aligned16(dlogits)) {
        dim3 grid((unsigned)cdiv(cdiv(lddl, 8), threads), (unsigned)rows);
        if (grid.x > 16) grid.x = 16;
        softmax_ce_bwd_bf16_kernel<<<grid, threads, 0, ctx->stream>>>(logits, ldl, targets, lse, dloss,
                                                                     (__nv_bfloat16*)dlogits, lddl, rows, V);
    } else {
        dim3 grid((unsigned)cdiv(lddl, threads), (unsigned)rows);
        if (grid.x > 64) grid.x = 64;
        if (dl_dtype == GK_F32)
            softmax_ce_bwd_kernel<float><<<grid, threads, 0, ctx->stream>>>(logits, ldl, targets, lse, dloss,
                                                                          (float*)dlogits, lddl, rows, V);
        else
            softmax_ce_bwd_kernel<__nv_bfloat16><<<grid, threads, 0, ctx->stream>>>(
                logits, ldl, targets, lse, dloss, (__nv_bfloat16*)dlogits, lddl, rows, V);
    }
    return launched(ctx, "softmax_ce_bwd");
}

gk_status gk_to_bf16(gk_ctx* ctx, const float* x, uint16_t* y, uint16_t* y_lo, int64_t n) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, x && y && n >= 0, GK_ERR_ARG, "gk_to_bf16: bad argument");
    if (n == 0) return GK_OK;
    to_bf16_kernel<<<grid_for(ctx, n, 256), 256, 0, ctx->stream>>>(x, (__nv_bfloat16*)y, (__nv_bfloat16*)y_lo, n);
    return launched(ctx, "to_bf16");
}

gk_status gk_adamw_step(gk_ctx* ctx, const gk_param* params, int n_params, float lr, float beta1, float beta2,
                        float eps, float wd, int step, int zero_grad) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, params && n_params >= 0 && step >= 1, GK_ERR_ARG, "gk_adamw_step: bad argument");
    double bc1 = 1.0 - pow((double)beta1, (double)step);
    double bc2 = 1.0 - pow((double)beta2, (double)step);
    float ib1 = (float)(1.0 / bc1), ib2 = (float)(1.0 / bc2);
    for (int k = 0; k < n_params; ++k) {
        const gk_param& q = params[k];
        GK_REQUIRE(ctx, q.p && q.g && q.m && q.v && q.n >= 0, GK_ERR_ARG, "gk_adamw_step: bad block %d", k);
        GK_REQUIRE(ctx, aligned16(q.p) && aligned16(q.g) && aligned16(q.m) && aligned16(q.v) &&
                            (!q.p_bf16 || ((uintptr_t)q.p_bf16 & 7) == 0) &&
                            (!q.p_bf16_lo || (q.p_bf16 && ((uintptr_t)q.p_bf16_lo & 7) == 0)),
                   GK_ERR_ALIGN, "gk_adamw_step: block %d not 16-byte aligned", k);
        if (q.n == 0) continue;
        adamw_kernel<<<grid_for(ctx, q.n / 4 + 1, 256, 8), 256, 0, ctx->stream>>>(
            q.p, q.g, q.m, q.v, (__nv_bfloat16*)q.p_bf16, (__nv_bfloat16*)q.p_bf16_lo, q.n, lr, beta1, beta2, eps,
            q.decay ? wd : 0.f, ib1, ib2,
            zero_grad);
        GK_TRY(launched(ctx, "adamw"));
    }
    return GK_OK;
}

}  // extern "C"

// ------------------------------------------------- LayerNorm backward without allocation
// Some callers cannot call cudaMalloc at all: a host framework that owns every byte of device
// memory through its own pool, a latency-critical loop that must never enter the allocator,
// or a plugin loaded into a process whose memory budget was fixed before it arrived. They can
// pass the inputs and outputs they own, but not the scratch this operation needs for its
// per-block partial sums of dgamma and dbeta. gk_layernorm_bwd_noalloc takes that scratch
// from one fixed array compiled into the library instead of from a context's workspace.
//
// The array is file-scope device memory of GK_LN_NOALLOC_SCRATCH_FLOATS floats (4 MiB). Every
// GPU that loads this library keeps it until the process exits. In host code its name only
// stands for it: the device address comes from cudaGetSymbolAddress, looked up once per device
// on the first call made with that device current.
namespace {
constexpr int64_t GK_LN_NOALLOC_SCRATCH_FLOATS = 1 << 20;
static __device__ __align__(256) float g_ln_noalloc_scratch[GK_LN_NOALLOC_SCRATCH_FLOATS];

// Per-device cache of the array's device address. Host threads making their first call at the
// same time may both look it up; they store the same value, and the atomics make that well
// defined. The cache assumes the device is not reset (cudaDeviceReset) while the library is
// loaded: a reset would invalidate the address.
constexpr int NOALLOC_MAX_DEVICES = 64;
std::atomic<float*> g_ln_noalloc_addr[NOALLOC_MAX_DEVICES];

gk_status ln_noalloc_scratch(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return GK_ERR_CUDA;
    float* a = g_ln_noalloc_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ln_noalloc_scratch) != cudaSuccess || !p) return GK_ERR_CUDA;
        a = static_cast<float*>(p);
        g_ln_noalloc_addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return GK_OK;
}
}  // namespace

extern "C" gk_status gk_layernorm_bwd_noalloc(void* cuda_stream, const float* x, const float* gamma,
                                              const float* mean, const float* rstd, const float* dy, float* dx,
                                              int accumulate_dx, uint16_t* dx_bf16, float* dgamma, float* dbeta,
                                              int64_t rows, int C) {
    if (!x || !gamma || !mean || !rstd || !dy || !dx || rows <= 0 || C <= 0) return GK_ERR_ARG;
    // at least one partial slot of 2 x C floats must fit in the fixed array
    if ((int64_t)2 * C > GK_LN_NOALLOC_SCRATCH_FLOATS) return GK_ERR_WORKSPACE;
    // an error left pending by earlier, unrelated CUDA work is reported (and left pending)
    // instead of being read back below as this call's launch status
    if (cudaPeekAtLastError() != cudaSuccess) return GK_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    bool want_partials = dgamma || dbeta;
    float* partial = nullptr;
    if (want_partials) GK_TRY(ln_noalloc_scratch(&partial));
    int64_t slots = GK_LN_NOALLOC_SCRATCH_FLOATS / ((int64_t)2 * C);
    int num_sms = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GK_ERR_CUDA;
    bool warp_path = (C % 128 == 0) && C <= 1024 && aligned16(x) && aligned16(dy) && aligned16(dx) &&
                     aligned16(gamma) && (!dx_bf16 || ((uintptr_t)dx_bf16 & 7) == 0);
    int nparts;
    if (warp_path) {
        nparts = (int)std::min<int64_t>(std::min<int64_t>(cdiv(rows, 8), (int64_t)num_sms * 4),
                                        std::min<int64_t>(1216, slots));
        int vpt = C / 128;
        size_t smem = want_partials ? (size_t)8 * 2 * C * sizeof(float) : 0;
        switch (vpt) {
#define LN_NA_CASE(V)                                                                                        \
    case V:                                                                                                  \
        if (cudaFuncSetAttribute(layernorm_bwd_warp_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                                 (int)smem) != cudaSuccess)                                                  \
            return GK_ERR_CUDA;                                                                              \
        layernorm_bwd_warp_kernel<V><<<nparts, 8 * 32, smem, stream>>>(                                      \
            x, gamma, mean, rstd, dy, dx, accumulate_dx, (__nv_bfloat16*)dx_bf16, partial, 2, rows, C);      \
        break;
            LN_NA_CASE(1) LN_NA_CASE(2) LN_NA_CASE(3) LN_NA_CASE(4)
            LN_NA_CASE(5) LN_NA_CASE(6) LN_NA_CASE(7) LN_NA_CASE(8)
#undef LN_NA_CASE
        }
    } else {
        nparts = (int)std::min<int64_t>(rows, std::min<int64_t>(1216, slots));
        layernorm_bwd_block_kernel<<<nparts, 512, 0, stream>>>(x, gamma, mean, rstd, dy, dx, accumulate_dx,
                                                              (__nv_bfloat16*)dx_bf16, partial, 2, rows, C);
    }
    if (cudaGetLastError() != cudaSuccess) return GK_ERR_CUDA;
    if (want_partials) {
        // every slot the reduction reads was written in full by the kernel above
        reduce_partials_kernel<<<dim3((unsigned)cdiv(C, 32), 2), RP_WARPS * 32, 0, stream>>>(partial, nparts, 2, C, dgamma,
                                                                                  dbeta, nullptr);
        if (cudaGetLastError() != cudaSuccess) return GK_ERR_CUDA;
    }
    return GK_OK;
}
