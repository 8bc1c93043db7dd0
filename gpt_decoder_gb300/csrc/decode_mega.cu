// One decode step of the KV-cache generator as a single persistent kernel.
// [LM4] = arabroot.io, "Build a language model in C# from scratch (4): running GPT-2 weights",
// "Generation with a KV cache": per token, the embedding of the token at its position, then per
// layer LayerNorm, the QKV product with the new key and value appended to the cache, attention
// of the query over every cached position (no mask: the cache holds only the past), the output
// projection and the MLP, each with its residual; then ln_f and the tied LM head.
//
// A step reads every weight once (about 495 MB for GPT-2-124M in float32): it is bound by HBM
// bandwidth, and at batch 1 by latency, since each product needs the whole output of the one
// before it. One block per SM runs the whole step (a cooperative launch, so all blocks are
// resident), and the steps' data dependencies become grid barriers: five per layer. The
// weights do not depend on the activations, so every block loads its tiles of the NEXT weight
// matrix into shared memory by TMA while the current phase computes and the barrier settles
// (double buffer, one phase ahead): after a barrier a block finds its weights in shared memory
// and only the activation vectors (a few KB, in L2) are on the critical path.
//
// Products: out[b, n] = sum_k xh[b, k] W[k, n] with W [K, N] as stored ([in, out]). The matrix
// is cut into tiles of cw columns x krows rows (one TMA box per 256 rows); a block takes tiles
// blockIdx.x, + gridDim.x, ... With more than one K split, each split writes its partial sums
// and the last split of a column group to finish (atomic ticket) adds them in split order and
// applies the epilogue; no block waits on another inside a phase. Attention: work items
// (batch row, head, chunk of 32 keys), one per warp, write (max, sum, unnormalised output)
// partials; the last chunk of a (row, head) combines them in chunk order. All sums run in a
// fixed order, so a step is deterministic. The cache runs this kernel for batches of one or
// two rows of models narrower than 512; wider batches and models keep the per-layer launches
// (decode.cu), which are faster there.
//
// Every wait is bounded (one second): a barrier or TMA wait that expires records
// GK_ERR_TIMEOUT, raises the abort word so the other blocks leave at their next barrier, waits
// (bounded) for the block's own TMA copies in flight and returns. After that error the cache
// must be recreated.
#include <math.h>

#include <algorithm>

#include "decode.cuh"
#include "tcgen05.cuh"

namespace gk {
namespace {

using namespace tc;

constexpr int MT = 256;                          // threads per block (8 warps)
constexpr int MAXL = 24;                         // layers the kernel parameters have room for
// Shared memory per batch width NB: two weight buffers (this phase, next), the staged activation
// rows (NB rows of up to 3072 values), and the per-warp partial sums of a tile (8 warps x NB x
// 64 columns; also the LayerNorm gain and bias). Narrow batches leave more room for weights,
// so their products need fewer K splits.
template <int NB>
struct Smem {
    static constexpr uint32_t XS = (NB * 12 < 48 ? NB * 12 : 48) * 1024;
    static constexpr uint32_t RED = (NB * 2 > 8 ? NB * 2 : 8) * 1024;
    static constexpr uint32_t BUF = ((224 * 1024 - XS - RED) / 2) & ~1023u;
    static constexpr size_t BYTES = 2 * (size_t)BUF + XS + RED + 128;
};
constexpr int KW = 32;                           // keys per attention work item (one warp)
constexpr int MEGA_MAX_B = 2;                    // widest batch the persistent step runs
constexpr int MEGA_MAX_C = 512;                  // widest model (C) the persistent step runs
constexpr uint64_t LIMIT_NS = 1000000000ull;     // bounded waits: 1 s
constexpr uint64_t DRAIN_NS = 200000000ull;

// Tiles of one weight kind ([K, N]; the same for every layer).
struct Tiling {
    int K, N;
    int cw;        // columns per tile: 4 to 64 (the TMA box's inner extent)
    int krows;     // rows per K split (a multiple of rows_box)
    int rows_box;  // TMA box rows (<= 256)
    int ks;        // K splits
    int ngroups;   // column groups
    int ntiles;    // ngroups * ks
};

struct LayerOff {
    int64_t ln1_w, ln1_b, attn_b, proj_b, ln2_w, ln2_b, fc_b, mproj_b;
};

enum { W_QKV = 0, W_PROJ = 1, W_FC = 2, W_MPROJ = 3 };

struct MegaArgs {
    CUtensorMap wm[MAXL][4];  // per layer: c_attn, attn c_proj, c_fc, mlp c_proj weights
    Tiling t[4];
    LayerOff lo[MAXL];
    const float* p;  // the flat float32 parameters
    int64_t off_wte, off_wpe, off_lnf_w, off_lnf_b;
    int B, C, H, hs, L, V, Tmax, nchunks_cap;
    const int32_t* tokens;
    const int* state;
    float* cache;
    float *x, *qkv, *y, *h;
    float* logits;
    int64_t ldl;
    float* partial;
    int* tickets;  // [0, 1024) column groups, [1024, 2048) attention (row, head)
    float* attn_part;
    unsigned* bar;
    int* err;
};

__device__ __forceinline__ int64_t cache_at(const MegaArgs& a, int l, int kv, int b, int h, int t) {
    return ((((int64_t)(l * 2 + kv) * a.B + b) * a.H + h) * a.Tmax + t) * a.hs;
}

// ---------------------------------------------------------------- grid barrier
// Arrival counter, never reset: a 64-bit count of every block's arrivals since the cache was
// created. A launch starts at a multiple of the block count (every earlier barrier completed),
// so barrier i of this launch is passed when the count reaches base + (i + 1) * gridDim.x. The
// abort word sits on its own 128-byte line.
constexpr int ABORT_WORD = 32;  // unsigned index of the abort word in the barrier block

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void raise_abort(const MegaArgs& a, int code) {
    report(a.err, code);
    atomicExch(a.bar + ABORT_WORD, 1u);
}

// Returns false if the wait expired or another block aborted (thread 0's verdict, block-wide).
__device__ bool grid_barrier(const MegaArgs& a, unsigned long long& target) {
    __shared__ int ok_s;
    __syncthreads();
    target += gridDim.x;
    if (threadIdx.x == 0) {
        unsigned long long* count = reinterpret_cast<unsigned long long*>(a.bar);
        volatile unsigned* abort_w = a.bar + ABORT_WORD;
        bool ok = *abort_w == 0;
        if (ok) {
            // arrival with release semantics: the block's writes of the phase (ordered before it
            // by the block barrier above) are visible to whoever acquires the count after it
            asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(count) : "memory");
            const uint64_t t0 = globaltimer();
            while (ld_acquire_u64(count) < target) {
                if (*abort_w) {
                    ok = false;
                    break;
                }
                if (globaltimer() - t0 > LIMIT_NS) {
                    raise_abort(a, GK_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
            }
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// ---------------------------------------------------------------- helpers
constexpr int MAXC = 1024;  // widest row the kernel holds in registers (float4 per lane: MAXC / 128)

// Element k of row b of the first layer's input: the token's embedding at the position (zero for
// an id outside the vocabulary or a full cache, which the kernel also reports).
__device__ __forceinline__ float4 embed4(const MegaArgs& a, int b, int k, int pos) {
    const int id = a.tokens[b];
    if (id < 0 || id >= a.V || pos >= a.Tmax) return make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 t = *reinterpret_cast<const float4*>(a.p + a.off_wte + (int64_t)id * a.C + k);
    const float4 q = *reinterpret_cast<const float4*>(a.p + a.off_wpe + (int64_t)pos * a.C + k);
    return make_float4(t.x + q.x, t.y + q.y, t.z + q.z, t.w + q.w);
}

// Mean and rstd (biased variance, eps 1e-5) of rows b < B of the step's input (layer 0: the
// embedding), into st[2b], st[2b + 1]: one warp per row, the row held in registers (every
// load issued before the first use), variance from the deviations (two passes over registers).
__device__ void row_stats(const MegaArgs& a, const float* src, bool embed, int pos, float* st) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int b = warp; b < a.B; b += MT / 32) {
        float4 v[MAXC / 128];
#pragma unroll
        for (int i = 0; i < MAXC / 128; ++i) {
            const int k = i * 128 + lane * 4;
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < a.C) v[i] = embed ? embed4(a, b, k, pos) : __ldcg(reinterpret_cast<const float4*>(src + (int64_t)b * a.C + k));
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < MAXC / 128; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
        const float mean = warp_sum(s) / a.C;
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < MAXC / 128; ++i) {
            if (i * 128 + lane * 4 < a.C) {
                const float d0 = v[i].x - mean, d1 = v[i].y - mean, d2 = v[i].z - mean, d3 = v[i].w - mean;
                q += (d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3);
            }
        }
        const float var = warp_sum(q) / a.C;
        if (lane == 0) {
            st[2 * b] = mean;
            st[2 * b + 1] = rsqrtf(var + 1e-5f);
        }
    }
}

// Phase inputs of a product.
struct GemvIn {
    const float* src;  // [B, K] (global; produced in this kernel)
    bool embed;        // layer 0's first product: the rows are the token embeddings
    const float* ln_w;
    const float* ln_b;  // LayerNorm applied to the rows when not null
};

// Phase outputs of a product.
struct GemvOut {
    const float* bias;  // [N]
    float* y;           // [B, N]
    bool residual;      // y[b, n] += value (in place)
    bool gelu;
    bool append;        // columns [C, 3C) also go to the cache (keys, values)
    int layer;
};

// bias[n] + (residual: y[b, n]), the value the epilogue adds to the product
__device__ __forceinline__ float epilogue_addend(const GemvOut& o, int b, int n, int N) {
    float t = o.bias[n];
    if (o.residual) t += __ldcg(o.y + (int64_t)b * N + n);
    return t;
}

// y[b, n] = act(v + addend) (and the key / value append)
__device__ __forceinline__ float gemv_epilogue(const MegaArgs& a, const GemvOut& o, int b, int n, int N, float v,
                                               float addend, int pos) {
    v += addend;
    float* yp = o.y + (int64_t)b * N + n;
    if (o.gelu) v = gelu_tanh(v);
    *yp = v;
    if (o.append && n >= a.C && pos < a.Tmax) {
        const int which = n / a.C - 1, c = n % a.C;
        a.cache[cache_at(a, o.layer, which, b, c / a.hs, pos) + c % a.hs] = v;
    }
    return v;
}

// Stage rows b < NB of src ([B, ld] in global memory) columns [k0, k0 + kn) into xs [NB][xld]
// (zero past B and kn): float4 pieces (every offset and length a multiple of 4), up to SU loads
// in flight per thread (one round for the staging sizes used here). Layer 0's first product
// reads the embedding instead.
template <int NB>
__device__ void stage_rows(const MegaArgs& a, const float* src, bool embed, int64_t ld, int k0, int kn, int xld,
                           int pos, float* xs) {
    constexpr int SU = NB >= 8 ? 12 : 4 * NB > 4 ? 4 * NB : 4;
    const int q4 = xld / 4, total = NB * q4;
    for (int e0 = threadIdx.x; e0 < total; e0 += SU * MT) {
        float4 v[SU];
#pragma unroll
        for (int u = 0; u < SU; ++u) {
            const int e = e0 + u * MT;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < total) {
                const int b = e / q4, kk = (e - b * q4) * 4;
                if (b < a.B && kk < kn)
                    v[u] = embed ? embed4(a, b, k0 + kk, pos)
                                 : __ldcg(reinterpret_cast<const float4*>(src + (int64_t)b * ld + k0 + kk));
            }
        }
#pragma unroll
        for (int u = 0; u < SU; ++u) {
            const int e = e0 + u * MT;
            if (e < total) *reinterpret_cast<float4*>(xs + e * 4) = v[u];
        }
    }
}

// One product phase (weights already requested into `wb` on barrier `wbar`). Returns false
// if a wait gave up. With LayerNorm the whole rows are staged once (one round of loads), their
// statistics taken from shared memory and the rows normalised in place; otherwise each tile
// stages its own K range.
template <int NB>
__device__ bool gemv_phase(const MegaArgs& a, const Tiling& T, const GemvIn& in, const GemvOut& o, const float* wb,
                           uint64_t* wbar, int wpar, float* xs, float* red, float* st, int pos) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ int last_s;
    if ((int)blockIdx.x >= T.ntiles) return true;
    const bool full_rows = in.ln_w != nullptr;  // K = C: [NB][C] fits the staging area
    // the epilogue's bias (+ residual) of this thread's output in each of the block's first
    // PRE tiles, requested now so that its latency hides behind the staging and the products
    constexpr int PRE = 4;
    float pre[PRE];
    const bool early = T.ks == 1 && tid < NB * T.cw;
#pragma unroll
    for (int i = 0; i < PRE; ++i) {
        const int tile = blockIdx.x + i * gridDim.x, b = tid / T.cw, n = (tile % T.ngroups) * T.cw + tid % T.cw;
        pre[i] = (early && tile < T.ntiles && b < a.B && n < T.N) ? epilogue_addend(o, b, n, T.N) : 0.f;
    }
    if (full_rows) {
        // the LayerNorm gain and bias (into the reduction area, free until the products) and the
        // rows, every load issued before the first store
        const int c4 = T.K / 4;
        float4 gw[MAXC / 128 / 2], gb[MAXC / 128 / 2];
#pragma unroll
        for (int u = 0; u < MAXC / 128 / 2; ++u) {
            const int e = tid + u * MT;
            if (e < c4) {
                gw[u] = *reinterpret_cast<const float4*>(in.ln_w + 4 * e);
                gb[u] = *reinterpret_cast<const float4*>(in.ln_b + 4 * e);
            }
        }
        stage_rows<NB>(a, in.src, in.embed, T.K, 0, T.K, T.K, pos, xs);
#pragma unroll
        for (int u = 0; u < MAXC / 128 / 2; ++u) {
            const int e = tid + u * MT;
            if (e < c4) {
                reinterpret_cast<float4*>(red)[e] = gw[u];
                reinterpret_cast<float4*>(red + T.K)[e] = gb[u];
            }
        }
        __syncthreads();
        for (int b = warp; b < a.B; b += MT / 32) {
            const float* xr = xs + b * T.K;
            float s = 0.f;
            for (int k = lane; k < T.K; k += 32) s += xr[k];
            const float mean = warp_sum(s) / T.K;
            float q = 0.f;
            for (int k = lane; k < T.K; k += 32) {
                const float d = xr[k] - mean;
                q = fmaf(d, d, q);
            }
            const float var = warp_sum(q) / T.K;
            if (lane == 0) {
                st[2 * b] = mean;
                st[2 * b + 1] = rsqrtf(var + 1e-5f);
            }
        }
        __syncthreads();
        for (int e = tid; e < a.B * T.K; e += MT) {
            const int b = e / T.K, k = e - b * T.K;
            xs[e] = (xs[e] - st[2 * b]) * st[2 * b + 1] * red[k] + red[T.K + k];
        }
        __syncthreads();  // normalised rows in place; the reduction area is free again
    } else {
        // the first tile's rows, in the same round of loads as the epilogue's values above: the
        // block barrier below waits for both
        const int k0 = (blockIdx.x / T.ngroups) * T.krows;
        stage_rows<NB>(a, in.src, false, T.K, k0, min(T.krows, T.K - k0), T.krows, pos, xs);
    }
    // the outcome is made block-wide before anyone leaves: every thread then takes the same path
    const bool landed = mbar_wait(wbar, (uint32_t)wpar, nullptr, LIMIT_NS);
    if (__syncthreads_or(!landed)) {
        if (tid == 0) raise_abort(a, GK_ERR_TIMEOUT);
        return false;
    }
    const int G = T.cw / 4;       // float4 column groups of a tile
    const int KL = MT / G;        // k-lanes
    const int g4 = tid % G, kl = tid / G;
    int i = 0;
    for (int tile = blockIdx.x; tile < T.ntiles; tile += gridDim.x, ++i) {
        const int grp = tile % T.ngroups, split = tile / T.ngroups;
        const int k0 = split * T.krows, kn = min(T.krows, T.K - k0), n0 = grp * T.cw;
        const float* w = wb + (size_t)i * T.krows * T.cw;
        const float* xt;  // this tile's rows: xt[b * xld + k], k < kn
        int xld;
        if (full_rows) {
            xt = xs + k0;
            xld = T.K;
        } else {
            if (i > 0) {  // the first tile was staged before the weights' wait
                stage_rows<NB>(a, in.src, false, T.K, k0, kn, T.krows, pos, xs);
                __syncthreads();
            }
            xt = xs;
            xld = T.krows;
        }
        float acc[NB][4];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0.f;
        for (int k = kl; k < kn; k += KL) {
            const float4 wv = *reinterpret_cast<const float4*>(w + (size_t)k * T.cw + 4 * g4);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float xv = xt[b * xld + k];
                acc[b][0] = fmaf(xv, wv.x, acc[b][0]);
                acc[b][1] = fmaf(xv, wv.y, acc[b][1]);
                acc[b][2] = fmaf(xv, wv.z, acc[b][2]);
                acc[b][3] = fmaf(xv, wv.w, acc[b][3]);
            }
        }
        // k-lanes of the same column group inside a warp: lanes differing in bits >= log2(G); the
        // level loop outside, so each level's 4 NB shuffles are independent
        for (int off = 16; off >= G; off >>= 1) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[b][j] += __shfl_xor_sync(0xffffffffu, acc[b][j], off);
        }
        if (lane < G) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int j = 0; j < 4; ++j) red[(warp * NB + b) * T.cw + 4 * g4 + j] = acc[b][j];
        }
        __syncthreads();
        // warps in order: the tile's value for (b, c)
        for (int e = tid; e < NB * T.cw; e += MT) {
            const int b = e / T.cw, c = e - b * T.cw, n = n0 + c;
            if (b >= a.B || n >= T.N) continue;
            float v = 0.f;
            for (int ww = 0; ww < MT / 32; ++ww) v += red[(ww * NB + b) * T.cw + c];
            if (T.ks == 1) {
                float add = 0.f;
#pragma unroll
                for (int u = 0; u < PRE; ++u)
                    if (u == i) add = pre[u];
                if (i >= PRE || e != tid) add = epilogue_addend(o, b, n, T.N);
                gemv_epilogue(a, o, b, n, T.N, v, add, pos);
            } else
                a.partial[((int64_t)split * a.B + b) * T.N + n] = v;
        }
        if (T.ks > 1) {
            __threadfence();
            __syncthreads();
            if (tid == 0) last_s = atomicAdd(&a.tickets[grp], 1) == T.ks - 1;
            __syncthreads();
            if (last_s) {
                __threadfence();
                for (int e = tid; e < a.B * T.cw; e += MT) {
                    const int b = e / T.cw, n = n0 + (e - b * T.cw);
                    if (n >= T.N) continue;
                    float v = 0.f;
                    for (int s0 = 0; s0 < T.ks; s0 += 8) {
                        float pv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            pv[u] = s0 + u < T.ks ? __ldcg(a.partial + ((int64_t)(s0 + u) * a.B + b) * T.N + n) : 0.f;
#pragma unroll
                        for (int u = 0; u < 8; ++u) v += pv[u];
                    }
                    gemv_epilogue(a, o, b, n, T.N, v, epilogue_addend(o, b, n, T.N), pos);
                }
                if (tid == 0) a.tickets[grp] = 0;
            }
        }
        __syncthreads();  // the staging and reduction areas are free for the next tile
    }
    return true;
}

// Attention of the new token's query over keys 0 .. n-1 of layer l. A work item is (row, head,
// chunk of KW = 32 keys) and runs on one warp, so a block has eight items in flight: lane j
// scores key j (its row read whole, every load issued first), the warp's max / sum come from
// shuffles, and for the output lane d takes dimensions d, d + 32, ... over the chunk's keys,
// the probabilities broadcast by shuffles. The item writes (max, sum, unnormalised output);
// the last item of a (row, head) to finish (atomic ticket) combines the chunks in chunk order
// (online rescaling over batches of 32 chunks).
__device__ void attention_phase(const MegaArgs& a, int l, int pos, float* xs) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = min(pos + 1, a.Tmax);
    const int nch = (n + KW - 1) / KW;
    const int items = a.B * a.H * nch;
    const int hs = a.hs, C = a.C;
    float* q = xs + warp * 128;  // this warp's query [hs <= 128]
    const float scale = rsqrtf((float)hs);
    // items spread over the blocks first (warp w of block k takes k + w * gridDim.x, ...)
    for (int item = warp * gridDim.x + blockIdx.x; item < items; item += gridDim.x * (MT / 32)) {
        const int bh = item / nch, ch = item - bh * nch, b = bh / a.H, hd = bh - b * a.H;
        __syncwarp();  // the previous item's reads of q are done
        const int j = ch * KW + lane;
        const float* kp = a.cache + cache_at(a, l, 0, b, hd, j < n ? j : 0);
        const int kn = min(KW, n - ch * KW);  // keys of this chunk
        float* out = a.attn_part + ((int64_t)bh * a.nchunks_cap + ch) * (hs + 2);
        const float* vp = a.cache + cache_at(a, l, 1, b, hd, ch * KW);
        if (hs <= 64) {
            // the key row and this lane's value dimensions (lane, lane + 32) of every key, all
            // loaded before the first use
            float4 kr[16];
            float v0[KW], v1[KW];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                kr[u] = (j < n && 4 * u < hs) ? __ldcg(reinterpret_cast<const float4*>(kp + 4 * u))
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < KW; ++t) {
                v0[t] = (t < kn && lane < hs) ? __ldcg(vp + (int64_t)t * hs + lane) : 0.f;
                v1[t] = (t < kn && lane + 32 < hs) ? __ldcg(vp + (int64_t)t * hs + lane + 32) : 0.f;
            }
            // the query (written by this layer's QKV product), requested after the cache rows
            for (int d = lane; d < hs; d += 32) q[d] = __ldcg(a.qkv + (int64_t)b * 3 * C + hd * hs + d);
            __syncwarp();
            float sc = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (4 * u < hs) {
                    const float4 qv = *reinterpret_cast<const float4*>(q + 4 * u);
                    sc = fmaf(qv.x, kr[u].x, fmaf(qv.y, kr[u].y, fmaf(qv.z, kr[u].z, fmaf(qv.w, kr[u].w, sc))));
                }
            }
            sc = j < n ? sc * scale : -INFINITY;
            const float m = warp_max(sc);
            const float p = j < n ? expf(sc - m) : 0.f;
            const float ls = warp_sum(p);
            float o0 = 0.f, o1 = 0.f;
#pragma unroll
            for (int t = 0; t < KW; ++t) {
                const float pt = __shfl_sync(0xffffffffu, p, t);
                o0 = fmaf(pt, v0[t], o0);
                o1 = fmaf(pt, v1[t], o1);
            }
            if (lane < hs) out[2 + lane] = o0;
            if (lane + 32 < hs) out[2 + lane + 32] = o1;
            if (lane == 0) {
                out[0] = m;
                out[1] = ls;
            }
        } else {
        for (int d = lane; d < hs; d += 32) q[d] = __ldcg(a.qkv + (int64_t)b * 3 * C + hd * hs + d);
        __syncwarp();
        float sc = 0.f;
        for (int d0 = 0; d0 < hs; d0 += 64) {  // 64 dimensions (16 float4) in flight at a time
            float4 kr[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                kr[u] = (j < n && d0 + 4 * u < hs) ? __ldcg(reinterpret_cast<const float4*>(kp + d0 + 4 * u))
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (d0 + 4 * u < hs) {
                    const float4 qv = *reinterpret_cast<const float4*>(q + d0 + 4 * u);
                    sc = fmaf(qv.x, kr[u].x, fmaf(qv.y, kr[u].y, fmaf(qv.z, kr[u].z, fmaf(qv.w, kr[u].w, sc))));
                }
            }
        }
        sc = j < n ? sc * scale : -INFINITY;
        const float m = warp_max(sc);
        const float p = j < n ? expf(sc - m) : 0.f;
        const float ls = warp_sum(p);
        for (int d0 = 0; d0 < hs; d0 += 32) {
            const int d = d0 + lane;
            float o = 0.f;
            for (int t0 = 0; t0 < kn; t0 += 16) {  // sixteen value rows in flight
                float vv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) vv[u] = (t0 + u < kn && d < hs) ? __ldcg(vp + (int64_t)(t0 + u) * hs + d) : 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float pt = __shfl_sync(0xffffffffu, p, (t0 + u) & 31);
                    o = fmaf(t0 + u < kn ? pt : 0.f, vv[u], o);
                }
            }
            if (d < hs) out[2 + d] = o;
        }
        if (lane == 0) {
            out[0] = m;
            out[1] = ls;
        }
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&a.tickets[1024 + bh], 1) == nch - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) continue;
        __threadfence();
        const float* pp = a.attn_part + (int64_t)bh * a.nchunks_cap * (hs + 2);
        float M = -INFINITY, L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};  // dimensions lane + 32 i
        for (int c0 = 0; c0 < nch; c0 += 32) {
            const int c = c0 + lane;
            const float mc = c < nch ? __ldcg(pp + (int64_t)c * (hs + 2)) : -INFINITY;
            const float lc = c < nch ? __ldcg(pp + (int64_t)c * (hs + 2) + 1) : 0.f;
            const float Mb = fmaxf(M, warp_max(mc));
            const float r = M == -INFINITY ? 0.f : expf(M - Mb);
            const float ec = mc == -INFINITY ? 0.f : expf(mc - Mb);
            L = L * r + warp_sum(lc * ec);
            const int nb = min(32, nch - c0);
            for (int i4 = 0; i4 < 4; i4 += 2) {  // two dimension groups' loads in flight together
                if (32 * i4 >= hs) break;
                const int d0 = lane + 32 * i4, d1 = d0 + 32;
                float ov0[32], ov1[32];
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    ov0[u] = (u < nb && d0 < hs) ? __ldcg(pp + (int64_t)(c0 + u) * (hs + 2) + 2 + d0) : 0.f;
                    ov1[u] = (u < nb && d1 < hs) ? __ldcg(pp + (int64_t)(c0 + u) * (hs + 2) + 2 + d1) : 0.f;
                }
                float t0 = acc[i4] * r, t1 = acc[i4 + 1] * r;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const float e = __shfl_sync(0xffffffffu, ec, u);
                    t0 = fmaf(e, ov0[u], t0);
                    t1 = fmaf(e, ov1[u], t1);
                }
                acc[i4] = t0;
                acc[i4 + 1] = t1;
            }
            M = Mb;
        }
        for (int i4 = 0; i4 < 4; ++i4) {
            const int d = lane + 32 * i4;
            if (d < hs) a.y[(int64_t)b * C + hd * hs + d] = acc[i4] / L;
        }
        if (lane == 0) a.tickets[1024 + bh] = 0;
    }
}

// ln_f and the tied head: logits[b, v] = sum_c lnf(x)[b, c] wte[v, c] for this block's rows.
template <int NB>
__device__ void head_phase(const MegaArgs& a, float* xs, float* st) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = a.C;
    row_stats(a, a.x, false, 0, st);
    __syncthreads();
    for (int e = tid; e < NB * C; e += MT) {
        const int b = e / C, c = e - b * C;
        float v = 0.f;
        if (b < a.B) v = (__ldcg(a.x + (int64_t)b * C + c) - st[2 * b]) * st[2 * b + 1] * a.p[a.off_lnf_w + c] +
                         a.p[a.off_lnf_b + c];
        xs[e] = v;
    }
    __syncthreads();
    const int per = (a.V + gridDim.x - 1) / gridDim.x;
    const int v_begin = blockIdx.x * per, v_end = min(a.V, v_begin + per);
    const float* wte = a.p + a.off_wte;
    // RH vocabulary rows per warp and pass, all of their loads in flight (C <= MAXC)
    constexpr int RH = NB <= 4 ? 4 : 2;
    for (int v0 = v_begin + warp * RH; v0 < v_end; v0 += (MT / 32) * RH) {
        float acc[RH][NB];
#pragma unroll
        for (int r = 0; r < RH; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
        float4 w[RH][MAXC / 128];
#pragma unroll
        for (int r = 0; r < RH; ++r)
#pragma unroll
            for (int i = 0; i < MAXC / 128; ++i) {
                const int c = i * 128 + lane * 4;
                w[r][i] = (v0 + r < v_end && c < C) ? *reinterpret_cast<const float4*>(wte + (int64_t)(v0 + r) * C + c)
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int i = 0; i < MAXC / 128; ++i) {
            const int c = i * 128 + lane * 4;
            if (c >= C) break;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float4 xb = *reinterpret_cast<const float4*>(xs + b * C + c);
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    acc[r][b] = fmaf(w[r][i].x, xb.x, fmaf(w[r][i].y, xb.y, fmaf(w[r][i].z, xb.z, fmaf(w[r][i].w, xb.w, acc[r][b]))));
            }
        }
#pragma unroll
        for (int r = 0; r < RH; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[r][b] = warp_sum(acc[r][b]);
#pragma unroll
        for (int r = 0; r < RH; ++r) {
            if (lane < NB && lane < a.B && v0 + r < v_end) {
                float o = 0.f;
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    if (b == lane) o = acc[r][b];
                a.logits[(int64_t)lane * a.ldl + v0 + r] = o;
            }
        }
    }
}

template <int NB>
__global__ void __launch_bounds__(MT, 1) decode_mega_kernel(const __grid_constant__ MegaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    float* wbuf0 = reinterpret_cast<float*>(smem);
    using SM = Smem<NB>;
    float* wbuf1 = reinterpret_cast<float*>(smem + SM::BUF);
    float* xs = reinterpret_cast<float*>(smem + 2 * SM::BUF);
    float* red = reinterpret_cast<float*>(smem + 2 * SM::BUF + SM::XS);
    __shared__ __align__(8) uint64_t wbar[2];
    __shared__ float st[2 * 16];
    __shared__ unsigned long long bar_base;
    const int tid = threadIdx.x;
    const int pos = __ldcg(a.state);
    const int nw = 4 * a.L;  // weight phases
    if (tid == 0) {
        // the arrival count stands at a multiple of the grid size plus this launch's arrivals
        // at its first barrier so far (fewer than the grid size)
        const unsigned long long c0 = ld_acquire_u64(reinterpret_cast<const unsigned long long*>(a.bar));
        bar_base = c0 - c0 % gridDim.x;
        mbar_init(&wbar[0], 1);
        mbar_init(&wbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (blockIdx.x == 0) {
            for (int b = 0; b < a.B; ++b) {
                const int id = a.tokens[b];
                if (pos >= a.Tmax) report(a.err, GK_ERR_OVERFLOW);
                else if (id < 0 || id >= a.V) report(a.err, GK_ERR_INDEX);
            }
        }
    }
    __syncthreads();
    // TMA bookkeeping (thread 0): uses of each buffer's barrier, and whether a use is pending
    uint32_t uses[2] = {0u, 0u};
    int pend[2] = {-1, -1};  // parity of a requested, not yet consumed fill
    auto issue = [&](int w) {
        if (w >= nw) return;
        const int l = w >> 2, j = w & 3, bi = w & 1;
        const Tiling& T = a.t[j];
        uint32_t bytes = 0;
        for (int tile = blockIdx.x; tile < T.ntiles; tile += gridDim.x) bytes += (uint32_t)T.krows * T.cw * 4u;
        if (bytes == 0) return;
        pend[bi] = (int)(uses[bi] & 1u);
        uses[bi]++;
        if (tid == 0) {
            float* dst0 = bi ? wbuf1 : wbuf0;
            fence_proxy_async_smem();  // earlier generic reads of this buffer before the async writes
            mbar_expect_tx(&wbar[bi], bytes);
            int i = 0;
            for (int tile = blockIdx.x; tile < T.ntiles; tile += gridDim.x, ++i) {
                const int grp = tile % T.ngroups, split = tile / T.ngroups;
                float* dst = dst0 + (size_t)i * T.krows * T.cw;
                for (int bx = 0; bx < T.krows / T.rows_box; ++bx)
                    tma_load_2d(&a.wm[l][j], &wbar[bi], dst + (size_t)bx * T.rows_box * T.cw, grp * T.cw,
                                split * T.krows + bx * T.rows_box);
            }
        }
    };
    // parity to wait for before reading phase w's buffer; the request stays pending (for the
    // abort drain) until the phase has waited for it
    auto parity = [&](int w) -> int { return pend[w & 1]; };
    auto consumed = [&](int w) { pend[w & 1] = -1; };
    unsigned long long target = bar_base;
    bool ok = true;
    issue(0);
    const int C = a.C;
    for (int l = 0; l < a.L && ok; ++l) {
        const LayerOff& lo = a.lo[l];
        const float* P = a.p;
        // LN1 + QKV (+ key / value append); layer 0 reads the embedding, block 0 stores it
        if (l == 0 && blockIdx.x == 0) {
            for (int e = tid; e < a.B * C; e += MT) {
                const int b = e / C, k = e - b * C, id = a.tokens[b];
                const bool okid = id >= 0 && id < a.V && pos < a.Tmax;
                a.x[e] = okid ? P[a.off_wte + (int64_t)id * C + k] + P[a.off_wpe + (int64_t)pos * C + k] : 0.f;
            }
        }
        issue(4 * l + 1);
        {
            const int par = parity(4 * l);
            GemvIn in{a.x, l == 0, P + lo.ln1_w, P + lo.ln1_b};
            GemvOut o{P + lo.attn_b, a.qkv, false, false, true, l};
            ok = gemv_phase<NB>(a, a.t[W_QKV], in, o, wbuf0, &wbar[0], par, xs, red, st, pos);
            if (ok) consumed(4 * l);
        }
        if (!ok || !(ok = grid_barrier(a, target))) break;
        attention_phase(a, l, pos, xs);
        if (!(ok = grid_barrier(a, target))) break;
        // attention projection + residual
        issue(4 * l + 2);
        {
            const int par = parity(4 * l + 1);
            GemvIn in{a.y, false, nullptr, nullptr};
            GemvOut o{P + lo.proj_b, a.x, true, false, false, l};
            ok = gemv_phase<NB>(a, a.t[W_PROJ], in, o, wbuf1, &wbar[1], par, xs, red, st, pos);
            if (ok) consumed(4 * l + 1);
        }
        if (!ok || !(ok = grid_barrier(a, target))) break;
        // LN2 + MLP up + GELU
        issue(4 * l + 3);
        {
            const int par = parity(4 * l + 2);
            GemvIn in{a.x, false, P + lo.ln2_w, P + lo.ln2_b};
            GemvOut o{P + lo.fc_b, a.h, false, true, false, l};
            ok = gemv_phase<NB>(a, a.t[W_FC], in, o, wbuf0, &wbar[0], par, xs, red, st, pos);
            if (ok) consumed(4 * l + 2);
        }
        if (!ok || !(ok = grid_barrier(a, target))) break;
        // MLP down + residual
        issue(4 * l + 4);
        {
            const int par = parity(4 * l + 3);
            GemvIn in{a.h, false, nullptr, nullptr};
            GemvOut o{P + lo.mproj_b, a.x, true, false, false, l};
            ok = gemv_phase<NB>(a, a.t[W_MPROJ], in, o, wbuf1, &wbar[1], par, xs, red, st, pos);
            if (ok) consumed(4 * l + 3);
        }
        if (!ok || !(ok = grid_barrier(a, target))) break;
    }
    if (ok) head_phase<NB>(a, xs, st);
    if (!ok && tid == 0) {
        // let this block's requested copies land before its shared memory is released
        for (int bi = 0; bi < 2; ++bi)
            if (pend[bi] >= 0) mbar_wait(&wbar[bi], (uint32_t)pend[bi], nullptr, DRAIN_NS);
    }
}

// ------------------------------------------------------------------- host side
// 2-D float32 map of a [K, N] row-major matrix, box {cw, rows_box}, no swizzle.
bool make_weight_map(CUtensorMap* map, const float* base, int K, int N, int cw, int rows_box) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)K};
    cuuint64_t strides[1] = {(cuuint64_t)N * 4};
    cuuint32_t box[2] = {(cuuint32_t)cw, (cuuint32_t)rows_box};
    cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tiles of a [K, N] weight over nblk blocks for NB batch rows: fewest K splits first (a split
// adds a round of partial sums and a ticket), then fewest tiles per block, then the smallest
// share of weights per block; every tile of a block, its staged rows and its reduction must fit.
bool choose_tiling(int K, int N, int nblk, int NB, uint32_t buf, uint32_t xsb, uint32_t redb, Tiling* out) {
    bool found = false;
    long best_key[3] = {0, 0, 0};
    for (int cw : {4, 8, 16, 32, 64}) {
        const int ngroups = (int)cdiv(N, cw);
        if (ngroups > 1024) continue;  // one ticket per column group
        for (int ks0 = 1; ks0 <= std::max(1, K / 8); ++ks0) {
            int krows = (int)cdiv(K, ks0);
            const int nbox = (int)cdiv(krows, 256);
            const int rows_box = (int)cdiv(cdiv(krows, nbox), 4) * 4;  // float4 staging needs krows % 4 == 0
            krows = rows_box * nbox;
            const int ks = (int)cdiv(K, krows);
            const int ntiles = ngroups * ks;
            const int per = (int)cdiv(ntiles, nblk);
            const long bytes = (long)per * krows * cw * 4;
            if (bytes > (long)buf) continue;
            if ((long)NB * krows * 4 > (long)xsb || (long)(MT / 32) * NB * cw * 4 > (long)redb) continue;
            const long key[3] = {ks, per, bytes};
            if (!found || std::lexicographical_compare(key, key + 3, best_key, best_key + 3)) {
                found = true;
                std::copy(key, key + 3, best_key);
                *out = Tiling{K, N, cw, krows, rows_box, ks, ngroups, ntiles};
            }
            break;  // the first K split count that fits is this width's best
        }
    }
    return found;
}

struct Plan {
    uint32_t buf, xs, red;
    size_t bytes;
};
template <int NB>
Plan plan_of() {
    return Plan{Smem<NB>::BUF, Smem<NB>::XS, Smem<NB>::RED, Smem<NB>::BYTES};
}
Plan plan_for(int nb) {
    switch (nb) {
        case 1: return plan_of<1>();
        case 2: return plan_of<2>();
        case 4: return plan_of<4>();
        case 8: return plan_of<8>();
        default: return plan_of<16>();
    }
}

template <int NB>
bool mega_supported(gk_ctx* ctx, const gk_kv* kv, int* blocks) {
    const gk_gpt_cfg& c = kv->cfg;
    const int hs = c.C / c.H;
    if (c.L > MAXL || c.C % 4 || hs % 4 || hs > 128 || (int64_t)kv->B * c.H > 1024) return false;
    using SM = Smem<NB>;
    if ((size_t)NB * c.C * 4 > SM::XS) return false;  // ln_f rows staged whole
    // rows of ln_f / LayerNorm staged whole; their gain and bias in the reduction area; eight
    // queries of the attention items
    if (c.C > MAXC || (size_t)2 * c.C * 4 > SM::RED || (MT / 32) * 128 * 4 > SM::XS) return false;
    int dev_coop = 0;
    if (cudaDeviceGetAttribute(&dev_coop, cudaDevAttrCooperativeLaunch, ctx->device) != cudaSuccess || !dev_coop)
        return false;
    if (cudaFuncSetAttribute(decode_mega_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::BYTES) !=
        cudaSuccess)
        return false;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mega_kernel<NB>, MT, SM::BYTES) != cudaSuccess ||
        per_sm < 1)
        return false;
    *blocks = ctx->num_sms;
    const int nb = *blocks;
    Tiling t;
    const int C = c.C;
    const uint32_t b = SM::BUF, x = SM::XS, r = SM::RED;
    return choose_tiling(C, 3 * C, nb, NB, b, x, r, &t) && choose_tiling(C, C, nb, NB, b, x, r, &t) &&
           choose_tiling(C, 4 * C, nb, NB, b, x, r, &t) && choose_tiling(4 * C, C, nb, NB, b, x, r, &t);
}

int nb_of(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16; }

}  // namespace

void mega_setup(gk_ctx* ctx, gk_kv* kv) {
    int blocks = 0;
    bool ok = false;
    switch (nb_of(kv->B)) {
        case 1: ok = mega_supported<1>(ctx, kv, &blocks); break;
        case 2: ok = mega_supported<2>(ctx, kv, &blocks); break;
        case 4: ok = mega_supported<4>(ctx, kv, &blocks); break;
        case 8: ok = mega_supported<8>(ctx, kv, &blocks); break;
        default: ok = mega_supported<16>(ctx, kv, &blocks); break;
    }
    cudaGetLastError();
    // measured on GB300 (GPT-2-124M, 512-token prompt), against the per-layer launches as they
    // were before their GEMVs finished on clusters: the persistent step was faster at batch 1
    // and 2 (457 vs 535 and 510 vs 559 us per step), the per-layer launches from batch 4 on
    // (705 vs 835 us at 4, 1508 vs 1625 us at 16; they now take 815 us at 16): the persistent
    // kernel's phases are latency bound at small batches, while its one block per SM limits
    // wide batches' arithmetic. With the GEMVs on clusters the per-layer launches also win for
    // GPT-2-124M (C = 768) at batch 1: 0.376 vs 0.471 ms per step; the persistent step is kept
    // for narrower models at batch 1-2
    kv->mega = ok && kv->bar && kv->B <= MEGA_MAX_B && kv->cfg.C < MEGA_MAX_C;
}

gk_status mega_step(gk_ctx* ctx, gk_kv* kv, const float* params, const int32_t* tokens, float* logits) {
    const gk_gpt_cfg& c = kv->cfg;
    const int nb = nb_of(kv->B), nblk = ctx->num_sms, C = c.C;
    const Plan plan = plan_for(nb);
    MegaArgs a;
    memset(&a, 0, sizeof(a));
    const int KN[4][2] = {{C, 3 * C}, {C, C}, {C, 4 * C}, {4 * C, C}};
    const int which[4] = {GK_T_ATTN_W, GK_T_ATTNPROJ_W, GK_T_FC_W, GK_T_MLPPROJ_W};
    for (int j = 0; j < 4; ++j)
        GK_REQUIRE(ctx, choose_tiling(KN[j][0], KN[j][1], nblk, nb, plan.buf, plan.xs, plan.red, &a.t[j]),
                   GK_ERR_UNSUPPORTED,
                   "decode: no tiling for a %dx%d weight", KN[j][0], KN[j][1]);
    for (int l = 0; l < c.L; ++l) {
        for (int j = 0; j < 4; ++j)
            GK_REQUIRE(ctx,
                       make_weight_map(&a.wm[l][j], params + gk_gpt_offset(&c, which[j], l), KN[j][0], KN[j][1],
                                       a.t[j].cw, a.t[j].rows_box),
                       GK_ERR_UNSUPPORTED, "decode: weight tensor map rejected");
        LayerOff& o = a.lo[l];
        o.ln1_w = gk_gpt_offset(&c, GK_T_LN1_W, l);
        o.ln1_b = gk_gpt_offset(&c, GK_T_LN1_B, l);
        o.attn_b = gk_gpt_offset(&c, GK_T_ATTN_B, l);
        o.proj_b = gk_gpt_offset(&c, GK_T_ATTNPROJ_B, l);
        o.ln2_w = gk_gpt_offset(&c, GK_T_LN2_W, l);
        o.ln2_b = gk_gpt_offset(&c, GK_T_LN2_B, l);
        o.fc_b = gk_gpt_offset(&c, GK_T_FC_B, l);
        o.mproj_b = gk_gpt_offset(&c, GK_T_MLPPROJ_B, l);
    }
    a.p = params;
    a.off_wte = gk_gpt_offset(&c, GK_T_WTE, 0);
    a.off_wpe = gk_gpt_offset(&c, GK_T_WPE, 0);
    a.off_lnf_w = gk_gpt_offset(&c, GK_T_LNF_W, 0);
    a.off_lnf_b = gk_gpt_offset(&c, GK_T_LNF_B, 0);
    a.B = kv->B; a.C = C; a.H = c.H; a.hs = C / c.H; a.L = c.L; a.V = c.V; a.Tmax = kv->Tmax;
    a.nchunks_cap = (int)cdiv(kv->Tmax, KW);
    a.tokens = tokens; a.state = kv->state; a.cache = kv->cache;
    a.x = kv->x; a.qkv = kv->qkv; a.y = kv->y; a.h = kv->h;
    a.logits = logits; a.ldl = c.V;
    a.partial = kv->partial; a.tickets = kv->tickets; a.attn_part = kv->attn_part;
    a.bar = kv->bar; a.err = ctx->d_err;
    size_t need = 0;
    for (int j = 0; j < 4; ++j) need = std::max(need, (size_t)a.t[j].ks * kv->B * a.t[j].N);
    GK_REQUIRE(ctx, need <= kv->partial_floats, GK_ERR_WORKSPACE, "decode: partial buffer too small");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)nblk);
    cfg.blockDim = dim3(MT);
    cfg.dynamicSmemBytes = plan.bytes;
    cfg.stream = ctx->stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaSuccess;
    switch (nb) {
        case 1: e = cudaLaunchKernelEx(&cfg, decode_mega_kernel<1>, a); break;
        case 2: e = cudaLaunchKernelEx(&cfg, decode_mega_kernel<2>, a); break;
        case 4: e = cudaLaunchKernelEx(&cfg, decode_mega_kernel<4>, a); break;
        case 8: e = cudaLaunchKernelEx(&cfg, decode_mega_kernel<8>, a); break;
        default: e = cudaLaunchKernelEx(&cfg, decode_mega_kernel<16>, a); break;
    }
    if (e != cudaSuccess) return fail(ctx, GK_ERR_CUDA, "decode step launch failed: %s", cudaGetErrorString(e));
    return launched(ctx, "decode_mega");
}

}  // namespace gk
