// Causal attention forward on the tensor cores (tcgen05), head size 64, bf16 q/k/v.
// [LM1] = "Build a language model in C# from scratch (1)", op table (BatchMatMulT,
// CausalSoftmax, BatchMatMul); [LM4] = "... (4): running GPT-2 weights", "The 12 tensors we do
// not use" (the causal mask by arithmetic) and "Generation with a KV cache" (1/sqrt(hs)).
//
// One CTA of 128 threads per (128-query tile, batch, head). Q is loaded once by TMA; K and V
// tiles of 128 keys stream through a double buffer. For each key tile:
//   S = Q K^T        one tcgen05 MMA chain (M=128, N=128, K=64) into TMEM columns 0..127;
//   softmax          each thread owns one query row: it reads its S row from TMEM twice
//                    (row max, then exp2 and row sum), applies the causal mask, and writes
//                    P = exp(S - m) as bf16 into shared memory in the 128-byte-swizzled
//                    K-major layout the MMA reads;
//   O_tile = P V     a second MMA chain (M=128, N=64, K=128; V is the MN-major operand) into
//                    TMEM columns 128..191, which the thread adds into its register
//                    accumulator after rescaling by exp(m_old - m_new).
// The result is O / l (bf16) and the row log-sum-exp (float32, natural log) for backward.
// All mbarrier waits are bounded (timeout -> GK_ERR_TIMEOUT in the error word).
#include <math.h>

#include "tcgen05.cuh"

namespace gk {
namespace {

using namespace tc;

constexpr int QT = 128, KT = 128, HS = 64, THREADS = 128;
constexpr uint32_t TILE = 128 * 64 * 2;                 // one 128 x 64 bf16 tile, 16 KB
constexpr size_t SMEM_BYTES = 7 * TILE + 1024 + 128;    // Q, K[2], V[2], P (two tiles)
constexpr uint32_t TMEM_COLS = 256;                     // S: 0..127, O tile: 128..191
constexpr uint64_t WAIT_NS = 1000000000ull;

// Byte offset of element (row r, column c) of a [128 x 128] bf16 tile stored as two K-major
// 128-byte-swizzle halves (columns 0..63, 64..127), each 128 rows x 128 bytes.
__device__ __forceinline__ uint32_t p_offset(int r, int c) {
    int half = c >> 6, byte = (c & 63) * 2;
    int chunk = byte >> 4;
    return (uint32_t)(half * 16384 + r * 128 + (((chunk ^ (r & 7)) << 4) | (byte & 15)));
}

__global__ void __launch_bounds__(THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, __nv_bfloat16* __restrict__ y,
                       float* __restrict__ lse, int T, int H, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = smem + TILE;       // two stages
    uint8_t* sV = smem + 3 * TILE;   // two stages
    uint8_t* sP = smem + 5 * TILE;   // two halves
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 7 * TILE);
    uint64_t* bar_q = bars;
    uint64_t* bar_kv = bars + 1;     // [2]
    uint64_t* bar_s = bars + 3;
    uint64_t* bar_o = bars + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 5);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int C = H * HS;
    const int qt = gridDim.x - 1 - blockIdx.x;  // heaviest (latest) query tiles first
    const int q0 = qt * QT;
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int row0 = b * T;
    const int n_kt = min((T + KT - 1) / KT, (q0 + QT - 1) / KT + 1);

    if (tid == 0) {
        mbar_init(bar_q, 1);
        mbar_init(&bar_kv[0], 1);
        mbar_init(&bar_kv[1], 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_qkv) : "memory");
        mbar_expect_tx(bar_q, TILE);
        tma_load_2d(&tm_qkv, bar_q, sQ, h * HS, row0 + q0);
        mbar_expect_tx(&bar_kv[0], 2 * TILE);
        tma_load_2d(&tm_qkv, &bar_kv[0], sK, C + h * HS, row0);
        tma_load_2d(&tm_qkv, &bar_kv[0], sV, 2 * C + h * HS, row0);
    }

    const uint32_t idesc_s = instr_desc_bf16(false, false, 128, 128);
    const uint32_t idesc_o = instr_desc_bf16(false, true, 128, 64);
    const float sl2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
    const int r = warp * 32 + (tid & 31);            // this thread's query row (TMEM lane)
    const int qq = q0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    float o[HS];
#pragma unroll
    for (int d = 0; d < HS; ++d) o[d] = 0.f;
    float m = -INFINITY, l = 0.f;
    bool aborted = false;
    int kv_pending[2] = {1, 0};  // thread 0: TMA loads issued and not yet waited for
    int q_pending = 1;

    for (int j = 0; j < n_kt; ++j) {
        const int st = j & 1;
        const uint32_t kph = (j >> 1) & 1, ph = j & 1;
        bool fail = false;
        if (tid == 0) {
            bool w = (j > 0 || mbar_wait(bar_q, 0, nullptr, WAIT_NS)) && mbar_wait(&bar_kv[st], kph, nullptr, WAIT_NS);
            if (w) {
                q_pending = 0;
                kv_pending[st] = 0;
                tc_fence_after();
                uint32_t q_a = saddr(sQ), k_a = saddr(sK + st * TILE);
#pragma unroll
                for (int k = 0; k < HS / 16; ++k)
                    umma_bf16(tmem, smem_desc(q_a + k * 32, 16, 1024), smem_desc(k_a + k * 32, 16, 1024), idesc_s,
                              k > 0);
                umma_commit(bar_s);
                if (j + 1 < n_kt) {
                    // the other stage's last readers (tile j-1's MMAs) completed before bar_o
                    int ns = st ^ 1;
                    mbar_expect_tx(&bar_kv[ns], 2 * TILE);
                    tma_load_2d(&tm_qkv, &bar_kv[ns], sK + ns * TILE, C + h * HS, row0 + (j + 1) * KT);
                    tma_load_2d(&tm_qkv, &bar_kv[ns], sV + ns * TILE, 2 * C + h * HS, row0 + (j + 1) * KT);
                    kv_pending[ns] = 1;
                }
            }
            fail = !w;
        }
        // every break decision is taken by the whole block together (__syncthreads_or)
        if (__syncthreads_or(fail)) {
            aborted = true;
            break;
        }
        if (__syncthreads_or(!mbar_wait(bar_s, ph, nullptr, WAIT_NS))) {
            aborted = true;
            break;
        }
        tc_fence_after();
        // pass 1: row max of the scaled, masked scores of this key tile
        const int k0 = j * KT;
        float tmax = -INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < KT; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                int kk = k0 + c0 + i;
                float t = __uint_as_float(v[i]) * sl2;
                if (kk <= qq && kk < T) tmax = fmaxf(tmax, t);
            }
        }
        const float m_new = fmaxf(m, tmax);
        const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m - m_new);
        // pass 2: P = exp2(t - m_new) as bf16 into the swizzled P tile; row sum in float32
        float psum = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < KT; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + c0, v);
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    int kk = k0 + c0 + i + e;
                    float t = __uint_as_float(v[i + e]) * sl2;
                    pv[e] = (kk <= qq && kk < T && m_new != -INFINITY) ? exp2f(t - m_new) : 0.f;
                    psum += pv[e];
                }
                uint4 pk;
                uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __nv_bfloat162 t2 = __floats2bfloat162_rn(pv[2 * e], pv[2 * e + 1]);
                    pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                }
                *reinterpret_cast<uint4*>(sP + p_offset(r, c0 + i)) = pk;
            }
        }
        l = l * corr + psum;
        m = m_new;
        fence_proxy_async_smem();  // P's generic-proxy stores -> visible to the tensor core
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            uint32_t p_a = saddr(sP), v_a = saddr(sV + st * TILE);
#pragma unroll
            for (int k = 0; k < KT / 16; ++k)
                umma_bf16(tmem + 128, smem_desc(p_a + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                          smem_desc(v_a + k * 2048, 8192, 1024), idesc_o, k > 0);
            umma_commit(bar_o);
        }
        if (__syncthreads_or(!mbar_wait(bar_o, ph, nullptr, WAIT_NS))) {
            aborted = true;
            break;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < HS; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + 128 + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[c0 + i] = o[c0 + i] * corr + __uint_as_float(v[i]);
        }
        tc_fence_before();
    }
    if (aborted && tid == 0) {
        // let this CTA's TMA copies and MMAs in flight finish before TMEM and shared memory go
        if (q_pending) mbar_wait(bar_q, 0, nullptr, WAIT_NS / 5);
        for (int s2 = 0; s2 < 2; ++s2)
            if (kv_pending[s2]) mbar_wait(&bar_kv[s2], 0, nullptr, WAIT_NS / 5), mbar_wait(&bar_kv[s2], 1, nullptr, WAIT_NS / 5);
        umma_commit(bar_s);
        mbar_wait(bar_s, 0, nullptr, WAIT_NS / 5);
        mbar_wait(bar_s, 1, nullptr, WAIT_NS / 5);
    }
    if (aborted) {
        if (tid == 0) report(err, GK_ERR_TIMEOUT);
    } else if (qq < T) {
        const float inv = 1.f / l;
        __nv_bfloat16* yr = y + (int64_t)(row0 + qq) * C + h * HS;
#pragma unroll
        for (int d = 0; d < HS; d += 8) {
            uint4 pk;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 t2 = __floats2bfloat162_rn(o[d + 2 * e] * inv, o[d + 2 * e + 1] * inv);
                pw[e] = *reinterpret_cast<uint32_t*>(&t2);
            }
            *reinterpret_cast<uint4*>(yr + d) = pk;
        }
        lse[(int64_t)bh * T + qq] = (m + log2f(l)) * 0.6931471805599453f;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

// Returns GK_ERR_UNSUPPORTED when this kernel does not take the request (the caller then
// uses the CUDA-core kernel).
gk_status attn_fwd_tc(gk_ctx* ctx, const void* qkv, void* y, float* lse, int B, int T, int H, int hs) {
    if (hs != HS) return GK_ERR_UNSUPPORTED;
    int64_t C = (int64_t)H * hs;
    if (!aligned16(qkv) || !aligned16(y)) return GK_ERR_UNSUPPORTED;
    CUtensorMap map;
    if (!make_map(&map, qkv, 3 * C, (int64_t)B * T, 3 * C, 128)) return GK_ERR_UNSUPPORTED;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        attr = true;
    }
    dim3 grid((unsigned)cdiv(T, QT), (unsigned)(B * H));
    attn_fwd_tc_kernel<<<grid, THREADS, SMEM_BYTES, ctx->stream>>>(map, static_cast<__nv_bfloat16*>(y), lse, T, H,
                                                                 ctx->d_err);
    return launched(ctx, "attn_fwd_tc");
}

}  // namespace gk
