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
constexpr uint64_t WAIT_NS = 1000000000ull;

// Byte offset of element (row r, column c) of a [128 x 128] bf16 tile stored as two K-major
// 128-byte-swizzle halves (columns 0..63, 64..127), each 128 rows x 128 bytes.
__device__ __forceinline__ uint32_t p_offset(int r, int c) {
    int half = c >> 6, byte = (c & 63) * 2;
    int chunk = byte >> 4;
    return (uint32_t)(half * 16384 + r * 128 + (((chunk ^ (r & 7)) << 4) | (byte & 15)));
}

// Forward, two query tiles per CTA played against each other ("ping-pong"): warps 0-3 own
// query tile A, warps 4-7 tile B (the next one), warp 8 streams K/V tiles (shared by both) through
// a 2-stage ring, warp 9 issues the MMAs. While one group turns its S tile into P, the tensor
// core computes the other group's P V and its next S, so the softmax runs in the MMAs' shadow.
// TMEM: S_A 0..127, S_B 128..255, O_A 256..319, O_B 320..383.
constexpr int FWD_THREADS = 320;
constexpr size_t FWD_SMEM_BYTES = 10 * TILE + 1024 + 256;  // Q_A, Q_B, K[2], V[2], P_A, P_B

__global__ void __maxnreg__(200)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, __nv_bfloat16* __restrict__ y,
                       float* __restrict__ lse, int T, int H, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;              // [2] (A, B)
    uint8_t* sK = smem + 2 * TILE;   // [2] stages
    uint8_t* sV = smem + 4 * TILE;   // [2] stages
    uint8_t* sP = smem + 6 * TILE;   // [2] groups x two halves
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 10 * TILE);
    uint64_t* bar_q = bars;          // Q_A and Q_B landed
    uint64_t* kv_full = bars + 1;    // [2]
    uint64_t* kv_empty = bars + 3;   // [2]
    uint64_t* bar_s = bars + 5;      // [2] S_g ready
    uint64_t* bar_p = bars + 7;      // [2] P_g written (128 arrivals)
    uint64_t* bar_o = bars + 9;      // [2] O_g tile ready
    uint64_t* bar_drain = bars + 11;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = H * HS;
    const int n_qt = (T + QT - 1) / QT;
    const int pair = gridDim.x - 1 - blockIdx.x;  // heaviest pairs first
    const int qa = 2 * pair;
    const bool has_b = qa + 1 < n_qt;
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int row0 = b * T;
    const int n_kv = has_b ? qa + 2 : qa + 1;      // key tiles the CTA needs (B needs one more)

    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&bar_s[i], 1);
            mbar_init(&bar_p[i], 128);
            mbar_init(&bar_o[i], 1);
        }
        mbar_init(bar_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 9) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;

    if (warp == 8) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_qkv) : "memory");
            mbar_expect_tx(bar_q, has_b ? 2 * TILE : TILE);
            tma_load_2d(&tm_qkv, bar_q, sQ, h * HS, row0 + qa * QT);
            if (has_b) tma_load_2d(&tm_qkv, bar_q, sQ + TILE, h * HS, row0 + (qa + 1) * QT);
            int last_ph[2] = {-1, -1};
            for (int j = 0; j < n_kv; ++j) {
                int st = j & 1;
                uint32_t ph = (j >> 1) & 1;
                if (!mbar_wait(&kv_empty[st], ph ^ 1, nullptr, WAIT_NS)) {
                    failed = true;
                    break;
                }
                mbar_expect_tx(&kv_full[st], 2 * TILE);
                tma_load_2d(&tm_qkv, &kv_full[st], sK + st * TILE, C + h * HS, row0 + j * KT);
                tma_load_2d(&tm_qkv, &kv_full[st], sV + st * TILE, 2 * C + h * HS, row0 + j * KT);
                last_ph[st] = (int)ph;
            }
            if (failed) {
                // let this CTA's copies in flight land before shared memory is released
                mbar_wait(bar_q, 0, nullptr, WAIT_NS / 5);
                for (int st = 0; st < 2; ++st)
                    if (last_ph[st] >= 0) mbar_wait(&kv_full[st], (uint32_t)last_ph[st], nullptr, WAIT_NS / 5);
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            const uint32_t id_s = instr_desc_bf16(false, false, 128, 128);
            const uint32_t id_o = instr_desc_bf16(false, true, 128, 64);
            const int nA = qa + 1, nB = has_b ? qa + 2 : 0;
            bool issued = false;
            bool ok = mbar_wait(bar_q, 0, nullptr, WAIT_NS) && mbar_wait(&kv_full[0], 0, nullptr, WAIT_NS);
            if (ok) {
                tc_fence_after();
                for (int g = 0; g < (has_b ? 2 : 1); ++g) {
                    uint32_t q_a = saddr(sQ + g * TILE), k_a = saddr(sK);
#pragma unroll
                    for (int k = 0; k < HS / 16; ++k)
                        umma_bf16(tmem + g * 128, smem_desc(q_a + k * 32, 16, 1024), smem_desc(k_a + k * 32, 16, 1024),
                                  id_s, k > 0);
                    umma_commit(&bar_s[g]);
                }
                issued = true;
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                for (int g = 0; g < 2 && ok; ++g) {
                    const int ng = g ? nB : nA;
                    if (j >= ng) continue;
                    ok = mbar_wait(&bar_p[g], j & 1, nullptr, WAIT_NS);
                    if (!ok) break;
                    tc_fence_after();
                    // O_g(j) = P_g V_j
                    uint32_t p_a = saddr(sP + g * 2 * TILE), v_a = saddr(sV + (j & 1) * TILE);
#pragma unroll
                    for (int k = 0; k < KT / 16; ++k)
                        umma_bf16(tmem + 256 + g * 64, smem_desc(p_a + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                                  smem_desc(v_a + k * 2048, 8192, 1024), id_o, k > 0);
                    umma_commit(&bar_o[g]);
                    // the last reader of K/V stage j frees it for the tile j + 2
                    if (g == 1 || j >= nB) umma_commit(&kv_empty[j & 1]);
                    // S_g(j + 1), once K_{j+1} has landed
                    if (j + 1 < ng) {
                        if (g == 0 || j + 1 >= nA) {
                            ok = mbar_wait(&kv_full[(j + 1) & 1], ((j + 1) >> 1) & 1, nullptr, WAIT_NS);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        uint32_t q_a = saddr(sQ + g * TILE), k_a = saddr(sK + ((j + 1) & 1) * TILE);
#pragma unroll
                        for (int k = 0; k < HS / 16; ++k)
                            umma_bf16(tmem + g * 128, smem_desc(q_a + k * 32, 16, 1024),
                                      smem_desc(k_a + k * 32, 16, 1024), id_s, k > 0);
                        umma_commit(&bar_s[g]);
                    }
                }
            }
            if (!ok) {
                failed = true;
                if (issued) {
                    umma_commit(bar_drain);
                    mbar_wait(bar_drain, 0, nullptr, WAIT_NS / 5);
                }
            }
        }
    } else {
        const int g = warp >> 2;          // group: 0 = tile A, 1 = tile B
        const int r = (warp & 3) * 32 + lane;
        const int q0 = (qa + g) * QT;
        const int qq = q0 + r;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
        uint8_t* myP = sP + g * 2 * TILE;
        float o[HS];
#pragma unroll
        for (int d = 0; d < HS; ++d) o[d] = 0.f;
        float m = -INFINITY, l = 0.f;
        const int my_kt = g ? (has_b ? qa + 2 : 0) : qa + 1;
        for (int j = 0; j < my_kt; ++j) {
            if (!mbar_wait(&bar_s[g], j & 1, nullptr, WAIT_NS)) {
                failed = true;
                break;
            }
            tc_fence_after();
            const int k0 = j * KT;
            float tmax = -INFINITY;
#pragma unroll 1
            for (int c0 = 0; c0 < KT; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_addr + g * 128 + c0, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    int kk = k0 + c0 + i;
                    float t = __uint_as_float(v[i]) * sl2;
                    if (kk <= qq && kk < T) tmax = fmaxf(tmax, t);
                }
            }
            const float m_new = fmaxf(m, tmax);
            const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m - m_new);
            float psum = 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < KT; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_addr + g * 128 + c0, v);
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
                    *reinterpret_cast<uint4*>(myP + p_offset(r, c0 + i)) = pk;
                }
            }
            l = l * corr + psum;
            m = m_new;
            fence_proxy_async_smem();  // P's generic-proxy stores -> visible to the tensor core
            tc_fence_before();
            mbar_arrive(&bar_p[g]);
            if (!mbar_wait(&bar_o[g], j & 1, nullptr, WAIT_NS)) {
                failed = true;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < HS; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_addr + 256 + g * 64 + c0, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[c0 + i] = o[c0 + i] * corr + __uint_as_float(v[i]);
            }
            tc_fence_before();
        }
        if (!failed && my_kt > 0 && qq < T) {
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
    }
    if (failed) report(err, GK_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------ backward
// One CTA of 128 threads per (128-key tile, batch, head), looping over the query tiles at or
// after its keys. Thread r owns key row r for S^T, dP^T, dV and dK, and query row r for the
// per-tile dQ. Per query tile:
//   S^T = K Q^T, dP^T = V dO^T      (M=128 keys, N=128 queries, K=64)        -> TMEM 0..255
//   P^T = exp(S^T / sqrt(hs) - lse), dS^T = P^T (dP^T - D)  as bf16 into shared memory
//   dV += P^T dO, dK += dS^T Q       (M=128 keys, N=64, K=128 queries)       -> TMEM 256..383
//   dQ_tile = dS K                   (M=128 queries, N=64, K=128 keys)       -> TMEM 384..447
// dQ_tile is added (float atomics) into a float32 accumulator; dK and dV are stored once.
constexpr size_t BWD_SMEM_BYTES = 10 * TILE + 2048 + 1024 + 128;  // K, V, Q[2], dO[2], P^T, dS^T, lse/D

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_dy,
                       const float* __restrict__ lse, const float* __restrict__ dvec, __nv_bfloat16* __restrict__ dqkv,
                       float* __restrict__ dq_acc, int T, int H, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem;
    uint8_t* sV = smem + TILE;
    uint8_t* sQ = smem + 2 * TILE;    // two stages
    uint8_t* sO = smem + 4 * TILE;    // dO, two stages
    uint8_t* sPT = smem + 6 * TILE;   // two halves
    uint8_t* sDS = smem + 8 * TILE;   // two halves
    float* sL = reinterpret_cast<float*>(smem + 10 * TILE);
    float* sD = sL + 128;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 10 * TILE + 2048);
    uint64_t* bar_kv = bars;
    uint64_t* bar_qo = bars + 1;      // [2]
    uint64_t* bar_1 = bars + 3;
    uint64_t* bar_2 = bars + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 5);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int C = H * HS;
    const int kt = blockIdx.x;  // heaviest (earliest keys) first
    const int k0 = kt * KT;
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int row0 = b * T;
    const int n_qt = (T + QT - 1) / QT;
    const int first_qt = k0 / QT;

    if (tid == 0) {
        mbar_init(bar_kv, 1);
        mbar_init(&bar_qo[0], 1);
        mbar_init(&bar_qo[1], 1);
        mbar_init(bar_1, 1);
        mbar_init(bar_2, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int pending_qo[2] = {0, 0}, pending_kv = 0;
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_qkv) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_dy) : "memory");
        mbar_expect_tx(bar_kv, 2 * TILE);
        tma_load_2d(&tm_qkv, bar_kv, sK, C + h * HS, row0 + k0);
        tma_load_2d(&tm_qkv, bar_kv, sV, 2 * C + h * HS, row0 + k0);
        pending_kv = 1;
        if (first_qt < n_qt) {
            mbar_expect_tx(&bar_qo[0], 2 * TILE);
            tma_load_2d(&tm_qkv, &bar_qo[0], sQ, h * HS, row0 + first_qt * QT);
            tma_load_2d(&tm_dy, &bar_qo[0], sO, h * HS, row0 + first_qt * QT);
            pending_qo[0] = 1;
        }
    }
    const uint32_t id_s = instr_desc_bf16(false, false, 128, 128);  // S^T, dP^T
    const uint32_t id_kv = instr_desc_bf16(false, true, 128, 64);   // dV, dK: B (dO, Q) MN-major
    const uint32_t id_q = instr_desc_bf16(true, true, 128, 64);     // dQ: A (dS) and B (K) MN-major
    const float sl2 = 0.125f * 1.4426950408889634f;
    const float L2E = 1.4426950408889634f;
    const int r = warp * 32 + (tid & 31);
    const int kk = k0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    bool aborted = false;

    // prologue: S^T and dP^T of the first query tile
    bool fail0 = false;
    if (tid == 0) {
        bool w = mbar_wait(bar_kv, 0, nullptr, WAIT_NS) && mbar_wait(&bar_qo[0], 0, nullptr, WAIT_NS);
        if (w) {
            pending_kv = 0;
            pending_qo[0] = 0;
            tc_fence_after();
            uint32_t k_a = saddr(sK), v_a = saddr(sV), q_a = saddr(sQ), o_a = saddr(sO);
#pragma unroll
            for (int k = 0; k < HS / 16; ++k)
                umma_bf16(tmem, smem_desc(k_a + k * 32, 16, 1024), smem_desc(q_a + k * 32, 16, 1024), id_s, k > 0);
#pragma unroll
            for (int k = 0; k < HS / 16; ++k)
                umma_bf16(tmem + 128, smem_desc(v_a + k * 32, 16, 1024), smem_desc(o_a + k * 32, 16, 1024), id_s,
                          k > 0);
            umma_commit(bar_1);
            if (first_qt + 1 < n_qt) {
                mbar_expect_tx(&bar_qo[1], 2 * TILE);
                tma_load_2d(&tm_qkv, &bar_qo[1], sQ + TILE, h * HS, row0 + (first_qt + 1) * QT);
                tma_load_2d(&tm_dy, &bar_qo[1], sO + TILE, h * HS, row0 + (first_qt + 1) * QT);
                pending_qo[1] = 1;
            }
        }
        fail0 = !w;
    }
    if (__syncthreads_or(fail0)) aborted = true;

    for (int qt = first_qt; !aborted && qt < n_qt; ++qt) {
        const int it = qt - first_qt;
        const int st = it & 1;
        const uint32_t ph = it & 1;
        const int q0 = qt * QT;
        {
            int q = q0 + r;
            sL[r] = q < T ? lse[(int64_t)bh * T + q] * L2E : 0.f;
            sD[r] = q < T ? dvec[(int64_t)bh * T + q] : 0.f;
        }
        // (the barrier below also orders these shared-memory writes before their use)
        if (__syncthreads_or(!mbar_wait(bar_1, ph, nullptr, WAIT_NS))) {
            aborted = true;
            break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < QT; c0 += 32) {
            uint32_t sv[32], dv[32];
            tmem_ld32(lane_addr + c0, sv);
            tmem_ld32(lane_addr + 128 + c0, dv);
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                float pv[8], dsv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    int c = c0 + i + e, q = q0 + c;
                    bool vis = q >= kk && q < T && kk < T;
                    float pp = vis ? exp2f(__uint_as_float(sv[i + e]) * sl2 - sL[c]) : 0.f;
                    pv[e] = pp;
                    dsv[e] = pp * (__uint_as_float(dv[i + e]) - sD[c]);
                }
                uint4 pk, dk;
                uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
                uint32_t* dw = reinterpret_cast<uint32_t*>(&dk);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __nv_bfloat162 t2 = __floats2bfloat162_rn(pv[2 * e], pv[2 * e + 1]);
                    __nv_bfloat162 u2 = __floats2bfloat162_rn(dsv[2 * e], dsv[2 * e + 1]);
                    pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                    dw[e] = *reinterpret_cast<uint32_t*>(&u2);
                }
                *reinterpret_cast<uint4*>(sPT + p_offset(r, c0 + i)) = pk;
                *reinterpret_cast<uint4*>(sDS + p_offset(r, c0 + i)) = dk;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        bool fail = false;
        if (tid == 0) {
            tc_fence_after();
            uint32_t pt_a = saddr(sPT), ds_a = saddr(sDS), k_a = saddr(sK), v_a = saddr(sV);
            uint32_t q_a = saddr(sQ + st * TILE), o_a = saddr(sO + st * TILE);
#pragma unroll
            for (int k = 0; k < QT / 16; ++k) {
                uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
                umma_bf16(tmem + 256, smem_desc(pt_a + koff, 16, 1024), smem_desc(o_a + k * 2048, 8192, 1024), id_kv,
                          (it > 0 || k > 0));
                umma_bf16(tmem + 320, smem_desc(ds_a + koff, 16, 1024), smem_desc(q_a + k * 2048, 8192, 1024), id_kv,
                          (it > 0 || k > 0));
            }
#pragma unroll
            for (int k = 0; k < KT / 16; ++k)
                umma_bf16(tmem + 384, smem_desc(ds_a + k * 2048, 16384, 1024), smem_desc(k_a + k * 2048, 8192, 1024),
                          id_q, k > 0);
            umma_commit(bar_2);
            // S^T and dP^T of the next query tile right behind: they overlap the dQ accumulation
            if (qt + 1 < n_qt) {
                int ns = st ^ 1;
                bool w = mbar_wait(&bar_qo[ns], ((it + 1) >> 1) & 1, nullptr, WAIT_NS);
                if (w) {
                    pending_qo[ns] = 0;
                    tc_fence_after();
                    uint32_t nq_a = saddr(sQ + ns * TILE), no_a = saddr(sO + ns * TILE);
#pragma unroll
                    for (int k = 0; k < HS / 16; ++k)
                        umma_bf16(tmem, smem_desc(k_a + k * 32, 16, 1024), smem_desc(nq_a + k * 32, 16, 1024), id_s,
                                  k > 0);
#pragma unroll
                    for (int k = 0; k < HS / 16; ++k)
                        umma_bf16(tmem + 128, smem_desc(v_a + k * 32, 16, 1024), smem_desc(no_a + k * 32, 16, 1024),
                                  id_s, k > 0);
                    umma_commit(bar_1);
                }
                fail = !w;
            }
        }
        if (__syncthreads_or(fail || !mbar_wait(bar_2, ph, nullptr, WAIT_NS))) {
            aborted = true;
            break;
        }
        tc_fence_after();
        // stage st (Q, dO of this tile) is free now: prefetch the tile after next into it
        if (tid == 0 && qt + 2 < n_qt) {
            mbar_expect_tx(&bar_qo[st], 2 * TILE);
            tma_load_2d(&tm_qkv, &bar_qo[st], sQ + st * TILE, h * HS, row0 + (qt + 2) * QT);
            tma_load_2d(&tm_dy, &bar_qo[st], sO + st * TILE, h * HS, row0 + (qt + 2) * QT);
            pending_qo[st] = 1;
        }
        {
            int q = q0 + r;
#pragma unroll
            for (int c0 = 0; c0 < HS; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_addr + 384 + c0, v);
                if (q < T) {
                    float* dst = dq_acc + (int64_t)(row0 + q) * C + h * HS + c0;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        atomicAdd(reinterpret_cast<float4*>(dst + i),
                                  make_float4(__uint_as_float(v[i]) * 0.125f, __uint_as_float(v[i + 1]) * 0.125f,
                                              __uint_as_float(v[i + 2]) * 0.125f, __uint_as_float(v[i + 3]) * 0.125f));
                }
            }
        }
        tc_fence_before();
    }
    if (aborted) {
        if (tid == 0) {
            report(err, GK_ERR_TIMEOUT);
            if (pending_kv) mbar_wait(bar_kv, 0, nullptr, WAIT_NS / 5);
            for (int s2 = 0; s2 < 2; ++s2)
                if (pending_qo[s2]) mbar_wait(&bar_qo[s2], 0, nullptr, WAIT_NS / 5), mbar_wait(&bar_qo[s2], 1, nullptr, WAIT_NS / 5);
            umma_commit(bar_1);
            mbar_wait(bar_1, 0, nullptr, WAIT_NS / 5);
            mbar_wait(bar_1, 1, nullptr, WAIT_NS / 5);
        }
    } else if (first_qt < n_qt) {
        uint32_t v[32];
        __nv_bfloat16* base = dqkv + (int64_t)(row0 + kk) * 3 * C + h * HS;
#pragma unroll
        for (int c0 = 0; c0 < HS; c0 += 32) {
            tmem_ld32(lane_addr + 256 + c0, v);   // dV
            if (kk < T) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 pk;
                    uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 t2 = __floats2bfloat162_rn(__uint_as_float(v[i + 2 * e]), __uint_as_float(v[i + 2 * e + 1]));
                        pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                    }
                    *reinterpret_cast<uint4*>(base + 2 * C + c0 + i) = pk;
                }
            }
            tmem_ld32(lane_addr + 320 + c0, v);   // dK (times 1/sqrt(hs))
            if (kk < T) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 pk;
                    uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 t2 = __floats2bfloat162_rn(__uint_as_float(v[i + 2 * e]) * 0.125f,
                                                                  __uint_as_float(v[i + 2 * e + 1]) * 0.125f);
                        pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                    }
                    *reinterpret_cast<uint4*>(base + C + c0 + i) = pk;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// D[b,h,t] = sum_d dy * y over one head's 64 columns (one warp per (row, head)); also zeroes
// that head's slice of the float32 dQ accumulator.
__global__ void attn_dvec_zero_kernel(const __nv_bfloat16* __restrict__ y, const __nv_bfloat16* __restrict__ dy,
                                      float* __restrict__ dvec, float* __restrict__ dq_acc, int64_t rows, int T, int H) {
    int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (wid >= rows * H) return;
    int64_t r = wid / H;
    int h = (int)(wid % H);
    int64_t C = (int64_t)H * HS;
    int64_t off = r * C + h * HS + lane * 2;
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(dy + off);
    __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(y + off);
    float s = __bfloat162float(a.x) * __bfloat162float(c.x) + __bfloat162float(a.y) * __bfloat162float(c.y);
    s = warp_sum(s);
    *reinterpret_cast<float2*>(dq_acc + off) = make_float2(0.f, 0.f);
    if (lane == 0) dvec[((r / T) * H + h) * T + (r % T)] = s;
}

// dqkv[:, 0:C] (bf16) = dq_acc (float32)
__global__ void attn_dq_store_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dqkv, int64_t rows,
                                     int C) {
    int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= rows * C) return;
    int64_t r = i / C, c = i % C;
    float4 v = *reinterpret_cast<const float4*>(dq_acc + i);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dqkv + r * 3 * C + c) = pk;
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
        cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FWD_SMEM_BYTES);
        attr = true;
    }
    dim3 grid((unsigned)cdiv(cdiv(T, QT), 2), (unsigned)(B * H));
    attn_fwd_tc_kernel<<<grid, FWD_THREADS, FWD_SMEM_BYTES, ctx->stream>>>(map, static_cast<__nv_bfloat16*>(y), lse,
                                                                         T, H, ctx->d_err);
    return launched(ctx, "attn_fwd_tc");
}

}  // namespace gk

namespace gk {

gk_status attn_bwd_tc(gk_ctx* ctx, const void* qkv, const void* y, const float* lse, const void* dy, void* dqkv,
                      int B, int T, int H, int hs) {
    if (hs != HS) return GK_ERR_UNSUPPORTED;
    int64_t C = (int64_t)H * hs, rows = (int64_t)B * T;
    if (!aligned16(qkv) || !aligned16(dy) || !aligned16(dqkv) || !aligned16(y)) return GK_ERR_UNSUPPORTED;
    size_t dvec_bytes = ((size_t)B * H * T * sizeof(float) + 255) & ~size_t(255);
    size_t need = dvec_bytes + (size_t)rows * C * sizeof(float);
    char* ws = (char*)workspace(ctx, need);
    GK_REQUIRE(ctx, ws, GK_ERR_WORKSPACE, "gk_attn_bwd: needs %zu workspace bytes", need);
    float* dvec = (float*)ws;
    float* dq_acc = (float*)(ws + dvec_bytes);
    CUtensorMap map_qkv, map_dy;
    if (!make_map(&map_qkv, qkv, 3 * C, rows, 3 * C, 128) || !make_map(&map_dy, dy, C, rows, C, 128))
        return GK_ERR_UNSUPPORTED;
    attn_dvec_zero_kernel<<<(unsigned)cdiv(rows * H * 32, 256), 256, 0, ctx->stream>>>(
        (const __nv_bfloat16*)y, (const __nv_bfloat16*)dy, dvec, dq_acc, rows, T, H);
    GK_TRY(launched(ctx, "attn_dvec_zero"));
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BWD_SMEM_BYTES);
        attr = true;
    }
    dim3 grid((unsigned)cdiv(T, KT), (unsigned)(B * H));
    attn_bwd_tc_kernel<<<grid, THREADS, BWD_SMEM_BYTES, ctx->stream>>>(map_qkv, map_dy, lse, dvec,
                                                                    (__nv_bfloat16*)dqkv, dq_acc, T, H, ctx->d_err);
    GK_TRY(launched(ctx, "attn_bwd_tc"));
    attn_dq_store_kernel<<<(unsigned)cdiv(rows * C / 4, 256), 256, 0, ctx->stream>>>(dq_acc, (__nv_bfloat16*)dqkv,
                                                                                    rows, (int)C);
    return launched(ctx, "attn_dq_store");
}

}  // namespace gk
