// Causal attention forward on the tensor cores (tcgen05), head size 64, bf16 q/k/v.
// [LM1] = "Build a language model in C# from scratch (1)", op table (BatchMatMulT,
// CausalSoftmax, BatchMatMul); [LM4] = "... (4): running GPT-2 weights", "The 12 tensors we do
// not use" (the causal mask by arithmetic) and "Generation with a KV cache" (1/sqrt(hs)).
//
// Forward: two 128-query tiles per CTA; K and V tiles of 128 keys stream through a double
// buffer. For each key tile and query tile:
//   S = Q K^T        tcgen05 MMA chain (M=128, N=128, K=64) into TMEM;
//   softmax          each thread owns one query row: one read of its 128 S values from TMEM,
//                    the causal mask on the diagonal tile only, P = 2^(S/sqrt(hs)*log2(e) - m)
//                    as bf16 into shared memory in the 128-byte-swizzled K-major layout the MMA
//                    reads; m moves only when the row maximum exceeds it by more than 8 (then O
//                    is rescaled in TMEM), so P <= 2^8;
//   O += P V         second MMA chain (M=128, N=64, K=128; V is the MN-major operand)
//                    accumulating in TMEM across key tiles.
// The result is O / l (bf16) and the row log-sum-exp (float32, natural log) for backward.
// All mbarrier waits are bounded (timeout -> GK_ERR_TIMEOUT in the error word).
#include <math.h>

#include <algorithm>

#include "tcgen05.cuh"

namespace gk {
namespace {

using namespace tc;

constexpr int QT = 128, KT = 128, HS = 64;
constexpr uint32_t TILE = 128 * 64 * 2;                 // one 128 x 64 bf16 tile, 16 KB
constexpr uint64_t WAIT_NS = 1000000000ull;

// One of two descriptors (kept in registers: an indexed array would live in local memory).
__device__ __forceinline__ uint64_t pick(uint64_t d0, uint64_t d1, int i) { return i ? d1 : d0; }

// Byte offset of element (row r, column c) of a [128 x 128] bf16 tile stored as two K-major
// 128-byte-swizzle halves (columns 0..63, 64..127), each 128 rows x 128 bytes.
__device__ __forceinline__ uint32_t p_offset(int r, int c) {
    int half = c >> 6, byte = (c & 63) * 2;
    int chunk = byte >> 4;
    return (uint32_t)(half * 16384 + r * 128 + (((chunk ^ (r & 7)) << 4) | (byte & 15)));
}

// Forward, two query tiles per work item played against each other ("ping-pong"): warps 0-3
// own query tile A, warps 4-7 tile B (the next one), warp 8 streams Q and the K/V tiles (shared
// by both) through shared memory, warp 9 issues the MMAs. While one group turns its S tile into
// P, the tensor core computes the other group's P V and its next S, so the softmax runs in the
// MMAs' shadow. The MMA warp issues S_g(j+1) after P_g V_j, so S_g(j+1) landing also means O_g
// and P_g are free again. TMEM: S_A 0..127, S_B 128..255, O_A 256..319, O_B 320..383.
//
// The kernel is persistent: one CTA per SM walks a list of work items (batch x head, pair of
// query tiles), so the tensor memory, the barriers and the pipeline are set up once, and the
// next item's Q and K/V tiles load while the current one finishes (Q is double-buffered: the
// items alternate between two Q sets; the K/V ring runs on across items). The items are ordered
// heaviest first (the last query tiles see the most keys) and dealt to the CTAs in snake order
// (round r: CTA c takes item r G + c for even r, r G + G - 1 - c for odd r), which evens out the
// CTAs' total work. Every role walks the same item sequence and keeps its barrier phases running
// across items.
// Registers are granted to a block in groups of four warps, so 9- or 10-warp blocks are
// budgeted as 12 warps: 168 registers per thread at most (hence __maxnreg__(168)).
constexpr int FWD_THREADS = 320;
constexpr size_t FWD_SMEM_BYTES = 8 * TILE + 1024 + 256;  // Q[2 sets][A, B], K[2], V[2]

// The r-th work item of this CTA, or -1 when it has no more: item k runs query-tile pair
// n_pairs - 1 - k / BH of (batch x head) k % BH.
__device__ __forceinline__ int fwd_item(int r, int n_items) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    const int k = r * G + ((r & 1) ? G - 1 - c : c);
    return k < n_items ? k : -1;
}

__global__ void __maxnreg__(168)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, __nv_bfloat16* __restrict__ y,
                       float* __restrict__ lse, int T, int H, int BH, int n_items, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;              // [2 sets][A, B]
    uint8_t* sK = smem + 4 * TILE;   // [2] stages
    uint8_t* sV = smem + 6 * TILE;   // [2] stages
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 8 * TILE);
    uint64_t* bar_q = bars;          // [2] Q set landed
    uint64_t* q_empty = bars + 2;    // [2] Q set free again (the item's MMAs are done)
    uint64_t* kv_full = bars + 4;    // [2]
    uint64_t* kv_empty = bars + 6;   // [2]
    uint64_t* bar_s = bars + 8;      // [2] S_g ready
    uint64_t* bar_p = bars + 10;     // [2] P_g written (128 arrivals)
    uint64_t* bar_o = bars + 12;     // [2] O_g tile ready
    uint64_t* bar_drain = bars + 14;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = H * HS;
    const int n_qt = (T + QT - 1) / QT;
    const int n_pairs = (n_qt + 1) / 2;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_q[i], 1);
            mbar_init(&q_empty[i], 1);
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
            int kvj = 0;  // K/V tiles issued so far (all items)
            int last_kv[2] = {-1, -1}, last_q[2] = {-1, -1};
            for (int r = 0, it = 0;; ++r, ++it) {
                const int k = fwd_item(r, n_items);
                if (k < 0) break;
                const int qa = 2 * (n_pairs - 1 - k / BH), bh = k % BH;
                const bool has_b = qa + 1 < n_qt;
                const int h = bh % H, row0 = (bh / H) * T;
                const int n_kv = has_b ? qa + 2 : qa + 1;
                const int qs = it & 1;
                if (it >= 2 && !mbar_wait(&q_empty[qs], ((it >> 1) - 1) & 1, nullptr, WAIT_NS)) {
                    failed = true;
                    break;
                }
                mbar_expect_tx(&bar_q[qs], has_b ? 2 * TILE : TILE);
                tma_load_2d(&tm_qkv, &bar_q[qs], sQ + 2 * qs * TILE, h * HS, row0 + qa * QT);
                if (has_b) tma_load_2d(&tm_qkv, &bar_q[qs], sQ + (2 * qs + 1) * TILE, h * HS, row0 + (qa + 1) * QT);
                last_q[qs] = (it >> 1) & 1;
                for (int j = 0; j < n_kv && !failed; ++j, ++kvj) {
                    const int st = kvj & 1;
                    const uint32_t ph = (kvj >> 1) & 1;
                    if (!mbar_wait(&kv_empty[st], ph ^ 1, nullptr, WAIT_NS)) {
                        failed = true;
                        break;
                    }
                    mbar_expect_tx(&kv_full[st], 2 * TILE);
                    tma_load_2d(&tm_qkv, &kv_full[st], sK + st * TILE, C + h * HS, row0 + j * KT);
                    tma_load_2d(&tm_qkv, &kv_full[st], sV + st * TILE, 2 * C + h * HS, row0 + j * KT);
                    last_kv[st] = (int)ph;
                }
                if (failed) break;
            }
            if (failed) {
                // let this CTA's copies in flight land before shared memory is released
                for (int i = 0; i < 2; ++i) {
                    if (last_q[i] >= 0) mbar_wait(&bar_q[i], (uint32_t)last_q[i], nullptr, WAIT_NS / 5);
                    if (last_kv[i] >= 0) mbar_wait(&kv_full[i], (uint32_t)last_kv[i], nullptr, WAIT_NS / 5);
                }
            }
        }
    } else if (warp == 9) {
        // The whole warp walks the schedule (warp-uniform descriptors); one elected lane
        // issues each group of MMAs together with the commits that track them.
        const uint32_t id_s = instr_desc_bf16(false, false, 128, 128);
        const uint32_t id_o = instr_desc_bf16(false, true, 128, 64);
        const uint64_t k_d0 = smem_desc(saddr(sK), 16, 1024), k_d1 = smem_desc(saddr(sK + TILE), 16, 1024);
        const uint64_t v_d0 = smem_desc(saddr(sV), 8192, 1024), v_d1 = smem_desc(saddr(sV + TILE), 8192, 1024);
        bool issued = false, ok = true;
        int kvj = 0, pc[2] = {0, 0}, it = 0;
        for (int r = 0; ok; ++r, ++it) {
            const int k = fwd_item(r, n_items);
            if (k < 0) break;
            const int qa = 2 * (n_pairs - 1 - k / BH);
            const bool has_b = qa + 1 < n_qt;
            const int nA = qa + 1, nB = has_b ? qa + 2 : 0, n_kv = has_b ? qa + 2 : qa + 1;
            const int qs = it & 1;
            const uint64_t q_d0 = smem_desc(saddr(sQ + 2 * qs * TILE), 16, 1024);
            const uint64_t q_d1 = smem_desc(saddr(sQ + (2 * qs + 1) * TILE), 16, 1024);
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_q[qs], (it >> 1) & 1, nullptr, WAIT_NS) &&
                                             mbar_wait(&kv_full[kvj & 1], (kvj >> 1) & 1, nullptr, WAIT_NS));
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                for (int g = 0; g < (has_b ? 2 : 1); ++g) {
#pragma unroll
                    for (int kk = 0; kk < HS / 16; ++kk)
                        umma_bf16(tmem + g * 128, desc_add(pick(q_d0, q_d1, g), kk * 32),
                                  desc_add(pick(k_d0, k_d1, kvj & 1), kk * 32), id_s, kk > 0);
                    umma_commit(&bar_s[g]);
                }
            }
            __syncwarp();
            issued = true;
            for (int j = 0; ok && j < n_kv; ++j) {
                const int sj = (kvj + j) & 1, sn = (kvj + j + 1) & 1;
                for (int g = 0; g < 2 && ok; ++g) {
                    const int ng = g ? nB : nA;
                    if (j >= ng) continue;
                    ok = __all_sync(0xffffffffu, mbar_wait(&bar_p[g], pc[g] & 1, nullptr, WAIT_NS));
                    if (!ok) break;
                    ++pc[g];
                    tc_fence_after();
                    // O_g(j) = P_g V_j, P_g read from TMEM (bf16 pairs over S_g's first 64 columns)
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < KT / 16; ++kk)
                            umma_bf16_ts(tmem + 256 + g * 64, tmem + g * 128 + kk * 8,
                                         desc_add(pick(v_d0, v_d1, sj), kk * 2048), id_o, (j > 0 || kk > 0) ? 1u : 0u);
                        if (j == ng - 1) umma_commit(&bar_o[g]);
                        // the last reader of K/V stage j frees it for the tile two ahead
                        if (g == 1 || j >= nB) umma_commit(&kv_empty[sj]);
                    }
                    __syncwarp();
                    // S_g(j + 1), once K_{j+1} has landed
                    if (j + 1 < ng) {
                        if (g == 0 || j + 1 >= nA) {
                            ok = __all_sync(0xffffffffu,
                                            mbar_wait(&kv_full[sn], ((kvj + j + 1) >> 1) & 1, nullptr, WAIT_NS));
                            if (!ok) break;
                            tc_fence_after();
                        }
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < HS / 16; ++kk)
                                umma_bf16(tmem + g * 128, desc_add(pick(q_d0, q_d1, g), kk * 32),
                                          desc_add(pick(k_d0, k_d1, sn), kk * 32), id_s, kk > 0);
                            umma_commit(&bar_s[g]);
                        }
                        __syncwarp();
                    }
                }
            }
            if (!ok) break;
            // every MMA of the item that reads this Q set has been issued
            if (elect_one()) umma_commit(&q_empty[qs]);
            __syncwarp();
            kvj += n_kv;
        }
        // the last item's MMAs (and the commits tracking them) complete before the CTA exits
        if (ok && it > 0) ok = __all_sync(0xffffffffu, mbar_wait(&q_empty[(it - 1) & 1], ((it - 1) >> 1) & 1, nullptr, WAIT_NS));
        if (!ok) {
            failed = true;
            if (issued) {
                if (elect_one()) {
                    umma_commit(bar_drain);
                    mbar_wait(bar_drain, 0, nullptr, WAIT_NS / 5);
                }
                __syncwarp();
            }
        }
    } else {
        // softmax warps: thread r of group g owns query row q0 + r of each item
        const int g = warp >> 2;          // group: 0 = tile A, 1 = tile B
        const int rr = (warp & 3) * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t o_addr = lane_addr + 256 + g * 64;
        const float sl2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
        int sc = 0, oc = 0;  // S_g tiles and O_g results waited for so far
        for (int r = 0; !failed; ++r) {
            const int k = fwd_item(r, n_items);
            if (k < 0) break;
            const int qa = 2 * (n_pairs - 1 - k / BH), bh = k % BH;
            const bool has_b = qa + 1 < n_qt;
            const int h = bh % H, row0 = (bh / H) * T;
            const int q0 = (qa + g) * QT;
            const int qq = q0 + rr;
            const int my_kt = g ? (has_b ? qa + 2 : 0) : qa + 1;
            if (my_kt == 0) continue;
            // m_ref: the reference the row's P and running sum l are taken against, in log2
            // units; it moves (and O in TMEM is rescaled) only when the row maximum exceeds it
            // by more than 8, so P <= 2^8 and most key tiles skip the rescale.
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < my_kt; ++j) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_s[g], sc & 1, nullptr, WAIT_NS))) {
                    failed = true;
                    break;
                }
                ++sc;
                tc_fence_after();
                // S row (128 keys) in one go; S_g(j) complete also means P_g V_{j-1} is complete
                uint32_t sv[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32_nowait(lane_addr + g * 128 + c * 32, sv[c]);
                tmem_wait_ld_only();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence32(sv[c]);
                // keys k0 + i, i < lim, are visible to this row (causal; the diagonal tile only)
                const int k0 = j * KT;
                const bool diag = j == qa + g;
                const int lim = diag ? min(qq, T - 1) - k0 + 1 : KT;
                if (diag) {  // hidden keys -> -inf, so their P is exactly 0 below
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c * 32 + i >= lim) sv[c][i] = 0xff800000u;
                }
                float mx[8];  // eight independent partial maxima instead of one 128-long chain
#pragma unroll
                for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(sv[0][e]);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(sv[c][i]));
                const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                const float m_new = fmaxf(m_ref, mt * sl2);
                // move the reference (O is rescaled after P is written, when the S row is dead)
                float corr = 1.f;
                const bool rescale = m_new > m_ref + 8.f;
                if (rescale) {
                    corr = ex2_hw(m_ref - m_new);  // 0 while the row was empty
                    l *= corr;
                    m_ref = m_new;
                }
                // P = 2^(S * sl2 - m_ref) as bf16 pairs into TMEM over S_g's first 64 columns
                // (this thread's row, already read), where the P V product takes its A operand
                float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float p0 = ex2_hw(fmaf(__uint_as_float(sv[c][2 * e]), sl2, -m_ref));
                        float p1 = ex2_hw(fmaf(__uint_as_float(sv[c][2 * e + 1]), sl2, -m_ref));
                        ps[(2 * e) & 7] += p0;
                        ps[(2 * e + 1) & 7] += p1;
                        __nv_bfloat162 t2 = __floats2bfloat162_rn(p0, p1);
                        pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                    }
                    tmem_st16(lane_addr + g * 128 + c * 16, pw);
                }
                l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                // tcgen05.ld / st are warp-collective: the warp rescales if any of its rows must
                // (corr = 1 for the others)
                if (j > 0 && __any_sync(0xffffffffu, rescale)) {  // O row, two 32-column halves
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t ov[32];
                        tmem_ld32_nowait(o_addr + c * 32, ov);
                        tmem_wait_ld_only();
                        reg_fence32(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * corr);
                        tmem_st32(o_addr + c * 32, ov);
                    }
                }
                tmem_wait_st();  // P (and a rescaled O) in TMEM before the MMA warp is told
                tc_fence_before();
                mbar_arrive(&bar_p[g]);
            }
            if (failed) break;
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_o[g], oc & 1, nullptr, WAIT_NS))) {
                failed = true;
                break;
            }
            ++oc;
            tc_fence_after();
            uint32_t ov[2][32];
            tmem_ld32_nowait(o_addr, ov[0]);
            tmem_ld32_nowait(o_addr + 32, ov[1]);
            tmem_wait_ld_only();
            reg_fence32(ov[0]);
            reg_fence32(ov[1]);
            if (qq < T) {
                const float inv = 1.f / l;
                __nv_bfloat16* yr = y + (int64_t)(row0 + qq) * C + h * HS;
#pragma unroll
                for (int d = 0; d < HS; d += 8) {
                    uint32_t pw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int dd = d + 2 * e;
                        __nv_bfloat162 t2 = __floats2bfloat162_rn(__uint_as_float(ov[dd >> 5][dd & 31]) * inv,
                                                                  __uint_as_float(ov[(dd + 1) >> 5][(dd + 1) & 31]) * inv);
                        pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                    }
                    *reinterpret_cast<uint4*>(yr + d) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                }
                lse[(int64_t)bh * T + qq] = (m_ref + log2f(l)) * 0.6931471805599453f;
            }
            // O_g is read: the next item's first P_g V (which overwrites it) is issued only after
            // this warp arrives on bar_p[g] again
            tc_fence_before();
        }
        tc_fence_before();
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
// Persistent: one CTA per SM walks work items (128-key tile, batch, head) — the earliest key
// tiles, which meet the most queries, first, dealt in snake order — and for each loops over
// the query tiles at or after its keys,
// each cut into two 64-query sub-tiles u (tile u / 2, half u % 2). Warps 0-7 compute: warp w
// owns key rows 32 (w % 4) .. + 31 (its TMEM lane quarter) and 32 query columns (w / 4) of
// each sub-tile. Warp 8 issues the TMA copies and the MMAs. Per sub-tile u:
//   S^T = K Q_u^T, dP^T = V dO_u^T   (M=128 keys, N=64 queries, K=64)   -> TMEM buffer u % 2
//   P^T = 2^(S^T / sqrt(hs) log2(e) - lse log2(e)), dS^T = P^T (dP^T - D)
//                                    bf16 into shared memory (K-major, 128-byte swizzle)
//   dV += P^T dO_u, dK += dS^T Q_u   (M=128 keys, N=64, K=64 queries)   -> TMEM 256..383
// and per query tile, after its second half:
//   dQ_tile = dS K                   (M=128 queries, N=64, K=128 keys)  -> TMEM 384 + 64 (tile % 2)
// With two S^T/dP^T buffers the tensor core computes one sub-tile while the compute warps turn
// the other into P^T and dS^T. dQ_tile, double-buffered in TMEM, goes through a swizzled
// shared-memory tile into a float32 accumulator by TMA reduce-add at the end of the next tile
// (while the tensor core works on that tile's last products); dK and dV are stored once at
// the end. TMEM: S^T/dP^T buffers 0..255, dV 256..319, dK 320..383, dQ 384..511. The barrier
// phases, the Q/dO stages and the dQ buffers run on across items (counted in query tiles); an
// item's K and V are loaded once the previous item's products are complete, while the compute
// warps store that item's dV and dK.
constexpr int BWD_THREADS = 288;
// K, V, Q[2], dO[2], P^T, dS^T, dQ staging (a 4 KB box per compute warp), lse/D (512 B per warp)
constexpr size_t BWD_SMEM_BYTES = 12 * TILE + 4096 + 1024 + 256;

// The r-th work item of this CTA (snake order, as fwd_item), or -1: item k is key tile k / BH of
// (batch x head) k % BH.
__device__ __forceinline__ int bwd_item(int r, int n_items) { return fwd_item(r, n_items); }

__global__ void __maxnreg__(168)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_dy,
                       const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse,
                       const float* __restrict__ dvec, __nv_bfloat16* __restrict__ dqkv, int T, int H, int BH,
                       int n_items, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem;
    uint8_t* sV = smem + TILE;
    uint8_t* sQ = smem + 2 * TILE;    // two stages (query tiles)
    uint8_t* sO = smem + 4 * TILE;    // dO, two stages
    uint8_t* sPT = smem + 6 * TILE;   // two halves (query columns 0..63, 64..127)
    uint8_t* sDS = smem + 8 * TILE;   // two halves
    uint8_t* sDQ = smem + 10 * TILE;  // per compute warp a 32-row x 32-column float32 box, 128-byte swizzle
    float* sLD = reinterpret_cast<float*>(smem + 12 * TILE);  // per compute warp [2 buffers][lse 32 | D 32]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 12 * TILE + 4096);
    uint64_t* bar_kv = bars;
    uint64_t* bar_qo = bars + 1;      // [2] Q, dO of a query tile landed
    uint64_t* bar_s = bars + 3;       // [2] S^T, dP^T of a sub-tile in TMEM buffer
    uint64_t* bar_p = bars + 5;       // [2] P^T, dS^T of a half written (256 arrivals)
    uint64_t* bar_mm = bars + 7;      // dQ of a query tile (and every product before it) done
    uint64_t* bar_drain = bars + 8;
    uint64_t* bar_st = bars + 9;      // a query tile's last dV, dK done: its Q/dO stage is free
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 11);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = H * HS;
    const int n_qt = (T + QT - 1) / QT;

    if (tid == 0) {
        mbar_init(bar_kv, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_qo[i], 1);
            mbar_init(&bar_s[i], 1);
            mbar_init(&bar_p[i], 256);
        }
        mbar_init(bar_mm, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_st, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 8) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // TMA copies and MMAs. The whole warp walks the schedule (warp-uniform descriptors);
        // one elected lane issues each group of copies or MMAs with the commits that track them.
        const uint32_t id_s = instr_desc_bf16(false, false, 128, 64);   // S^T, dP^T of a sub-tile
        const uint32_t id_kv = instr_desc_bf16(false, true, 128, 64);   // dV, dK: B (dO, Q) MN-major
        const uint32_t id_q = instr_desc_bf16(true, true, 128, 64);     // dQ: A (dS) and B (K) MN-major
        const uint64_t k_d = smem_desc(saddr(sK), 16, 1024), v_d = smem_desc(saddr(sV), 16, 1024);
        const uint64_t kq_d = smem_desc(saddr(sK), 8192, 1024);    // K as dQ's MN-major B
        const uint64_t ds_d = smem_desc(saddr(sDS), 16384, 1024);  // dS as dQ's MN-major A
        const uint64_t pt_d = smem_desc(saddr(sPT), 16, 1024), dst_d = smem_desc(saddr(sDS), 16, 1024);
        // Q / dO stages: K-major (S^T, dP^T) and MN-major (dK, dV) views
        const uint64_t q_d0 = smem_desc(saddr(sQ), 16, 1024), q_d1 = smem_desc(saddr(sQ + TILE), 16, 1024);
        const uint64_t o_d0 = smem_desc(saddr(sO), 16, 1024), o_d1 = smem_desc(saddr(sO + TILE), 16, 1024);
        const uint64_t qm_d0 = smem_desc(saddr(sQ), 8192, 1024), qm_d1 = smem_desc(saddr(sQ + TILE), 8192, 1024);
        const uint64_t om_d0 = smem_desc(saddr(sO), 8192, 1024), om_d1 = smem_desc(saddr(sO + TILE), 8192, 1024);
        if (elect_one()) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_qkv) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_dy) : "memory");
        }
        __syncwarp();
        int gt = 0;                // query tiles of the items before this one
        int pend[2] = {-1, -1};    // phase of the Q/dO load in flight per stage
        int kv_pend = -1;          // phase of the K/V load in flight
        bool ok = true, issued = false;
        for (int r = 0, ii = 0; ok; ++r, ++ii) {
            const int item = bwd_item(r, n_items);
            if (item < 0) break;
            const int kt = item / BH, bh = item % BH, h = bh % H;
            const int row0 = (bh / H) * T, k0 = kt * KT, first_qt = k0 / QT;
            const int n_it = n_qt - first_qt, n_u = 2 * n_it;
            // the previous item's products are complete (its last commit): K, V, both Q/dO stages
            // and the S^T/dP^T buffers are free again
            if (ii > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_st, (gt - 1) & 1, abort_flag, WAIT_NS))))
                break;
            if (elect_one()) {
                mbar_expect_tx(bar_kv, 2 * TILE);
                tma_load_2d(&tm_qkv, bar_kv, sK, C + h * HS, row0 + k0);
                tma_load_2d(&tm_qkv, bar_kv, sV, 2 * C + h * HS, row0 + k0);
                for (int i = 0; i < 2 && i < n_it; ++i) {
                    const int st = (gt + i) & 1;
                    mbar_expect_tx(&bar_qo[st], 2 * TILE);
                    tma_load_2d(&tm_qkv, &bar_qo[st], sQ + st * TILE, h * HS, row0 + (first_qt + i) * QT);
                    tma_load_2d(&tm_dy, &bar_qo[st], sO + st * TILE, h * HS, row0 + (first_qt + i) * QT);
                }
            }
            __syncwarp();
            kv_pend = ii & 1;
            for (int i = 0; i < 2 && i < n_it; ++i) pend[(gt + i) & 1] = ((gt + i) >> 1) & 1;
            // S^T and dP^T of sub-tile u into TMEM buffer u % 2 (its tile's Q/dO must have landed)
            auto issue_s = [&](int u) {
                const int st = (gt + (u >> 1)) & 1, hq = u & 1;
                const uint32_t d = tmem + (uint32_t)hq * 128;
#pragma unroll
                for (int k = 0; k < HS / 16; ++k)
                    umma_bf16(d, desc_add(k_d, k * 32), desc_add(pick(q_d0, q_d1, st), hq * 8192 + k * 32), id_s, k > 0);
#pragma unroll
                for (int k = 0; k < HS / 16; ++k)
                    umma_bf16(d + 64, desc_add(v_d, k * 32), desc_add(pick(o_d0, o_d1, st), hq * 8192 + k * 32), id_s, k > 0);
                umma_commit(&bar_s[hq]);
            };
            ok = __all_sync(0xffffffffu, mbar_wait(bar_kv, ii & 1, abort_flag, WAIT_NS) &&
                                             mbar_wait(&bar_qo[gt & 1], (gt >> 1) & 1, abort_flag, WAIT_NS));
            if (!ok) break;
            kv_pend = -1;
            pend[gt & 1] = -1;
            tc_fence_after();
            if (elect_one()) {
                issue_s(0);
                issue_s(1);
            }
            __syncwarp();
            issued = true;
            for (int u = 0; ok && u < n_u; ++u) {
                const int it = u >> 1, hq = u & 1, tg = gt + it, st = tg & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_p[hq], tg & 1, abort_flag, WAIT_NS))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    if (hq == 1) {
                        // dQ of the tile first (both dS halves are in): its completion frees the
                        // P^T / dS^T buffers for the next tile's first half
#pragma unroll
                        for (int k = 0; k < KT / 16; ++k)
                            umma_bf16(tmem + 384 + (uint32_t)(tg & 1) * 64, desc_add(ds_d, k * 2048),
                                      desc_add(kq_d, k * 2048), id_q, k > 0);
                        umma_commit(bar_mm);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t acc = (u > 0 || k > 0) ? 1u : 0u;
                        umma_bf16(tmem + 256, desc_add(pt_d, hq * 16384 + k * 32),
                                  desc_add(pick(om_d0, om_d1, st), hq * 8192 + k * 2048), id_kv, acc);
                        umma_bf16(tmem + 320, desc_add(dst_d, hq * 16384 + k * 32),
                                  desc_add(pick(qm_d0, qm_d1, st), hq * 8192 + k * 2048), id_kv, acc);
                    }
                    if (hq == 1) umma_commit(bar_st);
                }
                __syncwarp();
                if (u + 2 < n_u) {
                    if (hq == 0) {  // the next tile's Q/dO
                        const int ns = (tg + 1) & 1;
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(&bar_qo[ns], ((tg + 1) >> 1) & 1, abort_flag, WAIT_NS))) {
                            ok = false;
                            break;
                        }
                        pend[ns] = -1;
                        tc_fence_after();
                    }
                    if (elect_one()) issue_s(u + 2);
                    __syncwarp();
                }
                if (hq == 1 && it + 2 < n_it) {
                    // stage st (this tile's Q, dO) is free once the tile's last dV, dK are done
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_st, tg & 1, abort_flag, WAIT_NS))) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        mbar_expect_tx(&bar_qo[st], 2 * TILE);
                        tma_load_2d(&tm_qkv, &bar_qo[st], sQ + st * TILE, h * HS, row0 + (first_qt + it + 2) * QT);
                        tma_load_2d(&tm_dy, &bar_qo[st], sO + st * TILE, h * HS, row0 + (first_qt + it + 2) * QT);
                    }
                    __syncwarp();
                    pend[st] = ((tg + 2) >> 1) & 1;
                }
            }
            gt += n_it;
        }
        if (!ok) {
            if (elect_one()) {
                *abort_flag = 1;
                report(err, GK_ERR_TIMEOUT);
                // let this CTA's copies and MMAs in flight finish before shared memory and
                // TMEM are released
                if (kv_pend >= 0) mbar_wait(bar_kv, (uint32_t)kv_pend, nullptr, WAIT_NS / 5);
                for (int i = 0; i < 2; ++i)
                    if (pend[i] >= 0) mbar_wait(&bar_qo[i], (uint32_t)pend[i], nullptr, WAIT_NS / 5);
                if (issued) {
                    umma_commit(bar_drain);
                    mbar_wait(bar_drain, 0, nullptr, WAIT_NS / 5);
                }
            }
            __syncwarp();
        }
    } else {
        const int qd = warp & 3, hf = warp >> 2;
        const int r = qd * 32 + lane;  // key row of S^T / dP^T / dV / dK; query row of dQ
        const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
        const float sl2 = 0.125f * 1.4426950408889634f;
        const float L2E = 1.4426950408889634f;
        // No block barrier in this loop: each warp loads its own lse / D values and drains
        // its own 32 x 32 box of dQ. A failed wait only skips the warp's work and raises the
        // abort flag, so every other wait in the CTA ends quickly.
        bool fail = false;
        auto note_fail = [&](bool ok_) {
            if (!ok_) {
                fail = true;
                *abort_flag = 1;
            }
        };
        float* myLD = sLD + warp * 128;            // [2 buffers][lse 32 | D 32]
        uint8_t* myDQ = sDQ + warp * 4096;         // 32 rows x 128 bytes
        int gt = 0;                                // query tiles of the items before this one
        for (int ri = 0; !fail; ++ri) {
            const int item = bwd_item(ri, n_items);
            if (item < 0) break;
            const int kt = item / BH, bh = item % BH, h = bh % H;
            const int row0 = (bh / H) * T, k0 = kt * KT, first_qt = k0 / QT;
            const int n_it = n_qt - first_qt, n_u = 2 * n_it;
            const int kk = k0 + r;
            // lane c's lse (log2 units) and D for query column c of this warp in sub-tile v
            auto ld_pair = [&](int v, float& lv, float& dvv) {
                const int q = (first_qt + (v >> 1)) * QT + (v & 1) * 64 + hf * 32 + lane;
                lv = q < T ? lse[(int64_t)bh * T + q] * L2E : 0.f;
                dvv = q < T ? dvec[(int64_t)bh * T + q] : 0.f;
            };
            float nl = 0.f, nd = 0.f;
            ld_pair(0, nl, nd);
            // dQ of this item's query tile t (TMEM buffer (gt + t) % 2, complete): this warp's
            // 32 rows x 32 columns through its swizzled staging box into the float32
            // accumulator by TMA reduce-add
            auto drain_dq = [&](int t) {
                if (lane == 0) bulk_wait_read<0>();  // this warp's previous reduce has read the box
                __syncwarp();
                tc_fence_after();
                uint32_t qv[32];
                tmem_ld32_nowait(lane_addr + 384 + (uint32_t)((gt + t) & 1) * 64 + hf * 32, qv);
                tmem_wait_ld_only();
                reg_fence32(qv);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4*>(myDQ + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                        make_float4(__uint_as_float(qv[4 * j]) * 0.125f, __uint_as_float(qv[4 * j + 1]) * 0.125f,
                                    __uint_as_float(qv[4 * j + 2]) * 0.125f, __uint_as_float(qv[4 * j + 3]) * 0.125f);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // rows past this sequence carry dS = 0 (masked), so the whole box is added
                    tma_reduce_add_2d(&tm_dq, myDQ, h * HS + hf * 32, row0 + (first_qt + t) * QT + qd * 32);
                    bulk_commit();
                }
            };
            for (int u = 0; u < n_u; ++u) {
                const int it = u >> 1, hq = u & 1, tg = gt + it;
                const int q0 = (first_qt + it) * QT;
                // this sub-tile's lse / D into the warp's buffer u % 2; the next sub-tile's on the way
                float* L = myLD + (u & 1) * 64;
                L[lane] = nl;
                L[32 + lane] = nd;
                if (u + 1 < n_u) ld_pair(u + 1, nl, nd);
                __syncwarp();
                if (!fail) note_fail(__all_sync(0xffffffffu, mbar_wait(&bar_s[hq], tg & 1, abort_flag, WAIT_NS)));
                if (!fail) {
                    tc_fence_after();
                    uint32_t sv[32], dv[32];
                    tmem_ld32_nowait(lane_addr + hq * 128 + hf * 32, sv);
                    tmem_ld32_nowait(lane_addr + hq * 128 + 64 + hf * 32, dv);
                    tmem_wait_ld_only();
                    reg_fence32(sv);
                    reg_fence32(dv);
                    // this warp's 32 query columns: tile columns cbase .. cbase + 31; visible c
                    // (0..31) satisfy lo <= c < hi
                    const int cbase = hq * 64 + hf * 32;
                    int lo = 0, hi = 32;
                    if (q0 == k0) lo = r - cbase;                 // causal: query >= key on the diagonal
                    hi = min(hi, T - q0 - cbase);                 // ragged last query tile
                    if (kk >= T) hi = 0;                          // padding key rows
                    const bool masked = lo > 0 || hi < 32;
                    const float* D = L + 32;
                    uint32_t pw[16], qw[16];
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) {
                        const float4 l0 = *reinterpret_cast<const float4*>(L + c8);
                        const float4 l1 = *reinterpret_cast<const float4*>(L + c8 + 4);
                        const float4 d0 = *reinterpret_cast<const float4*>(D + c8);
                        const float4 d1 = *reinterpret_cast<const float4*>(D + c8 + 4);
                        const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
                        const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const int c = c8 + e;
                            float p0 = ex2_hw(fmaf(__uint_as_float(sv[c]), sl2, -lv[e]));
                            float p1 = ex2_hw(fmaf(__uint_as_float(sv[c + 1]), sl2, -lv[e + 1]));
                            float ds0 = p0 * (__uint_as_float(dv[c]) - dd[e]);
                            float ds1 = p1 * (__uint_as_float(dv[c + 1]) - dd[e + 1]);
                            if (masked) {  // hidden pairs contribute exactly zero
                                const bool v0 = c >= lo && c < hi, v1 = c + 1 >= lo && c + 1 < hi;
                                p0 = v0 ? p0 : 0.f;
                                ds0 = v0 ? ds0 : 0.f;
                                p1 = v1 ? p1 : 0.f;
                                ds1 = v1 ? ds1 : 0.f;
                            }
                            __nv_bfloat162 t2 = __floats2bfloat162_rn(p0, p1);
                            __nv_bfloat162 u2 = __floats2bfloat162_rn(ds0, ds1);
                            pw[c >> 1] = *reinterpret_cast<uint32_t*>(&t2);
                            qw[c >> 1] = *reinterpret_cast<uint32_t*>(&u2);
                        }
                    }
                    // the P^T / dS^T buffers are free for a new tile once the previous tile's dQ
                    // (issued after its last dS) is done; the half-1 products of the previous tile
                    // finished before this tile's S^T of half 1 (waited above). An item's first
                    // tile follows the previous item's last products, waited for at its end.
                    if (hq == 0 && it > 0)
                        note_fail(__all_sync(0xffffffffu, mbar_wait(bar_mm, (tg - 1) & 1, abort_flag, WAIT_NS)));
                    if (!fail) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            *reinterpret_cast<uint4*>(sPT + p_offset(r, cbase + 8 * j)) =
                                make_uint4(pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
                            *reinterpret_cast<uint4*>(sDS + p_offset(r, cbase + 8 * j)) =
                                make_uint4(qw[4 * j], qw[4 * j + 1], qw[4 * j + 2], qw[4 * j + 3]);
                        }
                        fence_proxy_async_smem();  // P^T, dS^T generic stores -> visible to the tensor core
                        tc_fence_before();
                        mbar_arrive(&bar_p[hq]);
                    }
                }
                // the previous tile's dQ (double-buffered in TMEM; waited above) while the tensor
                // core runs this tile's dQ, dV and dK
                if (hq == 1 && it > 0 && !fail) drain_dq(it - 1);
            }
            if (!fail) {  // the last tile's dQ
                note_fail(__all_sync(0xffffffffu, mbar_wait(bar_mm, (gt + n_it - 1) & 1, abort_flag, WAIT_NS)));
                if (!fail) drain_dq(n_it - 1);
            }
            if (lane == 0) bulk_wait_all();
            __syncwarp();
            // dV and dK: the last tile's dV, dK products follow its dQ, so they are waited for on
            // their own barrier (whose previous phase completed before bar_mm's last one); their
            // completion also frees every buffer of this item for the next one
            if (!fail)
                note_fail(__all_sync(0xffffffffu, mbar_wait(bar_st, (gt + n_it - 1) & 1, abort_flag, WAIT_NS)));
            if (fail) break;
            // lane r = key row kk
            tc_fence_after();
            uint32_t v[32];
            __nv_bfloat16* base = dqkv + (int64_t)(row0 + kk) * 3 * C + h * HS + hf * 32;
            tmem_ld32(lane_addr + 256 + hf * 32, v);  // dV
            if (kk < T) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint32_t pw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 t2 =
                            __floats2bfloat162_rn(__uint_as_float(v[i + 2 * e]), __uint_as_float(v[i + 2 * e + 1]));
                        pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                    }
                    *reinterpret_cast<uint4*>(base + 2 * C + i) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                }
            }
            tmem_ld32(lane_addr + 320 + hf * 32, v);  // dK (times 1/sqrt(hs))
            if (kk < T) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint32_t pw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 t2 = __floats2bfloat162_rn(__uint_as_float(v[i + 2 * e]) * 0.125f,
                                                                  __uint_as_float(v[i + 2 * e + 1]) * 0.125f);
                        pw[e] = *reinterpret_cast<uint32_t*>(&t2);
                    }
                    *reinterpret_cast<uint4*>(base + C + i) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                }
            }
            // dV, dK are read: the next item's first dV / dK products (issued after this warp's
            // next bar_p arrival) may overwrite them
            tc_fence_before();
            gt += n_it;
        }
        if (fail) {
            *abort_flag = 1;
            report(err, GK_ERR_TIMEOUT);
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// D[b,h,t] = sum_d dy * y over each head's 64 columns, one warp per row: lane l takes the
// 16-byte pieces l, l + 32, ... of the row (piece p lies in head p / 8), the 8 lanes of a
// head add their dot products by shuffles. The warp also zeroes the row of the float32 dQ
// accumulator.
__global__ void attn_dvec_zero_kernel(const __nv_bfloat16* __restrict__ y, const __nv_bfloat16* __restrict__ dy,
                                      float* __restrict__ dvec, float* __restrict__ dq_acc, int64_t rows, int T, int H) {
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const int C = H * HS, pieces = C / 8;
    const int64_t b = r / T, t = r % T;
    for (int p0 = 0; p0 < pieces; p0 += 32) {
        const int p = p0 + lane;
        float s = 0.f;
        if (p < pieces) {
            const uint4 a = *reinterpret_cast<const uint4*>(dy + r * C + p * 8);
            const uint4 c = *reinterpret_cast<const uint4*>(y + r * C + p * 8);
            const __nv_bfloat162* ah = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* ch = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                s += __low2float(ah[k]) * __low2float(ch[k]) + __high2float(ah[k]) * __high2float(ch[k]);
            float4* z = reinterpret_cast<float4*>(dq_acc + r * C + p * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // pieces p0 .. p0 + 31 hold heads p0 / 8 .. p0 / 8 + 3, eight lanes each
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        if ((lane & 7) == 0 && p < pieces) dvec[(b * H + p / 8) * T + t] = s;
    }
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
    // persistent: one CTA per SM (each holds all 512 TMEM columns) over the work items
    const int BH = B * H, n_items = BH * (int)cdiv(cdiv(T, QT), 2);
    if (n_items == 0) return GK_OK;
    const int grid = std::min(n_items, ctx->num_sms);
    attn_fwd_tc_kernel<<<grid, FWD_THREADS, FWD_SMEM_BYTES, ctx->stream>>>(map, static_cast<__nv_bfloat16*>(y), lse,
                                                                         T, H, BH, n_items, ctx->d_err);
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
    CUtensorMap map_qkv, map_dy, map_dq;
    if (!make_map(&map_qkv, qkv, 3 * C, rows, 3 * C, 128) || !make_map(&map_dy, dy, C, rows, C, 128) ||
        !make_map_f32(&map_dq, dq_acc, C, rows, C, 32, 32))
        return GK_ERR_UNSUPPORTED;
    attn_dvec_zero_kernel<<<(unsigned)cdiv(rows * 32, 256), 256, 0, ctx->stream>>>(
        (const __nv_bfloat16*)y, (const __nv_bfloat16*)dy, dvec, dq_acc, rows, T, H);
    GK_TRY(launched(ctx, "attn_dvec_zero"));
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BWD_SMEM_BYTES);
        attr = true;
    }
    // persistent: one CTA per SM over the (key tile, batch x head) items, heaviest first
    const int BH = B * H, n_items = BH * (int)cdiv(T, KT);
    const int grid = std::min(n_items, ctx->num_sms);
    attn_bwd_tc_kernel<<<grid, BWD_THREADS, BWD_SMEM_BYTES, ctx->stream>>>(map_qkv, map_dy, map_dq, lse, dvec,
                                                                        (__nv_bfloat16*)dqkv, T, H, BH, n_items,
                                                                        ctx->d_err);
    GK_TRY(launched(ctx, "attn_bwd_tc"));
    attn_dq_store_kernel<<<(unsigned)cdiv(rows * C / 4, 256), 256, 0, ctx->stream>>>(dq_acc, (__nv_bfloat16*)dqkv,
                                                                                    rows, (int)C);
    return launched(ctx, "attn_dq_store");
}

}  // namespace gk
