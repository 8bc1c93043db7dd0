// Tensor-core GEMM for sm_103a: C[M,N] (=|+=) epi(A B + bias + residual) with bfloat16 A and
// B of either majorness, float32 accumulation in tensor memory (TMEM).
//
// Persistent kernel, one 192-thread CTA per SM, 128 x 256 output tiles:
//   warp 0     TMA producer: streams 64-deep K slices of A and B into a 4-stage shared-memory
//              ring (128-byte swizzled tiles), arriving on full[s] with the byte count;
//   warp 1     MMA issuer: one thread issues tcgen05.mma (M=128, N=256, K=16, kind::f16) into
//              one of two TMEM accumulators, commits stage releases to empty[s] and a finished
//              accumulator to tmem_full[b]; the warp also allocates and frees the 512 TMEM
//              columns;
//   warps 2-5  epilogue: tcgen05.ld of their 32 accumulator rows, bias / residual / GELU /
//              GELU-backward, store, then arrive on tmem_empty[b] so the next tile's MMAs can
//              reuse the accumulator while this one is drained.
// Work units are (tile, K split); split K is used only for plain float32 accumulation
// (dW += ...), whose epilogue adds with atomics.
// Every mbarrier wait is bounded (about one second): on expiry the CTA records GK_ERR_TIMEOUT
// in the context's error word, waits briefly for its own TMA copies and MMAs in flight, frees
// its TMEM and returns.
#include "gemm.cuh"
#include "tcgen05.cuh"

namespace gk {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, THREADS = 320;  // 2 + 8 epilogue warps
constexpr uint32_t A_BYTES = BM * BK * 2;         // 16 KB per operand tile
constexpr uint32_t B_BYTES = BN * BK * 2;         // 32 KB per operand tile
constexpr uint32_t TMEM_COLS = 2 * BN;            // two float32 accumulators of 128 x 256

// Stage layout per split mode: bit 0 = A has a low bf16 plane, bit 1 = B has one. A stage
// holds [A_hi | A_lo? | B_hi | B_lo?]; the ring shrinks to keep within 227 KB of shared memory.
template <int SPLIT>
struct StageCfg {
    static constexpr bool A_LO = (SPLIT & 1) != 0, B_LO = (SPLIT & 2) != 0;
    static constexpr uint32_t A_SLOT = A_BYTES * (A_LO ? 2 : 1);
    static constexpr uint32_t B_SLOT = B_BYTES * (B_LO ? 2 : 1);
    static constexpr uint32_t STAGE = A_SLOT + B_SLOT;
    static constexpr int STAGES = SPLIT == 0 ? 4 : (SPLIT == 1 ? 3 : 2);
    static constexpr uint32_t EPI = 8 * 32 * 32 * 4;  // 4 KB per epilogue warp
    static constexpr size_t SMEM = (size_t)STAGES * STAGE + EPI + 1024 + 256;
};
constexpr uint64_t WAIT_NS = 1000000000ull;       // bounded waits: 1 s
constexpr uint64_t DRAIN_NS = 200000000ull;       // after an abort: 0.2 s per drain wait

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, splits, kbps, kblocks;
    int a_kmajor, b_kmajor;
    void* C;
    int64_t ldc;
    int c_dtype, accumulate, atomic_out;
    const float* bias;
    const float* residual;
    int64_t ldr;
    int epi;
    void* aux;
    int64_t ldaux;
    int aux_dtype;
    int64_t c_plane;  // > 0: bf16 C also gets its low plane (v - bf16(v)) at C + c_plane
    int vec;          // every epilogue pointer 16-byte aligned and every stride a multiple of 4
    int fast_act;     // bf16 output without a low plane: GELU through the hardware tanh
    int* err;
};

// --------------------------------------------------------------------- epilogue
// GELU (tanh form) with the hardware tanh.approx.f32 instead of tanhf: its error (about
// 2^-11 relative) is below the bf16 rounding of the outputs it is used for.
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float gelu_hw(float x) {
    const float k = 0.7978845608028654f;
    return 0.5f * x * (1.0f + tanh_hw(k * (x + 0.044715f * x * x * x)));
}
__device__ __forceinline__ float gelu_grad_hw(float x) {
    const float k = 0.7978845608028654f;
    float t = tanh_hw(k * (x + 0.044715f * x * x * x));
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * k * (1.0f + 3.0f * 0.044715f * x * x);
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

template <typename TC>
__device__ __forceinline__ float4 ld4c(const TC* p) {
    if constexpr (sizeof(TC) == 4) {
        return *reinterpret_cast<const float4*>(p);
    } else {
        uint2 u = *reinterpret_cast<const uint2*>(p);
        __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x), b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
        return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
    }
}

__device__ __forceinline__ void st4_bf16(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}

// Epilogue of one element (the scalar path for edges and unaligned operands).
template <typename TC>
__device__ __forceinline__ void epi1(const TcParams& p, int64_t m, int64_t n, float v) {
    int64_t ci = m * p.ldc + n;
    if (p.atomic_out) {
        atomicAdd(static_cast<float*>(p.C) + ci, v);
        return;
    }
    TC* C = static_cast<TC*>(p.C);
    if (p.accumulate) v += load_as_f32(C + ci);
    if (p.bias) v += p.bias[n];
    if (p.residual) v += p.residual[m * p.ldr + n];
    if (p.epi == EPI_GELU) {
        if (p.aux_dtype == GK_F32)
            static_cast<float*>(p.aux)[m * p.ldaux + n] = v;
        else
            static_cast<__nv_bfloat16*>(p.aux)[m * p.ldaux + n] = __float2bfloat16_rn(v);
        v = gelu_tanh(v);
    } else if (p.epi == EPI_DGELU) {
        float pre = p.aux_dtype == GK_F32 ? static_cast<const float*>(p.aux)[m * p.ldaux + n]
                                          : __bfloat162float(static_cast<const __nv_bfloat16*>(p.aux)[m * p.ldaux + n]);
        v *= gelu_tanh_grad(pre);
    }
    store_from_f32(C + ci, v);
    if (p.c_plane) {
        __nv_bfloat16* Cb = static_cast<__nv_bfloat16*>(p.C);
        Cb[ci + p.c_plane] = __float2bfloat16_rn(v - __bfloat162float(Cb[ci]));
    }
}

// Epilogue of 4 consecutive columns n .. n+3 of row m (16-byte accesses when allowed).
template <typename TC>
__device__ __forceinline__ void epi4(const TcParams& p, int64_t m, int64_t n, float4 v) {
    if (m >= p.M || n >= p.N) return;
    if (!p.vec || n + 3 >= p.N) {
        float t[4] = {v.x, v.y, v.z, v.w};
        for (int j = 0; j < 4 && n + j < p.N; ++j) epi1<TC>(p, m, n + j, t[j]);
        return;
    }
    int64_t ci = m * p.ldc + n;
    if (p.atomic_out) {
        atomicAdd(reinterpret_cast<float4*>(static_cast<float*>(p.C) + ci), v);
        return;
    }
    TC* C = static_cast<TC*>(p.C);
    if (p.accumulate) {
        float4 c = ld4c<TC>(C + ci);
        v.x += c.x; v.y += c.y; v.z += c.z; v.w += c.w;
    }
    if (p.bias) {
        float4 b = ld4(p.bias + n);
        v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
    }
    if (p.residual) {
        float4 r = ld4(p.residual + m * p.ldr + n);
        v.x += r.x; v.y += r.y; v.z += r.z; v.w += r.w;
    }
    if (p.epi == EPI_GELU) {
        if (p.aux_dtype == GK_F32)
            *reinterpret_cast<float4*>(static_cast<float*>(p.aux) + m * p.ldaux + n) = v;
        else
            st4_bf16(static_cast<__nv_bfloat16*>(p.aux) + m * p.ldaux + n, v);
        if (p.fast_act)
            v = make_float4(gelu_hw(v.x), gelu_hw(v.y), gelu_hw(v.z), gelu_hw(v.w));
        else
            v = make_float4(gelu_tanh(v.x), gelu_tanh(v.y), gelu_tanh(v.z), gelu_tanh(v.w));
    } else if (p.epi == EPI_DGELU) {
        float4 pre = p.aux_dtype == GK_F32 ? ld4(static_cast<const float*>(p.aux) + m * p.ldaux + n)
                                           : ld4c<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(p.aux) + m * p.ldaux + n);
        if (p.fast_act) {
            v.x *= gelu_grad_hw(pre.x); v.y *= gelu_grad_hw(pre.y);
            v.z *= gelu_grad_hw(pre.z); v.w *= gelu_grad_hw(pre.w);
        } else {
            v.x *= gelu_tanh_grad(pre.x); v.y *= gelu_tanh_grad(pre.y);
            v.z *= gelu_tanh_grad(pre.z); v.w *= gelu_tanh_grad(pre.w);
        }
    }
    if constexpr (sizeof(TC) == 4) {
        *reinterpret_cast<float4*>(C + ci) = v;
    } else {
        __nv_bfloat16* Cb = reinterpret_cast<__nv_bfloat16*>(C);
        st4_bf16(Cb + ci, v);
        if (p.c_plane) {
            float4 h = ld4c<__nv_bfloat16>(Cb + ci);
            st4_bf16(Cb + ci + p.c_plane, make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w));
        }
    }
}

__device__ __forceinline__ void unit_coords(const TcParams& p, int u, int& tm, int& tn, int& kb0, int& kb1) {
    int split = u % p.splits, tile = u / p.splits;
    tm = tile % p.tiles_m;
    tn = tile / p.tiles_m;
    kb0 = split * p.kbps;
    kb1 = min(p.kblocks, kb0 + p.kbps);
}

template <typename TC, int SPLIT>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA_lo, const __grid_constant__ CUtensorMap tmB_lo,
                   const TcParams p) {
    using SC = StageCfg<SPLIT>;
    constexpr int STAGES = SC::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // stage s: A_hi at smem + s*STAGE, A_lo at + A_BYTES, B_hi at + A_SLOT, B_lo at + A_SLOT + B_BYTES
    float* epi_stage = reinterpret_cast<float*>(smem + STAGES * SC::STAGE);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * SC::STAGE + SC::EPI);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = bars + 2 * STAGES + 2;
    uint64_t* drain = bars + 2 * STAGES + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 6);

    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int units = p.tiles_m * p.tiles_n * p.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 256);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
            if (SC::A_LO) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA_lo) : "memory");
            if (SC::B_LO) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB_lo) : "memory");
            uint32_t it = 0;
            int issued_ph[STAGES];
            for (int s = 0; s < STAGES; ++s) issued_ph[s] = -1;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int tm, tn, kb0, kb1;
                unit_coords(p, u, tm, tn, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    int s = it % STAGES;
                    uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, WAIT_NS)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&full[s], SC::STAGE);
                    uint8_t* a = smem + s * SC::STAGE;
                    uint8_t* b = a + SC::A_SLOT;
#pragma unroll
                    for (int pl = 0; pl < (SC::A_LO ? 2 : 1); ++pl) {
                        const CUtensorMap* ma = pl ? &tmA_lo : &tmA;
                        uint8_t* dst = a + pl * A_BYTES;
                        if (p.a_kmajor) {
                            tma_load_2d(ma, &full[s], dst, kb * BK, tm * BM);
                        } else {
                            tma_load_2d(ma, &full[s], dst, tm * BM, kb * BK);
                            tma_load_2d(ma, &full[s], dst + 8192, tm * BM + 64, kb * BK);
                        }
                    }
#pragma unroll
                    for (int pl = 0; pl < (SC::B_LO ? 2 : 1); ++pl) {
                        const CUtensorMap* mb = pl ? &tmB_lo : &tmB;
                        uint8_t* dst = b + pl * B_BYTES;
                        if (p.b_kmajor) {
                            tma_load_2d(mb, &full[s], dst, kb * BK, tn * BN);
                        } else {
#pragma unroll
                            for (int j = 0; j < BN / 64; ++j)
                                tma_load_2d(mb, &full[s], dst + j * 8192, tn * BN + 64 * j, kb * BK);
                        }
                    }
                    issued_ph[s] = (int)ph;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                report(p.err, GK_ERR_TIMEOUT);
                // let this CTA's copies in flight land before shared memory is released
                for (int s = 0; s < STAGES; ++s)
                    if (issued_ph[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_ph[s], nullptr, DRAIN_NS);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = instr_desc_bf16(!p.a_kmajor, !p.b_kmajor, BM, BN);
            // per 16-deep K step: K-major operands advance 32 bytes inside the swizzled row,
            // MN-major operands advance two 8-row core-matrix groups (2 x 1024 bytes)
            const uint32_t a_step = p.a_kmajor ? 32u : 2048u;
            const uint32_t b_step = p.b_kmajor ? 32u : 2048u;
            const uint32_t a_lbo = p.a_kmajor ? 16u : 8192u, b_lbo = p.b_kmajor ? 16u : 8192u;
            uint32_t it = 0, j = 0;
            bool ok = true, issued = false;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
                int tm, tn, kb0, kb1;
                unit_coords(p, u, tm, tn, kb0, kb1);
                uint32_t buf = j & 1, aph = (j >> 1) & 1;
                if (!mbar_wait(&tempty[buf], aph ^ 1, abort_flag, WAIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    int s = it % STAGES;
                    uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(&full[s], ph, abort_flag, WAIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t a0 = saddr(smem + s * SC::STAGE), b0 = a0 + SC::A_SLOT;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        uint64_t ad = smem_desc(a0 + k * a_step, a_lbo, 1024);
                        uint64_t bd = smem_desc(b0 + k * b_step, b_lbo, 1024);
                        umma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        // split operands: + A_hi B_lo + A_lo B_hi (the A_lo B_lo term is dropped)
                        if (SC::B_LO)
                            umma_bf16(d_tmem, ad, smem_desc(b0 + B_BYTES + k * b_step, b_lbo, 1024), idesc, 1u);
                        if (SC::A_LO)
                            umma_bf16(d_tmem, smem_desc(a0 + A_BYTES + k * a_step, a_lbo, 1024), bd, idesc, 1u);
                    }
                    issued = true;
                    umma_commit(&empty[s]);
                }
                if (!ok) break;
                umma_commit(&tfull[buf]);
            }
            if (!ok) {
                *abort_flag = 1;
                report(p.err, GK_ERR_TIMEOUT);
                if (issued) {
                    umma_commit(drain);
                    mbar_wait(drain, 0, nullptr, DRAIN_NS);
                }
            }
        }
    } else {
        // epilogue warps 2..9; a warp may read TMEM lanes 32 * (warp % 4) .. + 31; two warps
        // share each lane quarter and take alternate halves of the tile's columns
        int q = warp & 3;
        int half = (warp - 2) >> 2;
        uint32_t j = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
            int tm, tn, kb0, kb1;
            unit_coords(p, u, tm, tn, kb0, kb1);
            uint32_t buf = j & 1, aph = (j >> 1) & 1;
            if (!mbar_wait(&tfull[buf], aph, abort_flag, WAIT_NS)) {
                *abort_flag = 1;
                report(p.err, GK_ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            // Each 32 x 32 block of this warp's rows goes through a private, 16-byte-chunk
            // XOR-swizzled staging tile: written one row per lane (as tcgen05.ld delivers it),
            // read back row-contiguously (8 lanes x 4 columns per row) so that bias, residual
            // and the stores are coalesced 16-byte accesses.
            float* stg = epi_stage + (warp - 2) * 1024;
            const int64_t mrow0 = (int64_t)tm * BM + q * 32;
            for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + c0, r);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<float4*>(stg + lane * 32 + ((c ^ (lane & 7)) << 2)) =
                        make_float4(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]),
                                    __uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3]));
                __syncwarp();
                const int64_t n0 = (int64_t)tn * BN + c0;
                if (n0 < p.N) {
#pragma unroll 4
                    for (int pass = 0; pass < 8; ++pass) {
                        int rr = pass * 4 + (lane >> 3), c = lane & 7;
                        float4 v = *reinterpret_cast<const float4*>(stg + rr * 32 + ((c ^ (rr & 7)) << 2));
                        epi4<TC>(p, mrow0 + rr, n0 + c * 4, v);
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            mbar_arrive(&tempty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <typename TC, int SPLIT>
void launch_one(gk_ctx* ctx, int grid, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& al,
                const CUtensorMap& bl, const TcParams& p) {
    static bool attr = false;
    constexpr size_t smem = StageCfg<SPLIT>::SMEM;
    if (!attr) {
        cudaFuncSetAttribute(gemm_tc_kernel<TC, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr = true;
    }
    gemm_tc_kernel<TC, SPLIT><<<grid, THREADS, smem, ctx->stream>>>(a, b, al, bl, p);
}

template <typename TC>
void launch_split(gk_ctx* ctx, int split, int grid, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& al,
                  const CUtensorMap& bl, const TcParams& p) {
    switch (split) {
        case 0: launch_one<TC, 0>(ctx, grid, a, b, al, bl, p); break;
        case 1: launch_one<TC, 1>(ctx, grid, a, b, al, bl, p); break;
        case 2: launch_one<TC, 2>(ctx, grid, a, b, al, bl, p); break;
        default: launch_one<TC, 3>(ctx, grid, a, b, al, bl, p); break;
    }
}

}  // namespace

gk_status gemm_tc(gk_ctx* ctx, const Gemm& g) {
    if (g.ab_dtype != GK_BF16) return GK_ERR_UNSUPPORTED;
    if (!aligned16(g.A) || !aligned16(g.B) || (g.lda & 7) || (g.ldb & 7)) return GK_ERR_UNSUPPORTED;
    if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.M >= (1ll << 31) || g.N >= (1ll << 31) || g.K >= (1ll << 31))
        return GK_ERR_UNSUPPORTED;
    CUtensorMap ta, tb;
    bool ok = g.a_kmajor ? make_map(&ta, g.A, g.K, g.M, g.lda, BM) : make_map(&ta, g.A, g.M, g.K, g.lda, 64);
    ok = ok && (g.b_kmajor ? make_map(&tb, g.B, g.K, g.N, g.ldb, BN) : make_map(&tb, g.B, g.N, g.K, g.ldb, 64));
    if (!ok) return GK_ERR_UNSUPPORTED;
    TcParams p{};
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.tiles_m = (int)cdiv(g.M, BM);
    p.tiles_n = (int)cdiv(g.N, BN);
    p.kblocks = (int)cdiv(g.K, BK);
    p.a_kmajor = g.a_kmajor;
    p.b_kmajor = g.b_kmajor;
    p.C = g.C;
    p.ldc = g.ldc;
    p.c_dtype = g.c_dtype;
    p.accumulate = g.accumulate;
    p.bias = g.bias;
    p.residual = g.residual;
    p.ldr = g.ldr;
    p.epi = g.epi;
    p.aux = g.aux;
    p.ldaux = g.ldaux;
    p.aux_dtype = g.aux_dtype;
    p.err = ctx->d_err;
    p.c_plane = g.c_plane;
    p.fast_act = g.c_dtype == GK_BF16 && g.c_plane == 0;
    p.vec = aligned16(g.C) && (g.ldc % 4 == 0) && (!g.bias || aligned16(g.bias)) &&
            (!g.residual || (aligned16(g.residual) && g.ldr % 4 == 0)) &&
            (!g.aux || (aligned16(g.aux) && g.ldaux % 4 == 0)) && (g.c_plane % 4 == 0);
    if ((g.A_lo && (!aligned16(g.A_lo))) || (g.B_lo && !aligned16(g.B_lo))) return GK_ERR_UNSUPPORTED;
    int64_t tiles = (int64_t)p.tiles_m * p.tiles_n;
    p.splits = 1;
    bool plain_acc = g.accumulate && g.c_dtype == GK_F32 && !g.bias && !g.residual && g.epi == EPI_NONE;
    if (plain_acc && tiles < ctx->num_sms) {
        int want = (int)cdiv(2 * (int64_t)ctx->num_sms, tiles);
        int maxs = std::max(1, p.kblocks / 4);
        p.splits = std::max(1, std::min(want, maxs));
    }
    p.kbps = (int)cdiv(p.kblocks, p.splits);
    p.splits = (int)cdiv(p.kblocks, p.kbps);
    p.atomic_out = p.splits > 1;
    int64_t units = tiles * p.splits;
    int grid = (int)std::min<int64_t>(units, ctx->num_sms);
    int split = (g.A_lo ? 1 : 0) | (g.B_lo ? 2 : 0);
    CUtensorMap ta_lo = ta, tb_lo = tb;
    if (g.A_lo && !(g.a_kmajor ? make_map(&ta_lo, g.A_lo, g.K, g.M, g.lda, BM) : make_map(&ta_lo, g.A_lo, g.M, g.K, g.lda, 64)))
        return GK_ERR_UNSUPPORTED;
    if (g.B_lo && !(g.b_kmajor ? make_map(&tb_lo, g.B_lo, g.K, g.N, g.ldb, BN) : make_map(&tb_lo, g.B_lo, g.N, g.K, g.ldb, 64)))
        return GK_ERR_UNSUPPORTED;
    if (g.c_dtype == GK_F32)
        launch_split<float>(ctx, split, grid, ta, tb, ta_lo, tb_lo, p);
    else
        launch_split<__nv_bfloat16>(ctx, split, grid, ta, tb, ta_lo, tb_lo, p);
    return launched(ctx, "gemm_tc");
}

}  // namespace gk
