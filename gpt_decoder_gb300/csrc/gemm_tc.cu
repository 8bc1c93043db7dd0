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

// Stage layout per mode: bit 0 = A has a low bf16 plane, bit 1 = B has one; mode PAIR_MODE is
// a CTA pair sharing 256 x 256 tiles (each CTA holds its 128 rows of A and 128 of the 256
// columns of B). A stage holds [A_hi | A_lo? | B_hi | B_lo?]; the ring is as deep as 227 KB of
// shared memory allows. PAIR4_MODE: clusters of two pairs on tiles with the same columns (B):
// each CTA loads its A rows and half of its B columns, and multicasts that half to the CTA of
// the other pair that needs the same columns, so a CTA requests 24 of the 32 KB it receives per
// stage.
constexpr int PAIR_MODE = 4, PAIR4_MODE = 5;
template <int SPLIT>
struct StageCfg {
    static constexpr bool MC = SPLIT == PAIR4_MODE;
    static constexpr bool PAIR = SPLIT == PAIR_MODE || MC;
    static constexpr bool A_LO = !PAIR && (SPLIT & 1) != 0, B_LO = !PAIR && (SPLIT & 2) != 0;
    static constexpr uint32_t A_SLOT = A_BYTES * (A_LO ? 2 : 1);
    static constexpr uint32_t B_TILE = PAIR ? B_BYTES / 2 : B_BYTES;  // the B columns this CTA loads
    static constexpr uint32_t B_SLOT = B_TILE * (B_LO ? 2 : 1);
    static constexpr uint32_t STAGE = A_SLOT + B_SLOT;
    static constexpr int STAGES = PAIR ? 6 : SPLIT == 0 ? 4 : (SPLIT == 1 ? 3 : 2);
    static constexpr uint32_t EPI = 8 * 32 * 32 * 4;  // 4 KB per epilogue warp
    static constexpr size_t SMEM = (size_t)STAGES * STAGE + EPI + 1024 + 512;
};
constexpr uint64_t WAIT_NS = 1000000000ull;       // bounded waits: 1 s
constexpr uint64_t DRAIN_NS = 200000000ull;       // after an abort: 0.2 s per drain wait

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, splits, kbps, kblocks;
    int pair, tiles_m2;  // CTA pairs: a unit is a 256-row tile pair; tiles_m2 = ceil(tiles_m / 2)
    int n_fast;          // tile order: column tiles of a row block consecutive (else row tiles)
    int mc, tiles_m4;    // clusters of two pairs: a unit is two pair tiles in one column block
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
    // Epilogue through shared memory and TMA (every plane has C's element type): each warp
    // drains 32 rows x 64 bytes per chunk into a swizzled 2 KB slot that one TMA store (or
    // float32 reduce-add) writes out; an input plane is fetched by TMA a chunk ahead.
    int tma_epi;
    int in_kind;      // IN_NONE / IN_C (accumulate by load) / IN_RES (residual) / IN_AUX (GELU backward)
    int reduce_out;   // C += v by TMA reduce-add (float32 C)
    int out_aux;      // GELU: the pre-activation plane is stored too
    int out_lo;       // bf16 C: its low plane is stored too
    // fused softmax cross-entropy (see Gemm::ce_mode)
    int ce_mode, ce_nparts;
    int64_t ce_col0;
    const int32_t* ce_tgt;
    float2* ce_part;
    float* ce_tgt_logit;
    const float* ce_lse;
    const float* ce_dloss;
    float ce_scale;
    int* err;
    // a batch of products (see Gemm::nz)
    int nz, zh, z0;
    int zo[3][2][3];
};

enum { IN_NONE = 0, IN_C = 1, IN_RES = 2, IN_AUX = 3 };
constexpr uint32_t SLOT = 2048;  // one epilogue chunk: 32 rows x 64 bytes

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

constexpr float LOG2E_F = 1.4426950408889634f;

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
    if (p.accumulate) v += load_as_f32(C + ci);
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
    if (p.accumulate) {
        float4 c = ld4c<TC>(C + ci);
        v.x += c.x; v.y += c.y; v.z += c.z; v.w += c.w;
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

// Two-phase form of epi4 for a whole chunk: every global operand the epilogue reads (C when
// accumulating, the residual, the GELU pre-activation) is loaded first for all rows of the
// chunk, then the values are combined and stored; stores to C could alias those operands,
// so this ordering is what lets the loads overlap instead of paying one latency per row.
struct EpiIn {
    float4 c, r, a;
};

template <typename TC>
__device__ __forceinline__ bool epi_vec_ok(const TcParams& p, int64_t m, int64_t n) {
    return m < p.M && p.vec && n + 3 < p.N;
}

template <typename TC>
__device__ __forceinline__ void epi_load(const TcParams& p, int64_t m, int64_t n, EpiIn& e) {
    if (!epi_vec_ok<TC>(p, m, n) || p.atomic_out) return;
    if (p.accumulate) e.c = ld4c<TC>(static_cast<const TC*>(p.C) + m * p.ldc + n);
    if (p.residual) e.r = ld4(p.residual + m * p.ldr + n);
    if (p.epi == EPI_DGELU)
        e.a = p.aux_dtype == GK_F32 ? ld4(static_cast<const float*>(p.aux) + m * p.ldaux + n)
                                    : ld4c<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(p.aux) + m * p.ldaux + n);
}

template <typename TC>
__device__ __forceinline__ void epi_finish(const TcParams& p, int64_t m, int64_t n, float4 v, const EpiIn& e) {
    if (m >= p.M || n >= p.N) return;
    if (!epi_vec_ok<TC>(p, m, n) || p.atomic_out) {
        epi4<TC>(p, m, n, v);
        return;
    }
    int64_t ci = m * p.ldc + n;
    TC* C = static_cast<TC*>(p.C);
    if (p.bias) {
        float4 b = ld4(p.bias + n);
        v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
    }
    if (p.residual) { v.x += e.r.x; v.y += e.r.y; v.z += e.r.z; v.w += e.r.w; }
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
        if (p.fast_act) {
            v.x *= gelu_grad_hw(e.a.x); v.y *= gelu_grad_hw(e.a.y);
            v.z *= gelu_grad_hw(e.a.z); v.w *= gelu_grad_hw(e.a.w);
        } else {
            v.x *= gelu_tanh_grad(e.a.x); v.y *= gelu_tanh_grad(e.a.y);
            v.z *= gelu_tanh_grad(e.a.z); v.w *= gelu_tanh_grad(e.a.w);
        }
    }
    if (p.accumulate) { v.x += e.c.x; v.y += e.c.y; v.z += e.c.z; v.w += e.c.w; }
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

// Units of work of this CTA: u = unit_first(p), + unit_step(p), ... Both CTAs of a pair walk
// the same units; tm is this CTA's own 128-row tile.
__device__ __forceinline__ int unit_first(const TcParams& p) {
    return p.mc ? (int)(blockIdx.x >> 2) : p.pair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
}
__device__ __forceinline__ int unit_step(const TcParams& p) {
    return p.mc ? (int)(gridDim.x >> 2) : p.pair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
}
// BATCH: the kernel may run a batch of products (p.nz > 1; only the float32-operand kernels are
// built for it, so the others keep no trace of the batch arithmetic).
template <bool BATCH>
__device__ __forceinline__ void unit_coords(const TcParams& p, int u, int& tm, int& tn, int& kb0, int& kb1) {
    int split = u % p.splits, tile = u / p.splits;
    if (BATCH && p.nz > 1) tile %= p.tiles_m * p.tiles_n;  // the tile within its product of the batch
    const int rows = p.mc ? p.tiles_m4 : p.pair ? p.tiles_m2 : p.tiles_m;
    const int tr = p.n_fast ? tile / p.tiles_n : tile % rows;
    tn = p.n_fast ? tile % p.tiles_n : tile / rows;
    // a cluster of two pairs takes pair rows 2 tr and 2 tr + 1 (bit 1 of the CTA's index)
    const int tp = p.mc ? tr * 2 + (int)((blockIdx.x >> 1) & 1) : tr;
    tm = p.pair ? tp * 2 + (int)(blockIdx.x & 1) : tp;
    kb0 = split * p.kbps;
    kb1 = min(p.kblocks, kb0 + p.kbps);
}

// Batch position of unit u, and the TMA coordinate shift of operand o along c (0 = x, 1 = y).
template <bool BATCH>
__device__ __forceinline__ int unit_z(const TcParams& p, int u) {
    return BATCH && p.nz > 1 ? (u / p.splits) / (p.tiles_m * p.tiles_n) : 0;
}
template <bool BATCH>
__device__ __forceinline__ int zshift(const TcParams& p, int o, int c, int zl) {
    if (!BATCH || p.nz <= 1) return 0;
    const int zg = p.z0 + zl;
    return (zg % p.zh) * p.zo[o][c][0] + (zg / p.zh) * p.zo[o][c][1] + zl * p.zo[o][c][2];
}

// ------------------------------------------------------------ TMA epilogue
// Chunks of this warp's part of a tile: rows 32q .. 32q+31 of the tile, columns
// half*128 .. +127 cut into chunks of W = 64 / sizeof(TC) columns; chunks wholly outside
// the matrix are skipped.
template <typename TC>
__device__ __forceinline__ int epi_chunks(const TcParams& p, int tm, int tn, int q, int half) {
    constexpr int W = 64 / (int)sizeof(TC);
    if (tm * BM + q * 32 >= p.M) return 0;
    int rem = p.N - (tn * BN + half * (BN / 2));
    if (rem <= 0) return 0;
    return min((BN / 2) / W, (rem + W - 1) / W);
}

// Advance (u, ch) to this warp's next chunk, possibly in a later unit of this CTA.
template <typename TC, bool BATCH>
__device__ __forceinline__ bool epi_next(const TcParams& p, int units, int& u, int& ch, int q, int half) {
    int tm, tn, kb0, kb1;
    unit_coords<BATCH>(p, u, tm, tn, kb0, kb1);
    if (ch + 1 < epi_chunks<TC>(p, tm, tn, q, half)) {
        ++ch;
        return true;
    }
    for (int v = u + unit_step(p); v < units; v += unit_step(p)) {
        unit_coords<BATCH>(p, v, tm, tn, kb0, kb1);
        if (epi_chunks<TC>(p, tm, tn, q, half) > 0) {
            u = v;
            ch = 0;
            return true;
        }
    }
    return false;
}

// Slot rows are 64 bytes in the TMA 64-byte swizzle: 16-byte piece j of row r sits at piece
// j ^ ((r >> 1) & 3). Each lane owns one row.
__device__ __forceinline__ uint8_t* slot_piece(uint8_t* slot, int row, int j) {
    return slot + row * 64 + ((j ^ ((row >> 1) & 3)) << 4);
}

template <typename TC>
__device__ __forceinline__ void slot_write(uint8_t* slot, int row, const float (&v)[32]) {
    if constexpr (sizeof(TC) == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 w;
            __nv_bfloat162 a = __floats2bfloat162_rn(v[8 * j], v[8 * j + 1]);
            __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * j + 2], v[8 * j + 3]);
            __nv_bfloat162 c = __floats2bfloat162_rn(v[8 * j + 4], v[8 * j + 5]);
            __nv_bfloat162 d = __floats2bfloat162_rn(v[8 * j + 6], v[8 * j + 7]);
            w.x = *reinterpret_cast<uint32_t*>(&a);
            w.y = *reinterpret_cast<uint32_t*>(&b);
            w.z = *reinterpret_cast<uint32_t*>(&c);
            w.w = *reinterpret_cast<uint32_t*>(&d);
            *reinterpret_cast<uint4*>(slot_piece(slot, row, j)) = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4*>(slot_piece(slot, row, j)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
}

template <typename TC>
__device__ __forceinline__ void slot_read(uint8_t* slot, int row, float (&v)[32]) {
    if constexpr (sizeof(TC) == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 w = *reinterpret_cast<const uint4*>(slot_piece(slot, row, j));
            uint32_t u4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u4[k]);
                v[8 * j + 2 * k] = __low2float(h);
                v[8 * j + 2 * k + 1] = __high2float(h);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 f = *reinterpret_cast<const float4*>(slot_piece(slot, row, j));
            v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
        }
    }
}

struct EpiMaps {
    const CUtensorMap* C;
    const CUtensorMap* aux;
    const CUtensorMap* lo;
    const CUtensorMap* in;  // the input plane's map (C, residual or aux), or null
};

// Epilogue warp (one of 8) of the TMA path. Returns false if it gave up on a wait.
// An epilogue warp hands its accumulator buffer back to the MMA issuer (the even CTA of a pair).
// Its TMEM loads are complete (tcgen05.wait::ld) before it gets here.
__device__ __forceinline__ void release_accumulator(const TcParams& p, uint64_t* bar, int lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if (p.pair && (blockIdx.x & 1))
            mbar_arrive_cluster_relaxed(mapa_shared(saddr(bar), cluster_ctarank() & ~1u));
        else
            mbar_arrive(bar);
    }
}

template <typename TC, bool BATCH>
__device__ bool epilogue_tma(const TcParams& p, const EpiMaps& mp, uint8_t* slots, uint64_t* inbar, uint64_t* tfull,
                             uint64_t* tempty, volatile int* abort_flag, uint32_t tmem_base, int warp, int lane,
                             int units) {
    constexpr int W = 64 / (int)sizeof(TC);
    const int q = warp & 3, half = (warp - 2) >> 2;
    const bool has_in = p.in_kind != IN_NONE;
    uint32_t g = 0;       // chunks processed by this warp
    uint32_t kst = 0;     // single-slot stores issued (output-only path)
    int pend_slot = -1;   // lane 0: slot of the input load in flight, for the abort drain
    uint32_t pend_par = 0;
    bool ok = true;

    // the first chunk's input
    if (has_in && lane == 0) {
        int u0 = unit_first(p), c0 = -1;
        bool any = false;
        for (int v = unit_first(p); v < units && !any; v += unit_step(p)) {
            int tm, tn, kb0, kb1;
            unit_coords<BATCH>(p, v, tm, tn, kb0, kb1);
            if (epi_chunks<TC>(p, tm, tn, q, half) > 0) {
                u0 = v;
                c0 = 0;
                any = true;
            }
        }
        if (any) {
            int tm, tn, kb0, kb1;
            unit_coords<BATCH>(p, u0, tm, tn, kb0, kb1);
            mbar_expect_tx(&inbar[0], SLOT);
            tma_load_2d(mp.in, &inbar[0], slots, tn * BN + half * (BN / 2) + c0 * W, tm * BM + q * 32);
            pend_slot = 0;
            pend_par = 0;
        }
    }

    uint32_t j = 0;
    for (int u = unit_first(p); u < units && ok; u += unit_step(p), ++j) {
        int tm, tn, kb0, kb1;
        unit_coords<BATCH>(p, u, tm, tn, kb0, kb1);
        const uint32_t buf = j & 1, aph = (j >> 1) & 1;
        // warp-uniform outcome: every lane leaves together or none does
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[buf], aph, abort_flag, WAIT_NS))) {
            ok = false;
            break;
        }
        tc_fence_after();
        const int nch = epi_chunks<TC>(p, tm, tn, q, half);
        // warm L2 with the next unit's input while this tile drains
        if (has_in && lane == 0 && u + unit_step(p) < units) {
            int tm2, tn2, a2, b2;
            unit_coords<BATCH>(p, u + unit_step(p), tm2, tn2, a2, b2);
            const int n2 = epi_chunks<TC>(p, tm2, tn2, q, half);
            for (int c = 0; c < n2; ++c)
                tma_prefetch_l2_2d(mp.in, tn2 * BN + half * (BN / 2) + c * W, tm2 * BM + q * 32);
        }
        const int y = tm * BM + q * 32;
        const int zl = unit_z<BATCH>(p, u), cxs = zshift<BATCH>(p, 2, 0, zl), cys = zshift<BATCH>(p, 2, 1, zl);  // batch: C's shift
        // fused cross-entropy: this lane's row (y + lane) state over the tile's columns
        float ce_m = -INFINITY, ce_s = 0.f, ce_l2 = 0.f, ce_g = 0.f;
        int ce_t = -1;
        if (p.ce_mode != CE_NONE && y + lane < p.M) {
            ce_t = p.ce_tgt[y + lane];
            if (p.ce_mode == CE_DLOGITS) {
                ce_l2 = p.ce_lse[y + lane] * LOG2E_F;
                ce_g = (p.ce_dloss ? *p.ce_dloss : 1.f) * p.ce_scale;
            }
        }
        for (int ch = 0; ch < nch; ++ch, ++g) {
            const int x = tn * BN + half * (BN / 2) + ch * W;
            const uint32_t s = g & 1;
            // the next chunk's input goes into the other slot once its last store has read it
            if (has_in && lane == 0) {
                int nu = u, nc = ch;
                if (epi_next<TC, BATCH>(p, units, nu, nc, q, half)) {
                    int tm2, tn2, a2, b2;
                    unit_coords<BATCH>(p, nu, tm2, tn2, a2, b2);
                    bulk_wait_read<0>();
                    mbar_expect_tx(&inbar[s ^ 1], SLOT);
                    tma_load_2d(mp.in, &inbar[s ^ 1], slots + (s ^ 1) * SLOT, tn2 * BN + half * (BN / 2) + nc * W,
                                tm2 * BM + q * 32);
                    pend_slot = (int)(s ^ 1);
                    pend_par = ((g + 1) >> 1) & 1;
                }
            }
            uint32_t r[32];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + half * (BN / 2) + ch * W;
            if constexpr (W == 32)
                tmem_ld32_nowait(taddr, r);
            else
                tmem_ld16_nowait(taddr, r);
            float v[32];
            if (p.bias) {
                if (p.vec && x + W <= p.N) {
#pragma unroll
                    for (int i = 0; i < W / 4; ++i) {
                        float4 b = ld4(p.bias + x + 4 * i);
                        v[4 * i] = b.x; v[4 * i + 1] = b.y; v[4 * i + 2] = b.z; v[4 * i + 3] = b.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < W; ++i) v[i] = x + i < p.N ? p.bias[x + i] : 0.f;
                }
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i) v[i] = 0.f;
            }
            tmem_wait_ld(r);
#pragma unroll
            for (int i = 0; i < W; ++i) v[i] += __uint_as_float(r[i]);

            if (p.ce_mode == CE_LSE) {
                // online log-sum-exp of this row over its valid columns (log2 units), and the
                // target's logit when it falls in this chunk
                const int nv = min(W, p.N - x);
                float cm = -INFINITY;
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (i < nv) cm = fmaxf(cm, v[i] * LOG2E_F);
                if (cm > ce_m) {
                    ce_s *= ex2_hw(ce_m - cm);
                    ce_m = cm;
                }
                float cs = 0.f;
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (i < nv) cs += ex2_hw(fmaf(v[i], LOG2E_F, -ce_m));
                ce_s += cs;
                const int64_t tc = (int64_t)ce_t - p.ce_col0 - x;
                if (tc >= 0 && tc < nv) {
                    float tv = v[0];
#pragma unroll
                    for (int i = 1; i < W; ++i)
                        if (i == tc) tv = v[i];
                    p.ce_tgt_logit[y + lane] = tv;
                }
                continue;
            }
            if (p.ce_mode == CE_DLOGITS) {
                // (dloss / rows) * (softmax - one-hot) of this row's logits
                const int64_t tc = (int64_t)ce_t - p.ce_col0 - x;
#pragma unroll
                for (int i = 0; i < W; ++i) {
                    const float pr = ex2_hw(fmaf(v[i], LOG2E_F, -ce_l2));
                    v[i] = ce_g * (pr - (i == tc ? 1.f : 0.f));
                }
            }

            if (has_in) {
                if (!__all_sync(0xffffffffu, mbar_wait(&inbar[s], (g >> 1) & 1, abort_flag, WAIT_NS))) {
                    ok = false;
                    break;
                }
                if (lane == 0 && pend_slot == (int)s) pend_slot = -1;
                float in[32];
                slot_read<TC>(slots + s * SLOT, lane, in);
                if (p.in_kind == IN_RES) {
#pragma unroll
                    for (int i = 0; i < W; ++i) v[i] += in[i];
                } else if (p.in_kind == IN_AUX) {
                    if (p.fast_act) {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[i] *= gelu_grad_hw(in[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[i] *= gelu_tanh_grad(in[i]);
                    }
                } else {  // IN_C: accumulate by load
#pragma unroll
                    for (int i = 0; i < W; ++i) v[i] += in[i];
                }
                __syncwarp();  // every lane has read its row before the slot is overwritten
                slot_write<TC>(slots + s * SLOT, lane, v);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (p.reduce_out)
                        tma_reduce_add_2d(mp.C, slots + s * SLOT, x, y);
                    else
                        tma_store_2d(mp.C, slots + s * SLOT, x, y);
                    bulk_commit();
                }
            } else {
                // up to three planes (GELU pre-activation, C, C's low plane), each through the
                // slot whose previous store has finished reading it
                if (p.out_aux) {
                    const uint32_t sl = kst++ & 1;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    slot_write<TC>(slots + sl * SLOT, lane, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(mp.aux, slots + sl * SLOT, x, y);
                        bulk_commit();
                    }
                    if (p.fast_act) {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[i] = gelu_hw(v[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[i] = gelu_tanh(v[i]);
                    }
                }
                {
                    const uint32_t sl = kst++ & 1;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    slot_write<TC>(slots + sl * SLOT, lane, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (p.reduce_out)
                            tma_reduce_add_2d(mp.C, slots + sl * SLOT, x + cxs, y + cys);
                        else
                            tma_store_2d(mp.C, slots + sl * SLOT, x + cxs, y + cys);
                        bulk_commit();
                    }
                }
                if (p.out_lo) {
#pragma unroll
                    for (int i = 0; i < W; ++i) v[i] -= __bfloat162float(__float2bfloat16_rn(v[i]));
                    const uint32_t sl = kst++ & 1;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    slot_write<TC>(slots + sl * SLOT, lane, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(mp.lo, slots + sl * SLOT, x, y);
                        bulk_commit();
                    }
                }
            }
        }
        if (p.ce_mode == CE_LSE && ok && y + lane < p.M)
            p.ce_part[(int64_t)(y + lane) * p.ce_nparts + 2 * tn + half] = make_float2(ce_m, ce_s);
        release_accumulator(p, &tempty[buf], lane);
    }
    if (lane == 0) {
        if (pend_slot >= 0) mbar_wait(&inbar[pend_slot], pend_par, nullptr, DRAIN_NS);
        bulk_wait_all();
    }
    __syncwarp();
    return ok;
}

// F32OP: the operands are float32 containers of TF32 values (K-major, hi and lo planes; SPLIT
// is 3): kind::tf32 MMAs, 32-deep K slices of the same 128-byte rows.
template <typename TC, int SPLIT, bool F32OP>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA_lo, const __grid_constant__ CUtensorMap tmB_lo,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmAux,
                   const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmLo,
                   const TcParams p) {
    using SC = StageCfg<SPLIT>;
    constexpr int STAGES = SC::STAGES;
    constexpr bool PAIR = SC::PAIR;
    constexpr int BKE = F32OP ? BK / 2 : BK;  // K elements per 128-byte row of a stage
    static_assert(!F32OP || (SPLIT == 3 && !PAIR), "TF32 operands come as hi and lo planes");
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
    uint64_t* inbars = bars + 2 * STAGES + 5;  // 2 per epilogue warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 21);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 22);

    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int units = (SC::MC ? p.tiles_m4 : PAIR ? p.tiles_m2 : p.tiles_m) * p.tiles_n * p.splits * p.nz;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const uint32_t prank = rank & 1u, leader = rank & ~1u;  // rank within the pair, the pair's even CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], SC::MC ? 2 : 1);  // with multicast both pairs read every stage
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], PAIR ? 16 : 8);  // one arrival per epilogue warp (of both CTAs)
        }
        mbar_init(drain, 1);
        for (int i = 0; i < 16; ++i) mbar_init(&inbars[i], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        if (PAIR)
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
        else
            tmem_alloc(tmem_slot, TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // the peer's barriers are initialised before anything arrives on them
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
            for (int u = unit_first(p); u < units && ok; u += unit_step(p)) {
                int tm, tn, kb0, kb1;
                unit_coords<F32OP>(p, u, tm, tn, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    int s = it % STAGES;
                    uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, WAIT_NS)) {
                        ok = false;
                        break;
                    }
                    // a pair's stage is complete when both CTAs' copies have landed: all of them
                    // count on the even CTA's full[s], which the even CTA arms for both
                    const uint32_t fb = PAIR ? mapa_shared(saddr(&full[s]), leader) : 0u;
                    if (!PAIR || prank == 0) mbar_expect_tx(&full[s], PAIR ? 2 * SC::STAGE : SC::STAGE);
                    auto load = [&](const CUtensorMap* map, void* dst, int x, int y) {
                        if (PAIR)
                            tma_load_2d_pair(map, fb, dst, x, y);
                        else
                            tma_load_2d(map, &full[s], dst, x, y);
                    };
                    uint8_t* a = smem + s * SC::STAGE;
                    uint8_t* b = a + SC::A_SLOT;
                    const int zl = unit_z<F32OP>(p, u);
                    const int axs = zshift<F32OP>(p, 0, 0, zl), ays = zshift<F32OP>(p, 0, 1, zl);
                    const int bxs = zshift<F32OP>(p, 1, 0, zl), bys = zshift<F32OP>(p, 1, 1, zl);
#pragma unroll
                    for (int pl = 0; pl < (SC::A_LO ? 2 : 1); ++pl) {
                        const CUtensorMap* ma = pl ? &tmA_lo : &tmA;
                        uint8_t* dst = a + pl * A_BYTES;
                        if (F32OP || p.a_kmajor) {
                            load(ma, dst, kb * BKE + axs, tm * BM + ays);
                        } else {
                            load(ma, dst, tm * BM, kb * BK);
                            load(ma, dst + 8192, tm * BM + 64, kb * BK);
                        }
                    }
#pragma unroll
                    for (int pl = 0; pl < (SC::B_LO ? 2 : 1); ++pl) {
                        const CUtensorMap* mb = pl ? &tmB_lo : &tmB;
                        uint8_t* dst = b + pl * SC::B_TILE;
                        // this CTA's columns of the tile's B (all of them, or its half in a pair)
                        constexpr int BNC = (int)(SC::B_TILE / (BK * 2));
                        const int n0 = tn * BN + (int)prank * BNC;
                        if constexpr (SC::MC) {
                            // this CTA's B columns in two 64-column halves: it loads half `pair
                            // index` for itself and the same CTA of the other pair
                            const int j = (int)(rank >> 1);
                            const uint16_t mask = (uint16_t)((1u << rank) | (1u << (rank ^ 2u)));
                            if (p.b_kmajor)
                                tma_load_2d_pair_mc(mb, fb, dst + j * 8192, kb * BK, n0 + 64 * j, mask);
                            else
                                tma_load_2d_pair_mc(mb, fb, dst + j * 8192, n0 + 64 * j, kb * BK, mask);
                        } else if (F32OP || p.b_kmajor) {
                            load(mb, dst, kb * BKE + bxs, n0 + bys);
                        } else {
#pragma unroll
                            for (int j = 0; j < BNC / 64; ++j) load(mb, dst + j * 8192, n0 + 64 * j, kb * BK);
                        }
                    }
                    issued_ph[s] = (int)ph;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                report(p.err, GK_ERR_TIMEOUT);
                // let this CTA's copies in flight land before shared memory is released (the odd
                // CTA of a pair cannot see their completion: it gives them a millisecond)
                if (PAIR && prank != 0) {
                    const uint64_t t0 = globaltimer();
                    while (globaltimer() - t0 < 1000000ull) {
                    }
                } else {
                    for (int s = 0; s < STAGES; ++s)
                        if (issued_ph[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_ph[s], nullptr, DRAIN_NS);
                }
            }
        }
    } else if (PAIR && warp == 1 && prank != 0) {
        // odd CTA of a pair: the even CTA issues the MMAs
    } else if (warp == 1) {
        // The whole warp walks the loop in step (so the descriptors stay warp-uniform) and one
        // elected lane issues the MMAs and commits. In a pair this is the even CTA, issuing
        // 256-row MMAs whose commits reach both CTAs' barriers.
        const uint32_t idesc = F32OP ? instr_desc_tf32(BM, BN)
                                     : instr_desc_bf16(!p.a_kmajor, !p.b_kmajor, PAIR ? 2 * BM : BM, BN);
        // per 16-deep K step: K-major operands advance 32 bytes inside the swizzled row,
        // MN-major operands advance two 8-row core-matrix groups (2 x 1024 bytes)
        const uint32_t a_step = p.a_kmajor ? 32u : 2048u;
        const uint32_t b_step = p.b_kmajor ? 32u : 2048u;
        const uint32_t a_lbo = p.a_kmajor ? 16u : 8192u, b_lbo = p.b_kmajor ? 16u : 8192u;
        uint32_t it = 0, j = 0;
        bool ok = true, issued = false;
        for (int u = unit_first(p); u < units && ok; u += unit_step(p), ++j) {
            int tm, tn, kb0, kb1;
            unit_coords<F32OP>(p, u, tm, tn, kb0, kb1);
            uint32_t buf = j & 1, aph = (j >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&tempty[buf], aph ^ 1, abort_flag, WAIT_NS))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t d_tmem = tmem_base + buf * BN;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                int s = it % STAGES;
                uint32_t ph = (it / STAGES) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, abort_flag, WAIT_NS))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = saddr(smem + s * SC::STAGE), b0 = a0 + SC::A_SLOT;
                const uint64_t ad0 = smem_desc(a0, a_lbo, 1024), bd0 = smem_desc(b0, b_lbo, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = desc_add(ad0, k * a_step), bd = desc_add(bd0, k * b_step);
                        const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
                        if constexpr (F32OP) {
                            // 3xTF32: A_hi B_hi + A_hi B_lo + A_lo B_hi (A_lo B_lo, about 2^-22
                            // relative, is dropped)
                            umma_tf32(d_tmem, ad, bd, idesc, acc);
                            umma_tf32(d_tmem, ad, desc_add(bd0, B_BYTES + k * b_step), idesc, 1u);
                            umma_tf32(d_tmem, desc_add(ad0, A_BYTES + k * a_step), bd, idesc, 1u);
                        } else if (PAIR) {
                            umma_bf16_pair(d_tmem, ad, bd, idesc, acc);
                        } else {
                            umma_bf16(d_tmem, ad, bd, idesc, acc);
                            // split operands: + A_hi B_lo + A_lo B_hi (the A_lo B_lo term is dropped)
                            if (SC::B_LO) umma_bf16(d_tmem, ad, desc_add(bd0, B_BYTES + k * b_step), idesc, 1u);
                            if (SC::A_LO) umma_bf16(d_tmem, desc_add(ad0, A_BYTES + k * a_step), bd, idesc, 1u);
                        }
                    }
                    // commits track the MMAs of the thread that issues them: same lane, same block
                    if (PAIR) {
                        // the stage is free once every pair that reads it is done with it
                        umma_commit_pair_mc(&empty[s], SC::MC ? 0xF : 3);
                        if (kb == kb1 - 1) umma_commit_pair_mc(&tfull[buf], (uint16_t)(3u << leader));
                    } else {
                        umma_commit(&empty[s]);
                        if (kb == kb1 - 1) umma_commit(&tfull[buf]);
                    }
                }
                __syncwarp();
                issued = true;
            }
        }
        if (!ok) {
            if (elect_one()) {
                *abort_flag = 1;
                report(p.err, GK_ERR_TIMEOUT);
                if (issued) {
                    if (PAIR)
                        umma_commit_pair(drain);
                    else
                        umma_commit(drain);
                    mbar_wait(drain, 0, nullptr, DRAIN_NS);
                }
            }
            __syncwarp();
        }
    } else if (p.tma_epi) {
        EpiMaps mp{&tmC, &tmAux, &tmLo,
                   p.in_kind == IN_C ? &tmC : p.in_kind == IN_RES ? &tmR : p.in_kind == IN_AUX ? &tmAux : nullptr};
        uint8_t* slots = reinterpret_cast<uint8_t*>(epi_stage) + (warp - 2) * 2 * SLOT;
        if (!epilogue_tma<TC, F32OP>(p, mp, slots, inbars + 2 * (warp - 2), tfull, tempty, abort_flag, tmem_base, warp, lane,
                              units)) {
            *abort_flag = 1;
            report(p.err, GK_ERR_TIMEOUT);
        }
    } else {
        // epilogue warps 2..9; a warp may read TMEM lanes 32 * (warp % 4) .. + 31; two warps
        // share each lane quarter and take alternate halves of the tile's columns
        int q = warp & 3;
        int half = (warp - 2) >> 2;
        uint32_t j = 0;
        for (int u = unit_first(p); u < units; u += unit_step(p), ++j) {
            int tm, tn, kb0, kb1;
            unit_coords<F32OP>(p, u, tm, tn, kb0, kb1);
            uint32_t buf = j & 1, aph = (j >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull[buf], aph, abort_flag, WAIT_NS))) {
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
                    const int c = lane & 7;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float4 v[4];
                        EpiIn e[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            int rr = (half * 4 + i) * 4 + (lane >> 3);
                            v[i] = *reinterpret_cast<const float4*>(stg + rr * 32 + ((c ^ (rr & 7)) << 2));
                            epi_load<TC>(p, mrow0 + rr, n0 + c * 4, e[i]);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            epi_finish<TC>(p, mrow0 + (half * 4 + i) * 4 + (lane >> 3), n0 + c * 4, v[i], e[i]);
                    }
                }
                __syncwarp();
            }
            release_accumulator(p, &tempty[buf], lane);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // no MMA, commit or arrival of the pair is still in flight
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (PAIR) cluster_sync();
}

struct Maps {
    CUtensorMap a, b, al, bl, c, aux, r, lo;
};

template <typename TC, int SPLIT, bool F32OP = false>
void launch_one(gk_ctx* ctx, int grid, const Maps& m, const TcParams& p) {
    static bool attr = false;
    constexpr size_t smem = StageCfg<SPLIT>::SMEM;
    if (!attr) {
        cudaFuncSetAttribute(gemm_tc_kernel<TC, SPLIT, F32OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr = true;
    }
    if constexpr (StageCfg<SPLIT>::PAIR) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = ctx->stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = StageCfg<SPLIT>::MC ? 4 : 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, gemm_tc_kernel<TC, SPLIT, false>, m.a, m.b, m.al, m.bl, m.c, m.aux, m.r, m.lo, p);
    } else {
        gemm_tc_kernel<TC, SPLIT, F32OP><<<grid, THREADS, smem, ctx->stream>>>(m.a, m.b, m.al, m.bl, m.c, m.aux, m.r,
                                                                                m.lo, p);
    }
}

template <typename TC>
void launch_split(gk_ctx* ctx, int split, int grid, const Maps& m, const TcParams& p) {
    switch (split) {
        case 0: launch_one<TC, 0>(ctx, grid, m, p); break;
        case 1: launch_one<TC, 1>(ctx, grid, m, p); break;
        case 2: launch_one<TC, 2>(ctx, grid, m, p); break;
        case 3: launch_one<TC, 3>(ctx, grid, m, p); break;
        case PAIR_MODE: launch_one<TC, PAIR_MODE>(ctx, grid, m, p); break;
        default: launch_one<TC, PAIR4_MODE>(ctx, grid, m, p); break;
    }
}

// How many CTA pairs of the pair kernel can be resident at once (clusters need both SMs of a
// pair free); 0 if the query fails.
template <typename TC, int MODE = PAIR_MODE>
int max_pairs() {
    static int n = -1;
    if (n < 0) {
        constexpr size_t smem = StageCfg<MODE>::SMEM;
        constexpr int CS = StageCfg<MODE>::MC ? 4 : 2;
        cudaFuncSetAttribute(gemm_tc_kernel<TC, MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        cudaFuncSetAttribute(gemm_tc_kernel<TC, MODE, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(CS);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = CS;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int c = 0;
        n = cudaOccupancyMaxActiveClusters(&c, gemm_tc_kernel<TC, MODE, false>, &cfg) == cudaSuccess ? c : 0;
        cudaGetLastError();
    }
    return n;
}

// Decide whether the TMA epilogue takes this GEMM and build its tensor maps: every plane
// (C, the GELU pre-activation, the residual, C's low plane) has C's element type, 16-byte
// aligned bases and strides, and at most one plane is read.
bool setup_tma_epilogue(const Gemm& g, TcParams& p, Maps& m) {
    if (g.ce_mode == CE_LSE) {  // nothing is stored through TMA; rows and columns come from the tile
        p.reduce_out = p.out_aux = p.out_lo = 0;
        p.in_kind = IN_NONE;
        return g.ce_tgt && g.ce_part && g.ce_tgt_logit && !g.bias && !g.residual && g.epi == EPI_NONE &&
               !g.accumulate && !g.c_plane;
    }
    if (g.ce_mode == CE_DLOGITS &&
        (g.c_dtype != GK_BF16 || !g.ce_tgt || !g.ce_lse || g.bias || g.residual || g.epi != EPI_NONE ||
         g.accumulate || g.c_plane))
        return false;
    const bool bf = g.c_dtype == GK_BF16;
    if (g.c_dtype != GK_BF16 && g.c_dtype != GK_F32) return false;
    const int esz = bf ? 2 : 4, W = 64 / esz;
    auto ok_plane = [&](const void* base, int64_t ld) {
        return base && aligned16(base) && (ld * esz) % 16 == 0 && ld >= g.N;
    };
    if (!ok_plane(g.C, g.ldc)) return false;
    if (g.bias && !aligned16(g.bias)) return false;
    if (g.epi != EPI_NONE && (!g.aux || g.aux_dtype != g.c_dtype || !ok_plane(g.aux, g.ldaux))) return false;
    if (g.residual && (bf || !ok_plane(g.residual, g.ldr))) return false;
    if (g.c_plane && (!bf || (g.c_plane * 2) % 16 != 0)) return false;
    p.reduce_out = g.accumulate && !bf && !g.c_plane;
    int inputs = (g.residual ? 1 : 0) + (g.epi == EPI_DGELU ? 1 : 0) + (g.accumulate && !p.reduce_out ? 1 : 0);
    // a chunk with an input plane is rewritten in place: one output plane only
    if (inputs > 1 || (inputs == 1 && (g.epi == EPI_GELU || g.c_plane))) return false;
    p.in_kind = g.residual ? IN_RES : g.epi == EPI_DGELU ? IN_AUX : (g.accumulate && !p.reduce_out) ? IN_C : IN_NONE;
    p.out_aux = g.epi == EPI_GELU;
    p.out_lo = g.c_plane != 0;
    const int64_t cn = g.nz > 1 ? g.c_ext[0] : g.N, cm = g.nz > 1 ? g.c_ext[1] : g.M;
    if (!make_map_epi(&m.c, bf, g.C, cn, cm, g.ldc, W)) return false;
    m.aux = m.r = m.lo = m.c;
    if (g.epi != EPI_NONE && !make_map_epi(&m.aux, bf, g.aux, g.N, g.M, g.ldaux, W)) return false;
    if (g.residual && !make_map_epi(&m.r, false, g.residual, g.N, g.M, g.ldr, W)) return false;
    if (g.c_plane && !make_map_epi(&m.lo, true, static_cast<const __nv_bfloat16*>(g.C) + g.c_plane, g.N, g.M, g.ldc, W))
        return false;
    return true;
}

}  // namespace

gk_status gemm_tc(gk_ctx* ctx, const Gemm& g) {
    const bool f32op = g.tf32;  // TF32 hi / lo planes in float32 containers, K-major
    if (f32op) {
        if (g.ab_dtype != GK_F32 || !g.a_kmajor || !g.b_kmajor || !g.A_lo || !g.B_lo || g.ce_mode != CE_NONE ||
            g.c_dtype != GK_F32 || (g.lda & 3) || (g.ldb & 3) || !aligned16(g.A_lo) || !aligned16(g.B_lo))
            return GK_ERR_UNSUPPORTED;
    } else if (g.ab_dtype != GK_BF16 || (g.lda & 7) || (g.ldb & 7)) {
        return GK_ERR_UNSUPPORTED;
    }
    if (!aligned16(g.A) || !aligned16(g.B)) return GK_ERR_UNSUPPORTED;
    if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.M >= (1ll << 31) || g.N >= (1ll << 31) || g.K >= (1ll << 31))
        return GK_ERR_UNSUPPORTED;
    const int split = (g.A_lo ? 1 : 0) | (g.B_lo ? 2 : 0);
    // CTA pairs (256 x 256 tiles, half of B per CTA) for the single-plane products with at least
    // four 128-row tiles; the split-precision products keep one CTA per tile
    const bool c_f32 = g.ce_mode != CE_LSE && g.c_dtype == GK_F32;
    const bool batched = g.nz > 1;
    if (batched && (g.bias || g.residual || g.accumulate || g.epi != EPI_NONE || g.ce_mode != CE_NONE || g.c_plane ||
                    g.M % BM != 0 || g.N % (64 / (g.c_dtype == GK_F32 ? 4 : 2)) != 0 || g.zh < 1 || g.z0 < 0 ||
                    (int64_t)g.nz * cdiv(g.M, BM) * cdiv(g.N, BN) >= (1ll << 31)))
        return GK_ERR_UNSUPPORTED;
    const int pairs = !batched && split == 0 && cdiv(g.M, BM) >= 4
                          ? (c_f32 ? max_pairs<float>() : max_pairs<__nv_bfloat16>())
                          : 0;
    const bool pair = pairs > 0;
    // clusters of two pairs (B multicast) when there are at least two pair rows of tiles;
    // not for the GELU forward, whose epilogue sets its time (36 clusters of four hold 144
    // SMs against 152 for pairs). Measured at 16384 rows: QKV 49.9 -> 47.7 us, MLP down with
    // residual 64.2 -> 62.1, GELU-backward dX 201 -> 181; GELU forward 84.6 -> 88.7.
    const int quads = pair && cdiv(g.M, BM) >= 8 && g.epi != EPI_GELU
                          ? (c_f32 ? max_pairs<float, PAIR4_MODE>() : max_pairs<__nv_bfloat16, PAIR4_MODE>())
                          : 0;
    const bool mc = quads >= 16;
    CUtensorMap ta, tb;
    bool ok;
    // a batch indexes into whole buffers: their maps span them
    const int64_t ak = batched ? g.a_ext[0] : g.K, am = batched ? g.a_ext[1] : g.M;
    const int64_t bk = batched ? g.b_ext[0] : g.K, bn = batched ? g.b_ext[1] : g.N;
    if (batched && (!f32op || ak <= 0 || am <= 0 || bk <= 0 || bn <= 0 || g.c_ext[0] <= 0 || g.c_ext[1] <= 0))
        return GK_ERR_UNSUPPORTED;
    if (f32op) {
        ok = make_map_f32(&ta, g.A, ak, am, g.lda, BK / 2, BM) && make_map_f32(&tb, g.B, bk, bn, g.ldb, BK / 2, BN);
    } else {
        ok = g.a_kmajor ? make_map(&ta, g.A, g.K, g.M, g.lda, BM) : make_map(&ta, g.A, g.M, g.K, g.lda, 64);
        ok = ok && (g.b_kmajor ? make_map(&tb, g.B, g.K, g.N, g.ldb, mc ? BN / 4 : pair ? BN / 2 : BN)
                               : make_map(&tb, g.B, g.N, g.K, g.ldb, 64));
    }
    if (!ok) return GK_ERR_UNSUPPORTED;
    TcParams p{};
    p.pair = pair ? 1 : 0;
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.tiles_m = (int)cdiv(g.M, BM);
    p.tiles_n = (int)cdiv(g.N, BN);
    p.tiles_m2 = (int)cdiv(p.tiles_m, 2);
    p.mc = mc ? 1 : 0;
    p.tiles_m4 = (int)cdiv(p.tiles_m2, 2);
    // Units run in waves of one per CTA (pair), in unit order. With few column tiles and A the
    // larger operand (M > N: activations against weights, or the LM head's dlogits), the column
    // tiles of a row block go consecutively, so the CTAs that need a block of A rows load it
    // at the same time and A comes from DRAM once; in row order each column tile would stream
    // all of A again.
    p.n_fast = g.M > g.N && p.tiles_n <= 8;
    p.kblocks = (int)cdiv(g.K, f32op ? BK / 2 : BK);
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
    p.nz = batched ? g.nz : 1;
    p.zh = g.zh;
    p.z0 = g.z0;
    for (int o = 0; o < 3; ++o)
        for (int c = 0; c < 2; ++c)
            for (int t = 0; t < 3; ++t) p.zo[o][c][t] = g.zo[o][c][t];
    p.c_plane = g.c_plane;
    p.fast_act = g.c_dtype == GK_BF16 && g.c_plane == 0;
    p.vec = aligned16(g.C) && (g.ldc % 4 == 0) && (!g.bias || aligned16(g.bias)) &&
            (!g.residual || (aligned16(g.residual) && g.ldr % 4 == 0)) &&
            (!g.aux || (aligned16(g.aux) && g.ldaux % 4 == 0)) && (g.c_plane % 4 == 0);
    if ((g.A_lo && (!aligned16(g.A_lo))) || (g.B_lo && !aligned16(g.B_lo))) return GK_ERR_UNSUPPORTED;
    // persistent grid: one CTA per SM, or one pair per resident cluster
    const int slots = mc ? quads : pair ? pairs : ctx->num_sms;
    int64_t tiles = (int64_t)(mc ? p.tiles_m4 : pair ? p.tiles_m2 : p.tiles_m) * p.tiles_n;
    p.splits = 1;
    bool plain_acc = !batched && g.accumulate && g.c_dtype == GK_F32 && !g.bias && !g.residual && g.epi == EPI_NONE;
    if (plain_acc && tiles < slots) {
        int want = (int)cdiv(2 * (int64_t)slots, tiles);
        int maxs = std::max(1, p.kblocks / 4);
        p.splits = std::max(1, std::min(want, maxs));
    }
    p.kbps = (int)cdiv(p.kblocks, p.splits);
    p.splits = (int)cdiv(p.kblocks, p.kbps);
    p.atomic_out = p.splits > 1;
    int64_t units = tiles * p.splits * p.nz;
    int grid = (int)std::min<int64_t>(units, slots) * (mc ? 4 : pair ? 2 : 1);
    const int mode = mc ? PAIR4_MODE : pair ? PAIR_MODE : split;
    Maps m;
    m.a = ta;
    m.b = tb;
    m.al = ta;
    m.bl = tb;
    if (f32op) {
        if (!make_map_f32(&m.al, g.A_lo, ak, am, g.lda, BK / 2, BM) ||
            !make_map_f32(&m.bl, g.B_lo, bk, bn, g.ldb, BK / 2, BN))
            return GK_ERR_UNSUPPORTED;
    } else {
        if (g.A_lo && !(g.a_kmajor ? make_map(&m.al, g.A_lo, g.K, g.M, g.lda, BM)
                                   : make_map(&m.al, g.A_lo, g.M, g.K, g.lda, 64)))
            return GK_ERR_UNSUPPORTED;
        if (g.B_lo && !(g.b_kmajor ? make_map(&m.bl, g.B_lo, g.K, g.N, g.ldb, BN)
                                   : make_map(&m.bl, g.B_lo, g.N, g.K, g.ldb, 64)))
            return GK_ERR_UNSUPPORTED;
    }
    p.ce_mode = g.ce_mode;
    p.ce_nparts = g.ce_nparts;
    p.ce_col0 = g.ce_col0;
    p.ce_tgt = g.ce_tgt;
    p.ce_part = g.ce_part;
    p.ce_tgt_logit = g.ce_tgt_logit;
    p.ce_lse = g.ce_lse;
    p.ce_dloss = g.ce_dloss;
    p.ce_scale = g.ce_scale;
    if (g.ce_mode == CE_LSE) {
        m.c = m.aux = m.r = m.lo = ta;
        p.tma_epi = setup_tma_epilogue(g, p, m);
        if (!p.tma_epi) return GK_ERR_UNSUPPORTED;
        launch_split<__nv_bfloat16>(ctx, mode, grid, m, p);  // 32-column chunks; nothing is stored
        return launched(ctx, "gemm_tc");
    }
    p.tma_epi = setup_tma_epilogue(g, p, m);
    if (!p.tma_epi && (g.ce_mode != CE_NONE || batched)) return GK_ERR_UNSUPPORTED;
    if (!p.tma_epi) {
        m.c = m.aux = m.r = m.lo = ta;
        p.in_kind = IN_NONE;
        p.reduce_out = p.out_aux = p.out_lo = 0;
    }
    if (f32op)
        launch_one<float, 3, true>(ctx, grid, m, p);
    else if (g.c_dtype == GK_F32)
        launch_split<float>(ctx, mode, grid, m, p);
    else
        launch_split<__nv_bfloat16>(ctx, mode, grid, m, p);
    return launched(ctx, "gemm_tc");
}

}  // namespace gk
