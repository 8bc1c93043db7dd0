// Internal GEMM interface: C[M,N] (=|+=) epi(sum_k A(m,k) B(k,n) + bias[n] + residual[m,n]);
// with `accumulate` the epilogue's result is added to C (C_old + epi(...)).
//
// Operand majorness covers every product of the decoder step without transpose passes:
//   A(m,k) = A[m*lda + k] when a_kmajor, else A[k*lda + m];
//   B(k,n) = B[n*ldb + k] when b_kmajor, else B[k*ldb + n].
// A bf16 operand may come with a low plane (split bf16, about 16 significant bits); see Gemm.
// Epilogues: EPI_GELU stores the pre-activation v to `aux` and gelu(v) to C; EPI_DGELU
// stores v * gelu'(aux) (the backward of a GELU fused into the GEMM producing its input
// gradient).
#pragma once

#include "common.cuh"

namespace gk {

enum Epi { EPI_NONE = 0, EPI_GELU = 1, EPI_DGELU = 2 };

struct Gemm {
    int64_t M = 0, N = 0, K = 0;
    const void* A = nullptr;
    int64_t lda = 0;
    bool a_kmajor = true;
    const void* B = nullptr;
    int64_t ldb = 0;
    bool b_kmajor = true;
    int ab_dtype = GK_F32;
    void* C = nullptr;
    int64_t ldc = 0;
    int c_dtype = GK_F32;
    bool accumulate = false;
    const float* bias = nullptr;
    const float* residual = nullptr;
    int64_t ldr = 0;
    int epi = EPI_NONE;
    void* aux = nullptr;
    int64_t ldaux = 0;
    int aux_dtype = GK_F32;
    // split-bf16 operands: a low plane (value - bf16(value)) with the same layout as A / B;
    // the product then adds A_hi B_lo + A_lo B_hi to A_hi B_hi (bf16 operands only)
    const void* A_lo = nullptr;
    const void* B_lo = nullptr;
    // > 0 with bf16 C: C's low plane (v - bf16(v)) is also written, at C + c_plane elements
    int64_t c_plane = 0;
    // tf32: A, A_lo, B, B_lo are float32 containers of TF32 values, hi and lo planes of float32
    // operands (value = hi + lo), both K-major; the tensor-core kernel then adds the three
    // products A_hi B_hi + A_hi B_lo + A_lo B_hi (3xTF32)
    bool tf32 = false;
    // nz > 1: nz independent products of the same shape (a batch), all through the same tensor
    // maps. For product zl (global index zg = z0 + zl) the TMA coordinates of operand o (0 = A,
    // 1 = B, 2 = C) are shifted along x (inner) and y (outer) by
    //   (zg % zh) * zo[o][c][0] + (zg / zh) * zo[o][c][1] + zl * zo[o][c][2]   (c = 0: x, 1: y),
    // e.g. zg = batch row * heads + head. Plain stores only (no bias, residual, accumulate or
    // epilogue function); M a multiple of 128 and N of the store chunk, so that no tile crosses
    // into a neighbouring product.
    int nz = 1, zh = 1, z0 = 0;
    int zo[3][2][3] = {};
    // with nz > 1: the extents (inner, outer) of the whole buffers A, B and C that the products
    // index into, for their tensor maps
    int64_t a_ext[2] = {0, 0}, b_ext[2] = {0, 0}, c_ext[2] = {0, 0};
    // Softmax cross-entropy fused into a vocabulary-projection epilogue (tensor-core kernel,
    // TMA epilogue only). Column n of this GEMM is vocabulary entry ce_col0 + n, and
    // ce_tgt[m] is row m's target entry.
    //   CE_LSE: C is not written; per row and (256-column tile, column half) the epilogue
    //     leaves (max, sum of 2^(v log2 e - max)) in ce_part[m * ce_nparts + 2 * tile + half]
    //     (max in log2 units) and the target's logit in ce_tgt_logit[m].
    //   CE_DLOGITS: C (bf16) = (*ce_dloss * ce_scale) * (exp(v - ce_lse[m]) - [n == target]).
    int ce_mode = 0;
    const int32_t* ce_tgt = nullptr;
    int64_t ce_col0 = 0;
    float2* ce_part = nullptr;
    int ce_nparts = 0;
    float* ce_tgt_logit = nullptr;
    const float* ce_lse = nullptr;
    const float* ce_dloss = nullptr;
    float ce_scale = 1.f;
};

enum CeMode { CE_NONE = 0, CE_LSE = 1, CE_DLOGITS = 2 };

// CUDA-core (SIMT) kernel: float32 or bfloat16 operands, float32 FMA accumulation.
gk_status gemm_simt(gk_ctx* ctx, const Gemm& g);
// Tensor-core kernel (tcgen05 + TMA + TMEM), bfloat16 operands, float32 accumulation.
// Returns GK_ERR_UNSUPPORTED for shapes or alignments it does not take.
gk_status gemm_tc(gk_ctx* ctx, const Gemm& g);
// Dispatch by operand type, arithmetic mode and shape.
gk_status gemm(gk_ctx* ctx, const Gemm& g);
// Float32 operands (either majorness) in 3xTF32 on the tensor cores: each operand is split
// into TF32 hi / lo planes (K-major, in the context's workspace, in chunks of the output or of
// K when the whole does not fit), then gemm_tc adds the three products.
gk_status gemm_3xtf32(gk_ctx* ctx, const Gemm& g);
// TF32 hi / lo planes [R][ldp] of rows row0 .. row0 + R - 1 and K range k0 .. k0 + kc - 1 of a
// float32 operand (K-major: element (i, k) at src[i * ld + k]; else at src[k * ld + i]).
gk_status split_planes(gk_ctx* ctx, const float* src, int64_t ld, bool kmajor, int64_t row0, int64_t k0, int64_t R,
                       int64_t kc, float* hi, float* lo, int64_t ldp);

// x = hi + lo with hi = tf32(x) (round to nearest, ties away from zero) and lo = tf32(x - hi);
// x - hi is exact in float32.
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
__device__ __forceinline__ void tf32_split(float x, float& hi, float& lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - hi);
}

// Faithful-mode (float32) causal attention with its products as batched 3xTF32 tensor-core
// products (T a multiple of 128, head size a multiple of 32); GK_ERR_UNSUPPORTED for other shapes
// or when the context's workspace cannot hold one head's score buffers (the float32 CUDA-core
// kernels then run).
gk_status attn_fwd_3xtf32(gk_ctx* ctx, const float* qkv, float* y, float* lse, int B, int T, int H, int hs);
gk_status attn_bwd_3xtf32(gk_ctx* ctx, const float* qkv, const float* y, const float* lse, const float* dy, float* dqkv,
                          int B, int T, int H, int hs);
// Tensor-core causal attention forward (bf16 q/k/v, head size 64); GK_ERR_UNSUPPORTED otherwise.
gk_status attn_fwd_tc(gk_ctx* ctx, const void* qkv, void* y, float* lse, int B, int T, int H, int hs);
// Tensor-core causal attention backward (bf16, head size 64); GK_ERR_UNSUPPORTED otherwise.
gk_status attn_bwd_tc(gk_ctx* ctx, const void* qkv, const void* y, const float* lse, const void* dy, void* dqkv,
                      int B, int T, int H, int hs);

// dst[n] += sum over rows of src[r, n] (deterministic, float32 result).
gk_status colsum_add(gk_ctx* ctx, const void* src, int64_t ld, int dtype, int64_t rows, int64_t cols, float* dst);

}  // namespace gk
