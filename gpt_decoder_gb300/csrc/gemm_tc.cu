// Tensor-core GEMM for sm_103a (tcgen05 + TMA + TMEM). Not yet enabled: every call falls
// back to the CUDA-core kernel.
#include "gemm.cuh"

namespace gk {

gk_status gemm_tc(gk_ctx* ctx, const Gemm& g) {
    (void)ctx;
    (void)g;
    return GK_ERR_UNSUPPORTED;
}

}  // namespace gk
