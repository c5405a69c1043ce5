// tcgen05 (kind::tf32) GEMM -- not built yet: every shape reports "unsupported".
#include "gemm.cuh"

namespace spco {

bool gemm_tc_supported(int64_t, int64_t, int64_t, Operand, Operand) { return false; }

int gemm_tc(int64_t, int64_t, int64_t, Operand, Operand, const Epilogue &, cudaStream_t) {
    return fail(SPECOPTIM_ERR_NOT_IMPLEMENTED, "tcgen05 GEMM not built");
}

}  // namespace spco
