// SVD refresh of the anchor momentum (svd.cu).
#pragma once

#include "common.cuh"

namespace spco {

struct SvdArgs {
    const float *M;  // m x n anchor momentum
    int m, n;
    float *U, *s, *V, *d;  // outputs: U m x r, s r, V n x r, d r (written only on success)
    float *work;           // svd_workspace_floats(r) floats, 16-byte aligned
    float tau;
    int max_sweeps;
    float tol;
};

size_t svd_workspace_floats(int m, int n);
int svd_refresh_run(const SvdArgs &args, cudaStream_t stream, int *sweeps_out);

}  // namespace spco
