// SVD refresh of the anchor momentum (svd.cu).
#pragma once

#include "common.cuh"

namespace spco {

// One matrix of a (batched) refresh.
struct SvdJob {
    const float *M;        // m x n anchor momentum
    int m, n;
    float *U, *s, *V, *d;  // outputs: U m x r, s r, V n x r, d r (written only on success)
    float *work;           // svd_workspace_floats(m, n) floats, 16-byte aligned
    const float *warm;     // previous short-side factor (r x r) to start from, or null
    float tau, tol;
    int max_sweeps;
    int inner_sweeps;      // Jacobi sweeps per 64 x 64 subproblem and round
    int sweeps;            // out: Jacobi sweeps run
    int status;            // out: SPECOPTIM_OK or SPECOPTIM_ERR_NOT_CONVERGED
};

size_t svd_workspace_floats(int m, int n);
// Refreshes up to 16 matrices; their Jacobi rounds share kernel launches.
int svd_refresh_batch(SvdJob *jobs, int count, cudaStream_t stream);

// The same refresh in two phases.  start: the Gram matrices and the Jacobi
// sweeps of every job on the library's own streams, ordered after the work
// already on `stream`; with `async` a library thread runs the sweep loop (it
// waits on each sweep's convergence test) and the call returns at once.
// complete: waits (host) for that loop, orders `stream` after its kernels,
// writes the factors of the converged jobs on `stream`, fills jobs[i].sweeps
// and .status and frees the run.  One run at a time per process.
struct SvdRun;
int svd_refresh_start(const SvdJob *jobs, int count, cudaStream_t stream, bool async, SvdRun **out);
int svd_refresh_complete(SvdRun *run, SvdJob *jobs, cudaStream_t stream);

}  // namespace spco
