// C-ABI of the spectral-corrected optimizer ("Communication-Efficient LLM
// Adaptation over Decentralized GPU Meshes", key designs 2 and 3): handle
// lifecycle, anchor EMA, SVD refresh, and the step orchestration.
//
// Step (key design 3, projection + blend equations, then AdamW).  The filter
//   G_filt = U diag(d) U^T G V diag(d) V^T = P_L G P_R,
//   P_L = U diag(d) U^T (m x m),  P_R = V diag(d) V^T (n x n),
// is evaluated in the association that needs the fewest flops for the shape;
// the projectors it uses are formed once per SVD refresh (fp32-accurate
// 3xTF32 products).  Every operand is stored K-contiguous (the layout the
// tcgen05 path reads with TMA; the SIMT path reads the same buffers):
//   m = n:            T^T = P_R G^T     (n x m, K = n)      G read as the K-contiguous operand
//                     Gf  = P_L T       (m x n, K = m)      blend + AdamW in the epilogue
//   m > n (r = n):    G^T = transpose(G)
//                     T1  = U^T G       (r x n, K = m)
//                     T2^T= P_R T1^T D  (n x r, K = n)      diag(d) on the columns in the epilogue
//                     Gf  = U T2        (m x n, K = r)      blend + AdamW in the epilogue
//   m < n (r = m):    T1^T= V^T G^T     (r x m, K = n)
//                     T2  = P_L T1 D    (m x r, K = m)      diag(d) on the columns in the epilogue
//                     Gf  = T2 V^T      (m x n, K = r)      blend + AdamW in the epilogue
// Flops: 4 n^3 (square), 4 m n^2 + 2 n^3 (tall), 4 m^2 n + 2 m^3 (wide), against
// 8 n^3 and 4 r^2 max(m,n) + 4 r^3 for U^T G V and U X V^T in sequence.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "elementwise.cuh"
#include "gemm.cuh"
#include "svd.cuh"

struct specoptim {
    specoptim_config cfg;
    int m, n, r;
    bool tall;
    int64_t t;
    float *M, *U, *s, *V, *d, *m1, *m2;
    float *Uo, *UTo, *Vo, *VTo;  // GEMM operand copies of the factors (TF32-rounded on the TC path)
    float *PL, *PR;              // projectors U diag(d) U^T (m <= n) and V diag(d) V^T (m >= n)
    float *ws_g, *ws_a, *ws_x;   // step workspace: G^T (tall), T1/Z^T or T^T/Y, Xf
    float *ws_svd;
    bool have_factors;
    struct PendingRefresh *pending;  // refresh begun and not yet ended (svd_refresh_begin / _end)
};

// A refresh between specoptim_svd_refresh_begin and _end: its handles in call
// order, their jobs and the run of svd.cu.
struct PendingRefresh {
    int count;
    specoptim_t *h[16];
    spco::SvdJob jobs[16];
    spco::SvdRun *run;
};

namespace spco {

static thread_local std::string g_last_error;

void set_error(const std::string &msg) { g_last_error = msg; }
void clear_error() { g_last_error.clear(); }

static __device__ unsigned g_timeout_flag;

unsigned *device_flag_ptr() {
    static unsigned *ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_timeout_flag) == cudaSuccess) ptr = static_cast<unsigned *>(p);
    });
    return ptr;
}

int check_device_flag(cudaStream_t st) {
    if (int rc = bind_device()) return rc;
    unsigned *p = device_flag_ptr();
    if (!p) return SPECOPTIM_OK;
    unsigned v = 0;
    SPECOPTIM_CUDA(cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, st));
    SPECOPTIM_CUDA(cudaStreamSynchronize(st));
    if (v) {
        unsigned zero = 0;
        cudaMemcpyAsync(p, &zero, sizeof(zero), cudaMemcpyHostToDevice, st);
        cudaStreamSynchronize(st);
        if (v & 0x80000000u)  // only the checked build (-DSPECOPTIM_CHECK) sets bit 31
            return fail(SPECOPTIM_ERR_BOUNDS, "an index check of the checked build failed (site " +
                                                  std::to_string(v & 0x7FFFFFFFu) + ")");
        return fail(SPECOPTIM_ERR_TIMEOUT, "a bounded device-side wait gave up (code " +
                                               std::to_string(v) + ")");
    }
    return SPECOPTIM_OK;
}

int transpose_run(const float *src, float *dst, int rows, int cols, bool round, cudaStream_t st);
int gemm_tc(int64_t M, int64_t N, int64_t K, Operand A, Operand B, const Epilogue &epi,
            cudaStream_t stream);
bool gemm_tc_supported(int64_t M, int64_t N, int64_t K, Operand A, Operand B);

}  // namespace spco

using namespace spco;

namespace {

int validate_cfg(const specoptim_config *c) {
    if (!c) return fail(SPECOPTIM_ERR_INVALID_ARG, "config is null");
    if (c->m < 1 || c->n < 1) return fail(SPECOPTIM_ERR_INVALID_ARG, "m and n must be >= 1");
    if ((int64_t)c->m * c->n > (int64_t)1 << 34) return fail(SPECOPTIM_ERR_INVALID_ARG, "matrix too large");
    if (!(c->tau_p > 0.f) || !std::isfinite(c->tau_p))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "tau_p must be finite and > 0");
    if (!(c->alpha >= 0.f && c->alpha <= 1.f)) return fail(SPECOPTIM_ERR_INVALID_ARG, "alpha must be in [0,1]");
    if (!(c->beta_anc >= 0.f && c->beta_anc <= 1.f))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "beta_anc must be in [0,1]");
    if (!(c->beta1 >= 0.f && c->beta1 < 1.f) || !(c->beta2 >= 0.f && c->beta2 < 1.f))
        return fail(SPECOPTIM_ERR_INVALID_ARG, "AdamW betas must be in [0,1)");
    if (!(c->eps >= 0.f)) return fail(SPECOPTIM_ERR_INVALID_ARG, "eps must be >= 0");
    if (c->precision != SPECOPTIM_PREC_TF32 && c->precision != SPECOPTIM_PREC_FP32)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "unknown precision");
    if (c->svd_max_sweeps < 1) return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_max_sweeps must be >= 1");
    if (!(c->svd_tol >= 0.f)) return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_tol must be >= 0");
    if (c->svd_inner_sweeps < 1 || c->svd_inner_sweeps > 16)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_inner_sweeps must be in [1, 16]");
    return SPECOPTIM_OK;
}

void free_all(specoptim_t *h) {
    float *bufs[] = {h->M, h->U, h->s, h->V, h->d, h->m1, h->m2, h->Uo, h->UTo,
                     h->Vo, h->VTo, h->ws_g, h->ws_a, h->ws_x, h->ws_svd, h->PL, h->PR};
    for (float *p : bufs)
        if (p) cudaFree(p);
}

}  // namespace

extern "C" const char *specoptim_last_error(void) { return g_last_error.c_str(); }

extern "C" int specoptim_config_default(specoptim_config *cfg, int32_t m, int32_t n) {
    clear_error();
    if (!cfg) return fail(SPECOPTIM_ERR_INVALID_ARG, "config is null");
    std::memset(cfg, 0, sizeof(*cfg));
    cfg->m = m;
    cfg->n = n;
    cfg->beta_anc = 0.9f;
    cfg->tau_p = 1e-3f;
    cfg->alpha = 0.3f;
    cfg->beta1 = 0.9f;
    cfg->beta2 = 0.999f;
    cfg->eps = 1e-8f;
    cfg->weight_decay = 0.01f;
    cfg->precision = SPECOPTIM_PREC_TF32;
    cfg->svd_max_sweeps = 20;
    cfg->svd_tol = 1e-5f;
    cfg->svd_inner_sweeps = 1;
    return SPECOPTIM_OK;
}

extern "C" int specoptim_create(specoptim_t **out, const specoptim_config *cfg, void *stream) {
    clear_error();
    if (!out) return fail(SPECOPTIM_ERR_INVALID_ARG, "out is null");
    *out = nullptr;
    int rc = validate_cfg(cfg);
    if (rc) return rc;
    if ((rc = bind_device())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    specoptim_t *h = new specoptim_t();
    std::memset(h, 0, sizeof(*h));
    h->cfg = *cfg;
    h->m = cfg->m;
    h->n = cfg->n;
    h->r = std::min(cfg->m, cfg->n);
    h->tall = cfg->m > cfg->n;
    const size_t mn = (size_t)h->m * h->n, mr = (size_t)h->m * h->r, nr = (size_t)h->n * h->r;
    const size_t rr = (size_t)h->r * h->r;
    struct {
        float **p;
        size_t count;
    } plan[] = {
        {&h->M, mn}, {&h->U, mr}, {&h->s, (size_t)h->r}, {&h->V, nr}, {&h->d, (size_t)h->r},
        {&h->m1, mn}, {&h->m2, mn}, {&h->Uo, mr}, {&h->UTo, mr}, {&h->Vo, nr}, {&h->VTo, nr},
        {&h->ws_g, h->tall ? mn : 4}, {&h->ws_a, h->tall ? (size_t)h->n * h->r : mr},
        {&h->ws_x, rr}, {&h->ws_svd, svd_workspace_floats(h->m, h->n)},
        {&h->PL, h->m <= h->n ? (size_t)h->m * h->m : 4}, {&h->PR, h->m >= h->n ? (size_t)h->n * h->n : 4},
    };
    for (auto &b : plan) {
        cudaError_t e = cudaMalloc(reinterpret_cast<void **>(b.p), b.count * sizeof(float));
        if (e == cudaSuccess) e = cudaMemsetAsync(*b.p, 0, b.count * sizeof(float), st);
        if (e != cudaSuccess) {
            free_all(h);
            delete h;
            return cuda_status(e, "specoptim_create: allocation");
        }
    }
    *out = h;
    return SPECOPTIM_OK;
}

extern "C" int specoptim_destroy(specoptim_t *h) {
    clear_error();
    if (!h) return SPECOPTIM_OK;
    if (h->pending)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "destroy: an SVD refresh of this handle is in progress "
                                               "(end it with specoptim_svd_refresh_end first)");
    cudaDeviceSynchronize();
    free_all(h);
    delete h;
    return SPECOPTIM_OK;
}

extern "C" int specoptim_anchor_update(specoptim_t *h, const float *G_anc, void *stream) {
    clear_error();
    if (!h || !G_anc) return fail(SPECOPTIM_ERR_INVALID_ARG, "anchor_update: null argument");
    if (!aligned16(G_anc)) return fail(SPECOPTIM_ERR_MISALIGNED, "anchor_update: G_anc not 16-byte aligned");
    if (h->pending)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "anchor_update: the anchor momentum is being decomposed "
                                               "(call specoptim_svd_refresh_end first)");
    return ema_run(h->M, G_anc, (int64_t)h->m * h->n, h->cfg.beta_anc,
                   static_cast<cudaStream_t>(stream));
}

namespace {

// P = X diag(d) X^T (rows x rows) for a factor X (rows x r): X diag(d) into
// `tmp`, then one fp32-accurate 3xTF32 product, rounded to TF32 when it feeds
// the tensor-core step
int form_projector(const float *X, const float *d, int rows, int r, float *P, float *tmp, bool round,
                   cudaStream_t st) {
    int rc = scale_cols_run(X, d, rows, r, tmp, st);
    if (rc) return rc;
    float *ws = nullptr;
    if ((rc = scratch_floats(gemm3_workspace_floats(rows, rows, r), &ws))) return rc;
    Epilogue e;
    e.C = P;
    e.ldc = rows;
    e.round_tf32 = round;
    return gemm_fp32x3(rows, rows, r, Operand{X, r, false}, Operand{tmp, r, true}, e, ws, st);
}

}  // namespace

namespace {

int check_handles(specoptim_t *const *handles, int32_t count, const char *what) {
    if (!handles || count < 1 || count > 16)
        return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": 1 to 16 handles");
    for (int i = 0; i < count; ++i) {
        if (!handles[i]) return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": null handle");
        for (int k = 0; k < i; ++k)
            if (handles[k] == handles[i])
                return fail(SPECOPTIM_ERR_INVALID_ARG, std::string(what) + ": repeated handle");
    }
    return SPECOPTIM_OK;
}

void fill_jobs(specoptim_t *const *handles, int32_t count, SvdJob *jobs) {
    for (int i = 0; i < count; ++i) {
        specoptim_t *h = handles[i];
        SvdJob &a = jobs[i];
        a.M = h->M;
        a.m = h->m;
        a.n = h->n;
        a.U = h->U;
        a.s = h->s;
        a.V = h->V;
        a.d = h->d;
        a.work = h->ws_svd;
        a.warm = h->have_factors ? (h->tall || h->m == h->n ? h->V : h->U) : nullptr;
        a.tau = h->cfg.tau_p;
        a.tol = h->cfg.svd_tol;
        a.max_sweeps = h->cfg.svd_max_sweeps;
        a.inner_sweeps = h->cfg.svd_inner_sweeps;
        a.sweeps = 0;
        a.status = SPECOPTIM_OK;
    }
}

// After the factors of a refresh are written (svd_refresh_complete returned
// rc): the step's operand copies and projector of every converged handle.
int install_factors(specoptim_t *const *handles, int32_t count, const SvdJob *jobs, int rc,
                    cudaStream_t st, int32_t *sweeps_out) {
    if (sweeps_out)
        for (int i = 0; i < count; ++i) sweeps_out[i] = jobs[i].sweeps;
    if (rc && rc != SPECOPTIM_ERR_NOT_CONVERGED) return rc;
    std::string err = rc ? std::string(specoptim_last_error()) : std::string();
    for (int i = 0; i < count; ++i) {
        specoptim_t *h = handles[i];
        if (jobs[i].status != SPECOPTIM_OK) continue;
        // operand copies for the step's GEMMs
        const bool round = h->cfg.precision == SPECOPTIM_PREC_TF32;
        int r2;
        if ((r2 = transpose_run(h->U, h->UTo, h->m, h->r, round, st))) return r2;
        if ((r2 = transpose_run(h->V, h->VTo, h->n, h->r, round, st))) return r2;
        if ((r2 = transpose_run(h->UTo, h->Uo, h->r, h->m, false, st))) return r2;
        if ((r2 = transpose_run(h->VTo, h->Vo, h->r, h->n, false, st))) return r2;
        if (h->m <= h->n && (r2 = form_projector(h->U, h->d, h->m, h->r, h->PL, h->ws_svd, round, st))) return r2;
        if (h->m >= h->n && (r2 = form_projector(h->V, h->d, h->n, h->r, h->PR, h->ws_svd, round, st))) return r2;
        h->have_factors = true;
    }
    int r3 = check_device_flag(st);
    if (r3) return r3;
    if (rc) return fail(rc, err);
    return SPECOPTIM_OK;
}

}  // namespace

extern "C" int specoptim_svd_refresh_many(specoptim_t *const *handles, int32_t count, void *stream,
                                          int32_t *sweeps_out) {
    clear_error();
    int rc = check_handles(handles, count, "svd_refresh_many");
    if (rc) return rc;
    for (int i = 0; i < count; ++i)
        if (handles[i]->pending)
            return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_refresh_many: a refresh of this handle is in progress");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SvdJob jobs[16];
    fill_jobs(handles, count, jobs);
    rc = svd_refresh_batch(jobs, count, st);
    return install_factors(handles, count, jobs, rc, st, sweeps_out);
}

extern "C" int specoptim_svd_refresh_begin(specoptim_t *const *handles, int32_t count, void *stream) {
    clear_error();
    int rc = check_handles(handles, count, "svd_refresh_begin");
    if (rc) return rc;
    for (int i = 0; i < count; ++i)
        if (handles[i]->pending)
            return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_refresh_begin: a refresh of this handle is in progress");
    PendingRefresh *P = new PendingRefresh();
    P->count = count;
    for (int i = 0; i < count; ++i) P->h[i] = handles[i];
    fill_jobs(handles, count, P->jobs);
    if ((rc = svd_refresh_start(P->jobs, count, static_cast<cudaStream_t>(stream), true, &P->run))) {
        delete P;
        return rc;
    }
    for (int i = 0; i < count; ++i) handles[i]->pending = P;
    return SPECOPTIM_OK;
}

extern "C" int specoptim_svd_refresh_end(specoptim_t *const *handles, int32_t count, void *stream,
                                         int32_t *sweeps_out) {
    clear_error();
    int rc = check_handles(handles, count, "svd_refresh_end");
    if (rc) return rc;
    PendingRefresh *P = handles[0]->pending;
    bool same = P && P->count == count;
    for (int i = 0; same && i < count; ++i) same = P->h[i] == handles[i];
    if (!same)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "svd_refresh_end: the handles are not those of a refresh begun "
                                               "with specoptim_svd_refresh_begin (same handles, same order)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = svd_refresh_complete(P->run, P->jobs, st);
    for (int i = 0; i < count; ++i) handles[i]->pending = nullptr;
    SvdJob jobs[16];
    std::memcpy(jobs, P->jobs, sizeof(SvdJob) * count);
    delete P;
    return install_factors(handles, count, jobs, rc, st, sweeps_out);
}

extern "C" int specoptim_svd_refresh(specoptim_t *h, void *stream, int32_t *sweeps_out) {
    return specoptim_svd_refresh_many(&h, 1, stream, sweeps_out);
}

namespace {

// The products of one handle's step (two or three) with their epilogues, in
// slots first .. last: slot 0 holds every handle's first product, so that the
// square matrices' last (AdamW) product shares slot 1 with the others' middle
// products and slot 2 holds the AdamW products of the rest (grouped step_many
// runs one launch per slot; this spreads the AdamW epilogue's memory traffic
// over two of them).  `transpose` is set when G^T must be formed first (m > n).
constexpr int kSlots = 3;
struct StepPlan {
    GemmProblem stage[kSlots];
    int first, last;  // used slots
    bool transpose;
    const float *G;
    float *GT;
    int m, n;
    bool round;
};

int check_step_args(const specoptim_t *h, const float *W, const float *G_mask, float lr,
                    const float *G_filt_out, const float *G_proj_out) {
    if (!h || !W || !G_mask) return fail(SPECOPTIM_ERR_INVALID_ARG, "step: null argument");
    if (!aligned16(W) || !aligned16(G_mask) || (G_filt_out && !aligned16(G_filt_out)) ||
        (G_proj_out && !aligned16(G_proj_out)))
        return fail(SPECOPTIM_ERR_MISALIGNED, "step: pointers must be 16-byte aligned");
    if (!std::isfinite(lr)) return fail(SPECOPTIM_ERR_INVALID_ARG, "step: lr is not finite");
    return SPECOPTIM_OK;
}

// Advances the step counter and fills the plan (C = A . B^T problems, every
// operand K-contiguous).
StepPlan plan_step(specoptim_t *h, float *W, const float *G_mask, float lr, float *G_filt_out,
                   float *G_proj_out) {
    const int64_t m = h->m, n = h->n, r = h->r;
    StepPlan P;
    P.round = h->cfg.precision == SPECOPTIM_PREC_TF32;
    P.G = G_mask;
    P.GT = h->ws_g;
    P.m = h->m;
    P.n = h->n;
    P.transpose = h->tall;
    h->t += 1;
    const AdamWScalars sc = adamw_scalars(h->t, lr, h->cfg.beta1, h->cfg.beta2, h->cfg.eps,
                                          h->cfg.weight_decay);
    Epilogue plain;
    plain.round_tf32 = P.round;
    Epilogue scaled = plain;
    scaled.mode = EPI_SCALE;
    scaled.row_scale = h->d;
    scaled.col_scale = h->d;
    Epilogue last;
    last.mode = EPI_ADAMW;
    last.G = G_mask;
    last.W = W;
    last.m1 = h->m1;
    last.m2 = h->m2;
    last.Gf_out = G_filt_out;
    last.Gp_out = G_proj_out;
    last.ld = n;
    last.alpha = h->cfg.alpha;
    last.beta1 = sc.beta1;
    last.beta2 = sc.beta2;
    last.eps = sc.eps;
    last.decay = sc.decay;
    last.step_size = sc.step_size;
    last.inv_sqrt_bc2 = sc.inv_sqrt_bc2;
    auto nt = [](int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                 int64_t ldb, const Epilogue &e) {
        return GemmProblem{M, N, K, Operand{A, lda, false}, Operand{B, ldb, true}, e};
    };
    Epilogue cols = plain;  // diag(d) on the columns
    cols.mode = EPI_SCALE;
    cols.col_scale = h->d;
    if (m == n) {
        float *TT = h->ws_a;
        plain.C = TT;
        plain.ldc = m;
        P.first = 0;
        P.last = 1;
        P.transpose = false;
        P.stage[0] = nt(n, m, n, h->PR, n, G_mask, n, plain);     // T^T = P_R G^T
        P.stage[1] = nt(m, n, m, h->PL, m, TT, m, last);          // G_filt = P_L T -> AdamW
    } else if (h->tall) {
        float *T1 = h->ws_a, *T2T = h->ws_x;
        plain.C = T1;
        plain.ldc = n;
        P.first = 0;
        P.last = 2;
        P.stage[0] = nt(r, n, m, h->UTo, m, P.GT, m, plain);      // T1 = U^T G
        cols.C = T2T;
        cols.ldc = r;
        P.stage[1] = nt(n, r, n, h->PR, n, T1, n, cols);          // T2^T = P_R T1^T D
        P.stage[2] = nt(m, n, r, h->Uo, r, T2T, r, last);         // G_filt = U T2 -> AdamW
    } else {
        float *T1T = h->ws_a, *T2 = h->ws_x;
        plain.C = T1T;
        plain.ldc = m;
        P.first = 0;
        P.last = 2;
        P.stage[0] = nt(r, m, n, h->VTo, n, G_mask, n, plain);    // T1^T = V^T G^T
        cols.C = T2;
        cols.ldc = r;
        P.stage[1] = nt(m, r, m, h->PL, m, T1T, m, cols);         // T2 = P_L T1 D
        P.stage[2] = nt(m, n, r, T2, r, h->Vo, r, last);          // G_filt = T2 V^T -> AdamW
    }
    return P;
}

int run_problem(int precision, const GemmProblem &q, cudaStream_t st) {
    if (precision == SPECOPTIM_PREC_TF32 && gemm_tc_supported(q.M, q.N, q.K, q.A, q.B))
        return gemm_tc(q.M, q.N, q.K, q.A, q.B, q.epi, st);
    return gemm_simt(q.M, q.N, q.K, q.A, q.B, q.epi, st);
}

}  // namespace

extern "C" int specoptim_step(specoptim_t *h, float *W, const float *G_mask, float lr,
                              void *stream, float *G_filt_out, float *G_proj_out) {
    clear_error();
    int rc = check_step_args(h, W, G_mask, lr, G_filt_out, G_proj_out);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const StepPlan P = plan_step(h, W, G_mask, lr, G_filt_out, G_proj_out);
    if (P.transpose && (rc = transpose_run(P.G, P.GT, P.m, P.n, P.round, st))) return rc;
    for (int s = P.first; s <= P.last; ++s)
        if ((rc = run_problem(h->cfg.precision, P.stage[s], st))) return rc;
    return SPECOPTIM_OK;
}

extern "C" int specoptim_step_many(specoptim_t *const *handles, int32_t count, float *const *W,
                                   const float *const *G_mask, float lr, void *stream) {
    clear_error();
    if (!handles || !W || !G_mask || count < 1 || count > 16)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "step_many: 1 to 16 handles with W and G_mask arrays");
    int rc;
    for (int i = 0; i < count; ++i) {
        if ((rc = check_step_args(handles[i], W[i], G_mask[i], lr, nullptr, nullptr))) return rc;
        for (int k = 0; k < i; ++k)
            if (handles[k] == handles[i]) return fail(SPECOPTIM_ERR_INVALID_ARG, "step_many: repeated handle");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    StepPlan plans[16];
    for (int i = 0; i < count; ++i) plans[i] = plan_step(handles[i], W[i], G_mask[i], lr, nullptr, nullptr);
    TransposeJob tj[16];
    int nt = 0;
    for (int i = 0; i < count; ++i)
        if (plans[i].transpose) tj[nt++] = TransposeJob{plans[i].G, plans[i].GT, plans[i].m, plans[i].n, plans[i].round};
    if (nt && (rc = transpose_many(nt, tj, st))) return rc;
    for (int s = 0; s < kSlots; ++s) {
        // tensor-core problems of this slot share launches (largest first, 8 per launch);
        // the rest run one by one on the SIMT path
        GemmProblem group[16];
        double work[16];
        int ng = 0;
        for (int i = 0; i < count; ++i) {
            if (s < plans[i].first || s > plans[i].last) continue;
            const GemmProblem &q = plans[i].stage[s];
            if (handles[i]->cfg.precision == SPECOPTIM_PREC_TF32 && gemm_tc_supported(q.M, q.N, q.K, q.A, q.B)) {
                group[ng] = q;
                work[ng] = (double)q.M * q.N * q.K;
                ++ng;
            } else if ((rc = gemm_simt(q.M, q.N, q.K, q.A, q.B, q.epi, st))) {
                return rc;
            }
        }
        for (int a = 1; a < ng; ++a)  // insertion sort by work, descending
            for (int b = a; b > 0 && work[b] > work[b - 1]; --b) {
                std::swap(work[b], work[b - 1]);
                std::swap(group[b], group[b - 1]);
            }
        for (int off = 0; off < ng; off += 8)
            if ((rc = gemm_tc_group(std::min(8, ng - off), group + off, st))) return rc;
    }
    return SPECOPTIM_OK;
}

extern "C" int specoptim_get_factors(const specoptim_t *h, float *U, float *s, float *V, float *d,
                                     void *stream) {
    clear_error();
    if (!h) return fail(SPECOPTIM_ERR_INVALID_ARG, "get_factors: null handle");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t mr = (size_t)h->m * h->r, nr = (size_t)h->n * h->r;
    if (U) SPECOPTIM_CUDA(cudaMemcpyAsync(U, h->U, mr * 4, cudaMemcpyDeviceToDevice, st));
    if (s) SPECOPTIM_CUDA(cudaMemcpyAsync(s, h->s, (size_t)h->r * 4, cudaMemcpyDeviceToDevice, st));
    if (V) SPECOPTIM_CUDA(cudaMemcpyAsync(V, h->V, nr * 4, cudaMemcpyDeviceToDevice, st));
    if (d) SPECOPTIM_CUDA(cudaMemcpyAsync(d, h->d, (size_t)h->r * 4, cudaMemcpyDeviceToDevice, st));
    return SPECOPTIM_OK;
}

extern "C" int specoptim_get_state(const specoptim_t *h, float *M, float *exp_avg,
                                   float *exp_avg_sq, int64_t *t, void *stream) {
    clear_error();
    if (!h) return fail(SPECOPTIM_ERR_INVALID_ARG, "get_state: null handle");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)h->m * h->n * 4;
    if (M) SPECOPTIM_CUDA(cudaMemcpyAsync(M, h->M, bytes, cudaMemcpyDeviceToDevice, st));
    if (exp_avg) SPECOPTIM_CUDA(cudaMemcpyAsync(exp_avg, h->m1, bytes, cudaMemcpyDeviceToDevice, st));
    if (exp_avg_sq) SPECOPTIM_CUDA(cudaMemcpyAsync(exp_avg_sq, h->m2, bytes, cudaMemcpyDeviceToDevice, st));
    if (t) *t = h->t;
    return SPECOPTIM_OK;
}

extern "C" int specoptim_set_state(specoptim_t *h, const float *M, const float *exp_avg,
                                   const float *exp_avg_sq, int64_t t, void *stream) {
    clear_error();
    if (!h || !M || !exp_avg || !exp_avg_sq || t < 0)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "set_state: null argument or t < 0");
    if (h->pending)
        return fail(SPECOPTIM_ERR_INVALID_ARG, "set_state: an SVD refresh of this handle is in progress "
                                               "(call specoptim_svd_refresh_end first)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)h->m * h->n * 4;
    SPECOPTIM_CUDA(cudaMemcpyAsync(h->M, M, bytes, cudaMemcpyDeviceToDevice, st));
    SPECOPTIM_CUDA(cudaMemcpyAsync(h->m1, exp_avg, bytes, cudaMemcpyDeviceToDevice, st));
    SPECOPTIM_CUDA(cudaMemcpyAsync(h->m2, exp_avg_sq, bytes, cudaMemcpyDeviceToDevice, st));
    h->t = t;
    return SPECOPTIM_OK;
}

extern "C" int specoptim_adamw(float *W, const float *g, float *exp_avg, float *exp_avg_sq,
                               int64_t numel, int64_t t, float lr, float beta1, float beta2,
                               float eps, float weight_decay, void *stream) {
    clear_error();
    if (numel < 0 || t < 1) return fail(SPECOPTIM_ERR_INVALID_ARG, "adamw: numel < 0 or t < 1");
    if (numel == 0) return SPECOPTIM_OK;
    if (!W || !g || !exp_avg || !exp_avg_sq) return fail(SPECOPTIM_ERR_INVALID_ARG, "adamw: null pointer");
    if (!aligned16(W) || !aligned16(g) || !aligned16(exp_avg) || !aligned16(exp_avg_sq))
        return fail(SPECOPTIM_ERR_MISALIGNED, "adamw: pointers must be 16-byte aligned");
    return adamw_run(W, g, exp_avg, exp_avg_sq, numel,
                     adamw_scalars(t, lr, beta1, beta2, eps, weight_decay),
                     static_cast<cudaStream_t>(stream));
}

extern "C" int specoptim_gemm_nt(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                 const float *B, int64_t ldb, float *C, int64_t ldc,
                                 int32_t precision, void *stream) {
    clear_error();
    if (M < 0 || N < 0 || K < 0) return fail(SPECOPTIM_ERR_INVALID_ARG, "gemm_nt: negative size");
    if (M == 0 || N == 0) return SPECOPTIM_OK;
    if (!A || !B || !C) return fail(SPECOPTIM_ERR_INVALID_ARG, "gemm_nt: null pointer");
    if (lda < K || ldb < K || ldc < N) return fail(SPECOPTIM_ERR_INVALID_ARG, "gemm_nt: leading dimension too small");
    Operand a{A, lda, false}, b{B, ldb, true};
    Epilogue e;
    e.C = C;
    e.ldc = ldc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (precision == SPECOPTIM_PREC_TF32) {
        if (!gemm_tc_supported(M, N, K, a, b))
            return fail(SPECOPTIM_ERR_NOT_IMPLEMENTED,
                        "gemm_nt: the tensor-core path needs K >= 1, lda/ldb multiples of 4 and 16-byte aligned A, B");
        return gemm_tc(M, N, K, a, b, e, st);
    }
    if (precision != SPECOPTIM_PREC_FP32) return fail(SPECOPTIM_ERR_INVALID_ARG, "gemm_nt: unknown precision");
    return gemm_simt(M, N, K, a, b, e, st);
}
