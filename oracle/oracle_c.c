/*
 * Test infrastructure: the CPU oracle (C part).  Plain, slow, float64 where
 * the arithmetic is floating point.  Only the tests, the smoke check and the
 * bench's CPU-baseline leg load this file's library; the product path never does.
 *
 * It holds the two pieces of the oracle that need loops too slow for Python:
 *
 *   1. The activation-mask index function g and the pack / unpack copies.
 *      Source: "Communication-Efficient LLM Adaptation over Decentralized GPU
 *      Meshes" (papernotes.org notes), key design 1, mask equation
 *      h~ = h (.) m with K = round((1-p)H) kept dims per token, and the
 *      backward equation dL/dh = (dL/dh~) m.  The pages require only that g be
 *      deterministic, shared, keyed by (layer, step, batch metadata, S, H) and
 *      keep exactly K dims per token; the concrete keyed permutation below is
 *      this project's definition of g (a uniform random K-subset per row):
 *
 *        sm64(z)   = SplitMix64 output for state z (Steele, Lea, Flood 2014):
 *                    z += 0x9e3779b97f4a7c15, then the two xor-shift-multiply
 *                    steps and a final xor-shift.
 *        fmix32(x) = MurmurHash3 32-bit finaliser (Appleby).
 *        seed      = sm64(sm64(sm64(layer) ^ step) ^ batch_id)
 *        rowkey    = sm64(seed ^ row)            row = flattened b*T + t
 *        k_i       = low 32 bits of sm64(rowkey + i), i = 0..3
 *        w         = ceil(log2 H) bits, split hi = w/2 bits, lo = w - w/2 bits
 *        E(x)      : four alternating Feistel rounds
 *                    hi ^= fmix32(lo ^ k0) & hi_mask
 *                    lo ^= fmix32(hi ^ k1) & lo_mask
 *                    hi ^= fmix32(lo ^ k2) & hi_mask
 *                    lo ^= fmix32(hi ^ k3) & lo_mask
 *                    (each round is invertible, so E permutes [0, 2^w))
 *        pi(k)     = E applied to k repeatedly until the value is < H
 *                    (cycle walking, Black & Rogaway 2002)
 *        kept set  = { pi(k) : 0 <= k < K }, packed in k order.
 *
 *      Off-mask values are written as +0 (all-zero bytes), never h*0.
 *
 *   2. A one-sided (Hestenes) Jacobi thin SVD in float64, for the SVD of the
 *      anchor momentum M_anc = U S V^T (same page, key design 3).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* mask function g                                                            */
/* ------------------------------------------------------------------------- */

uint64_t oracle_sm64(uint64_t z) {
    z += 0x9e3779b97f4a7c15ULL;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

uint32_t oracle_fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85ebca6bU;
    h ^= h >> 13;
    h *= 0xc2b2ae35U;
    h ^= h >> 16;
    return h;
}

uint64_t oracle_mask_seed(uint32_t layer, uint64_t step, uint64_t batch_id) {
    return oracle_sm64(oracle_sm64(oracle_sm64((uint64_t)layer) ^ step) ^ batch_id);
}

void oracle_mask_row_keys(uint64_t seed, uint64_t row, uint32_t keys[4]) {
    uint64_t rowkey = oracle_sm64(seed ^ row);
    for (int i = 0; i < 4; ++i) keys[i] = (uint32_t)oracle_sm64(rowkey + (uint64_t)i);
}

/* number of bits w with 2^w >= H (H >= 1) */
static int domain_bits(uint32_t H) {
    int w = 0;
    while (((uint64_t)1 << w) < (uint64_t)H) ++w;
    return w;
}

/* one application of the Feistel permutation E on [0, 2^w) */
static uint32_t feistel(const uint32_t keys[4], int w, uint32_t x) {
    int hi_bits = w / 2, lo_bits = w - w / 2;
    uint32_t hi_mask = (uint32_t)((1u << hi_bits) - 1u);
    uint32_t lo_mask = (uint32_t)((1u << lo_bits) - 1u);
    uint32_t hi = x >> lo_bits, lo = x & lo_mask;
    hi ^= oracle_fmix32(lo ^ keys[0]) & hi_mask;
    lo ^= oracle_fmix32(hi ^ keys[1]) & lo_mask;
    hi ^= oracle_fmix32(lo ^ keys[2]) & hi_mask;
    lo ^= oracle_fmix32(hi ^ keys[3]) & lo_mask;
    return (hi << lo_bits) | lo;
}

/* pi(k) for 0 <= k < H; walks the cycle of E until it lands inside [0, H) */
uint32_t oracle_mask_perm(const uint32_t keys[4], uint32_t H, uint32_t k) {
    int w = domain_bits(H);
    uint32_t x = feistel(keys, w, k);
    uint64_t guard = 0, limit = (uint64_t)1 << w;
    while (x >= H && guard++ < limit) x = feistel(keys, w, x);
    return x;
}

/* idx[r*K + k] = pi_r(k); returns 0, or 1 on bad arguments */
int oracle_mask_indices(int32_t *idx, int64_t rows, int32_t H, int32_t K, uint32_t layer,
                        uint64_t step, uint64_t batch_id) {
    if (rows < 0 || H < 1 || K < 0 || K > H) return 1;
    uint64_t seed = oracle_mask_seed(layer, step, batch_id);
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t keys[4];
        oracle_mask_row_keys(seed, (uint64_t)r, keys);
        for (int32_t k = 0; k < K; ++k)
            idx[r * K + k] = (int32_t)oracle_mask_perm(keys, (uint32_t)H, (uint32_t)k);
    }
    return 0;
}

/* packed[r][k] = dense[r][pi_r(k)] (a copy of elem_bytes bytes) */
int oracle_mask_pack(const void *dense, void *packed, int64_t rows, int32_t H, int32_t K,
                     int32_t elem_bytes, uint32_t layer, uint64_t step, uint64_t batch_id) {
    if (rows < 0 || H < 1 || K < 0 || K > H || (elem_bytes != 2 && elem_bytes != 4)) return 1;
    const unsigned char *src = (const unsigned char *)dense;
    unsigned char *dst = (unsigned char *)packed;
    uint64_t seed = oracle_mask_seed(layer, step, batch_id);
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t keys[4];
        oracle_mask_row_keys(seed, (uint64_t)r, keys);
        for (int32_t k = 0; k < K; ++k) {
            uint32_t j = oracle_mask_perm(keys, (uint32_t)H, (uint32_t)k);
            memcpy(dst + ((size_t)r * K + k) * elem_bytes, src + ((size_t)r * H + j) * elem_bytes,
                   (size_t)elem_bytes);
        }
    }
    return 0;
}

/* dense[r][j] = packed[r][k] where j = pi_r(k), else +0 (all-zero bytes) */
int oracle_mask_unpack(const void *packed, void *dense, int64_t rows, int32_t H, int32_t K,
                       int32_t elem_bytes, uint32_t layer, uint64_t step, uint64_t batch_id) {
    if (rows < 0 || H < 1 || K < 0 || K > H || (elem_bytes != 2 && elem_bytes != 4)) return 1;
    const unsigned char *src = (const unsigned char *)packed;
    unsigned char *dst = (unsigned char *)dense;
    memset(dst, 0, (size_t)rows * H * elem_bytes);
    uint64_t seed = oracle_mask_seed(layer, step, batch_id);
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t keys[4];
        oracle_mask_row_keys(seed, (uint64_t)r, keys);
        for (int32_t k = 0; k < K; ++k) {
            uint32_t j = oracle_mask_perm(keys, (uint32_t)H, (uint32_t)k);
            memcpy(dst + ((size_t)r * H + j) * elem_bytes, src + ((size_t)r * K + k) * elem_bytes,
                   (size_t)elem_bytes);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* one-sided Jacobi thin SVD, float64                                         */
/* ------------------------------------------------------------------------- */

static double dot(const double *a, const double *b, int64_t len) {
    double s = 0.0;
    for (int64_t i = 0; i < len; ++i) s += a[i] * b[i];
    return s;
}

/*
 * Thin SVD of M (m x n, row-major): M = U diag(s) V^T with r = min(m, n),
 * U (m x r) and V (n x r) row-major with orthonormal columns, s descending.
 *
 * Works on the tall orientation A (p x q, p >= q): A = M if m >= n else M^T.
 * Sweeps over column pairs (i < j) in cyclic order; a pair is rotated when
 * |a_i . a_j| > tol * |a_i| |a_j|.  The rotation is the 2x2 symmetric Schur
 * rotation of the pair's Gram matrix, applied to A and accumulated into W
 * (q x q, starts at I).  On convergence A = U S and W = V (of A).
 * Columns with s = 0 get unit vectors completed against the canonical basis
 * (modified Gram-Schmidt), so that U always has orthonormal columns.
 *
 * Returns 0 on convergence, 4 when max_sweeps ran out (outputs still filled),
 * 1 on bad arguments, 3 on allocation failure.
 */
int oracle_thin_svd(const double *M, int64_t m, int64_t n, double *U, double *s, double *V,
                    int32_t max_sweeps, double tol, int32_t *sweeps_out) {
    if (m < 1 || n < 1 || !M || !U || !s || !V) return 1;
    int transposed = m < n;
    int64_t p = transposed ? n : m, q = transposed ? m : n;
    double *A = (double *)malloc(sizeof(double) * (size_t)(p * q));   /* column-major: A + j*p */
    double *W = (double *)malloc(sizeof(double) * (size_t)(q * q));   /* column-major          */
    double *L = (double *)malloc(sizeof(double) * (size_t)(p * q));
    double *norms = (double *)malloc(sizeof(double) * (size_t)q);
    int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)q);
    if (!A || !W || !L || !norms || !order) {
        free(A); free(W); free(L); free(norms); free(order);
        return 3;
    }
    for (int64_t i = 0; i < p; ++i)
        for (int64_t j = 0; j < q; ++j)
            A[j * p + i] = transposed ? M[j * n + i] : M[i * n + j];
    for (int64_t j = 0; j < q * q; ++j) W[j] = 0.0;
    for (int64_t j = 0; j < q; ++j) W[j * q + j] = 1.0;

    int converged = 0, sweep = 0;
    for (sweep = 0; sweep < max_sweeps && !converged; ++sweep) {
        int64_t rotations = 0;
        for (int64_t i = 0; i < q - 1; ++i) {
            for (int64_t j = i + 1; j < q; ++j) {
                double *ai = A + i * p, *aj = A + j * p;
                double alpha = dot(ai, ai, p), beta = dot(aj, aj, p), gamma = dot(ai, aj, p);
                if (gamma == 0.0 || fabs(gamma) <= tol * sqrt(alpha * beta)) continue;
                double zeta = (beta - alpha) / (2.0 * gamma);
                double t = (zeta >= 0.0 ? 1.0 : -1.0) / (fabs(zeta) + sqrt(1.0 + zeta * zeta));
                double c = 1.0 / sqrt(1.0 + t * t), sn = c * t;
                for (int64_t k = 0; k < p; ++k) {
                    double x = ai[k], y = aj[k];
                    ai[k] = c * x - sn * y;
                    aj[k] = sn * x + c * y;
                }
                double *wi = W + i * q, *wj = W + j * q;
                for (int64_t k = 0; k < q; ++k) {
                    double x = wi[k], y = wj[k];
                    wi[k] = c * x - sn * y;
                    wj[k] = sn * x + c * y;
                }
                ++rotations;
            }
        }
        if (rotations == 0) converged = 1;
    }
    if (sweeps_out) *sweeps_out = sweep;

    for (int64_t j = 0; j < q; ++j) { norms[j] = sqrt(dot(A + j * p, A + j * p, p)); order[j] = j; }
    /* insertion sort of column order by descending norm (stable) */
    for (int64_t a = 1; a < q; ++a) {
        int64_t key = order[a], b = a - 1;
        while (b >= 0 && norms[order[b]] < norms[key]) { order[b + 1] = order[b]; --b; }
        order[b + 1] = key;
    }
    /* left vectors of A: columns of A / s, in sorted order, column-major in L */
    for (int64_t c = 0; c < q; ++c) {
        int64_t j = order[c];
        s[c] = norms[j];
        double *dst = L + c * p;
        if (norms[j] > 0.0) {
            for (int64_t k = 0; k < p; ++k) dst[k] = A[j * p + k] / norms[j];
        } else {
            /* complete with the first canonical vector not yet in the span */
            for (int64_t e = 0; e < p; ++e) {
                for (int64_t k = 0; k < p; ++k) dst[k] = (k == e) ? 1.0 : 0.0;
                for (int pass = 0; pass < 2; ++pass)
                    for (int64_t o = 0; o < c; ++o) {
                        double proj = dot(L + o * p, dst, p);
                        for (int64_t k = 0; k < p; ++k) dst[k] -= proj * L[o * p + k];
                    }
                double nrm = sqrt(dot(dst, dst, p));
                if (nrm > 0.5) { for (int64_t k = 0; k < p; ++k) dst[k] /= nrm; break; }
            }
        }
    }
    /* write out: for A = M, U = L, V = W; for A = M^T, U = W, V = L */
    int64_t r = q;
    for (int64_t c = 0; c < r; ++c) {
        int64_t j = order[c];
        for (int64_t k = 0; k < p; ++k) {
            if (transposed) V[k * r + c] = L[c * p + k];
            else U[k * r + c] = L[c * p + k];
        }
        for (int64_t k = 0; k < q; ++k) {
            if (transposed) U[k * r + c] = W[j * q + k];
            else V[k * r + c] = W[j * q + k];
        }
    }
    free(A); free(W); free(L); free(norms); free(order);
    return converged ? 0 : 4;
}
