/*
 * The activation mask fused with the ops at a pipeline-stage boundary of a
 * decoder (key design 1 of "Communication-Efficient LLM Adaptation over
 * Decentralized GPU Meshes", NeurIPS 2026, arXiv 2609.14339; papernotes.org
 * notes): only the K kept values of the boundary activation h~ = h (.) m and of
 * its gradient travel, and the backward pass reuses the same indices.  Here
 * the pack is folded into the op that produces the boundary value on the
 * sender (the decoder layer's residual sum) and the unpack into the op that
 * consumes it on the receiver (the next layer's RMSNorm), so the dense
 * boundary tensor is never written and read back just to be packed or
 * normalised.
 *
 * The mask function g and its arguments (layer, step, batch_id, H, K) are
 * exactly those of mask_pack / mask_unpack in specoptim.h: the fused ops and
 * the plain ones select the same dims.  Every tensor is bf16 (2-byte
 * elements), row-major: dense [rows][H], packed [rows][K], gamma [H].
 * Pointers are device pointers, 2-byte aligned; 0 <= K <= H <= 2^30.  Calls
 * are asynchronous on `stream` (a cudaStream_t as void*) and return the status
 * codes of specoptim.h (message in specoptim_last_error()).
 *
 * Arithmetic (this library's reading; the page leaves the model's ops to the
 * model): a bf16 sum is the float32 sum rounded to bf16, nearest even; RMSNorm
 * is the Llama form x = h / sqrt(mean_j h_j^2 + eps) * gamma, computed in fp32
 * and rounded once to bf16.  Off-mask entries of h~ are +0.
 */
#ifndef MASK_FUSED_H
#define MASK_FUSED_H

#include <stdint.h>

#include "specoptim.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Sender, forward: packed[r][k] = bf16(a + b)[r][pi_r(k)].  a, b: dense (the
 * residual stream and the layer's last projection); only the kept dims are
 * read and summed. */
int mask_pack_add(const void *a, const void *b, void *packed, int64_t rows, int32_t H, int32_t K,
                  uint32_t layer, uint64_t step, uint64_t batch_id, void *stream);

/* Receiver, forward: h_out = unpack(packed) (dense h~, kept for the residual
 * branch) and x_out = RMSNorm(h~) * gamma (dense, zero off the mask).  The
 * mean of squares is taken over all H dims of h~, i.e. over the K received
 * values divided by H. */
int mask_unpack_rmsnorm(const void *packed, const void *gamma, float eps, void *h_out, void *x_out,
                        int64_t rows, int32_t H, int32_t K, uint32_t layer, uint64_t step,
                        uint64_t batch_id, void *stream);

/* Receiver, backward: packed_grad[r][k] = dL/dh~ at dim pi_r(k), where
 *   dL/dh~_j = g_res_j + gamma_j dx_j / rr - h~_j (sum_i gamma_i dx_i h~_i) / (H rr^3),
 *   rr = sqrt(mean_j h~_j^2 + eps),
 * with h~ given by its packed values packed_h, dx the gradient of x_out and
 * g_res (may be NULL) the gradient reaching h~ through the residual branch.
 * Only the kept dims of dx and g_res are read. */
int mask_rmsnorm_backward_pack(const void *packed_h, const void *gamma, float eps, const void *dx,
                               const void *g_res, void *packed_grad, int64_t rows, int32_t H,
                               int32_t K, uint32_t layer, uint64_t step, uint64_t batch_id,
                               void *stream);

/* Sender, backward: g[r][pi_r(k)] <- bf16(g + packed[r][k]) in place; every
 * other entry of g is left as it is (the gradient of the boundary value adds
 * into the residual stream's gradient). */
int mask_unpack_add(const void *packed, void *g, int64_t rows, int32_t H, int32_t K, uint32_t layer,
                    uint64_t step, uint64_t batch_id, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MASK_FUSED_H */
