/*
 * exact_attention_51_gb300 -- C ABI of the attention backward pass.
 *
 * Gradients of O = softmax(scale * Q K^T [+ causal mask]) V for an upstream
 * gradient dO:
 *
 *     dV = P^T dO,   dS = P o (dP - D) with dP = dO V^T, D_i = sum_c dO_ic O_ic,
 *     dQ = scale * dS K,   dK = scale * dS^T Q,
 *
 * P recomputed tile by tile from the forward's log-sum-exp -- like the
 * forward, no N x N matrix is written to HBM.  The pages name the backward
 * pass only as the part the ~100-line kernel's author had not written ("Show
 * HN: Flash Attention in ~100 lines of CUDA"); these are the derivatives of
 * the forward definition (see include/attn_fwd.h for the conventions:
 * layouts, causal, streams, ownership, status codes).
 */
#ifndef EXACT_ATTENTION_51_GB300_ATTN_BWD_H
#define EXACT_ATTENTION_51_GB300_ATTN_BWD_H

#include <stddef.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Backward pass, Nq = Nk = N.
 *
 *   q, k, v     the forward's inputs, bf16 [B,H,N,d]
 *   o, lse      the forward's outputs for the same scale and causal flag
 *               (bf16 [B,H,N,d], fp32 [B,H,N])
 *   dout        upstream gradient of o, bf16 [B,H,N,d]
 *   dq, dk, dv  written, bf16 [B,H,N,d]; must not overlap any input, each
 *               other or the workspace.  16-byte aligned.
 *   d           64, 128 or 256; other d is ATTN_ERR_INVALID_ARG.  At 64 and
 *               128 one kernel forms dK and dV together (tensor memory holds
 *               S, dP and two d-wide accumulators); at 256 one d-wide
 *               accumulator fills half of it, so dV, dK and dQ each take a
 *               kernel of their own.
 *   workspace   device buffer of attn_bwd_workspace_size(B, H, N) bytes,
 *               256-byte aligned, scratch for the call (per-row D and
 *               LSE * log2 e).
 * Enqueues three kernels on `stream` (row statistics, dK/dV, dQ; four at
 * d = 256: row statistics, dV, dK, dQ) and returns.
 */
ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                      const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                      int H, int N, int d, float scale, int causal, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Workspace bytes for attn_bwd: two fp32 arrays of B*H*round_up(N, 128),
 * each 256-byte padded (0 for invalid sizes).  Host-only. */
ATTN_API size_t attn_bwd_workspace_size(int B, int H, int N);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_51_GB300_ATTN_BWD_H */
