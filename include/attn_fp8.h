/*
 * exact_attention_51_gb300 -- C ABI of the 8-bit (e4m3) attention forward.
 *
 * The same exact attention as attn_fwd (include/attn_fwd.h), with Q, K and V
 * given as OCP FP8 e4m3 codes and one dequantisation scale per tensor: the
 * computed quantity is
 *
 *     O = softmax(scale * (sq Q8) (sk K8)^T [+ causal mask]) (sv V8),
 *     LSE_i = log sum_j exp(scale * sq sk q8_i . k8_j)
 *
 * with sq, sk, sv the descale arguments and Q8, K8, V8 the decoded codes.
 * The products run on the tensor cores' 8-bit path (tcgen05.mma
 * kind::f8f6f4, fp32 accumulate).  P is rounded to e4m3 before P V (bf16 in
 * attn_fwd), so O carries a relative rounding of up to 2^-4 per softmax
 * weight; the running max, the row sum and LSE stay fp32.  The pages' FA-3
 * thread (HN item 40939030) argues for adapting the kernel to the hardware it
 * runs on; 8-bit operands at twice the bf16 tensor rate are that adaptation
 * here -- the pages themselves give no FP8 algorithm.
 */
#ifndef EXACT_ATTENTION_51_GB300_ATTN_FP8_H
#define EXACT_ATTENTION_51_GB300_ATTN_FP8_H

#include <stddef.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * e4m3 forward, Nq = Nk = N, d = 64, 128 or 256.
 *
 *   q, k, v     e4m3 codes, one byte per element, [B,H,N,d] contiguous,
 *               16-byte aligned; read only.
 *   descale_q, descale_k, descale_v
 *               finite and > 0: element x of Q means descale_q * e4m3(x).
 *   o           written, bf16 [B,H,N,d], 16-byte aligned.
 *   lse         written, fp32 [B,H,N] (natural log), 4-byte aligned.
 *   scale       softmax scale (finite, >= 0), as in attn_fwd.
 *   workspace   device buffer of attn_fwd_fp8_workspace_size(B, H, N, d)
 *               bytes, 256-byte aligned, when that size is not 0.  It is 0
 *               here (the kernel reads V as stored), so NULL and 0 are
 *               accepted; the argument is kept so that callers need not
 *               change if a later version needs scratch.  o, lse and
 *               workspace must not overlap each other or q, k, v.
 * Enqueues the fused forward on `stream` and returns; status codes as in
 * attn_fwd (d not 64, 128 or 256, a non-positive or non-finite descale, a
 * missing or short workspace: ATTN_ERR_INVALID_ARG).
 */
ATTN_API int attn_fwd_fp8(const void* q, const void* k, const void* v, float descale_q,
                          float descale_k, float descale_v, void* o, float* lse, int B, int H,
                          int N, int d, float scale, int causal, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Workspace bytes for attn_fwd_fp8: 0 (the kernel reads V as stored; 0 for
 * invalid sizes as well).  Host-only. */
ATTN_API size_t attn_fwd_fp8_workspace_size(int B, int H, int N, int d);

/*
 * e4m3 forward with separate query and key lengths (a KV cache), optionally
 * split over several CTAs per query block (split-KV, as attn_fwd_splitkv).
 *
 *   q           e4m3 [B,H,Nq,d]; k, v e4m3 [B,H,Nk,d]; o bf16 [B,H,Nq,d];
 *               lse fp32 [B,H,Nq].
 *   causal      query i sees keys j <= i + Nk - Nq (the queries are the last
 *               Nq positions of the sequence; needs Nk >= Nq), as
 *               attn_fwd_kvcache.
 *   num_splits  1..64; attn_fwd_fp8_kvcache_num_splits gives the
 *               split count the library's makespan model picks.
 *   workspace   attn_fwd_fp8_kvcache_workspace_size(B, H, Nq, Nk, d,
 *               num_splits) bytes, 256-byte aligned: (num_splits > 1) the
 *               fp32 partial O and LSE of every split; NULL when the size is
 *               0.
 * Other arguments, errors and asynchrony as attn_fwd_fp8; with num_splits >
 * 1 a merge kernel follows the fused kernel on `stream`.
 */
ATTN_API int attn_fwd_fp8_kvcache(const void* q, const void* k, const void* v, float descale_q,
                                  float descale_k, float descale_v, void* o, float* lse, int B,
                                  int H, int Nq, int Nk, int d, float scale, int causal,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* Workspace bytes for attn_fwd_fp8_kvcache (0 for invalid sizes).  Host-only. */
ATTN_API size_t attn_fwd_fp8_kvcache_workspace_size(int B, int H, int Nq, int Nk, int d,
                                                    int num_splits);

/* Split count for attn_fwd_fp8_kvcache from the makespan model of
 * attn_fwd_splitkv_num_splits, for the e4m3 tile shape.  Host-only. */
ATTN_API int attn_fwd_fp8_kvcache_num_splits(int B, int H, int Nq, int Nk, int d, int causal,
                                            int num_sms);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_51_GB300_ATTN_FP8_H */
