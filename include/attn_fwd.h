/*
 * exact_attention_51_gb300 -- C ABI of the fused exact attention forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (all entry points below compute or check this one):
 *
 *     O   = softmax(scale * Q K^T  [+ causal mask]) V
 *     LSE = ln sum_j exp(scale * q_i . k_j)          (over the visible keys j)
 *
 * computed exactly -- not approximated -- as ONE fused, tiled kernel: the
 * N x N score matrix is never written to HBM.  The softmax row dependency is
 * broken with the online-softmax trick: the kernel visits key/value tiles in
 * order, keeps a running row maximum and row sum, and rescales the partial
 * output whenever the maximum grows, which reaches the same result as the
 * plain three-pass softmax.  Sources: "Tri Dao: prediction" (podcast
 * transcript: I/O awareness, kernel fusion, tiling into fast memory, the
 * softmax row dependency and the online-softmax trick); "Show HN: Flash
 * Attention in ~100 lines of CUDA" (forward pass only; torch used only for
 * bindings); HN item 40939030, FlashAttention-3 thread (the softmax of the
 * triangular matrix, i.e. causal attention, and the FA2/FA3/ThunderKittens
 * prior art).
 *
 * Conventions shared by every entry point
 *   - Q, K, V, O: bf16, contiguous row-major [B, H, N, d] (d fastest), passed
 *     as device pointers to __nv_bfloat16 data typed void* so that callers
 *     need no CUDA headers.  Nq = Nk = N (self-attention shapes).
 *   - LSE: fp32, contiguous [B, H, N], natural logarithm, scale included.
 *   - d must be 64, 128 or 256.  B, H, N >= 1.
 *   - scale: finite and >= 0 (the softmax temperature, usually 1/sqrt(d)).
 *   - causal != 0: key j is visible to query i iff j <= i (top-left aligned
 *     lower triangle; the diagonal is visible, so no row is empty).
 *   - Ownership: the caller owns every buffer.  The library allocates no
 *     device memory per call and keeps no per-call state.
 *   - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *     Calls are asynchronous: they enqueue work and return without a host
 *     synchronisation.  Execution errors surface at the caller's next
 *     synchronisation, as for any CUDA launch.
 *   - Thread safety: every entry point may be called from several host
 *     threads at once.
 */
#ifndef EXACT_ATTENTION_51_GB300_ATTN_FWD_H
#define EXACT_ATTENTION_51_GB300_ATTN_FWD_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by the entry points. */
enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,        /* null pointer, size < 1, d not in {64,128,256},
                                      sizes whose products overflow the launch,
                                      non-finite or negative scale */
  ATTN_ERR_MISALIGNED = 2,         /* q/k/v/o not 16-byte aligned, lse not 4-byte aligned */
  ATTN_ERR_ALIAS = 3,              /* o or lse overlaps an input, or lse overlaps o */
  ATTN_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
  ATTN_ERR_LAUNCH = 5,             /* CUDA runtime/driver call failed; see attn_last_cuda_error */
  ATTN_ERR_TIMEOUT = 6,            /* a device-side wait gave up (see attn_fwd_device_status) */
  ATTN_ERR_NOALLOC_TOO_LARGE = 7   /* attn_fwd_splitkv_noalloc: the problem needs more
                                      workspace than ATTN_NOALLOC_WORKSPACE_BYTES */
};

/* Size of the fixed device workspace behind attn_fwd_splitkv_noalloc. */
#define ATTN_NOALLOC_WORKSPACE_BYTES (64u * 1024u * 1024u)

/*
 * Fused exact attention forward.
 *
 *   q, k, v  device pointers, bf16 [B,H,N,d], read only (they may alias each
 *            other).  16-byte aligned.
 *   o        device pointer, bf16 [B,H,N,d], written.  16-byte aligned; must
 *            not overlap q, k, v or lse.
 *   lse      device pointer, fp32 [B,H,N], written.  4-byte aligned; must not
 *            overlap q, k, v or o.
 *   scale    multiplies Q K^T before the softmax.
 *   causal   0 = full attention, nonzero = causal (j <= i).
 *   stream   cudaStream_t to enqueue on.
 *
 * Enqueues one kernel and returns.  On any validation error nothing is
 * launched and the status says why.  O rows are the probability-weighted
 * value rows rounded to bf16 (round to nearest even); LSE is fp32.
 *
 * One thread block owns 256 query rows of one head (128 for d = 256), so a
 * launch has B*H*ceil(N/256) blocks.  When that is below the number of
 * multiprocessors (152 on GB300) -- few heads, long rows -- and the model
 * of attn_fwd_splitkv_num_splits finds it faster, d = 64 and 128 run 128
 * query rows per block instead (twice the blocks; measured on B=1 H=4
 * N=8192 d=128 causal: 990 TFLOP/s, against 658 with 256-row blocks and 904
 * with attn_fwd_splitkv's 2 splits).  A launch that still leaves the GPU
 * half idle -- one or two heads, as in decoding -- runs faster through
 * attn_fwd_splitkv with the count from attn_fwd_splitkv_num_splits, which
 * shares each block's keys over several blocks.
 */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, float scale, int causal, void* stream);

/*
 * The host-side argument checks of attn_fwd, without touching the GPU or the
 * CUDA runtime: returns ATTN_OK or the status attn_fwd would return for these
 * arguments before its device check.  Pointers are only compared, never
 * dereferenced.
 */
ATTN_API int attn_fwd_check_args(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, int B, int H, int N, int d, float scale, int causal);

/*
 * Split-KV variant of attn_fwd.  The key tiles of each 128..256-row query
 * block are shared out over `num_splits` thread blocks, which raises the
 * number of blocks in flight when B*H*N is too small to fill the GPU; each
 * block writes a normalised fp32 partial output and its partial
 * log-sum-exp to `workspace`, and a second kernel on the same stream merges
 * them per row (L = ln sum_s exp(L_s), O = sum_s exp(L_s - L) O_s -- the
 * associative merge of softmax states the online-softmax trick rests on,
 * "Tri Dao: prediction"; the "algebraic aggregates" of HN item 40939030).
 * The result equals attn_fwd's up to rounding.
 *
 *   num_splits  1..64.  1 runs attn_fwd itself (workspace unused, may be
 *               NULL).
 *   workspace   device buffer of at least
 *               attn_fwd_splitkv_workspace_size(B, H, N, d, num_splits)
 *               bytes, 256-byte aligned, owned by the caller, not
 *               overlapping q, k, v, o or lse.  Its contents on entry do not
 *               matter; it is scratch until the merge kernel has run.
 *   other arguments and errors as attn_fwd; a missing, short or misplaced
 *   workspace or num_splits out of range is ATTN_ERR_INVALID_ARG /
 *   ATTN_ERR_MISALIGNED / ATTN_ERR_ALIAS.  Enqueues two kernels.
 */
ATTN_API int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int N, int d, float scale, int causal, int num_splits,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes attn_fwd_splitkv needs (0 for num_splits == 1 or invalid
 * sizes): num_splits * B*H*N * (d + 1) * 4 bytes, each part 256-byte padded.
 * Host-only. */
ATTN_API size_t attn_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits);

/* A split count (1..16) for attn_fwd_splitkv on a GPU with `num_sms`
 * multiprocessors: 1 when attn_fwd's query blocks already fill one wave;
 * otherwise the count with the shortest modelled run time (blocks cost
 * their key tiles plus a fixed overhead -- a key tile of a 256-row block
 * 1.6 times one of a 128-row block -- and start heaviest first on the
 * least-loaded multiprocessor; a split run pays 5 % for the merge).
 * Host-only. */
ATTN_API int attn_fwd_splitkv_num_splits(int B, int H, int N, int d, int causal, int num_sms);

/*
 * Attention with a key length of its own (KV-cache shapes): q and o are
 * [B,H,Nq,d], k and v [B,H,Nk,d], lse [B,H,Nq].  Causal puts the diagonal of
 * the score matrix at its bottom-right corner -- query i sees keys
 * j <= i + Nk - Nq, so the Nq queries act as the last Nq positions of a
 * sequence whose keys are all Nk (the plainest reading of "the softmax of the
 * triangular matrix", HN item 40939030, for a rectangular score matrix) --
 * and needs Nk >= Nq.  Nq = Nk = N gives attn_fwd / attn_fwd_splitkv.
 *
 *   num_splits  1..64, as attn_fwd_splitkv; a decode-like call (small Nq,
 *               long Nk) needs splits to occupy the GPU
 *               (attn_fwd_kvcache_num_splits suggests a count).
 *   workspace   as attn_fwd_splitkv, sized by
 *               attn_fwd_splitkv_workspace_size(B, H, Nq, d, num_splits).
 *   other arguments and errors as attn_fwd_splitkv; causal with Nk < Nq is
 *   ATTN_ERR_INVALID_ARG.
 */
ATTN_API int attn_fwd_kvcache(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Nq, int Nk, int d, float scale, int causal,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              void* stream);

/* attn_fwd_splitkv_num_splits for attn_fwd_kvcache shapes.  Host-only. */
ATTN_API int attn_fwd_kvcache_num_splits(int B, int H, int Nq, int Nk, int d, int causal,
                                         int num_sms);

/*
 * attn_fwd_splitkv without a caller-provided workspace.  The pages have no
 * counterpart of this entry point; it exists for callers that cannot
 * allocate device memory: a plugin whose host framework hands it only the
 * input and output buffers, or a serving loop that must keep cudaMalloc off
 * its hot path (cudaMalloc can synchronise the whole device, and where a
 * pool allocator owns the memory it can fail or fragment it).
 *
 * The split-KV workspace is a fixed array of ATTN_NOALLOC_WORKSPACE_BYTES
 * (64 MiB) of device memory inside the library.  Every device the library is
 * used on holds it from first use until the process exits.  The call
 * allocates nothing itself.
 *
 *   Arguments, results and errors as attn_fwd_splitkv (num_splits 1 needs
 *   no workspace and runs attn_fwd).  A problem whose workspace
 *   (attn_fwd_splitkv_workspace_size) exceeds ATTN_NOALLOC_WORKSPACE_BYTES
 *   is rejected with ATTN_ERR_NOALLOC_TOO_LARGE before anything is launched.
 *   The first call on a device looks up the array's device address with the
 *   CUDA runtime (a one-time set-up per device, made with that device
 *   current); make that first call before any stream capture.
 *   All calls share the one array, and it keeps what the last call left in
 *   it.  Nothing in it has to start at zero: each call writes every value it
 *   later reads.  Calls whose kernels overlap on the GPU (several streams,
 *   several host threads) race on the array and give wrong results: order
 *   them, for instance on one stream.
 */
ATTN_API int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int H, int N, int d, float scale,
                                      int causal, int num_splits, void* stream);

/* Static, NUL-terminated English text for a status code. */
ATTN_API const char* attn_status_string(int status);

/*
 * Every wait inside the kernel is bounded: a wait that does not complete
 * within about two seconds stops that thread block, records a diagnostic
 * code in a device-wide status word and lets the kernel return instead of
 * hanging.  This call synchronises `stream`, reads the status word of the
 * current device, clears it and returns ATTN_OK (no timeout since the last
 * call) or ATTN_ERR_TIMEOUT.  `detail`, if not NULL, receives the raw code
 * (0 when clean): 0x1xx for a wait that gave up (0x101 TMA producer, 0x11x
 * MMA warp, 0x12x elementwise / softmax warps, 0x131 draining in-flight work,
 * 0x1f1 attn_selftest_wait_timeout), 0x1f2 when a head-dim-256 backward
 * kernel found its shared memory not 1024-byte aligned (it then does no
 * work), 0x1f3 when one found its ring out of order.  Outputs of launches
 * that ran while the word was set are not valid.  attn_bwd shares the word.
 */
ATTN_API int attn_fwd_device_status(void* stream, unsigned int* detail);

/* The cudaError_t of the last failed CUDA call made by this host thread
 * inside the library (0 if none). */
ATTN_API int attn_last_cuda_error(void);

/*
 * Self-test of the bounded waits behind attn_fwd_device_status: enqueues one
 * small kernel whose single wait (on an mbarrier nothing arrives on) gives up
 * after `timeout_ms` (1..10000) milliseconds, records its code (0x1f1) in the
 * device status word and exits.  A following attn_fwd_device_status returns
 * ATTN_ERR_TIMEOUT with that code and clears the word; the CUDA context stays
 * usable.  The status word is shared with every attn_fwd launch on the
 * device, so run this only when no other launch of the library is in flight.
 */
ATTN_API int attn_selftest_wait_timeout(unsigned int timeout_ms, void* stream);

/*
 * Self-test of the fused kernel's own abort path (a test hook, not a way to
 * compute attention): runs attn_fwd on the given arguments, except that in
 * every thread block the TMA producer leaves out the copy of K/V ring
 * position `drop_load` (0 = K tile 0, 1 = V tile 0, 2 = K tile 1, ...) and
 * every bounded wait gives up after `timeout_ms` (1..10000) milliseconds.
 * Nothing arrives on that slot's barrier, so the MMA warp's wait for it (or a
 * wait that depends on it: the producer's for a free slot, the softmax's for
 * the next scores) runs out: the first to give up records its code (0x1xx:
 * 0x101 producer, 0x11x MMA warp, 0x12x softmax) in the device status word
 * and raises the block's abort flag; the other roles leave their waits, every
 * role lets the copies and tensor-core operations it started finish (bounded
 * again), tensor memory is freed and the kernel returns.  Blocks that see fewer ring
 * positions than `drop_load` run to the end as usual.  O and LSE are not
 * valid afterwards; attn_fwd_device_status returns ATTN_ERR_TIMEOUT with the
 * code and clears the word, and the CUDA context stays usable.  Arguments
 * and errors as attn_fwd, plus ATTN_ERR_INVALID_ARG for drop_load < 0 or a
 * limit out of range.  The status word is shared with every launch of the
 * library on the device, so run this only when no other is in flight.
 */
ATTN_API int attn_selftest_fwd_dropped_load(const void* q, const void* k, const void* v, void* o,
                                            float* lse, int B, int H, int N, int d, float scale,
                                            int causal, int drop_load, unsigned int timeout_ms,
                                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_51_GB300_ATTN_FWD_H */
