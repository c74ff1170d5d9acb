/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library libfa.so.
 *
 * The operations are those of FlashAttention-2 as described by
 *   [V2]  "6.2 FlashAttention V2 chi tiet" (infra-guide-du8.pages.dev),
 *   [CSDN] "FlashAttention-2" algorithm/parallelism article (blog.csdn.net),
 *   [FA3] "FlashAttention-3: Attention nhanh hon ..." summary (vi.news.hada.io),
 * with the precise section named at each entry point.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.   Q, O, dO, dQ: [B][Hq][N][d]; K, V, dK, dV: [B][Hkv][N][d]; d is
 *           contiguous, then N, then head, then batch (dense, no padding).
 *           LSE: [B][Hq][N] fp32.  Query head h reads key/value head
 *           h / (Hq / Hkv) (consecutive query heads share a key/value head).
 * Pointers. All tensor pointers are DEVICE pointers on the current device and
 *           must be 16-byte aligned.  The caller owns every buffer (inputs,
 *           outputs, workspace); the library never allocates, frees or
 *           synchronises device memory, except where an entry point says so.
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).  All
 *           compute entry points are asynchronous on that stream.
 * Sizes.    1 <= N; d in {64, 128}; Hq % Hkv == 0; B, Hq, Hkv >= 1; the
 *           row count B*N (packed batches: total) and B*Hq at most 2^31 - 1,
 *           and ceil(N / 128) * B * Hq at most 2^31 - 1 (one CTA per 128-row
 *           tile and head); a tensor may hold more than 2^31 elements.
 * Errors.   Invalid arguments are reported before anything is launched
 *           (FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_WORKSPACE) and
 *           leave every output untouched.  A failed launch returns
 *           FA_ERR_CUDA.  Device-side waits are bounded: a wait that runs out
 *           records FA_ERR_TIMEOUT in a per-device status (read it with
 *           fa_get_device_status) and the kernel returns instead of hanging.
 * Scores.   S = scale * Q K^T; causal masking is top-left aligned (query row r
 *           sees key c iff c <= r).  LSE is the natural-log log-sum-exp of the
 *           scaled, masked scores of each row.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, misaligned pointer */
    FA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d not 64/128) */
    FA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    FA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    FA_ERR_TIMEOUT = 5        /* a bounded device wait ran out (see status) */
} fa_status_t;

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype_t;

/*
 * Forward pass: O = softmax(scale Q K^T [causal mask]) V and LSE.
 * [V2] section 6.1 (full forward pseudocode: Q-tile outer loop, K/V inner
 * loop, running max m and sum l, unnormalised O~, single final diag(l)^-1
 * rescale, L = m + log l); section 5.3 (causal tile classes and early exit);
 * [CSDN] "parallelism / forward" (one thread block per Q tile x head x batch,
 * sequence-length parallelism) and 3.1.1 (the recurrence).
 *   q [B][Hq][N][d], k, v [B][Hkv][N][d]  (in, element type `dtype`)
 *   o [B][Hq][N][d]                       (out, element type `dtype`)
 *   lse [B][Hq][N]                        (out, fp32, natural log)
 * Short sequences (N <= 2048) run the kernel of fa_fwd_persistent, longer
 * ones one CTA per 256-row block; both give the same bits.  fa_fwd_local
 * with window <= 2048 and fa_fwd_varlen with max_seqlen <= 2048 (or a
 * window <= 2048) use the persistent kernel in the same way.
 */
fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o,
                   float *lse, int B, int Hq, int Hkv, int N, int d,
                   int causal, float scale, fa_dtype_t dtype, void *stream);

/*
 * The forward of fa_fwd as a persistent kernel with a dynamic block schedule.
 * [FA3] "remaining optimisations" (persistent kernel); the arithmetic is
 * fa_fwd's ([V2] section 6.1, [CSDN] 3.1.1), and for the same arguments O and
 * LSE are bit-identical to fa_fwd's.  The grid holds one CTA per 256-row
 * block in fa_fwd's longest-first order, but every CTA that runs keeps
 * running: it cancels CTAs that have not been launched yet (cluster launch
 * control) and works on their blocks, so blocks are handed out dynamically
 * with no counter in global memory, and each block's loads, first MMAs and
 * epilogue overlap the neighbouring block's work.  It pays off where blocks
 * are short (short sequences); fa_fwd itself uses it for the shapes where it
 * was measured faster.
 *   Arguments, layouts and errors as fa_fwd, except that o must be 32-byte
 *   aligned (its rows are stored 32 bytes at a time; FA_ERR_INVALID_ARG
 *   otherwise).  fa_fwd falls back to the one-CTA-per-block kernel when o is
 *   only 16-byte aligned.
 */
fa_status_t fa_fwd_persistent(const void *q, const void *k, const void *v,
                              void *o, float *lse, int B, int Hq, int Hkv,
                              int N, int d, int causal, float scale,
                              fa_dtype_t dtype, void *stream);

/*
 * Debug forward: fa_fwd with O written in fp32, i.e. O~ / l before any
 * rounding to the 16-bit type, so that the kernel's own arithmetic can be
 * checked without the output's rounding.  [V2] section 6.1 (the final
 * diag(l)^-1 rescale of O~).  Same kernel and schedule; each thread stores
 * its output row directly instead of staging a 16-bit tile for TMA.
 *   Arguments, layouts and errors as fa_fwd, except
 *   o_f32 [B][Hq][N][d] fp32 (out, 16-byte aligned).
 * O still carries the rounding of P to the 16-bit type that the P.V tensor
 * core product consumes.
 */
fa_status_t fa_fwd_f32_out(const void *q, const void *k, const void *v,
                           float *o_f32, float *lse, int B, int Hq, int Hkv,
                           int N, int d, int causal, float scale,
                           fa_dtype_t dtype, void *stream);

/*
 * Causal sliding-window ("local") forward: fa_fwd with causal = 1 and the
 * additional mask that query row r sees only the `window` most recent keys,
 * r - window + 1 .. r (its own key included).
 * [FA3] discussion of GQA and sliding-window attention (sliding-window
 * attention changes the attention mask, i.e. which queries see which keys;
 * the algorithm is otherwise unchanged); [V2] section 5.3 (tiles that lie
 * wholly outside the mask are skipped, boundary tiles are masked
 * element-wise) applied to the window's lower edge as well.
 *   Arguments, layouts and results as fa_fwd; window >= 1 (window >= N is
 *   plain causal attention), otherwise FA_ERR_INVALID_ARG.
 */
fa_status_t fa_fwd_local(const void *q, const void *k, const void *v, void *o,
                         float *lse, int B, int Hq, int Hkv, int N, int d,
                         int window, float scale, fa_dtype_t dtype,
                         void *stream);

/*
 * Bytes of device workspace fa_bwd needs: D (B*Hq*N fp32, rounded up to 256
 * bytes) followed by the fp32 dQ accumulator (B*Hq*N*d fp32).
 */
size_t fa_bwd_workspace_bytes(int B, int Hq, int N, int d);

/*
 * Backward pass from O, LSE and dO only.
 * [CSDN] 3.1.2 (step list: D = rowsum(dO o O); per K/V tile j and Q tile i:
 * S = Q_i K_j^T, P = exp(S - L_i), dV_j += P^T dO_i, dP = dO_i V_j^T,
 * dS = P o (dP - D_i), dQ_i += dS K_j, dK_j += dS^T Q_i) and "parallelism /
 * backward" (one thread block per K/V column block, dQ combined across blocks
 * by atomic addition); [V2] sections 7.1-7.3 (LSE instead of m and l; D
 * computed once by a separate preprocessing kernel); [CSDN] MQA/GQA paragraph
 * (dK, dV summed over the query heads of a group).  The scale factor enters
 * dQ and dK by the chain rule.
 *   q, k, v, o, lse, dO: as produced/consumed by fa_fwd (in)
 *   dq [B][Hq][N][d], dk, dv [B][Hkv][N][d]: out, element type `dtype`
 *   workspace: device buffer of at least fa_bwd_workspace_bytes(B,Hq,N,d)
 *   bytes, 256-byte aligned; its contents on entry do not matter.
 * dQ is accumulated with fp32 atomic reductions, so it is deterministic only
 * up to the order of those additions.
 * Short sequences (N <= 1024, with dK and dV 32-byte aligned) run a
 * persistent main kernel (work items handed out by cluster launch control,
 * as in fa_fwd_persistent); dK and dV are the same bits either way, dQ the
 * same up to the order of its fp32 atomic additions.
 */
fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o,
                   const float *lse, const void *dO, void *dq, void *dk,
                   void *dv, int B, int Hq, int Hkv, int N, int d, int causal,
                   float scale, fa_dtype_t dtype, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace fa_bwd_two_pass needs: D only (B*Hq*N fp32,
 * rounded up to 256 bytes).
 */
size_t fa_bwd_two_pass_workspace_bytes(int B, int Hq, int N, int d);

/*
 * Deterministic backward: the same results as fa_bwd, but dQ is formed by a
 * second pass instead of atomic addition, so repeated calls on the same
 * inputs give bit-identical dQ, dK and dV.
 * [V2] section 7.2 (dQ is combined across K/V column blocks either by atomic
 * addition or in two passes).  Pass 1 walks K/V column blocks as fa_bwd does
 * and produces dK and dV only.  Pass 2 walks Q row blocks: for Q tile i it
 * recomputes S = Q_i K_j^T, P = exp(S - L_i) and dS = P o (dP - D_i) for
 * every K/V tile j in order and forms dQ_i = scale * sum_j dS K_j on chip,
 * stored once.  S and dP are computed twice in total (once per pass).
 *   Arguments, layouts and results: as fa_bwd.
 *   workspace: device buffer of at least
 *   fa_bwd_two_pass_workspace_bytes(B,Hq,N,d) bytes, 256-byte aligned; its
 *   contents on entry do not matter.
 */
fa_status_t fa_bwd_two_pass(const void *q, const void *k, const void *v,
                            const void *o, const float *lse, const void *dO,
                            void *dq, void *dk, void *dv, int B, int Hq,
                            int Hkv, int N, int d, int causal, float scale,
                            fa_dtype_t dtype, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Backward of fa_fwd_local (same sliding-window mask), from O, LSE and dO.
 * [CSDN] 3.1.2 and [V2] section 7 as for fa_bwd, with the mask of
 * fa_fwd_local; K/V column blocks visit only the Q row blocks that see them
 * and Q row blocks only the K/V blocks they see.
 *   Arguments and layouts as fa_bwd; window >= 1.
 *   deterministic = 0: dQ by fp32 atomic addition (as fa_bwd), workspace of
 *   at least fa_bwd_workspace_bytes(B,Hq,N,d) bytes;
 *   deterministic = 1: dQ by a second pass (as fa_bwd_two_pass), workspace
 *   of at least fa_bwd_two_pass_workspace_bytes(B,Hq,N,d) bytes.
 */
fa_status_t fa_bwd_local(const void *q, const void *k, const void *v,
                         const void *o, const float *lse, const void *dO,
                         void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
                         int N, int d, int window, float scale,
                         fa_dtype_t dtype, int deterministic, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Forward over a batch of sequences of different lengths packed back to back
 * ("variable length sequence", named among the optimisations of [FA3]):
 * sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of the packed
 * tensors and attends only within itself, with the fa_fwd algorithm (causal
 * and sliding-window masks relative to the sequence start).
 *   q, o  [total][Hq][d], k, v [total][Hkv][d] (token-major, d contiguous)
 *   lse   [Hq][total] fp32 (natural log)
 *   cu_seqlens: DEVICE int32 [B + 1], cu_seqlens[0] = 0, non-decreasing,
 *   cu_seqlens[B] = total, every length <= max_seqlen (4-byte aligned).
 *   window: 0 = none, else >= 1 with causal = 1 (as fa_fwd_local).
 * The offsets are read on the device: lengths that break the rules above are
 * reported by fa_get_device_status as FA_ERR_INVALID_ARG and the affected
 * sequences are left unwritten.
 */
fa_status_t fa_fwd_varlen(const void *q, const void *k, const void *v, void *o,
                          float *lse, const int *cu_seqlens, int B,
                          int max_seqlen, int total, int Hq, int Hkv, int d,
                          int causal, int window, float scale,
                          fa_dtype_t dtype, void *stream);

/*
 * Workspace of fa_bwd_varlen: D ([Hq][total] fp32, rounded up to 256 bytes)
 * and, unless deterministic, the fp32 dQ accumulator ([total][Hq][d]).
 */
size_t fa_bwd_varlen_workspace_bytes(int total, int Hq, int d,
                                     int deterministic);

/*
 * Backward of fa_fwd_varlen: fa_bwd (deterministic = 0, atomic dQ) or
 * fa_bwd_two_pass (deterministic = 1) on the packed layout above.
 *   dq [total][Hq][d], dk, dv [total][Hkv][d] (out); other arguments as
 *   fa_fwd_varlen and fa_bwd; workspace of at least
 *   fa_bwd_varlen_workspace_bytes(total, Hq, d, deterministic) bytes,
 *   256-byte aligned.
 */
fa_status_t fa_bwd_varlen(const void *q, const void *k, const void *v,
                          const void *o, const float *lse, const void *dO,
                          void *dq, void *dk, void *dv, const int *cu_seqlens,
                          int B, int max_seqlen, int total, int Hq, int Hkv,
                          int d, int causal, int window, float scale,
                          fa_dtype_t dtype, int deterministic, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Size of the scratch buffer built into the library for fa_bwd_noalloc:
 * 64 MiB per device.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory (code that may not call cudaMalloc, such as a plugin handed
 * only tensor pointers by its host framework or a process whose memory pool
 * is fixed up front).  The pages have no counterpart to this entry point; it
 * exists only for such callers.
 *   Arguments, layouts and results are exactly those of fa_bwd, and invalid
 *   arguments get the same status codes as from fa_bwd.  The workspace is a
 *   buffer of FA_BWD_NOALLOC_SCRATCH_BYTES inside the library.  Problems
 *   whose fa_bwd_workspace_bytes(B, Hq, N, d) exceeds that size are refused
 *   with FA_ERR_WORKSPACE before anything touches the GPU (with d = 128 this
 *   allows B * Hq * N up to about 130,000 rows).
 *   When the memory is taken: the buffer's device memory is committed when
 *   the CUDA runtime loads the part of the library that holds it -- on the
 *   first call on a device (default lazy module loading), or when the
 *   library is loaded (CUDA_MODULE_LOADING=EAGER, on every device the
 *   process uses).  It is then held until the process exits.  Make the first
 *   call on each device (with that device current) before reserving a fixed
 *   memory pool and before any stream capture: that call also looks up the
 *   buffer's device address, and may fail with FA_ERR_CUDA if the device has
 *   no room left for the buffer.  Later calls allocate nothing.
 *   The looked-up address is cached per device and CUDA context, and looked
 *   up again if the device's current context changes (e.g. after
 *   cudaDeviceReset).
 *   All calls on a device share the one buffer: calls whose kernels may
 *   overlap on the GPU (e.g. on unordered streams) race and give wrong
 *   results.  Each call rewrites and re-zeroes what it uses, so nothing from
 *   an earlier call carries over.
 */
fa_status_t fa_bwd_noalloc(const void *q, const void *k, const void *v,
                           const void *o, const float *lse, const void *dO,
                           void *dq, void *dk, void *dv, int B, int Hq,
                           int Hkv, int N, int d, int causal, float scale,
                           fa_dtype_t dtype, void *stream);

/*
 * Bytes of workspace fa_hadamard_quant_fp8 needs (the fp32 amax cell).
 */
size_t fa_hadamard_quant_workspace_bytes(long rows, int d);

/*
 * Incoherent processing + per-tensor e4m3 quantisation of one tensor.
 * [FA3] "FP8 and incoherent processing": multiply by a random orthogonal
 * matrix, realised as a Hadamard transform with random signs, O(d log d) per
 * row; here x' = (x o s) H_d / sqrt(d) for every row of d values, then
 * sigma = amax(|x'|) / 448 over the whole tensor and x8 = e4m3(x' / sigma)
 * (round to nearest even, saturating).
 *   x_bf16  [rows][d] bf16 (in)
 *   signs   [d] fp32 of +-1 (in; only the sign of each entry is used), or
 *           NULL for no rotation (plain FP8)
 *   x_e4m3  [rows][d] e4m3 (out)
 *   descale one fp32 device scalar (out): sigma, so x' ~= sigma * x8
 *   workspace: >= fa_hadamard_quant_workspace_bytes(rows, d) bytes
 * d must be 64 or 128.
 */
fa_status_t fa_hadamard_quant_fp8(const void *x_bf16, const float *signs,
                                  void *x_e4m3, float *descale, long rows,
                                  int d, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * FP8 (e4m3) forward: the fa_fwd algorithm on e4m3 Q, K, V with fp32
 * descales (device scalars), producing bf16 O and fp32 LSE of the
 * *dequantised* scores: S = scale * q_descale * k_descale * Q8 K8^T,
 * O = softmax(S) (v_descale * V8).
 * [FA3] "FP8" (tensor-core throughput doubles at 8 bits) and the FP8 forward
 * figures of that page.  Q and K may have been rotated by the same random-sign
 * Hadamard matrix, which leaves Q K^T unchanged.
 *   q8 [B][Hq][N][d], k8, v8 [B][Hkv][N][d]: e4m3 bytes (in)
 *   q/k/v_descale: one fp32 device scalar each (in), as written by
 *   fa_hadamard_quant_fp8
 *   o_bf16 [B][Hq][N][d] bf16 (out); lse [B][Hq][N] fp32 (out)
 * d must be 128 (FA_ERR_UNSUPPORTED otherwise).  P is quantised to e4m3
 * before the P.V product, so O carries FP8 rounding of both operands.
 */
fa_status_t fa_fwd_fp8(const void *q8, const void *k8, const void *v8,
                       const float *q_descale, const float *k_descale,
                       const float *v_descale, void *o_bf16, float *lse,
                       int B, int Hq, int Hkv, int N, int d, int causal,
                       float scale, void *stream);

/*
 * Reads and clears the current device's status, which kernels set when
 * a bounded wait runs out, when packed sequence offsets read on the device
 * break the rules of fa_fwd_varlen, or when a kernel finds its shared-memory
 * window misaligned for its tiles (it then does nothing).  Synchronises
 * `stream` first.  Returns, in this order of precedence: FA_ERR_TIMEOUT (a
 * wait ran out), FA_ERR_CUDA (a kernel could not use its launch
 * configuration, or the copy of the status itself failed), FA_ERR_INVALID_ARG
 * (bad device-side offsets), else FA_OK.
 *   There is ONE status per device, shared by every caller, thread and
 *   stream of the process, and this call clears it for all of them.  With
 *   several streams or callers in flight, a status read on one stream may
 *   report a condition raised by work on another (and that other caller's
 *   later read then sees FA_OK).  Callers that need to attribute a failure
 *   must serialise their work and their reads of the status.
 */
fa_status_t fa_get_device_status(void *stream);

/*
 * Measurement aid: launches `blocks` blocks of 256 threads, each thread
 * running `iters` rounds of eight independent exp2 evaluations with the
 * instruction the softmax uses, and returns how many exp2 evaluations the
 * launch performs (or -1 for invalid arguments or a failed launch).  Timing
 * the launch on `stream` gives the exp2 throughput that bounds the softmax
 * ([FA3] "overlapping GEMM and softmax": the exponential runs on a separate
 * unit far slower than the tensor cores).
 *   sink [blocks * 256] fp32 (out, device, 16-byte aligned): per thread the
 *        sum of its eight chains, in [-8, -6.3], written so that the work
 *        is not removed
 *   blocks 1 .. 65535, iters 1 .. 2^24
 */
long long fa_probe_exp2(float *sink, int blocks, int iters, void *stream);

/*
 * Self-test of the bounded-wait machinery: launches one block that waits on a
 * barrier nothing will ever complete, with a limit of `timeout_us`
 * microseconds (1 .. 1000000).  The wait runs out, the kernel records
 * FA_ERR_TIMEOUT in the device status and returns; nothing faults or hangs.
 */
fa_status_t fa_selftest_bounded_wait(int timeout_us, void *stream);

/* Human-readable name of a status code (static storage). */
const char *fa_status_string(fa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
