/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention library, libattn.so.
 *
 * The operation is scaled dot-product attention, O = softmax(scale * Q K^T) V
 * per (batch, query head), from "Scheduling Data to Compute: Hierarchical Data
 * Pipelining for LLM Training on AMD GPUs", section 2.1, Eq. (1), computed the
 * FlashAttention way that the same section's Algorithm 0 describes: K/V tiles
 * stream through on-chip memory while the softmax state and the output
 * accumulator stay on chip. The backward pass is the exact gradient of Eq. (1)
 * for the three products whose operand layouts the paper's Table 3 lists
 * (scores, query gradient dS*K, key gradient dS^T*Q) plus dV = P^T*dO.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers on the current CUDA device,
 *    owned by the caller, contiguous, 16-byte aligned.
 *  - bf16 tensors use the [B, S, H, D] layout ("BSHD"): q, o, dO, dq are
 *    [B, S, Hq, D]; k, v, dk, dv are [B, S, Hkv, D].
 *  - lse is fp32 [B, Hq, S]: LSE_i = ln sum_j exp(scale * q_i . k_j) over the
 *    keys row i sees (natural log, scaled scores).
 *  - Grouped-query attention: Hq must be a multiple of Hkv; query head h
 *    reads key/value head h / (Hq / Hkv) (contiguous groups).
 *  - causal != 0: query i sees keys j <= i. causal == 0: all keys.
 *  - D must be 64 or 128. Any S >= 0 up to 2^24 is accepted. B == 0 or
 *    S == 0 (with otherwise valid sizes) is a no-op that returns ATTN_OK; the
 *    pointers are then not read and may be NULL.
 *  - Checks run in this order: sizes (INVALID_ARG / UNSUPPORTED), scale, the
 *    empty-problem no-op, pointers, workspace, device.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream). The library allocates no memory per call and never
 *    synchronises the host, except under ATTN_CHECK_STATUS=1 in the
 *    environment, where each call waits for its kernels and reads back the
 *    device status word.
 *  - Arguments are validated before any launch; a failed check launches
 *    nothing and returns the code named below.
 *  - The sparse top-k entry points (attn_sparse_*) take their own layouts
 *    (per-token lists over a key/value pool), stated at their declarations.
 */
#ifndef ATTN_GB300_ATTN_H_
#define ATTN_GB300_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size or scale */
  ATTN_ERR_UNSUPPORTED = 2, /* valid but unsupported: D not in {64,128}, not an sm_103 GPU */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
  ATTN_ERR_TIMEOUT = 4,     /* a kernel's bounded pipeline wait ran out (reported via status) */
  ATTN_ERR_WORKSPACE = 5,   /* workspace null, misaligned or smaller than attn_bwd_workspace_size */
  ATTN_ERR_BOUNDS = 6       /* bounds-checked build only (ATTN_DEBUG_BOUNDS): an index check
                               failed, the access was skipped (reported via status) */
} attn_status_t;

/*
 * Forward: o = softmax(scale * q k^T) v and the row log-sum-exp -- the
 * paper's section 2.1, Eq. (1), computed as that section's Algorithm 0
 * streams it (online softmax over K/V tiles, state kept on chip).
 *
 *   q     [B,S,Hq,D]  bf16, in
 *   k, v  [B,S,Hkv,D] bf16, in
 *   o     [B,S,Hq,D]  bf16, out (overwritten): O rounded to nearest bf16.
 *                     The probabilities enter P V as bf16 values, and O is
 *                     divided by the sum of those same bf16 values, so O is a
 *                     weighted mean of V rows whose weights are within bf16
 *                     rounding of the softmax weights.
 *   lse   [B,Hq,S]    fp32, out (overwritten); needed by attn_bwd. From the
 *                     fp32 probabilities: ln sum_j exp(scale q_i . k_j).
 *   scale finite, e.g. 1/sqrt(D)
 *
 * Errors: ATTN_ERR_INVALID_ARG for a null or non-16-byte-aligned pointer,
 * B, S < 0, Hq, Hkv <= 0, Hq % Hkv != 0, or a non-finite scale;
 * ATTN_ERR_UNSUPPORTED for D not in {64, 128}, S > 2^24, or a device that is
 * not sm_103; ATTN_ERR_CUDA if tensor-map encoding or a launch fails.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int S, int D, int causal, float scale, void* stream);

/*
 * Forward that also writes the low-order part of the output (same passage
 * as attn_fwd; the residual is this library's addition for the backward):
 *
 *   o_lo  [B,S,Hq,D]  bf16, out (overwritten): bf16(O_fp32 - o), so o + o_lo
 *                     carries the kernel's fp32 O to about 16 significant
 *                     bits. o and lse are bit for bit those of attn_fwd.
 *
 * Passing o_lo on to attn_bwd gives the backward Dvec = rowsum(dO * O) from
 * that O in its cheap preprocess pass; without it, attn_bwd computes Dvec in
 * an extra pass (attn_bwd_dvec), because bf16 o alone holds O to about 8
 * bits, too few for the gradient tolerance (max-abs error <= 5e-2 of the
 * exact gradient's rms) with a sharp softmax. Other arguments and errors as
 * attn_fwd (o_lo may not be NULL here).
 */
attn_status_t attn_fwd_residual(const void* q, const void* k, const void* v, void* o, void* o_lo,
                                float* lse, int B, int Hq, int Hkv, int S, int D, int causal,
                                float scale, void* stream);

/*
 * Size in bytes of the device workspace attn_bwd needs for these sizes (the
 * paper has no counterpart: this library's workspace convention; the
 * status word, and fp32 Dvec and log2-scaled LSE rows with the sequence
 * padded to a multiple of 128). Returns 0 for invalid or unsupported sizes,
 * and for empty problems.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int S, int D);

/*
 * Backward: the gradients of L = sum(dO * O) with respect to q, k and v,
 * written in fp32. The paper gives no backward equations; this is the exact
 * gradient of its Eq. (1) (section 2.1), with the operand layouts of its
 * Table 3 (scores Q K^T, query gradient dS K, key gradient dS^T Q) and
 * dV = P^T dO:
 *   dP = dO V^T, Dvec_i = sum_j P_ij dP_ij, dS = P * (dP - Dvec),
 *   dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
 *
 *   q, k, v, o, lse  as passed to / returned by attn_fwd (in)
 *   dO    [B,S,Hq,D]  bf16, in
 *   dq    [B,S,Hq,D]  fp32, out (overwritten)
 *   dk,dv [B,S,Hkv,D] fp32, out (overwritten; for GQA each sums over the
 *                     Hq/Hkv query heads of its group)
 *   o_lo  [B,S,Hq,D]  bf16, in, optional (NULL allowed): the residual from
 *                     attn_fwd_residual. Given, Dvec = rowsum(dO * (o + o_lo))
 *                     in the preprocess pass (two kernels run: preprocess and
 *                     main). NULL: Dvec = sum_j P_ij dP_ij from the attn_bwd_dvec
 *                     pass (three kernels: preprocess, Dvec pass, main; the
 *                     Dvec pass costs about as much as a forward).
 *   workspace        device memory of at least attn_bwd_workspace_size()
 *                    bytes, 256-byte aligned, owned by the caller; its
 *                    contents on entry do not matter and are clobbered,
 *                    except its status word: a timeout that an earlier call
 *                    recorded there stays until attn_check_status(workspace)
 *                    reads and clears it.
 *
 * Runs its kernels in order on `stream`: the preprocess pass (Dvec as above,
 * log2-scaled LSE, dq zeroed), the Dvec pass when o_lo is NULL, and the
 * KV-parallel main kernel (dK and dV per key tile; dQ added into dq by fp32
 * reductions, so dq is reproducible only up to fp32 summation order). Inside
 * the main kernel P and dS enter the gradient products as bf16 hi/lo pairs
 * (about 16 significant bits).
 *
 * Errors: as attn_fwd, plus ATTN_ERR_WORKSPACE for a null or misaligned
 * workspace or one smaller than attn_bwd_workspace_size().
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, void* dq, void* dk, void* dv, const void* o_lo, int B,
                       int Hq, int Hkv, int S, int D, int causal, float scale, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * The stages of attn_bwd as separate calls, for callers that time or
 * schedule them one by one (the same gradient of Eq. (1), section 2.1; the
 * split into stages is this library's). Arguments and errors are those of attn_bwd; each
 * stage reads what the previous one left in `workspace` and `dq`, so they
 * must run in order on one stream with the same arguments:
 *   attn_bwd_preprocess: Dvec = rowsum(dO * (o + o_lo)) (o alone when o_lo is
 *     NULL), the log2-scaled LSE rows, dq zeroed;
 *   attn_bwd_dvec (optional, between the two): overwrites Dvec with
 *     sum_j P_ij dP_ij computed from q, k, v, dO and the LSE rows -- what
 *     attn_bwd runs when o_lo is NULL (window as in attn_bwd_ex, 0 = none);
 *   attn_bwd_main: the gradient products.
 * Each attn_bwd_main call needs a fresh attn_bwd_preprocess before it: the
 * main stage adds into the dq that the preprocess zeroed, and the preprocess
 * also restarts the item counter that the main stage's persistent launch
 * takes its work from (a word of the workspace's status region).
 */
attn_status_t attn_bwd_preprocess(const void* o, const void* o_lo, const void* dO,
                                  const float* lse, void* dq, int B, int Hq, int Hkv, int S, int D,
                                  void* workspace, size_t workspace_bytes, void* stream);
attn_status_t attn_bwd_dvec(const void* q, const void* k, const void* v, const void* dO, int B,
                            int Hq, int Hkv, int S, int D, int causal, int window, float scale,
                            void* workspace, size_t workspace_bytes, void* stream);
attn_status_t attn_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dq,
                            void* dk, void* dv, int B, int Hq, int Hkv, int S, int D, int causal,
                            float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Sliding-window causal attention: forms of attn_fwd / attn_fwd_residual,
 * attn_bwd and attn_bwd_main with a `window` argument. The window is the
 * dense part of the sparse attention in "Scheduling Data to Compute:
 * Hierarchical Data Pipelining for LLM Training on AMD GPUs" (§4.1, Table 7
 * caption: every query attends to a 128-token sliding window; §3's cr0
 * kernels). With window = W > 0, query i sees keys i-W+1..i (at most W keys,
 * its own included); the kernels skip key tiles that no row of a query tile
 * sees. window = 0 is plain attention and gives the results of the calls
 * without `window`.
 *
 *   window  >= 0; a window > 0 needs causal != 0 (else ATTN_ERR_INVALID_ARG,
 *           checked right after the sizes). W >= S is plain causal attention.
 *   o_lo    (attn_fwd_ex) NULL for the inference forward of attn_fwd, or the
 *           residual output of attn_fwd_residual.
 *
 * Other arguments, results and errors are those of the calls without
 * `window`. The backward must get the same causal and window values as the
 * forward that produced lse (and o, o_lo).
 */
attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, void* o_lo,
                          float* lse, int B, int Hq, int Hkv, int S, int D, int causal, int window,
                          float scale, void* stream);
attn_status_t attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv,
                          const void* o_lo, int B, int Hq, int Hkv, int S, int D, int causal,
                          int window, float scale, void* workspace, size_t workspace_bytes,
                          void* stream);
attn_status_t attn_bwd_main_ex(const void* q, const void* k, const void* v, const void* dO,
                               void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D,
                               int causal, int window, float scale, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory. The paper has no counterpart: this is a packaging variant of
 * attn_bwd, not part of the method.
 *
 * Who needs it: code that runs inside a host framework or plugin interface
 * which hands it only the tensors of one call and owns every allocation
 * itself, and code on a latency-critical path where a cudaMalloc (which can
 * synchronise the device) is not allowed. Such callers cannot provide the
 * workspace that attn_bwd asks for.
 *
 * Instead of a caller workspace the call uses one scratch array compiled into
 * the library: 16 MiB of device memory, held on every GPU that has made such
 * a call until the process exits. Problems whose
 * attn_bwd_workspace_size(B, Hq, Hkv, S, D) exceeds 16 MiB (about
 * B * Hq * ceil(S/128)*128 > 2,097,000 query rows) are rejected with
 * ATTN_ERR_WORKSPACE before anything is launched.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress). Under CUDA's lazy module loading that
 * first call also loads the module holding the array, which reserves its
 * 16 MiB and may synchronise the device: make one warm-up call outside any
 * latency-critical path, and before any stream capture. After that the call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * The address is cached per device for the life of the process, so the call
 * does not survive cudaDeviceReset or a re-created primary context.
 *
 * A bounded wait that runs out inside it is reported by
 * attn_check_status(NULL), which reads the array's status word.
 *
 * All calls on a device share the one array, and it keeps the last call's
 * contents; each call rewrites every word it reads before reading it. Calls
 * whose kernels overlap on the GPU (different streams without ordering
 * between them) race on the array and give wrong results: order them.
 *
 * Arguments, results and the other errors are those of attn_bwd.
 */
attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const void* dO, const float* lse, void* dq, void* dk, void* dv,
                               const void* o_lo, int B, int Hq, int Hkv, int S, int D, int causal,
                               float scale, void* stream);

/*
 * Sparse top-k gather attention, forward ("Scheduling Data to Compute:
 * Hierarchical Data Pipelining for LLM Training on AMD GPUs", section 2.1:
 * each query token receives a top-k list of KV rows; the forward gathers them,
 * scores them and streams their values into the output; section 3 and
 * Table 7 for the list shapes: a 128-row window plus top-k compressed rows).
 *
 * For every batch b, token t and head h:
 *   O[b,t,h,:] = sum_j softmax_j(scale * q[b,t,h,:] . kp[b,idx[b,t,j],:])
 *                      * vp[b,idx[b,t,j],:]
 * over the slots j whose entry lies in [0, P); any other entry (e.g. -1) is an
 * empty slot. All heads of a token share its list and the one key/value pool
 * of its batch. A row listed twice counts twice.
 *   q   [B, T, H, DK] bf16      kp [B, P, DK] bf16     vp [B, P, DV] bf16
 *   idx [B, T, K] int32 (K a multiple of 4)
 *   o   [B, T, H, DV] bf16 (out)
 *   o_lo [B, T, H, DV] bf16 (out, optional): bf16(O - o), so that o + o_lo
 *        carries O to about 16 significant bits; NULL to skip.
 *   lse [B, H, T] fp32 (out): natural log-sum-exp of the scaled scores over
 *        the filled slots; a token with no filled slot gets O = 0 and
 *        LSE = -inf.
 * H is 1..128, DK and DV are 64 or 128 each (they may differ). Device
 * pointers, contiguous, 16-byte aligned; the caller owns every buffer.
 * Errors: ATTN_ERR_INVALID_ARG for bad sizes, null or misaligned pointers or
 * a non-finite scale; ATTN_ERR_UNSUPPORTED for other head dimensions or a
 * non-sm_103a device; ATTN_ERR_CUDA for a failed launch. B = 0 or T = 0 is a
 * no-op. Bounded pipeline waits report through attn_check_status(NULL).
 */
attn_status_t attn_sparse_fwd(const void* q, const void* kp, const void* vp, const int* idx,
                              void* o, void* o_lo, float* lse, int B, int T, int H, int P, int K,
                              int DK, int DV, float scale, void* stream);

/*
 * Sparse top-k gather attention, backward (same pages, section 2.1: the
 * backward gathers the listed vectors again for dQ and reduces a per-slot
 * dK/dV intermediate through the inverse of the top-k map).
 *
 * The exact gradient of sum(dO * O) for attn_sparse_fwd's O:
 *   dq  [B, T, H, DK] fp32 (out): scale * sum_j dS[h, j] kp[idx_j]
 *   dkp [B, P, DK] fp32 (out): for each pool row, the sum over every
 *       (token, slot) naming it of scale * sum_h dS[h, j] q[h]
 *   dvp [B, P, DV] fp32 (out): likewise of sum_h P[h, j] dO[h]
 * with P the forward's probabilities (recomputed from q, kp, vp and lse),
 * dS = P * (dP - Dvec), dP = dO vp^T, Dvec = rowsum(dO * O).
 * o [B, T, H, DV] bf16 and lse [B, H, T] are attn_sparse_fwd's outputs; o_lo
 * (optional, NULL to skip) its residual, which makes Dvec exact to about 16
 * bits; dO [B, T, H, DV] bf16. Empty slots and tokens without a filled slot
 * contribute nothing. Sizes, layouts and the other arguments are those of
 * attn_sparse_fwd. dkp and dvp are overwritten (zeroed, then accumulated);
 * repeated rows accumulate every occurrence.
 * workspace: device memory, 256-byte aligned, of at least
 * attn_sparse_bwd_workspace_size(B, T, H) bytes, owned by the caller; it also
 * holds the status word that attn_check_status(workspace) reads.
 * Errors: those of attn_sparse_fwd, and ATTN_ERR_WORKSPACE for a missing,
 * misaligned or small workspace.
 */
size_t attn_sparse_bwd_workspace_size(int B, int T, int H);
attn_status_t attn_sparse_bwd(const void* q, const void* kp, const void* vp, const int* idx,
                              const void* o, const void* o_lo, const void* dO, const float* lse,
                              float* dq, float* dkp, float* dvp, int B, int T, int H, int P, int K,
                              int DK, int DV, float scale, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Static, human-readable name of a status code (library convention; the paper
 * has no counterpart). */
const char* attn_status_string(attn_status_t status);

/*
 * Failure reporting of this library (the paper has no counterpart).
 * Reads (and clears) the device status words that the kernels set when a
 * bounded pipeline wait ran out: the forward kernels' word of the current
 * device, and the backward word of `workspace` -- or, with workspace NULL,
 * the word of attn_bwd_noalloc's scratch array (once a call on this device
 * has looked the array up). A recorded timeout stays in its word until this
 * call reads it. Synchronises the device. Returns ATTN_OK, ATTN_ERR_TIMEOUT,
 * ATTN_ERR_BOUNDS (a library built with ATTN_DEBUG_BOUNDS whose index check
 * failed; that code takes precedence), or ATTN_ERR_CUDA if the read itself
 * failed.
 */
attn_status_t attn_check_status(void* workspace);

/*
 * (Library control; the paper has no counterpart.)
 * Sets the time limit of every bounded wait inside the kernels launched after
 * this call on this process, in nanoseconds (default 2e9, i.e. 2 s; 0 restores
 * the default). A limit shorter than a pipeline step makes the kernels give
 * up and report ATTN_ERR_TIMEOUT instead of computing; it exists for testing
 * that path.
 */
void attn_set_wait_timeout_ns(uint64_t ns);

/*
 * Testing hook for the failure path (not part of the method): with bit 0 of
 * mask set, the forward kernels' MMA warp issues nothing; with bit 1 set, the
 * backward main kernel's does. The other warps' bounded waits then run out
 * after the wait time limit, the kernels stop early without touching their
 * outputs, and attn_check_status() reports ATTN_ERR_TIMEOUT. No fault, trap
 * or hang is involved; 0 restores normal operation.
 */
void attn_set_fault_injection(int mask);

#ifdef __cplusplus
}
#endif
#endif /* ATTN_GB300_ATTN_H_ */
