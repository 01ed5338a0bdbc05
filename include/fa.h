/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused exact-attention forward library
 *         libfa_gb300.so.
 *
 * The operation (fa_fwd) is the tiled exact-attention forward pass:
 *
 *   O   = softmax(Q K^T * scale) V          per (batch, head), row-wise softmax
 *   LSE = log(sum_j exp(scale * q_i . k_j)) per query row (natural log)
 *
 * as defined on the pages "llm-infra-atlas / FlashAttention 01: IO awareness
 * and online softmax" (section 1 for the three-operation definition, section 3
 * for the tiled forward loop that emits O and LSE = m + log l, section 5 for
 * LSE's role in the backward pass) and "lumenova research-attention"
 * (section 01 for the shapes, section 03 for the per-row recurrence).  The
 * optional causal mask keeps key j for query row i iff j <= i.
 *
 * All functions have C linkage, never throw, never print and never abort the
 * process.  None of them allocates device memory.
 *
 * The first call on a device records per-device state in the library (the
 * kernels' shared-memory opt-in, the multiprocessor count and L2 size, and
 * for fa_fwd_splitkv_noalloc the device address of its fixed array).
 * Resetting a device (cudaDeviceReset) after this library has used it is not
 * supported: that state would be stale.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,          /* a required pointer is NULL                                  */
  FA_ERR_ALIGN = 2,         /* a tensor base pointer is not 16-byte aligned                */
  FA_ERR_SHAPE = 3,         /* B, H, Nk <= 0, a negative Nq, or a size beyond the limits   */
  FA_ERR_HEADDIM = 4,       /* d is not 64 or 128                                          */
  FA_ERR_CAUSAL_SHAPE = 5,  /* causal = 1 with Nq != Nk                                    */
  FA_ERR_LAUNCH = 6,        /* the CUDA runtime refused the launch or a set-up call        */
  FA_ERR_DEVICE = 7,        /* the current device is not compute capability 10.3 (GB300)  */
  FA_ERR_TIMEOUT = 8,       /* a kernel wait gave up (reported by fa_fwd_status)           */
  FA_ERR_SCALE = 9,         /* scale is not a finite positive number                       */
  FA_ERR_POINTER = 10,      /* a tensor pointer is not device memory of the current device */
  FA_ERR_WORKSPACE = 11     /* split-KV workspace missing or smaller than required         */
} fa_status;

/*
 * fa_fwd -- fused attention forward on `stream` (asynchronous; no host sync).
 *
 * q    [B, H, Nq, d] bf16, contiguous row-major (d fastest), device memory.
 * k, v [B, H, Nk, d] bf16, contiguous, device memory.
 * o    [B, H, Nq, d] bf16 output, contiguous, device memory; must not overlap
 *      q, k, v or lse.
 * lse  [B, H, Nq] fp32 output: natural-log log-sum-exp of the scaled logits of
 *      each query row (so that P = exp(scale * q.k - LSE)).
 * d    head dimension, 64 or 128.
 * scale  multiplies q.k before the softmax (1/sqrt(d) for standard attention);
 *        must be finite and > 0.
 * causal 0: every key is visible; 1: key j is visible to row i iff j <= i
 *        (requires Nq == Nk).
 *
 * Arithmetic: bf16 products accumulated in fp32 on the tensor cores, softmax
 * in fp32 (base-2 exponentials with log2(e) folded into the scale), the
 * probabilities rounded to bf16 for the P.V product, fp32 accumulation of O,
 * one division at the end by the row sum with the row's largest probability
 * counted as rounded for P.V (so a row dominated by one key returns that
 * key's V), O rounded to bf16 (nearest even).  LSE uses the exact fp32 sum.
 *
 * Ownership: the caller owns all five buffers; the library keeps no pointer
 * after the call returns and allocates nothing.
 * Errors: argument problems return a code before anything is launched and
 * nothing is written.  Nq == 0 is a successful no-op; q, o and lse may then be
 * NULL (k and v may not).  FA_ERR_LAUNCH is
 * returned if the launch itself fails, and by every call of a build whose
 * forward kernels did not get the register count their warpgroup register
 * split assumes (checked once per device, before any launch); faults during
 * execution surface, as usual for CUDA, at the next synchronising call on
 * the stream.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
           int Nk, int d, float scale, int causal, cudaStream_t stream);

/*
 * fa_fwd_window -- fa_fwd under a sliding-window mask (the "sliding" mask that
 * "llm-infra-atlas / FlashAttention 01", section 3, names beside "causal" in
 * the tiled loop; the window form and its alignment are this library's
 * reading, the pages give no formula).
 *
 * Key j is visible to query row i iff
 *     i + (Nk - Nq) - window_left  <=  j  <=  i + (Nk - Nq) + window_right,
 * i.e. the window is aligned so that its diagonal ends at the last query and
 * the last key (bottom-right alignment); -1 leaves that side unbounded.
 * (-1, 0) is causal attention for any Nq and Nk; (-1, -1) is no mask.  A query
 * row that sees no key gets O = 0 and LSE = -inf.
 * Arguments otherwise as fa_fwd (no causal flag, Nq and Nk independent);
 * window_left or window_right below -1 returns FA_ERR_SHAPE.
 */
int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                  int Nk, int d, float scale, int window_left, int window_right, cudaStream_t stream);

/*
 * fa_fwd_splitkv -- the same operation as fa_fwd, with each query tile's K/V
 * range cut into n_splits slices processed by separate CTAs, for shapes whose
 * B * H * ceil(Nq / 256) CTAs would leave most of the GPU idle.
 *
 * Each slice s produces a partial result for its rows: O_s normalised by its
 * own row sum, and L_s = log2 of that row sum in base-2 scaled-logit units.
 * A second kernel on the same stream merges the slices by the rule under which
 * the online-softmax state (m, l, O) is insensitive to block order ("llm-infra-
 * atlas / FlashAttention 01", section 2).  It is launched as a programmatic
 * dependent of the first (it may be scheduled while the first one's last CTAs
 * run and waits on the device for its completion), so stream order and the
 * results are those of two plain launches:
 *   L = log2 sum_s 2^L_s,   O = sum_s 2^(L_s - L) O_s,   LSE = L * ln 2.
 * At d = 64 a CTA takes one query tile instead of two when the CTAs of tile
 * pairs would fill under half of the multiprocessors or more than all of
 * them; the slices, and so the results, are the same either way.
 *
 * Arguments as in fa_fwd, plus:
 * n_splits   requested slices, 1..64; the call uses ceil(n_kv / ceil(n_kv /
 *            n_splits)) of them, n_kv = ceil(Nk / 128).  With one slice this is
 *            exactly fa_fwd and the workspace is not touched.
 * workspace  device memory of at least fa_splitkv_workspace_bytes() bytes,
 *            16-byte aligned, owned by the caller, not read before it is
 *            written; it must not be used by anything else until the call's
 *            kernels have finished on `stream`.
 * Errors as fa_fwd, plus FA_ERR_SHAPE for n_splits outside 1..64 and
 * FA_ERR_WORKSPACE for a missing or short workspace.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                   int Nk, int d, float scale, int causal, int n_splits, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes fa_fwd_splitkv needs for these sizes (0 for invalid sizes):
 * fp32 partial O [splits, B*H*Nq, d] followed by fp32 partial L [splits, B*H*Nq]. */
size_t fa_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int n_splits);

/* Suggested n_splits for the current device: 1 when B * H * ceil(Nq / 256)
 * CTAs already cover its multiprocessors, otherwise enough slices (at most 16,
 * each of at least two K/V tiles) to fill them about once. */
int fa_splitkv_heuristic(int B, int H, int Nq, int Nk, int d, int causal);

/*
 * fa_bwd -- attention backward pass by recomputation from the forward's LSE
 * ("llm-infra-atlas / FlashAttention 01", section 5):
 *   P = exp(scale * Q K^T - LSE),  dV = P^T dO,  dP = dO V^T,
 *   D = rowsum(dO * O),  dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
 *
 * q, o, dout, dq  [B, H, Nq, d] bf16;  k, v, dk, dv  [B, H, Nk, d] bf16;
 * lse [B, H, Nq] fp32 as written by fa_fwd (natural log).  All contiguous,
 * 16-byte aligned device memory of the current device; outputs must not
 * overlap inputs.  causal as in fa_fwd (Nq == Nk).  Nq and Nk must be > 0.
 * workspace: device memory of at least fa_bwd_workspace_bytes(B, H, Nq)
 * bytes, owned by the caller (fp32 L = LSE * log2(e) and D per query, padded
 * to whole 128-row tiles); not read before it is written.
 * Two kernels run on `stream`: one per 128-row query tile for dQ (and L, D),
 * then one per 128-key tile for dK and dV; no atomics, so the result does not
 * depend on scheduling.  Errors as fa_fwd, plus FA_ERR_WORKSPACE.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_window -- fa_bwd under the sliding-window mask of fa_fwd_window (key j
 * kept for query row i iff i + (Nk - Nq) - window_left <= j <= i + (Nk - Nq) +
 * window_right; -1 leaves that side open, so (-1, 0) is the causal mask aligned
 * bottom-right, for any Nq and Nk).  o and lse must come from fa_fwd_window
 * with the same window: a row that keeps no key has lse = -inf and o = 0 there,
 * and its dQ is written as 0; a key that no row keeps gets dK = dV = 0.
 * Each kernel visits only the tiles its window reaches.
 * Arguments, workspace and errors as fa_bwd (no causal argument); a bound
 * below -1 is FA_ERR_SHAPE.
 */
int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int window_left,
                  int window_right, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes fa_bwd and fa_bwd_window need (0 for invalid sizes). */
size_t fa_bwd_workspace_bytes(int B, int H, int Nq);

/* Size of the fixed device array fa_fwd_splitkv_noalloc works in. */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv without a caller workspace and
 * without any allocation: the slice buffers live in a fixed 16 MiB array
 * (FA_NOALLOC_SCRATCH_BYTES) in the library's own device memory.  The pages
 * describe no counterpart; this entry point exists for callers that cannot
 * allocate device memory themselves, for instance code running inside a host
 * framework that owns the whole device memory pool, or a latency path where a
 * cudaMalloc and the synchronisation it implies are not allowed.
 *
 * Arguments and results as fa_fwd_splitkv.  Sizes whose workspace
 * (fa_splitkv_workspace_bytes) exceeds FA_NOALLOC_SCRATCH_BYTES return
 * FA_ERR_WORKSPACE before anything is launched.  No cudaMalloc, cudaFree or
 * other allocating call is made.
 * Every GPU that loads the library holds the array until the process exits.
 * The first call on a device looks up the array's device address there (with
 * that device current); make that first call before any stream capture.
 * All calls share the one array, which keeps whatever the last call left in
 * it: calls whose kernels overlap on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller.  Nothing has to
 * be cleared between calls: every value the merge reads is written earlier in
 * the same call.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                           int Nq, int Nk, int d, float scale, int causal, int n_splits, cudaStream_t stream);

/* Human-readable text for a status code (static storage, never NULL). */
const char* fa_strerror(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

/*
 * fa_fwd_status -- synchronise `stream`, then report whether any kernel of
 * this library (forward, split-KV, backward) on the current device gave up on
 * a wait (FA_ERR_TIMEOUT) since the last clear.  Every wait inside the kernels
 * is bounded (about 2 s); a wait that runs out records the failing role in the
 * device status word (bit 0, and bits 8.. = 1 softmax/compute, 2 producer,
 * 4 MMA issuer, 8 epilogue), the CTA drains its in-flight copies and MMAs,
 * frees its tensor memory and exits.  *detail (optional) receives the raw
 * status word.  clear != 0 resets the word.  Returns FA_OK, FA_ERR_TIMEOUT, or
 * FA_ERR_LAUNCH if synchronisation failed.
 */
int fa_fwd_status(cudaStream_t stream, unsigned int* detail, int clear);

/*
 * fa_probe_exp2 -- measure how many 2^x results per SM clock cycle the current
 * device produces (median over the SMs of one CTA per SM running independent
 * exp2 chains).  Not an operation of the pages: method 0 times ex2.approx on
 * the special-function unit, the denominator of the forward kernel's
 * exponential-unit roofline; method 1 times a cubic polynomial on the FMA and
 * integer pipes, the kind of offload that the page "pinghaoyang FlashAttention
 * 1-4 guide" (FA4 section, emulated exponential) describes for Blackwell.
 *
 * method      0 or 1 (anything else: FA_ERR_SHAPE).
 * per_clk_sm  host pointer receiving the rate.
 * stream      the probe runs on it; the call synchronises the stream.
 * Uses no caller memory.  Returns FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_DEVICE
 * (not compute capability 10.3) or FA_ERR_LAUNCH; the value is written only
 * on FA_OK.
 */
int fa_probe_exp2(int method, double* per_clk_sm, cudaStream_t stream);

/*
 * fa_selftest_wait -- exercise the bounded wait that every kernel of this
 * library uses, without any fault: one CTA waits on an mbarrier phase that
 * nothing completes.  Not an operation of the pages.
 *
 * mode 0: the wait must give up when its time limit (about 2 s) runs out;
 * mode 1: another warp raises the CTA's abort flag after about 1 ms and the
 *         wait must give up on it at once.
 * word     receives the self-test's status word: bit 0 set when the wait gave
 *          up; bits 8.. = 1 (time limit) or 2 (abort flag).
 * wait_ns  receives how long the wait lasted, in nanoseconds.
 * Synchronises `stream`; the device status word of the other kernels is not
 * touched.  Returns FA_ERR_NULL, FA_ERR_SHAPE (mode), FA_ERR_DEVICE or
 * FA_ERR_LAUNCH; the outputs are written only on FA_OK.
 */
int fa_selftest_wait(int mode, unsigned int* word, unsigned long long* wait_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
