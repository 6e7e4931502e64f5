/*
 * linattn.h - C ABI of the GB300 kernelized linear attention library (liblinattn.so).
 *
 * The library computes kernelized (linear) attention
 *
 *     out_i = phi(q_i)^T S / max(phi(q_i)^T z, eps),
 *     S = sum_j phi(k_j) v_j^T  in R^{r x d_v},   z = sum_j phi(k_j)  in R^r,
 *
 * ("Reassociate a feature-map kernel without claiming exact softmax", ¶1-2;
 *  "Performer - Random Feature Softmax Approximation", §2 Step 5 and §3),
 * in bidirectional form (j over the whole sequence) and causal form (j <= i,
 * the inclusive prefix recurrence of "The Kernel Zoo", §1.3 and §5.4), over
 * packed sequences whose state resets at every boundary ("Reassociate a
 * feature-map kernel", ¶4).  The denominator is clamped from below at eps,
 * as the "Performer" §3 sketch does (its .clamp(min=1e-6)).
 *
 * Feature maps phi:
 *   LA_MAP_IDENTITY  phi(x) = x, r = d_k            ("The Kernel Zoo", §1.3)
 *   LA_MAP_ELU1      phi(x) = elu(x) + 1, r = d_k   ("The Kernel Zoo", running example;
 *                    x + 1 for x > 0, exp(x) otherwise)
 *   LA_MAP_FAVOR     phi(x) = exp(Omega x - |x|^2/2) / sqrt(r), Omega in R^{r x d_k}
 *                    ("The Kernel Zoo", §4.2 and §5.4; "Performer", §2 Step 3)
 *   LA_MAP_DPFP      DPFP-nu: x~ = relu([x, -x]) in R^{2 d_k}; feature (s-1) 2 d_k + i
 *                    = x~_i x~_{(i+s) mod 2 d_k} for s = 1..nu; r = 2 d_k nu with
 *                    1 <= nu <= 2 d_k - 1 ("The Kernel Zoo", §6.3; Omega unused).
 *                    Causal bf16 calls with d_k = d_v = 64 and nu <= 2 run on the
 *                    tensor cores; every other DPFP call on CUDA cores.
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout.   q, k: [T, H, d_k]; v, out: [T, H, d_v]; all contiguous row-major
 *           (d innermost), T = total packed tokens.  Omega: [r, d_k] fp32
 *           row-major, shared by every head and sequence (the single omega of
 *           the "Performer" §3 sketch).  Element type of q, k, v and out is
 *           given by `dtype` (LA_F32: float, LA_BF16: bfloat16 bits).
 * Packing.  cu_seqlens: device int32 [nseq + 1], cu_seqlens[0] = 0,
 *           non-decreasing, cu_seqlens[nseq] = T.  Sequence s owns rows
 *           cu_seqlens[s] .. cu_seqlens[s+1]-1.  NULL means nseq sequences of
 *           T / nseq tokens each (a B x N batch).  Empty sequences are allowed.
 * Memory.   Every pointer is device memory owned by the caller, except where
 *           a call says "host".  The library allocates nothing and keeps no
 *           state between calls; calls on different streams with different
 *           workspaces may run concurrently.  Inputs are read only; `out` must
 *           not alias them.  Pointers must be aligned to their element size;
 *           16-byte aligned q/k/v/out/omega enable the tensor-core path.
 * Streams.  `stream` is a cudaStream_t (NULL: the legacy default stream).
 *           Compute calls only enqueue work and return; they never
 *           synchronise, except la_check_cu_seqlens and la_workspace_error.
 * Errors.   Argument checks run on the host before anything is enqueued and
 *           return LA_ERR_INVALID_ARG / LA_ERR_UNSUPPORTED / LA_ERR_WORKSPACE;
 *           nothing is written in that case.  A failed launch returns
 *           LA_ERR_CUDA.  Problems only the device can see (cu_seqlens contents
 *           that break the rules above, a bounded wait inside a kernel that ran
 *           out) are recorded in the workspace's error word and the affected
 *           work is skipped; read it with la_workspace_error.  No kernel traps.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(LA_BUILDING_LIBRARY)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size or a bad combination       */
    LA_ERR_UNSUPPORTED = 2,   /* valid, but beyond the library's size limits           */
    LA_ERR_WORKSPACE = 3,     /* workspace_bytes < la_workspace_bytes(...)             */
    LA_ERR_CUDA = 4,          /* a CUDA call or kernel launch failed                   */
    LA_ERR_DEVICE = 5         /* the device recorded an error (la_workspace_error)     */
} la_status;

typedef enum { LA_MAP_IDENTITY = 0, LA_MAP_ELU1 = 1, LA_MAP_FAVOR = 2, LA_MAP_DPFP = 3 } la_map;
typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

/*
 * Normalisation of the output (la_forward, la_decode_step):
 *   LA_NORM_ATTENTION  out = phi(q)^T S / max(phi(q)^T z, eps): a weighted
 *                      average of the values ("Reassociate a feature-map
 *                      kernel" ¶1-2; what la_forward_bidir/causal compute).
 *   LA_NORM_NONE       out = phi(q)^T S: the unnormalised fast-weight output
 *                      ("The Kernel Zoo" §1.2-1.4, the fast weight programmer).
 *   LA_NORM_SUM        every query and key feature vector is divided by the
 *                      sum of its components, phi'(x) = phi(x) /
 *                      max(sum_f phi(x)_f, eps), and out = phi'(q)^T S' with
 *                      S' built from phi'(k); there is no attention
 *                      denominator ("The Kernel Zoo" §7.2-7.4).  Meant for the
 *                      non-negative maps: LA_MAP_IDENTITY is rejected.
 */
typedef enum { LA_NORM_ATTENTION = 0, LA_NORM_NONE = 1, LA_NORM_SUM = 2 } la_norm;

/* Device error codes stored in the workspace error word. */
#define LA_DEVERR_NONE 0
#define LA_DEVERR_CU_SEQLENS 1    /* cu_seqlens broke the packing rules: nothing computed */
#define LA_DEVERR_WAIT_TIMEOUT 2  /* a bounded in-kernel wait ran out: output incomplete */
#define LA_DEVERR_RANGE 3         /* tensor-core path: a value fell outside what its fp16
                                     operands hold after scaling and was clamped; the result
                                     is finite but may be less accurate (reported only when
                                     neither error above was recorded) */

/* Size limits (checked on the host). */
#define LA_MAX_DK 256
#define LA_MAX_DV 256
#define LA_MAX_R 512

/*
 * la_feature_map - phi applied to every row of x.
 *   x:      [T, H, d] of dtype;  omega: [r, d] fp32 (FAVOR only, else may be NULL)
 *   phi:    [T, H, r] fp32 output
 *   map:    la_map;  r must equal d for identity and ELU+1, and be 2 d nu with
 *           1 <= nu <= 2d - 1 for DPFP (LA_ERR_INVALID_ARG otherwise).
 * Defined by "The Kernel Zoo" §4.2 boxed map (FAVOR+), the running example
 * (ELU+1), §1.3 (identity) and §6.3 boxed map (DPFP-nu).  For LA_BF16 input the values are those the
 * forward calls use before they round phi to bf16 for the tensor cores.
 */
LA_API la_status la_feature_map(const void* x, const float* omega, int map, int dtype,
                         int64_t T, int H, int d, int r, float* phi, void* stream);

/*
 * la_forward_bidir - bidirectional kernelized attention.
 *   For every sequence and head: S = Phi_K^T V, z = Phi_K^T 1 over the whole
 *   sequence, out_i = phi(q_i)^T S / max(phi(q_i)^T z, eps)
 *   ("Performer" §2 Step 5 and the §3 sketch; "Linear attention & kernelized
 *   approximations", "Build the state once").
 *   q, k: [T, H, d_k]; v, out: [T, H, d_v] (dtype); omega: [r, d_k] fp32 or NULL.
 *   eps >= 0.  workspace: device scratch of at least
 *   la_workspace_bytes(0, ...) bytes, 256-byte aligned; its contents on entry
 *   do not matter.  Sums over tokens are fp32 and run in a fixed order, so the
 *   result is deterministic for a given device.
 */
LA_API la_status la_forward_bidir(const void* q, const void* k, const void* v, const float* omega,
                           int map, int dtype, const int32_t* cu_seqlens, int nseq,
                           int64_t T, int H, int d_k, int d_v, int r, float eps,
                           void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_forward_causal - causal kernelized attention by prefix sums.
 *   S_i = sum_{j<=i} phi(k_j) v_j^T, z_i = sum_{j<=i} phi(k_j) within each
 *   sequence (key i is visible to query i), out_i = phi(q_i)^T S_i /
 *   max(phi(q_i)^T z_i, eps) ("The Kernel Zoo" §1.3 and §5.4; "Reassociate a
 *   feature-map kernel" ¶4; "Performer" §2, prefix-sum recurrence).  The state
 *   is carried in fp32.  Arguments as for la_forward_bidir, with
 *   la_workspace_bytes(1, ...).
 */
LA_API la_status la_forward_causal(const void* q, const void* k, const void* v, const float* omega,
                            int map, int dtype, const int32_t* cu_seqlens, int nseq,
                            int64_t T, int H, int d_k, int d_v, int r, float eps,
                            void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_forward - the general forward call: either form, a normalisation variant
 *   and a state carried between calls.
 *   causal:    1 as la_forward_causal, 0 as la_forward_bidir.
 *   norm:      la_norm (LA_ERR_INVALID_ARG for LA_NORM_SUM with the identity map).
 *   state_in:  NULL (every sequence starts from S = 0, z = 0) or fp32
 *              [nseq, H, r, d_v + 1]: row f of the (sequence, head) block holds
 *              S[f, 0 .. d_v-1] followed by z[f].  Causal: the state the
 *              sequence's first token adds to, so a long sequence can be run
 *              as consecutive calls ("The Kernel Zoo" §9.3: fast weights
 *              carried from one segment to the next).  Bidirectional: added to
 *              the whole-sequence sums that every query reads.  Under
 *              LA_NORM_SUM it holds sums of sum-normalised key features.
 *   state_out: NULL or the same layout: state_in (or 0) plus the sums over the
 *              whole sequence, i.e. the state after its last token.  Written
 *              for every sequence, empty ones included.  May be the same
 *              array as state_in (the call reads state_in before any of
 *              state_out is written); must not overlap q, k, v, out or the
 *              workspace otherwise.
 *   Other arguments as for la_forward_bidir / la_forward_causal, with
 *   la_workspace_bytes(causal, ...).  Both state arrays must be 4-byte aligned.
 *   LA_NORM_SUM on the tensor-core path (shapes la_selected_path reports as 1,
 *   no carried state): the plan phase computes the feature sums of every q and
 *   k row and writes v / max(sigma_k, eps) into `out`, the kernels form the
 *   unnormalised output of those values, and the output phase divides it by
 *   max(sigma_q, eps).  With a carried state it runs on the CUDA-core kernels.
 */
LA_API la_status la_forward(int causal, int norm, const void* q, const void* k, const void* v,
                            const float* omega, int map, int dtype, const int32_t* cu_seqlens, int nseq,
                            int64_t T, int H, int d_k, int d_v, int r, float eps,
                            const float* state_in, float* state_out, void* out, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * la_decode_step - one new token for each of B independent causal sequences:
 *   the recurrence's single step S += phi(k) v^T, z += phi(k), then the query
 *   reads the updated state, out = phi(q)^T S / max(phi(q)^T z, eps) (key i
 *   visible to query i: "Reassociate a feature-map kernel" ¶4; "The Kernel
 *   Zoo" §1.3).  norm as for la_forward.
 *   q, k:  [B, H, d_k]; v, out: [B, H, d_v] (dtype); omega as for la_forward.
 *   state: fp32 [B, H, r, d_v + 1] in the la_forward state layout, read and
 *          updated in place (the state_out of a causal la_forward call over
 *          the prompt continues directly).
 *   Computed in fp32 on CUDA cores for every dtype; bf16 outputs are rounded
 *   once.  B = 0 enqueues nothing.  Needs no workspace.
 */
LA_API la_status la_decode_step(const void* q, const void* k, const void* v, const float* omega, int map,
                                int dtype, int norm, int B, int H, int d_k, int d_v, int r, float eps,
                                float* state, void* out, void* stream);

/*
 * la_backward - gradients of L = sum(dout * out) with respect to q, k and v,
 *   where out is what la_forward(causal, norm, ...) returns for the same
 *   arguments without a carried state ("Reassociate a feature-map kernel" ¶5
 *   asks for errors in gradients as well as outputs).  With g_i the gradient
 *   with respect to num_i | den_i (dout_i / max(den_i, eps) and
 *   -(dout_i . out_i) / den_i, 0 where the clamp holds; dout_i and 0 without
 *   attention normalisation): dphi(q_i) = S_i g_i, dphi(k_j) = R_j [v_j | 1],
 *   dv_j = R_j^T phi(k_j) restricted to the first d_v entries, with S_i the
 *   forward state and R_j = sum_{i >= j} phi(q_i) g_i^T (every i for the
 *   bidirectional form), then the chain rule through the feature map (and the
 *   sum normalisation).  Omega is treated as a constant.
 *   dout: [T, H, d_v]; dq, dk: [T, H, d_k]; dv: [T, H, d_v], all of `dtype`,
 *   written for every row; must not overlap the inputs or each other.
 *   workspace: at least la_backward_workspace_bytes(...) bytes, 256-byte
 *   aligned.  Computed in fp32 on CUDA cores for every dtype (bf16 gradients
 *   are rounded once); the output is recomputed, not read.  Other arguments
 *   and errors as for la_forward.
 */
LA_API la_status la_backward(int causal, int norm, const void* q, const void* k, const void* v,
                             const float* omega, int map, int dtype, const int32_t* cu_seqlens,
                             int nseq, int64_t T, int H, int d_k, int d_v, int r, float eps,
                             const void* dout, void* dq, void* dk, void* dv, void* workspace,
                             size_t workspace_bytes, void* stream);

/* la_backward_workspace_bytes - scratch size for la_backward (0 for arguments it rejects). */
LA_API size_t la_backward_workspace_bytes(int causal, int map, int dtype, int has_cu_seqlens, int nseq,
                                          int64_t T, int H, int d_k, int d_v, int r);

/*
 * la_forward_phase - one phase of a forward call, for callers that time or
 *   interleave the kernels.  la_forward (and so la_forward_bidir /
 *   la_forward_causal) is exactly phases LA_PHASE_PLAN .. LA_PHASE_OUTPUT
 *   called in order with the same arguments and workspace:
 *     LA_PHASE_PLAN    split the packed sequences into segments (reads cu_seqlens)
 *     LA_PHASE_STATE   per-segment state sum_j phi(k_j) [v_j | 1]^T
 *     LA_PHASE_SCAN    state entering each segment (causal: exclusive prefix
 *                      over the sequence's segments; bidirectional: the sum)
 *     LA_PHASE_OUTPUT  outputs of every segment
 *   A phase that the call does not need (STATE and SCAN when every causal
 *   sequence is a single segment) enqueues nothing.  *launched (host, may be
 *   NULL) receives the number of kernels the phase enqueued.
 */
#define LA_PHASE_PLAN 0
#define LA_PHASE_STATE 1
#define LA_PHASE_SCAN 2
#define LA_PHASE_OUTPUT 3
#define LA_NUM_PHASES 4
LA_API la_status la_forward_phase(int causal, int phase, int norm, const void* q, const void* k,
                                  const void* v, const float* omega, int map, int dtype,
                                  const int32_t* cu_seqlens, int nseq, int64_t T, int H, int d_k,
                                  int d_v, int r, float eps, const float* state_in, float* state_out,
                                  void* out, void* workspace, size_t workspace_bytes, void* stream,
                                  int* launched);

/*
 * la_forward_causal_noalloc - la_forward_causal for callers that cannot
 *   allocate device memory.  The source pages have no counterpart: this is a
 *   deployment variant of the same computation, not part of the method.
 *
 *   Who needs it: code that must not call cudaMalloc (or any allocator) on
 *   its hot path - a real-time serving loop whose memory is budgeted up front,
 *   a plug-in inside a host framework that owns all device memory, or a
 *   caller whose allocator may not be entered while it issues work.  Such a
 *   caller passes q, k, v, omega, cu_seqlens and out as usual but no
 *   workspace.  The scratch lives in one fixed array of
 *   LA_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 *   loads the library keeps until the process exits.
 *
 *   Arguments and result are those of la_forward_causal without `workspace`
 *   and `workspace_bytes`.  Returns LA_ERR_WORKSPACE, before enqueuing
 *   anything, when the call would need more scratch than
 *   LA_NOALLOC_SCRATCH_BYTES (la_workspace_bytes(1, ...) gives the need).
 *   The first call on each device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  The cache lives as long as the process: cudaDeviceReset
 *   destroys the context that holds the array, so a program that resets a
 *   device must not call this entry point on that device afterwards (the
 *   cached address would no longer be the array's).  Every call on a device
 *   uses the same array and leaves its contents behind; each call rewrites
 *   whatever it reads before reading it, so nothing needs clearing, but calls
 *   whose work overlaps on the GPU (different streams, or different host
 *   threads) race on the array and must be serialised by the caller.
 *   Device-side errors of the latest call (cu_seqlens contents that break the
 *   packing rules, a bounded wait that ran out, a value clamped into the f16
 *   operand range) are read with la_noalloc_error.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define LA_NOALLOC_SCRATCH_BYTES (32u << 20)
LA_API la_status la_forward_causal_noalloc(const void* q, const void* k, const void* v,
                                    const float* omega, int map, int dtype,
                                    const int32_t* cu_seqlens, int nseq, int64_t T, int H,
                                    int d_k, int d_v, int r, float eps, void* out, void* stream);

/*
 * la_noalloc_error - the device error word that the latest
 *   la_forward_causal_noalloc call on the current device left in the
 *   library's scratch array, as la_workspace_error reports it for a
 *   workspace: LA_OK, or LA_ERR_DEVICE with the LA_DEVERR_* code in *code
 *   (host pointer, may be NULL).  Synchronises `stream` (pass the stream of
 *   that call).  Not a counterpart of anything on the source pages.
 */
LA_API la_status la_noalloc_error(int* code, void* stream);

/*
 * la_test_force_wait_timeout - test hook for the bounded waits (not part of
 *   the method).  With enable = 1, every later launch of the causal tensor-core
 *   output kernel on the current device makes its projection epilogue first
 *   wait on a barrier that nothing arrives at, with a 1 ms limit; the wait runs
 *   out, the kernel records LA_DEVERR_WAIT_TIMEOUT in the workspace error word,
 *   every role gives up on its own bounded waits (2 s each), drains the copies
 *   and MMAs it started, frees its tensor memory and returns: the outputs of that
 *   call are incomplete and the context stays usable.  enable = 0 restores normal
 *   operation.  Device-wide; not for concurrent use with other calls.  Returns
 *   LA_OK, or LA_ERR_CUDA when the device flag cannot be written.
 */
LA_API la_status la_test_force_wait_timeout(int enable);

/*
 * la_test_segment_plan - test hook for the planner's host logic (not part of the
 *   method; no device needed).  For an equal-length batch on the tensor-core path
 *   whose sequences have `nchunks` chunks of 128 tokens each, with `pairs`
 *   (sequence, head) pairs on `nsm` SMs: with force_chunks = 0, returns the segment
 *   length in chunks the forward call uses (0: no candidate, the call then keeps
 *   one wave of nsm / pairs segments per sequence); with force_chunks > 0, returns
 *   force_chunks.  *makespan (if not null) receives the simulated finish time, in
 *   chunk times, of the returned length's blocks: blocks taken longest first, each
 *   starting as an SM frees up, one chunk of set-up each.  Returns -1 for
 *   nchunks, pairs or nsm below 1.
 */
LA_API int64_t la_test_segment_plan(int64_t nchunks, int64_t pairs, int nsm, int64_t force_chunks,
                                    int64_t* makespan);

/*
 * la_workspace_bytes - scratch size for a forward call on the current device.
 *   causal: 1 for la_forward_causal, 0 for la_forward_bidir; `has_cu_seqlens`:
 *   1 when a cu_seqlens array will be passed.  Returns 0 for arguments the
 *   forward call would reject.  The size depends on the device's SM count and
 *   covers every kernel path a call with these arguments can take (any norm,
 *   any operand alignment, with or without state_in / state_out).
 */
LA_API size_t la_workspace_bytes(int causal, int map, int dtype, int has_cu_seqlens, int nseq,
                          int64_t T, int H, int d_k, int d_v, int r);

/*
 * la_check_cu_seqlens - validate cu_seqlens contents (device array).
 *   Returns LA_OK when cu_seqlens[0] = 0, the array does not decrease and
 *   cu_seqlens[nseq] = T; LA_ERR_INVALID_ARG otherwise.  Synchronises `stream`
 *   (it copies nseq + 1 integers to the host).
 */
LA_API la_status la_check_cu_seqlens(const int32_t* cu_seqlens, int nseq, int64_t T, void* stream);

/*
 * la_workspace_error - read the device error word a forward call left in its
 *   workspace.  Synchronises `stream`.  Returns LA_OK, or LA_ERR_DEVICE and the
 *   LA_DEVERR_* code in *code (host pointer, may be NULL).
 */
LA_API la_status la_workspace_error(const void* workspace, int* code, void* stream);

/*
 * la_orthogonal_features - build the FAVOR+ projection matrix from Gaussian draws.
 *   gauss_blocks:  [ceil(r/d), d, d] fp64, i.i.d. N(0,1) (device)
 *   gauss_lengths: [r, d] fp64, i.i.d. N(0,1) (device)
 *   omega:         [r, d] fp32 output (device)
 *   Each block's rows are orthonormalised in order by Gram-Schmidt; row i of
 *   the stacked result is scaled to the Euclidean length of gauss_lengths[i]
 *   (a chi(d) draw), and the first r rows are kept ("The Kernel Zoo" §5.1 and
 *   §5.3 Steps 1-3; "Performer" §2 Step 4, rows with Gaussian-distributed
 *   norms).  Computed in fp64 and rounded to fp32.  1 <= d <= 128.
 */
LA_API la_status la_orthogonal_features(const double* gauss_blocks, const double* gauss_lengths,
                                 int r, int d, float* omega, void* stream);

/*
 * la_selected_path - which kernels a forward call with these arguments runs:
 *   0 = fp32 CUDA-core kernels, 1 = tcgen05 tensor-core kernels.  Assumes
 *   16-byte aligned pointers and no carried state under LA_NORM_SUM.
 *   Returns -1 for arguments a call would reject.
 */
LA_API int la_selected_path(int causal, int map, int dtype, int d_k, int d_v, int r);

/* la_status_string - static description of a status code. */
LA_API const char* la_status_string(la_status status);

/* la_version - library version, major * 10000 + minor * 100 + patch. */
LA_API int la_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
