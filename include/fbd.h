/*
 * fbd.h -- C ABI of libfbd: exact softmax attention (causal, causal with a sliding
 * window, or full) on GB300 (sm_103a): forward, recompute backward (optional
 * GProj), and backward-over-backward (optional GProj).
 *
 * The N x N score matrix is never written to device memory.  All entry points
 * take plain device pointers owned by the caller; the library allocates and
 * frees nothing.
 *
 * Sources (cited by page title and section):
 *   [FA]   "Flash attention for trading models": "Why attention is memory-bound"
 *          (S = Q K^T / sqrt(d), softmax, O = P V), "The Flash Attention
 *          algorithm" (tiling into row and column blocks), "Online softmax
 *          recurrence", "Backward pass: recompute instead of store" (only O and
 *          the softmax statistics are kept), "Causal masking is where trading
 *          gets a discount", "Eight-line integration" (q, k, v shaped
 *          (batch, heads, seq, head_dim)).
 *   [GP]   "FlashAttention bf16 gradient and GProj": "Why the error appears late"
 *          (subtract the row max before scaling), "How the zero sum turns into a
 *          false gradient" (bf16 rounding of dS, GProj).
 *   [BoB]  "FlashBoB: second-order attention": "Why go backward through an
 *          already computed gradient" (definition of backward-over-backward),
 *          "Two scalar states replace quadratic tensors" (row pass, column pass).
 *
 * Conventions shared by every entry point
 *   Layout:     every [B,H,N,d] tensor is contiguous row-major (d fastest), the
 *               (batch, heads, seq, head_dim) order of [FA] "Eight-line
 *               integration".  Statistics are [B,H,N] float32, contiguous.
 *   Types:      desc->dtype selects the element type of every [B,H,N,d] tensor
 *               (inputs and outputs alike): ATTN_F32 = float, ATTN_BF16 =
 *               bfloat16.  Arithmetic is float32 throughout (bf16 tensor-core
 *               products accumulate in float32).
 *   Supported:  causal in {0, 1}; window >= 0 (> 0 only with causal = 1); any
 *               group dividing H; d in {32, 64, 96, 128, 256}; dtype in
 *               {ATTN_F32, ATTN_BF16}.  Anything else returns ATTN_ERR_UNSUPPORTED
 *               (or ATTN_ERR_INVALID_ARG) before any launch.
 *   Kernels:    the shape decides, never a failure: bf16 attn_fwd, attn_bwd and
 *               attn_bob at d in {32, 64, 96, 128}, and bf16 attn_fwd and attn_bwd
 *               (with or without GProj) at d = 256, run on the tcgen05/TMA tensor-core kernels
 *               (d = 32 and 96 on those of d = 64 and 128, the head dim zero-padded in
 *               shared memory); float32 inputs at every d run on tcgen05
 *               kind::tf32 kernels that form each product from the operands' tf32
 *               high and low parts (A_lo B_hi + A_hi B_lo + A_hi B_hi: about 2^-21
 *               relative per element product, fp32 accumulation; across blocks the
 *               sums are fp32 additions on the CUDA cores; past d = 64 the head dim
 *               is taken in chunks of 64 and the output columns are split over CTAs
 *               in parts of 64); the bf16 BoB at d = 256 runs on the same tf32 engine
 *               (bf16 inputs widened on load, dS and P rounded to bf16 where GProj
 *               reads them, outputs rounded once on store).
 *               GProj does not apply to float32 inputs (gproj is ignored: nothing is
 *               rounded to bf16).  The GProj diagnostic attn_bwd_projected_dS runs on
 *               CUDA cores.
 *   Scale:      desc->scale == 0 means 1/sqrt(d); otherwise it must be finite and
 *               positive (the row max is subtracted before scaling).
 *   Pointers:   device pointers, 16-byte aligned (ATTN_ERR_ALIGNMENT otherwise),
 *               non-NULL whenever B*H*N > 0 (ATTN_ERR_INVALID_ARG).  Outputs must
 *               not overlap inputs, each other, or the workspace
 *               (ATTN_ERR_INVALID_ARG).  Empty problems (B*H*N == 0) return
 *               ATTN_OK without touching memory.
 *   Streams:    `stream` is a cudaStream_t (NULL = the legacy default stream).
 *               Calls are asynchronous: argument errors are returned at once;
 *               a launch failure returns ATTN_ERR_LAUNCH; a device-side wait that
 *               gave up (bounded waits; never expected) is reported by
 *               attn_device_status().  Outputs are valid once the stream is
 *               synchronised.  Each output element is written exactly once.
 *   Ragged N:   any N >= 1 is accepted; tiles past N are zero-filled on load and
 *               never stored.
 *   Sliding window ([BoB] "When FlashBoB changes the engineering plan" lists
 *               flexible masks among the next extensions; the reading here is the
 *               banded causal mask): with W = desc->window > 0, query i sees the
 *               keys i - W < j <= i, and every operation (forward, backward with or
 *               without GProj, BoB) is that of attention under this mask; row
 *               blocks skip the key blocks wholly outside every row's window and
 *               column blocks the query blocks that see none of their keys.
 *   Document mask ([BoB] "When FlashBoB changes the engineering plan" lists flexible
 *               masks among the next extensions; the reading here is the mask of packed
 *               batches): with desc->seg_lo / seg_hi set (attn_segment_bounds), query i
 *               sees the keys j <= i of its own document, every operation is that of
 *               attention under this mask, and the passes skip the blocks no row of
 *               theirs can see, as for the window.
 *   Grouped key/value heads ([BoB] "When FlashBoB changes the engineering plan"
 *               lists shared keys and values among the next extensions; the reading
 *               here is the usual grouped-query one): with g = desc->group > 1 the tensors on the key
 *               side -- K, V and, for the backward and BoB, dK, dV, gdK, gdV, gK,
 *               gV -- are [B, H/g, N, d]; every other tensor keeps H heads.  The
 *               result equals plain attention with each key/value head repeated
 *               for its g query heads, and the gradients of a shared head (dK, dV,
 *               gK, gV) are sums over its g query heads; gdK and gdV, cotangents of
 *               those sums, enter each of the g heads unchanged.
 */
#ifndef FBD_H
#define FBD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* NULL/negative/overlapping arguments, non-finite scale,
                                group < 0 or not dividing H, window < 0, only one of
                                seg_lo / seg_hi set */
  ATTN_ERR_UNSUPPORTED = 2,  /* causal not 0 or 1, window > 0 or a document mask without
                                causal = 1, d not supported, unknown dtype */
  ATTN_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned */
  ATTN_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than the *_workspace_bytes query */
  ATTN_ERR_LAUNCH = 5,       /* CUDA rejected a launch or a tensor-map encode */
  ATTN_ERR_TIMEOUT = 6,      /* a bounded device-side wait gave up (see attn_device_status) */
  ATTN_ERR_DEVICE = 7        /* no usable CUDA device / driver entry point */
} attn_status_t;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype_t;

typedef struct {
  int64_t B, H, N, d;  /* batch, heads, sequence length, head dimension */
  float scale;         /* softmax scale s; 0 means 1/sqrt(d) */
  int32_t causal;      /* 1: key j is visible to query i iff j <= i ([FA] "Causal
                          masking is where trading gets a discount"); 0: every key
                          is visible to every query (a full softmax over the row) */
  int32_t dtype;       /* attn_dtype_t */
  int32_t group;       /* query heads per key/value head, g (0 and 1 both mean plain
                          multi-head attention; g must divide H; g == H is multi-query).
                          Query head h reads key/value head h / g (integer division);
                          see "Grouped key/value heads" above. */
  int32_t window;      /* causal sliding window W: with W >= 1 (and causal = 1) key j
                          is visible to query i iff i - W < j <= i; 0 means no window
                          (W >= N is the same as none).  A flexible mask ([BoB] "When
                          FlashBoB changes the engineering plan" lists flexible masks
                          among the next extensions); every operation honours it. */
  /* Document (segment) mask, the second flexible mask: device arrays [B, N] written by
     attn_segment_bounds from per-token segment ids (both NULL: no document mask; both
     set: causal must be 1).  Query i of batch row b sees key j iff
     seg_lo[b][i] <= j <= i, i.e. j <= i and seg[b][j] == seg[b][i]; combined with a
     window when both are given.  16-byte aligned, B*N int32 each, read only.  See
     "Document mask" above. */
  const int32_t* seg_lo;
  const int32_t* seg_hi;
} attn_desc_t;

/* Bounds of the document (segment) mask.  [BoB] "When FlashBoB changes the engineering
 * plan" lists flexible masks among the next extensions; this is the mask of packed
 * batches: documents laid back to back along N, each attending only within itself.
 *   In:  seg [B, N] int32 device array, the segment (document) id of every token, non-
 *        decreasing along each batch row (each document one run of equal ids).
 *   Out: seg_lo [B, N]: for token i, the first index of its run (its document's first key);
 *        seg_hi [B, N]: for token j, the last index of its run (its document's last query).
 *   One launch on `stream` (binary searches; the ids are read, nothing else).  Pass both
 *   outputs in attn_desc_t.seg_lo / seg_hi to every call of the same batch: query i then
 *   sees exactly the keys j <= i with seg[j] == seg[i].  For ids that are not non-
 *   decreasing the bounds are those of the searches (still lo <= i <= hi, every row keeps
 *   its own key), not that mask.  Errors: B or N negative, or B*N >= 2^40
 *   (ATTN_ERR_INVALID_ARG); NULL, unaligned (16 bytes) or overlapping arrays; B*N == 0 is
 *   ATTN_OK with no launch. */
attn_status_t attn_segment_bounds(int64_t B, int64_t N, const int32_t* seg, int32_t* seg_lo, int32_t* seg_hi,
                                  void* stream);

/* Forward.  [FA] "The Flash Attention algorithm", "Online softmax recurrence",
 * causal masking; [GP] "Why the error appears late" (max subtracted before the
 * scale is applied, so the row max maps to exactly exp(0) = 1).
 *   In:  Q, K, V [B,H,N,d].
 *   Out: O [B,H,N,d] = softmax(s Q K^T + mask) V (mask: causal, or none);
 *        lse [B,H,N] float32, lse_i = log sum_{j visible} exp(s q_i.k_j) (natural log),
 *        the single-number form of the softmax statistics (m, l) kept for the
 *        recompute backward ([FA] "Backward pass: recompute instead of store"). */
attn_status_t attn_fwd(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                       void* O, float* lse, void* stream);

/* Workspace for attn_bwd: 16 bytes per (b,h,row), the rows of each slice rounded
 * up to an even count: the row statistics (lse, D, GProj coefficient) read by the
 * column pass (layout internal to the library); for bf16 at d <= 64 without GProj
 * and N < 2^21 (the single-pass form of attn_bwd) 256 bytes more per (b,h,row) for an
 * fp32 dQ accumulator. */
size_t attn_bwd_workspace_bytes(const attn_desc_t* desc, int gproj);

/* Recompute backward.  [FA] "Backward pass: recompute instead of store": P is
 * rebuilt from Q, K and lse; nothing N x N is stored.  With
 *   dP = dO V^T, D_i = sum_k dO_ik O_ik, dS = P * (dP - D):
 *   dQ = s dS K,  dK = s dS^T Q,  dV = P^T dO          (all [B,H,N,d]).
 * Two launches on `stream`: a row pass (dQ and the row statistics) and a column
 * pass (dK, dV).  For bf16 at d <= 64 without GProj and N < 2^21, the single-pass form instead
 * ([FA] "FA2: parallelism": the work split over key blocks, the query gradient summed
 * across them): a launch forming D and the row statistics, one launch over key blocks
 * that writes dK, dV once and adds each key block's dS K share of dQ into an fp32
 * accumulator in the workspace (tensor reduce-adds in L2), and a launch that writes
 * dQ = s * accumulator once, rounded to bf16.  Every contraction then runs once.  (From
 * N = 2^21 on its reduce-adds of dQ shares slow down and the two passes are as fast or
 * faster, so those lengths take the two passes.)  The
 * shares are added in the order the key blocks reach a query block, so dQ may differ
 * between calls in its last bits (two bf16 steps at most); dK and dV, and every output
 * of the two-pass forms, are the same bits on every call.
 * gproj != 0 (bf16 only; ignored for ATTN_F32, whose dS is never rounded):
 *   [GP] "How the zero sum turns into a false gradient".  The row of dS is rounded
 *   to bf16 (dS^) before the dS K and dS^T Q products; its remaining mass
 *   r_i = sum_j dS^_ij is removed by subtracting r_i * P^_ij / sum_k P^_ik, where
 *   P^ is the bf16 probability row the kernel feeds to its products, so that the
 *   row the products see sums to zero.  The query correction is applied inside
 *   the row pass; the key correction needs r_i of complete rows and is applied in
 *   the column pass.
 *   workspace: >= attn_bwd_workspace_bytes(desc, gproj) bytes of device memory,
 *   16-byte aligned, contents ignored on entry; it holds row statistics after. */
attn_status_t attn_bwd(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                       const void* O, const void* dO, const float* lse,
                       void* dQ, void* dK, void* dV, int gproj,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Workspace for attn_bob: 16 bytes per (b,h,row), the rows of each slice rounded
 * up to an even count: the per-row states (lse, D, E, F) written by the row pass
 * for the column pass.  With gproj != 0 and bf16: as much again for the GProj
 * coefficients, plus, for d <= 128, 256 (d <= 64) or 512 bytes per (b,h,row) for the
 * rows' P^ b (layout internal to the library). */
size_t attn_bob_workspace_bytes(const attn_desc_t* desc, int gproj);

/* Backward over backward.  [BoB] "Why go backward through an already computed
 * gradient": with Phi(Q,K,V,dO) = (dQ,dK,dV) the first backward and cotangents
 * gdQ, gdK, gdV of its outputs, returns the vector-Jacobian product
 *   (gQ, gK, gV, gdO) = d/d(Q,K,V,dO) [ <gdQ,dQ> + <gdK,dK> + <gdV,dV> ].
 * With a = gdQ, b = gdK, c = gdV, G = s(a K^T + Q b^T), H = dO c^T and the two
 * per-row scalar states ([BoB] "Two scalar states replace quadratic tensors")
 *   E_i = sum_j P_ij G_ij,  F_i = sum_j P_ij (G_ij (dP_ij - D_i) - E_i dP_ij + H_ij):
 *   gQ  = s (dS b + Sbar K),   gK = s (dS^T a + Sbar^T Q),
 *   gV  = dPbar^T dO,          gdO = P c + dPbar V,
 *   dPbar = P (G - E),  Sbar = P (G (dP - D) - E dP + H - F).
 * Two launches: the row pass holds a block of query rows, streams keys, writes
 * gQ, gdO and (lse, D, E, F) per row; the column pass holds a block of keys,
 * streams rows, re-reads those states and writes gK, gV.
 * gproj != 0 (bf16 only; ignored for ATTN_F32): [GP] "How the zero sum turns into
 *   a false gradient", applied to the two products that contract dS, gQ's dS b and
 *   gK's dS^T a.  They see the bf16-rounded row dS^ projected back to zero sum,
 *   dS^ - rho_i P^, rho_i = sum_j dS^_ij / sum_k P^_ik (P^ the bf16 probability row
 *   the products use), as attn_bwd's GProj treats dQ and dK.  On the bf16
 *   tensor-core path a third launch precedes the row pass: it forms P^ b per row
 *   (into the workspace), which the row pass scales by rho_i (in fp32, so the rows
 *   gQ sees sum to zero); the column pass adds the key term with the correction
 *   -rho_i P_ij as one more bf16 operand (its rows then sum to zero up to the bf16
 *   rounding of that small correction).  Nothing else changes.
 *   O, lse: the forward's outputs for the same Q, K, V (attn_fwd).
 *   workspace: >= attn_bob_workspace_bytes(desc, gproj) bytes of device memory,
 *   16-byte aligned, contents ignored on entry; holds (lse, D, E, F) after (and
 *   with GProj the coefficients and P^ b). */
attn_status_t attn_bob(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                       const void* O, const void* dO, const float* lse,
                       const void* gdQ, const void* gdK, const void* gdV,
                       void* gQ, void* gK, void* gV, void* gdO, int gproj,
                       void* workspace, size_t workspace_bytes, void* stream);

/* attn_bob for callers that cannot allocate device memory.  The source pages have
 * no counterpart of this entry point.  Some callers cannot obtain device memory
 * of their own (for example a plugin inside a host application whose memory
 * manager owns the device, or a deployment with a fixed memory plan that forbids
 * allocation after start-up), so this variant takes no workspace: the row
 * statistics live in a file-scope device array of 16 MiB, 1,048,576 rows of 16
 * bytes, which holds problems with B*H*Np <= 1,048,576, Np = N rounded up to an
 * even count (the row statistics are stored in row pairs).  Larger problems return
 * ATTN_ERR_WORKSPACE without launching anything (use attn_bob with a caller
 * workspace instead).
 *   Arguments, outputs and errors are those of attn_bob with gproj = 0 and no
 *   workspace (this entry point has no GProj form); the descriptor is checked
 *   first, as attn_bob checks it.
 *   The array is held by every GPU that loads the library until process exit.
 *   Under CUDA's lazy module loading (the default) the 16 MiB are committed on a
 *   device when the array is first looked up there, which the first call on that
 *   device does: it looks up the array's device address with cudaGetSymbolAddress
 *   (that device must be current) and caches it.  Callers with a fixed memory
 *   plan should therefore make one call per device at start-up -- an empty
 *   problem (B*H*N == 0, NULL pointers) does the look-up and launches nothing --
 *   or run with CUDA_MODULE_LOADING=EAGER; make that first call before any stream
 *   capture.  The cached address assumes the device is not reset (cudaDeviceReset)
 *   while the library is in use.  No call allocates or frees memory itself.
 *   All calls share the one array, which keeps the last call's contents; nothing
 *   in it needs clearing (the row pass writes every entry the column pass reads).
 *   Calls whose executions overlap on the GPU (other streams, or other host
 *   threads) race on the array: serialise them. */
attn_status_t attn_bob_static(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                              const void* O, const void* dO, const float* lse,
                              const void* gdQ, const void* gdK, const void* gdV,
                              void* gQ, void* gK, void* gV, void* gdO, void* stream);

/* The two launches of attn_bwd / attn_bob, issued separately (for callers that
 * schedule or time the passes themselves).  passes = ATTN_ROW_PASS (backward: dQ
 * and the row statistics; BoB: gQ, gdO and the row states, after the P^ b launch
 * when gproj is set on the bf16 tensor-core path), ATTN_COL_PASS
 * (backward: dK, dV; BoB: gK, gV, both from the statistics the row pass left in
 * `workspace`), or both, which is exactly attn_bwd / attn_bob (for the backward the
 * single-pass form where attn_bwd uses it, so dQ then equals the two separate passes'
 * dQ up to the summation order).  A single pass needs only the statistics part of the
 * workspace: 16 bytes per (b,h,row), the rows of each slice rounded up to even.  A column pass
 * must follow, in stream order, a row pass over the same inputs and workspace.
 * Arguments and checks are those of attn_bwd / attn_bob (all pointers are
 * validated whichever pass runs); any other `passes` is ATTN_ERR_INVALID_ARG.
 * [BoB] "Two scalar states replace quadratic tensors" (row pass, then column pass);
 * [GP] "How the zero sum ..." (the key correction needs the finished rows). */
#define ATTN_ROW_PASS 1
#define ATTN_COL_PASS 2
attn_status_t attn_bwd_passes(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                              const void* O, const void* dO, const float* lse,
                              void* dQ, void* dK, void* dV, int gproj,
                              void* workspace, size_t workspace_bytes, int passes, void* stream);
attn_status_t attn_bob_passes(const attn_desc_t* desc, const void* Q, const void* K, const void* V,
                              const void* O, const void* dO, const float* lse,
                              const void* gdQ, const void* gdK, const void* gdV,
                              void* gQ, void* gK, void* gV, void* gdO, int gproj,
                              void* workspace, size_t workspace_bytes, int passes, void* stream);

/* Diagnostic export of the GProj-projected score gradient (bf16 only).
 * Writes dS_out [B,H,N,N] float32 with dS_out[i][j] = dS^_ij - rho_i P^_ij for
 * every visible key j (0 for j > i under the causal mask), where dS^, P^ and
 * rho_i = r_i / sum_k P^_ik are the
 * very values the GProj row pass feeds to its products.  Meant for small N:
 * the output is N x N per slice.  [GP] "How the zero sum turns into a false
 * gradient". */
attn_status_t attn_bwd_projected_dS(const attn_desc_t* desc, const void* Q, const void* K,
                                    const void* V, const void* O, const void* dO,
                                    const float* lse, float* dS_out, void* stream);

/* Synchronises `stream` and reports (then clears) the device-side status word:
 * ATTN_ERR_TIMEOUT if any kernel's bounded wait gave up since the last call,
 * ATTN_ERR_LAUNCH if the stream holds a CUDA error, else ATTN_OK. */
attn_status_t attn_device_status(void* stream);

/* Check of the failure-detection path, for tests and health checks.  Launches one
 * CTA on `stream` whose bounded wait (the kind every tensor-core kernel uses) waits
 * on a barrier that nothing completes; after 20 ms it gives up, records the timeout
 * in the library's device status word and returns, without any fault.  Returns
 * attn_device_status(stream): ATTN_ERR_TIMEOUT when the path works (the status is
 * then cleared, and the context stays usable), ATTN_ERR_LAUNCH if the launch failed. */
attn_status_t attn_check_wait_timeout(void* stream);

/* Static description of a status code (never NULL). */
const char* attn_status_string(attn_status_t status);

/* Human-readable detail of the most recent non-OK status on the calling thread
 * (e.g. which argument was rejected); empty string if none. */
const char* attn_last_error(void);

/* Library build identification string. */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FBD_H */
