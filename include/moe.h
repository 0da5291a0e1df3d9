/*
 * moe.h -- C ABI of the single-GPU MoE expert-layer forward (GB300, sm_103a).
 *
 * The layer is Algorithm 2 ("Single-GPU MoE Forward (OlmoeExperts)") of the
 * page "MoE 分布式推理基础（基于 vLLM）", §1.2 "MoE Forward": router GEMM,
 * softmax, TopK with optional renormalisation, the dispatch layout, the SwiGLU
 * expert GEMMs and the weighted scatter-add combine.  One extra call runs two
 * (or more) micro-batches on two CUDA streams so that one micro-batch's
 * dispatch and combine overlap another's expert GEMMs (the cross-micro-batch
 * schedule of the page "XTuner Domino EP", section "执行路径").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *    never allocates device memory on these calls and never synchronises the
 *    host; work is enqueued on the stream(s) given.  Only moe_check_status()
 *    blocks.
 *  - Argument errors are returned synchronously, before anything is enqueued:
 *    MOE_ERR_INVALID_ARG (null pointer, bad size, misaligned pointer),
 *    MOE_ERR_UNSUPPORTED (a size the library does not handle),
 *    MOE_ERR_WORKSPACE (workspace too small).  A failed launch returns
 *    MOE_ERR_CUDA.
 *  - Problems found on the device (an expert id outside [0, E), an
 *    inconsistent layout, a pipeline wait that ran out of time) are OR-ed
 *    into a caller-provided int32 status word as MOE_DEV_* bits; kernels then
 *    skip the offending access instead of faulting.  The status word is never
 *    cleared by the library except where stated; read it with
 *    moe_check_status().
 *  - Layouts are row-major.  Shapes (n tokens, hidden H, intermediate I,
 *    E experts, K experts per token):
 *        x       (n, H)        dtype
 *        w_gate  (H, E)        dtype
 *        bias    (E)           float32, optional per-expert logit bias
 *        w13     (E, H, 2I)    dtype; columns [0, I) gate, [I, 2I) up
 *        w2      (E, I, H)     dtype
 *        logits  (n, E)        float32
 *        topk_idx(n, K)        int32, slot order = descending logit
 *        topk_w  (n, K)        float32
 *        counts  (E), offsets (E+1), perm (n*K), inv_perm (n*K)   int32
 *        x_perm  (n*K, H), h (n*K, I), y_perm (n*K, H), y (n, H)   dtype
 *    dtype is float32 (MOE_F32) or bfloat16 (MOE_BF16).  Accumulation is
 *    float32 in every GEMM and in the combine.
 *  - bf16 layers need H % 64 == 0 and I % 128 == 0; float32 layers need
 *    H % 4 == 0 and I % 4 == 0.  E <= 256, 1 <= K <= min(E, 16).
 *    Pointers must be 16-byte aligned.
 */
#ifndef TOP_ROUTING_DISPATCH_GB300_MOE_H
#define TOP_ROUTING_DISPATCH_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 (NULL) is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_BAD_ROUTING = 4, /* from moe_check_status: an expert id was out of range */
  MOE_ERR_CUDA = 5,
  MOE_ERR_TIMEOUT = 6,     /* from moe_check_status: a device pipeline wait gave up */
  MOE_ERR_BAD_LAYOUT = 7   /* from moe_check_status: offsets/perm inconsistent */
} moe_status_t;

/* Bits of the device status word. */
#define MOE_DEV_BAD_ROUTING 0x1
#define MOE_DEV_BAD_LAYOUT 0x2
#define MOE_DEV_TIMEOUT 0x4

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

/*
 * Layout of the expert weights w13 (E,H,2I) and w2 (E,I,H) that the expert
 * entry points read.
 *   MOE_WEIGHTS_ROW_MAJOR: as stored by the caller, row-major (the layout of
 *     the pages' code: W13[e] is H x 2I with the gate columns first).
 *   MOE_WEIGHTS_TILED: the output of moe_prepare_weights -- the same values
 *     regrouped into contiguous 64 x 64 tiles (bf16 layers only; not accepted
 *     by moe_backward).  Results are bitwise those of the row-major layout.
 */
typedef enum { MOE_WEIGHTS_ROW_MAJOR = 0, MOE_WEIGHTS_TILED = 1 } moe_weight_layout_t;

typedef struct {
  int32_t n;              /* tokens (may be 0) */
  int32_t H;              /* hidden size */
  int32_t I;              /* expert intermediate size */
  int32_t E;              /* experts */
  int32_t K;              /* experts per token */
  int32_t dtype;          /* moe_dtype_t */
  int32_t norm_topk_prob; /* nonzero: divide the K weights by their sum */
  int32_t weight_layout;  /* moe_weight_layout_t of w13 and w2 */
  /* optional (bf16 layers): the router weight transposed, (E, H) bf16 device
   * memory made by moe_prepare_router from the w_gate passed to the calls,
   * or NULL.  The router's exact near-tie rescoring then reads each expert's
   * column of w_gate as one contiguous row of this copy instead of H
   * scattered values; the results are bitwise the same.  16-byte aligned
   * (else MOE_ERR_INVALID_ARG from every call).  Ignored for float32 layers. */
  const void *w_gate_t;
} moe_layer_desc_t;

/* Library version string and a human-readable name of a status code. */
const char *moe_version(void);
const char *moe_status_string(moe_status_t status);

/*
 * Router: Algorithm 2 steps 1-3 and the renormalisation of the router shown
 * in §1.2.  logits = x·w_gate (+ bias), p = softmax(logits) over E, then the
 * K experts of largest logit in descending order (an exact tie goes to the
 * lower expert index), topk_w = p at those experts, divided by their sum
 * when norm_topk_prob.
 *   x (n,H) dtype; w_gate (H,E) dtype; bias (E) float32 or NULL;
 *   topk_idx (n,K) int32 out; topk_w (n,K) float32 out; logits (n,E) float32 out.
 * The selection is made on float32 logits, except for tokens whose top-(K+1)
 * float32 logits lie closer than a rounding margin: their candidate experts
 * are rescored in double-float (about 48-bit) precision and selected on that.
 */
moe_status_t moe_route_topk(const moe_layer_desc_t *desc, const void *x, const void *w_gate,
                            const float *bias, int32_t *topk_idx, float *topk_w, float *logits,
                            moe_stream_t stream);

/*
 * Dispatch layout: Algorithm 2 steps 4-5 (hit counts n_e and the sets I_e),
 * in the expert-sorted form of the moe_align_block_size example of §2.3
 * (without block padding).  With f = t*K + k the flat index of a (token,
 * slot) pair:
 *   counts[e]   = number of pairs routed to e
 *   offsets[e]  = sum of counts[e'] for e' < e; offsets[E] = pairs with a valid id
 *   perm[r]     = f of the r-th pair after a stable sort by expert (ascending f
 *                 inside each expert)
 *   inv_perm[f] = r
 * Deterministic (integer only).  Pairs whose id is outside [0, E) set
 * MOE_DEV_BAD_ROUTING in *status_word and are placed after offsets[E], so
 * perm stays a permutation of [0, n*K).
 *   topk_idx (n,K) int32; status_word: one int32 (device), OR-ed into;
 *   ws: moe_layout_workspace_size(desc) bytes of device scratch (contents
 *   need no initialisation; not used after the call returns on the stream).
 */
size_t moe_layout_workspace_size(const moe_layer_desc_t *desc);
moe_status_t moe_dispatch_layout(const moe_layer_desc_t *desc, const int32_t *topk_idx,
                                 int32_t *counts, int32_t *offsets, int32_t *perm,
                                 int32_t *inv_perm, int32_t *status_word, void *ws,
                                 size_t ws_bytes, moe_stream_t stream);

/*
 * moe_dispatch_layout without a workspace argument: the same layout, computed
 * by the same kernels, for callers that cannot allocate device memory when
 * they run (a pre-planned memory pool with nothing left over, or a context in
 * which a cudaMalloc would stall the device or is not allowed).  There is no
 * counterpart of this call in the pages; it exists only for such callers.
 *   - Scratch: a fixed device array owned by the library (257 KiB per
 *     GPU that loads the library, kept until the process exits).  The call
 *     itself allocates nothing.
 *   - Limit: n*K <= MOE_NOALLOC_MAX_PAIRS (and E <= 256 as everywhere);
 *     larger layouts return MOE_ERR_WORKSPACE before anything is enqueued.
 *   - Every call looks up the array's address on the current device
 *     (cudaGetSymbolAddress, a host-side lookup), so the address stays valid
 *     after a cudaDeviceReset.  The first call on a device may load the
 *     library's device code: make that first call before capturing a stream.
 *   - All calls on a device share the array.  Calls must not overlap on the
 *     GPU: two of them running at once (e.g. on unordered streams) race on the
 *     scratch and give wrong layouts.  Calls ordered on one stream are safe.
 * Other arguments, results and errors are those of moe_dispatch_layout.
 */
#define MOE_NOALLOC_MAX_PAIRS 524288
moe_status_t moe_dispatch_layout_noalloc(const moe_layer_desc_t *desc, const int32_t *topk_idx,
                                         int32_t *counts, int32_t *offsets, int32_t *perm,
                                         int32_t *inv_perm, int32_t *status_word,
                                         moe_stream_t stream);

/*
 * Permute (the gather of Algorithm 2 step 7 for all experts at once):
 * x_perm[r] = x[perm[r] / K].  x (n,H), x_perm (n*K,H), perm (n*K).
 * A perm entry outside [0, n*K) gives a zero row and sets MOE_DEV_BAD_LAYOUT
 * in *status_word (status_word may be NULL, then such rows are only zeroed).
 */
moe_status_t moe_permute(const moe_layer_desc_t *desc, const void *x, const int32_t *perm,
                         void *x_perm, int32_t *status_word, moe_stream_t stream);

/*
 * The same permute in scatter form: x_perm[inv_perm[t*K + k]] = x[t] for
 * every token t and slot k (inv_perm from moe_dispatch_layout).  Each x row
 * is read once and written to its K rows, so x leaves DRAM once whatever the
 * L2 holds (the gather form re-reads each x row K times and relies on the L2
 * for the re-reads).  x_perm is bitwise equal to moe_permute's.  An inv_perm
 * entry outside [0, n*K) is skipped and sets MOE_DEV_BAD_LAYOUT (status_word
 * may be NULL); the row it would have written is left as it was.
 */
moe_status_t moe_permute_scatter(const moe_layer_desc_t *desc, const void *x,
                                 const int32_t *inv_perm, void *x_perm, int32_t *status_word,
                                 moe_stream_t stream);

/*
 * Grouped SwiGLU experts: Algorithm 2 steps 8-9 for every expert with a
 * non-empty segment [offsets[e], offsets[e+1]) of x_perm:
 *   [G | U] = x_perm[seg] · w13[e];  h[seg] = SiLU(G) * U;  y_perm[seg] = h[seg] · w2[e]
 * with SiLU(g) = g / (1 + exp(-g)).  h is rounded to dtype before the second
 * GEMM.  bf16 layers run on the tcgen05 tensor cores (TMA-fed, TMEM
 * accumulators, SiLU*up in the first GEMM's epilogue); float32 layers run on
 * float32 FMA units.  Rows of y_perm at or after offsets[E] are not written.
 * sm_reserve: number of SMs left free for work on other streams (0 = all).
 * offsets must be as produced by moe_dispatch_layout; an inconsistent table
 * sets MOE_DEV_BAD_LAYOUT and nothing is computed.  No workspace is needed.
 */
moe_status_t moe_grouped_swiglu(const moe_layer_desc_t *desc, const void *x_perm, const void *w13,
                                const void *w2, const int32_t *offsets, void *h, void *y_perm,
                                int sm_reserve, int32_t *status_word, moe_stream_t stream);

/*
 * The two halves of moe_grouped_swiglu as separate calls (same kernels, same
 * results): GEMM1 with the SwiGLU epilogue writes h; GEMM2 reads h and writes
 * y_perm.  Arguments as for moe_grouped_swiglu.
 */
moe_status_t moe_expert_gemm1_swiglu(const moe_layer_desc_t *desc, const void *x_perm,
                                     const void *w13, const int32_t *offsets, void *h,
                                     int sm_reserve, int32_t *status_word, moe_stream_t stream);
/*
 * GEMM1 + SwiGLU with the permute fused into it (bf16 layers only): the A
 * rows of expert e's segment are read straight from x, row r being token
 * perm[r] / K, by 16-byte cp.async copies from four gathering warps, so
 * x_perm is never written.  The gather of Algorithm 2 step 7 and step 8 in
 * one pass: the permute folded into the expert GEMM, as HybridEP's
 * dispatch_with_permute (DModel notes "0. goin", §2.4) and FLUX/COMET's
 * scatter-into-grouped-GEMM ("大模型系统中的通算融合", §4.2.4) do.  Results
 * are bitwise identical to moe_permute followed by moe_expert_gemm1_swiglu.
 * A perm entry outside [0, n*K) sets MOE_DEV_BAD_LAYOUT and leaves that row
 * of h unspecified.  It trades speed for memory: x_perm (n*K*H elements) is
 * never allocated, but A rows arrive through 16-byte cp.async gathers from
 * L2, slower than the TMA tile loads of a materialised x_perm, so
 * moe_forward_microbatches uses moe_permute + moe_expert_gemm1_swiglu.
 *   x (n,H) bf16; perm (n*K) int32 as from moe_dispatch_layout; other
 *   arguments as for moe_expert_gemm1_swiglu.  float32 layers:
 *   MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_expert_gemm1_swiglu_gather(const moe_layer_desc_t *desc, const void *x,
                                            const int32_t *perm, const void *w13,
                                            const int32_t *offsets, void *h, int sm_reserve,
                                            int32_t *status_word, moe_stream_t stream);
moe_status_t moe_expert_gemm2(const moe_layer_desc_t *desc, const void *h, const void *w2,
                              const int32_t *offsets, void *y_perm, int sm_reserve,
                              int32_t *status_word, moe_stream_t stream);

/*
 * Combine (Algorithm 2 steps 10-11, as a gather per token instead of a
 * scatter-add): y[t] = sum_{k=0..K-1} topk_w[t,k] * y_perm[inv_perm[t*K+k]],
 * accumulated in float32 in slot order k = 0..K-1 and rounded once.  No
 * atomics: the result is bitwise reproducible.  An inv_perm entry outside
 * [0, n*K) contributes nothing and sets MOE_DEV_BAD_LAYOUT (status_word may
 * be NULL).
 */
moe_status_t moe_combine(const moe_layer_desc_t *desc, const void *y_perm, const float *topk_w,
                         const int32_t *inv_perm, void *y, int32_t *status_word,
                         moe_stream_t stream);

/*
 * GEMM2 with the combine's weighting moved into its epilogue (bf16 layers):
 * for every row r of an expert segment, with f = perm[r] (the flat index
 * t*K + k of its (token, slot) pair),
 *   y_slot[f] = topk_w[f] * (h[r] . W2[e]),
 * rounded once to bf16.  The rows land in (token, slot) order, so the
 * combine becomes moe_combine_slots, a contiguous read of each token's K
 * rows: Algorithm 2 step 10's weighting done where Y_e is produced, as the
 * GEMM + gather + top-k reduce of FLUX/COMET ("大模型系统中的通算融合",
 * §4.2.5) does.  moe_forward_microbatches uses this pair for bf16 layers.
 *   h (n*K, I); perm and topk_w as from moe_dispatch_layout / moe_route_topk;
 *   y_slot (n*K, H).  A perm entry outside [0, n*K) sets MOE_DEV_BAD_LAYOUT and
 *   its row is not written; rows of pairs with an invalid expert id (at or
 *   after offsets[E]) are not written either.  float32 layers:
 *   MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_expert_gemm2_weighted(const moe_layer_desc_t *desc, const void *h,
                                       const void *w2, const int32_t *offsets,
                                       const int32_t *perm, const float *topk_w, void *y_slot,
                                       int sm_reserve, int32_t *status_word,
                                       moe_stream_t stream);

/*
 * Combine of slot-ordered, already weighted rows:
 *   y[t] = sum over k = 0..K-1 of y_slot[t*K + k]
 * accumulated in float32 in slot order and rounded once (Algorithm 2 step 11
 * as a per-token sum of K contiguous rows; deterministic, no atomics).
 *   y_slot (n*K, H) dtype, y (n, H) dtype.
 */
moe_status_t moe_combine_slots(const moe_layer_desc_t *desc, const void *y_slot, void *y,
                               moe_stream_t stream);

/*
 * Whole layer for num_mb micro-batches that share one set of weights,
 * scheduled on two streams as in "XTuner Domino EP" (执行路径) and the
 * two-micro-batch interleave of "大模型系统中的通算融合" §3.1:
 *   dispatch stream: route, layout, permute of micro-batch j+1 while the
 *                    compute stream runs micro-batch j's expert GEMMs;
 *                    combine of micro-batch j while the compute stream runs
 *                    micro-batch j+1's GEMMs.
 * Events order producer and consumer only; the host never waits.  When the
 * call returns, all work is enqueued; `compute` is made to wait for the last
 * combine, so completion of `compute` means every y[j] is final.  With
 * dispatch == compute (or NULL) everything runs in order on one stream.
 *   x[j], y[j]: arrays of num_mb device pointers, each (n,H) dtype.
 *   ws: num_mb * moe_workspace_size(desc) bytes, 256-byte aligned; it holds
 *   each micro-batch's intermediates (logits, topk, layout, x_perm, h, y_perm;
 *   for bf16 layers the y_perm slot holds moe_expert_gemm2_weighted's y_slot).
 *   status_word: one int32 (device) or NULL; cleared at the start of the call
 *   (stream-ordered) and then OR-ed into.  NULL uses a word inside ws.
 *   sm_reserve: SMs the GEMMs leave free for the dispatch stream.
 * Results are bitwise identical to running the micro-batches one after
 * another (no result depends on grid size or stream timing).
 */
size_t moe_workspace_size(const moe_layer_desc_t *desc);

/*
 * Kernel launches one micro-batch of moe_forward_microbatches enqueues for
 * this layer (router, dispatch layout, permute, the two expert GEMMs, combine),
 * for launch accounting; host-side, touches no device.  0 for an invalid
 * descriptor.
 */
int moe_forward_launches(const moe_layer_desc_t *desc);
moe_status_t moe_forward_microbatches(const moe_layer_desc_t *desc, int num_mb,
                                      const void *const *x, const void *w_gate, const float *bias,
                                      const void *w13, const void *w2, void *const *y, void *ws,
                                      size_t ws_bytes, int sm_reserve, int32_t *status_word,
                                      moe_stream_t compute, moe_stream_t dispatch);

/*
 * Device-side pointers into a micro-batch's slice of the workspace used by
 * moe_forward_microbatches (for inspection in tests).  `which`:
 * 0 logits, 1 topk_idx, 2 topk_w, 3 counts, 4 offsets, 5 perm, 6 inv_perm,
 * 7 x_perm, 8 h, 9 y_perm, 10 internal status word.  Returns NULL on a bad
 * argument.  No device access.
 */
void *moe_workspace_slot(const moe_layer_desc_t *desc, void *ws, int mb, int which);

/*
 * Backward of the layer for an upstream gradient dy = dL/dy (bf16 layers,
 * H % 256 == 0, I % 128 == 0), with the expert choice of the forward held
 * fixed (as differentiating a top-k selection does).  The pages give the
 * structure: in training the backward of dispatch is a combine and the
 * backward of combine is a dispatch ("大模型系统中的通算融合" §6.2.4), and
 * the top-k reduce and the routing scores have their own backward kernels
 * (DModel notes "0. goin", §2.3).  Steps:
 *   dY[r] = w[f] dy[t], dw[f] = <dy[t], Y[r]>          (f = t*K + k, r = inv_perm[f])
 *   dh = dY W2[e]^T;  dG = dh U s (1 + G (1 - s)), dU = dh G s  (s = sigmoid(G),
 *   G|U recomputed from x_perm W13[e]);  dX = [dG|dU] W13[e]^T
 *   dW2[e] = h_e^T dY_e;  dW13[e] = x_perm_e^T [dG|dU]_e
 *   dp from dw (through the renormalisation when norm_topk_prob),
 *   dlogits = p (dp - <p, dp>);  dx = sum_k dX[inv_perm[t*K+k]] + dlogits W_gate^T;
 *   dW_gate = x^T dlogits;  dbias = sum_t dlogits[t]
 * Inputs: the layer (x (n,H), w_gate (H,E), w13, w2), dy (n,H) bf16, and the
 * forward's intermediates as written by moe_route_topk (logits, topk_idx,
 * topk_w), moe_dispatch_layout (offsets, inv_perm), moe_permute (x_perm),
 * moe_expert_gemm1_swiglu (h) and the UNWEIGHTED moe_expert_gemm2 (y_perm).
 * Outputs: dx (n,H) bf16; dw_gate (H,E), dbias (E, or NULL), dw13 (E,H,2I),
 * dw2 (E,I,H) float32.  ws: moe_backward_workspace_size(desc) bytes, 256-byte
 * aligned.  Every sum has a fixed order (bitwise reproducible).  n = 0: the
 * weight gradients are zeroed and the token arrays (and ws) may be NULL.
 */
size_t moe_backward_workspace_size(const moe_layer_desc_t *desc);
moe_status_t moe_backward(const moe_layer_desc_t *desc, const void *x, const void *w_gate,
                          const void *w13, const void *w2, const void *dy, const float *logits,
                          const int32_t *topk_idx, const float *topk_w, const int32_t *offsets,
                          const int32_t *inv_perm, const void *x_perm, const void *h,
                          const void *y_perm, void *dx, float *dw_gate, float *dbias,
                          float *dw13, float *dw2, void *ws, size_t ws_bytes,
                          int32_t *status_word, moe_stream_t stream);

/*
 * Device bytes moe_forward_host needs: one layer workspace and two staging
 * slots (x and y of one call each).  0 for an invalid descriptor.
 */
size_t moe_host_workspace_size(const moe_layer_desc_t *desc);

/*
 * The whole layer (Algorithm 2, as moe_forward_microbatches with one
 * micro-batch) on host buffers, with the copies of consecutive calls
 * overlapped with the layer of their neighbours: the input-copy and
 * output-copy stages of a serving loop around the layer.
 *   x_host, y_host: (n,H) dtype in page-locked host memory (cudaHostAlloc or
 *   cudaHostRegister; pageable memory turns the copies synchronous).
 *   ws: moe_host_workspace_size(desc) bytes of device memory, 256-byte
 *   aligned, kept for the whole sequence of calls.
 *   call: the caller's running call number (>= 0); consecutive calls must
 *   alternate its parity, which selects the staging slot.
 *   copy_in / copy_out: streams for the host-to-device and device-to-host
 *   copies (NULL: `compute` carries them and nothing overlaps).
 * Per call: copy_in waits until the layer of the previous call on the same
 * slot has finished, copies x_host into the slot; compute waits for that copy
 * and for the slot's previous copy-out, runs the layer; copy_out waits for the
 * layer and copies y back to y_host.  y_host is complete once copy_out has
 * passed the work this call enqueued (record an event on copy_out after the
 * call, or synchronise copy_out).  The host never blocks.  Results are
 * bitwise those of moe_forward_microbatches on the same input.
 *   status_word: as for moe_forward_microbatches (NULL: a word inside ws).
 * The library keeps six CUDA events per (device, ws) pipeline for at most 64
 * pipelines; the 65th distinct ws replaces the least recently used one, after
 * waiting on the host for that pipeline's last enqueued copies and layer.
 */
moe_status_t moe_forward_host(const moe_layer_desc_t *desc, const void *x_host,
                              const void *w_gate, const float *bias, const void *w13,
                              const void *w2, void *y_host, void *ws, size_t ws_bytes,
                              long long call, int32_t *status_word, moe_stream_t compute,
                              moe_stream_t copy_in, moe_stream_t copy_out);

/*
 * One-time weight transform (untimed, before the layers run; the counterpart
 * of the weight pre-transform the pages describe for DeepGEMM's Mega MoE
 * kernel, "大模型系统中的通算融合" §4.4).  Writes w13 and w2 (row-major, bf16)
 * in MOE_WEIGHTS_TILED layout: each 64 x 64 block (64 rows of k, 64 columns)
 * of every expert's matrix becomes one contiguous 8 KB run, ordered by
 * expert, then row block, then column block:
 *   w13_tiled[((e*(H/64) + kb)*(2I/64) + nb)*4096 + r*64 + c]
 *     = w13[e][64 kb + r][64 nb + c]          (and likewise w2 with I, H)
 * so every tile the grouped GEMMs load is one contiguous DRAM run instead of
 * 64 runs of 128 bytes a matrix row apart.  w13_tiled and w2_tiled have the
 * sizes of w13 and w2 and must not overlap them.  desc: bf16, H % 64 == 0,
 * I % 128 == 0 (weight_layout is ignored).  Enqueued on `stream`.
 */
moe_status_t moe_prepare_weights(const moe_layer_desc_t *desc, const void *w13, const void *w2,
                                 void *w13_tiled, void *w2_tiled, moe_stream_t stream);

/*
 * One-time transform of the router weight (bf16 layers): w_gate_t[e][h] =
 * w_gate[h][e], (E, H) bf16, for moe_layer_desc_t.w_gate_t.  w_gate_t must
 * not overlap w_gate and must be 16-byte aligned.  Enqueued on `stream`.
 * MOE_ERR_UNSUPPORTED for float32 layers; MOE_ERR_INVALID_ARG for NULL or
 * misaligned pointers.
 */
moe_status_t moe_prepare_router(const moe_layer_desc_t *desc, const void *w_gate,
                                void *w_gate_t, moe_stream_t stream);

/*
 * Test control for the device timeout path (failure detection without a
 * fault): the number of SM clock cycles a pipeline wait of the tensor-core
 * grouped GEMMs (moe_expert_gemm1_swiglu, moe_expert_gemm2,
 * moe_expert_gemm2_weighted, moe_expert_gemm1_swiglu_gather, the forward and
 * moe_backward's GEMMs) and weight-gradient GEMMs waits before it gives up.
 * A wait that gives up ORs MOE_DEV_TIMEOUT into the status word; every role
 * of the CTA then stops, waits (with the full limit) for the copies and MMAs
 * it has in flight, frees its tensor memory and leaves, so the context stays
 * usable.  0 restores the default (2^31 cycles, about a second at 2 GHz).
 * Applies to launches enqueued after the call, from any host thread.
 * Returns MOE_ERR_INVALID_ARG for a negative value.
 */
moe_status_t moe_set_pipeline_wait_limit(long long cycles);

/*
 * Tuning control of the tensor-core grouped GEMMs (bf16: moe_expert_gemm1_swiglu,
 * moe_expert_gemm2, moe_expert_gemm2_weighted, the forward's GEMMs, and
 * moe_backward's dgrad, SwiGLU-backward and weight-gradient GEMMs; not
 * moe_expert_gemm1_swiglu_gather): enable != 0 (the default) runs them on CTA
 * pairs -- clusters of two CTAs on two SMs computing 256-row x 256-column
 * tiles with cta_group::2 MMAs, each CTA holding its own 128 rows of A and half
 * of the B tile, which gives six operand stages instead of four; enable == 0
 * runs one CTA per SM with 128-row tiles.  The results are bitwise the same
 * either way.  Applies to launches enqueued after the call, from any host
 * thread.  Always returns MOE_OK.
 */
moe_status_t moe_set_gemm_pairs(int enable);

/*
 * Tuning control of the forward grouped GEMMs on CTA pairs
 * (moe_expert_gemm1_swiglu, moe_expert_gemm2, moe_expert_gemm2_weighted and
 * the forward's GEMMs; without effect on single CTAs and on the backward):
 * "fused tails".  An expert whose segment ends 1..32 rows past a 256-row
 * window boundary, after at least one full window, computes those rows inside
 * its last full window's tiles, transposed: per k stage the pair adds
 * M = 256, N = 32 MMAs that reuse the stage's weight columns as A and take
 * the tail rows as B, instead of a 256-row window of their own (Algorithm 2
 * steps 8-9 of "MoE 分布式推理基础（基于 vLLM）" §1.2 are unchanged: every row
 * is multiplied by its expert's weights).  mode < 0 (the default) chooses per
 * launch: on when the layer averages 192..384 rows per expert (n*K/E), where
 * about half of the experts save a window; mode == 0 never, mode > 0 always.
 * The results are bitwise the same either way.  Applies to launches enqueued
 * after the call, from any host thread.  Always returns MOE_OK.
 */
moe_status_t moe_set_gemm_tails(int mode);

/*
 * Blocks until `stream` is idle, then reads *status_word and maps it to
 * MOE_OK, MOE_ERR_BAD_ROUTING, MOE_ERR_BAD_LAYOUT or MOE_ERR_TIMEOUT (first
 * match in that order).  Intended for tests and debugging.
 */
moe_status_t moe_check_status(const int32_t *status_word, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
