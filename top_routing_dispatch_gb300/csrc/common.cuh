// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxE = 256;
constexpr int kMaxK = 16;

// Near-tie margins of the router, relative to max(1, |largest logit|).  A
// token whose top K+1 float32 logits have an adjacent gap below the margin
// has its candidate experts rescored in double-float.  The margin must stay
// above twice the largest float32 logit error: for the FMA-unit logits
// (float32 chains of 32 products) and for the tensor-core logits (float32
// accumulation in the tensor cores) that error is measured by the GPU parity
// tests against the float64 oracle.
constexpr float kTieMarginSimt = 1e-3f;
constexpr float kTieMarginTc = 1e-4f;  // scaled by max(1, H / 2048): see tie_margin_tc

// The tensor cores' float32 accumulation error grows about linearly with the
// length of the sum (measured), so their margin scales with H.
__host__ __device__ inline float tie_margin_tc(int H) {
  return kTieMarginTc * (H > 2048 ? (float)H / 2048.f : 1.f);
}

struct Desc {
  int n, H, I, E, K;
  bool bf16;
  bool norm;
  bool tiled;  // expert weights in MOE_WEIGHTS_TILED layout
  const void *w_gate_t;  // optional (E, H) transposed router weight (bf16), or null
  long long nK() const { return (long long)n * K; }
};

inline size_t elem_bytes(const Desc &d) { return d.bf16 ? 2 : 4; }

// ---- router.cu (dispatches to router_mma.cu or router_tc.cu for bf16 layers)
// guest: launch the configuration that fits beside a persistent GEMM CTA on
// an SM (same results, shallower pipeline); only the warp-level MMA router has
// one, the other routers ignore it
cudaError_t launch_router(const Desc &d, const void *x, const void *w_gate, const float *bias,
                          int32_t *topk_idx, float *topk_w, float *logits, int32_t *status,
                          cudaStream_t s, bool guest = false);
bool router_tc_supported(const Desc &d);
// kernels launch_router enqueues for this layer
int router_launches(const Desc &d);
// router_mma.cu: warp-level MMA router (bf16, E = 64 or 128, K <= 8), one kernel
bool router_mma_supported(const Desc &d);
cudaError_t launch_router_mma(const Desc &d, const void *x, const void *w_gate, const float *bias,
                              int32_t *topk_idx, float *topk_w, float *logits, bool guest,
                              cudaStream_t s);
cudaError_t launch_router_tc(const Desc &d, const void *x, const void *w_gate, const float *bias,
                             int32_t *topk_idx, float *topk_w, float *logits, int32_t *status,
                             cudaStream_t s);

// ---- layout.cu
size_t layout_ws_bytes(const Desc &d);
cudaError_t launch_layout(const Desc &d, const int32_t *topk_idx, int32_t *counts,
                          int32_t *offsets, int32_t *perm, int32_t *inv_perm, int32_t *status,
                          void *ws, cudaStream_t s, bool guest = false);

// ---- permute_combine.cu
cudaError_t launch_permute(const Desc &d, const void *x, const int32_t *perm, void *x_perm,
                           int32_t *status, cudaStream_t s, bool guest = false);
// x_perm[inv_perm[t*K + k]] = x[t]: x read once (bitwise equal to launch_permute)
cudaError_t launch_permute_scatter(const Desc &d, const void *x, const int32_t *inv_perm,
                                   void *x_perm, int32_t *status, cudaStream_t s,
                                   bool guest = false);
cudaError_t launch_combine(const Desc &d, const void *y_perm, const float *topk_w,
                           const int32_t *inv_perm, void *y, int32_t *status, cudaStream_t s,
                           bool guest = false);

// ---- gemm_tc.cu (bf16, tcgen05) and gemm_simt.cu (float32)
cudaError_t launch_gemm1_tc(const Desc &d, const void *x_perm, const void *w13,
                            const int32_t *offsets, void *h, int sm_reserve, int32_t *status,
                            cudaStream_t s);
cudaError_t launch_gemm1_tc_gather(const Desc &d, const void *x, const int32_t *perm,
                                   const void *w13, const int32_t *offsets, void *h,
                                   int sm_reserve, int32_t *status, cudaStream_t s);
cudaError_t launch_gemm2_tc(const Desc &d, const void *h, const void *w2, const int32_t *offsets,
                            void *y_perm, int sm_reserve, int32_t *status, cudaStream_t s);
// The grouped GEMMs (every mode but the fused gather, and the weight
// gradients) run on CTA pairs (cta_group::2, 256-row tiles) unless single CTAs
// are selected (moe_set_gemm_pairs); bitwise the same results.
void set_gemm_single_cta(bool single);
bool gemm_single_cta();
// Fused tails of the forward pair GEMMs (moe_set_gemm_tails): -1 automatic,
// 0 off, 1 on.
void set_gemm_tails(int mode);
// GEMM2 with the routing weight applied and each row written to its
// (token, slot) position: y_slot[perm[r]] = topk_w[perm[r]] * (h W2[e])[r]
cudaError_t launch_gemm2_tc_weighted(const Desc &d, const void *h, const void *w2,
                                     const int32_t *offsets, const int32_t *perm,
                                     const float *topk_w, void *y_slot, int sm_reserve,
                                     int32_t *status, cudaStream_t s);
// y[t] = sum over k of y_slot[t*K + k] (float32, slot order, one rounding)
cudaError_t launch_combine_slots(const Desc &d, const void *y_slot, void *y, cudaStream_t s,
                                 bool guest = false);
// backward (backward.cu, gemm_tc.cu modes 5 and 6, gemm_wgrad.cu)
constexpr int kRouterBwdSplit = 16;  // token ranges of the dW_gate reduction
cudaError_t launch_combine_bwd(const Desc &d, const void *dy, const void *y_perm,
                               const float *topk_w, const int32_t *inv_perm, void *dY, float *dw,
                               int32_t *status, cudaStream_t s);
cudaError_t launch_router_bwd(const Desc &d, const void *x, const float *logits,
                              const int32_t *topk_idx, const float *topk_w, const float *dw,
                              float *dlogits, float *dw_part, float *dw_gate, float *dbias,
                              cudaStream_t s);
cudaError_t launch_dx_final(const Desc &d, const void *dx_perm, const float *dlogits,
                            const void *w_gate, const int32_t *inv_perm, void *dx,
                            cudaStream_t s);
cudaError_t launch_gemm_dgrad_tc(const Desc &d, const void *a, const void *w, int Kdim, int Nout,
                                 const int32_t *offsets, void *out, int32_t *status,
                                 cudaStream_t s);
cudaError_t launch_gemm1_swiglu_bwd_tc(const Desc &d, const void *x_perm, const void *w13,
                                       const int32_t *offsets, const void *dh, void *dgu,
                                       int32_t *status, cudaStream_t s);
size_t wgrad_tail_bytes(const Desc &d, int M, int N);
cudaError_t launch_wgrad_tc(const Desc &d, const void *a, int M, const void *b, int N,
                            const int32_t *offsets, void *tail, float *out, int32_t *status,
                            cudaStream_t s);
cudaError_t launch_gemm1_simt(const Desc &d, const void *x_perm, const void *w13,
                              const int32_t *offsets, void *h, int32_t *status, cudaStream_t s);
cudaError_t launch_gemm2_simt(const Desc &d, const void *h, const void *w2,
                              const int32_t *offsets, void *y_perm, int32_t *status,
                              cudaStream_t s);

// GEMM1 (+SwiGLU) then GEMM2 for the layer's dtype.
inline cudaError_t launch_experts(const Desc &d, const void *x_perm, const void *w13,
                                  const void *w2, const int32_t *offsets, void *h, void *y_perm,
                                  int sm_reserve, int32_t *status, cudaStream_t s) {
  cudaError_t e = d.bf16 ? launch_gemm1_tc(d, x_perm, w13, offsets, h, sm_reserve, status, s)
                         : launch_gemm1_simt(d, x_perm, w13, offsets, h, status, s);
  if (e != cudaSuccess) return e;
  return d.bf16 ? launch_gemm2_tc(d, h, w2, offsets, y_perm, sm_reserve, status, s)
                : launch_gemm2_simt(d, h, w2, offsets, y_perm, status, s);
}

// prepare.cu: w13 (E,H,2I) and w2 (E,I,H) into 64 x 64 tiles (MOE_WEIGHTS_TILED)
cudaError_t launch_prepare_weights(const Desc &d, const void *w13, const void *w2, void *w13t,
                                   void *w2t, cudaStream_t s);
// prepare.cu: w_gate (H, E) bf16 transposed into w_gate_t (E, H)
cudaError_t launch_prepare_router(const Desc &d, const void *w_gate, void *w_gate_t,
                                  cudaStream_t s);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Cycles a pipeline wait of the tcgen05 GEMM kernels waits before it gives up
// (moe_set_pipeline_wait_limit; default about a second).
long long pipeline_wait_limit();

}  // namespace moe

// ---- device helpers
namespace moe {

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation (launch_pdl) and starts with pdl_enter():
// it waits until the preceding kernel of its stream has completed and its
// writes are visible (griddepcontrol.wait, before any global-memory access),
// then lets the next kernel of the stream begin launching.  The next kernel's
// launch and set-up thus overlap this kernel's tail; no kernel reads or
// writes global memory before its predecessor has finished.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Launch on the dispatch stream of the two-stream schedule, beside the
// persistent GEMM of the other stream ("guest"): without programmatic stream
// serialisation, so no CTA of the stream's next kernel sits resident on an SM
// waiting for this one.  Otherwise as launch_pdl.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(bool guest, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                            size_t smem, cudaStream_t s, Args &&...args) {
  if (!guest) return launch_pdl(kernel, grid, block, smem, s, static_cast<Args &&>(args)...);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Prefer the largest shared-memory carveout for a kernel that may share an
// SM with the grouped GEMM (whose CTA needs ~210 KB): an SM that starts one of
// its CTAs then keeps the configuration the GEMM needs.  Set once per device.
template <typename... KArgs>
inline cudaError_t prefer_max_shared(void (*kernel)(KArgs...)) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

__device__ __forceinline__ void flag_status(int32_t *status, int bits) {
  if (status) atomicOr(status, bits);
}

// Number of m-tiles of `bm` rows for segment lengths given by offsets.
__device__ __forceinline__ int ceil_div_dev(int a, int b) { return (a + b - 1) / b; }

}  // namespace moe
