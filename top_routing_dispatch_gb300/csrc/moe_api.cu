// C ABI of the MoE layer: argument checks, workspace layout, and the
// two-stream micro-batch schedule.  Kernels live in the other .cu files.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <map>
#include <mutex>

#include "common.cuh"

namespace moe {

namespace {
std::atomic<long long> g_wait_limit{0};  // 0: the default
}  // namespace

long long pipeline_wait_limit() {
  const long long v = g_wait_limit.load(std::memory_order_relaxed);
  return v > 0 ? v : (1ll << 31);
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int sms = 1;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) cache[dev] = sms;
  return sms;
}

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared checks of the layer description.
moe_status_t check_desc(const moe_layer_desc_t *d, Desc *out) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->n < 0 || d->H < 1 || d->I < 1 || d->E < 1 || d->K < 1) return MOE_ERR_INVALID_ARG;
  if (d->K > d->E) return MOE_ERR_INVALID_ARG;
  if (d->dtype != MOE_F32 && d->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (d->weight_layout != MOE_WEIGHTS_ROW_MAJOR && d->weight_layout != MOE_WEIGHTS_TILED)
    return MOE_ERR_INVALID_ARG;
  if (d->E > kMaxE || d->K > kMaxK) return MOE_ERR_UNSUPPORTED;
  // the transposed router weight is read in 16-byte pieces
  if (d->w_gate_t && (reinterpret_cast<uintptr_t>(d->w_gate_t) & 15)) return MOE_ERR_INVALID_ARG;
  if ((long long)d->n * d->K > 0x7fffffffll) return MOE_ERR_UNSUPPORTED;
  const bool bf16 = d->dtype == MOE_BF16;
  // rows move as 16-byte vectors
  if (bf16 ? (d->H % 8) : (d->H % 4)) return MOE_ERR_UNSUPPORTED;
  out->n = d->n;
  out->H = d->H;
  out->I = d->I;
  out->E = d->E;
  out->K = d->K;
  out->bf16 = bf16;
  out->norm = d->norm_topk_prob != 0;
  out->tiled = d->weight_layout == MOE_WEIGHTS_TILED;
  out->w_gate_t = bf16 ? d->w_gate_t : nullptr;
  return MOE_OK;
}

moe_status_t check_gemm_shape(const Desc &d) {
  if (d.bf16) {
    if (d.H % 64 || d.I % 128) return MOE_ERR_UNSUPPORTED;
  } else {
    if (d.I % 4 || d.tiled) return MOE_ERR_UNSUPPORTED;  // float32 layers read row-major weights
  }
  return MOE_OK;
}

inline moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

constexpr size_t kAlign = 256;
// x larger than this (a quarter of the L2) is permuted in scatter form
constexpr size_t kScatterPermuteBytes = 32ull << 20;
inline size_t up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

enum Slot {
  S_LOGITS = 0, S_TOPK_IDX, S_TOPK_W, S_COUNTS, S_OFFSETS, S_PERM, S_INV_PERM,
  S_X_PERM, S_H, S_Y_PERM, S_STATUS, S_LAYOUT_WS, S_COUNT
};

void slot_sizes(const Desc &d, size_t sz[S_COUNT]) {
  const size_t nK = (size_t)d.nK(), eb = elem_bytes(d);
  sz[S_LOGITS] = (size_t)d.n * d.E * 4;
  sz[S_TOPK_IDX] = nK * 4;
  sz[S_TOPK_W] = nK * 4;
  sz[S_COUNTS] = (size_t)d.E * 4;
  sz[S_OFFSETS] = (size_t)(d.E + 1) * 4;
  sz[S_PERM] = nK * 4;
  sz[S_INV_PERM] = nK * 4;
  sz[S_X_PERM] = nK * d.H * eb;
  sz[S_H] = nK * d.I * eb;
  sz[S_Y_PERM] = nK * d.H * eb;
  sz[S_STATUS] = 4;
  sz[S_LAYOUT_WS] = layout_ws_bytes(d);
}

size_t mb_bytes(const Desc &d) {
  size_t sz[S_COUNT];
  slot_sizes(d, sz);
  size_t tot = 0;
  for (int i = 0; i < S_COUNT; ++i) tot += up(sz[i] ? sz[i] : 1);
  return tot;
}

uint8_t *slot_ptr(const Desc &d, void *ws, int mb, int which) {
  size_t sz[S_COUNT];
  slot_sizes(d, sz);
  size_t off = mb_bytes(d) * (size_t)mb;
  for (int i = 0; i < which; ++i) off += up(sz[i] ? sz[i] : 1);
  return reinterpret_cast<uint8_t *>(ws) + off;
}

// Events reused by moe_forward_microbatches, per device.  A wait captures the
// most recent record at the time it is enqueued, so reuse across calls is
// safe; the mutex serialises enqueueing from several host threads.
constexpr int kMaxMB = 64;
constexpr int kPoolEvents = 4 * kMaxMB + 3;
// Per device: the events of moe_forward_microbatches and the library's own
// dispatch stream, created at the highest stream priority.  The two-stream
// schedule runs its dispatch-side kernels there: the block scheduler then
// serves their CTAs before CTAs of the compute stream's next GEMM, which a
// programmatic launch makes pending while the current GEMM still holds every
// SM (at equal priority those pending GEMM CTAs hold back the small dispatch
// kernels until the GEMM ends).
struct EventPool {
  cudaEvent_t ev[kPoolEvents];
  cudaStream_t hi = nullptr;
  bool ready = false;
};
EventPool g_pools[64];
std::mutex g_pool_mu;

// events of one host pipeline (one workspace): per staging slot, x copied in,
// layer finished (x read, y written), y copied out
struct HostEvents {
  cudaEvent_t in[2], layer[2], out[2];
  unsigned long long last_use;
};
// At most kMaxHostPipelines pipelines keep their events; a new one replaces
// the least recently used, whose recorded work is waited for first (so its
// workspace's ordering is never lost while still in flight).
constexpr size_t kMaxHostPipelines = 64;
std::map<std::pair<int, const void *>, HostEvents> g_host_events;
unsigned long long g_host_clock = 0;
std::mutex g_host_mu;

void destroy_host_events(HostEvents &h) {
  for (int k = 0; k < 2; ++k) {
    cudaEvent_t evs[3] = {h.in[k], h.layer[k], h.out[k]};
    for (cudaEvent_t ev : evs) {
      cudaEventSynchronize(ev);
      cudaEventDestroy(ev);
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_version(void) { return "top_routing_dispatch_gb300 0.1 (sm_103a)"; }

const char *moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_BAD_ROUTING: return "expert id out of range in topk_idx";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MOE_ERR_BAD_LAYOUT: return "inconsistent dispatch layout";
  }
  return "unknown status";
}

moe_status_t moe_route_topk(const moe_layer_desc_t *desc, const void *x, const void *w_gate,
                            const float *bias, int32_t *topk_idx, float *topk_w, float *logits,
                            moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (d.n == 0) return MOE_OK;
  if (!x || !w_gate || !topk_idx || !topk_w || !logits) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_router(d, x, w_gate, bias, topk_idx, topk_w, logits, nullptr, stream));
}

size_t moe_layout_workspace_size(const moe_layer_desc_t *desc) {
  Desc d;
  if (check_desc(desc, &d) != MOE_OK) return 0;
  return layout_ws_bytes(d);
}

moe_status_t moe_dispatch_layout(const moe_layer_desc_t *desc, const int32_t *topk_idx,
                                 int32_t *counts, int32_t *offsets, int32_t *perm,
                                 int32_t *inv_perm, int32_t *status_word, void *ws,
                                 size_t ws_bytes, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (!counts || !offsets || !status_word) return MOE_ERR_INVALID_ARG;
  if (d.nK() > 0 && (!topk_idx || !perm || !inv_perm || !ws)) return MOE_ERR_INVALID_ARG;
  if (d.nK() > 0 && ws_bytes < layout_ws_bytes(d)) return MOE_ERR_WORKSPACE;
  return cuda_status(
      launch_layout(d, topk_idx, counts, offsets, perm, inv_perm, status_word, ws, stream));
}

moe_status_t moe_permute(const moe_layer_desc_t *desc, const void *x, const int32_t *perm,
                         void *x_perm, int32_t *status_word, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (d.nK() == 0) return MOE_OK;
  if (!x || !perm || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_permute(d, x, perm, x_perm, status_word, stream));
}

moe_status_t moe_permute_scatter(const moe_layer_desc_t *desc, const void *x,
                                 const int32_t *inv_perm, void *x_perm, int32_t *status_word,
                                 moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (d.nK() == 0) return MOE_OK;
  if (!x || !inv_perm || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_permute_scatter(d, x, inv_perm, x_perm, status_word, stream));
}

moe_status_t moe_grouped_swiglu(const moe_layer_desc_t *desc, const void *x_perm, const void *w13,
                                const void *w2, const int32_t *offsets, void *h, void *y_perm,
                                int sm_reserve, int32_t *status_word, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  st = check_gemm_shape(d);
  if (st != MOE_OK) return st;
  if (d.nK() == 0) return MOE_OK;
  if (!x_perm || !w13 || !w2 || !offsets || !h || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w13) || !aligned16(w2) || !aligned16(h) ||
      !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;
  if (sm_reserve < 0) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_experts(d, x_perm, w13, w2, offsets, h, y_perm, sm_reserve, status_word, stream));
}

moe_status_t moe_expert_gemm1_swiglu(const moe_layer_desc_t *desc, const void *x_perm,
                                     const void *w13, const int32_t *offsets, void *h,
                                     int sm_reserve, int32_t *status_word, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  st = check_gemm_shape(d);
  if (st != MOE_OK) return st;
  if (d.nK() == 0) return MOE_OK;
  if (!x_perm || !w13 || !offsets || !h || sm_reserve < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w13) || !aligned16(h)) return MOE_ERR_INVALID_ARG;
  return cuda_status(d.bf16 ? launch_gemm1_tc(d, x_perm, w13, offsets, h, sm_reserve,
                                              status_word, stream)
                            : launch_gemm1_simt(d, x_perm, w13, offsets, h, status_word, stream));
}

moe_status_t moe_expert_gemm1_swiglu_gather(const moe_layer_desc_t *desc, const void *x,
                                            const int32_t *perm, const void *w13,
                                            const int32_t *offsets, void *h, int sm_reserve,
                                            int32_t *status_word, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (!d.bf16) return MOE_ERR_UNSUPPORTED;
  st = check_gemm_shape(d);
  if (st != MOE_OK) return st;
  if (d.nK() == 0) return MOE_OK;
  if (!x || !perm || !w13 || !offsets || !h || sm_reserve < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(h)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_gemm1_tc_gather(d, x, perm, w13, offsets, h, sm_reserve, status_word, stream));
}

moe_status_t moe_expert_gemm2(const moe_layer_desc_t *desc, const void *h, const void *w2,
                              const int32_t *offsets, void *y_perm, int sm_reserve,
                              int32_t *status_word, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  st = check_gemm_shape(d);
  if (st != MOE_OK) return st;
  if (d.nK() == 0) return MOE_OK;
  if (!h || !w2 || !offsets || !y_perm || sm_reserve < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w2) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  return cuda_status(d.bf16 ? launch_gemm2_tc(d, h, w2, offsets, y_perm, sm_reserve, status_word,
                                              stream)
                            : launch_gemm2_simt(d, h, w2, offsets, y_perm, status_word, stream));
}

moe_status_t moe_expert_gemm2_weighted(const moe_layer_desc_t *desc, const void *h,
                                       const void *w2, const int32_t *offsets,
                                       const int32_t *perm, const float *topk_w, void *y_slot,
                                       int sm_reserve, int32_t *status_word,
                                       moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (!d.bf16) return MOE_ERR_UNSUPPORTED;
  st = check_gemm_shape(d);
  if (st != MOE_OK) return st;
  if (d.nK() == 0) return MOE_OK;
  if (!h || !w2 || !offsets || !perm || !topk_w || !y_slot || sm_reserve < 0)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w2) || !aligned16(y_slot)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gemm2_tc_weighted(d, h, w2, offsets, perm, topk_w, y_slot,
                                              sm_reserve, status_word, stream));
}

moe_status_t moe_combine_slots(const moe_layer_desc_t *desc, const void *y_slot, void *y,
                               moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (d.n == 0) return MOE_OK;
  if (!y_slot || !y || !aligned16(y_slot) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine_slots(d, y_slot, y, stream));
}

moe_status_t moe_combine(const moe_layer_desc_t *desc, const void *y_perm, const float *topk_w,
                         const int32_t *inv_perm, void *y, int32_t *status_word,
                         moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (d.n == 0) return MOE_OK;
  if (!y_perm || !topk_w || !inv_perm || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(d, y_perm, topk_w, inv_perm, y, status_word, stream));
}

size_t moe_workspace_size(const moe_layer_desc_t *desc) {
  Desc d;
  if (check_desc(desc, &d) != MOE_OK) return 0;
  return mb_bytes(d);
}

int moe_forward_launches(const moe_layer_desc_t *desc) {
  Desc d;
  if (check_desc(desc, &d) != MOE_OK) return 0;
  const bool pairs = d.nK() > 0;
  // router | layout count + scan/scatter | permute | GEMM1, GEMM2 | combine
  return router_launches(d) + (pairs ? 2 + 1 + 2 : 0) + (d.n > 0 ? 1 : 0);
}

void *moe_workspace_slot(const moe_layer_desc_t *desc, void *ws, int mb, int which) {
  Desc d;
  if (!ws || mb < 0 || which < 0 || which >= S_LAYOUT_WS) return nullptr;
  if (check_desc(desc, &d) != MOE_OK) return nullptr;
  return slot_ptr(d, ws, mb, which);
}

moe_status_t moe_forward_microbatches(const moe_layer_desc_t *desc, int num_mb,
                                      const void *const *x, const void *w_gate, const float *bias,
                                      const void *w13, const void *w2, void *const *y, void *ws,
                                      size_t ws_bytes, int sm_reserve, int32_t *status_word,
                                      moe_stream_t compute, moe_stream_t dispatch) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  st = check_gemm_shape(d);
  if (st != MOE_OK) return st;
  if (num_mb < 1 || num_mb > kMaxMB || !x || !y || sm_reserve < 0) return MOE_ERR_INVALID_ARG;
  if (!w_gate || !w13 || !w2 || !ws) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < mb_bytes(d) * (size_t)num_mb) return MOE_ERR_WORKSPACE;
  for (int j = 0; j < num_mb; ++j) {
    if (d.n > 0 && (!x[j] || !y[j] || !aligned16(x[j]) || !aligned16(y[j])))
      return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(w13) || !aligned16(w2)) return MOE_ERR_INVALID_ARG;
  int32_t *status = status_word ? status_word
                                : reinterpret_cast<int32_t *>(slot_ptr(d, ws, 0, S_STATUS));
  cudaStream_t sc = compute;
  cudaStream_t sd = dispatch ? dispatch : compute;  // replaced by the library's stream below
  const bool two = sd != sc;

  // guest: a dispatch-stream launch that runs beside the other stream's GEMM
  // (see launch_k); every result is the same either way
  auto route = [&](int j, cudaStream_t s, bool guest) -> cudaError_t {
    return launch_router(d, x[j], w_gate, bias, (int32_t *)slot_ptr(d, ws, j, S_TOPK_IDX),
                         (float *)slot_ptr(d, ws, j, S_TOPK_W),
                         (float *)slot_ptr(d, ws, j, S_LOGITS), status, s, guest);
  };
  auto route_layout = [&](int j, cudaStream_t s, bool guest) -> cudaError_t {
    cudaError_t e = route(j, s, guest);
    if (e == cudaSuccess)
      e = launch_layout(d, (const int32_t *)slot_ptr(d, ws, j, S_TOPK_IDX),
                        (int32_t *)slot_ptr(d, ws, j, S_COUNTS),
                        (int32_t *)slot_ptr(d, ws, j, S_OFFSETS),
                        (int32_t *)slot_ptr(d, ws, j, S_PERM),
                        (int32_t *)slot_ptr(d, ws, j, S_INV_PERM), status,
                        slot_ptr(d, ws, j, S_LAYOUT_WS), s, guest);
    return e;
  };
  // the permute in gather form (x rows re-read K times, from L2 while x fits
  // there) or scatter form (x read once): bitwise equal, chosen by the size of
  // x -- measured on GB300: gather 83 % / scatter 73 % of HBM at 16.8 MB of x,
  // gather 60 % / scatter 80 % at 117 MB
  const bool scatter = (size_t)d.n * d.H * elem_bytes(d) > kScatterPermuteBytes;
  auto permute = [&](int j, cudaStream_t s, bool guest) -> cudaError_t {
    if (scatter)
      return launch_permute_scatter(d, x[j], (const int32_t *)slot_ptr(d, ws, j, S_INV_PERM),
                                    slot_ptr(d, ws, j, S_X_PERM), status, s, guest);
    return launch_permute(d, x[j], (int32_t *)slot_ptr(d, ws, j, S_PERM),
                          slot_ptr(d, ws, j, S_X_PERM), status, s, guest);
  };
  auto front = [&](int j, cudaStream_t s, bool guest) -> cudaError_t {  // route, layout, permute
    cudaError_t e = route_layout(j, s, guest);
    if (e == cudaSuccess) e = permute(j, s, guest);
    return e;
  };
  // bf16: GEMM2 applies the routing weights and writes each row to its
  // (token, slot) position (slot y_perm of the workspace), and the combine
  // adds each token's K contiguous rows; float32: GEMM2 writes y_perm in
  // expert order and the combine gathers and weights
  const int reserve = two ? sm_reserve : 0;
  auto gemm1 = [&](int j, cudaStream_t s) -> cudaError_t {
    const int32_t *off = (const int32_t *)slot_ptr(d, ws, j, S_OFFSETS);
    return d.bf16 ? launch_gemm1_tc(d, slot_ptr(d, ws, j, S_X_PERM), w13, off,
                                    slot_ptr(d, ws, j, S_H), reserve, status, s)
                  : launch_gemm1_simt(d, slot_ptr(d, ws, j, S_X_PERM), w13, off,
                                      slot_ptr(d, ws, j, S_H), status, s);
  };
  auto gemm2 = [&](int j, cudaStream_t s) -> cudaError_t {
    const int32_t *off = (const int32_t *)slot_ptr(d, ws, j, S_OFFSETS);
    if (!d.bf16)
      return launch_gemm2_simt(d, slot_ptr(d, ws, j, S_H), w2, off, slot_ptr(d, ws, j, S_Y_PERM),
                               status, s);
    return launch_gemm2_tc_weighted(d, slot_ptr(d, ws, j, S_H), w2, off,
                                    (const int32_t *)slot_ptr(d, ws, j, S_PERM),
                                    (const float *)slot_ptr(d, ws, j, S_TOPK_W),
                                    slot_ptr(d, ws, j, S_Y_PERM), reserve, status, s);
  };
  auto experts = [&](int j, cudaStream_t s) -> cudaError_t {
    cudaError_t e = gemm1(j, s);
    return e == cudaSuccess ? gemm2(j, s) : e;
  };
  auto back = [&](int j, cudaStream_t s, bool guest) -> cudaError_t {
    if (d.bf16) return launch_combine_slots(d, slot_ptr(d, ws, j, S_Y_PERM), y[j], s, guest);
    return launch_combine(d, slot_ptr(d, ws, j, S_Y_PERM),
                          (const float *)slot_ptr(d, ws, j, S_TOPK_W),
                          (const int32_t *)slot_ptr(d, ws, j, S_INV_PERM), y[j], status, s,
                          guest);
  };

  if (!two) {
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), sc);
    for (int j = 0; j < num_mb && e == cudaSuccess; ++j) {
      e = front(j, sc, false);
      if (e == cudaSuccess) e = experts(j, sc);
      if (e == cudaSuccess) e = back(j, sc, false);
    }
    return cuda_status(e);
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  EventPool &pool = g_pools[dev];
  if (!pool.ready) {
    for (int i = 0; i < kPoolEvents; ++i)
      if (cudaEventCreateWithFlags(&pool.ev[i], cudaEventDisableTiming) != cudaSuccess)
        return MOE_ERR_CUDA;
    int lo = 0, hi = 0;
    if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess ||
        cudaStreamCreateWithPriority(&pool.hi, cudaStreamNonBlocking, hi) != cudaSuccess)
      return MOE_ERR_CUDA;
    pool.ready = true;
  }
  cudaEvent_t ev_start = pool.ev[4 * kMaxMB], ev_done = pool.ev[4 * kMaxMB + 1];
  cudaEvent_t ev_caller = pool.ev[4 * kMaxMB + 2];
  cudaEvent_t *ev_front = pool.ev, *ev_gemm = pool.ev + kMaxMB, *ev_g1 = pool.ev + 2 * kMaxMB;
  cudaStream_t caller_d = sd;
  sd = pool.hi;

  // Schedule (D = the library's high-priority dispatch stream, joined to the
  // caller's compute and dispatch streams by events; C = compute stream):
  //   D: front(0) | route+layout(1)  permute(1) | combine(0) route+layout(2) ...
  //   C:          | GEMM1(0)         GEMM2(0)   | GEMM1(1)   GEMM2(1)  ...
  // Micro-batch j+1's route and layout run beside GEMM1(j), its permute (which
  // writes x_perm, the largest stream of the dispatch) beside GEMM2(j), and
  // combine(j-1) beside GEMMs(j).  They are launched as guests: at most one
  // CTA per SM, each small enough (registers, shared memory, no TMEM) to sit
  // beside the persistent GEMM CTA, and without programmatic serialisation, so
  // no CTA of the next kernel on D waits resident on an SM.  front(0) and the
  // last combine have no GEMM to hide under and run at full width.
  cudaError_t e = cudaEventRecord(ev_start, sc);
  if (e == cudaSuccess) e = cudaEventRecord(ev_caller, caller_d);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, ev_caller, 0);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int32_t), sd);
  if (e == cudaSuccess) e = front(0, sd, false);
  if (e == cudaSuccess) e = cudaEventRecord(ev_front[0], sd);
  for (int j = 0; j < num_mb && e == cudaSuccess; ++j) {
    e = cudaStreamWaitEvent(sc, ev_front[j], 0);                   // GEMMs of j on C
    if (e == cudaSuccess) e = gemm1(j, sc);
    if (e == cudaSuccess) e = cudaEventRecord(ev_g1[j], sc);
    if (e == cudaSuccess) e = gemm2(j, sc);
    if (e == cudaSuccess) e = cudaEventRecord(ev_gemm[j], sc);
    if (j > 0) {                                                   // combine of j-1 on D
      if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, ev_gemm[j - 1], 0);
      if (e == cudaSuccess) e = back(j - 1, sd, true);
    }
    if (j + 1 < num_mb) {                                          // front of j+1 on D
      if (e == cudaSuccess) e = route_layout(j + 1, sd, true);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, ev_g1[j], 0);
      if (e == cudaSuccess) e = permute(j + 1, sd, true);
      if (e == cudaSuccess) e = cudaEventRecord(ev_front[j + 1], sd);
    }
  }
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, ev_gemm[num_mb - 1], 0);
  if (e == cudaSuccess) e = back(num_mb - 1, sd, false);
  if (e == cudaSuccess) e = cudaEventRecord(ev_done, sd);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, ev_done, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(caller_d, ev_done, 0);
  return cuda_status(e);
}

size_t moe_host_workspace_size(const moe_layer_desc_t *desc) {
  Desc d;
  if (check_desc(desc, &d) != MOE_OK) return 0;
  const size_t io = up((size_t)d.n * d.H * elem_bytes(d));
  return mb_bytes(d) + 4 * io;
}

moe_status_t moe_forward_host(const moe_layer_desc_t *desc, const void *x_host,
                              const void *w_gate, const float *bias, const void *w13,
                              const void *w2, void *y_host, void *ws, size_t ws_bytes,
                              long long call, int32_t *status_word, moe_stream_t compute,
                              moe_stream_t copy_in, moe_stream_t copy_out) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  st = check_gemm_shape(d);
  if (st != MOE_OK) return st;
  if (!ws || !w_gate || !w13 || !w2 || call < 0) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_host_workspace_size(desc)) return MOE_ERR_WORKSPACE;
  if (d.n == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  const size_t bytes = (size_t)d.n * d.H * elem_bytes(d);
  const size_t io = up(bytes);
  const int slot = (int)(call & 1);
  uint8_t *stage = reinterpret_cast<uint8_t *>(ws) + mb_bytes(d) + (size_t)slot * 2 * io;
  void *xs = stage, *ys = stage + io;
  cudaStream_t sc = compute;
  cudaStream_t si = copy_in ? copy_in : sc;
  cudaStream_t so = copy_out ? copy_out : sc;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_host_mu);
  auto it = g_host_events.find({dev, ws});
  if (it == g_host_events.end()) {
    if (g_host_events.size() >= kMaxHostPipelines) {
      auto lru = g_host_events.begin();
      for (auto j = g_host_events.begin(); j != g_host_events.end(); ++j)
        if (j->second.last_use < lru->second.last_use) lru = j;
      int cur = dev;
      if (lru->first.first != dev) cudaSetDevice(lru->first.first);
      destroy_host_events(lru->second);
      if (lru->first.first != dev) cudaSetDevice(cur);
      g_host_events.erase(lru);
    }
    HostEvents h = {};
    for (int k = 0; k < 2; ++k) {
      if (cudaEventCreateWithFlags(&h.in[k], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&h.layer[k], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&h.out[k], cudaEventDisableTiming) != cudaSuccess)
        return MOE_ERR_CUDA;
    }
    it = g_host_events.emplace(std::make_pair(dev, (const void *)ws), h).first;
  }
  HostEvents &ev = it->second;
  ev.last_use = ++g_host_clock;
  // copy in once the slot's previous layer has read its x
  cudaError_t e = cudaStreamWaitEvent(si, ev.layer[slot], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, si);
  if (e == cudaSuccess) e = cudaEventRecord(ev.in[slot], si);
  // the layer, once x is in and the slot's previous y has been copied out
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, ev.in[slot], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, ev.out[slot], 0);
  if (e != cudaSuccess) return cuda_status(e);
  const void *xv[1] = {xs};
  void *yv[1] = {ys};
  st = moe_forward_microbatches(desc, 1, xv, w_gate, bias, w13, w2, yv, ws, mb_bytes(d), 0,
                                status_word, sc, nullptr);
  if (st != MOE_OK) return st;
  e = cudaEventRecord(ev.layer[slot], sc);
  // copy out once the layer is done
  if (e == cudaSuccess) e = cudaStreamWaitEvent(so, ev.layer[slot], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(y_host, ys, bytes, cudaMemcpyDeviceToHost, so);
  if (e == cudaSuccess) e = cudaEventRecord(ev.out[slot], so);
  return cuda_status(e);
}

// backward workspace: dY (nK,H) bf16 | dw (nK) f32 | dh (nK,I) bf16 | dGU (nK,2I) bf16 |
// dx_perm (nK,H) bf16 | dlogits (n,E) f32 | dW_gate partials (16,H,E) and
// dbias partials (16,E) f32 | the weight gradients' zero-padded tail rows
// (E*16 rows of both operands, bf16)
namespace {
struct BwdSlots {
  size_t off[8];
  size_t total;
};
BwdSlots bwd_slots(const Desc &d) {
  const size_t nK = (size_t)d.nK();
  const size_t sz[8] = {nK * d.H * 2, nK * 4, nK * d.I * 2, nK * 2 * d.I * 2, nK * d.H * 2,
                        (size_t)d.n * d.E * 4,
                        (size_t)kRouterBwdSplit * (d.H + 1) * d.E * 4,
                        wgrad_tail_bytes(d, d.H, 2 * d.I)};  // >= the (I, H) pair's
  BwdSlots b;
  size_t o = 0;
  for (int i = 0; i < 8; ++i) {
    b.off[i] = o;
    o += up(sz[i]);
  }
  b.total = o;
  return b;
}
}  // namespace

size_t moe_backward_workspace_size(const moe_layer_desc_t *desc) {
  Desc d;
  if (check_desc(desc, &d) != MOE_OK) return 0;
  return bwd_slots(d).total;
}

moe_status_t moe_backward(const moe_layer_desc_t *desc, const void *x, const void *w_gate,
                          const void *w13, const void *w2, const void *dy, const float *logits,
                          const int32_t *topk_idx, const float *topk_w, const int32_t *offsets,
                          const int32_t *inv_perm, const void *x_perm,
                          const void *h, const void *y_perm, void *dx, float *dw_gate,
                          float *dbias, float *dw13, float *dw2, void *ws, size_t ws_bytes,
                          int32_t *status_word, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (!d.bf16 || d.H % 256 || d.I % 128 || d.tiled) return MOE_ERR_UNSUPPORTED;
  if (d.n == 0) {  // no tokens: every gradient is zero (token arrays may be NULL)
    if (!w_gate || !w13 || !w2 || !dw_gate || !dw13 || !dw2) return MOE_ERR_INVALID_ARG;
    const size_t E = d.E, H = d.H, I = d.I;
    cudaError_t e = cudaMemsetAsync(dw_gate, 0, H * E * 4, stream);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, E * 4, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw13, 0, E * H * 2 * I * 4, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, E * I * H * 4, stream);
    return cuda_status(e);
  }
  if (!x || !w_gate || !w13 || !w2 || !dy || !logits || !topk_idx || !topk_w || !offsets ||
      !inv_perm || !x_perm || !h || !y_perm || !dx || !dw_gate || !dw13 || !dw2 || !ws)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
  const void *aligned[] = {x, w_gate, w13, w2, dy, x_perm, h, y_perm, dx, dw13, dw2};
  for (const void *p : aligned)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  const BwdSlots b = bwd_slots(d);
  if (ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  uint8_t *w = reinterpret_cast<uint8_t *>(ws);
  void *dY = w + b.off[0];
  float *dwt = reinterpret_cast<float *>(w + b.off[1]);
  void *dh = w + b.off[2];
  void *dgu = w + b.off[3];
  void *dxp = w + b.off[4];
  float *dl = reinterpret_cast<float *>(w + b.off[5]);
  float *dwp = reinterpret_cast<float *>(w + b.off[6]);
  void *tails = w + b.off[7];
  cudaStream_t s = stream;
  cudaError_t e = cudaSuccess;
  // combine backward (a dispatch): dY = w dy in expert order, dw = <dy, Y>
  e = launch_combine_bwd(d, dy, y_perm, topk_w, inv_perm, dY, dwt, status_word, s);
  // expert backward: dh = dY W2^T; dG|dU from the recomputed G|U; dX = dGU W13^T
  if (e == cudaSuccess) e = launch_gemm_dgrad_tc(d, dY, w2, d.H, d.I, offsets, dh, status_word, s);
  if (e == cudaSuccess)
    e = launch_gemm1_swiglu_bwd_tc(d, x_perm, w13, offsets, dh, dgu, status_word, s);
  if (e == cudaSuccess)
    e = launch_gemm_dgrad_tc(d, dgu, w13, 2 * d.I, d.H, offsets, dxp, status_word, s);
  // weight gradients over each expert's rows
  if (e == cudaSuccess)
    e = launch_wgrad_tc(d, h, d.I, dY, d.H, offsets, tails, dw2, status_word, s);
  if (e == cudaSuccess)
    e = launch_wgrad_tc(d, x_perm, d.H, dgu, 2 * d.I, offsets, tails, dw13, status_word, s);
  // router backward, then dx = sum of the slots' dX rows (a combine) + router term
  if (e == cudaSuccess)
    e = launch_router_bwd(d, x, logits, topk_idx, topk_w, dwt, dl, dwp, dw_gate, dbias, s);
  if (e == cudaSuccess) e = launch_dx_final(d, dxp, dl, w_gate, inv_perm, dx, s);
  return cuda_status(e);
}

moe_status_t moe_prepare_router(const moe_layer_desc_t *desc, const void *w_gate,
                                void *w_gate_t, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (!d.bf16) return MOE_ERR_UNSUPPORTED;
  if (!w_gate || !w_gate_t || (reinterpret_cast<uintptr_t>(w_gate_t) & 15))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_prepare_router(d, w_gate, w_gate_t, stream));
}

moe_status_t moe_prepare_weights(const moe_layer_desc_t *desc, const void *w13, const void *w2,
                                 void *w13_tiled, void *w2_tiled, moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (!d.bf16 || d.H % 64 || d.I % 128) return MOE_ERR_UNSUPPORTED;
  if (!w13 || !w2 || !w13_tiled || !w2_tiled) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w13) || !aligned16(w2) || !aligned16(w13_tiled) || !aligned16(w2_tiled))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_prepare_weights(d, w13, w2, w13_tiled, w2_tiled, stream));
}

moe_status_t moe_set_pipeline_wait_limit(long long cycles) {
  if (cycles < 0) return MOE_ERR_INVALID_ARG;
  g_wait_limit.store(cycles, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_gemm_pairs(int enable) {
  set_gemm_single_cta(enable == 0);
  return MOE_OK;
}

moe_status_t moe_set_gemm_tails(int mode) {
  set_gemm_tails(mode);
  return MOE_OK;
}

moe_status_t moe_check_status(const int32_t *status_word, moe_stream_t stream) {
  if (!status_word) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, status_word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (v & MOE_DEV_BAD_ROUTING) return MOE_ERR_BAD_ROUTING;
  if (v & MOE_DEV_BAD_LAYOUT) return MOE_ERR_BAD_LAYOUT;
  if (v & MOE_DEV_TIMEOUT) return MOE_ERR_TIMEOUT;
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Dispatch layout without caller-provided scratch.
//
// For callers that cannot allocate device memory at call time -- for example
// a runtime whose memory is fully pre-planned, or code running where a
// cudaMalloc would synchronise the device or is simply not permitted -- the
// layout's scratch (the per-chunk histograms) lives in a
// fixed array that belongs to the library.  The array is a device global of
// this file: every GPU that loads the library holds it (257 KiB) until
// the process exits.  It is shared by every call on a device and keeps what
// the previous call left in it; the layout kernels overwrite every entry they
// read, so nothing needs clearing.  Two calls whose work overlaps on the GPU
// (on different streams without ordering) would use the same array at the same
// time and produce wrong results: order such calls on one stream.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int kNoAllocMaxChunks = 256;  // chunks of 2048 (token, slot) pairs
constexpr size_t kNoAllocScratchInts = (size_t)kNoAllocMaxChunks * (kMaxE + 1);

static __device__ __align__(256) int32_t g_layout_scratch[kNoAllocScratchInts];

// Device address of g_layout_scratch on the current device.  It is looked up
// on every call (a host-side table lookup once the module is loaded), so it
// stays right after cudaDeviceReset, which unloads the module and may place
// the array elsewhere when it is loaded again.
cudaError_t layout_scratch_address(void **out) {
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_layout_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_dispatch_layout_noalloc(const moe_layer_desc_t *desc,
                                                    const int32_t *topk_idx, int32_t *counts,
                                                    int32_t *offsets, int32_t *perm,
                                                    int32_t *inv_perm, int32_t *status_word,
                                                    moe_stream_t stream) {
  Desc d;
  moe_status_t st = check_desc(desc, &d);
  if (st != MOE_OK) return st;
  if (!counts || !offsets || !status_word) return MOE_ERR_INVALID_ARG;
  if (d.nK() > 0 && (!topk_idx || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  if (d.nK() > (long long)MOE_NOALLOC_MAX_PAIRS ||
      layout_ws_bytes(d) > kNoAllocScratchInts * sizeof(int32_t))
    return MOE_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (layout_scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(
      launch_layout(d, topk_idx, counts, offsets, perm, inv_perm, status_word, scratch, stream));
}
