// Permute (row gather into expert order) and combine (weighted per-token
// gather-reduce of the K expert rows).
//   permute: "MoE 分布式推理基础（基于 vLLM）" §1.2, Algorithm 2 step 7
//            (X_e = x[token ids of I_e]) done for all experts in one pass.
//   combine: the same section, steps 10-11 (y[i] += Y_e[idx(i)] * w_top[i,k]),
//            evaluated as a gather per token in slot order with float32
//            accumulation, as the top-k slot reduction of the MinimalAsyncEP
//            kernels listed in the DModel notes ("0. goin", §2.3) does.
// Both kernels are HBM-bound streams of 16-byte vectors: one warp per row,
// each lane moving whole 16-byte vectors, with every load of a row issued
// before its stores/accumulation so that many requests are in flight.
#include "common.cuh"

namespace moe {
namespace {

constexpr int PT = 256;   // threads per block
constexpr int PU = 8;     // 16-byte vectors in flight per lane

// Permute: warp w copies the contiguous row range [w*nK/W, (w+1)*nK/W) of
// x_perm (its writes are one contiguous block), two rows per step with every
// load of both rows issued before their stores.  The x_perm stores carry the
// streaming (evict-first) cache hint, so the written rows do not push x,
// which is re-read K times, out of L2 (measured: 30.5 -> 27.3 us at the
// OLMoE shape, 134.6 -> 126.9 us for the skewed layer).
// GUEST: the instantiation launched beside the grouped GEMM (its own kernel,
// so that its shared-memory carveout preference does not touch the other).
template <bool GUEST>
__global__ void __launch_bounds__(PT) permute_kernel(const uint4 *__restrict__ x,
                                                     const int32_t *__restrict__ perm,
                                                     uint4 *__restrict__ xp, long long nK, int K,
                                                     int V, int32_t *status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long W = ((long long)gridDim.x * PT) >> 5;
  const long long wid = ((long long)blockIdx.x * PT + threadIdx.x) >> 5;
  const long long r0 = wid * nK / W, r1 = (wid + 1) * nK / W;
  for (long long r = r0; r < r1; r += 2) {
    const bool two = r + 1 < r1;
    int f[2] = {__ldg(perm + r), two ? __ldg(perm + r + 1) : 0};
    bool ok[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      ok[q] = (q == 0 || two) && f[q] >= 0 && (long long)f[q] < nK;
      if ((q == 0 || two) && !ok[q] && lane == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
    }
    for (int v0 = 0; v0 < V; v0 += 32 * PU) {
      uint4 buf[2][PU];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 *src = x + (size_t)(ok[q] ? f[q] / K : 0) * V;
#pragma unroll
        for (int u = 0; u < PU; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < V) buf[q][u] = ok[q] ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (q == 1 && !two) break;
        uint4 *dst = xp + (size_t)(r + q) * V;
#pragma unroll
        for (int u = 0; u < PU; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < V) __stcs(dst + v, buf[q][u]);  // streaming: x stays in L2
        }
      }
    }
  }
}

// Scatter permute: warp w copies the tokens [w*n/W, (w+1)*n/W); for each
// token the K destination rows come from inv_perm (lane k holds slot k's),
// PU 16-byte vectors per lane are loaded once and stored to all K rows
// (streaming stores, as the gather form).
template <bool GUEST>
__global__ void __launch_bounds__(PT) permute_scatter_kernel(const uint4 *__restrict__ x,
                                                             const int32_t *__restrict__ inv,
                                                             uint4 *__restrict__ xp, int n,
                                                             int K, int V, long long nK,
                                                             int32_t *status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long W = ((long long)gridDim.x * PT) >> 5;
  const long long wid = ((long long)blockIdx.x * PT + threadIdx.x) >> 5;
  const long long t0 = wid * n / W, t1 = (wid + 1) * n / W;
  bool bad = false;
  for (long long t = t0; t < t1; ++t) {
    int dst = 0;
    bool ok = true;
    if (lane < K) {
      dst = __ldg(inv + t * K + lane);
      ok = dst >= 0 && (long long)dst < nK;
      bad |= !ok;
    }
    const unsigned okm = __ballot_sync(0xffffffffu, ok);
    const uint4 *src = x + (size_t)t * V;
    for (int v0 = 0; v0 < V; v0 += 32 * PU) {
      uint4 buf[PU];
#pragma unroll
      for (int u = 0; u < PU; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < V) buf[u] = __ldcs(src + v);  // read once: no need to keep it in L2
      }
      for (int k = 0; k < K; ++k) {
        const int r = __shfl_sync(0xffffffffu, dst, k);
        if (!(okm >> k & 1u)) continue;  // warp-uniform
        uint4 *d = xp + (size_t)r * V;
#pragma unroll
        for (int u = 0; u < PU; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < V) __stcs(d + v, buf[u]);
        }
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
}

__device__ __forceinline__ void acc_vec(float (&a)[8], uint4 v, float w, bool bf16) {
  if (bf16) {
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p[i]);
      a[2 * i] = fmaf(w, f.x, a[2 * i]);
      a[2 * i + 1] = fmaf(w, f.y, a[2 * i + 1]);
    }
  } else {
    const float *p = reinterpret_cast<const float *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = fmaf(w, p[i], a[i]);
  }
}

// Combine work item: one token's 64-vector chunk of a row (two 16-byte vectors
// per lane).  Warp w takes the contiguous item range [w*T/W, (w+1)*T/W), so
// the warps' loads differ by at most one item, and all K rows' vectors of an
// item are loaded before they are accumulated.
constexpr int CV = 64;  // vectors per combine item

// SLOTS: the rows of token t are t*K .. t*K+K-1 of an already weighted,
// slot-ordered array (GEMM2's weighted epilogue), added with weight 1.
template <bool BF16, int KM, bool SLOTS, bool GUEST>
__global__ void __launch_bounds__(PT) combine_kernel(const uint4 *__restrict__ yp,
                                                     const float *__restrict__ tw,
                                                     const int32_t *__restrict__ inv,
                                                     uint4 *__restrict__ y, int n, int K, int V,
                                                     long long nK, int32_t *status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int nseg = (V + CV - 1) / CV;
  const long long T = (long long)n * nseg;
  const long long W = ((long long)gridDim.x * PT) >> 5;
  const long long wid = ((long long)blockIdx.x * PT + threadIdx.x) >> 5;
  const long long i0 = wid * T / W, i1 = (wid + 1) * T / W;
  int cur = -1;
  int rows[KM];
  float ws[KM];
  unsigned okmask = 0u;
  for (long long i = i0; i < i1; ++i) {
    const int t = (int)(i / nseg);
    const int v0 = (int)(i - (long long)t * nseg) * CV + lane;
    if (t != cur) {  // the token's K rows and weights
      cur = t;
      int my_row = 0;
      float my_w = 0.f;
      bool my_ok = true;
      if (lane < K) {
        if (SLOTS) {
          my_row = t * K + lane;
          my_w = 1.f;
        } else {
          my_row = __ldg(inv + (size_t)t * K + lane);
          my_w = __ldg(tw + (size_t)t * K + lane);
          my_ok = my_row >= 0 && (long long)my_row < nK;
        }
      }
      okmask = __ballot_sync(0xffffffffu, my_ok);
      if (okmask != 0xffffffffu && lane == 0 && v0 == lane) flag_status(status, MOE_DEV_BAD_LAYOUT);
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        rows[k] = __shfl_sync(0xffffffffu, my_row, k);
        ws[k] = __shfl_sync(0xffffffffu, my_w, k);
      }
    }
    const bool in0 = v0 < V, in1 = v0 + 32 < V;
    uint4 b0[KM], b1[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k < K && (okmask >> k & 1u)) {
        const uint4 *r = yp + (size_t)rows[k] * V;
        if (in0) b0[k] = __ldg(r + v0);
        if (in1) b1[k] = __ldg(r + v0 + 32);
      }
    }
    uint4 *dst = y + (size_t)t * V;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!(h ? in1 : in0)) continue;
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < KM; ++k)
        if (k < K && (okmask >> k & 1u)) acc_vec(a, h ? b1[k] : b0[k], ws[k], BF16);
      uint4 o;
      if (BF16) {
        __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) p[q] = __floats2bfloat162_rn(a[2 * q], a[2 * q + 1]);
      } else {
        float *p = reinterpret_cast<float *>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) p[q] = a[q];
      }
      dst[v0 + 32 * h] = o;
    }
  }
}

// Blocks of the kernel that fit on the device at once (all CTAs in one wave);
// for the guest instantiation, one per SM, and the first call on a device sets
// its shared-memory carveout preference (see prefer_max_shared).
template <auto Kernel, bool GUEST>
int resident_grid() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int &c = cache[dev >= 0 && dev < 64 ? dev : 0];
  if (c == 0) {
    int per_sm = 0;
    if (GUEST) prefer_max_shared(Kernel);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, Kernel, PT, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    c = GUEST ? device_sm_count() : per_sm * device_sm_count();
  }
  return c;
}

template <bool BF16, int KM, bool SLOTS, bool GUEST>
cudaError_t combine_g(const Desc &d, const void *y_perm, const float *topk_w,
                      const int32_t *inv_perm, void *y, int32_t *status, cudaStream_t s) {
  const int V = (int)((size_t)d.H * elem_bytes(d) / 16);
  const long long items = (long long)d.n * ((V + CV - 1) / CV);
  const long long res = resident_grid<combine_kernel<BF16, KM, SLOTS, GUEST>, GUEST>();
  const long long want = (items + (PT / 32) - 1) / (PT / 32);
  const int grid = (int)(want < res ? want : res);
  return launch_k(GUEST, combine_kernel<BF16, KM, SLOTS, GUEST>, dim3(grid), dim3(PT), 0, s,
                  reinterpret_cast<const uint4 *>(y_perm), topk_w, inv_perm,
                  reinterpret_cast<uint4 *>(y), d.n, d.K, V, d.nK(), status);
}

template <bool BF16, int KM, bool SLOTS = false>
cudaError_t combine_k(const Desc &d, const void *y_perm, const float *topk_w,
                      const int32_t *inv_perm, void *y, int32_t *status, cudaStream_t s,
                      bool guest) {
  return guest ? combine_g<BF16, KM, SLOTS, true>(d, y_perm, topk_w, inv_perm, y, status, s)
               : combine_g<BF16, KM, SLOTS, false>(d, y_perm, topk_w, inv_perm, y, status, s);
}

template <bool BF16, bool SLOTS = false>
cudaError_t combine_dispatch_k(const Desc &d, const void *y_perm, const float *topk_w,
                               const int32_t *inv_perm, void *y, int32_t *status,
                               cudaStream_t s, bool guest) {
  if (d.K <= 2) return combine_k<BF16, 2, SLOTS>(d, y_perm, topk_w, inv_perm, y, status, s, guest);
  if (d.K <= 4) return combine_k<BF16, 4, SLOTS>(d, y_perm, topk_w, inv_perm, y, status, s, guest);
  if (d.K <= 8) return combine_k<BF16, 8, SLOTS>(d, y_perm, topk_w, inv_perm, y, status, s, guest);
  return combine_k<BF16, kMaxK, SLOTS>(d, y_perm, topk_w, inv_perm, y, status, s, guest);
}

}  // namespace

cudaError_t launch_permute(const Desc &d, const void *x, const int32_t *perm, void *x_perm,
                           int32_t *status, cudaStream_t s, bool guest) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  const int V = (int)((size_t)d.H * elem_bytes(d) / 16);
  const long long res =
      guest ? resident_grid<permute_kernel<true>, true>() : resident_grid<permute_kernel<false>, false>();
  const long long want = (nK + (PT / 32) - 1) / (PT / 32);
  return launch_k(guest, guest ? permute_kernel<true> : permute_kernel<false>,
                  dim3((int)(want < res ? want : res)), dim3(PT), 0, s,
                  reinterpret_cast<const uint4 *>(x), perm, reinterpret_cast<uint4 *>(x_perm), nK,
                  d.K, V, status);
}

cudaError_t launch_permute_scatter(const Desc &d, const void *x, const int32_t *inv_perm,
                                   void *x_perm, int32_t *status, cudaStream_t s, bool guest) {
  if (d.nK() == 0) return cudaSuccess;
  const int V = (int)((size_t)d.H * elem_bytes(d) / 16);
  const long long res = guest ? resident_grid<permute_scatter_kernel<true>, true>()
                              : resident_grid<permute_scatter_kernel<false>, false>();
  const long long want = ((long long)d.n + (PT / 32) - 1) / (PT / 32);
  return launch_k(guest, guest ? permute_scatter_kernel<true> : permute_scatter_kernel<false>,
                  dim3((int)(want < res ? want : res)), dim3(PT), 0, s,
                  reinterpret_cast<const uint4 *>(x), inv_perm, reinterpret_cast<uint4 *>(x_perm),
                  d.n, d.K, V, d.nK(), status);
}

cudaError_t launch_combine_slots(const Desc &d, const void *y_slot, void *y, cudaStream_t s,
                                 bool guest) {
  if (d.n == 0) return cudaSuccess;
  if (d.bf16)
    return combine_dispatch_k<true, true>(d, y_slot, nullptr, nullptr, y, nullptr, s, guest);
  return combine_dispatch_k<false, true>(d, y_slot, nullptr, nullptr, y, nullptr, s, guest);
}

cudaError_t launch_combine(const Desc &d, const void *y_perm, const float *topk_w,
                           const int32_t *inv_perm, void *y, int32_t *status, cudaStream_t s,
                           bool guest) {
  if (d.n == 0) return cudaSuccess;
  if (d.bf16) return combine_dispatch_k<true>(d, y_perm, topk_w, inv_perm, y, status, s, guest);
  return combine_dispatch_k<false>(d, y_perm, topk_w, inv_perm, y, status, s, guest);
}

}  // namespace moe
