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

__global__ void __launch_bounds__(PT) permute_kernel(const uint4 *__restrict__ x,
                                                     const int32_t *__restrict__ perm,
                                                     uint4 *__restrict__ xp, long long nK, int K,
                                                     int V, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const long long w0 = ((long long)blockIdx.x * PT + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * PT) >> 5;
  for (long long r = w0; r < nK; r += nw) {
    const int f = __ldg(perm + r);
    uint4 *dst = xp + (size_t)r * V;
    if ((unsigned long long)(unsigned)f >= (unsigned long long)nK || f < 0) {
      if (lane == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
      for (int v = lane; v < V; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4 *src = x + (size_t)(f / K) * V;
    for (int v0 = 0; v0 < V; v0 += 32 * PU) {
      uint4 buf[PU];
#pragma unroll
      for (int u = 0; u < PU; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < V) buf[u] = __ldg(src + v);
      }
#pragma unroll
      for (int u = 0; u < PU; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < V) dst[v] = buf[u];
      }
    }
  }
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

template <bool BF16, int KM>
__global__ void __launch_bounds__(PT) combine_kernel(const uint4 *__restrict__ yp,
                                                     const float *__restrict__ tw,
                                                     const int32_t *__restrict__ inv,
                                                     uint4 *__restrict__ y, int n, int K, int V,
                                                     long long nK, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const long long w0 = ((long long)blockIdx.x * PT + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * PT) >> 5;
  for (long long t = w0; t < n; t += nw) {
    int my_row = 0;
    float my_w = 0.f;
    bool my_ok = true;
    if (lane < K) {
      my_row = __ldg(inv + t * K + lane);
      my_w = __ldg(tw + t * K + lane);
      my_ok = my_row >= 0 && (long long)my_row < nK;
    }
    const unsigned okmask = __ballot_sync(0xffffffffu, my_ok);
    if (okmask != 0xffffffffu && lane == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
    int rows[KM];
    float ws[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      rows[k] = __shfl_sync(0xffffffffu, my_row, k);
      ws[k] = __shfl_sync(0xffffffffu, my_w, k);
    }
    uint4 *dst = y + (size_t)t * V;
    for (int v = lane; v < V; v += 32) {
      uint4 buf[KM];
#pragma unroll
      for (int k = 0; k < KM; ++k)
        if (k < K && (okmask >> k & 1u)) buf[k] = __ldg(yp + (size_t)rows[k] * V + v);
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < KM; ++k)
        if (k < K && (okmask >> k & 1u)) acc_vec(a, buf[k], ws[k], BF16);
      uint4 o;
      if (BF16) {
        __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
      } else {
        float *p = reinterpret_cast<float *>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = a[i];
      }
      dst[v] = o;
    }
  }
}

inline int grid_for_rows(long long rows) {
  const long long want = (rows + (PT / 32) - 1) / (PT / 32);
  const long long cap = (long long)device_sm_count() * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

template <bool BF16, int KM>
cudaError_t combine_k(const Desc &d, const void *y_perm, const float *topk_w,
                      const int32_t *inv_perm, void *y, int32_t *status, cudaStream_t s) {
  const int V = (int)((size_t)d.H * elem_bytes(d) / 16);
  combine_kernel<BF16, KM><<<grid_for_rows(d.n), PT, 0, s>>>(
      reinterpret_cast<const uint4 *>(y_perm), topk_w, inv_perm, reinterpret_cast<uint4 *>(y),
      d.n, d.K, V, d.nK(), status);
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t combine_dispatch_k(const Desc &d, const void *y_perm, const float *topk_w,
                               const int32_t *inv_perm, void *y, int32_t *status,
                               cudaStream_t s) {
  if (d.K <= 2) return combine_k<BF16, 2>(d, y_perm, topk_w, inv_perm, y, status, s);
  if (d.K <= 4) return combine_k<BF16, 4>(d, y_perm, topk_w, inv_perm, y, status, s);
  if (d.K <= 8) return combine_k<BF16, 8>(d, y_perm, topk_w, inv_perm, y, status, s);
  return combine_k<BF16, kMaxK>(d, y_perm, topk_w, inv_perm, y, status, s);
}

}  // namespace

cudaError_t launch_permute(const Desc &d, const void *x, const int32_t *perm, void *x_perm,
                           int32_t *status, cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  const int V = (int)((size_t)d.H * elem_bytes(d) / 16);
  permute_kernel<<<grid_for_rows(nK), PT, 0, s>>>(reinterpret_cast<const uint4 *>(x), perm,
                                                  reinterpret_cast<uint4 *>(x_perm), nK, d.K, V,
                                                  status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Desc &d, const void *y_perm, const float *topk_w,
                           const int32_t *inv_perm, void *y, int32_t *status, cudaStream_t s) {
  if (d.n == 0) return cudaSuccess;
  if (d.bf16) return combine_dispatch_k<true>(d, y_perm, topk_w, inv_perm, y, status, s);
  return combine_dispatch_k<false>(d, y_perm, topk_w, inv_perm, y, status, s);
}

}  // namespace moe
