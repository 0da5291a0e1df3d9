// Backward of the MoE layer (bf16 layers): the element-wise, permutation and
// router parts.  The expert GEMMs of the backward run on the tensor cores in
// gemm_tc.cu (dgrad and SwiGLU-backward modes) and gemm_wgrad.cu (weight
// gradients).
//   "大模型系统中的通算融合" §6.2.4: in training the backward of dispatch is a
//   combine and the backward of combine is a dispatch; the DModel notes
//   ("0. goin", §2.3) list the backward of the top-k reduce and the
//   routing-score gradient beside the forward kernels.  With the expert
//   choice held fixed (as differentiating a top-k selection does):
//     combine backward  dY[inv(t,k)] = w[t,k] dy[t],  dw[t,k] = <dy[t], Y[inv(t,k)]>
//     permute backward  dx[t] = sum_k dx_perm[inv(t,k)]  (+ the router's term)
//     router backward   dp from dw (through the renormalisation), dlogits =
//                       p (dp - <p, dp>), dx += dlogits W_gate^T,
//                       dW_gate = x^T dlogits, dbias = sum_t dlogits[t]
// Every sum has a fixed order: results are bitwise reproducible.
#include "common.cuh"

namespace moe {
namespace {

constexpr int BT = 256;  // threads per block
constexpr int RB_SPLIT = kRouterBwdSplit;

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float (&f)[8]) {
  const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint4 o;
  __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return o;
}

__device__ __forceinline__ float warp_sum(float v) {  // fixed butterfly order
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per token: dy[t] is streamed once in 16-byte vectors; for each of
// the K slots the Y row is read, <dy, Y> accumulated per lane in float32, and
// dY = w dy written (bf16).  The K dot products are added over the lanes by a
// fixed butterfly.
template <int KM>
__global__ void __launch_bounds__(BT) combine_bwd_kernel(const uint4 *__restrict__ dy,
                                                         const uint4 *__restrict__ y_perm,
                                                         const float *__restrict__ topk_w,
                                                         const int32_t *__restrict__ inv,
                                                         uint4 *__restrict__ dY,
                                                         float *__restrict__ dw, int n, int K,
                                                         int V, long long nK, int32_t *status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long wid = ((long long)blockIdx.x * BT + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * BT) >> 5;
  for (long long t = wid; t < n; t += nw) {
    int rows[KM];
    float ws[KM], dot[KM];
    bool ok = true;
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      dot[k] = 0.f;
      rows[k] = 0;
      ws[k] = 0.f;
      if (k < K) {
        rows[k] = __ldg(inv + t * K + k);
        ws[k] = __ldg(topk_w + t * K + k);
        if (rows[k] < 0 || (long long)rows[k] >= nK) {
          ok = false;
          rows[k] = -1;
        }
      }
    }
    if (!ok && lane == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
    for (int v = lane; v < V; v += 32) {
      float g[8];
      bf16x8_to_f32(__ldg(dy + t * V + v), g);
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (k >= K || rows[k] < 0) continue;
        float yv[8];
        bf16x8_to_f32(__ldg(y_perm + (size_t)rows[k] * V + v), yv);
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dot[k] = fmaf(g[i], yv[i], dot[k]);
          o[i] = ws[k] * g[i];
        }
        dY[(size_t)rows[k] * V + v] = f32_to_bf16x8(o);
      }
    }
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k >= K) continue;
      const float s = warp_sum(dot[k]);
      if (lane == 0) dw[t * K + k] = s;
    }
  }
}

// One warp per token: softmax of the float32 logits, dp over the selected
// experts (through the renormalisation when norm), dlogits = p (dp - <p, dp>).
__global__ void __launch_bounds__(BT) router_bwd_kernel(const float *__restrict__ logits,
                                                        const int32_t *__restrict__ topk_idx,
                                                        const float *__restrict__ topk_w,
                                                        const float *__restrict__ dw,
                                                        float *__restrict__ dlogits, int n, int E,
                                                        int K, int norm) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long wid = ((long long)blockIdx.x * BT + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * BT) >> 5;
  for (long long t = wid; t < n; t += nw) {
    const float *lr = logits + t * E;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, lr[e]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float ssum = 0.f;
    for (int e = lane; e < E; e += 32) ssum += expf(lr[e] - m);
    ssum = warp_sum(ssum);
    // lanes < K hold slot k: its expert, probability, weight and dw
    int ek = -1;
    float pk = 0.f, wk = 0.f, dwk = 0.f;
    if (lane < K) {
      ek = topk_idx[t * K + lane];
      wk = topk_w[t * K + lane];
      dwk = dw[t * K + lane];
      pk = (ek >= 0 && ek < E) ? expf(lr[ek] - m) / ssum : 0.f;
    }
    float dpk = dwk;
    if (norm) {
      const float psel = warp_sum(pk);
      const float dww = warp_sum(dwk * wk);
      dpk = (dwk - dww) / psel;
    }
    const float pdp = warp_sum(pk * dpk);  // <p, dp> (dp is zero off the selection)
    for (int e = lane; e < E; e += 32) {
      const float p = expf(lr[e] - m) / ssum;
      float dpe = 0.f;
      for (int k = 0; k < K; ++k) {
        const int ekk = __shfl_sync(0xffffffffu, ek, k);
        const float dpkk = __shfl_sync(0xffffffffu, dpk, k);
        if (ekk == e) dpe = dpkk;
      }
      dlogits[t * E + e] = p * (dpe - pdp);
    }
  }
}

// C[m][n] = sum over k in [k0, k1) of A(m,k) B(k,n), float32 accumulate in
// ascending k, 32x32 output tiles, 256 threads (2x2 outputs each).
// A(m,k) = a[m*sam + k*sak], B(k,n) = b[k*sbk + n*sbn].  AK / BK: the
// operand's k stride is 1 (its tile is loaded with consecutive threads along
// k, else along m / n), so either layout is read in whole sectors.
// blockIdx.z selects the k range [z*kc, min(Kd, (z+1)*kc)) and the output
// c + z*M*N (split-K partials, added later in order).
template <typename TA, typename TB, bool AK, bool BK>
__global__ void __launch_bounds__(BT) small_gemm_kernel(const TA *__restrict__ a, long long sam,
                                                        long long sak, const TB *__restrict__ b,
                                                        long long sbk, long long sbn,
                                                        float *__restrict__ c, int M, int N,
                                                        int Kd, int kc) {
  pdl_enter();
  __shared__ float As[32][32 + 1];
  __shared__ float Bs[32][32 + 1];
  const int m0 = blockIdx.x * 32, n0 = blockIdx.y * 32;
  const int kb = blockIdx.z * kc, ke = min(Kd, kb + kc);
  c += (size_t)blockIdx.z * M * N;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[2][2] = {};
  for (int k0 = kb; k0 < ke; k0 += 32) {
    for (int i = threadIdx.x; i < 32 * 32; i += BT) {
      const int kk = AK ? i % 32 : i / 32, mm = AK ? i / 32 : i % 32;
      const int gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < ke) ? (float)a[(long long)gm * sam + (long long)gk * sak] : 0.f;
    }
    for (int i = threadIdx.x; i < 32 * 32; i += BT) {
      const int kk = BK ? i % 32 : i / 32, nn = BK ? i / 32 : i % 32;
      const int gn = n0 + nn, gk = k0 + kk;
      Bs[kk][nn] = (gn < N && gk < ke) ? (float)b[(long long)gk * sbk + (long long)gn * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
          acc[i][j] = fmaf(As[kk][ty * 2 + i], Bs[kk][tx * 2 + j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int gm = m0 + ty * 2 + i, gn = n0 + tx * 2 + j;
      if (gm < M && gn < N) c[(long long)gm * N + gn] = acc[i][j];
    }
}

// out[i] = sum over z = 0..S-1 of part[z][i] (ascending z)
__global__ void __launch_bounds__(BT) sum_parts_kernel(const float *__restrict__ part,
                                                       float *__restrict__ out, long long count,
                                                       int S) {
  pdl_enter();
  for (long long i = (long long)blockIdx.x * BT + threadIdx.x; i < count;
       i += (long long)gridDim.x * BT) {
    float s = 0.f;
    for (int z = 0; z < S; ++z) s += part[(size_t)z * count + i];
    out[i] = s;
  }
}

// partial column sums of dlogits: block (x, z) adds tokens [z*tc, (z+1)*tc)
// of experts [32x, 32x + 32) in 8 token groups (coalesced over experts), the
// group sums in order, into part[z][e]
__global__ void __launch_bounds__(BT) column_sum_kernel(const float *__restrict__ dl,
                                                        float *__restrict__ part, int n, int E,
                                                        int tc) {
  pdl_enter();
  __shared__ float grp[8][32];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + tx;
  const int t0 = blockIdx.z * tc, t1 = min(n, t0 + tc);
  float s = 0.f;
  if (e < E) {
#pragma unroll 4
    for (int t = t0 + ty; t < t1; t += 8) s += dl[(long long)t * E + e];
  }
  grp[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && e < E) {
    float r = 0.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) r += grp[g][tx];
    part[(size_t)blockIdx.z * E + e] = r;
  }
}

// dx[t] = sum_k dx_perm[inv(t,k)] (slot order) + dx_router[t], float32, one rounding
template <int KM>
__global__ void __launch_bounds__(BT) dx_gather_kernel(const uint4 *__restrict__ dxp,
                                                       const float4 *__restrict__ dxr,
                                                       const int32_t *__restrict__ inv,
                                                       uint4 *__restrict__ dx, int n, int K,
                                                       int V, long long nK) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long wid = ((long long)blockIdx.x * BT + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * BT) >> 5;
  for (long long t = wid; t < n; t += nw) {
    int rows[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      rows[k] = -1;
      if (k < K) {
        const int r = __ldg(inv + t * K + k);
        rows[k] = (r >= 0 && (long long)r < nK) ? r : -1;
      }
    }
    for (int v = lane; v < V; v += 32) {
      float acc[8];
      const float4 r0 = dxr[(t * V + v) * 2], r1 = dxr[(t * V + v) * 2 + 1];
      acc[0] = r0.x; acc[1] = r0.y; acc[2] = r0.z; acc[3] = r0.w;
      acc[4] = r1.x; acc[5] = r1.y; acc[6] = r1.z; acc[7] = r1.w;
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (k >= K || rows[k] < 0) continue;
        float f[8];
        bf16x8_to_f32(__ldg(dxp + (size_t)rows[k] * V + v), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += f[i];
      }
      dx[t * V + v] = f32_to_bf16x8(acc);
    }
  }
}

inline int grid_warps(long long items) {
  const long long want = (items + (BT / 32) - 1) / (BT / 32);
  const long long cap = (long long)device_sm_count() * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

template <int KM>
cudaError_t combine_bwd_k(const Desc &d, const void *dy, const void *y_perm, const float *topk_w,
                          const int32_t *inv, void *dY, float *dw, int32_t *status,
                          cudaStream_t s) {
  const int V = d.H * 2 / 16;
  return launch_pdl(combine_bwd_kernel<KM>, dim3(grid_warps(d.n)), dim3(BT), 0, s,
                    reinterpret_cast<const uint4 *>(dy), reinterpret_cast<const uint4 *>(y_perm),
                    topk_w, inv, reinterpret_cast<uint4 *>(dY), dw, d.n, d.K, V, d.nK(), status);
}

template <int KM>
cudaError_t dx_gather_k(const Desc &d, const void *dx_perm, const float *dx_router,
                        const int32_t *inv, void *dx, cudaStream_t s) {
  const int V = d.H * 2 / 16;
  return launch_pdl(dx_gather_kernel<KM>, dim3(grid_warps(d.n)), dim3(BT), 0, s,
                    reinterpret_cast<const uint4 *>(dx_perm),
                    reinterpret_cast<const float4 *>(dx_router), inv,
                    reinterpret_cast<uint4 *>(dx), d.n, d.K, V, d.nK());
}

}  // namespace

cudaError_t launch_combine_bwd(const Desc &d, const void *dy, const void *y_perm,
                               const float *topk_w, const int32_t *inv_perm, void *dY, float *dw,
                               int32_t *status, cudaStream_t s) {
  if (d.n == 0) return cudaSuccess;
  if (d.K <= 2) return combine_bwd_k<2>(d, dy, y_perm, topk_w, inv_perm, dY, dw, status, s);
  if (d.K <= 4) return combine_bwd_k<4>(d, dy, y_perm, topk_w, inv_perm, dY, dw, status, s);
  if (d.K <= 8) return combine_bwd_k<8>(d, dy, y_perm, topk_w, inv_perm, dY, dw, status, s);
  return combine_bwd_k<kMaxK>(d, dy, y_perm, topk_w, inv_perm, dY, dw, status, s);
}

cudaError_t launch_router_bwd(const Desc &d, const void *x, const void *w_gate,
                              const float *logits, const int32_t *topk_idx, const float *topk_w,
                              const float *dw, float *dlogits, float *dx_router,
                              float *dw_part, float *dw_gate, float *dbias, cudaStream_t s) {
  if (d.n == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(router_bwd_kernel, dim3(grid_warps(d.n)), dim3(BT), 0, s, logits,
                             topk_idx, topk_w, dw, dlogits, d.n, d.E, d.K, d.norm ? 1 : 0);
  if (e != cudaSuccess) return e;
  const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(x);
  const __nv_bfloat16 *wg = reinterpret_cast<const __nv_bfloat16 *>(w_gate);
  // dx_router[t][h] = sum_e dlogits[t][e] W_gate[h][e]   (both k-contiguous)
  e = launch_pdl(small_gemm_kernel<float, __nv_bfloat16, true, true>,
                 dim3((d.n + 31) / 32, (d.H + 31) / 32, 1), dim3(BT), 0, s,
                 (const float *)dlogits, (long long)d.E, 1ll, wg, 1ll, (long long)d.E, dx_router,
                 d.n, d.H, d.E, d.E);
  if (e != cudaSuccess) return e;
  // dW_gate[h][e] = sum_t x[t][h] dlogits[t][e]: the tokens split into
  // RB_SPLIT ranges (partials in dw_part), then added in order
  const int kc = (d.n + RB_SPLIT - 1) / RB_SPLIT;
  e = launch_pdl(small_gemm_kernel<__nv_bfloat16, float, false, false>,
                 dim3((d.H + 31) / 32, (d.E + 31) / 32, RB_SPLIT), dim3(BT), 0, s, xb, 1ll,
                 (long long)d.H, (const float *)dlogits, (long long)d.E, 1ll, dw_part, d.H, d.E,
                 d.n, kc);
  if (e != cudaSuccess) return e;
  const long long cnt = (long long)d.H * d.E;
  e = launch_pdl(sum_parts_kernel, dim3((int)((cnt + BT - 1) / BT)), dim3(BT), 0, s,
                 (const float *)dw_part, dw_gate, cnt, RB_SPLIT);
  if (e != cudaSuccess || !dbias) return e;
  // dbias: the same token ranges, partials after the dW_gate partials
  float *bpart = dw_part + (size_t)RB_SPLIT * d.H * d.E;
  e = launch_pdl(column_sum_kernel, dim3((d.E + 31) / 32, 1, RB_SPLIT), dim3(BT), 0, s,
                 (const float *)dlogits, bpart, d.n, d.E, kc);
  if (e != cudaSuccess) return e;
  return launch_pdl(sum_parts_kernel, dim3((d.E + BT - 1) / BT), dim3(BT), 0, s,
                    (const float *)bpart, dbias, (long long)d.E, RB_SPLIT);
}

cudaError_t launch_dx_gather(const Desc &d, const void *dx_perm, const float *dx_router,
                             const int32_t *inv_perm, void *dx, cudaStream_t s) {
  if (d.n == 0) return cudaSuccess;
  if (d.K <= 2) return dx_gather_k<2>(d, dx_perm, dx_router, inv_perm, dx, s);
  if (d.K <= 4) return dx_gather_k<4>(d, dx_perm, dx_router, inv_perm, dx, s);
  if (d.K <= 8) return dx_gather_k<8>(d, dx_perm, dx_router, inv_perm, dx, s);
  return dx_gather_k<kMaxK>(d, dx_perm, dx_router, inv_perm, dx, s);
}

}  // namespace moe
