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
//                       p (dp - <p, dp>), dx += dlogits W_gate^T (fused with the
//                       permute backward), dW_gate = x^T dlogits,
//                       dbias = sum_t dlogits[t]
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
// dY = w dy written (bf16).  All K row pieces of a vector are loaded before
// any dY piece is stored, so the loads overlap.  The K dot products are added
// over the lanes by a fixed butterfly.
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
      uint4 yr[KM];
#pragma unroll
      for (int k = 0; k < KM; ++k)
        yr[k] = (k < K && rows[k] >= 0) ? __ldg(y_perm + (size_t)rows[k] * V + v)
                                        : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (k >= K || rows[k] < 0) continue;
        float yv[8];
        bf16x8_to_f32(yr[k], yv);
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

// Partial dW_gate over one token range: part[z][h][e] = sum over t in
// [z*tc, min(n, (z+1)*tc)) of x[t][h] dlogits[t][e], ascending t, float32.
// A block computes 128 h x 64 e (each thread 8 h x 4 e: three 16-byte
// shared-memory loads per 32 FMAs); the tokens pass through shared memory 32
// at a time (x rows as 16-byte bf16 pieces, dlogits rows coalesced over e),
// the next chunk's global loads in flight while the current one is used.
constexpr int GW_T = 32, GW_H = 128, GW_E = 64;
__global__ void __launch_bounds__(BT) dw_gate_kernel(const __nv_bfloat16 *__restrict__ x,
                                                     const float *__restrict__ dl,
                                                     float *__restrict__ part, int n, int H,
                                                     int E, int tc) {
  pdl_enter();
  __shared__ __align__(16) float xs[GW_T][GW_H];
  __shared__ __align__(16) float ds[GW_T][GW_E];
  const int h0 = blockIdx.x * GW_H, e0 = blockIdx.y * GW_E;
  const int t0 = blockIdx.z * tc, t1 = min(n, t0 + tc);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[8][4] = {};
  // this thread's share of a chunk: 2 of the 512 16-byte pieces of x (32
  // tokens x 128 h) and 8 of the 2048 dlogits values (32 tokens x 64 e)
  constexpr int XP = GW_T * GW_H / 8 / BT, DP = GW_T * GW_E / BT;
  uint4 xv_next[XP];
  float dv_next[DP];
  auto fetch = [&](int tb) {
#pragma unroll
    for (int q = 0; q < XP; ++q) {
      const int i = tid + q * BT, r = i >> 4, c = i & 15;
      xv_next[q] = tb + r < t1 ? __ldg(reinterpret_cast<const uint4 *>(
                                     x + (size_t)(tb + r) * H + h0 + c * 8))
                               : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < DP; ++q) {
      const int i = tid + q * BT, r = i >> 6, c = i & 63;
      dv_next[q] = (tb + r < t1 && e0 + c < E) ? __ldg(dl + (size_t)(tb + r) * E + e0 + c) : 0.f;
    }
  };
  if (t0 < t1) fetch(t0);
  for (int tb = t0; tb < t1; tb += GW_T) {
#pragma unroll
    for (int q = 0; q < XP; ++q) {
      const int i = tid + q * BT, r = i >> 4, c = i & 15;
      float f[8];
      bf16x8_to_f32(xv_next[q], f);
      *reinterpret_cast<float4 *>(&xs[r][c * 8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4 *>(&xs[r][c * 8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    }
#pragma unroll
    for (int q = 0; q < DP; ++q) {
      const int i = tid + q * BT;
      ds[i >> 6][i & 63] = dv_next[q];
    }
    __syncthreads();
    if (tb + GW_T < t1) fetch(tb + GW_T);  // in flight while this chunk is used
#pragma unroll 4
    for (int tt = 0; tt < GW_T; ++tt) {
      const float4 x0 = *reinterpret_cast<const float4 *>(&xs[tt][ty * 8]);
      const float4 x1 = *reinterpret_cast<const float4 *>(&xs[tt][ty * 8 + 4]);
      const float4 dv = *reinterpret_cast<const float4 *>(&ds[tt][tx * 4]);
      const float xa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const float da[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], da[j], acc[i][j]);
    }
    __syncthreads();
  }
  float *out = part + (size_t)blockIdx.z * H * E;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) out[(size_t)(h0 + ty * 8 + i) * E + e] = acc[i][j];
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

// dx[t][h] = sum_e dlogits[t][e] W_gate[h][e] (ascending e) + sum_k
// dx_perm[inv(t,k)][h] (slot order), float32, one rounding to bf16: the
// router's term as a small GEMM (K = E) with the permute backward in its
// epilogue.  A block computes 128 tokens x 128 h; dlogits and W_gate pass
// through shared memory in chunks of 32 experts, transposed (expert-major) so
// that each k step is four 16-byte loads for 64 FMAs.  A thread holds 8
// tokens x two 4-wide h quads 64 apart (conflict-free loads; each quad of the
// gathered rows and of dx is an 8-byte piece of a 128-byte run).
constexpr int DX_T = 128, DX_H = 128, DX_E = 32, DX_P = DX_T + 4;
static_assert(DX_T == DX_H, "one padded row length for both tiles");

__device__ __forceinline__ void bf16x4_to_f32(uint2 v, float *f) {
  const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
  const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

__device__ __forceinline__ uint2 f32_to_bf16x4(const float *f) {
  uint2 o;
  __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&o);
  p[0] = __floats2bfloat162_rn(f[0], f[1]);
  p[1] = __floats2bfloat162_rn(f[2], f[3]);
  return o;
}

template <int KM>
__global__ void __launch_bounds__(BT) dx_final_kernel(const __nv_bfloat16 *__restrict__ dxp,
                                                      const float *__restrict__ dl,
                                                      const __nv_bfloat16 *__restrict__ wg,
                                                      const int32_t *__restrict__ inv,
                                                      __nv_bfloat16 *__restrict__ dx, int n, int K,
                                                      int E, int H, long long nK) {
  pdl_enter();
  __shared__ __align__(16) float ds[DX_E][DX_P];  // [e][token]
  __shared__ __align__(16) float ws[DX_E][DX_P];  // [e][h]
  __shared__ int srow[DX_T][KM];                   // the tokens' expert rows, -1: none
  const long long tb = (long long)blockIdx.x * DX_T;
  const int h0 = blockIdx.y * DX_H;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int i = threadIdx.x; i < DX_T * KM; i += BT) {
    const int t = i / KM, k = i % KM;
    int r = -1;
    if (tb + t < n && k < K) {
      r = __ldg(inv + (tb + t) * K + k);
      if (r < 0 || (long long)r >= nK) r = -1;
    }
    srow[t][k] = r;
  }
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int e0 = 0; e0 < E; e0 += DX_E) {
    for (int i = threadIdx.x; i < DX_T * DX_E; i += BT) {
      const int t = i / DX_E, e = i % DX_E;
      ds[e][t] = (tb + t < n && e0 + e < E) ? dl[(tb + t) * E + e0 + e] : 0.f;
      ws[e][t] = (e0 + e < E) ? __bfloat162float(wg[(size_t)(h0 + t) * E + e0 + e]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < DX_E; ++k) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&ds[k][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&ds[k][ty * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&ws[k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&ws[k][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  // + each token's K expert rows in slot order (slot outer: the 16 row pieces
  // of one slot are loaded before any is added), then one rounding
  const int hq0 = h0 + tx * 4, hq1 = h0 + 64 + tx * 4;
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    uint2 raw[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = srow[ty * 8 + i][k];
      raw[i][0] = raw[i][1] = make_uint2(0u, 0u);
      if (r >= 0) {
        raw[i][0] = __ldg(reinterpret_cast<const uint2 *>(dxp + (size_t)r * H + hq0));
        raw[i][1] = __ldg(reinterpret_cast<const uint2 *>(dxp + (size_t)r * H + hq1));
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float f[8];
      bf16x4_to_f32(raw[i][0], f);
      bf16x4_to_f32(raw[i][1], f + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] += f[j];
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const long long t = tb + ty * 8 + i;
    if (t < n) {
      *reinterpret_cast<uint2 *>(dx + t * H + hq0) = f32_to_bf16x4(acc[i]);
      *reinterpret_cast<uint2 *>(dx + t * H + hq1) = f32_to_bf16x4(acc[i] + 4);
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
cudaError_t dx_final_k(const Desc &d, const void *dx_perm, const float *dlogits,
                       const void *w_gate, const int32_t *inv, void *dx, cudaStream_t s) {
  return launch_pdl(dx_final_kernel<KM>, dim3((d.n + DX_T - 1) / DX_T, d.H / DX_H), dim3(BT), 0,
                    s, reinterpret_cast<const __nv_bfloat16 *>(dx_perm), dlogits,
                    reinterpret_cast<const __nv_bfloat16 *>(w_gate), inv,
                    reinterpret_cast<__nv_bfloat16 *>(dx), d.n, d.K, d.E, d.H, d.nK());
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

cudaError_t launch_router_bwd(const Desc &d, const void *x, const float *logits,
                              const int32_t *topk_idx, const float *topk_w, const float *dw,
                              float *dlogits, float *dw_part, float *dw_gate, float *dbias,
                              cudaStream_t s) {
  if (d.n == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(router_bwd_kernel, dim3(grid_warps(d.n)), dim3(BT), 0, s, logits,
                             topk_idx, topk_w, dw, dlogits, d.n, d.E, d.K, d.norm ? 1 : 0);
  if (e != cudaSuccess) return e;
  // dW_gate[h][e] = sum_t x[t][h] dlogits[t][e]: the tokens split into
  // RB_SPLIT ranges (partials in dw_part), then added in order
  const int kc = (d.n + RB_SPLIT - 1) / RB_SPLIT;
  e = launch_pdl(dw_gate_kernel, dim3(d.H / GW_H, (d.E + GW_E - 1) / GW_E, RB_SPLIT), dim3(BT), 0, s,
                 reinterpret_cast<const __nv_bfloat16 *>(x), (const float *)dlogits, dw_part, d.n,
                 d.H, d.E, kc);
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

cudaError_t launch_dx_final(const Desc &d, const void *dx_perm, const float *dlogits,
                            const void *w_gate, const int32_t *inv_perm, void *dx,
                            cudaStream_t s) {
  if (d.n == 0) return cudaSuccess;
  if (d.K <= 2) return dx_final_k<2>(d, dx_perm, dlogits, w_gate, inv_perm, dx, s);
  if (d.K <= 4) return dx_final_k<4>(d, dx_perm, dlogits, w_gate, inv_perm, dx, s);
  if (d.K <= 8) return dx_final_k<8>(d, dx_perm, dlogits, w_gate, inv_perm, dx, s);
  return dx_final_k<kMaxK>(d, dx_perm, dlogits, w_gate, inv_perm, dx, s);
}

}  // namespace moe
