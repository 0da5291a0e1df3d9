// Router: logits = x·W_gate (+ bias), softmax over experts, TopK, optional
// renormalisation.  "MoE 分布式推理基础（基于 vLLM）" §1.2, Algorithm 2 steps
// 1-3 and the router's norm_topk_prob branch.
//
// bf16 layers with E % 64 == 0 and K <= 8 use router_tc.cu (one kernel:
// tensor-core logits, softmax, TopK and near-tie rescoring).  Other layers
// use two kernels:
//  1. router_logits_kernel: SIMT tiled GEMM (n x H)·(H x E) with float32
//     accumulation in per-tile partial sums (32 products per partial, then
//     added to the running sum), bias added last.  Products of bf16 inputs are
//     exact in float32, so only the additions round.
//  2. router_topk_kernel: one warp per token.  Max, sum of exp and K+1 rounds
//     of a warp argmax (ties to the lower expert id) over the float32 logits.
//     If two of the top K+1 logits lie closer than a margin tau (far above the
//     float32 error of kernel 1), the experts that can still be in the top K
//     are rescored in double-float arithmetic (exact products, error-free
//     sums) and the K best are chosen on those values.  The choice therefore
//     matches an exact evaluation except for gaps near double-float rounding.
#include <math.h>

#include "common.cuh"
#include "df.cuh"

namespace moe {
namespace {

constexpr int RBM = 32, RBN = 64, RBK = 32, RTHREADS = 128;

template <bool BF16>
__device__ __forceinline__ float ld_in(const void *p, size_t i) {
  if constexpr (BF16)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  else
    return reinterpret_cast<const float *>(p)[i];
}

template <bool BF16>
__global__ void __launch_bounds__(RTHREADS) router_logits_kernel(
    const void *__restrict__ x, const void *__restrict__ wg, const float *__restrict__ bias,
    float *__restrict__ logits, int n, int H, int E) {
  pdl_enter();
  __shared__ float As[RBK][RBM + 4];  // k-major
  __shared__ float Bs[RBK][RBN + 4];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.x * RBM, n0 = blockIdx.y * RBN;
  const int tx = tid % 16, ty = tid / 16;  // 16 x 8 threads, 4x4 outputs each
  float total[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += RBK) {
    // A tile: 32 rows x 32 k; thread loads 8 consecutive k of one row
    {
      const int r = tid / 4, kk = (tid % 4) * 8;
      const int gm = m0 + r;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int gk = k0 + kk + j;
        As[kk + j][r] = (gm < n && gk < H) ? ld_in<BF16>(x, (size_t)gm * H + gk) : 0.f;
      }
    }
    // B tile: 32 k x 64 experts
#pragma unroll
    for (int j = 0; j < (RBK * RBN) / RTHREADS; ++j) {
      const int idx = tid + j * RTHREADS;
      const int kk = idx / RBN, c = idx % RBN;
      const int gk = k0 + kk, gn = n0 + c;
      Bs[kk][c] = (gk < H && gn < E) ? ld_in<BF16>(wg, (size_t)gk * E + gn) : 0.f;
    }
    __syncthreads();
    float part[4][4] = {};
#pragma unroll 8
    for (int kk = 0; kk < RBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = fmaf(a[i], b[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) total[i][j] += part[i][j];
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= n) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn < E) logits[(size_t)gm * E + gn] = total[i][j] + (bias ? bias[gn] : 0.f);
    }
  }
}

// (value, expert) argmax across the warp; ties to the lower expert id.
__device__ __forceinline__ void warp_argmax(float &v, int &e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oe = __shfl_xor_sync(0xffffffffu, e, o);
    if (ov > v || (ov == v && oe < e)) {
      v = ov;
      e = oe;
    }
  }
}

constexpr int TOPK_WARPS = 8;

constexpr int RG = 8;  // candidates rescored per pass over H
constexpr int RU = 4;  // rows of W_gate per lane per step of that pass

// only_flagged: finish only the tokens the tensor-core router flagged as
// near ties (topk_idx[t*K] < 0); other tokens are left as they are.
template <int EPL, bool BF16>
__global__ void __launch_bounds__(TOPK_WARPS * 32) router_topk_kernel(
    const float *__restrict__ logits, const void *__restrict__ x, const void *__restrict__ wg,
    const __nv_bfloat16 *__restrict__ wgt, const float *__restrict__ bias,
    int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int n, int H, int E, int K,
    int norm, int only_flagged) {
  pdl_enter();
  __shared__ float s_hi[TOPK_WARPS][kMaxK];
  __shared__ float s_lo[TOPK_WARPS][kMaxK];
  __shared__ int s_e[TOPK_WARPS][kMaxK];
  __shared__ int s_cand[TOPK_WARPS][kMaxE];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int t = blockIdx.x * TOPK_WARPS + wib;
  if (t >= n) return;
  if (only_flagged && topk_idx[(size_t)t * K] >= 0) return;
  const float NEG = -INFINITY;
  float v[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? logits[(size_t)t * E + e] : NEG;
  }
  float m = NEG;
#pragma unroll
  for (int j = 0; j < EPL; ++j) m = fmaxf(m, v[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < EPL; ++j)
    if (lane + 32 * j < E) s += expf(v[j] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);

  // K+1 rounds of argmax over the unselected experts
  const int R = K + 1 < E ? K + 1 : E;
  unsigned taken = 0;
  float top_v[kMaxK + 1];
  int top_e[kMaxK + 1];
#pragma unroll
  for (int r = 0; r < kMaxK + 1; ++r) {
    if (r >= R) break;
    float bv = NEG;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !(taken >> j & 1u) && (v[j] > bv || (v[j] == bv && e < be))) {
        bv = v[j];
        be = e;
      }
    }
    warp_argmax(bv, be);
    top_v[r] = bv;
    top_e[r] = be;
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
  }

  // near-tie check among the top K+1 (finite values only)
  const float tau = kTieMarginSimt * fmaxf(1.f, fabsf(top_v[0]));
  bool amb = false;
#pragma unroll
  for (int r = 0; r + 1 < kMaxK + 1; ++r) {
    if (r + 1 >= R) break;
    if (isfinite(top_v[r]) && isfinite(top_v[r + 1]) && top_v[r] - top_v[r + 1] < tau) amb = true;
  }

  if (amb) {  // warp-uniform: every lane holds the same top_v
    float vK = top_v[0];
#pragma unroll
    for (int r = 0; r < kMaxK; ++r)
      if (r == K - 1) vK = top_v[r];
    const float thr = vK - tau;
    // candidates, in ascending expert id: every expert that can still be in
    // the top K given the float32 error (< tau/2)
    int C = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const unsigned ball = __ballot_sync(0xffffffffu, lane + 32 * j < E && v[j] >= thr);
      if (ball >> lane & 1u) s_cand[wib][C + __popc(ball & ((1u << lane) - 1u))] = lane + 32 * j;
      C += __popc(ball);
    }
    __syncwarp();
    int cnt = 0;  // entries in the per-warp sorted list (uniform)
    for (int g0 = 0; g0 < C; g0 += RG) {
      int ce[RG];
#pragma unroll
      for (int c = 0; c < RG; ++c) ce[c] = g0 + c < C ? s_cand[wib][g0 + c] : -1;
      DF acc[RG];
#pragma unroll
      for (int c = 0; c < RG; ++c) acc[c] = DF{0.f, 0.f};
      // one pass over H for RG candidates: a lane reads x[h] once and the
      // candidates' weights from the same row of W_gate
      // RU rows per lane per step: all their loads are issued before the
      // double-float work, so many requests are in flight
      for (int h0 = lane; h0 < H; h0 += 32 * RU) {
        float xv[RU], wv[RU][RG];
#pragma unroll
        for (int u = 0; u < RU; ++u) {
          const int hh = h0 + 32 * u;
          const bool in = hh < H;
          xv[u] = in ? ld_in<BF16>(x, (size_t)t * H + hh) : 0.f;
#pragma unroll
          for (int c = 0; c < RG; ++c)
            // W_gate[hh][ce[c]]: from the transposed copy (bf16) when given
            wv[u][c] = !(in && ce[c] >= 0) ? 0.f
                       : (BF16 && wgt) ? __bfloat162float(wgt[(size_t)ce[c] * H + hh])
                                       : ld_in<BF16>(wg, (size_t)hh * E + ce[c]);
        }
#pragma unroll
        for (int u = 0; u < RU; ++u)
#pragma unroll
          for (int c = 0; c < RG; ++c)
            if (ce[c] >= 0) acc[c] = df_add(acc[c], two_prod(xv[u], wv[u][c]));
      }
#pragma unroll
      for (int c = 0; c < RG; ++c) {
        if (ce[c] < 0) break;  // uniform
        DF a = acc[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          DF other{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
          a = df_add(a, other);
        }
        const int e = ce[c];
        if (bias) {
          const float bb = bias[e];
          if (isinf(bb))
            a = DF{bb, 0.f};
          else
            a = df_add(a, DF{bb, 0.f});
        }
        // insert (a, e) into the warp's sorted list of at most K entries
        if (lane == 0) {
          int pos = cnt < K ? cnt : K;
          while (pos > 0 && df_greater(a, e, DF{s_hi[wib][pos - 1], s_lo[wib][pos - 1]},
                                       s_e[wib][pos - 1]))
            --pos;
          if (pos < K) {
            const int last = (cnt < K ? cnt : K - 1);
            for (int q = last; q > pos; --q) {
              s_hi[wib][q] = s_hi[wib][q - 1];
              s_lo[wib][q] = s_lo[wib][q - 1];
              s_e[wib][q] = s_e[wib][q - 1];
            }
            s_hi[wib][pos] = a.hi;
            s_lo[wib][pos] = a.lo;
            s_e[wib][pos] = e;
          }
        }
        cnt = cnt < K ? cnt + 1 : K;
        __syncwarp();
      }
    }
    // cnt >= K always: the K experts of largest float32 logit are candidates
#pragma unroll
    for (int r = 0; r < kMaxK; ++r)
      if (r < K) top_e[r] = s_e[wib][r];
    __syncwarp();
  }

  // weights: p at the chosen experts (float32 softmax), optional renormalisation
  float w = 0.f;
  int e_mine = 0;
  if (lane < K) {
#pragma unroll
    for (int r = 0; r < kMaxK; ++r)
      if (r == lane) e_mine = top_e[r];
    w = expf(logits[(size_t)t * E + e_mine] - m) / s;
  }
  if (norm) {
    float tot = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxK; ++r) {
      const float wr = __shfl_sync(0xffffffffu, w, r);
      if (r < K) tot += wr;
    }
    w = w / tot;
  }
  if (lane < K) {
    topk_idx[(size_t)t * K + lane] = e_mine;
    topk_w[(size_t)t * K + lane] = w;
  }
}

template <int EPL>
cudaError_t launch_topk(const Desc &d, const float *logits, const void *x, const void *wg,
                        const float *bias, int32_t *idx, float *w, int only_flagged,
                        cudaStream_t s) {
  dim3 grid((d.n + TOPK_WARPS - 1) / TOPK_WARPS);
  if (d.bf16)
    return launch_pdl(router_topk_kernel<EPL, true>, grid, dim3(TOPK_WARPS * 32), 0, s, logits, x,
                      wg, reinterpret_cast<const __nv_bfloat16 *>(d.w_gate_t), bias, idx, w, d.n,
                      d.H, d.E, d.K, d.norm, only_flagged);
  return launch_pdl(router_topk_kernel<EPL, false>, grid, dim3(TOPK_WARPS * 32), 0, s, logits, x,
                    wg, (const __nv_bfloat16 *)nullptr, bias, idx, w, d.n, d.H, d.E, d.K, d.norm,
                    only_flagged);
}

cudaError_t launch_topk_any(const Desc &d, const float *logits, const void *x, const void *wg,
                            const float *bias, int32_t *idx, float *w, int only_flagged,
                            cudaStream_t s) {
  if (d.E <= 32) return launch_topk<1>(d, logits, x, wg, bias, idx, w, only_flagged, s);
  if (d.E <= 64) return launch_topk<2>(d, logits, x, wg, bias, idx, w, only_flagged, s);
  if (d.E <= 128) return launch_topk<4>(d, logits, x, wg, bias, idx, w, only_flagged, s);
  return launch_topk<8>(d, logits, x, wg, bias, idx, w, only_flagged, s);
}

}  // namespace

int router_launches(const Desc &d) {
  if (d.n == 0) return 0;
  if (router_mma_supported(d)) return 1;  // one kernel: logits, TopK, near-tie rescoring
  return 2;  // tensor-core tile kernel + rescoring, or FMA logits + TopK
}

cudaError_t launch_router(const Desc &d, const void *x, const void *w_gate, const float *bias,
                          int32_t *topk_idx, float *topk_w, float *logits, int32_t *status,
                          cudaStream_t s, bool guest) {
  if (d.n == 0) return cudaSuccess;
  if (router_mma_supported(d)) {
    // warp-level MMA logits with softmax, TopK and near-tie rescoring in one
    // kernel that fits beside a persistent GEMM CTA on an SM
    return launch_router_mma(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
  }
  if (router_tc_supported(d)) {
    // tensor-core logits with softmax, TopK and near-tie rescoring fused
    return launch_router_tc(d, x, w_gate, bias, topk_idx, topk_w, logits, status, s);
  }
  dim3 grid((d.n + RBM - 1) / RBM, (d.E + RBN - 1) / RBN);
  cudaError_t err =
      d.bf16 ? launch_pdl(router_logits_kernel<true>, grid, dim3(RTHREADS), 0, s, x, w_gate, bias,
                          logits, d.n, d.H, d.E)
             : launch_pdl(router_logits_kernel<false>, grid, dim3(RTHREADS), 0, s, x, w_gate,
                          bias, logits, d.n, d.H, d.E);
  if (err != cudaSuccess) return err;
  return launch_topk_any(d, logits, x, w_gate, bias, topk_idx, topk_w, 0, s);
}

}  // namespace moe
