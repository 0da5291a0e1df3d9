// Grouped SwiGLU expert GEMMs for float32 layers on the float32 FMA units,
// "MoE 分布式推理基础（基于 vLLM）" §1.2, Algorithm 2 steps 8-9.  The tensor
// cores' float32 path (TF32, 10-bit mantissa) is too coarse for a float32
// layer, so float32 layers use this tiled FMA kernel; bf16 layers use the
// tcgen05 kernel.  Tiles never straddle experts: an m-tile is a 32-row window
// starting at an expert's segment start.  Each output is one float32 FMA
// chain over k in ascending order.
#include "common.cuh"

namespace moe {
namespace {

constexpr int SBM = 32, SBN = 32, SBK = 16;

struct SimtTiles {
  int off[kMaxE + 1];
  int tp[kMaxE + 1];
  int total;
  int ok;
};

__device__ void build_tiles(SimtTiles &s, const int32_t *offsets, int E, int nK) {
  for (int c = threadIdx.x; c <= E; c += blockDim.x) s.off[c] = offsets[c];
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = s.off[0] == 0 && s.off[E] <= nK;
    int run = 0;
    for (int e = 0; e < E; ++e) {
      const int len = s.off[e + 1] - s.off[e];
      ok = ok && len >= 0;
      s.tp[e] = run;
      run += len > 0 ? (len + SBM - 1) / SBM : 0;
    }
    s.tp[E] = run;
    s.total = run;
    s.ok = ok;
  }
  __syncthreads();
}

__device__ __forceinline__ int find_expert(const SimtTiles &s, int mt, int E) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tp[mid] <= mt)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// GEMM1 + SwiGLU: h[r, j] = SiLU(sum_k x[r,k] W13[e][k, j]) * (sum_k x[r,k] W13[e][k, I+j])
__global__ void __launch_bounds__(256) simt_gemm1(const float *__restrict__ xp,
                                                  const float *__restrict__ w13,
                                                  const int32_t *__restrict__ offsets, int E,
                                                  int nK, int H, int I, float *__restrict__ h,
                                                  int32_t *status) {
  pdl_enter();
  __shared__ SimtTiles s;
  __shared__ float As[SBK][SBM];
  __shared__ float Bg[SBK][SBN];
  __shared__ float Bu[SBK][SBN];
  build_tiles(s, offsets, E, nK);
  if (!s.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
      flag_status(status, MOE_DEV_BAD_LAYOUT);
    return;
  }
  const int mt = blockIdx.x;
  if (mt >= s.total) return;
  const int e = find_expert(s, mt, E);
  const int row0 = s.off[e] + (mt - s.tp[e]) * SBM;
  const int rows = min(SBM, s.off[e + 1] - row0);
  const int col0 = blockIdx.y * SBN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const float *W = w13 + (size_t)e * H * 2 * I;
  float g[2][2] = {}, u[2][2] = {};
  for (int k0 = 0; k0 < H; k0 += SBK) {
    for (int i = threadIdx.x; i < SBK * SBM; i += 256) {
      const int r = i / SBK, kk = i % SBK;
      As[kk][r] = (r < rows && k0 + kk < H) ? xp[(size_t)(row0 + r) * H + k0 + kk] : 0.f;
    }
    for (int i = threadIdx.x; i < SBK * SBN; i += 256) {
      const int kk = i / SBN, c = i % SBN;
      const bool in = k0 + kk < H && col0 + c < I;
      Bg[kk][c] = in ? W[(size_t)(k0 + kk) * 2 * I + col0 + c] : 0.f;
      Bu[kk][c] = in ? W[(size_t)(k0 + kk) * 2 * I + I + col0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float a = As[kk][ty * 2 + i];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          g[i][j] = fmaf(a, Bg[kk][tx * 2 + j], g[i][j]);
          u[i][j] = fmaf(a, Bu[kk][tx * 2 + j], u[i][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = ty * 2 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = col0 + tx * 2 + j;
      if (c < I) {
        const float gv = g[i][j];
        h[(size_t)(row0 + r) * I + c] = gv / (1.0f + expf(-gv)) * u[i][j];
      }
    }
  }
}

// GEMM2: y_perm[r, c] = sum_k h[r, k] W2[e][k, c]
__global__ void __launch_bounds__(256) simt_gemm2(const float *__restrict__ h,
                                                  const float *__restrict__ w2,
                                                  const int32_t *__restrict__ offsets, int E,
                                                  int nK, int H, int I, float *__restrict__ yp,
                                                  int32_t *status) {
  pdl_enter();
  __shared__ SimtTiles s;
  __shared__ float As[SBK][SBM];
  __shared__ float Bs[SBK][SBN];
  build_tiles(s, offsets, E, nK);
  if (!s.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
      flag_status(status, MOE_DEV_BAD_LAYOUT);
    return;
  }
  const int mt = blockIdx.x;
  if (mt >= s.total) return;
  const int e = find_expert(s, mt, E);
  const int row0 = s.off[e] + (mt - s.tp[e]) * SBM;
  const int rows = min(SBM, s.off[e + 1] - row0);
  const int col0 = blockIdx.y * SBN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const float *W = w2 + (size_t)e * I * H;
  float acc[2][2] = {};
  for (int k0 = 0; k0 < I; k0 += SBK) {
    for (int i = threadIdx.x; i < SBK * SBM; i += 256) {
      const int r = i / SBK, kk = i % SBK;
      As[kk][r] = (r < rows && k0 + kk < I) ? h[(size_t)(row0 + r) * I + k0 + kk] : 0.f;
    }
    for (int i = threadIdx.x; i < SBK * SBN; i += 256) {
      const int kk = i / SBN, c = i % SBN;
      Bs[kk][c] = (k0 + kk < I && col0 + c < H) ? W[(size_t)(k0 + kk) * H + col0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float a = As[kk][ty * 2 + i];
#pragma unroll
        for (int j = 0; j < 2; ++j) acc[i][j] = fmaf(a, Bs[kk][tx * 2 + j], acc[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = ty * 2 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = col0 + tx * 2 + j;
      if (c < H) yp[(size_t)(row0 + r) * H + c] = acc[i][j];
    }
  }
}

}  // namespace

namespace {
inline int simt_max_mtiles(const Desc &d) {
  return (int)((d.nK() + SBM - 1) / SBM) + d.E;  // >= sum_e ceil(n_e / SBM)
}
}  // namespace

cudaError_t launch_gemm1_simt(const Desc &d, const void *x_perm, const void *w13,
                              const int32_t *offsets, void *h, int32_t *status, cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  dim3 g(simt_max_mtiles(d), (d.I + SBN - 1) / SBN);
  return launch_pdl(simt_gemm1, g, dim3(256), 0, s, reinterpret_cast<const float *>(x_perm),
                    reinterpret_cast<const float *>(w13), offsets, d.E, (int)nK, d.H, d.I,
                    reinterpret_cast<float *>(h), status);
}

cudaError_t launch_gemm2_simt(const Desc &d, const void *h, const void *w2,
                              const int32_t *offsets, void *y_perm, int32_t *status,
                              cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  dim3 g(simt_max_mtiles(d), (d.H + SBN - 1) / SBN);
  return launch_pdl(simt_gemm2, g, dim3(256), 0, s, reinterpret_cast<const float *>(h),
                    reinterpret_cast<const float *>(w2), offsets, d.E, (int)nK, d.H, d.I,
                    reinterpret_cast<float *>(y_perm), status);
}

}  // namespace moe
