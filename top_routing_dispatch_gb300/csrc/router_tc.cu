// Router on the tcgen05 tensor cores with softmax and TopK fused into the
// epilogue, for bf16 layers with E % 64 == 0.  "MoE 分布式推理基础（基于
// vLLM）" §1.2, Algorithm 2 steps 1-3 and the router's renormalisation.
//
// One CTA per 128-token tile (persistent over tiles), 6 warps:
//   warp 0      TMA producer: x tile (128 tokens x 64 k) and E/64 boxes of
//               W_gate (64 k x 64 experts) per stage.
//   warp 1      TMEM allocator and MMA issuer: 128 x E x 16 bf16 MMAs into one
//               of two E-column float32 accumulators.
//   warps 2..5  epilogue, one thread per token (= TMEM lane): adds the bias,
//               stores the float32 logits, keeps the K+1 largest logits in
//               registers (descending, ties to the lower expert id), computes
//               max and sum of exp, and writes topk_idx / topk_w.  A token
//               whose top K+1 logits lie closer than the rounding margin tau
//               is flagged (topk_idx[t*K] = -1) and finished by the TopK kernel
//               of router.cu, which rescores its candidates in double-float.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int RT_BM = 128, RT_BK = 64, RT_STAGES = 4, RT_THREADS = 192;
constexpr int RT_A_BYTES = RT_BM * RT_BK * 2;   // 16 KB
constexpr int RT_BOX_BYTES = 64 * RT_BK * 2;    // 8 KB: 64 experts x 64 k

struct RtTail {
  uint64_t full[RT_STAGES];
  uint64_t empty[RT_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float bias[kMaxE];
};

inline size_t rt_smem_bytes(int E) {
  return 1024 + (size_t)RT_STAGES * (RT_A_BYTES + (E / 64) * RT_BOX_BYTES) + sizeof(RtTail);
}

__device__ __forceinline__ bool rt_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                        int32_t *status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > ptx::kWaitLimitCycles) {
      *abort_flag = 1;
      flag_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// (v, e) ranks above (w, f): larger value, or equal value and lower expert id
__device__ __forceinline__ bool ranks_above(float v, int e, float w, int f) {
  return v > w || (v == w && e < f);
}

template <int KM>  // K == KM: every list index is a compile-time constant
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const float *__restrict__ bias,
                     float *__restrict__ logits, int32_t *__restrict__ topk_idx,
                     float *__restrict__ topk_w, int n, int H, int E, int K, int norm,
                     uint32_t idesc, uint32_t tmem_cols, int32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nbox = E / 64;
  const int b_stage = nbox * RT_BOX_BYTES;
  uint8_t *smemA = smem;
  uint8_t *smemB = smem + RT_STAGES * RT_A_BYTES;
  RtTail &st = *reinterpret_cast<RtTail *>(smem + RT_STAGES * (RT_A_BYTES + b_stage));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (n + RT_BM - 1) / RT_BM;
  const int KB = H / RT_BK;
  if ((int)blockIdx.x >= n_tiles) return;

  if (tid == 0) {
    for (int s = 0; s < RT_STAGES; ++s) {
      ptx::mbar_init(&st.full[s], 1);
      ptx::mbar_init(&st.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&st.tfull[a], 1);
      ptx::mbar_init(&st.tempty[a], 4);
    }
    ptx::mbar_init(&st.drain, 1);
    st.abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  for (int e = tid; e < E; e += RT_THREADS) st.bias[e] = bias ? bias[e] : 0.f;
  __syncthreads();
  if (warp == 1) {
    ptx::tmem_alloc(&st.tmem_base, tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = st.tmem_base;
  volatile int *abort_flag = &st.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmX);
      ptx::prefetch_tmap(&tmW);
      int stage = 0;
      uint32_t phase = 0, used = 0, last_par = 0;
      const uint32_t tx_bytes = RT_A_BYTES + b_stage;
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        bool stop = false;
        for (int kb = 0; kb < KB; ++kb) {
          if (!rt_wait(&st.empty[stage], phase ^ 1u, abort_flag, status)) {
            stop = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(&st.full[stage], tx_bytes);
          ptx::tma_load_2d(smemA + stage * RT_A_BYTES, &tmX, &st.full[stage], kb * RT_BK,
                           t * RT_BM);
          for (int q = 0; q < nbox; ++q)
            ptx::tma_load_2d(smemB + stage * b_stage + q * RT_BOX_BYTES, &tmW, &st.full[stage],
                             q * 64, kb * RT_BK);
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == RT_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
      }
      for (int s = 0; s < RT_STAGES; ++s)
        if (used >> s & 1u) ptx::mbar_wait(&st.full[s], last_par >> s & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        if (!rt_wait(&st.tempty[acc], acc_phase ^ 1u, abort_flag, status)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * E);
        bool stop = false;
        for (int kb = 0; kb < KB; ++kb) {
          if (!rt_wait(&st.full[stage], phase, abort_flag, status)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smemA + stage * RT_A_BYTES);
          const uint32_t b0 = ptx::smem_u32(smemB + stage * b_stage);
#pragma unroll
          for (int kk = 0; kk < RT_BK / 16; ++kk) {
            const uint64_t adesc = ptx::smem_desc(a0 + kk * 32, 16, 1024);
            const uint64_t bdesc = ptx::smem_desc(b0 + kk * 2048, RT_BOX_BYTES, 1024);
            ptx::mma_bf16(d, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(&st.empty[stage]);
          if (++stage == RT_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
        ptx::mma_commit(&st.tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      ptx::mma_commit(&st.drain);
      ptx::mbar_wait(&st.drain, 0);
    }
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      if (!rt_wait(&st.tfull[acc], acc_phase, abort_flag, status)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + (uint32_t)(acc * E) + ((uint32_t)(q * 32) << 16);
      const int tok = t * RT_BM + r;
      const bool valid = tok < n;
      float *lrow = logits + (size_t)(valid ? tok : 0) * E;

      // pass 1: logits, running max, top K+1 list
      float lv[KM + 1];
      int li[KM + 1];
#pragma unroll
      for (int j = 0; j <= KM; ++j) {
        lv[j] = -INFINITY;
        li[j] = 0x7fffffff;
      }
      float last_v = -INFINITY;  // the (K+1)-th entry: the insertion threshold
      int last_i = 0x7fffffff;
      float m = -INFINITY;
      for (int c = 0; c < E / 8; ++c) {
        uint32_t raw[8];
        ptx::tmem_ld_32x32b_x8(tbase + c * 8, raw);
        ptx::tmem_ld_wait();
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(raw[i]) + st.bias[c * 8 + i];
        if (valid) {
          float4 *dst = reinterpret_cast<float4 *>(lrow + c * 8);
          dst[0] = make_float4(v[0], v[1], v[2], v[3]);
          dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          m = fmaxf(m, v[i]);
          const int e = c * 8 + i;
          if (ranks_above(v[i], e, last_v, last_i)) {
            float cv = v[i];
            int ci = e;
#pragma unroll
            for (int j = 0; j <= KM; ++j) {
              const bool gt = ranks_above(cv, ci, lv[j], li[j]);
              const float tv = gt ? lv[j] : cv;
              const int ti = gt ? li[j] : ci;
              lv[j] = gt ? cv : lv[j];
              li[j] = gt ? ci : li[j];
              cv = tv;
              ci = ti;
            }
            last_v = lv[KM];
            last_i = li[KM];
          }
        }
      }
      // pass 2: sum of exp(l - max)
      float ssum = 0.f;
      for (int c = 0; c < E / 32; ++c) {
        uint32_t raw[32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, raw);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          ssum += expf(__uint_as_float(raw[i]) + st.bias[c * 32 + i] - m);
      }
      // the accumulator can be reused by the next tile
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&st.tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;

      if (valid) {
        const int R = K + 1 < E ? K + 1 : E;
        const float tau = 1e-3f * fmaxf(1.f, fabsf(lv[0]));
        bool amb = false;
#pragma unroll
        for (int j = 0; j < KM; ++j)
          if (j + 1 < R && isfinite(lv[j]) && isfinite(lv[j + 1]) && lv[j] - lv[j + 1] < tau)
            amb = true;
        float w[KM];
        float wsum = 0.f;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          w[j] = j < K ? expf(lv[j] - m) / ssum : 0.f;
          wsum += w[j];
        }
        int32_t *irow = topk_idx + (size_t)tok * K;
        float *wrow = topk_w + (size_t)tok * K;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          if (j < K) {
            irow[j] = (j == 0 && amb) ? -1 : li[j];
            wrow[j] = norm ? w[j] / wsum : w[j];
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    __syncwarp();
    ptx::tmem_dealloc(tmem, tmem_cols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn rt_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool rt_map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
               uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = rt_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool router_tc_supported(const Desc &d) {
  return d.bf16 && d.E % 64 == 0 && d.E <= kMaxE && d.H % 64 == 0 && d.n > 0 && d.K >= 1 &&
         d.K <= 8 && d.K < d.E;
}

cudaError_t launch_router_tc(const Desc &d, const void *x, const void *w_gate, const float *bias,
                             int32_t *topk_idx, float *topk_w, float *logits, int32_t *status,
                             cudaStream_t s) {
  CUtensorMap mX, mW;
  if (!rt_map_2d(&mX, x, d.H, d.n, RT_BK, RT_BM) || !rt_map_2d(&mW, w_gate, d.E, d.H, 64, RT_BK))
    return cudaErrorInvalidValue;
  uint32_t cols = 32;
  while (cols < 2u * (uint32_t)d.E) cols <<= 1;
  const int n_tiles = (d.n + RT_BM - 1) / RT_BM;
  const int sms = device_sm_count();
  const int grid = n_tiles < sms ? n_tiles : sms;
  const uint32_t idesc = ptx::idesc_bf16_f32(RT_BM, d.E, false, true);
  auto run = [&](auto kernel) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rt_smem_bytes(kMaxE));
    if (e != cudaSuccess) return e;
    kernel<<<grid, RT_THREADS, rt_smem_bytes(d.E), s>>>(mX, mW, bias, logits, topk_idx, topk_w,
                                                        d.n, d.H, d.E, d.K, d.norm ? 1 : 0,
                                                        idesc, cols, status);
    return cudaSuccess;
  };
  cudaError_t e;
  switch (d.K) {
    case 1: e = run(router_tc_kernel<1>); break;
    case 2: e = run(router_tc_kernel<2>); break;
    case 3: e = run(router_tc_kernel<3>); break;
    case 4: e = run(router_tc_kernel<4>); break;
    case 5: e = run(router_tc_kernel<5>); break;
    case 6: e = run(router_tc_kernel<6>); break;
    case 7: e = run(router_tc_kernel<7>); break;
    default: e = run(router_tc_kernel<8>); break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
