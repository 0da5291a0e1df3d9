// Weight gradients of the expert GEMMs on the tcgen05 tensor cores:
//   dW2[e]  = h_e^T dY_e        (I x H)      dW13[e] = X_e^T [dG | dU]_e   (H x 2I)
// where _e are the rows [offsets[e], offsets[e+1]) of the expert-ordered
// arrays (the backward of Algorithm 2 steps 8-9 of "MoE 分布式推理基础（基于
// vLLM）" §1.2, with the expert's routed rows as the reduction dimension).
//
// C_e = A_e^T B_e with A (rows x M) and B (rows x N) row-major: both are
// MN-major UMMA operands (M or N contiguous), loaded by TMA as 64-wide,
// 64-row boxes with the 128-byte swizzle (the same layout as the forward's
// weight operand).  Tiles are (expert, 128 M rows, 256 N columns); the K loop
// runs over the expert's rows in blocks of 64, starting at the segment start.
// In the last block the rows past the segment belong to the next expert: the
// tensor cores must not see them.  That block is loaded as 16-row TMA boxes:
// whole 16-row groups of the segment from the operands themselves, and the
// last, partial group (rows % 16 rows) from a small zero-padded copy of each
// expert's last rows (wgrad_pack_tails_kernel, run just before); only the
// 16-row k steps that hold segment rows are issued.  No generic-proxy write
// ever reaches a pipeline stage, so no proxy fence sits in the MMA issue path
// (zeroing the rows in place with a fence there cost about 2 us per tile).  A
// tile of an expert without rows is written as zeros.  float32 output, one CTA
// per SM, persistent, double-buffered TMEM accumulators as in gemm_tc.cu.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int WM = 128, WN = 256, WK = 64, WSTAGES = 4;
constexpr int WA_BOX = 64 * WK * 2;               // 8 KB: 64 m x 64 k
constexpr int WA_STAGE = 2 * WA_BOX;              // 16 KB
constexpr int WB_BOX = 64 * WK * 2;               // 8 KB: 64 n x 64 k
constexpr int WB_STAGE = 4 * WB_BOX;              // 32 KB
constexpr int WSTAGE = WA_STAGE + WB_STAGE;
constexpr int W_THREADS = 192;
constexpr int W_TMEM = 512;
constexpr int W_GROUP = 16;                       // rows of one k step
constexpr int W_GROUP_BYTES = W_GROUP * 128;      // one 16-row slice of a 64-wide box

struct WTail {
  uint64_t full[WSTAGES];
  uint64_t empty[WSTAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ok;
  int off[kMaxE + 1];
  alignas(16) uint8_t epi[4][32 * 144];  // per epilogue warp: 32 rows x 128 B (+16 pad)
};

constexpr size_t W_SMEM = 1024 + (size_t)WSTAGES * WSTAGE + sizeof(WTail);
constexpr uint32_t W_IDESC = ptx::idesc_bf16_f32(WM, WN, /*a_mn=*/true, /*b_mn=*/true);

__device__ __forceinline__ bool w_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
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

struct WTile {
  int e, m0, n0, r0, rows, nkb;
};

__device__ __forceinline__ WTile w_decode(const WTail &st, int t, int mt, int nt) {
  WTile w;
  const int per = mt * nt;
  w.e = t / per;
  const int rem = t - w.e * per;
  w.m0 = (rem / nt) * WM;
  w.n0 = (rem % nt) * WN;
  w.r0 = st.off[w.e];
  w.rows = st.off[w.e + 1] - w.r0;
  w.nkb = (w.rows + WK - 1) / WK;
  return w;
}

__global__ void __launch_bounds__(W_THREADS, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmA16,
                    const __grid_constant__ CUtensorMap tmB16,
                    const __grid_constant__ CUtensorMap tmAt,
                    const __grid_constant__ CUtensorMap tmBt,
                    const int32_t *__restrict__ offsets, int E, int nK, int M, int N,
                    float *__restrict__ out, int32_t *status) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *smemA = smem;
  uint8_t *smemB = smem + WSTAGES * WA_STAGE;
  WTail &st = *reinterpret_cast<WTail *>(smem + WSTAGES * WSTAGE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = M / WM, nt = N / WN;

  if (tid == 0) {
    for (int s = 0; s < WSTAGES; ++s) {
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
  for (int c = tid; c <= E; c += W_THREADS) st.off[c] = offsets[c];
  __syncthreads();
  if (tid == 0) {
    bool ok = st.off[0] == 0 && st.off[E] <= nK;
    for (int e = 0; e < E; ++e) ok = ok && st.off[e + 1] >= st.off[e];
    st.ok = ok;
    if (!ok && blockIdx.x == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
  }
  __syncthreads();
  if (!st.ok) return;
  const int total = E * mt * nt;
  if ((int)blockIdx.x >= total) return;

  if (warp == 1) {
    ptx::tmem_alloc(&st.tmem_base, W_TMEM);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = st.tmem_base;
  volatile int *abort_flag = &st.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB);
      ptx::prefetch_tmap(&tmA16);
      ptx::prefetch_tmap(&tmB16);
      ptx::prefetch_tmap(&tmAt);
      ptx::prefetch_tmap(&tmBt);
      int stage = 0;
      uint32_t phase = 0, used = 0, last_par = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const WTile w = w_decode(st, t, mt, nt);
        bool stop = false;
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!w_wait(&st.empty[stage], phase ^ 1u, abort_flag, status)) {
            stop = true;
            break;
          }
          const int row = w.r0 + kb * WK;
          const int valid = min(WK, w.rows - kb * WK);
          uint8_t *sa = smemA + stage * WA_STAGE;
          uint8_t *sb = smemB + stage * WB_STAGE;
          if (valid == WK) {
            ptx::mbar_arrive_expect_tx(&st.full[stage], WSTAGE);
#pragma unroll
            for (int q = 0; q < 2; ++q)
              ptx::tma_load_2d(sa + q * WA_BOX, &tmA, &st.full[stage], w.m0 + q * 64, row);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              ptx::tma_load_2d(sb + q * WB_BOX, &tmB, &st.full[stage], w.n0 + q * 64, row);
          } else {
            // the segment's last rows: whole 16-row groups from the operands,
            // the partial group from the zero-padded tail rows of expert e
            const int groups = (valid + W_GROUP - 1) / W_GROUP;
            const bool partial = (valid % W_GROUP) != 0;
            ptx::mbar_arrive_expect_tx(&st.full[stage], groups * 6 * W_GROUP_BYTES);
            for (int g = 0; g < groups; ++g) {
              const bool tail = partial && g == groups - 1;
              const CUtensorMap *ma = tail ? &tmAt : &tmA16;
              const CUtensorMap *mb = tail ? &tmBt : &tmB16;
              const int r = tail ? w.e * W_GROUP : row + g * W_GROUP;
#pragma unroll
              for (int q = 0; q < 2; ++q)
                ptx::tma_load_2d(sa + q * WA_BOX + g * W_GROUP_BYTES, ma, &st.full[stage],
                                 w.m0 + q * 64, r);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                ptx::tma_load_2d(sb + q * WB_BOX + g * W_GROUP_BYTES, mb, &st.full[stage],
                                 w.n0 + q * 64, r);
            }
          }
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == WSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
      }
      for (int s = 0; s < WSTAGES; ++s)
        if (used >> s & 1u) ptx::mbar_wait(&st.full[s], last_par >> s & 1u);
    }
  } else if (warp == 1) {
    // one thread issues the MMAs; the rest of the warp waits at the end
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const WTile w = w_decode(st, t, mt, nt);
        if (!w_wait(&st.tempty[acc], acc_phase ^ 1u, abort_flag, status)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * WN);
        bool stop = false;
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!w_wait(&st.full[stage], phase, abort_flag, status)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          // k steps of 16 rows that hold segment rows (all four in a full block)
          const int ksteps = (min(WK, w.rows - kb * WK) + W_GROUP - 1) / W_GROUP;
          const uint32_t a0 = ptx::smem_u32(smemA + stage * WA_STAGE);
          const uint32_t b0 = ptx::smem_u32(smemB + stage * WB_STAGE);
          for (int kk = 0; kk < ksteps; ++kk) {
            // both MN-major SW128: 64-wide atoms one box apart, k step = 16 rows
            const uint64_t adesc = ptx::smem_desc(a0 + kk * W_GROUP_BYTES, WA_BOX, 1024);
            const uint64_t bdesc = ptx::smem_desc(b0 + kk * W_GROUP_BYTES, WB_BOX, 1024);
            ptx::mma_bf16(d, adesc, bdesc, W_IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(&st.empty[stage]);
          if (++stage == WSTAGES) {
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
    __syncwarp();
  } else {
    // epilogue warps 2..5 -> TMEM lane quarter (warp % 4) = 32 rows of M
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const WTile w = w_decode(st, t, mt, nt);
      if (!w_wait(&st.tfull[acc], acc_phase, abort_flag, status)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem + (uint32_t)(acc * WN) + ((uint32_t)(q * 32) << 16);
      // rows of this warp's 32-row slice; each 32-column chunk is staged in
      // shared memory and stored as whole 128-byte row segments (8 lanes a row)
      float *base = out + ((size_t)w.e * M + w.m0 + q * 32) * N + w.n0;
      uint8_t *eb = st.epi[warp - 2];
#pragma unroll 1
      for (int c = 0; c < WN / 32; ++c) {
        uint32_t a[32];
        if (w.nkb > 0) {  // uniform across the warp
          ptx::tmem_ld_32x32b_x32(tb + c * 32, a);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = 0u;
        }
        uint4 *mine = reinterpret_cast<uint4 *>(eb + lane * 144);
#pragma unroll
        for (int v = 0; v < 8; ++v) mine[v] = make_uint4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int p = lane + 32 * i;
          const int r = p >> 3, c16 = p & 7;
          const uint4 val = *reinterpret_cast<const uint4 *>(eb + r * 144 + c16 * 16);
          *reinterpret_cast<uint4 *>(base + (size_t)r * N + c * 32 + c16 * 4) = val;
        }
        __syncwarp();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&st.tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    __syncwarp();
    ptx::tmem_dealloc(tmem, W_TMEM);
  }
}

// Row e*16 + j of ta / tb = row offsets[e+1] - p + j of a / b for j < p,
// zero for j >= p, where p = (segment rows) % 16: the partial last 16-row
// group of expert e, zero-padded.  Experts whose row count is a multiple of
// 16 have no partial group and their tail rows are never read.  One block per
// (expert, row).
__global__ void __launch_bounds__(256)
    wgrad_pack_tails_kernel(const __nv_bfloat16 *__restrict__ a, int M,
                            const __nv_bfloat16 *__restrict__ b, int N,
                            const int32_t *__restrict__ offsets, int nK,
                            __nv_bfloat16 *__restrict__ ta, __nv_bfloat16 *__restrict__ tb) {
  pdl_enter();
  const int e = blockIdx.x / W_GROUP, j = blockIdx.x % W_GROUP;
  const int r0 = offsets[e], r1 = offsets[e + 1];
  if (r0 < 0 || r1 < r0 || r1 > nK) return;  // the GEMM reports the bad layout
  const int p = (r1 - r0) % W_GROUP;
  if (p == 0) return;
  const bool real = j < p;
  const size_t src = (size_t)(r1 - p + j), dst = (size_t)e * W_GROUP + j;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint4 *sa = reinterpret_cast<const uint4 *>(a) + src * (M / 8);
  uint4 *da = reinterpret_cast<uint4 *>(ta) + dst * (M / 8);
  for (int i = threadIdx.x; i < M / 8; i += blockDim.x) da[i] = real ? sa[i] : zero;
  const uint4 *sb = reinterpret_cast<const uint4 *>(b) + src * (N / 8);
  uint4 *db = reinterpret_cast<uint4 *>(tb) + dst * (N / 8);
  for (int i = threadIdx.x; i < N / 8; i += blockDim.x) db[i] = real ? sb[i] : zero;
}

typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                             const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                             const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                             CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn w_encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// rows x cols row-major bf16, boxes of 64 columns x box_rows rows, 128-byte
// swizzle
bool w_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeFn enc = w_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t wgrad_tail_bytes(const Desc &d, int M, int N) {
  return (size_t)d.E * W_GROUP * ((size_t)M + N) * 2;
}

// out[e] (M x N, float32) = a[seg_e]^T b[seg_e]; a (nK x M), b (nK x N) bf16;
// M % 128 == 0, N % 256 == 0; tail: wgrad_tail_bytes(d, M, N) bytes of
// scratch, 16-byte aligned
cudaError_t launch_wgrad_tc(const Desc &d, const void *a, int M, const void *b, int N,
                            const int32_t *offsets, void *tail, float *out, int32_t *status,
                            cudaStream_t s) {
  if (M % WM || N % WN) return cudaErrorInvalidValue;
  const long long nK = d.nK();
  __nv_bfloat16 *ta = reinterpret_cast<__nv_bfloat16 *>(tail);
  __nv_bfloat16 *tb = ta + (size_t)d.E * W_GROUP * M;
  CUtensorMap mA, mB, mA16, mB16, mAt, mBt;
  // a zero-row map is not encodable: point an empty layout at one row (no
  // expert has rows, so nothing is loaded; every tile writes zeros)
  const uint64_t rows = nK > 0 ? (uint64_t)nK : 1;
  const uint64_t trows = (uint64_t)d.E * W_GROUP;
  if (!w_map(&mA, a, M, rows, WK) || !w_map(&mB, b, N, rows, WK) ||
      !w_map(&mA16, a, M, rows, W_GROUP) || !w_map(&mB16, b, N, rows, W_GROUP) ||
      !w_map(&mAt, ta, M, trows, W_GROUP) || !w_map(&mBt, tb, N, trows, W_GROUP))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  static int done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !done[dev]) {
    e = cudaFuncSetAttribute(wgrad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)W_SMEM);
    if (e != cudaSuccess) return e;
    done[dev] = 1;
  }
  e = launch_pdl(wgrad_pack_tails_kernel, dim3(d.E * W_GROUP), dim3(256), 0, s,
                 (const __nv_bfloat16 *)a, M, (const __nv_bfloat16 *)b, N, offsets, (int)nK, ta,
                 tb);
  if (e != cudaSuccess) return e;
  const int total = d.E * (M / WM) * (N / WN);
  const int sms = device_sm_count();
  const int grid = total < sms ? total : sms;
  return launch_pdl(wgrad_tc_kernel, dim3(grid), dim3(W_THREADS), W_SMEM, s, mA, mB, mA16, mB16,
                    mAt, mBt, offsets, d.E, (int)nK, M, N, out, status);
}

}  // namespace moe
