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
// tile of an expert without rows is written as zeros.  float32 output, written
// by TMA tile stores from swizzled shared-memory staging buffers; persistent,
// double-buffered TMEM accumulators as in gemm_tc.cu.  Every CTA loads its own
// A and B boxes with plain (non-multicast) TMA copies.
//
// CTA pairs (PAIR, the default; moe_set_gemm_pairs): clusters of two CTAs on
// two SMs compute 256 M rows x 256 N columns with cta_group::2 MMAs, each CTA
// holding its own 128 M rows of A and half of the N columns of B, so six
// 32 KB operand stages fit where four 48 KB ones did.  The protocol is that of
// the grouped GEMM's pairs (gemm_tc.cu): the even CTA issues the MMAs and owns
// the operand-full barriers, which both CTAs' copies complete; its commits
// arrive on both CTAs' barriers; both CTAs' epilogue warps release the
// accumulator on its barriers; before the pair leaves it settles every stage
// whose two halves were not both loaded.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int WM = 128, WN = 256, WK = 64;
constexpr int WA_BOX = 64 * WK * 2;               // 8 KB: 64 m x 64 k
constexpr int WA_STAGE = 2 * WA_BOX;              // 16 KB
constexpr int WB_BOX = 64 * WK * 2;               // 8 KB: 64 n x 64 k
constexpr int W_MAX_STAGES = 6;

// Operand pipeline of one CTA: four stages of A (128 M) and all four B boxes
// (256 N), or (PAIR) six stages of A and half of B (two boxes, 128 N).
template <bool PAIR>
struct WPipe {
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int B_BOXES = PAIR ? 2 : 4;
  static constexpr int B_STAGE = B_BOXES * WB_BOX;
  static constexpr int STAGE = WA_STAGE + B_STAGE;
  static constexpr int UNIT_M = PAIR ? 2 * WM : WM;  // M rows of a work unit
};
constexpr int W_THREADS = 192;
constexpr int W_TMEM = 512;
constexpr int W_GROUP = 16;                       // rows of one k step
constexpr int W_GROUP_BYTES = W_GROUP * 128;      // one 16-row slice of a 64-wide box

constexpr int W_EPI_BYTES = 32 * 128;  // 32 rows x 32 float32 columns, 128-byte swizzle

struct WTail {
  uint64_t full[W_MAX_STAGES];
  uint64_t empty[W_MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ok;
  // PAIR: per stage, the phases this CTA's producer loaded and the bytes of
  // its last one; the leader also receives the odd CTA's
  int own_issued[W_MAX_STAGES], own_bytes[W_MAX_STAGES];
  int peer_issued[W_MAX_STAGES], peer_bytes[W_MAX_STAGES];
  int off[kMaxE + 1];
};

// stages | per epilogue warp two 1024-aligned staging buffers | WTail
template <bool PAIR>
constexpr size_t w_smem() {
  return 1024 + (size_t)WPipe<PAIR>::STAGES * WPipe<PAIR>::STAGE + 8 * W_EPI_BYTES +
         sizeof(WTail);
}
static_assert(w_smem<false>() <= 232448 && w_smem<true>() <= 232448,
              "wgrad shared memory above the per-block limit");
constexpr uint32_t W_IDESC = ptx::idesc_bf16_f32(WM, WN, /*a_mn=*/true, /*b_mn=*/true);
constexpr uint32_t W_IDESC_PAIR = ptx::idesc_bf16_f32(2 * WM, WN, /*a_mn=*/true, /*b_mn=*/true);

__device__ __forceinline__ bool w_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                       int32_t *status, long long limit) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      flag_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

struct WTile {
  int e, m0, n0, r0, rows, nkb;
};

// Work unit g: expert e, one M tile (128 rows, or 256 for a CTA pair, whose
// CTA `rank` takes rows [128 rank, 128 rank + 128)), one 256-column N tile.
template <bool PAIR = false>
__device__ __forceinline__ WTile w_decode(const WTail &st, int g, int mt, int nt, int rank = 0) {
  WTile w;
  const int per = mt * nt;
  w.e = g / per;
  const int rem = g - w.e * per;
  w.m0 = (rem / nt) * WPipe<PAIR>::UNIT_M + rank * WM;
  w.n0 = (rem % nt) * WN;
  w.r0 = st.off[w.e];
  w.rows = st.off[w.e + 1] - w.r0;
  w.nkb = (w.rows + WK - 1) / WK;
  return w;
}

// Persistent: one CTA per SM, or one CTA pair per two SMs (PAIR); work units
// are dealt round-robin.  A stage is refilled once the MMAs that read it have
// completed.
template <bool PAIR>
__global__ void __launch_bounds__(W_THREADS, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmA16,
                    const __grid_constant__ CUtensorMap tmB16,
                    const __grid_constant__ CUtensorMap tmAt,
                    const __grid_constant__ CUtensorMap tmBt,
                    const __grid_constant__ CUtensorMap tmOut,
                    const int32_t *__restrict__ offsets, int E, int nK, int M, int N,
                    int32_t *status, long long wait_limit) {
  using P = WPipe<PAIR>;
  constexpr int STAGES = P::STAGES;
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *smemA = smem;
  uint8_t *smemB = smem + STAGES * WA_STAGE;
  uint8_t *smemE = smem + STAGES * P::STAGE;
  WTail &st = *reinterpret_cast<WTail *>(smemE + 8 * W_EPI_BYTES);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = M / P::UNIT_M, nt = N / WN;
  const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
  const bool leader = rank == 0;
  const int cid = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ncl = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&st.full[s], 1);
      ptx::mbar_init(&st.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&st.tfull[a], 1);
      ptx::mbar_init(&st.tempty[a], PAIR ? 8 : 4);  // the epilogue warps (of both CTAs)
    }
    ptx::mbar_init(&st.drain, 1);
    for (int s = 0; s < W_MAX_STAGES; ++s)
      st.own_issued[s] = st.own_bytes[s] = st.peer_issued[s] = st.peer_bytes[s] = 0;
    st.abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  for (int c = tid; c <= E; c += W_THREADS) st.off[c] = offsets[c];
  // PAIR: both CTAs' barriers are initialised before either touches the other's
  if constexpr (PAIR)
    ptx::cluster_sync();
  else
    __syncthreads();
  if (tid == 0) {
    bool ok = st.off[0] == 0 && st.off[E] <= nK;
    for (int e = 0; e < E; ++e) ok = ok && st.off[e + 1] >= st.off[e];
    st.ok = ok;
    if (!ok && blockIdx.x == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
  }
  __syncthreads();
  if (!st.ok) return;  // the same decision in both CTAs of a pair
  // work units; the grid holds at most one CTA (pair) per unit
  const int total = E * mt * nt;

  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(&st.tmem_base, W_TMEM);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&st.tmem_base, W_TMEM);
      ptx::tmem_relinquish();
    }
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
      // PAIR: copies complete on the leader's operand-full barriers
      const uint32_t full0 = PAIR ? ptx::mapa_shared(ptx::smem_u32(&st.full[0]), 0) : 0u;
      // a box of this CTA's part: its own barrier, or the leader's (PAIR)
      auto load = [&](uint8_t *dst, const CUtensorMap *map, int stg, int c0, int c1) {
        if constexpr (PAIR)
          ptx::tma_load_2d_pair(dst, map, full0 + 8u * (uint32_t)stg, c0, c1);
        else
          ptx::tma_load_2d(dst, map, &st.full[stg], c0, c1);
      };
      // this CTA's B columns: all 256 of the unit, or (PAIR) its half
      const int nb0 = PAIR ? rank * (WN / 2) : 0;
      int stage = 0;
      uint32_t phase = 0, used = 0, last_par = 0;
      bool stop = false;
      for (int g = cid; g < total && !stop; g += ncl) {
        const WTile w = w_decode<PAIR>(st, g, mt, nt, rank);
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!w_wait(&st.empty[stage], phase ^ 1u, abort_flag, status, wait_limit)) {
            stop = true;
            break;
          }
          const int row = w.r0 + kb * WK;
          const int valid = min(WK, w.rows - kb * WK);
          uint8_t *sa = smemA + stage * WA_STAGE;
          uint8_t *sb = smemB + stage * P::B_STAGE;
          int bytes;  // this CTA's bytes of the stage
          if (valid == WK) {
            bytes = P::STAGE;
            if (!PAIR || leader)
              ptx::mbar_arrive_expect_tx(&st.full[stage], PAIR ? 2 * bytes : bytes);
#pragma unroll
            for (int q = 0; q < 2; ++q) load(sa + q * WA_BOX, &tmA, stage, w.m0 + q * 64, row);
#pragma unroll
            for (int q = 0; q < P::B_BOXES; ++q)
              load(sb + q * WB_BOX, &tmB, stage, w.n0 + nb0 + q * 64, row);
          } else {
            // the segment's last rows: whole 16-row groups from the operands,
            // the partial group from the zero-padded tail rows of expert e
            const int groups = (valid + W_GROUP - 1) / W_GROUP;
            const bool partial = (valid % W_GROUP) != 0;
            bytes = groups * (2 + P::B_BOXES) * W_GROUP_BYTES;
            if (!PAIR || leader)
              ptx::mbar_arrive_expect_tx(&st.full[stage], PAIR ? 2 * bytes : bytes);
            for (int gr = 0; gr < groups; ++gr) {
              const bool tail = partial && gr == groups - 1;
              const CUtensorMap *ma = tail ? &tmAt : &tmA16;
              const CUtensorMap *mb = tail ? &tmBt : &tmB16;
              const int r = tail ? w.e * W_GROUP : row + gr * W_GROUP;
#pragma unroll
              for (int q = 0; q < 2; ++q)
                load(sa + q * WA_BOX + gr * W_GROUP_BYTES, ma, stage, w.m0 + q * 64, r);
#pragma unroll
              for (int q = 0; q < P::B_BOXES; ++q)
                load(sb + q * WB_BOX + gr * W_GROUP_BYTES, mb, stage, w.n0 + nb0 + q * 64, r);
            }
          }
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if constexpr (PAIR) {
            ++st.own_issued[stage];
            st.own_bytes[stage] = bytes;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if constexpr (PAIR) {
        // copies still in flight are settled by the leader before the pair
        // leaves: it needs the odd CTA's counts
        if (!leader) {
          const uint32_t di = ptx::mapa_shared(ptx::smem_u32(&st.peer_issued[0]), 0);
          const uint32_t db = ptx::mapa_shared(ptx::smem_u32(&st.peer_bytes[0]), 0);
          for (int s2 = 0; s2 < STAGES; ++s2) {
            ptx::st_cluster_u32(di + 4u * s2, (uint32_t)st.own_issued[s2]);
            ptx::st_cluster_u32(db + 4u * s2, (uint32_t)st.own_bytes[s2]);
          }
        }
      } else {
        // never leave a TMA copy in flight: the last load of every stage has landed
        for (int s = 0; s < STAGES; ++s)
          if (used >> s & 1u) ptx::mbar_wait(&st.full[s], last_par >> s & 1u);
      }
    }
  } else if (warp == 1) {
    // one thread issues the MMAs (PAIR: the leader's); the rest of the warp
    // waits at the end
    if (lane == 0 && leader) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int g = cid; g < total; g += ncl) {
        const WTile w = w_decode<PAIR>(st, g, mt, nt, rank);
        if (!w_wait(&st.tempty[acc], acc_phase ^ 1u, abort_flag, status, wait_limit)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * WN);
        bool stop = false;
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!w_wait(&st.full[stage], phase, abort_flag, status, wait_limit)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          // k steps of 16 rows that hold segment rows (all four in a full block)
          const int ksteps = (min(WK, w.rows - kb * WK) + W_GROUP - 1) / W_GROUP;
          const uint32_t a0 = ptx::smem_u32(smemA + stage * WA_STAGE);
          const uint32_t b0 = ptx::smem_u32(smemB + stage * P::B_STAGE);
          for (int kk = 0; kk < ksteps; ++kk) {
            // both MN-major SW128: 64-wide atoms one box apart, k step = 16 rows
            const uint64_t adesc = ptx::smem_desc(a0 + kk * W_GROUP_BYTES, WA_BOX, 1024);
            const uint64_t bdesc = ptx::smem_desc(b0 + kk * W_GROUP_BYTES, WB_BOX, 1024);
            if constexpr (PAIR)
              ptx::mma_bf16_pair(d, adesc, bdesc, W_IDESC_PAIR, (kb | kk) != 0 ? 1u : 0u);
            else
              ptx::mma_bf16(d, adesc, bdesc, W_IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          if constexpr (PAIR)
            ptx::mma_commit_pair(&st.empty[stage], 0x3);
          else
            ptx::mma_commit(&st.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
        if constexpr (PAIR)
          ptx::mma_commit_pair(&st.tfull[acc], 0x3);
        else
          ptx::mma_commit(&st.tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if constexpr (PAIR)
        ptx::mma_commit_pair(&st.drain, 0x1);
      else
        ptx::mma_commit(&st.drain);
      ptx::mbar_wait(&st.drain, 0);
    }
    __syncwarp();
  } else {
    // epilogue warps 2..5 -> TMEM lane quarter (warp % 4) = 32 rows of M
    const int q = warp & 3;
    int acc = 0, nstore = 0;
    uint32_t acc_phase = 0;
    // PAIR: the odd CTA's warps release the accumulator on the leader's barrier
    const uint32_t tempty0 = PAIR ? ptx::mapa_shared(ptx::smem_u32(&st.tempty[0]), 0) : 0u;
    for (int g = cid; g < total; g += ncl) {
      const WTile w = w_decode<PAIR>(st, g, mt, nt, rank);
      if (!w_wait(&st.tfull[acc], acc_phase, abort_flag, status, wait_limit)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem + (uint32_t)(acc * WN) + ((uint32_t)(q * 32) << 16);
      // each 32-column chunk of this warp's 32 rows goes through a swizzled
      // staging buffer (lane = row; 16-byte piece j of row r at piece
      // j ^ (r % 8): conflict-free) and leaves as one TMA tile store
      const int orow = w.e * M + w.m0 + q * 32;
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
        uint8_t *buf = smemE + (2 * q + (nstore & 1)) * W_EPI_BYTES;
        // the store that last read this buffer (two chunks ago) must be done
        if (lane == 0) ptx::bulk_wait_group_read<1>();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4 *>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
              make_uint4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&tmOut, buf, w.n0 + c * 32, orow);
          ptx::bulk_commit_group();
        }
        ++nstore;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader)
          ptx::mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
        else
          ptx::mbar_arrive(&st.tempty[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) ptx::bulk_wait_group<0>();  // this warp's stores are complete
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncwarp();
  if constexpr (PAIR) {
    // every role of both CTAs is done and the odd CTA's counts are in the
    // leader: settle the stages whose two halves were not both loaded (the
    // halves of one phase have equal bytes), then wait for every copy
    ptx::cluster_sync();
    if (leader && tid == 0) {
      for (int s = 0; s < STAGES; ++s) {
        const int own = st.own_issued[s], peer = st.peer_issued[s];
        if (own == peer + 1)
          ptx::mbar_complete_tx(&st.full[s], (uint32_t)st.own_bytes[s]);
        else if (peer == own + 1)
          ptx::mbar_arrive_expect_tx(&st.full[s], (uint32_t)st.peer_bytes[s]);
        const int last = own > peer ? own : peer;
        if (last > 0) ptx::mbar_wait(&st.full[s], (uint32_t)(last - 1) & 1u);
      }
    }
    ptx::cluster_sync();  // no copy into either CTA is still in flight
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    __syncwarp();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem, W_TMEM);
    else
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

// out viewed as (rows x cols) float32, boxes of 32 columns x 32 rows, 128-byte
// swizzle (the epilogue's staging layout)
bool w_out_map(CUtensorMap *m, float *base, uint64_t cols, uint64_t rows) {
  EncodeFn enc = w_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct WgradArgs {
  CUtensorMap mA, mB, mA16, mB16, mAt, mBt, mOut;
  const int32_t *offsets;
  int E, nK, M, N;
  int32_t *status;
};

// Persistent launch: one CTA per SM, or as many CTA pairs as are resident at
// once (cached per device); at most one per work unit.
template <bool PAIR>
cudaError_t wgrad_launch(const WgradArgs &p, cudaStream_t s) {
  auto kernel = wgrad_tc_kernel<PAIR>;
  static int resident[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(W_THREADS);
  cfg.dynamicSmemBytes = w_smem<PAIR>();
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (!resident[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)w_smem<PAIR>());
    if (e != cudaSuccess) return e;
    int nc = device_sm_count();
    if (PAIR) {
      cfg.gridDim = dim3(2 * 16);
      cfg.attrs = attr;
      cfg.numAttrs = na;
      e = cudaOccupancyMaxActiveClusters(&nc, kernel, &cfg);
      if (e != cudaSuccess) return e;
    }
    if (nc < 1) return cudaErrorInvalidConfiguration;
    resident[dev] = nc;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const int units = p.E * (p.M / WPipe<PAIR>::UNIT_M) * (p.N / WN);
  const int n = units < resident[dev] ? units : resident[dev];
  cfg.gridDim = dim3((unsigned)((PAIR ? 2 : 1) * n));
  return cudaLaunchKernelEx(&cfg, kernel, p.mA, p.mB, p.mA16, p.mB16, p.mAt, p.mBt, p.mOut,
                            p.offsets, p.E, p.nK, p.M, p.N, p.status, pipeline_wait_limit());
}

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
  CUtensorMap mOut;
  if (!w_out_map(&mOut, out, N, (uint64_t)d.E * M)) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(wgrad_pack_tails_kernel, dim3(d.E * W_GROUP), dim3(256), 0, s,
                             (const __nv_bfloat16 *)a, M, (const __nv_bfloat16 *)b, N, offsets,
                             (int)nK, ta, tb);
  if (e != cudaSuccess) return e;
  const WgradArgs args{mA, mB, mA16, mB16, mAt, mBt, mOut, offsets, d.E, (int)nK, M, N, status};
  // CTA pairs need whole 256-row M units (M = H or I: multiples of 256 at the
  // usual sizes)
  if (!gemm_single_cta() && M % (2 * WM) == 0) return wgrad_launch<true>(args, s);
  return wgrad_launch<false>(args, s);
}

}  // namespace moe
