// Grouped SwiGLU expert GEMMs on the tcgen05 tensor cores (bf16 in, f32
// accumulate in TMEM), "MoE 分布式推理基础（基于 vLLM）" §1.2, Algorithm 2
// steps 8-9 and "SwiGLU expert 的两段 GEMM":
//   GEMM1: [G | U] = X_e · W13[e] (H x 2I), h = SiLU(G) * U   (fused epilogue)
//   GEMM2: Y_e = h · W2[e] (I x H)
// over the expert segments [offsets[e], offsets[e+1]) of the expert-sorted
// rows.  Putting SiLU*up in the first GEMM's epilogue follows the L1
// epilogue of the DeepGEMM Mega MoE kernel described in "大模型系统中的通算
// 融合" §4 (one L1 GEMM produces gate and up, the epilogue applies SwiGLU).
//
// Design (persistent, 6 warps per CTA):
//   warp 0      TMA producer: A tile (128 rows x 64 k) of the activations and
//               the expert's weight boxes (64 k x 64 n) per stage.
//   warp 1      TMEM allocator and MMA issuer: 4 x tcgen05.mma per stage into
//               one of two 256-column TMEM accumulators.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one row per thread),
//               SiLU(gate)*up (GEMM1) or plain conversion (GEMM2), bf16 stores
//               of the rows that belong to the tile's expert.
// Two forms, bitwise the same.  Single CTAs: one CTA per SM, 128x256x16 MMAs,
// four 48 KB stages (A + four B boxes).  CTA pairs (PAIR, the default): one
// cluster of two CTAs per two SMs, 256x256x16 cta_group::2 MMAs issued by the
// even CTA, each CTA holding its own 128 A rows and half of the weight tile
// (two B boxes), six 32 KB stages (see the kernel's comment for the protocol).
// A tile is (m-tile, n-tile).  m-tiles are 128-row windows that start at each
// expert's segment start, so every tile belongs to exactly one expert; its
// rows past the segment end are computed but not stored (TMA zero-fills rows
// past the tensor).  Tiles are dealt to CTAs round-robin; every tile costs the
// same (full K loop), so the static schedule balances.  Each tile is computed
// entirely by one CTA with a fixed k order: results do not depend on the grid
// size.
//
// B is the weight matrix as stored (k rows, n contiguous): an MN-major UMMA
// operand with 128-byte swizzle.  A is K-major with 128-byte swizzle.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BK = 64, UMMA_N = 256, UMMA_K = 16;
constexpr int A_STAGE_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;            // 8 KB: 64 n x 64 k
constexpr int kMaxStages = 6;

// Operand pipeline of one CTA.  Single CTAs: four stages of A (128 rows) and
// all four B boxes (256 n).  CTA pairs (PAIR): the pair computes a 256-row x
// 256-column tile with cta_group::2 MMAs; each CTA holds its own 128 A rows
// and half of B (two boxes, 128 n), so six 32 KB stages fit in the same
// shared memory.
template <bool PAIR>
struct Pipe {
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int B_BOXES = PAIR ? 2 : 4;
  static constexpr int B_STAGE = B_BOXES * B_BOX_BYTES;
  static constexpr int STAGE = A_STAGE_BYTES + B_STAGE;
  static constexpr int TILE_ROWS = PAIR ? 2 * BM : BM;  // rows of an m-tile (whole pair)
};
static_assert(Pipe<true>::STAGES <= kMaxStages && Pipe<false>::STAGES <= kMaxStages, "");
// warp 0: TMA producer, warp 1: MMA issuer, warps 2-5: epilogue; MODE 3 adds
// warps 6-9, which gather the A rows with cp.async
constexpr int NUM_THREADS = 192;
// MODE 3 copies a tile's 128 A rows with 16-byte cp.async from GATHER_WARPS
// extra warps (warps 6..9).
constexpr int GATHER_WARPS = BM / 32;
constexpr int threads_for(int mode) {
  return mode == 3 ? NUM_THREADS + 32 * GATHER_WARPS : NUM_THREADS;
}
constexpr int TMEM_COLS = 512;                      // two 256-column accumulators
constexpr int EPI_ROW_BYTES = 80, EPI_WARP_BYTES = 32 * EPI_ROW_BYTES;

struct SmemTail {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ok;
  int total_mtiles;
  int own_issued[kMaxStages];   // PAIR: phases this CTA's producer loaded, per stage
  int peer_issued[kMaxStages];  // PAIR (leader): the odd CTA's own_issued
  int off[kMaxE + 1];
  int tp[kMaxE + 1];  // first m-tile of each expert (exclusive prefix)
  alignas(16) uint8_t epi[4][EPI_WARP_BYTES];  // per epilogue warp staging
};

template <bool PAIR>
constexpr size_t smem_bytes() {
  return 1024 /*alignment slack*/ + (size_t)Pipe<PAIR>::STAGES * Pipe<PAIR>::STAGE +
         sizeof(SmemTail);
}
constexpr size_t SMEM_BYTES = smem_bytes<false>();
static_assert(smem_bytes<true>() <= 227 * 1024, "pair pipeline exceeds shared memory");

constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/true);
constexpr uint32_t IDESC_KB = ptx::idesc_bf16_f32(BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/false);
constexpr uint32_t IDESC_PAIR = ptx::idesc_bf16_f32(2 * BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/true);
constexpr uint32_t IDESC_PAIR_KB = ptx::idesc_bf16_f32(2 * BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/false);

// A pipeline wait: gives up after `limit` cycles (setting the abort flag and
// MOE_DEV_TIMEOUT), or at once when another role has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile int *abort_flag, int32_t *status,
                                              long long limit) {
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

struct TileInfo {
  int e, row0, rows, nt;
};

// Tile t: expert, first row and stored rows of this CTA's 128-row part
// (PAIR: rank 0 takes rows [0, 128) of the pair's 256-row window, rank 1 rows
// [128, 256); rows may be <= 0 when the segment ends in the first half).
template <bool PAIR = false>
__device__ __forceinline__ TileInfo decode_tile(const SmemTail &s, int t, int n_tiles, int E,
                                                int rank = 0) {
  TileInfo ti;
  const int mt = t / n_tiles;
  ti.nt = t - mt * n_tiles;
  int lo = 0, hi = E;  // largest e with tp[e] <= mt
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tp[mid] <= mt)
      lo = mid;
    else
      hi = mid;
  }
  ti.e = lo;
  ti.row0 = s.off[lo] + (mt - s.tp[lo]) * Pipe<PAIR>::TILE_ROWS + rank * BM;
  const int left = s.off[lo + 1] - ti.row0;
  ti.rows = left < BM ? left : BM;
  return ti;
}

// MODE 3: perm entry of tile row rr (0 past the segment: such rows are never
// stored and read token 0), and the token it names
__device__ __forceinline__ int tile_perm(const int32_t *__restrict__ perm, const TileInfo &ti,
                                         int rr) {
  return rr < ti.rows ? __ldg(perm + ti.row0 + rr) : 0;
}
__device__ __forceinline__ int perm_token(int f, int nK, int Kslots, bool &bad) {
  if ((unsigned)f < (unsigned)nK) return f / Kslots;
  bad = true;
  return 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// SiLU(g) = g / (1 + exp(-g)) with the fast exponential and divide (h is
// rounded to bf16 right after); the exponent is clamped so 1 + e stays finite.
__device__ __forceinline__ float silu(float g) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.f)));
}

// Epilogue staging: each epilogue warp puts its 32 rows x 32 columns (64 B per
// row) in shared memory, then stores them as whole 64-byte row segments, 8
// rows per store instruction.  Rows are 80 B apart so that both the row-wise
// writes and the segment-wise reads are (nearly) free of bank conflicts.

// my_dst: the output row of this lane's tile row (-1: do not store); the
// destination of tile row `row` is fetched from its lane.
__device__ __forceinline__ void store_tile_chunk(uint8_t *wbuf, const uint32_t (&pk)[16], int lane,
                                                 __nv_bfloat16 *out, size_t ld, int my_dst,
                                                 int rows, int col0) {
  uint4 *mine = reinterpret_cast<uint4 *>(wbuf + lane * EPI_ROW_BYTES);
#pragma unroll
  for (int v = 0; v < 4; ++v) mine[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = lane + 32 * i;
    const int row = p >> 2, c16 = p & 3;
    const int dst = __shfl_sync(0xffffffffu, my_dst, row);
    if (row < rows && dst >= 0) {
      const uint4 val = *reinterpret_cast<const uint4 *>(wbuf + row * EPI_ROW_BYTES + c16 * 16);
      *reinterpret_cast<uint4 *>(out + (size_t)dst * ld + col0 + c16 * 8) = val;
    }
  }
  __syncwarp();
}

// modes whose B is W13's gate/up column pairs (n-tile = 128 h columns)
__host__ __device__ constexpr bool gemm1_mode(int mode) {
  return mode == 1 || mode == 3 || mode == 6;
}
// mode 5: B stored n-major (rows n, k contiguous): a K-major UMMA operand
__host__ __device__ constexpr bool kmajor_b(int mode) { return mode == 5; }

// MODE 1: GEMM1 + SwiGLU (A = x_perm, B = W13, out = h, n-tile = 128 h columns)
// MODE 2: GEMM2          (A = h,      B = W2,  out = y_perm, n-tile = 256 columns)
// MODE 4: GEMM2 with the routing weight applied and the row scattered to its
//         (token, slot) position: out[perm[r]] = topk_w[perm[r]] * (h W2)[r],
//         so the combine reads each token's K rows as one contiguous block.
// MODE 3: GEMM1 + SwiGLU with the permute fused into the A loads: the A rows of
//         a tile are read straight from x (row perm[r] / K) by four gather
//         warps with 16-byte cp.async, written in the same 128-byte swizzled
//         layout the TMA produces; no x_perm exists.
//
// PAIR (modes 1, 2 and 4): clusters of two CTAs on two SMs compute 256-row x
// 256-column tiles with cta_group::2 MMAs.  The even CTA ("leader") issues the
// MMAs and owns the operand-full barriers: both CTAs' TMA copies complete on
// them, and it expects both CTAs' bytes.  Its MMA commits arrive on the
// operand-empty and accumulator-full barriers of both CTAs (multicast); both
// CTAs' epilogue warps arrive on the leader's accumulator-empty barriers.
// Each CTA drains the accumulator rows in its own TMEM.  Before the pair
// leaves, the leader settles every stage whose two halves were not both
// issued (a side that gave up early) and waits until every copy has landed.
template <int MODE, bool PAIR = false>
__global__ void __launch_bounds__(threads_for(MODE), 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const int32_t *__restrict__ offsets, int E, int nK, int Kdim, int I,
                           int Nout, __nv_bfloat16 *__restrict__ out, int32_t *status,
                           const int32_t *__restrict__ perm, int Kslots,
                           const __nv_bfloat16 *__restrict__ xg,
                           const float *__restrict__ tw,
                           const __nv_bfloat16 *__restrict__ aux, long long wait_limit,
                           int b_nb) {
  static_assert(!PAIR || MODE != 3, "CTA pairs: not with the cp.async gather of mode 3");
  using P = Pipe<PAIR>;
  constexpr int STAGES = P::STAGES;
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // single CTAs: A stages, then B stages; PAIR: B stages first, so that every
  // operand read of a stage stays inside the CTA's operand area
  uint8_t *smemA = PAIR ? smem + STAGES * P::B_STAGE : smem;
  uint8_t *smemB = PAIR ? smem : smem + STAGES * A_STAGE_BYTES;
  SmemTail &st = *reinterpret_cast<SmemTail *>(smem + STAGES * P::STAGE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = gemm1_mode(MODE) ? I / 128 : (Nout + UMMA_N - 1) / UMMA_N;
  const int KB = Kdim / BK;
  // PAIR: rank in the pair; tiles are dealt per pair
  const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
  const bool leader = rank == 0;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // MODE 3: the TMA producer's arrive (with the B bytes) + one completion
      // arrive per cp.async thread
      ptx::mbar_init(&st.full[s], MODE == 3 ? 1 + 32 * GATHER_WARPS : 1);
      ptx::mbar_init(&st.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&st.tfull[a], 1);
      ptx::mbar_init(&st.tempty[a], PAIR ? 8 : 4);  // the epilogue warps (of both CTAs)
    }
    ptx::mbar_init(&st.drain, 1);
    for (int s = 0; s < kMaxStages; ++s) st.own_issued[s] = st.peer_issued[s] = 0;
    st.abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  for (int c = tid; c <= E; c += NUM_THREADS) st.off[c] = offsets[c];
  // PAIR: both CTAs' barriers are initialised before either copies to or
  // arrives on the other's
  if constexpr (PAIR)
    ptx::cluster_sync();
  else
    __syncthreads();
  if (tid == 0) {
    bool ok = st.off[0] == 0 && st.off[E] <= nK;
    int run = 0;
    for (int e = 0; e < E; ++e) {
      const int len = st.off[e + 1] - st.off[e];
      ok = ok && len >= 0;
      st.tp[e] = run;
      run += len > 0 ? (len + P::TILE_ROWS - 1) / P::TILE_ROWS : 0;
    }
    st.tp[E] = run;
    st.total_mtiles = run;
    st.ok = ok;
    if (!ok && blockIdx.x == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
  }
  __syncthreads();
  // both CTAs of a pair read the same offsets, so they take the same exits
  if (!st.ok) return;
  const int total = st.total_mtiles * n_tiles;
  if (unit >= total) return;

  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(&st.tmem_base, TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&st.tmem_base, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = st.tmem_base;
  volatile int *abort_flag = &st.abort_flag;

  if (warp == 0 && PAIR) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB);
      // the leader's operand-full barriers, as shared::cluster addresses
      const uint32_t full0 = ptx::mapa_shared(ptx::smem_u32(&st.full[0]), 0);
      int stage = 0;
      uint32_t phase = 0;
      for (int t = unit; t < total; t += units) {
        const TileInfo ti = decode_tile<true>(st, t, n_tiles, E, rank);
        bool stop = false;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(&st.empty[stage], phase ^ 1u, abort_flag, status, wait_limit)) {
            stop = true;
            break;
          }
          if (leader) ptx::mbar_arrive_expect_tx(&st.full[stage], 2 * P::STAGE);
          const uint32_t bar = full0 + 8u * (uint32_t)stage;
          // a part with no rows of the expert (segment ends in the first
          // half) loads the expert's first rows: computed, never stored
          ptx::tma_load_2d_pair(smemA + stage * A_STAGE_BYTES, &tmA, bar, kb * BK,
                                ti.rows > 0 ? ti.row0 : st.off[ti.e]);
          if (kmajor_b(MODE)) {  // one box: 64 k x this CTA's 128 of the 256 n rows
            ptx::tma_load_3d_pair(smemB + stage * P::B_STAGE, &tmB, bar, kb * BK,
                                  ti.nt * UMMA_N + rank * (UMMA_N / 2), ti.e);
          } else {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            // this CTA's half of the 256 B columns: GEMM1 gate (rank 0) or up
            // (rank 1) columns of the 128 h columns; GEMM2 columns 128 * rank
            const int q = 2 * rank + j;
            const int ncol = gemm1_mode(MODE) ? (q < 2 ? 0 : I) + ti.nt * 128 + (q & 1) * 64
                                              : ti.nt * UMMA_N + q * 64;
            uint8_t *dst = smemB + stage * P::B_STAGE + j * B_BOX_BYTES;
            if (b_nb > 0)
              ptx::tma_load_2d_pair(dst, &tmB, bar, 0, ((ti.e * KB + kb) * b_nb + (ncol >> 6)) * 64);
            else
              ptx::tma_load_3d_pair(dst, &tmB, bar, ncol, kb * BK, ti.e);
          }
          }
          ++st.own_issued[stage];
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
      }
      // copies still in flight are settled by the leader before the pair
      // leaves: it needs the odd CTA's counts
      if (!leader) {
        const uint32_t dst0 = ptx::mapa_shared(ptx::smem_u32(&st.peer_issued[0]), 0);
        for (int s2 = 0; s2 < STAGES; ++s2)
          ptx::st_cluster_u32(dst0 + 4u * s2, (uint32_t)st.own_issued[s2]);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_par = 0;  // per stage: ever used, parity of last issue
      for (int t = unit; t < total; t += units) {
        const TileInfo ti = decode_tile(st, t, n_tiles, E);
        bool stop = false;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(&st.empty[stage], phase ^ 1u, abort_flag, status, wait_limit)) {
            stop = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(&st.full[stage], MODE == 3 ? P::B_STAGE : P::STAGE);
          if (MODE != 3)
            ptx::tma_load_2d(smemA + stage * A_STAGE_BYTES, &tmA, &st.full[stage], kb * BK,
                             ti.row0);
          if (kmajor_b(MODE)) {  // one box: 64 k x 256 n rows
            ptx::tma_load_3d(smemB + stage * P::B_STAGE, &tmB, &st.full[stage], kb * BK,
                             ti.nt * UMMA_N, ti.e);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              int ncol;
              if (gemm1_mode(MODE))
                ncol = (q < 2 ? 0 : I) + ti.nt * 128 + (q & 1) * 64;
              else
                ncol = ti.nt * UMMA_N + q * 64;
              uint8_t *dst = smemB + stage * P::B_STAGE + q * B_BOX_BYTES;
              if (b_nb > 0)  // tiled weights: the 64 x 64 tile is one contiguous run
                ptx::tma_load_2d(dst, &tmB, &st.full[stage], 0,
                                 ((ti.e * KB + kb) * b_nb + (ncol >> 6)) * 64);
              else
                ptx::tma_load_3d(dst, &tmB, &st.full[stage], ncol, kb * BK, ti.e);
            }
          }
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
      }
      // never leave a TMA copy in flight: wait for the last load of every stage
      for (int s = 0; s < STAGES; ++s)
        if (used >> s & 1u) ptx::mbar_wait(&st.full[s], last_par >> s & 1u);
    }
  } else if (warp == 1) {
    // PAIR: the leader alone issues the pair's MMAs
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = unit; t < total; t += units) {
        if (!wait_or_abort(&st.tempty[acc], acc_phase ^ 1u, abort_flag, status, wait_limit)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * UMMA_N);
        bool stop = false;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(&st.full[stage], phase, abort_flag, status, wait_limit)) {
            stop = true;
            break;
          }
          // MODE 3: A was written by cp.async (generic proxy); the barrier
          // made it visible to this thread, the proxy fence makes it visible
          // to the tensor cores' async-proxy reads issued below
          if (MODE == 3) ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smemA + stage * A_STAGE_BYTES);
          const uint32_t b0 = ptx::smem_u32(smemB + stage * P::B_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // A: K-major SW128, k step of 16 elements = 32 bytes inside the atom
            const uint64_t adesc = ptx::smem_desc(a0 + kk * 32, 16, 1024);
            // B: MN-major SW128, 64-wide n atoms 8 KB apart, k step = 16 rows;
            // or (mode 5) K-major SW128 like A, 256 n rows
            const uint64_t bdesc = kmajor_b(MODE) ? ptx::smem_desc(b0 + kk * 32, 16, 1024)
                                                  : ptx::smem_desc(b0 + kk * 2048, B_BOX_BYTES, 1024);
            // PAIR: each CTA's half of B is two of these atoms (128 n)
            if constexpr (PAIR)
              ptx::mma_bf16_pair(d, adesc, bdesc, kmajor_b(MODE) ? IDESC_PAIR_KB : IDESC_PAIR,
                                 (kb | kk) != 0 ? 1u : 0u);
            else
              ptx::mma_bf16(d, adesc, bdesc, kmajor_b(MODE) ? IDESC_KB : IDESC,
                            (kb | kk) != 0 ? 1u : 0u);
          }
          // the stage is free in both CTAs once these MMAs have read it
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
      // wait until every MMA this thread issued has finished
      if constexpr (PAIR)
        ptx::mma_commit_pair(&st.drain, 0x1);
      else
        ptx::mma_commit(&st.drain);
      ptx::mbar_wait(&st.drain, 0);
    }
  } else if (warp < 6) {
    // epilogue warps 2..5 -> TMEM lane quarter (warp % 4)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    // PAIR: the odd CTA's warps release the accumulator on the leader's barrier
    const uint32_t tempty0 = PAIR ? ptx::mapa_shared(ptx::smem_u32(&st.tempty[0]), 0) : 0u;
    for (int t = unit; t < total; t += units) {
      const TileInfo ti = decode_tile<PAIR>(st, t, n_tiles, E, rank);
      if (!wait_or_abort(&st.tfull[acc], acc_phase, abort_flag, status, wait_limit)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + (uint32_t)(acc * UMMA_N) + ((uint32_t)(q * 32) << 16);
      // rows of this warp's 32-row slice that belong to the tile's expert
      const int wrows = ti.rows - q * 32;
      const int wrow0 = ti.row0 + q * 32;
      uint8_t *wbuf = st.epi[q];
      // output row of this lane's tile row, and its routing weight (MODE 4)
      int my_dst = wrow0 + lane;
      float wscale = 1.f;
      if (MODE == 4) {
        my_dst = -1;
        if (lane < wrows) {
          const int f = __ldg(perm + wrow0 + lane);
          if ((unsigned)f < (unsigned)nK) {
            my_dst = f;
            wscale = __ldg(tw + f);
          } else {
            flag_status(status, MOE_DEV_BAD_LAYOUT);
          }
        }
      }
      if (gemm1_mode(MODE)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32x32b_x32(tbase + c * 32, g);
          ptx::tmem_ld_32x32b_x32(tbase + 128 + c * 32, u);
          ptx::tmem_ld_wait();
          const int col = ti.nt * 128 + c * 32;
          if (MODE == 6) {
            // SwiGLU backward: dG = dh U s (1 + G (1 - s)), dU = dh G s, s = sigmoid(G)
            float dh[32];
            if (lane < wrows) {
              const uint4 *src = reinterpret_cast<const uint4 *>(aux + (size_t)(wrow0 + lane) * I + col);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint4 q4 = __ldg(src + v);
                const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&q4);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const float2 f = __bfloat1622float2(b2[j]);
                  dh[8 * v + 2 * j] = f.x;
                  dh[8 * v + 2 * j + 1] = f.y;
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) dh[i] = 0.f;
            }
            uint32_t pg[16], pu[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float dg[2], du[2];
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const float gv = __uint_as_float(g[2 * i + j]), uv = __uint_as_float(u[2 * i + j]);
                const float sg = __fdividef(1.f, 1.f + __expf(fminf(-gv, 80.f)));
                const float d = dh[2 * i + j];
                dg[j] = d * uv * sg * (1.f + gv * (1.f - sg));
                du[j] = d * gv * sg;
              }
              pg[i] = pack_bf16x2(dg[0], dg[1]);
              pu[i] = pack_bf16x2(du[0], du[1]);
            }
            store_tile_chunk(wbuf, pg, lane, out, (size_t)Nout, my_dst, wrows, col);
            store_tile_chunk(wbuf, pu, lane, out, (size_t)Nout, my_dst, wrows, I + col);
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
              pk[i] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
            }
            store_tile_chunk(wbuf, pk, lane, out, (size_t)I, my_dst, wrows, col);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < UMMA_N / 32; ++c) {
          if (ti.nt * UMMA_N + c * 32 >= Nout) break;  // uniform across the warp
          uint32_t a[32];
          ptx::tmem_ld_32x32b_x32(tbase + c * 32, a);
          ptx::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0 = __uint_as_float(a[2 * i]), a1 = __uint_as_float(a[2 * i + 1]);
            if (MODE == 4) {
              a0 *= wscale;
              a1 *= wscale;
            }
            pk[i] = pack_bf16x2(a0, a1);
          }
          store_tile_chunk(wbuf, pk, lane, out, (size_t)Nout, my_dst, wrows,
                           ti.nt * UMMA_N + c * 32);
        }
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
  } else if (MODE == 3) {
    // cp.async gatherers: warp g fills tile rows [32g, 32g + 32).  Lane =
    // 8 * sub + chunk moves 16-byte chunk `chunk` of rows 32g + 4i + sub
    // (i = 0..7), so one warp instruction copies four whole 128-byte row
    // segments.  The chunk lands where the TMA's 128-byte swizzle puts it:
    // chunk c of row r at r * 128 + ((c ^ (r % 8)) * 16).  Every thread's
    // copies of a stage end in a completion arrive on that stage's full
    // barrier.  Perm entries of the next tile are loaded while the current
    // tile streams.
    const int g = warp - 6;
    const int sub = lane >> 3, chunk = lane & 7;
    const uint32_t a_base = ptx::smem_u32(smemA);
    int stage = 0;
    uint32_t phase = 0;
    bool bad = false;
    int fnext[8];
    {
      const TileInfo t0 = decode_tile(st, blockIdx.x, n_tiles, E);
#pragma unroll
      for (int i = 0; i < 8; ++i) fnext[i] = tile_perm(perm, t0, g * 32 + i * 4 + sub);
    }
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const __nv_bfloat16 *src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        src[i] = xg + (size_t)perm_token(fnext[i], nK, Kslots, bad) * Kdim + chunk * 8;
      if (t + (int)gridDim.x < total) {
        const TileInfo tn = decode_tile(st, t + gridDim.x, n_tiles, E);
#pragma unroll
        for (int i = 0; i < 8; ++i) fnext[i] = tile_perm(perm, tn, g * 32 + i * 4 + sub);
      }
      bool stop = false;
      for (int kb = 0; kb < KB; ++kb) {
        int ok = 1;
        if (lane == 0) ok = wait_or_abort(&st.empty[stage], phase ^ 1u, abort_flag, status, wait_limit);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        const uint32_t sb = a_base + stage * A_STAGE_BYTES;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = g * 32 + i * 4 + sub;
          ptx::cp_async_cg16(sb + rr * 128 + ((chunk ^ (rr & 7)) << 4), src[i] + kb * BK);
        }
        ptx::cp_async_arrive_noinc(&st.full[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (stop) break;
    }
    ptx::cp_async_wait<0>();  // no copy stays in flight
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, MOE_DEV_BAD_LAYOUT);
  }

  ptx::tc_fence_before();
  __syncwarp();
  if constexpr (PAIR) {
    // every role of both CTAs is done (the leader's MMAs have completed) and
    // the odd CTA's load counts are in the leader
    ptx::cluster_sync();
    if (leader && tid == 0) {
      // Both producers follow the same empty barriers, so per stage their
      // counts differ by at most one phase when one side gave up early: the
      // leader completes that last phase for the side that never came (its
      // bytes, or its own arrival), then waits until every copy has landed.
      for (int s = 0; s < STAGES; ++s) {
        const int own = st.own_issued[s], peer = st.peer_issued[s];
        if (own == peer + 1)
          ptx::mbar_complete_tx(&st.full[s], P::STAGE);
        else if (peer == own + 1)
          ptx::mbar_arrive_expect_tx(&st.full[s], P::STAGE);
        const int last = own > peer ? own : peer;
        if (last > 0) ptx::mbar_wait(&st.full[s], (uint32_t)(last - 1) & 1u);
      }
    }
    // no copy into either CTA is still in flight
    ptx::cluster_sync();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    __syncwarp();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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

bool make_map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = get_encode_fn();
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

bool make_map_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint32_t b0, uint32_t b1) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B operand map of the expert weights w (E matrices of rows x cols, bf16) for
// 64 x 64 boxes: a 3-D map over the row-major matrices, or, for tiled weights
// (moe_prepare_weights), a 2-D map over the contiguous 64 x 64 tiles (64
// columns, one 64-row box per tile).  *b_nb: tiles per tile row (cols / 64)
// for tiled weights, 0 otherwise (the kernel's b_nb argument).
bool weight_map(CUtensorMap *m, const void *w, const Desc &d, uint64_t rows, uint64_t cols,
                int *b_nb) {
  if (d.tiled) {
    *b_nb = (int)(cols / 64);
    return make_map_2d(m, w, 64, (uint64_t)d.E * rows * (cols / 64), 64, BK);
  }
  *b_nb = 0;
  return make_map_3d(m, w, cols, rows, d.E, 64, BK);
}

template <int MODE, bool PAIR = false>
cudaError_t set_smem_attr() {
  static int done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc_kernel<MODE, PAIR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bytes<PAIR>());
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

int gemm_grid(int sm_reserve) {
  const int g = device_sm_count() - (sm_reserve > 0 ? sm_reserve : 0);
  return g < 1 ? 1 : g;
}

// 0: CTA pairs for the grouped GEMMs (all modes but 3), 1: single CTAs
// (moe_set_gemm_pairs)
std::atomic<int> g_single_cta{0};

// CTA pairs of MODE's kernel that can be resident at once (cached per device)
template <int MODE>
cudaError_t pair_clusters(int *out) {
  static int cached[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!cached[dev]) {
    e = set_smem_attr<MODE, true>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 16);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem_bytes<true>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    e = cudaOccupancyMaxActiveClusters(&nc, grouped_gemm_tc_kernel<MODE, true>, &cfg);
    if (e != cudaSuccess) return e;
    if (nc < 1) return cudaErrorInvalidConfiguration;
    cached[dev] = nc;
  }
  *out = cached[dev];
  return cudaSuccess;
}

// Persistent launch of a grouped GEMM: one CTA per SM, or (pairs) as many CTA
// pairs as are resident at once within the SMs sm_reserve leaves.
template <int MODE, typename... Args>
cudaError_t launch_gemm(bool pair, int sm_reserve, cudaStream_t s, Args &&...args) {
  if (!pair) {
    cudaError_t e = set_smem_attr<MODE>();
    if (e != cudaSuccess) return e;
    return launch_pdl(grouped_gemm_tc_kernel<MODE>, dim3(gemm_grid(sm_reserve)),
                      dim3(NUM_THREADS), SMEM_BYTES, s, static_cast<Args &&>(args)...);
  }
  int nc = 0;
  cudaError_t e = pair_clusters<MODE>(&nc);
  if (e != cudaSuccess) return e;
  const int avail = gemm_grid(sm_reserve) / 2;
  if (avail < nc) nc = avail < 1 ? 1 : avail;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * nc);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes<true>();
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<MODE, true>,
                            static_cast<Args &&>(args)...);
}

}  // namespace

void set_gemm_single_cta(bool single) { g_single_cta.store(single ? 1 : 0); }
bool gemm_single_cta() { return g_single_cta.load() != 0; }

cudaError_t launch_gemm1_tc(const Desc &d, const void *x_perm, const void *w13,
                            const int32_t *offsets, void *h, int sm_reserve, int32_t *status,
                            cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  int BNB = 0;
  if (!make_map_2d(&mA, x_perm, d.H, nK, BK, BM) || !weight_map(&mB, w13, d, d.H, 2ull * d.I, &BNB))
    return cudaErrorInvalidValue;
  return launch_gemm<1>(!gemm_single_cta(), sm_reserve, s, mA, mB, offsets, d.E, (int)nK, d.H, d.I, d.I,
                                reinterpret_cast<__nv_bfloat16 *>(h), status,
                                (const int32_t *)nullptr, 0, (const __nv_bfloat16 *)nullptr,
                                (const float *)nullptr, (const __nv_bfloat16 *)nullptr,
                                pipeline_wait_limit(), BNB);
}

cudaError_t launch_gemm1_tc_gather(const Desc &d, const void *x, const int32_t *perm,
                                   const void *w13, const int32_t *offsets, void *h,
                                   int sm_reserve, int32_t *status, cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mB;  // A is gathered with cp.async: no tensor map for x
  int BNB = 0;
  if (!weight_map(&mB, w13, d, d.H, 2ull * d.I, &BNB)) return cudaErrorInvalidValue;
  cudaError_t e = set_smem_attr<3>();
  if (e != cudaSuccess) return e;
  return launch_pdl(grouped_gemm_tc_kernel<3>, dim3(gemm_grid(sm_reserve)), dim3(threads_for(3)),
                    SMEM_BYTES, s, mB, mB, offsets, d.E, (int)nK, d.H, d.I, d.I,
                    reinterpret_cast<__nv_bfloat16 *>(h), status, perm, d.K,
                    reinterpret_cast<const __nv_bfloat16 *>(x), nullptr, nullptr, pipeline_wait_limit(), BNB);
}

cudaError_t launch_gemm2_tc(const Desc &d, const void *h, const void *w2, const int32_t *offsets,
                            void *y_perm, int sm_reserve, int32_t *status, cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  int BNB = 0;
  if (!make_map_2d(&mA, h, d.I, nK, BK, BM) || !weight_map(&mB, w2, d, d.I, d.H, &BNB))
    return cudaErrorInvalidValue;
  return launch_gemm<2>(!gemm_single_cta(), sm_reserve, s, mA, mB, offsets, d.E, (int)nK, d.I, d.I, d.H,
                                reinterpret_cast<__nv_bfloat16 *>(y_perm), status,
                                (const int32_t *)nullptr, 0, (const __nv_bfloat16 *)nullptr,
                                (const float *)nullptr, (const __nv_bfloat16 *)nullptr,
                                pipeline_wait_limit(), BNB);
}

cudaError_t launch_gemm2_tc_weighted(const Desc &d, const void *h, const void *w2,
                                     const int32_t *offsets, const int32_t *perm,
                                     const float *topk_w, void *y_slot, int sm_reserve,
                                     int32_t *status, cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  int BNB = 0;
  if (!make_map_2d(&mA, h, d.I, nK, BK, BM) || !weight_map(&mB, w2, d, d.I, d.H, &BNB))
    return cudaErrorInvalidValue;
  return launch_gemm<4>(!gemm_single_cta(), sm_reserve, s, mA, mB, offsets, d.E, (int)nK, d.I, d.I, d.H,
                                reinterpret_cast<__nv_bfloat16 *>(y_slot), status, perm, d.K,
                                (const __nv_bfloat16 *)nullptr, topk_w,
                                (const __nv_bfloat16 *)nullptr, pipeline_wait_limit(), BNB);
}

cudaError_t launch_gemm_dgrad_tc(const Desc &d, const void *a, const void *w, int Kdim, int Nout,
                                 const int32_t *offsets, void *out, int32_t *status,
                                 cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  // A (nK, Kdim) K-major; W[e] (Nout, Kdim): rows n with k contiguous, one box
  // of 256 n rows per stage (CTA pairs: each CTA's 128)
  const bool pair = !gemm_single_cta();  // read once: the box and the kernel must agree
  const uint32_t box_n = pair ? UMMA_N / 2 : UMMA_N;
  if (!make_map_2d(&mA, a, Kdim, nK, BK, BM) ||
      !make_map_3d(&mB, w, Kdim, Nout, d.E, BK, box_n))
    return cudaErrorInvalidValue;
  return launch_gemm<5>(pair, 0, s, mA, mB, offsets, d.E, (int)nK, Kdim, 0, Nout,
                        reinterpret_cast<__nv_bfloat16 *>(out), status, (const int32_t *)nullptr,
                        0, (const __nv_bfloat16 *)nullptr, (const float *)nullptr,
                        (const __nv_bfloat16 *)nullptr, pipeline_wait_limit(), 0);
}

cudaError_t launch_gemm1_swiglu_bwd_tc(const Desc &d, const void *x_perm, const void *w13,
                                       const int32_t *offsets, const void *dh, void *dgu,
                                       int32_t *status, cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  if (!make_map_2d(&mA, x_perm, d.H, nK, BK, BM) ||
      !make_map_3d(&mB, w13, 2ull * d.I, d.H, d.E, 64, BK))
    return cudaErrorInvalidValue;
  return launch_gemm<6>(!gemm_single_cta(), 0, s, mA, mB, offsets, d.E, (int)nK, d.H, d.I, 2 * d.I,
                        reinterpret_cast<__nv_bfloat16 *>(dgu), status, (const int32_t *)nullptr,
                        0, (const __nv_bfloat16 *)nullptr, (const float *)nullptr,
                        reinterpret_cast<const __nv_bfloat16 *>(dh), pipeline_wait_limit(), 0);
}

}  // namespace moe
