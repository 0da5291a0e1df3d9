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
// (two B boxes), six 32 KB stages (see the kernel's comment for the protocol);
// in the forward modes optionally with fused tails (TAILS: an expert's last
// 1..32 rows computed transposed inside its last full window's tiles).
// A tile is (m-tile, n-tile).  m-tiles are 128-row windows (256 for a pair)
// that start at each expert's segment start, so every tile belongs to exactly
// one expert; its rows past the segment end are computed but not stored (TMA
// zero-fills rows past the tensor).  Tiles are dealt to CTAs (pairs)
// round-robin in expert order (the fused-tail GEMM1 walks the experts that
// fuse a tail first); a tile without a tail costs a full K loop, so the static
// schedule balances.  Each tile is computed entirely by one CTA (pair) with a
// fixed k order: results do not depend on the grid size.
//
// B is the weight matrix as stored (k rows, n contiguous): an MN-major UMMA
// operand with 128-byte swizzle (or, tiled by moe_prepare_weights, one 64 x 64
// tile per box).  A is K-major with 128-byte swizzle.
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
// epilogue staging per warp: 32 rows of 80 B (bf16 output rows)
constexpr int EPI_ROW_BYTES = 80, EPI_WARP_BYTES = 32 * EPI_ROW_BYTES;
// GEMM1 tails: a gate warp's 32 x 32 SiLU values for its up warp, 144-byte rows
constexpr int XCH_ROW_BYTES = 144, XCH_WARP_BYTES = 32 * XCH_ROW_BYTES;

// Fused tails (CTA pairs, forward modes 1, 2 and 4).  An expert whose
// segment ends 1..TAIL_ROWS rows past a 256-row window boundary, after at
// least one full window, computes those rows inside its last full window's
// tiles, transposed: in every k stage, beside the tile's 256 x 256 MMAs, the
// leader issues M = 256, N = TAIL_ROWS MMAs that take the same weight columns
// (each CTA's 128, MN-major) as A and the tail rows (TAIL_HALF per CTA,
// K-major) as B, accumulating D^T into the first TAIL_ROWS columns of the
// other TMEM accumulator.  The tail adds MMAs (an N = 32 MMA takes about
// 0.4 of an N = 256 one: it reads the same A) but no weight traffic, where a
// window of its own would repeat the whole tile.  The epilogue releases each
// accumulator's first TAIL_ROWS columns (its "head") apart from the rest, as
// soon as it has read them, and drains a tail before its tile's own
// accumulator, so a tile with a tail waits only for the head of the other
// accumulator.  A kernel variant (TAILS); launches choose it by the layer's
// rows per expert (tails_auto).
constexpr int TAIL_ROWS = 32, TAIL_HALF = TAIL_ROWS / 2;
constexpr int TAIL_BYTES = TAIL_HALF * BK * 2;  // 2 KB per CTA and stage
__host__ __device__ constexpr bool tail_mode(int mode) {
  return mode == 1 || mode == 2 || mode == 4;
}
// compile-time flag for the k loops specialised on "this tile has a tail"
template <bool B>
struct BoolC {
  static constexpr bool value = B;
};

struct SmemTail {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t hempty[2];  // TAILS: columns [0, TAIL_ROWS) of the accumulator read
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ok;
  int total_mtiles;
  int own_issued[kMaxStages];   // PAIR: phases this CTA's producer loaded, per stage
  int own_bytes[kMaxStages];    // PAIR: bytes per CTA of the last phase loaded, per stage
  int peer_issued[kMaxStages];  // PAIR (leader): the odd CTA's own_issued
  int peer_bytes[kMaxStages];   // PAIR (leader): the odd CTA's own_bytes
  int epi_ok[4];                // GEMM1 tails: each epilogue warp's go-ahead
  int off[kMaxE + 1];
  int tp[kMaxE + 1];  // first m-tile of each expert (exclusive prefix)
  alignas(16) uint8_t epi[4][EPI_WARP_BYTES];  // per epilogue warp staging
};

// TAILS: the stages are followed by a TAIL_BYTES slot per stage for the fused
// tail rows, the two gate warps' exchange buffers and the expert order
// the order in which the fused-tail variant walks the experts (uint16 each)
constexpr int ORD_BYTES = ((kMaxE + 1) * 2 + 15) / 16 * 16;
template <bool PAIR, bool TAILS = false>
__host__ __device__ constexpr size_t tails_bytes() {
  return TAILS ? (size_t)Pipe<PAIR>::STAGES * TAIL_BYTES + 2 * XCH_WARP_BYTES + ORD_BYTES : 0;
}
template <bool PAIR, bool TAILS = false>
constexpr size_t smem_bytes() {
  return 1024 /*alignment slack*/ + (size_t)Pipe<PAIR>::STAGES * Pipe<PAIR>::STAGE +
         tails_bytes<PAIR, TAILS>() + sizeof(SmemTail);
}
constexpr size_t SMEM_BYTES = smem_bytes<false>();
static_assert(smem_bytes<true, true>() <= 227 * 1024, "pair pipeline exceeds shared memory");

constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/true);
constexpr uint32_t IDESC_KB = ptx::idesc_bf16_f32(BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/false);
constexpr uint32_t IDESC_PAIR = ptx::idesc_bf16_f32(2 * BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/true);
constexpr uint32_t IDESC_PAIR_KB = ptx::idesc_bf16_f32(2 * BM, UMMA_N, /*a_mn=*/false, /*b_mn=*/false);
// fused tail: A = the weight columns (MN-major), B = the tail rows (K-major)
constexpr uint32_t IDESC_TAIL = ptx::idesc_bf16_f32(2 * BM, TAIL_ROWS, /*a_mn=*/true, /*b_mn=*/false);

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
  int tail, t0;  // fused tail: its rows (0: none) and first row
};

// TAILS: the expert's rows past its last full window (1..TAIL_ROWS of them)
// are fused into that window's tiles
template <bool PAIR, bool TAILS>
__host__ __device__ constexpr bool fused_tail(int len) {
  return PAIR && TAILS && len > Pipe<PAIR>::TILE_ROWS && len % Pipe<PAIR>::TILE_ROWS != 0 &&
         len % Pipe<PAIR>::TILE_ROWS <= TAIL_ROWS;
}
// m-tiles of an expert with len rows
template <bool PAIR, bool TAILS>
__host__ __device__ constexpr int mtiles_of(int len) {
  return len > 0 ? (len + Pipe<PAIR>::TILE_ROWS - 1) / Pipe<PAIR>::TILE_ROWS -
                       (fused_tail<PAIR, TAILS>(len) ? 1 : 0)
                 : 0;
}

// Tile t: expert, first row and stored rows of this CTA's 128-row part
// (PAIR: rank 0 takes rows [0, 128) of the pair's 256-row window, rank 1 rows
// [128, 256); rows may be <= 0 when the segment ends in the first half).
template <bool PAIR = false, bool TAILS = false>
// ord (TAILS): the expert at each position of the walk; tp is per position.
__device__ __forceinline__ TileInfo decode_tile(const SmemTail &s, int t, int n_tiles, int E,
                                                int rank = 0, const uint16_t *ord = nullptr) {
  TileInfo ti;
  const int mt = t / n_tiles;
  ti.nt = t - mt * n_tiles;
  int lo = 0, hi = E;  // largest position p with tp[p] <= mt
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tp[mid] <= mt)
      lo = mid;
    else
      hi = mid;
  }
  const int j = mt - s.tp[lo];
  const int e = (TAILS && ord) ? (int)ord[lo] : lo;
  ti.e = e;
  const int w0 = s.off[e] + j * Pipe<PAIR>::TILE_ROWS;
  ti.row0 = w0 + rank * BM;
  const int left = s.off[e + 1] - ti.row0;
  ti.rows = left < BM ? left : BM;
  ti.tail = 0;
  ti.t0 = 0;
  if constexpr (PAIR && TAILS) {
    const int len = s.off[e + 1] - s.off[e];
    if (fused_tail<PAIR, TAILS>(len) && j == len / Pipe<PAIR>::TILE_ROWS - 1) {
      ti.t0 = w0 + Pipe<PAIR>::TILE_ROWS;
      ti.tail = s.off[e + 1] - ti.t0;
    }
  }
  return ti;
}

// Barrier of the gate warp q and the up warp q + 2 (q = 0, 1) in a GEMM1
// tail's epilogue: named barrier 1 or 2, 64 threads.
__device__ __forceinline__ void epi_pair_bar(int q) {
  if (q & 1)
    ptx::named_bar_sync<2, 64>();
  else
    ptx::named_bar_sync<1, 64>();
}


// One epilogue warp's arrival (lane 0) on accumulator barrier bars[a]; the odd
// CTA of a pair arrives on the leader's (remote0: its bars[0] in the cluster).
__device__ __forceinline__ void epi_arrive(uint64_t *bars, uint32_t remote0, int a, bool remote) {
  if (remote)
    ptx::mbar_arrive_cluster(remote0 + 8u * (uint32_t)a);
  else
    ptx::mbar_arrive(&bars[a]);
}
// The warp has read accumulator a's head (its first TAIL_ROWS columns).  The
// arrival is relaxed: the reads are complete (tcgen05.wait::ld) and ordered
// before it (tcgen05.fence::before_thread_sync), and no memory write of the
// warp needs to reach the waiting MMA issuer.
__device__ __forceinline__ void head_release(uint64_t *bars, uint32_t remote0, int a, bool remote,
                                             int lane) {
  ptx::tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (remote)
      ptx::mbar_arrive_cluster_relaxed(remote0 + 8u * (uint32_t)a);
    else
      ptx::mbar_arrive_relaxed(&bars[a]);
  }
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
// Stores the staged 32 rows x 64 B: row r goes to out[dst of lane r] at col0.
__device__ __forceinline__ void store_staged(const uint8_t *wbuf, int lane, __nv_bfloat16 *out,
                                             size_t ld, int my_dst, int rows, int col0) {
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

__device__ __forceinline__ void store_tile_chunk(uint8_t *wbuf, const uint32_t (&pk)[16], int lane,
                                                 __nv_bfloat16 *out, size_t ld, int my_dst,
                                                 int rows, int col0) {
  uint4 *mine = reinterpret_cast<uint4 *>(wbuf + lane * EPI_ROW_BYTES);
#pragma unroll
  for (int v = 0; v < 4; ++v) mine[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
  __syncwarp();
  store_staged(wbuf, lane, out, ld, my_dst, rows, col0);
}

// Fused tails: this lane holds one output column (col0 + lane) for 32
// consecutive rows; staged as row i = those rows' 32 columns, then stored
// like a row-major chunk.
__device__ __forceinline__ void store_tile_chunk_t(uint8_t *wbuf, const float (&v)[32], int lane,
                                                   __nv_bfloat16 *out, size_t ld, int my_dst,
                                                   int rows, int col0) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    *reinterpret_cast<__nv_bfloat16 *>(wbuf + i * EPI_ROW_BYTES + lane * 2) = __float2bfloat16_rn(v[i]);
  __syncwarp();
  store_staged(wbuf, lane, out, ld, my_dst, rows, col0);
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
template <int MODE, bool PAIR = false, bool TAILS = false>
__global__ void __launch_bounds__(threads_for(MODE), 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmA2,
                           const int32_t *__restrict__ offsets, int E, int nK, int Kdim, int I,
                           int Nout, __nv_bfloat16 *__restrict__ out, int32_t *status,
                           const int32_t *__restrict__ perm, int Kslots,
                           const __nv_bfloat16 *__restrict__ xg,
                           const float *__restrict__ tw,
                           const __nv_bfloat16 *__restrict__ aux, long long wait_limit,
                           int b_nb) {
  static_assert(!PAIR || MODE != 3, "CTA pairs: not with the cp.async gather of mode 3");
  static_assert(!TAILS || (PAIR && tail_mode(MODE)), "fused tails: CTA pairs, forward modes");
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
  uint8_t *smemT = smem + STAGES * P::STAGE;  // TAILS: the fused tail rows, per stage
  uint8_t *xch = smemT + STAGES * TAIL_BYTES;  // TAILS: the gate warps' exchange buffers
  // TAILS: the experts in walk order.  GEMM1 takes those with a fused tail
  // first, so their heavier tiles are dealt evenly over the pairs (measured:
  // DeepSeek-V3-sized GEMM1 3.01 -> 2.77 ms); GEMM2, whose tiles are half as
  // long, keeps the index order (fused-first measured 3 % slower there).
  uint16_t *ord = TAILS ? reinterpret_cast<uint16_t *>(xch + 2 * XCH_WARP_BYTES) : nullptr;
  constexpr bool FUSED_FIRST = TAILS && MODE == 1;
  SmemTail &st = *reinterpret_cast<SmemTail *>(smemT + tails_bytes<PAIR, TAILS>());
  // PAIR, GEMM1: each CTA's half of the weight tile is 64 gate columns and the
  // 64 matching up columns (a tail's SwiGLU then stays inside the CTA)
  constexpr bool SPLIT_GU = PAIR && MODE == 1;

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
      ptx::mbar_init(&st.hempty[a], PAIR ? 8 : 4);
    }
    ptx::mbar_init(&st.drain, 1);
    for (int s = 0; s < kMaxStages; ++s)
      st.own_issued[s] = st.peer_issued[s] = st.own_bytes[s] = st.peer_bytes[s] = 0;
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
    if constexpr (TAILS) {
      for (int e = 0; e < E; ++e) ok = ok && st.off[e + 1] - st.off[e] >= 0;
      int pos = 0;
      for (int pass = FUSED_FIRST ? 0 : 1; pass < 2; ++pass)
        for (int e = 0; e < E; ++e) {
          const int len = st.off[e + 1] - st.off[e];
          if (ok && (!FUSED_FIRST || fused_tail<PAIR, TAILS>(len) == (pass == 0))) {
            ord[pos] = (uint16_t)e;
            st.tp[pos++] = run;
            run += mtiles_of<PAIR, TAILS>(len);
          }
        }
    } else {
      for (int e = 0; e < E; ++e) {
        const int len = st.off[e + 1] - st.off[e];
        ok = ok && len >= 0;
        st.tp[e] = run;
        run += mtiles_of<PAIR, TAILS>(len);
      }
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
      if (TAILS) ptx::prefetch_tmap(&tmA2);
      // the leader's operand-full barriers, as shared::cluster addresses
      const uint32_t full0 = ptx::mapa_shared(ptx::smem_u32(&st.full[0]), 0);
      int stage = 0;
      uint32_t phase = 0;
      for (int t = unit; t < total; t += units) {
        const TileInfo ti = decode_tile<true, TAILS>(st, t, n_tiles, E, rank, ord);
        // the k loop, compiled apart for tiles with a fused tail (TL): the
        // per-stage path of the others stays as short as without tails
        auto k_loop = [&](auto tl) {
          constexpr bool TL = decltype(tl)::value;
          constexpr int bytes = P::STAGE + (TL ? TAIL_BYTES : 0);  // per CTA and stage
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(&st.empty[stage], phase ^ 1u, abort_flag, status, wait_limit))
            return true;
          if (leader) ptx::mbar_arrive_expect_tx(&st.full[stage], 2 * bytes);
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
            // this CTA's half of the 256 B columns: GEMM1 (mode 1) 64 gate and
            // the 64 matching up columns, (mode 6) the gate (rank 0) or up
            // (rank 1) columns of the 128 h columns; GEMM2 columns 128 * rank
            const int q = 2 * rank + j;
            const int ncol = SPLIT_GU ? j * I + ti.nt * 128 + rank * 64
                             : gemm1_mode(MODE) ? (q < 2 ? 0 : I) + ti.nt * 128 + (q & 1) * 64
                                                : ti.nt * UMMA_N + q * 64;
            uint8_t *dst = smemB + stage * P::B_STAGE + j * B_BOX_BYTES;
            if (b_nb > 0)
              ptx::tma_load_2d_pair(dst, &tmB, bar, 0, ((ti.e * KB + kb) * b_nb + (ncol >> 6)) * 64);
            else
              ptx::tma_load_3d_pair(dst, &tmB, bar, ncol, kb * BK, ti.e);
          }
          }
          // fused tail: this CTA's TAIL_HALF of the tail rows (rows past the
          // tensor read zeros; rows of the next expert are never stored)
          if constexpr (TL)
            ptx::tma_load_2d_pair(smemT + stage * TAIL_BYTES, &tmA2, bar, kb * BK,
                                  ti.t0 + rank * TAIL_HALF);
          ++st.own_issued[stage];
          st.own_bytes[stage] = bytes;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
          return false;
        };
        const bool stop = ti.tail ? k_loop(BoolC<TAILS>{}) : k_loop(BoolC<false>{});
        if (stop) break;
      }
      // copies still in flight are settled by the leader before the pair
      // leaves: it needs the odd CTA's counts
      if (!leader) {
        const uint32_t dst0 = ptx::mapa_shared(ptx::smem_u32(&st.peer_issued[0]), 0);
        const uint32_t dstb = ptx::mapa_shared(ptx::smem_u32(&st.peer_bytes[0]), 0);
        for (int s2 = 0; s2 < STAGES; ++s2) {
          ptx::st_cluster_u32(dst0 + 4u * s2, (uint32_t)st.own_issued[s2]);
          ptx::st_cluster_u32(dstb + 4u * s2, (uint32_t)st.own_bytes[s2]);
        }
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
      // bit a: parity of the uses so far of accumulator a (uses: use u waits
      // for the epilogue's release u - 1), and of the waits for its head's
      // releases (huses)
      uint32_t uses = 0, huses = 0;
      bool prev_tail = false;  // the previous tile put a tail in this tile's head
      constexpr uint32_t idesc = PAIR ? (kmajor_b(MODE) ? IDESC_PAIR_KB : IDESC_PAIR)
                                      : (kmajor_b(MODE) ? IDESC_KB : IDESC);
      int p_cur = 0;  // walk position of the current tile's expert (tiles come in order)
      for (int t = unit; t < total; t += units) {
        bool tail = false;
        if constexpr (TAILS) {
          const int mt = t / n_tiles;
          while (p_cur + 1 < E && st.tp[p_cur + 1] <= mt) ++p_cur;
          const int e = ord[p_cur];
          const int len = st.off[e + 1] - st.off[e];
          tail = fused_tail<PAIR, TAILS>(len) && mt - st.tp[p_cur] == len / P::TILE_ROWS - 1;
        }
        if (!wait_or_abort(&st.tempty[acc], (uses >> acc & 1u) ^ 1u, abort_flag, status,
                           wait_limit))
          break;
        uses ^= 1u << acc;
        // Head releases come only around tails, each with one wait here: the
        // drain of a tail releases the head it used (awaited by the next
        // tile, whose accumulator that is), and the drain of a tile followed
        // by a tile with a tail releases its own head after its first chunk
        // (awaited by that tile, whose tail goes there).  The whole-accumulator
        // release covers every other case.
        if (TAILS && prev_tail) {
          if (!wait_or_abort(&st.hempty[acc], huses >> acc & 1u, abort_flag, status, wait_limit))
            break;
          huses ^= 1u << acc;
        }
        // the tail's D^T goes to the other accumulator's head (free before the
        // unit's first tile)
        if (TAILS && tail && t != unit) {
          if (!wait_or_abort(&st.hempty[acc ^ 1], huses >> (acc ^ 1) & 1u, abort_flag, status,
                             wait_limit))
            break;
          huses ^= 1u << (acc ^ 1);
        }
        prev_tail = tail;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * UMMA_N);
        const uint32_t dt = tmem + (uint32_t)((acc ^ 1) * UMMA_N);  // the tail's D^T
        // the k loop, compiled apart for tiles with a fused tail (TL)
        auto k_loop = [&](auto tl) {
          constexpr bool TL = decltype(tl)::value;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_or_abort(&st.full[stage], phase, abort_flag, status, wait_limit)) return true;
          // MODE 3: A was written by cp.async (generic proxy); the barrier
          // made it visible to this thread, the proxy fence makes it visible
          // to the tensor cores' async-proxy reads issued below
          if (MODE == 3) ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smemA + stage * A_STAGE_BYTES);
          const uint32_t b0 = ptx::smem_u32(smemB + stage * P::B_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // the activation rows: K-major SW128, k step of 16 elements = 32
            // bytes inside the atom
            const uint64_t xdesc = ptx::smem_desc(a0 + kk * 32, 16, 1024);
            // the weights: MN-major SW128, 64-wide n atoms 8 KB apart, k step
            // = 16 rows; or (mode 5) K-major SW128 like the rows, 256 n rows
            const uint64_t wdesc = kmajor_b(MODE) ? ptx::smem_desc(b0 + kk * 32, 16, 1024)
                                                  : ptx::smem_desc(b0 + kk * 2048, B_BOX_BYTES, 1024);
            // PAIR: each CTA's half of the weights is two of these atoms (128 n)
            if constexpr (PAIR)
              ptx::mma_bf16_pair(d, xdesc, wdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
            else
              ptx::mma_bf16(d, xdesc, wdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          if constexpr (TL) {
            // the same weight atoms as the 256-row A operand (MN-major), the
            // tail rows (TAIL_HALF per CTA, K-major) as a TAIL_ROWS-column B
            const uint32_t r0 = ptx::smem_u32(smemT + stage * TAIL_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              ptx::mma_bf16_pair(dt, ptx::smem_desc(b0 + kk * 2048, B_BOX_BYTES, 1024),
                                 ptx::smem_desc(r0 + kk * 32, 16, 1024), IDESC_TAIL,
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
          return false;
        };
        const bool stop = tail ? k_loop(BoolC<TAILS>{}) : k_loop(BoolC<false>{});
        if (stop) break;
        if constexpr (PAIR)
          ptx::mma_commit_pair(&st.tfull[acc], 0x3);
        else
          ptx::mma_commit(&st.tfull[acc]);
        acc ^= 1;
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
    uint32_t fills = 0;  // bit a: parity of the fills of accumulator a drained so far
    // PAIR: the odd CTA's warps release the accumulator on the leader's barrier
    const uint32_t tempty0 = PAIR ? ptx::mapa_shared(ptx::smem_u32(&st.tempty[0]), 0) : 0u;
    const uint32_t hempty0 = PAIR ? ptx::mapa_shared(ptx::smem_u32(&st.hempty[0]), 0) : 0u;
    for (int t = unit; t < total; t += units) {
      const TileInfo ti = decode_tile<PAIR, TAILS>(st, t, n_tiles, E, rank, ord);
      const bool tail = TAILS && ti.tail > 0;
      // the next tile puts its tail in this tile's head: release it early
      const bool next_tail = TAILS && t + units < total &&
                             decode_tile<PAIR, TAILS>(st, t + units, n_tiles, E, rank, ord).tail > 0;
      bool ok = wait_or_abort(&st.tfull[acc], fills >> acc & 1u, abort_flag, status, wait_limit);
      if (gemm1_mode(MODE) && tail) {
        // the gate and up warps of a GEMM1 tail wait on each other below:
        // they go on together or not at all
        const int wok = __all_sync(0xffffffffu, ok) ? 1 : 0;
        if (lane == 0) st.epi_ok[q] = wok;
        epi_pair_bar(q);
        const volatile int *eo = st.epi_ok;
        ok = eo[q & 1] && eo[(q & 1) + 2];
      }
      if (!ok) break;
      fills ^= 1u << acc;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + (uint32_t)(acc * UMMA_N) + ((uint32_t)(q * 32) << 16);
      uint8_t *wbuf = st.epi[q];
      if (TAILS && tail) {
        // first the fused tail's D^T, in the other accumulator's head: lane =
        // weight column, TMEM column i = tail row t0 + i
        const uint32_t tt = tmem + (uint32_t)((acc ^ 1) * UMMA_N) + ((uint32_t)(q * 32) << 16);
        const int r = lane < ti.tail ? ti.t0 + lane : -1;  // this lane's tail row
        if (gemm1_mode(MODE)) {
          // warps 4, 5 (lanes 0-63) hold this CTA's 64 gate columns, warps 2,
          // 3 (lanes 64-127) the matching up columns: each gate warp passes
          // SiLU(gate) to its up warp through an exchange buffer
          float4 *xrow =
              reinterpret_cast<float4 *>(xch + (q & 1) * XCH_WARP_BYTES + lane * XCH_ROW_BYTES);
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tt, v);
          ptx::tmem_ld_wait();
          // the other accumulator's head is free again
          head_release(st.hempty, hempty0, acc ^ 1, PAIR && !leader, lane);
          if (q < 2) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              xrow[i] = make_float4(silu(__uint_as_float(v[4 * i])), silu(__uint_as_float(v[4 * i + 1])),
                                    silu(__uint_as_float(v[4 * i + 2])), silu(__uint_as_float(v[4 * i + 3])));
            epi_pair_bar(q);  // staged
            epi_pair_bar(q);  // read by the up warp
          } else {
            epi_pair_bar(q);
            float hv[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 sv = xrow[i];
              hv[4 * i] = sv.x * __uint_as_float(v[4 * i]);
              hv[4 * i + 1] = sv.y * __uint_as_float(v[4 * i + 1]);
              hv[4 * i + 2] = sv.z * __uint_as_float(v[4 * i + 2]);
              hv[4 * i + 3] = sv.w * __uint_as_float(v[4 * i + 3]);
            }
            epi_pair_bar(q);
            store_tile_chunk_t(wbuf, hv, lane, out, (size_t)I, r, ti.tail,
                               ti.nt * 128 + rank * 64 + (q - 2) * 32);
          }
        } else {
          const bool live = ti.nt * UMMA_N + rank * 128 + q * 32 < Nout;  // uniform across the warp
          uint32_t a[32];
          if (live) {
            ptx::tmem_ld_32x32b_x32(tt, a);
            ptx::tmem_ld_wait();
          }
          head_release(st.hempty, hempty0, acc ^ 1, PAIR && !leader, lane);
          if (live) {
            // this lane's tail row: its output row and routing weight (MODE 4)
            int dst = r;
            float wt = 1.f;
            if (MODE == 4 && r >= 0) {
              const int f = __ldg(perm + r);
              if ((unsigned)f < (unsigned)nK) {
                dst = f;
                wt = __ldg(tw + f);
              } else {
                dst = -1;
                flag_status(status, MOE_DEV_BAD_LAYOUT);
              }
            }
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = __uint_as_float(a[i]);
              if (MODE == 4) v[i] *= __shfl_sync(0xffffffffu, wt, i);
            }
            store_tile_chunk_t(wbuf, v, lane, out, (size_t)Nout, dst, ti.tail,
                               ti.nt * UMMA_N + rank * 128 + q * 32);
          }
        }
      }
      // rows of this warp's 32-row slice that belong to the tile's expert
      const int wrows = ti.rows - q * 32;
      const int wrow0 = ti.row0 + q * 32;
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
          // SPLIT_GU: accumulator columns [128 r, 128 r + 64) are the gate and
          // [128 r + 64, 128 r + 128) the up columns of h columns [64 r, 64 r + 64)
          const int gc = SPLIT_GU ? (c >> 1) * 128 + (c & 1) * 32 : c * 32;
          const int uc = SPLIT_GU ? gc + 64 : 128 + c * 32;
          uint32_t g[32], u[32];
          ptx::tmem_ld_32x32b_x32(tbase + gc, g);
          ptx::tmem_ld_32x32b_x32(tbase + uc, u);
          ptx::tmem_ld_wait();
          if (TAILS && next_tail && c == 0)
            head_release(st.hempty, hempty0, acc, PAIR && !leader, lane);
          const int col = ti.nt * 128 + (SPLIT_GU ? (c >> 1) * 64 + (c & 1) * 32 : c * 32);
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
          if (TAILS && next_tail && c == 0)
            head_release(st.hempty, hempty0, acc, PAIR && !leader, lane);
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
      if (lane == 0) epi_arrive(st.tempty, tempty0, acc, PAIR && !leader);
      acc ^= 1;
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
        if (own == peer + 1)  // both load the same tile in a phase: the same bytes
          ptx::mbar_complete_tx(&st.full[s], (uint32_t)st.own_bytes[s]);
        else if (peer == own + 1)
          ptx::mbar_arrive_expect_tx(&st.full[s], (uint32_t)st.peer_bytes[s]);
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

template <int MODE, bool PAIR = false, bool TAILS = false>
cudaError_t set_smem_attr() {
  static int done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc_kernel<MODE, PAIR, TAILS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bytes<PAIR, TAILS>());
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
// fused tails of the forward pair GEMMs (moe_set_gemm_tails): -1 chosen per
// launch (tails_auto), 0 never, 1 always
std::atomic<int> g_tails{-1};

// Fused tails pay where a typical expert holds about one 256-row window and a
// remainder: then a tail of at most 32 rows saves a whole window in about
// half of the experts (measured: the grouped GEMMs of the DeepSeek-V3-sized
// layer, 256 rows per expert on average, 16 % faster).  With two or more
// windows per expert the saving is a smaller share, and the fused-tail kernel
// runs its windows without a tail a few per cent slower (measured on the
// OLMoE-shaped layer, 512 rows per expert: 7 % slower overall), so it is not
// used there.
bool tails_auto(long long nK, int E) {
  const long long a = E > 0 ? nK / E : 0;
  return a >= 192 && a <= 384;
}
bool use_tails(long long nK, int E) {
  const int m = g_tails.load();
  return m < 0 ? tails_auto(nK, E) : m != 0;
}

// CTA pairs of MODE's kernel that can be resident at once (cached per device)
template <int MODE, bool TAILS = false>
cudaError_t pair_clusters(int *out) {
  static int cached[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!cached[dev]) {
    e = set_smem_attr<MODE, true, TAILS>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 16);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem_bytes<true, TAILS>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    e = cudaOccupancyMaxActiveClusters(&nc, grouped_gemm_tc_kernel<MODE, true, TAILS>, &cfg);
    if (e != cudaSuccess) return e;
    if (nc < 1) return cudaErrorInvalidConfiguration;
    cached[dev] = nc;
  }
  *out = cached[dev];
  return cudaSuccess;
}

// Launch of the pair kernel: as many CTA pairs as are resident at once within
// the SMs sm_reserve leaves.
template <int MODE, bool TAILS, typename... Args>
cudaError_t launch_pairs(int sm_reserve, cudaStream_t s, Args &&...args) {
  int nc = 0;
  cudaError_t e = pair_clusters<MODE, TAILS>(&nc);
  if (e != cudaSuccess) return e;
  const int avail = gemm_grid(sm_reserve) / 2;
  if (avail < nc) nc = avail < 1 ? 1 : avail;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * nc);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes<true, TAILS>();
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
  return cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<MODE, true, TAILS>,
                            static_cast<Args &&>(args)...);
}

// Persistent launch of a grouped GEMM: one CTA per SM, or CTA pairs (with
// fused tails in the forward modes when `tails`).
template <int MODE, typename... Args>
cudaError_t launch_gemm(bool pair, bool tails, int sm_reserve, cudaStream_t s, Args &&...args) {
  if (!pair) {
    cudaError_t e = set_smem_attr<MODE>();
    if (e != cudaSuccess) return e;
    return launch_pdl(grouped_gemm_tc_kernel<MODE>, dim3(gemm_grid(sm_reserve)),
                      dim3(NUM_THREADS), SMEM_BYTES, s, static_cast<Args &&>(args)...);
  }
  if constexpr (tail_mode(MODE)) {
    if (tails) return launch_pairs<MODE, true>(sm_reserve, s, static_cast<Args &&>(args)...);
  }
  return launch_pairs<MODE, false>(sm_reserve, s, static_cast<Args &&>(args)...);
}

}  // namespace

void set_gemm_single_cta(bool single) { g_single_cta.store(single ? 1 : 0); }
void set_gemm_tails(int mode) { g_tails.store(mode < 0 ? -1 : (mode ? 1 : 0)); }
bool gemm_single_cta() { return g_single_cta.load() != 0; }

cudaError_t launch_gemm1_tc(const Desc &d, const void *x_perm, const void *w13,
                            const int32_t *offsets, void *h, int sm_reserve, int32_t *status,
                            cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mA, mB, mA2;
  int BNB = 0;
  if (!make_map_2d(&mA, x_perm, d.H, nK, BK, BM) ||
      !make_map_2d(&mA2, x_perm, d.H, nK, BK, TAIL_HALF) ||
      !weight_map(&mB, w13, d, d.H, 2ull * d.I, &BNB))
    return cudaErrorInvalidValue;
  return launch_gemm<1>(!gemm_single_cta(), use_tails(nK, d.E), sm_reserve, s, mA, mB, mA2, offsets, d.E, (int)nK, d.H, d.I, d.I,
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
                    SMEM_BYTES, s, mB, mB, mB, offsets, d.E, (int)nK, d.H, d.I, d.I,
                    reinterpret_cast<__nv_bfloat16 *>(h), status, perm, d.K,
                    reinterpret_cast<const __nv_bfloat16 *>(x), nullptr, nullptr, pipeline_wait_limit(), BNB);
}

cudaError_t launch_gemm2_tc(const Desc &d, const void *h, const void *w2, const int32_t *offsets,
                            void *y_perm, int sm_reserve, int32_t *status, cudaStream_t s) {
  const long long nK = d.nK();
  if (nK == 0) return cudaSuccess;
  CUtensorMap mA, mB, mA2;
  int BNB = 0;
  if (!make_map_2d(&mA, h, d.I, nK, BK, BM) || !make_map_2d(&mA2, h, d.I, nK, BK, TAIL_HALF) ||
      !weight_map(&mB, w2, d, d.I, d.H, &BNB))
    return cudaErrorInvalidValue;
  return launch_gemm<2>(!gemm_single_cta(), use_tails(nK, d.E), sm_reserve, s, mA, mB, mA2, offsets, d.E, (int)nK, d.I, d.I, d.H,
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
  CUtensorMap mA, mB, mA2;
  int BNB = 0;
  if (!make_map_2d(&mA, h, d.I, nK, BK, BM) || !make_map_2d(&mA2, h, d.I, nK, BK, TAIL_HALF) ||
      !weight_map(&mB, w2, d, d.I, d.H, &BNB))
    return cudaErrorInvalidValue;
  return launch_gemm<4>(!gemm_single_cta(), use_tails(nK, d.E), sm_reserve, s, mA, mB, mA2, offsets, d.E, (int)nK, d.I, d.I, d.H,
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
  return launch_gemm<5>(pair, false, 0, s, mA, mB, mA, offsets, d.E, (int)nK, Kdim, 0, Nout,
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
  return launch_gemm<6>(!gemm_single_cta(), false, 0, s, mA, mB, mA, offsets, d.E, (int)nK, d.H, d.I, 2 * d.I,
                        reinterpret_cast<__nv_bfloat16 *>(dgu), status, (const int32_t *)nullptr,
                        0, (const __nv_bfloat16 *)nullptr, (const float *)nullptr,
                        reinterpret_cast<const __nv_bfloat16 *>(dh), pipeline_wait_limit(), 0);
}

}  // namespace moe
