// Dispatch layout: per-expert counts, offsets and the stable expert-sorted
// permutation of the flat (token, slot) pairs f = t*K + k.
// "MoE 分布式推理基础（基于 vLLM）" §1.2 (Algorithm 2 steps 4-5, hit counts
// n_e and sets I_e) and §2.3 (moe_align_block_size: pairs sorted by expert,
// ascending flat index inside an expert, as in its worked example).
//
// Two integer-only kernels, so the result is deterministic:
//  1. layout_count:        each block histograms a chunk of CH pairs (+1
//                          bucket for ids outside [0, E)).
//  2. layout_scan_scatter: each block scans the per-chunk histograms itself
//                          (counts, offsets, its chunk's first position per
//                          expert), then each warp walks its 256-pair slice
//                          in order and scatters it stably.
#include "common.cuh"

namespace moe {
namespace {

constexpr int LT = 256;               // threads per block
constexpr int LW = LT / 32;           // warps per block
constexpr int SLICE = 256;            // pairs per warp
constexpr int CH = LW * SLICE;        // pairs per block (2048)

// GUEST: the instantiation launched beside the grouped GEMM (own carveout
// preference, see prefer_max_shared)
template <bool GUEST>
__global__ void __launch_bounds__(LT) layout_count(const int32_t *__restrict__ idx, long long nK,
                                                   int E, int32_t *__restrict__ cnt,
                                                   int32_t *status) {
  pdl_enter();
  __shared__ int hist[kMaxE + 1];
  for (int c = threadIdx.x; c <= E; c += LT) hist[c] = 0;
  __syncthreads();
  const long long base = (long long)blockIdx.x * CH;
  bool bad = false;
  int ev[CH / LT];  // all loads first, then the counting
#pragma unroll
  for (int j = 0; j < CH / LT; ++j) {
    const long long f = base + j * LT + threadIdx.x;
    ev[j] = f < nK ? __ldg(idx + f) : -1;
  }
#pragma unroll
  for (int j = 0; j < CH / LT; ++j) {
    if (base + j * LT + threadIdx.x >= nK) break;
    const bool ok = (unsigned)ev[j] < (unsigned)E;
    bad |= !ok;
    atomicAdd(&hist[ok ? ev[j] : E], 1);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, MOE_DEV_BAD_ROUTING);
  for (int c = threadIdx.x; c <= E; c += LT) cnt[(size_t)blockIdx.x * (E + 1) + c] = hist[c];
}

// Scan and scatter.  Every block reads the per-chunk histograms, forms the
// bucket totals, their exclusive scan and the first position of each bucket
// inside its own chunk (block 0 also writes counts and offsets).  Each warp
// then counts its 256-pair slice, takes running positions after the earlier
// warps of the block, and re-walks the slice in order: inside a 32-pair step
// the lanes holding one expert find each other through a per-warp bit mask
// per expert (atomicOr of the lane bit), a pair's rank is the number of lower
// lanes with its expert, so the order inside an expert follows the flat index.
template <bool GUEST>
__global__ void __launch_bounds__(LT) layout_scan_scatter(const int32_t *__restrict__ idx,
                                                          long long nK, int E, int nb,
                                                          const int32_t *__restrict__ cnt,
                                                          int32_t *__restrict__ counts,
                                                          int32_t *__restrict__ offsets,
                                                          int32_t *__restrict__ perm,
                                                          int32_t *__restrict__ inv_perm) {
  pdl_enter();
  __shared__ int tot[kMaxE + 1];
  __shared__ int pre[kMaxE + 1];
  __shared__ int run[LW][kMaxE + 1];
  __shared__ unsigned mask[LW][kMaxE + 1];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long slice0 = (long long)blockIdx.x * CH + (long long)w * SLICE;
  for (int c = threadIdx.x; c <= E; c += LT) {
    int t = 0, p = 0;
    for (int b = 0; b < nb; ++b) {
      const int v = cnt[(size_t)b * (E + 1) + c];
      t += v;
      p += b < (int)blockIdx.x ? v : 0;
    }
    tot[c] = t;
    pre[c] = p;
  }
  for (int c = lane; c <= E; c += 32) {
    run[w][c] = 0;
    mask[w][c] = 0u;
  }
  __syncthreads();
  // exclusive scan of the bucket totals (warp 0, 32 buckets per step)
  if (w == 0) {
    int carry = 0;
    for (int c0 = 0; c0 <= E; c0 += 32) {
      const int c = c0 + lane;
      const int v = c <= E ? tot[c] : 0;
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (c <= E) {
        const int start = carry + inc - v;
        if (blockIdx.x == 0) {
          if (c < E) {
            counts[c] = v;
            offsets[c] = start;
          } else {
            offsets[E] = start;  // pairs with a valid id; invalid ones follow
          }
        }
        pre[c] += start;  // first position of bucket c in this block's chunk
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  // pass 1: the slice's buckets (kept in registers for pass 2) and this
  // warp's histogram
  constexpr int NS = SLICE / 32;
  int key[NS];
#pragma unroll
  for (int j = 0; j < NS; ++j) {  // -1 past the end; E for an id outside [0, E)
    const long long f = slice0 + 32 * j + lane;
    const int e = f < nK ? __ldg(idx + f) : 0;
    key[j] = f < nK ? ((unsigned)e < (unsigned)E ? e : E) : -1;
  }
#pragma unroll
  for (int j = 0; j < NS; ++j)
    if (key[j] >= 0) atomicAdd(&run[w][key[j]], 1);
  __syncthreads();
  // running positions: chunk base + counts of the earlier warps of this block
  for (int c = threadIdx.x; c <= E; c += LT) {
    int r = pre[c];
    for (int ww = 0; ww < LW; ++ww) {
      const int h = run[ww][c];
      run[ww][c] = r;
      r += h;
    }
  }
  __syncthreads();
  // pass 2: stable scatter
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < NS; ++j) {
    const long long f = slice0 + 32 * j + lane;
    const int k = key[j];
    if (k >= 0) atomicOr(&mask[w][k], 1u << lane);
    __syncwarp();
    const unsigned peers = k >= 0 ? mask[w][k] : 0u;
    __syncwarp();
    if (k >= 0) {
      const int pos = run[w][k] + __popc(peers & lt_mask);
      perm[pos] = (int32_t)f;
      inv_perm[f] = pos;
    }
    __syncwarp();
    if (k >= 0 && (peers & lt_mask) == 0) {  // the lowest lane of the expert
      run[w][k] += __popc(peers);
      mask[w][k] = 0u;
    }
    __syncwarp();
  }
}

inline int num_chunks(long long nK) { return (int)((nK + CH - 1) / CH); }

}  // namespace

size_t layout_ws_bytes(const Desc &d) {
  const int nb = num_chunks(d.nK()) > 0 ? num_chunks(d.nK()) : 1;
  return (size_t)nb * (d.E + 1) * sizeof(int32_t);
}

cudaError_t launch_layout(const Desc &d, const int32_t *topk_idx, int32_t *counts,
                          int32_t *offsets, int32_t *perm, int32_t *inv_perm, int32_t *status,
                          void *ws, cudaStream_t s, bool guest) {
  const long long nK = d.nK();
  const int nb = num_chunks(nK);
  if (nb == 0) {  // no tokens: all counts and offsets are zero
    cudaError_t e1 = cudaMemsetAsync(counts, 0, sizeof(int32_t) * d.E, s);
    if (e1 != cudaSuccess) return e1;
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d.E + 1), s);
  }
  int32_t *cnt = reinterpret_cast<int32_t *>(ws);
  if (guest) {
    static bool carveout[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 && !carveout[dev]) {
      cudaError_t e = prefer_max_shared(layout_count<true>);
      if (e == cudaSuccess) e = prefer_max_shared(layout_scan_scatter<true>);
      if (e != cudaSuccess) return e;
      carveout[dev] = true;
    }
  }
  cudaError_t e = launch_k(guest, guest ? layout_count<true> : layout_count<false>, dim3(nb),
                           dim3(LT), 0, s, topk_idx, nK, d.E, cnt, status);
  if (e != cudaSuccess) return e;
  return launch_k(guest, guest ? layout_scan_scatter<true> : layout_scan_scatter<false>, dim3(nb),
                  dim3(LT), 0, s, topk_idx, nK, d.E, nb, cnt, counts, offsets, perm, inv_perm);
}

}  // namespace moe
