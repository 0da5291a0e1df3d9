// Dispatch layout: per-expert counts, offsets and the stable expert-sorted
// permutation of the flat (token, slot) pairs f = t*K + k.
// "MoE 分布式推理基础（基于 vLLM）" §1.2 (Algorithm 2 steps 4-5, hit counts
// n_e and sets I_e) and §2.3 (moe_align_block_size: pairs sorted by expert,
// ascending flat index inside an expert, as in its worked example).
//
// Three integer-only kernels, so the result is deterministic:
//  1. layout_count:   each block histograms a chunk of CH pairs (+1 bucket for
//                     ids outside [0, E)).
//  2. layout_scan:    one block turns the per-chunk histograms into counts,
//                     offsets and the first output position of every
//                     (chunk, expert).
//  3. layout_scatter: each warp walks its 256-pair slice in order; pairs of
//                     one expert inside a 32-wide step are ranked with
//                     __match_any_sync, so order within an expert follows f.
#include "common.cuh"

namespace moe {
namespace {

constexpr int LT = 256;               // threads per block
constexpr int LW = LT / 32;           // warps per block
constexpr int SLICE = 256;            // pairs per warp
constexpr int CH = LW * SLICE;        // pairs per block (2048)

__global__ void __launch_bounds__(LT) layout_count(const int32_t *__restrict__ idx, long long nK,
                                                   int E, int32_t *__restrict__ cnt,
                                                   int32_t *status) {
  __shared__ int hist[kMaxE + 1];
  for (int c = threadIdx.x; c <= E; c += LT) hist[c] = 0;
  __syncthreads();
  const long long base = (long long)blockIdx.x * CH;
  bool bad = false;
  for (int i = threadIdx.x; i < CH; i += LT) {
    const long long f = base + i;
    if (f >= nK) break;
    const int e = idx[f];
    const bool ok = (unsigned)e < (unsigned)E;
    bad |= !ok;
    atomicAdd(&hist[ok ? e : E], 1);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, MOE_DEV_BAD_ROUTING);
  for (int c = threadIdx.x; c <= E; c += LT) cnt[(size_t)blockIdx.x * (E + 1) + c] = hist[c];
}

__global__ void __launch_bounds__(LT) layout_scan(const int32_t *__restrict__ cnt, int nb, int E,
                                                  int32_t *__restrict__ counts,
                                                  int32_t *__restrict__ offsets,
                                                  int32_t *__restrict__ base) {
  __shared__ int tot[kMaxE + 1];
  __shared__ int start[kMaxE + 1];
  for (int c = threadIdx.x; c <= E; c += LT) {
    int s = 0;
    for (int b = 0; b < nb; ++b) s += cnt[(size_t)b * (E + 1) + c];
    tot[c] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int c = 0; c <= E; ++c) {
      start[c] = run;
      run += tot[c];
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c <= E; c += LT) {
    if (c < E) {
      counts[c] = tot[c];
      offsets[c] = start[c];
    } else {
      offsets[E] = start[E];  // pairs with a valid id; invalid ones follow
    }
    int run = start[c];
    for (int b = 0; b < nb; ++b) {
      base[(size_t)b * (E + 1) + c] = run;
      run += cnt[(size_t)b * (E + 1) + c];
    }
  }
}

__global__ void __launch_bounds__(LT) layout_scatter(const int32_t *__restrict__ idx, long long nK,
                                                     int E, const int32_t *__restrict__ base,
                                                     int32_t *__restrict__ perm,
                                                     int32_t *__restrict__ inv_perm) {
  __shared__ int run[LW][kMaxE + 1];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long slice0 = (long long)blockIdx.x * CH + (long long)w * SLICE;
  for (int c = lane; c <= E; c += 32) run[w][c] = 0;
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  // pass 1: this warp's histogram
  for (int s = 0; s < SLICE; s += 32) {
    const long long f = slice0 + s + lane;
    int key = -1;
    if (f < nK) {
      const int e = idx[f];
      key = (unsigned)e < (unsigned)E ? e : E;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (peers & lt_mask) == 0) run[w][key] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // running positions: chunk base + counts of the earlier warps of this block
  for (int c = threadIdx.x; c <= E; c += LT) {
    int r = base[(size_t)blockIdx.x * (E + 1) + c];
    for (int ww = 0; ww < LW; ++ww) {
      const int h = run[ww][c];
      run[ww][c] = r;
      r += h;
    }
  }
  __syncthreads();
  // pass 2: stable scatter
  for (int s = 0; s < SLICE; s += 32) {
    const long long f = slice0 + s + lane;
    int key = -1;
    if (f < nK) {
      const int e = idx[f];
      key = (unsigned)e < (unsigned)E ? e : E;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0) {
      const int pos = run[w][key] + __popc(peers & lt_mask);
      perm[pos] = (int32_t)f;
      inv_perm[f] = pos;
    }
    __syncwarp();
    if (key >= 0 && (peers & lt_mask) == 0) run[w][key] += __popc(peers);
    __syncwarp();
  }
}

inline int num_chunks(long long nK) { return (int)((nK + CH - 1) / CH); }

}  // namespace

size_t layout_ws_bytes(const Desc &d) {
  const int nb = num_chunks(d.nK()) > 0 ? num_chunks(d.nK()) : 1;
  return 2 * (size_t)nb * (d.E + 1) * sizeof(int32_t);
}

cudaError_t launch_layout(const Desc &d, const int32_t *topk_idx, int32_t *counts,
                          int32_t *offsets, int32_t *perm, int32_t *inv_perm, int32_t *status,
                          void *ws, cudaStream_t s) {
  const long long nK = d.nK();
  const int nb = num_chunks(nK);
  if (nb == 0) {  // no tokens: all counts and offsets are zero
    cudaError_t e1 = cudaMemsetAsync(counts, 0, sizeof(int32_t) * d.E, s);
    if (e1 != cudaSuccess) return e1;
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d.E + 1), s);
  }
  int32_t *cnt = reinterpret_cast<int32_t *>(ws);
  int32_t *base = cnt + (size_t)nb * (d.E + 1);
  layout_count<<<nb, LT, 0, s>>>(topk_idx, nK, d.E, cnt, status);
  layout_scan<<<1, LT, 0, s>>>(cnt, nb, d.E, counts, offsets, base);
  layout_scatter<<<nb, LT, 0, s>>>(topk_idx, nK, d.E, base, perm, inv_perm);
  return cudaGetLastError();
}

}  // namespace moe
