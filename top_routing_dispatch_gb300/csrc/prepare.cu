// One-time weight transforms.  For the grouped GEMMs (the pre-transform of
// expert weights that the pages describe for DeepGEMM's Mega MoE kernel,
// "大模型系统中的通算融合" §4.4): every 64 x 64 tile (64 rows of k, 64
// columns) of each expert matrix becomes one contiguous 8 KB run, ordered by
// expert, row block, column block.  The GEMMs then fetch each tile they stage
// as a single DRAM run (the row-major layout gives 64 runs of 128 bytes, one
// matrix row apart).  For the router: w_gate transposed, so the exact
// near-tie rescoring reads an expert's column as one contiguous row.  Pure
// copies: results are bitwise those of the weights as stored.
#include "common.cuh"

namespace moe {
namespace {

constexpr int TT = 256;  // threads per CTA; a tile is 512 pieces of 16 bytes

__global__ void __launch_bounds__(TT) tile_weights_kernel(const uint4 *__restrict__ w,
                                                          uint4 *__restrict__ out, int E,
                                                          int rows, int cols) {
  pdl_enter();
  const int kbn = rows / 64, nbn = cols / 64, vpr = cols / 8;  // 16-byte pieces per row
  const long long tiles = (long long)E * kbn * nbn;
  for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int nb = (int)(t % nbn);
    const long long rem = t / nbn;
    const int kb = (int)(rem % kbn);
    const int e = (int)(rem / kbn);
    const uint4 *src = w + ((size_t)e * rows + (size_t)kb * 64) * vpr + nb * 8;
    uint4 *dst = out + (size_t)t * 512;
#pragma unroll
    for (int i = threadIdx.x; i < 512; i += TT) dst[i] = __ldg(src + (size_t)(i >> 3) * vpr + (i & 7));
  }
}

cudaError_t tile_one(const void *w, void *out, int E, int rows, int cols, cudaStream_t s) {
  const long long tiles = (long long)E * (rows / 64) * (cols / 64);
  const long long cap = 8ll * device_sm_count();
  return launch_pdl(tile_weights_kernel, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(TT), 0,
                    s, reinterpret_cast<const uint4 *>(w), reinterpret_cast<uint4 *>(out), E, rows,
                    cols);
}

// w_gate_t[e][h] = w_gate[h][e]: 32 x 32 blocks through shared memory (one
// padding column keeps the column reads free of bank conflicts).
__global__ void __launch_bounds__(256) transpose_gate_kernel(const __nv_bfloat16 *__restrict__ w,
                                                             __nv_bfloat16 *__restrict__ wt,
                                                             int H, int E) {
  pdl_enter();
  __shared__ __nv_bfloat16 blk[32][33];
  const int h0 = blockIdx.y * 32, e0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  for (int r = ty; r < 32; r += 8) {
    const int h = h0 + r, e = e0 + tx;
    if (h < H && e < E) blk[r][tx] = w[(size_t)h * E + e];
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int e = e0 + r, h = h0 + tx;
    if (e < E && h < H) wt[(size_t)e * H + h] = blk[tx][r];
  }
}

}  // namespace

cudaError_t launch_prepare_router(const Desc &d, const void *w_gate, void *w_gate_t,
                                  cudaStream_t s) {
  dim3 grid((unsigned)((d.E + 31) / 32), (unsigned)((d.H + 31) / 32));
  return launch_pdl(transpose_gate_kernel, grid, dim3(256), 0, s,
                    reinterpret_cast<const __nv_bfloat16 *>(w_gate),
                    reinterpret_cast<__nv_bfloat16 *>(w_gate_t), d.H, d.E);
}

cudaError_t launch_prepare_weights(const Desc &d, const void *w13, const void *w2, void *w13t,
                                   void *w2t, cudaStream_t s) {
  cudaError_t e = tile_one(w13, w13t, d.E, d.H, 2 * d.I, s);
  if (e != cudaSuccess) return e;
  return tile_one(w2, w2t, d.E, d.I, d.H, s);
}

}  // namespace moe
