// Router on the tcgen05 tensor cores with softmax, TopK and the near-tie
// rescoring fused into one kernel, for bf16 layers with E % 64 == 0 and
// K <= 8.  "MoE 分布式推理基础（基于 vLLM）" §1.2, Algorithm 2 steps 1-3 and
// the router's renormalisation.
//
// One CTA per 128-token tile (persistent over tiles), 18 warps:
//   warp 0       TMA producer: x tile (128 tokens x 64 k) and E/64 boxes of
//                W_gate (64 k x 64 experts) per stage.
//   warp 1       TMEM allocator and MMA issuer: 128 x E x 16 bf16 MMAs into one
//                of two E-column float32 accumulators.
//   warps 2..17  epilogue: 4 TMEM lane quarters x 4 column slices.  Each
//                thread owns one token and E/4 experts: it adds the bias,
//                stores those float32 logits, keeps the K+1 largest in
//                registers (descending, ties to the lower expert id), and
//                computes their max and sum of exp.  After a barrier one
//                thread per token merges the four slices.  Tokens whose top
//                K+1 logits lie closer than the margin tau are rescored by all
//                512 epilogue threads in double-float (exact products,
//                error-free sums) over the experts within tau of the K-th
//                logit, and chosen on those values.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "df.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int RT_BM = 128, RT_BK = 64, RT_MAX_STAGES = 8;
constexpr int RT_SLICES = 4;                          // column slices per token
constexpr int RT_EPI_WARPS = 4 * RT_SLICES;           // 16
constexpr int RT_EPI_THREADS = 32 * RT_EPI_WARPS;     // 512
constexpr int RT_THREADS = 64 + RT_EPI_THREADS;       // 576
constexpr int RT_A_BYTES = RT_BM * RT_BK * 2;         // 16 KB
constexpr int RT_BOX_BYTES = 64 * RT_BK * 2;          // 8 KB: 64 experts x 64 k
constexpr int RT_PIPE_BYTES = 168 * 1024;             // operand stages
constexpr int RS_SLOTS = 256;                         // candidate slots per rescoring sweep
constexpr int RS_MAXF = 16;                           // flagged tokens per sweep

struct RtTail {
  uint64_t full[RT_MAX_STAGES];
  uint64_t empty[RT_MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float bias[kMaxE];
};

template <int KM>
struct EpiSmem {
  union {
    struct {                             // selection: one list per (slice, token)
      float pv[RT_SLICES][RT_BM][KM + 1];  // per-slice top K+1 values
      int pi[RT_SLICES][RT_BM][KM + 1];    // ... and expert ids
    } sel;
    struct {                             // rescoring of the tile's flagged tokens
      float phi[RT_EPI_THREADS];           // per-thread partial sums
      float plo[RT_EPI_THREADS];
      float chi[RS_SLOTS], clo[RS_SLOTS];  // per slot: summed over row groups + bias
      int cexp[RS_SLOTS];                  // expert of each slot
      int ctok[RS_SLOTS];                  // token (index in the sweep) of each slot
      int tbase[RS_MAXF + 1];              // first slot of each token
      int S, nb;                           // slots and tokens of the sweep
    } res;
  } u;
  float pm[RT_SLICES][RT_BM];          // per-slice max
  float ps[RT_SLICES][RT_BM];          // per-slice sum of exp(l - slice max)
  int stop;                            // set by an epilogue thread whose wait gave up
  int nflag;                           // flagged tokens of the tile
  int ftok[RT_BM];
  float fm[RT_BM], fS[RT_BM], fvK[RT_BM];
};

__host__ __device__ inline int rt_stages(int E) {
  const int s = RT_PIPE_BYTES / (RT_A_BYTES + (E / 64) * RT_BOX_BYTES);
  return s < RT_MAX_STAGES ? s : RT_MAX_STAGES;
}

// the tail (mbarriers) follows the epilogue area at a 16-byte boundary
template <int KM>
__host__ __device__ constexpr size_t epi_bytes() {
  return (sizeof(EpiSmem<KM>) + 15) & ~size_t(15);
}

template <int KM>
inline size_t rt_smem_bytes(int E) {
  return 1024 + (size_t)rt_stages(E) * (RT_A_BYTES + (E / 64) * RT_BOX_BYTES) + epi_bytes<KM>() +
         sizeof(RtTail);
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

// barrier among the 512 epilogue threads only
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(RT_EPI_THREADS) : "memory");
}

// (v, e) ranks above (w, f): larger value, or equal value and lower expert id
__device__ __forceinline__ bool ranks_above(float v, int e, float w, int f) {
  return v > w || (v == w && e < f);
}

// Rescoring of the tile's flagged tokens by the 512 epilogue threads.  A
// sweep takes up to 16 flagged tokens and their candidate experts (within tau
// of the token's K-th float32 logit), one slot per (token, candidate), at most
// 256 slots.  Thread et serves slot et mod Sp (Sp = slots rounded up to a
// power of two) over the rows h congruent to et / Sp modulo 512 / Sp,
// accumulating x[t,h] * W_gate[h,e] in double-float (four interleaved
// accumulators).  The 32 threads of a warp serve consecutive slots of the same
// row, so their W_gate loads fall in the few sectors of that row.  The
// partial sums are added in a fixed order, the bias is added, and one warp per
// token keeps the K largest.
template <int KM>
__device__ __forceinline__ void rescore_tile(EpiSmem<KM> &ep, const float *__restrict__ bias_s,
                                             const __nv_bfloat16 *__restrict__ x,
                                             const __nv_bfloat16 *__restrict__ wg,
                                             const float *__restrict__ logits,
                                             int32_t *__restrict__ topk_idx,
                                             float *__restrict__ topk_w, int H, int E, int norm,
                                             float tau_rel, int ew, int lane, int et) {
  constexpr int K = KM;
  auto &rs = ep.u.res;
  const int nflag = ep.nflag;
  for (int b0 = 0; b0 < nflag;) {
    // slots of this sweep (warp 0), in ascending expert order per token
    if (ew == 0) {
      int total = 0, nb = 0;
      for (int g = b0; g < nflag && nb < RS_MAXF; ++g) {
        const int ft = ep.ftok[g];
        const float thr = ep.fvK[g] - tau_rel * fmaxf(1.f, fabsf(ep.fm[g]));
        int C = 0;
        for (int j = 0; j < E / 32; ++j)
          C += __popc(__ballot_sync(0xffffffffu, logits[(size_t)ft * E + lane + 32 * j] >= thr));
        if (nb > 0 && total + C > RS_SLOTS) break;
        int pos = total;
        for (int j = 0; j < E / 32; ++j) {
          const int e = lane + 32 * j;
          const unsigned ball = __ballot_sync(0xffffffffu, logits[(size_t)ft * E + e] >= thr);
          if (ball >> lane & 1u) {
            const int sl = pos + __popc(ball & ((1u << lane) - 1u));
            rs.cexp[sl] = e;
            rs.ctok[sl] = nb;
          }
          pos += __popc(ball);
        }
        if (lane == 0) rs.tbase[nb] = total;
        total += C;
        ++nb;
      }
      if (lane == 0) {
        rs.tbase[nb] = total;
        rs.S = total;
        rs.nb = nb;
      }
    }
    epi_bar();
    const int S = rs.S, nb = rs.nb;
    int Sp = 1;
    while (Sp < S) Sp <<= 1;
    const int G = RT_EPI_THREADS / Sp;  // row groups
    const int s_id = et & (Sp - 1), g_id = et / Sp;
    const bool active = s_id < S;
    const int e_s = active ? rs.cexp[s_id] : 0;
    const int f_s = active ? rs.ctok[s_id] : 0;
    DF acc{0.f, 0.f};
    if (active) {
      const __nv_bfloat16 *xr = x + (size_t)ep.ftok[b0 + f_s] * H;
      const __nv_bfloat16 *wc = wg + e_s;
      DF a4[4] = {DF{0.f, 0.f}, DF{0.f, 0.f}, DF{0.f, 0.f}, DF{0.f, 0.f}};
      int h = g_id;
      for (; h + 7 * G < H; h += 8 * G) {
        float xv[8], wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          xv[u] = __bfloat162float(xr[h + u * G]);
          wv[u] = __bfloat162float(wc[(size_t)(h + u * G) * E]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) a4[u & 3] = df_add(a4[u & 3], two_prod(xv[u], wv[u]));
      }
      for (; h < H; h += G)
        a4[0] = df_add(a4[0], two_prod(__bfloat162float(xr[h]), __bfloat162float(wc[(size_t)h * E])));
      acc = df_add(df_add(a4[0], a4[1]), df_add(a4[2], a4[3]));
    }
    rs.phi[et] = acc.hi;
    rs.plo[et] = acc.lo;
    epi_bar();
    for (int sl = et; sl < S; sl += RT_EPI_THREADS) {
      DF sum{0.f, 0.f};
      for (int g = 0; g < G; ++g) sum = df_add(sum, DF{rs.phi[g * Sp + sl], rs.plo[g * Sp + sl]});
      const float bb = bias_s[rs.cexp[sl]];
      sum = isinf(bb) ? DF{bb, 0.f} : df_add(sum, DF{bb, 0.f});
      rs.chi[sl] = sum.hi;
      rs.clo[sl] = sum.lo;
    }
    epi_bar();
    // warp f keeps the K best of the sweep's token f
    if (ew < nb && lane == 0) {
      const int g = b0 + ew;
      const int ft = ep.ftok[g];
      DF lv[K];
      int li[K];
#pragma unroll
      for (int z = 0; z < K; ++z) {
        lv[z] = DF{-INFINITY, 0.f};
        li[z] = 0x7fffffff;
      }
      for (int sl = rs.tbase[ew]; sl < rs.tbase[ew + 1]; ++sl) {
        DF cv{rs.chi[sl], rs.clo[sl]};
        int ci = rs.cexp[sl];
#pragma unroll
        for (int z = 0; z < K; ++z) {
          const bool gt = df_greater(cv, ci, lv[z], li[z]);
          const DF tv = gt ? lv[z] : cv;
          const int ti = gt ? li[z] : ci;
          lv[z] = gt ? cv : lv[z];
          li[z] = gt ? ci : li[z];
          cv = tv;
          ci = ti;
        }
      }
      float w[K];
      float wsum = 0.f;
#pragma unroll
      for (int z = 0; z < K; ++z) {
        w[z] = expf(logits[(size_t)ft * E + li[z]] - ep.fm[g]) / ep.fS[g];
        wsum += w[z];
      }
#pragma unroll
      for (int z = 0; z < K; ++z) {
        topk_idx[(size_t)ft * K + z] = li[z];
        topk_w[(size_t)ft * K + z] = norm ? w[z] / wsum : w[z];
      }
    }
    epi_bar();  // the slots and staging buffers are reused by the next sweep
    b0 += nb;
  }
}

template <int KM>
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW,
                     const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ wg,
                     const float *__restrict__ bias, float *__restrict__ logits,
                     int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int n, int H,
                     int E, int norm, uint32_t idesc, uint32_t tmem_cols, int32_t *status) {
  constexpr int K = KM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nbox = E / 64;
  const int b_stage = nbox * RT_BOX_BYTES;
  const int STAGES = rt_stages(E);
  uint8_t *smemA = smem;
  uint8_t *smemB = smem + STAGES * RT_A_BYTES;
  EpiSmem<KM> &ep = *reinterpret_cast<EpiSmem<KM> *>(smem + STAGES * (RT_A_BYTES + b_stage));
  RtTail &st = *reinterpret_cast<RtTail *>(reinterpret_cast<uint8_t *>(&ep) + epi_bytes<KM>());

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (n + RT_BM - 1) / RT_BM;
  const int KB = H / RT_BK;
  if ((int)blockIdx.x >= n_tiles) return;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&st.full[s], 1);
      ptx::mbar_init(&st.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&st.tfull[a], 1);
      ptx::mbar_init(&st.tempty[a], RT_EPI_WARPS);
    }
    ptx::mbar_init(&st.drain, 1);
    st.abort_flag = 0;
    ep.nflag = 0;
    ep.stop = 0;
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
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
      }
      for (int s = 0; s < STAGES; ++s)
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
          if (++stage == STAGES) {
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
    const int ew = warp - 2;              // epilogue warp 0..15
    const int q = warp & 3;               // TMEM lane quarter this warp may read
    const int sl = ew >> 2;               // column slice 0..3
    const int r = q * 32 + lane;          // token row in the tile
    const int et = ew * 32 + lane;        // 0..511
    const int cols = E / RT_SLICES;
    const int c0 = sl * cols;
    const float tau_rel = tie_margin_tc(H);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      // all 512 threads take every barrier below; a thread whose wait gave up
      // raises ep.stop before the first one, so all leave together
      if (!rt_wait(&st.tfull[acc], acc_phase, abort_flag, status)) ep.stop = 1;
      epi_bar();
      if (ep.stop) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + (uint32_t)(acc * E + c0) + ((uint32_t)(q * 32) << 16);
      const int tok = t * RT_BM + r;
      const bool valid = tok < n;
      float *lrow = logits + (size_t)(valid ? tok : 0) * E;

      // this slice: logits, max, top K+1 (descending, ties to the lower id)
      float lv[K + 1];
      int li[K + 1];
#pragma unroll
      for (int j = 0; j <= K; ++j) {
        lv[j] = -INFINITY;
        li[j] = 0x7fffffff;
      }
      float last_v = -INFINITY;
      int last_i = 0x7fffffff;
      float m = -INFINITY;
      for (int c = 0; c < cols / 8; ++c) {
        uint32_t raw[8];
        ptx::tmem_ld_32x32b_x8(tbase + c * 8, raw);
        ptx::tmem_ld_wait();
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(raw[i]) + st.bias[c0 + c * 8 + i];
        if (valid) {
          float4 *dst = reinterpret_cast<float4 *>(lrow + c0 + c * 8);
          dst[0] = make_float4(v[0], v[1], v[2], v[3]);
          dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          m = fmaxf(m, v[i]);
          const int e = c0 + c * 8 + i;
          if (ranks_above(v[i], e, last_v, last_i)) {
            float cv = v[i];
            int ci = e;
#pragma unroll
            for (int j = 0; j <= K; ++j) {
              const bool gt = ranks_above(cv, ci, lv[j], li[j]);
              const float tv = gt ? lv[j] : cv;
              const int ti = gt ? li[j] : ci;
              lv[j] = gt ? cv : lv[j];
              li[j] = gt ? ci : li[j];
              cv = tv;
              ci = ti;
            }
            last_v = lv[K];
            last_i = li[K];
          }
        }
      }
      float ssum = 0.f;
      for (int c = 0; c < cols / 8; ++c) {
        uint32_t raw[8];
        ptx::tmem_ld_32x32b_x8(tbase + c * 8, raw);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          ssum += expf(__uint_as_float(raw[i]) + st.bias[c0 + c * 8 + i] - m);
      }
      // the accumulator is free for the next tile
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&st.tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;

#pragma unroll
      for (int j = 0; j <= K; ++j) {
        ep.u.sel.pv[sl][r][j] = lv[j];
        ep.u.sel.pi[sl][r][j] = li[j];
      }
      ep.pm[sl][r] = m;
      ep.ps[sl][r] = ssum;
      __threadfence_block();  // the logits rows are read back below
      epi_bar();

      // merge the four slices: one thread per token
      if (sl == 0 && valid) {
        float fv[K + 1];
        int fi[K + 1];
        int h0 = 0, h1 = 0, h2 = 0, h3 = 0;
#pragma unroll
        for (int j = 0; j <= K; ++j) {
          float bv = h0 <= K ? ep.u.sel.pv[0][r][h0] : -INFINITY;
          int bi = h0 <= K ? ep.u.sel.pi[0][r][h0] : 0x7fffffff;
          int bw = 0;
          const float v1 = h1 <= K ? ep.u.sel.pv[1][r][h1] : -INFINITY;
          const int i1 = h1 <= K ? ep.u.sel.pi[1][r][h1] : 0x7fffffff;
          if (ranks_above(v1, i1, bv, bi)) { bv = v1; bi = i1; bw = 1; }
          const float v2 = h2 <= K ? ep.u.sel.pv[2][r][h2] : -INFINITY;
          const int i2 = h2 <= K ? ep.u.sel.pi[2][r][h2] : 0x7fffffff;
          if (ranks_above(v2, i2, bv, bi)) { bv = v2; bi = i2; bw = 2; }
          const float v3 = h3 <= K ? ep.u.sel.pv[3][r][h3] : -INFINITY;
          const int i3 = h3 <= K ? ep.u.sel.pi[3][r][h3] : 0x7fffffff;
          if (ranks_above(v3, i3, bv, bi)) { bv = v3; bi = i3; bw = 3; }
          fv[j] = bv;
          fi[j] = bi;
          h0 += bw == 0;
          h1 += bw == 1;
          h2 += bw == 2;
          h3 += bw == 3;
        }
        float M = ep.pm[0][r];
#pragma unroll
        for (int w = 1; w < RT_SLICES; ++w) M = fmaxf(M, ep.pm[w][r]);
        float S = 0.f;
#pragma unroll
        for (int w = 0; w < RT_SLICES; ++w) S += ep.ps[w][r] * expf(ep.pm[w][r] - M);
        const float tau = tau_rel * fmaxf(1.f, fabsf(M));
        bool amb = false;
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (isfinite(fv[j]) && isfinite(fv[j + 1]) && fv[j] - fv[j + 1] < tau) amb = true;
        if (!amb) {
          float w[K];
          float wsum = 0.f;
#pragma unroll
          for (int j = 0; j < K; ++j) {
            w[j] = expf(fv[j] - M) / S;
            wsum += w[j];
          }
#pragma unroll
          for (int j = 0; j < K; ++j) {
            topk_idx[(size_t)tok * K + j] = fi[j];
            topk_w[(size_t)tok * K + j] = norm ? w[j] / wsum : w[j];
          }
        } else {
          const int slot = atomicAdd(&ep.nflag, 1);
          ep.ftok[slot] = tok;
          ep.fm[slot] = M;
          ep.fS[slot] = S;
          ep.fvK[slot] = fv[K - 1];
        }
      }
      epi_bar();

      // rescoring of the tile's flagged tokens (all 512 epilogue threads)
      rescore_tile<KM>(ep, st.bias, x, wg, logits, topk_idx, topk_w, H, E, norm, tau_rel, ew, lane,
                       et);
      epi_bar();  // the rescoring lists alias the next tile's selection lists
      if (et == 0) ep.nflag = 0;
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
  const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(x);
  const __nv_bfloat16 *wb = reinterpret_cast<const __nv_bfloat16 *>(w_gate);
  auto run = [&](auto kernel, size_t smem_max, size_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_max);
    if (e != cudaSuccess) return e;
    kernel<<<grid, RT_THREADS, smem, s>>>(mX, mW, xb, wb, bias, logits, topk_idx, topk_w, d.n,
                                          d.H, d.E, d.norm ? 1 : 0, idesc, cols, status);
    return cudaGetLastError();
  };
#define MOE_RT_CASE(KK)                                                              \
  case KK:                                                                           \
    return run(router_tc_kernel<KK>, rt_smem_bytes<KK>(64) > rt_smem_bytes<KK>(256) \
                                         ? rt_smem_bytes<KK>(64)                     \
                                         : rt_smem_bytes<KK>(256),                   \
               rt_smem_bytes<KK>(d.E));
  switch (d.K) {
    MOE_RT_CASE(1)
    MOE_RT_CASE(2)
    MOE_RT_CASE(3)
    MOE_RT_CASE(4)
    MOE_RT_CASE(5)
    MOE_RT_CASE(6)
    MOE_RT_CASE(7)
    MOE_RT_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef MOE_RT_CASE
}

}  // namespace moe
