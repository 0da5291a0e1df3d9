// Router on the tcgen05 tensor cores with softmax, TopK and the near-tie
// rescoring fused into one kernel, for bf16 layers with E % 64 == 0 and
// K <= 8.  "MoE 分布式推理基础（基于 vLLM）" §1.2, Algorithm 2 steps 1-3 and
// the router's renormalisation.
//
// A cluster of 4 CTAs per 128-token tile (6 warps each):
//   warp 0      TMA producer: x tile (128 tokens x 64 k) and E/64 boxes of
//               W_gate (64 k x 64 experts) per stage, for this CTA's quarter
//               of the k-blocks.
//   warp 1      TMEM allocator and MMA issuer: 128 x E x 16 bf16 MMAs into
//               one E-column float32 accumulator.
//   warps 2..5  exchange of the partial logits through distributed shared
//               memory, then the TopK epilogue of this CTA's 32 tokens.
// Tokens whose top K+1 logits lie closer than the margin tau are rescored by
// router_rescore_kernel in double-float (exact products, error-free sums) over
// the experts whose order the float32 logits leave open.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "df.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int RT_BM = 128, RT_BK = 64, RT_MAX_STAGES = 8;
constexpr int RC = 4;                                 // CTAs per tile (cluster): K split 4 ways
constexpr int RT_ROWS = RT_BM / RC;                   // tokens a CTA finalises (32)
constexpr int RT_SLICES = 4;                          // column slices per token (= epilogue warps)
constexpr int RT_EPI_THREADS = 32 * RT_SLICES;        // 128
constexpr int RT_THREADS = 64 + RT_EPI_THREADS;       // 192
constexpr int RT_A_BYTES = RT_BM * RT_BK * 2;         // 16 KB
constexpr int RT_BOX_BYTES = 64 * RT_BK * 2;          // 8 KB: 64 experts x 64 k
constexpr int RT_PIPE_BYTES = 168 * 1024;             // operand stages
constexpr int RR_THREADS = 256;                       // rescoring kernel: threads per CTA

struct RtTail {
  uint64_t full[RT_MAX_STAGES];
  uint64_t empty[RT_MAX_STAGES];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float bias[kMaxE];
};

template <int KM>
struct EpiSmem {
  float pv[RT_SLICES][RT_ROWS][KM + 1];  // per-slice top K+1 values
  int pi[RT_SLICES][RT_ROWS][KM + 1];    // ... and expert ids
  float pm[RT_SLICES][RT_ROWS];          // per-slice max
  float ps[RT_SLICES][RT_ROWS];          // per-slice sum of exp(l - slice max)
};

__host__ __device__ inline int rt_stages(int E) {
  const int s = RT_PIPE_BYTES / (RT_A_BYTES + (E / 64) * RT_BOX_BYTES);
  return s < RT_MAX_STAGES ? s : RT_MAX_STAGES;
}

// float32 partial logits received from the cluster: [RC][RT_ROWS][E + 4]
// (rows padded by 16 bytes against bank conflicts); aliases the operand
// stages, which are idle once every MMA of the cluster has finished
__host__ __device__ inline size_t red_bytes(int E) {
  return (size_t)RC * RT_ROWS * (E + 4) * sizeof(float);
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

// barrier among the epilogue threads only
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(RT_EPI_THREADS) : "memory");
}

// (v, e) ranks above (w, f): larger value, or equal value and lower expert id
__device__ __forceinline__ bool ranks_above(float v, int e, float w, int f) {
  return v > w || (v == w && e < f);
}

// Exact TopK of the tokens the tile kernel flagged (topk_idx[t][0] == -1).
// One CTA per flagged token (grid-stride over the tokens; each CTA first
// collects its flagged tokens with one parallel pass over the markers).
// Thread e ranks expert e among all E by float32 logit (larger first, ties to
// the lower id); the rank K-1 expert gives the threshold, and the experts
// within tau of it form the candidate list L (a prefix of that order), which
// holds every expert that can be in the exact top K since the logits' error
// is below tau / 2.  A position of L whose gap to a neighbour is below tau is
// uncertain; every other position already holds the expert the exact order
// puts there (neighbours tau apart cannot swap).  Only the uncertain experts
// are rescored: x[t,:] . W_gate[:,e] in double-float (exact products,
// error-free sums), thread j serving expert j mod Sp over the rows h congruent
// to j / Sp modulo G = 256 / Sp; the G partial sums of an expert are added by
// a butterfly inside each warp and then over the warps in order, and the bias
// is added.  Each run of consecutive uncertain positions is re-sorted by those
// values (larger first, ties to the lower id) and the first K of L are the
// token's experts.  Weights: softmax of the float32 logits.
template <int KM>
__global__ void __launch_bounds__(RR_THREADS)
    router_rescore_kernel(const __nv_bfloat16 *__restrict__ x,
                          const __nv_bfloat16 *__restrict__ wg,
                          const __nv_bfloat16 *__restrict__ wgt, const float *__restrict__ bias,
                          const float *__restrict__ logits, int32_t *__restrict__ topk_idx,
                          float *__restrict__ topk_w, int n, int H, int E, int norm,
                          float tau_rel) {
  pdl_enter();
  static_assert(RR_THREADS >= kMaxE, "one thread per expert");
  constexpr int K = KM;
  constexpr int MAXT = 64;  // tokens one CTA inspects per pass
  __shared__ float lg[kMaxE];
  __shared__ float cv[kMaxE];   // L's float values, in rank order
  __shared__ int ce[kMaxE];     // L's experts, in rank order
  __shared__ int unc[kMaxE];    // position of L is uncertain
  __shared__ int uslot[kMaxE];  // slot of an uncertain position
  __shared__ int ue[kMaxE];     // expert of each slot
  __shared__ float phi[RR_THREADS], plo[RR_THREADS];
  __shared__ float fhi[kMaxE], flo[kMaxE];  // exact value of each slot
  __shared__ int flagged[MAXT];
  __shared__ int nfl, shU;
  __shared__ float shM, shS, shThr, shTau;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int t0 = blockIdx.x; t0 < n; t0 += gridDim.x * MAXT) {
    // this pass's tokens t0 + i * gridDim.x, i < MAXT: collect the flagged ones
    if (tid == 0) nfl = 0;
    __syncthreads();
    if (tid < MAXT) {
      const long long t = (long long)t0 + (long long)tid * gridDim.x;
      if (t < n && topk_idx[t * K] < 0) flagged[atomicAdd(&nfl, 1)] = (int)t;
    }
    __syncthreads();
    const int nf = nfl;
    for (int q = 0; q < nf; ++q) {
      const int t = flagged[q];
      const bool ex = tid < E;  // this thread's expert e = tid
      const float v = ex ? logits[(size_t)t * E + tid] : -INFINITY;
      if (ex) lg[tid] = v;
      __syncthreads();
      int rk = 0;
      if (ex) {
#pragma unroll 4
        for (int f = 0; f < E; ++f) rk += ranks_above(lg[f], f, v, tid);
      }
      if (warp == 0) {  // softmax statistics
        float m = -INFINITY;
        for (int e = lane; e < E; e += 32) m = fmaxf(m, lg[e]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sm = 0.f;
        for (int e = lane; e < E; e += 32) sm += expf(lg[e] - m);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
        if (lane == 0) {
          shM = m;
          shS = sm;
          shTau = tau_rel * fmaxf(1.f, fabsf(m));
        }
      }
      __syncthreads();
      if (ex && rk == K - 1) shThr = v - shTau;
      __syncthreads();
      const float thr = shThr, tau = shTau;
      const bool inL = ex && v >= thr;  // L = ranks 0 .. C-1
      if (inL) {
        cv[rk] = v;
        ce[rk] = tid;
      }
      const int C = __syncthreads_count(inL);
      if (tid < C)
        unc[tid] = (tid > 0 && cv[tid - 1] - cv[tid] < tau) ||
                   (tid + 1 < C && cv[tid] - cv[tid + 1] < tau);
      __syncthreads();
      if (warp == 0) {  // slots of the uncertain positions, in position order
        int base = 0;
        for (int p0 = 0; p0 < C; p0 += 32) {
          const int p = p0 + lane;
          const bool u = p < C && unc[p];
          const unsigned b = __ballot_sync(0xffffffffu, u);
          if (u) {
            const int sl = base + __popc(b & ((1u << lane) - 1u));
            uslot[p] = sl;
            ue[sl] = ce[p];
          }
          base += __popc(b);
        }
        if (lane == 0) shU = base;
      }
      __syncthreads();
      const int U = shU;
      // double-float dot products of the uncertain experts
      int Sp = 1;
      while (Sp < U) Sp <<= 1;
      const int G = RR_THREADS / Sp;
      const int s_id = tid & (Sp - 1), g_id = tid / Sp;
      DF acc{0.f, 0.f};
      if (s_id < U) {
        const __nv_bfloat16 *xr = x + (size_t)t * H;
        // expert ue[s_id]'s column of W_gate: a contiguous row of the
        // transposed copy when there is one, else every E-th value of W_gate
        const __nv_bfloat16 *wc = wgt ? wgt + (size_t)ue[s_id] * H : wg + ue[s_id];
        const size_t ws = wgt ? 1 : (size_t)E;
        const int nrows = (H - g_id + G - 1) / G;  // rows g_id + i * G, i < nrows
        DF a4[4] = {DF{0.f, 0.f}, DF{0.f, 0.f}, DF{0.f, 0.f}, DF{0.f, 0.f}};
        float xv[8], wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const bool in = u < nrows;
          const int h = g_id + u * G;
          xv[u] = in ? __bfloat162float(xr[h]) : 0.f;
          wv[u] = in ? __bfloat162float(wc[(size_t)h * ws]) : 0.f;
        }
        for (int i0 = 0; i0 < nrows; i0 += 8) {
          float xn[8], wn[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = i0 + 8 + u;
            const bool in = i < nrows;
            const int h = g_id + i * G;
            xn[u] = in ? __bfloat162float(xr[h]) : 0.f;
            wn[u] = in ? __bfloat162float(wc[(size_t)h * ws]) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) a4[u & 3] = df_add(a4[u & 3], two_prod(xv[u], wv[u]));
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            xv[u] = xn[u];
            wv[u] = wn[u];
          }
        }
        acc = df_add(df_add(a4[0], a4[1]), df_add(a4[2], a4[3]));
      }
      // the G partial sums of each slot: butterfly over the lanes of a warp
      // that serve the slot, then the warps in order
      int ng = G;
      if (Sp < 32) {
        for (int o = Sp; o < 32; o <<= 1) {
          const DF other{__shfl_xor_sync(0xffffffffu, acc.hi, o),
                         __shfl_xor_sync(0xffffffffu, acc.lo, o)};
          acc = df_add(acc, other);
        }
        if (lane < Sp) {
          phi[warp * Sp + lane] = acc.hi;
          plo[warp * Sp + lane] = acc.lo;
        }
        ng = RR_THREADS / 32;
      } else {
        phi[tid] = acc.hi;
        plo[tid] = acc.lo;
      }
      __syncthreads();
      if (tid < U) {
        DF sum{0.f, 0.f};
        for (int g = 0; g < ng; ++g) sum = df_add(sum, DF{phi[g * Sp + tid], plo[g * Sp + tid]});
        const float bb = bias ? bias[ue[tid]] : 0.f;
        sum = isinf(bb) ? DF{bb, 0.f} : df_add(sum, DF{bb, 0.f});
        fhi[tid] = sum.hi;
        flo[tid] = sum.lo;
      }
      __syncthreads();
      // runs of uncertain positions re-sorted by the exact values; first K out
      if (tid == 0) {
        int out[K];
        int k = 0;
        for (int p = 0; p < C && k < K;) {
          if (!unc[p]) {
            out[k++] = ce[p++];
            continue;
          }
          int r = p;
          while (r < C && unc[r]) ++r;
          for (int a = p + 1; a < r; ++a) {  // insertion sort of [p, r)
            const int ea = ce[a], sa = uslot[a];
            const DF va{fhi[sa], flo[sa]};
            int b = a - 1;
            while (b >= p && df_greater(va, ea, DF{fhi[uslot[b]], flo[uslot[b]]}, ce[b])) {
              ce[b + 1] = ce[b];
              uslot[b + 1] = uslot[b];
              --b;
            }
            ce[b + 1] = ea;
            uslot[b + 1] = sa;
          }
          for (int a = p; a < r && k < K; ++a) out[k++] = ce[a];
          p = r;
        }
        float w[K];
        float wsum = 0.f;
#pragma unroll
        for (int z = 0; z < K; ++z) {
          w[z] = expf(lg[out[z]] - shM) / shS;
          wsum += w[z];
        }
#pragma unroll
        for (int z = 0; z < K; ++z) {
          topk_idx[(size_t)t * K + z] = out[z];
          topk_w[(size_t)t * K + z] = norm ? w[z] / wsum : w[z];
        }
      }
      __syncthreads();
    }
  }
}

// Tile kernel.  A cluster of RC = 4 CTAs takes one 128-token tile; CTA c of
// the cluster runs the k-blocks [c*KB/4, (c+1)*KB/4) of the 128 x E router
// GEMM into its own TMEM accumulator, so the four CTAs stream disjoint
// quarters of x and W_gate.  After a cluster barrier (every MMA of the cluster
// done, so the operand stages are idle) each CTA's epilogue warps send row
// quarter q of their partial logits to CTA q's shared memory; after a second
// barrier CTA c adds the four partials of its 32 tokens in k order, adds the
// bias, and runs the TopK epilogue on them: 4 warps = 4 column slices of E/4
// experts, one token per lane; each thread stores its float32 logits, keeps
// their K+1 largest (descending, ties to the lower id), their max and sum of
// exp; one thread per token merges the four slices.  A token whose top K+1
// logits lie closer than the margin tau gets topk_idx[t][0] = -1 and is
// decided by router_rescore_kernel.  Every thread passes both cluster
// barriers on every path (also after a timed-out wait), so no CTA waits on a
// peer that left.
template <int KM>
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW,
                     const float *__restrict__ bias, float *__restrict__ logits,
                     int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int n, int H,
                     int E, int norm, uint32_t idesc, uint32_t tmem_cols, int32_t *status) {
  pdl_enter();
  constexpr int K = KM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nbox = E / 64;
  const int b_stage = nbox * RT_BOX_BYTES;
  const int STAGES = rt_stages(E);
  uint8_t *smemA = smem;
  uint8_t *smemB = smem + STAGES * RT_A_BYTES;
  float *red = reinterpret_cast<float *>(smem);  // after the first cluster barrier
  EpiSmem<KM> &ep = *reinterpret_cast<EpiSmem<KM> *>(smem + STAGES * (RT_A_BYTES + b_stage));
  RtTail &st = *reinterpret_cast<RtTail *>(reinterpret_cast<uint8_t *>(&ep) + epi_bytes<KM>());

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)ptx::cluster_ctarank();
  const int tile = blockIdx.x / RC;
  const int KB = H / RT_BK;
  const int kb0 = rank * KB / RC, kb1 = (rank + 1) * KB / RC;
  const bool has_k = kb1 > kb0;
  const int RS = E + 4;  // row stride of red (floats)

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&st.full[s], 1);
      ptx::mbar_init(&st.empty[s], 1);
    }
    ptx::mbar_init(&st.tfull, 1);
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
  bool acc_ok = has_k;

  if (warp == 0) {
    if (lane == 0 && has_k) {
      ptx::prefetch_tmap(&tmX);
      ptx::prefetch_tmap(&tmW);
      int stage = 0;
      uint32_t phase = 0, used = 0, last_par = 0;
      const uint32_t tx_bytes = RT_A_BYTES + b_stage;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!rt_wait(&st.empty[stage], phase ^ 1u, abort_flag, status)) break;
        ptx::mbar_arrive_expect_tx(&st.full[stage], tx_bytes);
        ptx::tma_load_2d(smemA + stage * RT_A_BYTES, &tmX, &st.full[stage], kb * RT_BK,
                         tile * RT_BM);
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
      // never leave a TMA copy in flight
      for (int s = 0; s < STAGES; ++s)
        if (used >> s & 1u) ptx::mbar_wait(&st.full[s], last_par >> s & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && has_k) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!rt_wait(&st.full[stage], phase, abort_flag, status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(smemA + stage * RT_A_BYTES);
        const uint32_t b0 = ptx::smem_u32(smemB + stage * b_stage);
#pragma unroll
        for (int kk = 0; kk < RT_BK / 16; ++kk) {
          const uint64_t adesc = ptx::smem_desc(a0 + kk * 32, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc(b0 + kk * 2048, RT_BOX_BYTES, 1024);
          ptx::mma_bf16(tmem, adesc, bdesc, idesc, (kb > kb0 || kk) ? 1u : 0u);
        }
        ptx::mma_commit(&st.empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      (void)ok;
      // the accumulator (complete, or abandoned after a timeout) and the end
      // of every MMA this thread issued
      ptx::mma_commit(&st.tfull);
      ptx::mma_commit(&st.drain);
      ptx::mbar_wait(&st.drain, 0);
    }
    __syncwarp();
  } else {
    if (has_k) acc_ok = rt_wait(&st.tfull, 0, abort_flag, status) && !*abort_flag;
    acc_ok = __all_sync(0xffffffffu, acc_ok);  // tcgen05.ld below is warp-wide
  }

  // #1: every MMA of the cluster has finished, the operand stages are idle
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp >= 2) {
    // row quarter q of this CTA's partial -> CTA q, slot `rank`
    const int q = warp & 3;
    const uint32_t dst = ptx::mapa_shared(
        ptx::smem_u32(red + ((size_t)rank * RT_ROWS + lane) * RS), (uint32_t)q);
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    for (int c = 0; c < E; c += 8) {
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (acc_ok) {  // warp-uniform
        uint32_t raw[8];
        ptx::tmem_ld_32x32b_x8(tq + c, raw);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(raw[i]);
      }
      ptx::st_cluster_v4(dst + c * 4, v[0], v[1], v[2], v[3]);
      ptx::st_cluster_v4(dst + c * 4 + 16, v[4], v[5], v[6], v[7]);
    }
  }
  // #2: this CTA's 32 rows hold the four partials
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();

  if (warp >= 2) {
    const int sl = warp - 2;             // column slice 0..3
    const int r = lane;                  // token row among this CTA's 32
    const int cols = E / RT_SLICES;
    const int c0 = sl * cols;
    const float tau_rel = tie_margin_tc(H);
    const int tok = tile * RT_BM + rank * RT_ROWS + r;
    const bool valid = tok < n;
    float *lrow = logits + (size_t)(valid ? tok : 0) * E;

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
    for (int c = 0; c < cols; c += 4) {
      float4 sum = *reinterpret_cast<const float4 *>(red + (size_t)r * RS + c0 + c);
#pragma unroll
      for (int p = 1; p < RC; ++p) {  // k order
        const float4 pv = *reinterpret_cast<const float4 *>(red + ((size_t)p * RT_ROWS + r) * RS + c0 + c);
        sum.x += pv.x;
        sum.y += pv.y;
        sum.z += pv.z;
        sum.w += pv.w;
      }
      const float v[4] = {sum.x + st.bias[c0 + c], sum.y + st.bias[c0 + c + 1],
                          sum.z + st.bias[c0 + c + 2], sum.w + st.bias[c0 + c + 3]};
      if (valid) *reinterpret_cast<float4 *>(lrow + c0 + c) = make_float4(v[0], v[1], v[2], v[3]);
      // keep the logits for the sum of exp (same smem row, partial 0's slot)
      *reinterpret_cast<float4 *>(red + (size_t)r * RS + c0 + c) = make_float4(v[0], v[1], v[2], v[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, v[i]);
        const int e = c0 + c + i;
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
    for (int c = 0; c < cols; ++c) ssum += expf(red[(size_t)r * RS + c0 + c] - m);
#pragma unroll
    for (int j = 0; j <= K; ++j) {
      ep.pv[sl][r][j] = lv[j];
      ep.pi[sl][r][j] = li[j];
    }
    ep.pm[sl][r] = m;
    ep.ps[sl][r] = ssum;
    epi_bar();

    // merge the four slices: one thread per token
    if (sl == 0 && valid) {
      float fv[K + 1];
      int fi[K + 1];
      int h0 = 0, h1 = 0, h2 = 0, h3 = 0;
#pragma unroll
      for (int j = 0; j <= K; ++j) {
        float bv = h0 <= K ? ep.pv[0][r][h0] : -INFINITY;
        int bi = h0 <= K ? ep.pi[0][r][h0] : 0x7fffffff;
        int bw = 0;
        const float v1 = h1 <= K ? ep.pv[1][r][h1] : -INFINITY;
        const int i1 = h1 <= K ? ep.pi[1][r][h1] : 0x7fffffff;
        if (ranks_above(v1, i1, bv, bi)) { bv = v1; bi = i1; bw = 1; }
        const float v2 = h2 <= K ? ep.pv[2][r][h2] : -INFINITY;
        const int i2 = h2 <= K ? ep.pi[2][r][h2] : 0x7fffffff;
        if (ranks_above(v2, i2, bv, bi)) { bv = v2; bi = i2; bw = 2; }
        const float v3 = h3 <= K ? ep.pv[3][r][h3] : -INFINITY;
        const int i3 = h3 <= K ? ep.pi[3][r][h3] : 0x7fffffff;
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
        topk_idx[(size_t)tok * K] = -1;  // flagged: router_rescore_kernel decides
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
  // the received partials must fit in the idle operand stages
  if (red_bytes(d.E) > (size_t)rt_stages(d.E) * (RT_A_BYTES + (d.E / 64) * RT_BOX_BYTES))
    return cudaErrorInvalidValue;
  uint32_t cols = 32;
  while (cols < (uint32_t)d.E) cols <<= 1;
  const int n_tiles = (d.n + RT_BM - 1) / RT_BM;
  const uint32_t idesc = ptx::idesc_bf16_f32(RT_BM, d.E, false, true);
  const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(x);
  const __nv_bfloat16 *wb = reinterpret_cast<const __nv_bfloat16 *>(w_gate);
  // one CTA per token: a CTA whose token is not flagged leaves after one load,
  // and the flagged tokens (8 % at the DeepSeek-V3 size) are rescored in
  // parallel across the SMs instead of several after one another in one CTA
  const int rgrid = d.n;
  const float tau_rel = tie_margin_tc(d.H);
  // the tile kernel (clusters of RC CTAs), then the exact rescoring of the
  // tokens it flagged
  auto run = [&](auto kernel, auto rescore, size_t smem_max, size_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_max);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(RC * n_tiles));
    cfg.blockDim = dim3(RT_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = RC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kernel, mX, mW, bias, logits, topk_idx, topk_w, d.n, d.H, d.E,
                           d.norm ? 1 : 0, idesc, cols, status);
    if (e != cudaSuccess) return e;
    return launch_pdl(rescore, dim3(rgrid), dim3(RR_THREADS), 0, s, xb, wb,
                      reinterpret_cast<const __nv_bfloat16 *>(d.w_gate_t), bias, logits,
                      topk_idx, topk_w, d.n, d.H, d.E, d.norm ? 1 : 0, tau_rel);
  };
#define MOE_RT_CASE(KK)                                                                    \
  case KK:                                                                                 \
    return run(router_tc_kernel<KK>, router_rescore_kernel<KK>,                            \
               rt_smem_bytes<KK>(64) > rt_smem_bytes<KK>(256) ? rt_smem_bytes<KK>(64)      \
                                                              : rt_smem_bytes<KK>(256),    \
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
