// Router for bf16 layers with E = 64 or 128 experts and K <= 8: logits,
// softmax, TopK (with renormalisation) and the exact decision of near ties in
// ONE kernel, "MoE 分布式推理基础（基于 vLLM）" §1.2, Algorithm 2 steps 1-3 and
// the OlmoeTopKRouter code of that section.
//
// The kernel uses the warp-level tensor-core MMA (mma.sync m16n8k16, bf16 in,
// f32 accumulate) and no TMEM, so it can share an SM with the persistent
// grouped-GEMM CTA, which holds all of TMEM and ~210 KB of shared memory.  Its
// pipeline depth (STAGES) is a launch choice that does not touch the
// arithmetic: the deep configuration runs the router alone at full speed, the
// two-stage configuration (20 KB of shared memory at E = 64) fits beside a
// GEMM CTA, and both give bitwise equal results.
//
// A CTA takes 16 (or 32) tokens and all E experts (8 warps, 256 threads):
//   k loop      the x tile (the CTA's tokens x S k) and the W_gate block
//               (S k x E) of each stage are copied by cp.async into shared
//               memory (16-byte pieces, XOR-swizzled so the ldmatrix reads
//               below are free of bank conflicts), STAGES - 1 stages ahead, the
//               k range rotated per 32-token block so the CTAs do not all read
//               the same rows of W_gate at once.  Warp w takes the k16 steps g
//               with g % 8 == w for every expert (all E/8 MMA n-tiles): the A
//               fragments with ldmatrix, the B fragments with ldmatrix.trans
//               (W_gate is k-major with experts contiguous), one MMA chain per
//               warp in k order.
//   partials    the eight warps' partial logits are added in the fixed tree
//               ((p0 + p4) + (p2 + p6)) + ((p1 + p5) + (p3 + p7)) through
//               shared memory, so no result depends on the stage width, the
//               pipeline depth or the tile height.
//   logits      + bias, stored (shared memory for the TopK, and global).
//   TopK        warp w decides tokens w and w + 8: K+1 rounds of a warp argmax
//               by redux.sync (larger first, ties to the lower expert id), max
//               and sum of exp for the softmax.  If two of the top K+1 logits
//               lie closer than tau (far above the logits' float32 error) the
//               token is flagged: the warp lists the candidates (every expert
//               within tau of the K-th logit), and the positions of that list
//               whose order the float32 values leave open.
//   rescoring   the uncertain experts of every flagged token of the CTA are
//               evaluated by the whole CTA in double-float (exact products,
//               error-free sums, partial sums added in a fixed order); each
//               run of uncertain positions is re-sorted by those values, so the
//               choice is that of an exact evaluation.
#include <math.h>

#include "common.cuh"
#include "df.cuh"

namespace moe {
namespace {

constexpr int RM_WARPS = 8;
constexpr int RM_THREADS = 32 * RM_WARPS;
constexpr int RM_CAP = 64;                  // uncertain entries the CTA rescores together
constexpr int RM_UG = 4;                    // entries per pass of the CTA-wide dot products
constexpr int RM_RB = 8;                    // rows per thread per batch of those passes
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte cp.async (L2 only); valid == false writes zeros
__device__ __forceinline__ void cp16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}

// D (16x8 f32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// W_gate[h][e] for the rescoring is read at base[col(e) + h * stride]: from the
// transposed copy when there is one (expert e's column is a contiguous row of
// it: col = e * H, stride 1), else from W_gate itself (col = e, stride E).
// The same value either way.
// col(e) < 0 marks an unused entry.
struct GateCols {
  const __nv_bfloat16 *base;
  int stride;
  bool t;
  __device__ __forceinline__ int col(int e, int H) const { return e < 0 ? -1 : t ? e * H : e; }
};
__device__ __forceinline__ GateCols gate_cols(const __nv_bfloat16 *wg, const __nv_bfloat16 *wgt,
                                              int E) {
  return wgt ? GateCols{wgt, 1, true} : GateCols{wg, E, false};
}

// An order-preserving map of float32 onto uint32 (-0 taken as +0): a larger
// key is a larger value.
__device__ __forceinline__ unsigned fkey(float v) {
  const unsigned b = __float_as_uint(v + 0.f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float fkey_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The best expert not yet taken (warp-uniform): the largest value, ties to
// the lower expert id.  Lane l holds experts l + 32j in v[j]; bit j of
// `taken` marks expert l + 32j as taken.
template <int NV>
__device__ __forceinline__ void next_best(const float (&v)[NV], unsigned taken, int lane,
                                          float &bv, int &be) {
  unsigned bk = 0u;
  unsigned le = 0xffffffffu;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const unsigned k = fkey(v[j]);
    if (!(taken >> j & 1u) && (k > bk || (k == bk && (unsigned)(lane + 32 * j) < le))) {
      bk = k;
      le = (unsigned)(lane + 32 * j);
    }
  }
  const unsigned m = __reduce_max_sync(FULL, bk);
  be = (int)__reduce_min_sync(FULL, bk == m ? le : 0xffffffffu);
  bv = fkey_value(m);
}

// Index of the set bit of `m` that has `r` set bits below it (r < popc(m)).
__device__ __forceinline__ int nth_bit(unsigned m, int r) {
  for (int i = 0; i < r; ++i) m &= m - 1u;
  return __ffs(m) - 1;
}

// Per-token state of the TopK between its phases.  Position p of the rank
// order is held in slot p / 32 of lane p % 32.
template <int NV>
struct Tok {
  float m, S, tau;
  float pv[NV];
  int pe[NV];
  unsigned ub[NV];  // uncertain positions, one bit per lane per slot
  int run[NV];      // run of consecutive uncertain positions (id)
  int C, U, base;   // positions that matter, uncertain entries, first CTA entry (-1: own)
  unsigned taken;   // experts already placed (bit j of lane l: expert l + 32j)
  float vK, vK1;    // the K-th and (K+1)-th largest logits
  bool flagged;
};

// Phase 1 for the TT tokens of a warp, their rounds interleaved: rank order
// positions 0..K, softmax statistics and the near-tie flag.  lg: the CTA's
// logits rows (stride E + 4); tl[i]: the tokens' rows; valid tokens only.
template <int NV, int K, int TT>
__device__ __forceinline__ void tok_rank(Tok<NV> (&st)[TT], const float *lg, const int (&tl)[TT],
                                         int lane, float tau_rel) {
  constexpr int E = 32 * NV;
  float v[TT][NV];
#pragma unroll
  for (int i = 0; i < TT; ++i) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      v[i][j] = lg[tl[i] * (E + 4) + lane + 32 * j];
      st[i].pv[j] = -INFINITY;
      st[i].pe[j] = 0x7fffffff;
      st[i].ub[j] = 0u;
      st[i].run[j] = 0;
    }
    st[i].taken = 0u;
    st[i].flagged = false;
    st[i].C = K;
    st[i].U = 0;
    st[i].base = -1;
  }
  float prev[TT];
#pragma unroll
  for (int r = 0; r <= K; ++r) {  // K < E: K + 1 rounds
#pragma unroll
    for (int i = 0; i < TT; ++i) {
      float bv;
      int be;
      next_best<NV>(v[i], st[i].taken, lane, bv, be);
      if (lane == r) {  // r <= 8: slot 0
        st[i].pv[0] = bv;
        st[i].pe[0] = be;
      }
      if ((be & 31) == lane) st[i].taken |= 1u << (be >> 5);
      if (r == 0) {
        st[i].m = bv;
        st[i].tau = tau_rel * fmaxf(1.f, fabsf(bv));
      } else if (isfinite(prev[i]) && isfinite(bv) && prev[i] - bv < st[i].tau) {
        st[i].flagged = true;
      }
      if (r == K - 1) st[i].vK = bv;
      if (r == K) st[i].vK1 = bv;
      prev[i] = bv;
    }
  }
#pragma unroll
  for (int i = 0; i < TT; ++i) {
    float S = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) S += expf(v[i][j] - st[i].m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(FULL, S, o);
    st[i].S = S;
  }
}

// Phase 1 continued for a flagged token: the candidate list L (every expert
// within tau of the K-th logit), its uncertain positions and their entries in
// the CTA's rescoring list (ent_t, ent_e; count).
template <int NV, int K>
__device__ __forceinline__ void tok_extend(Tok<NV> &s, const float *lrow, int tl, int lane,
                                           int *ent_t, int *ent_e, int *count) {
  constexpr int E = 32 * NV;
  float v[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) v[j] = lrow[lane + 32 * j];
  unsigned taken = s.taken;
  const float tau = s.tau;
  const float thr = s.vK - tau;
  int C = K;
  if (s.vK1 >= thr) {
    // local copies: positions written inside a loop of unknown length stay
    // in registers
    float pv[NV];
    int pe[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      pv[j] = s.pv[j];
      pe[j] = s.pe[j];
    }
    C = K + 1;
    while (C < E) {
      float bv;
      int be;
      next_best<NV>(v, taken, lane, bv, be);
      if (!(bv >= thr)) break;
      const bool mine = lane == (C & 31);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const bool here = mine && j == (C >> 5);
        pv[j] = here ? bv : pv[j];
        pe[j] = here ? be : pe[j];
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      ++C;
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      s.pv[j] = pv[j];
      s.pe[j] = pe[j];
    }
  }
  s.C = C;
  // uncertain positions: a gap below tau to a neighbour in L
  bool unc[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int p = 32 * j + lane;
    float prev = __shfl_up_sync(FULL, s.pv[j], 1);
    float next = __shfl_down_sync(FULL, s.pv[j], 1);
    if (j > 0) {
      const float pl = __shfl_sync(FULL, s.pv[j - 1], 31);
      if (lane == 0) prev = pl;
    }
    if (j + 1 < NV) {
      const float nf = __shfl_sync(FULL, s.pv[j + 1], 0);
      if (lane == 31) next = nf;
    }
    unc[j] = p < C && ((p > 0 && prev - s.pv[j] < tau) || (p + 1 < C && s.pv[j] - next < tau));
    s.ub[j] = __ballot_sync(FULL, unc[j]);
  }
  // runs of consecutive uncertain positions: run id = run starts at or before p
  int nstart = 0, nunc = 0;
  const unsigned upto = (2u << lane) - 1u;
  const unsigned below = (1u << lane) - 1u;
  int rank_in_list[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const unsigned prevbit = (s.ub[j] << 1) | (j > 0 ? s.ub[j - 1] >> 31 : 0u);
    const unsigned sb = s.ub[j] & ~prevbit;
    s.run[j] = nstart + __popc(sb & upto);
    nstart += __popc(sb);
    rank_in_list[j] = nunc + __popc(s.ub[j] & below);
    nunc += __popc(s.ub[j]);
  }
  s.U = nunc;
  // entries in the CTA's rescoring list, in position order
  int base = 0;
  if (lane == 0) base = atomicAdd(count, nunc);
  base = __shfl_sync(FULL, base, 0);
  const bool fits = base + nunc <= RM_CAP;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    if (unc[j]) {
      const int d = base + rank_in_list[j];
      if (d < RM_CAP) {  // an entry that does not fit is marked unused
        ent_t[d] = fits ? tl : 0;
        ent_e[d] = fits ? s.pe[j] : -1;
      }
    }
  }
  s.base = fits ? base : -1;
}

// Exact logits of up to RM_UG uncertain experts of one flagged token, by one
// warp (used when the CTA's list is full): double-float products over H.
template <int NV>
__device__ __forceinline__ void warp_rescore(const Tok<NV> &s, float (&ex_hi)[NV], float (&ex_lo)[NV], int lane,
                             const __nv_bfloat16 *__restrict__ xr,
                             const __nv_bfloat16 *__restrict__ wg,
                             const __nv_bfloat16 *__restrict__ wgt, const float *__restrict__ bias,
                             int E, int H) {
  constexpr int UG = RM_UG, RU = 8;
  for (int u0 = 0; u0 < s.U; u0 += UG) {
    int eu[UG], pu[UG];
#pragma unroll
    for (int i = 0; i < UG; ++i) {  // position and expert of uncertain entry u0 + i
      int rem = u0 + i, pos = -1, ex = 0;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int cnt = __popc(s.ub[j]);
        const bool here = pos < 0 && rem < cnt;  // warp-uniform
        const int ln = here ? nth_bit(s.ub[j], rem) : 0;
        const int te = __shfl_sync(FULL, s.pe[j], ln);
        if (here) {
          pos = 32 * j + ln;
          ex = te;
        } else if (pos < 0) {
          rem -= cnt;
        }
      }
      pu[i] = pos;
      eu[i] = pos >= 0 ? ex : -1;
    }
    DF acc[UG];
#pragma unroll
    for (int i = 0; i < UG; ++i) acc[i] = DF{0.f, 0.f};
    const GateCols gc = gate_cols(wg, wgt, E);
    int wcol[UG];
#pragma unroll
    for (int i = 0; i < UG; ++i) wcol[i] = gc.col(eu[i], H);
    for (int h0 = lane; h0 < H; h0 += 32 * RU) {
      float xv[RU], wv[RU][UG];
#pragma unroll
      for (int r = 0; r < RU; ++r) {
        const int hh = h0 + 32 * r;
        const bool in = hh < H;
        xv[r] = in ? __bfloat162float(xr[hh]) : 0.f;
#pragma unroll
        for (int i = 0; i < UG; ++i)
          wv[r][i] = (in && wcol[i] >= 0)
                         ? __bfloat162float(gc.base[(size_t)wcol[i] + (size_t)hh * gc.stride])
                         : 0.f;
      }
#pragma unroll
      for (int r = 0; r < RU; ++r)
#pragma unroll
        for (int i = 0; i < UG; ++i) acc[i] = df_add(acc[i], two_prod(xv[r], wv[r][i]));
    }
#pragma unroll
    for (int i = 0; i < UG; ++i) {
      DF a = acc[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const DF other{__shfl_xor_sync(FULL, a.hi, o), __shfl_xor_sync(FULL, a.lo, o)};
        a = df_add(a, other);
      }
      if (eu[i] >= 0) {
        if (bias) {
          const float bb = bias[eu[i]];
          a = isinf(bb) ? DF{bb, 0.f} : df_add(a, DF{bb, 0.f});
        }
#pragma unroll
        for (int j = 0; j < NV; ++j)
          if (j == (pu[i] >> 5) && lane == (pu[i] & 31)) {
            ex_hi[j] = a.hi;
            ex_lo[j] = a.lo;
          }
      }
    }
  }
}

// Phase 3 for one token: the exact values of its uncertain positions (from
// the CTA's list, or computed by this warp), the final order, and the K
// experts with their softmax weights.
template <int NV, int K>
__device__ __forceinline__ void tok_finish(const Tok<NV> &s, int t, int lane,
                                           const float *ex_hi_l, const float *ex_lo_l,
                                           const __nv_bfloat16 *__restrict__ x,
                                           const __nv_bfloat16 *__restrict__ wg,
                                           const __nv_bfloat16 *__restrict__ wgt,
                                           const float *__restrict__ bias, int E, int H, int norm,
                                           int32_t *__restrict__ topk_idx,
                                           float *__restrict__ topk_w) {
  int fin[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) fin[j] = 32 * j + lane;
  if (s.flagged) {  // warp-uniform
    float ex_hi[NV], ex_lo[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      ex_hi[j] = 0.f;
      ex_lo[j] = 0.f;
    }
    if (s.base >= 0) {
      int nunc = 0;
      const unsigned below = (1u << lane) - 1u;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        if (s.ub[j] >> lane & 1u) {
          const int d = s.base + nunc + __popc(s.ub[j] & below);
          ex_hi[j] = ex_hi_l[d];
          ex_lo[j] = ex_lo_l[d];
        }
        nunc += __popc(s.ub[j]);
      }
    } else {
      warp_rescore<NV>(s, ex_hi, ex_lo, lane, x + (size_t)t * H, wg, wgt, bias, E, H);
    }
    // an uncertain position moves inside its run by (members ranked above it
    // by the exact values) - (members before it)
    int shift[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) shift[j] = 0;
    for (int u = 0; u < s.U; ++u) {
      int rem = u, pos = -1;
      float uh = 0.f, ul = 0.f;
      int ue = 0, ur = 0;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int cnt = __popc(s.ub[j]);
        const bool here = pos < 0 && rem < cnt;  // warp-uniform
        const int ln = here ? nth_bit(s.ub[j], rem) : 0;
        const float th = __shfl_sync(FULL, ex_hi[j], ln);
        const float tl = __shfl_sync(FULL, ex_lo[j], ln);
        const int te = __shfl_sync(FULL, s.pe[j], ln);
        const int tr = __shfl_sync(FULL, s.run[j], ln);
        if (here) {
          pos = 32 * j + ln;
          uh = th;
          ul = tl;
          ue = te;
          ur = tr;
        } else if (pos < 0) {
          rem -= cnt;
        }
      }
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int p = 32 * j + lane;
        if ((s.ub[j] >> lane & 1u) && s.run[j] == ur && p != pos) {
          if (df_greater(DF{uh, ul}, ue, DF{ex_hi[j], ex_lo[j]}, s.pe[j])) ++shift[j];
          if (pos < p) --shift[j];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) fin[j] += shift[j];
  }
  // weights of the K chosen experts: softmax of the float32 logits
  float w[NV];
  float tot = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const bool chosen = 32 * j + lane < s.C && fin[j] < K;
    w[j] = chosen ? expf(s.pv[j] - s.m) / s.S : 0.f;
    tot += w[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    if (32 * j + lane < s.C && fin[j] < K) {
      topk_idx[(size_t)t * K + fin[j]] = s.pe[j];
      topk_w[(size_t)t * K + fin[j]] = norm ? w[j] / tot : w[j];
    }
  }
}

// The arithmetic of one logit: warp w accumulates the k16 steps g with
// g % 8 == w in order (one MMA chain per warp), and the eight partial sums are
// added as ((p0 + p4) + (p2 + p6)) + ((p1 + p5) + (p3 + p7)).  The tile shape
// (MT m-tiles of 16 tokens per CTA), the stage width S and the pipeline depth
// STAGES only decide how the operands reach shared memory, so every
// configuration gives the same bits.
template <int EG, int K, int MT, int S, int STAGES>
__device__ __forceinline__ void route_tile(const __nv_bfloat16 *__restrict__ x,
                                           const __nv_bfloat16 *__restrict__ wg,
                                           const __nv_bfloat16 *__restrict__ wgt,
                                           const float *__restrict__ bias,
                                           float *__restrict__ logits,
                                           int32_t *__restrict__ topk_idx,
                                           float *__restrict__ topk_w, int n, int H, int norm,
                                           float tau_rel, int t0, uint8_t *rm_smem);

// One CTA per tile of 16 MT tokens (a grid-stride loop over the tiles when the
// grid is smaller).
template <int EG, int K, int MT, int S, int STAGES>
__global__ void __launch_bounds__(RM_THREADS)
    router_mma_kernel(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ wg,
                      const __nv_bfloat16 *__restrict__ wgt, const float *__restrict__ bias,
                      float *__restrict__ logits,
                      int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int n, int H,
                      int norm, float tau_rel) {
  static_assert(STAGES >= 2 && S % 64 == 0, "stages of whole 128-byte x rows");
  constexpr int TOK = 16 * MT;
  extern __shared__ __align__(128) uint8_t rm_smem[];
  pdl_enter();
  const int ntile = (n + TOK - 1) / TOK;
  for (int tile = blockIdx.x; tile < ntile; tile += gridDim.x) {
    if (tile != (int)blockIdx.x) __syncthreads();  // the previous tile is done with smem
    route_tile<EG, K, MT, S, STAGES>(x, wg, wgt, bias, logits, topk_idx, topk_w, n, H, norm,
                                     tau_rel, tile * TOK, rm_smem);
  }
}

template <int EG, int K, int MT, int S, int STAGES>
__device__ __forceinline__ void route_tile(const __nv_bfloat16 *__restrict__ x,
                                           const __nv_bfloat16 *__restrict__ wg,
                                           const __nv_bfloat16 *__restrict__ wgt,
                                           const float *__restrict__ bias,
                                           float *__restrict__ logits,
                                           int32_t *__restrict__ topk_idx,
                                           float *__restrict__ topk_w, int n, int H, int norm,
                                           float tau_rel, int t0, uint8_t *rm_smem) {
  constexpr int E = 64 * EG;
  constexpr int NV = E / 32;
  constexpr int NT = E / 8;                       // n-tiles, all held by every warp
  constexpr int TOK = 16 * MT;
  constexpr int XB = TOK * S * 2, SB = XB + S * E * 2;
  constexpr int XROW = S * 2, WROW = E * 2;       // bytes per staged row
  constexpr int TT = TOK / RM_WARPS;              // tokens per warp in the TopK
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(rm_smem);

  // Stage st holds k [k0, k0 + S) with the k range rotated by `rot` blocks of
  // 128 (the same for every configuration: it depends on the 32-token block),
  // so the CTAs do not all read the same rows of W_gate at the same time.
  const int nst = H / S;
  const int rot = ((t0 / 32) % (H / 128)) * (128 / S);
  auto load_stage = [&](int st, int buf) {
    const int k0 = ((st + rot) % nst) * S;
    const uint32_t xs = sbase + buf * SB, ws = xs + XB;
#pragma unroll
    for (int i = tid; i < TOK * (S / 8); i += RM_THREADS) {  // x: TOK rows x S/8 pieces
      const int t = i / (S / 8), j = i % (S / 8);
      const bool ok = t0 + t < n;
      cp16(xs + t * XROW + ((j ^ (t & 7)) << 4), x + (ok ? (size_t)(t0 + t) * H + k0 + 8 * j : 0),
           ok);
    }
#pragma unroll
    for (int i = tid; i < S * (E / 8); i += RM_THREADS) {  // W_gate: S rows x E/8 pieces
      const int k = i / (E / 8), j = i % (E / 8);
      cp16(ws + k * WROW + ((j ^ (k & 7)) << 4), wg + (size_t)(k0 + k) * E + 8 * j, true);
    }
  };
  float acc[MT][NT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[m][t][j] = 0.f;
#pragma unroll
  for (int i = 0; i < STAGES - 1; ++i) {
    if (i < nst) load_stage(i, i);
    cp_commit();
  }
  // this lane's ldmatrix rows: A (x4): token row (lane & 7) + 8 ((lane >> 3) & 1)
  // of an m-tile, k half lane >> 4; B (x4.trans): k row (lane & 7) + 8 ((lane >> 3)
  // & 1), n-tile (pair member) lane >> 4
  const int a_t = (lane & 7) + 8 * ((lane >> 3) & 1), a_h = lane >> 4;
  const int b_k = (lane & 7) + 8 * ((lane >> 3) & 1), b_n = lane >> 4;
  for (int it = 0; it < nst; ++it) {
    cp_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nx = it + STAGES - 1;
      if (nx < nst) load_stage(nx, nx % STAGES);
      cp_commit();
    }
    const uint32_t xs = sbase + (it % STAGES) * SB, ws = xs + XB;
    // this warp's k16 step of the stage, if it has one: the step g of the
    // rotated order with g % 8 == warp
    const int s = (warp - it * (S / 16)) & 7;
    if (s < S / 16) {  // warp-uniform
      uint32_t a[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int t = 16 * m + a_t;
        ldsm_x4(xs + t * XROW + (((2 * s + a_h) ^ (t & 7)) << 4), a[m][0], a[m][1], a[m][2],
                a[m][3]);
      }
      const int k = 16 * s + b_k;
#pragma unroll
      for (int p = 0; p < NT / 2; ++p) {
        uint32_t b0, b1, b2, b3;
        const int nt = 2 * p + b_n;
        ldsm_x4_t(ws + k * WROW + ((nt ^ (k & 7)) << 4), b0, b1, b2, b3);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          mma16816(acc[m][2 * p], a[m][0], a[m][1], a[m][2], a[m][3], b0, b1);
          mma16816(acc[m][2 * p + 1], a[m][0], a[m][1], a[m][2], a[m][3], b2, b3);
        }
      }
    }
  }
  cp_wait<0>();
  __syncthreads();  // every stage consumed: the areas below alias them

  // ---- partial sums of the eight warps, added in a fixed tree
  constexpr int RS = E + 4;  // row stride (floats) of a partial tile
  float *red = reinterpret_cast<float *>(rm_smem);
  const int g = lane >> 2, q = lane & 3;
#pragma unroll 1
  for (int half = 4; half >= 1; half >>= 1) {
    if (warp >= half && warp < 2 * half) {
      float *b = red + (size_t)(warp - half) * TOK * RS;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          *reinterpret_cast<float2 *>(b + (16 * m + g) * RS + 8 * t + 2 * q) =
              make_float2(acc[m][t][0], acc[m][t][1]);
          *reinterpret_cast<float2 *>(b + (16 * m + g + 8) * RS + 8 * t + 2 * q) =
              make_float2(acc[m][t][2], acc[m][t][3]);
        }
    }
    __syncthreads();
    if (warp < half) {
      const float *b = red + (size_t)warp * TOK * RS;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float2 u = *reinterpret_cast<const float2 *>(b + (16 * m + g) * RS + 8 * t + 2 * q);
          const float2 w = *reinterpret_cast<const float2 *>(b + (16 * m + g + 8) * RS + 8 * t + 2 * q);
          acc[m][t][0] += u.x;
          acc[m][t][1] += u.y;
          acc[m][t][2] += w.x;
          acc[m][t][3] += w.y;
        }
    }
    __syncthreads();
  }
  // ---- logits (+ bias) from warp 0: rows of lg (same positions it just read)
  float *lg = red;  // [TOK][E + 4]
  int *ent_t = reinterpret_cast<int *>(lg + TOK * RS);
  int *ent_e = ent_t + RM_CAP;
  float *ex_hi = reinterpret_cast<float *>(ent_e + RM_CAP);
  float *ex_lo = ex_hi + RM_CAP;
  float *part_hi = ex_lo + RM_CAP;
  float *part_lo = part_hi + RM_WARPS * RM_UG;
  int *count = reinterpret_cast<int *>(part_lo + RM_WARPS * RM_UG);
  if (warp == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int e = 8 * t + 2 * q;
      const float b0 = bias ? bias[e] : 0.f, b1 = bias ? bias[e + 1] : 0.f;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        *reinterpret_cast<float2 *>(lg + (16 * m + g) * RS + e) =
            make_float2(acc[m][t][0] + b0, acc[m][t][1] + b1);
        *reinterpret_cast<float2 *>(lg + (16 * m + g + 8) * RS + e) =
            make_float2(acc[m][t][2] + b0, acc[m][t][3] + b1);
      }
    }
  }
  if (tid == 0) *count = 0;
  __syncthreads();
  for (int i = tid; i < TOK * (E / 4); i += RM_THREADS) {
    const int r = i / (E / 4), c4 = i % (E / 4);
    if (t0 + r < n)
      *reinterpret_cast<float4 *>(logits + (size_t)(t0 + r) * E + 4 * c4) =
          *reinterpret_cast<const float4 *>(lg + r * RS + 4 * c4);
  }

  // ---- TopK: warp w takes tokens w + 8 i, two at a time with their rounds
  // interleaved; each pair of rounds has its own rescoring pass
  const int nvalid = n - t0;  // tokens of this CTA that exist (>= 1)
#pragma unroll 1
  for (int grp = 0; grp < TT; grp += 2) {
    if (grp > 0) {
      __syncthreads();  // the previous pair is done with the rescoring area
      if (tid == 0) *count = 0;
      __syncthreads();
    }
    Tok<NV> st[2];
    const int tl[2] = {warp + RM_WARPS * grp, warp + RM_WARPS * (grp + 1)};
    tok_rank<NV, K, 2>(st, lg, tl, lane, tau_rel);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (tl[i] < nvalid && st[i].flagged)  // warp-uniform
        tok_extend<NV, K>(st[i], lg + tl[i] * RS, tl[i], lane, ent_t, ent_e, count);
    __syncthreads();
    // CTA-wide double-float dot products of the listed uncertain experts
    const int D = min(*count, RM_CAP);
    for (int d0 = 0; d0 < D; d0 += RM_UG) {
      int ee[RM_UG];
      const __nv_bfloat16 *xr[RM_UG];
#pragma unroll
      for (int i = 0; i < RM_UG; ++i) {
        const int d = d0 + i;
        ee[i] = d < D ? ent_e[d] : -1;
        xr[i] = x + (size_t)(t0 + (d < D ? ent_t[d] : 0)) * H;
      }
      DF a[RM_UG];
#pragma unroll
      for (int i = 0; i < RM_UG; ++i) a[i] = DF{0.f, 0.f};
      const GateCols gc = gate_cols(wg, wgt, E);
      int wcol[RM_UG];
      int my_e = -1;  // thread tid < RM_UG adds up entry d0 + tid below
#pragma unroll
      for (int i = 0; i < RM_UG; ++i) {
        wcol[i] = gc.col(ee[i], H);
        if (tid == i) my_e = ee[i];
      }
      for (int h0 = 0; h0 < H; h0 += RM_THREADS * RM_RB) {
        float xv[RM_RB][RM_UG], wv[RM_RB][RM_UG];
#pragma unroll
        for (int rr = 0; rr < RM_RB; ++rr) {
          const int h = h0 + rr * RM_THREADS + tid;
#pragma unroll
          for (int i = 0; i < RM_UG; ++i) {
            const bool in = h < H && wcol[i] >= 0;
            xv[rr][i] = in ? __bfloat162float(xr[i][h]) : 0.f;
            wv[rr][i] = in ? __bfloat162float(gc.base[(size_t)wcol[i] + (size_t)h * gc.stride])
                           : 0.f;
          }
        }
#pragma unroll
        for (int rr = 0; rr < RM_RB; ++rr)
#pragma unroll
          for (int i = 0; i < RM_UG; ++i) a[i] = df_add(a[i], two_prod(xv[rr][i], wv[rr][i]));
      }
#pragma unroll
      for (int i = 0; i < RM_UG; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const DF other{__shfl_xor_sync(FULL, a[i].hi, o), __shfl_xor_sync(FULL, a[i].lo, o)};
          a[i] = df_add(a[i], other);
        }
        if (lane == 0) {
          part_hi[warp * RM_UG + i] = a[i].hi;
          part_lo[warp * RM_UG + i] = a[i].lo;
        }
      }
      __syncthreads();
      if (tid < RM_UG && my_e >= 0) {  // the warps' partial sums in order, then the bias
        DF sum{0.f, 0.f};
        for (int w = 0; w < RM_WARPS; ++w)
          sum = df_add(sum, DF{part_hi[w * RM_UG + tid], part_lo[w * RM_UG + tid]});
        if (bias) {
          const float bb = bias[my_e];
          sum = isinf(bb) ? DF{bb, 0.f} : df_add(sum, DF{bb, 0.f});
        }
        ex_hi[d0 + tid] = sum.hi;
        ex_lo[d0 + tid] = sum.lo;
      }
      __syncthreads();
    }
    // final order and weights
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (tl[i] < nvalid)
        tok_finish<NV, K>(st[i], t0 + tl[i], lane, ex_hi, ex_lo, x, wg, wgt, bias, E, H, norm,
                          topk_idx, topk_w);
  }
}

// Shared memory of a configuration: the stages, or the partial-sum tree and
// the TopK area that alias them afterwards, whichever is larger.
__host__ __device__ constexpr int rm_smem_bytes(int E, int MT, int S, int stages) {
  const int pipe = stages * (16 * MT * S * 2 + S * E * 2);
  const int red = 4 * 16 * MT * (E + 4) * 4;
  const int epi = 16 * MT * (E + 4) * 4 + 4 * RM_CAP * 4 + 2 * RM_WARPS * RM_UG * 4 + 16;
  const int tail = red > epi ? red : epi;
  return pipe > tail ? pipe : tail;
}

// Configurations (every one gives the same bits): beside a GEMM CTA ("guest"),
// 16 tokens per CTA and two 64-wide stages (20 KB of shared memory at E = 64);
// alone, four stages 128 wide at E = 64 (64 wide at E = 128), with 16 tokens
// per CTA while the tiles fit in one wave of two CTAs per SM, else 32 (E = 64:
// each CTA then reads W_gate for twice the tokens).
template <int EG, int K, int MT, int S, int STAGES>
cudaError_t launch_cfg(const Desc &d, const void *x, const void *w_gate, const float *bias,
                       int32_t *topk_idx, float *topk_w, float *logits, bool guest,
                       cudaStream_t s) {
  constexpr int E = 64 * EG;
  auto kernel = router_mma_kernel<EG, K, MT, S, STAGES>;
  constexpr int smem = rm_smem_bytes(E, MT, S, STAGES);
  if (d.H % S) return cudaErrorInvalidValue;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    if (smem > 48 * 1024)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = prefer_max_shared(kernel);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int tiles = (d.n + 16 * MT - 1) / (16 * MT);
  const int sms = device_sm_count();
  const int grid = guest && tiles > sms ? sms : tiles;
  return launch_k(guest, kernel, dim3(grid), dim3(RM_THREADS), (size_t)smem, s,
                  reinterpret_cast<const __nv_bfloat16 *>(x),
                  reinterpret_cast<const __nv_bfloat16 *>(w_gate),
                  reinterpret_cast<const __nv_bfloat16 *>(d.w_gate_t), bias, logits, topk_idx,
                  topk_w, d.n, d.H, d.norm ? 1 : 0, tie_margin_tc(d.H));
}

template <int EG, int K>
cudaError_t launch_mma(const Desc &d, const void *x, const void *w_gate, const float *bias,
                       int32_t *topk_idx, float *topk_w, float *logits, bool guest,
                       cudaStream_t s) {
  if (guest)
    return launch_cfg<EG, K, 1, 64, 2>(d, x, w_gate, bias, topk_idx, topk_w, logits, true, s);
  if constexpr (EG == 2) {
    return launch_cfg<EG, K, 1, 64, 4>(d, x, w_gate, bias, topk_idx, topk_w, logits, false, s);
  } else {
    if ((d.n + 15) / 16 <= 2 * device_sm_count())
      return launch_cfg<EG, K, 1, 128, 4>(d, x, w_gate, bias, topk_idx, topk_w, logits, false, s);
    return launch_cfg<EG, K, 2, 128, 4>(d, x, w_gate, bias, topk_idx, topk_w, logits, false, s);
  }
}

template <int EG>
cudaError_t launch_mma_k(const Desc &d, const void *x, const void *w_gate, const float *bias,
                         int32_t *topk_idx, float *topk_w, float *logits, bool guest,
                         cudaStream_t s) {
  switch (d.K) {
    case 1: return launch_mma<EG, 1>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    case 2: return launch_mma<EG, 2>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    case 3: return launch_mma<EG, 3>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    case 4: return launch_mma<EG, 4>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    case 5: return launch_mma<EG, 5>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    case 6: return launch_mma<EG, 6>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    case 7: return launch_mma<EG, 7>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    case 8: return launch_mma<EG, 8>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool router_mma_supported(const Desc &d) {
  return d.bf16 && (d.E == 64 || d.E == 128) && d.H % 128 == 0 && d.n > 0 && d.K >= 1 &&
         d.K <= 8 && d.K < d.E;
}

cudaError_t launch_router_mma(const Desc &d, const void *x, const void *w_gate, const float *bias,
                              int32_t *topk_idx, float *topk_w, float *logits, bool guest,
                              cudaStream_t s) {
  if (!router_mma_supported(d)) return cudaErrorInvalidValue;
  if (d.E == 64) return launch_mma_k<1>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
  return launch_mma_k<2>(d, x, w_gate, bias, topk_idx, topk_w, logits, guest, s);
}

}  // namespace moe
