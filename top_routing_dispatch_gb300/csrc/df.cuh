// Double-float ("float-float") arithmetic for rescoring near-tie router
// logits: a value is an unevaluated sum hi + lo of two floats (about 48
// significant bits).  Products of two floats are exact as hi + lo (fma), and
// additions use the error-free two-sum, so a dot product of bf16 or float
// inputs accumulates with an error near 2^-46 of its magnitude.  The
// intrinsics below forbid FMA contraction and reassociation.
#pragma once

namespace moe {

struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  err = __fadd_rn(err, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s, err);
  return DF{hi, __fsub_rn(err, __fsub_rn(hi, s))};
}

__device__ __forceinline__ DF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return DF{p, fmaf(a, b, -p)};
}

// (a, ea) ranks above (b, eb): larger value, ties to the lower expert id
__device__ __forceinline__ bool df_greater(DF a, int ea, DF b, int eb) {
  if (a.hi != b.hi) return a.hi > b.hi;
  if (a.lo != b.lo) return a.lo > b.lo;
  return ea < eb;
}

}  // namespace moe
