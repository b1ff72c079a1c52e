// Mergeable per-row acceptance statistics: the argmax of a logit row and,
// for typical acceptance, the softmax sums at a temperature, over any subset
// of the vocabulary.  Used by the LM head's fused epilogue (records per
// vocabulary group) and by the acceptance that merges them.
#pragma once

#include <math.h>

#include "common.cuh"

namespace medusa {

struct StatRec {
  float v;  // max logit
  int i;    // its index (lowest among equal maxima)
  float S;  // sum e^(y - m), y = logit * inv_temp, m = v * inv_temp (0: empty)
  float A;  // sum e^(y - m) (y - m)
};

MDEV StatRec stat_empty() {
  StatRec r;
  r.v = -INFINITY; r.i = 0x7fffffff; r.S = 0.f; r.A = 0.f;
  return r;
}
MDEV StatRec stat_load(float4 x) {
  StatRec r;
  r.v = x.x; r.i = __float_as_int(x.y); r.S = x.z; r.A = x.w;
  return r;
}
MDEV float4 stat_store(const StatRec& r) { return make_float4(r.v, __int_as_float(r.i), r.S, r.A); }

// Symmetric in its arguments, bit for bit (lane pairs that merge the same two
// records get the same result).  max y = (max logit) * inv_temp since a
// positive scale is monotone in floating point.
template <bool TYP>
MDEV StatRec stat_merge(const StatRec& a, const StatRec& b, float inv_temp) {
  StatRec r;
  const bool tb = b.v > a.v || (b.v == a.v && b.i < a.i);
  r.v = tb ? b.v : a.v;
  r.i = tb ? b.i : a.i;
  r.S = 0.f;
  r.A = 0.f;
  if (TYP) {
    const float ma = a.v * inv_temp, mb = b.v * inv_temp, M = fmaxf(ma, mb);
    const float ea = a.S > 0.f ? expf(ma - M) : 0.f, eb = b.S > 0.f ? expf(mb - M) : 0.f;
    r.S = a.S * ea + b.S * eb;
    r.A = (a.S > 0.f ? ea * (a.A + (ma - M) * a.S) : 0.f) + (b.S > 0.f ? eb * (b.A + (mb - M) * b.S) : 0.f);
  }
  return r;
}

}  // namespace medusa
