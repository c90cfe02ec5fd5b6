// Arithmetic shared by the sampling-adjustment selection and the acceptance
// kernels, so that both see the same probabilities bit for bit.
//
// Lecture 6 "Optimizing Autoregressive Decode" section 7.3: temperature, top-k
// and top-p are all sampling from an adjusted distribution, and speculative
// sampling run on the adjusted p (and the draft's q, adjusted the same way)
// follows the adjusted p.  Here the adjustment of one row is described by a
// SelRow: the kept tokens are those whose probability key (the fp32 bit pattern
// of p, which orders like p for p >= 0) is above t, or equal to t with a token
// index <= cut; kept token v gets fl32(fl64(R_v) * fl64(1 / Z)) with
// R_v = floor(p_v * 2^40) and Z the kept tokens' summed R.  Z == 0 marks a row
// without adjustment (p is used as it is).
#pragma once

#include "common.cuh"

namespace spec {

struct SelRow {
  uint32_t t;              // probability key of the last kept rank
  int32_t cut;             // tokens with key == t are kept up to this index
  unsigned long long Z;    // summed 2^-40 masses of the kept tokens; 0 = no adjustment
};

// Probability of token v from its logit and the row's softmax statistics.  The
// operations are pinned (no contraction), so every kernel gets the same value.
SPEC_DEVICE_INLINE float prob_from_logit(float logit, float row_max, float inv_temp, float row_z) {
  return __fdiv_rn(expf(__fmul_rn(__fsub_rn(logit, row_max), inv_temp)), row_z);
}

SPEC_DEVICE_INLINE uint32_t prob_key(float pv) { return pv > 0.f ? __float_as_uint(pv) : 0u; }

// floor(r * 2^40) for 0 <= r <= 1: exact (power-of-two scaling, then floor).
SPEC_DEVICE_INLINE unsigned long long grid_mass(float r) {
  return (unsigned long long)floorf(r * 1099511627776.0f);
}

SPEC_DEVICE_INLINE unsigned long long key_mass(uint32_t key) { return grid_mass(__uint_as_float(key)); }

SPEC_DEVICE_INLINE double sel_inv_z(const SelRow& s) { return s.Z ? __ddiv_rn(1.0, (double)s.Z) : 0.0; }

// Adjusted probability of token v whose unadjusted probability is pv.
SPEC_DEVICE_INLINE float adjusted_prob(float pv, int v, const SelRow& s, double inv_z) {
  if (s.Z == 0ull) return pv;
  const uint32_t key = prob_key(pv);
  const bool kept = key > s.t || (key == s.t && v <= s.cut);
  return kept ? __double2float_rn(__dmul_rn((double)key_mass(key), inv_z)) : 0.f;
}

}  // namespace spec
