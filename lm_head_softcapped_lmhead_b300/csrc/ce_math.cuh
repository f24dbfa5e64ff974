// ce_math.cuh -- the cross-entropy arithmetic shared by the forward finalize
// and the forward + dh pass's drain.
#pragma once

namespace lmce {

// nll = -ln p_t = log1p(S_other / e^{s_t}) in fp32 from the row's sum of e^s
// over the non-target columns and the target's term: relative-precise as
// p_t -> 1.  Where the ratio passes fp32's range (a softcap above about 40
// with saturated logits: up to V e^{2c}), ln S_other - ln e^{s_t} gives the
// same value to a few ulp of a result above 87.
__device__ __forceinline__ float nll_from_sums(float S_other, float et) {
  const float r = S_other / et;
  return r <= 1e37f ? log1pf(r) : logf(S_other) - logf(et);
}

}  // namespace lmce
