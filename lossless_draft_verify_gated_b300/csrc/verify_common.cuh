// verify_common.cuh -- device helpers shared by the verifier kernels
// (verify.cu: the block verifier and draft sampler; tree.cu: the tree
// sampler; lm_head.cu: the LM head's decide and race kernels): the online
// (max, sum exp) of a logit row and the candidates of the exponential race.
#pragma once

#include <cmath>
#include <cstdint>

namespace uno {
namespace vfy {

struct MS {
  float m, s;  // running max and sum of exp(x - m)
};

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, a.s + b.s};
  return {m, a.s * __expf(a.m - m) + b.s * __expf(b.m - m)};
}

// Fold four logits into a running (max, sum).  NaN poisons s; +inf makes
// s NaN through inf - inf; -inf entries contribute exactly 0.
__device__ __forceinline__ void ms_add4(MS& a, float x0, float x1, float x2, float x3) {
  const float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  if (mx > a.m) {
    a.s *= __expf(a.m - mx);
    a.m = mx;
  }
  if (a.m != -INFINITY) {
    a.s += __expf(x0 - a.m) + __expf(x1 - a.m) + __expf(x2 - a.m) + __expf(x3 - a.m);
  } else if (isnan(x0) || isnan(x1) || isnan(x2) || isnan(x3)) {
    a.s = NAN;
  }
}

__device__ __forceinline__ void ms_add1(MS& a, float x) {
  ms_add4(a, x, -INFINITY, -INFINITY, -INFINITY);
}

__device__ __forceinline__ MS warp_merge(MS a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS b{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o)};
    a = ms_merge(a, b);
  }
  return a;
}

struct Cand {
  float s;  // race score
  int v;    // vocab id, -1 = none
};

__device__ __forceinline__ Cand cand_best(Cand a, Cand b) {
  if (b.s > a.s || (b.s == a.s && b.v >= 0 && (a.v < 0 || b.v < a.v))) return b;
  return a;
}

__device__ __forceinline__ Cand warp_best(Cand a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand b{__shfl_xor_sync(0xffffffffu, a.s, o), __shfl_xor_sync(0xffffffffu, a.v, o)};
    a = cand_best(a, b);
  }
  return a;
}

// Candidates as 64-bit keys whose unsigned order is cand_best's: the score
// (IEEE bits made order-preserving; NaN lowest) above the id (2^31 - v for
// a token, 0 for none, so a lower id and a token over none win ties).  The
// race's chunk winners then merge by atomic max, in any order.
__device__ __forceinline__ unsigned long long cand_key(Cand c) {
  uint32_t u = __float_as_uint(c.s);
  u = isnan(c.s) ? 0u : (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  const uint32_t lo = c.v >= 0 ? 0x80000000u - uint32_t(c.v) : 0u;
  return (static_cast<unsigned long long>(u) << 32) | lo;
}
__device__ __forceinline__ Cand cand_of_key(unsigned long long k) {
  const uint32_t hi = uint32_t(k >> 32), lo = uint32_t(k);
  const uint32_t u = (hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi;
  return Cand{__uint_as_float(u), lo ? int(0x80000000u - lo) : -1};
}

struct RacePart {
  float sr;  // best residual score in the chunk (0 if no positive residual)
  int vr;
  float sp;  // best score of the AR row itself (fallback and bonus race)
  int vp;
};
// (inverse CDF) the same slot holds the chunk's residual and AR weight sums
static_assert(sizeof(RacePart) == sizeof(longlong2), "chunk sums share the race slot");

}  // namespace vfy
}  // namespace uno
