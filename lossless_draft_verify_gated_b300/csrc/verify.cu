// verify.cu -- block verifier and draft sampler of the Psi-Spec linear sampler.
//
// "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
// (aifromscratch.in), section "The Psi-Spec Sampler": a block drafted in
// parallel is checked against the AR model by rejection sampling (as in
// speculative decoding): drafts are kept up to the first rejection and the
// emitted tokens follow the AR model's distribution; the linear sampler draws
// a single token at each position.  "Uno Uses Discrete Diffusion to Accelerate LLMs Without Loss"
// (cctest.ai), section "What 'lossless' means here": the AR model rejects or
// adjusts candidates.
//
// The verifier is bound by HBM: every AR and draft logit is read once (8 bytes
// per (position, vocab entry)).  Two launches:
//   stats  -- one CTA per (row, vocab chunk); 128-bit streaming loads, an
//             online (max, sum exp) per thread, warp-shuffle merge, one
//             partial per CTA.  Rows of all sequences are spread over the grid,
//             and short rows are split so the grid fills the 148 SMs.
//   finish -- one CTA per (sequence, vocab chunk); every CTA of a sequence
//             merges the partials of that sequence (identically), takes the
//             accept decisions and the prefix length n, then races its chunk
//             of the residual row (or the bonus row), folds its winners into
//             the sequence's two 64-bit keys by atomic max, and counts in; the
//             last CTA to arrive (atomic counter, no waiting) reads the keys
//             and writes the outputs.
// Sampling variants (uno_verify_block_ex) are separate instantiations of both
// kernels: logits scaled by 1/T, and optionally the single-uniform inverse CDF
// in place of the race (exact fixed-point chunk sums; the last CTA finds the
// crossing).  The temperature-1 race keeps the plain instantiations.
// Nothing spins, nothing traps: bad data sets a per-sequence status.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include "uno_internal.h"
#include "verify_common.cuh"

namespace uno {
namespace {

using namespace vfy;

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Statistics pass: CPS CTAs resident on an SM at once, each thread with
// 32 / CPS float4 loads in flight.  Eight CTAs per SM, except for at most 64
// rows (a sequence or two), where four fatter CTAs per SM start sooner
// (batch 1: 13.8 -> 12.8 us per call; batch 8 was 0.5 us slower that way).
constexpr int kStatsCtasPerSm = 8;
constexpr int kStatsCtasPerSmFew = 4;
constexpr int64_t kStatsFewRows = 64;
constexpr int kFinishCtasPerSm = 4;  // finish CTAs resident on an SM at once
constexpr int kRace = 0, kInverseCdf = 1;  // resample modes (uno.h: UNO_RESAMPLE_*)

// Row j of sequence b: j < Kp is AR row j, else draft row j - Kp.
__device__ __forceinline__ const float* row_ptr(const float* p, const float* q, int64_t b,
                                                int64_t j, int64_t K, int64_t Kp, int64_t V) {
  return j < Kp ? p + (b * Kp + j) * V : q + (b * K + (j - Kp)) * V;
}

// kEx: logits at a temperature other than 1 (the plain kernel is kept as it was)
// CPS: CTAs per SM -- the registers a thread may use (32 at 8 CTAs) so that
// the grid the plan sizes for small batches runs as a single wave.
template <bool kEx, int CPS>
__global__ void __launch_bounds__(kThreads, CPS)
verify_stats_kernel(const float* __restrict__ p, const float* __restrict__ q,
                    const int32_t* __restrict__ draft, int64_t K, int64_t Kp, int64_t V,
                    int splits, int64_t chunk, float inv_t, float2* __restrict__ part,
                    float* __restrict__ gathered, int* __restrict__ counter,
                    unsigned long long* __restrict__ keys, int key_stride) {
  const int64_t unit = blockIdx.x;
  const int64_t row = unit / splits;
  const int split = int(unit - row * splits);
  const int64_t per_seq = Kp + K;
  const int64_t b = row / per_seq;
  const int64_t j = row - b * per_seq;
  grid_dependency_wait();
  if (j == 0 && split == 0 && threadIdx.x == 0) {
    counter[b] = 0;  // finish kernel's arrival count
    if (keys) keys[b * key_stride] = keys[b * key_stride + 1] = 0ull;  // its race winners
  }
  // This CTA's chunk [v0, v0 + n) of the row, addressed from its start with
  // 32-bit offsets (a chunk holds < 2^31 elements).
  const int64_t v0 = int64_t(split) * chunk;
  const float* r = row_ptr(p, q, b, j, K, Kp, V) + v0;
  const int n = int(min(V - v0, chunk));
  // The drafted token of this row's position (AR row j or draft row j - Kp):
  // the CTA whose chunk holds it stores its logit for the acceptance test.
  const int64_t pos = j < Kp ? j : j - Kp;
  if (pos < K && threadIdx.x == 0) {
    const int64_t xd = int64_t(draft[b * K + pos]) - v0;
    if (xd >= 0 && xd < n) gathered[row] = r[xd];
  }
  // 16-byte aligned body [head, head + 4 * nv), scalar head and tail.
  const int head_raw = int(((16 - (reinterpret_cast<uintptr_t>(r) & 15)) & 15) >> 2);
  const int head = head_raw < n ? head_raw : n;
  const int nv = (n - head) >> 2;
  const int tail = head + nv * 4;

  MS acc{-INFINITY, 0.f};
  const int tid = threadIdx.x;
  if (tid < head) {
    const float x = r[tid];
    ms_add1(acc, kEx ? x * inv_t : x);
  }
  if (tail + tid < n) {
    const float x = r[tail + tid];
    ms_add1(acc, kEx ? x * inv_t : x);
  }
  const float4* vp = reinterpret_cast<const float4*>(r + head);
  constexpr int kUnroll = 32 / CPS;  // float4 loads in flight per thread
  for (int i = tid; i < nv; i += kThreads * kUnroll) {
    float4 t[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int idx = i + u * kThreads;
      t[u] = idx < nv ? __ldcs(vp + idx) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (kEx)
        ms_add4(acc, t[u].x * inv_t, t[u].y * inv_t, t[u].z * inv_t, t[u].w * inv_t);
      else
        ms_add4(acc, t[u].x, t[u].y, t[u].z, t[u].w);
    }
  }

  acc = warp_merge(acc);
  __shared__ MS red[kWarps];
  if ((tid & 31) == 0) red[tid >> 5] = acc;
  __syncthreads();
  if (tid == 0) {
    MS t = red[0];
    for (int w = 1; w < kWarps; ++w) t = ms_merge(t, red[w]);
    part[unit] = make_float2(t.m, t.s);
    // The finish kernel's CTAs may now be scheduled (they wait for this grid
    // to complete before reading what it wrote).  Signalled at the end, not
    // the start, so that they do not take SM slots this grid's wave needs.
    grid_launch_dependents();
  }
}

constexpr int kMaxRows = 2 * 256 + 1;  // Kp + K rows of one sequence held in smem

// Arrival count of a last-arriver merge: the add releases this CTA's earlier
// stores and acquires those of every CTA that arrived before it.
__device__ __forceinline__ int arrive_acq_rel(int* p) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

// kEx: temperature other than 1 or the inverse-CDF resample
template <bool kEx>
__global__ void __launch_bounds__(kThreads, kFinishCtasPerSm)
verify_finish_kernel(const float* __restrict__ p, const float* __restrict__ q,
                     const int32_t* __restrict__ draft, const float* __restrict__ u_acc,
                     const float* __restrict__ u_res, int64_t K, int64_t Kp, int64_t V,
                     int splits, int race_splits, int64_t race_chunk, float inv_t, int mode,
                     const float2* __restrict__ part, const float* __restrict__ gathered,
                     RacePart* __restrict__ rpart, unsigned long long* __restrict__ keys,
                     int key_stride, int* __restrict__ counter, int32_t* __restrict__ n_acc,
                     int32_t* __restrict__ out_tokens, int32_t* __restrict__ n_emit,
                     int32_t* __restrict__ status) {
  __shared__ float s_m[kMaxRows];    // row max
  __shared__ float s_lz[kMaxRows];   // row max + ln(sum)
  __shared__ float s_iz[kMaxRows];   // 1 / sum
  __shared__ int s_bad;
  __shared__ int s_n;
  __shared__ int s_last;
  __shared__ Cand s_cr[kWarps], s_cp[kWarps];

  constexpr int kRaceUnroll = 4;
  const int tid = threadIdx.x;
  const int64_t b = blockIdx.x / race_splits;
  const int split = int(blockIdx.x - b * race_splits);
  const int64_t per_seq = Kp + K;
  // Inputs the statistics pass does not write, read before waiting for it:
  // this thread's drafted token and accept uniform (K <= kThreads) and its
  // first batch of race uniforms.
  const bool has_i = tid < K;
  const int32_t x_t = has_i ? draft[b * K + tid] : 0;
  const float ua_t = has_i ? u_acc[b * K + tid] : 0.f;
  const float* ub = u_res + b * V;  // (race) this sequence's uniforms
  const int64_t v0 = int64_t(split) * race_chunk;
  const int64_t v1 = min(V, v0 + race_chunk);
  float u_pre[kRaceUnroll];
#pragma unroll
  for (int i = 0; i < kRaceUnroll; ++i) {
    const int64_t vi = v0 + tid + int64_t(i) * kThreads;
    u_pre[i] = ((!kEx || mode == kRace) && vi < v1) ? ub[vi] : 0.5f;
  }
  if (tid == 0) s_bad = 0;
  grid_dependency_wait();  // the statistics pass's partials, gathered logits and counters
  // the drafted tokens' logits (position tid), in flight during step 1
  const float g_q = has_i ? gathered[b * per_seq + Kp + tid] : 0.f;
  const float g_p = has_i ? gathered[b * per_seq + tid] : 0.f;
  __syncthreads();

  // 1. Row normalisers of this sequence from the statistics partials: eight
  //    threads per row (32 rows at a time), each merging every eighth chunk
  //    partial, then three shuffle rounds inside the group of eight.
  {
    const int sub = tid & 7;
    for (int64_t j0 = 0; j0 < per_seq; j0 += kThreads / 8) {
      const int64_t j = j0 + (tid >> 3);
      MS t{-INFINITY, 0.f};
      if (j < per_seq) {
        const float2* pj = part + (b * per_seq + j) * splits;
        for (int s0 = sub; s0 < splits; s0 += 32) {
          float2 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int sx = s0 + 8 * u;
            v[u] = sx < splits ? pj[sx] : make_float2(-INFINITY, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) t = ms_merge(t, MS{v[u].x, v[u].y});
        }
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        const MS u{__shfl_xor_sync(0xffffffffu, t.m, o), __shfl_xor_sync(0xffffffffu, t.s, o)};
        t = ms_merge(t, u);
      }
      if (sub == 0 && j < per_seq) {
        const bool bad = isnan(t.s) || !(t.m > -INFINITY) || !(t.m < INFINITY) || !(t.s > 0.f);
        if (bad) atomicOr(&s_bad, 2);
        s_m[j] = t.m;
        s_lz[j] = t.m + logf(t.s);
        s_iz[j] = 1.0f / t.s;
      }
    }
  }
  // 2. Draft ids and acceptance flags.
  if (has_i && (x_t < 0 || x_t >= V)) atomicOr(&s_bad, 1);
  __syncthreads();
  const int bad = s_bad;
  int32_t* out = out_tokens + b * (K + 1);
  if (bad) {
    if (split == 0) {
      for (int64_t i = tid; i <= K; i += kThreads) out[i] = -1;
      if (tid == 0) {
        n_acc[b] = 0;
        n_emit[b] = 0;
        status[b] = (bad & 1) ? UNO_SEQ_BAD_DRAFT : UNO_SEQ_NONFINITE;
      }
    }
    return;
  }
  // Accept x_i iff u_i < min(1, p_i(x_i)/q_i(x_i)), the ratio taken in the
  // log domain so that neither probability underflows.
  if (tid == 0) s_n = int(K);
  __syncthreads();
  if (has_i) {
    const int i = tid;
    // logits of the drafted token, gathered by the statistics pass
    const float lq = g_q;
    bool accept;
    if (lq == -INFINITY) {
      accept = true;  // q_i(x) = 0: ratio +inf
    } else {
      const float lp = g_p;
      const float lr = kEx ? (lp * inv_t - s_lz[i]) - (lq * inv_t - s_lz[Kp + i])
                           : (lp - s_lz[i]) - (lq - s_lz[Kp + i]);
      const float thr = fminf(1.0f, expf(lr));
      accept = ua_t < thr;
    }
    if (!accept) atomicMin(&s_n, i);
  }
  __syncthreads();
  const int n = s_n;

  const bool residual = n < K;
  const bool bonus = !residual && Kp == K + 1;
  if (!residual && !bonus) {
    if (split == 0) {
      for (int64_t i = tid; i <= K; i += kThreads) out[i] = i < K ? x_t : -1;
      if (tid == 0) {
        n_acc[b] = n;
        n_emit[b] = n;
        status[b] = UNO_SEQ_OK;
      }
    }
    return;
  }

  // 3. Exponential race over this CTA's vocab chunk:
  //    residual: argmax_v max(0, p_n(v) - q_n(v)) / (-ln u_v), falling back
  //    to p_n if no entry is positive; bonus: argmax_v p_K(v) / (-ln u_v).
  const int64_t prow = residual ? n : K;
  const float* pr = p + (b * Kp + prow) * V;
  const float* qr = q + (b * K + n) * V;  // only read when residual
  const float mp = s_m[prow], izp = s_iz[prow];
  const float mq = residual ? s_m[Kp + n] : 0.f, izq = residual ? s_iz[Kp + n] : 0.f;
  // Each thread keeps its best score as a fraction num/den and compares by
  // cross-multiplication (den = -ln u > 0), dividing once at the end;
  // probabilities come from exp2 of the scaled, max-shifted logit.
  constexpr float kLog2e = 1.4426950408889634f;
  if constexpr (kEx) if (mode == kInverseCdf) {
    // 3'. Inverse CDF with one uniform u: the token is the smallest v whose
    //     cumulative weight exceeds u * S, in vocabulary order; weights
    //     max(0, p_n - q_n) (p_n should those sum to 0), or p_K for the bonus
    //     token.  Weights (at most 1, summing to at most about 1) are summed
    //     exactly as integers in units of 2^-46 (round to nearest): every order
    //     of summation gives the same sums, which the integer units compute at
    //     full rate.  This CTA's
    //     chunk is summed first; the last CTA to arrive scans the chunk sums in
    //     chunk order, then searches the chunk holding the crossing.
    __shared__ long long s_d[2][kWarps];  // per-warp sums
    __shared__ long long s_pick;          // chosen chunk, then chosen token
    __shared__ long long s_base;          // weight before the chosen chunk
    __shared__ long long s_loc[2][kThreads];
    constexpr float kFx = 70368744177664.0f;  // 2^46
    auto fx = [](float w) { return __float2ll_rn(w * kFx); };
    auto w_p = [&](int64_t v) { return exp2f((pr[v] * inv_t - mp) * kLog2e) * izp; };
    auto w_r = [&](int64_t v) {
      const float rv = w_p(v) - exp2f((qr[v] * inv_t - mq) * kLog2e) * izq;
      return rv > 0.f ? rv : 0.f;
    };
    long long sr = 0, sp = 0;
    for (int64_t v = v0 + tid; v < v1; v += kThreads) {
      sp += fx(w_p(v));
      if (residual) sr += fx(w_r(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sr += __shfl_xor_sync(0xffffffffu, sr, o);
      sp += __shfl_xor_sync(0xffffffffu, sp, o);
    }
    if ((tid & 31) == 0) {
      s_d[0][tid >> 5] = sr;
      s_d[1][tid >> 5] = sp;
    }
    __syncthreads();
    longlong2* csum = reinterpret_cast<longlong2*>(rpart) + b * race_splits;
    if (tid == 0) {
      long long a = 0, c = 0;
      for (int w = 0; w < kWarps; ++w) {
        a += s_d[0][w];
        c += s_d[1][w];
      }
      csum[split] = make_longlong2(a, c);
      s_last = arrive_acq_rel(&counter[b]) == race_splits - 1;
    }
    // thread 0's acquire, then the barrier, order the loads below after
    // every other CTA's chunk sums
    __syncthreads();
    if (!s_last) return;
    // (a) the chunk holding the crossing
    const int per = (race_splits + kThreads - 1) / kThreads;
    const int c_lo = min(race_splits, tid * per), c_hi = min(race_splits, c_lo + per);
    long long lr = 0, lpp = 0;
    for (int c = c_lo; c < c_hi; ++c) {
      const longlong2 t = __ldcg(csum + c);
      lr += t.x;
      lpp += t.y;
    }
    s_loc[0][tid] = lr;
    s_loc[1][tid] = lpp;
    __syncthreads();
    if (tid == 0) {
      long long a = 0, c = 0;
      for (int t = 0; t < kThreads; ++t) {
        const long long x = s_loc[0][t], y = s_loc[1][t];
        s_loc[0][t] = a;
        s_loc[1][t] = c;
        a += x;
        c += y;
      }
      s_d[0][0] = a;
      s_d[1][0] = c;
      s_pick = -1;
    }
    __syncthreads();
    const bool use_r = residual && s_d[0][0] > 0;
    const long long S = use_r ? s_d[0][0] : s_d[1][0];
    // cumulative weight C crosses u * S where C > floor(u * S) (u < 1, so at
    // most S - 1 even where the product rounds up)
    const long long target =
        S > 0 ? min(S - 1, (long long)floor(double(u_res[b]) * double(S))) : 0;
    {
      const long long E = s_loc[use_r ? 0 : 1][tid];
      long long loc = 0;
      for (int c = c_lo; c < c_hi; ++c) {
        const longlong2 t = __ldcg(csum + c);
        const long long before = E + loc;
        loc += use_r ? t.x : t.y;
        if (before <= target && target < E + loc) {
          s_pick = c;
          s_base = before;
        }
      }
    }
    __syncthreads();
    int64_t tok = -1;
    if (s_pick >= 0) {
      // (b) the entry of that chunk where the cumulative weight crosses u * S
      const int64_t cv0 = s_pick * race_chunk, cv1 = min(V, cv0 + race_chunk);
      const long long base = s_base;
      const int64_t per2 = (cv1 - cv0 + kThreads - 1) / kThreads;
      const int64_t e_lo = min(cv1, cv0 + tid * per2), e_hi = min(cv1, e_lo + per2);
      long long l = 0;
      for (int64_t v = e_lo; v < e_hi; ++v) l += fx(use_r ? w_r(v) : w_p(v));
      __syncthreads();
      s_loc[0][tid] = l;
      __syncthreads();
      if (tid == 0) {
        long long a = 0;
        for (int t = 0; t < kThreads; ++t) {
          const long long x = s_loc[0][t];
          s_loc[0][t] = a;
          a += x;
        }
        s_pick = -1;
      }
      __syncthreads();
      long long cum = base + s_loc[0][tid];
      int64_t last_pos = -1;
      for (int64_t v = e_lo; v < e_hi; ++v) {
        const long long wv = fx(use_r ? w_r(v) : w_p(v));
        if (wv > 0) last_pos = v;
        if (cum <= target && target < cum + wv) s_pick = v;
        cum += wv;
      }
      s_loc[1][tid] = last_pos;
      __syncthreads();
      tok = s_pick;
      if (tok < 0) {
        // the sums are exact, so only a chunk whose weights all rounded to 0
        // can miss: its last entry with positive weight, if any
        for (int t = kThreads - 1; t >= 0 && tok < 0; --t)
          if (s_loc[1][t] >= 0) tok = s_loc[1][t];
      }
    }
    if (tid == 0) {
      counter[b] = 0;
      n_acc[b] = n;
      n_emit[b] = n + 1;
      status[b] = UNO_SEQ_OK;
    }
    for (int64_t i = tid; i <= K; i += kThreads)
      out[i] = i < n ? x_t : (i == n ? int32_t(tok) : -1);
    return;
  }
  float pn = -1.f, pd = 1.f, rn = 0.f, rd = 1.f;
  int pvid = -1, rvid = -1;
  for (int64_t v = v0 + tid; v < v1; v += int64_t(kThreads) * kRaceUnroll) {
    float uu[kRaceUnroll], lp[kRaceUnroll], lq[kRaceUnroll];
    const bool first = v == v0 + tid;
#pragma unroll
    for (int i = 0; i < kRaceUnroll; ++i) {
      const int64_t vi = v + int64_t(i) * kThreads;
      const bool in = vi < v1;
      uu[i] = first ? u_pre[i] : (in ? ub[vi] : 0.5f);
      lp[i] = in ? pr[vi] : -INFINITY;
      lq[i] = (in && residual) ? qr[vi] : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < kRaceUnroll; ++i) {
      const int64_t vi = v + int64_t(i) * kThreads;
      if (vi >= v1) break;
      const float e = -logf(uu[i]);
      const float pv = exp2f(((kEx ? lp[i] * inv_t : lp[i]) - mp) * kLog2e) * izp;
      if (pv * pd > pn * e) {  // pv / e > pn / pd; ties keep the lower id
        pn = pv;
        pd = e;
        pvid = int(vi);
      }
      if (residual) {
        const float rv = pv - exp2f(((kEx ? lq[i] * inv_t : lq[i]) - mq) * kLog2e) * izq;
        if (rv > 0.f && rv * rd > rn * e) {
          rn = rv;
          rd = e;
          rvid = int(vi);
        }
      }
    }
  }
  Cand cr{rvid >= 0 ? rn / rd : 0.f, rvid}, cp{pvid >= 0 ? pn / pd : -1.f, pvid};
  cr = warp_best(cr);
  cp = warp_best(cp);
  if ((tid & 31) == 0) {
    s_cr[tid >> 5] = cr;
    s_cp[tid >> 5] = cp;
  }
  __syncthreads();
  if (tid == 0) {
    cr = s_cr[0];
    cp = s_cp[0];
    for (int w = 1; w < kWarps; ++w) {
      cr = cand_best(cr, s_cr[w]);
      cp = cand_best(cp, s_cp[w]);
    }
    int last = 1;
    if (race_splits > 1) {
      // The chunk winners merge by atomic max of their keys; the count's
      // release orders this CTA's maxima before it, and the last CTA's
      // acquire orders every CTA's before its loads of the two keys.
      unsigned long long* kk = keys + b * key_stride;
      atomicMax(kk, cand_key(cr));
      atomicMax(kk + 1, cand_key(cp));
      last = arrive_acq_rel(&counter[b]) == race_splits - 1;
      if (last) {
        cr = cand_of_key(__ldcg(kk));
        cp = cand_of_key(__ldcg(kk + 1));
        counter[b] = 0;
      }
    }
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  if (tid == 0) {
    n_acc[b] = n;
    n_emit[b] = n + 1;
    status[b] = UNO_SEQ_OK;
    s_n = (residual && cr.v >= 0) ? cr.v : cp.v;
  }
  __syncthreads();
  const int tok = s_n;
  for (int64_t i = tid; i <= K; i += kThreads)
    out[i] = i < n ? x_t : (i == n ? tok : -1);
}

// One CTA per row: Gumbel-max form of the race, argmax_v l_v - ln(-ln u_v),
// which equals argmax_v softmax(l)(v) / (-ln u_v) (the normaliser cancels).
__global__ void __launch_bounds__(kThreads)
draft_sample_kernel(const float* __restrict__ logits, const float* __restrict__ u, int64_t V,
                    int32_t* __restrict__ tokens, int32_t* __restrict__ status) {
  __shared__ Cand s_c[kWarps];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  const int64_t r = blockIdx.x;
  const float* lr = logits + r * V;
  const float* ur = u + r * V;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  Cand c{-INFINITY, -1};
  bool bad = false;
  for (int64_t v = tid; v < V; v += kThreads) {
    const float l = __ldcs(lr + v);
    bad |= isnan(l) || l == INFINITY;
    if (l > -INFINITY) c = cand_best(c, Cand{l - logf(-logf(__ldcs(ur + v))), int(v)});
  }
  if (bad) atomicOr(&s_bad, 1);
  c = warp_best(c);
  if ((tid & 31) == 0) s_c[tid >> 5] = c;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kWarps; ++w) c = cand_best(c, s_c[w]);
    if (s_bad || c.v < 0) {
      tokens[r] = -1;
      status[r] = UNO_SEQ_NONFINITE;
    } else {
      tokens[r] = c.v;
      status[r] = UNO_SEQ_OK;
    }
  }
}

}  // namespace

VerifyPlan plan_verify(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int sms) {
  VerifyPlan pl{};
  pl.rows = Bn * (Kp + K);
  // Statistics pass: one wave of stats_cps CTAs of 256 threads per SM;
  // split rows only while each chunk keeps at least 2048 logits.
  pl.stats_cps = pl.rows <= kStatsFewRows ? kStatsCtasPerSmFew : kStatsCtasPerSm;
  const int64_t target = int64_t(sms) * pl.stats_cps;
  int64_t s = pl.rows > 0 ? target / pl.rows : 1;  // (rounded down: no second, nearly empty wave)
  s = std::max<int64_t>(1, std::min<int64_t>(s, (V + 2047) / 2048));
  int64_t chunk = (V + s - 1) / s;
  chunk = (chunk + 3) & ~int64_t(3);
  pl.chunk = chunk;
  pl.splits = int((V + chunk - 1) / chunk);
  // Race pass: at most kFinishCtasPerSm CTAs per SM (one wave), chunks of at
  // least 1024 entries (one batch of loads per thread at small batch).
  const int64_t rt = int64_t(sms) * kFinishCtasPerSm;
  int64_t s2 = Bn > 0 ? rt / Bn : 1;
  s2 = std::max<int64_t>(1, std::min<int64_t>(s2, (V + 1023) / 1024));
  pl.race_chunk = (V + s2 - 1) / s2;
  pl.race_splits = int((V + pl.race_chunk - 1) / pl.race_chunk);
  // Inverse CDF: the same, but chunks of at most 8192 entries, so that the
  // last CTA's search of the chunk holding the crossing stays short.
  const int64_t s3 = std::min<int64_t>(std::max<int64_t>(s2, (V + 8191) / 8192), (V + 1023) / 1024);
  pl.icdf_chunk = (V + s3 - 1) / s3;
  pl.icdf_splits = int((V + pl.icdf_chunk - 1) / pl.icdf_chunk);
  pl.off_stats = 0;
  pl.off_gather = align_up(pl.off_stats + size_t(pl.rows) * pl.splits * sizeof(float2), 256);
  pl.off_race = align_up(pl.off_gather + size_t(pl.rows) * sizeof(float), 256);
  pl.off_count = align_up(pl.off_race + size_t(Bn) * std::max(pl.race_splits, pl.icdf_splits) *
                                            sizeof(RacePart),
                          256);
  pl.bytes = align_up(pl.off_count + size_t(Bn) * sizeof(int), 256);
  return pl;
}

cudaError_t launch_verify(const float* p, const float* q, const int32_t* draft,
                          const float* u_acc, const float* u_res, int64_t Bn, int64_t K,
                          int64_t Kp, int64_t V, int32_t* n_acc, int32_t* out_tokens,
                          int32_t* n_emit, int32_t* status, void* ws, const VerifyPlan& pl,
                          cudaStream_t st, float inv_t, int mode) {
  const bool ex = inv_t != 1.0f || mode != kRace;
  char* w = static_cast<char*>(ws);
  float2* part = reinterpret_cast<float2*>(w + pl.off_stats);
  float* gathered = reinterpret_cast<float*>(w + pl.off_gather);
  RacePart* rpart = reinterpret_cast<RacePart*>(w + pl.off_race);
  int* counter = reinterpret_cast<int*>(w + pl.off_count);
  const int64_t g1 = pl.rows * pl.splits;
  // The finish kernel is launched with programmatic stream serialization: it
  // may start while the statistics pass drains, and waits for it
  // (griddepcontrol.wait) before it reads what that pass writes; the
  // statistics CTAs signal it only as they end, so its CTAs become resident
  // as the statistics wave drains, not during it.  The statistics kernel
  // itself is launched in plain stream order: placed early beside a
  // still-running projection launch, its CTAs found fewer free slots per SM
  // than the plan's single wave assumes (a batch-32 step in one graph took
  // 0.498 ms that way against 0.475 ms).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(unsigned(g1));
  cfg.numAttrs = 0;  // (statistics: plain stream order)
  // race winners' keys: the first 16 bytes of each sequence's race slots
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(rpart);
  const int key_stride = 2 * std::max(pl.race_splits, pl.icdf_splits);
  const bool few = pl.stats_cps == kStatsCtasPerSmFew;
  auto kern = ex ? (few ? verify_stats_kernel<true, kStatsCtasPerSmFew> : verify_stats_kernel<true, kStatsCtasPerSm>)
                 : (few ? verify_stats_kernel<false, kStatsCtasPerSmFew> : verify_stats_kernel<false, kStatsCtasPerSm>);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p, q, draft, K, Kp, V, pl.splits, pl.chunk, inv_t, part,
                                     gathered, counter, keys, key_stride);
  if (e != cudaSuccess) return e;
  cfg.numAttrs = 1;  // (finish: chained to the statistics pass)
  const bool icdf = mode == kInverseCdf;
  const int rs = icdf ? pl.icdf_splits : pl.race_splits;
  const int64_t rc = icdf ? pl.icdf_chunk : pl.race_chunk;
  cfg.gridDim = dim3(unsigned(Bn * rs));
  e = ex ? cudaLaunchKernelEx(&cfg, verify_finish_kernel<true>, p, q, draft, u_acc, u_res, K, Kp, V,
                              pl.splits, rs, rc, inv_t, mode,
                              (const float2*)part, (const float*)gathered, rpart, keys, key_stride,
                              counter, n_acc, out_tokens, n_emit, status)
         : cudaLaunchKernelEx(&cfg, verify_finish_kernel<false>, p, q, draft, u_acc, u_res, K, Kp,
                              V, pl.splits, pl.race_splits, pl.race_chunk, inv_t, mode,
                              (const float2*)part, (const float*)gathered, rpart, keys, key_stride,
                              counter, n_acc, out_tokens, n_emit, status);
  return e;
}

cudaError_t launch_row_stats(const float* p, const float* q, const int32_t* draft, int64_t Bn,
                             int64_t K, int64_t Kp, int64_t V, const VerifyPlan& pl, void* ws,
                             cudaStream_t st, unsigned long long* keys, int key_stride) {
  char* w = static_cast<char*>(ws);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 0;  // plain stream order, as in launch_verify
  cfg.gridDim = dim3(unsigned(pl.rows * pl.splits));
  auto kern = pl.stats_cps == kStatsCtasPerSmFew ? verify_stats_kernel<false, kStatsCtasPerSmFew>
                                                 : verify_stats_kernel<false, kStatsCtasPerSm>;
  return cudaLaunchKernelEx(&cfg, kern, p, q, draft, K, Kp, V, pl.splits,
                            pl.chunk, 1.0f, reinterpret_cast<float2*>(w + pl.off_stats),
                            reinterpret_cast<float*>(w + pl.off_gather),
                            reinterpret_cast<int*>(w + pl.off_count), keys, key_stride);
}

cudaError_t launch_draft_sample(const float* logits, const float* u, int64_t R, int64_t V,
                                int32_t* tokens, int32_t* status, cudaStream_t st) {
  draft_sample_kernel<<<dim3(unsigned(R)), kThreads, 0, st>>>(logits, u, V, tokens, status);
  return cudaGetLastError();
}

}  // namespace uno
