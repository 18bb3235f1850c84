// lm_head.cu -- the LM head that feeds the block verifier, with the
// verifier's statistics computed in the GEMM's epilogue.
//
// "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
// (aifromscratch.in), section "The Psi-Spec Sampler", and the aiany.app
// summary's "Key Findings": the AR model checks the whole drafted block in a
// single forward pass, which ends in the LM head (logits = h . W^T over the
// vocabulary) and the rejection test of the linear sampler.  The verifier
// needs of every logit row only its (max, sum exp) and the logit of the
// drafted token; the full row is needed again only for the one position per
// sequence that is resampled.  Three strategies, the same result:
//
//   PLAIN       the head GEMM stores fp32 logits, the verifier of verify.cu
//               reads them;
//   STATS_STORE the GEMM's epilogue leaves the statistics (per row and
//               vocabulary tile) and also stores the logits; a decide kernel
//               takes the accept decisions from the statistics and a race
//               kernel reads back only the rows it resamples;
//   STATS_RECOMPUTE
//               the epilogue leaves only the statistics (no logit is written
//               to memory); the decide kernel gathers the hidden states of the
//               resampled rows (AR row n or K, draft row n) and a second GEMM
//               recomputes just those 2 rows per sequence for the race.
//
// Rows of h and of the logits: all AR rows (sequence b, position j at
// b*Kp + j), then all draft rows (b, i) at Bn*Kp + b*K + i, so the logits of
// PLAIN are the verifier's p [Bn, Kp, V] followed by its q [Bn, K, V].
#include <cuda_bf16.h>

#include <algorithm>

#include "ptx.cuh"
#include "uno_internal.h"
#include "verify_common.cuh"

namespace uno {
namespace {

using namespace vfy;

constexpr int kLT = 256;
constexpr int kLW = kLT / 32;
constexpr int kLMaxRows = 2 * 256 + 1;
constexpr float kLog2e = 1.4426950408889634f;

// The decision of one sequence, for the race.
struct SeqDecision {
  int n;          // accepted prefix length
  int race;       // 1: a token is drawn (residual row n, or bonus row K)
  int residual;   // 1: from max(0, p_n - q_n); 0: from p_K
  int pad;
  float mp, izp;  // max and 1/sum of the AR row raced
  float mq, izq;  // the same for draft row n (residual only)
};

// One CTA per sequence: merges the statistics partials of its rows, takes
// the accept decisions and n, writes the outputs of sequences that draw no
// token, and (recompute) copies the hidden states of the rows to race.
__global__ void __launch_bounds__(kLT)
lm_decide_kernel(const __nv_bfloat16* __restrict__ h, const int32_t* __restrict__ draft,
                 const float* __restrict__ u_acc, int64_t Bn, int64_t K, int64_t Kp, int64_t V,
                 int64_t d, int nvt, const float2* __restrict__ part,
                 const float* __restrict__ gathered, __nv_bfloat16* __restrict__ hc,
                 SeqDecision* __restrict__ dec, int* __restrict__ counter,
                 unsigned long long* __restrict__ keys, int key_stride,
                 int32_t* __restrict__ n_acc, int32_t* __restrict__ out_tokens,
                 int32_t* __restrict__ n_emit, int32_t* __restrict__ status) {
  __shared__ float s_m[kLMaxRows], s_lz[kLMaxRows], s_iz[kLMaxRows];
  __shared__ int s_bad, s_n;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t b = blockIdx.x;
  const int64_t per = Kp + K, Rp = Bn * Kp;
  const bool has_i = tid < K;
  const int32_t x_t = has_i ? draft[b * K + tid] : 0;
  const float ua_t = has_i ? u_acc[b * K + tid] : 0.f;
  if (tid == 0) {
    s_bad = 0;
    s_n = int(K);
  }
  ptx::grid_dependency_wait();  // the GEMM's statistics
  __syncthreads();
  // local row j: AR rows 0..Kp-1, then draft rows
  for (int64_t j = warp; j < per; j += kLW) {
    const int64_t r = j < Kp ? b * Kp + j : Rp + b * K + (j - Kp);
    MS t{-INFINITY, 0.f};
    for (int s = lane; s < nvt; s += 32) {
      const float2 v = part[r * nvt + s];
      t = ms_merge(t, MS{v.x, v.y});
    }
    t = warp_merge(t);
    if (lane == 0) {
      if (isnan(t.s) || !(t.m > -INFINITY) || !(t.m < INFINITY) || !(t.s > 0.f)) atomicOr(&s_bad, 2);
      s_m[j] = t.m;
      s_lz[j] = t.m + logf(t.s);
      s_iz[j] = 1.0f / t.s;
    }
  }
  if (has_i && (x_t < 0 || x_t >= V)) atomicOr(&s_bad, 1);
  __syncthreads();
  const int bad = s_bad;
  if (!bad && has_i) {
    const int i = tid;
    const float lq = gathered[Rp + b * K + i];
    bool accept;
    if (lq == -INFINITY) {
      accept = true;  // q_i(x) = 0: ratio +inf
    } else {
      const float lp = gathered[b * Kp + i];
      const float lr = (lp - s_lz[i]) - (lq - s_lz[Kp + i]);
      accept = ua_t < fminf(1.0f, expf(lr));
    }
    if (!accept) atomicMin(&s_n, i);
  }
  __syncthreads();
  const int n = s_n;
  const bool residual = n < K;
  const bool race = !bad && (residual || Kp == K + 1);
  int32_t* out = out_tokens + b * (K + 1);
  if (!race) {
    for (int64_t i = tid; i <= K; i += kLT) out[i] = (!bad && i < K) ? x_t : -1;
    if (tid == 0) {
      n_acc[b] = bad ? 0 : n;
      n_emit[b] = bad ? 0 : n;
      status[b] = bad ? ((bad & 1) ? UNO_SEQ_BAD_DRAFT : UNO_SEQ_NONFINITE) : UNO_SEQ_OK;
    }
  }
  const int64_t prow = residual ? n : K;
  if (tid == 0) {
    SeqDecision sd{};
    sd.n = n;
    sd.race = race;
    sd.residual = residual;
    sd.mp = s_m[prow];
    sd.izp = s_iz[prow];
    sd.mq = residual ? s_m[Kp + n] : 0.f;
    sd.izq = residual ? s_iz[Kp + n] : 0.f;
    dec[b] = sd;
    counter[b] = 0;
    keys[b * key_stride] = keys[b * key_stride + 1] = 0ull;  // the race's winners
  }
  if (hc != nullptr) {
    // hidden states of the rows to race: hc[2b] = AR row prow, hc[2b+1] =
    // draft row n (zeros when there is none)
    const uint4* src_p = reinterpret_cast<const uint4*>(h + (b * Kp + prow) * d);
    const uint4* src_q = reinterpret_cast<const uint4*>(h + (Rp + b * K + (residual ? n : 0)) * d);
    uint4* dp = reinterpret_cast<uint4*>(hc + (2 * b) * d);
    uint4* dq = reinterpret_cast<uint4*>(hc + (2 * b + 1) * d);
    const int64_t n16 = d / 8;
    for (int64_t k = tid; k < n16; k += kLT) {
      dp[k] = race ? src_p[k] : make_uint4(0, 0, 0, 0);
      dq[k] = (race && residual) ? src_q[k] : make_uint4(0, 0, 0, 0);
    }
  }
}

// One CTA per (sequence, vocabulary chunk): the exponential race over this
// chunk of the residual row (or the bonus row) and folds its winners into the
// sequence's 64-bit keys by atomic max; the last CTA to arrive reads the keys
// and writes the outputs (atomic count, no waiting).
__global__ void __launch_bounds__(kLT)
lm_race_kernel(const float* __restrict__ logits, int recompute, const int32_t* __restrict__ draft,
               const float* __restrict__ u_res, int64_t Bn, int64_t K, int64_t Kp, int64_t V,
               int race_splits, int64_t race_chunk, const SeqDecision* __restrict__ dec,
               unsigned long long* __restrict__ keys, int key_stride, int* __restrict__ counter,
               int32_t* __restrict__ n_acc, int32_t* __restrict__ out_tokens,
               int32_t* __restrict__ n_emit, int32_t* __restrict__ status) {
  __shared__ Cand s_cr[kLW], s_cp[kLW];
  __shared__ int s_last, s_tok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t b = blockIdx.x / race_splits;
  const int split = int(blockIdx.x - b * race_splits);
  ptx::grid_dependency_wait();
  const SeqDecision sd = dec[b];
  if (!sd.race) return;
  const int n = sd.n;
  const bool residual = sd.residual != 0;
  const int64_t Rp = Bn * Kp;
  const float* pr = recompute ? logits + (2 * b) * V : logits + (b * Kp + (residual ? n : K)) * V;
  const float* qr = recompute ? logits + (2 * b + 1) * V : logits + (Rp + b * K + (residual ? n : 0)) * V;
  const float* ub = u_res + b * V;
  const int64_t v0 = int64_t(split) * race_chunk;
  const int64_t v1 = min(V, v0 + race_chunk);
  float pn = -1.f, pd = 1.f, rn = 0.f, rd = 1.f;
  int pvid = -1, rvid = -1;
  for (int64_t v = v0 + 4 * tid; v < v1; v += 4 * kLT) {
    const float4 u4 = *reinterpret_cast<const float4*>(ub + v);
    const float4 p4 = *reinterpret_cast<const float4*>(pr + v);
    const float4 q4 = residual ? *reinterpret_cast<const float4*>(qr + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
    const float lp[4] = {p4.x, p4.y, p4.z, p4.w};
    const float lq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float e = -logf(uu[j]);
      const float pv = exp2f((lp[j] - sd.mp) * kLog2e) * sd.izp;
      if (pv * pd > pn * e) {  // pv / e > pn / pd; ties keep the lower id
        pn = pv;
        pd = e;
        pvid = int(v + j);
      }
      if (residual) {
        const float rv = pv - exp2f((lq[j] - sd.mq) * kLog2e) * sd.izq;
        if (rv > 0.f && rv * rd > rn * e) {
          rn = rv;
          rd = e;
          rvid = int(v + j);
        }
      }
    }
  }
  Cand cr{rvid >= 0 ? rn / rd : 0.f, rvid}, cp{pvid >= 0 ? pn / pd : -1.f, pvid};
  cr = warp_best(cr);
  cp = warp_best(cp);
  if (lane == 0) {
    s_cr[warp] = cr;
    s_cp[warp] = cp;
  }
  __syncthreads();
  if (tid == 0) {
    cr = s_cr[0];
    cp = s_cp[0];
    for (int w = 1; w < kLW; ++w) {
      cr = cand_best(cr, s_cr[w]);
      cp = cand_best(cp, s_cp[w]);
    }
    int last = 1;
    if (race_splits > 1) {
      // chunk winners merge by atomic max of their keys (verify_common.cuh)
      unsigned long long* kk = keys + b * key_stride;
      atomicMax(kk, cand_key(cr));
      atomicMax(kk + 1, cand_key(cp));
      __threadfence();
      last = atomicAdd(&counter[b], 1) == race_splits - 1;
      if (last) {
        __threadfence();
        cr = cand_of_key(__ldcg(kk));
        cp = cand_of_key(__ldcg(kk + 1));
      }
    }
    s_last = last;
    s_tok = (residual && cr.v >= 0) ? cr.v : cp.v;
  }
  __syncthreads();
  if (!s_last) return;
  const int tok = s_tok;
  int32_t* out = out_tokens + b * (K + 1);
  for (int64_t i = tid; i <= K; i += kLT) out[i] = i < n ? draft[b * K + i] : (i == n ? tok : -1);
  if (tid == 0) {
    n_acc[b] = n;
    n_emit[b] = n + 1;
    status[b] = UNO_SEQ_OK;
  }
}

cudaLaunchConfig_t pdl_config(dim3 grid, cudaStream_t st, cudaLaunchAttribute* attr) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kLT);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

LmPlan plan_lm_head(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int64_t d, int mode, int sms) {
  LmPlan L{};
  L.mode = mode == UNO_LM_AUTO ? (Bn >= kLmStatsMinBatch ? UNO_LM_STATS_STORE : UNO_LM_PLAIN) : mode;
  L.rows = Bn * (Kp + K);
  uno_lora_problem p{};
  p.d_in = d;
  p.d_out = V;
  size_t o = 0;
  L.off_gemm = o;
  L.gemm_bytes = lora_group_workspace_bytes(1, &p, L.rows, UNO_BF16, sms);
  o = align_up(o + L.gemm_bytes, 256);
  if (L.mode == UNO_LM_PLAIN || L.mode == UNO_LM_STATS_STORE) {
    L.off_logits = o;
    o = align_up(o + size_t(L.rows) * size_t(V) * 4, 256);
  }
  if (L.mode == UNO_LM_PLAIN) {
    L.vplan = plan_verify(Bn, K, Kp, V, sms);
    L.off_verify = o;
    o = align_up(o + L.vplan.bytes, 256);
    L.bytes = o;
    return L;
  }
  L.nvt = logit_gemm_tiles(L.rows, d, V, sms);
  L.off_part = o;
  o = align_up(o + size_t(L.rows) * size_t(L.nvt) * sizeof(float2), 256);
  L.off_gather = o;
  o = align_up(o + size_t(L.rows) * sizeof(float), 256);
  L.off_dec = o;
  o = align_up(o + size_t(Bn) * sizeof(SeqDecision), 256);
  // race: about four CTAs per SM, chunks of at least 1024 entries (multiples of 4)
  int64_t s2 = (int64_t(sms) * 4 + Bn - 1) / Bn;
  s2 = std::max<int64_t>(1, std::min<int64_t>(s2, (V + 1023) / 1024));
  L.race_chunk = (((V + s2 - 1) / s2) + 3) & ~int64_t(3);
  L.race_splits = int((V + L.race_chunk - 1) / L.race_chunk);
  L.off_race = o;
  o = align_up(o + size_t(Bn) * L.race_splits * sizeof(RacePart), 256);
  L.off_count = o;
  o = align_up(o + size_t(Bn) * sizeof(int), 256);
  if (L.mode == UNO_LM_STATS_RECOMPUTE) {
    L.off_hc = o;
    o = align_up(o + size_t(2 * Bn) * size_t(d) * 2, 256);
    L.off_lc = o;
    o = align_up(o + size_t(2 * Bn) * size_t(V) * 4, 256);
    L.off_gemm2 = o;
    L.gemm2_bytes = lora_group_workspace_bytes(1, &p, 2 * Bn, UNO_BF16, sms);
    o = align_up(o + L.gemm2_bytes, 256);
  }
  L.bytes = o;
  return L;
}

int launch_lm_head_verify(const void* h, const void* W, const int32_t* draft, const float* u_acc,
                          const float* u_res, int64_t Bn, int64_t K, int64_t Kp, int64_t V,
                          int64_t d, int32_t* n_acc, int32_t* out_tokens, int32_t* n_emit,
                          int32_t* status, void* ws, size_t ws_bytes, const LmPlan& L,
                          cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  const int64_t Rp = Bn * Kp;
  uno_lora_problem pr{};
  pr.x = h;
  pr.W = W;
  pr.d_in = d;
  pr.d_out = V;
  pr.rank = 0;
  pr.alpha = 0.f;
  LinearEpilogue epi{};
  epi.K = K;
  epi.Kp = Kp;
  epi.Rp = Rp;
  epi.draft = draft;
  if (L.mode == UNO_LM_PLAIN) {
    float* logits = reinterpret_cast<float*>(w + L.off_logits);
    pr.y = logits;
    epi.f32out = 1;
    int rc = launch_logit_gemm(pr, L.rows, w + L.off_gemm, L.gemm_bytes, st, epi);
    if (rc != UNO_OK) return rc;
    const cudaError_t e = launch_verify(logits, logits + Rp * V, draft, u_acc, u_res, Bn, K, Kp, V,
                                        n_acc, out_tokens, n_emit, status, w + L.off_verify,
                                        L.vplan, st);
    return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
  }
  const bool store = L.mode == UNO_LM_STATS_STORE;
  float* logits = store ? reinterpret_cast<float*>(w + L.off_logits) : nullptr;
  pr.y = store ? static_cast<void*>(logits) : w + L.off_part;  // (unused without the store)
  epi.f32out = 1;
  epi.stats = 1;
  epi.stats_store = store;
  epi.nvt = L.nvt;
  epi.part = reinterpret_cast<float2*>(w + L.off_part);
  epi.gathered = reinterpret_cast<float*>(w + L.off_gather);
  int rc = launch_logit_gemm(pr, L.rows, w + L.off_gemm, L.gemm_bytes, st, epi);
  if (rc != UNO_OK) return rc;
  SeqDecision* dec = reinterpret_cast<SeqDecision*>(w + L.off_dec);
  int* counter = reinterpret_cast<int*>(w + L.off_count);
  __nv_bfloat16* hc = store ? nullptr : reinterpret_cast<__nv_bfloat16*>(w + L.off_hc);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(unsigned(Bn)), st, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, lm_decide_kernel,
                                     static_cast<const __nv_bfloat16*>(h), draft, u_acc, Bn, K, Kp,
                                     V, d, L.nvt, const_cast<const float2*>(epi.part),
                                     const_cast<const float*>(epi.gathered), hc, dec, counter,
                                     reinterpret_cast<unsigned long long*>(w + L.off_race),
                                     2 * L.race_splits, n_acc, out_tokens, n_emit, status);
  if (e != cudaSuccess) return UNO_ERR_CUDA;
  const float* race_rows = logits;
  if (!store) {
    // the two rows per sequence that the race reads, recomputed
    float* lc = reinterpret_cast<float*>(w + L.off_lc);
    uno_lora_problem p2 = pr;
    p2.x = hc;
    p2.y = lc;
    LinearEpilogue e2{};
    e2.f32out = 1;
    rc = launch_logit_gemm(p2, 2 * Bn, w + L.off_gemm2, L.gemm2_bytes, st, e2);
    if (rc != UNO_OK) return rc;
    race_rows = lc;
  }
  cfg = pdl_config(dim3(unsigned(Bn * L.race_splits)), st, attr);
  e = cudaLaunchKernelEx(&cfg, lm_race_kernel, race_rows, store ? 0 : 1, draft, u_res, Bn, K, Kp, V,
                         L.race_splits, L.race_chunk, const_cast<const SeqDecision*>(dec),
                         reinterpret_cast<unsigned long long*>(w + L.off_race), 2 * L.race_splits,
                         counter, n_acc, out_tokens, n_emit, status);
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}

}  // namespace uno
