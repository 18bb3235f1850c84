// verify_fused.cu -- the block verifier in ONE launch, for small batches.
//
// Same rule as the two-launch verifier in verify.cu ("Unlocking Lossless
// Speedups in LLMs via Discrete Diffusion", aifromscratch.in, section "The
// Psi-Spec Sampler": drafts are kept up to the first rejection of a
// speculative-decoding style rejection test, and the emitted tokens follow the
// AR model's distribution).  At a small batch the two launches cost more in
// launch gaps and dependent round trips than in HBM time (batch 1 reads 16 MB
// of logits, 2.6 us at full bandwidth), so this kernel runs the whole verifier
// as one cooperative launch of one CTA per SM:
//
//   1. statistics: the logit rows of the batch (all AR rows, then all draft
//      rows) form one element range, cut into equal, 16-byte aligned slices,
//      one per CTA.  A CTA streams its slice through a shared-memory ring with
//      bulk asynchronous copies (cp.async.bulk, one thread issuing, mbarrier
//      completion) and keeps an online (max, sum exp) per thread, reduced per
//      row segment; the thread that meets a row's drafted token keeps its logit.
//   2. grid barrier (co-residency is guaranteed by the cooperative launch; the
//      wait is bounded all the same), then every CTA merges the partials of
//      every row (fixed order, so every CTA gets identical normalisers), takes
//      the accept decisions and the prefix length n of every sequence.
//   3. race: the rows to resample (max(0, p_n - q_n) at a rejection, p_K for a
//      bonus token) form a second element range, cut the same way; every CTA
//      races its slice, and the last CTA to arrive for a sequence (atomic
//      count, no waiting) merges the slice winners and writes the outputs.
//      A batch of 16 MB or less is still in L2 from step 1, so the rows
//      re-read here come from L2.
// Used for T = 1 with the race, a vocabulary size divisible by 4 and 16-byte
// aligned logit and uniform rows; other calls take the two-launch path.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "uno_internal.h"
#include "verify_common.cuh"

namespace uno {

// bit 0: a grid barrier of the fused verifier gave up waiting (outputs invalid)
__device__ int g_verify_error;

namespace {

using namespace vfy;

constexpr int kFT = 256;
constexpr int kFW = kFT / 32;
constexpr int kFStages = 6;    // even: stage s always belongs to issuing thread s % 2
constexpr int kFChunk = 8192;  // floats per ring stage (32 KB)
constexpr uint32_t kFRingBytes = uint32_t(kFStages) * kFChunk * 4;
constexpr uint64_t kFWaitNs = 1000000000ull;  // 1 s: the barrier's partners are co-resident
constexpr int kFMaxG = 160;    // CTAs of the launch (one per SM)
constexpr int kFRaceUnroll = 4;
constexpr int kFMaxRowsPerSlice = 64;  // rows whose drafted token a CTA keeps in shared memory

struct FusedArgs {
  const float* p;         // [Bn, Kp, V]
  const float* q;         // [Bn, K, V]
  const int32_t* draft;   // [Bn, K]
  const float* u_acc;     // [Bn, K]
  const float* u_res;     // [Bn, V]
  int64_t Bn, K, Kp, V;
  int64_t E;              // elements of all rows: Bn * (Kp + K) * V
  int64_t Np;             // elements of the AR rows: Bn * Kp * V
  int G;                  // CTAs of the launch
  int Gs;                 // CTAs with a statistics slice (each slice >= 4 elements)
  int S;                  // statistics slots per row (most CTAs a row can span)
  float2* part;           // [rows][S] (max, sum exp) of each CTA's segment of the row
  float* gathered;        // [rows] logit of the row's drafted token
  RacePart* rpart;        // [Bn][G] slice winners of each race row
  int* sync;              // [0] grid barrier arrivals, [1 + i] arrivals at race row i
  int32_t* n_acc;
  int32_t* out_tokens;
  int32_t* n_emit;
  int32_t* status;
  int64_t sstart[kFMaxG + 1];  // statistics slices: CTA c streams [sstart[c], sstart[c+1])
};

// First element of slice c when `total` elements (a multiple of 4) are cut into
// `n` slices of at least 4 elements, each starting on a multiple of 4.
__host__ __device__ __forceinline__ int64_t slice_start(int64_t total, int n, int c) {
  return c >= n ? total : ((int64_t(c) * total) / n) & ~int64_t(3);
}

// Slice of a start table holding element e (0 <= e < table[n]): binary search.
__device__ __forceinline__ int table_owner(const int64_t* table, int n, int64_t e) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (table[mid] <= e) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The drafted token whose logit row r holds (rows: all AR rows, then all draft rows).
__device__ __forceinline__ int64_t row_draft(const FusedArgs& a, int64_t r) {
  const int64_t Rp = a.Bn * a.Kp;
  if (r < Rp) {
    const int64_t b = r / a.Kp, j = r - b * a.Kp;
    return j < a.K ? int64_t(a.draft[b * a.K + j]) : -1;
  }
  return int64_t(a.draft[r - Rp]);  // draft row (b, i) is row Rp + b*K + i
}

// Walks the chunks of a statistics slice: at most kFChunk elements each, never
// across a row boundary (the AR and draft regions meet at a row boundary too).
struct ChunkCursor {
  int64_t cur, row, row_end, end, V;
  uint32_t idx;
  __device__ __forceinline__ void init(int64_t e0, int64_t e1, int64_t V_) {
    cur = e0;
    end = e1;
    V = V_;
    row = e0 / V_;
    row_end = (row + 1) * V_;
    idx = 0;
  }
  __device__ __forceinline__ int64_t len() const { return min(int64_t(kFChunk), min(row_end, end) - cur); }
  __device__ __forceinline__ void next() {
    cur += len();
    ++idx;
    if (cur == row_end) {
      ++row;
      row_end += V;
    }
  }
};

__global__ void __launch_bounds__(kFT, 1) verify_fused_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ uint8_t fsmem_raw[];
  float* ring = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(fsmem_raw) + 127) & ~uintptr_t(127));
  __shared__ uint64_t full[kFStages];
  __shared__ MS red[kFW];
  __shared__ Cand s_cr[kFW], s_cp[kFW];
  __shared__ int64_t s_rstart[kFMaxG + 1];
  __shared__ int s_last, s_tok, s_timeout, s_cf, s_cl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t V = a.V, K = a.K, Kp = a.Kp, Bn = a.Bn;
  const int64_t e0 = c < a.Gs ? a.sstart[c] : 0, e1 = c < a.Gs ? a.sstart[c + 1] : 0;

  // Inputs read before anything else: the drafted token of every row this
  // CTA streams, and this thread's accept inputs of step 2.
  __shared__ int32_t s_xd[kFMaxRowsPerSlice];
  const int64_t row0 = e0 / V;
  const int nrows = e0 < e1 ? int(min(int64_t(kFMaxRowsPerSlice), (e1 - 1) / V - row0 + 1)) : 0;
  if (tid < nrows) s_xd[tid] = int32_t(row_draft(a, row0 + tid));
  // (the first of this thread's accept tests; any further ones load in step 2)
  const int32_t x_pre = tid < Bn * K ? a.draft[tid] : 0;
  const float u_pre = tid < Bn * K ? a.u_acc[tid] : 0.f;
  if (tid == 0) {
    for (int s = 0; s < kFStages; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
    s_timeout = 0;
  }
  __syncthreads();

  // ------------------------------------------------------------ 1. statistics
  // Lane 0 of warps 0 and 1 issue the bulk copies of the even and odd chunks
  // (one issuing thread sustains too few copies); all threads consume.
  const bool producer = lane == 0 && warp < 2;
  ChunkCursor pk;  // (producers) the next chunk to consider issuing
  pk.init(e0, e1, V);
  uint32_t issued_hi = 0;  // (producers) one past the last chunk this thread issued
  auto issue_upto = [&](uint32_t j) {  // issue this thread's chunks with index <= j
    while (pk.cur < e1 && pk.idx <= j) {
      if ((pk.idx & 1u) == uint32_t(warp)) {
        const int slot = int(pk.idx % kFStages);
        const int64_t len = pk.len();
        const float* src = pk.cur < a.Np ? a.p + pk.cur : a.q + (pk.cur - a.Np);
        ptx::mbar_arrive_expect_tx(&full[slot], uint32_t(len) * 4u);
        ptx::bulk_load(ring + size_t(slot) * kFChunk, src, uint32_t(len) * 4u, &full[slot]);
        issued_hi = pk.idx + 1;
      }
      pk.next();
    }
  };
  if (producer) issue_upto(kFStages - 1);

  MS acc{-INFINITY, 0.f};
  ChunkCursor ck;
  ck.init(e0, e1, V);
  int64_t cur_row = ck.row;
  auto flush_row = [&]() {
    // block-reduce the running segment of row cur_row into its slot: this
    // CTA's rank among the row's CTAs; the row's first CTA pads the slots no
    // CTA fills
    const MS m = warp_merge(acc);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (tid == 0) {
      MS t = red[0];
      for (int w = 1; w < kFW; ++w) t = ms_merge(t, red[w]);
      const int cf = table_owner(a.sstart, a.Gs, cur_row * V);
      a.part[cur_row * a.S + (c - cf)] = make_float2(t.m, t.s);
      if (cf == c) {
        const int cl = table_owner(a.sstart, a.Gs, (cur_row + 1) * V - 1);
        for (int k = cl - cf + 1; k < a.S; ++k) a.part[cur_row * a.S + k] = make_float2(-INFINITY, 0.f);
      }
    }
    __syncthreads();
    acc = MS{-INFINITY, 0.f};
  };
  auto draft_of = [&](int64_t r) -> int64_t {
    return r - row0 < kFMaxRowsPerSlice ? int64_t(s_xd[r - row0]) : row_draft(a, r);
  };
  int64_t xd = e0 < e1 ? draft_of(cur_row) : -1;
  uint32_t i = 0;
  for (; ck.cur < e1; ++i) {
    const int64_t len = ck.len();
    if (ck.row != cur_row) {
      flush_row();
      cur_row = ck.row;
      xd = draft_of(cur_row);
    }
    const int slot = int(i % kFStages);
    // one thread waits for the stage (many threads polling the barrier slow
    // the copies landing in the same shared memory), then releases the block
    if (tid == 0 && !ptx::mbar_wait(&full[slot], (i / kFStages) & 1, kFWaitNs)) s_timeout = 1;
    __syncthreads();
    const int64_t v0 = ck.cur - cur_row * V;
    const float4* st4 = reinterpret_cast<const float4*>(ring + size_t(slot) * kFChunk);
    const int n4 = int(len >> 2);
    const int xq = (xd >= v0 && xd < v0 + len) ? int((xd - v0) >> 2) : -1;
    for (int k = tid; k < n4; k += kFT) {
      const float4 t = st4[k];
      ms_add4(acc, t.x, t.y, t.z, t.w);
      if (k == xq) {
        const int cc = int((xd - v0) & 3);
        a.gathered[cur_row] = cc == 0 ? t.x : cc == 1 ? t.y : cc == 2 ? t.z : t.w;
      }
    }
    __syncthreads();  // every thread is done with the slot before it is refilled
    if (s_timeout) break;
    if (producer) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // reads before the refill
      issue_upto(i + kFStages);
    }
    ck.next();
  }
  if (s_timeout) {
    // a copy did not land in time: issue nothing more, let this thread's
    // copies in flight land (bounded) before the CTA exits, report the failure
    if (producer) {
      for (uint32_t j = i; j < issued_hi; ++j)
        if ((j & 1u) == uint32_t(warp)) ptx::mbar_wait(&full[j % kFStages], (j / kFStages) & 1, kFWaitNs);
      if (warp == 0) atomicOr(&g_verify_error, 1);
    }
    return;
  }
  if (e0 < e1) flush_row();

  // ------------------------------------------------------------ grid barrier
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(&a.sync[0], 1);
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ld_acquire_gpu(&a.sync[0]) < a.G) {
      __nanosleep(32);
      if (ptx::globaltimer_ns() - t0 > kFWaitNs) {
        s_timeout = 1;
        break;
      }
    }
  }
  __syncthreads();
  if (s_timeout) {
    if (tid == 0) atomicOr(&g_verify_error, 1);
    return;
  }

  // ------------------------------------------------------------ 2. decisions
  // Row normalisers of every row, in the ring (idle now): max, max + ln(sum),
  // 1/sum; bad rows flag their sequence.
  const int64_t R = Bn * (Kp + K);
  const int64_t Rp = Bn * Kp;
  float* s_m = ring;
  float* s_lz = ring + R;
  float* s_iz = ring + 2 * R;
  int* s_n = reinterpret_cast<int*>(ring + 3 * R);  // [Bn] prefix length
  int* s_bad = s_n + Bn;                             // [Bn] status bits
  int* s_list = s_bad + Bn;                          // [Bn] sequences that race, in order
  int* s_nr = s_list + Bn;
  for (int64_t b = tid; b < Bn; b += kFT) {
    s_n[b] = int(K);
    s_bad[b] = 0;
  }
  __syncthreads();
  // one thread per row, its slots merged in slot order (loads of many rows in flight)
  for (int64_t r = tid; r < R; r += kFT) {
    MS t{-INFINITY, 0.f};
    for (int k0 = 0; k0 < a.S; k0 += 8) {
      float2 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = k0 + k < a.S ? __ldcg(a.part + r * a.S + k0 + k) : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) t = ms_merge(t, MS{v[k].x, v[k].y});
    }
    const int64_t b = r < Rp ? r / Kp : (r - Rp) / K;
    const bool bad = isnan(t.s) || !(t.m > -INFINITY) || !(t.m < INFINITY) || !(t.s > 0.f);
    if (bad) atomicOr(&s_bad[b], 2);
    s_m[r] = t.m;
    s_lz[r] = t.m + logf(t.s);
    s_iz[r] = 1.0f / t.s;
  }
  __syncthreads();
  for (int64_t t = tid; t < Bn * K; t += kFT) {
    const int64_t b = t / K, i2 = t - b * K;
    const int32_t x = t == tid ? x_pre : a.draft[t];
    if (x < 0 || x >= V) {
      atomicOr(&s_bad[b], 1);
      continue;
    }
    // accept x_i iff u_i < min(1, p_i(x_i)/q_i(x_i)), the ratio in the log domain
    const float lq = __ldcg(a.gathered + Rp + t);
    bool accept;
    if (lq == -INFINITY) {
      accept = true;  // q_i(x) = 0: ratio +inf
    } else {
      const float lp = __ldcg(a.gathered + b * Kp + i2);
      const float lr = (lp - s_lz[b * Kp + i2]) - (lq - s_lz[Rp + t]);
      accept = (t == tid ? u_pre : a.u_acc[t]) < fminf(1.0f, expf(lr));
    }
    if (!accept) atomicMin(&s_n[b], int(i2));
  }
  __syncthreads();
  if (tid == 0) {
    int nr = 0;
    for (int64_t b = 0; b < Bn; ++b)
      if (!s_bad[b] && (s_n[b] < K || Kp == K + 1)) s_list[nr++] = int(b);
    *s_nr = nr;
  }
  __syncthreads();
  // Sequences that draw no token (all accepted without a bonus row, or bad
  // data) are written here, each by one CTA.
  for (int64_t b = c; b < Bn; b += a.G) {
    const int bad = s_bad[b];
    const int n = s_n[b];
    if (!bad && (n < K || Kp == K + 1)) continue;
    int32_t* out = a.out_tokens + b * (K + 1);
    for (int64_t i2 = tid; i2 <= K; i2 += kFT) out[i2] = (!bad && i2 < K) ? a.draft[b * K + i2] : -1;
    if (tid == 0) {
      a.n_acc[b] = bad ? 0 : n;
      a.n_emit[b] = bad ? 0 : n;
      a.status[b] = bad ? ((bad & 1) ? UNO_SEQ_BAD_DRAFT : UNO_SEQ_NONFINITE) : UNO_SEQ_OK;
    }
  }

  // ------------------------------------------------------------ 3. race
  // residual: argmax_v max(0, p_n(v) - q_n(v)) / (-ln u_v), falling back to
  // p_n if no entry is positive; bonus: argmax_v p_K(v) / (-ln u_v).  Scores
  // are kept as fractions and compared by cross-multiplication.  The rows to
  // race form one range cut into Gr slices of at least 4 elements.
  const int nr = *s_nr;
  const int64_t RE = int64_t(nr) * V;
  const int Gr = int(max(int64_t(1), min(int64_t(a.G), RE / 4)));
  for (int k = tid; k <= Gr; k += kFT) s_rstart[k] = slice_start(RE, Gr, k);
  __syncthreads();
  const int64_t r0 = c < Gr ? s_rstart[c] : 0, r1 = c < Gr ? s_rstart[c + 1] : 0;
  constexpr float kLog2e = 1.4426950408889634f;
  for (int64_t rc = r0; rc < r1;) {
    const int idx = int(rc / V);
    const int64_t v0 = rc - int64_t(idx) * V;
    const int64_t v1 = min(V, r1 - int64_t(idx) * V);
    rc = int64_t(idx) * V + v1;
    const int64_t b = s_list[idx];
    const int n = s_n[b];
    const bool residual = n < K;
    const int64_t prow = residual ? n : K;
    const float* pr = a.p + (b * Kp + prow) * V;
    const float* qr = a.q + (b * K + (residual ? n : 0)) * V;
    const float* ub = a.u_res + b * V;
    const float mp = s_m[b * Kp + prow], izp = s_iz[b * Kp + prow];
    const float mq = residual ? s_m[Rp + b * K + n] : 0.f;
    const float izq = residual ? s_iz[Rp + b * K + n] : 0.f;
    float pn = -1.f, pd = 1.f, rn = 0.f, rd = 1.f;
    int pvid = -1, rvid = -1;
    const int64_t n4 = (v1 - v0) >> 2;
    for (int64_t k0 = tid; k0 < n4; k0 += int64_t(kFT) * kFRaceUnroll) {
      float4 u4[kFRaceUnroll], p4[kFRaceUnroll], q4[kFRaceUnroll];
#pragma unroll
      for (int w = 0; w < kFRaceUnroll; ++w) {
        const int64_t k = k0 + int64_t(w) * kFT;
        const bool in = k < n4;
        const int64_t v = v0 + 4 * k;
        u4[w] = in ? __ldcg(reinterpret_cast<const float4*>(ub + v)) : make_float4(0.5f, 0.5f, 0.5f, 0.5f);
        p4[w] = in ? __ldcg(reinterpret_cast<const float4*>(pr + v))
                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        q4[w] = (in && residual) ? __ldcg(reinterpret_cast<const float4*>(qr + v))
                                 : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int w = 0; w < kFRaceUnroll; ++w) {
        const int64_t k = k0 + int64_t(w) * kFT;
        if (k >= n4) break;
        const int64_t v = v0 + 4 * k;
        const float uu[4] = {u4[w].x, u4[w].y, u4[w].z, u4[w].w};
        const float lp[4] = {p4[w].x, p4[w].y, p4[w].z, p4[w].w};
        const float lq[4] = {q4[w].x, q4[w].y, q4[w].z, q4[w].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float e = -logf(uu[j]);
          const float pv = exp2f((lp[j] - mp) * kLog2e) * izp;
          if (pv * pd > pn * e) {  // pv / e > pn / pd; ties keep the lower id
            pn = pv;
            pd = e;
            pvid = int(v + j);
          }
          if (residual) {
            const float rv = pv - exp2f((lq[j] - mq) * kLog2e) * izq;
            if (rv > 0.f && rv * rd > rn * e) {
              rn = rv;
              rd = e;
              rvid = int(v + j);
            }
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
      for (int w = 1; w < kFW; ++w) {
        cr = cand_best(cr, s_cr[w]);
        cp = cand_best(cp, s_cp[w]);
      }
      // the CTAs whose slices overlap race row idx (every slice is non-empty)
      const int cf = table_owner(s_rstart, Gr, int64_t(idx) * V);
      const int cl = table_owner(s_rstart, Gr, int64_t(idx + 1) * V - 1);
      s_cf = cf;
      s_cl = cl;
      a.rpart[int64_t(idx) * a.G + (c - cf)] = RacePart{cr.s, cr.v, cp.s, cp.v};
      __threadfence();
      s_last = atomicAdd(&a.sync[1 + idx], 1) == cl - cf;
    }
    __syncthreads();
    const bool last = s_last != 0;
    if (last) {
      // the last CTA to arrive merges the slice winners, loads spread over the block
      __threadfence();
      const int ncon = s_cl - s_cf + 1;
      Cand br{0.f, -1}, bp{-1.f, -1};
      for (int k = tid; k < ncon; k += kFT) {
        const int4 t = __ldcg(reinterpret_cast<const int4*>(a.rpart + int64_t(idx) * a.G + k));
        br = cand_best(br, Cand{__int_as_float(t.x), t.y});
        bp = cand_best(bp, Cand{__int_as_float(t.z), t.w});
      }
      br = warp_best(br);
      bp = warp_best(bp);
      __syncthreads();
      if (lane == 0) {
        s_cr[warp] = br;
        s_cp[warp] = bp;
      }
      __syncthreads();
      if (tid == 0) {
        br = s_cr[0];
        bp = s_cp[0];
        for (int w = 1; w < kFW; ++w) {
          br = cand_best(br, s_cr[w]);
          bp = cand_best(bp, s_cp[w]);
        }
        a.n_acc[b] = n;
        a.n_emit[b] = n + 1;
        a.status[b] = UNO_SEQ_OK;
        s_tok = (residual && br.v >= 0) ? br.v : bp.v;
      }
      __syncthreads();
      const int tok = s_tok;
      int32_t* out = a.out_tokens + b * (K + 1);
      for (int64_t i2 = tid; i2 <= K; i2 += kFT)
        out[i2] = i2 < n ? a.draft[b * K + i2] : (i2 == n ? tok : -1);
    }
    __syncthreads();
  }
}

int fused_smem_bytes() { return int(kFRingBytes) + 128; }

}  // namespace

// Host plan of the fused path (pl.fused false when the sizes rule it out).
void plan_verify_fused(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int sms, VerifyPlan& pl) {
  pl.fused = false;
  pl.fused_bytes = 0;
  const int64_t R = Bn * (Kp + K);
  // the ring holds the normalisers of every row and three ints per sequence
  if (Bn < 1 || Bn > kFusedMaxBatch || K < 1 || V % 4 != 0 || sms < 1 ||
      (3 * R + 4 * Bn) * 4 > int64_t(kFRingBytes))
    return;
  const int G = std::min(sms, kFMaxG);
  const int64_t E = R * V;
  const int Gs = int(std::max<int64_t>(1, std::min<int64_t>(G, E / 4)));
  // a slice holds at least floor(E / Gs) - 3 elements: the most slices one row can meet
  const int64_t smin = std::max<int64_t>(1, E / Gs - 3);
  pl.fused_G = G;
  pl.fused_Gs = Gs;
  pl.fused_S = int(std::min<int64_t>(Gs, (V + smin - 1) / smin + 1));
  size_t o = 0;
  pl.off_fpart = o;
  o = align_up(o + size_t(R) * pl.fused_S * sizeof(float2), 256);
  pl.off_fgather = o;
  o = align_up(o + size_t(R) * sizeof(float), 256);
  pl.off_frace = o;
  o = align_up(o + size_t(Bn) * G * sizeof(RacePart), 256);
  pl.off_fsync = o;
  o = align_up(o + size_t(1 + Bn) * sizeof(int), 256);
  pl.fused_bytes = o;
  pl.fused = true;
}

cudaError_t launch_verify_fused(const float* p, const float* q, const int32_t* draft,
                                const float* u_acc, const float* u_res, int64_t Bn, int64_t K,
                                int64_t Kp, int64_t V, int32_t* n_acc, int32_t* out_tokens,
                                int32_t* n_emit, int32_t* status, void* ws, const VerifyPlan& pl,
                                cudaStream_t st) {
  static std::once_flag once[64];
  static cudaError_t attr_err[64] = {};
  static int resident[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  dev &= 63;
  std::call_once(once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(verify_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, fused_smem_bytes());
    if (attr_err[dev] == cudaSuccess)
      attr_err[dev] = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident[dev], verify_fused_kernel,
                                                                    kFT, fused_smem_bytes());
  });
  if (attr_err[dev] != cudaSuccess) return attr_err[dev];
  if (resident[dev] < 1) return cudaErrorCooperativeLaunchTooLarge;
  char* w = static_cast<char*>(ws);
  FusedArgs a{};
  a.p = p;
  a.q = q;
  a.draft = draft;
  a.u_acc = u_acc;
  a.u_res = u_res;
  a.Bn = Bn;
  a.K = K;
  a.Kp = Kp;
  a.V = V;
  a.E = Bn * (Kp + K) * V;
  a.Np = Bn * Kp * V;
  a.G = pl.fused_G;
  a.Gs = pl.fused_Gs;
  a.S = pl.fused_S;
  for (int c = 0; c <= kFMaxG; ++c) a.sstart[c] = c <= a.Gs ? slice_start(a.E, a.Gs, c) : a.E;
  a.part = reinterpret_cast<float2*>(w + pl.off_fpart);
  a.gathered = reinterpret_cast<float*>(w + pl.off_fgather);
  a.rpart = reinterpret_cast<RacePart*>(w + pl.off_frace);
  a.sync = reinterpret_cast<int*>(w + pl.off_fsync);
  a.n_acc = n_acc;
  a.out_tokens = out_tokens;
  a.n_emit = n_emit;
  a.status = status;
  cudaError_t e = cudaMemsetAsync(a.sync, 0, size_t(1 + Bn) * sizeof(int), st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(a.G));
  cfg.blockDim = dim3(kFT);
  cfg.dynamicSmemBytes = size_t(fused_smem_bytes());
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_fused_kernel, a);
}

int read_verify_error(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_verify_error, sizeof(int)) != cudaSuccess) return UNO_ERR_CUDA;
  if (reset) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_verify_error, &z, sizeof(int)) != cudaSuccess) return UNO_ERR_CUDA;
  }
  return v;
}

}  // namespace uno
