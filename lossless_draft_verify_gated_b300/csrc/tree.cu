// tree.cu -- verification half of the Psi-Spec tree sampler.
//
// "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
// (aifromscratch.in), section "The Psi-Spec Sampler": the tree sampler takes
// several candidates (the top K) at each position and verifies them in a
// prefix tree, for low batch sizes, while the emitted tokens keep the AR
// model's distribution.  Every drafted node is a deterministic candidate (a
// point-mass draft), for which the speculative rule reads: at the current node,
// with residual r (initially p at that node, mass S = 1), accept a child whose
// token is x with probability r(x)/S; on a rejection drop x from r (S -= r(x))
// and test the next child in index (rank) order; on an acceptance emit x and
// move to that child; when every child is rejected (or there is none) draw one
// token from r by the exponential race and stop.
//
// Two launches, as the linear verifier:
//   stats  -- the statistics pass of verify.cu over the N+1 node rows of every
//             sequence (per row (max, sum exp) partials);
//   finish -- one CTA per (sequence, vocab chunk): every CTA of a sequence
//             merges its rows' partials, and warp 0 walks the tree (children
//             found 32 at a time with a ballot, tested in index order); then
//             each CTA races its chunk of the final node's row with the
//             rejected tokens excluded (winners folded into 64-bit keys by
//             atomic max), and the last CTA to arrive (atomic count, no
//             waiting) reads the keys and writes the outputs.
// Nothing spins, nothing traps: a malformed tree or a non-finite row on the
// walked path sets the sequence's status.
#include <algorithm>

#include "ptx.cuh"
#include "uno_internal.h"
#include "verify_common.cuh"

namespace uno {
namespace {

using namespace vfy;

constexpr int kTT = 256;
constexpr int kTW = kTT / 32;
constexpr int kMaxNodeRows = int(kTreeMaxNodes) + 1;
static_assert(kMaxNodeRows <= kTT, "one thread per node row");

__global__ void __launch_bounds__(kTT)
tree_finish_kernel(const float* __restrict__ logits, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ token, const float* __restrict__ u_acc,
                   const float* __restrict__ u_res, int64_t N, int64_t V, int splits,
                   int race_splits, int64_t race_chunk, const float2* __restrict__ part,
                   unsigned long long* __restrict__ keys, int key_stride, int* __restrict__ counter,
                   int32_t* __restrict__ n_acc, int32_t* __restrict__ path,
                   int32_t* __restrict__ out_tokens, int32_t* __restrict__ n_emit,
                   int32_t* __restrict__ status) {
  __shared__ float s_m[kMaxNodeRows], s_lz[kMaxNodeRows], s_iz[kMaxNodeRows];
  __shared__ int s_rowbad[kMaxNodeRows];
  __shared__ int s_par[kMaxNodeRows], s_tok[kMaxNodeRows];
  __shared__ float s_u[kMaxNodeRows], s_lg[kMaxNodeRows];
  __shared__ int s_rej[kMaxNodeRows];   // tokens rejected at the final node, sorted
  __shared__ int s_path[kMaxNodeRows];  // accepted node ids by depth
  __shared__ int s_cur, s_depth, s_stat, s_nrej, s_last, s_tok_out;
  __shared__ Cand s_cr[kTW], s_cp[kTW];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t b = blockIdx.x / race_splits;
  const int split = int(blockIdx.x - b * race_splits);
  const int64_t N1 = N + 1;
  const float* lb = logits + b * N1 * V;

  // Inputs the statistics pass does not write, read before waiting for it:
  // this thread's node (parent, token, accept uniform) and, for a well-formed
  // node, the logit of its token in its parent's row.
  bool node_ok = true;
  if (tid < N1) {
    const int32_t pj = parent[b * N1 + tid];
    const int32_t xj = token[b * N1 + tid];
    s_par[tid] = pj;
    s_tok[tid] = xj;
    s_u[tid] = u_acc[b * N1 + tid];
    if (tid == 0) {
      node_ok = pj == -1;
    } else {
      node_ok = pj >= 0 && pj < tid && xj >= 0 && xj < V;
      s_lg[tid] = node_ok ? lb[int64_t(pj) * V + xj] : 0.f;
    }
  }
  const int64_t v0 = int64_t(split) * race_chunk;
  const int64_t v1 = min(V, v0 + race_chunk);
  const bool tree_ok = __syncthreads_and(node_ok) != 0;
  ptx::grid_dependency_wait();  // the statistics pass's partials and counters

  int32_t* out = out_tokens + b * N1;
  int32_t* pth = path + b * N;
  if (!tree_ok) {
    if (split == 0) {
      for (int64_t i = tid; i < N1; i += kTT) out[i] = -1;
      for (int64_t i = tid; i < N; i += kTT) pth[i] = -1;
      if (tid == 0) {
        n_acc[b] = 0;
        n_emit[b] = 0;
        status[b] = UNO_SEQ_BAD_DRAFT;
      }
    }
    return;
  }

  // 1. Row normalisers of the sequence's node rows: one warp per row, lanes
  //    over the chunk partials.
  for (int64_t j = warp; j < N1; j += kTW) {
    MS t{-INFINITY, 0.f};
    for (int s = lane; s < splits; s += 32) {
      const float2 v = part[(b * N1 + j) * splits + s];
      t = ms_merge(t, MS{v.x, v.y});
    }
    t = warp_merge(t);
    if (lane == 0) {
      s_rowbad[j] = isnan(t.s) || !(t.m > -INFINITY) || !(t.m < INFINITY) || !(t.s > 0.f);
      s_m[j] = t.m;
      s_lz[j] = t.m + logf(t.s);
      s_iz[j] = 1.0f / t.s;
    }
  }
  __syncthreads();

  // 2. The walk (warp 0; every value below is the same in all its lanes).
  if (warp == 0) {
    int cur = 0, depth = 0, stat = UNO_SEQ_OK, nrej = 0;
    while (true) {
      if (s_rowbad[cur]) {
        stat = UNO_SEQ_NONFINITE;
        break;
      }
      const float lzc = s_lz[cur];
      float S = 1.0f;
      int acc = -1;
      nrej = 0;
      for (int j0 = cur + 1; j0 <= N && acc < 0; j0 += 32) {
        const int j = j0 + lane;
        unsigned mask = __ballot_sync(0xffffffffu, j <= N && s_par[j] == cur);
        while (mask != 0u && acc < 0) {
          const int jj = j0 + __ffs(mask) - 1;
          mask &= mask - 1u;
          const int x = s_tok[jj];
          bool dup = false;  // x was rejected at this node already: its residual is 0
          for (int k = lane; k < nrej; k += 32) dup |= s_rej[k] == x;
          dup = __any_sync(0xffffffffu, dup);
          const float rx = dup ? 0.f : expf(s_lg[jj] - lzc);
          const float thr = S > 0.f ? rx / S : 0.f;
          if (s_u[jj] < thr) {
            acc = jj;
          } else {
            S -= rx;
            if (!dup) {
              if (lane == 0) s_rej[nrej] = x;
              ++nrej;
            }
            __syncwarp();
          }
        }
      }
      if (acc < 0) break;
      if (lane == 0) s_path[depth] = acc;
      ++depth;
      cur = acc;
    }
    if (lane == 0) {
      // the race skips rejected tokens by a forward scan: sort them
      for (int a = 1; a < nrej; ++a) {
        const int x = s_rej[a];
        int k = a - 1;
        while (k >= 0 && s_rej[k] > x) {
          s_rej[k + 1] = s_rej[k];
          --k;
        }
        s_rej[k + 1] = x;
      }
      s_cur = cur;
      s_depth = depth;
      s_stat = stat;
      s_nrej = nrej;
    }
  }
  __syncthreads();
  const int stat = s_stat;
  if (stat != UNO_SEQ_OK) {
    if (split == 0) {
      for (int64_t i = tid; i < N1; i += kTT) out[i] = -1;
      for (int64_t i = tid; i < N; i += kTT) pth[i] = -1;
      if (tid == 0) {
        n_acc[b] = 0;
        n_emit[b] = 0;
        status[b] = stat;
      }
    }
    return;
  }

  // 3. Race over this CTA's chunk of the final node's row: argmax_v p(v)/(-ln u_v)
  //    over the tokens not rejected there (cr), and over all of p (cp) should
  //    the rejected tokens have held all of p's mass.
  const int cur = s_cur;
  const int nrej = s_nrej;
  const float* pr = lb + int64_t(cur) * V;
  const float* ub = u_res + b * V;
  const float mp = s_m[cur], izp = s_iz[cur];
  constexpr float kLog2e = 1.4426950408889634f;
  float pn = -1.f, pd = 1.f, rn = 0.f, rd = 1.f;
  int pvid = -1, rvid = -1;
  int ptr = 0;  // first rejected token >= v (v grows along this thread's loop)
  constexpr int kU = 4;  // loads in flight per thread
  for (int64_t v0t = v0 + tid; v0t < v1; v0t += int64_t(kTT) * kU) {
    float uu[kU], lp[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int64_t v = v0t + int64_t(k) * kTT;
      uu[k] = v < v1 ? ub[v] : 0.5f;
      lp[k] = v < v1 ? pr[v] : -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int64_t v = v0t + int64_t(k) * kTT;
      if (v >= v1) break;
      const float e = -logf(uu[k]);
      const float pv = exp2f((lp[k] - mp) * kLog2e) * izp;
      while (ptr < nrej && s_rej[ptr] < v) ++ptr;
      const bool rejected = ptr < nrej && s_rej[ptr] == v;
      if (pv * pd > pn * e) {  // pv / e > pn / pd; ties keep the lower id
        pn = pv;
        pd = e;
        pvid = int(v);
      }
      if (!rejected && pv > 0.f && pv * rd > rn * e) {
        rn = pv;
        rd = e;
        rvid = int(v);
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
    for (int w = 1; w < kTW; ++w) {
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
        counter[b] = 0;
      }
    }
    s_last = last;
    s_tok_out = (cr.v >= 0) ? cr.v : cp.v;
  }
  __syncthreads();
  if (!s_last) return;
  const int depth = s_depth;
  const int tok = s_tok_out;
  for (int64_t i = tid; i < N1; i += kTT)
    out[i] = i < depth ? s_tok[s_path[i]] : (i == depth ? tok : -1);
  for (int64_t i = tid; i < N; i += kTT) pth[i] = i < depth ? s_path[i] : -1;
  if (tid == 0) {
    n_acc[b] = depth;
    n_emit[b] = depth + 1;
    status[b] = UNO_SEQ_OK;
  }
}

}  // namespace

cudaError_t launch_tree_verify(const float* logits, const int32_t* parent, const int32_t* token,
                               const float* u_acc, const float* u_res, int64_t Bn, int64_t N,
                               int64_t V, int32_t* n_acc, int32_t* path, int32_t* out_tokens,
                               int32_t* n_emit, int32_t* status, void* ws, const VerifyPlan& pl,
                               cudaStream_t st) {
  // node rows as the AR rows of a block with no draft rows (K = 0, Kp = N + 1)
  // (the statistics pass also zeroes the race's arrival counts and winner keys)
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + pl.off_race);
  const int key_stride = 2 * std::max(pl.race_splits, pl.icdf_splits);
  cudaError_t e = launch_row_stats(logits, logits, parent, Bn, 0, N + 1, V, pl, ws, st, keys, key_stride);
  if (e != cudaSuccess) return e;
  char* w = static_cast<char*>(ws);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(Bn * pl.race_splits));
  cfg.blockDim = dim3(kTT);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // (see launch_verify)
  return cudaLaunchKernelEx(&cfg, tree_finish_kernel, logits, parent, token, u_acc, u_res, N, V,
                            pl.splits, pl.race_splits, pl.race_chunk,
                            reinterpret_cast<const float2*>(w + pl.off_stats),
                            keys, key_stride,
                            reinterpret_cast<int*>(w + pl.off_count), n_acc, path, out_tokens,
                            n_emit, status);
}

}  // namespace uno
