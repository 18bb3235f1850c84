// gemm.cu -- gated-LoRA linear projections on the tcgen05 tensor cores.
//
//   y = x.W^T + gate_row * (alpha/rank) * (x.A^T).B^T
// "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
// (aifromscratch.in), section "Two Decoupled Weight Sets": rows of the draft
// pathway (gate 1) get theta_AR plus the rank-128, alpha-256 adapter
// theta_Delta; verification rows (gate 0) get theta_AR alone.
//
// One persistent, warp-specialised kernel computes a whole group of
// projections (for example the seven projections of a transformer layer):
//
//   * Work is a flat sequence of 64-wide K-blocks: first the down-projection
//     tiles of every problem, T = bf16(gate * alpha/rank * x.A^T), then the
//     main tiles, each made of its d_in/64 base K-blocks followed by its
//     rank/64 adapter K-blocks (A-operand B, B-operand T).  The adapter
//     therefore accumulates into the same TMEM accumulator as x.W^T: W is
//     streamed from HBM once and y is written once.
//   * CTA c of G takes the contiguous K-block range [c*Tot/G, (c+1)*Tot/G)
//     ("stream-K"), so every SM streams the same number of K-blocks whatever
//     the shapes.  A tile cut by range boundaries is finished by the last of
//     its CTAs to arrive, which sums the partials in CTA order
//     (deterministic results, nobody waits).
//   * A main tile's adapter K-blocks need T: the producer waits (bounded) on
//     the flag its down tile sets.  Down tiles come first in the sequence and
//     never wait, so the wait always ends; the launch is cooperative so all
//     CTAs are resident.
//
// Roles (192 threads): warp 0 lane 0 issues TMA (cp.async.bulk.tensor, 128-byte
// swizzle) into a STAGES-deep shared-memory ring; warp 1 owns TMEM and its
// lane 0 issues tcgen05.mma (M=128, N=bn, K=16, bf16 -> fp32) into one of two
// TMEM accumulators; warps 2-5 drain the other accumulator (tcgen05.ld) and
// store y, T or split-K partials, overlapping the next tile's MMAs.
// Decode-sized M (<= 256 token rows) swaps the operands so that the weights
// fill the 128-row MMA side and the tokens are N.
// Every wait is bounded (2 s): a timeout sets the device error word and the
// CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "ptx.cuh"
#include "uno_internal.h"

namespace uno {

__device__ int g_device_error;  // bit 0: a pipeline wait in the projection kernel timed out

namespace {

constexpr int kBM = 128;    // MMA M: A-operand rows per tile (= TMEM lanes)
constexpr int kBK = 64;     // K elements per K-block (one 128-byte swizzle row of bf16)
constexpr int kUmmaK = 16;  // K of one tcgen05.mma for 16-bit inputs
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMaxPhases = 2 * kMaxLoraProblems;

enum { MAP_X = 0, MAP_W = 1, MAP_A = 2, MAP_B = 3, MAP_T = 4, kMapsPerProblem = 5 };

struct Maps {
  CUtensorMap m[kMaxLoraProblems][kMapsPerProblem];
};

struct Phase {
  int64_t kb_start;  // first K-block of the phase in the global sequence
  int tiles;
  int tiles_a;       // tiles along the A-operand rows
  int nkb;           // K-blocks per tile
  int nkb_base;      // of which over d_in; the rest are adapter K-blocks
  int prob;
  int down;          // 1: T = gate*scale*x.A^T;  0: y = x.W^T + T.B^T
  int bn;            // MMA N (B-operand rows per tile)
};

struct Prob {
  void* y;
  void* t;
  const uint8_t* gate;
  float scale;
  int d_out;
  int r;
  int flag_base;
  int down_tiles;
};

struct Params {
  Phase ph[kMaxPhases];
  Prob pb[kMaxLoraProblems];
  int nph;
  int swap;
  int M;
  int out_f32;
  int grid;
  int bnmax;
  int64_t total;
  float* partial;  // [grid][2][bnmax * 128], layout [column/4][row][4]
  int* counters;   // [grid]
  int* flags;      // [sum of down tiles]
};

// Tuning constants: K-blocks per pipeline stage (a stage holds KPS consecutive
// 64-wide K slices, so a weight row is read as KPS*128 contiguous bytes) and
// the shared-memory budget of the ring.
#ifndef UNO_KPS_DECODE
#define UNO_KPS_DECODE 1
#endif
#ifndef UNO_MAX_STAGES
#define UNO_MAX_STAGES 8
#endif
constexpr uint32_t kRingBudget = 200 * 1024;

template <int BNMAX>
__host__ __device__ constexpr int kps_for() {
  return BNMAX <= 64 ? UNO_KPS_DECODE : 1;
}
template <int BNMAX, int KPS>
__host__ __device__ constexpr uint32_t stage_bytes() {
  return uint32_t(KPS) * uint32_t(kBM * kBK * 2 + BNMAX * kBK * 2);
}
template <int BNMAX, int KPS>
__host__ __device__ constexpr int stages_for() {
  return int(kRingBudget / stage_bytes<BNMAX, KPS>()) < UNO_MAX_STAGES
             ? int(kRingBudget / stage_bytes<BNMAX, KPS>())
             : UNO_MAX_STAGES;
}
template <int BNMAX, int KPS>
__host__ __device__ constexpr uint32_t smem_bytes_for() {
  return uint32_t(stages_for<BNMAX, KPS>()) * stage_bytes<BNMAX, KPS>() + 1024 + 256;
}

__device__ __forceinline__ int64_t range_lo(int c, int G, int64_t T) { return int64_t(c) * T / G; }
// CTA whose range holds K-block k: the largest c with range_lo(c) <= k.
__device__ __forceinline__ int cta_of(int64_t k, int G, int64_t T) {
  return int(((k + 1) * G - 1) / T);
}

struct Seg {
  int ph, tile;
  int64_t tstart, tend, s, e;
};

__device__ __forceinline__ Seg locate(const Params& P, int64_t k, int64_t hi) {
  Seg g;
  int p = 0;
  while (p + 1 < P.nph && P.ph[p + 1].kb_start <= k) ++p;
  const Phase& f = P.ph[p];
  g.ph = p;
  g.tile = int((k - f.kb_start) / f.nkb);
  g.tstart = f.kb_start + int64_t(g.tile) * f.nkb;
  g.tend = g.tstart + f.nkb;
  g.s = k;
  g.e = hi < g.tend ? hi : g.tend;
  return g;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async;" ::: "memory");
}
__device__ __forceinline__ void epi_sync() {  // named barrier of the 4 epilogue warps
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}
__device__ __forceinline__ bool wait_flag(const int* f, uint64_t limit_ns) {
  if (ld_acquire(f)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ld_acquire(f)) {
    __nanosleep(100);
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Stores 16 consecutive accumulator columns (c0 .. c0+15) of TMEM lane `row`.
__device__ __forceinline__ void store16(const Params& P, const Phase& f, const Prob& pb, int ta,
                                       int tb, int row, int c0, const float (&v)[16]) {
  const int ncols = f.down ? pb.r : pb.d_out;
  __nv_bfloat16* dst16 = static_cast<__nv_bfloat16*>(f.down ? pb.t : pb.y);
  if (P.swap) {
    // lane = output column n, accumulator column = token m
    const int n = ta * kBM + row;
    if (n >= ncols) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int m = tb * f.bn + c0 + j;
      if (m >= P.M) break;
      float x = v[j];
      if (f.down) x *= float(pb.gate[m]) * pb.scale;
      if (!f.down && P.out_f32)
        static_cast<float*>(pb.y)[int64_t(m) * ncols + n] = x;
      else
        dst16[int64_t(m) * ncols + n] = __float2bfloat16_rn(x);
    }
  } else {
    // lane = token m, accumulator column = output column n
    const int m = ta * kBM + row;
    if (m >= P.M) return;
    const int n0 = tb * f.bn + c0;
    const float gs = f.down ? float(pb.gate[m]) * pb.scale : 1.f;
    if (!f.down && P.out_f32) {
      float* d = static_cast<float*>(pb.y) + int64_t(m) * ncols;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (n0 + j < ncols) d[n0 + j] = v[j];
    } else if (n0 + 16 <= ncols) {
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j] * gs, v[2 * j + 1] * gs);
        w[j] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint4* d = reinterpret_cast<uint4*>(dst16 + int64_t(m) * ncols + n0);
      d[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (n0 + j < ncols) dst16[int64_t(m) * ncols + n0 + j] = __float2bfloat16_rn(v[j] * gs);
    }
  }
}

template <int BNMAX, int KPS>
__global__ void __launch_bounds__(kThreads, 1)
grouped_lora_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Params P) {
  constexpr int STAGES = stages_for<BNMAX, KPS>();
  constexpr uint32_t kABytes = kBM * kBK * 2;            // one A sub-tile (128 x 64)
  constexpr uint32_t kBSub = BNMAX * kBK * 2;            // one B sub-tile slot (BNMAX x 64)
  constexpr uint32_t kStage = stage_bytes<BNMAX, KPS>();  // KPS A sub-tiles, then KPS B slots
  constexpr uint32_t kTmemCols = 2 * BNMAX < 32 ? 32 : 2 * BNMAX;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2] accumulator ready
  uint64_t* tempty = tfull + 2;      // [2] accumulator drained
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = P.grid;
  const int64_t lo = range_lo(blockIdx.x, G, P.total);
  const int64_t hi = range_lo(blockIdx.x + 1, G, P.total);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], kEpiThreads / 32);
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol_first = ptx::policy_evict_first();
      const uint64_t pol_last = ptx::policy_evict_last();
      // swap: A = weights (streamed once), B = tokens (reused by every tile);
      // otherwise A = tokens, B = weights, both reused across tiles from L2.
      const uint64_t polA = P.swap ? pol_first : pol_last;
      const uint64_t polB = pol_last;
      uint32_t it = 0;
      for (int64_t k = lo; k < hi && !*abort_flag;) {
        const Seg g = locate(P, k, hi);
        const Phase& f = P.ph[g.ph];
        const Prob& pb = P.pb[f.prob];
        const CUtensorMap* mp = maps.m[f.prob];
        const int ta = g.tile % f.tiles_a, tb = g.tile / f.tiles_a;
        const uint32_t bytes = kABytes + uint32_t(f.bn) * kBK * 2;  // per K-block
        bool t_ready = false;
        for (int64_t kk = g.s; kk < g.e; ++it) {
          const int s = int(it % STAGES);
          const int n = int(g.e - kk < KPS ? g.e - kk : KPS);  // K-blocks in this stage
          if (it >= STAGES && !ptx::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          if (!f.down && !t_ready && int(kk + n - 1 - g.tstart) >= f.nkb_base) {
            // The rows of T this tile reads must be complete before TMA reads them.
            bool ok = true;
            if (P.swap) {
              for (int i = 0; i < pb.down_tiles && ok; ++i)
                ok = wait_flag(P.flags + pb.flag_base + i, kWaitLimitNs);
            } else {
              ok = wait_flag(P.flags + pb.flag_base + ta, kWaitLimitNs);
            }
            if (!ok) {
              *abort_flag = 1;
              break;
            }
            fence_proxy_async();
            t_ready = true;
          }
          uint8_t* sa = smem + s * kStage;
          ptx::mbar_arrive_expect_tx(&full[s], bytes * uint32_t(n));
          for (int j = 0; j < n; ++j, ++kk) {
            const int kl = int(kk - g.tstart);
            const CUtensorMap *ma, *mb;
            int kc;
            if (f.down) {
              ma = &mp[P.swap ? MAP_A : MAP_X];
              mb = &mp[P.swap ? MAP_X : MAP_A];
              kc = kl * kBK;
            } else if (kl < f.nkb_base) {
              ma = &mp[P.swap ? MAP_W : MAP_X];
              mb = &mp[P.swap ? MAP_X : MAP_W];
              kc = kl * kBK;
            } else {
              ma = &mp[P.swap ? MAP_B : MAP_T];
              mb = &mp[P.swap ? MAP_T : MAP_B];
              kc = (kl - f.nkb_base) * kBK;
            }
            ptx::tma_load_2d(sa + j * kABytes, ma, &full[s], kc, ta * kBM, polA);
            ptx::tma_load_2d(sa + KPS * kABytes + j * kBSub, mb, &full[s], kc, tb * f.bn, polB);
          }
        }
        k = g.e;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA can exit
        const uint32_t first = it > uint32_t(STAGES) ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i)
          ptx::mbar_wait(&full[i % STAGES], (i / STAGES) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      uint32_t it = 0;
      int seg = 0;
      for (int64_t k = lo; k < hi && !*abort_flag; ++seg) {
        const Seg g = locate(P, k, hi);
        const Phase& f = P.ph[g.ph];
        const int acc = seg & 1;
        if (seg >= 2 && !ptx::mbar_wait(&tempty[acc], ((seg >> 1) - 1) & 1, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + uint32_t(acc * BNMAX);
        const uint32_t idesc = ptx::idesc_bf16_f32(kBM, f.bn);
        for (int64_t kk = g.s; kk < g.e; ++it) {
          const int s = int(it % STAGES);
          const int n = int(g.e - kk < KPS ? g.e - kk : KPS);
          if (!ptx::mbar_wait(&full[s], (it / STAGES) & 1, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(smem + s * kStage);
          const uint32_t sb = sa + KPS * kABytes;
          for (int j = 0; j < n; ++j, ++kk) {
#pragma unroll
            for (int u = 0; u < kBK / kUmmaK; ++u)
              ptx::umma_f16(d, ptx::sw128_kmajor_desc(sa + j * kABytes + u * 32),
                            ptx::sw128_kmajor_desc(sb + j * kBSub + u * 32), idesc,
                            (kk > g.s || u > 0) ? 1u : 0u);
          }
          ptx::umma_commit(&empty[s]);
        }
        ptx::umma_commit(&tfull[acc]);
        k = g.e;
      }
      // once this arrives, every MMA issued by this thread has completed
      ptx::umma_commit(mma_done);
      ptx::mbar_wait(mma_done, 0, kWaitLimitNs);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 64;
    int seg = 0;
    for (int64_t k = lo; k < hi; ++seg) {
      const Seg g = locate(P, k, hi);
      const Phase& f = P.ph[g.ph];
      const Prob& pb = P.pb[f.prob];
      const int ta = g.tile % f.tiles_a, tb = g.tile / f.tiles_a;
      const int acc = seg & 1;
      if (!ptx::mbar_wait(&tfull[acc], (seg >> 1) & 1, kWaitLimitNs)) *abort_flag = 1;
      epi_sync();
      if (*abort_flag) break;
      ptx::tc_fence_after();
      const uint32_t tq = tmem + uint32_t(acc * BNMAX) + (uint32_t(q * 32) << 16);
      const bool whole = (g.s == g.tstart && g.e == g.tend);
      bool finish = whole;
      if (whole) {
        for (int c = 0; c < f.bn; c += 16) {
          uint32_t r[16];
          ptx::tmem_ld_32x32b_x16(tq + c, r);
          ptx::tmem_ld_wait(r);
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
          store16(P, f, pb, ta, tb, row, c, v);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
      } else {
        // Part of a tile: leave a partial; the last CTA of the tile to arrive
        // adds the partials in CTA order and writes the result.
        const int slot = (g.s == lo) ? 0 : 1;
        // partial layout [column/4][row][4]: each thread moves float4s and a
        // warp touches 512 contiguous bytes per access
        float4* dst = reinterpret_cast<float4*>(
            P.partial + (size_t(blockIdx.x) * 2 + slot) * (size_t(P.bnmax) * kBM));
        for (int c = 0; c < f.bn; c += 16) {
          uint32_t r[16];
          ptx::tmem_ld_32x32b_x16(tq + c, r);
          ptx::tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcg(dst + ((c >> 2) + i) * kBM + row,
                   make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                               __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
        __threadfence();
        epi_sync();
        const int c0 = cta_of(g.tstart, G, P.total);
        const int c1 = cta_of(g.tend - 1, G, P.total);
        if (et == 0) *last_flag = atomicAdd(P.counters + c0, 1) == c1 - c0;
        epi_sync();
        finish = *last_flag != 0;
        if (finish) {
          __threadfence();
          // Sum the partials in CTA order: 32 columns of up to 4 CTAs in flight.
          for (int c = 0; c < f.bn; c += 32) {
            float4 sum[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cb = c0; cb <= c1; cb += 4) {
              float4 t[4][8];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int cc = cb + u;
                const float4* src = nullptr;
                if (cc <= c1) {
                  const int sl = range_lo(cc, G, P.total) >= g.tstart ? 0 : 1;
                  src = reinterpret_cast<const float4*>(
                      P.partial + (size_t(cc) * 2 + sl) * (size_t(P.bnmax) * kBM));
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  t[u][i] = (src && c + 4 * i < f.bn) ? __ldcg(src + ((c >> 2) + i) * kBM + row)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  sum[i].x += t[u][i].x;
                  sum[i].y += t[u][i].y;
                  sum[i].z += t[u][i].z;
                  sum[i].w += t[u][i].w;
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (c + 16 * h >= f.bn) break;
              float v[16];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                v[4 * i] = sum[4 * h + i].x;
                v[4 * i + 1] = sum[4 * h + i].y;
                v[4 * i + 2] = sum[4 * h + i].z;
                v[4 * i + 3] = sum[4 * h + i].w;
              }
              store16(P, f, pb, ta, tb, row, c + 16 * h, v);
            }
          }
          if (et == 0) P.counters[c0] = 0;
        }
      }
      if (f.down && finish) {
        // publish this down tile: its part of T is in global memory
        fence_proxy_async();
        __threadfence();
        epi_sync();
        if (et == 0) st_release(P.flags + pb.flag_base + ta, 1);
      }
      k = g.e;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicOr(&g_device_error, 1);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void cast_f32_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                     int64_t n) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    out[i] = __float2bfloat16_rn(in[i]);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor [outer, inner] (inner contiguous), boxes of 64 x box_outer,
// 128-byte swizzle, out-of-range elements read as zero.
bool encode_bf16(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  cuuint64_t strides[1] = {cuuint64_t(inner) * 2};
  cuuint32_t box[2] = {uint32_t(kBK), uint32_t(box_outer)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pick_bn(int64_t n) {
  for (int bn : {16, 32, 64, 128}) if (n <= bn) return bn;
  return 256;
}

struct Layout {
  Params P;
  size_t off_t[kMaxLoraProblems];
  size_t off_partial, off_sync, sync_bytes;
  size_t off_cast[kMaxLoraProblems][4];  // fp32 mode: bf16 copies of x, W, A, B
  size_t bytes;
};

// Host-side schedule: phases of the global K-block sequence, grid size and
// workspace layout.  Depends only on shapes and the SM count.
bool make_layout(int n, const uno_lora_problem* pr, int64_t M, int dtype, int sms, Layout& L) {
  if (n < 1 || n > kMaxLoraProblems) return false;
  std::memset(&L, 0, sizeof(L));
  Params& P = L.P;
  P.M = int(M);
  P.swap = M <= 256 ? 1 : 0;
  P.out_f32 = dtype == UNO_F32;
  const int bn_tok = pick_bn(M);
  int64_t kb = 0;
  int nph = 0, flags = 0, bnmax = 16;
  for (int p = 0; p < n; ++p) {  // down-projection phases first
    Prob& b = P.pb[p];
    b.d_out = int(pr[p].d_out);
    b.r = int(pr[p].rank);
    b.scale = pr[p].rank > 0 ? pr[p].alpha / float(pr[p].rank) : 0.f;
    b.flag_base = flags;
    if (pr[p].rank == 0) continue;
    Phase& f = P.ph[nph++];
    f.kb_start = kb;
    f.prob = p;
    f.down = 1;
    f.nkb = f.nkb_base = int((pr[p].d_in + kBK - 1) / kBK);
    if (P.swap) {
      f.tiles_a = int((pr[p].rank + kBM - 1) / kBM);
      f.bn = bn_tok;
    } else {
      f.tiles_a = int((M + kBM - 1) / kBM);
      f.bn = pick_bn(pr[p].rank);
    }
    f.tiles = f.tiles_a;
    b.down_tiles = f.tiles;
    flags += f.tiles;
    kb += int64_t(f.tiles) * f.nkb;
    bnmax = std::max(bnmax, f.bn);
  }
  for (int p = 0; p < n; ++p) {  // then the main phases
    Phase& f = P.ph[nph++];
    f.kb_start = kb;
    f.prob = p;
    f.down = 0;
    f.nkb_base = int((pr[p].d_in + kBK - 1) / kBK);
    f.nkb = f.nkb_base + int((pr[p].rank + kBK - 1) / kBK);
    if (P.swap) {
      f.tiles_a = int((pr[p].d_out + kBM - 1) / kBM);
      f.bn = bn_tok;
      f.tiles = f.tiles_a;
    } else {
      f.tiles_a = int((M + kBM - 1) / kBM);
      f.bn = pick_bn(pr[p].d_out);
      f.tiles = f.tiles_a * int((pr[p].d_out + f.bn - 1) / f.bn);
    }
    kb += int64_t(f.tiles) * f.nkb;
    bnmax = std::max(bnmax, f.bn);
  }
  P.nph = nph;
  P.total = kb;
  P.bnmax = bnmax;
  // One CTA per SM, at least 4 K-blocks each.
  P.grid = int(std::max<int64_t>(1, std::min<int64_t>(sms, kb / 4)));
  size_t o = 0;
  for (int p = 0; p < n; ++p) {
    L.off_t[p] = o;
    o = align_up(o + size_t(M) * size_t(pr[p].rank) * 2, 256);
  }
  L.off_partial = o;
  o = align_up(o + size_t(P.grid) * 2 * size_t(bnmax) * kBM * sizeof(float), 256);
  L.off_sync = o;
  L.sync_bytes = align_up((size_t(P.grid) + size_t(flags)) * sizeof(int), 256);
  o += L.sync_bytes;
  if (dtype == UNO_F32) {
    for (int p = 0; p < n; ++p) {
      const size_t sz[4] = {size_t(M) * pr[p].d_in, size_t(pr[p].d_out) * pr[p].d_in,
                            size_t(pr[p].rank) * pr[p].d_in, size_t(pr[p].d_out) * pr[p].rank};
      for (int i = 0; i < 4; ++i) {
        L.off_cast[p][i] = o;
        o = align_up(o + sz[i] * 2, 256);
      }
    }
  }
  L.bytes = std::max<size_t>(o, 256);
  return true;
}

cudaError_t cast_to_bf16(const void* in, void* out, int64_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 148 * 16);
  cast_f32_bf16_kernel<<<unsigned(blocks), 256, 0, st>>>(static_cast<const float*>(in),
                                                        static_cast<__nv_bfloat16*>(out), n);
  return cudaGetLastError();
}

template <int BNMAX>
cudaError_t launch_grouped(const Maps& maps, const Params& P, cudaStream_t st) {
  constexpr int KPS = kps_for<BNMAX>();
  static std::once_flag once[64];
  static cudaError_t attr_err[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  dev &= 63;
  std::call_once(once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(grouped_lora_gemm_kernel<BNMAX, KPS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem_bytes_for<BNMAX, KPS>()));
  });
  if (attr_err[dev] != cudaSuccess) return attr_err[dev];
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(P.grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for<BNMAX, KPS>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_lora_gemm_kernel<BNMAX, KPS>, maps, P);
}

}  // namespace

size_t lora_group_workspace_bytes(int n, const uno_lora_problem* pr, int64_t M, int dtype,
                                  int sms) {
  Layout L;
  if (!make_layout(n, pr, M, dtype, sms, L)) return 0;
  return L.bytes;
}

int launch_lora_group(int n, const uno_lora_problem* pr, int64_t M, int dtype, void* ws,
                      size_t ws_bytes, cudaStream_t st) {
  Layout L;
  if (!make_layout(n, pr, M, dtype, sm_count(), L)) return UNO_ERR_ARG;
  if (ws_bytes < L.bytes) return UNO_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  Params& P = L.P;
  P.partial = reinterpret_cast<float*>(w + L.off_partial);
  P.counters = reinterpret_cast<int*>(w + L.off_sync);
  P.flags = P.counters + P.grid;
  Maps maps;
  std::memset(&maps, 0, sizeof(maps));
  for (int p = 0; p < n; ++p) {
    const uno_lora_problem& q = pr[p];
    const void *x = q.x, *W = q.W, *A = q.A, *B = q.B;
    if (dtype == UNO_F32) {
      void* c[4];
      for (int i = 0; i < 4; ++i) c[i] = w + L.off_cast[p][i];
      if (cast_to_bf16(q.x, c[0], M * q.d_in, st) != cudaSuccess ||
          cast_to_bf16(q.W, c[1], q.d_out * q.d_in, st) != cudaSuccess ||
          (q.rank > 0 && (cast_to_bf16(q.A, c[2], q.rank * q.d_in, st) != cudaSuccess ||
                          cast_to_bf16(q.B, c[3], q.d_out * q.rank, st) != cudaSuccess)))
        return UNO_ERR_CUDA;
      x = c[0];
      W = c[1];
      A = c[2];
      B = c[3];
    }
    Prob& b = P.pb[p];
    b.y = q.y;
    b.t = w + L.off_t[p];
    b.gate = q.gate;
    int bn_main = 0, bn_down = 0;
    for (int i = 0; i < P.nph; ++i)
      if (P.ph[i].prob == p) (P.ph[i].down ? bn_down : bn_main) = P.ph[i].bn;
    CUtensorMap* m = maps.m[p];
    const bool sw = P.swap != 0;
    bool ok = encode_bf16(&m[MAP_X], x, q.d_in, M, sw ? bn_main : kBM) &&
              encode_bf16(&m[MAP_W], W, q.d_in, q.d_out, sw ? kBM : bn_main);
    if (ok && q.rank > 0) {
      ok = encode_bf16(&m[MAP_A], A, q.d_in, q.rank, sw ? kBM : bn_down) &&
           encode_bf16(&m[MAP_B], B, q.rank, q.d_out, sw ? kBM : bn_main) &&
           encode_bf16(&m[MAP_T], b.t, q.rank, M, sw ? bn_main : kBM);
    } else {
      m[MAP_A] = m[MAP_B] = m[MAP_T] = m[MAP_X];
    }
    if (!ok) return UNO_ERR_CUDA;
  }
  if (cudaMemsetAsync(w + L.off_sync, 0, L.sync_bytes, st) != cudaSuccess) return UNO_ERR_CUDA;
  cudaError_t e;
  switch (P.bnmax) {
    case 16: e = launch_grouped<16>(maps, P, st); break;
    case 32: e = launch_grouped<32>(maps, P, st); break;
    case 64: e = launch_grouped<64>(maps, P, st); break;
    case 128: e = launch_grouped<128>(maps, P, st); break;
    default: e = launch_grouped<256>(maps, P, st); break;
  }
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}

int read_device_error(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return UNO_ERR_CUDA;
  if (reset) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(int)) != cudaSuccess) return UNO_ERR_CUDA;
  }
  return v;
}

}  // namespace uno
