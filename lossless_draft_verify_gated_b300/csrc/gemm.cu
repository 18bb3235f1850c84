// gemm.cu -- gated-LoRA linear projections on the tcgen05 tensor cores.
//
//   y = x.W^T + gate_row * (alpha/rank) * (x.A^T).B^T
// "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
// (aifromscratch.in), section "Two Decoupled Weight Sets": rows of the draft
// pathway (gate 1) get theta_AR plus the rank-128, alpha-256 adapter
// theta_Delta; verification rows (gate 0) get theta_AR alone.
//
// One persistent, warp-specialised kernel computes a whole group of
// projections (for example the seven projections of a transformer layer).
//
// Work is split into 64-wide K-blocks, in two sections:
//   * the down section (token-row order only): tiles of
//     T = bf16(gate * alpha/rank * x.A^T), one run of tiles per problem with
//     a nonzero rank;
//   * the main section: tiles of y, each a flat run of rank/64 adapter
//     K-blocks (A-operand B, B-operand T) followed by d_in/64 base K-blocks
//     (x.W^T).  The adapter accumulates into the same TMEM accumulator as
//     x.W^T, so W is streamed from HBM once and y is written once.
// CTA c owns a contiguous range of each section (stream-K): the down section
// is spread over enough CTAs that each does a few K-blocks, first thing, so
// T is complete early; the main ranges are sized so that every CTA streams
// the same number of K-blocks in total.  Inside a range piece a CTA runs the
// base K-blocks first and the adapter K-blocks last, so T is needed only at
// the end of a piece.
//
// A tile cut between CTAs is finished by the CTA that owns its first K-block
// (for that CTA it is always the last piece of the section).  The other
// owners hold their piece of the tile as the first piece of their range:
// they leave it as an fp32 partial and raise a flag.  The finisher adds the
// partials in CTA order to its own accumulator (deterministic).  Every wait
// points at a CTA with a higher index or at a flag raised before any wait of
// its raiser, so waits always end once all CTAs are resident (see
// launch_grouped).  A main tile's adapter K-blocks wait for the flags of the
// T tiles they read.
//
// Roles (224 threads): lane 0 of warps 0 and 6 issue TMA (cp.async.bulk.tensor,
// 128-byte swizzle) into the even and odd stages of a shared-memory ring;
// warp 1 owns TMEM and its lane 0 issues tcgen05.mma (M=128, N=bn, K=16,
// bf16 -> fp32) into one of two TMEM accumulators; warps 2-5 drain the other
// accumulator (tcgen05.ld) and store y, T or partials, overlapping the next
// piece's MMAs.
// Decode-sized M (<= 128 token rows) swaps the operands so that the weights
// fill the 128-row MMA side and the tokens are N, and computes T by split K
// in the epilogue warps, which are idle until a CTA's first accumulator is
// full: CTA c computes the partial T of one chunk of one problem's d_in with
// warp-level MMAs, then, once every chunk of that problem is in, sums a slice
// of T over the chunks in a fixed order and publishes it; the weight stream
// never carries the down matrix and no T tile waits on a merge.  Larger
// M takes tiles of 128 tokens x 256 (or 128) outputs and, with at least one
// tile per CTA, deals whole tiles out in data-parallel waves (no splits); a
// split T tile of that order is merged by slices over its pieces when a
// CTA's share of K-blocks is short.  With 256-token tiles for at least half
// of the CTA pairs and little padding, a launch runs instead as clusters of
// two CTAs (pair_gemm_kernel, below): 256 x 256 tiles by the pair MMA, each
// CTA loading half of every operand.
// Launches are chained with programmatic dependent launch: each CTA lets the
// next launch in the stream start at once, and waits (griddepcontrol.wait)
// for the previous one before it touches global memory, except for L2
// prefetch hints of its first weight tiles (L2 is the coherence point, so a
// hint can never return stale data).  A one-CTA kernel before each launch
// clears the schedule's flags once the previous launch has finished.
// Every wait is bounded (2 s): a timeout sets the device error word and the
// CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <atomic>
#include <vector>
#include <mutex>

#include "ptx.cuh"
#include "uno_internal.h"
#include "verify_common.cuh"

namespace uno {

__device__ int g_device_error;  // bit 0: a pipeline wait in the projection kernel timed out

namespace {

constexpr int kBM = 128;    // MMA M: A-operand rows per tile (= TMEM lanes)
constexpr int kBK = 64;     // K elements per K-block (one 128-byte swizzle row of bf16)
constexpr int kUmmaK = 16;  // K of one tcgen05.mma for 16-bit inputs
constexpr int kThreads = 224;  // warps: 0 and 6 TMA, 1 MMA, 2-5 epilogue
constexpr int kEpiThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMaxPhases = 4 * kMaxLoraProblems;
constexpr int kMaxGrid = 160;  // CTAs of one launch (one per SM)
constexpr int kPrefetchKBlocks = 8;  // weight tiles hinted into L2 before the previous launch ends
constexpr int64_t kTSliceMaxShare = 160;  // K-blocks a CTA, for T tiles merged by slices
constexpr int64_t kLocalTMaxWeightBytes = int64_t(80) << 20;
constexpr int64_t kSwapMaxRows = 128;  // above this many token rows, tokens are the A operand
constexpr bool kPairMma = true;       // large M: data-parallel tiles by CTA pairs (pair MMA)
constexpr bool kSplitKAdapter = true;  // decode order: T by split K in the epilogue warps
// (up to 64 token rows: the operands of a chunk are staged in the finisher
// staging area, which exists for tiles of at most 64 tokens)
constexpr int64_t kSplitKMaxRows = 64;
constexpr int kDown = 0, kMain = 1;

// MAP_W2 / MAP_B2: (pair order) W and B with 64-row boxes, for the 128-wide
// tiles that finish a launch's last wave
enum { MAP_X = 0, MAP_W = 1, MAP_A = 2, MAP_B = 3, MAP_T = 4, MAP_W2 = 5, MAP_B2 = 6, kMapsPerProblem = 7 };

struct Maps {
  CUtensorMap m[kMaxLoraProblems][kMapsPerProblem];
};

// A run of equally shaped tiles of one problem inside a section.
struct Phase {
  int64_t kb_start;  // first K-block of the phase in its stream-K section
  int tile0;         // first tile of the phase in its problem's tile grid
  int tbase;         // (data-parallel phases) first tile in the combined tile list
  int tiles;
  int tiles_a;       // tiles along the A-operand rows
  int tiles_all;     // tiles of the problem's whole grid (tiles_a x tiles along B)
  int nkb;           // K-blocks per tile
  int na;            // of which adapter K-blocks, first in the flat order (large-M path)
  int nad;           // adapter K-blocks appended to every piece (swap path)
  int prob;
  int down;          // 1: T = gate*scale*x.A^T;  0: y = T.B^T + x.W^T
  int bn;            // MMA N (B-operand rows per tile)
  int n0;            // (pair order) first output column of the phase's tiles
};

struct Prob {
  void* y;
  void* t;
  const uint8_t* gate;
  float scale;
  int d_in;
  int d_out;
  int r;
  int tflag0;  // first T-ready flag of the problem (split-K adapter: [chunks in, slices out])
  int ttiles;  // T tiles of the problem
  int f32out;  // store y as fp32 (bf16 operands)
  // Statistics epilogue (logit rows of the verifier, rank 0): instead of (or
  // besides, st_store) storing y, every finished tile leaves per row the
  // (max, sum exp) of its columns in st_part[row * st_nvt + vocab tile] and
  // the logit of the row's drafted token in st_gather[row].  Rows are grouped
  // per sequence as st_Kp AR rows then st_K draft rows.
  int st_store;
  int st_K, st_Kp, st_Rp, st_nvt;
  const int32_t* st_draft;
  float2* st_part;
  float* st_gather;
};

struct Params {
  Phase ph[kMaxPhases];
  Prob pb[kMaxLoraProblems];
  int ph0[2], ph1[2];  // stream-K section s holds phases [ph0[s], ph1[s])
  int dp0, dp1;        // data-parallel phases [dp0, dp1) (large M)
  int dp_tiles;        // tiles of the data-parallel waves: tile t goes to CTA t % grid
  int nprob;           // problems of the launch
  int swap;
  int localt;  // swap path with per-piece adapter
  int tslice;  // (token-rows order) split T tiles merge and publish by slices
  int pair;    // pair order: data-parallel tiles of 256 tokens by CTA pairs (pair_gemm_kernel)
  // Split-K adapter (decode order): the epilogue warps of CTA c < tchunks
  // compute the partial T of chunk c (tkpc K-blocks of one problem's d_in;
  // problem p owns chunks [tch0[p], tch0[p+1])), then reduce a slice of T.
  int tsplit;
  int tkpc;
  int tchunks;
  int tbn;  // rows of the x boxes (tokens, rounded up to the tile width)
  int tch0[kMaxLoraProblems + 1];
  int64_t tpart_stride;  // floats between chunk partials ([M][r] each)
  float* tpart;
  int M;
  int out_f32;
  int grid;
  int bnmax;
  int64_t lo[2][kMaxGrid + 1];  // CTA c owns K-blocks [lo[s][c], lo[s][c+1]) of section s
  float* partial;  // [grid][2][bnmax * 128], layout [column/4][row][4]
  int* ready;      // [2][grid]: the first piece of CTA c in section s left its partial
  int* tflag;      // [T tiles]: the rows of T of the tile are written (a count of
                   // slices for a split T tile of the token-rows order)
  int* tcnt;       // [T tiles] (token-rows order): pieces of a split T tile whose partial is in
};

// Shared memory (per CTA): a ring of STAGES stages, each one K-block of the
// A operand (128 x 64), the B operand (BNMAX x 64) and, when each piece
// computes its own share of the adapter (LOCALT), a 128 x 64 slice of the
// down matrix; with LOCALT, the piece's adapter input T' as the B operand of
// its up-projection (two 64-wide K-blocks); then, for decode-sized tiles
// (N <= 64), a staging area into which a finisher bulk-copies its
// contributors' partials.
constexpr int kMaxStages = 10;
constexpr uint32_t kABytes = kBM * kBK * 2;  // one 128 x 64 bf16 sub-tile
constexpr int kMaxLocalRank = 128;           // LOCALT keeps T' for ranks <= 128
constexpr int64_t kSharedTStaging = 96 * 1024;  // staging of decode tiles with a shared T

template <int BNMAX>
__host__ __device__ constexpr bool pre_merge() {
  return BNMAX <= 64;
}
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr uint32_t staging_bytes() {
  return pre_merge<BNMAX>() ? (LOCALT ? 64u * 1024 : uint32_t(kSharedTStaging)) : 0u;
}
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr int staging_slots() {  // partials the staging area holds at once
  return pre_merge<BNMAX>() ? int(staging_bytes<BNMAX, LOCALT>() / (uint32_t(BNMAX) * 128 * 4)) : 0;
}
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr uint32_t stage_bytes() {
  return kABytes + uint32_t(BNMAX) * kBK * 2 + (LOCALT ? kABytes : 0u);
}
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr uint32_t tprime_bytes() {
  return LOCALT ? uint32_t(BNMAX) * 128u * uint32_t(kMaxLocalRank / kBK) : 0u;
}
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr int stages_for() {
  return int((216 * 1024 - staging_bytes<BNMAX, LOCALT>() - tprime_bytes<BNMAX, LOCALT>()) /
             stage_bytes<BNMAX, LOCALT>()) < kMaxStages
             ? int((216 * 1024 - staging_bytes<BNMAX, LOCALT>() - tprime_bytes<BNMAX, LOCALT>()) /
                   stage_bytes<BNMAX, LOCALT>())
             : kMaxStages;
}
// TMEM accumulators: y (double-buffered when TMEM allows) and, with LOCALT,
// the piece's T.
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr int acc_bufs() {
  return (LOCALT && 3 * BNMAX > 512) ? 1 : 2;
}
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr uint32_t tmem_cols() {
  return (acc_bufs<BNMAX, LOCALT>() + (LOCALT ? 1 : 0)) * BNMAX <= 32    ? 32u
         : (acc_bufs<BNMAX, LOCALT>() + (LOCALT ? 1 : 0)) * BNMAX <= 64  ? 64u
         : (acc_bufs<BNMAX, LOCALT>() + (LOCALT ? 1 : 0)) * BNMAX <= 128 ? 128u
         : (acc_bufs<BNMAX, LOCALT>() + (LOCALT ? 1 : 0)) * BNMAX <= 256 ? 256u
                                                                         : 512u;
}
// Barriers and the TMEM slot, then a copy of the kernel parameters.
constexpr uint32_t kBarrierBytes = 512;
constexpr uint32_t kParamsBytes = (uint32_t(sizeof(Params)) + 15u) & ~15u;
// Decode order: the gates of every problem's tokens, staged once per CTA,
// then the split-K adapter's reduction scratch (one float4 per epilogue thread).
constexpr uint32_t kGateOnlyBytes = uint32_t(kMaxLoraProblems) * uint32_t(kSwapMaxRows);
constexpr uint32_t kGateBytes = kGateOnlyBytes + 2048;
template <int BNMAX, bool LOCALT>
__host__ __device__ constexpr uint32_t smem_bytes_for() {
  return uint32_t(stages_for<BNMAX, LOCALT>()) * stage_bytes<BNMAX, LOCALT>() +
         tprime_bytes<BNMAX, LOCALT>() + staging_bytes<BNMAX, LOCALT>() + kBarrierBytes + kParamsBytes +
         kGateBytes + 1024;
}

// A piece: K-blocks [s, e) of tile `tile` (whose K-blocks are [tstart, tend)),
// in stream-K section `sec`, or a whole data-parallel tile (sec = -1).
struct Seg {
  int ph, tile, sec;
  int64_t tstart, tend, s, e;
};

__device__ __forceinline__ Seg locate(const Params& P, int sec, int64_t k, int64_t hi) {
  Seg g;
  int p = P.ph0[sec];
  while (p + 1 < P.ph1[sec] && P.ph[p + 1].kb_start <= k) ++p;
  const Phase& f = P.ph[p];
  const int local = int((k - f.kb_start) / f.nkb);
  g.ph = p;
  g.sec = sec;
  g.tile = f.tile0 + local;
  g.tstart = f.kb_start + int64_t(local) * f.nkb;
  g.tend = g.tstart + f.nkb;
  g.s = k;
  g.e = hi < g.tend ? hi : g.tend;
  return g;
}

// Tile coordinates (A-operand rows ta, B-operand rows tb) of tile `tile` of a
// phase.  Tiles run through bands of up to 16 A-row tiles, all B-row tiles
// of a band before the next band, so that the tiles of a wave in flight
// share a compact set of operand tiles in L2.
__device__ __forceinline__ void tile_coords(const Phase& f, int tile, int& ta, int& tb) {
  const int tiles_b = f.tiles_all / f.tiles_a;
  const int S = f.tiles_a < 16 ? f.tiles_a : 16;
  const int band = tile / (S * tiles_b);
  const int r = tile - band * S * tiles_b;
  const int rows = f.tiles_a - band * S < S ? f.tiles_a - band * S : S;
  ta = band * S + r % rows;
  tb = r / rows;
}

// The pieces of one CTA, in order: its data-parallel tiles (t = cta, cta +
// grid, ...), then its ranges of the two stream-K sections.
struct PieceIter {
  int t, sec;
  int64_t k, hi;
  __device__ __forceinline__ PieceIter(const Params& P, int cta)
      : t(cta), sec(0), k(P.lo[0][cta]), hi(P.lo[0][cta + 1]) {}
  __device__ __forceinline__ bool next(const Params& P, int cta, Seg& g) {
    if (t < P.dp_tiles) {
      int p = P.dp0;
      while (p + 1 < P.dp1 && P.ph[p + 1].tbase <= t) ++p;
      const Phase& f = P.ph[p];
      g.ph = p;
      g.sec = -1;
      g.tile = f.tile0 + (t - f.tbase);
      g.tstart = g.s = 0;
      g.tend = g.e = f.nkb;
      t += P.grid;
      return true;
    }
    while (sec < 2) {
      if (k < hi) {
        g = locate(P, sec, k, hi);
        k = g.e;
        return true;
      }
      if (++sec < 2) {
        k = P.lo[sec][cta];
        hi = P.lo[sec][cta + 1];
      }
    }
    return false;
  }
};

// Flat position of the i-th K-block a CTA runs in piece g: base K-blocks
// first, then the adapter K-blocks (flat positions [tstart, tstart + na)).
__device__ __forceinline__ int64_t piece_kb(const Seg& g, int na, int64_t i) {
  const int64_t bs = g.s > g.tstart + na ? g.s : g.tstart + na;
  const int64_t nb = g.e > bs ? g.e - bs : 0;
  return i < nb ? bs + i : g.s + (i - nb);
}

// CTA whose range of section `sec` holds K-block k (ranges may be empty).
__device__ __forceinline__ int owner_of(const Params& P, int sec, int64_t k) {
  int a = 0, b = P.grid - 1;
  while (a < b) {
    const int m = (a + b + 1) >> 1;
    if (P.lo[sec][m] <= k) a = m; else b = m - 1;
  }
  return a;
}

// Token-rows order: the CTAs [c0, c0 + np) that hold the pieces of T tile
// `ta` of problem `prob` in the down section, one piece each (np = 1, c0 = -1
// for a T tile that is not split).
__device__ __forceinline__ void t_tile_span(const Params& P, int prob, int ta, int& c0, int& np) {
  c0 = -1;
  np = 1;
  if (!P.tslice) return;  // a split T tile has one finisher, which publishes it
  for (int p = P.ph0[kDown]; p < P.ph1[kDown]; ++p) {
    const Phase& f = P.ph[p];
    const int t = ta - f.tile0;
    if (f.prob != prob || t < 0 || t >= f.tiles) continue;
    const int64_t kb0 = f.kb_start + int64_t(t) * f.nkb;
    c0 = owner_of(P, kDown, kb0);
    np = owner_of(P, kDown, kb0 + f.nkb - 1) - c0 + 1;
    return;
  }
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
// Barrier of the 4 epilogue warps that also ORs `v` over them: every thread
// gets the same answer.
__device__ __forceinline__ bool epi_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(v)), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void red_add_relaxed(int* p, int v) {
  asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Waits until the counter at f reaches target (acquire), for at most limit_ns.
__device__ __forceinline__ bool wait_count(const int* f, int target, uint64_t limit_ns) {
  if (ld_acquire(f) >= target) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ld_acquire(f) < target) {
    __nanosleep(64);
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
__device__ __forceinline__ bool wait_flag(const int* f, uint64_t limit_ns) {
  if (ld_acquire(f)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ld_acquire(f)) {
    __nanosleep(64);
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// Waits (bounded) until every CTA in [c_from, c_to] whose range of section
// `sec` is not empty has raised its ready flag.  The flags of up to 16 CTAs
// are loaded at once (relaxed) and one fence then gives them acquire
// semantics, so a batch costs one round trip to L2 instead of one per CTA.
__device__ __forceinline__ bool wait_ready(const Params& P, int sec, int c_from, int c_to,
                                           uint64_t limit_ns) {
  const int* flags = P.ready + sec * P.grid;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (int c = c_from; c <= c_to; c += 16) {
    while (true) {
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        v[i] = (c + i <= c_to && P.lo[sec][c + i] < P.lo[sec][c + i + 1]) ? ld_relaxed(flags + c + i) : 1;
      int ok = 1;
#pragma unroll
      for (int i = 0; i < 16; ++i) ok &= v[i] != 0;
      if (ok) break;
      if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
      __nanosleep(32);
    }
  }
  fence_acq_rel_gpu();
  return true;
}

// Stores 16 consecutive accumulator columns (c0 .. c0+15) of TMEM lane `row`.
// Must be called by all 32 lanes of the warp (the swap path shuffles).
__device__ __forceinline__ void store16(const Params& P, const Phase& f, const Prob& pb, int ta,
                                       int tb, int row, int c0, const float (&v)[16],
                                       const uint8_t* gate_s) {
  const int ncols = f.down ? pb.r : pb.d_out;
  __nv_bfloat16* dst16 = static_cast<__nv_bfloat16*>(f.down ? pb.t : pb.y);
  if (P.swap) {
    // lane = output column, accumulator column = token.  An 8x8 transpose
    // by xor-shuffles inside each group of 8 lanes leaves lane 8k+i with 8
    // consecutive output columns of one token: one 16-byte store per lane.
    const int lane = row & 31;
    const int i = lane & 7;
    const int n = ta * kBM + (row & ~7);  // first output column of this lane group
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      float r[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) r[j] = v[8 * g + j];
#pragma unroll
      for (int sh = 4; sh > 0; sh >>= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j & sh) continue;
          const float send = (i & sh) ? r[j] : r[j + sh];
          const float got = __shfl_xor_sync(0xffffffffu, send, sh);
          if (i & sh) r[j] = got; else r[j + sh] = got;
        }
      }
      const int m = tb * f.bn + c0 + 8 * g + i;  // token of this lane
      if (m >= P.M || n >= ncols) continue;
      if (f.down) {
        const float gs = float(gate_s[f.prob * int(kSwapMaxRows) + m]) * pb.scale;
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] *= gs;
      }
      if (!f.down && (P.out_f32 || pb.f32out)) {
        float4* d = reinterpret_cast<float4*>(static_cast<float*>(pb.y) + int64_t(m) * ncols + n);
        d[0] = make_float4(r[0], r[1], r[2], r[3]);
        d[1] = make_float4(r[4], r[5], r[6], r[7]);
      } else {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __nv_bfloat162 h = __floats2bfloat162_rn(r[2 * j], r[2 * j + 1]);
          w[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(dst16 + int64_t(m) * ncols + n) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {
    // lane = token m, accumulator column = output column n
    const int m = ta * kBM + row;
    if (m >= P.M) return;
    const int n0 = f.n0 + tb * f.bn + c0;
    const float gs = f.down ? float(pb.gate[m]) * pb.scale : 1.f;
    if (!f.down && (P.out_f32 || pb.f32out)) {
      float* d = static_cast<float*>(pb.y) + int64_t(m) * ncols;
      if (n0 + 16 <= ncols && (reinterpret_cast<uintptr_t>(d + n0) & 31u) == 0) {
        // two 256-bit stores (full 32-byte sectors)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(d + n0 + 8 * h),
                       "f"(v[8 * h]), "f"(v[8 * h + 1]), "f"(v[8 * h + 2]), "f"(v[8 * h + 3]),
                       "f"(v[8 * h + 4]), "f"(v[8 * h + 5]), "f"(v[8 * h + 6]), "f"(v[8 * h + 7])
                       : "memory");
      } else if (n0 + 16 <= ncols) {  // ncols and n0 are multiples of 8: 16-byte stores
        float4* d4 = reinterpret_cast<float4*>(d + n0);
#pragma unroll
        for (int j = 0; j < 4; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (n0 + j < ncols) d[n0 + j] = v[j];
      }
    } else if (n0 + 16 <= ncols) {
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j] * gs, v[2 * j + 1] * gs);
        w[j] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint4* d = reinterpret_cast<uint4*>(dst16 + int64_t(m) * ncols + n0);
      // a lane's 16 outputs are one 32-byte sector: one 256-bit store when aligned
      if ((reinterpret_cast<uintptr_t>(d) & 31u) == 0) {
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(d), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
      } else {
        d[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (n0 + j < ncols) dst16[int64_t(m) * ncols + n0 + j] = __float2bfloat16_rn(v[j] * gs);
    }
  }
}

__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  ptx::tmem_ld_32x32b_x16(taddr, r);
  ptx::tmem_ld_wait(r);
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Split-K adapter, run by the 128 epilogue threads of CTA `cta` < tchunks
// before their first accumulator arrives (they are idle until then):
//   1. the partial T_c[m][j] = sum_{k in chunk c} x[m,k] A[j,k] of the CTA's
//      chunk: TMA brings the chunk's K-blocks of A and x into the staging
//      area (128-byte swizzle, as for the main operands) in as few rounds as
//      it holds; warp w multiplies rank rows 32w..32w+31 of every 128 with
//      warp-level MMAs; the partial is stored as fp32 [M][r] and counted in;
//   2. once all nch chunks of the problem are in, slice idx of the [M][r]
//      entries summed over the chunks -- each thread a fixed stride of
//      chunks, then the stride groups in order, so every run adds in the same
//      order -- and stored as T = bf16(gate[m] * alpha/r * sum), counted out.
// A main tile's adapter K-blocks wait for every slice of their problem.
// Counts are released by a fence and a relaxed add (one fence, not two).
// Returns false if a wait gave up.
__device__ bool tsplit_run(const Params& P, const Maps& maps, int cta, int et,
                           const uint8_t* gate_s, float4* red, uint8_t* stg, uint32_t stg_bytes,
                           uint64_t* stg_bar, uint32_t& stg_phase) {
  const int ch = cta;
  int p = 0;
  while (P.tch0[p + 1] <= ch) ++p;
  const Prob& pb = P.pb[p];
  const int nch = P.tch0[p + 1] - P.tch0[p];
  const int idx = ch - P.tch0[p];
  const int r = pb.r, M = P.M;
  const int nkb_p = (pb.d_in + kBK - 1) / kBK;
  const int kb0 = idx * P.tkpc;
  const int kb1 = min(nkb_p, kb0 + P.tkpc);
  int* cnt = P.tflag + pb.tflag0;  // [0] chunks in, [1] slices out
  {
    const int rt = (r + kBM - 1) / kBM;                  // 128-row tiles of A
    const uint32_t xbytes = uint32_t(P.tbn) * kBK * 2;   // one K-block of x
    const uint32_t per_kb = uint32_t(rt) * kABytes + xbytes;
    const int kb_round = int(stg_bytes / per_kb);        // K-blocks per round (>= 1)
    float* part = P.tpart + int64_t(ch) * P.tpart_stride;
    const int wq = et >> 5, lane = et & 31, g = lane >> 2, t2 = 2 * (lane & 3);
    const CUtensorMap* mp = maps.m[p];
    const uint32_t sbase = ptx::smem_u32(stg);
    // 32-bit word (two bf16) at (row, k) of a 128-byte-swizzled [rows][64] tile
    auto lds = [](uint32_t tile, int row, int k) -> uint32_t {
      uint32_t v;
      const uint32_t a = tile + uint32_t(row) * 128u + (uint32_t(((k >> 3) ^ row) & 7) << 4) +
                         uint32_t(k & 7) * 2u;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
      return v;
    };
    // K-blocks [kr, kr + nk) into the staging area; every thread takes part
    // (the barrier before the copies: the area is free; the one after the
    // wait: every thread gets the same answer)
    auto load_round = [&](int kr, int nk) -> bool {
      epi_sync();
      if (et == 0) {
        fence_proxy_async();
        ptx::mbar_arrive_expect_tx(stg_bar, uint32_t(nk) * per_kb);
        for (int i = 0; i < nk; ++i) {
          uint8_t* d = stg + size_t(i) * per_kb;
          for (int t = 0; t < rt; ++t)
            ptx::tma_load_2d(d + size_t(t) * kABytes, &mp[MAP_A], stg_bar, (kr + i) * kBK, t * kBM,
                             ptx::policy_evict_first());
          ptx::tma_load_2d(d + size_t(rt) * kABytes, &mp[MAP_X], stg_bar, (kr + i) * kBK, 0,
                           ptx::policy_evict_last());
        }
      }
      const bool ok = ptx::mbar_wait(stg_bar, stg_phase & 1, kWaitLimitNs);
      ++stg_phase;
      return !epi_sync_or(!ok);
    };
    const bool once = kb1 - kb0 <= kb_round;  // the whole chunk fits: one round
    if (once && !load_round(kb0, kb1 - kb0)) return false;
    // passes over rank rows (128 at a time) and tokens (32 at a time), the
    // same for every warp; a warp whose rows start beyond the rank idles
    for (int jp = 0; jp < r; jp += kBM) {
      for (int n0 = 0; n0 < M; n0 += 32) {
        const int j0 = jp + wq * 32;
        const bool active = j0 < r;
        const int ti = jp / kBM;  // A tile of this pass
        float acc[2][4][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int ni = 0; ni < 4; ++ni)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mi][ni][i] = 0.f;
        for (int kr = kb0; kr < kb1; kr += kb_round) {
          const int nk = min(kb_round, kb1 - kr);
          if (!once && !load_round(kr, nk)) return false;
          if (!active) continue;
          for (int i = 0; i < nk; ++i) {
            const uint32_t ta = sbase + uint32_t(i) * per_kb + uint32_t(ti) * kABytes;
            const uint32_t tx = sbase + uint32_t(i) * per_kb + uint32_t(rt) * kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK; kk += 16) {
              uint32_t a[2][4], b[4][2];
#pragma unroll
              for (int mi = 0; mi < 2; ++mi) {
                const int row = wq * 32 + 16 * mi + g;  // row in the A tile (rows >= r are zero)
                a[mi][0] = lds(ta, row, kk + t2);
                a[mi][1] = lds(ta, row + 8, kk + t2);
                a[mi][2] = lds(ta, row, kk + 8 + t2);
                a[mi][3] = lds(ta, row + 8, kk + 8 + t2);
              }
#pragma unroll
              for (int ni = 0; ni < 4; ++ni) {
                const int m = n0 + 8 * ni + g;  // token rows M .. tbn-1 are the tile's zero fill
                b[ni][0] = m < P.tbn ? lds(tx, m, kk + t2) : 0u;
                b[ni][1] = m < P.tbn ? lds(tx, m, kk + 8 + t2) : 0u;
              }
#pragma unroll
              for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) ptx::mma_bf16_16816(acc[mi][ni], a[mi], b[ni]);
            }
          }
        }
        if (!active) continue;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int ni = 0; ni < 4; ++ni) {
            const int j = j0 + 16 * mi + g, m = n0 + 8 * ni + t2;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int jj = j + 8 * h;
              if (jj >= r) continue;
              if (m < M) part[int64_t(m) * r + jj] = acc[mi][ni][2 * h];
              if (m + 1 < M) part[int64_t(m + 1) * r + jj] = acc[mi][ni][2 * h + 1];
            }
          }
      }
    }
  }
  epi_sync();
  if (et == 0) {
    fence_acq_rel_gpu();
    red_add_relaxed(cnt, 1);
  }
  bool ok = true;
  if (et == 0) ok = wait_count(cnt, nch, kWaitLimitNs);
  if (epi_sync_or(!ok)) return false;
  {
    const int64_t E4 = int64_t(M) * r / 4;  // r is a multiple of 8
    const int64_t s0 = E4 * idx / nch, s1 = E4 * (idx + 1) / nch;
    const float4* base = reinterpret_cast<const float4*>(P.tpart + int64_t(P.tch0[p]) * P.tpart_stride);
    const int64_t cs4 = P.tpart_stride / 4;
    __nv_bfloat16* T = static_cast<__nv_bfloat16*>(pb.t);  // [M][r]
    for (int64_t e0 = s0; e0 < s1; e0 += kEpiThreads) {
      const int S = int(s1 - e0 < kEpiThreads ? s1 - e0 : int64_t(kEpiThreads));
      const int G2 = kEpiThreads / S;  // chunk strides
      const int e = et % S, cg = et / S;
      float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (cg < G2) {
#pragma unroll 8
        for (int c = cg; c < nch; c += G2) {
          const float4 v = __ldcg(base + int64_t(c) * cs4 + e0 + e);
          a4.x += v.x;
          a4.y += v.y;
          a4.z += v.z;
          a4.w += v.w;
        }
      }
      red[et] = a4;
      epi_sync();
      if (et < S) {
        float4 sum = red[et];
        for (int q2 = 1; q2 < G2; ++q2) {
          const float4 v = red[q2 * S + et];
          sum.x += v.x;
          sum.y += v.y;
          sum.z += v.z;
          sum.w += v.w;
        }
        const int64_t ei = (e0 + et) * 4;
        const int m = int(ei / r), j = int(ei - int64_t(m) * r);
        const float gs = float(gate_s[p * int(kSwapMaxRows) + m]) * pb.scale;
        __nv_bfloat162 lo = __floats2bfloat162_rn(sum.x * gs, sum.y * gs);
        __nv_bfloat162 hi = __floats2bfloat162_rn(sum.z * gs, sum.w * gs);
        *reinterpret_cast<uint2*>(T + int64_t(m) * r + j) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      }
      epi_sync();
    }
  }
  // T is read next by TMA in other CTAs
  fence_proxy_async();
  epi_sync();
  if (et == 0) {
    fence_acq_rel_gpu();
    red_add_relaxed(cnt + 1, 1);
  }
  return true;
}

// ---------------------------------------------------------- statistics epilogue
// Drafted token of logit row m (-1 for a bonus AR row).  Rows: the st_Rp AR
// rows (sequence b, position j at b*Kp + j), then the draft rows (b, i) at
// st_Rp + b*K + i.
__device__ __forceinline__ int row_draft_token(const Prob& pb, int m) {
  if (m < pb.st_Rp) {
    const int b = m / pb.st_Kp, j = m - b * pb.st_Kp;
    return j < pb.st_K ? pb.st_draft[int64_t(b) * pb.st_K + j] : -1;
  }
  return pb.st_draft[m - pb.st_Rp];
}

// Decode order (lane = vocabulary entry n, accumulator column = token): the
// (max, sum exp) of 16 tokens over this warp's 32 entries by butterflies, then
// over the tile's 4 warps through shared memory; one partial per (token, tile).
// All 128 epilogue threads call it together.
__device__ __forceinline__ void stats16_swap(const Params& P, const Phase& f, const Prob& pb, int ta,
                                             int tb, int row, int c0, const float (&v)[16],
                                             const int* xd_s, float2* red, int et) {
  const int n = ta * kBM + row;
  const bool okn = n < pb.d_out;
  const int lane = row & 31, q = row >> 5;
  float mx[16], sm[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) mx[j] = okn ? v[j] : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < 16; ++j) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], o));
#pragma unroll
  for (int j = 0; j < 16; ++j) sm[j] = (okn && mx[j] != -INFINITY) ? __expf(v[j] - mx[j]) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < 16; ++j) sm[j] += __shfl_xor_sync(0xffffffffu, sm[j], o);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int m = tb * f.bn + c0 + j;
    if (okn && m < P.M && xd_s[m] == n) pb.st_gather[m] = v[j];
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < 16; ++j) red[q * 16 + j] = make_float2(mx[j], sm[j]);
  }
  epi_sync();
  if (et < 16) {
    const int m = tb * f.bn + c0 + et;
    vfy::MS t{-INFINITY, 0.f};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 r = red[w * 16 + et];
      t = vfy::ms_merge(t, vfy::MS{r.x, r.y});
    }
    if (m < P.M) pb.st_part[int64_t(m) * pb.st_nvt + ta] = make_float2(t.m, t.s);
  }
  epi_sync();
}

// Large-M order (lane = token row m, accumulator column = vocabulary entry):
// a running (max, sum exp) per thread over the tile's columns; stats_end
// writes it once the tile's last columns are in.
__device__ __forceinline__ void stats16_rows(const Phase& f, const Prob& pb, int tb, int c0,
                                             const float (&v)[16], int xd, int m_ok, float* gather_m,
                                             vfy::MS& acc) {
  const int n0 = tb * f.bn + c0;
  float x[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = n0 + j < pb.d_out ? v[j] : -INFINITY;
#pragma unroll
  for (int j = 0; j < 16; j += 4) vfy::ms_add4(acc, x[j], x[j + 1], x[j + 2], x[j + 3]);
  if (m_ok && xd >= n0 && xd < n0 + 16) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (xd == n0 + j) *gather_m = v[j];
  }
}

// SWAP: decode-sized M, the weights are the A operand (128 rows of W per
// tile) and the tokens are N.  LOCALT (swap only): every piece computes its
// own share of T = x.A^T and applies it; otherwise T is computed once per
// T tile in the down section and read back by TMA.
// STATS: the statistics epilogue of the verifier's logit rows (rank 0 only).
template <int BNMAX, bool SWAP, bool LOCALT, bool STATS>
__global__ void __launch_bounds__(kThreads, 1)
grouped_lora_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Params Pk) {
  static_assert(SWAP || !LOCALT, "per-piece adapter needs the swapped operands");
  static_assert(!(STATS && LOCALT), "the statistics epilogue has no adapter");
  constexpr int STAGES = stages_for<BNMAX, LOCALT>();
  constexpr uint32_t kStage = stage_bytes<BNMAX, LOCALT>();  // A sub-tile, B slot, (LOCALT) down slice
  constexpr uint32_t kBSlot = uint32_t(BNMAX) * kBK * 2;
  constexpr uint32_t kTmemCols = tmem_cols<BNMAX, LOCALT>();
  constexpr int kAcc = acc_bufs<BNMAX, LOCALT>();
  constexpr size_t kSlot = size_t(BNMAX) * kBM;  // floats of one partial slot
  // Decode-sized tiles: a finisher sums its contributors' partials while its
  // own last piece is still in the tensor cores.
  constexpr bool kPreMerge = pre_merge<BNMAX>();
  constexpr int kSlots = staging_slots<BNMAX, LOCALT>();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* tprime = smem + STAGES * kStage;  // [2][BNMAX][128 B] (LOCALT)
  float* staging = reinterpret_cast<float*>(tprime + tprime_bytes<BNMAX, LOCALT>());
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(staging) +
                                               staging_bytes<BNMAX, LOCALT>());
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2] y accumulator ready
  uint64_t* tempty = tfull + 2;      // [2] y accumulator drained
  uint64_t* mma_done = tempty + 2;
  uint64_t* stg_bar = mma_done + 1;  // staging area filled
  uint64_t* t_ready = stg_bar + 1;   // (LOCALT) the piece's T accumulator is complete
  uint64_t* t_smem = t_ready + 1;    // (LOCALT) T' is in shared memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_smem + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // The schedule is read with run-time indices all through the kernel: keep a
  // copy in shared memory rather than in the (small) constant cache.
  Params* sp = reinterpret_cast<Params*>(reinterpret_cast<uint8_t*>(full) + kBarrierBytes);
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&Pk);
    uint32_t* dst = reinterpret_cast<uint32_t*>(sp);
    for (uint32_t i = threadIdx.x; i < sizeof(Params) / 4; i += kThreads) dst[i] = src[i];
  }
  const Params& P = *sp;
  uint8_t* gate_s = reinterpret_cast<uint8_t*>(sp) + kParamsBytes;  // [problem][token] (swap)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  static_assert((2 * STAGES + 8) * 8 + 16 <= kBarrierBytes, "barrier area");
  static_assert(smem_bytes_for<BNMAX, LOCALT>() <= 227 * 1024, "shared memory per CTA");
  // one CTA per SM: the schedule's waits rely on it (see launch_grouped)
  static_assert(smem_bytes_for<BNMAX, LOCALT>() > 114 * 1024, "more than half an SM's shared memory");
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
    ptx::mbar_init(stg_bar, 1);
    ptx::mbar_init(t_ready, 1);
    ptx::mbar_init(t_smem, kEpiThreads / 32);
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
  const uint32_t tmem_t = tmem + uint32_t(kAcc * BNMAX);  // (LOCALT) T accumulator
  if (threadIdx.x == 0) ptx::grid_launch_dependents();

  if (threadIdx.x == 0) {
    // Before the previous launch has finished: L2 prefetch hints for the
    // weight tiles of this CTA's first K-blocks.
    int left = kPrefetchKBlocks;
    PieceIter pit(P, cta);
    Seg g;
    while (left > 0 && pit.next(P, cta, g)) {
      {
        const Phase& f = P.ph[g.ph];
        const CUtensorMap* mp = maps.m[f.prob];
        int ta, tb;
        tile_coords(f, g.tile, ta, tb);
        for (int64_t i = 0; i < g.e - g.s && left > 0; ++i, --left) {
          const int kl = int(piece_kb(g, f.na, i) - g.tstart);
          if (f.down)
            ptx::tma_prefetch_l2_2d(&mp[MAP_A], kl * kBK, SWAP ? ta * kBM : tb * f.bn);
          else if (kl >= f.na)
            ptx::tma_prefetch_l2_2d(&mp[MAP_W], (kl - f.na) * kBK, SWAP ? ta * kBM : tb * f.bn);
        }
      }
    }
  }
  if (SWAP && !LOCALT && P.tsplit && cta < P.tchunks && threadIdx.x == 64) {
    // the same hints for the split-K adapter's chunk (down matrix and tokens)
    int p = 0;
    while (P.tch0[p + 1] <= cta) ++p;
    const CUtensorMap* mp = maps.m[p];
    const int kb0 = (cta - P.tch0[p]) * P.tkpc;
    const int kb1 = min((P.pb[p].d_in + kBK - 1) / kBK, kb0 + P.tkpc);
    for (int kb = kb0; kb < kb1; ++kb) {
      for (int t = 0; t * kBM < P.pb[p].r; ++t) ptx::tma_prefetch_l2_2d(&mp[MAP_A], kb * kBK, t * kBM);
      ptx::tma_prefetch_l2_2d(&mp[MAP_X], kb * kBK, 0);
    }
  }
  // Everything below may read what the previous launch wrote.
  ptx::grid_dependency_wait();

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------------------ producers
      // Two threads in two warps share the ring: warp 0 fills the even
      // stages, warp 6 the odd ones (one issuing thread sustains only so
      // many copies in flight).
      const uint32_t mine = warp == 0 ? 0u : 1u;
      // swap: A = weights (streamed once), B = tokens (reused by every tile);
      // otherwise A = tokens, B = weights, both reused across tiles from L2.
      const uint64_t polA = SWAP ? ptx::policy_evict_first() : ptx::policy_evict_last();
      const uint64_t polB = ptx::policy_evict_last();
      uint32_t it = 0;
      PieceIter pit(P, cta);
      Seg g;
      while (!*abort_flag && pit.next(P, cta, g)) {
        {
          const Phase& f = P.ph[g.ph];
          const Prob& pb = P.pb[f.prob];
          const CUtensorMap* mp = maps.m[f.prob];
          int ta, tb;
        tile_coords(f, g.tile, ta, tb);
          // LOCALT: base K-blocks carry the down slice; then the piece's
          // adapter K-blocks bring the up-projection's rows (A operand only)
          const int64_t n = (g.e - g.s) + (LOCALT ? f.nad : 0);
          bool t_ready_flag = false;
          for (int64_t i = 0; i < n; ++i, ++it) {
            const bool local_ad = LOCALT && i >= g.e - g.s;
            const int kl = local_ad ? 0 : int(piece_kb(g, f.na, i) - g.tstart);
            const bool adapter = !LOCALT && kl < f.na;
            if ((it & 1u) != mine) continue;  // the other producer's stage
            const int s = int(it % STAGES);
            if (it >= STAGES && !ptx::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, kWaitLimitNs)) {
              *abort_flag = 1;
              break;
            }
            uint8_t* sa = smem + s * kStage;
            if (local_ad) {
              const int j = int(i - (g.e - g.s));
              ptx::mbar_arrive_expect_tx(&full[s], kABytes);
              ptx::tma_load_2d(sa, &mp[MAP_B], &full[s], j * kBK, ta * kBM, polB);
              continue;
            }
            const CUtensorMap *ma, *mb;
            int kc;
            if (f.down) {
              ma = &mp[SWAP ? MAP_A : MAP_X];
              mb = &mp[SWAP ? MAP_X : MAP_A];
              kc = kl * kBK;
            } else if (!adapter) {
              ma = &mp[SWAP ? MAP_W : MAP_X];
              mb = &mp[SWAP ? MAP_X : MAP_W];
              kc = (kl - f.na) * kBK;
            } else {
              ma = &mp[SWAP ? MAP_B : MAP_T];
              mb = &mp[SWAP ? MAP_T : MAP_B];
              kc = kl * kBK;
            }
            const bool down_slice = LOCALT && pb.r > 0;
            ptx::mbar_arrive_expect_tx(
                &full[s], kABytes + uint32_t(f.bn) * kBK * 2 + (down_slice ? kABytes : 0u));
            // an adapter K-block's weight tile (the up-projection rows) goes out first
            if (adapter) ptx::tma_load_2d(SWAP ? sa : sa + kABytes, SWAP ? ma : mb, &full[s], kc,
                                          SWAP ? ta * kBM : tb * f.bn, SWAP ? polA : polB);
            if (adapter && !t_ready_flag) {
              // The rows of T this tile reads must be complete before TMA reads
              // them.  Should the wait give up, T is loaded all the same (the
              // stage must complete before the CTA may exit) and the launch aborts.
              bool ok = true;
              if (SWAP && P.tsplit) {
                ok = wait_count(P.tflag + pb.tflag0 + 1, P.tch0[f.prob + 1] - P.tch0[f.prob],
                                kWaitLimitNs);
              } else if (SWAP) {
                for (int j = 0; j < pb.ttiles && ok; ++j)
                  ok = wait_flag(P.tflag + pb.tflag0 + j, kWaitLimitNs);
              } else {
                int c0t, np;
                t_tile_span(P, f.prob, ta, c0t, np);
                ok = wait_count(P.tflag + pb.tflag0 + ta, np, kWaitLimitNs);
              }
              if (!ok) *abort_flag = 1;
              fence_proxy_async();
              t_ready_flag = true;
            }
            if (!adapter || !SWAP) ptx::tma_load_2d(sa, ma, &full[s], kc, ta * kBM, polA);
            if (!adapter || SWAP) ptx::tma_load_2d(sa + kABytes, mb, &full[s], kc, tb * f.bn, polB);
            if (*abort_flag) {
              ++it;  // this stage's copies are in flight: the exit path waits for them
              break;
            }
            if (down_slice) ptx::tma_load_2d(sa + kABytes + kBSlot, &mp[MAP_A], &full[s], kc, 0, polB);
          }
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA can exit
        const uint32_t first = it > uint32_t(STAGES) ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i)
          if ((i & 1u) == mine) ptx::mbar_wait(&full[i % STAGES], (i / STAGES) & 1, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      uint32_t it = 0, tcount = 0;
      int seg = 0;
      PieceIter pit(P, cta);
      Seg g;
      for (; !*abort_flag && pit.next(P, cta, g); ++seg) {
        {
          const Phase& f = P.ph[g.ph];
          const Prob& pb = P.pb[f.prob];
          const int acc = seg % kAcc, use = seg / kAcc;
          if (seg >= kAcc && !ptx::mbar_wait(&tempty[acc], (use - 1) & 1, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem + uint32_t(acc * BNMAX);
          const uint32_t idesc = ptx::idesc_bf16_f32(kBM, f.bn);
          const bool local_t = LOCALT && pb.r > 0;
          const int64_t nb = g.e - g.s;
          bool ok = true;
          for (int64_t i = 0; i < nb; ++i, ++it) {
            const int s = int(it % STAGES);
            if (!ptx::mbar_wait(&full[s], (it / STAGES) & 1, kWaitLimitNs)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = ptx::smem_u32(smem + s * kStage);
            const uint32_t sb = sa + kABytes;
#pragma unroll
            for (int u = 0; u < kBK / kUmmaK; ++u)
              ptx::umma_f16(d, ptx::sw128_kmajor_desc(sa + u * 32), ptx::sw128_kmajor_desc(sb + u * 32),
                            idesc, (i > 0 || u > 0) ? 1u : 0u);
            if (local_t) {
              // this piece's share of T: down slice x tokens, into its own accumulator
#pragma unroll
              for (int u = 0; u < kBK / kUmmaK; ++u)
                ptx::umma_f16(tmem_t, ptx::sw128_kmajor_desc(sb + kBSlot + u * 32),
                              ptx::sw128_kmajor_desc(sb + u * 32), idesc, (i > 0 || u > 0) ? 1u : 0u);
            }
            ptx::umma_commit(&empty[s]);
          }
          if (ok && local_t) {
            // T' = bf16(gate * scale * T) comes back through shared memory;
            // then y += (up-projection rows) . T'^T
            ptx::umma_commit(t_ready);
            if (!ptx::mbar_wait(t_smem, tcount & 1, kWaitLimitNs)) ok = false;
            ++tcount;
            ptx::tc_fence_after();
            const uint32_t st = ptx::smem_u32(tprime);
            for (int j = 0; j < f.nad && ok; ++j, ++it) {
              const int s = int(it % STAGES);
              if (!ptx::mbar_wait(&full[s], (it / STAGES) & 1, kWaitLimitNs)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              const uint32_t sa = ptx::smem_u32(smem + s * kStage);
              const uint32_t tb = st + uint32_t(j) * uint32_t(BNMAX) * 128u;
#pragma unroll
              for (int u = 0; u < kBK / kUmmaK; ++u)
                ptx::umma_f16(d, ptx::sw128_kmajor_desc(sa + u * 32), ptx::sw128_kmajor_desc(tb + u * 32),
                              idesc, 1u);
              ptx::umma_commit(&empty[s]);
            }
          }
          if (!ok) {
            *abort_flag = 1;
            break;
          }
          ptx::umma_commit(&tfull[acc]);
        }
      }
      // once this arrives, every MMA issued by this thread has completed
      ptx::umma_commit(mma_done);
      ptx::mbar_wait(mma_done, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 64;
    uint32_t stg_phase = 0;  // phases of stg_bar used so far
    uint32_t tcount = 0;     // (swap) T drains so far
    // (STATS, decode order) the drafted token of every row, and the shared
    // area of the cross-warp reduction, in place of the gates
    int* xd_s = reinterpret_cast<int*>(gate_s);
    float2* st_red = reinterpret_cast<float2*>(gate_s + kSwapMaxRows * 4);
    if (SWAP && !STATS) {
      // the gates, read where they are needed, are one shared-memory load away
      // (a problem without an adapter reads none: its gate may be absent)
      for (int p = 0; p < P.nprob; ++p)
        for (int m = et; m < P.M; m += kEpiThreads)
          gate_s[p * int(kSwapMaxRows) + m] = P.pb[p].r > 0 ? P.pb[p].gate[m] : uint8_t(0);
      epi_sync();
      if constexpr (kPreMerge && !LOCALT) {
        if (P.tsplit && cta < P.tchunks &&
            !tsplit_run(P, maps, cta, et, gate_s, reinterpret_cast<float4*>(gate_s + kGateOnlyBytes),
                        reinterpret_cast<uint8_t*>(staging), staging_bytes<BNMAX, LOCALT>(), stg_bar,
                        stg_phase))
          *abort_flag = 1;
      }
    }
    if (SWAP && STATS) {
      for (int m = et; m < P.M; m += kEpiThreads) xd_s[m] = row_draft_token(P.pb[0], m);
      epi_sync();
    }
    int seg = 0;
    PieceIter pit(P, cta);
    Seg g;
    for (; pit.next(P, cta, g); ++seg) {
      const int sec = g.sec;
      {
        const Phase& f = P.ph[g.ph];
        const Prob& pb = P.pb[f.prob];
        int ta, tb;
        tile_coords(f, g.tile, ta, tb);
        const int acc = seg % kAcc, use = seg / kAcc;
        const bool whole = g.s == g.tstart && g.e == g.tend;
        // a piece of a split T tile in token-rows order (see below)
        const bool tslice = !SWAP && P.tslice && f.down && !whole;
        const bool finisher = !whole && !tslice && g.s == g.tstart;
        const int c1 = finisher ? owner_of(P, sec, g.tend - 1) : cta;
        bool fail = false;
        // The tile's final values leave through emit (16 columns at a time, in
        // column order) and emit_end (after its last columns).
        vfy::MS sacc{-INFINITY, 0.f};
        const int m_row = ta * kBM + row;  // (large-M order) this thread's token row
        const int xd_row = (STATS && !SWAP && m_row < P.M) ? row_draft_token(pb, m_row) : -1;
        float dummy_gather;
        auto emit = [&](int c0, const float (&v)[16]) {
          if constexpr (STATS) {
            if (pb.st_store) store16(P, f, pb, ta, tb, row, c0, v, gate_s);
            if constexpr (SWAP) {
              stats16_swap(P, f, pb, ta, tb, row, c0, v, xd_s, st_red, et);
            } else {
              stats16_rows(f, pb, tb, c0, v, xd_row, m_row < P.M,
                           m_row < P.M ? pb.st_gather + m_row : &dummy_gather, sacc);
            }
          } else {
            store16(P, f, pb, ta, tb, row, c0, v, gate_s);
          }
        };
        auto emit_end = [&]() {
          if constexpr (STATS && !SWAP) {
            if (m_row < P.M) pb.st_part[int64_t(m_row) * pb.st_nvt + tb] = make_float2(sacc.m, sacc.s);
          }
        };
        if (LOCALT && pb.r > 0) {
          // The piece's T (lane = rank, column = token) becomes T' =
          // bf16(gate * scale * T) in shared memory, K-major with the 128-byte
          // swizzle, as the B operand of the up-projection.
          if (!ptx::mbar_wait(t_ready, tcount & 1, kWaitLimitNs)) fail = true;
          ++tcount;
          if (epi_sync_or(fail || *abort_flag)) {
            *abort_flag = 1;
            goto done;
          }
          ptx::tc_fence_after();
          if (row < f.nad * kBK) {
            const uint32_t tq = tmem_t + (uint32_t(q * 32) << 16);
            uint8_t* tk = tprime + (row >> 6) * (BNMAX * 128);
            const int jj = row & 63;
            for (int c0 = 0; c0 < f.bn; c0 += 16) {
              float v[16];
              tmem_ld16f(tq + c0, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int m = c0 + j;
                const float gs = m < P.M ? float(gate_s[f.prob * int(kSwapMaxRows) + m]) * pb.scale : 0.f;
                const __nv_bfloat16 h = __float2bfloat16_rn(v[j] * gs);
                *reinterpret_cast<__nv_bfloat16*>(tk + m * 128 + ((((jj >> 3) ^ (m & 7))) << 4) +
                                                  (jj & 7) * 2) = h;
              }
            }
          }
          // generic-proxy stores, read next by the tensor cores
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(t_smem);
        }
        // A wide tile's finisher in its CTA's last piece merges through the
        // ring, which is idle once the piece's MMAs are done (no piece
        // follows it).  Decode-width finishers fetch their partials into the
        // staging area instead, while their own accumulator is still being
        // filled: that overlap measured faster, for T tiles too, than one
        // round through the ring after it.
        const bool last_piece = sec == kMain || P.lo[kMain][cta] == P.lo[kMain][cta + 1];
        const bool ring = finisher && last_piece && !kPreMerge;
        float pre[kPreMerge ? BNMAX : 1];
        if (ring) {
          if (et == 0) fail = !wait_ready(P, sec, cta + 1, c1, kWaitLimitNs);
        } else if (finisher) {
          if constexpr (kPreMerge) {
            // While the tensor cores finish this piece, bring the contributors'
            // partials into shared memory (one bulk copy each) and sum them in
            // CTA order.
            const uint32_t bytes = uint32_t(f.bn) * kBM * 4;
            bool any = false;
            int c = cta + 1;
            while (c <= c1) {
              int nb = 0, cs = c;
              for (; cs <= c1 && nb < kSlots; ++cs) nb += P.lo[sec][cs] < P.lo[sec][cs + 1];
              if (nb == 0) break;
              if (et == 0) {
                // first batch: wait for every contributor at once (they finish together)
                if (c == cta + 1) fail = !wait_ready(P, sec, cta + 1, c1, kWaitLimitNs);
                fence_proxy_async();
                ptx::mbar_arrive_expect_tx(stg_bar, fail ? 0u : bytes * uint32_t(nb));
                int i = 0;
                for (int cc = c; cc < cs && !fail; ++cc) {
                  if (P.lo[sec][cc] == P.lo[sec][cc + 1]) continue;
                  ptx::bulk_load(staging + size_t(i) * BNMAX * kBM,
                                 P.partial + (size_t(cc) * 2 + sec) * kSlot, bytes, stg_bar);
                  ++i;
                }
              }
              if (!ptx::mbar_wait(stg_bar, stg_phase & 1, kWaitLimitNs)) fail = true;
              ++stg_phase;
              if (!fail) {
                const float4* st4 = reinterpret_cast<const float4*>(staging);
                for (int i = 0; i < nb; ++i) {
#pragma unroll
                  for (int j = 0; j < BNMAX / 4; ++j) {
                    if (4 * j < f.bn) {
                      const float4 t = st4[(size_t(i) * BNMAX / 4 + j) * kBM + row];
                      pre[4 * j] = any ? pre[4 * j] + t.x : t.x;
                      pre[4 * j + 1] = any ? pre[4 * j + 1] + t.y : t.y;
                      pre[4 * j + 2] = any ? pre[4 * j + 2] + t.z : t.z;
                      pre[4 * j + 3] = any ? pre[4 * j + 3] + t.w : t.w;
                    }
                  }
                  any = true;
                }
              }
              // every thread is done with the slots before they are refilled
              fail = epi_sync_or(fail);
              if (fail) break;
              c = cs;
            }
            if (!any) {
#pragma unroll
              for (int j = 0; j < (kPreMerge ? BNMAX : 1); ++j) pre[j] = 0.f;
            }
          } else {
            // The contributors left their pieces as the first piece of their
            // ranges; their flags are normally up long before this point.
            fail = !wait_ready(P, sec, cta + 1, c1, kWaitLimitNs);
          }
        }
        if (!ptx::mbar_wait(&tfull[acc], use & 1, kWaitLimitNs)) fail = true;
        if (epi_sync_or(fail || *abort_flag)) {
          *abort_flag = 1;
          goto done;
        }
        ptx::tc_fence_after();
        {
          const uint32_t tq = tmem + uint32_t(acc * BNMAX) + (uint32_t(q * 32) << 16);
          if (whole) {
            for (int c0 = 0; c0 < f.bn; c0 += 16) {
              float v[16];
              tmem_ld16f(tq + c0, v);
              emit(c0, v);
            }
            emit_end();
          } else if (tslice) {
            // Split T tile (token-rows order): every piece leaves its partial
            // and counts in; once all np pieces are in, piece i sums slice i of
            // the tile (8-column units) over the pieces in CTA order -- the
            // order in which one finisher would add them -- and stores it as
            // T' = bf16(gate * scale * T).  The merge and the publication are
            // spread over the pieces; consumers wait for np slices.
            int c0t, np;
            t_tile_span(P, f.prob, ta, c0t, np);
            float4* dst = reinterpret_cast<float4*>(P.partial + (size_t(cta) * 2 + sec) * kSlot);
            for (int c0 = 0; c0 < f.bn; c0 += 16) {
              float v[16];
              tmem_ld16f(tq + c0, v);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                __stcg(dst + ((c0 >> 2) + i) * kBM + row,
                       make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
            }
            // the accumulator is free for the CTA's next piece at once
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
            epi_sync();
            int* cnt = P.tcnt + pb.tflag0 + ta;
            bool ok = true;
            if (et == 0) {
              fence_acq_rel_gpu();
              red_add_relaxed(cnt, 1);
              ok = wait_count(cnt, np, kWaitLimitNs);
            }
            // thread 0's acquire, then the barrier, order the loads below
            // after every piece's partial
            if (epi_sync_or(!ok)) {
              *abort_flag = 1;
              goto done;
            }
            const int nu = pb.r >> 3;
            const int pi = cta - c0t;
            const int u0 = pi * nu / np, u1 = (pi + 1) * nu / np;
            const int m = ta * kBM + row;
            const float gs = m < P.M ? float(pb.gate[m]) * pb.scale : 0.f;
            for (int u = u0; u < u1; ++u) {
              float sum[8];
              for (int k0 = 0; k0 < np; k0 += 4) {
                float4 t[4][2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float4* src = reinterpret_cast<const float4*>(
                      P.partial + (size_t(c0t + (k0 + k < np ? k0 + k : 0)) * 2 + sec) * kSlot);
                  t[k][0] = __ldcg(src + (2 * u) * kBM + row);
                  t[k][1] = __ldcg(src + (2 * u + 1) * kBM + row);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  if (k0 + k >= np) break;
                  const float x[8] = {t[k][0].x, t[k][0].y, t[k][0].z, t[k][0].w,
                                      t[k][1].x, t[k][1].y, t[k][1].z, t[k][1].w};
#pragma unroll
                  for (int j = 0; j < 8; ++j) sum[j] = (k0 + k == 0) ? x[j] : sum[j] + x[j];
                }
              }
              if (m < P.M) {
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  __nv_bfloat162 h = __floats2bfloat162_rn(sum[2 * j] * gs, sum[2 * j + 1] * gs);
                  w[j] = *reinterpret_cast<uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(pb.t) + int64_t(m) * pb.r + 8 * u) =
                    make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
            // T' is read next by TMA in other CTAs: async-proxy fence, then
            // the release of this slice
            fence_proxy_async();
            epi_sync();
            if (et == 0) {
              fence_acq_rel_gpu();
              red_add_relaxed(P.tflag + pb.tflag0 + ta, 1);
            }
          } else if (!finisher) {
            // contributor: leave the piece as a partial and raise this CTA's flag
            float4* dst = reinterpret_cast<float4*>(P.partial + (size_t(cta) * 2 + sec) * kSlot);
            for (int c0 = 0; c0 < f.bn; c0 += 16) {
              float v[16];
              tmem_ld16f(tq + c0, v);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                __stcg(dst + ((c0 >> 2) + i) * kBM + row,
                       make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
            }
          } else if (ring) {
            // The CTA's MMAs are done and its producers finished, so the idle
            // ring stages a column slice of as many contributors' partials as
            // it holds per round (bulk copies), summed in CTA order after the
            // CTA's own accumulator.
            constexpr uint32_t kRing = uint32_t(STAGES) * kStage;
            int nc = 0;
            for (int c = cta + 1; c <= c1; ++c) nc += P.lo[sec][c] < P.lo[sec][c + 1];
            int wcols = f.bn;
            while (wcols > 16 && uint32_t(nc) * uint32_t(wcols) * kBM * 4 > kRing) wcols >>= 1;
            // contributors per round: all of them unless the slice is 16 wide
            const int cap = int(kRing / (uint32_t(wcols) * kBM * 4));
            float* ringf = reinterpret_cast<float*>(smem);
            const float4* ring4 = reinterpret_cast<const float4*>(smem);
            for (int cw = 0; cw < f.bn; cw += wcols) {
              float v[16];
              for (int b0 = 0; b0 == 0 || b0 < nc; b0 += cap) {
                const int nb = std::min(cap, nc - b0);
                if (nb > 0) {
                  if (et == 0) {
                    fence_proxy_async();
                    ptx::mbar_arrive_expect_tx(stg_bar, uint32_t(nb) * uint32_t(wcols) * kBM * 4);
                    int i = 0, k = 0;
                    for (int c = cta + 1; c <= c1 && i < nb; ++c) {
                      if (P.lo[sec][c] == P.lo[sec][c + 1]) continue;
                      if (k++ < b0) continue;
                      ptx::bulk_load(ringf + size_t(i) * wcols * kBM,
                                     P.partial + (size_t(c) * 2 + sec) * kSlot + size_t(cw) * kBM,
                                     uint32_t(wcols) * kBM * 4, stg_bar);
                      ++i;
                    }
                  }
                  const bool bad = !ptx::mbar_wait(stg_bar, stg_phase & 1, kWaitLimitNs);
                  ++stg_phase;
                  if (epi_sync_or(bad)) {
                    *abort_flag = 1;
                    goto done;
                  }
                }
                for (int c0 = cw; c0 < cw + wcols; c0 += 16) {
                  if (b0 == 0) tmem_ld16f(tq + c0, v);
                  for (int i = 0; i < nb; ++i) {
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                      const float4 t = ring4[(size_t(i) * wcols / 4 + (c0 - cw) / 4 + j4) * kBM + row];
                      v[4 * j4] += t.x;
                      v[4 * j4 + 1] += t.y;
                      v[4 * j4 + 2] += t.z;
                      v[4 * j4 + 3] += t.w;
                    }
                  }
                  if (b0 + nb >= nc) emit(c0, v);
                }
                if (nb > 0) epi_sync();  // the ring is refilled only once every thread has read it
              }
            }
            emit_end();
          } else if constexpr (kPreMerge) {
#pragma unroll
            for (int c0 = 0; c0 < BNMAX; c0 += 16) {
              if (c0 < f.bn) {
                float v[16];
                tmem_ld16f(tq + c0, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += pre[c0 + j];
                emit(c0, v);
              }
            }
            emit_end();
          } else {
            // finisher of a wide tile: own accumulator, then the partials of
            // up to four contributors at a time, in CTA order
            for (int c0 = 0; c0 < f.bn; c0 += 16) {
              float v[16];
              tmem_ld16f(tq + c0, v);
              for (int cb = cta + 1; cb <= c1; cb += 4) {
                float4 t[4][4];
                bool use4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int c = cb + u;
                  use4[u] = c <= c1 && P.lo[sec][c] < P.lo[sec][c + 1];
                  const float4* src = reinterpret_cast<const float4*>(
                      P.partial + (size_t(use4[u] ? c : cta) * 2 + sec) * kSlot);
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    t[u][i] = use4[u] ? __ldcg(src + ((c0 >> 2) + i) * kBM + row)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  if (use4[u]) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                      v[4 * i] += t[u][i].x;
                      v[4 * i + 1] += t[u][i].y;
                      v[4 * i + 2] += t[u][i].z;
                      v[4 * i + 3] += t[u][i].w;
                    }
                  }
              }
              emit(c0, v);
            }
            emit_end();
          }
          if (!tslice) {
            // the accumulator may be reused
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
          }
          // A partial (read by the finisher's bulk copies) or a finished T tile
          // (read by TMA in other CTAs) is published with a release: every
          // thread orders its stores before the async proxy, the barrier
          // orders them before thread 0, whose fence and flag store release them.
          const bool publish_partial = !whole && !finisher && !tslice;
          const bool publish_t = f.down && (whole || finisher);
          if (publish_partial || publish_t) {
            fence_proxy_async();
            epi_sync();
            if (et == 0) {
              fence_acq_rel_gpu();
              st_release(publish_partial ? P.ready + sec * P.grid + cta : P.tflag + pb.tflag0 + ta, 1);
            }
          }
        }
      }
    }
  done:;
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicOr(&g_device_error, 1);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- pair order
// Large M with at least a wave of tiles: tiles of 256 tokens x bn outputs
// (y: bn = 256; T: bn = the rank) in data-parallel waves, each computed by a
// cluster of two CTAs with the pair MMA (M = 256).  CTA r of the pair loads
// the tile's token rows [128 r, 128 r + 128) and its output rows
// [r bn/2, (r + 1) bn/2) with plain TMA, every copy completing on the even
// (leader) CTA's barrier; the leader's MMA thread multiplies both CTAs'
// halves and its commits arrive on both CTAs' barriers; each CTA's TMEM
// receives the accumulator rows of its own tokens, which its epilogue warps
// store as in the token-rows order.  Per CTA and K-block 32 KB cross from L2
// to shared memory instead of 48 KB for a 128 x 256 tile.  Tiles are dealt
// t = pair, pair + pairs, ...; T tiles come first, so a y tile's adapter
// K-blocks (the last of its K order) only wait for tiles that never wait.
constexpr int kPairStages = 6;
constexpr uint32_t kPairStage = 2 * kABytes;  // token half + output half (at most 128 rows)
constexpr uint32_t kPairSmem = kPairStages * kPairStage + kBarrierBytes + kParamsBytes + 1024;
constexpr uint32_t kPairTmemCols = 512;  // two 256-column accumulators

// STATS: the statistics epilogue of the verifier's logit rows (rank 0 only),
// as in the CTA-per-tile order.
template <bool STATS>
__global__ void __launch_bounds__(kThreads, 1)
pair_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Params Pk) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStage);
  uint64_t* empty = full + kPairStages;
  uint64_t* tfull = empty + kPairStages;  // [2] accumulator ready (both CTAs)
  uint64_t* tempty = tfull + 2;           // [2] accumulator drained (leader: both CTAs' warps)
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  Params* sp = reinterpret_cast<Params*>(reinterpret_cast<uint8_t*>(full) + kBarrierBytes);
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&Pk);
    uint32_t* dst = reinterpret_cast<uint32_t*>(sp);
    for (uint32_t i = threadIdx.x; i < sizeof(Params) / 4; i += kThreads) dst[i] = src[i];
  }
  const Params& P = *sp;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  static_assert((2 * kPairStages + 6) * 8 + 16 <= kBarrierBytes, "barrier area");
  static_assert(kPairSmem <= 227 * 1024 && kPairSmem > 114 * 1024, "one CTA per SM");

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 2 * (kEpiThreads / 32));
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, kPairTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other's
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();

  // Tile t of the data-parallel list: phase, token-tile pair and output tile.
  auto tile_of = [&](int t, int& ph, int& ta2, int& tb) {
    int p = P.dp0;
    while (p + 1 < P.dp1 && P.ph[p + 1].tbase <= t) ++p;
    ph = p;
    tile_coords(P.ph[p], P.ph[p].tile0 + (t - P.ph[p].tbase), ta2, tb);
  };

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------------------ producers
      const uint32_t mine = warp == 0 ? 0u : 1u;
      const uint64_t pol = ptx::policy_evict_last();
      uint32_t it = 0;
      for (int t = pair; !*abort_flag && t < P.dp_tiles; t += npairs) {
        int ph, ta2, tb;
        tile_of(t, ph, ta2, tb);
        const Phase& f = P.ph[ph];
        const Prob& pb = P.pb[f.prob];
        const CUtensorMap* mp = maps.m[f.prob];
        const int nb = f.nkb - f.na;  // base K-blocks, then the adapter's
        const uint32_t bytes = 2u * (kABytes + uint32_t(f.bn / 2) * kBK * 2u);
        const int tok = ta2 * 2 * kBM + int(rank) * kBM;
        const int outr = f.n0 + tb * f.bn + int(rank) * (f.bn / 2);
        const bool narrow = !f.down && f.bn == 128;  // 64-row boxes
        bool t_ok = false;
        for (int i = 0; i < f.nkb; ++i, ++it) {
          if ((it & 1u) != mine) continue;
          const int s = int(it % kPairStages);
          if (it >= uint32_t(kPairStages) &&
              !ptx::mbar_wait(&empty[s], ((it / kPairStages) - 1) & 1, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          const bool adapter = !f.down && i >= nb;
          const int kc = (adapter ? i - nb : i) * kBK;
          if (adapter && !t_ok) {
            // both halves of the T tile of these 256 tokens are written
            if (!wait_count(P.tflag + pb.tflag0 + ta2, 2, kWaitLimitNs)) *abort_flag = 1;
            fence_proxy_async();
            t_ok = true;
          }
          uint8_t* sa = smem + s * kPairStage;
          const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&full[s]), 0);
          if (leader) ptx::mbar_arrive_expect_tx(&full[s], bytes);
          ptx::tma_load_2d_pair(sa, &mp[adapter ? MAP_T : MAP_X], bar, kc, tok, pol);
          ptx::tma_load_2d_pair(sa + kABytes,
                                &mp[f.down ? MAP_A : adapter ? (narrow ? MAP_B2 : MAP_B) : (narrow ? MAP_W2 : MAP_W)],
                                bar, kc, f.down ? int(rank) * (f.bn / 2) : outr, pol);
        }
      }
      // The leader's MMAs have read every stage this thread filled (their
      // commits arrive here): no copy or arrival is left in flight at exit.
      for (uint32_t j = it > uint32_t(kPairStages) ? it - kPairStages : 0; j < it; ++j)
        if ((j & 1u) == mine) ptx::mbar_wait(&empty[j % kPairStages], (j / kPairStages) & 1, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer
      uint32_t it = 0;
      int seg = 0;
      for (int t = pair; !*abort_flag && t < P.dp_tiles; t += npairs, ++seg) {
        int ph, ta2, tb;
        tile_of(t, ph, ta2, tb);
        const Phase& f = P.ph[ph];
        const int acc = seg & 1, use = seg >> 1;
        if (seg >= 2 && !ptx::mbar_wait(&tempty[acc], (use - 1) & 1, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + uint32_t(acc * 256);
        const uint32_t idesc = ptx::idesc_bf16_f32(2 * kBM, f.bn);
        bool ok = true;
        for (int i = 0; i < f.nkb; ++i, ++it) {
          const int s = int(it % kPairStages);
          if (!ptx::mbar_wait(&full[s], (it / kPairStages) & 1, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(smem + s * kPairStage);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int u = 0; u < kBK / kUmmaK; ++u)
            ptx::umma_pair_f16(d, ptx::sw128_kmajor_desc(sa + u * 32), ptx::sw128_kmajor_desc(sb + u * 32),
                               idesc, (i > 0 || u > 0) ? 1u : 0u);
          ptx::umma_pair_commit(&empty[s], 3);
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        ptx::umma_pair_commit(&tfull[acc], 3);
      }
      ptx::umma_pair_commit(mma_done, 1);
      ptx::mbar_wait(mma_done, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 64;
    int seg = 0;
    for (int t = pair; t < P.dp_tiles; t += npairs, ++seg) {
      int ph, ta2, tb;
      tile_of(t, ph, ta2, tb);
      const Phase& f = P.ph[ph];
      const Prob& pb = P.pb[f.prob];
      const int acc = seg & 1, use = seg >> 1;
      const bool fail = !ptx::mbar_wait(&tfull[acc], use & 1, kWaitLimitNs);
      if (epi_sync_or(fail || *abort_flag)) {
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tq = tmem + uint32_t(acc * 256) + (uint32_t(q * 32) << 16);
      const int ta = ta2 * 2 + int(rank);  // this CTA's 128-token tile
      const int m_row = ta * kBM + row;
      if constexpr (STATS) {
        // (max, sum exp) of the row's columns in this vocabulary tile, and the
        // logit of the row's drafted token where the tile holds it
        const int xd_row = m_row < P.M ? row_draft_token(pb, m_row) : -1;
        float dummy_gather;
        vfy::MS sacc{-INFINITY, 0.f};
        for (int c0 = 0; c0 < f.bn; c0 += 16) {
          float v[16];
          tmem_ld16f(tq + c0, v);
          if (pb.st_store) store16(P, f, pb, ta, tb, row, c0, v, nullptr);
          stats16_rows(f, pb, tb, c0, v, xd_row, m_row < P.M,
                       m_row < P.M ? pb.st_gather + m_row : &dummy_gather, sacc);
        }
        if (m_row < P.M) pb.st_part[int64_t(m_row) * pb.st_nvt + tb] = make_float2(sacc.m, sacc.s);
      } else {
        for (int c0 = 0; c0 < f.bn; c0 += 16) {
          float v[16];
          tmem_ld16f(tq + c0, v);
          store16(P, f, pb, ta, tb, row, c0, v, nullptr);
        }
      }
      // the accumulator may be reused: one arrival per warp on the leader's barrier
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&tempty[acc]), 0));
      if (f.down) {
        // this CTA's half of the T tile, read next by TMA in other CTAs
        fence_proxy_async();
        epi_sync();
        if (et == 0) {
          fence_acq_rel_gpu();
          red_add_relaxed(P.tflag + pb.tflag0 + ta2, 1);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // neither CTA leaves while the other may still signal it
  if (*abort_flag && threadIdx.x == 0) atomicOr(&g_device_error, 1);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kPairTmemCols);
  }
}

// Clears the schedule's flags once the previous launch in the stream has
// finished, letting the projection kernel that follows start right away.
// (16-byte aligned, n16 16-byte words)
__global__ void sync_reset_kernel(int4* __restrict__ sync, int n16) {
  if (threadIdx.x == 0) ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  for (int i = threadIdx.x; i < n16; i += blockDim.x) sync[i] = make_int4(0, 0, 0, 0);
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
  int tflags;
  size_t off_t[kMaxLoraProblems];
  size_t off_tpart;  // split-K adapter partials
  size_t off_partial, off_sync, sync_bytes;
  size_t off_cast[kMaxLoraProblems][4];  // fp32 mode: bf16 copies of x, W, A, B
  size_t bytes;
};

// Host-side schedule: the phases of both sections, the grid, each CTA's
// ranges and the workspace layout.  Depends only on shapes and the SM count.
// Clusters of two CTAs that can be resident at once on this device for the
// pair kernel (0 until the first launch has asked the runtime).
std::atomic<int> g_pair_cap{0};

bool make_layout(int n, const uno_lora_problem* pr, int64_t M, int dtype, int sms, Layout& L,
                 bool allow_pair = true, bool no_narrow = false) {
  if (n < 1 || n > kMaxLoraProblems) return false;
  std::memset(&L, 0, sizeof(L));
  Params& P = L.P;
  P.M = int(M);
  // Decode-sized M swaps the operands (weights fill the 128-row MMA side)
  // and computes the adapter input T by split K in the epilogue warps, which
  // leaves the weight stream alone; larger M computes T once per T tile in
  // the down section.  (The per-piece adapter, LOCALT, remains for launches
  // built without the split-K adapter.)
  P.swap = M <= kSwapMaxRows ? 1 : 0;
  int64_t wbytes = 0;
  bool small_rank = true, any_rank = false;
  for (int p = 0; p < n; ++p) {
    wbytes += 2 * pr[p].d_in * pr[p].d_out;
    small_rank = small_rank && pr[p].rank <= kMaxLocalRank;
    any_rank = any_rank || pr[p].rank > 0;
  }
  // (the split-K adapter needs a CTA per adapted problem at least)
  int n_adapted = 0;
  int64_t swap_kb = 0;
  for (int p = 0; p < n; ++p) {
    n_adapted += pr[p].rank > 0;
    swap_kb += ((pr[p].d_out + kBM - 1) / kBM) *
               ((pr[p].rank + kBK - 1) / kBK + (pr[p].d_in + kBK - 1) / kBK);
  }
  const int64_t g_swap = std::max<int64_t>(1, std::min<int64_t>(std::min(sms, kMaxGrid), swap_kb / 4));
  P.tsplit = (kSplitKAdapter && M <= kSplitKMaxRows && any_rank && n_adapted <= g_swap) ? 1 : 0;
  P.localt = (!P.tsplit && P.swap && any_rank && small_rank && wbytes < kLocalTMaxWeightBytes) ? 1 : 0;
  P.out_f32 = dtype == UNO_F32;
  const int bn_tok = pick_bn(M);

  // Pair order (pair_gemm_kernel): token-rows M whose 256-token tiles waste
  // at most a tenth of M in padding rows (the pair MMA computes them: at 384
  // rows gate/up took 117 us against 107 us per CTA), a tile for at least half
  // of the CTA pairs (a partly filled wave still beats stream-K's merges: the
  // down projection at 1024 rows, 68 tiles for 74 pairs, 98 us against 123 us),
  // and every rank a multiple of 32 up to 256.
  if (kPairMma && allow_pair && !P.swap && g_pair_cap.load() >= 0) {
    const int cap = g_pair_cap.load();
    const int pairs = std::min(std::min(sms, kMaxGrid) / 2, cap > 0 ? cap : kMaxGrid);
    const int64_t ta2 = (M + 2 * kBM - 1) / (2 * kBM);
    bool ranks_ok = true;
    int64_t ptiles = 0;
    for (int p = 0; p < n; ++p) {
      ranks_ok = ranks_ok && pr[p].rank % 32 == 0 && pr[p].rank <= 256;
      ptiles += (pr[p].rank > 0 ? ta2 : 0) + ta2 * ((pr[p].d_out + 255) / 256);
    }
    const bool pad_ok = (ta2 * 2 * kBM - M) * 10 <= M;
    if (pairs >= 1 && ranks_ok && pad_ok && 2 * ptiles >= pairs && ptiles < (int64_t(1) << 30) &&
        3 * n <= kMaxPhases) {
      P.pair = 1;
      P.grid = 2 * pairs;
      P.bnmax = 256;
      P.nprob = n;
      int nph = 0, tflags = 0, tbase = 0;
      for (int p = 0; p < n; ++p) {
        Prob& b = P.pb[p];
        b.d_in = int(pr[p].d_in);
        b.d_out = int(pr[p].d_out);
        b.r = int(pr[p].rank);
        b.scale = pr[p].rank > 0 ? pr[p].alpha / float(pr[p].rank) : 0.f;
        b.tflag0 = tflags;
        if (pr[p].rank == 0) continue;
        Phase f{};
        f.prob = p;
        f.down = 1;
        f.nkb = int((pr[p].d_in + kBK - 1) / kBK);
        f.tiles_a = int(ta2);
        f.bn = int(pr[p].rank);
        f.tiles = f.tiles_all = f.tiles_a;
        f.tbase = tbase;
        b.ttiles = f.tiles;
        tflags += f.tiles;
        tbase += f.tiles;
        P.ph[nph++] = f;
      }
      // y tiles 256 wide, except that when the last wave would keep at most
      // half of the pairs busy, trailing 256-column groups (of the last
      // problems first) become 128-wide tiles, dealt after all others, so
      // that they fill the last wave: the count is the one whose simulated
      // makespan (tiles dealt t -> pair t mod pairs; a 128-wide tile costs
      // 3/4 of a 256-wide one per K-block) is least.  Not for the statistics
      // epilogue, whose per-row partials assume one tile width.
      int cols[kMaxLoraProblems];
      int64_t total_cols = 0;
      for (int p = 0; p < n; ++p) total_cols += cols[p] = int((pr[p].d_out + 255) / 256);
      auto split_of = [&](int64_t c, int (&conv)[kMaxLoraProblems]) {
        for (int p = n - 1; p >= 0; --p) {
          conv[p] = int(std::min<int64_t>(c, cols[p]));
          c -= conv[p];
        }
      };
      auto makespan = [&](int64_t c) {
        int conv[kMaxLoraProblems];
        split_of(c, conv);
        std::vector<double> load(size_t(pairs), 0.0);
        int64_t t = 0;
        auto deal = [&](int64_t count, double cost) {
          for (int64_t i = 0; i < count; ++i, ++t) load[size_t(t % pairs)] += cost;
        };
        for (int p = 0; p < n; ++p)
          if (pr[p].rank > 0) deal(ta2, double((pr[p].d_in + kBK - 1) / kBK) * 0.75);
        for (int p = 0; p < n; ++p)
          deal(ta2 * (cols[p] - conv[p]), double((pr[p].rank + kBK - 1) / kBK + (pr[p].d_in + kBK - 1) / kBK));
        for (int p = 0; p < n; ++p)
          if (conv[p] > 0) {
            const int64_t n0 = int64_t(cols[p] - conv[p]) * 256;
            deal(ta2 * ((pr[p].d_out - n0 + 127) / 128),
                 0.75 * double((pr[p].rank + kBK - 1) / kBK + (pr[p].d_in + kBK - 1) / kBK));
          }
        return *std::max_element(load.begin(), load.end());
      };
      int64_t best_c = 0;
      if (!no_narrow && (ptiles % pairs) * 2 <= pairs && ptiles % pairs != 0) {
        double best = makespan(0);
        const int64_t cmax = std::min<int64_t>(total_cols, (pairs + ta2 - 1) / ta2 + 1);
        for (int64_t c = 1; c <= cmax; ++c) {
          const double m = makespan(c);
          if (m < best * 0.999) {
            best = m;
            best_c = c;
          }
        }
      }
      int conv[kMaxLoraProblems];
      split_of(best_c, conv);
      for (int p = 0; p < n; ++p) {
        if (cols[p] - conv[p] == 0) continue;
        Phase f{};
        f.prob = p;
        f.na = int((pr[p].rank + kBK - 1) / kBK);
        f.nkb = f.na + int((pr[p].d_in + kBK - 1) / kBK);
        f.tiles_a = int(ta2);
        f.bn = 256;
        f.tiles = f.tiles_all = int(ta2 * (cols[p] - conv[p]));
        f.tbase = tbase;
        tbase += f.tiles;
        P.ph[nph++] = f;
      }
      for (int p = 0; p < n; ++p) {
        if (conv[p] == 0) continue;
        Phase f{};
        f.prob = p;
        f.na = int((pr[p].rank + kBK - 1) / kBK);
        f.nkb = f.na + int((pr[p].d_in + kBK - 1) / kBK);
        f.tiles_a = int(ta2);
        f.bn = 128;
        f.n0 = (cols[p] - conv[p]) * 256;
        f.tiles = f.tiles_all = int(ta2 * ((pr[p].d_out - f.n0 + 127) / 128));
        f.tbase = tbase;
        tbase += f.tiles;
        P.ph[nph++] = f;
      }
      P.dp0 = 0;
      P.dp1 = nph;
      P.dp_tiles = tbase;
      P.ph0[0] = P.ph1[0] = P.ph0[1] = P.ph1[1] = nph;
      L.tflags = tflags;
      size_t o = 0;
      for (int p = 0; p < n; ++p) {
        L.off_t[p] = o;
        o = align_up(o + size_t(M) * size_t(pr[p].rank) * 2, 256);
      }
      L.off_tpart = L.off_partial = L.off_sync = o;
      L.sync_bytes = align_up((2 * size_t(P.grid) + 2 * size_t(tflags)) * sizeof(int), 256);
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
  }

  // Tile list: the T tiles of every adapted problem (unless each piece makes
  // its own), then the y tiles of every problem.
  Phase tl[2 * kMaxLoraProblems];
  int nt = 0, tflags = 0, bnmax = 16, max_down_nkb = 0;
  int64_t total_kb = 0, tiles_total = 0;
  for (int p = 0; p < n; ++p) {
    Prob& b = P.pb[p];
    b.d_in = int(pr[p].d_in);
    b.d_out = int(pr[p].d_out);
    b.r = int(pr[p].rank);
    b.scale = pr[p].rank > 0 ? pr[p].alpha / float(pr[p].rank) : 0.f;
    b.tflag0 = tflags;
    if (P.tsplit && pr[p].rank > 0) tflags += 2;  // chunks in, slices out
    if (pr[p].rank == 0 || P.localt || P.tsplit) continue;
    Phase f{};
    f.prob = p;
    f.down = 1;
    f.nkb = int((pr[p].d_in + kBK - 1) / kBK);
    // one tile along N: bn covers every token (swap) or the whole rank
    f.tiles_a = int(((P.swap ? pr[p].rank : M) + kBM - 1) / kBM);
    f.bn = P.swap ? bn_tok : pick_bn(pr[p].rank);
    f.tiles = f.tiles_all = f.tiles_a;
    b.ttiles = f.tiles;
    tflags += f.tiles;
    max_down_nkb = std::max(max_down_nkb, f.nkb);
    tl[nt++] = f;
  }
  const int n_down = nt;
  // Large M: 256-wide output tiles, or 128-wide ones when those cost less.
  // The mainloop is bound by operand traffic (a 128 x 64 token tile plus bn
  // rows of weights per K-block), so a launch's cost is counted per CTA in
  // those bytes: whole waves of tiles when there are at least as many tiles
  // as CTAs (data-parallel order); otherwise (stream-K) an even share of all
  // tiles' bytes plus the merge of the split tiles' fp32 partials, weighted
  // four times their bytes (measured: a merge costs L2 round trips, not only
  // bandwidth -- at 256 rows the split launches took 43 us with 128-wide
  // tiles against 68 us with 256-wide ones).
  int bn_large = 256;
  if (!P.swap) {
    auto cost = [&](int bn) {
      double tiles = 0, bytes = 0;
      for (int i = 0; i < n_down; ++i) {
        tiles += tl[i].tiles;
        bytes += double(tl[i].tiles) * tl[i].nkb * (double(kABytes) + tl[i].bn * 128.0);
      }
      for (int p = 0; p < n; ++p) {
        const double t = double((M + kBM - 1) / kBM) * double((pr[p].d_out + bn - 1) / bn);
        tiles += t;
        bytes += t * double((pr[p].rank + kBK - 1) / kBK + (pr[p].d_in + kBK - 1) / kBK) *
                 (double(kABytes) + bn * 128.0);
      }
      const double G0 = double(std::min(sms, kMaxGrid));
      if (tiles >= G0) return std::ceil(tiles / G0) * (bytes / tiles);
      return bytes / G0 + 4.0 * (G0 - tiles) / tiles * (double(kBM) * bn * 4.0);
    };
    if (cost(128) < cost(256)) bn_large = 128;
  }
  for (int p = 0; p < n; ++p) {
    Phase f{};
    f.prob = p;
    f.na = P.localt ? 0 : int((pr[p].rank + kBK - 1) / kBK);
    f.nad = P.localt ? int((pr[p].rank + kBK - 1) / kBK) : 0;
    f.nkb = f.na + int((pr[p].d_in + kBK - 1) / kBK);
    if (P.swap) {
      f.tiles_a = int((pr[p].d_out + kBM - 1) / kBM);
      f.bn = bn_tok;
      f.tiles = f.tiles_a;
    } else {
      f.tiles_a = int((M + kBM - 1) / kBM);
      f.bn = std::min(pick_bn(pr[p].d_out), bn_large);
      f.tiles = f.tiles_a * int((pr[p].d_out + f.bn - 1) / f.bn);
    }
    f.tiles_all = f.tiles;
    tl[nt++] = f;
  }
  for (int i = 0; i < nt; ++i) {
    tl[i].tbase = int(tiles_total);
    tiles_total += tl[i].tiles;
    total_kb += int64_t(tl[i].tiles) * tl[i].nkb;
    bnmax = std::max(bnmax, tl[i].bn);
  }
  P.bnmax = bnmax;
  L.tflags = tflags;
  // One CTA per SM, at least 4 K-blocks each.
  const int G = int(std::max<int64_t>(1, std::min<int64_t>(std::min(sms, kMaxGrid), total_kb / 4)));
  P.grid = G;
  // Split-K adapter: chunks of tkpc K-blocks, no more chunks than CTAs.
  if (P.tsplit) {
    int64_t kbt = 0;
    for (int p = 0; p < n; ++p)
      if (pr[p].rank > 0) kbt += (pr[p].d_in + kBK - 1) / kBK;
    int kpc = int(std::max<int64_t>(1, (kbt + G - 1) / G));
    while (true) {
      int c = 0;
      for (int p = 0; p < n; ++p) {
        P.tch0[p] = c;
        if (pr[p].rank > 0) c += int(((pr[p].d_in + kBK - 1) / kBK + kpc - 1) / kpc);
      }
      P.tch0[n] = c;
      if (c <= G) break;
      ++kpc;
    }
    for (int p = n + 1; p <= kMaxLoraProblems; ++p) P.tch0[p] = P.tch0[n];
    P.tkpc = kpc;
    P.tbn = bn_tok;
    P.tchunks = P.tch0[n];
    int max_rank = 0;
    for (int p = 0; p < n; ++p) max_rank = std::max(max_rank, int(pr[p].rank));
    P.tpart_stride = int64_t(align_up(size_t(M) * size_t(max_rank), 64));
  }

  // Large M: whole tiles in data-parallel waves (tile t to CTA t % G, so the
  // tiles in flight at once share their operands in L2).  Merging a split
  // 128 x 256 tile costs more than the idle part of a last wave, so a launch
  // with at least a wave of tiles splits none; fewer tiles than CTAs, and
  // every decode launch, use stream-K.
  int nph = 0;
  int64_t dp_tiles = 0;
  if (!P.swap) {
    dp_tiles = tiles_total >= G ? tiles_total : 0;
    P.dp0 = nph;
    for (int i = 0; i < nt; ++i) P.ph[nph++] = tl[i];
    P.dp1 = nph;
  }
  P.dp_tiles = int(dp_tiles);
  P.nprob = n;
  // Stream-K sections over the remaining tiles: 0 = T tiles, 1 = y tiles.
  int64_t sec_kb[2] = {0, 0};
  for (int sec = 0; sec < 2; ++sec) {
    P.ph0[sec] = nph;
    for (int i = sec ? n_down : 0; i < (sec ? nt : n_down); ++i) {
      const int64_t first = std::max<int64_t>(tl[i].tbase, dp_tiles);
      const int64_t last = int64_t(tl[i].tbase) + tl[i].tiles;
      if (first >= last) continue;
      Phase f = tl[i];
      f.tile0 = int(first - tl[i].tbase);
      f.tiles = int(last - first);
      f.kb_start = sec_kb[sec];
      sec_kb[sec] += int64_t(f.tiles) * f.nkb;
      P.ph[nph++] = f;
    }
    P.ph1[sec] = nph;
  }
  const int64_t D = sec_kb[kDown], Mn = sec_kb[kMain], Wt = D + Mn;
  // Down section: a few K-blocks per CTA so that T is complete early, but a
  // T tile in no more pieces than its finisher's staging area holds at once
  // (one round of bulk copies); at large M, where T tiles are many and cheap,
  // whole tiles up to half a CTA's share.
  // Token-rows order, split T tiles: merged by slices over their pieces when a
  // CTA's share of K-blocks is short (the pieces' waits and slice sums are
  // then what T waits for), else by one finisher that takes no main work
  // (measured: the down projection at 512 and 1024 rows, 201 and 207 K-blocks
  // a CTA, took 82 and 123 us that way against 88 and 168 us by slices).
  P.tslice = (!P.swap && D > 0 && Wt / G <= kTSliceMaxShare) ? 1 : 0;
  int Gd = 0;
  if (D > 0 && !P.tslice) {
    const int64_t slots =
        bnmax <= 64 ? std::max<int64_t>(1, kSharedTStaging / (int64_t(bnmax) * kBM * 4)) : 16;
    int64_t kd = std::max<int64_t>(4, (max_down_nkb + slots - 1) / slots);
    // a long T tile (down projection of a wide input) may take two rounds:
    // shorter pieces finish T sooner than one more round of copies costs
    if (P.swap && kd > 16) kd = (kd + 1) / 2;
    if (!P.swap) kd = std::max<int64_t>(kd, std::min<int64_t>(max_down_nkb, Wt / G / 2));
    Gd = int(std::max<int64_t>(1, std::min<int64_t>(G, (D + kd - 1) / kd)));
  }
  for (int c = 0; c <= G; ++c) P.lo[kDown][c] = c <= Gd && Gd > 0 ? int64_t(c) * D / Gd : D;
  if (P.tslice) {
    // Token-rows order: every T tile in pieces of about a quarter of a CTA's
    // share of K-blocks (at least 4), one piece per CTA, so that T is
    // complete early; the pieces merge and publish the tile together, each a
    // slice of it, so that more pieces cost no longer merge.
    int64_t kd = std::max<int64_t>(4, (Wt / G + 3) / 4);
    auto pieces = [&](int64_t k) {
      int64_t n_pc = 0;
      for (int p = P.ph0[kDown]; p < P.ph1[kDown]; ++p)
        n_pc += int64_t(P.ph[p].tiles) * ((P.ph[p].nkb + k - 1) / k);
      return n_pc;
    };
    while (pieces(kd) > G) ++kd;
    int c = 0;
    for (int p = P.ph0[kDown]; p < P.ph1[kDown]; ++p) {
      const Phase& f = P.ph[p];
      const int64_t np = (f.nkb + kd - 1) / kd;
      for (int t = 0; t < f.tiles; ++t)
        for (int64_t i = 0; i < np; ++i)
          P.lo[kDown][c++] = f.kb_start + int64_t(t) * f.nkb + i * f.nkb / np;
    }
    for (; c <= G; ++c) P.lo[kDown][c] = D;
  }
  // Main section: CTA c's range ends where the first c+1 CTAs have streamed
  // (c+1)/G of the section's K-blocks, down ones included -- except that a CTA
  // finishing a split T tile alone (it waits for and merges the tile's pieces,
  // then publishes T) takes no main work, which the others share.
  bool t_fin[kMaxGrid + 1] = {};
  int n_fin = 0;
  for (int c = 0; c < G && D > 0 && !P.tslice; ++c) {
    const int64_t lo0 = P.lo[kDown][c], hi0 = P.lo[kDown][c + 1];
    if (lo0 >= hi0) continue;
    // the CTA's last down piece starts a T tile that continues beyond it
    int p = P.ph0[kDown];
    int64_t k = hi0 - 1;
    while (p + 1 < P.ph1[kDown] && P.ph[p + 1].kb_start <= k) ++p;
    const Phase& f = P.ph[p];
    const int64_t ts = f.kb_start + (k - f.kb_start) / f.nkb * f.nkb;
    if (ts >= lo0 && ts + f.nkb > hi0) {
      t_fin[c] = true;
      ++n_fin;
    }
  }
  if (n_fin >= G) n_fin = 0, std::memset(t_fin, 0, sizeof(t_fin));
  P.lo[kMain][0] = 0;
  int64_t share_before = 0;  // weighted CTAs before c
  for (int c = 1; c < G; ++c) {
    share_before += t_fin[c - 1] ? 0 : 1;
    const int64_t v = share_before * Wt / (G - n_fin) - P.lo[kDown][c];
    P.lo[kMain][c] = std::min(Mn, std::max(P.lo[kMain][c - 1], v));
  }
  P.lo[kMain][G] = Mn;
  // A boundary inside a tile's adapter K-blocks (the first na of its flat
  // order) moves back to the tile's start: only the tile's finisher then
  // runs adapter K-blocks, and no contributor's first piece waits for T.
  for (int c = 1; c < G; ++c) {
    const int64_t k = P.lo[kMain][c];
    if (k <= 0 || k >= Mn || t_fin[c]) continue;  // (a T tile's finisher keeps no main work)
    int p = P.ph0[kMain];
    while (p + 1 < P.ph1[kMain] && P.ph[p + 1].kb_start <= k) ++p;
    const Phase& f = P.ph[p];
    const int64_t ts = f.kb_start + (k - f.kb_start) / f.nkb * f.nkb;
    if (k > ts && k < ts + f.na) P.lo[kMain][c] = std::max(P.lo[kMain][c - 1], ts);
  }
  size_t o = 0;
  for (int p = 0; p < n; ++p) {
    L.off_t[p] = o;
    o = align_up(o + size_t(M) * size_t(pr[p].rank) * 2, 256);
  }
  L.off_tpart = o;
  if (P.tsplit) o = align_up(o + size_t(P.tchunks) * size_t(P.tpart_stride) * sizeof(float), 256);
  L.off_partial = o;
  o = align_up(o + size_t(G) * 2 * size_t(bnmax) * kBM * sizeof(float), 256);
  L.off_sync = o;
  L.sync_bytes = align_up((2 * size_t(G) + 2 * size_t(tflags)) * sizeof(int), 256);
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

template <int BNMAX, bool SWAP, bool LOCALT, bool STATS>
cudaError_t launch_grouped(const Maps& maps, const Params& P, cudaStream_t st) {
  static std::once_flag once[64];
  static cudaError_t attr_err[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  dev &= 63;
  std::call_once(once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(grouped_lora_gemm_kernel<BNMAX, SWAP, LOCALT, STATS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem_bytes_for<BNMAX, LOCALT>()));
  });
  if (attr_err[dev] != cudaSuccess) return attr_err[dev];
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(P.grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for<BNMAX, LOCALT>();
  cfg.stream = st;
  // Not a cooperative launch: the grid is at most one CTA per SM (each CTA
  // takes more than half of an SM's shared memory), every wait points at a
  // higher CTA of this grid or at a flag raised without waiting, and a launch
  // chained after this one starts only once all of this grid's CTAs have
  // started (they trigger at entry), so all CTAs become resident without the
  // guarantee -- and the next launch can take each SM as soon as it is freed.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_lora_gemm_kernel<BNMAX, SWAP, LOCALT, STATS>, maps, P);
}

// The pair kernel's launch: clusters of two CTAs, chained like the others.
template <bool STATS>
cudaError_t pair_kernel_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(pair_gemm_kernel<STATS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(kPairSmem));
  });
  return err;
}

// Clusters of two that can be resident at once (asked once per process, on
// the first launch; the schedule uses no more).
void query_pair_cap() {
  if (!kPairMma || g_pair_cap.load() != 0) return;
  int n = 0;
  if (pair_kernel_attr<false>() == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(2 * std::max(1, sm_count() / 2)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPairSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, pair_gemm_kernel<false>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  g_pair_cap.store(n > 0 ? n : -1);  // -1: no pair launches
}

template <bool STATS>
cudaError_t launch_pair(const Maps& maps, const Params& P, cudaStream_t st) {
  const cudaError_t a = pair_kernel_attr<STATS>();
  if (a != cudaSuccess) return a;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(P.grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<STATS>, maps, P);
}

}  // namespace

size_t lora_group_workspace_bytes(int n, const uno_lora_problem* pr, int64_t M, int dtype,
                                  int sms) {
  // enough for the pair order and for the CTA-per-tile order (a launch with
  // the statistics epilogue takes the latter)
  auto Lp = std::make_unique<Layout>(), Lq = std::make_unique<Layout>();
  if (!make_layout(n, pr, M, dtype, sms, *Lp)) return 0;
  if (!make_layout(n, pr, M, dtype, sms, *Lq, false)) return 0;
  return std::max(Lp->bytes, Lq->bytes);
}

// Host-side invariants of the schedule make_layout builds for `sms` CTAs
// (no GPU involved): 0 when all hold, else the number of the first that fails.
int lora_plan_check(int n, const uno_lora_problem* pr, int64_t M, int dtype, int sms) {
  auto Lp = std::make_unique<Layout>();
  Layout& L = *Lp;
  if (!make_layout(n, pr, M, dtype, sms, L)) return 1;
  const Params& P = L.P;
  const int G = P.grid;
  // 2: one CTA per SM, at most the grid the kernel is built for
  if (G < 1 || G > std::min(sms, kMaxGrid)) return 2;
  // 3: the phase table: data-parallel phases, then the two stream-K sections
  if (P.dp0 < 0 || P.dp1 < P.dp0 || P.ph0[0] != P.dp1 || P.ph1[0] < P.ph0[0] ||
      P.ph0[1] != P.ph1[0] || P.ph1[1] < P.ph0[1] || P.ph1[1] > kMaxPhases)
    return 3;
  // 4: data-parallel waves only in tokens-as-M order, and then over every tile
  if (P.dp_tiles > 0) {
    int64_t t = 0;
    for (int p = P.dp0; p < P.dp1; ++p) t += P.ph[p].tiles;
    if (P.swap || t != P.dp_tiles || P.dp_tiles < (P.pair ? (G / 2 + 1) / 2 : G)) return 4;
  }
  int64_t sec_total[2] = {0, 0};
  for (int sec = 0; sec < 2; ++sec) {
    // 5: a section's phases are contiguous runs of whole tiles
    for (int p = P.ph0[sec]; p < P.ph1[sec]; ++p) {
      const Phase& f = P.ph[p];
      if (f.kb_start != sec_total[sec] || f.tiles < 1 || f.nkb < 1 || (f.down != 0) != (sec == kDown))
        return 5;
      sec_total[sec] += int64_t(f.tiles) * f.nkb;
    }
    // 6: CTA ranges partition the section's K-blocks in CTA order
    if (P.lo[sec][0] != 0 || P.lo[sec][G] != sec_total[sec]) return 6;
    for (int c = 0; c < G; ++c)
      if (P.lo[sec][c + 1] < P.lo[sec][c]) return 6;
  }
  // 7: a per-piece adapter needs no T tiles
  if (P.localt && sec_total[kDown] > 0) return 7;
  // 8: (one finisher per split T tile) a CTA that finishes a split T tile
  // has no main work (unless all do)
  int n_fin = 0, n_fin_busy = 0;
  for (int c = 0; c < G && !P.tslice; ++c) {
    const int64_t lo0 = P.lo[kDown][c], hi0 = P.lo[kDown][c + 1];
    if (lo0 >= hi0) continue;
    for (int p = P.ph0[kDown]; p < P.ph1[kDown]; ++p) {
      const Phase& f = P.ph[p];
      const int64_t end = f.kb_start + int64_t(f.tiles) * f.nkb;
      if (hi0 - 1 < f.kb_start || hi0 - 1 >= end) continue;
      const int64_t ts = f.kb_start + (hi0 - 1 - f.kb_start) / f.nkb * f.nkb;
      if (ts >= lo0 && ts + f.nkb > hi0) {
        ++n_fin;
        n_fin_busy += P.lo[kMain][c] < P.lo[kMain][c + 1];
      }
    }
  }
  if (n_fin_busy > 0 && n_fin < G) return 8;
  // 13: (T tiles merged by slices) only in token-rows order; the down
  // section's CTA ranges are pieces of single T tiles, one per CTA, with every
  // piece of a tile in consecutive CTAs, and the T counters fit the sync area
  if (P.tslice && (P.swap || sec_total[kDown] == 0)) return 13;
  if (P.tslice) {
    int c = 0;
    for (int p = P.ph0[kDown]; p < P.ph1[kDown]; ++p) {
      const Phase& f = P.ph[p];
      for (int t = 0; t < f.tiles; ++t) {
        const int64_t kb0 = f.kb_start + int64_t(t) * f.nkb, kb1 = kb0 + f.nkb;
        if (P.lo[kDown][c] != kb0) return 13;
        while (c < G && P.lo[kDown][c + 1] < kb1) {
          if (P.lo[kDown][c + 1] <= P.lo[kDown][c]) return 13;
          ++c;
        }
        if (c >= G || P.lo[kDown][c + 1] != kb1) return 13;
        ++c;
      }
    }
    for (; c < G; ++c)
      if (P.lo[kDown][c] != P.lo[kDown][c + 1]) return 13;
    if ((2 * size_t(G) + 2 * size_t(L.tflags)) * sizeof(int) > L.sync_bytes) return 13;
  }
  // 14: pair order: an even grid of at most one CTA per SM, data-parallel
  // phases only (T tiles first, of the whole rank; y tiles 256 wide), tiles of
  // 256 tokens, ranks that split into two TMA boxes, one T flag per T tile
  if (P.pair) {
    if (G % 2 || G < 2 || P.dp0 != 0 || P.ph0[0] != P.dp1 || sec_total[0] || sec_total[1] || P.swap ||
        P.tsplit || P.localt || P.tslice)
      return 14;
    int flags = 0;
    bool seen_y = false;
    for (int p = P.dp0; p < P.dp1; ++p) {
      const Phase& f = P.ph[p];
      const Prob& b = P.pb[f.prob];
      if (f.tiles_a != int((M + 2 * kBM - 1) / (2 * kBM)) || f.tiles != f.tiles_all) return 14;
      if (f.down) {
        if (seen_y || f.bn != b.r || b.r % 32 || b.r > 256 || f.na || b.tflag0 != flags) return 14;
        flags += f.tiles;
      } else {
        seen_y = true;
        if ((f.bn != 256 && f.bn != 128) || f.na != (b.r + kBK - 1) / kBK || f.n0 % 256 ||
            f.tiles_all % f.tiles_a)
          return 14;
      }
    }
    // every problem's output columns are covered once, in ascending phases
    for (int q = 0; q < n; ++q) {
      int64_t next = 0;
      for (int p = P.dp0; p < P.dp1; ++p) {
        const Phase& f = P.ph[p];
        if (f.down || f.prob != q) continue;
        if (f.n0 != next) return 14;
        next = f.n0 + int64_t(f.tiles_all / f.tiles_a) * f.bn;
      }
      if (next < pr[q].d_out || next - pr[q].d_out >= 256) return 14;
    }
    if (flags != L.tflags || (2 * size_t(G) + 2 * size_t(flags)) * sizeof(int) > L.sync_bytes) return 14;
  }
  // 9: decode order only for decode-sized M
  if (P.swap != (M <= kSwapMaxRows ? 1 : 0)) return 9;
  // 10: workspace regions in order and inside the total
  if (L.off_partial > L.off_sync || L.off_sync + L.sync_bytes > L.bytes) return 10;
  // 11: the partial slots hold a tile of the widest phase
  for (int p = 0; p < P.ph1[1]; ++p)
    if (P.ph[p].bn > P.bnmax) return 11;
  // 12: split-K adapter only in decode order and without T tiles; its chunks,
  // in problem order and at most one per CTA, cover every adapted problem's
  // K-blocks; its partials fit their workspace region
  if (P.tsplit) {
    if (!P.swap || P.localt || sec_total[kDown] > 0 || P.tkpc < 1 || P.bnmax > 64 ||
        P.tbn != P.bnmax || M > P.tbn)
      return 12;
    if (P.tch0[0] != 0 || P.tch0[n] != P.tchunks || P.tchunks > G) return 12;
    int64_t max_r = 0;
    for (int p = 0; p < n; ++p) {
      const int64_t nkb = (pr[p].d_in + kBK - 1) / kBK;
      const int64_t want = pr[p].rank > 0 ? (nkb + P.tkpc - 1) / P.tkpc : 0;
      if (P.tch0[p + 1] - P.tch0[p] != want) return 12;
      max_r = std::max<int64_t>(max_r, pr[p].rank);
    }
    if (P.tpart_stride < M * max_r || P.tpart_stride % 4 ||
        L.off_tpart + size_t(P.tchunks) * size_t(P.tpart_stride) * sizeof(float) > L.off_partial)
      return 12;
  }
  return 0;
}

namespace {
int launch_linear(int n, const uno_lora_problem* pr, int64_t M, int dtype, void* ws,
                  size_t ws_bytes, cudaStream_t st, const LinearEpilogue* epi);
}  // namespace

int launch_lora_group(int n, const uno_lora_problem* pr, int64_t M, int dtype, void* ws,
                      size_t ws_bytes, cudaStream_t st) {
  return launch_linear(n, pr, M, dtype, ws, ws_bytes, st, nullptr);
}

int launch_logit_gemm(const uno_lora_problem& pr, int64_t M, void* ws, size_t ws_bytes,
                      cudaStream_t st, const LinearEpilogue& epi) {
  return launch_linear(1, &pr, M, UNO_BF16, ws, ws_bytes, st, &epi);
}

namespace {
// Vocabulary tiles per logit row in a layout (the statistics epilogue leaves
// one (max, sum exp) per row and tile).
int layout_vocab_tiles(const Layout& L, int64_t V) {
  for (int i = 0; i < L.P.ph1[kMain]; ++i)
    if (!L.P.ph[i].down) {
      const int w = L.P.swap ? kBM : L.P.ph[i].bn;
      return int((V + w - 1) / w);
    }
  return 0;
}
}  // namespace

int logit_gemm_tiles(int64_t M, int64_t d, int64_t V, int sms) {
  uno_lora_problem p{};
  p.d_in = d;
  p.d_out = V;
  query_pair_cap();  // the same schedule as the launch
  auto L = std::make_unique<Layout>();
  if (!make_layout(1, &p, M, UNO_BF16, sms, *L, true, true)) return 0;  // (the statistics epilogue's)
  return layout_vocab_tiles(*L, V);
}

namespace {
// The schedule and the encoded tensor maps of a launch depend only on the
// problems' pointers and shapes, the epilogue, the workspace pointer, the
// device and its SM count: a small per-process cache spares repeated calls
// with the same arguments (every decode step of a serving loop) the host work
// of building them.
struct PlanKey {
  int n, dtype, dev, sms, has_epi;
  int64_t M;
  void* ws;
  uno_lora_problem pr[kMaxLoraProblems];
  LinearEpilogue epi;
};
struct PlanEntry {
  bool valid;
  PlanKey key;
  Layout L;
  Maps maps;
};
constexpr int kPlanCache = 16;
PlanEntry g_plans[kPlanCache];
int g_plan_next = 0;
std::mutex g_plan_mu;

int build_plan(int n, const uno_lora_problem* pr, int64_t M, int dtype, char* w, size_t ws_bytes,
               int sms, const LinearEpilogue* epi, Layout& L, Maps& maps) {
  if (!make_layout(n, pr, M, dtype, sms, L, true, epi && epi->stats)) return UNO_ERR_ARG;
  if (ws_bytes < L.bytes) return UNO_ERR_WORKSPACE;
  Params& P = L.P;
  P.partial = reinterpret_cast<float*>(w + L.off_partial);
  P.tpart = reinterpret_cast<float*>(w + L.off_tpart);
  P.ready = reinterpret_cast<int*>(w + L.off_sync);
  P.tflag = P.ready + 2 * P.grid;
  P.tcnt = P.tflag + L.tflags;
  std::memset(&maps, 0, sizeof(maps));
  for (int p = 0; p < n; ++p) {
    const uno_lora_problem& q = pr[p];
    const void *x = q.x, *W = q.W, *A = q.A, *B = q.B;
    if (dtype == UNO_F32) {  // operands read from their bf16 copies in the workspace
      x = w + L.off_cast[p][0];
      W = w + L.off_cast[p][1];
      A = w + L.off_cast[p][2];
      B = w + L.off_cast[p][3];
    }
    Prob& b = P.pb[p];
    b.y = q.y;
    b.t = w + L.off_t[p];
    b.gate = q.gate;

    if (epi) {
      b.f32out = epi->f32out;
      b.st_store = epi->stats_store;
      b.st_K = int(epi->K);
      b.st_Kp = int(epi->Kp);
      b.st_Rp = int(epi->Rp);
      b.st_nvt = epi->nvt;
      b.st_draft = epi->draft;
      b.st_part = epi->part;
      b.st_gather = epi->gathered;
    }
    int bn_main = 0, bn_down = 0;  // the widest tiles of the problem (pair order: also 128-wide ones)
    for (int i = 0; i < P.ph1[kMain]; ++i)
      if (P.ph[i].prob == p) {
        int& w = P.ph[i].down ? bn_down : bn_main;
        w = std::max(w, P.ph[i].bn);
      }
    CUtensorMap* m = maps.m[p];
    const bool sw = P.swap != 0;
    // pair order: each CTA loads half of a tile's output rows (bn / 2)
    if (P.pair) {
      bn_main /= 2;
      bn_down /= 2;
    }
    bool ok = encode_bf16(&m[MAP_X], x, q.d_in, M, sw ? bn_main : kBM) &&
              encode_bf16(&m[MAP_W], W, q.d_in, q.d_out, sw ? kBM : bn_main);
    if (ok && q.rank > 0) {
      ok = encode_bf16(&m[MAP_A], A, q.d_in, q.rank, sw ? kBM : bn_down) &&
           encode_bf16(&m[MAP_B], B, q.rank, q.d_out, sw ? kBM : bn_main) &&
           encode_bf16(&m[MAP_T], b.t, q.rank, M, sw ? bn_main : kBM);
    } else {
      m[MAP_A] = m[MAP_B] = m[MAP_T] = m[MAP_X];
    }
    // (pair order) 64-row boxes of W and B for the 128-wide tiles
    if (ok && P.pair) {
      ok = encode_bf16(&m[MAP_W2], W, q.d_in, q.d_out, 64) &&
           (q.rank == 0 || encode_bf16(&m[MAP_B2], B, q.rank, q.d_out, 64));
      if (q.rank == 0) m[MAP_B2] = m[MAP_W2];
    } else {
      m[MAP_W2] = m[MAP_B2] = m[MAP_X];
    }
    if (!ok) return UNO_ERR_CUDA;
  }
  return UNO_OK;
}

int launch_linear(int n, const uno_lora_problem* pr, int64_t M, int dtype, void* ws,
                  size_t ws_bytes, cudaStream_t st, const LinearEpilogue* epi) {
  char* w = static_cast<char*>(ws);
  auto key = std::make_unique<PlanKey>();
  std::memset(key.get(), 0, sizeof(PlanKey));
  key->n = n;
  key->dtype = dtype;
  cudaGetDevice(&key->dev);
  key->sms = sm_count();
  key->M = M;
  key->ws = ws;
  for (int p = 0; p < n; ++p) {
    uno_lora_problem& k = key->pr[p];
    k.x = pr[p].x;
    k.W = pr[p].W;
    k.A = pr[p].A;
    k.B = pr[p].B;
    k.gate = pr[p].gate;
    k.y = pr[p].y;
    k.d_in = pr[p].d_in;
    k.d_out = pr[p].d_out;
    k.rank = pr[p].rank;
    k.alpha = pr[p].alpha;
  }
  if (epi) {
    key->has_epi = 1;
    LinearEpilogue& e = key->epi;
    e.f32out = epi->f32out;
    e.stats = epi->stats;
    e.stats_store = epi->stats_store;
    e.K = epi->K;
    e.Kp = epi->Kp;
    e.Rp = epi->Rp;
    e.nvt = epi->nvt;
    e.draft = epi->draft;
    e.part = epi->part;
    e.gathered = epi->gathered;
  }
  query_pair_cap();
  auto Lp = std::make_unique<Layout>();
  Layout& L = *Lp;
  Maps maps;
  bool hit = false;
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (int i = 0; i < kPlanCache && !hit; ++i)
      if (g_plans[i].valid && std::memcmp(&g_plans[i].key, key.get(), sizeof(PlanKey)) == 0) {
        L = g_plans[i].L;
        maps = g_plans[i].maps;
        hit = true;
      }
  }
  if (!hit) {
    const int rc = build_plan(n, pr, M, dtype, w, ws_bytes, key->sms, epi, L, maps);
    if (rc != UNO_OK) return rc;
    {
      std::lock_guard<std::mutex> lock(g_plan_mu);
      PlanEntry& e = g_plans[g_plan_next];
      g_plan_next = (g_plan_next + 1) % kPlanCache;
      e.key = *key;
      e.L = L;
      e.maps = maps;
      e.valid = true;
    }
  }
  if (ws_bytes < L.bytes) return UNO_ERR_WORKSPACE;
  Params& P = L.P;
  if (dtype == UNO_F32) {
    for (int p = 0; p < n; ++p) {
      const uno_lora_problem& q = pr[p];
      if (cast_to_bf16(q.x, w + L.off_cast[p][0], M * q.d_in, st) != cudaSuccess ||
          cast_to_bf16(q.W, w + L.off_cast[p][1], q.d_out * q.d_in, st) != cudaSuccess ||
          (q.rank > 0 && (cast_to_bf16(q.A, w + L.off_cast[p][2], q.rank * q.d_in, st) != cudaSuccess ||
                          cast_to_bf16(q.B, w + L.off_cast[p][3], q.d_out * q.rank, st) != cudaSuccess)))
        return UNO_ERR_CUDA;
    }
  }
  {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (reinterpret_cast<uintptr_t>(w + L.off_sync) & 15u) return UNO_ERR_WORKSPACE;
    if (cudaLaunchKernelEx(&cfg, sync_reset_kernel, reinterpret_cast<int4*>(w + L.off_sync),
                           int(L.sync_bytes / 16)) != cudaSuccess)
      return UNO_ERR_CUDA;
  }
  cudaError_t e;
  // one instantiation per (tile width, operand order, adapter mode, epilogue)
#define UNO_DISPATCH(SW, LT, ST)                                         \
  switch (P.bnmax) {                                                     \
    case 16: e = launch_grouped<16, SW, LT, ST>(maps, P, st); break;     \
    case 32: e = launch_grouped<32, SW, LT, ST>(maps, P, st); break;     \
    case 64: e = launch_grouped<64, SW, LT, ST>(maps, P, st); break;     \
    case 128: e = launch_grouped<128, SW, LT, ST>(maps, P, st); break;   \
    default: e = launch_grouped<256, SW, LT, ST>(maps, P, st); break;    \
  }
  // the statistics partials are laid out by the vocabulary tiles the caller
  // planned for: a launch whose tiles differ would write past them
  if (epi && epi->stats && layout_vocab_tiles(L, pr[0].d_out) != epi->nvt) return UNO_ERR_ARG;
  if (P.pair) {
    if (epi && epi->stats) {
      if (n != 1 || pr[0].rank != 0) return UNO_ERR_UNSUPPORTED;
      e = launch_pair<true>(maps, P, st);
    } else {
      e = launch_pair<false>(maps, P, st);
    }
  } else if (epi && epi->stats) {
    if (n != 1 || P.localt || pr[0].rank != 0) return UNO_ERR_UNSUPPORTED;
    if (P.swap) {
      UNO_DISPATCH(true, false, true)
    } else {
      UNO_DISPATCH(false, false, true)
    }
  } else if (P.localt) {
    UNO_DISPATCH(true, true, false)
  } else if (P.swap) {
    UNO_DISPATCH(true, false, false)
  } else {
    UNO_DISPATCH(false, false, false)
  }
#undef UNO_DISPATCH
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}
}  // namespace

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
