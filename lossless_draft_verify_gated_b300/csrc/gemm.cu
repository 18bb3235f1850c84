// gemm.cu -- gated-LoRA linear projection on the tcgen05 tensor cores.
//
//   y = x.W^T + gate_row * (alpha/rank) * (x.A^T).B^T
// "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
// (aifromscratch.in), section "Two Decoupled Weight Sets": draft rows (gate 1)
// use theta_AR plus the rank-128, alpha=256 LoRA adapter theta_Delta;
// verification rows (gate 0) use theta_AR only.
//
// Two launches of one warp-specialised kernel:
//   1. T = bf16(gate * alpha/rank * x.A^T)          (down-projection, [M, rank])
//   2. y = x.W^T + T.B^T                             (base GEMM)
//      The up-projection is not a second pass over y: its rank/64 K-blocks
//      are appended to the base GEMM's K loop and accumulate into the same
//      TMEM accumulator, so W is streamed from HBM exactly once and y is
//      written exactly once.  Gate-0 rows of T are exact zeros, so gate-0 rows
//      of y are the plain x.W^T of the same kernel.
//
// Kernel anatomy (one output tile per CTA, 128 threads):
//   warp 0 lane 0  TMA producer: 128-byte-swizzled 64-wide K slices of both
//                  operands into a STAGES-deep shared-memory ring (mbarrier
//                  full/empty pairs); weights with an L2 evict-first policy.
//   warp 1         allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=BN,
//                  K=16, bf16 x bf16 -> fp32) and commits each stage back to
//                  the producer.
//   warps 0-3      epilogue: tcgen05.ld of their TMEM lane quadrant, optional
//                  per-row gate scale, bf16/fp32 store; split-K partials are
//                  summed in a fixed order by the last CTA of each tile
//                  (atomic arrival count, nobody waits), so results are
//                  deterministic.
// Decode-sized M (<= 256 token rows) swaps operands: the weight tile fills the
// 128-row MMA side and the tokens are the MMA's N, and the K loop is split
// across CTAs so that every SM streams weights.
// Every mbarrier wait is bounded (2 s); a timeout sets a device error word
// and the CTA unwinds instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "ptx.cuh"
#include "uno_internal.h"

namespace uno {

__device__ int g_device_error;  // bit 0: an mbarrier wait in the GEMM timed out

namespace {

constexpr int kBM = 128;     // MMA M: A-operand rows per tile (= TMEM lanes)
constexpr int kBK = 64;      // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kUmmaK = 16;   // K per tcgen05.mma for 16-bit inputs
constexpr int kThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct MainArgs {
  int nkb_base;      // K-blocks of the base product (over d_in)
  int nkb_lora;      // K-blocks of the adapter product (over rank), appended
  int splits;        // CTAs sharing one output tile along K
  int kb_per_split;
  int tiles_a;       // tiles along the A-operand rows
  int swap;          // 1: A-operand rows are output columns, B-operand rows are tokens
  int pdl_wait;      // griddepcontrol.wait before the first adapter K-block
};

struct EpiArgs {
  void* out;            // [M, ldo], bf16 or fp32
  int64_t ldo;
  int64_t M;            // token rows
  int64_t N;            // output columns
  int out_f32;
  const uint8_t* gate;  // optional per-token-row multiplier gate[m] * gscale
  float gscale;
  float* partial;       // split-K partials [tiles][splits][BN][128] (null if splits == 1)
  int* counters;        // [tiles], zero on entry, returned to zero
};

__device__ __forceinline__ void store_out(const EpiArgs& e, int64_t m, int64_t n, float v) {
  if (m >= e.M || n >= e.N) return;
  if (e.gate) v *= float(e.gate[m]) * e.gscale;
  if (e.out_f32)
    static_cast<float*>(e.out)[m * e.ldo + n] = v;
  else
    static_cast<__nv_bfloat16*>(e.out)[m * e.ldo + n] = __float2bfloat16_rn(v);
}

template <int BN>
constexpr int stages_for() {
  return BN <= 64 ? 8 : (BN == 128 ? 6 : 4);
}
template <int BN>
constexpr uint32_t smem_bytes_for() {
  return uint32_t(stages_for<BN>()) * uint32_t(kBM * kBK * 2 + BN * kBK * 2) + 1024 + 256;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
gated_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mB0,
                  const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mB1,
                  const MainArgs a, const EpiArgs e) {
  constexpr int STAGES = stages_for<BN>();
  constexpr uint32_t kABytes = kBM * kBK * 2;
  constexpr uint32_t kBBytes = BN * kBK * 2;
  constexpr uint32_t kStage = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = BN < 32 ? 32 : BN;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* accum = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* last_flag = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x % a.splits;
  const int tile = blockIdx.x / a.splits;
  const int ta = tile % a.tiles_a;
  const int tb = tile / a.tiles_a;
  const int nkb = a.nkb_base + a.nkb_lora;
  const int kb0 = split * a.kb_per_split;
  const int nk = min(nkb, kb0 + a.kb_per_split) - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(accum, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&mA0);
    ptx::prefetch_tensormap(&mB0);
    if (a.nkb_lora) {
      ptx::prefetch_tensormap(&mA1);
      ptx::prefetch_tensormap(&mB1);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::grid_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- producer
    const uint64_t pol_stream = ptx::policy_evict_first();
    const uint64_t pol_keep = ptx::policy_evict_last();
    const uint64_t polA = a.swap ? pol_stream : pol_keep;  // weights are streamed once
    const uint64_t polB = a.swap ? pol_keep : pol_stream;
    bool waited = false;
    int issued = 0;
    for (int i = 0; i < nk; ++i) {
      const int s = i % STAGES;
      if (i >= STAGES && !ptx::mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, kWaitLimitNs)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      const int kb = kb0 + i;
      uint8_t* sa = smem + s * kStage;
      uint8_t* sb = sa + kABytes;
      if (kb < a.nkb_base) {
        ptx::mbar_arrive_expect_tx(&full[s], kStage);
        ptx::tma_load_2d(sa, &mA0, &full[s], kb * kBK, ta * kBM, polA);
        ptx::tma_load_2d(sb, &mB0, &full[s], kb * kBK, tb * BN, polB);
      } else {
        if (a.pdl_wait && !waited) {
          ptx::grid_dependency_wait();
          waited = true;
        }
        const int kl = (kb - a.nkb_base) * kBK;
        ptx::mbar_arrive_expect_tx(&full[s], kStage);
        ptx::tma_load_2d(sa, &mA1, &full[s], kl, ta * kBM, pol_keep);
        ptx::tma_load_2d(sb, &mB1, &full[s], kl, tb * BN, pol_keep);
      }
      ++issued;
    }
    if (*abort_flag) {
      // Let copies already in flight land before the CTA can exit.
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        ptx::mbar_wait(&full[i % STAGES], (i / STAGES) & 1, kWaitLimitNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    for (int i = 0; i < nk; ++i) {
      const int s = i % STAGES;
      if (!ptx::mbar_wait(&full[s], (i / STAGES) & 1, kWaitLimitNs)) {
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t sa = ptx::smem_u32(smem + s * kStage);
      const uint32_t sb = sa + kABytes;
#pragma unroll
      for (int k = 0; k < kBK / kUmmaK; ++k)
        ptx::umma_f16(tmem, ptx::sw128_kmajor_desc(sa + k * 32), ptx::sw128_kmajor_desc(sb + k * 32),
                      kIdesc, (i | k) != 0);
      ptx::umma_commit(&empty[s]);
    }
    ptx::umma_commit(accum);
  }
  __syncwarp();

  // ------------------------------------------------------------ epilogue
  bool ok = ptx::mbar_wait(accum, 0, kWaitLimitNs);
  ok = __syncthreads_and(ok && !*abort_flag) != 0;  // uniform: tcgen05.ld is warp-collective
  ptx::tc_fence_after();
  if (!ok && threadIdx.x == 0) atomicOr(&g_device_error, 1);
  const int row = warp * 32 + lane;  // TMEM lane = A-operand row within the tile
  const uint32_t tq = tmem + (uint32_t(warp * 32) << 16);
  const int64_t a_row = int64_t(ta) * kBM + row;
  const int64_t b_row0 = int64_t(tb) * BN;
  if (ok) {
    if (a.splits == 1) {
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(tq + c, r);
        ptx::tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int64_t br = b_row0 + c + j;
          if (a.swap)
            store_out(e, br, a_row, __uint_as_float(r[j]));
          else
            store_out(e, a_row, br, __uint_as_float(r[j]));
        }
      }
    } else {
      float* P = e.partial + (size_t(tile) * a.splits + split) * (BN * kBM);
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(tq + c, r);
        ptx::tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) __stcg(P + (c + j) * kBM + row, __uint_as_float(r[j]));
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (!ok || a.splits == 1) return;

  // Split-K: the last CTA of the tile sums the partials in split order.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *last_flag = atomicAdd(&e.counters[tile], 1) == a.splits - 1;
  __syncthreads();
  if (!*last_flag) return;
  __threadfence();
  const float* P0 = e.partial + size_t(tile) * a.splits * (BN * kBM);
#pragma unroll 1
  for (int j = 0; j < BN; ++j) {
    float acc = 0.f;
#pragma unroll 4
    for (int s = 0; s < a.splits; ++s) acc += __ldcg(P0 + size_t(s) * (BN * kBM) + j * kBM + row);
    const int64_t br = b_row0 + j;
    if (a.swap)
      store_out(e, br, a_row, acc);
    else
      store_out(e, a_row, br, acc);
  }
  if (threadIdx.x == 0) e.counters[tile] = 0;
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

struct GemmPlan {
  int swap, BN;
  int tiles_a, tiles_b, splits, kb_per_split;
  int nkb_base, nkb_lora;
  size_t partial_bytes, counter_bytes;
  int tiles() const { return tiles_a * tiles_b; }
};

int pick_bn(int64_t n) {
  for (int bn : {16, 32, 64, 128}) if (n <= bn) return bn;
  return 256;
}

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K_base, int64_t K_lora, int sms) {
  GemmPlan p{};
  p.nkb_base = int((K_base + kBK - 1) / kBK);
  p.nkb_lora = int((K_lora + kBK - 1) / kBK);
  const int nkb = p.nkb_base + p.nkb_lora;
  if (M <= 256) {
    p.swap = 1;
    p.BN = pick_bn(M);
    p.tiles_a = int((N + kBM - 1) / kBM);
    p.tiles_b = 1;
  } else {
    p.swap = 0;
    p.BN = pick_bn(N);
    p.tiles_a = int((M + kBM - 1) / kBM);
    p.tiles_b = int((N + p.BN - 1) / p.BN);
  }
  int splits = 1;
  if (p.tiles() < sms) splits = std::max(1, std::min({sms / p.tiles(), std::max(1, nkb / 4), 32}));
  p.kb_per_split = (nkb + splits - 1) / splits;
  p.splits = (nkb + p.kb_per_split - 1) / p.kb_per_split;
  p.partial_bytes = p.splits > 1 ? size_t(p.tiles()) * p.splits * p.BN * kBM * sizeof(float) : 0;
  p.counter_bytes = p.splits > 1 ? size_t(p.tiles()) * sizeof(int) : 0;
  return p;
}

template <int BN>
cudaError_t launch_bn(const GemmPlan& p, const CUtensorMap* maps, const MainArgs& ma,
                      const EpiArgs& ea, cudaStream_t st, bool pdl) {
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(gated_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(smem_bytes_for<BN>()));
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(p.tiles() * p.splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for<BN>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gated_gemm_kernel<BN>, maps[0], maps[1], maps[2], maps[3], ma, ea);
}

cudaError_t launch_gemm(const GemmPlan& p, const CUtensorMap* maps, const EpiArgs& ea,
                        cudaStream_t st, bool pdl_wait) {
  MainArgs ma{};
  ma.nkb_base = p.nkb_base;
  ma.nkb_lora = p.nkb_lora;
  ma.splits = p.splits;
  ma.kb_per_split = p.kb_per_split;
  ma.tiles_a = p.tiles_a;
  ma.swap = p.swap;
  ma.pdl_wait = pdl_wait ? 1 : 0;
  switch (p.BN) {
    case 16: return launch_bn<16>(p, maps, ma, ea, st, pdl_wait);
    case 32: return launch_bn<32>(p, maps, ma, ea, st, pdl_wait);
    case 64: return launch_bn<64>(p, maps, ma, ea, st, pdl_wait);
    case 128: return launch_bn<128>(p, maps, ma, ea, st, pdl_wait);
    default: return launch_bn<256>(p, maps, ma, ea, st, pdl_wait);
  }
}

struct LoraLayout {
  GemmPlan down, main;
  size_t off_t, off_down_part, off_main_part, off_counters, off_cast, bytes;
  size_t cast_x, cast_w, cast_a, cast_b;  // offsets of bf16 copies (fp32 mode)
};

LoraLayout lora_layout(int64_t M, int64_t d_in, int64_t d_out, int64_t rank, int dtype, int sms) {
  LoraLayout L{};
  if (rank > 0) L.down = plan_gemm(M, rank, d_in, 0, sms);
  L.main = plan_gemm(M, d_out, d_in, rank, sms);
  size_t o = 0;
  L.off_t = o;
  o = align_up(o + size_t(M) * size_t(rank) * 2, 256);
  L.off_down_part = o;
  o = align_up(o + L.down.partial_bytes, 256);
  L.off_main_part = o;
  o = align_up(o + L.main.partial_bytes, 256);
  L.off_counters = o;
  o = align_up(o + L.down.counter_bytes + L.main.counter_bytes, 256);
  L.off_cast = o;
  if (dtype == UNO_F32) {
    L.cast_x = o;
    o = align_up(o + size_t(M) * d_in * 2, 256);
    L.cast_w = o;
    o = align_up(o + size_t(d_out) * d_in * 2, 256);
    L.cast_a = o;
    o = align_up(o + size_t(rank) * d_in * 2, 256);
    L.cast_b = o;
    o = align_up(o + size_t(d_out) * rank * 2, 256);
  }
  L.bytes = std::max<size_t>(o, 256);
  return L;
}

cudaError_t cast_to_bf16(const void* in, void* out, int64_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 148 * 16);
  cast_f32_bf16_kernel<<<unsigned(blocks), 256, 0, st>>>(static_cast<const float*>(in),
                                                        static_cast<__nv_bfloat16*>(out), n);
  return cudaGetLastError();
}

}  // namespace

size_t lora_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int64_t rank, int dtype,
                            int sms) {
  return lora_layout(M, d_in, d_out, rank, dtype, sms).bytes;
}

int launch_gated_lora_linear(const void* x, const void* W, const void* A, const void* B,
                             const uint8_t* gate, int64_t M, int64_t d_in, int64_t d_out,
                             int64_t rank, float alpha, int dtype, void* y, void* ws,
                             size_t ws_bytes, cudaStream_t st) {
  const LoraLayout L = lora_layout(M, d_in, d_out, rank, dtype, sm_count());
  if (ws_bytes < L.bytes) return UNO_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  const void *xb = x, *Wb = W, *Ab = A, *Bb = B;
  if (dtype == UNO_F32) {
    if (cast_to_bf16(x, w + L.cast_x, M * d_in, st) != cudaSuccess) return UNO_ERR_CUDA;
    if (cast_to_bf16(W, w + L.cast_w, d_out * d_in, st) != cudaSuccess) return UNO_ERR_CUDA;
    if (rank > 0) {
      if (cast_to_bf16(A, w + L.cast_a, rank * d_in, st) != cudaSuccess) return UNO_ERR_CUDA;
      if (cast_to_bf16(B, w + L.cast_b, d_out * rank, st) != cudaSuccess) return UNO_ERR_CUDA;
    }
    xb = w + L.cast_x;
    Wb = w + L.cast_w;
    Ab = w + L.cast_a;
    Bb = w + L.cast_b;
  }
  int* counters = reinterpret_cast<int*>(w + L.off_counters);
  const size_t cbytes = L.down.counter_bytes + L.main.counter_bytes;
  if (cbytes && cudaMemsetAsync(counters, 0, cbytes, st) != cudaSuccess) return UNO_ERR_CUDA;
  void* T = w + L.off_t;

  CUtensorMap maps[4];
  std::memset(maps, 0, sizeof(maps));
  if (rank > 0) {
    // T = bf16(gate * alpha/rank * x.A^T): tokens x rank, K = d_in.
    const GemmPlan& p = L.down;
    const void* rows_a = p.swap ? Ab : xb;
    const void* rows_b = p.swap ? xb : Ab;
    const int64_t na = p.swap ? rank : M, nb = p.swap ? M : rank;
    if (!encode_bf16(&maps[0], rows_a, d_in, na, kBM) || !encode_bf16(&maps[1], rows_b, d_in, nb, p.BN))
      return UNO_ERR_CUDA;
    maps[2] = maps[0];
    maps[3] = maps[1];
    EpiArgs e{};
    e.out = T;
    e.ldo = rank;
    e.M = M;
    e.N = rank;
    e.out_f32 = 0;
    e.gate = gate;
    e.gscale = alpha / float(rank);
    e.partial = reinterpret_cast<float*>(w + L.off_down_part);
    e.counters = counters;
    if (launch_gemm(p, maps, e, st, false) != cudaSuccess) return UNO_ERR_CUDA;
  }
  {
    // y = x.W^T + T.B^T, adapter K-blocks appended to the base K loop.
    const GemmPlan& p = L.main;
    const void* a0 = p.swap ? Wb : xb;
    const void* b0 = p.swap ? xb : Wb;
    const int64_t na = p.swap ? d_out : M, nb = p.swap ? M : d_out;
    if (!encode_bf16(&maps[0], a0, d_in, na, kBM) || !encode_bf16(&maps[1], b0, d_in, nb, p.BN))
      return UNO_ERR_CUDA;
    if (rank > 0) {
      const void* a1 = p.swap ? Bb : T;
      const void* b1 = p.swap ? T : Bb;
      if (!encode_bf16(&maps[2], a1, rank, na, kBM) || !encode_bf16(&maps[3], b1, rank, nb, p.BN))
        return UNO_ERR_CUDA;
    } else {
      maps[2] = maps[0];
      maps[3] = maps[1];
    }
    EpiArgs e{};
    e.out = y;
    e.ldo = d_out;
    e.M = M;
    e.N = d_out;
    e.out_f32 = dtype == UNO_F32;
    e.gate = nullptr;
    e.gscale = 1.f;
    e.partial = reinterpret_cast<float*>(w + L.off_main_part);
    e.counters = reinterpret_cast<int*>(w + L.off_counters + L.down.counter_bytes);
    if (launch_gemm(p, maps, e, st, rank > 0) != cudaSuccess) return UNO_ERR_CUDA;
  }
  return UNO_OK;
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
