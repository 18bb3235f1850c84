// api.cu -- the extern "C" boundary of libuno.so (declared in include/uno.h):
// argument validation, workspace queries and dispatch to the kernels.
// Everything here runs on the host and touches no device memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "uno_internal.h"

namespace uno {

int read_device_error(int reset);  // gemm.cu

namespace {
// SMs of the current context's SM resource when the driver reports one (a
// green context may own fewer SMs than the device); 0 when it does not.
int context_sm_count() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetDevResource_v12040 get_res = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetDevResource", &p, 12040, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_res = reinterpret_cast<PFN_cuCtxGetDevResource_v12040>(p);
    cudaGetLastError();
  });
  if (!get_cur || !get_res) return 0;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  CUdevResource r{};
  if (get_res(ctx, &r, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return 0;
  return int(r.sm.smCount);
}
}  // namespace

// SMs the persistent kernels may size their grids for: the device's, or the
// current context's SM resource where that is smaller.  (An MPS client's
// thread-percentage limit is not visible here; the kernels' bounded waits
// and the device error word cover that case.)
int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 148;
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 148;
    }
    cached[dev] = n;
  }
  const int c = context_sm_count();
  return c > 0 && c < cached[dev] ? c : cached[dev];
}

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

bool lora_shape_ok(int64_t M, int64_t d_in, int64_t d_out, int64_t rank, int dtype) {
  if (M < 0 || d_in < 1 || d_out < 1 || rank < 0 || rank > 256) return false;
  if (d_in % 8 || d_out % 8 || rank % 8) return false;
  if (dtype != UNO_F32 && dtype != UNO_BF16) return false;
  if (M > (int64_t(1) << 31) - 1 || d_in > (int64_t(1) << 31) - 1 || d_out > (int64_t(1) << 31) - 1)
    return false;
  return true;
}

}  // namespace

bool verify_shape_ok(int64_t Bn, int64_t K, int64_t Kp, int64_t V) {
  if (Bn < 0 || K < 0 || K > 256 || V < 1 || V >= (int64_t(1) << 31)) return false;
  if (Kp != K && Kp != K + 1) return false;
  if (Kp < 1) return false;
  if (Bn > (int64_t(1) << 24)) return false;
  return true;
}

}  // namespace uno

using namespace uno;

extern "C" {

int uno_version(void) { return 100; }

const char* uno_status_string(int code) {
  switch (code) {
    case UNO_OK: return "ok";
    case UNO_ERR_ARG: return "invalid argument (null pointer, bad size or unsupported shape)";
    case UNO_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
    case UNO_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case UNO_ERR_WORKSPACE: return "workspace too small or misaligned";
    case UNO_ERR_CUDA: return "CUDA runtime or driver call failed";
    default: return "unknown status";
  }
}

size_t uno_gated_lora_linear_workspace(int64_t M, int64_t d_in, int64_t d_out, int64_t rank,
                                       int dtype) {
  if (!lora_shape_ok(M, d_in, d_out, rank, dtype)) return 0;
  uno_lora_problem p{};
  p.d_in = d_in;
  p.d_out = d_out;
  p.rank = rank;
  return lora_group_workspace_bytes(1, &p, M, dtype, sm_count());
}

int uno_gated_lora_linear(const void* x, const void* W, const void* A, const void* B,
                          const uint8_t* gate, int64_t M, int64_t d_in, int64_t d_out,
                          int64_t rank, float alpha, int dtype, void* y, void* workspace,
                          size_t ws_bytes, uno_stream_t stream) {
  uno_lora_problem p{};
  p.x = x;
  p.W = W;
  p.A = A;
  p.B = B;
  p.gate = gate;
  p.y = y;
  p.d_in = d_in;
  p.d_out = d_out;
  p.rank = rank;
  p.alpha = alpha;
  return uno_gated_lora_linear_batched(1, &p, M, dtype, workspace, ws_bytes, stream);
}

size_t uno_gated_lora_linear_batched_workspace(int n, const uno_lora_problem* problems, int64_t M,
                                               int dtype) {
  if (n < 1 || n > UNO_MAX_LORA_PROBLEMS || !problems) return 0;
  for (int i = 0; i < n; ++i)
    if (!lora_shape_ok(M, problems[i].d_in, problems[i].d_out, problems[i].rank, dtype)) return 0;
  return lora_group_workspace_bytes(n, problems, M, dtype, sm_count());
}

int uno_lora_plan_check(int n, const uno_lora_problem* problems, int64_t M, int dtype, int sms) {
  if (dtype != UNO_F32 && dtype != UNO_BF16) return UNO_ERR_UNSUPPORTED;
  if (n < 1 || n > UNO_MAX_LORA_PROBLEMS || !problems || sms < 1 || M < 1) return UNO_ERR_ARG;
  for (int i = 0; i < n; ++i)
    if (!lora_shape_ok(M, problems[i].d_in, problems[i].d_out, problems[i].rank, dtype))
      return UNO_ERR_ARG;
  return lora_plan_check(n, problems, M, dtype, sms);
}

int uno_gated_lora_linear_batched(int n, const uno_lora_problem* problems, int64_t M, int dtype,
                                  void* workspace, size_t ws_bytes, uno_stream_t stream) {
  if (dtype != UNO_F32 && dtype != UNO_BF16) return UNO_ERR_UNSUPPORTED;
  if (n < 1 || n > UNO_MAX_LORA_PROBLEMS || !problems) return UNO_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    const uno_lora_problem& p = problems[i];
    if (!lora_shape_ok(M, p.d_in, p.d_out, p.rank, dtype)) return UNO_ERR_ARG;
    if (!(p.alpha == p.alpha) || p.alpha == INFINITY || p.alpha == -INFINITY) return UNO_ERR_ARG;
  }
  if (M == 0) return UNO_OK;
  for (int i = 0; i < n; ++i) {
    const uno_lora_problem& p = problems[i];
    if (!p.x || !p.W || !p.gate || !p.y) return UNO_ERR_ARG;
    if (p.rank > 0 && (!p.A || !p.B)) return UNO_ERR_ARG;
    if (!aligned16(p.x) || !aligned16(p.W) || !aligned16(p.y) ||
        (p.rank > 0 && (!aligned16(p.A) || !aligned16(p.B))))
      return UNO_ERR_ALIGN;
  }
  if (!workspace) return UNO_ERR_ARG;
  if (!aligned256(workspace)) return UNO_ERR_WORKSPACE;
  return launch_lora_group(n, problems, M, dtype, workspace, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream));
}

size_t uno_verify_block_workspace(int64_t Bn, int64_t K, int64_t Kp, int64_t V) {
  if (!verify_shape_ok(Bn, K, Kp, V)) return 0;
  return plan_verify(Bn, K, Kp, V, sm_count()).bytes;
}

int uno_verify_block(const float* p_logits, const float* q_logits, const int32_t* draft,
                     const float* u_accept, const float* u_resample, int64_t Bn, int64_t K,
                     int64_t Kp, int64_t V, int32_t* n_accepted, int32_t* out_tokens,
                     int32_t* n_emitted, int32_t* status, void* workspace, size_t ws_bytes,
                     uno_stream_t stream) {
  if (!verify_shape_ok(Bn, K, Kp, V)) return UNO_ERR_ARG;
  if (Bn == 0) return UNO_OK;
  if (!p_logits || !u_resample || !n_accepted || !out_tokens || !n_emitted || !status || !workspace)
    return UNO_ERR_ARG;
  if (K > 0 && (!q_logits || !draft || !u_accept)) return UNO_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(p_logits) | reinterpret_cast<uintptr_t>(q_logits) |
       reinterpret_cast<uintptr_t>(u_resample) | reinterpret_cast<uintptr_t>(u_accept)) & 3u)
    return UNO_ERR_ALIGN;
  if (!aligned256(workspace)) return UNO_ERR_WORKSPACE;
  const VerifyPlan pl = plan_verify(Bn, K, Kp, V, sm_count());
  if (ws_bytes < pl.bytes) return UNO_ERR_WORKSPACE;
  const cudaError_t e = launch_verify(p_logits, q_logits, draft, u_accept, u_resample, Bn, K, Kp, V,
                                      n_accepted, out_tokens, n_emitted, status, workspace, pl,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}

int uno_verify_block_ex(const float* p_logits, const float* q_logits, const int32_t* draft,
                        const float* u_accept, const float* u_resample, int64_t Bn, int64_t K,
                        int64_t Kp, int64_t V, float temperature, int resample,
                        int32_t* n_accepted, int32_t* out_tokens, int32_t* n_emitted,
                        int32_t* status, void* workspace, size_t ws_bytes, uno_stream_t stream) {
  if (!(temperature > 0.0f) || !(temperature < INFINITY)) return UNO_ERR_ARG;
  if (resample != UNO_RESAMPLE_RACE && resample != UNO_RESAMPLE_INVERSE_CDF) return UNO_ERR_ARG;
  if (!verify_shape_ok(Bn, K, Kp, V)) return UNO_ERR_ARG;
  if (Bn == 0) return UNO_OK;
  if (!p_logits || !u_resample || !n_accepted || !out_tokens || !n_emitted || !status || !workspace)
    return UNO_ERR_ARG;
  if (K > 0 && (!q_logits || !draft || !u_accept)) return UNO_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(p_logits) | reinterpret_cast<uintptr_t>(q_logits) |
       reinterpret_cast<uintptr_t>(u_resample) | reinterpret_cast<uintptr_t>(u_accept)) & 3u)
    return UNO_ERR_ALIGN;
  if (!aligned256(workspace)) return UNO_ERR_WORKSPACE;
  const VerifyPlan pl = plan_verify(Bn, K, Kp, V, sm_count());
  if (ws_bytes < pl.bytes) return UNO_ERR_WORKSPACE;
  // logits are scaled by 1/T in fp32 (exact for T == 1)
  const float inv_t = temperature == 1.0f ? 1.0f : 1.0f / temperature;
  const cudaError_t e = launch_verify(p_logits, q_logits, draft, u_accept, u_resample, Bn, K, Kp, V,
                                      n_accepted, out_tokens, n_emitted, status, workspace, pl,
                                      reinterpret_cast<cudaStream_t>(stream), inv_t, resample);
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}

namespace {
bool lm_shape_ok(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int64_t d, int mode) {
  if (!verify_shape_ok(Bn, K, Kp, V)) return false;
  if (d < 8 || d % 8 || V % 8 || d > (int64_t(1) << 31) - 1) return false;
  if (mode < UNO_LM_AUTO || mode > UNO_LM_STATS_RECOMPUTE) return false;
  if (Bn * (Kp + K) > (int64_t(1) << 31) - 1) return false;
  return true;
}
}  // namespace

size_t uno_lm_head_verify_workspace(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int64_t d,
                                    int mode) {
  if (!lm_shape_ok(Bn, K, Kp, V, d, mode) || Bn == 0) return 0;
  return plan_lm_head(Bn, K, Kp, V, d, mode, sm_count()).bytes;
}

int uno_lm_head_verify(const void* h, const void* W, const int32_t* draft, const float* u_accept,
                       const float* u_resample, int64_t Bn, int64_t K, int64_t Kp, int64_t V,
                       int64_t d, int mode, int32_t* n_accepted, int32_t* out_tokens,
                       int32_t* n_emitted, int32_t* status, void* workspace, size_t ws_bytes,
                       uno_stream_t stream) {
  if (!lm_shape_ok(Bn, K, Kp, V, d, mode)) return UNO_ERR_ARG;
  if (Bn == 0) return UNO_OK;
  if (!h || !W || !u_resample || !n_accepted || !out_tokens || !n_emitted || !status || !workspace)
    return UNO_ERR_ARG;
  if (K > 0 && (!draft || !u_accept)) return UNO_ERR_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(u_resample) ||
      (reinterpret_cast<uintptr_t>(u_accept) & 3u))
    return UNO_ERR_ALIGN;
  if (!aligned256(workspace)) return UNO_ERR_WORKSPACE;
  const LmPlan L = plan_lm_head(Bn, K, Kp, V, d, mode, sm_count());
  if (ws_bytes < L.bytes) return UNO_ERR_WORKSPACE;
  return launch_lm_head_verify(h, W, draft, u_accept, u_resample, Bn, K, Kp, V, d, n_accepted,
                               out_tokens, n_emitted, status, workspace, ws_bytes, L,
                               reinterpret_cast<cudaStream_t>(stream));
}

size_t uno_tree_verify_workspace(int64_t Bn, int64_t N, int64_t V) {
  if (Bn < 0 || Bn > (int64_t(1) << 24) || N < 0 || N > kTreeMaxNodes || V < 1 ||
      V >= (int64_t(1) << 31))
    return 0;
  return plan_verify(Bn, 0, N + 1, V, sm_count()).bytes;
}

int uno_tree_verify(const float* logits, const int32_t* parent, const int32_t* token,
                    const float* u_accept, const float* u_resample, int64_t Bn, int64_t N,
                    int64_t V, int32_t* n_accepted, int32_t* path, int32_t* out_tokens,
                    int32_t* n_emitted, int32_t* status, void* workspace, size_t ws_bytes,
                    uno_stream_t stream) {
  if (Bn < 0 || Bn > (int64_t(1) << 24) || N < 0 || N > kTreeMaxNodes || V < 1 ||
      V >= (int64_t(1) << 31))
    return UNO_ERR_ARG;
  if (Bn == 0) return UNO_OK;
  if (!logits || !parent || !token || !u_accept || !u_resample || !n_accepted ||
      (N > 0 && !path) || !out_tokens || !n_emitted || !status || !workspace)
    return UNO_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(u_resample) |
       reinterpret_cast<uintptr_t>(u_accept)) & 3u)
    return UNO_ERR_ALIGN;
  if (!aligned256(workspace)) return UNO_ERR_WORKSPACE;
  const VerifyPlan pl = plan_verify(Bn, 0, N + 1, V, sm_count());
  if (ws_bytes < pl.bytes) return UNO_ERR_WORKSPACE;
  const cudaError_t e = launch_tree_verify(logits, parent, token, u_accept, u_resample, Bn, N, V,
                                           n_accepted, path, out_tokens, n_emitted, status,
                                           workspace, pl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}

int uno_draft_sample(const float* logits, const float* u, int64_t R, int64_t V, int32_t* tokens,
                     int32_t* status, uno_stream_t stream) {
  if (R < 0 || V < 1 || V >= (int64_t(1) << 31) || R >= (int64_t(1) << 31)) return UNO_ERR_ARG;
  if (R == 0) return UNO_OK;
  if (!logits || !u || !tokens || !status) return UNO_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(u)) & 3u)
    return UNO_ERR_ALIGN;
  const cudaError_t e =
      launch_draft_sample(logits, u, R, V, tokens, status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}

int uno_device_error(int reset) { return read_device_error(reset); }

}  // extern "C"
