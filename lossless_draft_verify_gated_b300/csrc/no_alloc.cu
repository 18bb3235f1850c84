// no_alloc.cu -- the block verifier for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a plugin or custom op inside
// another inference runtime that is given only its input and output buffers, a
// serving loop whose memory is owned by a framework pool it may not grow, or code
// running under rules that forbid cudaMalloc on the request path.  For them this
// entry point runs the same verifier kernels with their scratch in a fixed,
// file-scope device array instead of a caller workspace.
//
// The array (kNoAllocScratchBytes) lives in every GPU that loads libuno.so until
// the process exits.  Its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on that
// device; make that first call before any stream capture.  Every call shares the
// array: calls that may overlap on the GPU (two streams, two threads) race on it
// and must be serialised by the caller.  The looked-up address belongs to the
// device's context of the time: after cudaDeviceReset the library must not be
// called again in the same process.  The only scratch that must start at zero
// (the per-sequence arrival counters) is cleared by the first kernel of each call;
// every other scratch word is written before it is read.
#include <mutex>

#include "uno_internal.h"

namespace uno {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace uno

using namespace uno;

extern "C" {

size_t uno_verify_block_no_alloc_max_scratch(void) { return kNoAllocScratchBytes; }

int uno_verify_block_no_alloc(const float* p_logits, const float* q_logits, const int32_t* draft,
                              const float* u_accept, const float* u_resample, int64_t Bn,
                              int64_t K, int64_t Kp, int64_t V, int32_t* n_accepted,
                              int32_t* out_tokens, int32_t* n_emitted, int32_t* status,
                              uno_stream_t stream) {
  if (!verify_shape_ok(Bn, K, Kp, V)) return UNO_ERR_ARG;
  if (Bn == 0) return UNO_OK;
  if (!p_logits || !u_resample || !n_accepted || !out_tokens || !n_emitted || !status)
    return UNO_ERR_ARG;
  if (K > 0 && (!q_logits || !draft || !u_accept)) return UNO_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(p_logits) | reinterpret_cast<uintptr_t>(q_logits) |
       reinterpret_cast<uintptr_t>(u_resample) | reinterpret_cast<uintptr_t>(u_accept)) & 3u)
    return UNO_ERR_ALIGN;
  const VerifyPlan pl = plan_verify(Bn, K, Kp, V, sm_count());
  if (pl.bytes > kNoAllocScratchBytes) return UNO_ERR_WORKSPACE;  // batch too large for the array
  void* ws = scratch_on_current_device();
  if (!ws) return UNO_ERR_CUDA;
  const cudaError_t e = launch_verify(p_logits, q_logits, draft, u_accept, u_resample, Bn, K, Kp, V,
                                      n_accepted, out_tokens, n_emitted, status, ws, pl,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? UNO_OK : UNO_ERR_CUDA;
}

}  // extern "C"
