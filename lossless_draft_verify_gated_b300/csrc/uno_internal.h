// uno_internal.h -- declarations shared by the C-ABI layer (api.cu) and the
// kernel translation units.  Not installed; the public surface is include/uno.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "uno.h"

namespace uno {

// Number of SMs of the current device (cached per device); 148 when no
// device can be queried (workspace queries on a machine without a GPU).
int sm_count();

// Rounds n up to a multiple of a (a power of two).
inline size_t align_up(size_t n, size_t a) { return (n + a - 1) & ~(a - 1); }

// ---------------------------------------------------------------- verifier
struct VerifyPlan {
  int64_t rows;      // Bn * (Kp + K): AR rows then draft rows of each sequence
  int splits;        // vocab chunks per row in the statistics pass
  int64_t chunk;     // elements per chunk (multiple of 4)
  int race_splits;   // vocab chunks per sequence in the resampling race
  int64_t race_chunk;
  size_t off_stats, off_gather, off_race, off_count, bytes;
};
VerifyPlan plan_verify(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int sms);

cudaError_t launch_verify(const float* p, const float* q, const int32_t* draft,
                          const float* u_acc, const float* u_res, int64_t Bn,
                          int64_t K, int64_t Kp, int64_t V, int32_t* n_acc,
                          int32_t* out_tokens, int32_t* n_emit, int32_t* status,
                          void* ws, const VerifyPlan& plan, cudaStream_t st,
                          float inv_t = 1.0f, int mode = 0);  // 1/temperature, UNO_RESAMPLE_*

cudaError_t launch_draft_sample(const float* logits, const float* u, int64_t R,
                                int64_t V, int32_t* tokens, int32_t* status,
                                cudaStream_t st);

// -------------------------------------------------------------- projection
constexpr int kMaxLoraProblems = UNO_MAX_LORA_PROBLEMS;
size_t lora_group_workspace_bytes(int n, const uno_lora_problem* pr, int64_t M, int dtype, int sms);
int launch_lora_group(int n, const uno_lora_problem* pr, int64_t M, int dtype, void* ws,
                      size_t ws_bytes, cudaStream_t st);
int lora_plan_check(int n, const uno_lora_problem* pr, int64_t M, int dtype, int sms);

}  // namespace uno
