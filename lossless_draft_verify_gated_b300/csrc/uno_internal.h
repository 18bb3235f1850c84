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
// Sizes every verifier entry point accepts (include/uno.h): K <= 256,
// Kp in {K, K+1} with Kp >= 1, 1 <= V < 2^31, 0 <= Bn <= 2^24.
bool verify_shape_ok(int64_t Bn, int64_t K, int64_t Kp, int64_t V);

struct VerifyPlan {
  int64_t rows;      // Bn * (Kp + K): AR rows then draft rows of each sequence
  int stats_cps;     // statistics CTAs per SM (the kernel's occupancy and load depth)
  int splits;        // vocab chunks per row in the statistics pass
  int64_t chunk;     // elements per chunk (multiple of 4)
  int race_splits;   // vocab chunks per sequence in the resampling race
  int64_t race_chunk;
  int icdf_splits;   // the same for the inverse-CDF resample (smaller chunks: the
  int64_t icdf_chunk;  // last CTA searches one of them for the crossing)
  size_t off_stats, off_gather, off_race, off_count, bytes;
};
VerifyPlan plan_verify(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int sms);

cudaError_t launch_verify(const float* p, const float* q, const int32_t* draft,
                          const float* u_acc, const float* u_res, int64_t Bn,
                          int64_t K, int64_t Kp, int64_t V, int32_t* n_acc,
                          int32_t* out_tokens, int32_t* n_emit, int32_t* status,
                          void* ws, const VerifyPlan& plan, cudaStream_t st,
                          float inv_t = 1.0f, int mode = 0);  // 1/temperature, UNO_RESAMPLE_*

// The statistics pass alone over the rows of a plan (Bn sequences of Kp rows
// of p then K rows of q); K = 0 gives plain per-row (max, sum exp) partials.
// It zeroes each sequence's arrival count and, when `keys` is given, the two
// race-winner keys at keys[b * key_stride] for the race that follows.
cudaError_t launch_row_stats(const float* p, const float* q, const int32_t* draft, int64_t Bn,
                             int64_t K, int64_t Kp, int64_t V, const VerifyPlan& pl, void* ws,
                             cudaStream_t st, unsigned long long* keys = nullptr, int key_stride = 0);

// ------------------------------------------------------------ tree sampler
constexpr int64_t kTreeMaxNodes = 255;  // drafted nodes per sequence (N); N + 1 rows
cudaError_t launch_tree_verify(const float* logits, const int32_t* parent, const int32_t* token,
                               const float* u_acc, const float* u_res, int64_t Bn, int64_t N,
                               int64_t V, int32_t* n_acc, int32_t* path, int32_t* out_tokens,
                               int32_t* n_emit, int32_t* status, void* ws, const VerifyPlan& pl,
                               cudaStream_t st);

cudaError_t launch_draft_sample(const float* logits, const float* u, int64_t R,
                                int64_t V, int32_t* tokens, int32_t* status,
                                cudaStream_t st);

// -------------------------------------------------------------- projection
constexpr int kMaxLoraProblems = UNO_MAX_LORA_PROBLEMS;
size_t lora_group_workspace_bytes(int n, const uno_lora_problem* pr, int64_t M, int dtype, int sms);
int launch_lora_group(int n, const uno_lora_problem* pr, int64_t M, int dtype, void* ws,
                      size_t ws_bytes, cudaStream_t st);
int lora_plan_check(int n, const uno_lora_problem* pr, int64_t M, int dtype, int sms);

// Epilogue options of the projection kernel for internal callers (the LM head
// feeding the verifier): fp32 output from bf16 operands, and the statistics
// epilogue of logit rows (per row and vocabulary tile the (max, sum exp) of
// the tile's logits, plus each row's drafted-token logit), with or without
// the logits themselves stored.
struct LinearEpilogue {
  int f32out;         // y as fp32
  int stats;          // statistics epilogue (one problem, rank 0)
  int stats_store;    // (stats) also store y
  int64_t K, Kp;      // AR rows per sequence (Kp) and draft rows per sequence (K)
  int64_t Rp;         // AR rows of the launch: rows [0, Rp) are AR rows b*Kp + j,
                      // rows Rp + b*K + i are draft rows
  int nvt;            // vocabulary tiles per row (logit_gemm_tiles)
  const int32_t* draft;  // [sequences, K]
  float2* part;       // [rows, nvt]
  float* gathered;    // [rows]
};
// One bf16 GEMM y[M, V] = h[M, d] . W[V, d]^T with the given epilogue.
int launch_logit_gemm(const uno_lora_problem& pr, int64_t M, void* ws, size_t ws_bytes,
                      cudaStream_t st, const LinearEpilogue& epi);
// Vocabulary tiles per row of that GEMM's schedule (the statistics partials per row).
int logit_gemm_tiles(int64_t M, int64_t d, int64_t V, int sms);

// -------------------------------------------------------------- LM head
// Batches from which UNO_LM_AUTO takes the verifier's statistics in the head
// GEMM's epilogue (the logits are still stored, which the tensor-bound GEMM
// hides, and only the resampled rows are read back); below it, where the
// head's weights dominate the traffic, the plain path is as fast.
constexpr int64_t kLmStatsMinBatch = 8;

struct LmPlan {
  int mode;          // UNO_LM_PLAIN, UNO_LM_STATS_STORE or UNO_LM_STATS_RECOMPUTE
  int64_t rows;      // Bn * (Kp + K)
  int nvt;           // statistics partials per row
  int race_splits;
  int64_t race_chunk;
  VerifyPlan vplan;  // (plain) the verifier's own plan
  size_t gemm_bytes, gemm2_bytes;
  size_t off_gemm, off_logits, off_verify, off_part, off_gather, off_dec, off_race, off_count,
      off_hc, off_lc, off_gemm2, bytes;
};
LmPlan plan_lm_head(int64_t Bn, int64_t K, int64_t Kp, int64_t V, int64_t d, int mode, int sms);
int launch_lm_head_verify(const void* h, const void* W, const int32_t* draft, const float* u_acc,
                          const float* u_res, int64_t Bn, int64_t K, int64_t Kp, int64_t V,
                          int64_t d, int32_t* n_acc, int32_t* out_tokens, int32_t* n_emit,
                          int32_t* status, void* ws, size_t ws_bytes, const LmPlan& L,
                          cudaStream_t st);

}  // namespace uno
