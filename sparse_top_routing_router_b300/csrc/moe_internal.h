// Internal interfaces between the C-ABI layer (abi.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxE = 512;
constexpr int kMaxK = 32;
constexpr size_t kWsHeader = 256;     // status word + padding
constexpr int kDispatchChunk = 256;   // tokens per dispatch CTA

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout, shared by every call of one forward:
//   [0, 256)              status word (int32) + padding
//   router logits         T*E fp32
//   dispatch chunk table  2 * nchunks * E int32
//   expert activations h  (T*k + T) * I elements (bf16, or fp32 for the fp32 path)
struct WsLayout {
  size_t logits, chunk_counts, chunk_base, h, total;
};

inline WsLayout ws_layout(int T, int H, int E, int I, int k, int dtype, int has_shared) {
  (void)H;
  WsLayout L;
  size_t off = kWsHeader;
  L.logits = off;
  off = align_up(off + (size_t)T * E * 4, 256);
  const size_t nchunks = ((size_t)T + kDispatchChunk - 1) / kDispatchChunk;
  L.chunk_counts = off;
  off = align_up(off + nchunks * E * 4, 256);
  L.chunk_base = off;
  off = align_up(off + nchunks * E * 4, 256);
  L.h = off;
  const size_t rows = (size_t)T * k + (has_shared ? (size_t)T : 0);
  off = align_up(off + rows * I * (dtype == MOE_DTYPE_BF16 ? 2 : 4), 256);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------- launch helpers
struct RouterArgs {
  int T, H, E, k, score, renorm, x_dtype;
  const void* X;
  const float* Wg;
  const float* bias;
  const float* logit_bias;
  float* logits;       // workspace [T, E]
  int32_t* idx;
  float* gate;
  float* gap;
  double* colsum;
  int* status;
};
cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t s);
cudaError_t launch_router_select(const RouterArgs& a, cudaStream_t s);

struct DispatchArgs {
  int T, k, E, H, x_dtype, capacity;
  const int32_t* idx;
  const void* X;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_of_slot;
  int32_t* slot_of_row;
  void* Xperm;
  int32_t* chunk_counts;
  int32_t* chunk_base;
  int* status;
};
cudaError_t launch_dispatch_count(const DispatchArgs& a, cudaStream_t s);
cudaError_t launch_dispatch_scan(const DispatchArgs& a, cudaStream_t s);
cudaError_t launch_dispatch_scatter(const DispatchArgs& a, cudaStream_t s);
cudaError_t launch_dispatch_gather(const DispatchArgs& a, cudaStream_t s);

struct ExpertArgs {
  int T, H, E, I, k, has_shared, num_sms;
  const void* X;
  const void* Xperm;
  const int32_t* offsets;
  const void* W_gate;
  const void* W_up;
  const void* W_down;
  const void* Ws_gate;
  const void* Ws_up;
  const void* Ws_down;
  void* h;            // workspace [(T*k + T), I]
  float* O;
  float* O_shared;
  int* status;
  int test_hook;                  // MOE_TEST_HOOK_* (0 in normal use)
  unsigned long long wait_limit_ns;
};
// bf16 tensor-core path.  `encode` is the driver's cuTensorMapEncodeTiled.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
// Returns cudaErrorInvalidValue (with *encode_failed set) when a tensor map cannot be
// encoded.
cudaError_t launch_expert_gate_up_tc(const ExpertArgs& a, EncodeTiledFn encode,
                                     bool* encode_failed, cudaStream_t s);
cudaError_t launch_expert_down_tc(const ExpertArgs& a, EncodeTiledFn encode,
                                  bool* encode_failed, cudaStream_t s);
// fp32 CUDA-core path.
cudaError_t launch_expert_gate_up_f32(const ExpertArgs& a, cudaStream_t s);
cudaError_t launch_expert_down_f32(const ExpertArgs& a, cudaStream_t s);

struct CombineArgs {
  int T, k, H;
  const float* O;
  const float* O_shared;
  const int32_t* row_of_slot;
  const float* gate;
  float* Y;
  void* Y_bf16;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

struct StatsArgs {
  int T, k, E;
  const int32_t* counts;
  const int32_t* offsets;
  const double* colsum;
  double alpha;
  double* f;
  double* p;
  double* out;
};
cudaError_t launch_balance_stats(const StatsArgs& a, cudaStream_t s);

}  // namespace moe
