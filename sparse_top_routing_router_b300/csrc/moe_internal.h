// Internal interfaces between the C-ABI layer (abi.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda_bf16.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"

namespace moe {

// Error reporting shared by every entry point (defined in abi.cu): fail() records the
// text that moe_last_error_detail() returns to this thread and passes `code` through;
// ok() clears it and returns MOE_OK.
int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int ok();
int cuda_fail(cudaError_t e, const char* what);

// An NVTX range named after the entry point around each compute call, so a profiler can
// group the kernels of one call (host-side only; a no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kMaxE = 512;
constexpr int kMaxK = 32;
constexpr size_t kWsHeader = 256;     // status word + padding
constexpr int kDispatchChunk = 256;   // tokens per dispatch CTA
constexpr int kGridSms = 148;         // B300 SMs: sizes the grids of the small-batch splits

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The router's reduction over H is split into S slices.  On the CUDA cores the split
// gives a small batch enough CTAs; on the tensor cores it also bounds the length of each
// fp32 accumulation chain to kRouterTcMaxK products (the MMA accumulator's rounding error
// grows with the chain).  Each CUDA-core slice leaves an fp32 (hi, lo) partial per (token,
// expert), each tensor-core slice a plain fp32 one (so up to 2 (cap - 1) of them fit
// behind slice 0); a reduce kernel adds the S partials in slice order.
constexpr int kRouterTcMaxK = 3072;
inline int router_split_cap(int T, int H) {      // sizes the workspace
  int s = 1;
  if (T > 0 && T < 16384) s = 16384 / T < 2 ? 2 : 16384 / T;
  const int tc = (3 * H + kRouterTcMaxK - 1) / kRouterTcMaxK;
  if (tc > s) s = tc;
  return s > 64 ? 64 : s;
}
// Tensor-core router with at most 128 experts: the three W_g pieces of a 64-wide block of
// H share one X box, so a k-block carries 3 * 64 products (else 64 of the [X, X, X] row).
inline bool router_tc_fused(int E) { return E <= 128; }
inline int router_splits(int T, int H) {          // CUDA-core logits
  const int s = router_split_cap(T, H);
  const int max_by_h = H / 128 > 0 ? H / 128 : 1;
  return s < max_by_h ? s : max_by_h;
}

// Workspace layout, shared by every call of one forward (each region's offset depends
// only on arguments every call that uses it receives):
//   [0, 256)              status word (int32 at 0), rows re-decided by the last router
//                         call (int32 at 4), padding
//   router partial logits S*T*E float2 (S <= router_split_cap(T, H))
//   router refine list    T int4 (rows listed for exact re-decision: t, band limits)
//   router weight pieces  E * 3H bf16 (tensor-core router: W_g split into hi, mid, lo)
//   dispatch chunk table  2 * nchunks * E int32
//   expert activations h  (T*k + T) * I elements (bf16, or fp32 for the fp32 path)
struct WsLayout {
  size_t logits, refine, wsplit, chunk_counts, chunk_base, h;
  // expert-choice routing: affinities by column, exact affinities of listed tokens,
  // token flags and lists, column list and limits, counters
  size_t ec_st, ec_exs, ec_need, ec_tok, ec_col, ec_info, ec_ctr;
  size_t total;
};

inline WsLayout ws_layout(int T, int H, int E, int I, int k, int dtype, int has_shared) {
  WsLayout L;
  size_t off = kWsHeader;
  L.logits = off;
  off = align_up(off + (size_t)router_split_cap(T, H) * T * E * 8, 256);
  L.refine = off;
  off = align_up(off + (size_t)T * 16, 256);
  L.wsplit = off;
  off = align_up(off + (size_t)E * 3 * H * 2, 256);
  const size_t nchunks = ((size_t)T + kDispatchChunk - 1) / kDispatchChunk;
  L.chunk_counts = off;
  off = align_up(off + nchunks * E * 4, 256);
  L.chunk_base = off;
  off = align_up(off + nchunks * E * 4, 256);
  L.ec_st = off;
  off = align_up(off + (size_t)T * E * 4, 256);
  L.ec_exs = off;
  off = align_up(off + (size_t)T * E * 8, 256);
  L.ec_need = off;
  off = align_up(off + (size_t)T * 4, 256);
  L.ec_tok = off;
  off = align_up(off + (size_t)T * 4, 256);
  L.ec_col = off;
  off = align_up(off + (size_t)E * 4, 256);
  L.ec_info = off;
  off = align_up(off + (size_t)E * 16, 256);
  L.ec_ctr = off;
  off = align_up(off + 16, 256);
  L.h = off;   // last: the only region whose size depends on I
  const size_t rows = (size_t)T * k + (has_shared ? (size_t)T : 0);
  off = align_up(off + rows * I * (dtype == MOE_DTYPE_BF16 ? 2 : 4), 256);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------- launch helpers
struct RouterArgs {
  int T, H, E, k, score, renorm, x_dtype;
  int n_groups, topk_groups;   // group-limited routing (n_groups > 1), else 0
  const void* X;
  const float* Wg;
  const float* bias;
  const float* logit_bias;
  float2* logits;      // workspace [S, T, E] (hi, lo) partial sums; slice 0 the result
  float* logits_part;  // tensor-core split-K: fp32 partials [S, T, E] after slice 0, or null
  int splits;          // S
  __nv_bfloat16* wsplit;   // tensor-core router: W_g as [E][3H] bf16 pieces, else null
  float eps_rel;       // fp32 logit error bound per unit of max(1, max|l|) * sqrt(H/1024)
  int num_sms;
  unsigned long long wait_limit_ns;
  int32_t* idx;
  float* gate;
  float* gap;
  double* colsum;
  int* status;
  int* refined;        // counter of rows re-decided from exact dot products
  int4* refine_list;   // [T] (t, lower band limit, sure limit, 0) of those rows, or
                       // (t, candidate group mask, fp32 group margin, 1) when group-limited
};
cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t s);
// Tensor-core router logits (x bf16, E % 8 == 0, H % 64 == 0, T >= 256): splits W_g into bf16
// pieces in a.wsplit, then one GEMM [T, 3H] x [3H, E] with split-K partials.
typedef CUresult (*EncodeTiledFnR)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
cudaError_t launch_router_split(const RouterArgs& a, cudaStream_t s);
cudaError_t launch_router_tc(const RouterArgs& a, EncodeTiledFnR enc, bool* encode_failed,
                             cudaStream_t s);
cudaError_t launch_router_select(const RouterArgs& a, cudaStream_t s);
// sums split-K partial logits into slot 0 (a.splits > 1); returns the args with splits = 1
cudaError_t launch_router_reduce(RouterArgs& a, cudaStream_t s);

// Expert-choice routing: every expert takes the C tokens of largest affinity.
constexpr int kEcMaxT = 32768;   // one expert's column of keys sits in shared memory
struct ExpertChoiceArgs {
  RouterArgs r;        // logits (reduced), shapes, X, W_g, logit offset, error bound
  int C;
  float* St;           // [E][T] fp32 affinities, one column per expert
  double* exS;         // [T][E] exact affinities of the listed tokens
  int* need;           // [T] 1 = the token's exact affinities are needed
  int* tok_list;       // [T] those tokens
  int* col_list;       // [E] experts whose choice waits for exact affinities
  int4* col_info;      // [E] (band low, band high, fp32 margin, 0) of those experts
  int* ctr;            // [0] listed tokens, [1] listed experts, [2] max rel err, [3] max abs err
  int32_t* offsets;    // [E+1]
  int32_t* row_of_slot;  // [T*E], slot t*E + e
  int32_t* slot_of_row;  // [E*C]
  float* gate;         // [T*E]
  float* gap;          // [E] nullable
};
cudaError_t launch_expert_choice(const ExpertChoiceArgs& a, cudaStream_t s);

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
// Xperm[r] = X[slot_of_row[r] / k] for r < R (one warp per row)
cudaError_t launch_gather_rows(int R, int k, int row_bytes, const int32_t* slot_of_row,
                               const void* X, void* Xperm, int* status, int T,
                               cudaStream_t s);

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
// FP8 (E4M3) weights with per-output-channel fp32 scales: CUDA-core GEMVs for
// decode-sized batches (bf16 activations).
struct Fp8Args {
  int T, H, E, I, k, has_shared;
  const void* X;
  const void* Xperm;
  const int32_t* offsets;
  const uint8_t *Q_gate, *Q_up, *Q_down;      // [E][I][H], [E][I][H], [E][H][I] codes
  const float *S_gate, *S_up, *S_down;        // [E][I], [E][I], [E][H] scales
  const uint8_t *Qs_gate, *Qs_up, *Qs_down;   // shared expert
  const float *Ss_gate, *Ss_up, *Ss_down;
  void* h;
  float* O;
  float* O_shared;
  int* status;
};
cudaError_t launch_quantize_fp8_rows(int rows, int cols, int w_dtype, const void* W,
                                     uint8_t* q, float* scale, cudaStream_t s);
// TMA-fed: `encode` is the driver's cuTensorMapEncodeTiled (cudaErrorInvalidValue with
// *encode_failed set when a tensor map cannot be encoded); waits give up after
// wait_limit_ns.
cudaError_t launch_expert_gate_up_fp8(const Fp8Args& a, EncodeTiledFn encode,
                                      bool* encode_failed, unsigned long long wait_limit_ns,
                                      cudaStream_t s);
cudaError_t launch_expert_down_fp8(const Fp8Args& a, EncodeTiledFn encode, bool* encode_failed,
                                   unsigned long long wait_limit_ns, cudaStream_t s);
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

struct BiasArgs {
  int E;
  long long slots;   // T * k
  const int32_t* counts;
  float gamma;
  float* bias;
};
cudaError_t launch_bias_update(const BiasArgs& a, cudaStream_t s);

}  // namespace moe
