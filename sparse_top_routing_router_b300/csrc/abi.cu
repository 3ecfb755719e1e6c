// The C ABI of libmoe.so (declared in include/moe.h): argument checks, workspace
// carving, kernel launches on the caller's stream, optional per-kernel event timing.
// Nothing here allocates device memory and nothing here synchronises, except
// moe_get_device_status and moe_ctx_trace_read, which are documented to.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "moe_internal.h"

using namespace moe;

namespace {
constexpr unsigned long long kWaitLimitDefaultNs = 2000000000ull;
// Error bounds the router's exactness guard assumes for its fp32 logits, per unit of
// max(1, max|l|) * sqrt(H/1024): CUDA-core logits sum 32-term fp32 blocks with
// compensation; tensor-core logits accumulate exact bf16 x bf16 products in the MMA's
// fp32 accumulator, chains of at most 3072 products.  They are empirical, not worst-case
// bounds: on the benchmarked shapes the GPU tests require the true error below a quarter
// of 2^-19 (CUDA cores) and of 2^-17 (tensor cores, half the bound used here), and
// measure at most 0.13 of those.
constexpr float kRouterEpsCuda = 1.9073486328125e-06f;     // 2^-19
constexpr float kRouterEpsTensor = 1.52587890625e-05f;     // 2^-16
}

namespace {
thread_local std::string g_detail;
}

namespace moe {

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_detail = buf;
  return code;
}

int ok() {
  g_detail.clear();
  return MOE_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace moe

struct moe_ctx {
  int device = 0;
  int num_sms = 0;
  EncodeTiledFn encode = nullptr;
  bool tracing = false;
  int test_hook = MOE_TEST_HOOK_NONE;
  unsigned long long wait_limit_ns = kWaitLimitDefaultNs;
  struct Rec {
    int id;
    int kernels;   // kernels the bracketed launch function enqueued
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  std::mutex mu;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaEvent_t take_event(moe_ctx* c) {
  if (!c->pool.empty()) {
    cudaEvent_t e = c->pool.back();
    c->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launches `fn` (which enqueues `kernels` kernels) with optional event bracketing on `s`.
template <typename F>
cudaError_t traced(moe_ctx* c, int id, cudaStream_t s, F&& fn, int kernels = 1) {
  if (!c->tracing) return fn();
  std::lock_guard<std::mutex> lk(c->mu);
  cudaEvent_t a = take_event(c), b = take_event(c);
  if (a) cudaEventRecord(a, s);
  cudaError_t e = fn();
  if (b) cudaEventRecord(b, s);
  if (a && b) c->recs.push_back({id, kernels, a, b});
  return e;
}

int check_ctx(moe_ctx* c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "ctx is null");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess)
    return fail(MOE_ERR_CUDA, "cudaGetDevice failed");
  if (dev != c->device)
    return fail(MOE_ERR_INVALID_ARG, "current device %d is not the context's device %d", dev,
                c->device);
  return MOE_OK;
}

int check_shape(int T, int E, int k) {
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
  if (E < 1 || E > kMaxE) return fail(MOE_ERR_UNSUPPORTED, "E = %d outside [1, %d]", E, kMaxE);
  if (k < 1 || k > E || k > kMaxK)
    return fail(MOE_ERR_UNSUPPORTED, "k = %d outside [1, min(E, %d)]", k, kMaxK);
  if ((long long)T * k > 0x7fffffffLL) return fail(MOE_ERR_UNSUPPORTED, "T*k exceeds int32");
  return MOE_OK;
}

// Router scoring shared by token-choice and expert-choice routing: fills the logits part
// of `a` (shapes, inputs, workspace pointers, split-K choice, error bound) and launches the
// logit kernels (traced as router_logits).  The caller has validated d and the buffers.
int router_logits_stage(moe_ctx* ctx, const moe_router_desc* d, const void* X,
                        const float* Wg, const float* logit_bias, void* ws, size_t ws_bytes,
                        const WsLayout& L, RouterArgs& a, cudaStream_t s) {
  // the tensor-core router also needs the W_g pieces; the fp32 CUDA-core one does not
  const bool use_tc = d->x_dtype == MOE_DTYPE_BF16 && d->E % 8 == 0 &&
                      d->H % 64 == 0 && d->T >= 256 && ws_bytes >= L.chunk_counts;
  a = RouterArgs{};
  a.T = d->T;
  a.H = d->H;
  a.E = d->E;
  a.k = d->k;
  a.score = d->score;
  a.renorm = d->renorm;
  a.x_dtype = d->x_dtype;
  a.X = X;
  a.Wg = Wg;
  a.logit_bias = logit_bias;
  a.logits = reinterpret_cast<float2*>(static_cast<char*>(ws) + L.logits);
  a.num_sms = ctx->num_sms;
  a.wait_limit_ns = ctx->wait_limit_ns;
  a.wsplit = use_tc ? reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + L.wsplit)
                    : nullptr;
  a.logits_part = nullptr;
  if (use_tc) {
    // Every slice at most kRouterTcMaxK products long.  Among the slice counts the
    // workspace holds, take the one with the least time per slice-wave: tiles * S work
    // units over num_sms CTAs take ceil(tiles * S / num_sms) rounds of 1/S of a tile each.
    const int tiles = ((d->T + 127) / 128) * ((d->E + 255) / 256);
    const bool fused = router_tc_fused(d->E);
    const int nkb = (fused ? 1 : 3) * d->H / 64;
    const int kb_chain = kRouterTcMaxK / (fused ? 3 * 64 : 64);   // k-blocks per chain
    const int need = (nkb + kb_chain - 1) / kb_chain;
    const int cap = router_split_cap(d->T, d->H);
    int hi = cap >= 2 ? 2 * (cap - 1) : 1;   // fp32 partials behind slice 0
    if (hi > nkb) hi = nkb;
    const int sms = ctx->num_sms > 0 ? ctx->num_sms : 1;
    int best = need > hi ? hi : need;
    double best_t = 1e30;
    for (int sp = best; sp <= hi; ++sp) {
      const double t = (double)((tiles * sp + sms - 1) / sms) / sp;
      if (t < best_t - 1e-12) {
        best_t = t;
        best = sp;
      }
    }
    a.splits = best;
    if (best > 1)
      a.logits_part = reinterpret_cast<float*>(a.logits + (size_t)d->T * d->E);
    a.eps_rel = kRouterEpsTensor;
  } else {
    a.splits = router_splits(d->T, d->H);
    a.eps_rel = kRouterEpsCuda;
  }
  a.status = static_cast<int*>(ws);
  a.refined = static_cast<int*>(ws) + 1;
  a.refine_list = reinterpret_cast<int4*>(static_cast<char*>(ws) + L.refine);
  cudaError_t e;
  if ((e = cudaMemsetAsync(a.refined, 0, sizeof(int), s))) return cuda_fail(e, "cudaMemsetAsync");
  if (use_tc) {
    bool bad = false;
    e = traced(ctx, MOE_K_ROUTER_LOGITS, s, [&] {
      cudaError_t r = launch_router_split(a, s);
      return r != cudaSuccess ? r : launch_router_tc(a, ctx->encode, &bad, s);
    }, 2);
    if (bad) return fail(MOE_ERR_INVALID_ARG, "tensor map encoding failed (router)");
    if (e) return cuda_fail(e, "router_logits launch");
  } else if ((e = traced(ctx, MOE_K_ROUTER_LOGITS, s,
                         [&] { return launch_router_logits(a, s); }))) {
    return cuda_fail(e, "router_logits launch");
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_version(void) { return 10400; }

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_INDEX: return "device index out of range";
    default: return "unknown status";
  }
}

// Text describing the last failure of a call made by this thread ("" after success).
const char* moe_last_error_detail(void) { return g_detail.c_str(); }

const char* moe_kernel_name(int id) {
  static const char* names[MOE_KERNEL_COUNT] = {
      "router_logits",    "router_select",    "dispatch_count", "dispatch_scan",
      "dispatch_scatter", "dispatch_gather",  "expert_gate_up", "expert_down",
      "combine",          "balance_stats",    "bias_update"};
  return (id >= 0 && id < MOE_KERNEL_COUNT) ? names[id] : "unknown";
}

int moe_ctx_create(moe_ctx** out, int device) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  int n = 0;
  cudaError_t e = cudaGetDeviceCount(&n);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device < 0 || device >= n)
    return fail(MOE_ERR_INVALID_ARG, "device %d outside [0, %d)", device, n);
  int sms = 0, major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return fail(MOE_ERR_CUDA, "cannot resolve cuTensorMapEncodeTiled");
  moe_ctx* c = new moe_ctx();
  c->device = device;
  c->num_sms = sms;
  c->encode = reinterpret_cast<EncodeTiledFn>(fn);
  *out = c;
  (void)major;
  (void)minor;
  return ok();
}

void moe_ctx_destroy(moe_ctx* c) {
  if (!c) return;
  for (auto& r : c->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : c->pool) cudaEventDestroy(e);
  delete c;
}

size_t moe_workspace_bytes(int T, int H, int E, int I, int k, int dtype, int has_shared) {
  if (T < 0 || H < 0 || E < 0 || I < 0 || k < 0) return 0;
  return ws_layout(T, H, E, I, k, dtype, has_shared).total;
}

int moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < kWsHeader) return fail(MOE_ERR_INVALID_ARG, "workspace too small");
  cudaError_t e = cudaMemsetAsync(ws, 0, kWsHeader, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "cudaMemsetAsync");
}

int moe_capacity(double c, int T, int k, int E) {
  if (!isfinite(c) || c < 0.0) return fail(MOE_ERR_INVALID_ARG, "capacity factor %g", c);
  if (T < 0 || k < 1 || E < 1) return fail(MOE_ERR_INVALID_ARG, "bad T/k/E");
  if (c == 0.0 || T == 0) return 0;
  // c = mant * 2^ex exactly
  int e2 = 0;
  const double f = frexp(c, &e2);                      // c = f * 2^e2, f in [0.5, 1)
  const unsigned long long mant = (unsigned long long)ldexp(f, 53);
  const int ex = e2 - 53;
  typedef unsigned __int128 u128;
  u128 num = (u128)mant * (u128)(unsigned)T * (u128)(unsigned)k;
  u128 q;
  if (ex >= 0) {
    // q = num * 2^ex.  E < 2^31, so any q >= 2^64 makes C > INT32_MAX: reject it before
    // the shift, which could otherwise wrap past 2^128 to a small (wrong) capacity.
    if (ex > 30 || (num >> (64 - ex)) != 0)
      return fail(MOE_ERR_INVALID_ARG, "capacity overflows");
    q = num << ex;
  } else {
    const int s = -ex;
    q = (s >= 127) ? (num > 0 ? 1 : 0) : ((num + (((u128)1 << s) - 1)) >> s);   // ceil
  }
  const u128 C = (q + (u128)(unsigned)E - 1) / (u128)(unsigned)E;           // ceil
  if (C > (u128)0x7fffffff) return fail(MOE_ERR_INVALID_ARG, "capacity overflows int32");
  g_detail.clear();
  return (int)C;
}

int moe_router_topk(moe_ctx* ctx, const moe_router_desc* d, const void* X, const float* Wg,
                    const float* bias, const float* logit_bias, int32_t* topk_idx,
                    float* topk_gate, float* key_gap, double* prob_colsum, void* ws,
                    size_t ws_bytes, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (!d) return fail(MOE_ERR_INVALID_ARG, "desc is null");
  int r = check_shape(d->T, d->E, d->k);
  if (r) return r;
  if (d->H < 1) return fail(MOE_ERR_INVALID_ARG, "H = %d", d->H);
  if (d->score != MOE_SCORE_SOFTMAX && d->score != MOE_SCORE_SIGMOID)
    return fail(MOE_ERR_INVALID_ARG, "score = %d", d->score);
  if (d->x_dtype != MOE_DTYPE_BF16 && d->x_dtype != MOE_DTYPE_F32)
    return fail(MOE_ERR_INVALID_ARG, "x_dtype = %d", d->x_dtype);
  // group-limited routing: n_groups <= 1, or every group allowed, is plain top-k
  int n_groups = d->n_groups, topk_groups = d->topk_groups;
  if (n_groups < 0 || topk_groups < 0)
    return fail(MOE_ERR_INVALID_ARG, "n_groups = %d, topk_groups = %d", n_groups, topk_groups);
  if (n_groups > 1) {
    if (n_groups > 32 || d->E % n_groups != 0)
      return fail(MOE_ERR_UNSUPPORTED, "n_groups = %d must divide E = %d and be <= 32",
                  n_groups, d->E);
    const int gs = d->E / n_groups;
    if (topk_groups < 1 || topk_groups > n_groups || d->k % topk_groups != 0 ||
        d->k / topk_groups > gs)
      return fail(MOE_ERR_INVALID_ARG,
                  "topk_groups = %d needs 1 <= topk_groups <= n_groups = %d, k = %d a "
                  "multiple of it and k / topk_groups <= E / n_groups = %d",
                  topk_groups, n_groups, d->k, gs);
    if (topk_groups == n_groups) n_groups = topk_groups = 0;
  } else {
    n_groups = topk_groups = 0;
  }
  if (d->T > 0 && (!X || !Wg || !topk_idx || !topk_gate))
    return fail(MOE_ERR_INVALID_ARG, "X, Wg, topk_idx and topk_gate are required");
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is null");
  if (!aligned16(X) || !aligned16(Wg) || !aligned16(ws))
    return fail(MOE_ERR_INVALID_ARG, "X, Wg and ws must be 16-byte aligned");
  const WsLayout L = ws_layout(d->T, d->H, d->E, 0, d->k, d->x_dtype, 0);
  if (ws_bytes < L.wsplit) return fail(MOE_ERR_INVALID_ARG, "workspace too small");
  if ((r = check_ctx(ctx))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (prob_colsum && (e = cudaMemsetAsync(prob_colsum, 0, sizeof(double) * d->E, s)))
    return cuda_fail(e, "cudaMemsetAsync");
  if (d->T == 0) return ok();
  RouterArgs a;
  if ((r = router_logits_stage(ctx, d, X, Wg, logit_bias, ws, ws_bytes, L, a, s))) return r;
  a.bias = bias;
  a.n_groups = n_groups;
  a.topk_groups = topk_groups;
  a.idx = topk_idx;
  a.gate = topk_gate;
  a.gap = key_gap;
  a.colsum = prob_colsum;
  // selection and exact re-decision, after a reduce kernel that sums split-K partials
  if ((e = traced(ctx, MOE_K_ROUTER_SELECT, s, [&] { return launch_router_select(a, s); },
                  a.splits > 1 ? 3 : 2)))
    return cuda_fail(e, "router_select launch");
  return ok();
}

int moe_expert_choice(moe_ctx* ctx, const moe_router_desc* d, const void* X, const float* Wg,
                      const float* logit_bias, int32_t* offsets, int32_t* row_of_slot,
                      int32_t* slot_of_row, float* slot_gate, float* col_gap, void* ws,
                      size_t ws_bytes, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (!d) return fail(MOE_ERR_INVALID_ARG, "desc is null");
  int r = check_shape(d->T, d->E, d->k);
  if (r) return r;
  if (d->H < 1) return fail(MOE_ERR_INVALID_ARG, "H = %d", d->H);
  if (d->score != MOE_SCORE_SOFTMAX && d->score != MOE_SCORE_SIGMOID)
    return fail(MOE_ERR_INVALID_ARG, "score = %d", d->score);
  if (d->x_dtype != MOE_DTYPE_BF16 && d->x_dtype != MOE_DTYPE_F32)
    return fail(MOE_ERR_INVALID_ARG, "x_dtype = %d", d->x_dtype);
  if (d->n_groups > 1)
    return fail(MOE_ERR_UNSUPPORTED, "expert-choice routing takes no expert groups");
  if (((long long)d->T * d->k) % d->E != 0)
    return fail(MOE_ERR_INVALID_ARG, "E = %d must divide T*k = %lld (C = T*k/E)", d->E,
                (long long)d->T * d->k);
  if (d->T > kEcMaxT)
    return fail(MOE_ERR_UNSUPPORTED, "expert-choice routing takes T <= %d tokens", kEcMaxT);
  if ((long long)d->T * d->E > 0x7fffffffLL)
    return fail(MOE_ERR_UNSUPPORTED, "T*E exceeds int32");
  if (d->T > 0 && (!X || !Wg || !offsets || !row_of_slot || !slot_of_row || !slot_gate))
    return fail(MOE_ERR_INVALID_ARG,
                "X, Wg, offsets, row_of_slot, slot_of_row and slot_gate are required");
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is null");
  if (!aligned16(X) || !aligned16(Wg) || !aligned16(ws))
    return fail(MOE_ERR_INVALID_ARG, "X, Wg and ws must be 16-byte aligned");
  const WsLayout L = ws_layout(d->T, d->H, d->E, 0, d->k, d->x_dtype, 0);
  if (ws_bytes < L.h) return fail(MOE_ERR_INVALID_ARG, "workspace too small");
  if ((r = check_ctx(ctx))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  const int C = (int)((long long)d->T * d->k / d->E);
  if (d->T == 0) {
    if (offsets && (e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d->E + 1), s)))
      return cuda_fail(e, "cudaMemsetAsync");
    return ok();
  }
  ExpertChoiceArgs a;
  if ((r = router_logits_stage(ctx, d, X, Wg, logit_bias, ws, ws_bytes, L, a.r, s))) return r;
  char* w = static_cast<char*>(ws);
  a.C = C;
  a.St = reinterpret_cast<float*>(w + L.ec_st);
  a.exS = reinterpret_cast<double*>(w + L.ec_exs);
  a.need = reinterpret_cast<int*>(w + L.ec_need);
  a.tok_list = reinterpret_cast<int*>(w + L.ec_tok);
  a.col_list = reinterpret_cast<int*>(w + L.ec_col);
  a.col_info = reinterpret_cast<int4*>(w + L.ec_info);
  a.ctr = reinterpret_cast<int*>(w + L.ec_ctr);
  a.offsets = offsets;
  a.row_of_slot = row_of_slot;
  a.slot_of_row = slot_of_row;
  a.gate = slot_gate;
  a.gap = col_gap;
  const size_t slots = (size_t)d->T * d->E;
  if ((e = cudaMemsetAsync(a.ctr, 0, 16, s)) ||
      (e = cudaMemsetAsync(a.need, 0, sizeof(int) * d->T, s)) ||
      (e = cudaMemsetAsync(row_of_slot, 0xff, sizeof(int32_t) * slots, s)) ||
      (e = cudaMemsetAsync(slot_gate, 0, sizeof(float) * slots, s)))
    return cuda_fail(e, "cudaMemsetAsync");
  // the split-K reduce, affinities, per-expert selection, exact rows, fix-up
  if ((e = traced(ctx, MOE_K_ROUTER_SELECT, s, [&] {
         cudaError_t q = launch_router_reduce(a.r, s);
         return q != cudaSuccess ? q : launch_expert_choice(a, s);
       }, a.r.splits > 1 ? 5 : 4)))
    return cuda_fail(e, "expert-choice launch");
  // the diagnostic counter: experts re-decided from exact affinities
  if ((e = cudaMemcpyAsync(static_cast<int*>(ws) + 1, a.ctr + 1, sizeof(int),
                           cudaMemcpyDeviceToDevice, s)))
    return cuda_fail(e, "cudaMemcpyAsync");
  return ok();
}

int moe_gather_rows(moe_ctx* ctx, int R, int k, int H, int x_dtype, const int32_t* slot_of_row,
                    const void* X, int T, void* Xperm, void* ws, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (R < 0 || k < 1 || k > kMaxE || T < 0)
    return fail(MOE_ERR_INVALID_ARG, "R = %d, k = %d, T = %d", R, k, T);
  if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32)
    return fail(MOE_ERR_INVALID_ARG, "x_dtype = %d", x_dtype);
  if (H < 1 || (H * (x_dtype == MOE_DTYPE_BF16 ? 2 : 4)) % 16 != 0)
    return fail(MOE_ERR_UNSUPPORTED, "row of H = %d elements is not a multiple of 16 B", H);
  if (R > 0 && (!slot_of_row || !X || !Xperm || !ws))
    return fail(MOE_ERR_INVALID_ARG, "slot_of_row, X, Xperm and ws are required");
  if (!aligned16(X) || !aligned16(Xperm))
    return fail(MOE_ERR_INVALID_ARG, "X and Xperm must be 16-byte aligned");
  int r = check_ctx(ctx);
  if (r) return r;
  cudaStream_t s = (cudaStream_t)stream;
  const int row_bytes = H * (x_dtype == MOE_DTYPE_BF16 ? 2 : 4);
  cudaError_t e = traced(ctx, MOE_K_DISPATCH_GATHER, s, [&] {
    return launch_gather_rows(R, k, row_bytes, slot_of_row, X, Xperm, static_cast<int*>(ws),
                              T, s);
  });
  return e ? cuda_fail(e, "gather launch") : ok();
}

int moe_dispatch(moe_ctx* ctx, int T, int k, int E, int H, int x_dtype, int capacity,
                 const int32_t* topk_idx, const void* X, int32_t* counts, int32_t* offsets,
                 int32_t* row_of_slot, int32_t* slot_of_row, void* Xperm, void* ws,
                 size_t ws_bytes, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int r = check_shape(T, E, k);
  if (r) return r;
  if (!counts || !offsets || !ws) return fail(MOE_ERR_INVALID_ARG, "counts/offsets/ws null");
  if (H < 1) return fail(MOE_ERR_INVALID_ARG, "H = %d (it also sizes the workspace layout)", H);
  if (T > 0 && (!topk_idx || !row_of_slot || !slot_of_row))
    return fail(MOE_ERR_INVALID_ARG, "topk_idx/row_of_slot/slot_of_row null");
  if ((X == nullptr) != (Xperm == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "X and Xperm must be given together");
  if (Xperm) {
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32)
      return fail(MOE_ERR_INVALID_ARG, "x_dtype = %d", x_dtype);
    if (H < 1 || (H * (x_dtype == MOE_DTYPE_BF16 ? 2 : 4)) % 16 != 0)
      return fail(MOE_ERR_UNSUPPORTED, "row of H = %d elements is not a multiple of 16 B", H);
    if (!aligned16(X) || !aligned16(Xperm))
      return fail(MOE_ERR_INVALID_ARG, "X and Xperm must be 16-byte aligned");
  }
  if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "ws must be 16-byte aligned");
  const WsLayout L = ws_layout(T, H, E, 0, k, MOE_DTYPE_BF16, 0);
  if (ws_bytes < L.h) return fail(MOE_ERR_INVALID_ARG, "workspace too small");
  if ((r = check_ctx(ctx))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (T == 0) {
    if ((e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s)) ||
        (e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s)))
      return cuda_fail(e, "cudaMemsetAsync");
    return ok();
  }
  DispatchArgs a;
  a.T = T;
  a.k = k;
  a.E = E;
  a.H = H;
  a.x_dtype = x_dtype;
  a.capacity = capacity < 0 ? -1 : capacity;
  a.idx = topk_idx;
  a.X = X;
  a.counts = counts;
  a.offsets = offsets;
  a.row_of_slot = row_of_slot;
  a.slot_of_row = slot_of_row;
  a.Xperm = Xperm;
  a.chunk_counts = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.chunk_counts);
  a.chunk_base = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.chunk_base);
  a.status = static_cast<int*>(ws);
  if ((e = traced(ctx, MOE_K_DISPATCH_COUNT, s, [&] { return launch_dispatch_count(a, s); })))
    return cuda_fail(e, "dispatch_count launch");
  if ((e = traced(ctx, MOE_K_DISPATCH_SCAN, s, [&] { return launch_dispatch_scan(a, s); })))
    return cuda_fail(e, "dispatch_scan launch");
  if ((e = traced(ctx, MOE_K_DISPATCH_SCATTER, s,
                  [&] { return launch_dispatch_scatter(a, s); })))
    return cuda_fail(e, "dispatch_scatter launch");
  if (Xperm &&
      (e = traced(ctx, MOE_K_DISPATCH_GATHER, s, [&] { return launch_dispatch_gather(a, s); })))
    return cuda_fail(e, "dispatch_gather launch");
  return ok();
}

int moe_grouped_swiglu(moe_ctx* ctx, const moe_expert_desc* d, const void* X,
                       const void* Xperm, const int32_t* offsets, const void* W_gate,
                       const void* W_up, const void* W_down, const void* Ws_gate,
                       const void* Ws_up, const void* Ws_down, float* O, float* O_shared,
                       void* ws, size_t ws_bytes, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (!d) return fail(MOE_ERR_INVALID_ARG, "desc is null");
  int r = check_shape(d->T, d->E, d->k);
  if (r) return r;
  if (d->H < 1 || d->I < 1) return fail(MOE_ERR_INVALID_ARG, "H = %d, I = %d", d->H, d->I);
  if (d->dtype == MOE_DTYPE_BF16) {
    if (d->H % 64 || d->I % 64)
      return fail(MOE_ERR_UNSUPPORTED, "bf16 experts need H %% 64 == 0 and I %% 64 == 0");
  } else if (d->dtype == MOE_DTYPE_F32) {
    if (d->H % 4 || d->I % 4)
      return fail(MOE_ERR_UNSUPPORTED, "fp32 experts need H %% 4 == 0 and I %% 4 == 0");
  } else {
    return fail(MOE_ERR_INVALID_ARG, "dtype = %d", d->dtype);
  }
  if (d->T == 0) {
    int rc = check_ctx(ctx);
    return rc ? rc : ok();
  }
  if (!offsets || !W_gate || !W_up || !W_down || !O || !Xperm || !ws)
    return fail(MOE_ERR_INVALID_ARG, "offsets, weights, Xperm, O and ws are required");
  if (d->has_shared && (!X || !Ws_gate || !Ws_up || !Ws_down || !O_shared))
    return fail(MOE_ERR_INVALID_ARG, "the shared expert needs X, Ws_* and O_shared");
  const void* ptrs[] = {X, Xperm, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, O, O_shared, ws};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(MOE_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const WsLayout L = ws_layout(d->T, d->H, d->E, d->I, d->k, d->dtype, d->has_shared);
  if (ws_bytes < L.total) return fail(MOE_ERR_INVALID_ARG, "workspace too small");
  if ((r = check_ctx(ctx))) return r;
  if (d->T == 0) return ok();
  cudaStream_t s = (cudaStream_t)stream;
  ExpertArgs a;
  a.T = d->T;
  a.H = d->H;
  a.E = d->E;
  a.I = d->I;
  a.k = d->k;
  a.has_shared = d->has_shared ? 1 : 0;
  a.num_sms = ctx->num_sms;
  a.X = X;
  a.Xperm = Xperm;
  a.offsets = offsets;
  a.W_gate = W_gate;
  a.W_up = W_up;
  a.W_down = W_down;
  a.Ws_gate = Ws_gate;
  a.Ws_up = Ws_up;
  a.Ws_down = Ws_down;
  a.h = static_cast<char*>(ws) + L.h;
  a.O = O;
  a.O_shared = O_shared;
  a.status = static_cast<int*>(ws);
  a.test_hook = ctx->test_hook;
  a.wait_limit_ns = ctx->wait_limit_ns;
  cudaError_t e;
  if (d->dtype == MOE_DTYPE_BF16) {
    bool bad = false;
    e = traced(ctx, MOE_K_EXPERT_GATE_UP, s,
               [&] { return launch_expert_gate_up_tc(a, ctx->encode, &bad, s); });
    if (bad) return fail(MOE_ERR_INVALID_ARG, "tensor map encoding failed (gate/up)");
    if (e) return cuda_fail(e, "expert_gate_up launch");
    e = traced(ctx, MOE_K_EXPERT_DOWN, s,
               [&] { return launch_expert_down_tc(a, ctx->encode, &bad, s); });
    if (bad) return fail(MOE_ERR_INVALID_ARG, "tensor map encoding failed (down)");
    if (e) return cuda_fail(e, "expert_down launch");
  } else {
    if ((e = traced(ctx, MOE_K_EXPERT_GATE_UP, s,
                    [&] { return launch_expert_gate_up_f32(a, s); })))
      return cuda_fail(e, "expert_gate_up launch");
    if ((e = traced(ctx, MOE_K_EXPERT_DOWN, s, [&] { return launch_expert_down_f32(a, s); })))
      return cuda_fail(e, "expert_down launch");
  }
  return ok();
}

int moe_quantize_fp8(moe_ctx* ctx, int rows, int cols, int w_dtype, const void* W,
                     uint8_t* q, float* scale, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (rows < 0 || cols < 2 || cols % 2)
    return fail(MOE_ERR_INVALID_ARG, "rows = %d, cols = %d (cols even and >= 2)", rows, cols);
  if (w_dtype != MOE_DTYPE_BF16 && w_dtype != MOE_DTYPE_F32)
    return fail(MOE_ERR_INVALID_ARG, "w_dtype = %d", w_dtype);
  if (rows > 0 && (!W || !q || !scale))
    return fail(MOE_ERR_INVALID_ARG, "W, q and scale are required");
  int r = check_ctx(ctx);
  if (r) return r;
  cudaError_t e = launch_quantize_fp8_rows(rows, cols, w_dtype, W, q, scale,
                                           (cudaStream_t)stream);
  return e ? cuda_fail(e, "quantize_fp8 launch") : ok();
}

int moe_grouped_swiglu_fp8(moe_ctx* ctx, const moe_expert_desc* d, const void* X,
                           const void* Xperm, const int32_t* offsets, const uint8_t* Q_gate,
                           const float* S_gate, const uint8_t* Q_up, const float* S_up,
                           const uint8_t* Q_down, const float* S_down, const uint8_t* Qs_gate,
                           const float* Ss_gate, const uint8_t* Qs_up, const float* Ss_up,
                           const uint8_t* Qs_down, const float* Ss_down, float* O,
                           float* O_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (!d) return fail(MOE_ERR_INVALID_ARG, "desc is null");
  int r = check_shape(d->T, d->E, d->k);
  if (r) return r;
  if (d->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "FP8 expert weights take bf16 activations");
  if (d->H < 64 || d->I < 64 || d->H % 64 || d->I % 64)
    return fail(MOE_ERR_UNSUPPORTED, "FP8 experts need H %% 64 == 0 and I %% 64 == 0");
  if (d->T > 0 && (!offsets || !Q_gate || !S_gate || !Q_up || !S_up || !Q_down || !S_down ||
                   !O || !Xperm || !ws))
    return fail(MOE_ERR_INVALID_ARG, "offsets, codes, scales, Xperm, O and ws are required");
  if (d->T > 0 && d->has_shared &&
      (!X || !Qs_gate || !Ss_gate || !Qs_up || !Ss_up || !Qs_down || !Ss_down || !O_shared))
    return fail(MOE_ERR_INVALID_ARG, "the shared expert needs X, its codes, scales and O_shared");
  const void* ptrs[] = {X, Xperm, Q_gate, Q_up, Q_down, Qs_gate, Qs_up, Qs_down, O, O_shared, ws};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(MOE_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const WsLayout L = ws_layout(d->T, d->H, d->E, d->I, d->k, d->dtype, d->has_shared);
  if (ws_bytes < L.total) return fail(MOE_ERR_INVALID_ARG, "workspace too small");
  if ((r = check_ctx(ctx))) return r;
  if (d->T == 0) return ok();
  cudaStream_t s = (cudaStream_t)stream;
  Fp8Args a;
  a.T = d->T;
  a.H = d->H;
  a.E = d->E;
  a.I = d->I;
  a.k = d->k;
  a.has_shared = d->has_shared ? 1 : 0;
  a.X = X;
  a.Xperm = Xperm;
  a.offsets = offsets;
  a.Q_gate = Q_gate;
  a.Q_up = Q_up;
  a.Q_down = Q_down;
  a.S_gate = S_gate;
  a.S_up = S_up;
  a.S_down = S_down;
  a.Qs_gate = Qs_gate;
  a.Qs_up = Qs_up;
  a.Qs_down = Qs_down;
  a.Ss_gate = Ss_gate;
  a.Ss_up = Ss_up;
  a.Ss_down = Ss_down;
  a.h = static_cast<char*>(ws) + L.h;
  a.O = O;
  a.O_shared = O_shared;
  a.status = static_cast<int*>(ws);
  cudaError_t e;
  bool bad = false;
  e = traced(ctx, MOE_K_EXPERT_GATE_UP, s, [&] {
    return launch_expert_gate_up_fp8(a, ctx->encode, &bad, ctx->wait_limit_ns, s);
  });
  if (bad) return fail(MOE_ERR_INVALID_ARG, "tensor map encoding failed (fp8 gate/up)");
  if (e) return cuda_fail(e, "expert_gate_up (fp8) launch");
  e = traced(ctx, MOE_K_EXPERT_DOWN, s, [&] {
    return launch_expert_down_fp8(a, ctx->encode, &bad, ctx->wait_limit_ns, s);
  });
  if (bad) return fail(MOE_ERR_INVALID_ARG, "tensor map encoding failed (fp8 down)");
  if (e) return cuda_fail(e, "expert_down (fp8) launch");
  return ok();
}

int moe_combine(moe_ctx* ctx, int T, int k, int H, const float* O, const float* O_shared,
                const int32_t* row_of_slot, const float* topk_gate, float* Y, void* Y_bf16,
                moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (T < 0 || k < 1 || k > kMaxE) return fail(MOE_ERR_INVALID_ARG, "T = %d, k = %d", T, k);
  if (H < 4 || H % 4) return fail(MOE_ERR_UNSUPPORTED, "combine needs H %% 4 == 0");
  if (T > 0 && (!O || !row_of_slot || !topk_gate || !Y))
    return fail(MOE_ERR_INVALID_ARG, "O, row_of_slot, topk_gate and Y are required");
  if (!aligned16(O) || !aligned16(O_shared) || !aligned16(Y) || !aligned16(Y_bf16))
    return fail(MOE_ERR_INVALID_ARG, "O, O_shared, Y, Y_bf16 must be 16-byte aligned");
  int r = check_ctx(ctx);
  if (r) return r;
  if (T == 0) return ok();
  cudaStream_t s = (cudaStream_t)stream;
  CombineArgs a{T, k, H, O, O_shared, row_of_slot, topk_gate, Y, Y_bf16};
  cudaError_t e = traced(ctx, MOE_K_COMBINE, s, [&] { return launch_combine(a, s); });
  return e ? cuda_fail(e, "combine launch") : ok();
}

int moe_balance_stats(moe_ctx* ctx, int T, int k, int E, const int32_t* counts,
                      const int32_t* offsets, const double* prob_colsum, double alpha,
                      double* f, double* p, double* out, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int r = check_shape(T, E, k);
  if (r) return r;
  if (!counts || !prob_colsum || !f || !p || !out)
    return fail(MOE_ERR_INVALID_ARG, "counts, prob_colsum, f, p and out are required");
  if ((r = check_ctx(ctx))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  StatsArgs a{T, k, E, counts, offsets, prob_colsum, alpha, f, p, out};
  cudaError_t e = traced(ctx, MOE_K_BALANCE_STATS, s, [&] { return launch_balance_stats(a, s); });
  return e ? cuda_fail(e, "balance_stats launch") : ok();
}

int moe_bias_update(moe_ctx* ctx, int T, int k, int E, const int32_t* counts, float gamma,
                    float* bias, moe_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int r = check_shape(T, E, k);
  if (r) return r;
  if (!counts || !bias) return fail(MOE_ERR_INVALID_ARG, "counts and bias are required");
  if (!(gamma == gamma) || gamma - gamma != 0.f)
    return fail(MOE_ERR_INVALID_ARG, "gamma must be finite");
  if ((r = check_ctx(ctx))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  BiasArgs a{E, (long long)T * k, counts, gamma, bias};
  cudaError_t e = traced(ctx, MOE_K_BIAS_UPDATE, s, [&] { return launch_bias_update(a, s); });
  return e ? cuda_fail(e, "bias_update launch") : ok();
}

int moe_get_device_status(moe_ctx* ctx, void* ws, int* status, int reset,
                          moe_stream_t stream) {
  if (!ws || !status) return fail(MOE_ERR_INVALID_ARG, "ws and status are required");
  int r = check_ctx(ctx);
  if (r) return r;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e) return cuda_fail(e, "cudaStreamSynchronize");
  if ((e = cudaMemcpy(status, ws, sizeof(int), cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "cudaMemcpy");
  if (reset && (e = cudaMemset(ws, 0, sizeof(int)))) return cuda_fail(e, "cudaMemset");
  return ok();
}

int moe_ctx_set_test_hook(moe_ctx* ctx, int hook, int wait_limit_ms) {
  if (!ctx) return fail(MOE_ERR_INVALID_ARG, "ctx is null");
  if (hook != MOE_TEST_HOOK_NONE && hook != MOE_TEST_HOOK_WITHHOLD_LOAD)
    return fail(MOE_ERR_INVALID_ARG, "hook = %d", hook);
  if (wait_limit_ms < 0) return fail(MOE_ERR_INVALID_ARG, "wait_limit_ms < 0");
  ctx->test_hook = hook;
  ctx->wait_limit_ns =
      wait_limit_ms ? (unsigned long long)wait_limit_ms * 1000000ull : kWaitLimitDefaultNs;
  return ok();
}

int moe_ctx_set_tracing(moe_ctx* ctx, int enable) {
  if (!ctx) return fail(MOE_ERR_INVALID_ARG, "ctx is null");
  ctx->tracing = enable != 0;
  return ok();
}

int moe_ctx_trace_read(moe_ctx* ctx, int* launches, double* total_ms, int n) {
  if (!ctx || !launches || !total_ms || n < MOE_KERNEL_COUNT)
    return fail(MOE_ERR_INVALID_ARG, "bad trace buffers");
  std::lock_guard<std::mutex> lk(ctx->mu);
  for (int i = 0; i < n; ++i) {
    launches[i] = 0;
    total_ms[i] = 0.0;
  }
  int rc = MOE_OK;
  for (auto& rec : ctx->recs) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(rec.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, rec.a, rec.b);
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaEventElapsedTime");
    launches[rec.id] += rec.kernels;
    total_ms[rec.id] += ms;
    ctx->pool.push_back(rec.a);
    ctx->pool.push_back(rec.b);
  }
  ctx->recs.clear();
  return rc ? rc : ok();
}

}  // extern "C"
