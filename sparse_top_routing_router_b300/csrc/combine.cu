// Step 6 of the MoE forward and the balance statistics.
//
// combine: "LLM Internals §14.2.1 step 6" - weight each expert output by its gate, write
// it back to the token's position through the inverse of the step-4 permutation, add the
// shared expert; "AI Knowledge Map - MoE": y = sum over S of g_e E_e(x).  One CTA per
// token, 16-byte vector loads, a fixed summation order (choices j ascending, then the
// shared expert), so the result is bitwise reproducible.
//
// balance_stats: §14.2.3 L = alpha * N * sum f_i p_i and the three monitoring signals it
// names (routing entropy, per-expert load, drop rate), plus the load CV of the
// "AI Knowledge Map - MoE" page.  One CTA, float64.
#include <math.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  const int t = blockIdx.x;
  __shared__ int s_row[kMaxK];
  __shared__ float s_g[kMaxK];
  if (threadIdx.x < a.k) {
    s_row[threadIdx.x] = a.row_of_slot[(size_t)t * a.k + threadIdx.x];
    s_g[threadIdx.x] = a.gate[(size_t)t * a.k + threadIdx.x];
  }
  __syncthreads();
  const int nv = a.H / 4;
  float4* Y = reinterpret_cast<float4*>(a.Y + (size_t)t * a.H);
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < a.k; ++j) {
      const int r = s_row[j];
      if (r < 0) continue;
      const float g = s_g[j];
      const float4 o = reinterpret_cast<const float4*>(a.O + (size_t)r * a.H)[v];
      acc.x = fmaf(g, o.x, acc.x);
      acc.y = fmaf(g, o.y, acc.y);
      acc.z = fmaf(g, o.z, acc.z);
      acc.w = fmaf(g, o.w, acc.w);
    }
    if (a.O_shared) {
      const float4 o = reinterpret_cast<const float4*>(a.O_shared + (size_t)t * a.H)[v];
      acc.x += o.x;
      acc.y += o.y;
      acc.z += o.z;
      acc.w += o.w;
    }
    Y[v] = acc;
    if (a.Y_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.Y_bf16) + (size_t)t * a.H)[v] =
          pk;
    }
  }
}

__global__ void __launch_bounds__(kMaxE) balance_stats_kernel(StatsArgs a) {
  __shared__ double red[kMaxE];
  const int e = threadIdx.x;
  const double slots = (double)a.T * a.k;
  const bool in = e < a.E;
  const double m = in ? (double)a.counts[e] : 0.0;
  const double f = (in && slots > 0) ? m / slots : 0.0;
  const double p = (in && a.T > 0) ? a.colsum[e] / a.T : 0.0;
  if (in) {
    a.f[e] = f;
    a.p[e] = p;
  }
  auto block_sum = [&](double v) -> double {
    red[e] = v;
    __syncthreads();
    for (int s = kMaxE / 2; s > 0; s >>= 1) {
      if (e < s) red[e] += red[e + s];
      __syncthreads();
    }
    const double r = red[0];
    __syncthreads();
    return r;
  };
  const double sum_fp = block_sum(f * p);
  const double sum_m = block_sum(m);
  const double mean = a.E > 0 ? sum_m / a.E : 0.0;
  const double sq = block_sum(in ? (m - mean) * (m - mean) : 0.0);
  const double ent = block_sum(f > 0 ? -f * log(f) : 0.0);
  if (e == 0) {
    a.out[0] = a.alpha * a.E * sum_fp;
    a.out[1] = (a.offsets && slots > 0) ? (slots - (double)a.offsets[a.E]) / slots : 0.0;
    a.out[2] = mean > 0 ? sqrt(sq / a.E) / mean : 0.0;
    a.out[3] = ent;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  combine_kernel<<<a.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_balance_stats(const StatsArgs& a, cudaStream_t s) {
  balance_stats_kernel<<<1, kMaxE, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
