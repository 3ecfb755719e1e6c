// Step 6 of the MoE forward and the balance statistics.
//
// combine: "LLM Internals §14.2.1 step 6" - weight each expert output by its gate, write
// it back to the token's position through the inverse of the step-4 permutation, add the
// shared expert; "AI Knowledge Map - MoE": y = sum over S of g_e E_e(x).  One CTA per
// token (and column chunk, for small batches), 16-byte vector loads, a fixed summation
// order (choices j ascending, then the shared expert), so the result is bitwise
// reproducible.
//
// balance_stats: §14.2.3 L = alpha * N * sum f_i p_i and the three monitoring signals it
// names (routing entropy, per-expert load, drop rate), plus the load CV of the
// "AI Knowledge Map - MoE" page.  One CTA, float64.
//
// bias_update: §14.2.3 bias-adjusted selection, the balancing step after a batch: an
// expert whose load m_e (router choices before capacity) is above the balanced load
// T k / E loses gamma from its selection bias, one below it gains gamma, one exactly at it
// keeps its bias.  The comparison is exact in integers (E m_e against T k); the update is
// one float32 addition.
#include <math.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  const int t = blockIdx.x;
  // the token's live slots (row >= 0) in ascending slot order: k is at most kMaxK for
  // token-choice routing and E for expert-choice routing, where most slots are empty
  __shared__ int s_row[kMaxE];
  __shared__ float s_g[kMaxE];
  __shared__ int s_n;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int n = 0;
    for (int base = 0; base < a.k; base += 32) {
      const int j = base + lane;
      const int r = j < a.k ? a.row_of_slot[(size_t)t * a.k + j] : -1;
      const uint32_t live = __ballot_sync(0xffffffffu, r >= 0);
      if (r >= 0) {
        const int pos = n + __popc(live & ((1u << lane) - 1u));
        s_row[pos] = r;
        s_g[pos] = a.gate[(size_t)t * a.k + j];
      }
      n += __popc(live);
    }
    if (lane == 0) s_n = n;
  }
  __syncthreads();
  const int nlive = s_n;
  const int nv = a.H / 4;
  const int per = (nv + gridDim.y - 1) / gridDim.y;   // column chunk of this CTA
  const int v0 = blockIdx.y * per, v1 = min(nv, v0 + per);
  float4* Y = reinterpret_cast<float4*>(a.Y + (size_t)t * a.H);
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < nlive; ++j) {
      const int r = s_row[j];
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

// One thread per expert, ceil(E/32) warps: warp-shuffle sums, then one cross-warp pass.
__global__ void __launch_bounds__(kMaxE) balance_stats_kernel(StatsArgs a) {
  __shared__ double part[kMaxE / 32][3];
  __shared__ double s_mean;
  const int e = threadIdx.x, lane = e & 31, w = e >> 5, nw = blockDim.x >> 5;
  const double slots = (double)a.T * a.k;
  const bool in = e < a.E;
  double m = 0.0, f = 0.0, p = 0.0, fp = 0.0, ent = 0.0;
  if (in) {
    m = (double)a.counts[e];
    if (slots > 0) f = m / slots;
    if (a.T > 0) p = a.colsum[e] / a.T;
    a.f[e] = f;
    a.p[e] = p;
    fp = f * p;
    if (f > 0) ent = -f * log(f);
  }
  auto warp_sum = [](double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };
  fp = warp_sum(fp);
  const double msum = warp_sum(m);
  ent = warp_sum(ent);
  if (lane == 0) {
    part[w][0] = fp;
    part[w][1] = msum;
    part[w][2] = ent;
  }
  __syncthreads();
  if (e == 0) {
    double t = 0.0;
    for (int q = 0; q < nw; ++q) t += part[q][1];
    s_mean = a.E > 0 ? t / a.E : 0.0;
  }
  __syncthreads();
  const double mean = s_mean;
  double sq = in ? (m - mean) * (m - mean) : 0.0;
  sq = warp_sum(sq);
  __syncthreads();
  if (lane == 0) part[w][1] = sq;
  __syncthreads();
  if (e == 0) {
    double sfp = 0.0, ssq = 0.0, sent = 0.0;
    for (int q = 0; q < nw; ++q) {
      sfp += part[q][0];
      ssq += part[q][1];
      sent += part[q][2];
    }
    a.out[0] = a.alpha * a.E * sfp;
    a.out[1] = (a.offsets && slots > 0) ? (slots - (double)a.offsets[a.E]) / slots : 0.0;
    a.out[2] = mean > 0 ? sqrt(ssq / a.E) / mean : 0.0;
    a.out[3] = sent;
  }
}

__global__ void __launch_bounds__(256) bias_update_kernel(BiasArgs a) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= a.E) return;
  const long long load = (long long)a.counts[e] * a.E;
  if (load > a.slots) a.bias[e] = a.bias[e] - a.gamma;
  else if (load < a.slots) a.bias[e] = a.bias[e] + a.gamma;
}

}  // namespace

cudaError_t launch_bias_update(const BiasArgs& a, cudaStream_t s) {
  bias_update_kernel<<<(a.E + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  // CTA per token and column chunk: a small batch is split along H so that the GPU gets
  // about two CTAs per SM, each chunk at least 256 float4 wide
  const int nv = a.H / 4;
  const int ymax = nv / 256 > 0 ? nv / 256 : 1;
  int ysplit = (2 * kGridSms + a.T - 1) / (a.T > 0 ? a.T : 1);
  ysplit = ysplit < 1 ? 1 : (ysplit > ymax ? ymax : ysplit);
  combine_kernel<<<dim3(a.T, ysplit), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_balance_stats(const StatsArgs& a, cudaStream_t s) {
  balance_stats_kernel<<<1, 32 * ((a.E + 31) / 32), 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
