// Steps 2-3 of the MoE forward ("LLM Internals §14.2.1": router scoring X[T,H] x
// W_g[H,E], then top-k per row and normalisation among the k chosen; "AI Knowledge Map
// - MoE": score, softmax, top-k hard selection, renormalise).
//
// Two kernels (the first in a wide and a narrow form):
//  router_logits  fp32 CUDA-core GEMM l = X W_g (+ logit offset).  Each 32-long block
//                 of the reduction is summed with fp32 FMA, and the block partials are
//                 folded into a (hi, lo) pair with TwoSum (Knuth), so the error is that of
//                 32-term fp32 sums, not of an H-term one.
//  router_select  one warp per token: keys, top-(k+1) by warp argmax (ties to the lower
//                 expert index), and an exactness guard: when the k-th/(k+1)-th margin
//                 is within the fp32 error bound, every expert that could still be in
//                 the top k gets its logit recomputed as a float64 dot product and the
//                 row is re-decided on those.  Then gates, key gap, row probabilities.
#include <math.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTM = 64;   // tokens per CTA tile
constexpr int kTE = 64;   // experts per CTA tile
constexpr int kTK = 32;   // reduction block

__device__ __forceinline__ void two_sum(float& hi, float& lo, float b) {
  const float s = hi + b;
  const float bp = s - hi;
  const float err = (hi - (s - bp)) + (b - bp);
  hi = s;
  lo += err;
}

template <typename TX>
__device__ __forceinline__ void load_x8(const TX* X, size_t off, float (&v)[8]);

template <>
__device__ __forceinline__ void load_x8<__nv_bfloat16>(const __nv_bfloat16* X, size_t off,
                                                        float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(X + off);
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

template <>
__device__ __forceinline__ void load_x8<float>(const float* X, size_t off, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(X + off);
  const float4 b = *reinterpret_cast<const float4*>(X + off + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename TX>
__device__ __forceinline__ float load_x1(const TX* X, size_t off);
template <>
__device__ __forceinline__ float load_x1<__nv_bfloat16>(const __nv_bfloat16* X, size_t off) {
  return __bfloat162float(X[off]);
}
template <>
__device__ __forceinline__ float load_x1<float>(const float* X, size_t off) {
  return X[off];
}

// 256 threads; thread (ty, tx) owns tokens ty*4..+3 and experts tx*4..+3 of the tile.
template <typename TX>
__global__ void __launch_bounds__(256) router_logits_kernel(RouterArgs a) {
  __shared__ __align__(16) float sX[kTK][kTM + 4];
  __shared__ __align__(16) float sW[kTK][kTE];
  const TX* X = static_cast<const TX*>(a.X);
  const int T = a.T, H = a.H, E = a.E;
  const int t0 = blockIdx.x * kTM, e0 = blockIdx.y * kTE;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const bool vec_x = (H % 8) == 0;
  const bool vec_w = (E % 4) == 0;

  float hi[4][4], lo[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) hi[i][j] = lo[i][j] = 0.f;

  for (int kb = 0; kb < H; kb += kTK) {
    // X tile [64 tokens][32 h] -> sX[h][token]; one 8-element segment per thread.
    {
      const int r = tid >> 2, c0 = (tid & 3) * 8;
      const int t = t0 + r, h = kb + c0;
      float v[8];
      if (t < T && vec_x && h + 8 <= H) {
        load_x8<TX>(X, (size_t)t * H + h, v);
      } else {
#pragma unroll
        for (int m = 0; m < 8; ++m)
          v[m] = (t < T && h + m < H) ? load_x1<TX>(X, (size_t)t * H + h + m) : 0.f;
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) sX[c0 + m][r] = v[m];
    }
    // W tile [32 h][64 experts]
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int i = tid + q * 256;           // 512 float4 slots
      const int r = i >> 4, c = (i & 15) * 4;
      const int h = kb + r, e = e0 + c;
      float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
      if (h < H) {
        if (vec_w && e + 4 <= E) {
          w = *reinterpret_cast<const float4*>(a.Wg + (size_t)h * E + e);
        } else {
          const float* row = a.Wg + (size_t)h * E;
          w.x = (e + 0 < E) ? row[e + 0] : 0.f;
          w.y = (e + 1 < E) ? row[e + 1] : 0.f;
          w.z = (e + 2 < E) ? row[e + 2] : 0.f;
          w.w = (e + 3 < E) ? row[e + 3] : 0.f;
        }
      }
      *reinterpret_cast<float4*>(&sW[r][c]) = w;
    }
    __syncthreads();

    float p[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) p[i][j] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      const float4 xv = *reinterpret_cast<const float4*>(&sX[kk][ty * 4]);
      const float4 wv = *reinterpret_cast<const float4*>(&sW[kk][tx * 4]);
      const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
      const float ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) p[i][j] = fmaf(xs[i], ws[j], p[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) two_sum(hi[i][j], lo[i][j], p[i][j]);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e >= E) continue;
      float h = hi[i][j], l = lo[i][j];
      if (a.logit_bias) two_sum(h, l, a.logit_bias[e]);
      a.logits[(size_t)t * E + e] = h + l;
    }
  }
}

// Narrow routers (E <= 16): a CTA owns 32 tokens and walks H in chunks of 256 (128 for
// E > 8); thread
// (token, g) sums h = g, g+8, ... of the chunk (32 or 16 terms) for every expert, folds the
// block partial into its (hi, lo) pair, and the 8 partial pairs of a token are merged with
// TwoSum across lanes.  Same error class as router_logits_kernel, 16x less padding work.
template <typename TX, int EP>
__global__ void __launch_bounds__(256) router_logits_narrow_kernel(RouterArgs a) {
  constexpr int TM = 32, HC = EP <= 8 ? 256 : 128;   // static shared memory under 48 KB
  __shared__ __align__(16) float sX[TM][HC + 8];
  __shared__ __align__(16) float sW[HC][EP];
  const TX* X = static_cast<const TX*>(a.X);
  const int T = a.T, H = a.H, E = a.E;
  const int tid = threadIdx.x, tl = tid >> 3, g = tid & 7;
  const int t0 = blockIdx.x * TM;
  const bool vec_x = (H % 8) == 0;
  float hi[EP], lo[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) hi[e] = lo[e] = 0.f;

  for (int kb = 0; kb < H; kb += HC) {
#pragma unroll
    for (int q = 0; q < TM * HC / 8 / 256; ++q) {
      const int v = tid + q * 256;
      const int r = v / (HC / 8), c = (v % (HC / 8)) * 8;
      const int t = t0 + r, h = kb + c;
      float x[8];
      if (t < T && vec_x && h + 8 <= H) {
        load_x8<TX>(X, (size_t)t * H + h, x);
      } else {
#pragma unroll
        for (int m = 0; m < 8; ++m)
          x[m] = (t < T && h + m < H) ? load_x1<TX>(X, (size_t)t * H + h + m) : 0.f;
      }
      *reinterpret_cast<float4*>(&sX[r][c]) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(&sX[r][c + 4]) = make_float4(x[4], x[5], x[6], x[7]);
    }
    for (int i = tid; i < HC * EP; i += 256) {
      const int r = i / EP, e = i % EP;
      const int h = kb + r;
      sW[r][e] = (h < H && e < E) ? a.Wg[(size_t)h * E + e] : 0.f;
    }
    __syncthreads();
    float p[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) p[e] = 0.f;
#pragma unroll 8
    for (int j = 0; j < HC / 8; ++j) {
      const int h = g + 8 * j;
      const float x = sX[tl][h];
#pragma unroll
      for (int q = 0; q < EP / 4; ++q) {
        const float4 w = *reinterpret_cast<const float4*>(&sW[h][4 * q]);
        p[4 * q + 0] = fmaf(x, w.x, p[4 * q + 0]);
        p[4 * q + 1] = fmaf(x, w.y, p[4 * q + 1]);
        p[4 * q + 2] = fmaf(x, w.z, p[4 * q + 2]);
        p[4 * q + 3] = fmaf(x, w.w, p[4 * q + 3]);
      }
    }
#pragma unroll
    for (int e = 0; e < EP; ++e) two_sum(hi[e], lo[e], p[e]);
    __syncthreads();
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      const float h2 = __shfl_xor_sync(0xffffffffu, hi[e], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, lo[e], o);
      two_sum(hi[e], lo[e], h2);
      lo[e] += l2;
    }
  }
  const int t = t0 + tl;
  if (g == 0 && t < T) {
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      if (e >= E) break;
      float h = hi[e], l = lo[e];
      if (a.logit_bias) two_sum(h, l, a.logit_bias[e]);
      a.logits[(size_t)t * E + e] = h + l;
    }
  }
}

// ------------------------------------------------------------------ selection

struct Best {
  float key;
  int idx;
};

__device__ __forceinline__ bool better(float k1, int i1, float k2, int i2) {
  return k1 > k2 || (k1 == k2 && i1 < i2);
}

__device__ __forceinline__ Best warp_best(Best b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float k2 = __shfl_xor_sync(0xffffffffu, b.key, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, b.idx, o);
    if (better(k2, i2, b.key, b.idx)) {
      b.key = k2;
      b.idx = i2;
    }
  }
  return b;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// float64 dot product of token t with router column e, the whole warp cooperating.
template <typename TX>
__device__ double exact_logit(const RouterArgs& a, const TX* X, int t, int e, int lane) {
  double acc0 = 0.0, acc1 = 0.0;
  const TX* xr = X + (size_t)t * a.H;
  int h = lane;
  for (; h + 32 < a.H; h += 64) {
    acc0 = fma((double)load_x1<TX>(xr, h), (double)a.Wg[(size_t)h * a.E + e], acc0);
    acc1 = fma((double)load_x1<TX>(xr, h + 32), (double)a.Wg[(size_t)(h + 32) * a.E + e],
               acc1);
  }
  if (h < a.H) acc0 = fma((double)load_x1<TX>(xr, h), (double)a.Wg[(size_t)h * a.E + e], acc0);
  double s = warp_sum_d(acc0 + acc1);
  if (a.logit_bias) s += (double)a.logit_bias[e];
  return s;
}

constexpr int kSelWarps = 8;
constexpr int kTokPerWarp = 8;

template <typename TX, int NJ>
__global__ void __launch_bounds__(kSelWarps * 32) router_select_kernel(RouterArgs a) {
  __shared__ float s_col[kSelWarps][NJ * 32];
  const TX* X = static_cast<const TX*>(a.X);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int E = a.E, k = a.k;
  const bool sigm = a.score == MOE_SCORE_SIGMOID;
  const float h_scale = sqrtf(fmaxf(1.f, a.H / 1024.f));

  float col[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) col[j] = 0.f;

  const int tbeg = (blockIdx.x * kSelWarps + w) * kTokPerWarp;
  for (int t = tbeg; t < min(tbeg + kTokPerWarp, a.T); ++t) {
    float l[NJ], key[NJ];
    float lmax = -INFINITY, amax = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E) {
        l[j] = a.logits[(size_t)t * E + e];
        lmax = fmaxf(lmax, l[j]);
        amax = fmaxf(amax, fabsf(l[j]));
        float kv;
        if (sigm) {
          kv = 1.f / (1.f + expf(-l[j]));
          if (a.bias) kv += a.bias[e];
        } else {
          kv = l[j];
        }
        key[j] = (kv != kv) ? -INFINITY : kv;
      } else {
        l[j] = -INFINITY;
        key[j] = -INFINITY;
      }
    }
    lmax = warp_max_f(lmax);
    amax = warp_max_f(amax);

    // top-(k+1) by repeated warp argmax
    uint32_t taken = 0;   // bit j: expert lane+32j already chosen in this pass
    float kth = 0.f, k1th = -INFINITY;
    int sel_lane_j[kMaxK];   // chosen experts, descending key
    const int rounds = (k < E) ? k + 1 : k;
    for (int r = 0; r < rounds; ++r) {
      Best b{-INFINITY, 0x7fffffff};
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !(taken >> j & 1u) && better(key[j], e, b.key, b.idx)) {
          b.key = key[j];
          b.idx = e;
        }
      }
      b = warp_best(b);
      if (r < k) {
        sel_lane_j[r] = b.idx;
        if ((b.idx & 31) == lane) taken |= 1u << (b.idx >> 5);
        kth = b.key;
      } else {
        k1th = b.key;
      }
    }

    float gap = (k < E) ? kth - k1th : INFINITY;
    // error bound of the fp32 logits and of the fp32 keys derived from them
    const float eps_l = ldexpf(1.f, -19) * fmaxf(1.f, amax) * h_scale;
    const float eps = sigm ? 0.25f * eps_l + ldexpf(1.f, -20) : eps_l;

    if (k < E && !(gap > 2.f * eps)) {
      // Exactness guard: every expert whose key could still belong to the top k.
      const float lim = kth - 2.f * eps;
      double ex[NJ];
      uint32_t cand = 0;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        ex[j] = -INFINITY;
        if (e < E && key[j] >= lim) cand |= 1u << j;
      }
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        uint32_t m = __ballot_sync(0xffffffffu, (cand >> j) & 1u);
        while (m) {
          const int src = __ffs(m) - 1;
          m &= m - 1;
          const int e = src + 32 * j;
          const double le = exact_logit<TX>(a, X, t, e, lane);
          double kv = le;
          if (sigm) {
            kv = 1.0 / (1.0 + exp(-le));
            if (a.bias) kv += (double)a.bias[e];
          }
          if (lane == src) ex[j] = kv;
        }
      }
      // re-decide among the candidates on the float64 keys
      uint32_t tk = 0;
      double dk = 0.0, dk1 = -INFINITY;
      for (int r = 0; r <= k; ++r) {
        double bk = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int e = lane + 32 * j;
          if ((cand >> j & 1u) && !(tk >> j & 1u) &&
              (ex[j] > bk || (ex[j] == bk && e < bi))) {
            bk = ex[j];
            bi = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const double k2 = __shfl_xor_sync(0xffffffffu, bk, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
          if (k2 > bk || (k2 == bk && i2 < bi)) {
            bk = k2;
            bi = i2;
          }
        }
        if (bi == 0x7fffffff) break;   // fewer than k+1 candidates (cannot happen)
        if (r < k) {
          if ((bi & 31) == lane) tk |= 1u << (bi >> 5);
          dk = bk;
        } else {
          dk1 = bk;
        }
      }
      // the first k rounds always succeed: the candidates include the approximate top
      // k+1; rebuild the chosen list from tk
      int n = 0;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const uint32_t m = __ballot_sync(0xffffffffu, (tk >> j) & 1u);
        uint32_t mm = m;
        while (mm) {
          const int src = __ffs(mm) - 1;
          mm &= mm - 1;
          if (n < k) sel_lane_j[n] = src + 32 * j;
          ++n;
        }
      }
      gap = (float)(dk - dk1);
    }

    // gates of the chosen experts (fp32, from the fp32 logits)
    float zsum = 0.f, ssum = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < E) {
        if (sigm) ssum += 1.f / (1.f + expf(-l[j]));
        else zsum += expf(l[j] - lmax);
      }
    }
    zsum = warp_sum_f(zsum);
    ssum = warp_sum_f(ssum);

    // lane r < k takes chosen expert r and fetches its logit from the owner lane
    int my_e = 0x7fffffff;
    float lv = 0.f;
    for (int r = 0; r < k; ++r) {
      const int e = sel_lane_j[r];          // warp-uniform
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if ((e >> 5) == j) v = l[j];
      v = __shfl_sync(0xffffffffu, v, e & 31);
      if (lane == r) {
        lv = v;
        my_e = e;
      }
    }
    float my_v = 0.f;
    if (lane < k) my_v = sigm ? 1.f / (1.f + expf(-lv)) : expf(lv - lmax);
    const float chosen_sum = warp_sum_f(my_v);
    float g;
    if (a.renorm) g = my_v / chosen_sum;
    else g = sigm ? my_v : my_v / zsum;
    // write in ascending expert order
    int rank = 0;
    for (int r = 0; r < k; ++r) {
      const int e = __shfl_sync(0xffffffffu, my_e, r);
      if (e < my_e) ++rank;
    }
    if (lane < k) {
      a.idx[(size_t)t * k + rank] = my_e;
      a.gate[(size_t)t * k + rank] = g;
    }
    if (lane == 0 && a.gap) a.gap[t] = gap;

    // row probabilities for the balance statistics
    if (a.colsum) {
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        if (e < E) col[j] += sigm ? (1.f / (1.f + expf(-l[j]))) / ssum
                                  : expf(l[j] - lmax) / zsum;
      }
    }
  }

  if (a.colsum) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) s_col[w][lane + 32 * j] = col[j];
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      double s = 0.0;
#pragma unroll
      for (int q = 0; q < kSelWarps; ++q) s += (double)s_col[q][e];
      atomicAdd(a.colsum + e, s);
    }
  }
}

template <typename TX>
cudaError_t launch_select_t(const RouterArgs& a, cudaStream_t s) {
  const int per_cta = kSelWarps * kTokPerWarp;
  const dim3 grid((a.T + per_cta - 1) / per_cta);
  const dim3 block(kSelWarps * 32);
  if (a.E <= 32) router_select_kernel<TX, 1><<<grid, block, 0, s>>>(a);
  else if (a.E <= 64) router_select_kernel<TX, 2><<<grid, block, 0, s>>>(a);
  else if (a.E <= 128) router_select_kernel<TX, 4><<<grid, block, 0, s>>>(a);
  else if (a.E <= 256) router_select_kernel<TX, 8><<<grid, block, 0, s>>>(a);
  else router_select_kernel<TX, 16><<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t s) {
  if (a.E <= 16) {
    const dim3 g((a.T + 31) / 32);
    const bool bf = a.x_dtype == MOE_DTYPE_BF16;
    if (a.E <= 8) {
      if (bf) router_logits_narrow_kernel<__nv_bfloat16, 8><<<g, 256, 0, s>>>(a);
      else router_logits_narrow_kernel<float, 8><<<g, 256, 0, s>>>(a);
    } else {
      if (bf) router_logits_narrow_kernel<__nv_bfloat16, 16><<<g, 256, 0, s>>>(a);
      else router_logits_narrow_kernel<float, 16><<<g, 256, 0, s>>>(a);
    }
    return cudaGetLastError();
  }
  const dim3 grid((a.T + kTM - 1) / kTM, (a.E + kTE - 1) / kTE);
  if (a.x_dtype == MOE_DTYPE_BF16)
    router_logits_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
  else
    router_logits_kernel<float><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_router_select(const RouterArgs& a, cudaStream_t s) {
  return a.x_dtype == MOE_DTYPE_BF16 ? launch_select_t<__nv_bfloat16>(a, s)
                                     : launch_select_t<float>(a, s);
}

}  // namespace moe
