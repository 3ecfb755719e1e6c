// Steps 2-3 of the MoE forward ("LLM Internals §14.2.1": router scoring X[T,H] x
// W_g[H,E], then top-k per row and normalisation among the k chosen; "AI Knowledge Map
// - MoE": score, softmax, top-k hard selection, renormalise).
//
// Kernels:
//  router_logits  fp32 CUDA-core GEMM l = X W_g (a wide and a narrow form).  Each 32-long
//                 block of the reduction is summed with fp32 FMA, and the block partials
//                 are folded into a (hi, lo) pair with TwoSum (Knuth), so the error is that
//                 of 32-term fp32 sums, not of an H-term one.  (The tensor-core form of
//                 the logits lives with the expert GEMMs; router_split_kernel prepares its
//                 exact bf16 pieces of W_g.)
//  router_reduce  sums the split-K partials in slice order.
//  router_select  one warp per token: logit offset, keys, top-(k+1) by warp argmax (ties
//                 to the lower expert index), gates, key gap, row probabilities.  A row
//                 whose k-th/(k+1)-th margin is within the fp32 error bound is listed.
//  router_refine  one CTA per listed row: every expert that could still be in the top k
//                 gets its logit recomputed exactly (to ~48 bits) and the row is
//                 re-decided on those.
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
  // this CTA's slice of the reduction: whole 32-blocks [b0, b1)
  const int nblk = (H + kTK - 1) / kTK;
  const int b0 = (int)((long long)nblk * blockIdx.z / gridDim.z);
  const int b1 = (int)((long long)nblk * (blockIdx.z + 1) / gridDim.z);

  float hi[4][4], lo[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) hi[i][j] = lo[i][j] = 0.f;

  for (int kb = b0 * kTK; kb < b1 * kTK; kb += kTK) {
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
      a.logits[((size_t)blockIdx.z * T + t) * E + e] = make_float2(h, l);
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
  const int nch = (H + HC - 1) / HC;
  const int c0 = (int)((long long)nch * blockIdx.y / gridDim.y);
  const int c1 = (int)((long long)nch * (blockIdx.y + 1) / gridDim.y);
  float hi[EP], lo[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) hi[e] = lo[e] = 0.f;

  for (int kb = c0 * HC; kb < c1 * HC; kb += HC) {
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
      a.logits[((size_t)blockIdx.y * T + t) * E + e] = make_float2(h, l);
    }
  }
}

// W_g [H, E] fp32 -> pieces [E][3H] bf16 with w = hi + mid + lo exactly: hi = bf16(w),
// mid = bf16(w - hi), lo = w - hi - mid (8 significant bits at most, so bf16-exact).  The
// transpose goes through a 32x32 shared tile so both the read and the write coalesce.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ Wg, int H,
                                                           int E, __nv_bfloat16* __restrict__ out) {
  __shared__ __nv_bfloat16 t[3][32][33];
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int r = ty; r < 32; r += 8) {
    const int h = h0 + r, e = e0 + tx;
    const float w = (h < H && e < E) ? Wg[(size_t)h * E + e] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    t[0][tx][r] = hi;
    t[1][tx][r] = mid;
    t[2][tx][r] = __float2bfloat16_rn(r2);
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int e = e0 + r, h = h0 + tx;
    if (e < E && h < H) {
      __nv_bfloat16* row = out + (size_t)e * 3 * H;
      row[h] = t[0][r][tx];
      row[H + h] = t[1][r][tx];
      row[2 * H + h] = t[2][r][tx];
    }
  }
}

// Sum of the S split-K partials of every (token, expert) in slice order: G consecutive
// lanes share one element, lane r adding the r-th contiguous run of slices with TwoSum,
// then the G runs are combined in lane order (a fixed order, so the result does not vary
// between runs).  G > 1 when there are too few elements to keep the GPU's loads in
// flight; the result goes to slice 0 as a (hi, lo) pair.  F32 selects plain fp32
// partials in `q` (tensor-core slices), else (hi, lo) partials in `p` itself.
template <bool F32, int G>
__global__ void __launch_bounds__(256) router_reduce_kernel(float2* __restrict__ p,
                                                            const float* __restrict__ q,
                                                            size_t n, int S) {
  const size_t gid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t i = gid / G;
  const int r = (int)(gid % G);
  const bool live = i < n;
  const int per = (S + G - 1) / G;
  const int z_lo = min(S, r * per), z_hi = min(S, z_lo + per);
  float hs = 0.f, ls = 0.f;
  if (live) {
    for (int z0 = z_lo; z0 < z_hi; z0 += 8) {
      float2 v[8];
#pragma unroll
      for (int z = 0; z < 8; ++z) {
        v[z] = make_float2(0.f, 0.f);
        if (z0 + z < z_hi) {
          if (F32) v[z].x = q[(size_t)(z0 + z) * n + i];
          else v[z] = p[(size_t)(z0 + z) * n + i];
        }
      }
#pragma unroll
      for (int z = 0; z < 8; ++z) {
        two_sum(hs, ls, v[z].x);
        ls += v[z].y;
      }
    }
  }
  if (G > 1) {
    // lane r takes lane r + o's sum, o = 1, 2, 4: the runs are added in slice order
#pragma unroll
    for (int o = 1; o < G; o <<= 1) {
      const float h2 = __shfl_down_sync(0xffffffffu, hs, o, G);
      const float l2 = __shfl_down_sync(0xffffffffu, ls, o, G);
      if ((r & (2 * o - 1)) == 0) {
        two_sum(hs, ls, h2);
        ls += l2;
      }
    }
  }
  if (live && r == 0) p[i] = make_float2(hs, ls);
}

// ------------------------------------------------------------------ selection

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

// Order-preserving map of a float key to uint32 (larger key -> larger integer), so the
// warp's hardware integer max reduction finds the largest key in one instruction.  -0 is
// folded to +0 first so the two compare equal, as the floats do.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_of(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 u, float (&v)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// ------------------------------------------------------------------ exact re-decision
// Rows whose k-th/(k+1)-th margin lies inside the fp32 error bound are listed by the
// selection kernel and re-decided by router_refine_kernel, one CTA per listed row.  The
// CTA's threads share the reduction over H: each product x*w is split exactly by FMA
// (p + e = x*w) and added to a double-fp32 (hi, lo) accumulator with TwoSum (Knuth); the
// per-thread pairs are combined by warp shuffles, then across warps in a fixed order.
// The sums carry ~48 significant bits - far below the 1e-6 key margins that matter - and
// no float64 arithmetic runs in the loop.
constexpr int kRefineBatch = 8;       // band experts per pass over H
constexpr int kRefineThreads = 256;
constexpr int kRefineWarps = kRefineThreads / 32;

template <typename TX>
__device__ void exact_logits_cta(const RouterArgs& a, int t, const int* ce, int nb,
                                 float2 (*part)[kRefineBatch], double* out) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  float sh[kRefineBatch], sl[kRefineBatch];
#pragma unroll
  for (int c = 0; c < kRefineBatch; ++c) sh[c] = sl[c] = 0.f;
  const TX* xr = static_cast<const TX*>(a.X) + (size_t)t * a.H;
  if (a.wsplit) {
    // transposed bf16 pieces (tensor-core path: bf16 X, H % 64 == 0); 8 consecutive h per
    // 16-byte load; w = hi + mid + lo is exact in fp32
    const int nvec = a.H / 8;
    const uint4* x4 = reinterpret_cast<const uint4*>(xr);
    for (int v = tid; v < nvec; v += kRefineThreads) {
      float x[8];
      unpack_bf16x8(x4[v], x);
#pragma unroll
      for (int c = 0; c < kRefineBatch; ++c) {
        if (c < nb) {
          const uint4* w4 = reinterpret_cast<const uint4*>(a.wsplit + (size_t)ce[c] * 3 * a.H);
          float w0[8], w1[8], w2[8];
          unpack_bf16x8(w4[v], w0);
          unpack_bf16x8(w4[v + nvec], w1);
          unpack_bf16x8(w4[v + 2 * nvec], w2);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float wv = (w0[i] + w1[i]) + w2[i];
            const float p = x[i] * wv;
            const float e = fmaf(x[i], wv, -p);   // exact rounding error of the product
            two_sum(sh[c], sl[c], p);
            sl[c] += e;
          }
        }
      }
    }
  } else {
    for (int h = tid; h < a.H; h += kRefineThreads) {
      const float x = load_x1<TX>(xr, h);
      const float* wr = a.Wg + (size_t)h * a.E;
#pragma unroll
      for (int c = 0; c < kRefineBatch; ++c) {
        if (c < nb) {
          const float wv = wr[ce[c]];
          const float p = x * wv;
          const float e = fmaf(x, wv, -p);
          two_sum(sh[c], sl[c], p);
          sl[c] += e;
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kRefineBatch; ++c) {
    float h0 = sh[c], l0 = sl[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float h2 = __shfl_xor_sync(0xffffffffu, h0, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l0, o);
      two_sum(h0, l0, h2);
      l0 += l2;
    }
    if (lane == 0) part[w][c] = make_float2(h0, l0);
  }
  __syncthreads();
  if (tid < nb) {
    float h0 = part[0][tid].x, l0 = part[0][tid].y;
#pragma unroll
    for (int q = 1; q < kRefineWarps; ++q) {
      two_sum(h0, l0, part[q][tid].x);
      l0 += part[q][tid].y;
    }
    double v = (double)h0 + (double)l0;
    if (a.logit_bias) v += (double)a.logit_bias[ce[tid]];
    out[tid] = v;
  }
  __syncthreads();
}

constexpr int kSelWarps = 8;

// One row as the warp sees it: lane `lane` owns experts lane + 32 j, j < NJ.
template <int NJ>
struct RowKeys {
  float l[NJ], sg[NJ];
  uint32_t ok[NJ];     // order-preserving integer form of the fp32 selection key
  uint32_t have;       // bit j: expert lane + 32 j exists
  float lmax, amax;
};

// Logits and fp32 keys of row t.  first: slot 0 holds the (hi, lo) sum of the split-K
// partials; the fixed logit offset is added and (l, 0) written back.  Otherwise slot 0
// already holds (l, 0).
template <int NJ>
__device__ __forceinline__ void load_row(const RouterArgs& a, int t, int lane, bool first,
                                         RowKeys<NJ>& r) {
  const bool sigm = a.score == MOE_SCORE_SIGMOID;
  r.have = 0;
  r.lmax = -INFINITY;
  r.amax = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    r.l[j] = -INFINITY;
    r.sg[j] = 0.f;
    r.ok[j] = 0u;
    if (e < a.E) {
      const float2 pz = a.logits[(size_t)t * a.E + e];
      float hs = pz.x, ls = pz.y;
      if (first && a.logit_bias) two_sum(hs, ls, a.logit_bias[e]);
      const float lv = hs + ls;
      if (first) a.logits[(size_t)t * a.E + e] = make_float2(lv, 0.f);
      r.l[j] = lv;
      r.lmax = fmaxf(r.lmax, lv);
      r.amax = fmaxf(r.amax, fabsf(lv));
      float kv = lv;
      if (sigm) {
        r.sg[j] = __fdividef(1.f, 1.f + __expf(-lv));
        kv = r.sg[j] + (a.bias ? a.bias[e] : 0.f);
      }
      r.ok[j] = ordered_key(kv != kv ? -INFINITY : kv);
      r.have |= 1u << j;
    }
  }
  r.lmax = warp_max_f(r.lmax);
  r.amax = warp_max_f(r.amax);
}

// Top-k (and the (k+1)-th key if `next`) by repeated warp max: hardware max of the
// ordered keys, then the lowest expert index holding that key.  Returns the chosen set as
// a per-lane bitmask.  Only experts with their `have` bit set take part.
template <int NJ>
__device__ __forceinline__ uint32_t topk_row(const RowKeys<NJ>& r, int k, bool next, int lane,
                                             float& kth, float& k1th) {
  uint32_t taken = 0;
  kth = 0.f;
  k1th = -INFINITY;
  const int rounds = next ? k + 1 : k;
  for (int q = 0; q < rounds; ++q) {
    uint32_t mine = 0u;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if ((r.have & ~taken) >> j & 1u) mine = max(mine, r.ok[j]);
    const uint32_t best = __reduce_max_sync(0xffffffffu, mine);
    uint32_t my_e = 0xffffffffu;
#pragma unroll
    for (int j = NJ - 1; j >= 0; --j)
      if (((r.have & ~taken) >> j & 1u) && r.ok[j] == best) my_e = lane + 32 * j;
    const uint32_t win = __reduce_min_sync(0xffffffffu, my_e);
    if (q < k) {
      if (win != 0xffffffffu && (int)(win & 31u) == lane) taken |= 1u << (win >> 5);
      kth = key_of(best);
    } else {
      k1th = key_of(best);
    }
  }
  return taken;
}

// Gates of the chosen experts (each computed by the lane that owns the expert), written
// in ascending expert order with the key gap; optionally the row's probabilities are
// added to `col`.
template <int NJ>
__device__ __forceinline__ void finish_row(const RouterArgs& a, int t, int lane,
                                           const RowKeys<NJ>& r, uint32_t taken, float gap,
                                           float (*col)[NJ]) {
  const bool sigm = a.score == MOE_SCORE_SIGMOID;
  const int k = a.k;
  const uint32_t lt_mask = (1u << lane) - 1u;
  float zsum = 0.f, ssum = 0.f, csum = 0.f;
  float num[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    num[j] = 0.f;
    if (r.have >> j & 1u) {
      if (sigm) {
        ssum += r.sg[j];
        num[j] = r.sg[j];
      } else {
        num[j] = __expf(r.l[j] - r.lmax);
        zsum += num[j];
      }
      if (taken >> j & 1u) csum += num[j];
    }
  }
  zsum = warp_sum_f(zsum);
  ssum = warp_sum_f(ssum);
  csum = warp_sum_f(csum);
  uint32_t B[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) B[j] = __ballot_sync(0xffffffffu, (taken >> j) & 1u);
  int base = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    if (taken >> j & 1u) {
      const int pos = base + __popc(B[j] & lt_mask);
      float g;
      if (a.renorm) g = __fdividef(num[j], csum);
      else g = sigm ? num[j] : __fdividef(num[j], zsum);
      a.idx[(size_t)t * k + pos] = lane + 32 * j;
      a.gate[(size_t)t * k + pos] = g;
    }
    base += __popc(B[j]);
  }
  if (lane == 0 && a.gap) a.gap[t] = gap;
  if (col) {
    const float inv = __fdividef(1.f, sigm ? ssum : zsum);
#pragma unroll
    for (int j = 0; j < NJ; ++j) (*col)[j] += num[j] * inv;
  }
}

// ------------------------------------------------------------------ group-limited routing
// "LLM Internals §14.2.3" (node-limited routing) and "MoE 03: efficiency frontiers"
// (DeepSeek's hardware-aware design): the experts sit in n_groups groups of consecutive
// indices; a group's score is the sum of its k / topk_groups largest affinities (the
// unbiased sigmoid s, or the softmax probability); a token may use only the experts of
// its topk_groups best groups (ties to the lower group), and takes its top k keys among
// them.

struct GroupPick {
  uint32_t sel;    // bit g: group g is used
  uint32_t cand;   // bit g: group g's score is within 2 err of the M-th (a superset of sel)
  float gap;       // S_(M) - S_(M+1), +inf if every group is used
};

// Scores of all groups from fp32 affinities (lane g < G ends up with group g's score),
// then the M best.  err: error bound of one group score.
template <int NJ>
__device__ __forceinline__ GroupPick pick_groups(const RouterArgs& a, uint32_t have,
                                                 const float (&aff)[NJ], int lane, float err) {
  const int G = a.n_groups, M = a.topk_groups, gs = a.E / G, n = a.k / M;
  uint32_t oa[NJ];
  int grp[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    oa[j] = ordered_key(aff[j]);
    grp[j] = (lane + 32 * j) / gs;
  }
  float my_s = 0.f;
  for (int g = 0; g < G; ++g) {
    uint32_t left = 0;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if ((have >> j & 1u) && grp[j] == g) left |= 1u << j;
    float sum = 0.f;
    for (int q = 0; q < n; ++q) {   // largest first; which of equal values goes is moot
      uint32_t mine = 0u;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (left >> j & 1u) mine = max(mine, oa[j]);
      const uint32_t best = __reduce_max_sync(0xffffffffu, mine);
      uint32_t my_e = 0xffffffffu;
#pragma unroll
      for (int j = NJ - 1; j >= 0; --j)
        if ((left >> j & 1u) && oa[j] == best) my_e = lane + 32 * j;
      const uint32_t win = __reduce_min_sync(0xffffffffu, my_e);
      if (win != 0xffffffffu && (int)(win & 31u) == lane) left &= ~(1u << (win >> 5));
      sum += key_of(best);
    }
    if (lane == g) my_s = sum;
  }
  GroupPick gp;
  gp.sel = 0u;
  const uint32_t os = ordered_key(my_s);
  bool in = lane < G;
  float sM = 0.f, sM1 = -INFINITY;
  const int rounds = M < G ? M + 1 : M;
  for (int q = 0; q < rounds; ++q) {
    const uint32_t best = __reduce_max_sync(0xffffffffu, in ? os : 0u);
    const uint32_t win =
        __reduce_min_sync(0xffffffffu, (in && os == best) ? (uint32_t)lane : 0xffffffffu);
    if (q < M) {
      gp.sel |= 1u << win;
      sM = key_of(best);
      if (lane == (int)win) in = false;
    } else {
      sM1 = key_of(best);
    }
  }
  gp.gap = M < G ? sM - sM1 : INFINITY;
  gp.cand = __ballot_sync(0xffffffffu, lane < G && my_s >= sM - 2.f * err);
  return gp;
}

// Per-lane mask of the experts (lane + 32 j) that belong to a group of `groups`.
template <int NJ>
__device__ __forceinline__ uint32_t experts_of(const RouterArgs& a, uint32_t have,
                                               uint32_t groups, int lane) {
  const int gs = a.E / a.n_groups;
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if ((have >> j & 1u) && (groups >> ((lane + 32 * j) / gs) & 1u)) m |= 1u << j;
  return m;
}

// One warp per token: keys, top-(k+1), gates, key gap, row probabilities.  A row whose
// margin is within twice the error bound of its fp32 keys (or, group-limited, of its group
// scores) is listed for router_refine_kernel; its outputs here are provisional.
// GRP: group-limited routing (a separate instantiation: the plain kernel keeps its
// registers).
template <typename TX, int NJ, bool GRP>
__global__ void __launch_bounds__(kSelWarps * 32) router_select_kernel(RouterArgs a,
                                                                      int tok_per_warp) {
  __shared__ float s_col[kSelWarps][NJ * 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int E = a.E, k = a.k;
  const bool sigm = a.score == MOE_SCORE_SIGMOID;
  const float h_scale = sqrtf(fmaxf(1.f, a.H / 1024.f));

  float col[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) col[j] = 0.f;

  const int tbeg = (blockIdx.x * kSelWarps + w) * tok_per_warp;
  for (int t = tbeg; t < min(tbeg + tok_per_warp, a.T); ++t) {
    RowKeys<NJ> r;
    load_row<NJ>(a, t, lane, true, r);
    // error bound of the fp32 logits and of the fp32 keys derived from them
    const float eps_l = a.eps_rel * fmaxf(1.f, r.amax) * h_scale;
    const float eps = sigm ? 0.25f * eps_l + ldexpf(1.f, -20) : eps_l;
    if (GRP) {
      // affinities: s, or p = exp(l - lmax) / sum (moves by <= 2.01 eps_l p when every
      // logit moves by eps_l, plus fp32 rounding of exp, the row sum and the quotient)
      float aff[NJ];
      float zs = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        aff[j] = 0.f;
        if (r.have >> j & 1u) aff[j] = sigm ? r.sg[j] : __expf(r.l[j] - r.lmax);
        if (aff[j] != aff[j]) aff[j] = 0.f;
        zs += aff[j];
      }
      if (!sigm) {
        zs = warp_sum_f(zs);
#pragma unroll
        for (int j = 0; j < NJ; ++j) aff[j] = __fdividef(aff[j], zs);
      }
      const int n = k / a.topk_groups;
      const float eps_a = sigm ? eps : 2.5f * eps_l + ldexpf(1.f, -18);
      const float err_g = n * (eps_a + n * ldexpf(1.f, -23));
      const GroupPick gp = pick_groups<NJ>(a, r.have, aff, lane, err_g);
      RowKeys<NJ> re = r;
      re.have = experts_of<NJ>(a, r.have, gp.sel, lane);
      const bool next = a.topk_groups * (E / a.n_groups) > k;
      float kth, k1th;
      const uint32_t taken = topk_row<NJ>(re, k, next, lane, kth, k1th);
      const float k_gap = next ? kth - k1th : INFINITY;
      if ((!(gp.gap > 2.f * err_g) || !(k_gap > 2.f * eps)) && lane == 0) {
        // Exactness guard.  A group whose fp32 score is below S_(M) - 2 err is below the
        // M groups chosen here in exact arithmetic too, so the exact choice lies among
        // the candidate groups; the refine kernel re-decides from their exact logits.
        const int slot = atomicAdd(a.refined, 1);
        a.refine_list[slot] = make_int4(t, (int)gp.cand, __float_as_int(gp.gap), 1);
      }
      finish_row<NJ>(a, t, lane, r, taken, fminf(gp.gap, k_gap), a.colsum ? &col : nullptr);
      continue;
    }
    float kth, k1th;
    const uint32_t taken = topk_row<NJ>(r, k, k < E, lane, kth, k1th);
    const float gap = (k < E) ? kth - k1th : INFINITY;
    if (k < E && !(gap > 2.f * eps) && lane == 0) {
      // Exactness guard.  With |approx - exact| <= eps for every key, an expert whose
      // approximate key exceeds k1th + 2 eps beats every expert outside the approximate
      // top k, so it is in the exact top k ("sure"); any other member of the exact top k
      // has an approximate key >= kth - 2 eps.  Only the band between the two limits
      // needs exact keys.
      const int slot = atomicAdd(a.refined, 1);
      a.refine_list[slot] = make_int4(t, __float_as_int(kth - 2.f * eps),
                                      __float_as_int(k1th + 2.f * eps), 0);
    }
    finish_row<NJ>(a, t, lane, r, taken, gap, a.colsum ? &col : nullptr);
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

// Warp-wide argmax of a double per lane (ties to the lower index); bi = 0x7fffffff if
// no lane offers a value.
__device__ __forceinline__ void warp_argmax_d(double& bk, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double k2 = __shfl_xor_sync(0xffffffffu, bk, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (k2 > bk || (k2 == bk && i2 < bi)) {
      bk = k2;
      bi = i2;
    }
  }
}

// The n-th largest of the ordered values oa[j] over the experts in `members` (per-lane
// masks), as a float; -inf if there are fewer than n.
template <int NJ>
__device__ __forceinline__ float nth_largest(const uint32_t (&oa)[NJ], uint32_t members, int n,
                                             int lane) {
  float v = -INFINITY;
  for (int q = 0; q < n; ++q) {
    uint32_t mine = 0u;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (members >> j & 1u) mine = max(mine, oa[j]);
    const uint32_t best = __reduce_max_sync(0xffffffffu, mine);
    uint32_t my_e = 0xffffffffu;
#pragma unroll
    for (int j = NJ - 1; j >= 0; --j)
      if ((members >> j & 1u) && oa[j] == best) my_e = lane + 32 * j;
    const uint32_t win = __reduce_min_sync(0xffffffffu, my_e);
    if (win == 0xffffffffu) return -INFINITY;
    if ((int)(win & 31u) == lane) members &= ~(1u << (win >> 5));
    v = key_of(best);
  }
  return v;
}

// Writes the experts of the per-lane masks `m` to s_ce in ascending order; returns the
// count (all lanes).
template <int NJ>
__device__ __forceinline__ int list_experts(uint32_t m, int lane, int* s_ce) {
  const uint32_t lt_mask = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const uint32_t B = __ballot_sync(0xffffffffu, (m >> j) & 1u);
    if (m >> j & 1u) s_ce[base + __popc(B & lt_mask)] = lane + 32 * j;
    base += __popc(B);
  }
  return base;
}

// Reads back into lane registers the exact logits of the experts listed by list_experts(m).
template <int NJ>
__device__ __forceinline__ void take_exact(uint32_t m, int lane, const double* s_ex,
                                           double (&ex)[NJ]) {
  const uint32_t lt_mask = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const uint32_t B = __ballot_sync(0xffffffffu, (m >> j) & 1u);
    if (m >> j & 1u) ex[j] = s_ex[base + __popc(B & lt_mask)];
    base += __popc(B);
  }
}

// Group-limited re-decision of row t, in two rounds of exact logits.
//  1. Group scores.  In a candidate group (cmask), an expert whose fp32 affinity is below
//     the group's n-th largest minus 2 eps_a is below n others in exact arithmetic too;
//     the exact top n of the group lies among the rest, so their exact logits give the
//     exact score.  The M best candidates by exact score are the groups used.
//  2. Experts.  Among the experts of those groups, the band of the fp32 keys
//     [kth - 2 eps, k1th + 2 eps] as in the plain re-decision: experts above it are sure
//     members, the band is ranked on exact keys (computed now unless step 1 did).
// approx_gap: the fp32 group margin, reported when no other candidate group is left to
// measure the exact margin against.
template <typename TX, int NJ>
__device__ void refine_group_row(const RouterArgs& a, int t, uint32_t cmask, float approx_gap,
                                 int* s_ce, double* s_ex, float2 (*s_part)[kRefineBatch],
                                 int* s_nband) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int k = a.k, G = a.n_groups, M = a.topk_groups, n = k / M;
  const bool sigm = a.score == MOE_SCORE_SIGMOID;
  const float h_scale = sqrtf(fmaxf(1.f, a.H / 1024.f));
  RowKeys<NJ> r;
  float zs = 1.f, eps = 0.f, kth = 0.f, k1th = -INFINITY, g_gap = approx_gap;
  uint32_t known = 0, cand2 = 0, sure = 0;
  double ex[NJ];
  if (w == 0) {
    load_row<NJ>(a, t, lane, false, r);
    const float eps_l = a.eps_rel * fmaxf(1.f, r.amax) * h_scale;
    eps = sigm ? 0.25f * eps_l + ldexpf(1.f, -20) : eps_l;
    const float eps_a = sigm ? eps : 2.5f * eps_l + ldexpf(1.f, -18);
    float aff[NJ];
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      aff[j] = 0.f;
      if (r.have >> j & 1u) aff[j] = sigm ? r.sg[j] : __expf(r.l[j] - r.lmax);
      if (aff[j] != aff[j]) aff[j] = 0.f;
      z += aff[j];
    }
    if (!sigm) {
      zs = warp_sum_f(z);
#pragma unroll
      for (int j = 0; j < NJ; ++j) aff[j] = __fdividef(aff[j], zs);
    }
    uint32_t oa[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) oa[j] = ordered_key(aff[j]);
    // with exactly M candidates the groups are already decided
    for (int g = 0; g < G && __popc(cmask) > M; ++g) {
      if (!(cmask >> g & 1u)) continue;
      const uint32_t mem = experts_of<NJ>(a, r.have, 1u << g, lane);
      const float lim = nth_largest<NJ>(oa, mem, n, lane) - 2.f * eps_a;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if ((mem >> j & 1u) && aff[j] >= lim) known |= 1u << j;
    }
    const int nb = list_experts<NJ>(known, lane, s_ce);
    if (lane == 0) *s_nband = nb;
  }
  __syncthreads();
  int nband = *s_nband;
  for (int b0 = 0; b0 < nband; b0 += kRefineBatch)
    exact_logits_cta<TX>(a, t, s_ce + b0, min(kRefineBatch, nband - b0), s_part, s_ex + b0);
  if (w == 0) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) ex[j] = 0.0;
    take_exact<NJ>(known, lane, s_ex, ex);
    // exact affinities (softmax: scaled by the row's fp32 maximum and sum, which orders
    // the groups as the exact probabilities do)
    double ea[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      ea[j] = !(known >> j & 1u) ? 0.0
              : sigm ? 1.0 / (1.0 + exp(-ex[j])) : exp(ex[j] - (double)r.lmax) / (double)zs;
    double my_s = -INFINITY;   // lane g: exact score of candidate group g
    for (int g = 0; g < G && __popc(cmask) > M; ++g) {
      if (!(cmask >> g & 1u)) continue;
      uint32_t left = experts_of<NJ>(a, known, 1u << g, lane);
      double sum = 0.0;
      for (int q = 0; q < n; ++q) {
        double bk = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
          if ((left >> j & 1u) && (ea[j] > bk || (ea[j] == bk && lane + 32 * j < bi))) {
            bk = ea[j];
            bi = lane + 32 * j;
          }
        warp_argmax_d(bk, bi);
        if (bi == 0x7fffffff) break;
        if ((bi & 31) == lane) left &= ~(1u << (bi >> 5));
        sum += bk;
      }
      if (lane == g) my_s = sum;
    }
    uint32_t sel = __popc(cmask) > M ? 0u : cmask;
    bool in = lane < G && (cmask >> lane & 1u);
    double sM = 0.0, sM1 = -INFINITY;
    for (int q = 0; q <= M && __popc(cmask) > M; ++q) {
      double bk = in ? my_s : -INFINITY;
      int bi = in ? lane : 0x7fffffff;
      warp_argmax_d(bk, bi);
      if (bi == 0x7fffffff) break;
      if (q < M) {
        sel |= 1u << bi;
        sM = bk;
        if (lane == bi) in = false;
      } else {
        sM1 = bk;
      }
    }
    if (sM1 != -INFINITY) g_gap = (float)(sM - sM1);
    // the key band among the experts of the chosen groups
    RowKeys<NJ> re = r;
    re.have = experts_of<NJ>(a, r.have, sel, lane);
    const bool next = M * (a.E / G) > k;
    topk_row<NJ>(re, k, next, lane, kth, k1th);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const float kv = key_of(r.ok[j]);
      if ((re.have >> j & 1u) && kv >= kth - 2.f * eps) {
        cand2 |= 1u << j;
        if (kv > k1th + 2.f * eps) sure |= 1u << j;
      }
    }
    const int nb = list_experts<NJ>(cand2 & ~sure & ~known, lane, s_ce);
    if (lane == 0) *s_nband = nb;
  }
  __syncthreads();
  const int nband2 = *s_nband;
  for (int b0 = 0; b0 < nband2; b0 += kRefineBatch)
    exact_logits_cta<TX>(a, t, s_ce + b0, min(kRefineBatch, nband2 - b0), s_part, s_ex + b0);
  if (w == 0) {
    take_exact<NJ>(cand2 & ~sure & ~known, lane, s_ex, ex);
    double ek[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (!(cand2 >> j & 1u)) {
        ek[j] = -INFINITY;
      } else if (sure >> j & 1u) {
        ek[j] = INFINITY;
      } else {
        ek[j] = sigm ? 1.0 / (1.0 + exp(-ex[j])) + (a.bias ? (double)a.bias[lane + 32 * j] : 0.0)
                     : ex[j];
      }
    }
    uint32_t tk = 0;
    double dk = 0.0, dk1 = -INFINITY;
    for (int q = 0; q <= k; ++q) {
      double bk = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        if ((cand2 >> j & 1u) && !(tk >> j & 1u) && (ek[j] > bk || (ek[j] == bk && e < bi))) {
          bk = ek[j];
          bi = e;
        }
      }
      warp_argmax_d(bk, bi);
      if (bi == 0x7fffffff) break;
      if (q < k) {
        if ((bi & 31) == lane) tk |= 1u << (bi >> 5);
        dk = bk;
      } else {
        dk1 = bk;
      }
    }
    // the exact key margin where the band decided it, else the fp32 one
    const float k_gap = dk1 == -INFINITY ? INFINITY
                        : (dk == INFINITY || dk1 == INFINITY) ? kth - k1th : (float)(dk - dk1);
    finish_row<NJ>(a, t, lane, r, tk, fminf(g_gap, k_gap), nullptr);
  }
  __syncthreads();   // s_ce / s_ex are reused by the next listed row
}

// One CTA per listed row (grid-stride over the list): exact logits of the band experts
// (CTA-wide), then warp 0 re-decides the row among its candidates on the exact keys
// (ties to the lower index; sure experts rank first) and rewrites its outputs.
template <typename TX, int NJ, bool GRP>
__global__ void __launch_bounds__(kRefineThreads) router_refine_kernel(RouterArgs a) {
  __shared__ int s_ce[kMaxE];        // band experts, ascending
  __shared__ double s_ex[kMaxE];     // their exact keys
  __shared__ float2 s_part[kRefineWarps][kRefineBatch];
  __shared__ int s_nband;
  const int n = *a.refined;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int k = a.k;
  const bool sigm = a.score == MOE_SCORE_SIGMOID;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int4 ent = a.refine_list[i];
    const int t = ent.x;
    if (GRP) {
      refine_group_row<TX, NJ>(a, t, (uint32_t)ent.y, __int_as_float(ent.z), s_ce, s_ex,
                               s_part, &s_nband);
      continue;
    }
    const float lim = __int_as_float(ent.y), sure = __int_as_float(ent.z);
    RowKeys<NJ> r;
    uint32_t cand = 0, band = 0;
    if (w == 0) {
      load_row<NJ>(a, t, lane, false, r);
      int base = 0;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const float kv = key_of(r.ok[j]);
        if ((r.have >> j & 1u) && kv >= lim) {
          cand |= 1u << j;
          if (!(kv > sure)) band |= 1u << j;
        }
        const uint32_t M = __ballot_sync(0xffffffffu, (band >> j) & 1u);
        if (band >> j & 1u) s_ce[base + __popc(M & lt_mask)] = lane + 32 * j;
        base += __popc(M);
      }
      if (lane == 0) s_nband = base;
    }
    __syncthreads();
    const int nband = s_nband;
    for (int b0 = 0; b0 < nband; b0 += kRefineBatch)
      exact_logits_cta<TX>(a, t, s_ce + b0, min(kRefineBatch, nband - b0), s_part, s_ex + b0);
    if (sigm) {
      for (int c = threadIdx.x; c < nband; c += blockDim.x) {
        double kv = 1.0 / (1.0 + exp(-s_ex[c]));
        if (a.bias) kv += (double)a.bias[s_ce[c]];
        s_ex[c] = kv;
      }
      __syncthreads();
    }
    if (w == 0) {
      double ex[NJ];
      int base = 0;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const uint32_t M = __ballot_sync(0xffffffffu, (band >> j) & 1u);
        ex[j] = !(cand >> j & 1u) ? -INFINITY
                : (band >> j & 1u) ? s_ex[base + __popc(M & lt_mask)] : INFINITY;
        base += __popc(M);
      }
      uint32_t tk = 0;
      double dk = 0.0, dk1 = -INFINITY;
      for (int q = 0; q <= k; ++q) {
        double bk = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int e = lane + 32 * j;
          if ((cand >> j & 1u) && !(tk >> j & 1u) && (ex[j] > bk || (ex[j] == bk && e < bi))) {
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
        if (bi == 0x7fffffff) break;
        if (q < k) {
          if ((bi & 31) == lane) tk |= 1u << (bi >> 5);
          dk = bk;
        } else {
          dk1 = bk;
        }
      }
      finish_row<NJ>(a, t, lane, r, tk, (float)(dk - dk1), nullptr);
    }
    __syncthreads();   // s_ce / s_ex are reused by the next listed row
  }
}

// ------------------------------------------------------------------ expert-choice routing
// "LLM Internals §14.2" (the two selection paradigms: expert-choice) and "MoE 03:
// efficiency frontiers" (Expert Choice Routing): every expert takes the C tokens of the
// batch with the largest affinity S[t, e] - the softmax probability over the experts, or
// the sigmoid s - with ties to the lower token index.  Exactness as for token choice: a
// column whose C-th/(C+1)-th margin lies within twice the error bound of its fp32
// affinities waits for the exact affinities of the tokens in its band.

constexpr int kEcThreads = 1024;

__device__ __forceinline__ uint64_t ordered_key64(double d) {
  const uint64_t u = (uint64_t)__double_as_longlong(d + 0.0);
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double key_of64(uint64_t o) {
  return __longlong_as_double((long long)((o >> 63) ? (o & 0x7fffffffffffffffull) : ~o));
}

// Exclusive prefix sum of one int per thread over a block of kEcThreads (32 warps).
__device__ __forceinline__ int block_excl_scan(int v, int* s_w) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[w] = x;
  __syncthreads();
  if (w == 0) {
    const int y = s_w[lane];
    int z = y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int q = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += q;
    }
    s_w[lane] = z - y;
  }
  __syncthreads();
  const int res = s_w[w] + x - v;
  __syncthreads();
  return res;
}

// The rank-th largest key (rank >= 1, at most the number of active items) among the
// items i < n for which get(i, key) is true: most significant byte first, one 256-bin
// histogram per byte.  Affinities crowd into a few bins (their leading bytes agree), so
// the lanes of a warp that fall into the same bin add to it once, with their count.
template <typename K, typename Get>
__device__ K block_radix_select(int n, int rank, Get get, int* hist, K* s_pre, int* s_rem) {
  K prefix = 0, mask = 0;
  int remaining = rank;
  const int lane = threadIdx.x & 31;
  for (int shift = (int)sizeof(K) * 8 - 8; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {   // the same trip count for all
      const int i = base + threadIdx.x;
      K key = 0;
      const bool act = i < n && get(i, key) && (key & mask) == prefix;
      const int digit = act ? (int)((key >> shift) & 255) : -1;
      const unsigned grp = __match_any_sync(0xffffffffu, digit);
      if (act && __ffs(grp) - 1 == lane) atomicAdd(&hist[digit], __popc(grp));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // the bin holding the rank-th largest: lane i sums bins 255 - 8i down to 248 - 8i,
      // a warp scan finds the lane where the count from the top reaches `remaining`,
      // and that lane walks its eight bins
      int c8 = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) c8 += hist[255 - 8 * lane - q];
      int incl = c8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
      const int src = hit ? __ffs(hit) - 1 : 31;
      if (lane == src) {
        int cum = incl - c8, d = 255 - 8 * lane;
        for (int q = 0; q < 7; ++q, --d) {
          if (cum + hist[d] >= remaining) break;
          cum += hist[d];
        }
        *s_pre = prefix | ((K)d << shift);
        *s_rem = remaining - cum;
      }
    }
    __syncthreads();
    prefix = *s_pre;
    remaining = *s_rem;
    mask |= (K)255 << shift;
    __syncthreads();
  }
  return prefix;
}

// fp32 affinities of token t (one warp per token), stored by column; the row's error
// bound |dS| <= abs + rel * S goes into the running maxima.  Softmax: S moves by at most
// (e^{2 eps} - 1) S when every logit moves by eps, plus the rounding of exp, the row sum
// and the quotient; sigmoid: by 0.25 eps plus the rounding of exp and the quotient.
template <int NJ>
__global__ void __launch_bounds__(256) ec_scores_kernel(ExpertChoiceArgs a) {
  const RouterArgs& r = a.r;
  const int lane = threadIdx.x & 31;
  // a warp past the last token takes the last token again (same values, same stores) so
  // that every warp reaches the block's barriers
  const int t = min(blockIdx.x * 8 + (threadIdx.x >> 5), r.T - 1);
  const bool sigm = r.score == MOE_SCORE_SIGMOID;
  float l[NJ];
  float lmax = -INFINITY, amax = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    l[j] = -INFINITY;
    if (e < r.E) {
      const float2 pz = r.logits[(size_t)t * r.E + e];
      float hs = pz.x, ls = pz.y;
      if (r.logit_bias) two_sum(hs, ls, r.logit_bias[e]);
      l[j] = hs + ls;
      lmax = fmaxf(lmax, l[j]);
      amax = fmaxf(amax, fabsf(l[j]));
    }
  }
  lmax = warp_max_f(lmax);
  amax = warp_max_f(amax);
  const float eps_l = r.eps_rel * fmaxf(1.f, amax) * sqrtf(fmaxf(1.f, r.H / 1024.f));
  float S[NJ];
  float z = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    S[j] = 0.f;
    if (lane + 32 * j < r.E)
      S[j] = sigm ? __fdividef(1.f, 1.f + __expf(-l[j])) : __expf(l[j] - lmax);
    z += S[j];
  }
  if (!sigm) {
    z = warp_sum_f(z);
#pragma unroll
    for (int j = 0; j < NJ; ++j) S[j] = __fdividef(S[j], z);
  }
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    if (e < r.E) a.St[(size_t)e * r.T + t] = S[j] == S[j] ? S[j] : 0.f;
  }
  // the block's largest bounds, then one update of the running maxima per block
  // (non-negative floats order as their bit patterns)
  __shared__ int s_rel, s_abs;
  if (threadIdx.x == 0) s_rel = s_abs = 0;
  __syncthreads();
  if (lane == 0) {
    const float rel = sigm ? 0.f : 2.1f * eps_l + ldexpf(1.f, -18);
    const float ab = sigm ? 0.25f * eps_l + ldexpf(1.f, -20) : ldexpf(1.f, -24);
    atomicMax(&s_rel, __float_as_int(rel));
    atomicMax(&s_abs, __float_as_int(ab));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicMax(&a.ctr[2], s_rel);
    atomicMax(&a.ctr[3], s_abs);
  }
}

struct EcShared {
  int hist[256];
  int w[32];
  int cnt[3];
  unsigned long long mx;
  uint64_t pre;
  int rem;
};

// Writes expert e's column from the membership flags s_in[t]: its rows e*C + i hold its
// tokens in ascending order.
__device__ void ec_write_column(const ExpertChoiceArgs& a, int e, const uint8_t* s_in,
                                const uint32_t* s_key, EcShared& sh) {
  const int T = a.r.T, E = a.r.E, C = a.C;
  const int per = (T + kEcThreads - 1) / kEcThreads;
  const int t0 = threadIdx.x * per, t1 = min(T, t0 + per);
  int c = 0;
  for (int t = t0; t < t1; ++t) c += s_in[t];
  int pos = block_excl_scan(c, sh.w);
  for (int t = t0; t < t1; ++t) {
    if (!s_in[t]) continue;
    if (pos >= C) break;   // cannot happen: exactly C members
    const int row = e * C + pos++;
    const int slot = t * E + e;
    a.slot_of_row[row] = slot;
    a.row_of_slot[slot] = row;
    a.gate[slot] = key_of(s_key[t]);
  }
}

// One CTA per expert: the C-th largest fp32 affinity of its column by radix select, the
// (C+1)-th, and either the column's tokens (margin above twice the error bound) or a
// listing of the column and of its band tokens for the exact path.
__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(ExpertChoiceArgs a) {
  extern __shared__ uint32_t s_key[];
  uint8_t* s_in = reinterpret_cast<uint8_t*>(s_key + a.r.T);
  __shared__ EcShared sh;
  const int e = blockIdx.x, T = a.r.T, C = a.C, tid = threadIdx.x;
  for (int t = tid; t < T; t += kEcThreads) s_key[t] = ordered_key(a.St[(size_t)e * T + t]);
  if (tid == 0) {
    a.offsets[e] = e * C;
    if (e == 0) a.offsets[a.r.E] = a.r.E * C;
    sh.cnt[0] = sh.cnt[1] = 0;
    sh.mx = 0ull;
  }
  __syncthreads();
  if (C == 0 || C >= T) {
    for (int t = tid; t < T; t += kEcThreads) s_in[t] = C > 0;
    __syncthreads();
    if (C > 0) ec_write_column(a, e, s_in, s_key, sh);
    if (tid == 0 && a.gap) a.gap[e] = INFINITY;
    return;
  }
  __shared__ uint32_t s_pre32;
  const uint32_t tau = block_radix_select<uint32_t>(
      T, C, [&](int i, uint32_t& k) { k = s_key[i]; return true; }, sh.hist, &s_pre32,
      &sh.rem);
  int gt = 0, eq = 0;
  uint32_t below = 0u;
  for (int t = tid; t < T; t += kEcThreads) {
    const uint32_t k = s_key[t];
    gt += k > tau;
    eq += k == tau;
    if (k < tau) below = max(below, k);
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  below = __reduce_max_sync(0xffffffffu, below);
  if ((tid & 31) == 0) {
    atomicAdd(&sh.cnt[0], gt);
    atomicAdd(&sh.cnt[1], eq);
    atomicMax(&sh.mx, (unsigned long long)below);
  }
  __syncthreads();
  gt = sh.cnt[0];
  eq = sh.cnt[1];
  const uint32_t next = gt + eq > C ? tau : (uint32_t)sh.mx;   // the (C+1)-th largest
  const float ftau = key_of(tau), fnext = key_of(next);
  const float err = __int_as_float(a.ctr[3]) + __int_as_float(a.ctr[2]) * ftau;
  const float gapf = ftau - fnext;
  if (!(gapf > 2.f * err)) {
    // Exactness guard.  With |dS| <= err near the boundary, a token above fnext + 2 err
    // is in the exact top C and one below ftau - 2 err is not; the band between needs
    // exact affinities.
    const float lo = ftau - 2.f * err, hi = fnext + 2.f * err;
    for (int t = tid; t < T; t += kEcThreads) {
      const float v = key_of(s_key[t]);
      if (v >= lo && !(v > hi) && atomicExch(&a.need[t], 1) == 0)
        a.tok_list[atomicAdd(&a.ctr[0], 1)] = t;
    }
    if (tid == 0) {
      a.col_list[atomicAdd(&a.ctr[1], 1)] = e;
      // the band limits themselves, so that the fix-up sees the very same band
      a.col_info[e] = make_int4(__float_as_int(lo), __float_as_int(hi), __float_as_int(gapf), 0);
    }
    return;
  }
  // members: every key above tau, then the C - gt lowest tokens whose key equals tau
  const int per = (T + kEcThreads - 1) / kEcThreads;
  const int t0 = tid * per, t1 = min(T, t0 + per);
  int ce = 0;
  for (int t = t0; t < t1; ++t) ce += s_key[t] == tau;
  int rank = block_excl_scan(ce, sh.w);
  for (int t = t0; t < t1; ++t) {
    const uint32_t k = s_key[t];
    s_in[t] = k > tau || (k == tau && rank++ < C - gt);
  }
  __syncthreads();
  ec_write_column(a, e, s_in, s_key, sh);
  if (tid == 0 && a.gap) a.gap[e] = gapf;
}

// One CTA per listed token: exact logits of all its experts, then its exact affinities.
template <typename TX>
__global__ void __launch_bounds__(kRefineThreads) ec_exact_rows_kernel(ExpertChoiceArgs a) {
  __shared__ int s_ce[kMaxE];
  __shared__ double s_ex[kMaxE];
  __shared__ float2 s_part[kRefineWarps][kRefineBatch];
  const int n = a.ctr[0], E = a.r.E;
  const bool sigm = a.r.score == MOE_SCORE_SIGMOID;
  for (int c = threadIdx.x; c < E; c += blockDim.x) s_ce[c] = c;
  __syncthreads();
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int t = a.tok_list[i];
    for (int b0 = 0; b0 < E; b0 += kRefineBatch)
      exact_logits_cta<TX>(a.r, t, s_ce + b0, min(kRefineBatch, E - b0), s_part, s_ex + b0);
    if (threadIdx.x == 0) {
      double* out = a.exS + (size_t)t * E;
      if (sigm) {
        for (int c = 0; c < E; ++c) out[c] = 1.0 / (1.0 + exp(-s_ex[c]));
      } else {
        double m = -INFINITY, z = 0.0;
        for (int c = 0; c < E; ++c) m = fmax(m, s_ex[c]);
        for (int c = 0; c < E; ++c) z += exp(s_ex[c] - m);
        for (int c = 0; c < E; ++c) out[c] = exp(s_ex[c] - m) / z;
      }
    }
    __syncthreads();
  }
}

// One CTA per listed expert: its sure members, then the best of its band tokens by exact
// affinity (ties to the lower token) up to C.
__global__ void __launch_bounds__(kEcThreads) ec_fix_kernel(ExpertChoiceArgs a) {
  extern __shared__ uint32_t s_key[];
  uint8_t* s_in = reinterpret_cast<uint8_t*>(s_key + a.r.T);
  __shared__ EcShared sh;
  const int n = a.ctr[1], T = a.r.T, E = a.r.E, C = a.C, tid = threadIdx.x;
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int e = a.col_list[i];
    const int4 info = a.col_info[e];
    const float lo = __int_as_float(info.x), hi = __int_as_float(info.y);
    for (int t = tid; t < T; t += kEcThreads) s_key[t] = ordered_key(a.St[(size_t)e * T + t]);
    if (tid == 0) {
      sh.cnt[0] = sh.cnt[1] = sh.cnt[2] = 0;
      sh.mx = 0ull;
    }
    __syncthreads();
    // 1 = sure member, 2 = band
    int nsure = 0, nband = 0;
    for (int t = tid; t < T; t += kEcThreads) {
      const float v = key_of(s_key[t]);
      const uint8_t f = v > hi ? 1 : (v >= lo ? 2 : 0);
      s_in[t] = f;
      nsure += f == 1;
      nband += f == 2;
    }
    nsure = __reduce_add_sync(0xffffffffu, nsure);
    nband = __reduce_add_sync(0xffffffffu, nband);
    if ((tid & 31) == 0) {
      atomicAdd(&sh.cnt[0], nsure);
      atomicAdd(&sh.cnt[1], nband);
    }
    __syncthreads();
    const int need = C - sh.cnt[0];
    const int band_n = sh.cnt[1];
    auto exkey = [&](int t) { return ordered_key64(a.exS[(size_t)t * E + e]); };
    uint64_t etau = 0ull;
    if (need > 0 && need <= band_n)
      etau = block_radix_select<uint64_t>(
          T, need,
          [&](int t, uint64_t& k) {
            if (s_in[t] != 2) return false;
            k = exkey(t);
            return true;
          },
          sh.hist, &sh.pre, &sh.rem);
    int gt = 0;
    for (int t = tid; t < T; t += kEcThreads)
      if (s_in[t] == 2 && exkey(t) > etau) ++gt;
    gt = __reduce_add_sync(0xffffffffu, gt);
    if ((tid & 31) == 0) atomicAdd(&sh.cnt[2], gt);
    __syncthreads();
    const int take_eq = need - sh.cnt[2];
    const int per = (T + kEcThreads - 1) / kEcThreads;
    const int t0 = tid * per, t1 = min(T, t0 + per);
    int ce = 0;
    for (int t = t0; t < t1; ++t) ce += s_in[t] == 2 && exkey(t) == etau;
    int rank = block_excl_scan(ce, sh.w);
    unsigned long long best_out = 0ull;   // largest exact key of the band left out
    for (int t = t0; t < t1; ++t) {
      const uint8_t f = s_in[t];
      bool in = f == 1;
      if (f == 2 && need > 0) {
        const uint64_t k = exkey(t);
        in = k > etau || (k == etau && rank++ < take_eq);
      }
      if (f == 2 && !in) best_out = max(best_out, (unsigned long long)exkey(t));
      s_in[t] = in;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best_out = max(best_out, __shfl_xor_sync(0xffffffffu, best_out, o));
    if ((tid & 31) == 0) atomicMax(&sh.mx, best_out);
    __syncthreads();
    ec_write_column(a, e, s_in, s_key, sh);
    if (tid == 0 && a.gap)
      a.gap[e] = (need > 0 && sh.mx) ? (float)(key_of64(etau) - key_of64(sh.mx))
                                     : __int_as_float(info.z);
    __syncthreads();   // shared memory is reused by the next listed expert
  }
}

template <int NJ>
cudaError_t launch_ec_scores(const ExpertChoiceArgs& a, cudaStream_t s) {
  ec_scores_kernel<NJ><<<(a.r.T + 7) / 8, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename TX, int NJ, bool GRP>
cudaError_t launch_select_grp(const RouterArgs& a, cudaStream_t s) {
  // one token per warp up to 2^14 tokens, then more: enough warps to fill the GPU, few
  // enough CTAs that the per-CTA column sums stay cheap
  const int tpw = a.T <= 16384 ? 1 : (a.T + 16383) / 16384;
  const int per_cta = kSelWarps * tpw;
  router_select_kernel<TX, NJ, GRP>
      <<<(a.T + per_cta - 1) / per_cta, kSelWarps * 32, 0, s>>>(a, tpw);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the listed rows are few; most of these CTAs find nothing to do and exit
  const int sms = a.num_sms > 0 ? a.num_sms : 1;
  const int grid = a.T < 8 * sms ? a.T : 8 * sms;
  router_refine_kernel<TX, NJ, GRP><<<grid, kRefineThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename TX, int NJ>
cudaError_t launch_select_nj(const RouterArgs& a, cudaStream_t s) {
  return a.n_groups > 1 ? launch_select_grp<TX, NJ, true>(a, s)
                        : launch_select_grp<TX, NJ, false>(a, s);
}

template <typename TX>
cudaError_t launch_select_t(const RouterArgs& a, cudaStream_t s) {
  if (a.E <= 32) return launch_select_nj<TX, 1>(a, s);
  if (a.E <= 64) return launch_select_nj<TX, 2>(a, s);
  if (a.E <= 128) return launch_select_nj<TX, 4>(a, s);
  if (a.E <= 256) return launch_select_nj<TX, 8>(a, s);
  return launch_select_nj<TX, 16>(a, s);
}

}  // namespace

cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t s) {
  if (a.E <= 16) {
    const dim3 g((a.T + 31) / 32, a.splits);
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
  const dim3 grid((a.T + kTM - 1) / kTM, (a.E + kTE - 1) / kTE, a.splits);
  if (a.x_dtype == MOE_DTYPE_BF16)
    router_logits_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
  else
    router_logits_kernel<float><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_router_split(const RouterArgs& a, cudaStream_t s) {
  const dim3 grid((a.H + 31) / 32, (a.E + 31) / 32);
  router_split_kernel<<<grid, 256, 0, s>>>(a.Wg, a.H, a.E, a.wsplit);
  return cudaGetLastError();
}

cudaError_t launch_expert_choice(const ExpertChoiceArgs& a, cudaStream_t s) {
  const int E = a.r.E;
  cudaError_t e = E <= 32 ? launch_ec_scores<1>(a, s)
                  : E <= 64 ? launch_ec_scores<2>(a, s)
                  : E <= 128 ? launch_ec_scores<4>(a, s)
                  : E <= 256 ? launch_ec_scores<8>(a, s)
                             : launch_ec_scores<16>(a, s);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)a.r.T * 5 + 16;
  for (const void* fn : {reinterpret_cast<const void*>(ec_select_kernel),
                         reinterpret_cast<const void*>(ec_fix_kernel)}) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  ec_select_kernel<<<E, kEcThreads, smem, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the listed tokens are few; most of these CTAs find nothing to do
  const int sms = a.r.num_sms > 0 ? a.r.num_sms : 1;
  const int grid = a.r.T < 2 * sms ? a.r.T : 2 * sms;
  if (a.r.x_dtype == MOE_DTYPE_BF16)
    ec_exact_rows_kernel<__nv_bfloat16><<<grid, kRefineThreads, 0, s>>>(a);
  else
    ec_exact_rows_kernel<float><<<grid, kRefineThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ec_fix_kernel<<<E, kEcThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_router_reduce(RouterArgs& a, cudaStream_t s) {
  if (a.splits <= 1) return cudaSuccess;
  const size_t n = (size_t)a.T * a.E;
  const size_t want = (size_t)2 * 2048 * (a.num_sms > 0 ? a.num_sms : 1);
  int G = 1;
  while (G < 8 && G < a.splits && n * G < want) G <<= 1;
  const unsigned blocks = (unsigned)((n * G + 255) / 256);
  const bool f32 = a.logits_part != nullptr;
#define MOE_REDUCE(GG)                                                                      \
  (f32 ? router_reduce_kernel<true, GG><<<blocks, 256, 0, s>>>(a.logits, a.logits_part, n,   \
                                                                a.splits)                   \
       : router_reduce_kernel<false, GG><<<blocks, 256, 0, s>>>(a.logits, nullptr, n, a.splits))
  if (G == 1) MOE_REDUCE(1);
  else if (G == 2) MOE_REDUCE(2);
  else if (G == 4) MOE_REDUCE(4);
  else MOE_REDUCE(8);
#undef MOE_REDUCE
  a.splits = 1;
  return cudaGetLastError();
}

cudaError_t launch_router_select(const RouterArgs& a, cudaStream_t s) {
  RouterArgs b = a;
  if (a.splits > 1) {
    const size_t n = (size_t)a.T * a.E;
    // lanes per element: enough threads for ~2 waves of loads, at most 8, at most S
    const size_t want = (size_t)2 * 2048 * (a.num_sms > 0 ? a.num_sms : 1);
    int G = 1;
    while (G < 8 && G < a.splits && n * G < want) G <<= 1;
    const unsigned blocks = (unsigned)((n * G + 255) / 256);
    const bool f32 = a.logits_part != nullptr;
#define MOE_REDUCE(GG)                                                                      \
  (f32 ? router_reduce_kernel<true, GG><<<blocks, 256, 0, s>>>(a.logits, a.logits_part, n,   \
                                                                a.splits)                   \
       : router_reduce_kernel<false, GG><<<blocks, 256, 0, s>>>(a.logits, nullptr, n, a.splits))
    if (G == 1) MOE_REDUCE(1);
    else if (G == 2) MOE_REDUCE(2);
    else if (G == 4) MOE_REDUCE(4);
    else MOE_REDUCE(8);
#undef MOE_REDUCE
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    b.splits = 1;
  }
  return b.x_dtype == MOE_DTYPE_BF16 ? launch_select_t<__nv_bfloat16>(b, s)
                                     : launch_select_t<float>(b, s);
}

}  // namespace moe
