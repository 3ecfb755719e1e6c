// FP8 expert weights for decode-sized batches ("LLM Internals §14.2.5": one expert is
// 44 MB in FP8, and a decode step reads each touched expert's weights for a handful of
// rows, so the step is bound by the bytes of weights it streams).
//
// Format: E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest
// finite value 448) with one fp32 scale per output channel, scale = amax / 448 over the
// channel's row (1 for an all-zero row), code = E4M3(w / scale) rounded to nearest even
// with saturation; both divisions are correctly rounded fp32.
//
// The expert GEMMs of a decode step do 2 b FLOP per weight byte for b rows per expert (a
// few): the step streams weights, and the arithmetic only has to keep pace with HBM.
// Each warp takes 16 weight rows against 8 rows of the expert (m16n8k16 bf16 mma.sync,
// fp32 accumulation), decoding the codes exactly to bf16 in registers on the way; a
// tcgen05 tile would spend its 128-row operand on 8 live rows and would need the codes
// converted in shared memory first.  The channel's scale multiplies the finished sum.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kFp8Threads = 256;      // 8 warps
constexpr int kFp8Rows = 8;           // expert rows per pass: the mma's N
constexpr int kMaxGroups8 = kMaxE + 1;

// ------------------------------------------------------------------ quantization

template <typename TW>
__device__ __forceinline__ float load_w(const TW* p);
template <>
__device__ __forceinline__ float load_w<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float load_w<float>(const float* p) {
  return *p;
}

// One CTA per row: amax, the scale, then the codes two at a time.
template <typename TW>
__global__ void __launch_bounds__(256) quantize_fp8_rows_kernel(int cols, const TW* W,
                                                                uint8_t* q, float* scale) {
  __shared__ float s_max[8];
  const size_t row = blockIdx.x;
  const TW* w = W + row * cols;
  float amax = 0.f;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(load_w<TW>(w + c)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, s_max[i]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (threadIdx.x == 0) scale[row] = s;
  uint16_t* q2 = reinterpret_cast<uint16_t*>(q + row * cols);
  for (int c = 2 * threadIdx.x; c < cols; c += 2 * blockDim.x) {
    const float2 v = make_float2(__fdiv_rn(load_w<TW>(w + c), s),
                                 __fdiv_rn(load_w<TW>(w + c + 1), s));
    q2[c >> 1] = (uint16_t)__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
  }
}

// ------------------------------------------------------------------ decode GEMVs

// Four E4M3 codes (one word, lowest byte first) -> two bf16x2 words, exactly: E4M3 ->
// fp16 and fp16 -> fp32 are exact, and a 4-bit significand fits bf16.
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2_raw a = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  const __half2_raw b = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&a));
  const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&b));
  const __nv_bfloat162 ba = __floats2bfloat162_rn(fa.x, fa.y);
  const __nv_bfloat162 bb = __floats2bfloat162_rn(fb.x, fb.y);
  lo = *reinterpret_cast<const uint32_t*>(&ba);
  hi = *reinterpret_cast<const uint32_t*>(&bb);
}

// D (16 x 8, fp32) += A (16 x 16, bf16, row) * B (16 x 8, bf16, col).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One warp: NT tiles of 16 weight rows (rows[q] + g and + 8 for lane g = lane / 4) times
// the 8 input rows xr + n * ldx (n < mr; zeros beyond), over K in 64-wide chunks.  The
// mma's k order inside a chunk is permuted - lane t = lane % 4 supplies k = 16 t + 4 s
// + 0..3 at step s for both operands - so each lane reads 16 contiguous codes of its two
// weight rows and 16 contiguous bf16 of its input row; a dot product does not depend on
// the order of its terms.  The next chunk's loads are issued before the current chunk's
// conversions and MMAs.  acc[q] is the mma's D fragment: (row g, cols 2t, 2t+1), (row g+8,
// cols 2t, 2t+1).
template <int NT>
__device__ __forceinline__ void gemv_mma(const uint8_t* const (&rows)[NT], size_t ldw,
                                         const __nv_bfloat16* xr, size_t ldx, int mr, int K,
                                         int lane, float (&acc)[NT][4]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int q = 0; q < NT; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[q][i] = 0.f;
  const uint8_t* w0[NT];
  const uint8_t* w8[NT];
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    w0[q] = rows[q] + (size_t)g * ldw + 16 * t;
    w8[q] = rows[q] + (size_t)(g + 8) * ldw + 16 * t;
  }
  const bool xin = g < mr;
  const __nv_bfloat16* xp = xr + (size_t)(xin ? g : 0) * ldx + 16 * t;
  uint4 c0[NT], c8[NT], cx0, cx1;
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    c0[q] = *reinterpret_cast<const uint4*>(w0[q]);
    c8[q] = *reinterpret_cast<const uint4*>(w8[q]);
  }
  cx0 = xin ? reinterpret_cast<const uint4*>(xp)[0] : make_uint4(0, 0, 0, 0);
  cx1 = xin ? reinterpret_cast<const uint4*>(xp)[1] : make_uint4(0, 0, 0, 0);
  for (int kb = 0; kb < K; kb += 64) {
    const int kn = kb + 64;
    uint4 n0[NT], n8[NT], nx0 = make_uint4(0, 0, 0, 0), nx1 = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      n0[q] = kn < K ? *reinterpret_cast<const uint4*>(w0[q] + kn) : make_uint4(0, 0, 0, 0);
      n8[q] = kn < K ? *reinterpret_cast<const uint4*>(w8[q] + kn) : make_uint4(0, 0, 0, 0);
    }
    if (xin && kn < K) {
      nx0 = reinterpret_cast<const uint4*>(xp + kn)[0];
      nx1 = reinterpret_cast<const uint4*>(xp + kn)[1];
    }
    const uint32_t xw[8] = {cx0.x, cx0.y, cx0.z, cx0.w, cx1.x, cx1.y, cx1.z, cx1.w};
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const uint32_t a0w[4] = {c0[q].x, c0[q].y, c0[q].z, c0[q].w};
      const uint32_t a8w[4] = {c8[q].x, c8[q].y, c8[q].z, c8[q].w};
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        uint32_t l0, h0, l8, h8;
        e4m3x4_to_bf16(a0w[st], l0, h0);
        e4m3x4_to_bf16(a8w[st], l8, h8);
        mma_16816(acc[q], l0, l8, h0, h8, xw[2 * st], xw[2 * st + 1]);
      }
    }
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      c0[q] = n0[q];
      c8[q] = n8[q];
    }
    cx0 = nx0;
    cx1 = nx1;
  }
}

struct Fp8Table {
  int ngroups, total;
  int start[kMaxGroups8 + 1];   // first work item of each group
  int rows[kMaxGroups8];
  int row0[kMaxGroups8];        // first input row (Xperm / X, or h)
  int out0[kMaxGroups8];        // first output row (h, or O / O_shared)
};

// Work items of one launch: per group, ceil(rows / kFp8Rows) row passes times n_blk
// channel blocks.  GATE_UP (mode 0): input rows Xperm (routed) or X (shared), output h
// rows offsets[e] / Tk + t.  DOWN (mode 1): input h rows, output O / O_shared rows.
__device__ void build_fp8_table(Fp8Table& S, const Fp8Args& a, int mode, int n_blk) {
  const int ngroups = a.E + (a.has_shared ? 1 : 0);
  const int Tk = a.T * a.k;
  for (int g = threadIdx.x; g < ngroups; g += blockDim.x) {
    int rows, row0, out0;
    if (g < a.E) {
      const int lo = a.offsets[g], hi = a.offsets[g + 1];
      if (lo < 0 || hi < lo || hi > Tk) {
        set_status(a.status, MOE_ERR_DEVICE_INDEX);
        rows = row0 = out0 = 0;
      } else {
        rows = hi - lo;
        row0 = lo;
        out0 = lo;
      }
    } else {
      rows = a.T;
      row0 = mode == 0 ? 0 : Tk;
      out0 = mode == 0 ? Tk : 0;
    }
    S.rows[g] = rows;
    S.row0[g] = row0;
    S.out0[g] = out0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int g = 0; g < ngroups; ++g) {
      S.start[g] = acc;
      acc += ((S.rows[g] + kFp8Rows - 1) / kFp8Rows) * n_blk;
    }
    S.start[ngroups] = acc;
    S.total = acc;
    S.ngroups = ngroups;
  }
  __syncthreads();
}

__device__ __forceinline__ int find_group8(const Fp8Table& S, int item) {
  int lo = 0, hi = S.ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.start[mid] <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

constexpr int kChanPerWarp = 16;
constexpr int kChanPerCta = kChanPerWarp * (kFp8Threads / 32);   // 128

// Gate/up: a warp takes 16 channels, their gate and up rows; h = SiLU(s_g a) * (s_u u),
// rounded to bf16 as in the tensor-core path.
__global__ void __launch_bounds__(kFp8Threads) fp8_gate_up_kernel(Fp8Args a) {
  __shared__ Fp8Table S;
  const int n_blk = (a.I + kChanPerCta - 1) / kChanPerCta;
  build_fp8_table(S, a, 0, n_blk);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const __nv_bfloat16* Xp = static_cast<const __nv_bfloat16*>(a.Xperm);
  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.X);
  __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.h);
  for (int item = blockIdx.x; item < S.total; item += gridDim.x) {
    const int grp = find_group8(S, item);
    const int local = item - S.start[grp];
    const int pass = local / n_blk, blk = local % n_blk;
    const int r0 = pass * kFp8Rows;
    const int mr = min(kFp8Rows, S.rows[grp] - r0);
    const int i0 = blk * kChanPerCta + w * kChanPerWarp;
    if (i0 >= a.I) continue;   // I % 64 == 0, so a started warp has all 16 channels
    const bool sh = grp >= a.E;
    const uint8_t* Wg = (sh ? a.Qs_gate : a.Q_gate + (size_t)grp * a.I * a.H) + (size_t)i0 * a.H;
    const uint8_t* Wu = (sh ? a.Qs_up : a.Q_up + (size_t)grp * a.I * a.H) + (size_t)i0 * a.H;
    const float* sg = (sh ? a.Ss_gate : a.S_gate + (size_t)grp * a.I) + i0;
    const float* su = (sh ? a.Ss_up : a.S_up + (size_t)grp * a.I) + i0;
    const uint8_t* const rows[2] = {Wg, Wu};
    const __nv_bfloat16* xr = (sh ? X : Xp) + (size_t)(S.row0[grp] + r0) * a.H;
    float acc[2][4];
    gemv_mma<2>(rows, a.H, xr, a.H, mr, a.H, lane, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = g + (i >= 2 ? 8 : 0);
      const int n = 2 * t + (i & 1);
      if (n < mr) {
        const float gv = sg[ch] * acc[0][i], uv = su[ch] * acc[1][i];
        h[(size_t)(S.out0[grp] + r0 + n) * a.I + i0 + ch] =
            __float2bfloat16_rn(gv / (1.f + __expf(-gv)) * uv);
      }
    }
  }
}

// Down: a warp takes 16 output channels of W_down; O = s_d * (h . code).
__global__ void __launch_bounds__(kFp8Threads) fp8_down_kernel(Fp8Args a) {
  __shared__ Fp8Table S;
  const int n_blk = (a.H + kChanPerCta - 1) / kChanPerCta;
  build_fp8_table(S, a, 1, n_blk);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(a.h);
  for (int item = blockIdx.x; item < S.total; item += gridDim.x) {
    const int grp = find_group8(S, item);
    const int local = item - S.start[grp];
    const int pass = local / n_blk, blk = local % n_blk;
    const int r0 = pass * kFp8Rows;
    const int mr = min(kFp8Rows, S.rows[grp] - r0);
    const int j0 = blk * kChanPerCta + w * kChanPerWarp;
    if (j0 >= a.H) continue;   // H % 64 == 0
    const bool sh = grp >= a.E;
    const uint8_t* Wd = (sh ? a.Qs_down : a.Q_down + (size_t)grp * a.H * a.I) + (size_t)j0 * a.I;
    const float* sd = (sh ? a.Ss_down : a.S_down + (size_t)grp * a.H) + j0;
    const uint8_t* const rows[1] = {Wd};
    const __nv_bfloat16* xr = h + (size_t)(S.row0[grp] + r0) * a.I;
    float acc[1][4];
    gemv_mma<1>(rows, a.I, xr, a.I, mr, a.I, lane, acc);
    float* out = sh ? a.O_shared : a.O;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = g + (i >= 2 ? 8 : 0);
      const int n = 2 * t + (i & 1);
      if (n < mr) out[(size_t)(S.out0[grp] + r0 + n) * a.H + j0 + ch] = sd[ch] * acc[0][i];
    }
  }
}

}  // namespace

cudaError_t launch_quantize_fp8_rows(int rows, int cols, int w_dtype, const void* W,
                                     uint8_t* q, float* scale, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (w_dtype == MOE_DTYPE_BF16)
    quantize_fp8_rows_kernel<__nv_bfloat16>
        <<<rows, 256, 0, s>>>(cols, static_cast<const __nv_bfloat16*>(W), q, scale);
  else
    quantize_fp8_rows_kernel<float><<<rows, 256, 0, s>>>(cols, static_cast<const float*>(W), q,
                                                         scale);
  return cudaGetLastError();
}

// A persistent grid: as many CTAs as fit on the GPU at once.
static int resident_grid(const void* fn) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kFp8Threads, 0) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  int dev = 0, sms = kGridSms;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return per_sm * (sms > 0 ? sms : kGridSms);
}

cudaError_t launch_expert_gate_up_fp8(const Fp8Args& a, cudaStream_t s) {
  static const int grid = resident_grid(reinterpret_cast<const void*>(fp8_gate_up_kernel));
  fp8_gate_up_kernel<<<grid, kFp8Threads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_expert_down_fp8(const Fp8Args& a, cudaStream_t s) {
  static const int grid = resident_grid(reinterpret_cast<const void*>(fp8_down_kernel));
  fp8_down_kernel<<<grid, kFp8Threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
