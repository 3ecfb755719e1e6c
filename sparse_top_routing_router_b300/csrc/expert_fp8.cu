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
// few): the step streams weights, and the arithmetic only has to keep pace with HBM.  Both
// GEMVs multiply 16 weight rows by up to 8 rows of the expert with m16n8k16 bf16 mma.sync
// (fp32 accumulation), decoding the codes exactly to bf16 in registers on the way; the
// channel's scale multiplies the finished sum.  (A tcgen05 tile would spend its 128-row
// operand on 8 live rows and would need the codes converted in shared memory first.)
// A work item is (expert, up to 8 of its rows, a block of output channels).  One CTA per
// SM: a producer warp streams the item's code rows (128-row TMA boxes) and input rows
// through a shared-memory ring (128-byte swizzle, 256 k per stage, 3 stages of about
// 68 KB), and 16 consumer warps run the mma on what lands:
//  gate/up  128 channels per item, gate and up rows; the warps form two k groups of eight,
//           each taking two of the four 64-wide k slices of every stage for 16 channels,
//           and the groups' partial sums are added in group order at the end of the item.
//  down     256 channels per item; every warp takes 16 channels over the whole k range,
//           so an item ends with no hand-over between warps.
#include <string.h>

#include <atomic>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

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

constexpr int kF8Chunk = 256;            // k per ring stage
constexpr int kF8Consumers = 16;         // consumer warps, 16 channels each
constexpr int kF8Threads = (kF8Consumers + 1) * 32;
constexpr int kXBox = kFp8Rows * 128;    // TMA box: 8 input rows x 64 bf16

// Shape of the ring kernel.  NMAT code matrices per item (2: gate and up; 1: W_down); KG
// k groups: the consumer warps split into KG groups of 16 / KG warps, group kg takes the
// 64-wide k slices kg, kg + KG, ... of every stage, and the groups' partial sums are added
// in group order at the end of an item.  An item covers 16 * 16 / KG channels; a stage
// holds, per matrix, the item's kCh code rows of k 0-127, then of k 128-255 (each loaded as
// TMA boxes of kBoxRows rows x 128 codes, 128 when the item has that many), then four
// input-row boxes (64 k each).
template <int NMAT, int KG>
struct F8Shape {
  static constexpr int kChanWarps = kF8Consumers / KG;
  static constexpr int kCh = 16 * kChanWarps;             // channels per item
  static constexpr int kBoxRows = kCh >= 128 ? 128 : 64;  // code rows per TMA box
  static constexpr int kHalfBytes = kCh * 128;            // one matrix, one 128-code k half
  static constexpr int kStageBytes = NMAT * 2 * kHalfBytes + 4 * kXBox;
  static constexpr int kStages = 210 * 1024 / kStageBytes < 5 ? 210 * 1024 / kStageBytes : 5;
};

template <int NMAT, int KG>
struct F8Smem {
  using Sh = F8Shape<NMAT, KG>;
  uint8_t ring[Sh::kStages][Sh::kStageBytes];
  uint64_t full[Sh::kStages];
  uint64_t empty[Sh::kStages];
  // KG > 1: the partial sums of k groups 1.. of the item that ended last; written by those
  // groups, read by group 0
  uint64_t part_written, part_read;
  int abort_flag;
  float part[KG > 1 ? KG - 1 : 1][KG > 1 ? Sh::kChanWarps : 1][NMAT * 4][32];
  Fp8Table T;
};

// 16 bytes at logical 16-byte chunk `c` of row `r` of a box written by TMA with the
// 128-byte swizzle (rows of 128 B; the chunk index is XORed with the row index mod 8).
__device__ __forceinline__ uint4 ld_sw128(const uint8_t* box, int r, int c) {
  return *reinterpret_cast<const uint4*>(box + r * 128 + ((c ^ (r & 7)) << 4));
}

// One 64-wide k slice of a stage.  Consumer warp w of a group holds rows w*16 + g and
// w*16 + g + 8 of each code box (g = lane / 4) and input row g; inside each 64-wide k slice
// lane t = lane % 4 supplies k = 16 t + 4 s + 0..3 at mma step s to both operands (a dot
// product does not depend on the order of its terms), i.e. 16 contiguous codes of each of
// its code rows and 16 contiguous bf16 of its input row.  acc[m] is the mma's D fragment
// for matrix m: (channel g, rows 2t, 2t+1), (channel g + 8, rows 2t, 2t+1).
template <int NMAT, int HALF>
__device__ __forceinline__ void f8_slice_mma(const uint8_t* st, int j, int w, int lane,
                                             float (&acc)[NMAT][4]) {
  const int g = lane >> 2, t = lane & 3;
  const int r_lo = w * 16 + g, r_hi = r_lo + 8;
  {                                         // 64-wide k slice j of the stage
    const uint8_t* xb = st + NMAT * 2 * HALF + j * kXBox;
    const uint4 x0 = ld_sw128(xb, g, 2 * t), x1 = ld_sw128(xb, g, 2 * t + 1);
    const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const int cb = (j & 1) * 4 + t;         // 16-byte chunk of the 128-code box row
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      const uint8_t* box = st + (m * 2 + (j >> 1)) * HALF;
      const uint4 c0 = ld_sw128(box, r_lo, cb), c8 = ld_sw128(box, r_hi, cb);
      const uint32_t a0w[4] = {c0.x, c0.y, c0.z, c0.w};
      const uint32_t a8w[4] = {c8.x, c8.y, c8.z, c8.w};
#pragma unroll
      for (int sstep = 0; sstep < 4; ++sstep) {
        uint32_t l0, h0, l8, h8;
        e4m3x4_to_bf16(a0w[sstep], l0, h0);
        e4m3x4_to_bf16(a8w[sstep], l8, h8);
        mma_16816(acc[m], l0, l8, h0, h8, xw[2 * sstep], xw[2 * sstep + 1]);
      }
    }
  }
}

struct F8Maps {
  CUtensorMap q0, q1, q0s, q1s;   // codes as [rows, K] uint8 (routed: E * N rows; shared: N)
  CUtensorMap x, xs;              // input rows [rows, K] bf16 (routed, shared expert)
};

// NMAT = 2: gate/up, h = SiLU(s_g a) * (s_u u) rounded to bf16 as in the tensor-core path.
// NMAT = 1: down, O = s_d * (h . code).
template <int NMAT, int KG>
__global__ void __launch_bounds__(kF8Threads, 1)
    fp8_gemv_kernel(const __grid_constant__ F8Maps mp, const Fp8Args a,
                    unsigned long long lim) {
  using Sh = F8Shape<NMAT, KG>;
  constexpr int kF8Stages = Sh::kStages, kF8Ch = Sh::kCh, kHalf = Sh::kHalfBytes;
  constexpr int kBoxR = Sh::kBoxRows;
  extern __shared__ uint8_t f8_raw[];
  F8Smem<NMAT, KG>& S = *reinterpret_cast<F8Smem<NMAT, KG>*>(
      (reinterpret_cast<uintptr_t>(f8_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kMode = NMAT == 2 ? 0 : 1;
  constexpr uint32_t kTx = (uint32_t)Sh::kStageBytes;
  const int N = NMAT == 2 ? a.I : a.H;      // output channels of one expert
  const int K = NMAT == 2 ? a.H : a.I;      // reduction length
  const int n_blk = (N + kF8Ch - 1) / kF8Ch;
  const int nchunks = (K + kF8Chunk - 1) / kF8Chunk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    S.abort_flag = 0;
    for (int q = 0; q < kF8Stages; ++q) {
      mbar_init(&S.full[q], 1);
      mbar_init(&S.empty[q], kF8Consumers);   // every consumer warp releases each stage
    }
    mbar_init(&S.part_written, (KG - 1) * Sh::kChanWarps);   // the warps of groups 1..
    mbar_init(&S.part_read, Sh::kChanWarps);                 // the warps of group 0
    fence_mbar_init();
  }
  build_fp8_table(S.T, a, kMode, n_blk);   // ends with __syncthreads
  const volatile int* abort_flag = &S.abort_flag;

  if (warp == kF8Consumers) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < S.T.total && ok; item += gridDim.x) {
        const int grp = find_group8(S.T, item);
        const int local = item - S.T.start[grp];
        const int r0 = (local / n_blk) * kFp8Rows, ch0 = (local % n_blk) * kF8Ch;
        const bool sh = grp >= a.E;
        const int qrow = sh ? ch0 : grp * N + ch0;
        const int xrow = S.T.row0[grp] + r0;
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait(&S.empty[stage], phase ^ 1u, abort_flag, lim)) {
            ok = false;
            break;
          }
          uint8_t* st = S.ring[stage];
          const int k0 = c * kF8Chunk;
          mbar_arrive_expect_tx(&S.full[stage], kTx);
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            const CUtensorMap* q = m == 0 ? (sh ? &mp.q0s : &mp.q0) : (sh ? &mp.q1s : &mp.q1);
#pragma unroll
            for (int b = 0; b < kF8Ch / kBoxR; ++b) {
              uint8_t* box = st + m * 2 * kHalf + b * kBoxR * 128;
              tma_load_2d(box, q, &S.full[stage], k0, qrow + kBoxR * b);
              tma_load_2d(box + kHalf, q, &S.full[stage], k0 + 128, qrow + kBoxR * b);
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tma_load_2d(st + NMAT * 2 * kHalf + j * kXBox, sh ? &mp.xs : &mp.x,
                        &S.full[stage], k0 + 64 * j, xrow);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kF8Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        S.abort_flag = 1;
        set_status(a.status, MOE_ERR_TIMEOUT);
        const int zero = 0;   // let every copy already issued land before leaving
        for (int q = 0; q < kF8Stages; ++q)
          if (issued_mask >> q & 1u) mbar_wait(&S.full[q], issued_parity >> q & 1u, &zero, lim);
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    // warp = kg * (16 / KG) + w: k group kg takes slices kg, kg + KG, ... of every stage,
    // w its 16 channels
    const int kg = warp / Sh::kChanWarps, w = warp % Sh::kChanWarps;
    const int g = lane >> 2, t = lane & 3;
    int stage = 0, n_items = 0;
    uint32_t phase = 0;
    bool ok = true;
    // a bounded wait of the whole warp; false (with the abort flag raised) if it gave up
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const bool got = mbar_wait(bar, parity, abort_flag, lim);
      if (__all_sync(0xffffffffu, got)) return true;
      S.abort_flag = 1;
      set_status(a.status, MOE_ERR_TIMEOUT);
      return false;
    };
    for (int item = blockIdx.x; item < S.T.total && ok; item += gridDim.x) {
      const int grp = find_group8(S.T, item);
      const int local = item - S.T.start[grp];
      const int r0 = (local / n_blk) * kFp8Rows, ch0 = (local % n_blk) * kF8Ch + w * 16;
      // N % 64 == 0, so a warp's 16 channels are all in range or all past the end (never
      // past it for 64-channel items); a warp past the end still takes part in every
      // stage's hand-over
      const bool live = kF8Ch == 64 || ch0 < N;
      const int mr = min(kFp8Rows, S.T.rows[grp] - r0);
      const bool sh = grp >= a.E;
      float acc[NMAT][4];
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;
      for (int c = 0; c < nchunks; ++c) {
        if (!warp_wait(&S.full[stage], phase)) {
          ok = false;
          break;
        }
        if (live) {
#pragma unroll
          for (int jj = 0; jj < 4 / KG; ++jj)
            f8_slice_mma<NMAT, kHalf>(S.ring[stage], kg + jj * KG, w, lane, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[stage]);
        if (++stage == kF8Stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      // The k groups' partial sums, added in group order by group 0.  Groups 1.. store
      // theirs and go on to the next item at once; before storing the next item's they wait
      // until group 0 has read these (it does so as soon as this item ends, so that wait is
      // normally over before it starts).
      if (KG > 1) {
        const uint32_t use = (uint32_t)n_items++;   // items this CTA finished before this one
        if (kg > 0) {
          if (use > 0 && !warp_wait(&S.part_read, (use - 1) & 1u)) break;
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) S.part[kg - 1][w][m * 4 + i][lane] = acc[m][i];
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.part_written);
          continue;
        }
        if (!warp_wait(&S.part_written, use & 1u)) break;
#pragma unroll
        for (int q = 0; q < KG - 1; ++q)
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[m][i] += S.part[q][w][m * 4 + i][lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.part_read);
      }
      if (!live) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ch = g + (i >= 2 ? 8 : 0);
        const int n = 2 * t + (i & 1);
        if (n >= mr) continue;
        const size_t orow = (size_t)(S.T.out0[grp] + r0 + n);
        if (NMAT == 2) {
          const float* sg = (sh ? a.Ss_gate : a.S_gate + (size_t)grp * a.I) + ch0;
          const float* su = (sh ? a.Ss_up : a.S_up + (size_t)grp * a.I) + ch0;
          const float gv = sg[ch] * acc[0][i], uv = su[ch] * acc[NMAT - 1][i];
          static_cast<__nv_bfloat16*>(a.h)[orow * a.I + ch0 + ch] =
              __float2bfloat16_rn(gv / (1.f + __expf(-gv)) * uv);
        } else {
          const float* sd = (sh ? a.Ss_down : a.S_down + (size_t)grp * a.H) + ch0;
          (sh ? a.O_shared : a.O)[orow * a.H + ch0 + ch] = sd[ch] * acc[0][i];
        }
      }
    }
  }
}

bool encode_f8(EncodeTiledFn enc, CUtensorMap* m, bool codes, const void* base, uint64_t K,
               uint64_t rows, uint32_t code_box_rows = 64) {
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * (codes ? 1 : 2)};
  const cuuint32_t box[2] = {codes ? 128u : 64u, codes ? code_box_rows : (cuuint32_t)kFp8Rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, codes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMAT, int KG>
cudaError_t launch_f8(const Fp8Args& a, EncodeTiledFn enc, bool* encode_failed,
                      unsigned long long lim, cudaStream_t s) {
  *encode_failed = false;
  const int Tk = a.T * a.k;
  F8Maps mp;
  memset(&mp, 0, sizeof(mp));
  bool ok = true;
  constexpr uint32_t br = F8Shape<NMAT, KG>::kBoxRows;
  if (NMAT == 2) {
    ok &= encode_f8(enc, &mp.q0, true, a.Q_gate, a.H, (uint64_t)a.E * a.I, br);
    ok &= encode_f8(enc, &mp.q1, true, a.Q_up, a.H, (uint64_t)a.E * a.I, br);
    ok &= encode_f8(enc, &mp.q0s, true, a.has_shared ? a.Qs_gate : a.Q_gate, a.H, a.I, br);
    ok &= encode_f8(enc, &mp.q1s, true, a.has_shared ? a.Qs_up : a.Q_up, a.H, a.I, br);
    ok &= encode_f8(enc, &mp.x, false, a.Xperm, a.H, Tk);
    ok &= encode_f8(enc, &mp.xs, false, a.has_shared ? a.X : a.Xperm, a.H,
                    a.has_shared ? a.T : Tk);
  } else {
    ok &= encode_f8(enc, &mp.q0, true, a.Q_down, a.I, (uint64_t)a.E * a.H, br);
    ok &= encode_f8(enc, &mp.q0s, true, a.has_shared ? a.Qs_down : a.Q_down, a.I, a.H, br);
    mp.q1 = mp.q0;
    mp.q1s = mp.q0s;
    ok &= encode_f8(enc, &mp.x, false, a.h, a.I, (uint64_t)Tk + (a.has_shared ? a.T : 0));
    mp.xs = mp.x;
  }
  if (!ok) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  const size_t smem = sizeof(F8Smem<NMAT, KG>) + 1024;
  auto* fn = fp8_gemv_kernel<NMAT, KG>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one resident wave of CTAs, computed once per device (the ordinals past the table are
  // queried every time)
  static std::atomic<int> grids[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  int grid = (dev >= 0 && dev < 64) ? grids[dev].load(std::memory_order_relaxed) : 0;
  if (!grid) {
    int per_sm = 0, sms = kGridSms;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kF8Threads, smem) !=
            cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    if (dev >= 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                        cudaSuccess) {
      cudaGetLastError();
      sms = kGridSms;
    }
    grid = per_sm * (sms > 0 ? sms : kGridSms);
    if (dev >= 0 && dev < 64) grids[dev].store(grid, std::memory_order_relaxed);
  }
  fn<<<grid, kF8Threads, smem, s>>>(mp, a, lim);
  return cudaGetLastError();
}

static_assert(sizeof(F8Smem<2, 2>) + 1024 <= 227 * 1024, "FP8 gate/up shared memory");
static_assert(sizeof(F8Smem<1, 1>) + 1024 <= 227 * 1024, "FP8 down shared memory");

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

cudaError_t launch_expert_gate_up_fp8(const Fp8Args& a, EncodeTiledFn enc,
                                      bool* encode_failed, unsigned long long wait_limit_ns,
                                      cudaStream_t s) {
  return launch_f8<2, 2>(a, enc, encode_failed, wait_limit_ns, s);
}

cudaError_t launch_expert_down_fp8(const Fp8Args& a, EncodeTiledFn enc, bool* encode_failed,
                                   unsigned long long wait_limit_ns, cudaStream_t s) {
  return launch_f8<1, 1>(a, enc, encode_failed, wait_limit_ns, s);
}

}  // namespace moe
