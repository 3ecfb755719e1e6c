// Step 5 of the MoE forward for fp32 hidden states and weights ("LLM Internals §14.2.1
// step 5"; §14.2.2 SwiGLU expert).  The tensor cores have no fp32 input kind, and a
// TF32 product would lose the 1e-4 relative accuracy asked of fp32 layers, so this path
// uses CUDA-core fp32 FMA: 32-row x 64-column tiles per CTA, the (group, n, m) work
// list enumerated on the device from the dispatch offsets as in the bf16 kernel.
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int FM = 32, FN = 64, FK = 32;
constexpr int kMaxGroups = kMaxE + 1;

struct F32Table {
  int ngroups, total;
  int tile_start[kMaxGroups + 1];
  int rows[kMaxGroups];
  int row0[kMaxGroups];
};

__device__ void build_table(F32Table& S, const int32_t* offsets, int E, int has_shared, int T,
                            int Tk, int shared_row0, int n_tiles_n, int* status) {
  const int ngroups = E + (has_shared ? 1 : 0);
  for (int g = threadIdx.x; g < ngroups; g += blockDim.x) {
    int rows, row0;
    if (g < E) {
      const int a = offsets[g], b = offsets[g + 1];
      if (a < 0 || b < a || b > Tk) {
        set_status(status, MOE_ERR_DEVICE_INDEX);
        rows = 0;
        row0 = 0;
      } else {
        rows = b - a;
        row0 = a;
      }
    } else {
      rows = T;
      row0 = shared_row0;
    }
    S.rows[g] = rows;
    S.row0[g] = row0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int g = 0; g < ngroups; ++g) {
      S.tile_start[g] = acc;
      acc += ((S.rows[g] + FM - 1) / FM) * n_tiles_n;
    }
    S.tile_start[ngroups] = acc;
    S.total = acc;
    S.ngroups = ngroups;
  }
  __syncthreads();
}

__device__ __forceinline__ int find_group(const F32Table& S, int tile) {
  int lo = 0, hi = S.ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// MODE 0: h = SiLU(A Wg^T) * (A Wu^T);  MODE 1: O = A Wd^T.
template <int MODE>
__global__ void __launch_bounds__(256) expert_f32_kernel(ExpertArgs a) {
  __shared__ F32Table S;
  __shared__ float sA[FK][FM + 1];
  __shared__ float sB0[FK][FN + 1];
  __shared__ float sB1[FK][FN + 1];
  const int Tk = a.T * a.k;
  const int K = MODE == 0 ? a.H : a.I;
  const int N = MODE == 0 ? a.I : a.H;
  const int n_tiles_n = (N + FN - 1) / FN;
  build_table(S, a.offsets, a.E, a.has_shared, a.T, Tk, MODE == 0 ? 0 : Tk, n_tiles_n,
              a.status);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  for (int tile = blockIdx.x; tile < S.total; tile += gridDim.x) {
    const int g = find_group(S, tile);
    const int rows = S.rows[g], row0 = S.row0[g];
    const int mt = (rows + FM - 1) / FM;
    const int local = tile - S.tile_start[g];
    const int m0 = (local % mt) * FM, n0 = (local / mt) * FN;
    const bool sh = g >= a.E;
    const float* A;
    if (MODE == 0) A = sh ? static_cast<const float*>(a.X) : static_cast<const float*>(a.Xperm);
    else A = static_cast<const float*>(a.h);
    const float *B0, *B1 = nullptr;
    if (MODE == 0) {
      B0 = sh ? static_cast<const float*>(a.Ws_gate)
              : static_cast<const float*>(a.W_gate) + (size_t)g * N * K;
      B1 = sh ? static_cast<const float*>(a.Ws_up)
              : static_cast<const float*>(a.W_up) + (size_t)g * N * K;
    } else {
      B0 = sh ? static_cast<const float*>(a.Ws_down)
              : static_cast<const float*>(a.W_down) + (size_t)g * N * K;
    }
    float c0[2][4] = {}, c1[2][4] = {};
    for (int kb = 0; kb < K; kb += FK) {
      for (int i = tid; i < FM * FK; i += 256) {
        const int r = i / FK, c = i % FK;
        const int m = m0 + r, kk = kb + c;
        sA[c][r] = (m < rows && kk < K) ? A[(size_t)(row0 + m) * K + kk] : 0.f;
      }
      for (int i = tid; i < FN * FK; i += 256) {
        const int r = i / FK, c = i % FK;   // r: output column, c: reduction index
        const int n = n0 + r, kk = kb + c;
        const bool in = n < N && kk < K;
        sB0[c][r] = in ? B0[(size_t)n * K + kk] : 0.f;
        if (MODE == 0) sB1[c][r] = in ? B1[(size_t)n * K + kk] : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < FK; ++kk) {
        const float x0 = sA[kk][ty * 2], x1 = sA[kk][ty * 2 + 1];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float w0 = sB0[kk][tx * 4 + j];
          c0[0][j] = fmaf(x0, w0, c0[0][j]);
          c0[1][j] = fmaf(x1, w0, c0[1][j]);
          if (MODE == 0) {
            const float w1 = sB1[kk][tx * 4 + j];
            c1[0][j] = fmaf(x0, w1, c1[0][j]);
            c1[1][j] = fmaf(x1, w1, c1[1][j]);
          }
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int m = m0 + ty * 2 + i;
      if (m >= rows) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tx * 4 + j;
        if (n >= N) continue;
        if (MODE == 0) {
          const float gv = c0[i][j], uv = c1[i][j];
          const size_t out_row = sh ? (size_t)Tk + m : (size_t)row0 + m;
          static_cast<float*>(a.h)[out_row * N + n] = gv / (1.f + expf(-gv)) * uv;
        } else {
          float* O = sh ? a.O_shared + (size_t)m * N : a.O + (size_t)(row0 + m) * N;
          O[n] = c0[i][j];
        }
      }
    }
  }
}

cudaError_t launch_f32(const ExpertArgs& a, int mode, cudaStream_t s) {
  const int Tk = a.T * a.k;
  const int N = mode == 0 ? a.I : a.H;
  const long long mt = (Tk + FM - 1) / FM + a.E + (a.has_shared ? (a.T + FM - 1) / FM : 0);
  const long long tiles = mt * ((N + FN - 1) / FN);
  const long long cap = 8LL * a.num_sms;
  const int grid = (int)(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
  if (mode == 0) expert_f32_kernel<0><<<grid, 256, 0, s>>>(a);
  else expert_f32_kernel<1><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_gate_up_f32(const ExpertArgs& a, cudaStream_t s) {
  return launch_f32(a, 0, s);
}
cudaError_t launch_expert_down_f32(const ExpertArgs& a, cudaStream_t s) {
  return launch_f32(a, 1, s);
}

}  // namespace moe
