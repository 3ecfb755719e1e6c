// Step 5 of the MoE forward on the 5th-generation tensor cores ("LLM Internals §14.2.1
// step 5": one GEMM per expert over its m_i rows, [m_i, H] x W_i[H, I] -> [m_i, I],
// then back to H; §14.2.2: the expert is a three-matrix SwiGLU).
//
// One persistent, warp-specialised kernel template serves both GEMMs of the expert:
//   GATE_UP: h = SiLU(x W_gate^T) * (x W_up^T), bf16 out.  One 128x256 accumulator holds
//            the gate tile (columns 0-127) and the up tile (128-255) of the same 128
//            rows, so the SwiGLU is applied in the epilogue straight from TMEM.
//   DOWN:    o = h W_down^T, fp32 out, 128x256 tiles.
// Work items are (group, n-tile, m-tile) with the m-tile fastest, enumerated on the
// device from the dispatch offsets (the host never learns m_i), assigned round-robin
// to one CTA per SM.  Neighbouring CTAs thus share the weight tile of an expert through
// L2.  The shared expert is one more group whose rows are all T tokens.
//
// Roles (192 threads):
//   warp 0      TMA producer: A rows [128 x 64] and two weight boxes [128 x 64] per
//               stage, 128-byte swizzle, 4-stage ring guarded by full/empty mbarriers
//   warp 1      TMEM allocation (512 columns = two 256-column accumulators) and, on one
//               lane, the tcgen05.mma issue loop (M=128, N=256, K=16 per instruction)
//   warps 2-5   epilogue: tcgen05.ld 32 columns at a time, SwiGLU or fp32 store
// Every mbarrier wait is bounded (see ptx.cuh); a timeout sets the status word and the
// CTA drains its in-flight copies and MMAs, frees TMEM and returns.
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;
constexpr int kBBoxBytes = 128 * BK * 2;
constexpr int kStageBytes = kABytes + 2 * kBBoxBytes;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kMaxGroups = kMaxE + 1;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, 256);

enum Mode { GATE_UP = 0, DOWN = 1 };

struct TcParams {
  const int32_t* offsets;
  int E, has_shared, T, Tk;
  int K;        // reduction length
  int N;        // output width
  int n_tile;   // output columns per tile: 128 (GATE_UP) or 256 (DOWN)
  __nv_bfloat16* h;
  float* O;
  float* O_shared;
  int* status;
  int test_hook;
  unsigned long long wait_limit_ns;
};

struct __align__(1024) Smem {
  uint8_t tiles[kStages][kStageBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ngroups;
  int total_tiles;
  int tile_start[kMaxGroups + 1];
  int grp_rows[kMaxGroups];
  int grp_row0[kMaxGroups];
};

struct TileInfo {
  int g, m0, n0, rows, row0;
};

__device__ __forceinline__ TileInfo decode_tile(const Smem& S, int tile, int n_tile) {
  int lo = 0, hi = S.ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  ti.g = lo;
  ti.rows = S.grp_rows[lo];
  ti.row0 = S.grp_row0[lo];
  const int mt = (ti.rows + BM - 1) / BM;
  const int local = tile - S.tile_start[lo];
  ti.m0 = (local % mt) * BM;
  ti.n0 = (local / mt) * n_tile;
  return ti;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mA,
                        const __grid_constant__ CUtensorMap mA_sh,
                        const __grid_constant__ CUtensorMap mB0,
                        const __grid_constant__ CUtensorMap mB1,
                        const __grid_constant__ CUtensorMap mB0_sh,
                        const __grid_constant__ CUtensorMap mB1_sh, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles_n = (p.N + p.n_tile - 1) / p.n_tile;
  const int nkb = (p.K + BK - 1) / BK;

  // ---------------------------------------------------------------- set-up
  const int ngroups = p.E + (p.has_shared ? 1 : 0);
  if (tid == 0) {
    S.ngroups = ngroups;
    S.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.tfull[b], 1);
      mbar_init(&S.tempty[b], 128);
    }
    mbar_init(&S.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  for (int g = tid; g < ngroups; g += kThreads) {
    int rows, row0;
    if (g < p.E) {
      const int a = p.offsets[g], b = p.offsets[g + 1];
      if (a < 0 || b < a || b > p.Tk) {
        set_status(p.status, MOE_ERR_DEVICE_INDEX);
        rows = 0;
        row0 = 0;
      } else {
        rows = b - a;
        row0 = a;
      }
    } else {
      rows = p.T;
      row0 = (MODE == GATE_UP) ? 0 : p.Tk;
    }
    S.grp_rows[g] = rows;
    S.grp_row0[g] = row0;
    S.tile_start[g] = ((rows + BM - 1) / BM) * n_tiles_n;   // count, scanned below
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < ngroups; base += 32) {
      const int g = base + lane;
      const int c = (g < ngroups) ? S.tile_start[g] : 0;
      int v = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (g < ngroups) S.tile_start[g] = carry + v - c;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
      S.tile_start[ngroups] = carry;
      S.total_tiles = carry;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_base;
  const int total = S.total_tiles;
  const volatile int* abort_flag = &S.abort_flag;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mB0);
    tma_prefetch_desc(&mB1);
    if (p.has_shared) {
      tma_prefetch_desc(&mA_sh);
      tma_prefetch_desc(&mB0_sh);
      tma_prefetch_desc(&mB1_sh);
    }
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile(S, tile, p.n_tile);
      const bool sh = ti.g >= p.E;
      const CUtensorMap* a_map = sh ? &mA_sh : &mA;
      const int ay = ti.row0 + ti.m0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&S.empty[stage], phase ^ 1u, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        uint8_t* st = S.tiles[stage];
        if (p.test_hook == MOE_TEST_HOOK_WITHHOLD_LOAD && tile == (int)blockIdx.x && kb == 0) {
          // test only: the first stage is never filled, so the MMA issuer's bounded wait
          // on it runs out and the CTA takes its timeout path
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        mbar_arrive_expect_tx(&S.full[stage], kStageBytes);
        tma_load_2d(st, a_map, &S.full[stage], kb * BK, ay);
        if (MODE == GATE_UP) {
          if (sh) {
            tma_load_2d(st + kABytes, &mB0_sh, &S.full[stage], kb * BK, ti.n0);
            tma_load_2d(st + kABytes + kBBoxBytes, &mB1_sh, &S.full[stage], kb * BK, ti.n0);
          } else {
            tma_load_3d(st + kABytes, &mB0, &S.full[stage], kb * BK, ti.n0, ti.g);
            tma_load_3d(st + kABytes + kBBoxBytes, &mB1, &S.full[stage], kb * BK, ti.n0,
                        ti.g);
          }
        } else {
          if (sh) {
            tma_load_2d(st + kABytes, &mB0_sh, &S.full[stage], kb * BK, ti.n0);
            tma_load_2d(st + kABytes + kBBoxBytes, &mB0_sh, &S.full[stage], kb * BK,
                        ti.n0 + 128);
          } else {
            tma_load_3d(st + kABytes, &mB0, &S.full[stage], kb * BK, ti.n0, ti.g);
            tma_load_3d(st + kABytes + kBBoxBytes, &mB0, &S.full[stage], kb * BK,
                        ti.n0 + 128, ti.g);
          }
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      S.abort_flag = 1;
      set_status(p.status, MOE_ERR_TIMEOUT);
      // let every copy already issued land before the CTA's shared memory goes away
      const int zero = 0;
      for (int s = 0; s < kStages; ++s)
        if (issued_mask >> s & 1u)
          mbar_wait(&S.full[s], issued_parity >> s & 1u, &zero, p.wait_limit_ns);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      if (!mbar_wait(&S.tempty[acc], acc_phase ^ 1u, abort_flag, p.wait_limit_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + acc * kAccCols;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&S.full[stage], phase, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(S.tiles[stage]);
        const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
        const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + kABytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16(d, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, (kb | kk) != 0);
        umma_commit(&S.empty[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit(&S.tfull[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok) {
      S.abort_flag = 1;
      set_status(p.status, MOE_ERR_TIMEOUT);
      // wait for the MMAs already issued before TMEM is released
      umma_commit(&S.drain);
      const int zero = 0;
      mbar_wait(&S.drain, 0, &zero, p.wait_limit_ns);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int r_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = decode_tile(S, tile, p.n_tile);
      const bool got = mbar_wait(&S.tfull[acc], acc_phase, abort_flag, p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        S.abort_flag = 1;
        set_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + acc * kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      const int m = ti.m0 + r_in_tile;
      const bool valid = m < ti.rows;
      const bool sh = ti.g >= p.E;
      if (MODE == GATE_UP) {
        const size_t out_row = sh ? (size_t)p.Tk + m : (size_t)ti.row0 + m;
        __nv_bfloat16* dst = p.h + out_row * p.N + ti.n0;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c, g);
          tmem_ld32(tb + 128 + c, u);
          tmem_ld_wait();
          if (valid && ti.n0 + c < p.N) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16(silu_mul(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                silu_mul(__uint_as_float(g[2 * i + 1]),
                                         __uint_as_float(u[2 * i + 1])));
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      } else {
        float* dst = sh ? p.O_shared + (size_t)m * p.N : p.O + ((size_t)ti.row0 + m) * p.N;
        dst += ti.n0;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t v[32];
          tmem_ld32(tb + c, v);
          tmem_ld_wait();
          if (valid && ti.n0 + c < p.N) {
            float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                  __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&S.tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ---------------------------------------------------------------- tear-down
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

bool encode_2d(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t inner,
               uint64_t outer, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {BK, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t inner,
               uint64_t mid, uint64_t outer) {
  const cuuint64_t dims[3] = {inner, mid, outer};
  const cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  const cuuint32_t box[3] = {BK, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_tc(const ExpertArgs& a, EncodeTiledFn enc, bool* encode_failed,
                      cudaStream_t s) {
  *encode_failed = false;
  const int Tk = a.T * a.k;
  const int K = (MODE == GATE_UP) ? a.H : a.I;
  const int N = (MODE == GATE_UP) ? a.I : a.H;
  const int n_tile = (MODE == GATE_UP) ? 128 : 256;
  const int h_rows = Tk + (a.has_shared ? a.T : 0);
  CUtensorMap mA, mA_sh, mB0, mB1, mB0_sh, mB1_sh;
  bool ok = true;
  if (MODE == GATE_UP) {
    ok &= encode_2d(enc, &mA, a.Xperm, K, Tk, BM);
    ok &= encode_2d(enc, &mA_sh, a.has_shared ? a.X : a.Xperm, K,
                    a.has_shared ? a.T : Tk, BM);
    ok &= encode_3d(enc, &mB0, a.W_gate, K, N, a.E);
    ok &= encode_3d(enc, &mB1, a.W_up, K, N, a.E);
    ok &= encode_2d(enc, &mB0_sh, a.has_shared ? a.Ws_gate : a.W_gate, K, N, 128);
    ok &= encode_2d(enc, &mB1_sh, a.has_shared ? a.Ws_up : a.W_up, K, N, 128);
  } else {
    ok &= encode_2d(enc, &mA, a.h, K, h_rows, BM);
    mA_sh = mA;
    ok &= encode_3d(enc, &mB0, a.W_down, K, N, a.E);
    mB1 = mB0;
    ok &= encode_2d(enc, &mB0_sh, a.has_shared ? a.Ws_down : a.W_down, K, N, 128);
    mB1_sh = mB0_sh;
  }
  if (!ok) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  TcParams p;
  p.offsets = a.offsets;
  p.E = a.E;
  p.has_shared = a.has_shared;
  p.T = a.T;
  p.Tk = Tk;
  p.K = K;
  p.N = N;
  p.n_tile = n_tile;
  p.h = static_cast<__nv_bfloat16*>(a.h);
  p.O = a.O;
  p.O_shared = a.O_shared;
  p.status = a.status;
  p.test_hook = a.test_hook;
  p.wait_limit_ns = a.wait_limit_ns;

  const int n_tiles_n = (N + n_tile - 1) / n_tile;
  const long long m_tiles_bound =
      (Tk + BM - 1) / BM + a.E + (a.has_shared ? (a.T + BM - 1) / BM : 0);
  const long long tiles_bound = m_tiles_bound * n_tiles_n;
  const int grid = (int)(tiles_bound < a.num_sms ? (tiles_bound > 0 ? tiles_bound : 1)
                                                 : a.num_sms);
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  grouped_gemm_kernel<MODE><<<grid, kThreads, smem, s>>>(mA, mA_sh, mB0, mB1, mB0_sh,
                                                         mB1_sh, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_gate_up_tc(const ExpertArgs& a, EncodeTiledFn enc,
                                     bool* encode_failed, cudaStream_t s) {
  return launch_tc<GATE_UP>(a, enc, encode_failed, s);
}

cudaError_t launch_expert_down_tc(const ExpertArgs& a, EncodeTiledFn enc,
                                  bool* encode_failed, cudaStream_t s) {
  return launch_tc<DOWN>(a, enc, encode_failed, s);
}

}  // namespace moe
