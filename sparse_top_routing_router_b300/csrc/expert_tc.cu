// Step 5 of the MoE forward on the 5th-generation tensor cores ("LLM Internals §14.2.1
// step 5": one GEMM per expert over its m_i rows, [m_i, H] x W_i[H, I] -> [m_i, I],
// then back to H; §14.2.2: the expert is a three-matrix SwiGLU).
//
// One persistent, warp-specialised kernel template serves both GEMMs of the expert:
//   GATE_UP: h = SiLU(x W_gate^T) * (x W_up^T), bf16 out.  One 256-column accumulator
//            holds the gate tile (columns 0-127) and the up tile (128-255) of the same
//            rows, so the SwiGLU is applied in the epilogue straight from TMEM.
//   DOWN:    o = h W_down^T, fp32 out, 256-column tiles.
// and two shapes of work unit:
//   single CTA (PAIR = false): 128-row tiles, tcgen05.mma.cta_group::1 M=128 N=256 (M=64
//            for a group's last tile of at most 64 rows); a stage holds A [128 x 64] and
//            both weight boxes [2 x 128 x 64] (48 KB), 4 stages.
//   CTA pair   (PAIR = true):  a cluster of 2 CTAs owns a 256-row tile; each CTA loads its
//            own 128 rows of A and one 128-row weight box (32 KB per stage, 6 stages),
//            the leader CTA issues tcgen05.mma.cta_group::2 M=256 N=256 over both CTAs'
//            shared memory, and each CTA's TMEM receives its 128 rows.  Per SM the
//            operand traffic per MMA cycle drops by a third and the ring is 1.5x deeper.
//   single-CTA clusters (MCA = true, the down GEMM): two CTAs take the two n-tiles of one
//            128-row block and each multicasts half of its A rows to both.
// Work items are (group, n-tile, m-tile) with the m-tile fastest, enumerated on the
// device from the dispatch offsets (the host never learns m_i), assigned round-robin
// to the resident CTAs (or CTA pairs).  Neighbouring units thus share the weight tile of
// an expert through L2.  The shared expert is one more group whose rows are all T tokens.
//
// Roles (192 threads per CTA):
//   warp 0      TMA producer (128-byte swizzle), full/empty mbarrier ring
//   warp 1      TMEM allocation (512 columns = two 256-column accumulators); one lane of
//               the (leader) CTA issues the MMAs
//   warps 2-5   epilogue: tcgen05.ld 32 columns at a time, SwiGLU or fp32 store
// Every mbarrier wait is bounded (see ptx.cuh); a timeout sets the status word and the
// CTA drains what it can of its in-flight copies and MMAs, frees TMEM and returns.
#include <string.h>

#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BK = 64;
constexpr int kBoxBytes = 128 * BK * 2;   // one [128 x 64] bf16 box
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kMaxGroups = kMaxE + 1;
constexpr int kMaxRing = 12;   // router tiles of a narrow N cut the same bytes into more stages

enum Mode { GATE_UP = 0, DOWN = 1, ROUTER = 2 };
// A group taller than kMBlockRows rows runs its m-tiles in blocks of kMBlockRows rows,
// every n-tile of a block before the next block, so that the block's A rows (29 MB at
// H = 7168) stay in L2 across its n-tiles.  Without the blocks a tall group - above all the
// shared expert, whose A is all of X - streams its A once per n-tile pass.
constexpr int kMBlockRows = 2048;

template <bool PAIR>
struct Cfg {
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kStageBytes = PAIR ? 2 * kBoxBytes : 3 * kBoxBytes;
  static constexpr int kTileM = PAIR ? 256 : 128;            // rows per work unit
  static constexpr int kTxBytes = PAIR ? 4 * kBoxBytes : 3 * kBoxBytes;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(PAIR ? 256 : 128, 256);
};
// bytes that complete one stage: single CTA A + 2 B boxes (48 KB); pair: 2 x (A + B) (64 KB)
static_assert(Cfg<false>::kTxBytes == 3 * kBoxBytes, "");
static_assert(Cfg<true>::kTxBytes == 4 * kBoxBytes, "");

struct TcParams {
  const int32_t* offsets;
  int E, has_shared, T, Tk;
  int K;        // reduction length
  int N;        // output width
  int n_tile;   // output columns per tile: 128 (GATE_UP), 256 (DOWN), E to 16 (ROUTER)
  __nv_bfloat16* h;
  float* O;
  float* O_shared;
  int* status;
  int test_hook;
  unsigned long long wait_limit_ns;
  // ROUTER: split-K factor, period of A's reduction coordinate, partial-logit output
  int splits;
  int a_kmod;
  float2* logits;       // splits == 1: (l, 0) per (token, expert)
  float* logits_part;   // splits > 1: fp32 partial per (slice, token, expert)
  int swap_rows;        // single CTA: tails of at most this many rows swap operands (0: none)
  int pieces;           // ROUTER: 3 = per 64 h one X box and three W_g-piece boxes;
                        // 1 = reduction over [X, X, X] . [hi; mid; lo] (K = 3H)
  uint32_t piece_bytes; // ROUTER, pieces == 3: bytes of one W_g-piece box
  uint32_t router_tx;   // bytes per stage: A box + the W_g-piece box(es)
  int ring;             // stages of the ring (ROUTER; the others use Cfg::kStages)
  uint32_t stage_bytes; // bytes between stages (ROUTER; a multiple of 1024)
};

template <bool PAIR>
struct __align__(1024) Smem {
  uint8_t tiles[Cfg<PAIR>::kStages][Cfg<PAIR>::kStageBytes];
  uint64_t full[kMaxRing];
  uint64_t empty[kMaxRing];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int ngroups;
  int total_tiles;
  int tile_start[kMaxGroups + 1];
  int grp_rows[kMaxGroups];
  int grp_row0[kMaxGroups];   // first A row of the group
  int grp_out0[kMaxGroups];   // first output row (h, O or O_shared) of the group
  float stage[4][32][33];     // epilogue: one 32 x 32 fp32 chunk per warp, padded rows
};

// dynamic shared memory of one CTA (+ 1 KB to align the tiles) within the 227 KB limit
static_assert(sizeof(Smem<false>) + 1024 <= 227 * 1024, "single-CTA shared memory");
static_assert(sizeof(Smem<true>) + 1024 <= 227 * 1024, "CTA-pair shared memory");

// The gate and up weights as 64-row boxes: a CTA pair's half tile takes them in the
// order [gate 0-63 | up 0-63 | gate 64-127 | up 64-127] (see half_tile).
struct HalfMaps {
  CUtensorMap gate, up, gate_sh, up_sh;
  // A (and the shared expert's A) with 64-row boxes: a tile of at most 64 live rows per
  // CTA (single-CTA tails of <= 64 rows, a pair's half tiles) loads only those rows
  CUtensorMap a64, a64_sh;
};

struct TileInfo {
  int g, m0, n0, rows, row0, out0, z;
};

template <bool PAIR>
__device__ __forceinline__ TileInfo decode_tile(const Smem<PAIR>& S, int tile, int n_tile,
                                                int n_tiles_n, int mblock) {
  int lo = 0, hi = S.ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  constexpr int TM = Cfg<PAIR>::kTileM;
  TileInfo ti;
  ti.g = lo;
  ti.rows = S.grp_rows[lo];
  ti.row0 = S.grp_row0[lo];
  ti.out0 = S.grp_out0[lo];
  const int mt = (ti.rows + TM - 1) / TM;
  const int local = tile - S.tile_start[lo];
  if (mblock > 0 && mt > mblock) {
    // a group taller than mblock m-tiles: blocks of mblock m-tiles, every n-tile of a block
    // before the next block, so that the block's A rows stay in L2 across the n-tiles
    const int per_block = mblock * n_tiles_n;
    const int b = local / per_block;
    const int in = local - b * per_block;
    const int bm = min(mblock, mt - b * mblock);
    ti.m0 = (b * mblock + in % bm) * TM;
    ti.n0 = (in / bm) * n_tile;
    ti.z = 0;
    return ti;
  }
  ti.m0 = (local % mt) * TM;
  const int rest = local / mt;                 // n-tile, then split-K slice (router)
  ti.n0 = (rest % n_tiles_n) * n_tile;
  ti.z = rest / n_tiles_n;
  return ti;
}

// Tiny tail tiles of the single-CTA kernel (at most kSwapRows rows left in the group, as
// in nearly every group of a decode-sized batch) swap the operands:
// D^T = W_box . X^T, one MMA per 128-row weight box, M = 128 weight rows and N = the
// live rows rounded up to 16.  A normal tile would spend a full M = 128 MMA on a handful
// of rows; the swapped one does about an eighth of the multiply-adds (less power under
// the board's cap) and reads fewer operand bytes.  Swapping larger tails was slower:
// every M = 128 MMA still reads its whole weight operand from shared memory, so two
// swapped MMAs per k-step cost as much as one full tile once N passes ~64.  Only batches
// of under 16 rows per expert on average use them (TcParams::swap_rows): in a skewed
// prefill (DSV3-shaped) the faster tiny tiles let the CTAs that share a weight tile drift
// apart, more weight loads then come from HBM, and the forward was 3 % slower (while the
// decode-sized layer gained 1.5 %).  The TMA loads are those of a normal tile.
// Accumulator columns: box 0 (gate, or W_down rows n0..) at 0, box 1 (up, or W_down rows
// n0+128..) at kSwapCol1.
constexpr int kSwapRows = 16;
constexpr int kSwapCol1 = 128;

__device__ __forceinline__ bool is_swapped_tail(const TileInfo& ti, int swap_rows) {
  return ti.rows - ti.m0 <= swap_rows;
}

__device__ __forceinline__ int swap_cols(const TileInfo& ti) {
  return (ti.rows - ti.m0 + 15) & ~15;   // 16..kSwapRows rounded up to 16
}

// Single-CTA tail tiles of at most 64 live rows run as M = 64 MMAs (half the multiply-adds
// of an M = 128 tile).  Their accumulator rows sit 16 to a TMEM lane quadrant: row r in
// lane 32 (r / 16) + r % 16, so epilogue warp q holds rows 16 q .. 16 q + 15 in its
// lanes 0-15.
__device__ __forceinline__ bool is_m64_tail(const TileInfo& ti) {
  return ti.rows - ti.m0 <= 64;
}

// CTA pairs: a group's last tile of at most 128 rows runs as M = 128 (64 rows from each
// CTA) instead of M = 256.  In that shape each CTA's TMEM holds its 64 rows twice over:
// lanes 0-63 with accumulator columns 0-127 and lanes 64-127 with columns 128-255, both in
// TMEM columns 0-127 (an in-bounds probe of the instruction's data-path layout
// established this), and a half tile loads gate and up as 64-row boxes (HalfMaps).
// Same-call A/Bs on the Mixtral-shaped layer (8 groups of 969-1073 rows, 5 with a tail of
// at most 128): 2.48-2.52 ms per forward before, 2.46-2.49 with half tiles.
template <bool PAIR>
__device__ __forceinline__ bool half_tile(const TileInfo& ti) {
  return PAIR && ti.rows - ti.m0 <= 128;
}

// A warp's 32 rows x 32 fp32 columns (thread = row, v = its 32 columns, as tcgen05.ld
// 32x32b returns them) to global memory row-contiguously: through the warp's padded
// shared-memory chunk (conflict-free both ways), then every store writes 4 rows x 128 B.
// A direct store from the TMEM layout would touch 32 rows x 16 B per instruction.
// dst0 = the chunk's (row 0, column 0); rows from nrows on are skipped.
__device__ __forceinline__ void store_chunk_f32(float (*stg)[33], const uint32_t (&v)[32],
                                                int lane, float* dst0, size_t ld, int nrows) {
#pragma unroll
  for (int i = 0; i < 32; ++i) stg[lane][i] = __uint_as_float(v[i]);
  __syncwarp();
  const int f = lane & 7;
#pragma unroll
  for (int pass = 0; pass < 8; ++pass) {
    const int r = pass * 4 + (lane >> 3);
    if (r < nrows)
      *reinterpret_cast<float4*>(dst0 + (size_t)r * ld + 4 * f) =
          make_float4(stg[r][4 * f], stg[r][4 * f + 1], stg[r][4 * f + 2], stg[r][4 * f + 3]);
  }
  __syncwarp();
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// SWAP: single-CTA launches of decode-sized batches, whose tiny tails swap operands; a
// separate instantiation, so that the other kernels keep their code unchanged.
// MCA: single-CTA tiles run by clusters of two CTAs that take the two n-tiles of one
// (group, n-tile pair, m-tile) unit; each CTA loads half of the unit's A rows and
// multicasts them to both, so A is read from L2 once for two tiles.  A ring stage is
// released only when both CTAs' MMAs have read it (each MMA issuer commits to both CTAs'
// empty barriers).
template <int MODE, bool PAIR, bool SWAP = false, bool MCA = false>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mA,
                        const __grid_constant__ CUtensorMap mA_sh,
                        const __grid_constant__ CUtensorMap mB0,
                        const __grid_constant__ CUtensorMap mB1,
                        const __grid_constant__ CUtensorMap mB0_sh,
                        const __grid_constant__ CUtensorMap mB1_sh,
                        const __grid_constant__ HalfMaps hm, const TcParams p) {
  using C = Cfg<PAIR>;
  const int kStages = MODE == ROUTER ? p.ring : C::kStages;
  const uint32_t stage_bytes = MODE == ROUTER ? p.stage_bytes : (uint32_t)C::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  Smem<PAIR>& S = *reinterpret_cast<Smem<PAIR>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkb = (p.K + BK - 1) / BK;
  static_assert(!MCA || (!PAIR && !SWAP && MODE != ROUTER), "MCA: single-CTA expert GEMMs");
  constexpr bool CL = PAIR || MCA;                         // launched as clusters of two
  const uint32_t rank = CL ? cluster_ctarank() : 0u;       // 0 = leader
  const int unit = CL ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_units = CL ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int mblock = MODE == ROUTER ? 0 : kMBlockRows / Cfg<PAIR>::kTileM;
  // MCA: a unit spans two n-tiles (the host launches MCA only for an even count)
  const int n_tile_u = MCA ? 2 * p.n_tile : p.n_tile;
  const int n_units_n = (p.N + n_tile_u - 1) / n_tile_u;
  auto decode = [&](int t) {
    TileInfo ti = decode_tile<PAIR>(S, t, n_tile_u, n_units_n, mblock);
    if (MCA) ti.n0 += (int)rank * p.n_tile;
    return ti;
  };

  // ---------------------------------------------------------------- set-up
  const int ngroups = (MODE == ROUTER) ? 1 : p.E + (p.has_shared ? 1 : 0);
  if (tid == 0) {
    S.ngroups = ngroups;
    S.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], MCA ? 2 : 1);   // MCA: both CTAs' MMAs release a stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.tfull[b], 1);
      mbar_init(&S.tempty[b], PAIR ? 256 : 128);
    }
    mbar_init(&S.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&S.tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&S.tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  constexpr int TM = C::kTileM;
  for (int g = tid; g < ngroups; g += kThreads) {
    int rows, row0, out0;
    if (MODE == ROUTER) {
      rows = p.T;
      row0 = 0;
      out0 = 0;
    } else if (g < p.E) {
      const int a = p.offsets[g], b = p.offsets[g + 1];
      if (a < 0 || b < a || b > p.Tk) {
        set_status(p.status, MOE_ERR_DEVICE_INDEX);
        rows = 0;
        row0 = 0;
      } else {
        rows = b - a;
        row0 = a;
      }
      out0 = row0;   // routed rows: h and O rows follow the permuted rows
    } else {
      rows = p.T;    // shared expert: A = X (gate/up) or h rows Tk.. (down)
      row0 = (MODE == GATE_UP) ? 0 : p.Tk;
      out0 = (MODE == GATE_UP) ? p.Tk : 0;   // h rows Tk.., O_shared rows 0..
    }
    S.grp_rows[g] = rows;
    S.grp_row0[g] = row0;
    S.grp_out0[g] = out0;
  }
  __syncthreads();
  for (int g = tid; g < ngroups; g += kThreads)
    S.tile_start[g] = ((S.grp_rows[g] + TM - 1) / TM) * n_units_n *
                      (MODE == ROUTER ? p.splits : 1);     // count, scanned below
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
  if (CL) cluster_sync();   // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_base;
  const int total = S.total_tiles;
  const volatile int* abort_flag = &S.abort_flag;
  const unsigned long long lim = p.wait_limit_ns;
  constexpr bool M64 = !PAIR && MODE != ROUTER;   // M = 64 tail tiles (single CTA)

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
    for (int tile = unit; tile < total && ok; tile += n_units) {
      const TileInfo ti = decode(tile);
      const bool sh = (MODE == ROUTER) || ti.g >= p.E;
      const CUtensorMap* a_map = sh ? &mA_sh : &mA;
      // a pair's half tile (M = 128) takes 64 rows from each CTA
      const int ay = ti.row0 + ti.m0 + (PAIR ? (half_tile<PAIR>(ti) ? 64 : 128) * (int)rank : 0);
      const int kb_lo = (MODE == ROUTER) ? (int)((long long)nkb * ti.z / p.splits) : 0;
      const int kb_hi = (MODE == ROUTER) ? (int)((long long)nkb * (ti.z + 1) / p.splits) : nkb;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!mbar_wait(&S.empty[stage], phase ^ 1u, abort_flag, lim)) {
          ok = false;
          break;
        }
        uint8_t* st = &S.tiles[0][0] + (size_t)stage * stage_bytes;
        if (p.test_hook == MOE_TEST_HOOK_WITHHOLD_LOAD && tile == unit && kb == kb_lo) {
          // test only: the first stage is never filled, so the MMA issuer's bounded wait
          // on it runs out and the CTA takes its timeout path
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        const int kx = kb * BK;
        if (MODE == ROUTER && p.pieces == 3) {
          // one X box and the hi, mid, lo boxes of the same 64 h
          mbar_arrive_expect_tx(&S.full[stage], p.router_tx);
          tma_load_2d(st, a_map, &S.full[stage], kx, ay);
#pragma unroll
          for (int q = 0; q < 3; ++q)
            tma_load_2d(st + kBoxBytes + q * p.piece_bytes, &mB0_sh, &S.full[stage],
                        kx + q * p.a_kmod, ti.n0);
        } else if (!PAIR) {
          // a tail of at most 64 rows (M = 64 or operand-swapped MMAs) reads A rows 0-63
          const bool a64 = MODE != ROUTER && is_m64_tail(ti);
          mbar_arrive_expect_tx(&S.full[stage],
                                MODE == ROUTER ? p.router_tx
                                               : (a64 ? C::kTxBytes - kBoxBytes / 2 : C::kTxBytes));
          // ROUTER over [X, X, X] . [hi; mid; lo]: the k-blocks run h-block by h-block,
          // the three pieces of a 64-wide block of h one after another, so a split-K slice
          // covers a range of h with all three pieces and each X box comes from DRAM once
          // (the next two loads of it hit L2)
          const int ka = MODE == ROUTER ? (kb / 3) * BK : kx;
          const int kw = MODE == ROUTER ? (kb % 3) * p.a_kmod + (kb / 3) * BK : kx;
          if (MCA) {
            // half of the unit's A rows from each CTA, multicast to both; a tail of at most
            // 64 rows comes whole from the leader
            const CUtensorMap* a_half = sh ? &hm.a64_sh : &hm.a64;
            if (!a64)
              tma_load_2d_mc(st + (int)rank * (kBoxBytes / 2), a_half, &S.full[stage], ka,
                             ay + 64 * (int)rank, 0x3);
            else if (rank == 0)
              tma_load_2d_mc(st, a_half, &S.full[stage], ka, ay, 0x3);
          } else {
            tma_load_2d(st, a64 ? (sh ? &hm.a64_sh : &hm.a64) : a_map, &S.full[stage], ka, ay);
          }
          const CUtensorMap* b0 = sh ? &mB0_sh : &mB0;
          const CUtensorMap* b1 = (MODE == GATE_UP) ? (sh ? &mB1_sh : &mB1) : b0;
          const int n1 = (MODE == GATE_UP) ? ti.n0 : ti.n0 + 128;
          if (sh) {
            tma_load_2d(st + kBoxBytes, b0, &S.full[stage], kw, ti.n0);
            // a router tile of at most 128 experts takes one box of n_tile rows
            if (MODE != ROUTER || p.n_tile > 128)
              tma_load_2d(st + 2 * kBoxBytes, b1, &S.full[stage], kw, n1);
          } else {
            tma_load_3d(st + kBoxBytes, b0, &S.full[stage], kx, ti.n0, ti.g);
            tma_load_3d(st + 2 * kBoxBytes, b1, &S.full[stage], kx, n1, ti.g);
          }
        } else {
          // both CTAs' copies count on the leader's barrier; the leader expects all bytes.
          // A half tile (M = 128) takes 64 rows of A from each CTA.
          const bool hf = half_tile<PAIR>(ti);
          if (rank == 0)
            mbar_arrive_expect_tx(&S.full[stage], hf ? C::kTxBytes - kBoxBytes : C::kTxBytes);
          const uint32_t bar = mapa_shared(smem_u32(&S.full[stage]), 0);
          tma_load_2d_pair(st, hf ? (sh ? &hm.a64_sh : &hm.a64) : a_map, bar, kx, ay);
          // weight half of this CTA.  GATE_UP full tile: rank 0 the gate rows, rank 1 the
          // up rows n0 .. + 127; half tile: gate rows n0 + 64 r .. + 63, then the up rows
          // of the same outputs (64-row boxes), so that every TMEM lane holds the gate and
          // up of the same outputs.  DOWN: output rows n0 + 128 r .. + 127.
          if (MODE == GATE_UP && half_tile<PAIR>(ti)) {
            const int ny = ti.n0 + 64 * (int)rank;
            if (sh) {
              tma_load_2d_pair(st + kBoxBytes, &hm.gate_sh, bar, kx, ny);
              tma_load_2d_pair(st + kBoxBytes + kBoxBytes / 2, &hm.up_sh, bar, kx, ny);
            } else {
              tma_load_3d_pair(st + kBoxBytes, &hm.gate, bar, kx, ny, ti.g);
              tma_load_3d_pair(st + kBoxBytes + kBoxBytes / 2, &hm.up, bar, kx, ny, ti.g);
            }
          } else if (MODE == GATE_UP) {
            const CUtensorMap* b = rank == 0 ? (sh ? &mB0_sh : &mB0) : (sh ? &mB1_sh : &mB1);
            if (sh) tma_load_2d_pair(st + kBoxBytes, b, bar, kx, ti.n0);
            else tma_load_3d_pair(st + kBoxBytes, b, bar, kx, ti.n0, ti.g);
          } else {
            const CUtensorMap* b = sh ? &mB0_sh : &mB0;
            const int ny = ti.n0 + 128 * (int)rank;
            if (sh) tma_load_2d_pair(st + kBoxBytes, b, bar, kx, ny);
            else tma_load_3d_pair(st + kBoxBytes, b, bar, kx, ny, ti.g);
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
      // (in a pair only the leader's barriers count the copies)
      const int zero = 0;
      if (!PAIR || rank == 0)
        for (int s = 0; s < kStages; ++s)
          if (issued_mask >> s & 1u) mbar_wait(&S.full[s], issued_parity >> s & 1u, &zero, lim);
    }
  } else if (warp == 1 && lane == 0 && (rank == 0 || !PAIR)) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    // the router's N is the expert count rounded up to 16 (at most 256)
    const uint32_t idesc = MODE == ROUTER ? idesc_bf16_f32(128, p.n_tile) : C::kIdesc;
    for (int tile = unit; tile < total && ok; tile += n_units) {
      int kb_lo = 0, kb_hi = nkb;
      bool swap = false;
      uint32_t sw_idesc = 0;
      uint32_t mma_idesc = idesc;
      if (MODE == ROUTER) {
        const TileInfo ti = decode(tile);
        kb_lo = (int)((long long)nkb * ti.z / p.splits);
        kb_hi = (int)((long long)nkb * (ti.z + 1) / p.splits);
      } else if (SWAP || M64) {
        const TileInfo ti = decode(tile);
        swap = SWAP && is_swapped_tail(ti, p.swap_rows);
        if (swap) sw_idesc = idesc_bf16_f32(128, swap_cols(ti));
        else if (M64 && is_m64_tail(ti)) mma_idesc = idesc_bf16_f32(64, 256);
      }
      uint32_t pair_idesc = C::kIdesc;
      if (PAIR && half_tile<PAIR>(decode(tile)))
        pair_idesc = idesc_bf16_f32(128, 256);
      const bool got = PAIR ? mbar_wait_cluster(&S.tempty[acc], acc_phase ^ 1u, abort_flag, lim)
                            : mbar_wait(&S.tempty[acc], acc_phase ^ 1u, abort_flag, lim);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + acc * kAccCols;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!mbar_wait(&S.full[stage], phase, abort_flag, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(&S.tiles[0][0] + (size_t)stage * stage_bytes);
        const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
        const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + kBoxBytes);
        if (MODE == ROUTER && p.pieces == 3) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
            for (int q = 0; q < 3; ++q) {
              const uint64_t bq = sdesc_kmajor_sw128(a_addr + kBoxBytes + q * p.piece_bytes);
              const uint32_t accum = (kb != kb_lo || kk != 0 || q != 0) ? 1u : 0u;
              umma_bf16(d, adesc + 2 * kk, bq + 2 * kk, idesc, accum);
            }
          }
        } else if (SWAP && MODE != ROUTER && swap) {
          // tiny tail: each weight box is the M = 128 operand, the rows the N operand
          const uint64_t bdesc1 = sdesc_kmajor_sw128(a_addr + 2 * kBoxBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t accum = (kb != kb_lo || kk != 0) ? 1u : 0u;
            umma_bf16(d, bdesc + 2 * kk, adesc + 2 * kk, sw_idesc, accum);
            umma_bf16(d + kSwapCol1, bdesc1 + 2 * kk, adesc + 2 * kk, sw_idesc, accum);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t accum = (kb != kb_lo || kk != 0) ? 1u : 0u;
            if (PAIR) umma_bf16_pair(d, adesc + 2 * kk, bdesc + 2 * kk, pair_idesc, accum);
            else umma_bf16(d, adesc + 2 * kk, bdesc + 2 * kk, mma_idesc, accum);
          }
        }
        if (PAIR) umma_commit_pair_mc(&S.empty[stage], 0x3);
        else if (MCA) umma_commit_mc(&S.empty[stage], 0x3);
        else umma_commit(&S.empty[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (PAIR) umma_commit_pair_mc(&S.tfull[acc], 0x3);
      else umma_commit(&S.tfull[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok) {
      S.abort_flag = 1;
      set_status(p.status, MOE_ERR_TIMEOUT);
      // wait for the MMAs already issued before TMEM is released
      if (PAIR) umma_commit_pair(&S.drain);
      else umma_commit(&S.drain);
      const int zero = 0;
      mbar_wait(&S.drain, 0, &zero, lim);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int r_in_tile = (PAIR ? 128 * (int)rank : 0) + q * 32 + lane;
    const uint32_t tempty_leader =
        PAIR ? mapa_shared(smem_u32(&S.tempty[0]), 0) : 0u;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = unit; tile < total; tile += n_units) {
      const TileInfo ti = decode(tile);
      const bool got = mbar_wait(&S.tfull[acc], acc_phase, abort_flag, lim);
      if (!__all_sync(0xffffffffu, got)) {
        S.abort_flag = 1;
        set_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + acc * kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      const bool m64 = M64 && is_m64_tail(ti) && !(SWAP && is_swapped_tail(ti, p.swap_rows));
      const int m = ti.m0 + (m64 ? q * 16 + (lane & 15) : r_in_tile);
      const bool valid = m < ti.rows && (!m64 || lane < 16);
      const bool sh = ti.g >= p.E;
      if (PAIR && MODE != ROUTER) {
        // A full tile (M = 256): this lane is row 128 r + q*32 + lane with all 256
        // accumulator columns (GATE_UP: gate 0-127, up 128-255).  A half tile (M = 128):
        // row 64 r + (q & 1)*32 + lane, and accumulator columns 128 (q >> 1) .. + 127 in
        // TMEM columns 0-127 (GATE_UP: [gate | up] per 64 outputs, see the producer).
        const bool hf = half_tile<PAIR>(ti);
        const int row = hf ? 64 * (int)rank + (q & 1) * 32 + lane : 128 * (int)rank + q * 32 + lane;
        const int mm = ti.m0 + row;
        const bool ok_row = mm < ti.rows;
        const int hc0 = hf ? (q >> 1) : 0, hc1 = hf ? (q >> 1) : 1;
        if (MODE == GATE_UP && !hf) {
          __nv_bfloat16* dst = p.h + ((size_t)ti.out0 + mm) * p.N + ti.n0;
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(tb + c, g);
            tmem_ld32(tb + 128 + c, u);
            tmem_ld_wait();
            if (ok_row && ti.n0 + c < p.N) {
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
        }
#pragma unroll 1
        for (int hc = hc0; hc <= hc1 && !(MODE == GATE_UP && !hf); ++hc) {
          const uint32_t tcol = hf ? 0u : 128u * (uint32_t)hc;
          if (MODE == GATE_UP) {
            __nv_bfloat16* dst = p.h + ((size_t)ti.out0 + mm) * p.N + ti.n0 + 64 * hc;
#pragma unroll 1
            for (int c = 0; c < 64; c += 32) {
              uint32_t g[32], u[32];
              tmem_ld32(tb + tcol + c, g);
              tmem_ld32(tb + tcol + 64 + c, u);
              tmem_ld_wait();
              if (ok_row && ti.n0 + 64 * hc + c < p.N) {
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
            // this warp's 32 rows start at row - lane
            const int wrow = ti.m0 + row - lane;
            const int nrows = min(32, max(0, ti.rows - wrow));
            float* dst = (sh ? p.O_shared : p.O) + ((size_t)ti.out0 + wrow) * p.N + ti.n0 +
                         128 * hc;
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
              uint32_t v[32];
              tmem_ld32(tb + tcol + c, v);
              tmem_ld_wait();
              if (ti.n0 + 128 * hc + c < p.N)
                store_chunk_f32(S.stage[q], v, lane, dst + c, p.N, nrows);
            }
          }
        }
      } else if (SWAP && MODE != ROUTER && is_swapped_tail(ti, p.swap_rows)) {
        // D^T: this lane holds weight row q*32+lane of each box, the columns are rows
        const int r = ti.rows - ti.m0;
        const int nn = q * 32 + lane;
        uint32_t v0[32], v1[32];
        tmem_ld32(tb, v0);                 // r <= kSwapRows <= 32: one load per box
        tmem_ld32(tb + kSwapCol1, v1);
        tmem_ld_wait();
        if (MODE == GATE_UP) {
          if (ti.n0 + nn < p.N) {
            __nv_bfloat16* dst = p.h + ((size_t)ti.out0 + ti.m0) * p.N + ti.n0 + nn;
#pragma unroll
            for (int i = 0; i < kSwapRows; ++i)
              if (i < r)
                dst[(size_t)i * p.N] = __float2bfloat16_rn(
                    silu_mul(__uint_as_float(v0[i]), __uint_as_float(v1[i])));
          }
        } else {
          float* dst = (sh ? p.O_shared : p.O) + ((size_t)ti.out0 + ti.m0) * p.N + ti.n0 + nn;
          const bool ok0 = ti.n0 + nn < p.N, ok1 = ti.n0 + 128 + nn < p.N;
#pragma unroll
          for (int i = 0; i < kSwapRows; ++i) {
            if (i < r) {
              if (ok0) dst[(size_t)i * p.N] = __uint_as_float(v0[i]);
              if (ok1) dst[(size_t)i * p.N + 128] = __uint_as_float(v1[i]);
            }
          }
        }
      } else if (MODE == ROUTER) {
        // one slice: the logits as (l, 0) pairs; several: fp32 partials for the reduce
        const size_t cell = ((size_t)ti.z * p.T + m) * p.N + ti.n0;
#pragma unroll 1
        for (int c = 0; c < p.n_tile; c += 32) {
          uint32_t v[32];
          tmem_ld32(tb + c, v);
          tmem_ld_wait();
          const int ncol = p.N - ti.n0 - c;   // live columns from c on
          if (!valid || ncol <= 0) continue;
          if (p.splits == 1) {
            float2* dst = p.logits + cell + c;
            if (ncol >= 32) {
              float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                d4[i] = make_float4(__uint_as_float(v[2 * i]), 0.f,
                                    __uint_as_float(v[2 * i + 1]), 0.f);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < ncol) dst[i] = make_float2(__uint_as_float(v[i]), 0.f);
            }
          } else {
            float* dst = p.logits_part + cell + c;
            if (ncol >= 32) {
              float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < ncol) dst[i] = __uint_as_float(v[i]);
            }
          }
        }
      } else if (MODE == GATE_UP) {
        const size_t out_row = (size_t)ti.out0 + m;
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
        // this warp's 32 rows start at m - lane
        const int wrow = m64 ? ti.m0 + q * 16 : m - lane;
        const int nrows = min(m64 ? 16 : 32, max(0, ti.rows - wrow));
        float* dst = (sh ? p.O_shared : p.O) + ((size_t)ti.out0 + wrow) * p.N + ti.n0;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t v[32];
          tmem_ld32(tb + c, v);
          tmem_ld_wait();
          if (ti.n0 + c < p.N) store_chunk_f32(S.stage[q], v, lane, dst + c, p.N, nrows);
        }
      }
      tc_fence_before();
      if (PAIR) mbar_arrive_cluster(tempty_leader + acc * (uint32_t)sizeof(uint64_t));
      else mbar_arrive(&S.tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ---------------------------------------------------------------- tear-down
  tc_fence_before();
  __syncthreads();
  if (CL) cluster_sync();   // no MMA, copy or arrival targets either CTA any more
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <typename Enc>
bool encode_2d(Enc enc, CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
               uint32_t box_rows = 128) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t inner,
               uint64_t mid, uint64_t outer, uint32_t box_rows = 128) {
  const cuuint64_t dims[3] = {inner, mid, outer};
  const cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  const cuuint32_t box[3] = {BK, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Number of clusters of two CTAs that can be resident at once (persistent grid), cached
// per kernel and SM count (thread-safe; a device with another SM count is queried anew).
int max_pairs(const void* fn, size_t smem, int num_sms) {
  static std::mutex mu;
  static const void* fns[16] = {};
  static int sms_of[16] = {};
  static int cached[16] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < 16; ++i)
      if (fns[i] == fn && sms_of[i] == num_sms) return cached[i];
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms & ~1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < 16; ++i)
    if (!fns[i]) {
      fns[i] = fn;
      sms_of[i] = num_sms;
      cached[i] = n;
      break;
    }
  return n;
}

template <int MODE, bool PAIR>
cudaError_t launch_tc(const ExpertArgs& a, EncodeTiledFn enc, bool* encode_failed,
                      cudaStream_t s) {
  *encode_failed = false;
  const int Tk = a.T * a.k;
  const int K = (MODE == GATE_UP) ? a.H : a.I;
  const int N = (MODE == GATE_UP) ? a.I : a.H;
  const int n_tile = (MODE == GATE_UP) ? 128 : 256;
  const int h_rows = Tk + (a.has_shared ? a.T : 0);
  CUtensorMap mA, mA_sh, mB0, mB1, mB0_sh, mB1_sh;
  HalfMaps hm;
  memset(&hm, 0, sizeof(hm));
  bool ok = true;
  if (MODE == GATE_UP) {
    ok &= encode_2d(enc, &mA, a.Xperm, K, Tk);
    ok &= encode_2d(enc, &mA_sh, a.has_shared ? a.X : a.Xperm, K, a.has_shared ? a.T : Tk);
    ok &= encode_3d(enc, &mB0, a.W_gate, K, N, a.E);
    ok &= encode_3d(enc, &mB1, a.W_up, K, N, a.E);
    ok &= encode_2d(enc, &mB0_sh, a.has_shared ? a.Ws_gate : a.W_gate, K, N);
    ok &= encode_2d(enc, &mB1_sh, a.has_shared ? a.Ws_up : a.W_up, K, N);
    if (PAIR) {   // 64-row boxes for the half tiles
      ok &= encode_3d(enc, &hm.gate, a.W_gate, K, N, a.E, 64);
      ok &= encode_3d(enc, &hm.up, a.W_up, K, N, a.E, 64);
      ok &= encode_2d(enc, &hm.gate_sh, a.has_shared ? a.Ws_gate : a.W_gate, K, N, 64);
      ok &= encode_2d(enc, &hm.up_sh, a.has_shared ? a.Ws_up : a.W_up, K, N, 64);
    }
    ok &= encode_2d(enc, &hm.a64, a.Xperm, K, Tk, 64);
    ok &= encode_2d(enc, &hm.a64_sh, a.has_shared ? a.X : a.Xperm, K, a.has_shared ? a.T : Tk,
                    64);
  } else {
    ok &= encode_2d(enc, &mA, a.h, K, h_rows);
    mA_sh = mA;
    ok &= encode_2d(enc, &hm.a64, a.h, K, h_rows, 64);
    hm.a64_sh = hm.a64;
    ok &= encode_3d(enc, &mB0, a.W_down, K, N, a.E);
    mB1 = mB0;
    ok &= encode_2d(enc, &mB0_sh, a.has_shared ? a.Ws_down : a.W_down, K, N);
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
  p.splits = 1;
  p.a_kmod = K;
  p.logits = nullptr;
  p.logits_part = nullptr;
  // decode-sized batches (under 16 rows per expert on average): swap the tiny tails
  p.swap_rows = (!PAIR && (long long)a.T * a.k < 16LL * a.E) ? kSwapRows : 0;
  p.pieces = 1;
  p.piece_bytes = 0;
  p.router_tx = 0;
  p.ring = Cfg<PAIR>::kStages;
  p.stage_bytes = Cfg<PAIR>::kStageBytes;

  constexpr int TM = Cfg<PAIR>::kTileM;
  const int n_tiles_n = (N + n_tile - 1) / n_tile;
  const long long m_tiles_bound =
      (Tk + TM - 1) / TM + a.E + (a.has_shared ? (a.T + TM - 1) / TM : 0);
  const long long tiles_bound = m_tiles_bound * n_tiles_n;
  const size_t smem = sizeof(Smem<PAIR>) + 1024;
  // The down GEMM's single CTAs run as clusters of two that share each A row block when
  // its reduction is short (K = I <= 2048) and the n-tile count is even.  Same-call A/Bs:
  // DSV3-shaped prefill (K = 2048) down 2.25 against 2.30 ms (20 steps) and 2.45 against
  // 2.52 ms (200 steps); but the Switch-shaped down GEMM (K = 8192) 0.683 against
  // 0.671 ms and the DSV3-shaped gate/up GEMM (K = 7168) 3.91 against 3.76 ms.
  // Decode-sized batches keep the operand-swapped kernel.
  constexpr bool kMcaMode = MODE == DOWN && !PAIR;
  const bool mca = kMcaMode && K <= 2048 && p.swap_rows == 0 && n_tiles_n % 2 == 0 &&
                   a.num_sms >= 2;
  auto* fn = p.swap_rows > 0 ? grouped_gemm_kernel<MODE, PAIR, !PAIR>
             : (mca ? grouped_gemm_kernel<MODE, PAIR, false, kMcaMode>
                    : grouped_gemm_kernel<MODE, PAIR, false>);
  cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (!PAIR && !mca) {
    const int grid = (int)(tiles_bound < a.num_sms ? (tiles_bound > 0 ? tiles_bound : 1)
                                                   : a.num_sms);
    fn<<<grid, kThreads, smem, s>>>(mA, mA_sh, mB0, mB1, mB0_sh, mB1_sh, hm, p);
    return cudaGetLastError();
  }
  const int pairs_max = max_pairs(reinterpret_cast<const void*>(fn), smem, a.num_sms);
  const long long units_bound = mca ? tiles_bound / 2 : tiles_bound;
  const int pairs = (int)(units_bound < pairs_max ? (units_bound > 0 ? units_bound : 1)
                                                  : pairs_max);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, mA, mA_sh, mB0, mB1, mB0_sh, mB1_sh, hm, p);
}

// CTA pairs pay off for large experts (>= 512 rows on average).  For smaller ones the
// 256-row pair tile pads too much (DSV3-shaped prefill, groups of 0 to 2113 rows: same-call
// A/B 7.6 ms single-CTA vs 8.3 ms pairs per forward).  Splitting a group between a pair
// launch and a single-CTA launch streams its weights from HBM twice, and sending whole
// groups to one launch or the other gained at most 1 % under the power cap.
bool use_pairs(const ExpertArgs& a) {
  return (long long)a.T * a.k >= 512LL * a.E && a.num_sms >= 2;
}

template <int MODE>
cudaError_t launch_expert(const ExpertArgs& a, EncodeTiledFn enc, bool* bad, cudaStream_t s) {
  return use_pairs(a) ? launch_tc<MODE, true>(a, enc, bad, s)
                      : launch_tc<MODE, false>(a, enc, bad, s);
}

}  // namespace

// Router logits on the tensor cores: A = X [T, H] (its reduction coordinate taken modulo
// H), B = W_g pieces [E][3H] (hi | mid | lo), so one fp32 accumulator receives
// sum_h x_h (hi + mid + lo)_h = sum_h x_h w_h with exact bf16 x bf16 products.
cudaError_t launch_router_tc(const RouterArgs& a, EncodeTiledFnR enc, bool* encode_failed,
                             cudaStream_t s) {
  *encode_failed = false;
  // MMA N = the expert count rounded up to 16 (at most 256); up to 128 experts the W_g
  // pieces come as one box of that many rows, beyond that as two 128-row boxes
  const int n_tile = a.E >= 256 ? 256 : (a.E + 15) & ~15;
  const uint32_t w_rows = n_tile > 128 ? 128u : (uint32_t)n_tile;
  CUtensorMap mX, mW;
  bool ok = encode_2d(enc, &mX, a.X, a.H, a.T);
  ok &= encode_2d(enc, &mW, a.wsplit, 3ull * a.H, a.E, w_rows);
  if (!ok) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  TcParams p = {};
  p.offsets = nullptr;
  p.E = 0;
  p.has_shared = 0;
  p.T = a.T;
  p.Tk = a.T;
  // up to 128 experts: per 64 h one X box and the three piece boxes (X read once);
  // beyond: the reduction runs over [X, X, X] . [hi; mid; lo] (the pieces would not fit
  // a stage together)
  const bool fused = router_tc_fused(a.E);
  p.pieces = fused ? 3 : 1;
  p.piece_bytes = w_rows * BK * 2;
  p.K = fused ? a.H : 3 * a.H;
  p.N = a.E;
  p.n_tile = n_tile;
  p.h = nullptr;
  p.O = nullptr;
  p.O_shared = nullptr;
  p.status = a.status;
  p.test_hook = MOE_TEST_HOOK_NONE;
  p.wait_limit_ns = a.wait_limit_ns;
  p.splits = a.splits;
  p.a_kmod = a.H;
  p.logits = a.logits;
  p.logits_part = a.logits_part;
  p.router_tx = fused ? kBoxBytes + 3u * p.piece_bytes
                      : kBoxBytes + (n_tile > 128 ? 2u * kBoxBytes : p.piece_bytes);
  // the ring's bytes cut into as many stages as fit (a narrow N leaves most of a 48 KB
  // stage unused, and more stages in flight hide more of the load latency)
  p.stage_bytes = (p.router_tx + 1023u) & ~1023u;
  constexpr uint32_t kRingBytes = (uint32_t)sizeof(Smem<false>::tiles);
  p.ring = (int)(kRingBytes / p.stage_bytes);
  if (p.ring > kMaxRing) p.ring = kMaxRing;
  const long long tiles =
      (long long)((a.T + 127) / 128) * ((a.E + p.n_tile - 1) / p.n_tile) * a.splits;
  const int grid = (int)(tiles < a.num_sms ? tiles : a.num_sms);
  const size_t smem = sizeof(Smem<false>) + 1024;
  auto* fn = grouped_gemm_kernel<ROUTER, false>;
  cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  HalfMaps hm;
  memset(&hm, 0, sizeof(hm));
  fn<<<grid, kThreads, smem, s>>>(mX, mX, mW, mW, mW, mW, hm, p);
  return cudaGetLastError();
}

cudaError_t launch_expert_gate_up_tc(const ExpertArgs& a, EncodeTiledFn enc,
                                     bool* encode_failed, cudaStream_t s) {
  return launch_expert<GATE_UP>(a, enc, encode_failed, s);
}

cudaError_t launch_expert_down_tc(const ExpertArgs& a, EncodeTiledFn enc,
                                  bool* encode_failed, cudaStream_t s) {
  return launch_expert<DOWN>(a, enc, encode_failed, s);
}

}  // namespace moe
