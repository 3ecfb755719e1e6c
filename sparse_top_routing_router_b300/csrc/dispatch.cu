// Step 4 of the MoE forward: the dispatch permutation ("LLM Internals §14.2.1 step 4":
// rows re-ordered by expert so that each expert's tokens are contiguous), with the
// optional capacity of "AI Knowledge Map - MoE" (C = ceil(c*N*k/E), overflow dropped,
// the lowest token indices kept).
//
// A stable counting sort of the T*k slots by expert, in four launches:
//  count    per 256-token chunk, per-expert slot counts (shared-memory histogram)
//  scan     per expert, exclusive scan over chunks; m_e; capacity clamp; offsets
//  scatter  per chunk, each slot's rank inside its expert = chunk base + the number of
//           earlier tokens of the chunk routed to the same expert (bitmap popcount);
//           row_of_slot / slot_of_row, or -1 beyond capacity
//  gather   one warp per token: its X row copied once to each of its kept rows, with
//           16-byte vector moves
#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kChunk = kDispatchChunk;   // 256 tokens, one per thread

__global__ void __launch_bounds__(kChunk) dispatch_count_kernel(DispatchArgs a) {
  __shared__ int hist[kMaxE];
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int t = c * kChunk + threadIdx.x;
  if (t < a.T) {
    for (int j = 0; j < a.k; ++j) {
      const int e = a.idx[(size_t)t * a.k + j];
      if (e >= 0 && e < a.E) atomicAdd(&hist[e], 1);
      else set_status(a.status, MOE_ERR_DEVICE_INDEX);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += blockDim.x)
    a.chunk_counts[(size_t)c * a.E + e] = hist[e];
}

// One CTA of 512 threads: thread e walks the chunks of expert e, 16 chunk counts loaded
// at a time (independent loads, then the running sums).
__global__ void __launch_bounds__(kMaxE) dispatch_scan_kernel(DispatchArgs a, int nchunks) {
  __shared__ int s_warp[kMaxE / 32];
  constexpr int kBatch = 16;
  const int e = threadIdx.x;
  int run = 0;
  if (e < a.E) {
    for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q)
        v[q] = (c0 + q < nchunks) ? a.chunk_counts[(size_t)(c0 + q) * a.E + e] : 0;
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (c0 + q < nchunks) a.chunk_base[(size_t)(c0 + q) * a.E + e] = run;
        run += v[q];
      }
    }
    a.counts[e] = run;
  }
  const int kept = (e < a.E) ? (a.capacity >= 0 ? min(run, a.capacity) : run) : 0;
  // block exclusive scan of kept over experts
  const int lane = e & 31, w = e >> 5;
  int v = kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) s_warp[w] = v;
  __syncthreads();
  if (w == 0) {
    int x = (lane < kMaxE / 32) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
    if (lane < kMaxE / 32) s_warp[lane] = x;   // inclusive warp totals
  }
  __syncthreads();
  const int excl = v - kept + (w > 0 ? s_warp[w - 1] : 0);
  if (e < a.E) a.offsets[e] = excl;
  if (e == a.E - 1) a.offsets[a.E] = excl + kept;
}

__global__ void __launch_bounds__(kChunk) dispatch_scatter_kernel(DispatchArgs a) {
  __shared__ uint32_t bits[kMaxE][kChunk / 32];
  const int c = blockIdx.x, tid = threadIdx.x;
  for (int i = tid; i < a.E * (kChunk / 32); i += blockDim.x) (&bits[0][0])[i] = 0u;
  __syncthreads();
  const int t = c * kChunk + tid;
  const int wd = tid >> 5;
  const uint32_t me = 1u << (tid & 31);
  if (t < a.T) {
    for (int j = 0; j < a.k; ++j) {
      const int e = a.idx[(size_t)t * a.k + j];
      // this thread alone sets bit `me`: finding it already set means the token named
      // expert e twice, which would give two slots one row (reported, not repaired)
      if (e >= 0 && e < a.E && (atomicOr(&bits[e][wd], me) & me))
        set_status(a.status, MOE_ERR_DEVICE_INDEX);
    }
  }
  __syncthreads();
  if (t >= a.T) return;
  for (int j = 0; j < a.k; ++j) {
    const size_t s = (size_t)t * a.k + j;
    const int e = a.idx[s];
    if (e < 0 || e >= a.E) {
      a.row_of_slot[s] = -1;
      continue;
    }
    int rank = a.chunk_base[(size_t)c * a.E + e] + __popc(bits[e][wd] & (me - 1u));
    for (int q = 0; q < wd; ++q) rank += __popc(bits[e][q]);
    if (a.capacity >= 0 && rank >= a.capacity) {
      a.row_of_slot[s] = -1;
    } else {
      const int row = a.offsets[e] + rank;
      a.row_of_slot[s] = row;
      a.slot_of_row[row] = (int)s;
    }
  }
}

// Warp per token and column chunk: the token's row is read once (16-byte vectors) and
// written to each of its kept rows.  gridDim.y splits the row into chunks so that a
// small batch still gives every SM several warps.
template <int VEC_BYTES>
__global__ void __launch_bounds__(256) dispatch_gather_kernel(DispatchArgs a,
                                                              int row_bytes) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.T) return;
  int rows[kMaxK];
  int nk = 0;
  for (int j = 0; j < a.k; ++j) {
    const int r = a.row_of_slot[(size_t)t * a.k + j];
    if (r >= 0) rows[nk++] = r;
  }
  if (nk == 0) return;
  const int nvec = row_bytes / 16;
  const int per = (nvec + gridDim.y - 1) / gridDim.y;
  const int v0 = blockIdx.y * per, v1 = min(nvec, v0 + per);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.X) +
                                                    (size_t)t * row_bytes);
  char* dst = static_cast<char*>(a.Xperm);
  for (int v = v0 + lane; v < v1; v += 32) {
    const uint4 x = src[v];
    for (int q = 0; q < nk; ++q)
      reinterpret_cast<uint4*>(dst + (size_t)rows[q] * row_bytes)[v] = x;
  }
}

// Warp per permuted row: Xperm[r] = X[slot_of_row[r] / k] (expert-choice routing, where
// a token may fill any number of rows).  A slot outside [0, T*k) is reported and its
// row left untouched.
__global__ void __launch_bounds__(256) gather_rows_kernel(int R, int k, int T, int row_bytes,
                                                          const int32_t* slot_of_row,
                                                          const void* X, void* Xperm,
                                                          int* status) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= R) return;
  const int slot = slot_of_row[r];
  if (slot < 0 || (long long)slot >= (long long)T * k) {
    if (lane == 0) set_status(status, MOE_ERR_DEVICE_INDEX);
    return;
  }
  const int t = slot / k;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(X) +
                                                    (size_t)t * row_bytes);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(Xperm) + (size_t)r * row_bytes);
  for (int v = lane; v < row_bytes / 16; v += 32) dst[v] = src[v];
}

}  // namespace

cudaError_t launch_gather_rows(int R, int k, int row_bytes, const int32_t* slot_of_row,
                               const void* X, void* Xperm, int* status, int T,
                               cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  gather_rows_kernel<<<(R + 7) / 8, 256, 0, s>>>(R, k, T, row_bytes, slot_of_row, X, Xperm,
                                                 status);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_count(const DispatchArgs& a, cudaStream_t s) {
  const int nchunks = (a.T + kChunk - 1) / kChunk;
  dispatch_count_kernel<<<nchunks, kChunk, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_scan(const DispatchArgs& a, cudaStream_t s) {
  const int nchunks = (a.T + kChunk - 1) / kChunk;
  dispatch_scan_kernel<<<1, kMaxE, 0, s>>>(a, nchunks);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_scatter(const DispatchArgs& a, cudaStream_t s) {
  const int nchunks = (a.T + kChunk - 1) / kChunk;
  dispatch_scatter_kernel<<<nchunks, kChunk, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_gather(const DispatchArgs& a, cudaStream_t s) {
  const int elt = a.x_dtype == MOE_DTYPE_BF16 ? 2 : 4;
  const int row_bytes = a.H * elt;
  // about 32 warps per SM in all: split rows into chunks of at least 32 vectors when the
  // batch alone gives fewer
  const int nvec = row_bytes / 16;
  const long long want = (long long)kGridSms * 32;
  int ysplit = (int)((want + a.T - 1) / (a.T > 0 ? a.T : 1));
  const int ymax = nvec / 32 > 0 ? nvec / 32 : 1;
  ysplit = ysplit < 1 ? 1 : (ysplit > ymax ? ymax : ysplit);
  dispatch_gather_kernel<16><<<dim3((a.T + 7) / 8, ysplit), 256, 0, s>>>(a, row_bytes);
  return cudaGetLastError();
}


// ---------------------------------------------------------------- allocation-free entry
//
// moe_dispatch_static: the same dispatch for callers that may not allocate device memory
// at the moment they dispatch - an inference engine or host runtime that owns all device
// memory and hands out only the buffers it planned, or a process whose allocator must
// never grow (cudaMalloc can also synchronise the device, which a latency-bound decode loop
// cannot afford).  Its scratch (the per-chunk count and base tables) lives in the array
// below, which the module holds on every GPU that loads the library until the process
// exits.

namespace {
constexpr int kStaticMaxT = 65536;                                   // tokens per call
constexpr int kStaticMaxChunks = kStaticMaxT / kDispatchChunk;       // 256
constexpr size_t kStaticScratchInts = 2ull * kStaticMaxChunks * kMaxE;  // 1 MiB of int32
constexpr int kMaxDevices = 64;
}  // namespace

static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchInts];

namespace {
std::mutex g_scratch_mu;
int32_t* g_scratch_addr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device, looked up once per device.
// In host code the array's name is only a host-side stand-in, so kernels must be given
// this address, never the name.
cudaError_t static_scratch(int32_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}
}  // namespace

}  // namespace moe

extern "C" int moe_dispatch_static(int T, int k, int E, int H, int x_dtype, int capacity,
                                   const int32_t* topk_idx, const void* X, int32_t* counts,
                                   int32_t* offsets, int32_t* row_of_slot,
                                   int32_t* slot_of_row, void* Xperm, moe_stream_t stream) {
  using namespace moe;
  const NvtxRange nvtx_range(__func__);
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
  if (E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK)
    return fail(MOE_ERR_INVALID_ARG, "E = %d, k = %d: need 1 <= k <= min(E, %d), E <= %d", E,
                k, kMaxK, kMaxE);
  if (T > kStaticMaxT)
    return fail(MOE_ERR_UNSUPPORTED, "T = %d exceeds the %d tokens the static scratch holds",
                T, kStaticMaxT);
  if (!counts || !offsets) return fail(MOE_ERR_INVALID_ARG, "counts/offsets null");
  if (T > 0 && (!topk_idx || !row_of_slot || !slot_of_row))
    return fail(MOE_ERR_INVALID_ARG, "topk_idx/row_of_slot/slot_of_row null");
  if ((X == nullptr) != (Xperm == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "X and Xperm must be given together");
  if (Xperm) {
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32)
      return fail(MOE_ERR_INVALID_ARG, "x_dtype = %d", x_dtype);
    if (H < 1 || (H * (x_dtype == MOE_DTYPE_BF16 ? 2 : 4)) % 16 != 0)
      return fail(MOE_ERR_UNSUPPORTED, "row of H = %d elements is not a multiple of 16 B", H);
    if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Xperm)) & 15u)
      return fail(MOE_ERR_INVALID_ARG, "X and Xperm must be 16-byte aligned");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* scratch = nullptr;
  cudaError_t e;
  if ((e = static_scratch(&scratch)) != cudaSuccess)
    return cuda_fail(e, "static scratch address lookup");
  if (T == 0) {
    if ((e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s)) != cudaSuccess ||
        (e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync");
    return ok();
  }
  const int nchunks = (T + kDispatchChunk - 1) / kDispatchChunk;
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
  // every entry of both tables is written by count / scan before it is read, so the
  // previous call's contents need no clearing
  a.chunk_counts = scratch;
  a.chunk_base = scratch + (size_t)nchunks * E;
  a.status = nullptr;
  if ((e = launch_dispatch_count(a, s)) != cudaSuccess) return cuda_fail(e, "dispatch_count launch");
  if ((e = launch_dispatch_scan(a, s)) != cudaSuccess) return cuda_fail(e, "dispatch_scan launch");
  if ((e = launch_dispatch_scatter(a, s)) != cudaSuccess)
    return cuda_fail(e, "dispatch_scatter launch");
  if (Xperm && (e = launch_dispatch_gather(a, s)) != cudaSuccess)
    return cuda_fail(e, "dispatch_gather launch");
  return ok();
}

