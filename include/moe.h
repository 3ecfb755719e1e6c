/*
 * moe.h - C ABI of libmoe.so: the forward of one sparse top-k routed Mixture-of-Experts
 * layer on one NVIDIA B300 (sm_103a).
 *
 * The five compute calls follow the six-step forward of "LLM Internals §14.2.1 (one MoE
 * forward: six steps and shapes)":
 *   step 1  input X[T, H]                                   (caller's buffer)
 *   step 2  router scoring X x W_g -> s[T, E]                moe_router_topk
 *   step 3  top-k per row and normalisation among the k     moe_router_topk
 *   step 4  dispatch permutation grouping rows by expert     moe_dispatch
 *   step 5  grouped GEMM per expert over variable m_i        moe_grouped_swiglu
 *   step 6  gate-weighted combine through the inverse
 *           permutation, plus the shared expert              moe_combine
 * and the monitoring signals of §14.2.3 (balance loss, per-expert load, drop rate,
 * routing entropy) with the load CV of "AI Knowledge Map - MoE": moe_balance_stats.
 *
 * Conventions for every call
 *  - Pointers are DEVICE pointers unless stated.  The caller owns every buffer.  The
 *    library allocates no device memory: scratch lives in a caller-provided workspace
 *    of moe_workspace_bytes() bytes whose first 256 bytes hold a device status word
 *    (int32 at byte 0) and must be zeroed once (moe_workspace_init) before first use.
 *    The int32 at byte 4 counts the rows the last moe_router_topk call (the experts the
 *    last moe_expert_choice call) re-decided from exact dot products (a diagnostic).
 *  - Every call is asynchronous on `stream`, performs no host synchronisation (except
 *    moe_get_device_status and moe_ctx_trace_read, which say so) and returns an int
 *    status: MOE_OK (0) or a negative MOE_ERR_*.  Argument checks run before anything is
 *    enqueued; a failed check enqueues nothing.  No C++ exception crosses the ABI.
 *  - Device-side failures (a bounded wait that timed out, an index out of range) are
 *    recorded in the workspace status word (first error wins) and read back with
 *    moe_get_device_status.  Kernels never trap.
 *  - Layouts are row-major.  Expert weights are stored output-major (the transpose of
 *    the [H, I] orientation in which §14.2.1 writes the product) so that both operands
 *    of every expert GEMM are contiguous along their reduction axis:
 *      W_gate, W_up : [E][I][H]     W_down : [E][H][I]
 *      Ws_gate, Ws_up : [I][H]      Ws_down : [H][I]      (shared expert)
 *  - Supported: 1 <= k <= min(E, 32), 1 <= E <= 512, T >= 0.  bf16 experts need
 *    H % 64 == 0 and I % 64 == 0; fp32 experts need H % 4 == 0 and I % 4 == 0.
 *    All pointers 16-byte aligned.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* moe_stream_t;

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer, small ws   */
  MOE_ERR_UNSUPPORTED = -2, /* valid request outside what the kernels implement      */
  MOE_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed                      */
  MOE_ERR_TIMEOUT = -4,     /* device: a bounded wait gave up                         */
  MOE_ERR_DEVICE_INDEX = -5 /* device: an index read from memory was out of range     */
};

enum moe_score { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum moe_dtype { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 };

typedef struct moe_ctx moe_ctx;

/* Shape and policy of the router (steps 2-3). */
typedef struct {
  int T, H, E, k;
  int score;   /* MOE_SCORE_SOFTMAX: key = logit, gate from softmax(l) ("AI Knowledge
                  Map - MoE", router steps 1-4).  MOE_SCORE_SIGMOID: s = sigmoid(l) per
                  cell (§14.2.1 step 2), key = s + bias (§14.2.3 eq. 16). */
  int renorm;  /* 1: gates renormalised over the k chosen (sum to 1); 0: raw softmax
                  probability / raw affinity. */
  int x_dtype; /* dtype of X: MOE_DTYPE_BF16 or MOE_DTYPE_F32 */
  int n_groups;    /* group-limited routing ("LLM Internals §14.2.3", node-limited routing;
                      "MoE 03: efficiency frontiers", DeepSeek's hardware-aware design):
                      the E experts form n_groups groups of E / n_groups consecutive
                      indices (the experts of one node).  0 or 1: off. */
  int topk_groups; /* groups a token may use: its topk_groups best groups by the sum of
                      their k / topk_groups largest unbiased affinities (sigmoid s, or the
                      softmax probability; ties to the lower group); the k experts are then
                      the top k keys among those groups' experts.  Needs n_groups <= 32
                      dividing E, 1 <= topk_groups <= n_groups, k a multiple of topk_groups
                      and k / topk_groups <= E / n_groups.  topk_groups == n_groups is plain
                      top-k. */
} moe_router_desc;

/* Shape of the expert stage (step 5). */
typedef struct {
  int T, H, E, I, k;
  int dtype;      /* dtype of X / Xperm and all expert weights */
  int has_shared; /* 1: one always-on shared expert of width I (§14.2.4) */
} moe_expert_desc;

/* ------------------------------------------------------------------ context */

/* Create a context bound to CUDA device `device` (reads its SM count, resolves the
 * tensor-map encoder of the driver).  *out is owned by the caller; free it with
 * moe_ctx_destroy.  Returns MOE_ERR_CUDA if the device cannot be queried. */
int moe_ctx_create(moe_ctx** out, int device);
void moe_ctx_destroy(moe_ctx* ctx);

/* Bytes of workspace the calls of one forward of this shape need (all five calls share
 * one workspace).  Host-only; never fails (returns 0 for negative sizes). */
size_t moe_workspace_bytes(int T, int H, int E, int I, int k, int dtype, int has_shared);

/* Zero the workspace header (status word) on `stream`. */
int moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Expert capacity C = ceil(c * T * k / E) ("AI Knowledge Map - MoE", capacity formula;
 * the GShard form of §14.2.3), evaluated exactly on the binary value of c.  Host-only.
 * Returns C >= 0, or MOE_ERR_INVALID_ARG for c < 0, non-finite c, T < 0, k < 1, E < 1 or
 * a result above INT32_MAX. */
int moe_capacity(double c, int T, int k, int E);

/* ------------------------------------------------------------------ steps 2-3 */

/* Router scoring, top-k and gates for all T tokens.
 *   X          [T, H] bf16 or fp32 (d->x_dtype)
 *   Wg         [H, E] fp32 router weight
 *   bias       [E] fp32 selection-only bias (sigmoid scoring; nullable = 0)
 *   logit_bias [E] fp32 offset added to every logit before scoring (nullable = 0)
 *   topk_idx   [T, k] int32 out: the k chosen experts of each token, ascending index
 *   topk_gate  [T, k] fp32 out: their gate weights, same order
 *   key_gap    [T] fp32 out (nullable): key_(k) - key_(k+1) of the row (+inf if k == E);
 *              group-limited: the smaller of the group margin S_(M) - S_(M+1) and the
 *              key margin among the allowed experts
 *   prob_colsum[E] fp64 out (nullable): sum over tokens of p[t, e] (softmax row, or the
 *              sigmoid affinities normalised over the row); zeroed by the call
 * Selection is exact: the logits are fp32 (bf16 X with E % 8 == 0, H % 64 == 0 and
 * T >= 256: tensor cores over exact bf16 pieces of W_g, accumulation chains of at most
 * 3072 products; otherwise CUDA-core fp32 with 32-term blocks and compensated
 * accumulation), and any row whose k-th/(k+1)-th margin (or group margin) falls inside
 * their error bound is re-decided from dot products carried to ~48 significant bits
 * (error-free products, double-fp32 sums).  Ties go to the lower expert index.
 * Returns MOE_ERR_UNSUPPORTED for n_groups > 32 or not dividing E, MOE_ERR_INVALID_ARG for
 * the other group-shape violations. */
int moe_router_topk(moe_ctx* ctx, const moe_router_desc* d, const void* X,
                    const float* Wg, const float* bias, const float* logit_bias,
                    int32_t* topk_idx, float* topk_gate, float* key_gap,
                    double* prob_colsum, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Expert-choice routing ("LLM Internals §14.2", the two selection paradigms: expert-
 * choice; "MoE 03: efficiency frontiers", Expert Choice Routing).  Instead of every token
 * choosing k experts, every expert takes the C = T*k/E tokens of the batch with the
 * largest affinity S[t, e]: the softmax probability over the experts (MOE_SCORE_SOFTMAX)
 * or the sigmoid s (MOE_SCORE_SIGMOID).  Ties go to the lower token index.  Every expert
 * carries exactly C rows and nothing is dropped, but a token may be taken by several
 * experts or by none.  Slots are (token, expert) pairs s = t*E + e, so steps 5-6 run
 * unchanged with E slots per token:
 *   offsets     [E+1] int32 out: e*C
 *   row_of_slot [T*E] int32 out: permuted row of slot t*E+e, -1 if e did not take t
 *   slot_of_row [T*k] int32 out: the slot of each row (rows by expert, then token)
 *   slot_gate   [T*E] fp32 out: S[t, e] where e took t, 0 elsewhere (moe_combine's gate)
 *   col_gap     [E] fp32 out (nullable): S_(C) - S_(C+1) down each expert's column
 *               (+inf if C is 0 or T)
 * d: T <= 32768, H, E, k (the average experts per token; E must divide T*k), score,
 * x_dtype.  renorm does not apply and there is no selection bias: a per-expert bias shifts
 * a whole column and changes no choice.  n_groups must be 0 or 1.  Exactness as for
 * moe_router_topk: a column whose C-th/(C+1)-th margin lies inside the error bound of its
 * fp32 affinities is re-decided from the exact affinities of its band tokens.
 * Then moe_gather_rows (R = T*k, k = E), moe_grouped_swiglu (k) and moe_combine (k = E,
 * row_of_slot, slot_gate). */
int moe_expert_choice(moe_ctx* ctx, const moe_router_desc* d, const void* X,
                      const float* Wg, const float* logit_bias, int32_t* offsets,
                      int32_t* row_of_slot, int32_t* slot_of_row, float* slot_gate,
                      float* col_gap, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Xperm[r] = X[slot_of_row[r] / k] for r < R: the row gather of a slot layout in which a
 * token may fill any number of rows (expert-choice routing, k = E).  X has T rows; a slot
 * outside [0, T*k) is recorded in the workspace status word (MOE_ERR_DEVICE_INDEX) and
 * its row left untouched.  The row size H * element size must be a multiple of 16 B. */
int moe_gather_rows(moe_ctx* ctx, int R, int k, int H, int x_dtype,
                    const int32_t* slot_of_row, const void* X, int T, void* Xperm, void* ws,
                    moe_stream_t stream);

/* ------------------------------------------------------------------ step 4 */

/* Group the T*k (token, choice) slots by expert (§14.2.1 step 4) under an optional
 * capacity ("AI Knowledge Map - MoE": overflow beyond C is dropped; the lowest token
 * indices of an expert are kept).
 *   capacity   < 0: dropless; >= 0: C (see moe_capacity)
 *   topk_idx   [T, k] int32 from moe_router_topk
 *   counts     [E] int32 out: m_e, slots routed to e BEFORE capacity
 *   offsets    [E+1] int32 out: first permuted row of each expert AFTER capacity;
 *              offsets[E] = R, the kept slot count
 *   row_of_slot[T*k] int32 out: permuted row of slot t*k+j, or -1 if dropped
 *   slot_of_row[T*k] int32 out: rows [0, R) hold the inverse; rows >= R untouched
 *   H          hidden size, >= 1 even without a gather (it sizes the workspace layout)
 *   X, Xperm   nullable pair: when both are given, Xperm[row] = X[slot / k] for every
 *              kept row (x_dtype element type, Xperm has T*k rows)
 * Rows are ordered by (expert ascending, token ascending).  The k experts of a token must
 * be distinct (moe_router_topk's always are): an index outside [0, E) or repeated within a
 * row is recorded in the workspace status word (MOE_ERR_DEVICE_INDEX), and the rows of
 * that expert are then unspecified (never out of bounds). */
int moe_dispatch(moe_ctx* ctx, int T, int k, int E, int H, int x_dtype, int capacity,
                 const int32_t* topk_idx, const void* X, int32_t* counts,
                 int32_t* offsets, int32_t* row_of_slot, int32_t* slot_of_row,
                 void* Xperm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Allocation-free dispatch.  The paper has no counterpart to this call.  It is for callers
 * that may not allocate device memory at the moment they dispatch: an inference engine or
 * host runtime that owns all device memory and hands out only the buffers it planned, or
 * a process whose allocator must never grow (cudaMalloc can also synchronise the device,
 * which a latency-bound decode loop cannot afford).  It does what moe_dispatch does, with
 * the same arguments minus the context and the workspace: its scratch (the per-chunk count
 * and base tables) is a file-scope static device array of 1 MiB that every GPU which loads
 * the library keeps until the process exits.
 *  - T may be at most 65536; larger T returns MOE_ERR_UNSUPPORTED and enqueues nothing.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - The first call on a device looks up the array's device address (once per device,
 *    with that device current) and caches it for the life of the process; make that first
 *    call before any stream capture begins.  The cache is keyed on the CURRENT device:
 *    `stream` must belong to it.  After a cudaDeviceReset (or anything else that destroys
 *    the device's primary context) the cached address is stale: do not call this entry
 *    point on that device again in the same process.
 *  - Every call shares the one array: calls whose work overlaps on the GPU (different
 *    streams, or different host threads on one device) race and corrupt each other; the
 *    array keeps the last call's contents, and each call rewrites every entry it reads.
 *  - Out-of-range or repeated expert indices are not reported (there is no workspace
 *    status word): out-of-range slots get -1, and a repeated expert's rows are
 *    unspecified (never out of bounds).
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA, with the reason
 * in moe_last_error_detail(). */
int moe_dispatch_static(int T, int k, int E, int H, int x_dtype, int capacity,
                        const int32_t* topk_idx, const void* X, int32_t* counts,
                        int32_t* offsets, int32_t* row_of_slot, int32_t* slot_of_row,
                        void* Xperm, moe_stream_t stream);

/* ------------------------------------------------------------------ step 5 */

/* Per-expert SwiGLU FFN over the permuted rows (§14.2.1 step 5, §14.2.2 three
 * matrices): for the rows [offsets[e], offsets[e+1]) of expert e,
 *   h = SiLU(x W_gate[e]^T) * (x W_up[e]^T),   o = h W_down[e]^T,
 * and for the shared expert (has_shared) the same over all T rows of X.
 *   X        [T, H]   (read only for the shared expert; nullable when has_shared = 0)
 *   Xperm    [T*k, H] permuted rows from moe_dispatch
 *   offsets  [E+1]    from moe_dispatch (read on the device; no host sync)
 *   O        [T*k, H] fp32 out: o of each kept row; rows >= R untouched
 *   O_shared [T, H]   fp32 out (has_shared): the shared expert's output
 * bf16: tcgen05 tensor cores, fp32 accumulation, h rounded to bf16.  fp32: CUDA-core
 * fp32 FMA throughout. */
int moe_grouped_swiglu(moe_ctx* ctx, const moe_expert_desc* d, const void* X,
                       const void* Xperm, const int32_t* offsets, const void* W_gate,
                       const void* W_up, const void* W_down, const void* Ws_gate,
                       const void* Ws_up, const void* Ws_down, float* O, float* O_shared,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* FP8 expert weights ("LLM Internals §14.2.5": one expert's three matrices are 44 MB in
 * FP8, and decode-sized batches read every touched expert's weights for a few rows).
 * The pages fix one byte per weight and no scale convention; this library stores E4M3
 * codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448)
 * with one fp32 scale per output channel (row of the output-major weight):
 *   scale[r] = amax_r / 448 (1 for an all-zero row), q[r][c] = E4M3(W[r][c] / scale[r]),
 * both divisions correctly rounded in fp32, the code rounded to nearest even and
 * saturated at 448.  The dequantized weight is scale[r] * value(q[r][c]).
 *
 * moe_quantize_fp8: W [rows, cols] (bf16 or fp32, w_dtype; cols even) -> q [rows, cols]
 * uint8 codes and scale [rows] fp32, all device memory.  For the expert weights call it
 * on W_gate / W_up as [E*I, H] and W_down as [E*H, I]. */
int moe_quantize_fp8(moe_ctx* ctx, int rows, int cols, int w_dtype, const void* W,
                     uint8_t* q, float* scale, moe_stream_t stream);

/* Step 5 with FP8 expert weights: as moe_grouped_swiglu (same X, Xperm, offsets, O,
 * O_shared, workspace and h rounding), the weights given as codes and scales:
 *   Q_gate, Q_up [E][I][H], S_gate, S_up [E][I]; Q_down [E][H][I], S_down [E][H];
 *   Qs_* / Ss_* the shared expert's ([I][H], [I]; [H][I], [H]; nullable without it).
 * h = SiLU(s_g (x . q_g)) * (s_u (x . q_u)), o = s_d (h . q_d): the codes decode exactly
 * and every dot product accumulates in fp32 on CUDA cores, a GEMV per weight row for up
 * to 8 rows of an expert at a time - the form of decode-sized batches (a few rows per
 * expert), where the step streams the touched weights once.  Needs bf16 activations and
 * H % 64 == 0, I % 64 == 0. */
int moe_grouped_swiglu_fp8(moe_ctx* ctx, const moe_expert_desc* d, const void* X,
                           const void* Xperm, const int32_t* offsets, const uint8_t* Q_gate,
                           const float* S_gate, const uint8_t* Q_up, const float* S_up,
                           const uint8_t* Q_down, const float* S_down, const uint8_t* Qs_gate,
                           const float* Ss_gate, const uint8_t* Qs_up, const float* Ss_up,
                           const uint8_t* Qs_down, const float* Ss_down, float* O,
                           float* O_shared, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------ step 6 */

/* Y[t] = sum over kept j of topk_gate[t, j] * O[row_of_slot[t*k+j]]  (+ O_shared[t])
 * (§14.2.1 step 6; "AI Knowledge Map - MoE" final weighted sum).  A dropped slot adds
 * nothing and the remaining gates are not renormalised.
 *   O_shared nullable; Y [T, H] fp32 out; Y_bf16 [T, H] nullable bf16 copy of Y.
 *   k: slots per token, at most 512 (E for expert-choice routing). */
int moe_combine(moe_ctx* ctx, int T, int k, int H, const float* O, const float* O_shared,
                const int32_t* row_of_slot, const float* topk_gate, float* Y,
                void* Y_bf16, moe_stream_t stream);

/* ------------------------------------------------------------------ balance signals */

/* Load-balance statistics of one routed batch (§14.2.3 balance loss and monitoring;
 * "AI Knowledge Map - MoE" load CV):
 *   f[e] = counts[e] / (T k)   (router choices before capacity; sums to 1)
 *   p[e] = prob_colsum[e] / T
 *   out[0] = alpha * E * sum_e f[e] p[e]        (Switch balance loss)
 *   out[1] = (T k - offsets[E]) / (T k)        (drop rate; 0 when offsets is null)
 *   out[2] = std(counts) / mean(counts)         (population std; load CV)
 *   out[3] = -sum_e f[e] ln f[e]                (routing entropy)
 * f, p: [E] fp64 out; out: [4] fp64 out.  With T == 0 everything is 0. */
int moe_balance_stats(moe_ctx* ctx, int T, int k, int E, const int32_t* counts,
                      const int32_t* offsets, const double* prob_colsum, double alpha,
                      double* f, double* p, double* out, moe_stream_t stream);

/* Auxiliary-loss-free balancing step ("LLM Internals §14.2.3", bias-adjusted selection):
 * after a batch, every expert whose load is above the balanced load loses gamma from its
 * selection bias and every expert below it gains gamma; the page gives gamma = 0.001 for
 * most of training and 0 at the end.  Load = counts[e] from moe_dispatch (router choices
 * before capacity); balanced load = T k / E, compared exactly (E counts[e] against T k);
 * an expert exactly at it keeps its bias.  Each updated entry is one float32 addition.
 *   counts [E] int32 (device), bias [E] fp32 (device, updated in place).
 * Returns MOE_ERR_INVALID_ARG for a null pointer or a non-finite gamma. */
int moe_bias_update(moe_ctx* ctx, int T, int k, int E, const int32_t* counts, float gamma,
                    float* bias, moe_stream_t stream);

/* ------------------------------------------------------------------ diagnostics */

/* Synchronise `stream`, copy the workspace status word into *status (host pointer) and,
 * if reset != 0, zero it.  Returns MOE_ERR_CUDA if the copy fails. */
int moe_get_device_status(moe_ctx* ctx, void* ws, int* status, int reset,
                          moe_stream_t stream);

/* Kernel timing.  With tracing on, every kernel a call launches is bracketed by CUDA
 * events recorded on that call's stream.  moe_ctx_trace_read synchronises those events
 * and writes, per kernel id, the number of kernel launches (the router's tensor-core
 * logits are two kernels, W_g split and GEMM; split-K router logits add a reduce kernel
 * to router_select) and their summed milliseconds
 * (host arrays of n entries, n >= MOE_KERNEL_COUNT), then clears the record. */
enum moe_kernel_id {
  MOE_K_ROUTER_LOGITS = 0,
  MOE_K_ROUTER_SELECT,
  MOE_K_DISPATCH_COUNT,
  MOE_K_DISPATCH_SCAN,
  MOE_K_DISPATCH_SCATTER,
  MOE_K_DISPATCH_GATHER,
  MOE_K_EXPERT_GATE_UP,
  MOE_K_EXPERT_DOWN,
  MOE_K_COMBINE,
  MOE_K_BALANCE_STATS,
  MOE_K_BIAS_UPDATE,
  MOE_KERNEL_COUNT
};
int moe_ctx_set_tracing(moe_ctx* ctx, int enable);
int moe_ctx_trace_read(moe_ctx* ctx, int* launches, double* total_ms, int n);
const char* moe_kernel_name(int id);

/* Failure-detection test hook (not for production use).  hook = MOE_TEST_HOOK_NONE
 * restores normal operation.  MOE_TEST_HOOK_WITHHOLD_LOAD makes the tensor-core expert
 * kernel skip the first operand load of each CTA, a barrier that nothing completes: the
 * bounded waits run out after wait_limit_ms (0 keeps the default 2000 ms), the kernel
 * records MOE_ERR_TIMEOUT in the workspace status word, frees its tensor memory and
 * returns, and the context stays usable.  Nothing faults, traps or hangs. */
enum moe_test_hook { MOE_TEST_HOOK_NONE = 0, MOE_TEST_HOOK_WITHHOLD_LOAD = 1 };
int moe_ctx_set_test_hook(moe_ctx* ctx, int hook, int wait_limit_ms);

const char* moe_status_string(int status);
/* Text describing why the last call made by this thread failed ("" after a success).
 * Host-only; the pointer stays valid until this thread's next call. */
const char* moe_last_error_detail(void);
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
