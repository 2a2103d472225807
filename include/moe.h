/*
 * moe.h -- C ABI of libmoe.so, the DeepSeekMoE layer forward for one B300
 * (sm_103a).
 *
 * The layer, as the deepseek-v3-jax pages describe it:
 *   "190行JAX复刻DeepSeek V3" (openai-hub.com), section "190行代码到底装进了什么":
 *     routed experts of which each token selects the top k, plus one shared
 *     expert that every token always passes through;
 *   same page, section "最有价值的实验:无辅助损失均衡真的有效":
 *     auxiliary-loss-free balancing -- after each step an over-loaded
 *     expert's bias is lowered and an idle expert's bias raised, speed
 *     gamma = 1e-3; the bias decides which experts are selected and never
 *     changes the gate value of a selected expert;
 *   "DeepSeek V3 viết lại bằng 190 dòng JAX thuần" (lehuy.net), section
 *     "Những gì đã được đơn giản hóa": the pages' code runs every expert on
 *     every token and zeroes the unselected ones, with no sparse dispatch.
 *     This library is truly sparse: each token reaches only its k experts.
 *
 * Per token t (x[t] a row of d numbers), with E routed experts:
 *   u[t,e]  = x[t] . W_r[e]                (fp32 accumulation)
 *   s[t,e]  = 1 / (1 + exp(-u[t,e]))       (sigmoid affinity)
 *   idx[t]  = the k experts with the largest s[t,e] + b[e], ordered by that
 *             biased score, descending; equal scores go to the lower index;
 *             a NaN score ranks below every number
 *   g[t,j]  = s[t,idx[t,j]] / sum_j' s[t,idx[t,j']]   (unbiased affinities)
 *   y[t]    = S(x[t]) + sum_j g[t,j] * R_{idx[t,j]}(x[t])
 *   where every expert is SwiGLU: F(x) = W_down (silu(W_gate x) * (W_up x)),
 *   silu(z) = z / (1 + exp(-z)).
 *   load[e] = #{(t,j) : idx[t,j] = e}
 * and, called separately after a step,
 *   b[e]   -= gamma * sgn(load[e] - T*k/E)     (sgn(0) = 0, fp32 result)
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *     and contiguous, 16-byte aligned.  The library allocates no device
 *     memory: all scratch comes from the caller's workspace.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously; nothing synchronises the host.
 *   - Return value: MOE_OK (0) once the work is enqueued, or a negative
 *     MOE_ERR_* code.  Argument errors are found on the host before anything
 *     is launched (nothing is written).  Errors that only the device can see
 *     (a pipeline wait that ran out of time) set a device error word which
 *     moe_last_error() returns after the caller has synchronised.
 *   - Thread safety: calls on different streams may run concurrently if they
 *     use different workspaces and outputs.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

/* Only the functions declared here are exported from libmoe.so. */
#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of x, y and the expert weights.  The router weights, the
 * bias, the gates and the load counts are always fp32 / int32. */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

enum {
  MOE_OK = 0,
  MOE_ERR_NULL = -1,           /* a required pointer is NULL */
  MOE_ERR_SHAPE = -2,          /* sizes out of range (see moe_desc) */
  MOE_ERR_ALIGN = -3,          /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = -4,      /* ws_bytes < moe_workspace_size(desc) */
  MOE_ERR_DTYPE = -5,          /* unknown dtype, or flags that the dtype does not support */
  MOE_ERR_LAUNCH = -6,         /* a kernel launch failed (cudaGetLastError) */
  MOE_ERR_DEVICE_TIMEOUT = -7, /* device-side wait ran out of time (moe_last_error) */
  MOE_ERR_DEVICE = -8,         /* no usable sm_103 device, or a CUDA runtime call failed */
};

/* Flags. */
#define MOE_ROUTE_ONLY   1u  /* router + load counts only: no dispatch, experts or
                                combine; y and the expert weights may be NULL */
#define MOE_SIMT_EXPERTS 2u  /* bf16 only: run the expert GEMMs on the CUDA-core
                                kernels instead of the tensor cores (a cross-check
                                of the tensor-core path; slow) */
#define MOE_TRAINING     4u  /* bf16 tensor-core path only: the workspace also holds
                                the backward's buffers, so that moe_backward can
                                follow moe_forward on it */
#define MOE_FP8_GATE_UP  8u  /* bf16 tensor-core path only, not with MOE_TRAINING:
                                the gate/up products run on e4m3 codes with one
                                fp32 scale per row (moe_quantize_rows_e4m3).
                                w_gate and w_up of experts and shared then point at
                                packed quantized matrices; w_down stays bf16; the
                                tokens are quantized per row inside the call */
/* (flag 16 is not used) */
#define MOE_GRAD_BF16   64u  /* with MOE_TRAINING: moe_backward writes the expert
                                weight gradients (d_gate, d_up, d_down of experts
                                and shared) in bf16 -- fp32 sums rounded once --
                                instead of fp32, half the bytes; the router
                                gradient stays fp32 */
#define MOE_FP8_BLOCK   32u  /* bf16 tensor-core path only, not with MOE_TRAINING or
                                MOE_FP8_GATE_UP: both expert products on
                                block-scaled e4m3 codes (moe_quantize_blocks_e4m3);
                                w_gate, w_up and w_down of experts and shared point
                                at packed block-quantized matrices; the tokens and
                                the hidden rows are quantized inside the call */

/* Problem description.
 *   T  tokens (>= 0)            d  model width          h  expert hidden width
 *   E  routed experts (1..1024) k  experts per token (1..min(E, 32))
 * Both dtypes need d and h to be multiples of 64; the bf16 tensor-core path
 * needs multiples of 128.  T*k*max(d,h) and (T*k+T)*max(d,h) must stay below
 * 2^31. */
typedef struct {
  int T, d, h, E, k;
  int dtype;        /* moe_dtype */
  unsigned flags;   /* MOE_ROUTE_ONLY | MOE_SIMT_EXPERTS | MOE_TRAINING |
                       MOE_FP8_GATE_UP | MOE_FP8_BLOCK | MOE_GRAD_BF16 */
} moe_desc;

/* Expert weights, element type desc->dtype.
 * Routed experts: w_gate [E, h, d], w_up [E, h, d], w_down [E, d, h].
 * Shared expert : w_gate [h, d],    w_up [h, d],    w_down [d, h].
 * (Each matrix is stored output-major: row i holds the weights of output i.)
 * With MOE_FP8_GATE_UP (w_gate, w_up) those pointers instead hold the packed
 * per-row e4m3 form of the same matrices, written by moe_quantize_rows_e4m3;
 * with MOE_FP8_BLOCK (all three) the packed block-scaled form written by
 * moe_quantize_blocks_e4m3 (layouts below). */
typedef struct {
  const void *w_gate, *w_up, *w_down;
} moe_expert_w;

/* FP8 gate/up weights with per-row scales.  The official V3 model computes
 * its expert products in FP8 ("DeepSeek V3 viết lại bằng 190 dòng JAX thuần",
 * section "Những gì đã được đơn giản hóa": the re-creation leaves FP8
 * training out), and so does the default path here.  With MOE_FP8_GATE_UP the
 * first expert GEMM multiplies e4m3 codes (tcgen05 kind::f8f6f4, fp32
 * accumulation) and applies the two rows' scales to each product before
 * SwiGLU.  Scaling unit: one row (a weight row, a token), with
 *   scale = amax(|row|) / 448 (1 for an all-zero row or a row with a NaN:
 *           the NaN stays in its own code and still makes that token's
 *           output NaN),
 *   code  = e4m3(row / scale), nearest-even, saturating at +-448,
 * both fp32 operations.
 *
 * Packed layout of a quantized [rows, cols] matrix, one device buffer of
 * moe_e4m3_packed_bytes(rows, cols) bytes:
 *   codes  [rows, cols] uint8 (e4m3 bit patterns) at byte 0,
 *   scales [rows]       fp32 at byte ceil(rows*cols / 256) * 256.
 * The routed gate (or up) weights are one matrix of E*h rows; the shared
 * expert's h rows. */
MOE_API size_t moe_e4m3_packed_bytes(long long rows, int cols);

/* Quantize a bf16 matrix a [rows, cols] (device, row-major, 16-byte aligned)
 * into `packed` (device, moe_e4m3_packed_bytes(rows, cols) bytes, 16-byte
 * aligned), enqueued on `stream`.  cols: a positive multiple of 8; rows >= 0.
 * MOE_ERR_NULL / MOE_ERR_SHAPE / MOE_ERR_ALIGN / MOE_ERR_DEVICE /
 * MOE_ERR_LAUNCH as for moe_forward.  The buffers must not overlap. */
MOE_API int moe_quantize_rows_e4m3(const void* a, long long rows, int cols, void* packed,
                                   void* stream);

/* Block-scaled FP8 experts (MOE_FP8_BLOCK): the official model's FP8 tile
 * granularity ("DeepSeek V3 viết lại bằng 190 dòng JAX thuần", section
 * "Những gì đã được đơn giản hóa": the re-creation leaves FP8 training out;
 * the pages give no scheme, so the granularity is a reading of this
 * library), on the B300's block-scaled MMA (tcgen05 kind::mxf8f6f4, fp32
 * accumulation).  Each expert weight matrix is cut into 128 x 128 blocks
 * (128 output rows x 128 inputs), each activation row -- a token for
 * gate/up, the hidden row of a (token, expert) pair for the down projection
 * -- into 1 x 128 blocks.  A block with largest magnitude amax gets the scale
 * 2^e, e the smallest integer with amax <= 448 * 2^e (0 for a block of zeros
 * or one whose maximum is not finite, clamped to [-127, 127]), and its codes
 * are e4m3(v / 2^e), nearest-even (NaN stays NaN, +-inf saturates to +-448).
 * The hidden rows are quantized from their fp32 values inside the first
 * expert GEMM; nothing rounds them to bf16 first.
 *
 * Packed layout of a block-quantized [rows, cols] matrix (rows and cols
 * multiples of 128), one device buffer of moe_e4m3_block_packed_bytes(rows,
 * cols) bytes:
 *   codes [rows, cols] uint8 (e4m3 bit patterns) at byte 0,
 *   exponent words [rows / 128][ceil(cols / 512)] uint32 at byte
 *   ceil(rows*cols / 256) * 256; byte j of word w of a block row holds e + 127
 *   of block 4 w + j along the row.
 * The routed gate (or up) weights are one matrix of E*h rows, the routed down
 * weights one of E*d rows; the shared expert's h (gate, up) or d (down) rows.
 * moe_e4m3_block_packed_bytes returns 0 for sizes that are not multiples of
 * 128. */
MOE_API size_t moe_e4m3_block_packed_bytes(long long rows, int cols);

/* Block-quantize a bf16 matrix a [rows, cols] (device, row-major, 16-byte
 * aligned) into `packed` (device, moe_e4m3_block_packed_bytes(rows, cols)
 * bytes, 16-byte aligned), enqueued on `stream`.  rows and cols: multiples of
 * 128 (rows / 128 <= 65535).  MOE_ERR_NULL / MOE_ERR_SHAPE / MOE_ERR_ALIGN /
 * MOE_ERR_DEVICE / MOE_ERR_LAUNCH as for moe_forward.  The buffers must not
 * overlap. */
MOE_API int moe_quantize_blocks_e4m3(const void* a, long long rows, int cols, void* packed,
                                     void* stream);

/* Bytes of device workspace that moe_forward needs for `desc` (flags
 * included).  Returns 0 for an invalid desc.  The value depends only on the
 * desc, so one buffer can be reused for every call with the same desc. */
MOE_API size_t moe_workspace_size(const moe_desc* desc);

/* One forward pass of the MoE layer.
 *   x          [T, d]   dtype         tokens (already normalised; the layer
 *                                     output excludes any residual)
 *   w_router   [E, d]   fp32          router weights W_r
 *   bias       [E]      fp32          selection bias b (read only here)
 *   experts, shared                   see moe_expert_w (may be NULL with
 *                                     MOE_ROUTE_ONLY)
 *   y          [T, d]   dtype   out   layer output (NULL allowed with
 *                                     MOE_ROUTE_ONLY)
 *   topk_idx   [T, k]   int32   out   selected experts, slot order as above
 *   gates      [T, k]   fp32    out   gate values g
 *   load_counts[E]      int32   out   tokens routed to each expert
 *   workspace  device buffer of ws_bytes >= moe_workspace_size(desc)
 * The bias is not updated here: call moe_bias_update after the step. */
MOE_API int moe_forward(const moe_desc* desc, const void* x, const float* w_router,
                const float* bias, const moe_expert_w* experts,
                const moe_expert_w* shared, void* y, int32_t* topk_idx,
                float* gates, int32_t* load_counts, void* workspace,
                size_t ws_bytes, void* stream);

/* Same pass with x and y in HOST memory (pinned memory lets the copies run
 * asynchronously).  x is copied to the device, the layer runs, y is copied
 * back, all enqueued on `stream`; the host buffers must stay valid until the
 * stream reaches that point.  Weights, router, bias and the small outputs are
 * device pointers as in moe_forward.  The workspace must hold
 * moe_workspace_size(desc) + moe_host_io_extra_bytes(desc) bytes. */
MOE_API size_t moe_host_io_extra_bytes(const moe_desc* desc);
MOE_API int moe_forward_host_io(const moe_desc* desc, const void* x_host,
                        const float* w_router, const float* bias,
                        const moe_expert_w* experts, const moe_expert_w* shared,
                        void* y_host, int32_t* topk_idx, float* gates,
                        int32_t* load_counts, void* workspace, size_t ws_bytes,
                        void* stream);

/* moe_forward with caller-owned CUDA events recorded on `stream` between the
 * phases of the pass, for timing each phase on the device:
 *   events[0] before the router (logits + top-k)
 *   events[1] before dispatch (ranks, scan, permute/gather)
 *   events[2] before expert GEMM 1 (gate/up + SwiGLU, shared expert included)
 *   events[3] before expert GEMM 2 (down projection)
 *   events[4] before the combine (gates, slot sums)
 *   events[5] after the combine
 * `events` points to MOE_N_PHASE_EVENTS cudaEvent_t handles (created by the
 * caller, not destroyed here).  Phases that do not run (route-only, T = 0)
 * still get their events recorded, back to back. */
#define MOE_N_PHASE_EVENTS 6
MOE_API int moe_forward_profiled(const moe_desc* desc, const void* x,
                                 const float* w_router, const float* bias,
                                 const moe_expert_w* experts,
                                 const moe_expert_w* shared, void* y,
                                 int32_t* topk_idx, float* gates,
                                 int32_t* load_counts, void* workspace,
                                 size_t ws_bytes, void* stream,
                                 void* const* events);

/* Auxiliary-loss-free bias update ("190行JAX复刻DeepSeek V3", section
 * "最有价值的实验:无辅助损失均衡真的有效"):
 *   bias[e] = fp32(bias[e] - fp32(gamma) * sgn(E*load_counts[e] - TK))
 * i.e. an expert above the mean load T*k/E loses gamma, one below gains it,
 * one exactly at the mean is unchanged.  load_counts [E] int32 and bias [E]
 * fp32 are device pointers; bias is updated in place.  TK = T*k of the step
 * the counts came from. */
MOE_API int moe_bias_update(const int32_t* load_counts, float* bias, float gamma,
                    int E, int TK, void* stream);

/* Sequence-wise balance loss of the routing that the last moe_forward (or
 * moe_forward_profiled, moe_forward_host_io) on `workspace` with the same
 * `desc` computed: the small auxiliary loss the pages keep beside the bias,
 * weight alpha = 1e-4 ("DeepSeek V3 viết lại bằng 190 dòng JAX thuần",
 * section "Những gì có trong 190 dòng code"), as the original report defines
 * it, for each sequence of seq_len consecutive tokens (the last one may be
 * shorter and uses its own length S):
 *   f_e = E/(k S) * #{t in the sequence : e among its selected experts}
 *   P_e = (1/S) * sum_t s[t,e] / sum_j s[t,j]   (s = sigmoid affinities)
 *   loss[q] = alpha * sum_e f_e * P_e
 * Reads the router's partial logits left in the workspace and topk_idx
 * [T, k] (device, int32, the selection of that forward); writes
 * loss[ceil(T / seq_len)] (device fp32).  Enqueue it on the same stream after
 * that forward and before the workspace is reused.  Deterministic.  Returns
 * MOE_ERR_SHAPE for seq_len < 1, MOE_ERR_NULL / MOE_ERR_WORKSPACE for missing
 * pointers or a short workspace; T = 0 enqueues nothing. */
MOE_API int moe_seq_balance_loss(const moe_desc* desc, int seq_len, float alpha,
                                 const int32_t* topk_idx, const void* workspace,
                                 size_t ws_bytes, float* loss, void* stream);

/* Gradients of expert weights (device, fp32 -- or bf16 with MOE_GRAD_BF16,
 * the pointers then holding bf16 arrays of the same shapes -- written in
 * full: experts that no token selected get zeros).  Routed: d_gate [E, h, d],
 * d_up [E, h, d], d_down [E, d, h]; shared: the same with E = 1. */
typedef struct {
  float *d_gate, *d_up, *d_down;
} moe_expert_grad;

/* Backward of the layer ("DeepSeek V3 viết lại bằng 190 dòng JAX thuần",
 * section "Những gì có trong 190 dòng code": the re-creation trains with this
 * layer) for the output gradient dy [T, d] (bf16, device): with the forward's
 * selection held fixed (it carries no gradient) and gates g = s_sel / sum s_sel
 * over the selected sigmoid affinities,
 *   dx [T, d]            (bf16) gradient of the tokens
 *   d_experts, d_shared  (fp32) gradients of the expert weights
 *   d_router [E, d]      (fp32) gradient of W_r (through the gates only)
 * The bias gets no gradient (moe_bias_update moves it).  Call it after
 * moe_forward on the same workspace, stream, desc (with MOE_TRAINING) and
 * inputs (x, w_router, experts, shared, and that forward's topk_idx and
 * gates), before the workspace is reused.  Deterministic (no atomics in any
 * sum).  bf16 with d, h multiples of 128 only (MOE_ERR_DTYPE / MOE_ERR_SHAPE
 * otherwise); argument errors as moe_forward. */
MOE_API int moe_backward(const moe_desc* desc, const void* x, const float* w_router,
                         const moe_expert_w* experts, const moe_expert_w* shared,
                         const int32_t* topk_idx, const float* gates, const void* dy,
                         void* dx, const moe_expert_grad* d_experts,
                         const moe_expert_grad* d_shared, float* d_router, void* workspace,
                         size_t ws_bytes, void* stream);

/* Device error word of the calls made so far (MOE_OK or
 * MOE_ERR_DEVICE_TIMEOUT), and reset it to MOE_OK.  It does not synchronise
 * the caller's stream: synchronise first.  Returns MOE_ERR_DEVICE if the
 * word cannot be read. */
MOE_API int moe_last_error(void);

/* In-band SM clock record of the tensor-core kernels.  Each CTA of those
 * kernels adds, on exit, the SM clock cycles (%clock64) and the wall time
 * (%globaltimer, ns) from its start to its end into one of MOE_CLOCK_SLOTS
 * per-process counter pairs; cycles / ns is the mean SM clock (GHz) at which
 * that kernel class ran -- under the board's power cap it falls below the
 * maximum clock within tens of milliseconds of load, sooner than nvidia-smi
 * reports it.  Slots: */
#define MOE_CLOCK_GATE_UP 0 /* the forward gate/up products (expert GEMM 1) */
#define MOE_CLOCK_DOWN    1 /* the forward down products (expert GEMM 2) */
#define MOE_CLOCK_BWD     2 /* the backward's tensor-core products */
#define MOE_CLOCK_ROUTER  3 /* the tensor-core router */
#define MOE_CLOCK_SLOTS   4
/* Copies the counters to out[2 * slot] (cycles) and out[2 * slot + 1] (ns)
 * for every slot (host array of 2 * MOE_CLOCK_SLOTS values) and, if reset is
 * non-zero, zeroes them.  Synchronous with respect to the device's legacy
 * default stream: synchronise the caller's stream first.  Counting costs two
 * atomic adds per CTA and launch.  Returns MOE_ERR_NULL for out == NULL,
 * MOE_ERR_DEVICE if the counters cannot be read. */
MOE_API int moe_sm_clock_record(unsigned long long* out, int reset);

/* Self-test of the failure path.  Every wait of the library's kernels on a
 * pipeline barrier is bounded: when it runs out (4 s), the kernel sets the
 * device error word and returns, and moe_last_error then reports
 * MOE_ERR_DEVICE_TIMEOUT; the context stays usable.  This call enqueues one
 * small kernel on `stream` whose single wait, on a barrier that nothing
 * arrives on, runs out after limit_ms (1..10000) milliseconds, so a caller or
 * a test can check that path end to end: synchronise, expect
 * MOE_ERR_DEVICE_TIMEOUT from moe_last_error, then MOE_OK from the next
 * call.  No fault or trap is involved.  Returns MOE_ERR_SHAPE for limit_ms
 * out of range, MOE_ERR_DEVICE / MOE_ERR_LAUNCH as moe_forward. */
MOE_API int moe_selftest_timeout(unsigned limit_ms, void* stream);

/* The expert epilogue's silu(z) = z / (1 + e^-z) (the gate/up products'
 * SwiGLU), applied elementwise to n fp32 device values z -> out, for
 * accuracy tests of the kernel's arithmetic.  Enqueued on `stream`.  Returns
 * MOE_ERR_SHAPE for n < 0, MOE_ERR_NULL for a NULL pointer with n > 0,
 * MOE_ERR_DEVICE / MOE_ERR_LAUNCH as moe_forward. */
MOE_API int moe_selftest_silu(const float* z, float* out, int n, void* stream);

/* Static string for a MOE_* code. */
MOE_API const char* moe_error_string(int code);

/* Byte offsets of the named scratch regions inside the workspace for
 * `desc`, for tests that inspect intermediate results.  `names` receives up
 * to `cap` entries of (name, offset, bytes); returns the number of regions
 * (or a negative MOE_ERR_*).  Region names: "router_part" (fp32 partial
 * logits), "router_w3" (the router weights as three bf16 terms, for the
 * tensor-core router; empty otherwise), "blk_hist", "pair_rank", "groups"
 * (int32 group table),
 * "perm" (permuted row -> token*k+slot), "inv" (token*k+slot -> permuted row),
 * "x_perm", "h", "y_perm" (the T*k routed rows in expert order, then the
 * shared expert's T rows in token order, in the element type), "x_q"
 * (MOE_FP8_GATE_UP: the tokens
 * quantized, packed as above; MOE_FP8_BLOCK: the tokens' codes [T, d], then
 * their exponent words [ceil(d / 512)][T] from byte ceil(T*d / 256) * 256;
 * empty otherwise), "h_q" (MOE_FP8_BLOCK: the hidden rows' codes [T*k + T,
 * h] and exponent words [ceil(h / 512)][T*k + T], laid out as x_q; empty
 * otherwise; with MOE_FP8_BLOCK "h" is empty). */
typedef struct {
  char name[16];
  size_t offset, bytes;
} moe_region;
MOE_API int moe_workspace_regions(const moe_desc* desc, moe_region* regions, int cap);

/* Routing without any device allocation.  The pages have no counterpart to
 * this entry point: it exists for callers that must not allocate device
 * memory and cannot hand the library a workspace -- for example a plugin
 * whose host framework owns every byte of device memory, or a runtime with
 * a fixed memory budget that forbids allocation once it has started.
 *
 * It computes what moe_forward computes with MOE_ROUTE_ONLY (router
 * affinities, biased top-k, gates, load counts; desc->flags is ignored and
 * the route-only pass is run), with the same kernels, so its outputs are
 * identical to that call's.  Its scratch is a static device array of
 * MOE_STATIC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits; the caller passes only inputs and outputs (all device
 * pointers, as in moe_forward).
 *
 *   - A desc whose route-only scratch (moe_workspace_size of the desc with
 *     MOE_ROUTE_ONLY) exceeds MOE_STATIC_SCRATCH_BYTES is rejected with
 *     MOE_ERR_WORKSPACE before anything is launched.  32 MiB covers, e.g.,
 *     T = 8192 tokens with E = 256 experts and d = 7168.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress)
 *     with the caller's device current.  With CUDA's lazy module loading
 *     (the default) the array is reserved on a device when the library's
 *     module is first loaded there, which may be during the first call of
 *     any entry point, this one included.  A caller with a fixed memory
 *     budget should therefore make one call at start-up, before the budget
 *     is fixed and before any stream capture; later calls reserve nothing.
 *   - Every call uses the same array, which keeps the previous call's
 *     contents.  Nothing in it needs to start at zero: each call writes
 *     every scratch byte it reads before reading it.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on the
 *     array: order them on one stream or synchronise between them. */
#define MOE_STATIC_SCRATCH_BYTES (32u << 20)
MOE_API int moe_route_noalloc(const moe_desc* desc, const void* x,
                              const float* w_router, const float* bias,
                              int32_t* topk_idx, float* gates,
                              int32_t* load_counts, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
