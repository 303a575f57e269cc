/*
 * fp.h — fused input projection on one GB300 (sm_103a): the C ABI of libfp.so.
 *
 * One call computes, for an activation x read in place through its strides,
 *
 *     Y = x W + b                         (one dense GEMM, fp32 accumulation)
 *     ff = act(Y[:, :F])                  (GELU-erf / GELU-tanh / SiLU / none)
 *     q, k = rotate_half_rope(Y[:, F:F+C]), rotate_half_rope(Y[:, F+C:F+2C])
 *     v = Y[:, F+2C:F+3C]
 *
 * and writes ff token-major and q, k, v head-major [B*heads, T, head_dim].
 *
 * What each piece follows:
 *  - reading a channels-first activation (b c h w d, optionally with a time
 *    axis) as [tokens, C] with no permuted copy, and one fused ff+q+k+v weight
 *    instead of per-token GEMVs: Walrus PR #12 "Make fused_ff_qkv contiguous"
 *    (opening comment and the profiler comparison that follows it);
 *  - bias and activation fused into the GEMM epilogue (w x + b, then the
 *    activation), and a projection that writes straight into three buffers:
 *    xformers PR #283 "[perf] Fused linear" (PR description; the comment on a
 *    dedicated attention-projection kernel);
 *  - rotate-half rotary embedding on q and k with no slice/cat/neg kernels:
 *    nvFuser issue #1597 "Improve performance on RoPE" (rope_one_entry and
 *    split_qkv listings);
 *  - the [batch*heads, tokens, head_dim] output layout: memory-efficient-
 *    attention issue #7 "Improve performance via batched-matmul and fused
 *    multiplies" (the layout conversion in the opening comment).
 *
 * Conventions shared by every entry point:
 *  - All data pointers are DEVICE pointers on the current CUDA device, owned
 *    by the caller; the library keeps no reference after a call returns.
 *    fp_forward_host and fp_backward_host are the exceptions: their
 *    activation, gradient and result buffers are page-locked host memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). fp_forward only enqueues work: it never synchronises.
 *  - Argument checks run on the host before any launch; a rejected call
 *    launches nothing and returns a non-zero fp_status. fp_last_error()
 *    then gives a one-line reason (thread-local).
 *  - Errors raised on the device (a bounded wait that ran out; with
 *    FP_OPT_BOUNDS_CHECK, a store that would leave its output buffer) are
 *    recorded in a per-plan status word and reported by fp_get_device_status.
 *  - Each call is bracketed by an NVTX range named after the entry point, so
 *    it shows in Nsight timelines; without an attached tool this costs nothing.
 */
#ifndef FP_H
#define FP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP_OK = 0,
  FP_ERR_INVALID_ARG = 1,        /* null/inconsistent argument, aliasing outputs */
  FP_ERR_UNSUPPORTED_LAYOUT = 2, /* strides the selected kernel cannot address */
  FP_ERR_MISALIGNED = 3,         /* pointer or stride not 16-byte aligned */
  FP_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
  FP_ERR_OUT_OF_MEMORY = 5,      /* plan scratch could not be allocated */
  FP_ERR_TIMEOUT = 6,            /* a device-side bounded wait ran out */
  FP_ERR_DEVICE_BOUNDS = 7       /* a store was stopped by FP_OPT_BOUNDS_CHECK */
} fp_status;

typedef enum {
  FP_ACT_NONE = 0,
  FP_ACT_GELU_ERF = 1,  /* 0.5 y (1 + erf(y / sqrt 2)) */
  FP_ACT_GELU_TANH = 2, /* 0.5 y (1 + tanh(sqrt(2/pi) (y + 0.044715 y^3))) */
  FP_ACT_SILU = 3,      /* y / (1 + exp(-y)) */
  FP_ACT_RELU2 = 4      /* max(y, 0)^2, squared ReLU */
} fp_act;

typedef enum { FP_BF16 = 0, FP_F32 = 1 } fp_dtype;

#define FP_MAX_DIMS 8

/*
 * Logical shape and element strides of x. Axis `channel_dim` holds C. The
 * other axes, in order, index the tokens row-major: the first `n_batch_dims`
 * of them form the batch index b, the rest the in-sequence index t, so token
 * m = b*T + t. Rotary positions restart at every b.
 * Examples: channels-first [B, T6, C, H, W, D] -> channel_dim 2, n_batch_dims 1;
 *           row-major [B, S, C] -> channel_dim 2, n_batch_dims 1;
 *           NCHW [B, C, H, W] -> channel_dim 1, n_batch_dims 1.
 */
typedef struct {
  int32_t dtype; /* fp_dtype: the dtype of x, W, b and of every output */
  int32_t ndim;  /* 1 .. FP_MAX_DIMS */
  int64_t sizes[FP_MAX_DIMS];
  int64_t strides[FP_MAX_DIMS]; /* in elements, >= 0 */
  int32_t channel_dim;
  int32_t n_batch_dims;
} fp_layout;

typedef struct fp_plan fp_plan;

/*
 * fp_create — a projection plan for fixed sizes. Host only: touches no GPU.
 *   C          channels (> 0)
 *   ff_hidden  F, width of the ff block (>= 0)
 *   heads      attention heads (>= 0); heads * head_dim must equal C
 *   head_dim   even, and ff_hidden a multiple of it; <= 128 with rotary embedding
 *   act        activation of the ff block
 *   rope_base  > 0: rotate q and k with theta_i = pos * rope_base^(-2i/head_dim);
 *              <= 0: no rotary embedding
 * The fused weight W is [C, N] row-major with N = F + 3*heads*head_dim and
 * column blocks [ff | q | k | v]; inside a block, column = head*head_dim + j.
 * Returns FP_ERR_INVALID_ARG for inconsistent sizes; *plan is set to NULL then.
 */
fp_status fp_create(fp_plan** plan, int C, int ff_hidden, int heads, int head_dim, fp_act act,
                    float rope_base);

/*
 * fp_create_ex — fp_create with the grouped-query column order and partial
 * rotary of the split_qkv / rope_one_entry listings (nvFuser issue #1597).
 *   n_query_groups  0: as fp_create. > 0: the q|k|v part of W's columns is
 *                   [group][q_per_kv query heads | 1 key head | 1 value head]
 *                   x head_dim, q_per_kv = heads / n_query_groups;
 *                   N = F + (heads + 2*n_query_groups) * head_dim, and out_k /
 *                   out_v are [B*n_query_groups, T, head_dim] (one head per group;
 *                   the listing's expand over q_per_kv is a broadcast, not data).
 *   rope_n_elem     0: rotate the whole head. Else an even count <= head_dim:
 *                   lanes [0, rope_n_elem) rotate with theta_i = pos *
 *                   base^(-2i/rope_n_elem), pairs (i, i + rope_n_elem/2); the
 *                   other lanes pass through.
 *   k_transposed    0: out_k is [B*kv, T, head_dim] like q and v. 1: out_k is
 *                   written pre-transposed, [B*kv, head_dim, T], the layout a
 *                   q k^T product wants (memory-efficient-attention issue #7,
 *                   the comments on transposing the key once, up front).
 */
typedef struct {
  int32_t C;
  int32_t ff_hidden;
  int32_t heads;
  int32_t head_dim;
  int32_t n_query_groups;
  int32_t rope_n_elem;
  int32_t act; /* fp_act */
  float rope_base;
  int32_t k_transposed;
} fp_config;

fp_status fp_create_ex(fp_plan** plan, const fp_config* config);

/*
 * fp_forward — enqueue one fused projection on `stream`.
 *   x        device pointer to element (0, ..., 0) of the activation; layout `x_layout`
 *   W        [C, N] row-major, dtype of x
 *   b        [N] or NULL (no bias), dtype of x
 *   pos      int32 [T] rotary positions, or NULL for 0 .. T-1 (ignored without rope)
 *   out_ff   [B*T, F] row-major, or NULL when F == 0
 *   out_q, out_k, out_v   [B*heads, T, head_dim] each (k, v: [B*n_query_groups, T,
 *            head_dim] with grouped-query columns), or NULL when heads == 0
 * All pointers must be 16-byte aligned. Outputs may not overlap each other or
 * any input. bf16 activations run on the tcgen05 tensor-core kernel when x has
 * unit stride on the channel axis or on its innermost token axis, its other
 * strides are 16-byte multiples, ff_hidden and head_dim are multiples of 16 and
 * the rotated half-width is a multiple of 16 (or 1, 2, 4, 8); otherwise, and
 * for f32, the FFMA kernel runs (TF32 off; any strides).
 * Rotary table: with pos == NULL the (cos, sin) table is a constant of the
 * plan and T; it is built by the first such call and reused by later ones
 * (calls on another stream are ordered after that build with an event).
 * Caller-given positions rebuild the table on every call, so such calls on
 * different streams must be ordered by the caller.
 * Device scratch: the first call on a plan, and a call that needs more table
 * room than the plan holds, grow the plan's scratch in stream order
 * (cudaMallocAsync and cudaMemsetAsync on `stream`, at least doubling the
 * table); later calls on other streams are ordered after that growth by an
 * event, and a replaced table is freed by fp_reserve or fp_destroy. Every other
 * call allocates nothing; fp_reserve sizes the scratch up front, and must be
 * used (or one call made) before the first call inside a stream capture. Inside
 * a capture, waits on events recorded outside it become external-event nodes.
 * Returns FP_OK once the work is enqueued.
 */
fp_status fp_forward(fp_plan* plan, const void* x, const fp_layout* x_layout, const void* W,
                     const void* b, const int32_t* pos, void* out_ff, void* out_q, void* out_k,
                     void* out_v, void* stream);

/*
 * fp_forward_host — fp_forward for an activation and outputs in host memory.
 * It is the same projection, with the host <-> device copies pipelined against
 * the compute.
 *   x_host                 host pointer to x, page-locked (cudaHostAlloc or
 *                          cudaHostRegister), layout `x_layout`
 *   W, b, pos              device pointers, as fp_forward
 *   out_*_host             page-locked host pointers, shapes as fp_forward's
 *                          outputs (NULL where fp_forward takes NULL)
 * When x is dense (row-major strides over its sizes) and its first axis is a
 * batch axis (channel_dim != 0, n_batch_dims >= 1), the call splits that axis
 * into up to 4 chunks. Each chunk is a contiguous range of x and of every
 * output. For chunk c: its x bytes are uploaded on the plan's upload stream,
 * projected on `stream` by fp_forward into device staging, and its outputs
 * downloaded on the plan's download stream. Two staging slots alternate, so
 * chunk c + 1's upload and compute overlap chunk c's download. Otherwise the
 * whole call is one chunk.
 * Staging (two chunks of x and of every output) is plan-owned device memory. It
 * is grown in stream order on `stream` (cudaMallocAsync) and freed by fp_reserve
 * or fp_destroy. Both side streams are forked from `stream` by an event, and
 * `stream` waits for the last download, so the work completes in `stream`
 * order. The host buffers must stay valid and unmodified until then. Host
 * calls on one plan run one after another: each starts after the previous
 * one's last download, whatever streams they are on. Inside a stream capture
 * only after a first call has sized the staging.
 * Errors: FP_ERR_INVALID_ARG for host buffers that are not page-locked host
 * memory, and every error of fp_forward (checked on the first chunk's staging
 * pointers before any copy is enqueued). Rotary positions: as fp_forward; with
 * caller positions the table is rebuilt per chunk. Returns FP_OK once the work
 * is enqueued; fp_last_launch_count counts the kernels of every chunk.
 */
fp_status fp_forward_host(fp_plan* plan, const void* x_host, const fp_layout* x_layout,
                          const void* W, const void* b, const int32_t* pos, void* out_ff_host,
                          void* out_q_host, void* out_k_host, void* out_v_host, void* stream);

/*
 * fp_forward_rope_table — fp_forward with caller-given rotary tables instead
 * of positions: the cos and sin inputs of the rope_one_entry listing (nvFuser
 * issue #1597 "Improve performance on RoPE"), [T, n_rot] with n_rot =
 * rope_n_elem (or head_dim), addressed through `layout` (the listing notes the
 * inner dimension need not be contiguous). Lane i < n_rot/2 of a rotated head
 * becomes x_i cos[t,i] - x_{i+n_rot/2} sin[t,i], lane i + n_rot/2 becomes
 * x_{i+n_rot/2} cos[t,i+n_rot/2] + x_i sin[t,i+n_rot/2]; t is the token's index
 * inside its batch element. The plan must have been created with rotary
 * embedding (its base is then unused). The tables are repacked on `stream` into
 * the plan's scratch (allocated on first use, 16 bytes per position and pair);
 * they must stay valid until the work completes. Other arguments as fp_forward.
 */
typedef struct {
  int32_t dtype;    /* fp_dtype of cos and sin */
  int64_t stride_t; /* elements between consecutive positions */
  int64_t stride_i; /* elements between consecutive lanes */
} fp_rope_table;

fp_status fp_forward_rope_table(fp_plan* plan, const void* x, const fp_layout* x_layout,
                                const void* W, const void* b, const void* rope_cos,
                                const void* rope_sin, const fp_rope_table* layout, void* out_ff,
                                void* out_q, void* out_k, void* out_v, void* stream);

/*
 * fp_backward_workspace_size — bytes of device workspace fp_backward needs for
 * an activation of layout `x_layout`: the gradient G at the fused output before
 * activation and rotation, [B*T, N] bf16 (rounded up to 256 bytes).
 */
fp_status fp_backward_workspace_size(const fp_plan* plan, const fp_layout* x_layout,
                                     size_t* bytes);

/*
 * fp_backward — enqueue the gradients of fp_forward's outputs with respect to
 * x, W and b on `stream`. The pages name this pass only as the part of the
 * fused linear that is left unfused and slow ("[perf] Fused linear", xformers
 * PR #283); it is the chain rule through the forward's steps in reverse:
 *   G[m, ff col]  = g_ff * act'(x W + b) at the recomputed pre-activation,
 *   G[m, q/k col] = the upstream gradient rotated back (the transpose of the
 *                   rotation: lane i: g_i cos + g_{i+h} sin, lane i+h:
 *                   g_{i+h} cos - g_i sin), v copied,
 *   dx = G W^T,  dW = X^T G,  db = sum over tokens of G.
 * Arguments:
 *   x, x_layout, W, b, pos   as for fp_forward (the same values as the forward)
 *   g_ff, g_q, g_k, g_v      upstream gradients, dtype of x, in the layouts of
 *                            out_ff, out_q, out_k, out_v (g_k pre-transposed
 *                            when the plan emits k that way); NULL exactly
 *                            where the forward output is NULL
 *   dx                       gradient of x, dtype of x, written through
 *                            x_layout's strides (a buffer laid out like x)
 *   dW                       float32 [C, N] row-major (overwritten)
 *   db                       float32 [N] (overwritten), or NULL to skip
 *   workspace                device buffer of fp_backward_workspace_size bytes,
 *                            256-byte aligned, owned by the caller
 * Runs on the tensor cores for bf16 layouts the forward's tcgen05 kernel
 * takes; other layouts and f32 return FP_ERR_UNSUPPORTED_LAYOUT. With no
 * tokens nothing is launched: dx (which may then be NULL) is empty and dW and
 * db are set to zero. dW and db
 * are sums whose order varies between runs (atomic adds across CTAs), so they
 * are reproducible to rounding, not bit for bit. Inputs must stay valid until
 * the work completes; nothing is allocated except, on first use, the plan's
 * status word and rotary table (as fp_forward) and, when both the ff
 * gradient and the q/k/v gather run, a second stream and two events of the
 * plan: the gather runs there beside the ff gradient, forked from `stream`
 * and joined back to it before the dx GEMM, so the call's work still
 * completes in `stream` order. A plan's calls are issued from one host
 * thread at a time. Returns FP_OK once enqueued.
 */
fp_status fp_backward(fp_plan* plan, const void* x, const fp_layout* x_layout, const void* W,
                      const void* b, const int32_t* pos, const void* g_ff, const void* g_q,
                      const void* g_k, const void* g_v, void* dx, float* dW, float* db,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * fp_backward_host — fp_backward for an activation, upstream gradients and
 * results in host memory, with the copies pipelined against the compute as in
 * fp_forward_host.
 *   x_host, g_*_host   page-locked host memory, layouts as fp_backward's x and
 *                      gradients (NULL exactly where fp_backward takes NULL)
 *   dx_host            page-locked host memory laid out like x
 *   dW_host, db_host   page-locked host float32 [C, N] and [N] (db_host NULL to
 *                      skip), overwritten
 *   W, b, pos          device pointers, as fp_backward
 * x must be dense (row-major strides over its sizes): dx comes back as whole
 * byte ranges. When the first axis is a batch axis (channel_dim != 0,
 * n_batch_dims >= 1) it is split into up to 4 chunks. For each chunk, x and
 * the gradients are uploaded on the plan's upload stream. The chunk's
 * gradients are computed on `stream`: dW and db are summed into plan-owned
 * device accumulators, cleared by the first chunk. dx is downloaded on the
 * plan's download stream, and dW and db after the last chunk. The staging,
 * the G workspace and the accumulators are plan-owned device memory, grown
 * and ordered as for fp_forward_host (shared with it). Errors: those of
 * fp_backward, FP_ERR_UNSUPPORTED_LAYOUT for a strided x, and
 * FP_ERR_INVALID_ARG for host buffers that are not page-locked. All are
 * checked before anything is enqueued. dW and db are sums whose order varies
 * between runs, as fp_backward's. Returns FP_OK once the work is enqueued.
 */
fp_status fp_backward_host(fp_plan* plan, const void* x_host, const fp_layout* x_layout,
                           const void* W, const void* b, const int32_t* pos,
                           const void* g_ff_host, const void* g_q_host, const void* g_k_host,
                           const void* g_v_host, void* dx_host, float* dW_host, float* db_host,
                           void* stream);

/*
 * fp_forward_noalloc — fp_forward for callers that may not allocate device
 * memory. The pages have no counterpart: it exists for callers such as a
 * plug-in running inside a host framework that owns every device byte through
 * its own pool, or a fixed-budget serving process that sizes memory once at
 * start-up, where a cudaMalloc during a call (which can also stall the device)
 * is not allowed. It takes the configuration directly (no plan) and runs the
 * same kernels as fp_forward, with their device scratch (two status words and
 * the rotary (cos, sin) table) in a static device array of 4 MiB + 256 bytes
 * that the library holds on every GPU that loads it, until process exit.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *   Sizes: the rotary table may need at most 524288 (cos, sin) entries, i.e.
 *   T * rope_n_elem/2 <= 524288 (T = tokens per batch element; rope_n_elem =
 *   head_dim when 0); larger problems are rejected with FP_ERR_INVALID_ARG and
 *   a message from fp_last_error(). Other arguments as fp_forward.
 *   Set-up: the first call on each device asks the runtime for the array's
 *   device address with that device current; make that first call before any
 *   stream capture.
 *   Sharing: every call uses the same array, which keeps the previous call's
 *   contents; each call clears the status words and rebuilds the table on its
 *   stream. Calls whose work overlaps on the GPU (other streams, other host
 *   threads) race on the array and must be serialised by the caller.
 *   Device-side timeouts still stop the kernels cleanly; the call cannot
 *   report them (it returns once the work is enqueued), but
 *   fp_get_device_status(NULL, stream) reads and clears these status words.
 *   The device address is cached per device ordinal for the life of the
 *   process: it assumes the device's primary context is not reset
 *   (cudaDeviceReset) while the library is loaded.
 */
fp_status fp_forward_noalloc(const fp_config* config, const void* x, const fp_layout* x_layout,
                             const void* W, const void* b, const int32_t* pos, void* out_ff,
                             void* out_q, void* out_k, void* out_v, void* stream);

/*
 * fp_attention — enqueue softmax attention over this plan's q, k, v outputs:
 *     out[z, i, :] = sum_t softmax_t(scale * q[z, i, :] . k[z', t, :]) v[z', t, :]
 * for every batch*head index z and query i, in the [batch*heads, tokens,
 * head_dim] layout of memory-efficient-attention issue #7 ("Improve
 * performance via batched-matmul and fused multiplies": the scaled scores of
 * its baddbmm, the softmax over the keys, its bmm with the values). The
 * queries are taken in chunks of 128 and the keys in chunks of 128 merged
 * under the running row maximum, as that page chunks them; with at most 128
 * keys there is one key chunk (the page's fast path). Both products run on
 * the tcgen05 tensor cores; bf16 in and out, fp32 scores and accumulation.
 *   q     [batch*heads, T_q, head_dim]
 *   k     [batch*kv, T_k, head_dim], or [batch*kv, head_dim, T_k] when the plan
 *         emits k pre-transposed (kv = n_query_groups, else heads; query head
 *         h uses k/v head h / (heads/kv) of its batch element)
 *   v     [batch*kv, T_k, head_dim]
 *   out   [batch*heads, T_q, head_dim], may not overlap q, k or v
 *   scale > 0: the softmax scale; <= 0: head_dim^(-1/2)
 * head_dim must be 64 or 128 (else FP_ERR_UNSUPPORTED_LAYOUT); with
 * pre-transposed k, T_k must be a multiple of 8 (its rows are TMA strides).
 * All pointers 16-byte aligned. Uses the plan's status word (device-side
 * timeouts surface through fp_get_device_status). Returns FP_OK once enqueued.
 * Work split: one CTA per 128-query block while whole waves of SMs fill; the
 * blocks past the last whole wave have their keys split over up to 16 CTAs
 * each, and a second launch merges those partial results (fp_last_launch_count
 * then reports 2). The partial results live in plan scratch, grown in stream
 * order like the rotary table (128 * (head_dim + 2) floats per split; freed by
 * fp_reserve or fp_destroy once replaced). Calls on one plan that overlap on
 * the GPU (different streams without ordering) share that scratch and must be
 * serialised by the caller.
 */
fp_status fp_attention(fp_plan* plan, const void* q, const void* k, const void* v, void* out,
                       int64_t batch, int64_t T_q, int64_t T_k, float scale, void* stream);

/*
 * fp_reserve — allocate, on the current device, the plan's device scratch
 * (status word and a rotary table for up to max_tokens_per_batch positions) so
 * that later fp_forward calls with T <= max_tokens_per_batch allocate nothing.
 * Unlike the calls that enqueue work, it waits for the allocation to complete;
 * if it replaces a table it first waits for the device to go idle and frees
 * every table the plan has retired.
 */
fp_status fp_reserve(fp_plan* plan, int64_t max_tokens_per_batch);

/*
 * fp_get_device_status — synchronise `stream`, then report and clear the
 * device-side status word: FP_OK, FP_ERR_TIMEOUT or FP_ERR_DEVICE_BOUNDS.
 * With plan == NULL it reads the status words of fp_forward_noalloc on the
 * current device (allocating nothing). Returns FP_ERR_CUDA if the
 * synchronisation itself failed.
 */
fp_status fp_get_device_status(fp_plan* plan, void* stream);

/* Number of kernels the plan's last successful fp_forward launched. */
int fp_last_launch_count(const fp_plan* plan);

/* Static description of the status code (never NULL). */
const char* fp_status_string(fp_status s);

/* Reason for the calling thread's most recent non-OK status ("" if none). */
const char* fp_last_error(void);

/*
 * fp_set_option — tuning and test hooks (not needed for normal use).
 *   FP_OPT_WAIT_LIMIT_NS   device-side bound on every wait (default 2e9 ns)
 *   FP_OPT_INJECT_STALL    1: the next bf16 launch's first CTA withholds one
 *                          operand load, so its consumers' bounded waits run
 *                          out and the launch reports FP_ERR_TIMEOUT (tests the
 *                          error path; the GPU stays usable). Cleared after use.
 *   FP_OPT_GROUP_M         tile rasterisation: M-tiles per group (>= 1)
 *   FP_OPT_MAX_CTAS        cap on the persistent grid (0 = one CTA per SM)
 *   FP_OPT_CLUSTER         2 (default): CTA pairs run 2-SM MMAs over one
 *                          256-column weight tile, each CTA loading its own half
 *                          of it and its own 128 token rows; 1: single CTAs,
 *                          each loading the whole weight tile
 *   FP_OPT_BOUNDS_CHECK    1: every output store whose address the kernels
 *                          compute themselves (ragged or batch-crossing tiles,
 *                          pre-transposed k, the FFMA kernel) is first checked
 *                          against its buffer; one that would leave it is
 *                          skipped and reported as FP_ERR_DEVICE_BOUNDS (stores
 *                          by TMA are confined by their tensor maps). 2: the same
 *                          against half of each buffer, a test of the check
 *                          itself (stores past the middle are reported, never
 *                          made). 0 (default): off. Forward calls only.
 *   FP_OPT_TILE_N          width of the tensor-core tiles without rotation: 0
 *                          (default) takes 256, or 192 where 256-column tiles
 *                          would compute at least 15 % more columns than N
 *                          (N = 384, 576, 960 ...); 256 or 192 forces it. CTA
 *                          pairs only; rotated layouts keep whole heads per tile
 */
typedef enum {
  FP_OPT_WAIT_LIMIT_NS = 1,
  FP_OPT_INJECT_STALL = 2,
  FP_OPT_GROUP_M = 3,
  FP_OPT_MAX_CTAS = 4,
  FP_OPT_CLUSTER = 5,
  FP_OPT_BOUNDS_CHECK = 6,
  FP_OPT_TILE_N = 7
} fp_option;
fp_status fp_set_option(fp_plan* plan, fp_option opt, int64_t value);

/* Release the plan and its device scratch. NULL is a no-op. */
void fp_destroy(fp_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* FP_H */
