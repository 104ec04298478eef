/*
 * moe_w4.h -- C ABI of the GB300 (sm_103a) W4A16 mixture-of-experts block.
 *
 * The block is the expert layer of a Qwen3.6-35B-A3B-style model as described
 * in "Perplexity libera Lily, un motor de IA que supera a MLX-LM en Apple
 * Silicon" (diariobitcoin.com):
 *   - section "Qwen3.6 combina tres cargas de trabajo": a router scores all E
 *     (256) experts and selects k (8) per token; one shared expert processes
 *     every token; weights are 4-bit affine with groups of 64, one bfloat16
 *     scale and one bfloat16 bias per group;
 *   - section "Las optimizaciones en el prefill": the grouped GEMM rebuilds
 *     weights block by block on chip and accumulates in FP32 (the dequantised
 *     array never exists in memory), and the routing histogram, prefix scan,
 *     scatter and block map stay on the GPU with no CPU synchronisation
 *     inside a layer.
 *
 * Conventions for every call:
 *   - All tensor arguments are DEVICE pointers owned by the caller, on the
 *     plan's device, 16-byte aligned. bf16 tensors are passed as uint16_t bit
 *     patterns. The library never frees or keeps caller memory past a call.
 *   - A plan owns only its device scratch, allocated once in moe_plan_create
 *     and sized for max_tokens.
 *   - Calls are stream-ordered and asynchronous: they enqueue kernels on
 *     `stream` (NULL = legacy default stream) and never wait for the device.
 *     Grid sizes never depend on routing results, so no value is read back.
 *   - Argument errors are found on the host before any launch and returned as
 *     a status; nothing is enqueued then. Errors found on the device (a
 *     bounded wait that ran out) are latched in a device word and reported by
 *     moe_get_error.
 *   - Weights (router weights, packed experts, scales, biases) are read by
 *     some kernels before they wait for the previous launch on the stream
 *     (programmatic dependent launch): no kernel running just before a call
 *     on the same stream may write them (record an event, or run any other
 *     launch in between). Token inputs are always read after that wait.
 *   - A plan is not thread-safe: calls on one plan must come from one host
 *     thread at a time, and calls that share a plan's scratch must be ordered
 *     on the device (same stream, or explicit events).
 *   - Operand precision. The pages fix only FP32 accumulation and the bf16
 *     scale and bias. The expert GEMMs multiply fp16 operands: token values
 *     are converted from bf16 to fp16 (exact for magnitudes up to 65504;
 *     below 2^-14 they become fp16 subnormals, an absolute error under
 *     2^-25, negligible against a unit-scale row), the tensor-core path
 *     rebuilds each weight as fp16(q * scale + bias) from fp16 copies of the
 *     scale and bias, and the SwiGLU activations are stored as fp16. The
 *     contract, checked on the device:
 *       |x| < 65536 for every token value (a larger one, an inf or a NaN is
 *         clamped to +-65504 and flagged), checked on every call;
 *       every scale is 0 or has magnitude in [2^-14, 2^12) and every bias
 *         has magnitude below 2^11 (then |q * scale + bias| < 65504 and no
 *         scale is an fp16 subnormal), checked once per weight set, by a
 *         kernel on the stream the first time a plan sees the set (by its
 *         scale and bias addresses; new values written in place at the
 *         same addresses are not checked again).
 *     A value outside the contract sets a bit in the plan's device error
 *     word that moe_get_error reports as MOE_ERR_OPERAND_RANGE; the call
 *     itself still completes with clamped values. The activations the
 *     block produces itself (RMS-normalised stack input, SwiGLU outputs of
 *     in-contract weights) stay far inside these bounds.
 */
#ifndef MOE_W4_H
#define MOE_W4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t compatible handle, so this header needs no CUDA headers */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, bad field */
  MOE_ERR_UNSUPPORTED = 2,    /* valid request this build has no kernel for */
  MOE_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  MOE_ERR_CAPACITY = 4,       /* T above the plan's max_tokens */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a device-side bounded wait ran out */
  MOE_ERR_OPERAND_RANGE = 6   /* an input outside the fp16 operand range (below) */
} moe_status;

/* Plan description. Sizes are in elements. */
typedef struct {
  int hidden;            /* H: model width (2048); multiple of group_size */
  int inter;             /* I: expert FFN width (512); multiple of group_size */
  int num_experts;       /* E: routed experts (256); 8..512, multiple of 8 */
  int top_k;             /* k: experts per token (8); 1..min(E, 32) */
  int group_size;        /* G: quantisation group along K; must be 64 */
  int has_shared;        /* 1: one always-on shared expert with weight 1 */
  int max_tokens;        /* capacity: scratch is sized for this T, once */
  int block_m;           /* rows per block-map tile; must be 128 */
  int gemm_path;         /* 0 auto, 1 tensor-core (tcgen05) path, 2 small-M path,
                            3 tensor-core path on SM pairs (tcgen05 cta_group::2;
                            falls back to 1 on a device without cluster launch) */
  int small_m_max_tokens;/* auto: T <= this uses the small-M path (default 16 if 0) */
  int wait_limit_ms;     /* device bounded-wait limit (default 1000 if 0) */
} moe_plan_desc;

typedef struct moe_plan* moe_plan_t;

/* One 4-bit affine matrix set for E experts, N output rows, K inputs.
 * Weight W[e][n][kk] = q * scale[e][n][kk/64] + bias[e][n][kk/64] where q is
 * nibble (kk % 8) -- bits 4*(kk%8) .. 4*(kk%8)+3 -- of qweight[e][n][kk/8],
 * read as an unsigned integer 0..15. */
typedef struct {
  const uint32_t* qweight;   /* [E][N][K/8] */
  const uint16_t* scales;    /* [E][N][K/64] bf16 */
  const uint16_t* biases;    /* [E][N][K/64] bf16 */
} moe_w4;

/* SwiGLU expert set: gate and up are N = inter, K = hidden; down is
 * N = hidden, K = inter. An expert computes
 *   a[n] = silu(sum_k x[k] Wg[n][k]) * sum_k x[k] Wu[n][k],
 *   out[m] = sum_n a[n] Wd[m][n]. */
typedef struct {
  moe_w4 gate, up, down;
} moe_experts;

/* Routing result. moe_route fills this with pointers into plan scratch that
 * stay valid until the next moe_route / moe_forward_layer on the plan. A
 * caller may also point it at its own device buffers with these layouts
 * (slot s = t*k + j, position = row in expert-contiguous order):
 *   topk_idx     int32 [T][k]  selected experts, rank order (logit desc,
 *                              lower index first on ties)
 *   topk_w       f32   [T][k]  softmax over all E, renormalised over the k
 *   counts       int32 [E]     histogram of selected experts
 *   offsets      int32 [E+1]   exclusive prefix scan of counts; [E] = T*k
 *   tile_offsets int32 [E+1]   exclusive scan of ceil(counts/block_m)
 *   perm         int32 [T*k]   position -> slot, stable in token order
 *   inv          int32 [T*k]   slot -> position
 *   block_map    int32 [tiles][3] (expert, first position, rows) per tile,
 *                              expert-major; shared-expert tiles excluded
 *   num_tiles    int32 [1]     number of block_map tiles
 *   logits       f32   [T][E]  router logits (moe_route only; may be NULL
 *                              when the struct is given to
 *                              moe_grouped_w4_ffn) */
typedef struct {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* tile_offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* block_map;
  int32_t* num_tiles;
  float* logits;
} moe_routing;

/* Create a plan on CUDA device `device`: validates `desc` (host only; no
 * CUDA call is made when it is invalid) and allocates the scratch. */
moe_status moe_plan_create(const moe_plan_desc* desc, int device, moe_plan_t* out);

/* Free the plan and its scratch. Waits for the device to finish using it. */
moe_status moe_plan_destroy(moe_plan_t plan);

/* Bytes of device scratch a plan with this description allocates (host only). */
moe_status moe_plan_scratch_bytes(const moe_plan_desc* desc, size_t* bytes);

/* Routing (histogram, prefix scan, scatter and block map in section "Las
 * optimizaciones en el prefill"; router and top-8 in section "Qwen3.6
 * combina tres cargas de trabajo"):
 *   logits[t][e] = sum_h x[t][h] * router_w[h][e] + router_bias[e]  (FP32)
 * then top-k, weights, counts, offsets, tile offsets, perm, inv, block map.
 * x: bf16 [T][H]; router_w: bf16 [H][E]; router_bias: f32 [E] or NULL.
 * `out` receives pointers into plan scratch. 1 <= T <= max_tokens. */
moe_status moe_route(moe_plan_t plan, const uint16_t* x, int T, const uint16_t* router_w,
                     const float* router_bias, moe_routing* out, moe_stream_t stream);

/* Experts on a given routing (the grouped GEMM with block-wise dequant in
 * section "Las optimizaciones en el prefill"):
 *   y[t] = shared(x[t]) + sum_j topk_w[t][j] * expert_{topk_idx[t][j]}(x[t])
 * x: bf16 [T][H]; routing: as moe_route produces (topk_w, perm, inv,
 * block_map and num_tiles are read); routed: E experts; shared: one expert
 * set with E = 1, or NULL (must be non-NULL iff desc.has_shared);
 * y: f32 [T][H], the block's FP32 sum (the pages accumulate in FP32; a bf16
 * rounding of y alone would cost about 1.5% of the output's rms at 4-sigma
 * values), must not overlap x. Dequantised weights exist only in on-chip
 * memory. Routed experts' outputs are weighted and kept in bf16 before the
 * combine; the shared expert's are kept in FP32. */
moe_status moe_grouped_w4_ffn(moe_plan_t plan, const uint16_t* x, int T,
                              const moe_routing* routing, const moe_experts* routed,
                              const moe_experts* shared, float* y, moe_stream_t stream);

/* moe_route followed by moe_grouped_w4_ffn: one MoE layer, no host sync. */
moe_status moe_forward_layer(moe_plan_t plan, const uint16_t* x, int T,
                             const uint16_t* router_w, const float* router_bias,
                             const moe_experts* routed, const moe_experts* shared,
                             float* y, moe_stream_t stream);

/* moe_forward_layer followed by moe_residual_add(x, y, T, alpha, x, xn_out)
 * in one call whose last pass updates the stack directly from the experts'
 * outputs, so y is never written (the FP32 [T][H] round trip is saved):
 *   y = moe(xn); x = bf16(x + alpha * y); xn_out = bf16(rmsnorm(x))
 * Bit-identical to the two calls. xn (the layer's input) and xn_out may be
 * the same buffer (the update runs after every read of xn); x must differ
 * from both. Layouts as in moe_forward_layer and moe_residual_add. */
moe_status moe_forward_layer_residual(moe_plan_t plan, const uint16_t* xn, int T,
                                      const uint16_t* router_w, const float* router_bias,
                                      const moe_experts* routed, const moe_experts* shared,
                                      float alpha, uint16_t* x, uint16_t* xn_out,
                                      moe_stream_t stream);

/* One layer of a stack for moe_forward_stack: its router and experts.
 * shared is ignored (may be NULL) when the plan has no shared expert. */
typedef struct {
  const uint16_t* router_w;     /* bf16 [H][E] */
  const float* router_bias;     /* f32 [E] or NULL */
  moe_experts routed;
  moe_experts shared;
} moe_layer;

/* A stack of MoE layers on a prompt of any length (chunked prefill; the
 * pages' engine prefills long prompts in chunks, "Las optimizaciones en el
 * prefill"). x is the residual stream, bf16 [T][H], updated in place:
 *   xn = bf16(rmsnorm(x));
 *   for each layer: x = bf16(x + alpha * moe_layer(xn)); xn = bf16(rmsnorm(x))
 * T may exceed the plan's max_tokens: the tokens go through all layers in
 * chunks of at most max_tokens rows, one chunk after the other (the block
 * treats every token on its own, so each chunk's result is the one of the
 * whole prompt). xn is caller scratch, bf16 [min(T, max_tokens)][H], and holds
 * the last chunk's normalised stream on return. Every layer of a chunk is one
 * moe_forward_layer_residual, except for decode-sized chunks (at most 8
 * tokens, on the small-M path): there every layer is one launch of a fused
 * kernel that takes the RMS norm, routes, runs both expert passes and
 * updates x (the same arithmetic up to rounding: the routed experts' outputs
 * stay FP32 until the combine; the routing lands in the plan's routing
 * arrays and y in its FP32 shared-output buffer, moe_debug_buffer 3).
 * Stream-ordered, no host sync. Errors: as for the per-layer calls (checked
 * for every layer before any launch); MOE_ERR_INVALID_ARG for num_layers < 1
 * or a NULL layers array. */
moe_status moe_forward_stack(moe_plan_t plan, uint16_t* x, uint16_t* xn, int T,
                             const moe_layer* layers, int num_layers, float alpha,
                             moe_stream_t stream);

/* Update between stacked layers (not part of the expert block itself):
 *   x_out[t] = bf16(x[t] + alpha * y[t])                 (skipped if y == NULL)
 *   xn_out[t] = bf16(x_out[t] / sqrt(mean_h x_out[t][h]^2 + 1e-6))
 *                                                        (skipped if NULL)
 * x, x_out, xn_out bf16 [T][H]; y f32 [T][H]; FP32 arithmetic, the mean of
 * squares over the bf16-rounded x_out. x_out may equal x (NULL means x);
 * xn_out must be a separate buffer. xn_out is the RMS-normalised input of
 * the next layer: without it the SwiGLU experts, quadratic in their input,
 * make a residual stack grow without bound. */
moe_status moe_residual_add(moe_plan_t plan, const uint16_t* x, const float* y, int T,
                            float alpha, uint16_t* x_out, uint16_t* xn_out,
                            moe_stream_t stream);

/* Routing without a plan and without any device allocation. The pages have
 * no counterpart: this entry point exists for callers that cannot call
 * cudaMalloc -- a host framework that hands out all device memory from its
 * own pool (an allocation behind its back can fail or fragment the memory
 * it budgets), runtimes with no device allocator at all, and latency-bound
 * callbacks that must not block (cudaMalloc can synchronise the device).
 * It computes exactly what moe_route computes, with the same kernels.
 * The caller passes x, router_w, router_bias (may be NULL) as for moe_route
 * and every output buffer in `out` (layouts as in moe_routing; block_map
 * must hold ceil(T*k/128) + E triples; logits is required, every buffer
 * 8-byte aligned; hidden a multiple of 64, num_experts a multiple of 8 and
 * at least 8, 1 <= top_k <= num_experts, otherwise MOE_ERR_INVALID_ARG;
 * top_k above 32 returns MOE_ERR_UNSUPPORTED as for a plan). Every input is
 * read only after the previous work on the stream has completed, so the
 * caller's own kernel just before may write x or the router weight.
 * The library's only scratch for this call is a fixed device array of
 * 128 x 512 int32 (256 KB) in the library image, present on every GPU that
 * loads the library until the process exits; hence T <= 4096 and
 * num_experts <= 512, and larger requests return MOE_ERR_CAPACITY. Nothing
 * in that array needs clearing between calls. The first call on a device
 * looks up the array's device address (a host-side runtime query, with that
 * device current) and keeps it for later calls. All calls share the array:
 * calls that can overlap on the GPU (different streams without ordering)
 * race and must not be made.
 * A bounded wait of the routing kernels that runs out (1 s) leaves the
 * outputs unspecified and is reported by moe_route_noalloc_get_error. */
moe_status moe_route_noalloc(const uint16_t* x, int T, int hidden, const uint16_t* router_w,
                             const float* router_bias, int num_experts, int top_k,
                             const moe_routing* out, moe_stream_t stream);

/* Reads and clears the device error word of moe_route_noalloc on the
 * current device (shared by every call on that device). Synchronises the
 * device: call it between steps, never inside one. Returns MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT, or MOE_ERR_CUDA if the context has failed. Not
 * part of the pages' method: the error path of the call above. */
moe_status moe_route_noalloc_get_error(void);

/* Launches, on `stream`, a kernel whose bounded wait can never be satisfied,
 * with the given limit (1 us .. 10 s) and the error word of
 * moe_route_noalloc: it gives up, latches MOE_ERR_DEVICE_TIMEOUT there and
 * exits, so a test can check moe_route_noalloc_get_error without faulting
 * or hanging the GPU. */
moe_status moe_route_noalloc_debug_wait_timeout(int limit_us, moe_stream_t stream);

/* Reads and clears the plan's device error word. Synchronises the device:
 * call it between layers or steps, never inside one. Returns MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT (a bounded wait ran out; reported first),
 * MOE_ERR_OPERAND_RANGE (an input outside the fp16 operand contract above),
 * or MOE_ERR_CUDA if the context has failed. */
moe_status moe_get_error(moe_plan_t plan);

/* Launch a kernel whose bounded wait can never be satisfied, with the given
 * limit: it must give up, latch MOE_ERR_DEVICE_TIMEOUT and exit. Lets a test
 * check the failure path without faulting or hanging the GPU. */
moe_status moe_debug_wait_timeout(moe_plan_t plan, int limit_us, moe_stream_t stream);

/* Kernel timing for profiling. When enabled, every kernel the plan launches
 * is bracketed by CUDA events on its stream. moe_read_timing synchronises,
 * adds up the elapsed times per kernel kind since the last read, and resets.
 * Kinds: 0 router logits, 1 scan, 2 scatter, 3 gather, 4 gate/up GEMM,
 * 5 down GEMM, 6 combine, 7 residual, 8 top-k selection, 9 fused decode
 * layer. */
#define MOE_NUM_KERNEL_KINDS 10
typedef struct {
  double ms[MOE_NUM_KERNEL_KINDS];
  long long launches[MOE_NUM_KERNEL_KINDS];
} moe_timing;
moe_status moe_enable_timing(moe_plan_t plan, int on);
moe_status moe_read_timing(moe_plan_t plan, moe_timing* out);

/* Introspection of plan scratch for tests and profiling: device address of
 * the gathered activations (which = 0: fp16 [rows][H], routed positions
 * first, then the shared expert's T rows), the SwiGLU activations (1: fp16
 * [rows][I]) -- both with each block of 8 columns stored in the order
 * (0,4,1,5,2,6,3,7) --, the weighted routed expert outputs (2: bf16 [T*k][H]) or the
 * shared expert's outputs (3: f32 [T][H]) of the last layer. NULL for an
 * unknown `which` or a plan without a shared expert (3). */
void* moe_debug_buffer(moe_plan_t plan, int which);

/* Which GEMM path the last layer call took: 1 tensor-core, 2 small-M, 3 the
 * fused decode layer of moe_forward_stack, 4 tensor-core on SM pairs. */
int moe_last_gemm_path(moe_plan_t plan);

/* Load balance of the tensor-core path for expert groups of very different
 * sizes (the grouped GEMM of section "Las optimizaciones en el prefill"
 * runs over groups whose sizes vary by expert); on = 1, off = 0 (the
 * default). Units (one
 * 128-token tile x one weight block pair) are dealt in rounds over the SMs,
 * and when the last round holds at most half as many units as SMs, each of
 * its units is cut along K into two halves on different SMs, whose fp32
 * partial sums the SM that finishes second adds (one addition, the same
 * bits whichever SM that is: the result is the same on every run).
 * A token's output then depends, in its last bits, on whether its tile fell
 * into the last round. Off, every tile is summed over K in one pass, so a
 * prompt run in chunks gives the bits of one pass. Off by default: on the
 * 2048- and 4096-token workloads the split measured slower (the halves'
 * partial sums cost more than the idle SMs of the last round). Host only;
 * takes effect from the next call. */
moe_status moe_set_tail_split(moe_plan_t plan, int on);

/* Text of a status code. */
const char* moe_status_string(moe_status s);

/* Library version, major*10000 + minor*100 + patch. */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4_H */
