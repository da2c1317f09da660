/*
 * ft_moe.h — C ABI of the NVFP4 mixture-of-experts layer for GB300 (sm_103a).
 *
 * The layer is the one a serving engine runs in every layer at every decode step
 * (FreeToken PR #84, "Effect in production": the NVFP4 MoE decode GEMV): router
 * softmax / top-k (FreeToken commit log, 512-expert entry: "non-power-of-2 top-k
 * router"), then per selected expert a W13 (gate|up) product on NVFP4 weights fused
 * with clamped SwiGLU (288-expert entry: "clamped-SwiGLU activation across the MoE
 * stack"), then a W2 product whose outputs are summed with the router weights, plus an
 * optional gated shared expert (512-expert entry: "512 NVFP4 ... routed experts
 * (top-10) plus a gated shared expert").
 *
 * Conventions for every entry point
 *  - All array pointers are DEVICE pointers owned by the caller; the library allocates
 *    nothing, frees nothing and never synchronises inside route / decode / prefill.
 *  - bf16 tensors are passed as uint16_t bit patterns (the upper half of an IEEE float).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Work is enqueued
 *    asynchronously on it; the call returns after enqueueing.
 *  - Host-side argument checks run before any launch; on failure nothing is enqueued
 *    and the call returns the error. A failed launch returns FT_ERR_CUDA.
 *  - Anomalies seen inside kernels (an expert id outside [0, E)) are OR-ed into an
 *    error word at the start of the workspace; ft_moe_get_error() reports and clears it.
 *  - Results are deterministic: the same inputs give the same output bits.
 *
 * NVFP4 weight layout (per expert, per projection; reduction dimension contiguous):
 *  - codes: uint8, two 4-bit E2M1 codes per byte, the even element in the low nibble
 *    (E2M1: sign bit 3, 2 exponent bits with bias 1, 1 mantissa bit; magnitudes
 *    0, 0.5, 1, 1.5, 2, 3, 4, 6);
 *  - block scales: one E4M3 (fn) byte per 16 consecutive elements of a row;
 *  - one FP32 tensor scale per expert and projection;
 *  - element value = e2m1(code) * e4m3(block scale) * tensor scale.
 *  W13 of expert e is [2I, H]: rows [0, I) are the gate projection, rows [I, 2I) the up
 *  projection. W2 of expert e is [H, I].
 */
#ifndef FT_MOE_H
#define FT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FT_OK = 0,
  FT_ERR_INVALID_ARG = 1,       /* null pointer, k < 1, k > E, T < 0, bad limit, ... */
  FT_ERR_UNSUPPORTED_SHAPE = 2, /* H or I not a multiple of 128, k > 32, E > 4096, ...  */
  FT_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment stated below          */
  FT_ERR_WORKSPACE_TOO_SMALL = 4,
  FT_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed                 */
  FT_ERR_DEVICE_FLAG = 6,       /* a kernel saw an expert id outside [0, E)             */
  FT_ERR_TIMEOUT = 7            /* reserved: a bounded device-side wait gave up         */
} ft_status;

/* Routed experts, all device pointers, 16-byte aligned:
 *   w13        uint8 [E, 2I, H/2]   w13_scale uint8 [E, 2I, H/16]   w13_gscale float [E]
 *   w2         uint8 [E, H,  I/2]   w2_scale  uint8 [E, H,  I/16]   w2_gscale  float [E]
 * (the gscale arrays need only 4-byte alignment). */
typedef struct {
  int32_t E, H, I;
  const uint8_t* w13;
  const uint8_t* w13_scale;
  const float* w13_gscale;
  const uint8_t* w2;
  const uint8_t* w2_scale;
  const float* w2_gscale;
} ft_nvfp4_experts;

/* Optional dense shared expert with the routed experts' H and I (same layouts without
 * the E dimension; the two gscale pointers point at one device float each) and its gate
 * vector gv (bf16 [H], 16-byte aligned). Its output is scaled by sigmoid(x_t . gv) and added to y_t. */
typedef struct {
  const uint8_t* w13;
  const uint8_t* w13_scale;
  const float* w13_gscale;
  const uint8_t* w2;
  const uint8_t* w2_scale;
  const float* w2_gscale;
  const uint16_t* gate;
} ft_nvfp4_shared_expert;

/* Version of this ABI (bumped on any incompatible change). */
int32_t ft_moe_abi_version(void);

/* Text for a status code (static storage, never NULL). */
const char* ft_status_string(ft_status s);

/*
 * ft_moe_route — router softmax -> top-k -> renormalise, one warp per token.
 *   logits    float [T, E] (4-byte aligned), must be finite
 *   topk_idx  int32 [T, k] out: the k experts with the largest logits, in descending
 *             logit order; equal logits go to the lower expert index. Ranking uses the
 *             fp32 logits themselves, so the choice is exact.
 *   topk_w    float [T, k] out: softmax over all E renormalised over the kept k, i.e.
 *             exp(l_j - l_max) / sum over kept i of exp(l_i - l_max).
 *   1 <= k <= min(E, 32), 1 <= E <= 4096, T >= 0. T = 0 (an empty batch) returns FT_OK
 *   without reading or writing anything; the pointers may then be NULL.
 */
ft_status ft_moe_route(const float* logits, int32_t T, int32_t E, int32_t k,
                       int32_t* topk_idx, float* topk_w, void* stream);

/*
 * ft_moe_router_logits — the router's logits l_t = W_router x_t, and the shared expert's gate
 * dot x_t . gv (the FreeToken commit log lists "moe router / shared gate" kernels beside the
 * MoE GEMV; the pages do not define them further: the plain reading is a bf16 matrix product
 * with float32 accumulation). Below 64 tokens one CUDA-core pass computes both; from 64 tokens
 * the logits run on the tensor cores (one launch) and the gate dot on the CUDA cores (a second
 * launch on the same stream).
 *   x         bf16 [T, H], w_router bf16 [E, H], gate bf16 [H] or NULL (16-byte aligned)
 *   logits    float [T, E] (4-byte aligned), fully overwritten
 *   gate_dot  float [T], written when gate is given (may be NULL otherwise)
 *   H a multiple of 8; E <= 4096. Products are exact in float32 and every sum runs in a fixed
 *   order for a given T (deterministic; the two forms may differ in the last bits). T = 0 is a
 *   no-op.
 */
ft_status ft_moe_router_logits(const uint16_t* x, int32_t T, int32_t H, const uint16_t* w_router,
                               int32_t E, const uint16_t* gate, float* logits, float* gate_dot,
                               void* stream);

/*
 * ft_moe_router_route — ft_moe_router_logits then ft_moe_route on those logits, enqueued by
 * one call (two launches): the routing slots from the activations and the router matrix.
 * logits [T, E] is the caller's buffer for the intermediate logits; the rest as for the two
 * calls.
 */
ft_status ft_moe_router_route(const uint16_t* x, int32_t T, int32_t H, const uint16_t* w_router,
                              int32_t E, const uint16_t* gate, int32_t k, float* logits,
                              float* gate_dot, int32_t* topk_idx, float* topk_w, void* stream);

/* Workspace bytes that decode (prefill = 0) or prefill (prefill = 1) needs for these
 * sizes on the current device; has_shared = 1 when a shared expert is passed. Without a
 * usable device the decode figure is an upper bound for any GPU. Returns 0 for invalid
 * sizes and for T = 0 (an empty batch needs no workspace). */
size_t ft_moe_workspace_bytes(int32_t T, int32_t k, int32_t E, int32_t H, int32_t I,
                              int32_t has_shared, int32_t prefill);

/* Dynamic shared memory per CTA that the decode kernel launches with for these sizes (one
 * CTA per SM, 512 threads): the plan, the activations when they are kept on chip, and the
 * weight rings. Host-only arithmetic, no device call; 0 for sizes decode does not accept. */
size_t ft_moe_decode_smem_bytes(int32_t T, int32_t k, int32_t E, int32_t H, int32_t I,
                                int32_t has_shared);

/* Zero a workspace once after allocating it. Enqueued on `stream`.
 * Only the first FT_MOE_WORKSPACE_HEAD_BYTES bytes (the error word and the barrier and
 * completion counters) must be zero before a call, and every call leaves them at zero
 * again; the rest is scratch that a call writes before it reads it, so its contents
 * (stale results, NaN bit patterns) never reach an output. */
#define FT_MOE_WORKSPACE_HEAD_BYTES 1024
ft_status ft_moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * ft_moe_nvfp4_decode — the expert part of the layer for a decode batch (0 <= T <= 64).
 *   T = 0 (an empty batch) returns FT_OK after the shape checks without reading or
 *   writing anything; x, topk_idx, topk_w, out and workspace may then be NULL.
 *   x            bf16 [T, H] (16-byte aligned)
 *   topk_idx     int32 [T, k], topk_w float [T, k]: as written by ft_moe_route (any
 *                source is accepted; an id outside [0, E) raises FT_ERR_DEVICE_FLAG in the
 *                workspace error word and that slot contributes nothing)
 *   ex           routed experts (see ft_nvfp4_experts); ex->H, ex->I multiples of 128,
 *                H <= 16384, I <= 8192
 *   sh           shared expert or NULL
 *   swiglu_limit L in (0, 128]: h = silu(min(g, L)) * clamp(u, -L, L)
 *   out          bf16 [T, H] (16-byte aligned), fully overwritten:
 *                y_t = sum_j topk_w[t,j] * W2_e (h_tj) [+ sigmoid(x_t.gv) * shared(x_t)]
 *   workspace    device scratch of at least ft_moe_workspace_bytes(T,k,E,H,I,sh!=0,0)
 *                bytes, 256-byte aligned, zeroed once by ft_moe_workspace_init; calls that
 *                share a workspace must be ordered on one stream.
 */
ft_status ft_moe_nvfp4_decode(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                              const float* topk_w, int32_t k, const ft_nvfp4_experts* ex,
                              const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                              uint16_t* out, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * ft_moe_nvfp4_decode_routed — route and decode in one call: the layer from the router
 * logits instead of the routing slots (the softmax -> top-k -> renormalise of
 * ft_moe_route, then ft_moe_nvfp4_decode). For T = 1 it is a single kernel launch in which
 * every CTA routes the token itself; for T >= 2 it enqueues the route kernel and then the
 * decode kernel. The experts, weights and output are bit-identical to ft_moe_route followed
 * by ft_moe_nvfp4_decode.
 *   logits        float [T, E] (4-byte aligned), must be finite
 *   topk_idx_out  int32 [T, k] or NULL; topk_w_out float [T, k] or NULL: when given, the
 *                 routing slots are written there (as ft_moe_route writes them)
 *   workspace     as for ft_moe_nvfp4_decode (ft_moe_workspace_bytes(T,k,E,H,I,sh!=0,0))
 *   other arguments, limits, T = 0 and errors: as ft_moe_nvfp4_decode.
 */
ft_status ft_moe_nvfp4_decode_routed(const uint16_t* x, int32_t T, const float* logits,
                                     int32_t k, const ft_nvfp4_experts* ex,
                                     const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                                     uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * ft_moe_nvfp4_prefill — the same layer for a multi-token chunk (any T >= 0), run as
 * grouped dense contractions: tokens are grouped by expert on the GPU, NVFP4 tiles are
 * dequantised to bf16 on chip and multiplied on the tensor cores. Arguments as for
 * decode, with workspace of at least ft_moe_workspace_bytes(T,k,E,H,I,sh!=0,1) bytes.
 */
ft_status ft_moe_nvfp4_prefill(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                               const float* topk_w, int32_t k, const ft_nvfp4_experts* ex,
                               const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                               uint16_t* out, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * ft_moe_nvfp4_decode_noalloc — ft_moe_nvfp4_decode for callers that cannot allocate
 * device memory: a host framework that owns the GPU's memory through its own pool, a
 * latency-bound serving loop that must not call cudaMalloc / cudaFree (they can
 * synchronise the device), or a plug-in handed only a stream and its tensors. The pages
 * have no counterpart: this is a deployment variant of the decode entry point.
 *   Arguments as for ft_moe_nvfp4_decode, without the workspace: the scratch is a fixed
 *   16 MiB array inside the library, held on every GPU that loads it until the process
 *   exits. Shapes whose decode scratch (ft_moe_workspace_bytes) exceeds it return
 *   FT_ERR_WORKSPACE_TOO_SMALL; nothing is allocated, by this call or by any library
 *   routine it uses.
 *   The first call on a device does a one-time set-up there (the array's device address
 *   and the SM count, with that device current); make that first call before any stream
 *   capture. Each call clears the array's error word and barrier counter on `stream`
 *   before its kernel; every call shares the array, so calls that overlap on the GPU
 *   (other streams, other host threads) race: order them on one stream. Device-side
 *   flags (bad expert ids, timeouts) are not reported by this variant.
 */
ft_status ft_moe_nvfp4_decode_noalloc(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                                      const float* topk_w, int32_t k,
                                      const ft_nvfp4_experts* ex,
                                      const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                                      uint16_t* out, void* stream);

/*
 * ft_moe_layer_from_host — the whole layer for T tokens whose activations and router
 * logits are in host memory, with the output returned to host memory: enqueues on `stream`
 * the copy of x and of the logits into the caller's device buffers, the layer (for T <= 64
 * ft_moe_nvfp4_decode_routed; for larger T ft_moe_route into topk_idx_dev / topk_w_dev, then
 * ft_moe_nvfp4_prefill), and the copy of the output back. Nothing is synchronised: the host
 * output is complete once `stream` has reached this point. The pages' engine runs the layer
 * on device-resident activations; this is the same layer with the host transfers of one
 * call attached, so that one C call serves a caller whose inputs start on the host.
 *   x_host       bf16 [T, H] in host memory, logits_host float [T, E]; out_host bf16 [T, H]
 *                (page-locked memory keeps the copies asynchronous; other host memory
 *                works but makes them synchronous)
 *   x_dev, logits_dev, out_dev  device buffers of those sizes (16-, 4- and 16-byte aligned)
 *   topk_idx_dev int32 [T, k], topk_w_dev float [T, k] on the device: required for T > 64
 *                (they receive the routing slots), optional (NULL) for T <= 64
 *   workspace    ft_moe_workspace_bytes(T, k, E, H, I, sh != 0, T > 64) bytes, as for the
 *                call it runs
 *   Other arguments and errors as for ft_moe_nvfp4_decode_routed / ft_moe_nvfp4_prefill; a
 *   failed copy returns FT_ERR_CUDA.
 */
ft_status ft_moe_layer_from_host(const uint16_t* x_host, const float* logits_host, int32_t T,
                                 int32_t k, const ft_nvfp4_experts* ex,
                                 const ft_nvfp4_shared_expert* sh, float swiglu_limit,
                                 uint16_t* out_host, uint16_t* x_dev, float* logits_dev,
                                 int32_t* topk_idx_dev, float* topk_w_dev, uint16_t* out_dev,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Block-FP8 routed experts, the other routed-expert format of the 512-expert model (FreeToken
 * commit log, 512-expert entry). The pages name the format without defining it; the reading
 * taken: one E4M3 (fn) byte per weight, one float32 scale per 128 x 128 tile of each weight
 * matrix (K, the reduction dimension, contiguous), no per-tensor scale, activations bf16.
 * All device pointers; codes 16-byte aligned, scales 4-byte aligned:
 *   w13  uint8 [E, 2I, H]   w13_scale float [E, 2I/128, H/128]
 *   w2   uint8 [E, H, I]    w2_scale  float [E, H/128, I/128]
 * element value = e4m3(code[r, c]) * scale[r / 128, c / 128]. H and I multiples of 128.
 */
typedef struct {
  int32_t E, H, I;
  const uint8_t* w13;
  const float* w13_scale;
  const uint8_t* w2;
  const float* w2_scale;
} ft_fp8block_experts;

/* Optional shared expert in block-FP8 (the same layouts without E) and its gate vector gv
 * (bf16 [H], 16-byte aligned): y_t += sigmoid(x_t . gv) * shared(x_t). */
typedef struct {
  const uint8_t* w13;
  const float* w13_scale;
  const uint8_t* w2;
  const float* w2_scale;
  const uint16_t* gate;
} ft_fp8block_shared_expert;

/* Workspace bytes of ft_moe_fp8block_decode for these sizes (0 when they are invalid). */
size_t ft_moe_fp8block_workspace_bytes(int32_t T, int32_t k, int32_t E, int32_t H, int32_t I,
                                       int32_t has_shared);

/*
 * ft_moe_fp8block_decode — the expert part of the layer for a decode batch (0 <= T <= 64)
 * with block-FP8 experts: y_t = sum_j topk_w[t,j] * W2_e (SwiGLU(W13_e x_t))
 * [+ sigmoid(x_t . gv) * shared(x_t)], the same layer as ft_moe_nvfp4_decode with the other
 * weight format. Arguments, routing slots, error flags (an id outside [0, E) or repeated in
 * a token raises FT_ERR_DEVICE_FLAG and that slot contributes nothing) and the workspace
 * rule (ft_moe_workspace_init once; calls sharing it ordered on one stream) as for
 * ft_moe_nvfp4_decode; workspace of ft_moe_fp8block_workspace_bytes bytes. Four kernels
 * (activations, W13 + SwiGLU, W2, ordered slot sum); deterministic.
 */
ft_status ft_moe_fp8block_decode(const uint16_t* x, int32_t T, const int32_t* topk_idx,
                                 const float* topk_w, int32_t k, const ft_fp8block_experts* ex,
                                 const ft_fp8block_shared_expert* sh, float swiglu_limit,
                                 uint16_t* out, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* Text of the last CUDA runtime error seen by this thread inside the library (the cause
 * behind an FT_ERR_CUDA); static storage, never NULL. */
const char* ft_moe_last_cuda_error(void);

/* Synchronise `stream`, read the workspace error word, clear it, and return FT_OK or the
 * first error flagged since the last call (FT_ERR_DEVICE_FLAG, FT_ERR_TIMEOUT). */
ft_status ft_moe_get_error(void* workspace, void* stream);

/* Test hook for the failure path; the pages have no counterpart. Sets, for this process,
 * how many times a decode kernel polls for the other CTAs' results (the grid barrier of
 * the several-token kernel, the slot-completion counters of the one-token kernel) before
 * it gives up: it then sets FT_ERR_TIMEOUT in the workspace error word, goes on with what
 * it has (the output is then undefined) and returns normally, and the workspace is left
 * ready for the next call. iterations < 0 restores the default bound (about a second of
 * waiting); 0 makes a wait give up at its first poll that finds the results incomplete.
 * Returns FT_OK. Not for production use: set it only while no decode call is being
 * enqueued by another thread. */
ft_status ft_moe_debug_set_wait_limit(int64_t iterations);

#ifdef __cplusplus
}
#endif

#endif /* FT_MOE_H */
