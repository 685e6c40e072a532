/*
 * libmoe — the mixture-of-experts FFN layer of a decoding LLM, with expert
 * weights in the GGUF IQ4_NL format, for one NVIDIA GB300 GPU (sm_103a).
 *
 * What the layer computes (per token t with activation x_t of H values):
 *   1. Router. s_e = W_r[e,:] . x_t for every routed expert e; p_e = sigmoid(s_e).
 *      The k experts with the largest p_e + b_e are chosen (ties: lower index);
 *      their combine weights are w_j = p_{e_j} / sum_i p_{e_i}. The bias b only
 *      selects. (PocketLLM page "Xing4.0-29B-A4B", Overview: a sigmoid-routed
 *      MoE with a shared expert, 64 experts activated top-4.)
 *   2. Experts. Each chosen expert and the always-on shared expert run a SwiGLU
 *      FFN: h = silu(W_g x) * (W_u x), o = W_d h.
 *   3. Combine. y_t = sum_j w_j o_{e_j}(x_t) + o_shared(x_t). The order of the
 *      sum is fixed (the page's "deterministic route reduction"): the shared
 *      expert first, then the routed experts in ascending id. It does not
 *      depend on the other tokens of the batch, so y_t is bit-identical
 *      whatever the batch (Red Lite, "What we learned", section 4: two requests
 *      in one pass give the answers of serving them in turn).
 *
 * IQ4_NL (GGML type 20; the Xing4.0 page's Overview table: "4.5 bits a weight,
 * 32 weights in 18 bytes"): a block is a little-endian fp16 scale d followed by
 * 16 bytes; the low nibble of byte j indexes weight j, the high nibble weight
 * j+16; weight = d * T[nibble] with the format's table
 * T = {-127,-104,-83,-65,-49,-35,-22,-10,1,13,25,38,53,69,89,113}.
 * A matrix with R rows and K inputs is R*K/32 consecutive blocks, row-major,
 * blocks along K (rows = output features), as GGUF stores it. Expert e of a
 * stacked tensor starts at block e*R*K/32.
 *
 * Conventions for every call below
 *  - Pointers are DEVICE pointers unless the comment says "host".
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). They allocate nothing, free nothing and never synchronise.
 *  - Arguments are checked on the host before any launch. A bad argument
 *    returns a negative moe_status and launches nothing ("refuse, don't
 *    ignore": the Xing4.0 page's option table refuses unsupported flags).
 *  - Kernels are launched with programmatic dependent launch: each kernel
 *    starts streaming constant weights while the previous kernel on the stream
 *    finishes, and waits for it before it reads any activation, route or
 *    workspace data. Work enqueued before a call must therefore not trigger
 *    programmatic completion (griddepcontrol.launch_dependents) before its
 *    outputs are written. moe_set_pdl(0) turns this off.
 *  - Nothing on the device traps. Device-side conditions are reported in the
 *    optional `status` word (device uint32, accumulated with atomicOr/atomicAdd,
 *    never cleared by libmoe): bits 0..15 count invalid routes (saturating),
 *    bit 31 (MOE_STATUS_TIMEOUT) means a bounded on-chip wait gave up.
 */
#ifndef LIBMOE_MOE_H
#define LIBMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* NULL pointer, size out of range, shape rule broken */
  MOE_ERR_UNSUPPORTED = -2,   /* valid for the format but not built here (see limits) */
  MOE_ERR_WORKSPACE = -3,     /* workspace NULL or smaller than moe_workspace_bytes() */
  MOE_ERR_MISALIGNED = -4,    /* a pointer breaks the alignment rule of its argument */
  MOE_ERR_CUDA = -5           /* a CUDA runtime call or launch failed */
} moe_status;

#define MOE_STATUS_INVALID_ROUTE_MASK 0x0000FFFFu
#define MOE_STATUS_TIMEOUT 0x80000000u

/* Limits of this build. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOP_K 16
#define MOE_MAX_DECODE_TOKENS 16
#define MOE_MAX_HIDDEN 8192
#define MOE_MAX_FFN 8192
#define MOE_MAX_LAYERS 128

/* Sizes of one MoE layer. hidden, ffn and ffn_shared are multiples of 64
 * (IQ4_NL needs 32; the kernels pair blocks) and at most 8192.
 * 1 <= n_experts <= 1024; 1 <= top_k <= min(n_experts, 16); n_shared is 0 or 1
 * (ffn_shared is ignored when n_shared == 0). */
typedef struct {
  int32_t hidden;      /* H */
  int32_t ffn;         /* F, width of each routed expert */
  int32_t ffn_shared;  /* Fs, width of the shared expert */
  int32_t n_experts;   /* E, routed experts */
  int32_t top_k;       /* k */
  int32_t n_shared;    /* 0 or 1 */
} moe_shape;

/* Expert weights of one layer, IQ4_NL, device memory, each pointer 16-byte
 * aligned (GGUF aligns tensor data to 32 bytes). Read only; libmoe streams
 * them while earlier work on the stream finishes, so they must not be written
 * by work still in flight when a call is enqueued.
 *   gate, up : [E][F][H/32] blocks     down : [E][H][F/32] blocks
 *   sh_gate, sh_up : [Fs][H/32]        sh_down : [H][Fs/32]  (NULL when n_shared == 0) */
typedef struct {
  const void* gate;
  const void* up;
  const void* down;
  const void* sh_gate;
  const void* sh_up;
  const void* sh_down;
} moe_expert_weights;

/* Router: scores, sigmoid, bias, top-k, renormalised weights.
 *   router_w : bf16 [E][H] (uint16 bit patterns), 16-byte aligned
 *   router_bias : fp32 [E] selection bias, or NULL for none
 *   x        : bf16 [T][H], 16-byte aligned
 *   T        : 0 <= T <= 1 << 20 (T == 0 launches nothing)
 *   ids      : out int32 [T][k], per token in descending p+b (ties: lower index)
 *   weights  : out fp32 [T][k], p_j / sum of the chosen p, same order
 * Scores accumulate in fp32 and the choice is made in fp32. No workspace. */
moe_status moe_route_topk(const moe_shape* shape, const uint16_t* router_w,
                          const float* router_bias, const uint16_t* x, int32_t T,
                          int32_t* ids, float* weights, void* stream);

/* Bytes of workspace that moe_iq4nl_decode (mode 0),
 * moe_iq4nl_prefill_grouped (mode 1) or moe_iq4nl_prefill_grouped_fp8
 * (mode 2) needs for up to max_tokens tokens.
 * Returns 0 for an invalid shape, mode or max_tokens. The workspace is
 * caller-owned device memory, 256-byte aligned, and MUST be zero-filled once
 * after allocation (cudaMemset); every call leaves its counter words at zero
 * again. One workspace serves any number of layers of the same shape run one
 * after another on one stream (the wpnews vLLM article's workspace sharing
 * keyed on shape). Calls that may overlap (other streams) need their own. */
size_t moe_workspace_bytes(const moe_shape* shape, int32_t max_tokens, int32_t mode);

/* Decode: the whole layer (experts + combine) for 1..16 tokens.
 *   x        : bf16 [T][H], 16-byte aligned
 *   ids      : int32 [T][k]; an id outside [0, E) is an invalid route: it is
 *              treated as expert 0 with weight 0 (wpnews vLLM article, route
 *              sanitising), i.e. it contributes nothing, and is counted in *status
 *   weights  : fp32 [T][k]
 *   y        : out fp32 [T][H], 16-byte aligned
 *   ws       : workspace of moe_workspace_bytes(shape, >= T, 0) bytes
 *   status   : device uint32 or NULL
 * Each distinct expert's weights are read once per call, whatever the number
 * of tokens routed to it; each IQ4_NL block is decoded once and used for every
 * such token. Arithmetic: fp32 accumulation of exact integer block dot
 * products; activations and h enter them as 16-bit integers with one power-of-
 * two scale per 32 values. */
moe_status moe_iq4nl_decode(const moe_shape* shape, const moe_expert_weights* w,
                            const uint16_t* x, int32_t T, const int32_t* ids,
                            const float* weights, float* y, void* ws, size_t ws_bytes,
                            uint32_t* status, void* stream);

/* Route + decode in one call: what moe_route_topk followed by moe_iq4nl_decode
 * computes, for 1..16 tokens, with the same outputs (ids, weights, y) and the
 * same arithmetic. For 1..4 tokens, at most 512 experts and hidden, ffn,
 * ffn_shared multiples of 256 it is a single persistent launch: the router runs
 * inside the layer kernel
 * (each CTA scores a slice of the experts, a grid-wide barrier, then every CTA
 * takes the top-k itself), which removes one kernel boundary per layer from the
 * critical path. The ids written here are always valid.
 *   router_w, router_bias, x: as for moe_route_topk;  w, y, ws, status: as for
 *   moe_iq4nl_decode;  ids, weights: out [T][k], as moe_route_topk writes them. */
moe_status moe_iq4nl_decode_routed(const moe_shape* shape, const uint16_t* router_w,
                                   const float* router_bias, const moe_expert_weights* w,
                                   const uint16_t* x, int32_t T, int32_t* ids, float* weights,
                                   float* y, void* ws, size_t ws_bytes, uint32_t* status,
                                   void* stream);

/* One layer's weights for moe_iq4nl_decode_layers: its experts and its router. */
typedef struct {
  moe_expert_weights experts;
  const uint16_t* router_w;     /* bf16 [E][H], 16-byte aligned */
  const float* router_bias;     /* fp32 [E] or NULL */
} moe_layer_weights;

/* Route + decode of n_layers consecutive MoE layers of one shape in one call:
 * for each layer l in order, what moe_iq4nl_decode_routed computes, with the
 * same arithmetic and the same outputs. The PocketLLM "Xing4.0-29B-A4B" page
 * (Performance) measures its decode step bound by kernel launches (11,536 a
 * step, 178 ms of host submission against 46.5 ms of device work); for 1..4
 * tokens, at most 512 experts and hidden, ffn, ffn_shared multiples of 256,
 * this call is ONE persistent launch over all the layers, with bounded
 * grid-wide waits between the phases of a layer and between layers (limit:
 * moe_set_barrier_wait_ns). Weights that do not depend on the routes (the
 * next layer's router rows and shared expert) are fetched a layer ahead.
 * Other sizes run layer by layer (router, then the layer), with the same
 * results.
 *   n_layers : 1..MOE_MAX_LAYERS
 *   layers   : HOST array [n_layers]; read during the call only (its pointers
 *              are copied into the launch); the device pointers it holds
 *              follow the rules of moe_expert_weights and moe_route_topk
 *   x        : bf16, 16-byte aligned: chained == 0: [n_layers][T][H], each
 *              layer's own input; chained == 1: [T][H], the first layer's
 *              input, layer l + 1's input then being bf16(y_l) (round to
 *              nearest even)
 *   ids, weights : out [n_layers][T][k], per layer as moe_route_topk writes them
 *   y        : out fp32 [n_layers][T][H], 16-byte aligned: every layer's output
 *   ws       : workspace of moe_workspace_bytes(shape, >= T, 0) bytes. Besides
 *              its counters, which return to zero, it keeps a call counter that
 *              tags the router scores of each call; zero-filling the whole
 *              workspace again is always allowed.
 *   status   : as for moe_iq4nl_decode
 * Layers run one after another in both modes (layer l + 1 starts once every
 * row of y_l is written). */
moe_status moe_iq4nl_decode_layers(const moe_shape* shape, int32_t n_layers,
                                   const moe_layer_weights* layers, const uint16_t* x,
                                   int32_t T, int32_t chained, int32_t* ids, float* weights,
                                   float* y, void* ws, size_t ws_bytes, uint32_t* status,
                                   void* stream);

/* Decode without a caller-provided workspace. This call has no counterpart on
 * the pages; it is a convenience of this library. It exists for callers that
 * cannot allocate device memory at the point where they run the layer: code
 * that runs while another component captures the stream into a CUDA graph
 * with its own memory pool, hosts that embed the library behind an allocator
 * they do not control, and runtimes that plan all device memory up front.
 *
 * It computes exactly what moe_iq4nl_decode computes (same arguments minus the
 * workspace, same outputs, same arithmetic), on a scratch area that is part of
 * the library: a fixed device array of MOE_STATIC_SCRATCH_BYTES (8 MiB) on
 * every GPU that loads the library, held until the process exits. It allocates
 * and frees nothing. A shape and token count whose
 * moe_workspace_bytes(shape, T, 0) exceeds that size is refused with
 * MOE_ERR_UNSUPPORTED (use moe_iq4nl_decode with your own workspace instead).
 *
 *  - Set-up: the first call on each device (with that device current) looks
 *    up the scratch's device address once (cudaGetSymbolAddress) and keeps it;
 *    a failure there returns MOE_ERR_CUDA. Make that first call before any
 *    stream capture begins.
 *  - Each call first clears the scratch's counter words on `stream` (a
 *    stream-ordered memset), then launches the decode kernels.
 *  - There is ONE scratch per device, shared by every caller in the process.
 *    Calls whose work may overlap on the GPU (other streams, other threads
 *    without ordering between their streams) race on it and give wrong
 *    results. Order them on one stream, or use moe_iq4nl_decode with a
 *    workspace each.
 *  - The kept address belongs to the device's current context. Do not call
 *    this function after cudaDeviceReset (or anything else that destroys that
 *    context) in the same process: the kept address is not looked up again
 *    and no longer names the scratch. Use moe_iq4nl_decode with a workspace
 *    in a process that resets its devices. */
#define MOE_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
moe_status moe_iq4nl_decode_static(const moe_shape* shape, const moe_expert_weights* w,
                                   const uint16_t* x, int32_t T, const int32_t* ids,
                                   const float* weights, float* y, uint32_t* status,
                                   void* stream);

/* Prefill: the whole layer for a chunk of 1..max_tokens tokens (at most 16384).
 * The Xolotl engine blog ("DeepSeek-V4.1-Flash at 27 Tokens/s on One RTX 4090",
 * section "Prompts: fast, and exact") runs a long prompt in chunks, streaming
 * each layer's experts once per chunk and running them as one batched multiply
 * on the tensor cores; this call is that step for one layer. Tokens are
 * bucketed by expert with a counting sort (no atomics decide any order), each
 * expert's tokens run as one grouped tensor-core contraction (tcgen05,
 * fp16 operands, fp32 accumulation) on weights dequantised on the fly, and a
 * gather-combine forms y in the fixed order above. Dequantised weights are
 * round-to-nearest-even fp16 of d*T[q]; x and h also enter as fp16.
 * Shape rule beyond moe_shape's: hidden, ffn and ffn_shared are multiples of
 * 128 (the contraction's 128-row weight tiles); other shapes are refused with
 * MOE_ERR_UNSUPPORTED and nothing is launched.
 * Arguments as for moe_iq4nl_decode; ws from moe_workspace_bytes(shape, >= T, 1). */
moe_status moe_iq4nl_prefill_grouped(const moe_shape* shape, const moe_expert_weights* w,
                                     const uint16_t* x, int32_t T, const int32_t* ids,
                                     const float* weights, float* y, void* ws,
                                     size_t ws_bytes, uint32_t* status, void* stream);

/* Prefill with 8-bit operands: the same step as moe_iq4nl_prefill_grouped on
 * 8-bit tensor cores (tcgen05 kind::f8f6f4, fp32 accumulation). The Xolotl
 * engine blog ("Prompts: fast, and exact") runs its prompt contraction on the
 * 4090's int8 tensor cores; on this GPU the 8-bit tensor format with a fast
 * rate is floating point, so the operands here are OCP E4M3 codes (bias 7,
 * largest finite 448), rounded to nearest even with finite overflow saturated:
 *   weights : row r of a matrix is scaled by 2^-E_r before rounding, E_r the
 *             largest floor(log2 d) over the row's block scales d (-14 for a
 *             zero or subnormal d), so w8 = 2^E_r e4m3(d T[q] 2^-E_r);
 *   x       : each token's row is scaled by 2^-X, X = floor(log2 max|x|) - 6
 *             (0 for an all-zero row), so its largest value lies in [64, 128);
 *   h       : each (token, expert) row of SwiGLU outputs the same way, from
 *             the row's fp32 h.
 * The fp32 accumulators are multiplied back by the powers of two: the weight
 * row's and x's in the contractions' epilogues, h's through the combine weight
 * (w 2^X, the same product while w 2^X is a normal fp32); the combine order is
 * that of moe_iq4nl_prefill_grouped. The result differs from the fp16-operand
 * call by the E4M3 rounding (about 2^-4 relative per operand). Inside each
 * 32-value block both operands keep K in the order of the IQ4_NL index bytes
 * (values j and j + 16 side by side); the sums do not depend on it.
 *   row_exp : device int8, the table moe_iq4nl_fp8_row_exponents wrote for
 *             these weights (it depends on the weights only: make it once).
 * Shape rule: hidden, ffn and ffn_shared are multiples of 256 (the operand
 * ring carries 256 weights of a row per copy); other shapes are refused with
 * MOE_ERR_UNSUPPORTED. ws from moe_workspace_bytes(shape, >= T, 2); the other
 * arguments as for moe_iq4nl_prefill_grouped. */
moe_status moe_iq4nl_prefill_grouped_fp8(const moe_shape* shape, const moe_expert_weights* w,
                                         const int8_t* row_exp, const uint16_t* x, int32_t T,
                                         const int32_t* ids, const float* weights, float* y,
                                         void* ws, size_t ws_bytes, uint32_t* status,
                                         void* stream);

/* Entries (int8, one per weight row) of the row-exponent table of a shape:
 * E*ffn (gate) + E*ffn (up) + E*hidden (down) and, with a shared expert,
 * ffn_shared (gate) + ffn_shared (up) + hidden (down), in that order. 0 for an
 * invalid shape. */
int64_t moe_fp8_row_exponent_count(const moe_shape* shape);

/* Write the row-exponent table (E_r above, in the order above) of a layer's
 * weights to row_exp (device, moe_fp8_row_exponent_count bytes). */
moe_status moe_iq4nl_fp8_row_exponents(const moe_shape* shape, const moe_expert_weights* w,
                                       int8_t* row_exp, void* stream);

/* The E4M3 weight decoder of moe_iq4nl_prefill_grouped_fp8 on its own, so
 * that it can be checked bit for bit: rows x K weights (K a multiple of 32;
 * rows of K/32 IQ4_NL blocks, 18 bytes each, packed) to row_exp[rows] (E_r as
 * above) and out[rows][K], the E4M3 code of d T[q] 2^-E_r for each weight, both
 * through the device functions the fp8 prefill runs.
 *   mat : device, 2-byte aligned   row_exp : device   out : device, 4-byte aligned */
moe_status moe_iq4nl_dequantize_e4m3(const void* mat, int64_t rows, int32_t K, int8_t* row_exp,
                                     uint8_t* out, void* stream);

/* Dequantise n_blocks consecutive IQ4_NL blocks (the block layout above),
 * through one of the block decoders the layer kernels use, so that each can be
 * checked bit for bit against the format's definition:
 *   MOE_DEQUANT_FP32           fp32 [n_blocks*32], the exact product d*T[q], through
 *                              the table lookup of the decode dot products for an
 *                              expert with several tokens;
 *   MOE_DEQUANT_FP16           fp16 [n_blocks*32], round-to-nearest-even of d*T[q],
 *                              through the decoder of the prefill contraction;
 *   MOE_DEQUANT_FP32_ONE_TOKEN fp32 [n_blocks*32], the exact product d*T[q], through
 *                              the split-table dot product of the decode path for
 *                              an expert with one token.
 *   blocks : device, 2-byte aligned        out : device, 4-byte aligned
 * Any other mode is refused with MOE_ERR_INVALID_ARG. */
#define MOE_DEQUANT_FP32 0
#define MOE_DEQUANT_FP16 1
#define MOE_DEQUANT_FP32_ONE_TOKEN 2
moe_status moe_iq4nl_dequantize(const void* blocks, int64_t n_blocks, int32_t mode,
                                void* out, void* stream);

/* The invalid-route rule on its own (wpnews vLLM article, route sanitising):
 * ids_out[i] = ids[i] if 0 <= ids[i] < n_experts else 0; weights_out[i] =
 * weights[i] if the id is valid else 0. Invalid routes are counted in *status.
 * In-place use (ids_out == ids, weights_out == weights) is allowed. */
moe_status moe_sanitize_routes(const int32_t* ids, const float* weights, int64_t n,
                               int32_t n_experts, int32_t* ids_out, float* weights_out,
                               uint32_t* status, void* stream);

/* Kernel launches one call makes for this shape and token count (host, no
 * device work): call 0 = moe_route_topk, 1 = moe_iq4nl_decode,
 * 2 = moe_iq4nl_decode_routed, 3 = moe_iq4nl_prefill_grouped,
 * 5 = moe_iq4nl_prefill_grouped_fp8, and
 * 4 + 2*n_layers + chained = moe_iq4nl_decode_layers of n_layers layers
 * (chained 0 or 1). Returns a negative moe_status for bad arguments. */
int32_t moe_launches_per_call(const moe_shape* shape, int32_t T, int32_t call);

/* 1 (default) launches kernels with programmatic dependent launch; 0 does not.
 * Host-side, process-wide. Returns the previous setting. */
int32_t moe_set_pdl(int32_t enable);

/* Limit, in nanoseconds, of a CTA's waits on the other CTAs of its grid: the
 * grid-wide barriers of the single-launch decode kernels (a CTA waits there
 * until every CTA has published its router scores, or its rows of h). Those
 * kernels launch one CTA per SM and check before launching that a CTA fits on
 * an SM (an occupancy query; otherwise the multi-kernel path runs), but a
 * device shared with other work (MPS, partitioned SMs) can still keep some
 * CTAs from starting; the limit bounds that wait instead of hanging the GPU.
 * A wait that reaches it gives up and sets MOE_STATUS_TIMEOUT in *status; the
 * call's outputs are then undefined, the kernel still waits for its own copies
 * in flight (on the fixed 2 s limit of waits on copies, not on this one) and
 * leaves the workspace ready for the next call. 0 makes a CTA give up the
 * first time it finds a barrier incomplete (a way for tests to take the
 * timeout path without a fault). Host-side, process-wide, read at each call;
 * the default is 2e9 (2 s). Returns the previous limit. */
uint64_t moe_set_barrier_wait_ns(uint64_t ns);

/* A static description of a status code (host). */
const char* moe_status_string(int32_t status);

/* Library version, e.g. "libmoe 0.1 sm_103a" (host, static string). */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBMOE_MOE_H */
