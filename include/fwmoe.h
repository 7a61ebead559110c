/*
 * fwmoe — the routed mixture-of-experts feed-forward step over Q8_0 weights,
 * on one NVIDIA GB300 (sm_103a). C ABI.
 *
 * The step (the Flyweight README, "flyweight-llm" 0.2.0, §Features: "sparse
 * MoE execution"; §Quantization: grouped routed-expert GPU kernels for Q8_0
 * among other formats; the pages print no formula, and the reading used here
 * is the standard top-k softmax router):
 *
 *   z[t,e]   = sum_h x[t,h] * router_w[e,h] + router_bias[e]        (fp32)
 *   ids[t,:] = the k largest z[t,.]; ties go to the lower expert id; ordered
 *              by descending z (equal z: lower id first)
 *   gates    = softmax of z[t,.] restricted to ids[t,:], renormalised to sum 1
 *   y_e(x)   = W_down,e ( SiLU(W_gate,e x) * (W_up,e x) ),  SiLU(a) = a/(1+e^-a)
 *   out[t]   = sum_j gates[t,j] * y_{ids[t,j]}(x_t)  (+ y_shared(x_t), weight 1)
 *
 * There is no residual add: out is the MoE output only.
 *
 * Q8_0 weight layout accepted by fw_moe_init (GGUF convention; the pages name
 * the format, §Quantization): each matrix row is cut along its input dimension
 * into blocks of 32 values, each block 34 bytes: a little-endian IEEE binary16
 * scale d, then 32 int8 codes q; the weight is d*q. Expert matrices are stored
 * back to back, expert-major: w_gate / w_up are E x [I rows x H/32 blocks],
 * w_down is E x [H rows x I/32 blocks].
 *
 * Conventions for every call:
 *  - Pointers named "device" are CUDA device pointers owned by the caller.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls enqueue
 *    asynchronously; none synchronises except fw_moe_init, fw_moe_free,
 *    fw_moe_status and fw_moe_forward_host.
 *  - Argument errors are reported before anything is enqueued. A failed call
 *    returns a negative fw_status and fw_moe_last_error() describes it.
 *  - There is no CPU fallback: without an sm_103 device, fw_moe_init fails
 *    with FW_EUNSUPPORTED.
 */
#ifndef FWMOE_H
#define FWMOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FW_OK = 0,
  FW_EINVAL = -1,       /* bad argument (null pointer, size, alignment) */
  FW_ENOMEM = -2,       /* device allocation failed */
  FW_ECUDA = -3,        /* a CUDA call or launch failed */
  FW_EUNSUPPORTED = -4, /* no sm_103 device, or a shape this build does not handle */
  FW_ESTATE = -5,       /* call order broken (e.g. ffn with a T other than the last route's) */
  FW_ETIMEOUT = -6,     /* a kernel gave up a bounded wait (see fw_moe_status) */
  FW_EDEVICE = -7       /* a kernel reported a failed index or layout check */
} fw_status;

typedef struct fw_moe_handle fw_moe_handle; /* opaque; one handle = one MoE layer */

/* Layer shape. H and I must be multiples of 64, not only of the Q8_0 block
 * length 32: the prefill GEMMs step K by 64 (two Q8_0 blocks per 128-byte
 * swizzled shared-memory row). Every Qwen/DeepSeek-shaped MoE layer the pages
 * speak of meets this. */
typedef struct {
  int32_t H;            /* hidden size; multiple of 64 */
  int32_t I;            /* per-expert intermediate size; multiple of 64 */
  int32_t E;            /* routed experts, 1..256 */
  int32_t k;            /* experts per token, 1..min(E, 16) */
  int32_t n_shared;     /* always-on shared experts: 0 or 1 */
  int32_t T_max;        /* largest T any call on this handle may pass (sizes the workspace) */
  int32_t decode_T_max; /* T <= this takes the decode (grouped GEMV) path; 0 = 16; at most 16.
                         * The decode kernel holds a call's x in shared memory: one token
                         * up to H = 14336, several up to H = 2048; calls past that take
                         * the prefill path whatever their T. */
  int32_t act_q8;       /* 0: bf16 activations (the default step). 1: Q8 activations on the
                         * decode path (the Flyweight README, §Quantization: Q8-activation
                         * dp4a decode kernels): each token's x quantised per 32-block and
                         * each expert's h = SiLU(g)*u per 16-block by the Q8_0 rule in fp32
                         * (d = amax/127, codes round-half-away(v/d)), integer dot products
                         * with the Q8_0 weights, scales applied per block. The prefill path
                         * keeps bf16 activations (sm_103a has no int8 tensor-core MMA). */
} fw_moe_config;

typedef struct { /* all DEVICE pointers, read only during fw_moe_init */
  const float *router_w;       /* [E, H] fp32 row-major */
  const float *router_bias;    /* [E] fp32 or NULL; added to the logits (selection and gates) */
  const uint8_t *w_gate;       /* E x [I x H/32] Q8_0 blocks */
  const uint8_t *w_up;         /* E x [I x H/32] Q8_0 blocks */
  const uint8_t *w_down;       /* E x [H x I/32] Q8_0 blocks */
  const uint8_t *shared_gate;  /* [I x H/32] Q8_0, or NULL when n_shared == 0 */
  const uint8_t *shared_up;    /* [I x H/32] Q8_0, or NULL when n_shared == 0 */
  const uint8_t *shared_down;  /* [H x I/32] Q8_0, or NULL when n_shared == 0 */
} fw_moe_weights;

/* Create a layer (the pages' runtime loads routed experts of GGUF Q8_0 models
 * onto the GPU for its grouped kernels: Flyweight README, §Quantization and
 * §Features): validates the shapes, copies the router and repacks every
 * Q8_0 matrix into the handle's own device memory (a byte-preserving change of
 * layout: int8 code planes plus binary16 scale planes), allocates the
 * workspace for T_max tokens and synchronises `stream` once. The caller may
 * free its weight buffers afterwards. *out receives the handle. */
fw_status fw_moe_init(const fw_moe_config *cfg, const fw_moe_weights *w, void *stream, fw_moe_handle **out);

/* The router step (Flyweight README, §Current limitations: dynamic MoE routing;
 * vOOM README, router/top-k substeps; the reading: fp32 logits, top-k with ties
 * to the lower id, softmax restricted to the k and renormalised).
 * Routing for T tokens (0 <= T <= T_max): x is DEVICE bf16 [T, H] row-major.
 * Writes expert_ids (DEVICE int32 [T, k]) and gates (DEVICE fp32 [T, k], may be
 * NULL), and keeps the routing and the token-to-expert grouping in the handle
 * for the next fw_moe_ffn. T == 0 is a no-op. */
fw_status fw_moe_route(fw_moe_handle *h, const void *x, int32_t T, int32_t *expert_ids, float *gates,
                       void *stream);

/* The routed-expert step (Flyweight README, §Features "sparse MoE execution",
 * §Quantization: grouped routed-expert kernels over Q8_0; vOOM README: SwiGLU
 * experts, shared experts): each selected expert's SiLU(gate) * up then down
 * projection, gate-weighted and summed in slot order (+ the shared expert).
 * Experts and combine for the routing made by the last fw_moe_route on this
 * handle: same x, same T, same stream. out is DEVICE bf16 [T, H] row-major.
 * A T different from the last route's returns FW_ESTATE. */
fw_status fw_moe_ffn(fw_moe_handle *h, const void *x, int32_t T, void *out, void *stream);

/* fw_moe_route followed by fw_moe_ffn (expert_ids may not be NULL; gates may). */
fw_status fw_moe_forward(fw_moe_handle *h, const void *x, int32_t T, int32_t *expert_ids, float *gates, void *out,
                         void *stream);

/* The whole step from and to HOST memory: copies x (bf16 [T, H]) to the device,
 * runs fw_moe_forward on the handle's own device buffers, copies expert_ids
 * (int32 [T, k]) and out (bf16 [T, H]) back and synchronises `stream`. Host
 * buffers should be pinned for the copies to be asynchronous. */
fw_status fw_moe_forward_host(fw_moe_handle *h, const void *x_host, int32_t T, int32_t *expert_ids_host,
                              void *out_host, void *stream);

/* The token-to-expert permutation the grouped kernels run on (Flyweight
 * README, §Runtime controls: block-table kernels for routed experts).
 * Token-to-expert grouping of the last route (for tests and tools): offsets
 * DEVICE int32 [E + 1], the exclusive prefix sum of the per-expert counts;
 * perm DEVICE int32 [T*k], the slot ids s = t*k + j grouped by ascending expert
 * and, within an expert, by ascending token; inv DEVICE int32 [T*k] (may be
 * NULL), inv[perm[p]] = p. */
fw_status fw_moe_get_permutation(fw_moe_handle *h, int32_t *offsets, int32_t *perm, int32_t *inv, void *stream);

/* Copy one repacked matrix of one expert back out in the GGUF Q8_0 layout
 * (which: 0 gate, 1 up, 2 down; expert E is the shared expert). blocks is
 * DEVICE memory of rows x K/32 x 34 bytes. Round-trips fw_moe_init's input. */
fw_status fw_moe_export_q8_0(fw_moe_handle *h, int32_t expert, int32_t which, uint8_t *blocks, void *stream);

/* A chain of layer calls captured once as one CUDA graph and replayed by a
 * single launch (Flyweight README, §Current limitations: host
 * synchronisation points of dynamic MoE routing, persistent layer kernels
 * listed as incomplete; §Features: CUDA-graph replay of decode). No call of
 * fw_moe_forward synchronises with the host -- routing, grouping and tile
 * lists stay on the device for both paths -- so n of them capture into one
 * graph. Call i runs fw_moe_forward(layers[i], x[i], T, expert_ids[i], NULL,
 * out[i]): x[i] and out[i] DEVICE bf16 [T, H_i], 16-byte aligned (out[i] may be
 * x[i + 1], chaining the layers); expert_ids[i] DEVICE int32 [T, k_i]. The
 * handles, T and every pointer are fixed at capture; the buffers' contents
 * are read at each launch. Capture runs on a stream of its own on the current
 * device, which must be every layer's. Replays of one graph, and other work
 * on its layers, must not overlap (they share each handle's workspace).
 * Errors: FW_EINVAL for arguments (before any CUDA call), FW_ESTATE if a layer
 * is profiling, else what a capture or instantiation reports. */
typedef struct fw_moe_graph fw_moe_graph;
fw_status fw_moe_graph_create(fw_moe_handle *const *layers, int32_t n, int32_t T, const void *const *x,
                              void *const *out, int32_t *const *expert_ids, fw_moe_graph **graph);
/* Enqueue one replay of the chain on `stream`. */
fw_status fw_moe_graph_launch(fw_moe_graph *graph, void *stream);
/* Release the graph (not its layers). NULL is a no-op. */
fw_status fw_moe_graph_destroy(fw_moe_graph *graph);

/* Synchronise `stream`, read and clear the handle's device status word.
 * FW_OK, FW_ETIMEOUT or FW_EDEVICE. */
fw_status fw_moe_status(fw_moe_handle *h, void *stream);

/* Kernel kinds reported by fw_moe_profile_end. */
enum {
  FW_KERNEL_ROUTE_DECODE = 0, /* decode router: GEMV, top-k, gates, grouping */
  FW_KERNEL_ROUTE_TILES = 1,  /* prefill router: tiled GEMM, top-k, per-tile counts */
  FW_KERNEL_ROUTE_SCAN = 2,   /* prefill grouping: offsets, tile lists */
  FW_KERNEL_ROUTE_SCATTER = 3,/* prefill grouping: stable scatter */
  FW_KERNEL_DECODE_EXPERTS = 4, /* decode experts: gate/up GEMV + SiLU, grid barrier, down GEMV + combine */
  FW_KERNEL_RESERVED_5 = 5,
  FW_KERNEL_PREFILL_GATEUP = 6,  /* prefill gate/up grouped GEMM (tcgen05) + SiLU */
  FW_KERNEL_PREFILL_DOWN = 7,    /* prefill down grouped GEMM (tcgen05) x gate */
  FW_KERNEL_PREFILL_COMBINE = 8, /* prefill un-permute and sum */
  FW_KERNEL_PREFILL_GATHER = 9, /* prefill: x rows gathered into grouped order */
  FW_KERNEL_PREFILL_GATEUP_SMALL = 10, /* prefill gate/up GEMM over the tiles of at most 64 rows */
  FW_KERNEL_PREFILL_DOWN_SMALL = 11,   /* prefill down GEMM over the tiles of at most 64 rows */
  FW_KERNEL_PREFILL_GATEUP_MID = 12,   /* prefill gate/up GEMM over the tiles of 65 to 96 rows */
  FW_KERNEL_PREFILL_DOWN_MID = 13,     /* prefill down GEMM over the tiles of 65 to 96 rows */
  FW_KERNEL_KINDS = 16
};

/* Optional per-kernel timing, for measurement tools. After
 * fw_moe_profile_begin, every kernel this handle launches (up to max_launches)
 * is bracketed by CUDA events recorded on its own stream; this serialises the
 * kernels (no programmatic overlap), so profile in a pass of its own.
 * fw_moe_profile_end synchronises, writes per kind (arrays of n_kinds, at most
 * FW_KERNEL_KINDS) the summed milliseconds and the launch count, and stops
 * recording. Creating the events happens in begin, not on the launch path. */
fw_status fw_moe_profile_begin(fw_moe_handle *h, int32_t max_launches);
fw_status fw_moe_profile_end(fw_moe_handle *h, int32_t n_kinds, float *total_ms, int32_t *launches);

/* Release the handle (no counterpart on the pages: resource management of
 * this library). Synchronises its device first. NULL is a no-op; a
 * handle already freed is detected (FW_EINVAL) as long as its memory has not
 * been reused. */
fw_status fw_moe_free(fw_moe_handle *h);

/* Text of the last failed call on this thread ("" if none). No counterpart
 * on the pages. */
const char *fw_moe_last_error(void);

/* Routing only (logits, top-k with ties to the lower id, renormalised gates)
 * for callers that must not allocate device memory: code that runs inside a
 * framework whose memory manager owns every byte of the device (a serving
 * engine's pool or a fixed arena), or on a latency path where cudaMalloc's
 * implicit synchronisation is not acceptable. It needs no handle: x is DEVICE
 * bf16 [T, H], router_w DEVICE fp32 [E, H] (16-byte aligned), router_bias
 * DEVICE fp32 [E] or NULL; writes expert_ids DEVICE int32 [T, k] and gates
 * DEVICE fp32 [T, k] (may be NULL), the same values fw_moe_route writes.
 * The pages have no counterpart: this is a convenience of this library.
 *
 * Its only scratch (the T x E logits and a ticket counter, 16.25 KiB) is a
 * file-scope __device__ array that every GPU loading this library holds until
 * process exit; limits: T <= 16, E <= 256, k <= min(E, 16), H % 4 == 0, beyond
 * which it returns FW_EINVAL with text. The first call on a device looks the
 * array's device address up (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture. Each call clears
 * the ticket in stream order. All calls share the one array and it keeps the
 * last call's contents: calls that can overlap on the GPU (other streams, or
 * other threads' streams) race and must be serialised by the caller. It calls
 * no cudaMalloc, cudaFree or allocating library routine. `stream` must belong
 * to the current device (checked: FW_EINVAL otherwise); the looked-up address
 * is kept for the life of the process, so after a cudaDeviceReset of the
 * device this entry point (like every handle) may no longer be used. */
fw_status fw_moe_route_noalloc(const void *x, int32_t T, int32_t H, const float *router_w, const float *router_bias,
                               int32_t E, int32_t k, int32_t *expert_ids, float *gates, void *stream);

/* A tool for preparing inputs, not a step of the MoE layer (the pages name
 * the GGUF Q8_0 format, Flyweight README §Quantization; the layer itself
 * never quantises). Quantise fp32 weights to Q8_0 on the GPU: w DEVICE [rows, K] row-major fp32,
 * K % 32 == 0; blocks DEVICE rows x K/32 x 34 bytes. Per block of 32:
 * amax = max|w|, d = amax/127 (fp64), q = round-half-away-from-zero(w/d)
 * clamped to +-127 (fp64), d stored as binary16 (round to nearest even);
 * an all-zero block stores zeros. */
fw_status fw_q8_0_quantize(const float *w, int64_t rows, int64_t K, uint8_t *blocks, void *stream);

#ifdef __cplusplus
}
#endif
#endif
