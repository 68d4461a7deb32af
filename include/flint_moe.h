/*
 * flint_moe — one Flint-shaped sparse mixture-of-experts layer on an sm_103a GPU (B300).
 *
 * The layer (Recursive Flint serving-kit post, section "The architecture, from the config";
 * news article "Recursive opens Flint, a 40B coding model with 2.5B active", section "What
 * runs on each token"): hidden size 2048; 256 routed experts, 6 chosen per token by sigmoid
 * router scores normalised over the chosen set ("normalized top-k, not softmax routing");
 * routed expert width 512; one shared expert of width 1024 that runs on every token.
 * Readings taken where the pages are silent: every expert is a SwiGLU MLP
 * E(x) = (silu(x Wg) * (x Wu)) Wd; an optional per-expert router bias is added to the logit
 * before the sigmoid and counts for both selection and gates; ties in score go to the lower
 * expert index; y = shared(x) + sum_j g_j E_{e_j}(x).
 *
 * Conventions for every call below:
 *   - All tensor pointers are caller-owned DEVICE memory unless the name ends in _host.
 *     The library never copies, repacks or frees them; weights are borrowed for the
 *     lifetime of the handle.
 *   - bf16 tensors are passed as `const void*` (IEEE bfloat16, row-major, densely packed,
 *     16-byte aligned base).  Matrices use the math orientation y = x W.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  route / forward make no host synchronisation and no allocation, so
 *     flint_moe_forward and flint_moe_stack_forward can be captured in a CUDA graph and
 *     replayed (each call leaves the workspace's counters at zero).
 *   - Argument errors are returned synchronously and nothing is enqueued.
 *   - Errors detected on the device (a bounded wait that ran out, an index out of range)
 *     are recorded in a status word inside the workspace; they are sticky until read by
 *     flint_moe_poll_device_status.
 *   - A handle may be used from one stream at a time.  Results are bitwise deterministic
 *     for identical inputs (no floating-point atomics).  Several handles (e.g. the layers of
 *     a stack) may share one workspace when all their calls are ordered on one stream: the
 *     workspace holds only per-call scratch, and its counters return to zero at the end of
 *     every call.
 *   - T <= 256 runs the decode-size path (one persistent cooperative kernel); larger T runs
 *     the tensor-core path (five kernels).  Pre-norm adds one RMSNorm kernel to either.
 *   - The only supported shape is the Flint layer's (hidden 2048, 256 experts, top-6,
 *     widths 512 / 1024); any other returns FLINT_MOE_ERR_UNSUPPORTED, as does a device
 *     that is not compute capability 10.3 (the serving kit likewise refuses configurations
 *     it cannot run correctly rather than degrade: serving-kit post, section "What isn't
 *     validated, and what the kit refuses to do").
 */
#ifndef FLINT_MOE_H
#define FLINT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct flint_moe_s* flint_moe_t;
typedef struct CUstream_st* flint_stream_t; /* identical to cudaStream_t */

typedef enum {
  FLINT_MOE_OK = 0,
  FLINT_MOE_ERR_INVALID_ARG = 1,    /* NULL / misaligned pointer, T out of range, ...   */
  FLINT_MOE_ERR_UNSUPPORTED = 2,    /* shape, flags or device not supported              */
  FLINT_MOE_ERR_WORKSPACE = 3,      /* workspace missing, misaligned or too small        */
  FLINT_MOE_ERR_CUDA = 4,           /* a CUDA runtime call failed                         */
  FLINT_MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait ran out                 */
  FLINT_MOE_ERR_DEVICE_BOUNDS = 6   /* a device-side index check failed                   */
} flint_moe_status;

/* config.flags */
#define FLINT_MOE_FLAG_PRE_RMSNORM 0x1u /* route and run the experts on r = x / rms(x)     */
#define FLINT_MOE_FLAG_RESIDUAL 0x2u    /* y = x + MoE(...) (y may alias x)                 */
/* For tests of the device-timeout path only: every route / forward call makes one bounded device
 * wait on a workspace word that nothing writes.  The wait gives up after 0.25 s (a quarter of
 * the 1 s limit of every other device wait, so the call's results are unaffected) and records
 * the timeout: flint_moe_poll_device_status then returns FLINT_MOE_ERR_DEVICE_TIMEOUT, and the
 * context stays usable.  It is not part of the method. */
#define FLINT_MOE_FLAG_TEST_WAIT_TIMEOUT 0x80000000u

typedef struct {
  int hidden;       /* must be 2048 */
  int n_experts;    /* must be 256 */
  int top_k;        /* must be 6 */
  int expert_inter; /* must be 512 */
  int shared_inter; /* must be 1024 */
  int max_tokens;   /* largest T any call on this handle will pass; 1..65536 */
  unsigned flags;   /* FLINT_MOE_FLAG_* */
  float rms_eps;    /* RMSNorm epsilon (used with FLINT_MOE_FLAG_PRE_RMSNORM), > 0 */
} flint_moe_config;

typedef struct {
  const void* w_router;     /* bf16 [hidden][n_experts]                            */
  const float* router_bias; /* fp32 [n_experts], or NULL for no bias                */
  const void* w_gate;       /* bf16 [n_experts][hidden][expert_inter]              */
  const void* w_up;         /* bf16 [n_experts][hidden][expert_inter]              */
  const void* w_down;       /* bf16 [n_experts][expert_inter][hidden]              */
  const void* ws_gate;      /* bf16 [hidden][shared_inter]                         */
  const void* ws_up;        /* bf16 [hidden][shared_inter]                         */
  const void* ws_down;      /* bf16 [shared_inter][hidden]                         */
} flint_moe_weights;

/* Human-readable name of a status code (static string, never NULL). */
const char* flint_moe_status_string(flint_moe_status s);

/* Bytes of device workspace a handle created with `cfg` needs (written to *bytes).
 * The caller allocates it (256-byte aligned) and keeps it alive until flint_moe_destroy. */
flint_moe_status flint_moe_workspace_bytes(const flint_moe_config* cfg, size_t* bytes);

/* Validates the configuration, the device (compute capability 10.3), pointer alignment
 * (16 bytes) and the workspace size; builds the TMA descriptors of the weights; zeroes
 * the workspace's counters and status word (a synchronous cudaMemset on the current
 * device).  On success *out receives a handle owning only host-side state. */
flint_moe_status flint_moe_create(const flint_moe_config* cfg, const flint_moe_weights* w,
                                  void* workspace, size_t workspace_bytes, flint_moe_t* out);

/* Router scoring, normalised top-k and the expert permutation only (serving-kit post, section
 * "The architecture, from the config": sigmoid router scoring with normalised top-k, 6 of 256
 * routed experts per token; the per-expert counts and the expert-sorted order are this
 * library's layout of the routed work).
 *   x        bf16 [T][hidden] (the layer input; with PRE_RMSNORM the routing uses rms(x))
 *   topk_idx int32 [T][top_k]: chosen experts, score descending, lower index first on ties
 *   topk_w   fp32 [T][top_k]: their normalised gates
 *   counts   int32 [n_experts] tokens per expert, or NULL
 * 1 <= T <= max_tokens. */
flint_moe_status flint_moe_route(flint_moe_t h, const void* x, int T, int32_t* topk_idx,
                                 float* topk_w, int32_t* counts, flint_stream_t stream);

/* The whole layer (serving-kit post, section "The architecture, from the config"; news article
 * "Recursive opens Flint, a 40B coding model with 2.5B active", section "What runs on each
 * token": the six chosen experts of width 512 plus one always-on shared expert of width 1024):
 * y bf16 [T][hidden] = shared(x') + sum_j g_j E_{e_j}(x') with x' = x, or
 * rms(x) under PRE_RMSNORM; plus x under RESIDUAL (then y may alias x).  topk_idx / topk_w
 * (same layout as flint_moe_route) receive the routing when not NULL.  1 <= T <= max_tokens. */
flint_moe_status flint_moe_forward(flint_moe_t h, const void* x, int T, void* y,
                                   int32_t* topk_idx, float* topk_w, flint_stream_t stream);

/* flint_moe_forward on HOST buffers: x_host and y_host are host memory (pinned for
 * asynchronous copies; pageable works but the copies then synchronise).  The input is
 * copied into the workspace, the layer runs, the output is copied back, all on `stream`;
 * the call returns once the work is enqueued (synchronise `stream` before reading y_host). */
flint_moe_status flint_moe_forward_host(flint_moe_t h, const void* x_host, int T, void* y_host,
                                        flint_stream_t stream);

/* Synchronises `stream`, then returns and clears the device status word
 * (FLINT_MOE_OK, FLINT_MOE_ERR_DEVICE_TIMEOUT or FLINT_MOE_ERR_DEVICE_BOUNDS). */
flint_moe_status flint_moe_poll_device_status(flint_moe_t h, flint_stream_t stream);

/* Profiling.  enable = 1: later forward calls record a CUDA event pair around every kernel
 * they launch (this serialises kernels that would otherwise overlap); flint_moe_kernel_times
 * synchronises on the last call's events and writes up to `cap` entries: names[i] (static
 * strings) and ms[i]; *n receives the count.  enable = 2: 24 slots per CTA in the workspace
 * record a trace -- at T <= 256 the decode-size kernel's GPU global timer stamps (ns) at its
 * phase boundaries; at T > 256 the wait profiles of the routed gate/up (slots 0-7), down (8-15)
 * and router (16-23) GEMMs: SM cycles the producer, the MMA issuer and the epilogue waited, the
 * global timer at start and end, tiles processed.  flint_moe_read_trace synchronises the device
 * and copies up to `cap` values (CTA-major) to host memory `out`.  enable = 0 turns both off. */
flint_moe_status flint_moe_enable_kernel_timing(flint_moe_t h, int enable);
flint_moe_status flint_moe_kernel_times(flint_moe_t h, const char** names, float* ms, int cap,
                                        int* n);
flint_moe_status flint_moe_read_trace(flint_moe_t h, unsigned long long* out, int cap, int* n);

/* Releases the handle's host state.  Does not touch the workspace or the weights. */
flint_moe_status flint_moe_destroy(flint_moe_t h);

/* ---------------------------------------------------------------- NVFP4 expert weights
 * The pages' four-bit builds (news article "Recursive opens Flint, a 40B coding model with 2.5B
 * active", section "Built with the Eureka Machine": the NVFP4 model; serving-kit post, section
 * "What isn't validated, and what the kit refuses to do": the quantized builds run on other
 * engines).  NVFP4, by the format's published definition: each weight is an FP4 E2M1 code, every
 * 16 consecutive weights along the contraction dimension share one FP8 E4M3 scale, and each
 * matrix has one fp32 tensor scale: w = e2m1 * e4m3 * tensor_scale.  Layouts (device memory,
 * 16-byte aligned), K-major, for a matrix W [K][N] of the math orientation y = x W (K the
 * contraction dimension):
 *   codes  uint8 [N][K/2]: byte (n, j) holds W[2j][n] in its low nibble, W[2j+1][n] in its high;
 *   scales uint8 [N][K/16]: E4M3 bits of the scale of W[16g .. 16g+15][n].
 * The routed experts' matrices are stacked as in flint_moe_weights, with one tensor scale per
 * expert and matrix (device fp32 arrays); the router stays bf16.  A handle made by
 * flint_moe_create_nvfp4 is used with flint_moe_route / flint_moe_forward / flint_moe_destroy
 * and the other per-handle calls; it runs the decode-size kernel, streaming the codes and scales
 * (4.5 bits per weight) and multiplying them in f16 (e2m1 * e4m3 is exact in f16; the layer input
 * and the SwiGLU activations are rounded to f16 for these products, so inputs must stay within
 * f16's range, |x| < 65504), with the tensor scale applied to each finished output in fp32.
 * Decode sizes only: max_tokens <= 64, else FLINT_MOE_ERR_UNSUPPORTED. */
typedef struct {
  const void* w_router;         /* bf16 [hidden][n_experts] */
  const float* router_bias;     /* fp32 [n_experts] or NULL */
  const uint8_t* gate_codes;    /* [n_experts][expert_inter][hidden / 2] */
  const uint8_t* up_codes;      /* [n_experts][expert_inter][hidden / 2] */
  const uint8_t* down_codes;    /* [n_experts][hidden][expert_inter / 2] */
  const uint8_t* gate_scales;   /* [n_experts][expert_inter][hidden / 16] */
  const uint8_t* up_scales;     /* [n_experts][expert_inter][hidden / 16] */
  const uint8_t* down_scales;   /* [n_experts][hidden][expert_inter / 16] */
  const float* gate_tscale;     /* device fp32 [n_experts] */
  const float* up_tscale;       /* device fp32 [n_experts] */
  const float* down_tscale;     /* device fp32 [n_experts] */
  const uint8_t* sgate_codes;   /* [shared_inter][hidden / 2] */
  const uint8_t* sup_codes;     /* [shared_inter][hidden / 2] */
  const uint8_t* sdown_codes;   /* [hidden][shared_inter / 2] */
  const uint8_t* sgate_scales;  /* [shared_inter][hidden / 16] */
  const uint8_t* sup_scales;    /* [shared_inter][hidden / 16] */
  const uint8_t* sdown_scales;  /* [hidden][shared_inter / 16] */
  float sgate_tscale, sup_tscale, sdown_tscale;
} flint_moe_nvfp4_weights;

flint_moe_status flint_moe_create_nvfp4(const flint_moe_config* cfg, const flint_moe_nvfp4_weights* w,
                                        void* workspace, size_t workspace_bytes, flint_moe_t* out);

/* The whole layer for callers that cannot allocate device memory where they run it (a host
 * program that owns all device memory and gives plugins no allocator, a runtime that plans
 * its memory at start-up and allows no allocation later, a latency path that cannot take the
 * implicit synchronisation of cudaMalloc).  The pages have no counterpart of this call: it is
 * a property of this library, not of the method.
 *   w, x, y, topk_idx, topk_w, stream: as for flint_moe_create / flint_moe_forward (no flags:
 *   no pre-norm, no residual); 1 <= T <= 4, a larger T returns FLINT_MOE_ERR_UNSUPPORTED.
 * Scratch memory comes from one fixed array of 25 MiB that the library declares in device
 * memory; every GPU that loads the library holds it until the process exits.  The call makes
 * no allocation.  The first call on a device (with that device current) looks up the array's
 * device address, sets the kernel's shared-memory limit, checks that one CTA fits on every SM
 * and clears the array's status word (synchronously); make that first call before any stream
 * capture.  The address is kept for the life of the process: after cudaDeviceReset (or any
 * other destruction of the device's primary context) do not call these entry points on that
 * device again.  All calls on a device share the array, and it keeps the last call's contents:
 * the barrier counters and tickets, which must start at zero, are cleared on `stream` at the
 * start of each call, and calls whose work overlaps on the GPU race on the array.  Device
 * errors (a bounded wait that ran out, an index out of range) are recorded in the array's
 * status word and stay there until flint_moe_noalloc_poll_device_status reads them. */
flint_moe_status flint_moe_forward_noalloc(const flint_moe_weights* w, const void* x, int T, void* y,
                                           int32_t* topk_idx, float* topk_w, flint_stream_t stream);

/* Synchronises `stream`, then returns and clears the status word of the current device's
 * fixed scratch array (FLINT_MOE_OK, FLINT_MOE_ERR_DEVICE_TIMEOUT or FLINT_MOE_ERR_DEVICE_BOUNDS):
 * the device errors of every flint_moe_forward_noalloc call on this device since the last poll
 * (the array is shared by all of them).  Allocates nothing; like flint_moe_forward_noalloc, a
 * first call on a device does that device's one-time set-up. */
flint_moe_status flint_moe_noalloc_poll_device_status(flint_stream_t stream);

/* ---------------------------------------------------------------- the layer stack
 * The model runs its MoE layers back to back: two dense layers, then 47 MoE layers (Recursive
 * Flint serving-kit post, section "The architecture, from the config"); the pages' own engine
 * fuses the decode forward pass into one kernel (news article "Recursive opens Flint, a 40B
 * coding model with 2.5B active", section "Built with the Eureka Machine").  A stack handle applies
 * n_layers MoE layers, each with its own weights, in place,
 *     x <- [x +] MoE_l([RMSNorm](x)),  l = 0 .. n_layers-1  (the config's flags, for every layer),
 * in ONE persistent cooperative kernel launch: each layer's steps as in flint_moe_forward, a
 * grid-wide barrier between layers instead of a kernel boundary, the next layer's pre-norm done by
 * the CTAs that combine each token row, and the next layer's router and shared-expert weights
 * requested into L2 while this layer's down step finishes.  The results are bitwise those of
 * n_layers successive flint_moe_forward calls (x in, y = x) with the same config on the layers'
 * weights.  Decode sizes only: cfg->max_tokens <= 256, else
 * FLINT_MOE_ERR_UNSUPPORTED. */
typedef struct flint_moe_stack_s* flint_moe_stack_t;

/* Workspace bytes for a stack of n_layers (>= 1) layers: one layer's scratch plus a device
 * table of the layers' tensor maps (about 1 KB per layer). */
flint_moe_status flint_moe_stack_workspace_bytes(const flint_moe_config* cfg, int n_layers, size_t* bytes);

/* layers: host array of n_layers weight sets (each as for flint_moe_create; borrowed, they must
 * stay valid).  workspace: caller-owned device memory, 256-byte aligned, at least
 * flint_moe_stack_workspace_bytes; the call writes the layer table into it (synchronously). */
flint_moe_status flint_moe_stack_create(const flint_moe_config* cfg, const flint_moe_weights* layers, int n_layers,
                                        void* workspace, size_t workspace_bytes, flint_moe_stack_t* out);

/* x: device bf16 [T][2048], 16-byte aligned, read and overwritten with the stack's output;
 * 1 <= T <= max_tokens.  topk_idx / topk_w: optional device [n_layers][T][6] copies of every
 * layer's routing (null to skip).  Asynchronous on `stream`; no allocation. */
flint_moe_status flint_moe_stack_forward(flint_moe_stack_t s, void* x, int T, int32_t* topk_idx, float* topk_w,
                                         flint_stream_t stream);

/* As flint_moe_poll_device_status, for the stack's workspace. */
flint_moe_status flint_moe_stack_poll_device_status(flint_moe_stack_t s, flint_stream_t stream);

/* As flint_moe_enable_kernel_timing / flint_moe_read_trace, for the stack's launches (the phase
 * trace holds the last layer's stamps). */
flint_moe_status flint_moe_stack_enable_kernel_timing(flint_moe_stack_t s, int enable);
flint_moe_status flint_moe_stack_read_trace(flint_moe_stack_t s, unsigned long long* out, int cap, int* n);

/* Releases the stack's host state (not the workspace or the weights). */
flint_moe_status flint_moe_stack_destroy(flint_moe_stack_t s);

/* ---------------------------------------------------------------- the dense MLP layers
 * The model's first two layers are dense SwiGLU MLP layers instead of MoE layers (serving-kit
 * post, section "The architecture, from the config": "2 dense MLP layers (mlp_only_layers: [0,
 * 1]), then 47 MoE layers"; the two "add about 75M" parameters).  The pages give no width; the
 * one their parameter count fixes is 6144 (2 x 3 x 2048 x 6144 = 75.5M), and the layer is read
 * as the same SwiGLU MLP as an expert: y = (silu(x' Wg) * (x' Wu)) Wd [+ x], x' = x or rms(x).
 * The conventions of the MoE calls above hold (caller-owned device memory, asynchronous on
 * `stream`, no allocation in forward, sticky device status, bitwise deterministic).  T <= 256
 * runs the decode-size kernel (the MoE kernel's shared-expert steps at this width), larger T
 * the tensor-core GEMMs. */
typedef struct flint_dense_s* flint_dense_t;

typedef struct {
  int hidden;       /* must be 2048 */
  int inter;        /* must be 6144 */
  int max_tokens;   /* largest T any call on this handle will pass; 1..65536 */
  unsigned flags;   /* FLINT_MOE_FLAG_PRE_RMSNORM, FLINT_MOE_FLAG_RESIDUAL (y may alias x),
                       FLINT_MOE_FLAG_TEST_WAIT_TIMEOUT */
  float rms_eps;    /* RMSNorm epsilon (with FLINT_MOE_FLAG_PRE_RMSNORM), > 0 */
} flint_dense_config;

typedef struct {
  const void* w_gate; /* bf16 [hidden][inter], 16-byte aligned */
  const void* w_up;   /* bf16 [hidden][inter] */
  const void* w_down; /* bf16 [inter][hidden] */
} flint_dense_weights;

/* Bytes of device workspace a dense layer with `cfg` needs (the caller allocates it, 256-byte
 * aligned, and keeps it alive until flint_dense_destroy). */
flint_moe_status flint_dense_workspace_bytes(const flint_dense_config* cfg, size_t* bytes);

/* As flint_moe_create: validates, builds the TMA descriptors, zeroes the workspace's counters
 * and status word (synchronously).  The weights are borrowed. */
flint_moe_status flint_dense_create(const flint_dense_config* cfg, const flint_dense_weights* w, void* workspace,
                                    size_t workspace_bytes, flint_dense_t* out);

/* y bf16 [T][hidden] = (silu(x' Wg) * (x' Wu)) Wd [+ x]; 1 <= T <= max_tokens; x, y device,
 * 16-byte aligned. */
flint_moe_status flint_dense_forward(flint_dense_t d, const void* x, int T, void* y, flint_stream_t stream);

/* As flint_moe_poll_device_status / flint_moe_enable_kernel_timing / flint_moe_kernel_times,
 * for a dense layer. */
flint_moe_status flint_dense_poll_device_status(flint_dense_t d, flint_stream_t stream);
flint_moe_status flint_dense_enable_kernel_timing(flint_dense_t d, int enable);
flint_moe_status flint_dense_kernel_times(flint_dense_t d, const char** names, float* ms, int cap, int* n);

/* Releases the handle's host state (not the workspace or the weights). */
flint_moe_status flint_dense_destroy(flint_dense_t d);

/* ---------------------------------------------------------------- sliding-window decode attention
 * One decode step of a sliding-window attention layer (serving-kit post, section "The
 * architecture, from the config": 35 layers attend to a 513-token window, the current token plus
 * 512 back; 32 query heads, 4 KV heads, head dimension 128; learned per-head attention sinks.
 * News article "Recursive opens Flint, a 40B coding model with 2.5B active", section "What runs
 * on each token": a sink is a slot that can take attention no real token needs).  For every
 * sequence b and query head h (KV head h / 8):
 *   out[b][h] = sum_j e^(s_j - m) v_j / (e^(sinks[h] - m) + sum_j e^(s_j - m)),
 *   s_j = q[b][h] . k_j / sqrt(128), m = max(sinks[h], s_j),
 * over the sequence's valid cache slots.  Readings taken: the sink is a logit of the softmax
 * denominator that carries no value; q and k are passed already normalised and rotated (the
 * per-head QK RMSNorm and RoPE belong to the projections).
 * Layouts (device memory, caller-owned, 16-byte aligned; bf16 row-major):
 *   q       [B][32][128]
 *   k_cache [B][513][4][128], v_cache the same: each sequence's ring of its last 513 tokens,
 *           position p in slot p mod 513, the current token's K and V already stored;
 *   sinks   fp32 [32];  pos int32 [B]: position of each sequence's current token (>= 0; the
 *           slots 0 .. min(pos + 1, 513) - 1 are valid; a negative pos is a device bounds error);
 *   out     [B][32][128] bf16.
 * One kernel launch, asynchronous on `stream`, no allocation, bitwise deterministic.  The
 * workspace (caller-owned, 256-byte aligned, flint_swa_workspace_bytes) holds chunk partials
 * and tickets; initialise it once with flint_swa_workspace_init (on each device that will run
 * decode calls: it also sets the kernel's shared-memory limit); its tickets return to zero at
 * the end of every call.  Calls sharing one workspace must be ordered on one stream. */
flint_moe_status flint_swa_workspace_bytes(int max_batch, size_t* bytes);
flint_moe_status flint_swa_workspace_init(void* workspace, size_t workspace_bytes, flint_stream_t stream);
flint_moe_status flint_swa_decode(void* workspace, size_t workspace_bytes, const void* q, const void* k_cache,
                                  const void* v_cache, const float* sinks, const int32_t* pos, int B, void* out,
                                  flint_stream_t stream);
/* Synchronises `stream`, then returns and clears the workspace's device status word. */
flint_moe_status flint_swa_poll_device_status(void* workspace, flint_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FLINT_MOE_H */
