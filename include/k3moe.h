/*
 * k3moe.h -- C ABI of the GB300 (sm_103a) MXFP4 mixture-of-experts layer library (libk3moe.so).
 *
 * The layer (Kimi-K3 style, as described by the kimi-k3-in-c review,
 * blog.123qwe.co.kr/?p=4411, tables "한눈에 보는 kimi-k3-in-c" and "KDA·MLA·MoE", and the
 * kimi-k3-in-c README, rosettalens.com/s/ko/kimi-k3-in-c, section "shard census"):
 *   for each token x (d_model values)
 *     logits  l_e = x . W_e (+ b_e)                      e = 0..n_routed-1      (router)
 *     top-k   the k largest logits, equal logits -> lower index first
 *     gates   w_i = exp(l_i - l_max) / sum_{j in top-k} exp(l_j - l_max)       (renormalised softmax)
 *     expert  o = W_down (SiLU(W_gate x) * (W_up x))     on MXFP4 weights        (SiLU-gated GLU)
 *     output  y = sum_i w_i o_{e_i} + sum_s o_s          (n_shared always-on experts, weight 1)
 *
 * MXFP4 (OCP MX v1.0): 4-bit E2M1 codes plus one E8M0 scale byte (2^(b-127), 0xFF = NaN) per
 * 32 consecutive weights along the reduction axis, 0.53125 B per weight. Expert record, one per
 * expert, contiguous, `record_stride` bytes apart (d = d_model, f = d_ff):
 *   [gate codes f x d/2][gate scales f x d/32][up codes f x d/2][up scales f x d/32]
 *   [down codes d x f/2][down scales d x f/32]
 * Codes are row-major, two per byte, the even column in the low nibble. A record of the
 * d_model 7168 / d_ff 1536 shape is 17,547,264 bytes (the census figure). This is the stored
 * order; the compute calls read records put in the device order by k3moe_pack_records (see
 * there), once, when the records are loaded onto the GPU.
 *
 * Conventions shared by every call below:
 *  - Pointers are DEVICE pointers unless marked "host". The caller owns all memory; nothing is
 *    allocated by a compute call and nothing is kept after it returns (one exception:
 *    k3moe_layer_static keeps its scratch array, and that array's address, between calls).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *  - Invalid arguments return K3MOE_ERR_INVALID_ARGUMENT synchronously and launch nothing:
 *    a NULL required pointer, T < 0, top_k < 1 or top_k > min(n_routed, 32), n_routed > 4096,
 *    n_shared < 0 or > 8, d_model or d_ff not a positive multiple of 32, record_stride < the
 *    record size or not a multiple of 4096 (records are 4 KiB aligned), a pointer not 16-byte
 *    aligned, or an unknown enum value.
 *    Legal configurations this library does not implement return K3MOE_ERR_UNSUPPORTED
 *    without launching anything: d_model or d_ff a multiple of 32 but not of 128 (the
 *    tensor-core tiles are 128 rows), d_model > 25600, act_mode K3MOE_ACT_MXFP4, and records
 *    in the stored order (record_order K3MOE_ORDER_STORED) given to a call that reads them
 *    (record_order describes the MXFP4 records; bf16 shared records have a single order).
 *    A workspace smaller than k3moe_workspace_bytes(cfg, T) returns K3MOE_ERR_WORKSPACE.
 *  - T = 0 is a no-op that returns K3MOE_OK.
 *  - Bad data found on the device (an expert index outside [0, n_routed) given to
 *    k3moe_expert_ffn, or an E8M0 scale byte 0xFF) sets a status word in the workspace; the
 *    affected output is not trusted. k3moe_check_device_status reports it as
 *    K3MOE_ERR_DEVICE_CHECK. Kernels never trap and never wait without a bound.
 *  - CUDA launch errors return K3MOE_ERR_CUDA.
 *  - The workspace (`ws`, `ws_bytes`) is scratch owned by the caller: size it with
 *    k3moe_workspace_bytes, zero-fill it once after allocation, and do not run two calls
 *    that share a workspace concurrently. Calls on different workspaces are independent.
 *    Other mutable global state: caches of tensor-map descriptors and device properties
 *    (guarded by a mutex), and k3moe_layer_static's scratch array, which all its calls share.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define K3MOE_API __attribute__((visibility("default")))
#else
#define K3MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  K3MOE_OK = 0,
  K3MOE_ERR_INVALID_ARGUMENT = 1,
  K3MOE_ERR_UNSUPPORTED = 2,
  K3MOE_ERR_WORKSPACE = 3,
  K3MOE_ERR_CUDA = 4,
  K3MOE_ERR_DEVICE_CHECK = 5,
  K3MOE_ERR_TIMEOUT = 6
} k3moe_status;

/* Router score function: softmax over the logits (the bias, if given, is added to the logits), or
   sigmoid of the unbiased logit with a selection-only bias (see k3moe_route). */
enum { K3MOE_SCORE_SOFTMAX = 0, K3MOE_SCORE_SIGMOID_BIAS = 1 };
/* Legal but not implemented: d_model > 25600 (the router stages whole rows in shared memory). */
/* Activation handling in the expert FFN. The activations x and h = SiLU(g) * u enter the tensor
   cores as sums of terms with E8M0 block scales (one per 32 elements), each term the rounding
   residual of the previous ones; the bounds below are of |v - sum of terms| against the maximum of
   the element's 32-element block.
   K3MOE_ACT_EXACT (the default): with 1 and 2 tokens, x and h as eight E2M1 terms, within 2^-23.
   From 3 tokens on, bf16 x as two E4M3 terms, exact for every element of at least 2^-13 of the
   block maximum (smaller ones within 2^-21); fp32 x and h as three E4M3 terms, within 2^-12
   (about 2^-14 over random blocks).
   K3MOE_ACT_BF16H: x as in the exact mode; from 3 tokens on, h enters the down projection as two
   E4M3 terms, within 2^-8, every element of at least 2^-13 of the block maximum to 2^-8 of itself
   (bf16's precision class), and the down projection's work groups hold 32 positions instead of 16. The layer output stays within the 2e-3 bound on max|y - y_exact| /
   max|y_exact| (measured 6e-4 to 1e-3 at the test shapes, against ~2e-5 exact) and the down
   projection runs ~2x faster at 4096 tokens. Below 3 tokens it is the exact mode.
   K3MOE_ACT_MXFP4 (activations quantised to MXFP4) is legal but not implemented. */
enum { K3MOE_ACT_EXACT = 0, K3MOE_ACT_MXFP4 = 1, K3MOE_ACT_BF16H = 2 };
/* Element type of the token activations x. */
enum { K3MOE_X_BF16 = 0, K3MOE_X_F32 = 1 };
/* Order of the bytes inside the expert records the caller passes: the stored order (the layout
   below, as the records are kept on disk) or the device order that k3moe_pack_records produces.
   The compute calls read the device order only; they refuse records marked as stored
   (K3MOE_ERR_UNSUPPORTED), so that records never packed cannot be used by mistake. A
   zero-initialised config says "stored". */
enum { K3MOE_ORDER_STORED = 0, K3MOE_ORDER_DEVICE = 1 };
/* Format of the shared experts' records: MXFP4 like the routed experts (the default), or bf16
   (the kimi-k3-in-c README's parameter budget counts every non-routed parameter in bfloat16). A bf16
   shared record is [gate f x d][up f x d][down d x f] bf16, row-major, 6 d f bytes, shared_stride
   bytes apart; it is used as stored (k3moe_pack_records is for MXFP4 records only). Its FFN runs as
   bf16 GEMMs on the tensor cores (fp32 accumulation; fp32 tokens and h enter as three bf16 parts,
   24 significant bits), after the routed experts, and the combine adds its output. */
enum { K3MOE_SHARED_MXFP4 = 0, K3MOE_SHARED_BF16 = 1 };

typedef struct {
  int32_t d_model;       /* hidden size d (7168 for the K3 shape) */
  int32_t d_ff;          /* expert intermediate size f (1536) */
  int32_t n_routed;      /* routed experts E (896) */
  int32_t top_k;         /* experts selected per token k (16) */
  int32_t n_shared;      /* always-on shared experts S (2) */
  int32_t score_func;    /* K3MOE_SCORE_* */
  int32_t act_mode;      /* K3MOE_ACT_* */
  int32_t x_dtype;       /* K3MOE_X_* */
  int32_t record_order;  /* K3MOE_ORDER_* of the records passed to the call */
  int32_t shared_format; /* K3MOE_SHARED_* */
  int64_t record_stride; /* bytes between expert records (>= record size, multiple of 4096) */
  int64_t shared_stride; /* bytes between shared records; 0: record_stride (MXFP4 shared records)
                            or the bf16 record size rounded up to 4096 (bf16 shared records) */
} k3moe_config;

/*
 * Device order of records. The block-scaled MMA of the tensor cores reads the E8M0 scales of 128
 * weight rows x 4 blocks as one 32 x 16-byte image (lane i of each 32-row quarter c holds the 4
 * scale bytes of row 32 c + i), and the gate/up kernel finishes h = SiLU(g) * u in its epilogue,
 * which needs the gate and up rows of the same h indices in one 128-row tile. In the device order:
 *  - gate/up: for u = 0 .. d_ff/128 - 1 and half h = 0, 1, the stacked tile 2u + h consists of gate
 *    rows 128u + 64h .. 128u + 64h + 63 (its rows 0-63) and up rows 128u + 64h .. +63 (rows
 *    64-127); stacked tile 2u takes the place of gate rows 128u .. 128u + 127 and stacked tile 2u + 1
 *    that of up rows 128u .. 128u + 127, for the codes and for the scale bytes. (For the codes this
 *    swaps gate rows 128u + 64 .. 128u + 127 with up rows 128u .. 128u + 63.)
 *  - down: codes unchanged.
 *  - every 128-row tile (stacked, or of the down matrix) stores its scale bytes as its image: the
 *    byte of tile row r = 32 c + i and block b = 4 g + e at tile_start + 512 g + 16 i + 4 c + e,
 *    so that the scales of one chunk of the reduction axis are a single contiguous copy.
 * The record size and the offsets of the six regions are those of the stored order.
 * k3moe_pack_records converts `n_records` records (record_stride bytes apart, 16-byte aligned
 * base) in place: to_device = 1 stored -> device order, 0 device -> stored order. Only d_model,
 * d_ff and record_stride of `cfg` are used (any valid config of that geometry). Asynchronous on
 * `stream`; the records must not be in use by another call meanwhile.
 */
K3MOE_API k3moe_status k3moe_pack_records(const k3moe_config* cfg /* host */, uint8_t* records, int64_t n_records,
                                          int32_t to_device, void* stream);

/* Bytes of one expert record for this config: 3 * d_model * d_ff * 17 / 32 (host only; 0 if invalid). */
K3MOE_API size_t k3moe_record_bytes(const k3moe_config* cfg /* host */);

/* Workspace bytes needed for calls of up to `max_tokens` tokens (host only; 0 if invalid). */
K3MOE_API size_t k3moe_workspace_bytes(const k3moe_config* cfg /* host */, int64_t max_tokens);

/*
 * Bytes of the router weights' three bf16 parts, 3 * n_routed * d_model * 2 (host only; 0 if the
 * config is invalid).
 */
K3MOE_API size_t k3moe_router_parts_bytes(const k3moe_config* cfg /* host */);

/*
 * Weight-loading step of the router (once per set of router weights, like k3moe_pack_records):
 * writes w_parts[3][n_routed][d_model] bf16 with W = W0 + W1 + W2, each part the bf16 rounding of
 * what the earlier parts leave (24 significant bits of every fp32 weight are kept). From 16 tokens
 * the router computes its logits on the tensor cores from these parts; k3moe_route and k3moe_layer
 * take them as `w_router_parts`. w_router [n_routed, d_model] fp32; w_parts 16-byte aligned,
 * k3moe_router_parts_bytes(cfg) bytes. Asynchronous on `stream`.
 */
K3MOE_API k3moe_status k3moe_prepare_router(const k3moe_config* cfg /* host */, const float* w_router,
                                            uint16_t* w_parts, void* stream);

/*
 * Router: softmax over the n_routed logits of each token, top-k, renormalised gates.
 * With score_func K3MOE_SCORE_SIGMOID_BIAS (the review's list of public-header invariants: the
 * routing bias skews only the selection, the combine weights come from the unbiased sigmoid score):
 * s_e = sigmoid(x . W_e), the k largest s_e + b_e are selected (equal values -> lower index first),
 * and the gates are s_e / sum over the selected of s.
 *   x        [T, d_model] bf16 or fp32 (cfg->x_dtype), row-major
 *   w_router [n_routed, d_model] fp32, row-major
 *   w_router_parts  [3, n_routed, d_model] bf16 from k3moe_prepare_router, or NULL: then calls of
 *            16 tokens or more split the weights into the workspace on every call
 *   bias     [n_routed] fp32, or NULL: softmax score: added to every logit before selection and
 *            softmax; sigmoid score: added to the sigmoid scores for the selection only
 *   topk_idx [T, top_k] int32 out: expert ids, descending ranked value, ties to the lower id
 *   topk_w   [T, top_k] fp32 out: gates, summing to 1 per token
 * Below 16 tokens the logits are fp32 dot products. From 16 tokens they come from the tensor cores
 * (three bf16 parts of the weights; the accumulation rounds by ~1e-5 at d_model 7168); every expert
 * whose place in the selection that rounding could decide is recomputed as an fp32 dot product, so
 * the indices are those of fp32 logits, and the other selected experts' gates carry the rounding
 * (measured below 2e-5).
 */
K3MOE_API k3moe_status k3moe_route(const k3moe_config* cfg /* host */, const void* x, int64_t T,
                         const float* w_router, const uint16_t* w_router_parts, const float* bias,
                         int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream);

/*
 * Expert FFN and combine for given routing (review, table "KDA·MLA·MoE": the experts multiply
 * MXFP4 nibbles directly; the layer's 2 shared experts run for every token).
 *   x              [T, d_model] bf16 or fp32
 *   topk_idx       [T, top_k] int32 expert ids in [0, n_routed) (checked on the device)
 *   topk_w         [T, top_k] fp32 gate weights
 *   routed_records n_routed records, record_stride bytes apart (16-byte aligned base), in the
 *                  device order (k3moe_pack_records)
 *   shared_records n_shared records: MXFP4, record_stride bytes apart, device order; or bf16
 *                  (shared_format K3MOE_SHARED_BF16), shared_stride bytes apart (may be NULL
 *                  if n_shared == 0)
 *   y              [T, d_model] fp32 out, overwritten
 */
K3MOE_API k3moe_status k3moe_expert_ffn(const k3moe_config* cfg /* host */, const void* x, int64_t T,
                              const int32_t* topk_idx, const float* topk_w,
                              const uint8_t* routed_records, const uint8_t* shared_records, float* y,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * The whole layer: k3moe_route followed by k3moe_expert_ffn, sharing one workspace.
 *   topk_idx_out / topk_w_out: optional [T, top_k] outputs of the routing (NULL to skip).
 */
K3MOE_API k3moe_status k3moe_layer(const k3moe_config* cfg /* host */, const void* x, int64_t T,
                         const float* w_router, const uint16_t* w_router_parts, const float* bias,
                         const uint8_t* routed_records, const uint8_t* shared_records, float* y,
                         int32_t* topk_idx_out, float* topk_w_out, void* ws, size_t ws_bytes, void* stream);

/*
 * k3moe_layer with an explicit bound on the waits of its tensor-core kernels: `wait_limit` polls of
 * a pipeline barrier before the waiting CTA gives up, sets K3MOE_ERR_TIMEOUT in the workspace's
 * status word (read by k3moe_check_device_status), stops its work, lets the copies and MMAs it
 * started complete, frees its tensor memory and exits. k3moe_layer uses 2^24 polls (seconds). A
 * limit of 1 makes the first wait that is not already satisfied give up: this is how the timeout
 * path is tested (the output of such a call is not trusted; the context stays usable). 0 is invalid.
 */
K3MOE_API k3moe_status k3moe_layer_bounded(const k3moe_config* cfg /* host */, const void* x, int64_t T,
                                           const float* w_router, const uint16_t* w_router_parts,
                                           const float* bias, const uint8_t* routed_records,
                                           const uint8_t* shared_records, float* y, void* ws, size_t ws_bytes,
                                           uint32_t wait_limit, void* stream);

/*
 * k3moe_layer with phase timing, for profiling: `events` points to 6 cudaEvent_t handles created by
 * the caller; they are recorded on `stream` before the router kernel, before the gate/up kernel
 * (which also finishes h), twice after it (once where a separate GLU kernel would end), before the
 * combine kernel and after it.
 * Same kernels and results as k3moe_layer (an event between two kernels only removes their overlap).
 */
K3MOE_API k3moe_status k3moe_layer_timed(const k3moe_config* cfg /* host */, const void* x, int64_t T,
                                         const float* w_router, const uint16_t* w_router_parts,
                                         const float* bias, const uint8_t* routed_records,
                                         const uint8_t* shared_records, float* y, int32_t* topk_idx_out,
                                         float* topk_w_out, void* ws, size_t ws_bytes, void* stream,
                                         void* const* events /* host */);

/*
 * The whole layer for callers that cannot allocate device memory (no counterpart in the pages:
 * an interface addition of this library). Some programs own every device allocation through
 * their own pool and forbid other cudaMalloc calls, and latency-critical callers cannot afford
 * cudaMalloc's device synchronisation; this call needs no workspace from them. Its scratch is a
 * fixed K3MOE_STATIC_SCRATCH_BYTES array in device memory declared by the library (resident on
 * every GPU that loads it until exit); calls needing more (k3moe_workspace_bytes(cfg, T) larger)
 * return K3MOE_ERR_WORKSPACE: at the 7168/1536/896 top-16 shape with 2 shared experts, T <= 6 is
 * served and T >= 7 is refused. It allocates nothing, clears the scratch it uses at the start of
 * each call, and otherwise behaves like k3moe_layer without the optional outputs (same argument
 * checks and status codes; the router weights are used as fp32, which is all that calls of this
 * size read). All calls on a device share the array: calls that overlap on the GPU race and give
 * wrong results. The first call on a device looks up the array's address; make it before any
 * stream capture, and do not reset the device after it. Device-side data checks are not reported.
 */
#define K3MOE_STATIC_SCRATCH_BYTES (4u << 20)
K3MOE_API k3moe_status k3moe_layer_static(const k3moe_config* cfg /* host */, const void* x, int64_t T,
                                          const float* w_router, const float* bias,
                                          const uint8_t* routed_records, const uint8_t* shared_records,
                                          float* y, void* stream);

/*
 * Pre-norm residual step of a stack of layers: xn = RMSNorm(x) with unit weight,
 * xn_j = x_j / sqrt(mean_j(x^2) + eps) (RMSNorm is one of the engine's ops in the review's
 * "k3_ops.c" row). x, xn: [T, d] fp32.
 */
K3MOE_API k3moe_status k3moe_rmsnorm(const float* x, int64_t T, int32_t d, float eps, float* xn, void* stream);

/* Residual add x += y over n fp32 values. */
K3MOE_API k3moe_status k3moe_residual_add(float* x, const float* y, int64_t n, void* stream);

/*
 * The step between two layers of a stack in one kernel: x += y (skipped if y is NULL), then
 * xn = RMSNorm(x) with unit weight. x, y, xn: [T, d] fp32, 16-byte aligned, d a multiple of 4.
 * Like every kernel of this library it is launched with programmatic stream serialization: it is
 * scheduled while the previous layer's last kernel drains, and the next layer's router kernel is
 * scheduled while it runs and streams its router weights (which nothing on the stream writes)
 * before it waits for xn. So layer l+1's router overlaps layer l's tail instead of starting cold.
 */
K3MOE_API k3moe_status k3moe_residual_rmsnorm(float* x, const float* y, int64_t T, int32_t d, float eps, float* xn,
                                              void* stream);

/*
 * Synchronise `stream`, read the workspace's device status word, clear it, and return
 * K3MOE_ERR_TIMEOUT if a bounded wait gave up since the last check, else K3MOE_ERR_DEVICE_CHECK if
 * bad data was seen, else K3MOE_OK (K3MOE_ERR_CUDA if the stream reports an error).
 */
K3MOE_API k3moe_status k3moe_check_device_status(void* ws, void* stream);

/* Static description of a status code (host only). */
K3MOE_API const char* k3moe_status_string(k3moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* K3MOE_H */
