// C ABI of libk3moe.so (declared in include/k3moe.h): argument validation, the workspace
// layout, and the launch sequence of each call. No call allocates memory.
#include <cstddef>
#include <cstdint>

#include "../../include/k3moe.h"
#include "k3moe_kernels.h"

namespace {

using k3::Cfg;
using k3::Ws;

constexpr long long kMaxE = 4096;
constexpr long long kMaxK = 32;
constexpr long long kMaxS = 8;
constexpr int kMaxDModel = 25600;
constexpr long long kMaxTerms = 3;     // E4M3 terms per activation block (x: 2 bf16 / 3 fp32; h: 3)
constexpr long long kMaxTermsFp4 = 8;  // E2M1 terms per activation block
constexpr long long kFp4MaxT = 2;      // the E2M1 / mxf4 path serves up to this many tokens
constexpr uint32_t kDefaultWaitLimit = 1u << 24;  // polls of a pipeline barrier before a CTA gives up

// E2M1 activation terms and kind::mxf4 MMAs for few tokens (d_model and d_ff multiples of 256).
bool use_fp4(const k3moe_config* c, long long T) {
  return T <= kFp4MaxT && c->d_model % 256 == 0 && c->d_ff % 256 == 0;
}

// Gate/up B tiles from the x terms in position order (one tensor copy per chunk) from kGatherMinT
// tokens on, where the loaders' 16-byte copies of rows gathered by token bound the projection. The
// gather costs P x xterms x d bytes written and read once more.
constexpr long long kGatherMinT = 256;
bool gather_x(const k3moe_config* c, long long T) { return !use_fp4(c, T) && T >= kGatherMinT; }

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

// Router logits on the tensor cores from kRouterTcMinT tokens, else on the CUDA cores. Below it the
// CUDA-core kernel reads the fp32 router weights once per 8-token tile. The tensor-core path reads
// their three bf16 parts instead (6 bytes per weight; prepared once by k3moe_prepare_router, else
// split per call, which writes and reads them first: 4x the fp32 bytes), then selects in a second
// kernel. The threshold was measured with the per-call split, at the K3 shape with bf16 tokens:
// 72 vs 85 us at 8 tokens, 163 vs 95 us at 32.
constexpr long long kRouterTcMinT = 16;
bool router_tc(const k3moe_config* c, long long T) {
  return T >= kRouterTcMinT && c->d_model % 64 == 0;
}

// Parts of the tensor-core router's reduction axis: enough (128 token x 256 expert) tiles x parts to
// fill the 152 SMs once, each part at least 16 of the 64-wide k-steps (the router kernel adds the
// parts up: fewer parts, fewer loads there); 1 on the CUDA-core path.
constexpr long long kRouterSplitSms = 152;
long long router_splits(const k3moe_config* c, long long T) {
  if (!router_tc(c, T)) return 1;
  const long long tiles = ((T + 127) / 128) * ((c->n_routed + 255) / 256);
  const long long nk = (c->x_dtype == K3MOE_X_F32 ? 6 : 3) * (c->d_model / 64);
  long long p = kRouterSplitSms / tiles;
  if (p > nk / 16) p = nk / 16;
  return p < 1 ? 1 : p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long record_bytes_of(const k3moe_config* c) {
  return 3LL * ((long long)c->d_model * c->d_ff / 2 + (long long)c->d_model * c->d_ff / 32);
}

bool shared_bf16(const k3moe_config* c) { return c->shared_format == K3MOE_SHARED_BF16 && c->n_shared > 0; }

long long shared_bf16_bytes(const k3moe_config* c) { return 6LL * c->d_model * c->d_ff; }

long long shared_stride_of(const k3moe_config* c) {
  if (c->shared_stride) return c->shared_stride;
  return c->shared_format == K3MOE_SHARED_BF16 ? (shared_bf16_bytes(c) + 4095) / 4096 * 4096 : c->record_stride;
}

// Every check of the config that returns K3MOE_ERR_INVALID_ARGUMENT, then those that return
// K3MOE_ERR_UNSUPPORTED, except the tile geometry (d_model and d_ff multiples of 128), which
// validate() adds.
k3moe_status validate_fields(const k3moe_config* c) {
  if (!c) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->d_model <= 0 || c->d_model % 32 || c->d_ff <= 0 || c->d_ff % 32) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->n_routed < 1 || c->n_routed > kMaxE) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->top_k < 1 || c->top_k > kMaxK || c->top_k > c->n_routed) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->n_shared < 0 || c->n_shared > kMaxS) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->score_func != K3MOE_SCORE_SOFTMAX && c->score_func != K3MOE_SCORE_SIGMOID_BIAS)
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->act_mode != K3MOE_ACT_EXACT && c->act_mode != K3MOE_ACT_MXFP4 && c->act_mode != K3MOE_ACT_BF16H)
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->x_dtype != K3MOE_X_BF16 && c->x_dtype != K3MOE_X_F32) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->record_order != K3MOE_ORDER_STORED && c->record_order != K3MOE_ORDER_DEVICE) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->shared_format != K3MOE_SHARED_MXFP4 && c->shared_format != K3MOE_SHARED_BF16) return K3MOE_ERR_INVALID_ARGUMENT;
  if ((long long)c->d_model * c->d_ff > (1LL << 40)) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->record_stride < record_bytes_of(c) || c->record_stride % 4096) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->shared_stride < 0 || c->shared_stride % 4096) return K3MOE_ERR_INVALID_ARGUMENT;
  const long long shared_need = c->shared_format == K3MOE_SHARED_BF16 ? shared_bf16_bytes(c) : record_bytes_of(c);
  if (c->shared_stride && c->shared_stride < shared_need) return K3MOE_ERR_INVALID_ARGUMENT;
  if (c->act_mode == K3MOE_ACT_MXFP4) return K3MOE_ERR_UNSUPPORTED;
  if (c->d_model > kMaxDModel) return K3MOE_ERR_UNSUPPORTED;  // router rows are staged in shared memory
  return K3MOE_OK;
}

k3moe_status validate(const k3moe_config* c) {
  const k3moe_status s = validate_fields(c);
  if (s != K3MOE_OK) return s;
  if (c->d_model % 128 || c->d_ff % 128) return K3MOE_ERR_UNSUPPORTED;  // 128-row tensor-core tiles
  return K3MOE_OK;
}

// The calls that read expert records read them in the device order only.
k3moe_status records_readable(const k3moe_config* c) {
  return c->record_order == K3MOE_ORDER_DEVICE ? K3MOE_OK : K3MOE_ERR_UNSUPPORTED;
}

bool tokens_ok(const k3moe_config* c, int64_t T) {
  return T >= 0 && T * (long long)(c->top_k + c->n_shared) < (1LL << 30) && T <= (1LL << 26);
}

// Upper bound on work groups for T tokens (work groups of one token: the largest count).
long long wg_bound(const k3moe_config* c, long long T) {
  long long slots = T * c->top_k;
  long long distinct = slots < c->n_routed ? slots : c->n_routed;
  return distinct + slots + (long long)c->n_shared * T + 1;
}

struct Layout {
  size_t ctrl, logits, topk_idx, topk_w, counts, cursor, offsets, wgoff, perm_tok, perm_w, inv, wgs, wgs_dn, xq, xs, xp, hq,
      hs, part, rtcnt, w3, x3, sgu, sh3, sho, total;
};

// Largest T' * parts(T') over T' <= T when parts(T') is constant on runs of 128 tokens (the tile rows)
// and 1 from kRouterSplitSms runs on: sized so, a region never shrinks as T grows.
template <typename F>
long long max_rows(long long T, F parts) {
  long long m = T * parts(T);
  for (long long j = 1; j <= kRouterSplitSms && 128 * j < T; ++j) {
    const long long r = 128 * j * parts(128 * j);
    m = r > m ? r : m;
  }
  return m;
}

Layout make_layout(const k3moe_config* c, long long T) {
  const long long E = c->n_routed, k = c->top_k, S = c->n_shared, d = c->d_model, f = c->d_ff;
  const long long P = T * (k + (shared_bf16(c) ? 0 : S));  // (bf16 shared experts take no positions)
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t& field, size_t bytes) {
    field = o;
    o = align_up(o + (bytes ? bytes : 1));
  };
  take(L.ctrl, sizeof(int) * k3::CTRL_WORDS);
  // partial logits: T x parts rows, sized for the largest row count over T' <= T
  take(L.logits, sizeof(float) * max_rows(T, [&](long long t) { return router_splits(c, t); }) * E);
  take(L.topk_idx, sizeof(int) * T * k);
  take(L.topk_w, sizeof(float) * T * k);
  take(L.counts, sizeof(int) * E);
  take(L.cursor, sizeof(int) * E);
  take(L.offsets, sizeof(int) * (E + 1));
  take(L.wgoff, sizeof(int) * (E + 1));
  take(L.perm_tok, sizeof(int) * P);
  take(L.perm_w, sizeof(float) * P);
  take(L.inv, sizeof(int) * T * k);
  take(L.wgs, sizeof(k3::WorkGroup) * wg_bound(c, T));
  take(L.wgs_dn, sizeof(k3::WorkGroup) * wg_bound(c, T));
  const bool fp4 = use_fp4(c, T);
  const long long terms = fp4 ? kMaxTermsFp4 : kMaxTerms;
  take(L.xq, (size_t)(T * terms * (fp4 ? d / 2 : d)));
  take(L.xs, (size_t)(T * terms * (d / 32)));
  take(L.xp, gather_x(c, T) ? (size_t)(P * terms * d) : 0);
  take(L.hq, (size_t)(P * terms * (fp4 ? f / 2 : f)));
  take(L.hs, (size_t)(P * terms * (f / 32)));
  take(L.part, sizeof(float) * P * d);
  take(L.rtcnt, sizeof(int) * T);  // one counter per router token tile (tiles of 1 to 8 tokens)
  take(L.w3, router_tc(c, T) ? (size_t)3 * E * d * 2 : 0);  // bf16 parts of the router weights
  // three bf16 parts of fp32 tokens (tensor-core router, bf16 shared experts)
  take(L.x3, (router_tc(c, T) || shared_bf16(c)) && c->x_dtype == K3MOE_X_F32 ? (size_t)3 * T * d * 2 : 0);
  // bf16 shared experts: partial sums of gate | up, h in three bf16 parts, partial sums of the outputs
  const bool sb = shared_bf16(c);
  const int xp = c->x_dtype == K3MOE_X_F32 ? 3 : 1;
  take(L.sgu, sb ? sizeof(float) * S * 2 * f *
                       max_rows(T, [&](long long t) { return (long long)k3::shared_gemm_splits(t, 2 * (int)f, (int)d, xp); })
                 : 0);
  take(L.sh3, sb ? (size_t)2 * S * 3 * T * f : 0);
  take(L.sho, sb ? sizeof(float) * S * d *
                       max_rows(T, [&](long long t) { return (long long)k3::shared_gemm_splits(t, (int)d, (int)f, 3); })
                 : 0);
  L.total = o;
  return L;
}

Ws bind(const Layout& L, void* base) {
  char* b = static_cast<char*>(base);
  Ws w;
  w.ctrl = reinterpret_cast<int*>(b + L.ctrl);
  w.logits = reinterpret_cast<float*>(b + L.logits);
  w.topk_idx = reinterpret_cast<int*>(b + L.topk_idx);
  w.topk_w = reinterpret_cast<float*>(b + L.topk_w);
  w.counts = reinterpret_cast<int*>(b + L.counts);
  w.cursor = reinterpret_cast<int*>(b + L.cursor);
  w.offsets = reinterpret_cast<int*>(b + L.offsets);
  w.wgoff = reinterpret_cast<int*>(b + L.wgoff);
  w.perm_tok = reinterpret_cast<int*>(b + L.perm_tok);
  w.perm_w = reinterpret_cast<float*>(b + L.perm_w);
  w.inv = reinterpret_cast<int*>(b + L.inv);
  w.wgs = reinterpret_cast<k3::WorkGroup*>(b + L.wgs);
  w.wgs_dn = reinterpret_cast<k3::WorkGroup*>(b + L.wgs_dn);
  w.xq = reinterpret_cast<uint8_t*>(b + L.xq);
  w.xs = reinterpret_cast<uint8_t*>(b + L.xs);
  w.xp = reinterpret_cast<uint8_t*>(b + L.xp);
  w.hq = reinterpret_cast<uint8_t*>(b + L.hq);
  w.hs = reinterpret_cast<uint8_t*>(b + L.hs);
  w.part = reinterpret_cast<float*>(b + L.part);
  w.rtcnt = reinterpret_cast<int*>(b + L.rtcnt);
  w.sgu = reinterpret_cast<float*>(b + L.sgu);
  w.sh3 = reinterpret_cast<uint8_t*>(b + L.sh3);
  w.sho = reinterpret_cast<float*>(b + L.sho);
  return w;
}

Cfg make_cfg(const k3moe_config* c, long long T) {
  Cfg k;
  k.d = c->d_model;
  k.f = c->d_ff;
  k.E = c->n_routed;
  k.k = c->top_k;
  k.S = shared_bf16(c) ? 0 : c->n_shared;  // MXFP4 shared experts run as work groups
  k.Sb = shared_bf16(c) ? c->n_shared : 0;
  k.nsp1 = k.Sb ? k3::shared_gemm_splits(T, 2 * c->d_ff, c->d_model, c->x_dtype == K3MOE_X_F32 ? 3 : 1) : 0;
  k.nsp2 = k.Sb ? k3::shared_gemm_splits(T, c->d_model, c->d_ff, 3) : 0;
  k.x_f32 = c->x_dtype == K3MOE_X_F32 ? 1 : 0;
  k.fp4 = use_fp4(c, T) ? 1 : 0;
  if (k.fp4) {
    k.xterms = 8;  // at most 2^-23 of the block maximum per element
    k.hterms = 8;
  } else {
    k.xterms = k.x_f32 ? 3 : 2;
    k.hterms = c->act_mode == K3MOE_ACT_BF16H ? 2 : 3;
  }
  // tokens per work group. Gate/up: 32 (16 with the E2M1 terms; 42, which reads an expert's record
  // fewer times, measured slower at prefill sizes, 16 slower from 256 tokens on; whole experts' token
  // lists of up to 128 tokens, MMA N 256 over two issuers, measured slower at 4096 tokens: 13.0 against
  // 10.3 ms in the same build, whose down projection gained 17 % from lists of 85 positions). Down:
  // 16, which keeps its MMA N at 48 with two issuers and two accumulator buffers (32, N = 96 with one
  // of either, measured 35 % slower at 64 tokens, 45 % at 512, 9 % at 4096; 8 slower than 16). With
  // two terms of h (K3MOE_ACT_BF16H) 32 positions make the gate/up projection's N = 64 and stream each
  // down record half as often (4096 tokens: down 7.6 -> 4.4 ms). Wider down groups at prefill sizes,
  // which read each record twice instead of three times at ~73 positions per expert, measured slower
  // still: 48 or 64 positions (N 96 / 128 on the general instance, one issuer) took the 4096-token
  // down projection from 3.3 ms to 4.3 ms with stages of two chunks, 5.2-5.7 ms with one.
  const long long wmax = k.fp4 ? 16 : 32, wmax_dn = (!k.fp4 && k.hterms == 2) ? 32 : 16;
  k.wgt = (int)(T < wmax ? T : wmax);
  k.wgt_dn = (int)(T < wmax_dn ? T : wmax_dn);
  k.rsplit = (int)router_splits(c, T);
  k.gx = gather_x(c, T) ? 1 : 0;
  k.wait_limit = kDefaultWaitLimit;
  k.stride = c->record_stride;
  k.sstride = shared_stride_of(c);
  return k;
}

k3moe_status check_ws(const k3moe_config* c, long long T, void* ws, size_t ws_bytes, Layout* L) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return K3MOE_ERR_INVALID_ARGUMENT;
  *L = make_layout(c, T);
  if (ws_bytes < L->total) return K3MOE_ERR_WORKSPACE;
  return K3MOE_OK;
}

k3moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA; }

}  // namespace

extern "C" {

size_t k3moe_record_bytes(const k3moe_config* cfg) {
  if (!cfg || cfg->d_model <= 0 || cfg->d_ff <= 0 || cfg->d_model % 32 || cfg->d_ff % 32) return 0;
  return (size_t)record_bytes_of(cfg);
}

size_t k3moe_router_parts_bytes(const k3moe_config* cfg) {
  const k3moe_status s = validate(cfg);
  if (s != K3MOE_OK && s != K3MOE_ERR_UNSUPPORTED) return 0;
  return (size_t)3 * cfg->n_routed * cfg->d_model * 2;
}

k3moe_status k3moe_prepare_router(const k3moe_config* cfg, const float* w_router, uint16_t* w_parts, void* stream) {
  const k3moe_status s = validate(cfg);
  if (s != K3MOE_OK) return s;
  if (!w_router || !w_parts || !aligned16(w_router) || !aligned16(w_parts)) return K3MOE_ERR_INVALID_ARGUMENT;
  return cuda_status(k3::launch_split_router(w_router, (long long)cfg->n_routed * cfg->d_model, w_parts,
                                             static_cast<cudaStream_t>(stream)));
}

size_t k3moe_workspace_bytes(const k3moe_config* cfg, int64_t max_tokens) {
  if (validate(cfg) != K3MOE_OK || !tokens_ok(cfg, max_tokens)) return 0;
  // the layout grows with T except, possibly, where the E2M1 activation form gives way to the E4M3
  // one (above kFp4MaxT tokens)
  const long long T = max_tokens < 1 ? 1 : max_tokens;
  const size_t a = make_layout(cfg, T).total, b = make_layout(cfg, T < kFp4MaxT ? T : kFp4MaxT).total;
  return a > b ? a : b;
}

k3moe_status k3moe_route(const k3moe_config* cfg, const void* x, int64_t T, const float* w_router,
                         const uint16_t* w_router_parts, const float* bias, int32_t* topk_idx, float* topk_w, void* ws,
                         size_t ws_bytes, void* stream) {
  k3moe_status s = validate(cfg);
  if (s != K3MOE_OK) return s;
  if (!tokens_ok(cfg, T)) return K3MOE_ERR_INVALID_ARGUMENT;
  if (!x || !w_router || !topk_idx || !topk_w) return K3MOE_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(w_router) || (bias && !aligned16(bias)) || !aligned16(topk_idx) ||
      !aligned16(topk_w) || (w_router_parts && !aligned16(w_router_parts)))
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (T == 0) return K3MOE_OK;
  Layout L;
  if ((s = check_ws(cfg, T, ws, ws_bytes, &L)) != K3MOE_OK) return s;
  const Cfg c = make_cfg(cfg, T);
  const Ws w = bind(L, ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int mode = k3::RM_USER_OUT | (cfg->score_func == K3MOE_SCORE_SIGMOID_BIAS ? k3::RM_SIGMOID : 0);
  if (router_tc(cfg, T)) {
    // (the sigmoid score adds its bias at the selection, not to the logits)
    cudaError_t e = k3::launch_router_tc(c, w, x, T, w_router, w_router_parts, (mode & k3::RM_SIGMOID) ? nullptr : bias,
                                         static_cast<char*>(ws) + L.w3, static_cast<char*>(ws) + L.x3, st);
    if (e != cudaSuccess) return cuda_status(e);
    mode |= k3::RM_LOGITS_READY;
  }
  return cuda_status(k3::launch_route(c, w, x, T, w_router, bias, topk_idx, topk_w, mode, st));
}

}  // extern "C"

namespace {

// The bf16 shared experts (their GEMMs on the tensor cores, after the routed projections), then the
// combine. fp32 tokens are split into three bf16 parts unless the tensor-core router already did.
cudaError_t shared_bf16_then_combine(const k3moe_config* cfg, const Cfg& c, const Ws& w, const Layout& L, const void* x,
                                     long long T, const uint8_t* shared, float* y, void* ws, bool x3_ready,
                                     cudaStream_t st) {
  char* x3 = static_cast<char*>(ws) + L.x3;
  cudaError_t e = cudaSuccess;
  if (c.x_f32 && !x3_ready) e = k3::launch_split_tokens(static_cast<const float*>(x), T * cfg->d_model, x3, st);
  if (e == cudaSuccess) e = k3::launch_shared_bf16(c, w, x, T, x3, shared, st);
  if (e == cudaSuccess) e = k3::launch_combine(c, w, y, T, st);
  return e;
}

}  // namespace

extern "C" {

k3moe_status k3moe_expert_ffn(const k3moe_config* cfg, const void* x, int64_t T, const int32_t* topk_idx,
                              const float* topk_w, const uint8_t* routed_records, const uint8_t* shared_records,
                              float* y, void* ws, size_t ws_bytes, void* stream) {
  k3moe_status s = validate(cfg);
  if (s != K3MOE_OK) return s;
  if (!tokens_ok(cfg, T)) return K3MOE_ERR_INVALID_ARGUMENT;
  if (!x || !topk_idx || !topk_w || !routed_records || !y || (cfg->n_shared > 0 && !shared_records))
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(routed_records) || !aligned16(y) ||
      (shared_records && !aligned16(shared_records)))
    return K3MOE_ERR_INVALID_ARGUMENT;
  if ((s = records_readable(cfg)) != K3MOE_OK) return s;
  if (T == 0) return K3MOE_OK;
  Layout L;
  if ((s = check_ws(cfg, T, ws, ws_bytes, &L)) != K3MOE_OK) return s;
  const Cfg c = make_cfg(cfg, T);
  const Ws w = bind(L, ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = k3::launch_prep(c, w, x, T, topk_idx, topk_w, st);
  if (e == cudaSuccess && c.gx) e = k3::launch_gather_x(c, w, T, st);
  if (e == cudaSuccess) e = k3::launch_gateup(c, w, routed_records, shared_records, y, T, wg_bound(cfg, T), st);
  if (e == cudaSuccess)
    e = k3::launch_down(c, w, routed_records, shared_records, y, T, wg_bound(cfg, T), st, nullptr, c.Sb == 0);
  if (e == cudaSuccess && c.Sb > 0) e = shared_bf16_then_combine(cfg, c, w, L, x, T, shared_records, y, ws, false, st);
  return cuda_status(e);
}

}  // extern "C"

namespace {

k3moe_status layer_impl(const k3moe_config* cfg, const void* x, int64_t T, const float* w_router,
                        const uint16_t* w_router_parts, const float* bias, const uint8_t* routed_records,
                        const uint8_t* shared_records, float* y, int32_t* topk_idx_out, float* topk_w_out, void* ws,
                        size_t ws_bytes, void* stream, void* const* events, uint32_t wait_limit) {
  k3moe_status s = validate(cfg);
  if (s != K3MOE_OK) return s;
  if (!tokens_ok(cfg, T)) return K3MOE_ERR_INVALID_ARGUMENT;
  if (!x || !w_router || !routed_records || !y || (cfg->n_shared > 0 && !shared_records))
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(w_router) || (bias && !aligned16(bias)) || !aligned16(routed_records) ||
      !aligned16(y) || (shared_records && !aligned16(shared_records)) || (topk_idx_out && !aligned16(topk_idx_out)) ||
      (topk_w_out && !aligned16(topk_w_out)) || (w_router_parts && !aligned16(w_router_parts)))
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (events)
    for (int i = 0; i < 6; ++i)
      if (!events[i]) return K3MOE_ERR_INVALID_ARGUMENT;
  if (wait_limit == 0) return K3MOE_ERR_INVALID_ARGUMENT;
  if ((s = records_readable(cfg)) != K3MOE_OK) return s;
  if (T == 0) return K3MOE_OK;
  Layout L;
  if ((s = check_ws(cfg, T, ws, ws_bytes, &L)) != K3MOE_OK) return s;
  Cfg c = make_cfg(cfg, T);
  c.wait_limit = wait_limit;
  const Ws w = bind(L, ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long wgb = wg_bound(cfg, T);
  cudaError_t e = cudaSuccess;
  if (events) e = cudaEventRecord(static_cast<cudaEvent_t>(events[0]), st);
  int mode = k3::RM_USER_OUT | k3::RM_XPREP | k3::RM_PERMUTE |
             (cfg->score_func == K3MOE_SCORE_SIGMOID_BIAS ? k3::RM_SIGMOID : 0);
  if (e == cudaSuccess && router_tc(cfg, T)) {
    e = k3::launch_router_tc(c, w, x, T, w_router, w_router_parts, (mode & k3::RM_SIGMOID) ? nullptr : bias,
                             static_cast<char*>(ws) + L.w3, static_cast<char*>(ws) + L.x3, st);
    mode |= k3::RM_LOGITS_READY;
  }
  if (e == cudaSuccess) e = k3::launch_route(c, w, x, T, w_router, bias, topk_idx_out, topk_w_out, mode, st);
  if (e == cudaSuccess && events) e = cudaEventRecord(static_cast<cudaEvent_t>(events[1]), st);
  auto evt = [&](int i) { return events ? static_cast<cudaEvent_t>(events[i]) : nullptr; };
  if (e == cudaSuccess && c.gx) e = k3::launch_gather_x(c, w, T, st);
  if (e == cudaSuccess) e = k3::launch_gateup(c, w, routed_records, shared_records, y, T, wgb, st, evt(2));
  if (e == cudaSuccess && events) e = cudaEventRecord(evt(3), st);
  if (e == cudaSuccess) e = k3::launch_down(c, w, routed_records, shared_records, y, T, wgb, st, evt(4), c.Sb == 0);
  if (e == cudaSuccess && c.Sb > 0)
    e = shared_bf16_then_combine(cfg, c, w, L, x, T, shared_records, y, ws, router_tc(cfg, T), st);
  if (e == cudaSuccess && events) e = cudaEventRecord(evt(5), st);
  return cuda_status(e);
}

}  // namespace

extern "C" {

k3moe_status k3moe_layer(const k3moe_config* cfg, const void* x, int64_t T, const float* w_router,
                         const uint16_t* w_router_parts, const float* bias, const uint8_t* routed_records,
                         const uint8_t* shared_records, float* y, int32_t* topk_idx_out, float* topk_w_out, void* ws,
                         size_t ws_bytes, void* stream) {
  return layer_impl(cfg, x, T, w_router, w_router_parts, bias, routed_records, shared_records, y, topk_idx_out,
                    topk_w_out, ws, ws_bytes, stream, nullptr, kDefaultWaitLimit);
}

k3moe_status k3moe_layer_bounded(const k3moe_config* cfg, const void* x, int64_t T, const float* w_router,
                                 const uint16_t* w_router_parts, const float* bias, const uint8_t* routed_records,
                                 const uint8_t* shared_records, float* y, void* ws, size_t ws_bytes, uint32_t wait_limit,
                                 void* stream) {
  return layer_impl(cfg, x, T, w_router, w_router_parts, bias, routed_records, shared_records, y, nullptr, nullptr, ws,
                    ws_bytes, stream, nullptr, wait_limit);
}

k3moe_status k3moe_layer_timed(const k3moe_config* cfg, const void* x, int64_t T, const float* w_router,
                               const uint16_t* w_router_parts, const float* bias, const uint8_t* routed_records,
                               const uint8_t* shared_records, float* y, int32_t* topk_idx_out, float* topk_w_out,
                               void* ws, size_t ws_bytes, void* stream, void* const* events) {
  if (!events) return K3MOE_ERR_INVALID_ARGUMENT;
  return layer_impl(cfg, x, T, w_router, w_router_parts, bias, routed_records, shared_records, y, topk_idx_out,
                    topk_w_out, ws, ws_bytes, stream, events, kDefaultWaitLimit);
}

k3moe_status k3moe_pack_records(const k3moe_config* cfg, uint8_t* records, int64_t n_records, int32_t to_device,
                                void* stream) {
  // only the record geometry matters here (d_model, d_ff, record_stride)
  k3moe_status s = validate_fields(cfg);
  if (s != K3MOE_OK && s != K3MOE_ERR_UNSUPPORTED) return s;
  if (!records || !aligned16(records) || n_records < 0 || (to_device != 0 && to_device != 1))
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (cfg->d_model % 128 || cfg->d_ff % 128) return K3MOE_ERR_UNSUPPORTED;
  if (n_records == 0) return K3MOE_OK;
  return cuda_status(k3::launch_pack_records(records, n_records, cfg->record_stride, cfg->d_model, cfg->d_ff, to_device,
                                            static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_rmsnorm(const float* x, int64_t T, int32_t d, float eps, float* xn, void* stream) {
  if (!x || !xn || T < 0 || d <= 0 || !(eps >= 0.0f)) return K3MOE_ERR_INVALID_ARGUMENT;
  if (T == 0) return K3MOE_OK;
  return cuda_status(k3::launch_rmsnorm(x, T, d, eps, xn, static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_residual_add(float* x, const float* y, int64_t n, void* stream) {
  if (!x || !y || n < 0) return K3MOE_ERR_INVALID_ARGUMENT;
  if (n == 0) return K3MOE_OK;
  return cuda_status(k3::launch_residual_add(x, y, n, static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_residual_rmsnorm(float* x, const float* y, int64_t T, int32_t d, float eps, float* xn,
                                    void* stream) {
  if (!x || !xn || T < 0 || d <= 0 || d % 4 || !(eps >= 0.0f) || !aligned16(x) || !aligned16(xn) ||
      (y && !aligned16(y)))
    return K3MOE_ERR_INVALID_ARGUMENT;
  if (T == 0) return K3MOE_OK;
  return cuda_status(k3::launch_residual_rmsnorm(x, y, T, d, eps, xn, static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_check_device_status(void* ws, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return K3MOE_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int flags = 0;
  if (cudaMemcpyAsync(&flags, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return K3MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return K3MOE_ERR_CUDA;
  if (flags == 0) return K3MOE_OK;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return K3MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return K3MOE_ERR_CUDA;
  return (flags & k3::ST_TIMEOUT) ? K3MOE_ERR_TIMEOUT : K3MOE_ERR_DEVICE_CHECK;
}

const char* k3moe_status_string(k3moe_status s) {
  switch (s) {
    case K3MOE_OK: return "ok";
    case K3MOE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case K3MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case K3MOE_ERR_WORKSPACE: return "workspace too small";
    case K3MOE_ERR_CUDA: return "CUDA error";
    case K3MOE_ERR_DEVICE_CHECK: return "bad data detected on the device";
    case K3MOE_ERR_TIMEOUT: return "bounded wait timed out on the device";
  }
  return "unknown status";
}

}  // extern "C"
