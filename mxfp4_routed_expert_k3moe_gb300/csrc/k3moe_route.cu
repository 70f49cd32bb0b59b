// Router (logits, top-k, renormalised softmax gates), activation preparation and the
// token -> expert permutation of the MXFP4 MoE layer.
//
// Router: logits l_e = x . W_e (+ b_e) over the n_routed experts; the k largest logits are
// selected (equal logits: lower expert id first) and the gates are the softmax restricted to the
// selected logits, which equals the full softmax renormalised over the selection. (Kimi-K3 layer
// shape from the kimi-k3-in-c review, table "한눈에 보는 kimi-k3-in-c": 896 experts, top-16.)
//
// Permutation: routed slots (t, i) are grouped by expert into "positions"; each expert's run of
// positions is cut into work groups of at most `wgt` tokens; the shared experts get one run of T
// positions each. The FFN kernels stream each work group's expert record once.
#include <cstdint>

#include "k3moe_kernels.h"

namespace k3 {

namespace {

constexpr int kMaxE = 4096;
constexpr int kRouteMaxSmem = 200 * 1024;  // router CTA: x tile + permutation scratch + candidates

__device__ __forceinline__ float load_x(const void* x, int x_f32, long long idx) {
  if (x_f32) return reinterpret_cast<const float*>(x)[idx];
  return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[idx] << 16);
}

// Activation terms of the 32-element block of token t starting at element j (lane = element).
__device__ __forceinline__ void xterms_block(const Cfg& c, const Ws& ws, float v, long long t, int j, int lane) {
  if (c.fp4)
    split_terms_fp4(v, c.xterms, ws.xq + (t * c.xterms) * (c.d / 2) + j / 2, c.d / 2,
                    ws.xs + (t * c.xterms) * (c.d / 32) + j / 32, c.d / 32, lane);
  else
    split_terms(v, c.xterms, ws.xq + (t * c.xterms) * c.d + j + lane, c.d,
                ws.xs + (t * c.xterms) * (c.d / 32) + j / 32, c.d / 32, lane);
}

// One warp per token: all activation terms of the token (used by k3moe_expert_ffn's preparation);
// eight blocks' elements are loaded before their terms are formed.
__device__ void xterms_rows(const Cfg& c, const Ws& ws, const void* x, long long T, long long first, long long step) {
  const int lane = threadIdx.x & 31;
  for (long long t = first; t < T; t += step)
    for (int j0 = 0; j0 < c.d; j0 += 8 * 32) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = j0 + 32 * u < c.d ? load_x(x, c.x_f32, t * c.d + j0 + 32 * u + lane) : 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (j0 + 32 * u < c.d) xterms_block(c, ws, v[u], t, j0 + 32 * u, lane);
    }
}

// Orderable 64-bit key: larger logit first, then lower expert id. Key 0 marks an empty entry. -0 is
// keyed as +0, so that the two zeros compare equal (and the lower id wins) as they do in the oracle.
__device__ __forceinline__ unsigned long long topk_key(float l, int e) {
  uint32_t u = __float_as_uint(l);
  if (u == 0x80000000u) u = 0u;
  uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
}
__device__ __forceinline__ int key_expert(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}
__device__ __forceinline__ float key_logit(unsigned long long key) {
  const uint32_t o = (uint32_t)(key >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

template <int R>
__device__ __forceinline__ unsigned long long local_max(const unsigned long long (&key)[R]) {
  unsigned long long t[R];
#pragma unroll
  for (int r = 0; r < R; ++r) t[r] = key[r];
#pragma unroll
  for (int h = R / 2; h >= 1; h /= 2)
#pragma unroll
    for (int r = 0; r < h; ++r) t[r] = t[r + h] > t[r] ? t[r + h] : t[r];
  return t[0];
}

// Warp-wide maximum of one 64-bit key per lane: the high words first, then the low words of the
// lanes that hold the maximal high word (two single-instruction reductions).
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long v) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32));
  const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32) == hi ? (uint32_t)v : 0u);
  return ((unsigned long long)hi << 32) | lo;
}

// One warp: the k largest keys held in registers (R per lane), in descending order; lane r < k
// returns the r-th (0 if fewer than r+1 keys exist). Each round takes the warp-wide maximum of the
// lanes' cached local maxima; only the lane that owned it clears the key and recomputes its maximum.
template <int R>
__device__ unsigned long long warp_topk(unsigned long long (&key)[R], int k) {
  const int lane = threadIdx.x & 31;
  unsigned long long lm = local_max<R>(key);
  unsigned long long mine = 0;
  for (int r = 0; r < k; ++r) {
    const unsigned long long best = warp_max_key(lm);
    if (lane == r) mine = best;
    if (best != 0ull && lm == best) {  // keys are unique: exactly one owner
#pragma unroll
      for (int q = 0; q < R; ++q) key[q] = (key[q] == best) ? 0ull : key[q];
      lm = local_max<R>(key);
    }
  }
  return mine;
}

// Keys of one thread for the block top-k: experts lane + 32 (warp + nw q), q < R. The logits are the
// sums of `np` partial logits `ls` floats apart, added in part order, the loads of KZ parts at a time.
__device__ __forceinline__ float sigmoid_score(float l) { return 1.0f / (1.0f + expf(-l)); }

// The value an expert is ranked by: its logit (softmax score), or with the sigmoid score (SIG)
// sigmoid(logit) + its selection bias (sel_bias, or none if NULL).
template <int R, int KZ, bool SIG>
__device__ __forceinline__ void load_keys(int E, const float* logits_t, long long ls, int np,
                                          const float* sel_bias, unsigned long long (&key)[R]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float l[R];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const int e = lane + 32 * (warp + nw * q);
    l[q] = (e < E) ? __ldcg(&logits_t[e]) : 0.0f;
  }
  for (int z0 = 1; z0 < np; z0 += KZ) {
    float pv[KZ][R];
#pragma unroll
    for (int u = 0; u < KZ; ++u)
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int e = lane + 32 * (warp + nw * q);
        pv[u][q] = (z0 + u < np && e < E) ? __ldcg(&logits_t[(z0 + u) * ls + e]) : 0.0f;
      }
#pragma unroll
    for (int u = 0; u < KZ; ++u)
      if (z0 + u < np)
#pragma unroll
        for (int q = 0; q < R; ++q) l[q] += pv[u][q];
  }
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const int e = lane + 32 * (warp + nw * q);
    float v = l[q];
    if (SIG && e < E) v = sigmoid_score(v) + (sel_bias ? __ldg(&sel_bias[e]) : 0.0f);
    key[q] = (e < E) ? topk_key(v, e) : 0ull;
  }
}

// The k largest keys of one token, in descending order, into sel[0..k). `cand` holds blockDim.x keys,
// `s_thr` 64.
//
// Threshold pass: every warp takes its m = ceil(k / nw) largest keys; these nw m distinct keys are
// all >= their minimum tau, so the k-th largest key is >= tau and the selection lies among the keys
// >= tau. Those candidates (the warps' own picks plus the rest of the keys >= tau; typically a few
// more than k) are gathered in shared memory and each is ranked by counting the candidates above
// it. If more candidates than threads turn up (ties at the threshold's scale, or tiny E), the
// two-stage selection runs instead: every warp's k best, then the k best of those.
template <int R, int KZ, bool SIG>
__device__ void topk_select(int E, int k, const float* logits_t, long long ls, int np, const float* sel_bias,
                            unsigned long long* cand, unsigned long long* sel, unsigned long long* s_thr, int* s_n) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int m = (k + nw - 1) / nw;
  unsigned long long key[R];
  load_keys<R, KZ, SIG>(E, logits_t, ls, np, sel_bias, key);
  const unsigned long long mine = warp_topk<R>(key, m);  // clears the picked keys in `key`
  if (lane < m) s_thr[warp * m + lane] = mine;
  if (threadIdx.x == 0) *s_n = 0;
  __syncthreads();
  // tau: the smallest of the warps' picks (every warp forms the minimum of all nw m picks)
  unsigned long long tv = ~0ull;
  for (int i = lane; i < nw * m; i += 32) tv = s_thr[i] < tv ? s_thr[i] : tv;
  const uint32_t tau_hi = __reduce_min_sync(0xffffffffu, (uint32_t)(tv >> 32));
  const uint32_t tau_lo = __reduce_min_sync(0xffffffffu, (uint32_t)(tv >> 32) == tau_hi ? (uint32_t)tv : 0xFFFFFFFFu);
  const unsigned long long tau = ((unsigned long long)tau_hi << 32) | tau_lo;
  const int cap = blockDim.x;
  // the candidates go to `cand` with one shared-memory atomic per warp: a lane's candidates take the
  // slots after those of the lanes below it
  int cnt = (lane < m && mine != 0ull) ? 1 : 0;
#pragma unroll
  for (int q = 0; q < R; ++q) cnt += (key[q] != 0ull && key[q] >= tau) ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  int base = 0;
  if (lane == 31 && incl > 0) base = atomicAdd(s_n, incl);
  int at = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
  if (lane < m && mine != 0ull) {
    if (at < cap) cand[at] = mine;
    ++at;
  }
#pragma unroll
  for (int q = 0; q < R; ++q)
    if (key[q] != 0ull && key[q] >= tau) {
      if (at < cap) cand[at] = key[q];
      ++at;
    }
  __syncthreads();
  const int n = *s_n;
  if (n <= cap) {
    if ((int)threadIdx.x < n) {
      const unsigned long long v = cand[threadIdx.x];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += (cand[j] > v) ? 1 : 0;
      if (rank < k) sel[rank] = v;
    }
    if ((int)threadIdx.x < k && (int)threadIdx.x >= n) sel[threadIdx.x] = 0ull;  // fewer than k experts
  } else {
    load_keys<R, KZ, SIG>(E, logits_t, ls, np, sel_bias, key);
    const unsigned long long top = warp_topk<R>(key, k);
    cand[warp * 32 + lane] = (lane < k) ? top : 0ull;
    __syncthreads();
    if (warp == 0) {
      unsigned long long c8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) c8[q] = (q < nw) ? cand[q * 32 + lane] : 0ull;
      const unsigned long long best = warp_topk<8>(c8, k);
      if (lane < k) sel[lane] = best;
    }
  }
  __syncthreads();
}

// Top-k and gates of one token, by the whole CTA (2 to 8 warps), from `np` partial logits `ls` floats
// apart. Softmax score (SIG false): ranked by logit, gates = softmax over the selected logits. Sigmoid
// score (kimi-k3-in-c review, list of public-header invariants: the routing bias skews only the
// selection, the combine weights come from the unbiased sigmoid): ranked by sigmoid(logit) + sel_bias,
// gates = the selected sigmoid scores renormalised. `cand` is shared memory for blockDim.x keys. Ends
// with __syncthreads.
// `idx_sm` / `w_sm` (shared memory, or NULL) receive a copy of the selection for the permutation.
// topk_select with the keys per thread that E needs (E <= 4096 with 8 warps).
template <int KZ, bool SIG>
__device__ void topk_select_any(int E, int k, const float* logits_t, long long ls, int np, const float* sel_bias,
                                unsigned long long* cand, unsigned long long* sel, unsigned long long* s_thr, int* s_n) {
  const int nw = blockDim.x >> 5;
  const int per_lane = (E + 32 * nw - 1) / (32 * nw);
  if (per_lane <= 1) topk_select<1, KZ, SIG>(E, k, logits_t, ls, np, sel_bias, cand, sel, s_thr, s_n);
  else if (per_lane <= 2) topk_select<2, KZ, SIG>(E, k, logits_t, ls, np, sel_bias, cand, sel, s_thr, s_n);
  else if (per_lane <= 4) topk_select<4, KZ, SIG>(E, k, logits_t, ls, np, sel_bias, cand, sel, s_thr, s_n);
  else if (per_lane <= 8) topk_select<8, KZ, SIG>(E, k, logits_t, ls, np, sel_bias, cand, sel, s_thr, s_n);
  else topk_select<16, KZ, SIG>(E, k, logits_t, ls, np, sel_bias, cand, sel, s_thr, s_n);
}

// Warp 0 after topk_select: lane r < k takes the r-th selected expert and its gate (written to the
// workspace's and the caller's top-k arrays); lanes >= k return expert -1.
template <bool SIG>
__device__ __forceinline__ void gates_warp(int k, const float* logits_t, long long ls, int np,
                                           const unsigned long long* sel, int* idx_out, float* w_out, int* idx_user,
                                           float* w_user, int& my_e, float& w) {
  const int lane = threadIdx.x & 31;
  const unsigned long long best = (lane < k) ? sel[lane] : 0ull;
  my_e = key_expert(best);
  float ex;
  if (SIG) {  // the unbiased score of the selected expert: its logit again, parts added in order
    float l = 0.0f;
    if (lane < k) {
      l = __ldcg(&logits_t[my_e]);
      for (int z = 1; z < np; ++z) l += __ldcg(&logits_t[z * ls + my_e]);
    }
    ex = (lane < k) ? sigmoid_score(l) : 0.0f;
  } else {
    const float my_l = (lane < k) ? key_logit(best) : 0.0f;  // the key holds the logit's bits
    const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
    ex = (lane < k) ? expf(my_l - lmax) : 0.0f;
  }
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  w = ex / sum;
  if (lane < k) {
    idx_out[lane] = my_e;
    w_out[lane] = w;
    if (idx_user) idx_user[lane] = my_e;
    if (w_user) w_user[lane] = w;
  } else {
    my_e = -1;
  }
}

template <int KZ, bool SIG>
__device__ void topk_block(int E, int k, const float* logits_t, long long ls, int np, const float* sel_bias,
                           unsigned long long* cand, int* idx_out, float* w_out, int* idx_user, float* w_user,
                           int* idx_sm, float* w_sm) {
  __shared__ unsigned long long s_sel[32], s_thr[64];
  __shared__ int s_n;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  topk_select_any<KZ, SIG>(E, k, logits_t, ls, np, sel_bias, cand, s_sel, s_thr, &s_n);
  if (warp == 0) {
    int my_e;
    float w;
    gates_warp<SIG>(k, logits_t, ls, np, s_sel, idx_out, w_out, idx_user, w_user, my_e, w);
    if (lane < k) {
      if (idx_sm) idx_sm[lane] = my_e;
      if (w_sm) w_sm[lane] = w;
    }
  }
  __syncthreads();
}

// One token (T = 1, k <= 32 <= ... selected experts all distinct and valid, as top_k <= n_routed):
// the top-k, the gates and the whole permutation in warp 0, from registers. It writes what the
// general builder writes for one token: routed slot r goes to position p_r = the number of selected
// experts with a lower id (positions sorted by expert), each position is a work group of one token
// in both lists, the shared experts' positions and groups follow at k, k + 1, ...
template <int KZ, bool SIG>
__device__ void topk_permute_one_token(const Cfg& c, const Ws& ws, const float* logits_t, long long ls, int np,
                                       const float* sel_bias, unsigned long long* cand, int* idx_user, float* w_user) {
  __shared__ unsigned long long s_sel[32], s_thr[64];
  __shared__ int s_n;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  topk_select_any<KZ, SIG>(c.E, c.k, logits_t, ls, np, sel_bias, cand, s_sel, s_thr, &s_n);
  if (warp != 0) return;
  int my_e;
  float w;
  gates_warp<SIG>(c.k, logits_t, ls, np, s_sel, ws.topk_idx, ws.topk_w, idx_user, w_user, my_e, w);
  int pos = 0;
  for (int j = 0; j < c.k; ++j) pos += (__shfl_sync(0xffffffffu, my_e, j) < my_e) ? 1 : 0;
  if (lane < c.k) {
    ws.perm_tok[pos] = 0;
    ws.perm_w[pos] = w;
    ws.inv[lane] = pos;
    ws.wgs[pos] = WorkGroup{my_e, pos, 1, 0};
    ws.wgs_dn[pos] = WorkGroup{my_e, pos, 1, 0};
  }
  if (lane < c.S) {
    const int p = c.k + lane;
    ws.perm_tok[p] = 0;
    ws.perm_w[p] = 1.0f;
    ws.wgs[p] = WorkGroup{c.E + lane, p, 1, 0};
    ws.wgs_dn[p] = WorkGroup{c.E + lane, p, 1, 0};
  }
  if (lane == 0) {
    ws.ctrl[CTRL_NWG] = c.k + c.S;
    ws.ctrl[CTRL_NWG_DN] = c.k + c.S;
    ws.ctrl[CTRL_NPOS] = c.k;
  }
}

// Logits from the tensor cores carry the rounding of the MMA's fp32 accumulation (measured ~1e-5 at
// d_model 7168, against ~1e-6 for fp32 dot products), enough to swap two experts whose logits differ
// by a little more than 1e-5, and to move the gates by ~1e-5. Before the final selection of a token,
// the experts whose place could depend on that rounding are recomputed on the CUDA cores and written
// over the partial logits (part 0 takes the value, the other parts zero, so the parts still add up to
// it exactly): where an unselected expert's ranked value (logit, or sigmoid + selection bias) lies
// within kRefineMargin of the k-th value (a tight boundary), those experts and the selected ones
// within the margin of the k-th value; and every selected expert within kRefineMargin of a selected
// neighbour. Every other selected expert stays more than the margin above its neighbours and, at a
// tight boundary, above the k-th value; every other expert more than the margin below the k-th value;
// so the selection and its order are those of exact logits. When nothing is recomputed (the usual
// case) the first selection stands and only its gates are formed. The gates of the experts not
// recomputed carry the tensor cores' rounding (~1e-5).
// (Recomputing every selected expert as well, for gates to ~1e-6, took 23 us per token at 64 tokens.)
// The whole CTA computes the candidates together, kRefineBatch at a time: thread i sums the fp32 products
// of its d / blockDim.x consecutive elements of x and of each candidate's fp32 router row, then the
// warps' sums and the per-warp partials are added in order (+ the bias for the softmax score). If
// more than blockDim.x experts lie within the margin (a token whose logits are all equal, x = 0), the
// tensor-core values stand: exact ties are then exact zeros.
constexpr float kRefineMargin = 2e-4f;
constexpr int kRefineBatch = 16;

template <int R, int KZ, bool SIG>
__device__ int refine_candidates_r(const Cfg& c, float* logits_t, long long ls, int np, const float* sel_bias,
                                    const float* W, const float* logit_bias, const uint8_t* xrow,
                                    const unsigned long long* sel, int* s_cid, int* s_nc,
                                    float (*s_red)[kRefineBatch]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned long long kth = sel[c.k - 1];
  const float vk = key_logit(kth);
  unsigned long long key[R];
  load_keys<R, KZ, SIG>(c.E, logits_t, ls, np, sel_bias, key);
  if (threadIdx.x == 0) *s_nc = 0;
  __syncthreads();
  // experts below the k-th within the margin (then the boundary is tight)
  bool below = false;
#pragma unroll
  for (int q = 0; q < R; ++q)
    if (key[q] != 0ull && key[q] < kth && key_logit(key[q]) >= vk - kRefineMargin) {
      below = true;
      const int at = atomicAdd(s_nc, 1);
      if (at < (int)blockDim.x) s_cid[at] = key_expert(key[q]);
    }
  const bool tight = __syncthreads_or(below);
  // selected experts within the margin of a tight boundary or of a selected neighbour (lane = rank)
  if (warp == 0 && lane < c.k && sel[lane] != 0ull) {
    const float v = key_logit(sel[lane]);
    const bool near = (tight && v - vk <= kRefineMargin) ||
                      (lane > 0 && key_logit(sel[lane - 1]) - v < kRefineMargin) ||
                      (lane + 1 < c.k && v - key_logit(sel[lane + 1]) < kRefineMargin);
    if (near) {
      const int at = atomicAdd(s_nc, 1);
      if (at < (int)blockDim.x) s_cid[at] = key_expert(sel[lane]);
    }
  }
  __syncthreads();
  const int n = *s_nc;
  if (n > (int)blockDim.x) return 0;  // (the tensor-core values stand)
  // this thread's slice of the reduction axis: [j0, j1), a multiple of 4 elements (d is a multiple of 128)
  const int per = ((c.d / 4 + blockDim.x - 1) / blockDim.x) * 4;
  const int j0 = min(c.d, (int)threadIdx.x * per), j1 = min(c.d, j0 + per);
  // one or two candidates (the usual case) and a slice of at most kRefineSlice 4-element steps: each
  // candidate's loads of the slice are all issued before its products (a loop over the steps waited
  // for each in turn)
  constexpr int kRefineSlice = 8;
  if (n <= 2 && j1 - j0 <= 4 * kRefineSlice) {
    for (int u = 0; u < n; ++u) {
      float4 wv[kRefineSlice];
#pragma unroll
      for (int v = 0; v < kRefineSlice; ++v) {
        const int j = j0 + 4 * v;
        wv[v] = j < j1 ? __ldg(reinterpret_cast<const float4*>(W + (long long)s_cid[u] * c.d + j))
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
      float acc = 0.0f;
#pragma unroll
      for (int v = 0; v < kRefineSlice; ++v) {
        const int j = j0 + 4 * v;
        if (j < j1) {  // the products in the order of the general loop below
          float xv[4];
          if (c.x_f32) {
            const float4 q4 = *reinterpret_cast<const float4*>(xrow + 4 * j);
            xv[0] = q4.x; xv[1] = q4.y; xv[2] = q4.z; xv[3] = q4.w;
          } else {
            const uint2 q2 = *reinterpret_cast<const uint2*>(xrow + 2 * j);
            xv[0] = __uint_as_float(q2.x << 16); xv[1] = __uint_as_float(q2.x & 0xFFFF0000u);
            xv[2] = __uint_as_float(q2.y << 16); xv[3] = __uint_as_float(q2.y & 0xFFFF0000u);
          }
          acc = fmaf(wv[v].x, xv[0], acc);
          acc = fmaf(wv[v].y, xv[1], acc);
          acc = fmaf(wv[v].z, xv[2], acc);
          acc = fmaf(wv[v].w, xv[3], acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) s_red[warp][u] = acc;
    }
    __syncthreads();
    if ((int)threadIdx.x < n) {
      const int e = s_cid[threadIdx.x];
      float v = 0.0f;
      for (int w = 0; w < nw; ++w) v += s_red[w][threadIdx.x];
      logits_t[e] = v + (logit_bias ? __ldg(&logit_bias[e]) : 0.0f);
      for (int z = 1; z < np; ++z) logits_t[z * ls + e] = 0.0f;
    }
    __threadfence_block();
    __syncthreads();
    return n;
  }
  for (int b0 = 0; b0 < n; b0 += kRefineBatch) {
    const int nb = min(kRefineBatch, n - b0);
    float acc[kRefineBatch];
#pragma unroll
    for (int u = 0; u < kRefineBatch; ++u) acc[u] = 0.0f;
    for (int j = j0; j < j1; j += 4) {
      float xv[4];
      if (c.x_f32) {
        const float4 q4 = *reinterpret_cast<const float4*>(xrow + 4 * j);
        xv[0] = q4.x; xv[1] = q4.y; xv[2] = q4.z; xv[3] = q4.w;
      } else {
        const uint2 q2 = *reinterpret_cast<const uint2*>(xrow + 2 * j);
        xv[0] = __uint_as_float(q2.x << 16); xv[1] = __uint_as_float(q2.x & 0xFFFF0000u);
        xv[2] = __uint_as_float(q2.y << 16); xv[3] = __uint_as_float(q2.y & 0xFFFF0000u);
      }
#pragma unroll
      for (int u = 0; u < kRefineBatch; ++u)
        if (u < nb) {
          const float4 w4 = __ldg(reinterpret_cast<const float4*>(W + (long long)s_cid[b0 + u] * c.d + j));
          acc[u] = fmaf(w4.x, xv[0], acc[u]);
          acc[u] = fmaf(w4.y, xv[1], acc[u]);
          acc[u] = fmaf(w4.z, xv[2], acc[u]);
          acc[u] = fmaf(w4.w, xv[3], acc[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < kRefineBatch; ++u) {
      float v = acc[u];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_red[warp][u] = v;
    }
    __syncthreads();
    if ((int)threadIdx.x < nb) {
      const int e = s_cid[b0 + threadIdx.x];
      float v = 0.0f;
      for (int w = 0; w < nw; ++w) v += s_red[w][threadIdx.x];
      logits_t[e] = v + (logit_bias ? __ldg(&logit_bias[e]) : 0.0f);
      for (int z = 1; z < np; ++z) logits_t[z * ls + e] = 0.0f;
    }
    __syncthreads();
  }
  __threadfence_block();
  __syncthreads();
  return n;
}

// One token: the selection on the tensor cores' partial logits, then the recomputation of the experts
// near its k-th value (above); the final selection runs on the corrected logits.
template <int KZ, bool SIG>
// Returns the number of experts recomputed (0: no logit changed, and the selection in s_sel stands).
__device__ int refine_candidates(const Cfg& c, float* logits_t, long long ls, int np, const float* sel_bias,
                                 const float* W, const float* logit_bias, const uint8_t* xrow,
                                 unsigned long long* cand, unsigned long long* s_sel) {
  __shared__ unsigned long long s_thr[64];
  __shared__ int s_n, s_nc, s_cid[256];
  __shared__ float s_red[8][kRefineBatch];
  topk_select_any<KZ, SIG>(c.E, c.k, logits_t, ls, np, sel_bias, cand, s_sel, s_thr, &s_n);
  const int nw = blockDim.x >> 5;
  const int per_lane = (c.E + 32 * nw - 1) / (32 * nw);
  if (per_lane <= 1) return refine_candidates_r<1, KZ, SIG>(c, logits_t, ls, np, sel_bias, W, logit_bias, xrow, s_sel, s_cid, &s_nc, s_red);
  if (per_lane <= 2) return refine_candidates_r<2, KZ, SIG>(c, logits_t, ls, np, sel_bias, W, logit_bias, xrow, s_sel, s_cid, &s_nc, s_red);
  if (per_lane <= 4) return refine_candidates_r<4, KZ, SIG>(c, logits_t, ls, np, sel_bias, W, logit_bias, xrow, s_sel, s_cid, &s_nc, s_red);
  if (per_lane <= 8) return refine_candidates_r<8, KZ, SIG>(c, logits_t, ls, np, sel_bias, W, logit_bias, xrow, s_sel, s_cid, &s_nc, s_red);
  return refine_candidates_r<16, KZ, SIG>(c, logits_t, ls, np, sel_bias, W, logit_bias, xrow, s_sel, s_cid, &s_nc, s_red);
}

// Exclusive block-wide scan of two int arrays of length n (in place into out0/out1, total at [n]).
__device__ void block_scan2(const int* in0, const int* in1, int* out0, int* out1, int n, int* s_tmp) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int per = (n + nt - 1) / nt;
  const int lo = tid * per, hi = min(n, lo + per);
  int a = 0, b = 0;
  for (int i = lo; i < hi; ++i) { a += in0[i]; b += in1[i]; }
  // inclusive warp scan
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int ta = __shfl_up_sync(0xffffffffu, ia, o), tb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += ta; ib += tb; }
  }
  if (lane == 31) { s_tmp[warp] = ia; s_tmp[32 + warp] = ib; }
  __syncthreads();
  if (tid == 0) {
    int ra = 0, rb = 0;
    for (int w = 0; w < nw; ++w) {
      int va = s_tmp[w], vb = s_tmp[32 + w];
      s_tmp[w] = ra; s_tmp[32 + w] = rb;
      ra += va; rb += vb;
    }
    out0[n] = ra;
    out1[n] = rb;
  }
  __syncthreads();
  int ra = s_tmp[warp] + ia - a, rb = s_tmp[32 + warp] + ib - b;
  for (int i = lo; i < hi; ++i) {
    int va = in0[i], vb = in1[i];
    out0[i] = ra; out1[i] = rb;
    ra += va; rb += vb;
  }
  __syncthreads();
}

// Ints of permutation scratch in shared memory (256-thread CTAs): the general builder's 6E + 4, the
// small one's 3 x 256 slots + 64.
__host__ __device__ constexpr size_t perm_ints(int E) {
  return 6 * (size_t)E + 4 > 3 * 256 + 64 ? 6 * (size_t)E + 4 : 3 * 256 + 64;
}

// Work groups of one run of n positions from p0 (expert e), at most W positions each, from list slot g.
__device__ __forceinline__ void write_groups(WorkGroup* list, int g, int e, long long p0, long long n, int W) {
  for (long long p = 0; p < n; p += W, ++g) list[g] = WorkGroup{e, (int)(p0 + p), (int)min((long long)W, n - p), 0};
}

// One CTA: positions, inverse map and the two work-group lists (wgt positions each for gate/up,
// wgt_dn for down) for T tokens' routed slots plus the shared experts. `sm` is shared-memory scratch
// of kPermInts(E) ints (counts, cursors, offsets, the two lists' group offsets, scan scratch). The
// slot loops read kPermBatch slots per thread before acting on them (one load latency per batch).
// The order of an expert's positions follows the shared-memory atomics; no result depends on it (the
// projections treat positions independently and the combine adds each token's slots in slot order).
__device__ void build_permutation(const Cfg& c, const Ws& ws, long long T, const int* idx, const float* w, int* sm) {
  __shared__ int s_tmp[64];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int E = c.E, k = c.k, W = c.wgt;
  const int Wd = c.wgt_dn;
  int* counts = sm;
  int* cursor = sm + E;
  int* offsets = sm + 2 * E;      // E + 1
  int* wgoff = sm + 3 * E + 1;    // E + 1
  int* wgoff_dn = sm + 4 * E + 2; // E + 1
  int* scratch = sm + 5 * E + 3;  // E + 1
  const long long nslot = T * k;
  for (int e = tid; e < E; e += nt) { counts[e] = 0; cursor[e] = 0; }
  __syncthreads();
  constexpr int kPermBatch = 8;
  for (long long s0 = tid; s0 < nslot; s0 += (long long)kPermBatch * nt) {
    int ev[kPermBatch];
#pragma unroll
    for (int u = 0; u < kPermBatch; ++u) {
      const long long s = s0 + (long long)u * nt;
      ev[u] = s < nslot ? __ldcg(&idx[s]) : 0;
    }
#pragma unroll
    for (int u = 0; u < kPermBatch; ++u) {
      if (s0 + (long long)u * nt >= nslot) continue;
      if (ev[u] < 0 || ev[u] >= E) set_status(ws.ctrl, ST_BAD_EXPERT);
      else atomicAdd(&counts[ev[u]], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += nt) cursor[e] = (counts[e] + W - 1) / W;  // work groups per expert
  __syncthreads();
  block_scan2(counts, cursor, offsets, wgoff, E, s_tmp);
  for (int e = tid; e < E; e += nt) cursor[e] = (counts[e] + Wd - 1) / Wd;  // down work groups per expert
  __syncthreads();
  block_scan2(cursor, cursor, wgoff_dn, scratch, E, s_tmp);
  for (int e = tid; e < E; e += nt) cursor[e] = 0;
  __syncthreads();
  for (long long s0 = tid; s0 < nslot; s0 += (long long)kPermBatch * nt) {
    int ev[kPermBatch];
    float wv[kPermBatch];
#pragma unroll
    for (int u = 0; u < kPermBatch; ++u) {
      const long long s = s0 + (long long)u * nt;
      ev[u] = s < nslot ? __ldcg(&idx[s]) : -1;
      wv[u] = s < nslot ? __ldcg(&w[s]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kPermBatch; ++u) {
      const long long s = s0 + (long long)u * nt;
      if (s >= nslot) continue;
      const int e = ev[u];
      if (e < 0 || e >= E) { ws.inv[s] = -1; continue; }
      const int pos = offsets[e] + atomicAdd(&cursor[e], 1);
      ws.perm_tok[pos] = (int)(s / k);
      ws.perm_w[pos] = wv[u];
      ws.inv[s] = pos;
    }
  }
  for (int e = tid; e < E; e += nt) {
    write_groups(ws.wgs, wgoff[e], e, offsets[e], counts[e], W);
    write_groups(ws.wgs_dn, wgoff_dn[e], e, offsets[e], counts[e], Wd);
  }
  const long long pr = nslot;  // shared positions start after all routed slots
  const int nwt = (int)((T + W - 1) / W), nwt_d = (int)((T + Wd - 1) / Wd);
  for (int q = tid; q < c.S * nwt; q += nt)
    write_groups(ws.wgs, wgoff[E] + q, E + q / nwt, pr + (long long)(q / nwt) * T + (long long)(q % nwt) * W,
                 min((long long)W, T - (long long)(q % nwt) * W), W);
  for (int q = tid; q < c.S * nwt_d; q += nt)
    write_groups(ws.wgs_dn, wgoff_dn[E] + q, E + q / nwt_d, pr + (long long)(q / nwt_d) * T + (long long)(q % nwt_d) * Wd,
                 min((long long)Wd, T - (long long)(q % nwt_d) * Wd), Wd);
  for (long long q = tid; q < (long long)c.S * T; q += nt) {
    ws.perm_tok[pr + q] = (int)(q % T);
    ws.perm_w[pr + q] = 1.0f;
  }
  if (tid == 0) {
    ws.ctrl[CTRL_NWG] = wgoff[E] + c.S * nwt;
    ws.ctrl[CTRL_NWG_DN] = wgoff_dn[E] + c.S * nwt_d;
    ws.ctrl[CTRL_NPOS] = offsets[E];
  }
  __syncthreads();
}

// The same permutation for at most blockDim.x routed slots, without arrays over the experts: slot s
// (thread s) finds its position by counting the valid slots that sort before it (expert id, then
// slot order), and starts a work group of either list when its rank within its expert is a multiple
// of that list's size; the groups are numbered by a block-wide count of the starts before each
// position.
__device__ void build_permutation_small(const Cfg& c, const Ws& ws, long long T, const int* idx, const float* w,
                                        int* sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int E = c.E, k = c.k, W = c.wgt, Wd = c.wgt_dn;
  const int n = (int)(T * k);
  int* s_e = sm;                // [n] expert of each slot (-1 if invalid)
  int* s_flag = sm + n;         // [n] by position: 1 if the position starts a gate/up group (then its number)
  int* s_flag_dn = sm + 2 * n;  // [n] the same for the down groups
  int* s_wsum = sm + 3 * n;     // [2][32] per-warp start counts
  int e = -1;
  if (tid < n) {
    e = idx[tid];
    if (e < 0 || e >= E) {
      set_status(ws.ctrl, ST_BAD_EXPERT);
      e = -1;
    }
    s_e[tid] = e;
  }
  const int npos = __syncthreads_count(tid < n && e >= 0);
  int pos = -1, same_before = 0, cnt_e = 0;
  if (tid < n && e >= 0) {
    int before = 0;
    for (int q = 0; q < n; ++q) {
      const int eq = s_e[q];
      if (eq < 0) continue;
      before += (eq < e || (eq == e && q < tid)) ? 1 : 0;
      cnt_e += (eq == e) ? 1 : 0;
      same_before += (eq == e && q < tid) ? 1 : 0;
    }
    pos = before;
    ws.perm_tok[pos] = tid / k;
    ws.perm_w[pos] = w[tid];
    s_flag[pos] = (same_before % W == 0) ? 1 : 0;
    s_flag_dn[pos] = (same_before % Wd == 0) ? 1 : 0;
  }
  if (tid < n) ws.inv[tid] = pos;
  __syncthreads();
  // exclusive counts of the work-group starts before each position
  const unsigned bal = __ballot_sync(0xffffffffu, tid < npos && s_flag[tid]);
  const unsigned bal_dn = __ballot_sync(0xffffffffu, tid < npos && s_flag_dn[tid]);
  if (lane == 0) {
    s_wsum[warp] = __popc(bal);
    s_wsum[32 + warp] = __popc(bal_dn);
  }
  __syncthreads();
  int base = 0, base_dn = 0, n_routed_wg = 0, n_routed_wg_dn = 0;
  for (int q = 0; q < nw; ++q) {
    base += (q < warp) ? s_wsum[q] : 0;
    base_dn += (q < warp) ? s_wsum[32 + q] : 0;
    n_routed_wg += s_wsum[q];
    n_routed_wg_dn += s_wsum[32 + q];
  }
  const unsigned below = (1u << lane) - 1u;
  __syncthreads();
  if (tid < npos) {  // now the group numbers of each position
    s_flag[tid] = base + __popc(bal & below);
    s_flag_dn[tid] = base_dn + __popc(bal_dn & below);
  }
  __syncthreads();
  if (tid < n && e >= 0 && same_before % W == 0) ws.wgs[s_flag[pos]] = WorkGroup{e, pos, min(W, cnt_e - same_before), 0};
  if (tid < n && e >= 0 && same_before % Wd == 0)
    ws.wgs_dn[s_flag_dn[pos]] = WorkGroup{e, pos, min(Wd, cnt_e - same_before), 0};
  const long long pr = (long long)n;  // shared positions start after all routed slots
  const int nwt = (int)((T + W - 1) / W), nwt_d = (int)((T + Wd - 1) / Wd);
  for (int q = tid; q < c.S * nwt; q += blockDim.x)
    write_groups(ws.wgs, n_routed_wg + q, E + q / nwt, pr + (long long)(q / nwt) * T + (long long)(q % nwt) * W,
                 min((long long)W, T - (long long)(q % nwt) * W), W);
  for (int q = tid; q < c.S * nwt_d; q += blockDim.x)
    write_groups(ws.wgs_dn, n_routed_wg_dn + q, E + q / nwt_d, pr + (long long)(q / nwt_d) * T + (long long)(q % nwt_d) * Wd,
                 min((long long)Wd, T - (long long)(q % nwt_d) * Wd), Wd);
  for (long long q = tid; q < (long long)c.S * T; q += blockDim.x) {
    ws.perm_tok[pr + q] = (int)(q % T);
    ws.perm_w[pr + q] = 1.0f;
  }
  if (tid == 0) {
    ws.ctrl[CTRL_NWG] = n_routed_wg + c.S * nwt;
    ws.ctrl[CTRL_NWG_DN] = n_routed_wg_dn + c.S * nwt_d;
    ws.ctrl[CTRL_NPOS] = npos;
  }
  __syncthreads();
}

__device__ void permute(const Cfg& c, const Ws& ws, long long T, const int* idx, const float* w, int* sm) {
  if (T * c.k <= (long long)blockDim.x) build_permutation_small(c, ws, T, idx, w, sm);
  else build_permutation(c, ws, T, idx, w, sm);
}

struct RouteArgs {
  Cfg c;
  Ws ws;
  const void* x;
  long long T;
  const float* W;
  const float* bias;
  int* out_idx;
  float* out_w;
  int mode;
};

// Shared-memory layout of the router CTA: [x tile | permutation scratch (aliased)][top-k candidates].
// The x tile is staged only when the CTA computes logits (stage_x).
__host__ __device__ __forceinline__ size_t route_tile_bytes(const Cfg& c, int tt, bool stage_x) {
  const size_t xt = stage_x ? (size_t)tt * c.d * (c.x_f32 ? 4 : 2) : 0;
  const size_t perm = sizeof(int) * perm_ints(c.E);
  const size_t m = xt > perm ? xt : perm;
  return (m + 15) & ~(size_t)15;
}

// Router CTA: 8 warps, two expert rows, each row's reduction axis split in four quarters (one warp
// each), so that every warp issues all router-weight loads of its quarter at once (the weights are
// read once and stream; the latency of one batch is paid, not four). The token tile of x is staged
// in shared memory meanwhile. Warps also produce the E4M3 terms of x, one 32-element block each.
// SIG: the sigmoid score (RM_SIGMOID), selected at launch.
template <int TT, bool SIG>
__global__ void __launch_bounds__(256, 3) k_route(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_last;
  __shared__ float s_part[8][TT];
  __shared__ int s_tk_idx[8 * 32];  // the selection of a single token tile, for the permutation
  __shared__ float s_tk_w[8 * 32];
  const Cfg& c = a.c;
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = warp >> 2, kq = warp & 3;
  // (launch_route gives precomputed logits to k_select; the mode flag is kept here, where the compiled
  // form of the dot-product path measured best, without spills)
  const bool dots = !(a.mode & RM_LOGITS_READY);
  const int e = dots ? blockIdx.x * 2 + r : c.E;
  const long long t0 = (long long)blockIdx.y * TT;
  const int ntt = (int)min((long long)TT, a.T - t0);
  const int esz = c.x_f32 ? 4 : 2;
  const int row_bytes = c.d * esz;
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem + route_tile_bytes(c, TT, dots));

  // quarter [jb, je) of row e: U float4 loads per lane per batch, all issued before any arithmetic
  constexpr int U = 14;
  const int qlen = c.d / 4, jb = kq * qlen, je = dots ? jb + qlen : jb;
  const float* wrow = a.W + (long long)(e < c.E ? e : 0) * c.d;
  uint4 wv[U];
  auto load_batch = [&](int j0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * 128 + lane * 4;
      wv[u] = (e < c.E && j < je) ? ld_stream_v4(wrow + j) : make_uint4(0, 0, 0, 0);
    }
  };
  // The router weights are not written by earlier kernels: the first batch is in flight before the
  // wait for the previous kernels, which may still use the workspace and produce x.
  load_batch(jb);
  pdl_wait();
  pdl_launch_dependents();

  // the token tile of x goes to shared memory (asynchronously, waited for below)
  if (dots) {
    const uint8_t* src = reinterpret_cast<const uint8_t*>(a.x) + t0 * row_bytes;
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(smem);
    const int bytes = ntt * row_bytes;
    for (int off = threadIdx.x * 16; off < bytes; off += blockDim.x * 16)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + off), "l"(src + off) : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  float acc[TT];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) acc[tt] = 0.0f;
  bool waited = false;
  for (int j0 = jb; j0 < je; j0 += 128 * U) {
    if (j0 != jb) load_batch(j0);
    if (!waited) {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();
      waited = true;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * 128 + lane * 4;
      if (j < je) {
        const float w4[4] = {__uint_as_float(wv[u].x), __uint_as_float(wv[u].y), __uint_as_float(wv[u].z),
                             __uint_as_float(wv[u].w)};
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
          if (tt < ntt) {
            float xv[4];
            const uint8_t* xr = smem + tt * row_bytes;
            if (c.x_f32) {
              const float4 q = *reinterpret_cast<const float4*>(xr + 4 * j);
              xv[0] = q.x; xv[1] = q.y; xv[2] = q.z; xv[3] = q.w;
            } else {
              const uint2 q = *reinterpret_cast<const uint2*>(xr + 2 * j);
              xv[0] = __uint_as_float(q.x << 16); xv[1] = __uint_as_float(q.x & 0xFFFF0000u);
              xv[2] = __uint_as_float(q.y << 16); xv[3] = __uint_as_float(q.y & 0xFFFF0000u);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[tt] = fmaf(w4[q], xv[q], acc[tt]);
          }
        }
      }
    }
  }
  if (!waited) {  // (only when the quarter is empty)
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
  }
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) {
    float v = acc[tt];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_part[warp][tt] = v;
  }
  __syncthreads();
  // row sums of the four quarters, in quarter order
  if (threadIdx.x < 2 * TT) {
    const int rr = threadIdx.x / TT, tt = threadIdx.x - rr * TT;
    const int er = blockIdx.x * 2 + rr;
    if (dots && er < c.E && tt < ntt) {
      const float v = ((s_part[4 * rr][tt] + s_part[4 * rr + 1][tt]) + s_part[4 * rr + 2][tt]) + s_part[4 * rr + 3][tt];
      a.ws.logits[(t0 + tt) * c.E + er] = v + (a.bias && !SIG ? a.bias[er] : 0.0f);  // (sigmoid: bias at selection)
    }
  }
  // E4M3 terms of x: warp gw of the grid takes the 32-element blocks gw, gw + 8 * gridDim.x, ...
  if (a.mode & RM_XPREP) {
    for (int blk = blockIdx.x * nw + warp; blk * 32 < c.d; blk += (int)gridDim.x * nw) {
      const int j = blk * 32;
      for (int tt = 0; tt < ntt; ++tt) {
        float v;
        if (dots) {  // from the staged tile
          const uint8_t* xr = smem + tt * row_bytes;
          v = c.x_f32 ? reinterpret_cast<const float*>(xr)[j + lane]
                      : __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(xr)[j + lane] << 16);
        } else {
          v = load_x(a.x, c.x_f32, (t0 + tt) * c.d + j + lane);
        }
        xterms_block(c, a.ws, v, t0 + tt, j, lane);
      }
    }
  }
  // the last CTA of each token tile selects the top-k of its tokens ...
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atom_add_acq_rel_gpu(&a.ws.rtcnt[blockIdx.y], 1);
    s_last = (prev == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  if (a.T == 1 && (a.mode & RM_PERMUTE)) {  // one token: selection and permutation in one warp
    topk_permute_one_token<2, SIG>(c, a.ws, a.ws.logits, a.T * c.E, dots ? 1 : c.rsplit, SIG ? a.bias : nullptr, cand,
                                   (a.mode & RM_USER_OUT) ? a.out_idx : nullptr,
                                   (a.mode & RM_USER_OUT) ? a.out_w : nullptr);
    if (threadIdx.x == 0) a.ws.rtcnt[0] = 0;
    return;
  }
  // one token tile whose routed slots fit the block: the permutation reads the selection from shared memory
  const bool tile_sm = gridDim.y == 1 && (long long)ntt * c.k <= (long long)blockDim.x && ntt * c.k <= 8 * 32;
  for (int tt = 0; tt < ntt; ++tt) {
    const long long t = t0 + tt;
    topk_block<2, SIG>(c.E, c.k, a.ws.logits + t * c.E, a.T * c.E, dots ? 1 : c.rsplit, SIG ? a.bias : nullptr,
                       cand, a.ws.topk_idx + t * c.k,
               a.ws.topk_w + t * c.k,
               (a.mode & RM_USER_OUT) && a.out_idx ? a.out_idx + t * c.k : nullptr,
               (a.mode & RM_USER_OUT) && a.out_w ? a.out_w + t * c.k : nullptr, tile_sm ? s_tk_idx + tt * c.k : nullptr,
               tile_sm ? s_tk_w + tt * c.k : nullptr);
  }
  if (threadIdx.x == 0) a.ws.rtcnt[blockIdx.y] = 0;
  // ... and the last token tile to finish builds the permutation (directly when there is one tile)
  if (gridDim.y > 1) {
    if (threadIdx.x < 32) __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int prev = atomicAdd(&a.ws.ctrl[CTRL_ROUTER_DONE], 1);
      s_last = (prev == (int)gridDim.y - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) a.ws.ctrl[CTRL_ROUTER_DONE] = 0;
  }
  if (a.mode & RM_PERMUTE) {
    if (tile_sm) permute(c, a.ws, a.T, s_tk_idx, s_tk_w, reinterpret_cast<int*>(smem));
    else permute(c, a.ws, a.T, a.ws.topk_idx, a.ws.topk_w, reinterpret_cast<int*>(smem));
  }
}

struct PrepArgs {
  Cfg c;
  Ws ws;
  const void* x;
  long long T;
  const int* idx;
  const float* w;
};

// Activation planes for k3moe_expert_ffn (CTAs 1..), permutation of the given routing (CTA 0).
__global__ void __launch_bounds__(256) k_prep(PrepArgs a) {
  extern __shared__ int s_perm[];  // perm_ints(E) ints
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0) {
    permute(a.c, a.ws, a.T, a.idx, a.w, s_perm);
    return;
  }
  const int warp = threadIdx.x >> 5;
  xterms_rows(a.c, a.ws, a.x, a.T, (long long)(blockIdx.x - 1) * 8 + warp, (long long)(gridDim.x - 1) * 8);
}

__global__ void __launch_bounds__(256) k_rmsnorm(const float* x, long long T, int d, float eps, float* out) {
  __shared__ float s_red[8];
  pdl_wait();
  pdl_launch_dependents();
  for (long long t = blockIdx.x; t < T; t += gridDim.x) {
    const float* xr = x + t * d;
    float ss = 0.0f;
    for (int j = threadIdx.x; j < d; j += blockDim.x) ss = fmaf(xr[j], xr[j], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_red[w];
    const float r = 1.0f / sqrtf(tot / (float)d + eps);
    for (int j = threadIdx.x; j < d; j += blockDim.x) out[t * d + j] = xr[j] * r;
    __syncthreads();
  }
}

__global__ void k_residual_add(float* x, const float* y, long long n) {
  pdl_wait();
  pdl_launch_dependents();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    x[i] += y[i];
}

// x += y (if y), then out = RMSNorm(x), one CTA per token row, 16-byte accesses (d a multiple of 4).
// The dependents are released at once: the next layer's router kernel is scheduled while this one
// runs and starts streaming its weights (which no kernel writes) before it waits for this one.
__global__ void __launch_bounds__(256) k_residual_rmsnorm(float* x, const float* y, long long T, int d, float eps,
                                                          float* out) {
  __shared__ float s_red[8];
  pdl_wait();
  pdl_launch_dependents();
  for (long long t = blockIdx.x; t < T; t += gridDim.x) {
    float* xr = x + t * d;
    float ss = 0.0f;
    for (int j = 4 * threadIdx.x; j < d; j += 4 * blockDim.x) {
      float4 v = *reinterpret_cast<const float4*>(xr + j);
      if (y) {
        const float4 u = *reinterpret_cast<const float4*>(y + t * d + j);
        v.x += u.x;
        v.y += u.y;
        v.z += u.z;
        v.w += u.w;
        *reinterpret_cast<float4*>(xr + j) = v;
      }
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_red[w];
    const float r = 1.0f / sqrtf(tot / (float)d + eps);
    for (int j = 4 * threadIdx.x; j < d; j += 4 * blockDim.x) {  // (the same thread's x values as above)
      const float4 v = *reinterpret_cast<const float4*>(xr + j);
      *reinterpret_cast<float4*>(out + t * d + j) = make_float4(v.x * r, v.y * r, v.z * r, v.w * r);
    }
    __syncthreads();
  }
}

// Selection with logits computed by the tensor cores (k_router_mma): grid (G, T). CTA (0, t) selects
// token t's top-k from the partial logits (added in part order) and the last of these CTAs builds the
// permutation; token t's activation terms are formed by CTAs (1 .. G-1, t), sharing its 32-blocks, or
// with G = 1 by CTA (0, t) first. G by token count (router phase, K3 shape): 5 below 256 tokens (one
// CTA per token spent ~18 us on the terms at 64 tokens, its warps taking 28 blocks in turn each), 2
// below 1024 (512 tokens: 112 us against 133 with G = 1), 1 from 1024 (4096 tokens: 557 us against
// 594 with G = 2 and 638 with G = 5).
__host__ __forceinline__ unsigned select_ctas(long long T) { return T < 256 ? 5u : (T < 1024 ? 2u : 1u); }
// KZ: partial logits loaded per round; MINB: CTAs per SM the registers are sized for (with one part,
// three CTAs per SM; with several, two, whose registers hold four parts' loads without spilling).
template <int KZ, int MINB, bool SIG>
__global__ void __launch_bounds__(256, MINB) k_select(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];  // [x row | permutation scratch][top-k candidates]
  __shared__ int s_last;
  const Cfg& c = a.c;
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long t = blockIdx.y;
  pdl_wait();
  pdl_launch_dependents();
  const int tc0 = gridDim.x > 1 ? 1 : 0;  // first term-forming CTA
  if (blockIdx.x >= tc0 && (a.mode & RM_XPREP)) {
    const int esz = c.x_f32 ? 4 : 2;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(a.x) + t * c.d * esz;
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(smem);
    for (int off = threadIdx.x * 16; off < c.d * esz; off += blockDim.x * 16)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + off), "l"(src + off) : "memory");
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const int n = (int)gridDim.x - tc0;
    for (int blk = ((int)blockIdx.x - tc0) * nw + warp; blk * 32 < c.d; blk += n * nw) {
      const int j = blk * 32;
      const float v = c.x_f32 ? reinterpret_cast<const float*>(smem)[j + lane]
                              : __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(smem)[j + lane] << 16);
      xterms_block(c, a.ws, v, t, j, lane);
    }
    __syncthreads();  // (with G = 1 the x row's shared memory is reused below)
  }
  if (blockIdx.x > 0) return;
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem + route_tile_bytes(c, 1, true));
  if (!(tc0 == 0 && (a.mode & RM_XPREP))) {  // the token's row of x, for the recomputed logits
    const int esz = c.x_f32 ? 4 : 2;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(a.x) + t * c.d * esz;
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(smem);
    for (int off = threadIdx.x * 16; off < c.d * esz; off += blockDim.x * 16)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + off), "l"(src + off) : "memory");
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncthreads();
  }
  __shared__ unsigned long long s_sel1[32];
  const int nref = refine_candidates<KZ, SIG>(c, a.ws.logits + t * c.E, a.T * c.E, c.rsplit, SIG ? a.bias : nullptr,
                                              a.W, SIG ? nullptr : a.bias, smem, cand, s_sel1);
  int* idx_user = (a.mode & RM_USER_OUT) && a.out_idx ? a.out_idx + t * c.k : nullptr;
  float* w_user = (a.mode & RM_USER_OUT) && a.out_w ? a.out_w + t * c.k : nullptr;
  if (nref == 0) {  // no logit changed: the first selection stands, and its gates are formed
    if (warp == 0) {
      int my_e;
      float w;
      gates_warp<SIG>(c.k, a.ws.logits + t * c.E, a.T * c.E, c.rsplit, s_sel1, a.ws.topk_idx + t * c.k,
                      a.ws.topk_w + t * c.k, idx_user, w_user, my_e, w);
    }
    __syncthreads();
  } else {
    topk_block<KZ, SIG>(c.E, c.k, a.ws.logits + t * c.E, a.T * c.E, c.rsplit, SIG ? a.bias : nullptr, cand,
                        a.ws.topk_idx + t * c.k, a.ws.topk_w + t * c.k, idx_user, w_user, nullptr, nullptr);
  }
  // the last selecting CTA builds the permutation
  if (threadIdx.x < 32) __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&a.ws.ctrl[CTRL_ROUTER_DONE], 1);
    s_last = (prev == (int)gridDim.y - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) a.ws.ctrl[CTRL_ROUTER_DONE] = 0;
  if (a.mode & RM_PERMUTE) permute(c, a.ws, a.T, a.ws.topk_idx, a.ws.topk_w, reinterpret_cast<int*>(smem));
}

bool g_route_attr_set = false;
template <int KZ, int MINB, bool SIG>
cudaError_t launch_select(const RouteArgs& a, cudaStream_t st) {
  const size_t smem = route_tile_bytes(a.c, 1, true) + sizeof(unsigned long long) * 256;
  if (smem > (size_t)kRouteMaxSmem) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_select<KZ, MINB, SIG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouteMaxSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(k_select<KZ, MINB, SIG>, dim3(select_ctas(a.T), (unsigned)a.T), dim3(256), smem, st, a);
}

}  // namespace

template <int TT, bool SIG>
cudaError_t launch_route_tt2(const RouteArgs& a, int warps, cudaStream_t st) {
  const size_t smem = route_tile_bytes(a.c, TT, !(a.mode & RM_LOGITS_READY)) + sizeof(unsigned long long) * 32 * warps;
  if (smem > (size_t)kRouteMaxSmem) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_route<TT, SIG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouteMaxSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  // with precomputed logits one CTA per token tile selects, writes the activation terms and permutes
  dim3 grid((a.mode & RM_LOGITS_READY) ? 1u : (unsigned)((a.c.E + 1) / 2), (unsigned)((a.T + TT - 1) / TT));
  return launch_pdl(k_route<TT, SIG>, grid, dim3(warps * 32), smem, st, a);
}

template <int TT>
cudaError_t launch_route_tt(const RouteArgs& a, int warps, cudaStream_t st) {
  return (a.mode & RM_SIGMOID) ? launch_route_tt2<TT, true>(a, warps, st) : launch_route_tt2<TT, false>(a, warps, st);
}

cudaError_t launch_route(const Cfg& c, const Ws& ws, const void* x, long long T, const float* W, const float* bias,
                         int* out_idx, float* out_w, int mode, cudaStream_t st) {
  RouteArgs a{c, ws, x, T, W, bias, out_idx, out_w, mode};
  // largest token tile (<= T) whose staged activations fit in shared memory
  auto fits = [&](int tt, int warps) {
    return route_tile_bytes(c, tt, !(mode & RM_LOGITS_READY)) + sizeof(unsigned long long) * 32 * warps <=
           (size_t)kRouteMaxSmem;
  };
  if (mode & RM_LOGITS_READY)  // selection and activation terms from the tensor cores' partial logits
    return (mode & RM_SIGMOID) ? (c.rsplit > 1 ? launch_select<4, 2, true>(a, st) : launch_select<1, 3, true>(a, st))
                     : (c.rsplit > 1 ? launch_select<4, 2, false>(a, st) : launch_select<1, 3, false>(a, st));
  if (T >= 8 && fits(8, 8)) return launch_route_tt<8>(a, 8, st);
  if (T >= 4 && fits(4, 8)) return launch_route_tt<4>(a, 8, st);
  if (T >= 2 && fits(2, 8)) return launch_route_tt<2>(a, 8, st);
  return launch_route_tt<1>(a, 8, st);
}

cudaError_t launch_prep(const Cfg& c, const Ws& ws, const void* x, long long T, const int* idx, const float* w,
                        cudaStream_t st) {
  PrepArgs a{c, ws, x, T, idx, w};
  long long ctas = 1 + (T + 7) / 8;
  if (ctas > 1 + 152 * 8) ctas = 1 + 152 * 8;
  if (!g_route_attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(int) * perm_ints(kMaxE)));
    if (e != cudaSuccess) return e;
    g_route_attr_set = true;
  }
  return launch_pdl(k_prep, dim3((unsigned)ctas), dim3(256), sizeof(int) * perm_ints(c.E), st, a);
}

// The E4M3 terms of x in position order: row p * xterms + j of xp is row perm_tok[p] * xterms + j of xq,
// for the routed positions below the routed count and every shared position (one warp per row, d bytes
// as 16-byte words). A gate/up work group's B rows are then consecutive rows of xp, one tensor copy
// per chunk, instead of rows gathered by token with 16-byte copies.
__global__ void __launch_bounds__(256) k_gather_x(Cfg c, Ws ws, long long T) {
  pdl_wait();
  pdl_launch_dependents();
  const long long PR = T * c.k, P = T * (c.k + c.S);
  const long long npos = __ldcg(&ws.ctrl[CTRL_NPOS]);
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31, words = c.d / 16;
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < P * c.xterms; r += nwarps) {
    const long long p = r / c.xterms;
    if (p >= npos && p < PR) continue;  // (slots without a valid expert)
    const long long src = (long long)__ldcg(&ws.perm_tok[p]) * c.xterms + (r - p * c.xterms);
    const uint4* s = reinterpret_cast<const uint4*>(ws.xq + src * c.d);
    uint4* o = reinterpret_cast<uint4*>(ws.xp + r * c.d);
    for (int v = lane; v < words; v += 32) o[v] = __ldcg(s + v);
  }
}

cudaError_t launch_gather_x(const Cfg& c, const Ws& ws, long long T, cudaStream_t st) {
  const long long rows = T * (c.k + c.S) * c.xterms;
  long long blocks = (rows + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  return launch_pdl(k_gather_x, dim3((unsigned)blocks), dim3(256), 0, st, c, ws, T);
}

cudaError_t launch_rmsnorm(const float* x, long long T, int d, float eps, float* out, cudaStream_t st) {
  const long long blocks = T < 152 * 16 ? T : 152 * 16;
  return launch_pdl(k_rmsnorm, dim3((unsigned)blocks), dim3(256), 0, st, x, T, d, eps, out);
}

cudaError_t launch_residual_add(float* x, const float* y, long long n, cudaStream_t st) {
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  return launch_pdl(k_residual_add, dim3((unsigned)blocks), dim3(256), 0, st, x, y, n);
}

cudaError_t launch_residual_rmsnorm(float* x, const float* y, long long T, int d, float eps, float* out,
                                    cudaStream_t st) {
  const long long blocks = T < 152 * 16 ? T : 152 * 16;
  return launch_pdl(k_residual_rmsnorm, dim3((unsigned)blocks), dim3(256), 0, st, x, y, T, d, eps, out);
}

}  // namespace k3
