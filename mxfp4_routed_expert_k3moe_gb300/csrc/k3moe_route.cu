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

constexpr int kRouteWarps = 4;  // expert rows per router CTA (one warp each)
constexpr int kRouteTT = 8;     // tokens per router warp
constexpr int kMaxE = 4096;

__device__ __forceinline__ float load_x(const void* x, int x_f32, long long idx) {
  if (x_f32) return reinterpret_cast<const float*>(x)[idx];
  uint32_t b = reinterpret_cast<const uint16_t*>(x)[idx];
  return __uint_as_float(b << 16);
}

// One warp per 32-element block of x: the block's fp16 plane(s) and its exponent.
__device__ void xprep_blocks(const Cfg& c, const Ws& ws, const void* x, long long T, long long first, long long step) {
  const int lane = threadIdx.x & 31;
  const int kb_per_row = c.d / 32;
  const long long nblk = T * kb_per_row;
  for (long long b = first; b < nblk; b += step) {
    const long long t = b / kb_per_row;
    const int kb = (int)(b - t * kb_per_row);
    const float v = load_x(x, c.x_f32, t * c.d + kb * 32 + lane);
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const int e = plane_exponent(a);
    const float s = v * pow2i(e);
    const __half hi = __float2half_rn(s);
    ws.xact[(t * c.xplanes) * c.d + kb * 32 + lane] = hi;
    if (c.xplanes == 2) ws.xact[(t * 2 + 1) * c.d + kb * 32 + lane] = __float2half_rn(s - __half2float(hi));
    if (lane == 0) ws.xexp[t * kb_per_row + kb] = (int8_t)e;
  }
}

// Orderable 64-bit key: larger logit first, then lower expert id. Key 0 marks a taken entry.
__device__ __forceinline__ unsigned long long topk_key(float l, int e) {
  uint32_t u = __float_as_uint(l);
  uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
}

// One warp: top-k of one token's logits and the renormalised softmax gates.
__device__ void topk_token(int E, int k, const float* logits_t, unsigned long long* keys, int* idx_out,
                           float* w_out, int* idx_user, float* w_user) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) keys[e] = topk_key(__ldcg(&logits_t[e]), e);
  __syncwarp();
  int my_e = 0;
  for (int r = 0; r < k; ++r) {
    unsigned long long best = 0;
    for (int e = lane; e < E; e += 32) best = keys[e] > best ? keys[e] : best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e_best = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    __syncwarp();
    if (lane == (e_best & 31)) keys[e_best] = 0ull;
    if (lane == r) my_e = e_best;
    __syncwarp();
  }
  const float my_l = (lane < k) ? __ldcg(&logits_t[my_e]) : 0.0f;
  const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = (lane < k) ? expf(my_l - lmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    const float w = ex / sum;
    idx_out[lane] = my_e;
    w_out[lane] = w;
    if (idx_user) idx_user[lane] = my_e;
    if (w_user) w_user[lane] = w;
  }
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

// One CTA: positions, inverse map and work groups for T tokens' routed slots plus the shared experts.
__device__ void build_permutation(const Cfg& c, const Ws& ws, long long T, const int* idx, const float* w) {
  __shared__ int s_tmp[64];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int E = c.E, k = c.k, W = c.wgt;
  const long long nslot = T * k;
  for (int e = tid; e < E; e += nt) { ws.counts[e] = 0; ws.cursor[e] = 0; }
  __syncthreads();
  for (long long s = tid; s < nslot; s += nt) {
    const int e = idx[s];
    if (e < 0 || e >= E) set_status(ws.ctrl, ST_BAD_EXPERT);
    else atomicAdd(&ws.counts[e], 1);
  }
  __syncthreads();
  // wg counts per expert go into `cursor` temporarily, then the scans
  for (int e = tid; e < E; e += nt) ws.cursor[e] = (ws.counts[e] + W - 1) / W;
  __syncthreads();
  block_scan2(ws.counts, ws.cursor, ws.offsets, ws.wgoff, E, s_tmp);
  for (int e = tid; e < E; e += nt) ws.cursor[e] = 0;
  __syncthreads();
  for (long long s = tid; s < nslot; s += nt) {
    const int e = idx[s];
    if (e < 0 || e >= E) { ws.inv[s] = -1; continue; }
    const int pos = ws.offsets[e] + atomicAdd(&ws.cursor[e], 1);
    ws.perm_tok[pos] = (int)(s / k);
    ws.perm_w[pos] = w[s];
    ws.inv[s] = pos;
  }
  for (int e = tid; e < E; e += nt) {
    const int n = ws.counts[e];
    int g = ws.wgoff[e];
    for (int p = 0; p < n; p += W, ++g) ws.wgs[g] = WorkGroup{e, ws.offsets[e] + p, min(W, n - p), 0};
  }
  const int n_routed_wg = ws.wgoff[E];
  const long long pr = nslot;  // shared positions start after all routed slots
  const int nwt = (int)((T + W - 1) / W);
  for (int q = tid; q < c.S * nwt; q += nt) {
    const int s = q / nwt, i = q % nwt;
    const long long p0 = (long long)i * W;
    ws.wgs[n_routed_wg + q] = WorkGroup{E + s, (int)(pr + (long long)s * T + p0), (int)min((long long)W, T - p0), 0};
  }
  for (long long q = tid; q < (long long)c.S * T; q += nt) {
    ws.perm_tok[pr + q] = (int)(q % T);
    ws.perm_w[pr + q] = 1.0f;
  }
  for (int rb = tid; rb < c.d / 32; rb += nt) ws.tilecnt[rb] = 0;
  if (tid == 0) ws.ctrl[CTRL_NWG] = n_routed_wg + c.S * nwt;
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

__global__ void __launch_bounds__(kRouteWarps * 32) k_route(RouteArgs a) {
  extern __shared__ unsigned long long s_keys[];  // [kRouteWarps][E], used by the last CTA only
  __shared__ int s_last;
  const Cfg& c = a.c;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long nblocks = (long long)gridDim.x * gridDim.y;
  const long long bid = (long long)blockIdx.y * gridDim.x + blockIdx.x;

  if (a.mode & RM_XPREP) xprep_blocks(c, a.ws, a.x, a.T, bid * kRouteWarps + warp, nblocks * kRouteWarps);

  // logits of expert row e for up to kRouteTT tokens
  const int e = blockIdx.x * kRouteWarps + warp;
  const long long t0 = (long long)blockIdx.y * kRouteTT;
  if (e < c.E) {
    float acc[kRouteTT];
#pragma unroll
    for (int tt = 0; tt < kRouteTT; ++tt) acc[tt] = 0.0f;
    const float* wrow = a.W + (long long)e * c.d;
    const int ntt = (int)min((long long)kRouteTT, a.T - t0);
#pragma unroll 2
    for (int j = lane * 4; j < c.d; j += 128) {
      const uint4 wv = ld_stream_v4(wrow + j);
      const float w0 = __uint_as_float(wv.x), w1 = __uint_as_float(wv.y), w2 = __uint_as_float(wv.z),
                  w3 = __uint_as_float(wv.w);
#pragma unroll
      for (int tt = 0; tt < kRouteTT; ++tt) {
        if (tt < ntt) {
          const long long xi = (t0 + tt) * c.d + j;
          float x0, x1, x2, x3;
          if (c.x_f32) {
            const float4 xv = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.x) + xi);
            x0 = xv.x; x1 = xv.y; x2 = xv.z; x3 = xv.w;
          } else {
            const uint2 xv = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(a.x) + xi);
            x0 = __uint_as_float(xv.x << 16); x1 = __uint_as_float(xv.x & 0xFFFF0000u);
            x2 = __uint_as_float(xv.y << 16); x3 = __uint_as_float(xv.y & 0xFFFF0000u);
          }
          acc[tt] = fmaf(w0, x0, acc[tt]);
          acc[tt] = fmaf(w1, x1, acc[tt]);
          acc[tt] = fmaf(w2, x2, acc[tt]);
          acc[tt] = fmaf(w3, x3, acc[tt]);
        }
      }
    }
    const float b = a.bias ? a.bias[e] : 0.0f;
#pragma unroll
    for (int tt = 0; tt < kRouteTT; ++tt) {
      float v = acc[tt];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && tt < ntt) a.ws.logits[(t0 + tt) * c.E + e] = v + b;
    }
  }

  // the last CTA to finish selects the top-k of every token and builds the permutation
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(&a.ws.ctrl[CTRL_ROUTER_DONE], 1);
    s_last = (prev == (int)nblocks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (long long t = warp; t < a.T; t += kRouteWarps) {
    topk_token(c.E, c.k, a.ws.logits + t * c.E, s_keys + (long long)warp * c.E, a.ws.topk_idx + t * c.k,
               a.ws.topk_w + t * c.k, (a.mode & RM_USER_OUT) && a.out_idx ? a.out_idx + t * c.k : nullptr,
               (a.mode & RM_USER_OUT) && a.out_w ? a.out_w + t * c.k : nullptr);
  }
  __syncthreads();
  if (a.mode & RM_PERMUTE) build_permutation(c, a.ws, a.T, a.ws.topk_idx, a.ws.topk_w);
  if (threadIdx.x == 0) a.ws.ctrl[CTRL_ROUTER_DONE] = 0;
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
  if (blockIdx.x == 0) {
    build_permutation(a.c, a.ws, a.T, a.idx, a.w);
    return;
  }
  const int warp = threadIdx.x >> 5;
  xprep_blocks(a.c, a.ws, a.x, a.T, (long long)(blockIdx.x - 1) * 8 + warp, (long long)(gridDim.x - 1) * 8);
}

__global__ void __launch_bounds__(256) k_rmsnorm(const float* x, long long T, int d, float eps, float* out) {
  __shared__ float s_red[8];
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
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    x[i] += y[i];
}

bool g_route_attr_set = false;

}  // namespace

cudaError_t launch_route(const Cfg& c, const Ws& ws, const void* x, long long T, const float* W, const float* bias,
                         int* out_idx, float* out_w, int mode, cudaStream_t st) {
  const size_t smem = sizeof(unsigned long long) * kRouteWarps * (size_t)c.E;
  if (!g_route_attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(unsigned long long) * kRouteWarps * kMaxE));
    if (e != cudaSuccess) return e;
    g_route_attr_set = true;
  }
  RouteArgs a{c, ws, x, T, W, bias, out_idx, out_w, mode};
  dim3 grid((c.E + kRouteWarps - 1) / kRouteWarps, (unsigned)((T + kRouteTT - 1) / kRouteTT));
  k_route<<<grid, kRouteWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prep(const Cfg& c, const Ws& ws, const void* x, long long T, const int* idx, const float* w,
                        cudaStream_t st) {
  PrepArgs a{c, ws, x, T, idx, w};
  long long nblk = T * (c.d / 32);
  long long ctas = 1 + (nblk + 7) / 8;
  if (ctas > 1 + 152 * 8) ctas = 1 + 152 * 8;
  k_prep<<<(unsigned)ctas, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* x, long long T, int d, float eps, float* out, cudaStream_t st) {
  long long blocks = T < 152 * 16 ? T : 152 * 16;
  k_rmsnorm<<<(unsigned)blocks, 256, 0, st>>>(x, T, d, eps, out);
  return cudaGetLastError();
}

cudaError_t launch_residual_add(float* x, const float* y, long long n, cudaStream_t st) {
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  k_residual_add<<<(unsigned)blocks, 256, 0, st>>>(x, y, n);
  return cudaGetLastError();
}

}  // namespace k3
