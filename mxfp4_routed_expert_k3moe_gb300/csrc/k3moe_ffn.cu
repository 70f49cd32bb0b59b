// Expert FFN of the MXFP4 MoE layer for small token counts per expert (decode):
//   gate/up:  g = W_gate x, u = W_up x, h = SiLU(g) * u        (k_gateup)
//   down:     o = W_down h, y[t] = sum_i w_i o_i + sum_s o_s   (k_down, deterministic combine)
// computed directly on the MXFP4 records (kimi-k3-in-c review, table "KDA·MLA·MoE": the
// experts multiply the 4-bit nibbles without a dequantised copy of the weights).
//
// Scheme (one warp per work item = 32 weight rows of one expert x up to a few tokens):
//  * Each lane streams 16-byte pieces of its weight rows with 128-bit non-allocating loads;
//    a 16-byte piece is exactly one 32-weight MXFP4 block of one row.
//  * E2M1 codes are converted in registers to exact f16 pairs (cvt.rn.f16x2.e2m1x2) and fed as
//    the A operand of mma.sync m16n8k16 (16 weight rows x 16 reduction elements).
//  * The reduction axis is permuted inside each 128-element chunk so that lane t of a quad owns
//    block 4j+t. The B operand (activations) puts block q's elements only into column q of each
//    4-column group, so C column q holds the partial dot product of block q alone; the block's
//    E8M0 scale and the activation block's exponent are then applied in fp32 to that column.
//    Products are exact (E2M1 x fp16) and accumulate in fp32.
//  * Activations enter as fp16 planes scaled by a power of two per 32-element block (bf16 x is
//    exact in one plane; fp32 x and h use a hi + lo pair of planes, ~22 significant bits).
#include <cstdint>

#include "k3moe_kernels.h"

namespace k3 {

namespace {

constexpr int kFfnWarps = 4;  // warps per CTA (independent items)

template <int NMAT, int NG>
struct Stage {
  uint4 w[NMAT][2][2];   // [matrix][16-row tile][row g / g+8] : one 32-weight block per lane
  uint32_t s[NMAT][2][2];  // scale bytes of blocks 4j..4j+3 for the same rows
  uint4 b[NG][4];        // activation block (32 fp16) for this lane's B column, or zeros
  uint32_t ae[NG];       // activation exponents of blocks 4j + q0, 4j + q0 + 1 (two int8)
};

struct ItemCtx {
  const uint8_t* codes[2];   // per matrix: [rows][K/2]
  const uint8_t* scales[2];  // per matrix: [rows][K/32]
  int K;
  int R0;                    // first of the 32 weight rows
};

template <int NMAT, int NG>
__device__ __forceinline__ void load_stage(Stage<NMAT, NG>& st, const ItemCtx& it, int j, int g, int t,
                                           const __half* const (&bsrc)[NG], const int8_t* const (&esrc)[NG]) {
  const int rowb = it.K / 2, rows_s = it.K / 32;
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int rs = 0; rs < 2; ++rs) {
        const long long r = it.R0 + 16 * tt + 8 * rs + g;
        st.w[m][tt][rs] = ld_stream_v4(it.codes[m] + r * rowb + 64 * j + 16 * t);
        st.s[m][tt][rs] = ld_nc_u32(it.scales[m] + r * rows_s + 4 * j);
      }
#pragma unroll
  for (int mg = 0; mg < NG; ++mg) {
    if (bsrc[mg]) {
      const __half* p = bsrc[mg] + 128 * j;
#pragma unroll
      for (int q = 0; q < 4; ++q) st.b[mg][q] = ld_v4(p + 8 * q);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) st.b[mg][q] = make_uint4(0, 0, 0, 0);
    }
    st.ae[mg] = esrc[mg] ? (uint32_t)(*reinterpret_cast<const uint16_t*>(esrc[mg] + 4 * j)) : 0u;
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int p) {
  return p == 0 ? v.x : p == 1 ? v.y : p == 2 ? v.z : v.w;
}

template <int NMAT, int NG>
__device__ __forceinline__ void compute_stage(const Stage<NMAT, NG>& st, float (&acc)[NG][2][NMAT][2], int t,
                                              int& bad_scale) {
  float c[NG][2][NMAT][4];
#pragma unroll
  for (int mg = 0; mg < NG; ++mg)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) c[mg][tt][m][q] = 0.0f;

#pragma unroll
  for (int p = 0; p < 4; ++p) {  // 32-bit word p of each lane's 16-byte block: MMAs i = 2p, 2p+1
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        uint32_t a0_0, a2_0, a0_1, a2_1, a1_0, a3_0, a1_1, a3_1;
        e2m1x8_to_f16x2(word_of(st.w[m][tt][0], p), a0_0, a2_0, a0_1, a2_1);
        e2m1x8_to_f16x2(word_of(st.w[m][tt][1], p), a1_0, a3_0, a1_1, a3_1);
#pragma unroll
        for (int mg = 0; mg < NG; ++mg) {
          const uint4& bq = st.b[mg][p];  // elements 8p .. 8p+7 of the block
          mma_f16_16816(c[mg][tt][m], a0_0, a1_0, a2_0, a3_0, bq.x, bq.y);
          mma_f16_16816(c[mg][tt][m], a0_1, a1_1, a2_1, a3_1, bq.z, bq.w);
        }
      }
  }
  // scales: C columns 2t, 2t+1 hold blocks q0 = 2(t&1), q0+1 of the chunk
  const int q0 = 2 * (t & 1);
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int rs = 0; rs < 2; ++rs) bad_scale |= (__vcmpeq4(st.s[m][tt][rs], 0xFFFFFFFFu) != 0u);
#pragma unroll
  for (int mg = 0; mg < NG; ++mg) {
    const int e0 = (int)(int8_t)(st.ae[mg] & 0xFFu), e1 = (int)(int8_t)((st.ae[mg] >> 8) & 0xFFu);
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const uint32_t sa = st.s[m][tt][0] >> (8 * q0), sb = st.s[m][tt][1] >> (8 * q0);
        const float fa0 = pow2i((int)(sa & 0xFFu) - 127 - e0), fa1 = pow2i((int)((sa >> 8) & 0xFFu) - 127 - e1);
        const float fb0 = pow2i((int)(sb & 0xFFu) - 127 - e0), fb1 = pow2i((int)((sb >> 8) & 0xFFu) - 127 - e1);
        acc[mg][tt][m][0] = fmaf(c[mg][tt][m][0], fa0, fmaf(c[mg][tt][m][1], fa1, acc[mg][tt][m][0]));
        acc[mg][tt][m][1] = fmaf(c[mg][tt][m][2], fb0, fmaf(c[mg][tt][m][3], fb1, acc[mg][tt][m][1]));
      }
  }
}

// Accumulate one pass: 32 weight rows x (2*NG column groups) over the full reduction axis.
template <int NMAT, int NG>
__device__ __forceinline__ void run_pass(const ItemCtx& it, int g, int t, const __half* const (&bsrc)[NG],
                                         const int8_t* const (&esrc)[NG], float (&acc)[NG][2][NMAT][2],
                                         int& bad_scale) {
#pragma unroll
  for (int mg = 0; mg < NG; ++mg)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int m = 0; m < NMAT; ++m) acc[mg][tt][m][0] = acc[mg][tt][m][1] = 0.0f;
  const int nch = it.K / 128;
  Stage<NMAT, NG> cur, nxt;
  load_stage(cur, it, 0, g, t, bsrc, esrc);
  for (int j = 0; j < nch; ++j) {
    if (j + 1 < nch) load_stage(nxt, it, j + 1, g, t, bsrc, esrc);
    compute_stage(cur, acc, t, bad_scale);
    cur = nxt;
  }
}

struct FfnArgs {
  Cfg c;
  Ws ws;
  const uint8_t* routed;
  const uint8_t* shared;
  float* y;
  long long T;
};

__device__ __forceinline__ const uint8_t* record_of(const FfnArgs& a, int expert) {
  return expert < a.c.E ? a.routed + (long long)expert * a.c.stride
                        : a.shared + (long long)(expert - a.c.E) * a.c.stride;
}

// ---------------------------------------------------------------------------- gate/up + GLU
// NPL: fp16 planes of x (1 for bf16 input, 2 for fp32 input). A pass covers NG MMA column groups
// pairs = NG * 2 / NPL tokens.
template <int NG, int NPL>
__global__ void __launch_bounds__(kFfnWarps * 32) k_gateup(FfnArgs a) {
  const Cfg& c = a.c;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const long long warps_total = (long long)gridDim.x * kFfnWarps;
  const long long gw = (long long)blockIdx.x * kFfnWarps + (threadIdx.x >> 5);
  const int n_wg = a.ws.ctrl[CTRL_NWG];
  const int nrb = c.f / 32;
  const long long n_items = (long long)n_wg * nrb;
  const long long nc = (long long)c.d * c.f / 2, ns = (long long)c.d * c.f / 32;
  const bool bactive = (t == (g & 3));
  constexpr int TP = NG * 2 / NPL;  // tokens per pass
  int bad_scale = 0;

  for (long long item = gw; item < n_items; item += warps_total) {
    const int wgi = (int)(item / nrb), rb = (int)(item % nrb);
    const WorkGroup wg = a.ws.wgs[wgi];
    const uint8_t* rec = record_of(a, wg.expert);
    ItemCtx it;
    it.codes[0] = rec;
    it.scales[0] = rec + nc;
    it.codes[1] = rec + nc + ns;
    it.scales[1] = rec + 2 * nc + ns;
    it.K = c.d;
    it.R0 = rb * 32;
    for (int p0 = 0; p0 < wg.ntok; p0 += TP) {
      const __half* bsrc[NG];
      const int8_t* esrc[NG];
#pragma unroll
      for (int mg = 0; mg < NG; ++mg) {
        // B-loading lanes: column group 2mg + (g >> 2); C-scaling lanes: 2mg + (t >> 1)
        const int cgb = 2 * mg + (g >> 2), cgc = 2 * mg + (t >> 1);
        const int tb = p0 + (NPL == 1 ? cgb : cgb / 2), tc = p0 + (NPL == 1 ? cgc : cgc / 2);
        bsrc[mg] = nullptr;
        esrc[mg] = nullptr;
        if (bactive && tb < wg.ntok) {
          const int tok = a.ws.perm_tok[wg.pos0 + tb];
          bsrc[mg] = a.ws.xact + ((long long)tok * NPL + (NPL == 1 ? 0 : (cgb & 1))) * c.d + 32 * t;
        }
        if (tc < wg.ntok) {
          const int tok = a.ws.perm_tok[wg.pos0 + tc];
          esrc[mg] = a.ws.xexp + (long long)tok * (c.d / 32) + 2 * (t & 1);
        }
      }
      float acc[NG][2][2][2];
      run_pass<2, NG>(it, g, t, bsrc, esrc, acc, bad_scale);

      // GLU epilogue and the fp16 hi/lo planes of h for the 32 rows (one exponent per token)
#pragma unroll
      for (int mg = 0; mg < NG; ++mg) {
        float hv[2][2];
        float amax = 0.0f;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
          for (int rs = 0; rs < 2; ++rs) {
            float gs = acc[mg][tt][0][rs], us = acc[mg][tt][1][rs];
            gs += __shfl_xor_sync(0xffffffffu, gs, 1);
            us += __shfl_xor_sync(0xffffffffu, us, 1);
            if (NPL == 2) {
              gs += __shfl_xor_sync(0xffffffffu, gs, 2);
              us += __shfl_xor_sync(0xffffffffu, us, 2);
            }
            hv[tt][rs] = silu(gs) * us;
            amax = fmaxf(amax, fabsf(hv[tt][rs]));
          }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int e = plane_exponent(amax);
        const float sc = pow2i(e);
        const int tl = p0 + (NPL == 1 ? 2 * mg + (t >> 1) : mg);
        if (tl < wg.ntok) {
          const long long pos = wg.pos0 + tl;
          // writers: NPL 1 -> lanes t, t^1 share a token: (t&1) picks the tile; NPL 2 -> t picks (tile, row)
#pragma unroll
          for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int rs = 0; rs < 2; ++rs) {
              const bool mine = (NPL == 1) ? (tt == (t & 1)) : (tt == (t >> 1) && rs == (t & 1));
              if (mine) {
                const int row = it.R0 + 16 * tt + 8 * rs + g;
                const float v = hv[tt][rs] * sc;
                const __half hi = __float2half_rn(v);
                a.ws.hact[(pos * 2) * c.f + row] = hi;
                a.ws.hact[(pos * 2 + 1) * c.f + row] = __float2half_rn(v - __half2float(hi));
              }
            }
          if (g == 0 && (NPL == 1 ? (t & 1) == 0 : t == 0)) a.ws.hexp[pos * nrb + rb] = (int8_t)e;
        }
      }
    }
  }
  if (bad_scale) set_status(a.ws.ctrl, ST_NAN_SCALE);
}

// ---------------------------------------------------------------------------- down + combine
// h enters as 2 planes (hi, lo): one token per MMA column-group pair, NG tokens per pass.
template <int NG>
__global__ void __launch_bounds__(kFfnWarps * 32) k_down(FfnArgs a) {
  const Cfg& c = a.c;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const long long warps_total = (long long)gridDim.x * kFfnWarps;
  const long long gw = (long long)blockIdx.x * kFfnWarps + (threadIdx.x >> 5);
  const int n_wg = a.ws.ctrl[CTRL_NWG];
  const int nrb = c.d / 32;
  const long long n_items = (long long)n_wg * nrb;
  const long long nc = (long long)c.d * c.f / 2, ns = (long long)c.d * c.f / 32;
  const bool bactive = (t == (g & 3));
  const long long P_R = a.T * c.k;
  int bad_scale = 0;

  if (n_wg == 0) {  // nothing routed and no shared experts: y = 0
    for (long long i = gw * 32 + lane; i < a.T * c.d; i += warps_total * 32) a.y[i] = 0.0f;
    return;
  }

  for (long long item = gw; item < n_items; item += warps_total) {
    const int wgi = (int)(item / nrb), rb = (int)(item % nrb);
    const WorkGroup wg = a.ws.wgs[wgi];
    const uint8_t* rec = record_of(a, wg.expert);
    ItemCtx it;
    it.codes[0] = rec + 2 * (nc + ns);
    it.scales[0] = rec + 2 * (nc + ns) + nc;
    it.codes[1] = it.codes[0];
    it.scales[1] = it.scales[0];
    it.K = c.f;
    it.R0 = rb * 32;
    for (int p0 = 0; p0 < wg.ntok; p0 += NG) {
      const __half* bsrc[NG];
      const int8_t* esrc[NG];
#pragma unroll
      for (int mg = 0; mg < NG; ++mg) {
        const int tk = p0 + mg;
        const long long pos = wg.pos0 + tk;
        bsrc[mg] = (bactive && tk < wg.ntok) ? a.ws.hact + (pos * 2 + (g >> 2)) * c.f + 32 * t : nullptr;
        esrc[mg] = (tk < wg.ntok) ? a.ws.hexp + pos * (c.f / 32) + 2 * (t & 1) : nullptr;
      }
      float acc[NG][2][1][2];
      run_pass<1, NG>(it, g, t, bsrc, esrc, acc, bad_scale);
#pragma unroll
      for (int mg = 0; mg < NG; ++mg) {
        const int tk = p0 + mg;
        float ov[2][2];
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
          for (int rs = 0; rs < 2; ++rs) {
            float o = acc[mg][tt][0][rs];
            o += __shfl_xor_sync(0xffffffffu, o, 1);
            o += __shfl_xor_sync(0xffffffffu, o, 2);
            ov[tt][rs] = o;
          }
        if (tk < wg.ntok) {
          const long long pos = wg.pos0 + tk;
          const float gwt = a.ws.perm_w[pos];
          const int tt = t >> 1, rs = t & 1;
          a.ws.part[pos * c.d + it.R0 + 16 * tt + 8 * rs + g] = ov[tt][rs] * gwt;
        }
      }
    }
    // the last work group to finish this 32-row block combines it for every token
    __syncwarp();
    __threadfence();
    int prev = 0;
    if (lane == 0) prev = atomicAdd(&a.ws.tilecnt[rb], 1);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev == n_wg - 1) {
      __threadfence();
      const int row = it.R0 + lane;
      for (long long tok = 0; tok < a.T; ++tok) {
        float s = 0.0f;
        for (int i = 0; i < c.k; ++i) {
          const int p = a.ws.inv[tok * c.k + i];
          if (p >= 0) s += __ldcg(&a.ws.part[(long long)p * c.d + row]);
        }
        for (int sh = 0; sh < c.S; ++sh) s += __ldcg(&a.ws.part[(P_R + (long long)sh * a.T + tok) * c.d + row]);
        a.y[tok * c.d + row] = s;
      }
      if (lane == 0) a.ws.tilecnt[rb] = 0;
    }
  }
  if (bad_scale) set_status(a.ws.ctrl, ST_NAN_SCALE);
}

template <typename K>
int blocks_per_sm(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kFfnWarps * 32, 0) != cudaSuccess || n < 1) n = 1;
  return n;
}

int g_num_sms = 0;

}  // namespace

namespace {
void init_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 1;
  }
}

unsigned grid_for(long long items, int bps) {
  long long need = (items + kFfnWarps - 1) / kFfnWarps;
  long long cap = (long long)g_num_sms * bps;
  return (unsigned)(need < cap ? (need > 0 ? need : 1) : cap);
}
}  // namespace

cudaError_t launch_gateup(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                          long long T, long long wg_max, cudaStream_t st) {
  init_sms();
  FfnArgs a{c, ws, routed, shared, y, T};
  const long long items = wg_max * (c.f / 32);
  const bool single = (c.wgt == 1);
  if (c.xplanes == 1) {
    if (single) {
      static int bps = blocks_per_sm(k_gateup<1, 1>);
      k_gateup<1, 1><<<grid_for(items, bps), kFfnWarps * 32, 0, st>>>(a);
    } else {
      static int bps = blocks_per_sm(k_gateup<2, 1>);
      k_gateup<2, 1><<<grid_for(items, bps), kFfnWarps * 32, 0, st>>>(a);
    }
  } else {
    if (single) {
      static int bps = blocks_per_sm(k_gateup<1, 2>);
      k_gateup<1, 2><<<grid_for(items, bps), kFfnWarps * 32, 0, st>>>(a);
    } else {
      static int bps = blocks_per_sm(k_gateup<2, 2>);
      k_gateup<2, 2><<<grid_for(items, bps), kFfnWarps * 32, 0, st>>>(a);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_down(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                        long long T, long long wg_max, cudaStream_t st) {
  init_sms();
  FfnArgs a{c, ws, routed, shared, y, T};
  const long long items = wg_max * (c.d / 32);
  if (c.wgt == 1) {
    static int bps = blocks_per_sm(k_down<1>);
    k_down<1><<<grid_for(items, bps), kFfnWarps * 32, 0, st>>>(a);
  } else {
    static int bps = blocks_per_sm(k_down<2>);
    k_down<2><<<grid_for(items, bps), kFfnWarps * 32, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace k3
