// Expert FFN of the MXFP4 MoE layer for small token counts per expert (decode):
//   gate/up:  g = W_gate x, u = W_up x, h = SiLU(g) * u        (k_ffn<GATEUP>)
//   down:     o = W_down h, y[t] = sum_i w_i o_i + sum_s o_s   (k_ffn<DOWN>, deterministic combine)
// computed directly on the MXFP4 records (kimi-k3-in-c review, table "KDA·MLA·MoE": the
// experts multiply the 4-bit nibbles without a dequantised copy of the weights).
//
// Scheme (one warp per work item = 32 weight rows of one expert x the tokens of a work group):
//  * Each warp streams its items through a private ring of S shared-memory stages filled with
//    16-byte cp.async copies (S-1 stages in flight, continuous across items). A lane's 16-byte
//    piece is exactly one 32-weight MXFP4 block of one row.
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

constexpr int kFfnWarps = 4;  // warps per CTA (independent streams)
enum { GATEUP = 0, DOWN = 1 };

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Shared-memory stage of one warp: weights, scale bytes, activation blocks, activation exponents.
// Both modes stream two 32-row weight blocks per chunk: gate/up rows R0..R0+31 of the gate and the
// up matrix, or down rows R0..R0+63 as two 32-row blocks.
template <int MODE, int NG>
struct StageLayout {
  static constexpr int NMAT = 2;
  static constexpr int kSlots = NMAT * 4;                 // (matrix, 16-row tile, row g / g+8)
  static constexpr int kW = 0;                            // [slot][lane] 16 B
  static constexpr int kSc = kW + kSlots * 512;           // [slot][g] 4 B (scale bytes of blocks 4j..4j+3)
  static constexpr int kB = kSc + kSlots * 32;            // [mg][g] 64 B (B column block, active lanes)
  static constexpr int kAe = kB + NG * 512;               // [mg][lane] 4 B (h block exponents, down only)
  static constexpr int kBytes = kAe + (MODE == DOWN ? NG * 128 : 0);
};

struct FfnArgs {
  Cfg c;
  Ws ws;
  const uint8_t* routed;
  const uint8_t* shared;
  float* y;
  long long T;
};

// Parts of the gate/up reduction axis: c.ks, but never more than the number of 128-element chunks.
__host__ __device__ __forceinline__ int gateup_parts(const Cfg& c) { return c.ks < c.d / 128 ? c.ks : c.d / 128; }

// Position in a warp's stream of (item, pass, chunk) steps. Gate/up items are
// (work group, 32-row block, reduction part); down items are (work group, 32-row block).
template <int MODE, int NG, int NPL>
struct Iter {
  static constexpr int TP = (MODE == GATEUP) ? NG * 2 / NPL : NG;  // tokens per pass
  long long item, n_items, stride;
  int nrb, parts, nch;
  int wgi, rb, kp, j, j1, pass, npass;
  WorkGroup wg;
  const uint8_t* wrow[2];  // per matrix: codes of row R0 + g, lane offset 16t included
  const uint8_t* srow[2];  // per matrix: scale bytes of row R0 + g
  const __half* bsrc[NG];  // B block of this lane for the current pass (null: zeros / not a B lane)
  const int8_t* esrc[NG];  // h block exponents of this lane's C columns (down only)
  bool vb[NG], vc[NG];

  __device__ void setup_pass(const FfnArgs& a, int lane) {
    const Cfg& c = a.c;
    const int g = lane >> 2, t = lane & 3;
    const bool bactive = (t == (g & 3));
#pragma unroll
    for (int mg = 0; mg < NG; ++mg) {
      const int cgb = 2 * mg + (g >> 2), cgc = 2 * mg + (t >> 1);
      const int tb = pass * TP + (NPL == 1 ? cgb : cgb / 2), tc = pass * TP + (NPL == 1 ? cgc : cgc / 2);
      vb[mg] = bactive && tb < wg.ntok;
      vc[mg] = tc < wg.ntok;
      bsrc[mg] = nullptr;
      esrc[mg] = nullptr;
      if (vb[mg]) {
        if (MODE == GATEUP) {
          const int tok = a.ws.perm_tok[wg.pos0 + tb];
          bsrc[mg] = a.ws.xact + ((long long)tok * NPL + (NPL == 1 ? 0 : (cgb & 1))) * c.d + 32 * t;
        } else {
          bsrc[mg] = a.ws.hact + ((long long)(wg.pos0 + tb) * 2 + (cgb & 1)) * c.f + 32 * t;
        }
      }
      if (MODE == DOWN && vc[mg]) esrc[mg] = a.ws.hexp + (long long)(wg.pos0 + tc) * (c.f / 32);
    }
  }
  __device__ void load(const FfnArgs& a, int lane) {
    if (item >= n_items) return;
    const Cfg& c = a.c;
    const int g = lane >> 2, t = lane & 3;
    const long long per_wg = (long long)nrb * parts;
    wgi = (int)(item / per_wg);
    const int rem = (int)(item - (long long)wgi * per_wg);
    rb = rem / parts;
    kp = rem - rb * parts;
    j = kp * nch / parts;
    j1 = (kp + 1) * nch / parts;
    wg = a.ws.wgs[wgi];
    const uint8_t* rec = wg.expert < c.E ? a.routed + (long long)wg.expert * c.stride
                                         : a.shared + (long long)(wg.expert - c.E) * c.stride;
    const long long nc = (long long)c.d * c.f / 2, ns = (long long)c.d * c.f / 32;
    const int K = (MODE == GATEUP) ? c.d : c.f;
    if (MODE == GATEUP) {
      const long long r = (long long)rb * 32 + g;
      wrow[0] = rec + r * (K / 2) + 16 * t;
      srow[0] = rec + nc + r * (K / 32);
      wrow[1] = rec + nc + ns + r * (K / 2) + 16 * t;
      srow[1] = rec + 2 * nc + ns + r * (K / 32);
    } else {
      const long long r = (long long)rb * 64 + g;
      wrow[0] = rec + 2 * (nc + ns) + r * (K / 2) + 16 * t;
      srow[0] = rec + 2 * (nc + ns) + nc + r * (K / 32);
      wrow[1] = wrow[0] + 32LL * (K / 2);
      srow[1] = srow[0] + 32LL * (K / 32);
    }
    npass = (wg.ntok + TP - 1) / TP;
    pass = 0;
    setup_pass(a, lane);
  }
  __device__ bool valid() const { return item < n_items; }
  __device__ bool last_chunk() const { return j + 1 == j1; }
  __device__ void advance(const FfnArgs& a, int lane) {
    if (++j == j1) {
      if (++pass == npass) {
        item += stride;
        load(a, lane);
      } else {
        j = kp * nch / parts;
        setup_pass(a, lane);
      }
    }
  }
};

template <int MODE, int NG, int NPL>
__device__ __forceinline__ void issue_step(const Iter<MODE, NG, NPL>& p, int K, uint32_t sb, int lane) {
  using SL = StageLayout<MODE, NG>;
  const int g = lane >> 2, t = lane & 3;
  const long long rowb = K / 2, rows_s = K / 32;
#pragma unroll
  for (int m = 0; m < SL::NMAT; ++m)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int rs = 0; rs < 2; ++rs) {
        const int slot = (m * 2 + tt) * 2 + rs;
        const int off = 16 * tt + 8 * rs;
        cp16(sb + SL::kW + slot * 512 + lane * 16, p.wrow[m] + off * rowb + 64 * p.j);
        if (t == 0) cp4(sb + SL::kSc + slot * 32 + g * 4, p.srow[m] + off * rows_s + 4 * p.j);
      }
#pragma unroll
  for (int mg = 0; mg < NG; ++mg) {
    if (p.bsrc[mg]) {
      const __half* src = p.bsrc[mg] + 128 * p.j;
#pragma unroll
      for (int q = 0; q < 4; ++q) cp16(sb + SL::kB + mg * 512 + g * 64 + q * 16, src + 8 * q);
    }
    if (MODE == DOWN && p.esrc[mg]) cp4(sb + SL::kAe + mg * 128 + lane * 4, p.esrc[mg] + 4 * p.j);
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int p) {
  return p == 0 ? v.x : p == 1 ? v.y : p == 2 ? v.z : v.w;
}

// 2^(b - 127) for the E8M0 byte q of word s (b = 0 gives 2^-127; b = 255 is flagged separately).
__device__ __forceinline__ float e8m0_byte(uint32_t s, int q) {
  const uint32_t bits = __byte_perm(s, 0u, 0x0444u | ((uint32_t)q << 12)) >> 1;
  return __uint_as_float(bits > 0x00400000u ? bits : 0x00400000u);
}

// 2^(b - 127 - e): E8M0 weight scale times the activation block's 2^-e.
__device__ __forceinline__ float e8m0_times_pow2(uint32_t s, int q, int e) {
  const int dd = (int)((s >> (8 * q)) & 0xFFu) - e;
  return ((unsigned)(dd - 1) < 254u) ? __int_as_float(dd << 23) : pow2i(dd - 127);
}

template <int MODE, int NG, int NPL>
__device__ __forceinline__ void consume_step(const Iter<MODE, NG, NPL>& cn, uint32_t sb, int lane,
                                             float (&acc)[NG][2][StageLayout<MODE, NG>::NMAT][2], int& bad_scale) {
  using SL = StageLayout<MODE, NG>;
  constexpr int NMAT = SL::NMAT;
  const int g = lane >> 2, t = lane & 3;
  uint4 w[NMAT][2][2];
  uint32_t s[NMAT][2][2];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int rs = 0; rs < 2; ++rs) {
        const int slot = (m * 2 + tt) * 2 + rs;
        w[m][tt][rs] = lds128(sb + SL::kW + slot * 512 + lane * 16);
        s[m][tt][rs] = lds32(sb + SL::kSc + slot * 32 + g * 4);
      }
  uint4 b[NG][4];
  uint32_t ae[NG];
#pragma unroll
  for (int mg = 0; mg < NG; ++mg) {
    if (cn.vb[mg]) {
#pragma unroll
      for (int q = 0; q < 4; ++q) b[mg][q] = lds128(sb + SL::kB + mg * 512 + g * 64 + q * 16);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) b[mg][q] = make_uint4(0, 0, 0, 0);
    }
    ae[mg] = (MODE == DOWN && cn.vc[mg]) ? lds32(sb + SL::kAe + mg * 128 + lane * 4) : 0u;
  }

  // two independent accumulator chains per (tile, matrix): MMAs i = 2p and i = 2p + 1
  float cc[NG][2][NMAT][4], cd[NG][2][NMAT][4];
#pragma unroll
  for (int mg = 0; mg < NG; ++mg)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) cc[mg][tt][m][q] = cd[mg][tt][m][q] = 0.0f;
#pragma unroll
  for (int p = 0; p < 4; ++p) {  // 32-bit word p of each lane's 16-byte block: MMAs i = 2p, 2p+1
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        uint32_t a0_0, a2_0, a0_1, a2_1, a1_0, a3_0, a1_1, a3_1;
        e2m1x8_to_f16x2(word_of(w[m][tt][0], p), a0_0, a2_0, a0_1, a2_1);
        e2m1x8_to_f16x2(word_of(w[m][tt][1], p), a1_0, a3_0, a1_1, a3_1);
#pragma unroll
        for (int mg = 0; mg < NG; ++mg) {
          const uint4& bq = b[mg][p];  // elements 8p .. 8p+7 of the block
          mma_f16_16816(cc[mg][tt][m], a0_0, a1_0, a2_0, a3_0, bq.x, bq.y);
          mma_f16_16816(cd[mg][tt][m], a0_1, a1_1, a2_1, a3_1, bq.z, bq.w);
        }
      }
  }
#pragma unroll
  for (int mg = 0; mg < NG; ++mg)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) cc[mg][tt][m][q] += cd[mg][tt][m][q];
  // scales: C columns 2t, 2t+1 hold blocks q0 = 2(t&1), q0+1 of the chunk
  const int q0 = 2 * (t & 1);
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int rs = 0; rs < 2; ++rs) bad_scale |= (__vcmpeq4(s[m][tt][rs], 0xFFFFFFFFu) != 0u);
  if constexpr (MODE == GATEUP) {
    // one activation exponent per token: applied in the epilogue
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const float fa0 = e8m0_byte(s[m][tt][0], q0), fa1 = e8m0_byte(s[m][tt][0], q0 + 1);
        const float fb0 = e8m0_byte(s[m][tt][1], q0), fb1 = e8m0_byte(s[m][tt][1], q0 + 1);
#pragma unroll
        for (int mg = 0; mg < NG; ++mg) {
          acc[mg][tt][m][0] = fmaf(cc[mg][tt][m][0], fa0, fmaf(cc[mg][tt][m][1], fa1, acc[mg][tt][m][0]));
          acc[mg][tt][m][1] = fmaf(cc[mg][tt][m][2], fb0, fmaf(cc[mg][tt][m][3], fb1, acc[mg][tt][m][1]));
        }
      }
  } else {
#pragma unroll
    for (int mg = 0; mg < NG; ++mg) {
      const int e0 = (int)(int8_t)((ae[mg] >> (8 * q0)) & 0xFFu), e1 = (int)(int8_t)((ae[mg] >> (8 * q0 + 8)) & 0xFFu);
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const float fa0 = e8m0_times_pow2(s[m][tt][0], q0, e0), fa1 = e8m0_times_pow2(s[m][tt][0], q0 + 1, e1);
          const float fb0 = e8m0_times_pow2(s[m][tt][1], q0, e0), fb1 = e8m0_times_pow2(s[m][tt][1], q0 + 1, e1);
          acc[mg][tt][m][0] = fmaf(cc[mg][tt][m][0], fa0, fmaf(cc[mg][tt][m][1], fa1, acc[mg][tt][m][0]));
          acc[mg][tt][m][1] = fmaf(cc[mg][tt][m][2], fb0, fmaf(cc[mg][tt][m][3], fb1, acc[mg][tt][m][1]));
        }
    }
  }
}

// Gate/up epilogue of one pass: partial sums of this reduction part -> gupart (scaled back by 2^-c_t).
template <int NG, int NPL>
__device__ __forceinline__ void epilogue_gateup(const FfnArgs& a, const Iter<GATEUP, NG, NPL>& cn, int lane,
                                                float (&acc)[NG][2][2][2]) {
  const Cfg& c = a.c;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mg = 0; mg < NG; ++mg) {
    float gv[2][2], uv[2][2];
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
        gv[tt][rs] = gs;
        uv[tt][rs] = us;
      }
    const int tl = cn.pass * Iter<GATEUP, NG, NPL>::TP + (NPL == 1 ? 2 * mg + (t >> 1) : mg);
    if (tl < cn.wg.ntok) {
      const long long pos = cn.wg.pos0 + tl;
      const float inv = pow2i(-(int)a.ws.xexp[a.ws.perm_tok[pos]]);
      float* dst = a.ws.gupart + (pos * c.ks + cn.kp) * 2 * c.f;
#pragma unroll
      for (int tt = 0; tt < 2; ++tt)
#pragma unroll
        for (int rs = 0; rs < 2; ++rs) {
          const bool mine = (NPL == 1) ? (tt == (t & 1)) : (tt == (t >> 1) && rs == (t & 1));
          if (mine) {
            const int row = cn.rb * 32 + 16 * tt + 8 * rs + g;
            dst[row] = gv[tt][rs] * inv;
            dst[c.f + row] = uv[tt][rs] * inv;
          }
        }
    }
  }
}

// The last reduction part of a (work group, 32-row block) to finish sums the parts in a fixed
// order, applies h = SiLU(g) * u and writes the fp16 hi/lo planes of h with the block's exponent.
__device__ void finish_gateup(const FfnArgs& a, const WorkGroup& wg, int rb, int parts, int lane) {
  const Cfg& c = a.c;
  const int row = rb * 32 + lane;
  for (int tl = 0; tl < wg.ntok; ++tl) {
    const long long pos = wg.pos0 + tl;
    const float* src = a.ws.gupart + pos * c.ks * 2 * c.f;
    float gs = 0.0f, us = 0.0f;
    for (int kp = 0; kp < parts; ++kp) {
      gs += __ldcg(src + (long long)kp * 2 * c.f + row);
      us += __ldcg(src + (long long)kp * 2 * c.f + c.f + row);
    }
    const float h = silu(gs) * us;
    float amax = fabsf(h);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = plane_exponent(amax);
    const float v = h * pow2i(e);
    const __half hi = __float2half_rn(v);
    a.ws.hact[(pos * 2) * c.f + row] = hi;
    a.ws.hact[(pos * 2 + 1) * c.f + row] = __float2half_rn(v - __half2float(hi));
    if (lane == 0) a.ws.hexp[pos * (c.f / 32) + rb] = (int8_t)e;
  }
}

// Down epilogue: gate-weighted outputs of the pass's tokens for 32 rows into the partial buffer.
template <int NG>
__device__ __forceinline__ void epilogue_down(const FfnArgs& a, const Iter<DOWN, NG, 2>& cn, int lane,
                                              float (&acc)[NG][2][2][2]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mg = 0; mg < NG; ++mg) {
    float ov[2][2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt)
#pragma unroll
        for (int rs = 0; rs < 2; ++rs) {
          float o = acc[mg][tt][m][rs];
          o += __shfl_xor_sync(0xffffffffu, o, 1);
          o += __shfl_xor_sync(0xffffffffu, o, 2);
          ov[m][tt][rs] = o;
        }
    const int tk = cn.pass * NG + mg;
    if (tk < cn.wg.ntok) {
      const long long pos = cn.wg.pos0 + tk;
      const float gwt = a.ws.perm_w[pos];
      const int tt = t >> 1, rs = t & 1;
#pragma unroll
      for (int m = 0; m < 2; ++m)
        a.ws.part[pos * a.c.d + cn.rb * 64 + 32 * m + 16 * tt + 8 * rs + g] = ov[m][tt][rs] * gwt;
    }
  }
}

// The last work group to finish a 32-row block of the down projection sums it for every token,
// in a fixed order (routed slots in top-k order, then shared experts).
__device__ void combine_rows(const FfnArgs& a, int rb, int lane) {
  const Cfg& c = a.c;
  const long long P_R = a.T * c.k;
  for (long long tok = 0; tok < a.T; ++tok) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = rb * 64 + 32 * half + lane;
      float s = 0.0f;
      for (int i = 0; i < c.k; ++i) {
        const int p = a.ws.inv[tok * c.k + i];
        if (p >= 0) s += __ldcg(&a.ws.part[(long long)p * c.d + row]);
      }
      for (int sh = 0; sh < c.S; ++sh) s += __ldcg(&a.ws.part[(P_R + (long long)sh * a.T + tok) * c.d + row]);
      a.y[tok * c.d + row] = s;
    }
  }
}

// Increment a completion counter; true for the warp that completes it (the counter is reset).
__device__ __forceinline__ bool last_arrival(int* cnt, int target, int lane) {
  __syncwarp();
  __threadfence();
  int prev = 0;
  if (lane == 0) prev = atomicAdd(cnt, 1);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != target - 1) return false;
  __threadfence();
  if (lane == 0) *cnt = 0;
  return true;
}

template <int MODE, int NG, int NPL, int S>
__global__ void __launch_bounds__(kFfnWarps * 32) k_ffn(FfnArgs a) {
  using SL = StageLayout<MODE, NG>;
  constexpr int NMAT = SL::NMAT;
  extern __shared__ __align__(128) uint8_t smem[];
  const Cfg& c = a.c;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_wg = a.ws.ctrl[CTRL_NWG];
  const int nrb = (MODE == GATEUP) ? c.f / 32 : c.d / 64;
  const int K = (MODE == GATEUP) ? c.d : c.f;
  // reduction parts: at most one per 128-element chunk, so that no part is empty
  const int parts = (MODE == GATEUP) ? gateup_parts(c) : 1;
  const long long n_items = (long long)n_wg * nrb * parts;
  const long long warps_total = (long long)gridDim.x * kFfnWarps;
  // interleave: consecutive items go to different CTAs (SMs) first
  const long long wid = (long long)warp * gridDim.x + blockIdx.x;
  const uint32_t ring = smem_addr(smem) + warp * (S * SL::kBytes);

  if (MODE == DOWN && n_wg == 0) {  // nothing routed and no shared experts: y = 0
    for (long long i = wid * 32 + lane; i < a.T * c.d; i += warps_total * 32) a.y[i] = 0.0f;
    return;
  }

  Iter<MODE, NG, NPL> prod, cons;
  prod.item = cons.item = wid;
  prod.n_items = cons.n_items = n_items;
  prod.stride = cons.stride = warps_total;
  prod.nrb = cons.nrb = nrb;
  prod.parts = cons.parts = parts;
  prod.nch = cons.nch = K / 128;
  prod.load(a, lane);
  cons.load(a, lane);

  int bad_scale = 0;
  for (int s = 0; s < S - 1; ++s) {  // prologue: S-1 stages in flight
    if (prod.valid()) {
      issue_step(prod, K, ring + s * SL::kBytes, lane);
      prod.advance(a, lane);
    }
    cp_commit();
  }
  float acc[NG][2][NMAT][2];
#pragma unroll
  for (int mg = 0; mg < NG; ++mg)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int m = 0; m < NMAT; ++m) acc[mg][tt][m][0] = acc[mg][tt][m][1] = 0.0f;

  uint32_t st_c = 0, st_p = S - 1;  // consumer / producer stage indices
  while (cons.valid()) {
    __syncwarp();  // every lane is done with the stage about to be refilled
    if (prod.valid()) {
      issue_step(prod, K, ring + st_p * SL::kBytes, lane);
      prod.advance(a, lane);
    }
    cp_commit();
    cp_wait<S - 1>();
    __syncwarp();
    consume_step(cons, ring + st_c * SL::kBytes, lane, acc, bad_scale);
    st_c = (st_c + 1 == S) ? 0 : st_c + 1;
    st_p = (st_p + 1 == S) ? 0 : st_p + 1;
    if (cons.last_chunk()) {
      if constexpr (MODE == GATEUP) epilogue_gateup<NG, NPL>(a, cons, lane, acc);
      else epilogue_down<NG>(a, cons, lane, acc);
#pragma unroll
      for (int mg = 0; mg < NG; ++mg)
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
          for (int m = 0; m < NMAT; ++m) acc[mg][tt][m][0] = acc[mg][tt][m][1] = 0.0f;
      if (cons.pass == cons.npass - 1) {
        if constexpr (MODE == GATEUP) {
          if (last_arrival(&a.ws.gucnt[(long long)cons.wgi * nrb + cons.rb], parts, lane))
            finish_gateup(a, cons.wg, cons.rb, parts, lane);
        } else {
          if (last_arrival(&a.ws.tilecnt[cons.rb], n_wg, lane)) combine_rows(a, cons.rb, lane);
        }
      }
    }
    cons.advance(a, lane);
  }
  cp_wait<0>();
  if (bad_scale) set_status(a.ws.ctrl, ST_NAN_SCALE);
}

int g_num_sms = 0;

void init_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 1;
  }
}

template <int MODE, int NG, int NPL, int S>
cudaError_t launch_one(const FfnArgs& a, long long items, cudaStream_t st) {
  constexpr int smem = kFfnWarps * S * StageLayout<MODE, NG>::kBytes;
  static int bps = -1;
  if (bps < 0) {
    cudaError_t e = cudaFuncSetAttribute(k_ffn<MODE, NG, NPL, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_ffn<MODE, NG, NPL, S>, kFfnWarps * 32, smem) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    bps = n;
  }
  long long need = (items + kFfnWarps - 1) / kFfnWarps;
  long long cap = (long long)g_num_sms * bps;
  unsigned grid = (unsigned)(need < cap ? (need > 0 ? need : 1) : cap);
  k_ffn<MODE, NG, NPL, S><<<grid, kFfnWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gateup(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                          long long T, long long wg_max, cudaStream_t st) {
  init_sms();
  FfnArgs a{c, ws, routed, shared, y, T};
  const long long items = wg_max * (c.f / 32) * gateup_parts(c);
  const bool single = (c.wgt == 1);
  if (c.xplanes == 1)
    return single ? launch_one<GATEUP, 1, 1, 3>(a, items, st) : launch_one<GATEUP, 2, 1, 3>(a, items, st);
  return single ? launch_one<GATEUP, 1, 2, 3>(a, items, st) : launch_one<GATEUP, 2, 2, 3>(a, items, st);
}

cudaError_t launch_down(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                        long long T, long long wg_max, cudaStream_t st) {
  init_sms();
  FfnArgs a{c, ws, routed, shared, y, T};
  const long long items = wg_max * (c.d / 64);
  return c.wgt == 1 ? launch_one<DOWN, 1, 2, 3>(a, items, st) : launch_one<DOWN, 2, 2, 3>(a, items, st);
}

}  // namespace k3
