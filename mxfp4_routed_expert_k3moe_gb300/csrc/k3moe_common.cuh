// Device-side definitions shared by the kernels of libk3moe.so (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace k3 {

// ----------------------------------------------------------------------------- configuration
struct Cfg {
  int d, f, E, k, S;  // d_model, d_ff, routed experts, top-k, MXFP4 shared experts (in the work groups)
  int Sb;             // bf16 shared experts (computed apart, added by the combine); S = 0 then
  int nsp1, nsp2;     // reduction parts of the bf16 shared experts' gate|up and down GEMMs
  int x_f32;          // 1 if x is fp32, 0 if bf16
  int wgt;            // max tokens per work group of the gate/up projection
  int wgt_dn;         // ... of the down projection (the permutation writes both lists)
  int fp4;           // 1: activations as E2M1 terms and kind::mxf4 MMAs (few tokens); 0: E4M3 terms, mxf8f6f4
  int xterms;         // terms per activation block of x (E4M3: 2 for bf16 x, 3 for fp32 x; E2M1: 8 or 16)
  int hterms;         // terms per block of h
  int rsplit;         // partial logits the router kernel adds up (parts of the tensor-core reduction; 1: final)
  int gx;             // 1: the gate/up B tiles come from xp (the x terms in position order) by tensor copies
  uint32_t wait_limit;  // polls of a pipeline barrier before a CTA gives up (K3MOE_ERR_TIMEOUT)
  long long stride;   // bytes between routed expert records
  long long sstride;  // bytes between shared expert records
};

// Control block at the start of the workspace (int32 slots).
enum CtrlSlot {
  CTRL_STATUS = 0,       // status bits, read and cleared by k3moe_check_device_status
  CTRL_ROUTER_DONE = 1,  // router token tiles whose top-k is done (the last builds the permutation)
  CTRL_NWG = 2,          // number of work groups built by the permutation
  CTRL_NPOS = 3,         // number of routed positions (slots with a valid expert id)
  CTRL_NWG_DN = 4,       // number of work groups of the down projection's list
  CTRL_WORDS = 64
};
enum StatusBits { ST_BAD_EXPERT = 1, ST_NAN_SCALE = 2, ST_TIMEOUT = 4 };

// Work group: one expert (routed id < E, shared id E + s) and a run of its token positions.
struct WorkGroup {
  int expert, pos0, ntok, pad;
};

// Device pointers into the caller's workspace (offsets computed on the host, see ws_layout).
struct Ws {
  int* ctrl;
  float* logits;      // [rsplit, T, E] partial logits (one part: the logits)
  int* topk_idx;      // [T, k]
  float* topk_w;      // [T, k]
  int* counts;        // [E] tokens per routed expert
  int* cursor;        // [E] fill cursors
  int* offsets;       // [E + 1] first position of each routed expert
  int* wgoff;         // [E + 1] first work group of each routed expert
  int* perm_tok;      // [P] token of each position (P = T*k routed + T*S shared)
  float* perm_w;      // [P] gate weight of each position (1 for shared)
  int* inv;           // [T*k] position of routed slot (t, i), -1 if the slot was rejected
  WorkGroup* wgs;     // [WGmax] work groups of the gate/up projection (wgt positions at most)
  WorkGroup* wgs_dn;  // [WGmax] work groups of the down projection (wgt_dn positions at most)
  uint8_t* xq;        // [T * xterms, d] E4M3 (or [.., d/2] packed E2M1) terms of x (row t*xterms + j)
  uint8_t* xs;        // [T * xterms, d/32] their E8M0 block scales
  uint8_t* xp;        // [P * xterms, d] E4M3 terms of x in position order (row p*xterms + j), when Cfg::gx
  uint8_t* hq;        // [P * hterms, f] E4M3 (or [.., f/2] packed E2M1) terms of h (row p*hterms + j)
  uint8_t* hs;        // [P * hterms, f/32] their E8M0 block scales
  float* part;        // [P, d] down-projection outputs per position (the combine weights them)
  int* rtcnt;         // [T] router CTAs finished per token tile (tiles of 1 to 8 tokens)
  float* sgu;         // [Sb][nsp1][T][2 f] bf16 shared experts: partial sums of gate | up
  uint8_t* sh3;       // [Sb][3][T][f] bf16: their h in three bf16 parts
  float* sho;         // [Sb][nsp2][T][d] partial sums of their outputs (added by the combine)
};

// ----------------------------------------------------------------------------- small helpers
__device__ __forceinline__ float pow2i(int e) {
  // exact 2^e; fast path for normal results
  if (e >= -126 && e <= 127) return __int_as_float((e + 127) << 23);
  return ldexpf(1.0f, e);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// The same kind of split into E2M1 terms (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and signs) with E8M0
// block scales, on a fixed exponent schedule: with E = floor(log2 max|v|) of the block, term j uses
// the scale 2^{E - 3j}. Every scaled residual then lies within [-2, 2], where E2M1 is spaced by 0.5,
// so each rounding leaves at most a quarter of the term's scale: |r_{j+1}| <= 2^{E - 3j - 2}, and the
// next term sees |r_{j+1}| / 2^{E - 3j - 3} <= 2 again. n terms leave at most 2^{E - 3n + 1}, i.e.
// 2^-23 of the block maximum for 8 terms, with one reduction for the block maximum in all. (Scales
// are clamped at 2^-127; elements below that stay unresolved.) Codes are packed two per byte (even
// element in the low nibble): lane l and l ^ 1 share a byte, which the even lane writes to
// codes[j * code_stride + lane / 2]; lane 0 writes the scales.
__device__ __forceinline__ void split_terms_fp4(float v, int terms, uint8_t* codes, long long code_stride,
                                                uint8_t* scales, long long scale_stride, int lane) {
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int E = 0;
  if (amax > 0.0f && amax <= 3.402823466e38f) E = ilogbf(amax);  // max|v| / 2^E in [1, 2)
  float r = v;
  for (int j = 0; j < terms; ++j) {
    int e = E - 3 * j;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    const float s = r * pow2i(-e);
    uint32_t code, dec;
    asm("{\n .reg .b8 t;\n .reg .b16 h;\n cvt.rn.satfinite.e2m1x2.f32 t, %2, %3;\n mov.b16 h, {t, t};\n"
        " cvt.u32.u16 %0, h;\n cvt.rn.f16x2.e2m1x2 %1, t;\n}\n"
        : "=r"(code), "=r"(dec)
        : "f"(0.0f), "f"(s));
    code &= 0xFu;
    r -= __half2float(__ushort_as_half((unsigned short)(dec & 0xFFFFu))) * pow2i(e);
    const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
    if ((lane & 1) == 0) codes[j * code_stride + (lane >> 1)] = (uint8_t)(code | (hi << 4));
    if (lane == 0) scales[j * scale_stride] = (uint8_t)(e + 127);
  }
}

// Programmatic dependent launch: kernels of the layer are launched so that the next one may be
// scheduled before the previous one ends; each waits here for its predecessor grid to complete
// (and its memory to be visible) before it touches anything the predecessor writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Split one 32-element block (one value per lane of the warp) into `terms` E4M3 terms with E8M0
// block scales: term j = RN_e4m3(r_j / 2^{e_j}) with e_j = floor(log2 max|r_j|) - 7 (so the block
// maximum maps into [128, 256), inside E4M3's range), r_0 = v, r_{j+1} = r_j - term_j 2^{e_j}.
// Lane l writes codes[j * code_stride] of its element; lane 0 writes scales[j * scale_stride].
__device__ __forceinline__ void split_terms(float v, int terms, uint8_t* codes, long long code_stride, uint8_t* scales,
                                            long long scale_stride, int lane) {
  float r = v;
  for (int j = 0; j < terms; ++j) {
    float amax = fabsf(r);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = 0;
    if (amax > 0.0f && amax <= 3.402823466e38f) e = ilogbf(amax) - 7;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    const float s = r * pow2i(-e);
    uint16_t q2;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q2) : "f"(0.0f), "f"(s));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q2));
    r -= __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * pow2i(e);
    codes[j * code_stride] = (uint8_t)(q2 & 0xFFu);
    if (lane == 0) scales[j * scale_stride] = (uint8_t)(e + 127);
  }
}

__device__ __forceinline__ void set_status(int* ctrl, int bits) { atomicOr(&ctrl[CTRL_STATUS], bits); }
// GPU-scope release-acquire add, for the last-CTA handshakes: between two CTA barriers, the release
// orders the CTA's earlier writes before the count, and the acquire in the CTA that reads the final
// count orders its later reads after it.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

}  // namespace k3
