// Device-side definitions shared by the kernels of libk3moe.so (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace k3 {

// ----------------------------------------------------------------------------- configuration
struct Cfg {
  int d, f, E, k, S;  // d_model, d_ff, routed experts, top-k, shared experts
  int xplanes;        // fp16 planes per activation row: 1 (bf16 x is exact in one plane) or 2 (fp32 x: hi + lo)
  int x_f32;          // 1 if x is fp32, 0 if bf16
  int wgt;            // max tokens per work group
  int ks;             // parts of the gate/up reduction axis (d) processed by separate warps
  long long stride;   // bytes between expert records
};

// Control block at the start of the workspace (int32 slots).
enum CtrlSlot {
  CTRL_STATUS = 0,       // status bits, read and cleared by k3moe_check_device_status
  CTRL_ROUTER_DONE = 1,  // router token tiles whose top-k is done (the last builds the permutation)
  CTRL_NWG = 2,          // number of work groups built by the permutation
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
  float* logits;      // [T, E]
  int* topk_idx;      // [T, k]
  float* topk_w;      // [T, k]
  int* counts;        // [E] tokens per routed expert
  int* cursor;        // [E] fill cursors
  int* offsets;       // [E + 1] first position of each routed expert
  int* wgoff;         // [E + 1] first work group of each routed expert
  int* perm_tok;      // [P] token of each position (P = T*k routed + T*S shared)
  float* perm_w;      // [P] gate weight of each position (1 for shared)
  int* inv;           // [T*k] position of routed slot (t, i), -1 if the slot was rejected
  WorkGroup* wgs;     // [WGmax]
  __half* xact;       // [T, xplanes, d] scaled fp16 planes of x
  int8_t* xexp;       // [T] per-token power-of-two exponent c: plane values = x * 2^c
  __half* hact;       // [P, 2, f] scaled fp16 hi/lo planes of h
  int8_t* hexp;       // [P, f/32]
  float* part;        // [P, d] gate-weighted down-projection outputs per position
  int* tilecnt;       // [d/32] work groups finished per 32-row block of the down projection
  float* gupart;      // [P, ks, 2, f] partial gate/up sums of the ks reduction-axis parts
  int* gucnt;         // [WGmax * f/32] parts finished per (work group, 32-row block)
  int* rtcnt;         // [ceil(T/8)] router CTAs finished per token tile
};

// ----------------------------------------------------------------------------- small helpers
__device__ __forceinline__ float pow2i(int e) {
  // exact 2^e; fast path for normal results
  if (e >= -126 && e <= 127) return __int_as_float((e + 127) << 23);
  return ldexpf(1.0f, e);
}

// Exponent c such that max|v| * 2^c lies in [2^14, 2^15): the block's fp16 plane is then exact
// for bf16 inputs and keeps 11 significant bits (22 with the lo plane) for fp32 values.
__device__ __forceinline__ int plane_exponent(float amax) {
  if (!(amax > 0.0f) || !(amax <= 3.402823466e38f)) return 0;
  int c = 14 - ilogbf(amax);
  return c > 120 ? 120 : c;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
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

// Four packed E2M1 pairs (one 32-bit word = 8 codes, even element in each low nibble) to four
// f16x2 registers holding the exact element values: out[b] = (elem 2b, elem 2b+1).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                uint32_t& o3) {
  asm("{\n"
      " .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}\n"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}

// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate (warp-wide).
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void set_status(int* ctrl, int bits) { atomicOr(&ctrl[CTRL_STATUS], bits); }

}  // namespace k3
