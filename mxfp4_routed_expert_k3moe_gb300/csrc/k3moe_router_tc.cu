// Router logits of many tokens on the 5th-generation tensor cores (tcgen05 kind::f16, sm_103a):
//   logits[t, e] = sum_j x[t, j] W[e, j] (+ b[e])
// (kimi-k3-in-c review, table "한눈에 보는 kimi-k3-in-c": 896 routed experts scored per token.)
// The fp32 router weights are split into three bf16 parts, W = W0 + W1 + W2, each the bf16 rounding
// of what the previous parts leave (the differences are exact in fp32), which keeps 24 significant
// bits of every weight; the parts go to the workspace as W3[3][E][d]. bf16 tokens enter the MMA
// exactly and meet the three parts: K = 3 d. fp32 tokens are split the same way into X3[3][T][d], and
// the products X_a W_b with a + b <= 2 are accumulated (6 pairs, K = 6 d); the pairs left out are
// below 2^-24 of the dot product's terms. Accumulation is fp32 in tensor memory. At prefill sizes
// this replaces the CUDA-core dot products, which read the whole router matrix once per tile of 8
// tokens.
//
// One CTA per (128-token tile, 256-expert tile, part of the reduction axis): warp 0 lane 0 issues the
// tensor copies of a 4-stage ring (x tile 128 x 64 and W part tile 256 x 64, bf16, 128-byte swizzle),
// warp 1 lane 0 issues the MMAs (M = 128 tokens, N = 256 experts, K = 16 each), and the four warps
// then read the accumulator (lane = token) and store the partial logits (the bias added to part 0).
// With few tokens the reduction axis is cut into parts so that the grid fills the SMs; the router
// kernel adds the parts, in part order, when it reads the logits. Every wait is bounded.
//
// The same kernel computes the bf16 shared experts' projections (the variant whose non-routed weights
// are bf16): C[t, n] = sum over parts a of A_a[t, :] . B[n, :], with A the tokens (one bf16 part, or
// three for fp32 tokens) or h in three bf16 parts, and B a bf16 weight matrix as stored (gate and up
// stacked as [2 f, d], or down [d, f]); k_shared_glu forms h = SiLU(g) * u between the two.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "k3moe_kernels.h"
#include "k3moe_ptx.cuh"

namespace k3 {

namespace {

using namespace ptx;

constexpr int kRM = 128;                  // tokens per tile (MMA M)
constexpr int kRN = 256;                  // experts per tile (MMA N)
constexpr int kRK = 64;                   // bf16 elements per stage along the reduction axis (one 128-byte row)
constexpr int kRStages = 4;
constexpr int kRThreads = 128;
constexpr int kRA = kRM * kRK * 2;        // 16 KB
constexpr int kRB = kRN * kRK * 2;        // 32 KB
constexpr uint32_t kRWaitLimit = 1u << 24;  // bound of the drain waits (the pipeline's come with the call)
constexpr uint32_t kRPollTestBelow = 64;    // pipeline bounds below this poll with test_wait

struct RCtl {
  uint64_t full[kRStages];
  uint64_t empty[kRStages];
  uint64_t done;
  uint32_t tmem;
  volatile int abort;
};

// Pipeline wait: at most `limit` polls, then ST_TIMEOUT and the CTA's abort flag.
__device__ __forceinline__ bool rwait(uint32_t bar, uint32_t parity, RCtl* ctl, int* status, uint32_t limit) {
  const bool test = limit < kRPollTestBelow;
  for (uint32_t it = 0; it < limit; ++it) {
    if (test ? mbar_test(bar, parity) : mbar_try(bar, parity)) return true;
    if (ctl->abort) return false;
    if (it > 256) __nanosleep(64);
  }
  ctl->abort = 1;
  atomicOr(&status[CTRL_STATUS], ST_TIMEOUT);
  return false;
}

// Wait for copies or MMAs this CTA started (bounded, not cut short by the abort flag).
__device__ __forceinline__ bool rdrain(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kRWaitLimit; ++it) {
    if (mbar_try(bar, parity)) return true;
    if (it > 256) __nanosleep(64);
  }
  return false;
}

// Pairs (token part, weight part) of the reduction, in order: bf16 tokens use the first three. With
// pair_b0 set (the shared experts' GEMMs) pair a is (A part a, B part 0).
__constant__ int kPairA[6] = {0, 0, 0, 1, 1, 2};
__constant__ int kPairB[6] = {0, 1, 2, 0, 1, 0};

// W3[p][i], p = 0, 1, 2: the three bf16 parts of W[i] (router weights or fp32 tokens); n a multiple of
// 4, W 16-byte aligned: four elements per thread and step (one 16-byte load, three 8-byte stores).
__global__ void __launch_bounds__(256) k_split_w(const float* W, long long n, __nv_bfloat16* w3) {
  pdl_wait();
  pdl_launch_dependents();
  for (long long i = 4 * ((long long)blockIdx.x * blockDim.x + threadIdx.x); i < n;
       i += 4LL * gridDim.x * blockDim.x) {
    const float4 w4 = __ldcs(reinterpret_cast<const float4*>(W + i));
    const float w[4] = {w4.x, w4.y, w4.z, w4.w};
    __nv_bfloat16 p[3][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      p[0][u] = __float2bfloat16_rn(w[u]);
      const float r1 = w[u] - __bfloat162float(p[0][u]);
      p[1][u] = __float2bfloat16_rn(r1);
      p[2][u] = __float2bfloat16_rn(r1 - __bfloat162float(p[1][u]));
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) *reinterpret_cast<uint2*>(w3 + q * n + i) = *reinterpret_cast<const uint2*>(p[q]);
  }
}

__global__ void __launch_bounds__(kRThreads, 1)
    k_router_mma(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                 const float* bias, float* logits, long long T, int E, int d, int npairs, int nsplit, int* status,
                 uint32_t wait_limit, int pair_b0) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  RCtl* ctl = reinterpret_cast<RCtl*>(smem + kRStages * (kRA + kRB));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, nt = blockIdx.y, z = blockIdx.z;
  pdl_wait();  // the weight parts come from the split kernel just before
  pdl_launch_dependents();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&ctl->tmem)), "r"(kRN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(su32(&ctl->full[s]), 1);
      mbar_init(su32(&ctl->empty[s]), 1);
    }
    mbar_init(su32(&ctl->done), 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const int kpp = d / kRK, nk = npairs * kpp;  // k-steps per (token part, weight part) pair, in all
  const int kb = (int)((long long)nk * z / nsplit), ke = (int)((long long)nk * (z + 1) / nsplit);  // this part
  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {  // tensor copies
      int filled = 0;  // stages filled (the last fill of stage s was round (filled - 1 - s) / kRStages)
      for (int ks = kb, s = 0; ks < ke && ok; ++ks) {
        const int i = ks - kb;
        const uint32_t round = (uint32_t)(i / kRStages);
        if (i >= kRStages && !rwait(su32(&ctl->empty[s]), (round - 1) & 1u, ctl, status, wait_limit)) {
          ok = false;
          break;
        }
        filled = i + 1;
        const int pair = ks / kpp, k0 = (ks - pair * kpp) * kRK;
        uint8_t* st = smem + (size_t)s * (kRA + kRB);
        mbar_expect_tx(su32(&ctl->full[s]), kRA + kRB);
        tma_load_3d(su32(st), &map_x, k0, mt * kRM, pair_b0 ? pair : kPairA[pair], su32(&ctl->full[s]));
        tma_load_3d(su32(st + kRA), &map_w, k0, nt * kRN, pair_b0 ? 0 : kPairB[pair], su32(&ctl->full[s]));
        if (++s == kRStages) s = 0;
      }
      // after a timeout, the last fill of every stage lands before the CTA frees its memory (earlier
      // fills were consumed by MMAs that completed before the stage was refilled)
      if (!ok)
        for (int s2 = 0; s2 < kRStages && s2 < filled; ++s2)
          rdrain(su32(&ctl->full[s2]), (uint32_t)((filled - 1 - s2) / kRStages) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMAs
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRN >> 3) << 17) | ((uint32_t)(kRM >> 4) << 24);
      for (int ks = kb, s = 0; ks < ke; ++ks) {
        if (!rwait(su32(&ctl->full[s]), (uint32_t)((ks - kb) / kRStages) & 1u, ctl, status, wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + (size_t)s * (kRA + kRB);
        const uint64_t da = sw128_desc(su32(st)), db = sw128_desc(su32(st + kRA));
#pragma unroll
        for (int k = 0; k < kRK / 16; ++k) tc_mma_bf16(tmem, da + 2 * k, db + 2 * k, idesc, (ks != kb || k) ? 1u : 0u);
        tc_commit(su32(&ctl->empty[s]));
        if (++s == kRStages) s = 0;
      }
      tc_commit(su32(&ctl->done));  // arrives when every MMA issued above has completed
    }
  }
  __syncwarp();
  // epilogue: the accumulator (lane = token, column = expert) goes through shared memory, whose stages
  // are free once every MMA completed (rows of kRN + 1 floats: conflict-free both ways), and each warp
  // then stores whole rows of logits (a thread per accumulator row stored 32 scattered rows per
  // instruction)
  // (every MMA issued has completed once `done` arrives, aborted or not: the wait is not cut short)
  const bool have = __syncthreads_and(__all_sync(0xffffffffu, rdrain(su32(&ctl->done), 0)) && !ctl->abort);
  tc_fence_after();
  float* tile = reinterpret_cast<float*>(smem);
  if (have) {
    const int r = 32 * warp + lane;
    for (int c0 = 0; c0 < kRN; c0 += 32) {
      uint32_t v[32];
      tc_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
      tc_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) tile[r * (kRN + 1) + c0 + j] = __uint_as_float(v[j]);
    }
  }
  __syncthreads();
  if (have) {
    const bool addb = bias && z == 0;
    for (int rr = warp; rr < kRM; rr += kRThreads / 32) {
      const long long t = (long long)mt * kRM + rr;
      if (t >= T) break;
      float* dst = logits + (long long)z * T * E + t * E + (long long)nt * kRN;
      for (int cc = lane; cc < kRN; cc += 32) {
        const int e = nt * kRN + cc;
        if (e < E) dst[cc] = tile[rr * (kRN + 1) + cc] + (addb ? __ldg(&bias[e]) : 0.0f);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRN));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode_r = nullptr;
std::mutex g_mu_r;

cudaError_t encode_fn() {
  std::lock_guard<std::mutex> lock(g_mu_r);
  if (g_encode_r) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
  g_encode_r = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_split_tokens(const float* x, long long n, void* parts, cudaStream_t st) {
  if (n % 4) return cudaErrorInvalidValue;
  return launch_pdl(k_split_w, dim3(4 * 152), dim3(256), 0, st, x, n, static_cast<__nv_bfloat16*>(parts));
}

cudaError_t launch_split_router(const float* W, long long n, void* parts, cudaStream_t st) {
  if (n % 4) return cudaErrorInvalidValue;
  return launch_pdl(k_split_w, dim3(4 * 152), dim3(256), 0, st, W, n, static_cast<__nv_bfloat16*>(parts));
}

cudaError_t launch_router_tc(const Cfg& c, const Ws& ws, const void* x, long long T, const float* W,
                             const void* w_parts, const float* bias, void* w3, void* x3, cudaStream_t st) {
  if (c.d % kRK != 0 || T > (1LL << 31) - kRM || (c.x_f32 && !x3) || c.rsplit < 1 ||
      c.rsplit > (c.x_f32 ? 6 : 3) * (c.d / kRK))
    return cudaErrorInvalidValue;
  cudaError_t e = encode_fn();
  if (e != cudaSuccess) return e;
  const long long n = (long long)c.E * c.d;
  if (w_parts) {  // prepared when the weights were loaded
    w3 = const_cast<void*>(w_parts);
  } else {
    e = launch_pdl(k_split_w, dim3(4 * 152), dim3(256), 0, st, W, n, static_cast<__nv_bfloat16*>(w3));
    if (e != cudaSuccess) return e;
  }
  if (c.x_f32) {  // fp32 tokens: three bf16 parts as well
    e = launch_pdl(k_split_w, dim3(4 * 152), dim3(256), 0, st, static_cast<const float*>(x), T * c.d,
                   static_cast<__nv_bfloat16*>(x3));
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mx, mw;
  {
    cuuint64_t gdim[3] = {(cuuint64_t)c.d, (cuuint64_t)T, (cuuint64_t)(c.x_f32 ? 3 : 1)};
    cuuint64_t gstr[2] = {(cuuint64_t)c.d * 2, (cuuint64_t)(T * c.d * 2)};
    cuuint32_t box[3] = {kRK, kRM, 1}, es[3] = {1, 1, 1};
    if (g_encode_r(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c.x_f32 ? x3 : const_cast<void*>(x), gdim, gstr, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t gdim[3] = {(cuuint64_t)c.d, (cuuint64_t)c.E, 3};
    cuuint64_t gstr[2] = {(cuuint64_t)c.d * 2, (cuuint64_t)n * 2};
    cuuint32_t box[3] = {kRK, kRN, 1}, es[3] = {1, 1, 1};
    if (g_encode_r(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w3, gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static bool attr = false;
  const size_t smem = (size_t)kRStages * (kRA + kRB) + sizeof(RCtl) + 1024;
  if (!attr) {
    if ((e = cudaFuncSetAttribute(k_router_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return e;
    attr = true;
  }
  dim3 grid((unsigned)((T + kRM - 1) / kRM), (unsigned)((c.E + kRN - 1) / kRN), (unsigned)c.rsplit);
  return launch_pdl(k_router_mma, grid, dim3(kRThreads), smem, st, mx, mw, bias, ws.logits, T, c.E, c.d,
                    c.x_f32 ? 6 : 3, c.rsplit, ws.ctrl, c.wait_limit, 0);
}

namespace {

// 3D map over parts of a bf16 matrix [parts][rows][K] (row-major, parts part_stride bytes apart),
// boxes of 64 elements x box_rows rows x 1 part, 128-byte swizzle.
cudaError_t bf16_map(const void* base, long long K, long long rows, long long parts, long long part_stride,
                     int box_rows, CUtensorMap* out) {
  cudaError_t e = encode_fn();
  if (e != cudaSuccess) return e;
  cuuint64_t gdim[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)parts};
  cuuint64_t gstr[2] = {(cuuint64_t)K * 2, (cuuint64_t)part_stride};
  cuuint32_t box[3] = {kRK, (cuuint32_t)box_rows, 1}, es[3] = {1, 1, 1};
  if (g_encode_r(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstr, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// h = SiLU(g) * u from the gate|up partial sums gu[z][t][0 .. 2f) (parts added in order), written as
// three bf16 parts h3[p][t][r] (each the rounding of what the earlier parts leave: 24 significant bits).
__global__ void __launch_bounds__(256) k_shared_glu(const float* gu, int nsp, long long T, int f, int S,
                                                    long long gu_stride, long long h3_stride, __nv_bfloat16* h3) {
  pdl_wait();
  pdl_launch_dependents();
  const long long n = (long long)S * T * f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long s = i / (T * f), rem = i - s * T * f, t = rem / f;
    const int r = (int)(rem - t * f);
    const float* g0 = gu + s * gu_stride + t * 2 * f;
    float g = 0.0f, u = 0.0f;
    for (int z = 0; z < nsp; ++z) {
      g += g0[(long long)z * T * 2 * f + r];
      u += g0[(long long)z * T * 2 * f + f + r];
    }
    const float h = silu(g) * u;
    const __nv_bfloat16 p0 = __float2bfloat16_rn(h);
    const float r1 = h - __bfloat162float(p0);
    const __nv_bfloat16 p1 = __float2bfloat16_rn(r1);
    const __nv_bfloat16 p2 = __float2bfloat16_rn(r1 - __bfloat162float(p1));
    __nv_bfloat16* hp = h3 + s * h3_stride + t * f + r;
    hp[0] = p0;
    hp[T * f] = p1;
    hp[2 * T * f] = p2;
  }
}

cudaError_t launch_bf16_gemm(const CUtensorMap& ma, const CUtensorMap& mb, float* out, long long T, int N, int K,
                             int npairs, int nsplit, int* status, uint32_t wait_limit, cudaStream_t st) {
  static bool attr = false;
  const size_t smem = (size_t)kRStages * (kRA + kRB) + sizeof(RCtl) + 1024;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_router_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((unsigned)((T + kRM - 1) / kRM), (unsigned)((N + kRN - 1) / kRN), (unsigned)nsplit);
  return launch_pdl(k_router_mma, grid, dim3(kRThreads), smem, st, ma, mb, (const float*)nullptr, out, T, N, K, npairs,
                    nsplit, status, wait_limit, 1);
}

}  // namespace

// Reduction parts of a shared-expert GEMM over T tokens: enough (128 x 256) tiles x parts to fill the
// SMs, each part at least 16 of the 64-wide k-steps.
int shared_gemm_splits(long long T, int N, int K, int npairs) {
  const long long tiles = ((T + kRM - 1) / kRM) * ((N + kRN - 1) / kRN);
  const long long nk = (long long)npairs * (K / kRK);
  long long p = 152 / tiles;
  if (p > nk / 16) p = nk / 16;
  return (int)(p < 1 ? 1 : p);
}

cudaError_t launch_shared_bf16(const Cfg& c, const Ws& ws, const void* x, long long T, const void* x3,
                               const uint8_t* shared, cudaStream_t st) {
  if (c.Sb <= 0) return cudaSuccess;
  const int d = c.d, f = c.f;
  const int xparts = c.x_f32 ? 3 : 1;
  const int nsp1 = shared_gemm_splits(T, 2 * f, d, xparts), nsp2 = shared_gemm_splits(T, d, f, 3);
  if (nsp1 != c.nsp1 || nsp2 != c.nsp2) return cudaErrorInvalidValue;  // (the workspace was laid out for these)
  CUtensorMap mx;
  cudaError_t e = bf16_map(c.x_f32 ? x3 : x, d, T, xparts, T * d * 2, kRM, &mx);
  if (e != cudaSuccess) return e;
  const long long gu_stride = (long long)nsp1 * T * 2 * f, h3_stride = 3LL * T * f, o_stride = (long long)nsp2 * T * d;
  for (int s = 0; s < c.Sb; ++s) {
    CUtensorMap mw;
    const uint8_t* rec = shared + (long long)s * c.sstride;
    if ((e = bf16_map(rec, d, 2 * f, 1, 2LL * f * d * 2, kRN, &mw)) != cudaSuccess) return e;
    if ((e = launch_bf16_gemm(mx, mw, ws.sgu + s * gu_stride, T, 2 * f, d, xparts, nsp1, ws.ctrl, c.wait_limit, st)) !=
        cudaSuccess)
      return e;
  }
  long long blocks = ((long long)c.Sb * T * f + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  e = launch_pdl(k_shared_glu, dim3((unsigned)blocks), dim3(256), 0, st, (const float*)ws.sgu, nsp1, T, f, c.Sb,
                 gu_stride, h3_stride, reinterpret_cast<__nv_bfloat16*>(ws.sh3));
  if (e != cudaSuccess) return e;
  for (int s = 0; s < c.Sb; ++s) {
    CUtensorMap mh, md;
    const uint8_t* rec = shared + (long long)s * c.sstride;
    if ((e = bf16_map(ws.sh3 + s * h3_stride * 2, f, T, 3, T * f * 2, kRM, &mh)) != cudaSuccess) return e;
    if ((e = bf16_map(rec + 4LL * f * d, f, d, 1, (long long)d * f * 2, kRN, &md)) != cudaSuccess) return e;
    if ((e = launch_bf16_gemm(mh, md, ws.sho + s * o_stride, T, d, f, 3, nsp2, ws.ctrl, c.wait_limit, st)) != cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

}  // namespace k3
