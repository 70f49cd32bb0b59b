// Host-side launch interface between the C-ABI layer (k3moe_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "k3moe_common.cuh"

namespace k3 {

// Launch with programmatic stream serialization: the kernel may be scheduled while the previous
// kernel of the stream still runs; it must call pdl_wait() before reading that kernel's results.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// k3moe_route.cu
// RM_SIGMOID: the sigmoid score with a selection-only bias (else softmax, the bias added to the logits)
enum RouteMode { RM_USER_OUT = 1, RM_XPREP = 2, RM_PERMUTE = 4, RM_LOGITS_READY = 8, RM_SIGMOID = 16 };
cudaError_t launch_route(const Cfg& c, const Ws& ws, const void* x, long long T, const float* W, const float* bias,
                         int* out_idx, float* out_w, int mode, cudaStream_t st);
cudaError_t launch_prep(const Cfg& c, const Ws& ws, const void* x, long long T, const int* idx, const float* w,
                        cudaStream_t st);
// x terms in position order (ws.xp, c.gx): after the permutation and the x terms, before gate/up.
cudaError_t launch_gather_x(const Cfg& c, const Ws& ws, long long T, cudaStream_t st);
cudaError_t launch_rmsnorm(const float* x, long long T, int d, float eps, float* out, cudaStream_t st);
cudaError_t launch_residual_rmsnorm(float* x, const float* y, long long T, int d, float eps, float* out,
                                    cudaStream_t st);

// k3moe_router_tc.cu: router logits on the tensor cores (the token counts where this runs are chosen
// in k3moe_api.cu). `w3` is workspace for the three bf16 parts of the router weights ([3, E, d]), `x3`
// for those of fp32 tokens ([3, T, d]); the logits are written as c.rsplit partial sums ([rsplit, T, E],
// see Cfg).
// `w_parts` ([3, E, d] bf16, prepared at weight-loading time) replaces the per-call split into w3 if given.
cudaError_t launch_router_tc(const Cfg& c, const Ws& ws, const void* x, long long T, const float* W,
                             const void* w_parts, const float* bias, void* w3, void* x3, cudaStream_t st);
// The three bf16 parts of n fp32 values (n a multiple of 4, both pointers 16-byte aligned).
cudaError_t launch_split_router(const float* W, long long n, void* parts, cudaStream_t st);
cudaError_t launch_residual_add(float* x, const float* y, long long n, cudaStream_t st);
// bf16 shared experts (c.Sb of them, records c.sstride bytes apart): gate|up GEMM on the tokens (x, or
// its three bf16 parts x3 for fp32 tokens), GLU into three bf16 parts of h, down GEMM; outputs in ws.sho.
int shared_gemm_splits(long long T, int N, int K, int npairs);
cudaError_t launch_shared_bf16(const Cfg& c, const Ws& ws, const void* x, long long T, const void* x3,
                               const uint8_t* shared, cudaStream_t st);
// The three bf16 parts of n fp32 values into `parts` ([3][n]), as the router does for fp32 tokens.
cudaError_t launch_split_tokens(const float* x, long long n, void* parts, cudaStream_t st);

// k3moe_tc.cu (tcgen05 expert FFN)
// `mid` (optional) is recorded between the projection kernel and the GLU / combine kernel.
cudaError_t launch_gateup(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                          long long T, long long wg_max, cudaStream_t st, cudaEvent_t mid = nullptr);
cudaError_t launch_down(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                        long long T, long long wg_max, cudaStream_t st, cudaEvent_t mid = nullptr,
                        bool combine = true);
// y = the gate-weighted routed outputs (slot order) + the shared experts' outputs.
cudaError_t launch_combine(const Cfg& c, const Ws& ws, float* y, long long T, cudaStream_t st);

// In-place conversion of the records' scale bytes between the stored and the device order.
cudaError_t launch_pack_records(uint8_t* records, long long n_rec, long long stride, int d, int f, int to_device,
                               cudaStream_t st);

}  // namespace k3
