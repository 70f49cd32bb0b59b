// Seeded synthetic inputs for the MXFP4 MoE layer: device-side byte generator.
//
// Bit-identical twin of synth_host.c (SplitMix64 used counter-based; same
// stream keys, same record layout). Holds none of the method's arithmetic: it
// only writes reproducible bytes into expert records that already live in
// device memory, so that 15.7 GB of weights per layer can be made in
// milliseconds instead of being copied from the host.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t stream_key(uint64_t seed, uint32_t kind, uint32_t layer,
                                               uint32_t expert, uint32_t matrix) {
  uint64_t tag = ((uint64_t)(kind & 0xFFu) << 56) | ((uint64_t)(layer & 0xFFFFu) << 40) |
                 ((uint64_t)expert << 8) | (uint64_t)(matrix & 0xFFu);
  return mix64(seed * kGamma ^ mix64(tag));
}

__device__ inline uint64_t value(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * kGamma); }

// One thread per 8-byte code word, or per scale byte, or per 8 padding bytes.
// Work units of one record: [3 x (nc/8 code words + ns scale bytes)] + pad words.
__global__ void fill_kernel(uint8_t* __restrict__ dst, int64_t nc, int64_t ns, int64_t stride,
                            int64_t rec, uint64_t seed, uint32_t layer, uint32_t e0, int64_t n) {
  const int64_t per_matrix = nc / 8 + ns;
  const int64_t pad_words = (stride - rec + 7) / 8;
  const int64_t per_record = 3 * per_matrix + pad_words;
  const int64_t total = per_record * n;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
       u += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = u / per_record;
    int64_t w = u - r * per_record;
    uint8_t* p = dst + r * stride;
    uint32_t e = e0 + (uint32_t)r;
    if (w < 3 * per_matrix) {
      uint32_t m = (uint32_t)(w / per_matrix);
      int64_t q = w - (int64_t)m * per_matrix;
      uint8_t* pm = p + (int64_t)m * (nc + ns);
      if (q < nc / 8) {
        uint64_t v = value(stream_key(seed, 1, layer, e, m), (uint64_t)q);
        *reinterpret_cast<uint64_t*>(pm + q * 8) = v;  // little-endian: byte b = v >> 8b
      } else {
        int64_t i = q - nc / 8;
        uint64_t v = value(stream_key(seed, 2, layer, e, m), (uint64_t)i);
        uint32_t e5 = (uint32_t)(((v >> 32) * 5ull) >> 32);
        pm[nc + i] = (uint8_t)(121u + e5);
      }
    } else {
      int64_t i = (w - 3 * per_matrix) * 8;
      for (int b = 0; b < 8 && rec + i + b < stride; ++b) p[rec + i + b] = 0;
    }
  }
}

}  // namespace

extern "C" {

// Fill n consecutive expert records (ids e0 .. e0+n-1 of `layer`) at device
// pointer dst, `stride` bytes apart, asynchronously on `stream`.
// Returns 0 on success, -1 on a bad argument, -2 on a CUDA launch error.
int k3s_fill_records_device(void* dst, int64_t d, int64_t f, uint64_t seed, uint32_t layer,
                            uint32_t e0, int64_t n, int64_t stride, void* stream) {
  int64_t rec = 3 * (d * f / 2 + d * f / 32);
  if (!dst || d <= 0 || f <= 0 || (d % 32) || (f % 32) || stride < rec || (stride % 8) || n < 0)
    return -1;
  if (reinterpret_cast<uintptr_t>(dst) % 16) return -1;
  if (n == 0) return 0;
  int64_t nc = d * f / 2, ns = d * f / 32;
  int64_t per_record = 3 * (nc / 8 + ns) + (stride - rec + 7) / 8;
  int64_t total = per_record * n;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      (uint8_t*)dst, nc, ns, stride, rec, seed, layer, e0, n);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // extern "C"
