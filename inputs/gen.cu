// Device twin of inputs/__init__.py: SplitMix64 in counter mode (Steele, Lea and
// Flood, OOPSLA 2014).  Fills large synthetic tensors (packed int4 weights and
// their fp32 scales) on the GPU with exactly the bytes the host generator gives.
// Input generation only: nothing here belongs to the W4AFP8 method.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t stream_key(uint64_t seed, uint32_t stream) {
  return mix64(((seed << 16) + stream + 1) * kGamma);
}

__global__ void fill_int4_kernel(uint8_t* out, int64_t start, int64_t count, uint64_t key) {
  const int64_t n4 = count / 4;
  uint32_t* out4 = reinterpret_cast<uint32_t*>(out);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t idx = static_cast<uint64_t>(start + 4 * i + j + 1);
      v |= static_cast<uint32_t>(mix64(key + idx * kGamma) >> 56) << (8 * j);
    }
    out4[i] = v;
  }
  if (blockIdx.x == 0 && threadIdx.x < count - 4 * n4) {
    const int64_t i = 4 * n4 + threadIdx.x;
    out[i] = static_cast<uint8_t>(mix64(key + static_cast<uint64_t>(start + i + 1) * kGamma) >> 56);
  }
}

__global__ void fill_scales_kernel(float* out, int64_t start, int64_t count, uint64_t key, float lo, float span) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t w = mix64(key + static_cast<uint64_t>(start + i + 1) * kGamma);
    const float u = static_cast<float>(static_cast<uint32_t>(w >> 40)) * 5.9604644775390625e-08f;  // 2^-24
    out[i] = __fadd_rn(lo, __fmul_rn(span, u));
  }
}

}  // namespace

extern "C" int w4a8gen_fill_int4(uint8_t* out, int64_t start, int64_t count, uint64_t seed, uint32_t stream,
                                 void* cuda_stream) {
  if (count <= 0) return 0;
  if (reinterpret_cast<uintptr_t>(out) & 3) return 1;
  fill_int4_kernel<<<1184, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(out, start, count,
                                                                           stream_key(seed, stream));
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int w4a8gen_fill_scales(float* out, int64_t start, int64_t count, uint64_t seed, uint32_t stream, float lo,
                                   float span, void* cuda_stream) {
  if (count <= 0) return 0;
  fill_scales_kernel<<<1184, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(out, start, count,
                                                                             stream_key(seed, stream), lo, span);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
