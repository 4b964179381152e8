// FP8 E4M3 quantisation per token per 128-column group, and SiLU-and-Mul with
// re-quantisation of the intermediate.
//
// One warp per (row, group): each lane owns 4 consecutive values (one 8-byte
// load per operand), the group's amax is a shuffle max, the scale amax/448 and
// the quotients x/s are IEEE fp32 divisions, and the codes come from the
// hardware cvt.rn.satfinite.e4m3x2 (round to nearest even, saturate to +-448,
// as on the PR #37796 page's fp8 write path).  The amax clamp to 1e-12 follows
// the DeepGEMM PR #53 page (padded rows would give 448/0).
#include <cuda_fp16.h>

#include "common.cuh"

namespace w4a8 {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {  // exact: E4M3 -> f16 -> f32
  uint32_t h2;  // the code in both bytes, so either half of the result holds its value
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code | (code << 8))));
  return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
}

// Quantise 4 values of one 128-group held by this lane; writes the codes and (lane 0) the
// scale and the group's correction term of the symmetric weight encoding:
//   gcorr = -1/2 * s * sum_k e4m3(code_k)  (lane sums, then a fixed xor-tree over lanes).
__device__ __forceinline__ void quant_group4(float f0, float f1, float f2, float f3, int lane, uint8_t* qdst,
                                             float* sdst, float* cdst) {
  float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
  amax = warp_max(amax);
  amax = fmaxf(amax, 1e-12f);
  const float s = __fdiv_rn(amax, 448.0f);
  const uint32_t lo = e4m3x2(__fdiv_rn(f0, s), __fdiv_rn(f1, s));
  const uint32_t hi = e4m3x2(__fdiv_rn(f2, s), __fdiv_rn(f3, s));
  const uint32_t codes = lo | (hi << 16);
  *reinterpret_cast<uint32_t*>(qdst + lane * 4) = codes;
  if (cdst) {
    float sum = (e4m3_value(codes & 0xFF) + e4m3_value((codes >> 8) & 0xFF)) +
                (e4m3_value((codes >> 16) & 0xFF) + e4m3_value(codes >> 24));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) *cdst = -0.5f * __fmul_rn(s, sum);
  }
  if (lane == 0) *sdst = s;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    quant_kernel(const uint16_t* __restrict__ x, int64_t K, const int32_t* __restrict__ row_index,
                 int64_t row_div, int64_t M_out, uint8_t* __restrict__ q, float* __restrict__ scales,
                 float* __restrict__ gcorr, int64_t ld) {
  const int64_t G = K / kGroup;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = gw / G;
  if (row >= M_out) return;
  const int64_t g = gw - row * G;
  const int64_t src = row_index ? static_cast<int64_t>(row_index[row]) / row_div : row;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + src * K + g * kGroup + lane * 4);
  const float f0 = __uint_as_float(raw.x << 16);
  const float f1 = __uint_as_float(raw.x & 0xFFFF0000u);
  const float f2 = __uint_as_float(raw.y << 16);
  const float f3 = __uint_as_float(raw.y & 0xFFFF0000u);
  quant_group4(f0, f1, f2, f3, lane, q + row * K + g * kGroup, scales + g * ld + row,
               gcorr ? gcorr + g * ld + row : nullptr);
}

// h = silu(gate) * up = gate / (1 + exp(-gate)) * up, fp32.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    silu_mul_requant_kernel(const uint16_t* __restrict__ gu, int64_t M, int64_t I, uint8_t* __restrict__ q,
                            float* __restrict__ scales, float* __restrict__ gcorr, int64_t ld) {
  const int64_t G = I / kGroup;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = gw / G;
  if (row >= M) return;
  const int64_t g = gw - row * G;
  const uint16_t* base = gu + row * 2 * I + g * kGroup + lane * 4;
  const uint2 gr = *reinterpret_cast<const uint2*>(base);
  const uint2 ur = *reinterpret_cast<const uint2*>(base + I);
  const float h0 = silu_mul(__uint_as_float(gr.x << 16), __uint_as_float(ur.x << 16));
  const float h1 = silu_mul(__uint_as_float(gr.x & 0xFFFF0000u), __uint_as_float(ur.x & 0xFFFF0000u));
  const float h2 = silu_mul(__uint_as_float(gr.y << 16), __uint_as_float(ur.y << 16));
  const float h3 = silu_mul(__uint_as_float(gr.y & 0xFFFF0000u), __uint_as_float(ur.y & 0xFFFF0000u));
  quant_group4(h0, h1, h2, h3, lane, q + row * I + g * kGroup, scales + g * ld + row,
               gcorr ? gcorr + g * ld + row : nullptr);
}

}  // namespace
}  // namespace w4a8

extern "C" int fp8_quant_per_token_group(const uint16_t* x, int64_t M_src, int64_t K, const int32_t* row_index,
                                         int64_t row_div, int64_t M_out, uint8_t* q, float* scales, float* gcorr,
                                         int64_t scale_ld, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(K > 0 && K % kGroup == 0, "K=%lld must be a positive multiple of 128", (long long)K);
  W4A8_REQUIRE(M_src >= 0 && M_out >= 0, "negative row count");
  W4A8_REQUIRE(row_index != nullptr || M_out == M_src, "without row_index M_out must equal M_src");
  W4A8_REQUIRE(row_index == nullptr || row_div >= 1, "row_div must be >= 1");
  W4A8_REQUIRE(scale_ld >= M_out && scale_ld % 4 == 0, "scale_ld must be >= M_out and a multiple of 4");
  if (M_out == 0) return W4A8_OK;
  W4A8_REQUIRE(x && q && scales, "null pointer");
  W4A8_REQUIRE(((uintptr_t)x & 7) == 0 && ((uintptr_t)q & 3) == 0 && ((uintptr_t)scales & 3) == 0 &&
                   ((uintptr_t)gcorr & 3) == 0,
               "x must be 8-byte and q, scales, gcorr 4-byte aligned");
  const int64_t warps = M_out * (K / kGroup);
  const int64_t blocks = ceil_div(warps, kWarpsPerBlock);
  W4A8_REQUIRE(blocks < (1ll << 31), "too many rows");
  quant_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      x, K, row_index, row_div, M_out, q, scales, gcorr, scale_ld);
  return check_launch("quant_kernel");
}

extern "C" int silu_mul_requant(const uint16_t* gate_up, int64_t M, int64_t I, uint8_t* q, float* scales,
                                float* gcorr, int64_t scale_ld, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(I > 0 && I % kGroup == 0, "I=%lld must be a positive multiple of 128", (long long)I);
  W4A8_REQUIRE(M >= 0, "negative row count");
  W4A8_REQUIRE(scale_ld >= M && scale_ld % 4 == 0, "scale_ld must be >= M and a multiple of 4");
  if (M == 0) return W4A8_OK;
  W4A8_REQUIRE(gate_up && q && scales, "null pointer");
  W4A8_REQUIRE(((uintptr_t)gate_up & 7) == 0 && ((uintptr_t)q & 3) == 0 && ((uintptr_t)scales & 3) == 0 &&
                   ((uintptr_t)gcorr & 3) == 0,
               "gate_up must be 8-byte and q, scales, gcorr 4-byte aligned");
  const int64_t blocks = ceil_div(M * (I / kGroup), kWarpsPerBlock);
  W4A8_REQUIRE(blocks < (1ll << 31), "too many rows");
  silu_mul_requant_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0,
                            static_cast<cudaStream_t>(stream)>>>(gate_up, M, I, q, scales, gcorr, scale_ld);
  return check_launch("silu_mul_requant_kernel");
}
