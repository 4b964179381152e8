// FP8 E4M3 quantisation per token per 128-column group, and SiLU-and-Mul with
// re-quantisation of the intermediate.
//
// 16 or 4 lanes per (row, group), whose values stay in registers between the
// amax pass and the quantisation pass (the SiLU-and-Mul kernel holds h).  The
// scale amax/448 is an IEEE fp32 division; the quotients x/s are the correctly
// rounded fp32 quotients; the codes come from the hardware
// cvt.rn.satfinite.e4m3x2 (round to nearest even, saturate to +-448, as on the
// PR #37796 page's fp8 write path).  The amax clamp to 1e-12 follows
// the DeepGEMM PR #53 page (padded rows would give 448/0).
#include "common.cuh"

namespace w4a8 {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// LANES consecutive lanes per (row, 128-group), 128 / LANES values each: the values stay in
// registers between the amax pass and the quantisation pass, and the group's amax and code sum
// take log2(LANES) shuffle steps.  amax is taken on the bf16 magnitude bits (same order as the values for non-NaN
// inputs).
// Lanes per group: 16 (8 values each) for small launches, 4 (32 values each) for large ones, where
// the SiLU kernel measured faster with 4 (0.19 vs 0.23 ms at 8192 tokens); the scatter quantisation
// always takes 16 (0.143 vs 0.175 ms at 8192 tokens: each group's codes go to k rows).
constexpr int kSmallLaunchGroups = 1 << 16;

// One (row, 128-group) quantised by its LANES lanes, lane `sub` holding values [sub*V, sub*V + V)
// (V = 128 / LANES) of the group at xg: the codes (4 per word) stay in registers, with the scale s
// and the group correction -1/2 * s * sum(E4M3 values) (when want_corr) returned to every lane.
template <int LANES>
__device__ __forceinline__ void quantize_group(const uint16_t* __restrict__ xg, int sub, bool want_corr,
                                               uint32_t (&code)[kGroup / LANES / 4], float& s, float& corr) {
  constexpr int kQuantVals = kGroup / LANES;  // values per lane
  const uint4* xp = reinterpret_cast<const uint4*>(xg + sub * kQuantVals);
  uint32_t w[kQuantVals / 2];
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < kQuantVals / 8; ++i) {
    const uint4 v = __ldg(xp + i);
    w[4 * i + 0] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
    mx = __vmaxu2(mx, __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu));
    mx = __vmaxu2(mx, __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
  const unsigned quad = ((1u << LANES) - 1u) << (threadIdx.x & (32 - LANES));  // this group's lanes
#pragma unroll
  for (int o = 1; o < LANES; o <<= 1) mx = max(mx, __shfl_xor_sync(quad, mx, o));
  const float amax = fmaxf(__uint_as_float(mx << 16), 1e-12f);
  s = __fdiv_rn(amax, 448.0f);
  const float r = __frcp_rn(s);
#pragma unroll
  for (int i = 0; i < kQuantVals / 8; ++i) {
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t v = w[4 * i + j];
      c[j] = e4m3x2(div_by_scale(bf16_lo(v), s, r), div_by_scale(bf16_hi(v), s, r));
    }
    code[2 * i] = c[0] | (c[1] << 16);
    code[2 * i + 1] = c[2] | (c[3] << 16);
  }
  corr = 0.0f;
  if (want_corr) {
    int u = code_units(code);
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) u += __shfl_xor_sync(quad, u, o);
    corr = corr_from_units(u, s);
  }
}

// The lane's codes of one group to q (16-byte stores when a lane holds a multiple of 16 codes).
template <int LANES>
__device__ __forceinline__ void store_codes(uint8_t* qp, const uint32_t (&code)[kGroup / LANES / 4]) {
  constexpr int kQuantVals = kGroup / LANES;
  if constexpr (kQuantVals % 16 == 0) {
#pragma unroll
    for (int i = 0; i < kQuantVals / 16; ++i)
      reinterpret_cast<uint4*>(qp)[i] = make_uint4(code[4 * i], code[4 * i + 1], code[4 * i + 2], code[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < kQuantVals / 8; ++i) reinterpret_cast<uint2*>(qp)[i] = make_uint2(code[2 * i], code[2 * i + 1]);
  }
}

// Output row `row` of q from input row row_index[row] / row_div (or row itself): a gather.
template <int LANES>
__global__ void __launch_bounds__(256)
    quant_quad_kernel(const uint16_t* __restrict__ x, int64_t K, const int32_t* __restrict__ row_index,
                      int64_t row_div, int64_t M_out, uint8_t* __restrict__ q, float* __restrict__ scales,
                      float* __restrict__ gcorr, int64_t ld) {
  constexpr int kQuantVals = kGroup / LANES;  // values per lane
  pdl_trigger();
  pdl_wait();
  const int64_t G = K / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t task = tid / LANES;
  const int sub = static_cast<int>(tid % LANES);
  // a group's lanes leave together (M_out * G * LANES threads are launched rounded up to the block)
  if (task >= M_out * G) return;
  const int64_t row = task / G;
  const int64_t g = task - row * G;
  const int64_t ri = row_index ? static_cast<int64_t>(row_index[row]) : row;
  if (ri < 0) return;  // no source row (a pair of a remote expert): left unwritten; the group's lanes leave together
  const int64_t src = row_index ? ri / row_div : row;
  uint32_t code[kQuantVals / 4];
  float s, corr;
  quantize_group<LANES>(x + src * K + g * kGroup, sub, gcorr != nullptr, code, s, corr);
  store_codes<LANES>(q + row * K + g * kGroup + sub * kQuantVals, code);
  if (sub == 0) {
    scales[g * ld + row] = s;
    if (gcorr) gcorr[g * ld + row] = corr;
  }
}

// The same quantisation, once per source row t, with the codes, scale and correction written to
// every destination row src2dst[t*k + j] (j < k; -1 and rows past M_out are skipped): in the MoE
// each token's row is quantised once instead of once per routed pair.
template <int LANES>
__global__ void __launch_bounds__(256)
    quant_scatter_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t K, const int32_t* __restrict__ src2dst,
                         int k, int64_t M_out, uint8_t* __restrict__ q, float* __restrict__ scales,
                         float* __restrict__ gcorr, int64_t ld) {
  constexpr int kQuantVals = kGroup / LANES;  // values per lane
  pdl_trigger();
  pdl_wait();
  const int64_t G = K / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t task = tid / LANES;
  const int sub = static_cast<int>(tid % LANES);
  if (task >= T * G) return;  // a group's lanes leave together
  const int64_t row = task / G;
  const int64_t g = task - row * G;
  uint32_t code[kQuantVals / 4];
  float s, corr;
  quantize_group<LANES>(x + row * K + g * kGroup, sub, gcorr != nullptr, code, s, corr);
  constexpr int kPre = 8;  // destinations fetched ahead (top-8 routing: all of them)
  for (int j0 = 0; j0 < k; j0 += kPre) {
    int64_t dst[kPre];
#pragma unroll
    for (int j = 0; j < kPre; ++j) dst[j] = j0 + j < k ? src2dst[row * k + j0 + j] : -1;
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const int64_t d = dst[j];  // the same for all of the group's lanes
      if (d < 0 || d >= M_out) continue;
      store_codes<LANES>(q + d * K + g * kGroup + sub * kQuantVals, code);
      if (sub == 0) {
        scales[g * ld + d] = s;
        if (gcorr) gcorr[g * ld + d] = corr;
      }
    }
  }
}

// SiLU-and-Mul + requantisation, four lanes per (row, 128-group) as in quant_quad_kernel: each
// lane computes its 32 values of h = silu(gate) * up into registers, then quantises them.
template <int LANES>
__global__ void __launch_bounds__(256)
    silu_quad_kernel(const uint16_t* __restrict__ gu, int64_t M, const int64_t* __restrict__ m_dev, int64_t I,
                     uint8_t* __restrict__ q, float* __restrict__ scales, float* __restrict__ gcorr, int64_t ld) {
  constexpr int kQuantVals = kGroup / LANES;  // values per lane
  pdl_trigger();
  pdl_wait();
  const int64_t G = I / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t task = tid / LANES;
  const int sub = static_cast<int>(tid % LANES);
  if (task >= M * G) return;  // a group's lanes leave together
  const int64_t row = task / G;
  if (m_dev && row >= *m_dev) return;  // rows past the device-side count are not produced
  const int64_t g = task - row * G;
  const uint4* gp = reinterpret_cast<const uint4*>(gu + row * 2 * I + g * kGroup + sub * kQuantVals);
  const uint4* up = reinterpret_cast<const uint4*>(gu + row * 2 * I + I + g * kGroup + sub * kQuantVals);
  float h[kQuantVals];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kQuantVals / 8; ++i) {
    const uint4 gv = __ldg(gp + i);
    const uint4 uv = __ldg(up + i);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[8 * i + 2 * j] = silu_mul(bf16_lo(gw[j]), bf16_lo(uw[j]));
      h[8 * i + 2 * j + 1] = silu_mul(bf16_hi(gw[j]), bf16_hi(uw[j]));
      amax = fmaxf(amax, fmaxf(fabsf(h[8 * i + 2 * j]), fabsf(h[8 * i + 2 * j + 1])));
    }
  }
  const unsigned quad = ((1u << LANES) - 1u) << (threadIdx.x & (32 - LANES));
#pragma unroll
  for (int o = 1; o < LANES; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(quad, amax, o));
  amax = fmaxf(amax, 1e-12f);
  const float s = __fdiv_rn(amax, 448.0f);
  const float r = __frcp_rn(s);
  uint8_t* qp = q + row * I + g * kGroup + sub * kQuantVals;
  uint32_t code[kQuantVals / 4];
#pragma unroll
  for (int i = 0; i < kQuantVals / 8; ++i) {
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      c[j] = e4m3x2(div_by_scale(h[8 * i + 2 * j], s, r), div_by_scale(h[8 * i + 2 * j + 1], s, r));
    code[2 * i] = c[0] | (c[1] << 16);
    code[2 * i + 1] = c[2] | (c[3] << 16);
    reinterpret_cast<uint2*>(qp)[i] = make_uint2(code[2 * i], code[2 * i + 1]);
  }
  float corr = 0.0f;
  if (gcorr) {
    int u = code_units(code);
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) u += __shfl_xor_sync(quad, u, o);
    corr = corr_from_units(u, s);
  }
  if (sub == 0) {
    scales[g * ld + row] = s;
    if (gcorr) gcorr[g * ld + row] = corr;
  }
}

// The corrections of stored codes: gcorr[g][m] = -1/2 * a_s[g][m] * (sum of the E4M3 values of A[m]'s
// group g), 16 lanes per (row, group), with the arithmetic of the quantisation kernels above (so the
// result equals what they emit for the same codes, bit for bit).  Tasks run group-major, so
// consecutive groups of 16 lanes write consecutive entries of one gcorr row.
__global__ void __launch_bounds__(256) gcorr_kernel(const uint8_t* __restrict__ A, int64_t M, int64_t K,
                                                    const float* __restrict__ a_s, int64_t ld,
                                                    float* __restrict__ gcorr) {
  pdl_trigger();
  pdl_wait();
  const int64_t G = K / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t task = tid / 16;
  const int sub = static_cast<int>(tid % 16);
  if (task >= M * G) return;  // a group's lanes leave together
  const int64_t g = task / M;
  const int64_t m = task - g * M;
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(A + m * K + g * kGroup + sub * 8));
  const uint32_t code[2] = {v.x, v.y};
  int u = code_units(code);
  const unsigned half = 0xFFFFu << (threadIdx.x & 16);
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) u += __shfl_xor_sync(half, u, o);
  if (sub == 0) gcorr[g * ld + m] = corr_from_units(u, a_s[g * ld + m]);
}

}  // namespace

int launch_gcorr(const uint8_t* A, int64_t M, int64_t K, const float* a_s, int64_t ld, float* gcorr,
                 cudaStream_t st) {
  const int64_t blocks = ceil_div(M * (K / kGroup) * 16, 256);
  W4A8_REQUIRE(blocks < (1ll << 31), "too many rows");
  if (M == 0) return W4A8_OK;
  return launch_pdl("gcorr_kernel", gcorr_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, A, M, K,
                    a_s, ld, gcorr);
}

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
  W4A8_REQUIRE(((uintptr_t)x & 15) == 0 && ((uintptr_t)q & 15) == 0 && ((uintptr_t)scales & 3) == 0 &&
                   ((uintptr_t)gcorr & 3) == 0,
               "x and q must be 16-byte, scales and gcorr 4-byte aligned");
  const int64_t groups = M_out * (K / kGroup);
  const bool small = groups < kSmallLaunchGroups;
  const int64_t blocks = ceil_div(groups * (small ? 16 : 4), 256);
  W4A8_REQUIRE(blocks < (1ll << 31), "too many rows");
  return launch_pdl("quant_quad_kernel", small ? quant_quad_kernel<16> : quant_quad_kernel<4>,
                    dim3(static_cast<unsigned>(blocks)), dim3(256), 0, static_cast<cudaStream_t>(stream), x, K,
                    row_index, row_div, M_out, q, scales, gcorr, scale_ld);
}

extern "C" int fp8_quant_scatter_per_token_group(const uint16_t* x, int64_t T, int64_t K, const int32_t* src2dst,
                                                 int k, int64_t M_out, uint8_t* q, float* scales, float* gcorr,
                                                 int64_t scale_ld, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(K > 0 && K % kGroup == 0, "K=%lld must be a positive multiple of 128", (long long)K);
  W4A8_REQUIRE(T >= 0 && M_out >= 0, "negative row count");
  W4A8_REQUIRE(k >= 1 && k <= 32, "k=%d must be in [1, 32]", k);
  W4A8_REQUIRE(scale_ld >= M_out && scale_ld % 4 == 0, "scale_ld must be >= M_out and a multiple of 4");
  if (T == 0 || M_out == 0) return W4A8_OK;
  W4A8_REQUIRE(x && src2dst && q && scales, "null pointer");
  W4A8_REQUIRE(((uintptr_t)x & 15) == 0 && ((uintptr_t)q & 15) == 0 && ((uintptr_t)scales & 3) == 0 &&
                   ((uintptr_t)gcorr & 3) == 0,
               "x and q must be 16-byte, scales and gcorr 4-byte aligned");
  const int64_t groups = T * (K / kGroup);
  const int64_t blocks = ceil_div(groups * 16, 256);
  W4A8_REQUIRE(blocks < (1ll << 31), "too many rows");
  return launch_pdl("quant_scatter_kernel", quant_scatter_kernel<16>,
                    dim3(static_cast<unsigned>(blocks)), dim3(256), 0, static_cast<cudaStream_t>(stream), x, T, K,
                    src2dst, k, M_out, q, scales, gcorr, scale_ld);
}

extern "C" int silu_mul_requant_rows(const uint16_t* gate_up, int64_t M, const int64_t* m_dev, int64_t I,
                                     uint8_t* q, float* scales, float* gcorr, int64_t scale_ld, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(I > 0 && I % kGroup == 0, "I=%lld must be a positive multiple of 128", (long long)I);
  W4A8_REQUIRE(M >= 0, "negative row count");
  W4A8_REQUIRE(scale_ld >= M && scale_ld % 4 == 0, "scale_ld must be >= M and a multiple of 4");
  if (M == 0) return W4A8_OK;
  W4A8_REQUIRE(gate_up && q && scales, "null pointer");
  W4A8_REQUIRE(((uintptr_t)gate_up & 15) == 0 && ((uintptr_t)q & 7) == 0 && ((uintptr_t)scales & 3) == 0 &&
                   ((uintptr_t)gcorr & 3) == 0,
               "gate_up must be 16-byte, q 8-byte and scales, gcorr 4-byte aligned");
  const int64_t groups = M * (I / kGroup);
  const bool small = groups < kSmallLaunchGroups;
  const int64_t blocks = ceil_div(groups * (small ? 16 : 4), 256);
  W4A8_REQUIRE(blocks < (1ll << 31), "too many rows");
  return launch_pdl("silu_quad_kernel", small ? silu_quad_kernel<16> : silu_quad_kernel<4>,
                    dim3(static_cast<unsigned>(blocks)), dim3(256), 0, static_cast<cudaStream_t>(stream), gate_up, M,
                    m_dev, I, q, scales, gcorr, scale_ld);
}

extern "C" int silu_mul_requant(const uint16_t* gate_up, int64_t M, int64_t I, uint8_t* q, float* scales,
                                float* gcorr, int64_t scale_ld, void* stream) {
  return silu_mul_requant_rows(gate_up, M, nullptr, I, q, scales, gcorr, scale_ld, stream);
}
