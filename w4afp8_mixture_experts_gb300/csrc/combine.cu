// Unpermute and combine (SGLang PR #7762 page: post-reordering of the outputs):
// out[t][c] = bf16( sum_j topk_w[t][j] * Y[src2dst[t*k+j]][c] ), fp32 in j order; slots with
// src2dst = -1 (routed to another expert-parallel shard) add nothing.
// CTA per token (and, for few tokens, per slice of 2048 columns); each thread loads the k rows' 8 bf16 of its
// columns with 16-byte loads.
#include "common.cuh"

namespace w4a8 {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    combine_kernel(const uint16_t* __restrict__ Y, const int32_t* __restrict__ s2d, const float* __restrict__ w,
                   int k, int64_t H, uint16_t* __restrict__ out) {
  __shared__ int64_t rows[32];
  __shared__ float ws[32];
  __shared__ int n_here;
  pdl_trigger();
  pdl_wait();
  const int64_t t = blockIdx.x;
  if (threadIdx.x < 32) {  // the token's placed pairs in slot order (src2dst = -1: another shard's expert)
    const int j = threadIdx.x;
    const int d = j < k ? s2d[t * k + j] : -1;
    const unsigned here = __ballot_sync(0xffffffffu, d >= 0);
    if (d >= 0) {
      const int pos = __popc(here & ((1u << j) - 1u));
      rows[pos] = static_cast<int64_t>(d) * H;
      ws[pos] = w[t * k + j];
    }
    if (j == 0) n_here = __popc(here);
  }
  __syncthreads();
  const int kh = n_here;
  for (int64_t c = (static_cast<int64_t>(blockIdx.y) * kThreads + threadIdx.x) * 8; c < H;
       c += static_cast<int64_t>(gridDim.y) * kThreads * 8) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 8
    for (int j = 0; j < kh; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(Y + rows[j] + c);
      const float wj = ws[j];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wj, __uint_as_float(u[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wj, __uint_as_float(u[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = static_cast<uint32_t>(float_to_bf16_bits(acc[2 * i])) |
             (static_cast<uint32_t>(float_to_bf16_bits(acc[2 * i + 1])) << 16);
    *reinterpret_cast<uint4*>(out + t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace
}  // namespace w4a8

extern "C" int moe_unpermute_combine(const uint16_t* Y, const int32_t* src2dst, const float* topk_w, int64_t T,
                                     int k, int64_t H, uint16_t* out, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(T >= 0 && T < (1ll << 31), "T out of range");
  W4A8_REQUIRE(k >= 1 && k <= 32, "k=%d must be in [1, 32]", k);
  W4A8_REQUIRE(H > 0 && H % 8 == 0, "H=%lld must be a positive multiple of 8", (long long)H);
  if (T == 0) return W4A8_OK;
  W4A8_REQUIRE(Y && src2dst && topk_w && out, "null pointer");
  W4A8_REQUIRE(aligned16(Y) && aligned16(out), "Y and out must be 16-byte aligned");
  // few tokens: also split the columns over CTAs, so that the SMs have work
  const int64_t slices = T >= 2 * num_sms() ? 1 : ceil_div(H, kThreads * 8);
  const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>(slices < 65535 ? slices : 65535));
  return launch_pdl("combine_kernel", combine_kernel, grid, dim3(kThreads), 0, static_cast<cudaStream_t>(stream), Y,
                    src2dst, topk_w, k, H, out);
}
