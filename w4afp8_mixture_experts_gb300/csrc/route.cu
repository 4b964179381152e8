// Router top-k: one warp per token, experts spread over the lanes, k rounds of
// a warp-wide (logit desc, expert id asc) arg-max by shuffles.
// The ids feed the permutation preprocess of the SGLang PR #7762 page
// (run_cutlass_moe_ep_preproess(topk_ids, ...)).
#include "common.cuh"

namespace w4a8 {
namespace {

template <int EPL>  // experts per lane
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  pdl_trigger();
  pdl_wait();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + static_cast<int64_t>(t) * E;
  float v[EPL];
  uint32_t taken = 0;  // bit i: expert lane + 32 i is selected or does not exist
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      v[i] = row[e];
    } else {
      v[i] = -INFINITY;
      taken |= 1u << i;
    }
  }
  int my_e = 0;
  float my_v = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (lane == j) {
      my_e = be;
      my_v = bv;
    }
    if ((be & 31) == lane && be < E) taken |= 1u << (be >> 5);
  }
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - vmax) : 0.f;
  float denom;
  if (renorm) {
    denom = ex;
  } else {
    denom = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) denom += expf(v[i] - vmax);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, o);
  if (lane < k) {
    ids[static_cast<int64_t>(t) * k + lane] = my_e;
    w[static_cast<int64_t>(t) * k + lane] = ex / denom;
  }
}

template <int EPL>
int launch_route(const float* logits, int64_t T, int64_t E, int k, int renorm, int32_t* ids, float* w,
                 cudaStream_t st) {
  const int blocks = static_cast<int>(ceil_div(T, 8));
  return launch_pdl("route_topk_kernel", route_topk_kernel<EPL>, dim3(blocks), dim3(256), 0, st, logits,
                    static_cast<int>(T), static_cast<int>(E), k, renorm, ids, w);
}

}  // namespace
}  // namespace w4a8

extern "C" int moe_route_topk(const float* logits, int64_t T, int64_t E, int k, int renormalize, int32_t* topk_ids,
                              float* topk_w, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(T >= 0 && T < (1ll << 26), "T=%lld out of range", (long long)T);
  W4A8_REQUIRE(E >= 1 && E <= 1024, "E=%lld must be in [1, 1024]", (long long)E);
  W4A8_REQUIRE(k >= 1 && k <= 32 && k <= E, "k=%d must be in [1, min(E, 32)]", k);
  if (T == 0) return W4A8_OK;
  W4A8_REQUIRE(logits && topk_ids && topk_w, "null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t epl = ceil_div(E, 32);
  if (epl <= 1) return launch_route<1>(logits, T, E, k, renormalize, topk_ids, topk_w, st);
  if (epl <= 2) return launch_route<2>(logits, T, E, k, renormalize, topk_ids, topk_w, st);
  if (epl <= 4) return launch_route<4>(logits, T, E, k, renormalize, topk_ids, topk_w, st);
  if (epl <= 8) return launch_route<8>(logits, T, E, k, renormalize, topk_ids, topk_w, st);
  if (epl <= 12) return launch_route<12>(logits, T, E, k, renormalize, topk_ids, topk_w, st);
  if (epl <= 16) return launch_route<16>(logits, T, E, k, renormalize, topk_ids, topk_w, st);
  return launch_route<32>(logits, T, E, k, renormalize, topk_ids, topk_w, st);
}
