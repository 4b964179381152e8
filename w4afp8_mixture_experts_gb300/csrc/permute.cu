// Permutation preprocess: the stable sort of the flat routed pairs by expert
// (SGLang PR #7762 page, review of ep_moe/kernels.py: torch.sort(..., stable=True),
// seg_indptr[E+1] int64, src2dst int32).  No sort is needed: a counting sort
// gives the same order.
//
// One CTA of 1024 threads: a shared-memory histogram, an exclusive scan into
// seg_indptr, then the pairs in chunks of 1024 in flat order.  Inside a chunk,
// a pair's rank among the chunk's earlier pairs of the same expert is its rank
// inside its warp (__match_any_sync) plus the counts of the lower warps, which
// one pass over a [32][E] table of per-warp counts turns into prefixes.
#include "common.cuh"

namespace w4a8 {
namespace {

constexpr int kThreads = 1024;
__device__ unsigned int g_permute_error;

__global__ void __launch_bounds__(kThreads, 1)
    permute_kernel(const int32_t* __restrict__ ids, int P, int E, int64_t* __restrict__ seg,
                   int32_t* __restrict__ src2dst, int32_t* __restrict__ dst2src) {
  extern __shared__ int sm[];
  int* run = sm;           // [E] counts, then running start of each expert
  int* wh = sm + E;        // [32][E] per-warp counts of the current chunk
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  for (int i = tid; i < E; i += kThreads) run[i] = 0;
  for (int i = tid; i < 32 * E; i += kThreads) wh[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int f = tid; f < P; f += kThreads) {
    const int e = ids[f];
    if (e < 0 || e >= E) {
      bad = true;
      continue;
    }
    atomicAdd(&run[e], 1);
  }
  if (bad) atomicOr(&g_permute_error, 2u);
  __syncthreads();

  // exclusive scan of run[0..E) (E <= 1024: one value per thread)
  const int c = tid < E ? run[tid] : 0;
  int v = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    warp_tot[lane] = t - warp_tot[lane];  // exclusive
  }
  __syncthreads();
  const int excl = v - c + warp_tot[warp];
  if (tid < E) {
    run[tid] = excl;
    seg[tid] = excl;
  }
  if (tid == E - 1) seg[E] = excl + c;
  __syncthreads();

  const unsigned lt = (1u << lane) - 1u;
  for (int base = 0; base < P; base += kThreads) {
    const int f = base + tid;
    int e = -1;
    if (f < P) {
      e = ids[f];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt);
    if (e >= 0 && rank == 0) wh[warp * E + e] = __popc(same);
    __syncthreads();
    for (int x = tid; x < E; x += kThreads) {
      int s = run[x];
#pragma unroll 8
      for (int w = 0; w < 32; ++w) {
        const int t = wh[w * E + x];
        wh[w * E + x] = s;
        s += t;
      }
      run[x] = s;
    }
    __syncthreads();
    if (e >= 0) {
      const int d = wh[warp * E + e] + rank;
      src2dst[f] = d;
      dst2src[d] = f;
    }
    __syncthreads();
    for (int i = tid; i < 32 * E; i += kThreads) wh[i] = 0;
    __syncthreads();
  }
}

int read_permute_error() {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_permute_error, sizeof(v));
  const unsigned int zero = 0;
  cudaMemcpyToSymbol(g_permute_error, &zero, sizeof(zero));
  return static_cast<int>(v);
}

struct Registrar {
  Registrar() { register_device_error_reader(&read_permute_error); }
} registrar;

}  // namespace
}  // namespace w4a8

extern "C" int moe_permute(const int32_t* topk_ids, int64_t T, int k, int64_t E, int64_t* seg_indptr,
                           int32_t* src2dst, int32_t* dst2src, void* ws, size_t ws_bytes, void* stream) {
  using namespace w4a8;
  (void)ws;
  (void)ws_bytes;
  W4A8_REQUIRE(T >= 0 && k >= 1 && T * k < (1ll << 31), "T*k out of range");
  W4A8_REQUIRE(E >= 1 && E <= 1024, "E=%lld must be in [1, 1024]", (long long)E);
  W4A8_REQUIRE(seg_indptr != nullptr, "seg_indptr is null");
  W4A8_REQUIRE(T == 0 || (topk_ids && src2dst && dst2src), "null pointer");
  const size_t smem = static_cast<size_t>(33 * E) * sizeof(int);
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 33 * 1024 * 4) !=
        cudaSuccess)
      return check_launch("cudaFuncSetAttribute(permute)");
    attr_set = true;
  }
  permute_kernel<<<1, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      topk_ids, static_cast<int>(T * k), static_cast<int>(E), seg_indptr, src2dst, dst2src);
  return check_launch("permute_kernel");
}
