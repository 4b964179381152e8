// Permutation preprocess: the stable sort of the flat routed pairs by expert
// (SGLang PR #7762 page, review of ep_moe/kernels.py: torch.sort(..., stable=True),
// seg_indptr[E+1] int64, src2dst int32).  No sort is needed: a counting sort
// gives the same order.
//
// Up to 8191 pairs: one CTA of 1024 threads builds a shared-memory histogram,
// scans it into seg_indptr and places the pairs.  From 8192 pairs: the pairs are
// cut into CTA chunks; pass 1 counts each chunk's experts into a workspace table,
// pass 2 derives every chunk's first position per expert from that table and
// places the chunk's pairs the same way.
//
// Expert-parallel shard (same page, review of ep_moe/layer.py: routed ids are
// translated through expert_map before the preprocess, which then runs over the
// local experts): with an expert map, a pair's expert is its local id; pairs of
// remote experts (map entry -1) are not placed (src2dst = -1) and dst2src holds
// -1 past the last local pair.
#include "common.cuh"

namespace w4a8 {
namespace {

constexpr int kThreads = 1024;
constexpr int kMultiMin = 8192;  // pairs from which the work is spread over several CTAs
__device__ unsigned int g_permute_error;

// Pairs per CTA of the multi-CTA path: a multiple of 1024, at least 2048, at most 1024 CTAs.
__host__ __device__ inline int64_t permute_chunk(int64_t P) {
  int64_t c = (P + 1023) / 1024;
  c = (c + 1023) / 1024 * 1024;
  return c < 2048 ? 2048 : c;
}

// Local expert of pair f: its routed id through the map (or the id itself without one); -1 for a
// pair of a remote expert, -2 for an id or map entry out of range (flagged, and the pair skipped).
__device__ __forceinline__ int local_expert(const int32_t* __restrict__ ids, const int32_t* __restrict__ emap, int f,
                                            int E, int EL) {
  const int e = ids[f];
  if (e < 0 || e >= E) return -2;
  const int l = emap ? emap[e] : e;
  return (l < -1 || l >= EL) ? -2 : l;
}

// Block-wide exclusive scan of v (one value per thread, E <= 1024 entries); returns the exclusive
// prefix and the total in *tot.
__device__ __forceinline__ int block_excl_scan(int c, int* warp_tot, int* tot) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    if (lane == 31) warp_tot[32] = t;     // grand total
  }
  __syncthreads();
  const int excl = v - c + warp_tot[warp];
  *tot = warp_tot[32];
  return excl;
}

// Sorted positions of the pairs [f0, f1) given run[e] = first free position of expert e: chunks of
// 1024 in flat order; inside a chunk a pair's rank among the chunk's earlier pairs of its expert is
// its rank inside its warp (__match_any_sync) plus the counts of the lower warps, which one pass
// over a [32][E] table of per-warp counts turns into prefixes.
__device__ void place_pairs(const int32_t* __restrict__ ids, const int32_t* __restrict__ emap, int E, int f0, int f1,
                            int EL, int* run, int* wh, int32_t* __restrict__ src2dst, int32_t* __restrict__ dst2src) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = f0; base < f1; base += kThreads) {
    const int f = base + tid;
    int e = -1;
    if (f < f1) {
      e = local_expert(ids, emap, f, E, EL);
      if (e < 0) {
        src2dst[f] = -1;  // remote (or invalid): not placed
        e = -1;
      }
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt);
    if (e >= 0 && rank == 0) wh[warp * EL + e] = __popc(same);
    __syncthreads();
    for (int x = tid; x < EL; x += kThreads) {
      int s = run[x];
#pragma unroll 8
      for (int w = 0; w < 32; ++w) {
        const int t = wh[w * EL + x];
        wh[w * EL + x] = s;
        s += t;
      }
      run[x] = s;
    }
    __syncthreads();
    if (e >= 0) {
      const int d = wh[warp * EL + e] + rank;
      src2dst[f] = d;
      dst2src[d] = f;
    }
    __syncthreads();
    for (int i = tid; i < 32 * EL; i += kThreads) wh[i] = 0;
    __syncthreads();
  }
}

// One CTA: histogram, scan into seg_indptr, placement.
__global__ void __launch_bounds__(kThreads, 1)
    permute_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ emap, int P, int E, int EL,
                   int64_t* __restrict__ seg, int32_t* __restrict__ src2dst, int32_t* __restrict__ dst2src) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sm[];
  int* run = sm;           // [EL] counts, then running start of each local expert
  int* wh = sm + EL;       // [32][EL] per-warp counts of the current chunk
  __shared__ int warp_tot[33];
  const int tid = threadIdx.x;

  for (int i = tid; i < EL; i += kThreads) run[i] = 0;
  for (int i = tid; i < 32 * EL; i += kThreads) wh[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int f = tid; f < P; f += kThreads) {
    const int e = local_expert(ids, emap, f, E, EL);
    if (e == -2) bad = true;
    if (e >= 0) atomicAdd(&run[e], 1);
  }
  if (bad) atomicOr(&g_permute_error, 2u);
  __syncthreads();
  const int c = tid < EL ? run[tid] : 0;
  int tot;
  const int excl = block_excl_scan(c, warp_tot, &tot);
  if (tid < EL) {
    run[tid] = excl;
    seg[tid] = excl;
  }
  if (tid == 0) seg[EL] = tot;
  for (int i = tot + tid; i < P; i += kThreads) dst2src[i] = -1;  // past the last placed pair
  __syncthreads();
  place_pairs(ids, emap, E, 0, P, EL, run, wh, src2dst, dst2src);
}

// Several CTAs, pass 1: CTA b counts the experts of pairs [b*C, (b+1)*C) into cnt[b][E].
__global__ void __launch_bounds__(kThreads)
    permute_count_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ emap, int P, int E, int EL,
                         int C, int* __restrict__ cnt) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int hist[];
  const int tid = threadIdx.x;
  for (int i = tid; i < EL; i += kThreads) hist[i] = 0;
  __syncthreads();
  const int f0 = blockIdx.x * C, f1 = min(P, f0 + C);
  bool bad = false;
  for (int f = f0 + tid; f < f1; f += kThreads) {
    const int e = local_expert(ids, emap, f, E, EL);
    if (e == -2) bad = true;
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
  if (bad) atomicOr(&g_permute_error, 2u);
  __syncthreads();
  for (int i = tid; i < EL; i += kThreads) cnt[static_cast<int64_t>(blockIdx.x) * EL + i] = hist[i];
}

// Pass 2: CTA b derives expert e's first position for its pairs (all pairs of lower experts, plus
// expert e's pairs in lower CTAs), CTA 0 writes seg_indptr, then places its pairs.
__global__ void __launch_bounds__(kThreads, 1)
    permute_place_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ emap, int P, int E, int EL,
                         int C, const int* __restrict__ cnt, int64_t* __restrict__ seg, int32_t* __restrict__ src2dst,
                         int32_t* __restrict__ dst2src) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sm[];
  int* run = sm;
  int* wh = sm + EL;
  __shared__ int warp_tot[33];
  const int tid = threadIdx.x;
  for (int i = tid; i < 32 * EL; i += kThreads) wh[i] = 0;
  int total = 0, before = 0;
  if (tid < EL) {
    for (int b = 0; b < static_cast<int>(gridDim.x); ++b) {
      const int v = cnt[static_cast<int64_t>(b) * EL + tid];
      if (b < static_cast<int>(blockIdx.x)) before += v;
      total += v;
    }
  }
  int tot;
  const int excl = block_excl_scan(tid < EL ? total : 0, warp_tot, &tot);
  if (tid < EL) run[tid] = excl + before;
  if (blockIdx.x == 0) {
    if (tid < EL) seg[tid] = excl;
    if (tid == 0) seg[EL] = tot;
  }
  for (int i = tot + static_cast<int>(blockIdx.x) * kThreads + tid; i < P; i += static_cast<int>(gridDim.x) * kThreads)
    dst2src[i] = -1;  // past the last placed pair
  __syncthreads();
  const int f0 = blockIdx.x * C;
  place_pairs(ids, emap, E, f0, min(P, f0 + C), EL, run, wh, src2dst, dst2src);
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

namespace w4a8 {

size_t permute_ws_bytes(int64_t P, int64_t E) {
  if (P < kMultiMin || E < 1) return 0;
  const int64_t blocks = (P + permute_chunk(P) - 1) / permute_chunk(P);
  return static_cast<size_t>(blocks * E) * sizeof(int);
}

}  // namespace w4a8

extern "C" int moe_permute_ep(const int32_t* topk_ids, int64_t T, int k, int64_t E, const int32_t* expert_map,
                              int64_t E_local, int64_t* seg_indptr, int32_t* src2dst, int32_t* dst2src, void* ws,
                              size_t ws_bytes, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(T >= 0 && k >= 1 && T * k < (1ll << 31), "T*k out of range");
  W4A8_REQUIRE(E >= 1 && E < (1ll << 31), "E=%lld out of range", (long long)E);
  W4A8_REQUIRE(E_local >= 1 && E_local <= 1024, "E_local=%lld must be in [1, 1024]", (long long)E_local);
  W4A8_REQUIRE(expert_map != nullptr || E_local == E, "without expert_map E_local must equal E");
  W4A8_REQUIRE(seg_indptr != nullptr, "seg_indptr is null");
  W4A8_REQUIRE(T == 0 || (topk_ids && src2dst && dst2src), "null pointer");
  const int64_t P = T * k;
  const size_t need = permute_ws_bytes(P, E_local);
  W4A8_REQUIRE(need == 0 || (ws != nullptr && ws_bytes >= need && (reinterpret_cast<uintptr_t>(ws) & 3) == 0),
               "workspace of %zu bytes (4-byte aligned) required for %lld pairs, got %zu", need, (long long)P,
               ws_bytes);
  const size_t smem = static_cast<size_t>(33 * E_local) * sizeof(int);
  static DeviceOnce attrs;  // the shared-memory limit is a per-device function attribute
  if (int rc = attrs.run([] {
        if (cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 33 * 1024 * 4) !=
                cudaSuccess ||
            cudaFuncSetAttribute(permute_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 33 * 1024 * 4) != cudaSuccess)
          return check_launch("cudaFuncSetAttribute(permute)");
        return static_cast<int>(W4A8_OK);
      }))
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int Ei = static_cast<int>(E), EL = static_cast<int>(E_local);
  if (need == 0) {
    return launch_pdl("permute_kernel", permute_kernel, dim3(1), dim3(kThreads), smem, st, topk_ids, expert_map,
                      static_cast<int>(P), Ei, EL, seg_indptr, src2dst, dst2src);
  }
  const int C = static_cast<int>(permute_chunk(P));
  const int blocks = static_cast<int>((P + C - 1) / C);
  int* cnt = static_cast<int*>(ws);
  if (int rc = launch_pdl("permute_count_kernel", permute_count_kernel, dim3(blocks), dim3(kThreads),
                          static_cast<size_t>(E_local) * sizeof(int), st, topk_ids, expert_map, static_cast<int>(P),
                          Ei, EL, C, cnt))
    return rc;
  return launch_pdl("permute_place_kernel", permute_place_kernel, dim3(blocks), dim3(kThreads), smem, st, topk_ids,
                    expert_map, static_cast<int>(P), Ei, EL, C, static_cast<const int*>(cnt), seg_indptr, src2dst,
                    dst2src);
}

extern "C" int moe_permute(const int32_t* topk_ids, int64_t T, int k, int64_t E, int64_t* seg_indptr,
                           int32_t* src2dst, int32_t* dst2src, void* ws, size_t ws_bytes, void* stream) {
  if (E > 1024) return w4a8::set_error(W4A8_ERR_INVALID_ARG, "E=%lld must be in [1, 1024]", (long long)E);
  return moe_permute_ep(topk_ids, T, k, E, nullptr, E, seg_indptr, src2dst, dst2src, ws, ws_bytes, stream);
}
