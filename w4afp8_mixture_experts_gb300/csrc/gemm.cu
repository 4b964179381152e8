// int4 x FP8 grouped GEMM and dense Linear on the 5th-generation tensor cores (sm_103a).
//
// Computes, per expert e and routed row j of that expert,
//   C[j][n] = bf16( sum_g a_s[g][j] * w_s[e][g][n] * sum_{k in g} e4m3(A[j][k]) * int4(W[e][n][k]) )
// which is the W4A8 grouped GEMM of the SGLang PR #7762 page (cutlass_w4a8_moe,
// group size / chunk_size 128) and, with one expert, the dense W4AFP8 Linear
// of the lyraW4AFp8 page.
//
// Design (one persistent CTA per SM, 14 warps):
//   * Operands are swapped so that the weights fill the 128-row M side of
//     tcgen05.mma and the few tokens of an expert sit on N (16..NMAX, any
//     multiple of 16).  Prior art: the swapAB small-batch path of the DeepGEMM
//     PR #53 page ("SM90 FP4 MegaMoE"); here it is the only mode, and N
//     shrinks to the expert's rows, so no row tile runs empty.
//   * warp 0   : TMA producer.  Per 128-K group it loads the token tile (E4M3,
//                128-byte swizzle), the packed int4 weight tile (64-byte
//                swizzle), and the fp32 scales of both, into a STAGES-deep ring.
//   * warps 2-5: converters.  Thread r owns weight row r of the tile, reads its
//                64 packed bytes and writes 128 E4M3 bytes (int4 -8..7 are all
//                exact in E4M3) with two 8-entry byte-permute lookups per 8
//                values, into the UMMA K-major 128-byte-swizzled layout (or into
//                tensor memory, A_TMEM).
//   * warp 1   : allocates tensor memory and issues 4 MMAs (K = 32 each) per
//                group into one of two fp32 accumulators P in tensor memory.
//   * warps 6-13: promotion.  The scales differ per 128-K group, so each
//                group's partial product leaves the tensor core (tcgen05.ld)
//                and is added in fp32: acc += (w_s * a_s) * P (the epilogue
//                FFMA promotion the DeepGEMM PR #53 page describes for SM90,
//                kept here because the scales are arbitrary fp32 values).  The
//                second P buffer lets the tensor core run the next group
//                meanwhile.  At the end of a tile the accumulators are rounded
//                to bf16 and stored.
//   * Tiles: (expert, token chunk, 128-row weight block); chunks split an
//     expert's rows evenly into pieces of at most NMAX; the schedule is built
//     in shared memory from seg_indptr by every CTA (no host synchronisation,
//     no workspace), and CTAs stride over it.
#include <algorithm>
#include <cstdio>
#include <cstring>

#include "common.cuh"

namespace w4a8 {
namespace {

constexpr int kBM = 128;      // weight rows per tile (MMA M)
constexpr int kKStep = 32;    // K per tcgen05.mma for 8-bit operands
constexpr int kWarpTma = 0;
constexpr int kConvSets = 2;                 // group sets: set c takes the groups with it % 2 == c
constexpr int kWarpMma = 1;                  // warps 1 .. kConvSets issue the MMAs of one set each
constexpr int kWarpConv0 = kWarpMma + kConvSets;
constexpr int kConvWarps = 4;                // converter warps per set: one per tensor-memory lane quarter
constexpr int kWarpEpi0 = kWarpConv0 + kConvSets * kConvWarps;
constexpr int kEpiWarps = 8;
constexpr int kWarps = kWarpEpi0 + kEpiWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxExperts = 1024;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s: no legitimate wait comes close

__device__ unsigned int g_gemm_error;

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int NMAX_, int STAGES_, int SSTAGES_, int ABUF_, int NP_, bool A_TMEM_>
struct Cfg {
  static constexpr int NMAX = NMAX_;        // token tile (MMA N upper bound)
  static constexpr int STAGES = STAGES_;    // main ring: token tile + packed weights
  static constexpr int SSTAGES = SSTAGES_;  // scale ring: token + weight scales (epilogue only)
  static constexpr int ABUF = ABUF_;        // converted weight buffers
  static constexpr int NP = NP_;            // fp32 partial-product buffers in tensor memory
  static constexpr bool A_TMEM = A_TMEM_;   // converted weights in tensor memory (else shared)
  static constexpr int kTokBytes = NMAX * 128;            // NMAX rows x 128 B, 128B swizzle
  static constexpr int kWpkBytes = kBM * 64;              // 128 rows x 64 B packed int4
  static constexpr int kABytes = kBM * 128;               // 128 rows x 128 B E4M3
  static constexpr int kWscOff = (NMAX * 4 + 127) / 128 * 128;          // weight scales in a slot
  static constexpr int kScBytes = kWscOff + kBM * 4;                      // one scale slot (128-B aligned)
  static constexpr int kOffTok = 0;
  static constexpr int kOffWpk = kOffTok + STAGES * kTokBytes;
  static constexpr int kOffA = kOffWpk + STAGES * kWpkBytes;
  static constexpr int kOffSc = kOffA + (A_TMEM ? 0 : ABUF * kABytes);
  static constexpr int kOffBar = kOffSc + SSTAGES * kScBytes;
  static constexpr int kNumBars = 2 * STAGES + 2 * SSTAGES + 2 * ABUF + NP;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffSched = kOffMisc + 64;
  static constexpr int kSmemBytes = kOffSched + 2 * (kMaxExperts + 1) * 4 + 1024;
  static constexpr int kAColBase = NP * NMAX;             // first tensor-memory column of A
  static constexpr uint32_t kTmemCols = pow2_at_least(NP * NMAX + (A_TMEM ? ABUF * 32 : 0));
  static constexpr int kChunkMax = NMAX - 3;              // rows of a chunk (tile starts 4-aligned)
  static_assert(NMAX % 16 == 0 && NMAX >= 16 && NMAX <= 256, "token tile");
  static_assert(kTokBytes % 1024 == 0 && kOffWpk % 1024 == 0 && kOffA % 1024 == 0, "alignment");
  static_assert(NP * NMAX + (A_TMEM ? ABUF * 32 : 0) <= 512, "tensor memory");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(ABUF % kConvSets == 0 && NP % kConvSets == 0, "each set owns every kConvSets-th buffer");
  static_assert(NP <= ABUF, "an A-buffer completion barrier must not run a phase ahead of the epilogue");
};

struct GemmParams {
  const int64_t* seg;  // [E+1] or nullptr (dense: one expert with M rows)
  uint16_t* C;
  int E, N, K, M;      // M: rows of A (dense) / M_total
};

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;             // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;     // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;             // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2u) << 61;             // SWIZZLE_128B
  return d;
}

// Instruction descriptor: D fp32, A and B E4M3, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_e4m3(uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// 8 int4 (two's complement nibbles, element i in bits 4i..4i+3) -> 8 E4M3 codes.
// Positive and negative codes come from two 8-entry tables selected with prmt;
// a prmt in sign-replicate mode turns each nibble's sign bit into a byte mask.
__device__ __forceinline__ void int4x8_to_e4m3x8(uint32_t w, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t kPos0 = 0x44403800u;  // E4M3 of 0, 1, 2, 3
  constexpr uint32_t kPos1 = 0x4E4C4A48u;  //          4, 5, 6, 7
  constexpr uint32_t kNeg0 = 0xCACCCED0u;  //         -8,-7,-6,-5
  constexpr uint32_t kNeg1 = 0xB8C0C4C8u;  //         -4,-3,-2,-1
  const uint32_t idx = w & 0x77777777u;
  const uint32_t idx_hi = idx >> 16;
  const uint32_t pl = prmt(kPos0, kPos1, idx);
  const uint32_t nl = prmt(kNeg0, kNeg1, idx);
  const uint32_t ph = prmt(kPos0, kPos1, idx_hi);
  const uint32_t nh = prmt(kNeg0, kNeg1, idx_hi);
  const uint32_t w4 = w << 4;
  const uint32_t ml = prmt(w4, w, 0xD9C8u);  // byte j = 0xFF if nibble j < 0 (j = 0..3)
  const uint32_t mh = prmt(w4, w, 0xFBEAu);  // byte j = 0xFF if nibble j+4 < 0
  lo = (pl & ~ml) | (nl & ml);
  hi = (ph & ~mh) | (nh & mh);
}

struct Sched {
  const int* prefix;  // [E+1] chunk prefix
  const int* start;   // [E+1] row starts
  int E, NMAX, nblk;
  __device__ __forceinline__ void decode(int item, int& e, int& nb, int& row0, int& rows) const {
    const int chunk = item / nblk;
    nb = item - chunk * nblk;
    int lo = 0, hi = E;  // prefix[lo] <= chunk < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= chunk) lo = mid; else hi = mid;
    }
    e = lo;
    const int nc = prefix[e + 1] - prefix[e];
    const int cnt = start[e + 1] - start[e];
    const int cs = (cnt + nc - 1) / nc;
    const int c = chunk - prefix[e];
    const int r0 = c * cs;
    row0 = start[e] + r0;
    rows = min(cs, cnt - r0);
  }
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 127u) == 127u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        atomicOr(&g_gemm_error, 1u);
        return false;
      }
    }
  }
}

template <int NCOL>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (NCOL == 8) {
    uint32_t (&r8)[8] = *reinterpret_cast<uint32_t(*)[8]>(r);
    tmem_ld8(taddr, r8);
  } else if constexpr (NCOL == 16) {
    tmem_ld16(taddr, r);
  } else {
    static_assert(NCOL % 32 == 0, "columns");
#pragma unroll
    for (int c = 0; c < NCOL; c += 32) tmem_ld32(taddr + c, r + c);
  }
}

// acc[0..1] += (ws * ts[0..1]) * p[0..1], two lanes of fp32 per instruction.
__device__ __forceinline__ void promote2(float& a0, float& a1, float ws, float t0, float t1, uint32_t p0,
                                         uint32_t p1) {
  uint64_t acc, c, ts, w2, pp;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ts) : "f"(t0), "f"(t1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(w2) : "f"(ws));
  asm("mov.b64 %0, {%1, %2};" : "=l"(pp) : "r"(p0), "r"(p1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(c) : "l"(w2), "l"(ts));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(c), "l"(pp));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

template <class CF>
__global__ void __launch_bounds__(kThreads, 1)
    w4a8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAS,
                     const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBS,
                     const GemmParams prm) {
  constexpr int NMAX = CF::NMAX;
  constexpr int STAGES = CF::STAGES;
  constexpr int SSTAGES = CF::SSTAGES;
  constexpr int ABUF = CF::ABUF;
  constexpr int NP = CF::NP;
  constexpr int NHALF = NMAX / 2;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_tok = smem + CF::kOffTok;
  uint8_t* s_wpk = smem + CF::kOffWpk;
  uint8_t* s_a = smem + CF::kOffA;
  uint8_t* s_sc = smem + CF::kOffSc;  // slot: NMAX token scales, then (128-B aligned) 128 weight scales
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* sfull = empty + STAGES;
  uint64_t* sempty = sfull + SSTAGES;
  uint64_t* mready = sempty + SSTAGES;  // [ABUF] converted weights (and their P buffer) ready for the MMA
  uint64_t* mdone = mready + ABUF;      // [ABUF] MMAs of the group done: A buffer free, partials ready
  uint64_t* pempty = mdone + ABUF;      // [NP] partial buffer read by the epilogue
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + CF::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + CF::kOffMisc + 4);
  int* s_prefix = reinterpret_cast<int*>(smem + CF::kOffSched);
  int* s_start = s_prefix + (kMaxExperts + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = prm.K / kGroup;
  const int nblk = prm.N / kBM;
  const int E = prm.seg ? prm.E : 1;

  // ---- prologue: barriers, tensor memory, schedule ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConvWarps + 1);
    }
    for (int s = 0; s < SSTAGES; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], kEpiWarps);
    }
    for (int b = 0; b < ABUF; ++b) {
      mbar_init(&mready[b], kConvWarps);
      mbar_init(&mdone[b], 1);
    }
    for (int b = 0; b < NP; ++b) mbar_init(&pempty[b], kEpiWarps);
    *s_abort = 0;
    mbar_fence_init();
  }
  if (warp == kWarpMma) {  // the first MMA warp owns the tensor-memory allocation
    tmem_alloc(s_tmem, CF::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmAS);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmBS);
  }
  if (warp == 2) {  // chunk prefix over experts (warp-wide scan)
    int carry = 0;
    if (lane == 0) s_prefix[0] = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int cnt = 0, st = 0;
      if (e < E) {
        if (prm.seg) {
          st = static_cast<int>(prm.seg[e]);
          cnt = static_cast<int>(prm.seg[e + 1]) - st;
        } else {
          st = 0;
          cnt = prm.M;
        }
        s_start[e] = st;
      }
      int v = (cnt + CF::kChunkMax - 1) / CF::kChunkMax;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (e < E) s_prefix[e + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_start[E] = prm.seg ? static_cast<int>(prm.seg[E]) : prm.M;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *s_tmem;
  Sched sch{s_prefix, s_start, E, NMAX, nblk};
  const int n_items = s_prefix[E] * nblk;

  // A tile covers rows [row0 & ~3, ...): the scale vectors then start 16-byte aligned.
  if (warp == kWarpTma) {
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      uint32_t it = 0;
      for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        int e, nb, row0, rows;
        sch.decode(item, e, nb, row0, rows);
        const int r4 = row0 & ~3;
        for (int g = 0; g < G; ++g, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          const int ss = it % SSTAGES;
          const uint32_t sph = (it / SSTAGES) & 1;
          if (!wait_bar(&empty[s], ph ^ 1, s_abort)) goto done;
          mbar_arrive_expect_tx(&full[s], CF::kTokBytes + CF::kWpkBytes);
          tma_load_2d(s_tok + s * CF::kTokBytes, &tmA, &full[s], g * kGroup, r4);
          tma_load_2d_hint(s_wpk + s * CF::kWpkBytes, &tmB, &full[s], g * (kGroup / 2), e * prm.N + nb * kBM,
                           pol_w);
          if (!wait_bar(&sempty[ss], sph ^ 1, s_abort)) goto done;
          uint8_t* sc = s_sc + ss * CF::kScBytes;
          mbar_arrive_expect_tx(&sfull[ss], NMAX * 4 + kBM * 4);
          tma_load_2d(sc, &tmAS, &sfull[ss], r4, g);
          tma_load_2d(sc + CF::kWscOff, &tmBS, &sfull[ss], nb * kBM, e * G + g);
        }
      }
    }
  } else if (warp < kWarpConv0) {
    // ---- MMA issue: one thread per group set ----
    const int mset = warp - kWarpMma;
    if (lane == 0) {
      uint32_t it = 0;
      for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        int e, nb, row0, rows;
        sch.decode(item, e, nb, row0, rows);
        const int ncol = (row0 - (row0 & ~3) + rows + 15) & ~15;
        const uint32_t idesc = idesc_e4m3(static_cast<uint32_t>(ncol));
        for (int g = 0; g < G; ++g, ++it) {
          if (static_cast<int>(it % kConvSets) != mset) continue;
          const int s = it % STAGES;
          const int b = it % ABUF;
          const uint32_t aph = (it / ABUF) & 1;
          const int pb = it % NP;
          // mready implies: token tile landed, weights converted, partial buffer free
          if (!wait_bar(&mready[b], aph, s_abort)) goto done;
          tc_fence_after();
          const uint32_t d = tmem_base + pb * NMAX;
          const uint32_t tok = smem_u32(s_tok + s * CF::kTokBytes);
#pragma unroll
          for (int kk = 0; kk < kGroup / kKStep; ++kk) {
            const uint64_t bdesc = sw128_desc(tok + kk * kKStep);
            if constexpr (CF::A_TMEM) {
              const uint32_t a_t = tmem_base + CF::kAColBase + b * 32 + kk * (kKStep / 4);
              mma_f8f6f4_ts(d, a_t, bdesc, idesc, kk > 0 ? 1u : 0u);
            } else {
              const uint64_t adesc = sw128_desc(smem_u32(s_a + b * CF::kABytes) + kk * kKStep);
              mma_f8f6f4_ss(d, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&empty[s]);
          mma_commit(&mdone[b]);
        }
      }
    }
  } else if (warp < kWarpEpi0) {
    // ---- converters: int4 -> E4M3; set `cset` takes every kConvSets-th group ----
    const int q4 = warp & 3;
    const int cset = (warp - kWarpConv0) / kConvWarps;
    const int r = q4 * 32 + lane;
    uint32_t it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      for (int g = 0; g < G; ++g, ++it) {
        if (static_cast<int>(it % kConvSets) != cset) continue;
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        const int b = it % ABUF;
        const uint32_t aph = (it / ABUF) & 1;
        const int pb = it % NP;
        const uint32_t pph = (it / NP) & 1;
        const bool ok = wait_bar(&full[s], ph, s_abort) && wait_bar(&mdone[b], aph ^ 1, s_abort) &&
                        wait_bar(&pempty[pb], pph ^ 1, s_abort);
        if (__any_sync(0xffffffffu, !ok)) goto done;  // warp-uniform; the warp is converged below
        const uint8_t* wrow = s_wpk + s * CF::kWpkBytes + r * 64;
        uint32_t in[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((j ^ ((r >> 1) & 3)) << 4));
          in[4 * j + 0] = v.x;
          in[4 * j + 1] = v.y;
          in[4 * j + 2] = v.z;
          in[4 * j + 3] = v.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        uint32_t out[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) int4x8_to_e4m3x8(in[i], out[2 * i], out[2 * i + 1]);
        if constexpr (CF::A_TMEM) {
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + CF::kAColBase + b * 32;
          tmem_st32(taddr, out);
          tmem_wait_st();
          tc_fence_before();
        } else {
          uint8_t* arow = s_a + b * CF::kABytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) =
                make_uint4(out[4 * c], out[4 * c + 1], out[4 * c + 2], out[4 * c + 3]);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&mready[b]);
      }
    }
  } else {
    // ---- promotion and epilogue ----
    const int q4 = warp & 3;
    const int half = (warp - kWarpEpi0) >> 2;
    const int r = q4 * 32 + lane;
    const int c0 = half * NHALF;
    const uint32_t t_lane = static_cast<uint32_t>(q4 * 32) << 16;
    constexpr int CH = NHALF < 16 ? NHALF : 16;
    uint32_t it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      int e, nb, row0, rows;
      sch.decode(item, e, nb, row0, rows);
      const int r4 = row0 & ~3;
      const int lo = row0 - r4;  // columns [lo, lo + rows) of the tile are this chunk's rows
      float acc[NHALF];
#pragma unroll
      for (int j = 0; j < NHALF; ++j) acc[j] = 0.f;
      for (int g = 0; g < G; ++g, ++it) {
        const int ss = it % SSTAGES;
        const uint32_t sph = (it / SSTAGES) & 1;
        const int pb = it % NP;
        const int b = it % ABUF;
        const uint32_t aph = (it / ABUF) & 1;
        const bool ok = wait_bar(&mdone[b], aph, s_abort) && wait_bar(&sfull[ss], sph, s_abort);
        if (__any_sync(0xffffffffu, !ok)) goto done;  // warp-uniform; tcgen05.ld needs a converged warp
        tc_fence_after();
        const float* sc = reinterpret_cast<const float*>(s_sc + ss * CF::kScBytes);
        const float ws = sc[CF::kWscOff / 4 + r];
#pragma unroll
        for (int c = 0; c < NHALF; c += CH) {
          uint32_t p[CH];
          tmem_load_cols<CH>(tmem_base + t_lane + pb * NMAX + c0 + c, p);
          tmem_wait_ld();
          if (c + CH >= NHALF) {  // last chunk read: hand the buffer back to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[pb]);
          }
#pragma unroll
          for (int j = 0; j < CH; j += 4) {
            const float4 t = *reinterpret_cast<const float4*>(sc + c0 + c + j);
            promote2(acc[c + j], acc[c + j + 1], ws, t.x, t.y, p[j], p[j + 1]);
            promote2(acc[c + j + 2], acc[c + j + 3], ws, t.z, t.w, p[j + 2], p[j + 3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[ss]);
      }
      uint16_t* crow = prm.C + static_cast<int64_t>(r4) * prm.N + nb * kBM + r;
#pragma unroll
      for (int j = 0; j < NHALF; ++j) {
        const int t = c0 + j;
        if (t >= lo && t < lo + rows) crow[static_cast<int64_t>(t) * prm.N] = float_to_bf16_bits(acc[j]);
      }
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, CF::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

int make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
                uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw,
                const char* name) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(W4A8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(W4A8_ERR_INVALID_ARG, "tensor map for %s rejected (CUresult %d)", name, (int)r);
  return W4A8_OK;
}

int read_gemm_error() {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v));
  const unsigned int zero = 0;
  cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero));
  return static_cast<int>(v);
}

struct Registrar {
  Registrar() { register_device_error_reader(&read_gemm_error); }
} registrar;

template <class CF>
int launch(const uint8_t* A, const float* a_s, int64_t a_ld, const uint8_t* B, const float* b_s,
           const int64_t* seg, int64_t E, int64_t N, int64_t K, int64_t M, uint16_t* C, cudaStream_t st) {
  const int64_t G = K / kGroup;
  CUtensorMap tA, tAS, tB, tBS;
  int rc;
  if ((rc = make_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, CF::NMAX,
                        CU_TENSOR_MAP_SWIZZLE_128B, "A")))
    return rc;
  if ((rc = make_map_2d(&tAS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a_s, a_ld, G, a_ld * 4, CF::NMAX, 1,
                        CU_TENSOR_MAP_SWIZZLE_NONE, "a_scales")))
    return rc;
  if ((rc = make_map_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K / 2, E * N, K / 2, 64, kBM,
                        CU_TENSOR_MAP_SWIZZLE_64B, "B")))
    return rc;
  if ((rc = make_map_2d(&tBS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, b_s, N, E * G, N * 4, kBM, 1,
                        CU_TENSOR_MAP_SWIZZLE_NONE, "b_scales")))
    return rc;
  static bool attr_set = false;  // per template instance
  if (!attr_set) {
    if (cudaFuncSetAttribute(w4a8_gemm_kernel<CF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             CF::kSmemBytes) != cudaSuccess)
      return check_launch("cudaFuncSetAttribute(gemm)");
    attr_set = true;
  }
  GemmParams p;
  p.seg = seg;
  p.C = C;
  p.E = static_cast<int>(E);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.M = static_cast<int>(M);
  w4a8_gemm_kernel<CF><<<num_sms(), kThreads, CF::kSmemBytes, st>>>(tA, tAS, tB, tBS, p);
  return check_launch("w4a8_gemm_kernel");
}

// decode: few rows per expert, weight streaming; converted weights in tensor memory
using CfgDecode = Cfg<16, 16, 24, 8, 8, true>;
// prefill: 128-row token tiles, four partial buffers fill tensor memory; weights in shared memory
using CfgPrefill = Cfg<128, 5, 16, 4, 4, false>;

int gemm_common(const uint8_t* A, const float* a_s, int64_t a_ld, const uint8_t* B, const float* b_s,
                const int64_t* seg, int64_t E, int64_t N, int64_t K, int64_t M, uint16_t* C, void* stream) {
  W4A8_REQUIRE(K > 0 && K % kGroup == 0, "K=%lld must be a positive multiple of 128", (long long)K);
  W4A8_REQUIRE(N > 0 && N % kBM == 0, "N=%lld must be a positive multiple of 128", (long long)N);
  W4A8_REQUIRE(M >= 0 && M < (1ll << 31), "M=%lld out of range", (long long)M);
  W4A8_REQUIRE(E >= 1 && E <= kMaxExperts, "E=%lld must be in [1, 1024]", (long long)E);
  W4A8_REQUIRE(E * N < (1ll << 31) && K < (1ll << 31), "E*N or K too large");
  W4A8_REQUIRE(a_ld >= M && a_ld % 4 == 0 && a_ld > 0, "a_scale_ld=%lld must be >= M and a multiple of 4",
               (long long)a_ld);
  W4A8_REQUIRE(A && a_s && B && b_s && C, "null pointer");
  W4A8_REQUIRE(aligned16(A) && aligned16(a_s) && aligned16(B) && aligned16(b_s) && aligned16(C),
               "device pointers must be 16-byte aligned");
  if (M == 0) return W4A8_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Few rows per expert: weight streaming, 16-wide token tiles and a deep ring.
  if (M <= 32 * E)
    return launch<CfgDecode>(A, a_s, a_ld, B, b_s, seg, E, N, K, M, C, st);
  return launch<CfgPrefill>(A, a_s, a_ld, B, b_s, seg, E, N, K, M, C, st);
}

}  // namespace
}  // namespace w4a8

extern "C" int w4a8_grouped_gemm(const uint8_t* A, const float* a_scales, int64_t a_scale_ld,
                                 const uint8_t* B_packed, const float* b_scales, const int64_t* seg_indptr,
                                 int64_t E, int64_t N, int64_t K, int64_t M_total, uint16_t* C, void* ws,
                                 size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  W4A8_REQUIRE(seg_indptr != nullptr, "seg_indptr is null");
  return w4a8::gemm_common(A, a_scales, a_scale_ld, B_packed, b_scales, seg_indptr, E, N, K, M_total, C,
                           stream);
}

extern "C" int w4a8_linear(const uint8_t* A, const float* a_scales, int64_t a_scale_ld, const uint8_t* B_packed,
                           const float* b_scales, int64_t M, int64_t N, int64_t K, uint16_t* C, void* ws,
                           size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  return w4a8::gemm_common(A, a_scales, a_scale_ld, B_packed, b_scales, nullptr, 1, N, K, M, C, stream);
}
