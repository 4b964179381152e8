// int4 x FP8 grouped GEMM and dense Linear on the 5th-generation tensor cores (sm_103a).
//
// Computes, per expert e and routed row j of that expert,
//   C[j][n] = bf16( sum_g a_s[g][j] * w_s[e][g][n] * sum_{k in g} e4m3(A[j][k]) * int4(W[e][n][k]) )
// which is the W4A8 grouped GEMM of the SGLang PR #7762 page (cutlass_w4a8_moe,
// group size / chunk_size 128) and, with one expert, the dense W4AFP8 Linear
// of the lyraW4AFp8 page.
//
// Design (one persistent CTA per SM; warp roles fixed per configuration):
//   * Operands are swapped so that the weights fill the 128-row M side of
//     tcgen05.mma and the few tokens of an expert sit on N (16..NMAX, any
//     multiple of 16).  Prior art: the swapAB small-batch path of the DeepGEMM
//     PR #53 page ("SM90 FP4 MegaMoE"); here it is the only mode, and N
//     shrinks to the expert's rows, so no row tile runs empty.
//   * The K loop runs in stages of gps 128-K groups of one tile.  A stage is
//     the unit of every barrier transaction below, so the fixed cost of a
//     hand-over (waits, fences, arrivals) is paid once per gps groups.
//   * warp 0: weight producer.  TMA loads the prepacked int4 tile of a stage
//     (64-byte swizzle, L2 evict-first) into a STAGES-deep ring.
//   * warp 1: token and scale producer.  TMA loads the E4M3 token tiles
//     (128-byte swizzle) into a TSTAGES ring and the fp32 token scales, group
//     corrections and weight scales into an SSTAGES ring.
//   * SETS x 4 converter warps: thread r owns weight row r, reads its 64
//     packed bytes per group and writes 128 E4M3 bytes of v + 1/2 (7 integer
//     operations per 8 weights, two 8-entry byte-permute lookups) into tensor
//     memory (A_TMEM) or the UMMA K-major 128-byte-swizzled shared layout.
//   * MMAS MMA warps: one thread each issues 4 tcgen05.mma (K = 32) per group
//     into that group's fp32 partial P in tensor memory.  An issuing thread
//     stalls about 120 cycles per tcgen05.mma whatever N is, so the groups of
//     a stage are dealt out to several issuing warps.
//   * epilogue warps: the scales differ per 128-K group, so each group's P
//     leaves the tensor core (tcgen05.ld) and is promoted in fp32:
//     acc += w_s * (a_s * P + gcorr), gcorr = -1/2 * a_s * sum(a) undoing the
//     +1/2 of the weight codes (the epilogue FFMA promotion the DeepGEMM PR #53
//     page describes for SM90, kept because the scales are arbitrary fp32
//     values).  At the end of a tile the accumulators are rounded to bf16.
//   * Every role walks all stages in order, splitting a stage's groups among
//     its warps, so each barrier's waiters meet its phases in order: the
//     condition under which a phase-parity wait cannot be satisfied by a stale
//     phase.
//   * Tiles: (expert, token chunk, 128-row weight block); chunks cut an
//     expert's rows on a grid of NMAX rows that starts at its first row rounded
//     down to a multiple of 4 (so scale vectors stay 16-byte aligned); the schedule is built
//     in shared memory from seg_indptr by every CTA (no host synchronisation,
//     no workspace), and CTAs stride over it.  Each CTA decodes its own tiles
//     once, in the prologue, into a shared-memory list that every role reads.
//   * Wide token tiles (128) promote from 16x256b tensor-memory fragments (4 rows
//     x 16 columns per thread, so a token scale read serves 4 rows) and move
//     registers from the producer/MMA and converter warpgroups to the epilogue
//     warpgroups with setmaxnreg.
//   * Configurations (host side, from the mean rows per expert and K): 16-wide
//     token tiles with 4 groups per stage for few rows per expert (4 MMA warps
//     for long K), 128-wide tiles with 2 groups per stage and the converted
//     weights in shared memory for many, both in two launches over disjoint
//     experts in between; split-K with fp32 partials for dense Linear calls
//     whose tiles leave SMs idle.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <atomic>
#include <cstring>

#include "common.cuh"

namespace w4a8 {
namespace {

constexpr int kBM = 128;      // weight rows per tile (MMA M)
constexpr int kKStep = 32;    // K per tcgen05.mma for 8-bit operands
constexpr int kWarpTma = 0;                  // producer of the weight ring
constexpr int kWarpTmaAct = 1;               // producer of the token and scale rings
constexpr int kWarpMma = 2;                  // warps 2 .. 1 + kMmaWarps issue the MMAs
constexpr int kConvWarps = 4;                // converter warps per set: one per tensor-memory lane quarter
constexpr int kMaxExperts = 1024;
constexpr int kMaxDynSmem = 227 * 1024;  // dynamic shared memory a CTA may use on sm_100 / sm_103
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s: no legitimate wait comes close

__device__ unsigned int g_gemm_error;

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// Every consumer works on whole pipeline stages (GPS 128-K groups of one tile): a stage is
// one barrier transaction for the converters, the MMA issue and the epilogue.
template <int NMAX_, int GPS_, int STAGES_, int TSTAGES_, int SSTAGES_, int ABUF_, int NP_, bool A_TMEM_, int SETS_,
          int MMAS_, int EPIW_, int EPIS_, bool FUSE_ = false>
struct Cfg {
  // warp roles: 0 weight producer | 1 token/scale producer | 2..1+MMAS MMA issue | SETS x 4 converters |
  // EPIW epilogue
  static constexpr int kConvSets = SETS_;   // converter sets: set c converts groups j % SETS == c of a stage
  static constexpr int kMmaWarps = MMAS_;   // MMA warps: warp m issues groups j % MMAS == m of a stage (a
                                            // thread stalls ~120 cycles per tcgen05.mma, so several
                                            // issuing warps keep the tensor core fed)
  static constexpr int kEpiWarps = EPIW_;   // 4 x column blocks x epilogue sets
  static constexpr int kEpiSets = EPIS_;    // epilogue sets: set c promotes groups j % EPIS == c of a stage
  static constexpr int kEpiSetWarps = EPIW_ / EPIS_;  // warps of one epilogue set (4 x column blocks)
  static constexpr int kEpiCols = NMAX_ * 4 / (EPIW_ / EPIS_);  // columns per epilogue warp
  static constexpr bool kEpi16 = NMAX_ >= 64 && EPIS_ == 1 && kEpiCols % 32 == 0;
  static constexpr int kWarpConv0 = kWarpMma + kMmaWarps;
  static constexpr int kWarpEpi0 = kWarpConv0 + kConvSets * kConvWarps;
  static constexpr int kWarps = kWarpEpi0 + kEpiWarps;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int NMAX = NMAX_;        // token tile (MMA N upper bound)
  static constexpr int GPS = GPS_;          // most 128-K groups per pipeline stage
  static constexpr int STAGES = STAGES_;    // weight ring: packed weights of a stage (freed by the converters)
  static constexpr int TSTAGES = TSTAGES_;  // token ring: token tiles of a stage (freed by the MMAs)
  static constexpr int SSTAGES = SSTAGES_;  // scale ring: token + weight scales of a stage (epilogue)
  static constexpr int ABUF = ABUF_;        // converted-weight slots (one stage each)
  static constexpr int NP = NP_;            // fp32 partial-product slots in tensor memory (one stage each)
  static constexpr bool A_TMEM = A_TMEM_;   // converted weights in tensor memory (else shared)
  static constexpr int kTokBytes = NMAX * 128;            // one group: NMAX rows x 128 B, 128B swizzle
  static constexpr int kWpkBytes = kBM * 64;              // one group: 128 rows x 64 B packed int4
  static constexpr int kABytes = kBM * 128;               // 128 rows x 128 B E4M3
  static constexpr int kTscBytes = (GPS * NMAX * 4 + 127) / 128 * 128;  // token scales (and corrections) of a slot
  static constexpr int kScBytes = 2 * kTscBytes + GPS * kBM * 4;        // one scale slot
  static constexpr int kOffTok = 0;
  static constexpr int kOffWpk = kOffTok + TSTAGES * GPS * kTokBytes;
  static constexpr int kOffA = kOffWpk + STAGES * GPS * kWpkBytes;
  static constexpr int kOffSc = kOffA + (A_TMEM ? 0 : ABUF * GPS * kABytes);
  // Fused SiLU-and-Mul requantisation (w13 only): gate and up tiles of the same 128 h-columns go to one
  // CTA in turn; the up tile's epilogue needs the E4M3 codes of its NMAX tokens staged as rows
  // [NMAX][kStageRow B] for coalesced stores, and per-lane-quarter partial amax and code sums [2][4][NMAX].
  static constexpr bool kFuse = FUSE_;
  static constexpr int kOffFuse = kOffSc + SSTAGES * kScBytes;
  static constexpr int kStageRow = 144;  // staged code row: 128 B + 16 B of padding (byte stores spread over banks)
  static constexpr int kFuseBytes = FUSE_ ? NMAX * kStageRow + 2 * 4 * NMAX * 4 : 0;
  // 16x256b epilogues without the fused requantisation: each epilogue warp's 1 KB tile-end staging block
  // (16 token rows x 64 B), through which stmatrix turns the weight-row-major fragments into token rows
  static constexpr int kOffEpiStg = kOffFuse + kFuseBytes;
  static constexpr int kEpiStgBytes = (kEpi16 && !FUSE_) ? EPIW_ * 1024 : 0;
  static constexpr int kOffBar = kOffEpiStg + kEpiStgBytes;
  // mbarrier area, in 8-byte slots: the rings, then xfull[2], xempty[2], hx[2] (used by the fused epilogue
  // only, always laid out) and mdrain[4]; the kernel takes every array's address from these offsets
  static constexpr int kBarFull = 0, kBarEmpty = kBarFull + STAGES;
  static constexpr int kBarTfull = kBarEmpty + STAGES, kBarTempty = kBarTfull + TSTAGES;
  static constexpr int kBarSfull = kBarTempty + TSTAGES, kBarSempty = kBarSfull + SSTAGES;
  static constexpr int kBarMready = kBarSempty + SSTAGES, kBarMdone = kBarMready + ABUF;
  static constexpr int kBarPfull = kBarMdone + ABUF, kBarPempty = kBarPfull + NP;
  static constexpr int kBarXfull = kBarPempty + NP, kBarXempty = kBarXfull + 2;
  static constexpr int kBarHx = kBarXempty + 2, kBarMdrain = kBarHx + 2;
  static constexpr int kNumBars = kBarMdrain + 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffSched = kOffMisc + 64;
  // schedule: [E+1] chunk prefix, [E+1] row starts, then (16-byte aligned) [cap] int4 tiles of this CTA
  __host__ __device__ static int tiles_off(int E) { return (kOffSched + 2 * (E + 1) * 4 + 15) & ~15; }
  static int smem_bytes(int E, int cap) { return tiles_off(E) + 16 * cap + 1024; }
  // tensor memory: [NP][GPS][NMAX] partials | [ABUF][GPS][32] converted weights (A_TMEM) |
  // with two epilogue sets, two NMAX-column slots (by tile parity) through which set 1 hands
  // its accumulators to set 0 at the end of a tile
  static constexpr int kAColBase = NP * GPS * NMAX;
  static constexpr int kXColBase = (kAColBase + (A_TMEM ? ABUF * GPS * 32 : 0) + 31) / 32 * 32;
  static constexpr int kTmemUsed = kXColBase + (EPIS_ > 1 ? 2 * NMAX : 0);
  static constexpr uint32_t kTmemCols = pow2_at_least(kTmemUsed);
  static_assert(NMAX % 16 == 0 && NMAX >= 16 && NMAX <= 256, "token tile");
  static_assert(kTokBytes % 1024 == 0 && kOffWpk % 1024 == 0 && kOffA % 1024 == 0, "alignment");
  static_assert(kOffSc % 128 == 0 && kScBytes % 128 == 0, "TMA destinations 128-byte aligned");
  static_assert(!FUSE_ || (NMAX_ == 128 && EPIS_ == 1 && EPIW_ == 8), "fused SiLU: 128-wide tiles, 8 epilogue warps");
  static_assert(kTmemUsed <= 512, "tensor memory");
  static_assert(EPIS_ == 1 || EPIS_ == 2, "one or two epilogue sets");
  static_assert(EPIW_ % (4 * EPIS_) == 0, "each epilogue set covers all four lane quarters");
  static_assert(kOffSched + 2 * 257 * 4 + 1024 <= 227 * 1024, "shared memory (256 experts)");
  // Wide tiles promote from 16x256b fragments: each epilogue thread holds 4 rows x 16 columns of a
  // 64-column block, so a token scale read from shared memory serves 4 rows (a 32x32b fragment, one
  // row per thread, makes every column's scale a 32-lane broadcast).  The fragments and the 64
  // accumulators need more registers than an even split gives, so these tiles also move registers
  // from the producer/MMA warpgroup and the converters to the epilogue warpgroups.
  static constexpr bool kRegSplit = kEpi16;
  // With one group per stage the MMA warps take whole stages in turn (warp m: stages st % MMAS == m)
  // instead of groups of a stage, and each stage's barriers get one commit.  A token or A slot is
  // then committed by one MMA warp only (its ring depth is a multiple of MMAS), so its phases
  // complete in order.  A partial slot may pass between MMA warps: the MMAs of stage st + NP wait
  // until the epilogue has read stage st, so its phases complete in order too, and an MMA warp
  // waiting on it is never two phases behind.
  static constexpr bool kMmaByStage = GPS_ == 1 && MMAS_ > 1;
  static constexpr int kMmaCommits = kMmaByStage ? 1 : MMAS_;
  static_assert(MMAS_ >= 1 && MMAS_ <= 4, "one to four MMA-issuing warps (one drain barrier each)");
  static_assert(!kMmaByStage || (TSTAGES_ % MMAS_ == 0 && ABUF_ % MMAS_ == 0),
                "stage-wise MMA warps: token and A ring depths must be multiples of the MMA warps");
  // Registers a thread gets at launch (the block's share of the 64 K register file, in steps of 8), and the
  // per-warpgroup budgets.  With two converter sets (640 threads) the converters work on quarter rows and
  // fit in 40 registers.
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8 > 255 ? 255 : (65536 / kThreads) / 8 * 8;
  static constexpr int kRegsCtl = SETS_ > 1 ? 48 : 72;   // warps 0-3: the two producers and the MMA warps
  static constexpr int kRegsConv = SETS_ > 1 ? 48 : 96;  // converter warpgroups
  static constexpr int kRegsEpi = 168;                   // epilogue warpgroups
  static_assert(!kRegSplit || (kWarpConv0 == 4 && kWarpEpi0 % 4 == 0 && kEpiWarps % 4 == 0),
                "register split: warp roles aligned to warpgroups");
  static_assert(!kRegSplit || 128 * kRegsCtl + 32 * kConvSets * kConvWarps * kRegsConv + 32 * EPIW_ * kRegsEpi <=
                                  kThreads * kLaunchRegs,
                "register split exceeds the registers the block is launched with");
};

struct GemmParams {
  const int64_t* seg;  // [E+1] or nullptr (dense: one expert with M rows)
  uint16_t* C;
  float* partial;      // split-K: fp32 partial sums [splits][M][N] instead of C (nullptr: write C)
  int E, N, K, M;      // M: rows of A (dense) / M_total
  int gps;             // 128-K groups per stage (divides K/128, <= Cfg::GPS)
  int splits;          // K splits per tile (1: none)
  int tile_cap;        // tiles per CTA the shared-memory tile list holds (0: decode each tile in place)
  int min_rows, max_rows;  // experts with a row count outside [min_rows, max_rows] are left to another launch
  // fused SiLU-and-Mul requantisation (N = 2 I): the gate tile's bf16 values go to gate [M][I] (scratch
  // read back by the same threads), the up tile's epilogue writes hq [M][I] E4M3, hs / hc [I/128][h_ld]
  uint16_t* gate;
  uint8_t* hq;
  float* hs;
  float* hc;
  int64_t h_ld;
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

// One prepacked 32-bit word (8 weights, see w4a8_prepack_weights) -> 8 E4M3 codes of v + 1/2.
// Nibble p holds the magnitude index m of element p in bits 0-2 (|v + 1/2| = m + 1/2) and,
// in bit 3, the sign of element 4 + p/2 (p even) or (p - 1)/2 (p odd): one 8-entry table
// serves both signs, and the sign bits sit on byte MSBs of w (elements 0-3) or w << 4 (4-7).
__device__ __forceinline__ void int4x8_to_e4m3x8(uint32_t w, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t kMag0 = 0x46423C30u;  // E4M3 of 0.5, 1.5, 2.5, 3.5
  constexpr uint32_t kMag1 = 0x4F4D4B49u;  //          4.5, 5.5, 6.5, 7.5
  const uint32_t idx = w & 0x77777777u;
  lo = prmt(kMag0, kMag1, idx) | (w & 0x80808080u);
  hi = prmt(kMag0, kMag1, idx >> 16) | ((w << 4) & 0x80808080u);
}

// Canonical packed int4 (byte b: element 2b in bits 0-3, 2b+1 in bits 4-7, two's complement)
// -> the prepacked word above.  Per element: s = sign bit, m = low three bits xor (s ? 7 : 0).
__global__ void __launch_bounds__(256) prepack_kernel(const uint32_t* __restrict__ in, uint32_t* __restrict__ out,
                                                      int64_t n_words) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t w = in[i];
    const uint32_t sgn = (w >> 3) & 0x11111111u;         // sign of element i in bit 4i
    const uint32_t m = (w ^ (sgn * 7u)) & 0x77777777u;     // magnitude index of element i in nibble i
    // sign of element e goes to bit 3 of nibble 2e+1 (e < 4) or 2(e-4) (e >= 4)
    uint32_t sb = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int p = e < 4 ? 2 * e + 1 : 2 * (e - 4);
      sb |= ((sgn >> (4 * e)) & 1u) << (4 * p + 3);
    }
    out[i] = m | sb;
  }
}

struct Sched {
  const int* prefix;  // [E+1] chunk prefix
  const int* start;   // [E+1] row starts
  const int4* tiles;  // this CTA's tiles {e, nb, row0, rows} in order, or nullptr (decode in place)
  int E, NMAX, nblk;
  int S, Gs, gps;     // K splits per tile, stages per tile, groups per stage
  int pairs;          // 1: tiles come in (gate block p, up block p + nblk / 2) pairs, a pair to one CTA
  // global item of this CTA's tile `it`: CTAs stride over items, or over pairs of items
  __device__ __forceinline__ int item_of(int it) const {
    return pairs ? 2 * (static_cast<int>(blockIdx.x) + (it >> 1) * static_cast<int>(gridDim.x)) + (it & 1)
                 : static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
  }
  // item = tile * S + split; split s covers stages [s*Gs/S, (s+1)*Gs/S) of the tile
  __device__ __forceinline__ void krange(int item, int& g_beg, int& g_end) const {
    const int sp = item % S;
    g_beg = (sp * Gs / S) * gps;
    g_end = ((sp + 1) * Gs / S) * gps;
  }
  __device__ __forceinline__ void decode(int item_, int& e, int& nb, int& row0, int& rows) const {
    const int item = item_ / S;
    int chunk;
    if (pairs) {  // item = 2 * (chunk * nblk / 2 + p) + half -> block p (gate) or p + nblk / 2 (up)
      const int np = nblk >> 1, pi = item >> 1;
      chunk = pi / np;
      nb = pi - chunk * np + (item & 1) * np;
    } else {
      chunk = item / nblk;
      nb = item - chunk * nblk;
    }
    int lo = 0, hi = E;  // prefix[lo] <= chunk < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= chunk) lo = mid; else hi = mid;
    }
    e = lo;
    // chunks sit on a grid of NMAX rows from the expert's first row rounded down to 4, so a
    // tile's token rows start 4-aligned (16-byte scale vectors) and only the first one is ragged
    const int st = start[e], end = start[e + 1];
    const int base = (st & ~3) + (chunk - prefix[e]) * NMAX;
    row0 = max(st, base);
    rows = min(end, base + NMAX) - row0;
  }
  // tile `it` of this CTA (item = blockIdx.x + it * gridDim.x)
  __device__ __forceinline__ void tile(int it, int item, int& e, int& nb, int& row0, int& rows) const {
    if (tiles) {
      const int4 t = tiles[it];
      e = t.x;
      nb = t.y;
      row0 = t.z;
      rows = t.w;
    } else {
      decode(item, e, nb, row0, rows);
    }
  }
};

// Waits for the phase of `bar` with the given parity, at most kTimeoutNs: on expiry it raises the CTA's
// abort flag and sets bit 0 of the device error word; it also gives up when another role has raised the
// flag.  Returns whether the phase completed.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t limit_ns = kTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 127u) == 127u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(&g_gemm_error, 1u);
        return false;
      }
    }
  }
}

// Waits (at most kTimeoutNs, whatever the abort flag) for an asynchronous operation this thread issued:
// after an abort the MMA-issuing threads let their MMAs finish, so that none writes tensor memory after
// the CTA has released it.  (On a normal exit the epilogue has waited for every MMA already.)  On expiry
// sets bit 2 of the error word.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      atomicOr(&g_gemm_error, 4u);
      return;
    }
  }
}

// An MMA-issuing thread after an abort: every MMA it issued has completed (a commit arrives once they have).
// (TMA loads already issued are not waited for: with a drain of the two producers' rings as well, the
// 16-row decode configuration measured 4 % slower, 0.620 -> 0.645 ms for the w13 launch.)
__device__ __forceinline__ void drain_mma(uint64_t* bar) {
  mma_commit(bar);
  drain_bar(bar, 0);
}

// A wait that nothing completes: thread 0 waits on a fresh mbarrier with the GEMM's bounded wait and a
// limit of limit_ns.  The wait gives up, raising the device error word as a timed-out GEMM wait does;
// *gave_up records it.  Lets a test run the timeout path without any TMA or MMA in flight.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns, int* gave_up) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) *gave_up = wait_bar(&bar, 0, &abort_flag, limit_ns) ? 0 : 1;
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

// acc2 += ws2 * ({t0, t1} * {p0, p1} + {k0, k1}): two fp32 lanes per instruction.  p is
// the tensor-core partial of (v + 1/2) * a, t the token scale and k = -1/2 * t * sum(a) the
// group correction, so t * p + k = t * sum(v * a); acc2 and ws2 = {ws, ws} are packed pairs.
__device__ __forceinline__ void promote2(uint64_t& acc2, uint64_t ws2, float t0, float t1, float k0, float k1,
                                         uint32_t p0, uint32_t p1) {
  uint64_t e, ts, ks, pp;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ts) : "f"(t0), "f"(t1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ks) : "f"(k0), "f"(k1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(pp) : "r"(p0), "r"(p1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(ts), "l"(pp), "l"(ks));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2) : "l"(ws2), "l"(e));
}

// The same promotion with the token scales and corrections already packed in pairs.
__device__ __forceinline__ void promote2p(uint64_t& acc2, uint64_t ws2, uint64_t ts2, uint64_t ks2, uint32_t p0,
                                          uint32_t p1) {
  uint64_t e, pp;
  asm("mov.b64 %0, {%1, %2};" : "=l"(pp) : "r"(p0), "r"(p1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(ts2), "l"(pp), "l"(ks2));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2) : "l"(ws2), "l"(e));
}

template <class CF, bool SPLIT>
__global__ void __launch_bounds__(CF::kThreads, 1)
    w4a8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAS,
                     const __grid_constant__ CUtensorMap tmAC, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmBS, const GemmParams prm) {
  constexpr int NMAX = CF::NMAX;
  constexpr int GPS = CF::GPS;
  constexpr int STAGES = CF::STAGES;
  constexpr int TSTAGES = CF::TSTAGES;
  constexpr int SSTAGES = CF::SSTAGES;
  constexpr int ABUF = CF::ABUF;
  constexpr int NP = CF::NP;
  constexpr int kConvSets = CF::kConvSets;
  constexpr int EPIS = CF::kEpiSets;
  constexpr int kWarpConv0 = CF::kWarpConv0;
  constexpr int kWarpEpi0 = CF::kWarpEpi0;
  constexpr int NHALF = NMAX * 4 / CF::kEpiSetWarps;  // columns per epilogue thread

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_tok = smem + CF::kOffTok;  // [TSTAGES][GPS][NMAX x 128 B]
  uint8_t* s_wpk = smem + CF::kOffWpk;  // [STAGES][GPS][128 x 64 B]
  uint8_t* s_a = smem + CF::kOffA;      // [ABUF][128 x 128 B]
  uint8_t* s_sc = smem + CF::kOffSc;    // [SSTAGES] slot: [GPS][NMAX] token scales, [GPS][NMAX] corrections,
                                        //   [GPS][128] weight scales
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::kOffBar);
  uint64_t* full = bars + CF::kBarFull;      // weight ring
  uint64_t* empty = bars + CF::kBarEmpty;
  uint64_t* tfull = bars + CF::kBarTfull;    // token ring
  uint64_t* tempty = bars + CF::kBarTempty;
  uint64_t* sfull = bars + CF::kBarSfull;    // scale ring
  uint64_t* sempty = bars + CF::kBarSempty;
  uint64_t* mready = bars + CF::kBarMready;  // [ABUF] converted weights of a stage ready for the MMAs
  uint64_t* mdone = bars + CF::kBarMdone;    // [ABUF] MMAs of the stage done: A slot free
  uint64_t* pfull = bars + CF::kBarPfull;    // [NP] MMAs of the stage done: partials ready
  uint64_t* pempty = bars + CF::kBarPempty;  // [NP] partial slot read by the epilogue
  uint64_t* xfull = bars + CF::kBarXfull;    // [2] epilogue set 1 -> set 0 hand-over slot written
  uint64_t* xempty = bars + CF::kBarXempty;  // [2] hand-over slot read
  uint64_t* hx = bars + CF::kBarHx;          // [2] fused SiLU: lane-quarter exchange of column block 0 / 1
  uint64_t* mdrain = bars + CF::kBarMdrain;  // [4] per MMA warp: its last MMAs complete (on leaving)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + CF::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + CF::kOffMisc + 4);
  const int E = prm.seg ? prm.E : 1;
  int* s_prefix = reinterpret_cast<int*>(smem + CF::kOffSched);  // [E+1]
  int* s_start = s_prefix + (E + 1);                              // [E+1]
  int4* s_tiles = reinterpret_cast<int4*>(smem + CF::tiles_off(E));  // [tile_cap]

  pdl_trigger();  // the next kernel may launch once every CTA has started (it waits for this grid)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = prm.K / kGroup;
  const int gps = prm.gps;
  const int nblk = prm.N / kBM;

  // ---- prologue: barriers, tensor memory, schedule ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConvSets * kConvWarps);  // every converter warp
    }
    for (int s = 0; s < TSTAGES; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], CF::kMmaCommits);  // one commit per MMA warp taking part in the stage
    }
    for (int s = 0; s < SSTAGES; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], CF::kEpiWarps);  // every epilogue warp
    }
    for (int b = 0; b < ABUF; ++b) {
      mbar_init(&mready[b], kConvSets * kConvWarps);
      mbar_init(&mdone[b], CF::kMmaCommits);
    }
    for (int b = 0; b < NP; ++b) {
      mbar_init(&pfull[b], CF::kMmaCommits);
      mbar_init(&pempty[b], CF::kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xfull[b], CF::kEpiSetWarps);
      mbar_init(&xempty[b], CF::kEpiSetWarps);
    }
    if constexpr (CF::kFuse) {
      mbar_init(&hx[0], 4);  // the four warps (lane quarters) of a 64-column block
      mbar_init(&hx[1], 4);
    }
    for (int m = 0; m < 4; ++m) mbar_init(&mdrain[m], 1);
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
    tma_prefetch_desc(&tmAC);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmBS);
  }
  // everything above touched only this CTA's own state; inputs written by earlier kernels from here on
  pdl_wait();
  if (warp == kWarpConv0) {  // chunk prefix over experts (warp-wide scan)
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
      int v = cnt > 0 ? ((st & 3) + cnt + NMAX - 1) / NMAX : 0;  // chunks on the NMAX-row grid
      if (cnt < prm.min_rows || cnt > prm.max_rows) v = 0;        // another launch's expert
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

  // This CTA's tiles, decoded once here by all threads (a tile's decode is a binary search over the
  // experts, a chain of dependent shared-memory loads that cost each role ~1500 cycles per tile
  // under load); every role then reads a tile with one 16-byte load.
  const int S = SPLIT ? prm.splits : 1;  // 1 folds the split arithmetic away
  Sched sch{s_prefix, s_start, nullptr, E, NMAX, nblk, S, G / gps, gps, CF::kFuse ? 1 : 0};
  // units the CTAs stride over: tiles (x K splits), or gate/up tile pairs
  const int n_units = s_prefix[E] * nblk * S / (CF::kFuse ? 2 : 1);
  const int n_mine_units = n_units > static_cast<int>(blockIdx.x)
                               ? (n_units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                     static_cast<int>(gridDim.x)
                               : 0;
  const int n_mine = n_mine_units * (CF::kFuse ? 2 : 1);  // this CTA's tiles
  if (n_mine <= prm.tile_cap) {
    for (int i = threadIdx.x; i < n_mine; i += blockDim.x) {
      int e, nb, row0, rows;
      sch.decode(sch.item_of(i), e, nb, row0, rows);
      s_tiles[i] = make_int4(e, nb, row0, rows);
    }
    sch.tiles = s_tiles;
  }
  __syncthreads();

  const uint32_t tmem_base = *s_tmem;

  // Counters: `it` counts 128-K groups, `st` counts stages of gps groups; stage st holds
  // groups [st*gps, st*gps + gps) of one tile (gps divides K/128, so stages never straddle
  // tiles).  A tile covers token rows [row0 & ~3, ...): the scale vectors start 16-byte aligned.
  // Warp roles, grouped by warpgroup; with a register split every warp of a warpgroup first executes
  // the same setmaxnreg instruction.
  if (warp < kWarpConv0) {
    if constexpr (CF::kRegSplit) regs_release<CF::kRegsCtl>();
    if (warp == kWarpTma) {
      // ---- weight ring producer: runs ahead of everything else ----
      if (lane == 0) {
        const uint64_t pol_w = l2_policy_evict_first();
        const uint32_t w_bytes = gps * CF::kWpkBytes;
        uint32_t st = 0;
        for (int it = 0; it < n_mine; ++it) {
          const int item = sch.item_of(it);
          int e, nb, row0, rows;
          sch.tile(it, item, e, nb, row0, rows);
          int g_beg, g_end;
          sch.krange(item, g_beg, g_end);
          for (int g0 = g_beg; g0 < g_end; g0 += gps, ++st) {
            const int s = st % STAGES;
            const uint32_t ph = (st / STAGES) & 1;
            if (!wait_bar(&empty[s], ph ^ 1, s_abort)) goto done;
            mbar_arrive_expect_tx(&full[s], w_bytes);
            tma_load_3d_hint(s_wpk + s * GPS * CF::kWpkBytes, &tmB, &full[s], 0, e * prm.N + nb * kBM, g0, pol_w);
          }
        }
      }
    } else if (warp == kWarpTmaAct) {
      // ---- token and scale ring producer ----
      if (lane == 0) {
        const uint32_t t_bytes = gps * CF::kTokBytes;
        const uint32_t sc_bytes = gps * (2 * NMAX * 4 + kBM * 4);
        uint32_t st = 0;
        for (int it = 0; it < n_mine; ++it) {
          const int item = sch.item_of(it);
          int e, nb, row0, rows;
          sch.tile(it, item, e, nb, row0, rows);
          const int r4 = row0 & ~3;
          int g_beg, g_end;
          sch.krange(item, g_beg, g_end);
          for (int g0 = g_beg; g0 < g_end; g0 += gps, ++st) {
            const int ts_ = st % TSTAGES;
            const uint32_t tph = (st / TSTAGES) & 1;
            const int ss = st % SSTAGES;
            const uint32_t sph = (st / SSTAGES) & 1;
            if (!wait_bar(&tempty[ts_], tph ^ 1, s_abort)) goto done;
            mbar_arrive_expect_tx(&tfull[ts_], t_bytes);
            tma_load_3d(s_tok + ts_ * GPS * CF::kTokBytes, &tmA, &tfull[ts_], 0, r4, g0);
            if (!wait_bar(&sempty[ss], sph ^ 1, s_abort)) goto done;
            uint8_t* sc = s_sc + ss * CF::kScBytes;
            mbar_arrive_expect_tx(&sfull[ss], sc_bytes);
            tma_load_2d(sc, &tmAS, &sfull[ss], r4, g0);
            tma_load_2d(sc + CF::kTscBytes, &tmAC, &sfull[ss], r4, g0);
            tma_load_2d(sc + 2 * CF::kTscBytes, &tmBS, &sfull[ss], nb * kBM, e * G + g0);
          }
        }
      }
    } else {
      // ---- MMA issue: every stage, warp m issuing the groups j with j % kMmaWarps == m; with one
      // group per stage, the stages st with st % kMmaWarps == m ----
      const int mset = warp - kWarpMma;
      if (lane == 0) {
        uint32_t st = 0;
        // the next tile's entry is loaded a tile ahead: a tile change costs the MMA issue no load latency
        int4 nxt = sch.tiles && n_mine > 0 ? sch.tiles[0] : make_int4(0, 0, 0, 0);
        for (int it = 0; it < n_mine; ++it) {
          const int item = sch.item_of(it);
          int e, nb, row0, rows;
          if (sch.tiles) {
            row0 = nxt.z;
            rows = nxt.w;
            if (it + 1 < n_mine) nxt = sch.tiles[it + 1];
          } else {
            sch.decode(item, e, nb, row0, rows);
          }
          const int ncol = (row0 - (row0 & ~3) + rows + 15) & ~15;
          const uint32_t idesc = idesc_e4m3(static_cast<uint32_t>(ncol));
          int g_beg, g_end;
          sch.krange(item, g_beg, g_end);
          for (int g0 = g_beg; g0 < g_end; g0 += gps, ++st) {
            if constexpr (CF::kMmaByStage) {
              if (static_cast<int>(st % CF::kMmaWarps) != mset) continue;
            }
            const int ts_ = st % TSTAGES;
            const uint32_t tph = (st / TSTAGES) & 1;
            const int a = st % ABUF;
            const uint32_t aph = (st / ABUF) & 1;
            const int pslot = st % NP;
            const uint32_t pph = (st / NP) & 1;
            // token tiles landed, weights converted, partial slot read by the epilogue
            const bool ok = mbar_test3(&tfull[ts_], tph, &mready[a], aph, &pempty[pslot], pph ^ 1) ||
                            (wait_bar(&tfull[ts_], tph, s_abort) && wait_bar(&mready[a], aph, s_abort) &&
                             wait_bar(&pempty[pslot], pph ^ 1, s_abort));
            if (!ok) goto m_drain;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < GPS; ++j) {
              if (j >= gps) break;
              if (!CF::kMmaByStage && j % CF::kMmaWarps != mset) continue;
              const uint32_t d = tmem_base + (pslot * GPS + j) * NMAX;
              const uint32_t tok = smem_u32(s_tok + (ts_ * GPS + j) * CF::kTokBytes);
#pragma unroll
              for (int kk = 0; kk < kGroup / kKStep; ++kk) {
                const uint64_t bdesc = sw128_desc(tok + kk * kKStep);
                if constexpr (CF::A_TMEM) {
                  const uint32_t a_t = tmem_base + CF::kAColBase + (a * GPS + j) * 32 + kk * (kKStep / 4);
                  mma_f8f6f4_ts(d, a_t, bdesc, idesc, kk > 0 ? 1u : 0u);
                } else {
                  const uint64_t adesc = sw128_desc(smem_u32(s_a + (a * GPS + j) * CF::kABytes) + kk * kKStep);
                  mma_f8f6f4_ss(d, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                }
              }
            }
            // a commit arrives once this thread's earlier MMAs are complete (at once if it issued none)
            mma_commit(&pfull[pslot]);
            mma_commit(&mdone[a]);
            mma_commit(&tempty[ts_]);
          }
        }
      m_drain:  // after an abort, the MMAs this thread issued complete before the CTA releases tensor memory
        if (*s_abort) drain_mma(&mdrain[mset]);
      }
    }
  } else if (warp < kWarpEpi0) {
    if constexpr (CF::kRegSplit) regs_release<CF::kRegsConv>();
    // ---- converters: every stage; set c converts the groups j with j % kConvSets == c ----
    const int q4 = warp & 3;
    const int cset = (warp - kWarpConv0) / kConvWarps;
    const int r = q4 * 32 + lane;
    uint32_t st = 0;
    for (int it = 0; it < n_mine; ++it) {
          const int item = sch.item_of(it);
      int g_beg, g_end;
      sch.krange(item, g_beg, g_end);
      for (int g0 = g_beg; g0 < g_end; g0 += gps, ++st) {
        const int s = st % STAGES;
        const uint32_t ph = (st / STAGES) & 1;
        const int a = st % ABUF;
        const uint32_t aph = (st / ABUF) & 1;
        // weights landed; the A slot's previous MMAs done
        bool ok = true;
        if (!mbar_try_wait(&full[s], ph) || !mbar_try_wait(&mdone[a], aph ^ 1))
          ok = wait_bar(&full[s], ph, s_abort) && wait_bar(&mdone[a], aph ^ 1, s_abort);
        if (__any_sync(0xffffffffu, !ok)) goto done;  // warp-uniform; the warp is converged below
#pragma unroll
        for (int j = 0; j < GPS; ++j) {
          if (j >= gps) break;
          if (j % kConvSets != cset) continue;
          const uint8_t* wrow = s_wpk + (s * GPS + j) * CF::kWpkBytes + r * 64;
          if constexpr (CF::A_TMEM) {
            // two halves of 64 weights: 8 packed words -> 16 E4M3 words -> 16 tensor-memory columns
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t in[8];
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const uint4 v = *reinterpret_cast<const uint4*>(wrow + (((2 * hh + q) ^ ((r >> 1) & 3)) << 4));
                in[4 * q + 0] = v.x;
                in[4 * q + 1] = v.y;
                in[4 * q + 2] = v.z;
                in[4 * q + 3] = v.w;
              }
              uint32_t out[16];
#pragma unroll
              for (int i = 0; i < 8; ++i) int4x8_to_e4m3x8(in[i], out[2 * i], out[2 * i + 1]);
              tmem_st16(tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + CF::kAColBase + (a * GPS + j) * 32 + 16 * hh,
                        out);
            }
          } else if constexpr (kConvSets > 1) {
            // quarter rows (16 packed bytes -> 32 E4M3 bytes at a time): few registers, several sets
            uint8_t* arow = s_a + (a * GPS + j) * CF::kABytes + r * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((q ^ ((r >> 1) & 3)) << 4));
              const uint32_t in[4] = {v.x, v.y, v.z, v.w};
              uint32_t out[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) int4x8_to_e4m3x8(in[i], out[2 * i], out[2 * i + 1]);
              *reinterpret_cast<uint4*>(arow + (((2 * q) ^ (r & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
              *reinterpret_cast<uint4*>(arow + (((2 * q + 1) ^ (r & 7)) << 4)) =
                  make_uint4(out[4], out[5], out[6], out[7]);
            }
          } else {
            uint32_t in[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((q ^ ((r >> 1) & 3)) << 4));
              in[4 * q + 0] = v.x;
              in[4 * q + 1] = v.y;
              in[4 * q + 2] = v.z;
              in[4 * q + 3] = v.w;
            }
            uint32_t out[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) int4x8_to_e4m3x8(in[i], out[2 * i], out[2 * i + 1]);
            uint8_t* arow = s_a + (a * GPS + j) * CF::kABytes + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) =
                  make_uint4(out[4 * c], out[4 * c + 1], out[4 * c + 2], out[4 * c + 3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // every packed byte this warp reads is in registers by now
        if constexpr (CF::A_TMEM) {
          tmem_wait_st();
          tc_fence_before();
        } else {
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&mready[a]);
      }
    }
  } else {
    if constexpr (CF::kRegSplit) regs_claim<CF::kRegsEpi>();
    if constexpr (CF::kEpi16) {
      // 16x256b fragments: thread t of the warp for lane quarter q4 and its NHALF columns from c0 holds,
      // for each 32-column block hb, rows q4*32 + t/4 + 8*rho (rho = 0..3) and columns
      // c0 + 32*hb + 8*v + 2*(t%4) + {0, 1} (v = 0..3): a token scale pair read from shared memory
      // serves four rows.  Same promotion, same order of groups as the 32x32b path below.
      constexpr int NB32 = NHALF / 32;
      const int ew = warp - kWarpEpi0;
      const int q4 = warp & 3;
      const int c0 = (ew >> 2) * NHALF;
      const int rq = q4 * 32 + (lane >> 2);
      const int cq = 2 * (lane & 3);
      const uint32_t t_lane = static_cast<uint32_t>(q4 * 32) << 16;
      uint32_t st = 0;
      uint32_t hx_phase = 0;  // fused SiLU: completed exchanges of this warp's column block
      for (int it = 0; it < n_mine; ++it) {
          const int item = sch.item_of(it);
        int e, nb, row0, rows;
        sch.tile(it, item, e, nb, row0, rows);
        const int r4 = row0 & ~3;
        const int lo = row0 - r4;    // columns [lo, lo + rows) of the tile are this chunk's rows
        const int need = lo + rows;  // 32-column blocks from `need` on are never stored: skipped
        uint64_t acc2[NB32][4][4];
#pragma unroll
        for (int hb = 0; hb < NB32; ++hb)
#pragma unroll
          for (int rho = 0; rho < 4; ++rho)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc2[hb][rho][v] = 0ull;
        int g_beg, g_end;
        sch.krange(item, g_beg, g_end);
        for (int g0 = g_beg; g0 < g_end; g0 += gps, ++st) {
          const int ss = st % SSTAGES;
          const uint32_t sph = (st / SSTAGES) & 1;
          const int pslot = st % NP;
          const uint32_t pph = (st / NP) & 1;
          const float* tsc = reinterpret_cast<const float*>(s_sc + ss * CF::kScBytes);
          const float* tcr = reinterpret_cast<const float*>(s_sc + ss * CF::kScBytes + CF::kTscBytes);
          const float* wsc = reinterpret_cast<const float*>(s_sc + ss * CF::kScBytes + 2 * CF::kTscBytes);
          bool ok = true;
          if (!mbar_try_wait(&sfull[ss], sph) || !mbar_try_wait(&pfull[pslot], pph))
            ok = wait_bar(&sfull[ss], sph, s_abort) && wait_bar(&pfull[pslot], pph, s_abort);
          if (__any_sync(0xffffffffu, !ok)) goto done;  // warp converged below
          tc_fence_after();
          if (gps == GPS && need >= c0 + NHALF) {
            // every 32-column block of every group of the stage is promoted: the next block's
            // tensor-memory read is issued before the current block is promoted (two buffers), so each
            // wait covers one read that has been in flight for a block's promotion
            uint32_t qa0[16], qb0[16], qa1[16], qb1[16];
            {
              const uint32_t pa0 = tmem_base + t_lane + (pslot * GPS) * NMAX + c0;
              tmem_ld16x256b_x4(pa0, qa0);
              tmem_ld16x256b_x4(pa0 + (16u << 16), qb0);
              tmem_wait_ld_pin<16>(qa0);
#pragma unroll
              for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(qb0[i]));
            }
            uint64_t ws2[4];
#pragma unroll
            for (int u = 0; u < GPS * NB32; ++u) {
              const int j = u / NB32, hb = u % NB32;
              uint32_t* ca = (u & 1) ? qa1 : qa0;
              uint32_t* cb = (u & 1) ? qb1 : qb0;
              uint32_t* na = (u & 1) ? qa0 : qa1;
              uint32_t* nbuf = (u & 1) ? qb0 : qb1;
              if (u + 1 < GPS * NB32) {
                const int j1 = (u + 1) / NB32, hb1 = (u + 1) % NB32;
                const uint32_t pa1 = tmem_base + t_lane + (pslot * GPS + j1) * NMAX + c0 + 32 * hb1;
                tmem_ld16x256b_x4(pa1, na);
                tmem_ld16x256b_x4(pa1 + (16u << 16), nbuf);
              }
              if (hb == 0) {
#pragma unroll
                for (int rho = 0; rho < 4; ++rho) {
                  const float w = wsc[j * kBM + rq + 8 * rho];
                  asm("mov.b64 %0, {%1, %1};" : "=l"(ws2[rho]) : "f"(w));
                }
              }
              const float* ts = tsc + j * NMAX + c0 + cq + 32 * hb;
              const float* tc = tcr + j * NMAX + c0 + cq + 32 * hb;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint64_t t2 = *reinterpret_cast<const uint64_t*>(ts + 8 * v);
                const uint64_t k2 = *reinterpret_cast<const uint64_t*>(tc + 8 * v);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                  for (int jj = 0; jj < 2; ++jj) {
                    const uint32_t* cur = h ? cb : ca;
                    const int i = 4 * v + 2 * jj;
                    promote2p(acc2[hb][2 * h + jj][v], ws2[2 * h + jj], t2, k2, cur[i], cur[i + 1]);
                  }
              }
              if (u + 1 < GPS * NB32) {
                tmem_wait_ld_pin<16>(na);
#pragma unroll
                for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(nbuf[i]));
              }
            }
          } else
#pragma unroll
          for (int j = 0; j < GPS; ++j) {
            if (j >= gps) break;
            const float* wsj = wsc + j * kBM + rq;
            const float* ts = tsc + j * NMAX + c0 + cq;
            const float* tc = tcr + j * NMAX + c0 + cq;
            if (c0 >= need) continue;  // warp-uniform: none of this warp's columns is stored
            uint64_t ws2[4];
#pragma unroll
            for (int rho = 0; rho < 4; ++rho) {
              const float w = wsj[8 * rho];
              asm("mov.b64 %0, {%1, %1};" : "=l"(ws2[rho]) : "f"(w));
            }
            // the partials in 32-column blocks, one tensor-memory wait each (reading them in 16-column
            // chunks, each chunk's read in flight while the previous one is promoted, measured 2 %
            // slower: a wait per 16 columns)
            const uint32_t pa = tmem_base + t_lane + (pslot * GPS + j) * NMAX + c0;
#pragma unroll
            for (int hb = 0; hb < NB32; ++hb) {
              if (c0 + 32 * hb >= need) continue;  // warp-uniform
              uint32_t qa[16], qb[16];  // lanes +0 and +16 of the quarter: rows rho = 0, 1 and 2, 3
              tmem_ld16x256b_x4(pa + 32 * hb, qa);
              tmem_ld16x256b_x4(pa + 32 * hb + (16u << 16), qb);
              tmem_wait_ld_pin<16>(qa);
#pragma unroll
              for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(qb[i]));
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint64_t t2 = *reinterpret_cast<const uint64_t*>(ts + 32 * hb + 8 * v);
                const uint64_t k2 = *reinterpret_cast<const uint64_t*>(tc + 32 * hb + 8 * v);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                  for (int jj = 0; jj < 2; ++jj) {
                    const uint32_t* cur = h ? qb : qa;
                    const int i = 4 * v + 2 * jj;
                    promote2p(acc2[hb][2 * h + jj][v], ws2[2 * h + jj], t2, k2, cur[i], cur[i + 1]);
                  }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&pempty[pslot]);
            mbar_arrive(&sempty[ss]);
          }
        }
        if constexpr (CF::kFuse) {
          // SiLU-and-Mul with FP8 requantisation fused into the w13 epilogue: tile `it` of a gate / up pair.
          // The gate tile's values, rounded to bf16 as the unfused path stores them, go to the gate
          // scratch; the same threads read them back in the up tile and form h = silu(gate) * up, the
          // amax and the E4M3 code sum of each token's 128 h-columns (own 4 rows, the 8 lanes of the
          // lane quarter by shuffles, the 4 quarters through shared memory), the codes, the scale and the
          // correction, with the arithmetic of the SiLU-and-Mul kernel (the same bits).
          const int np = nblk >> 1;
          const int I = prm.N >> 1;
          if (c0 >= need) continue;  // no row of this chunk in the warp's columns (the whole 64-column block)
          if (nb < np) {  // gate tile
#pragma unroll
            for (int rho = 0; rho < 4; ++rho)
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                float a[2];
                asm("mov.b64 {%0, %1}, %2;" : "=f"(a[0]), "=f"(a[1]) : "l"(acc2[v >> 2][rho][v & 3]));
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                  const int t = c0 + 8 * v + cq + q;
                  if (t < lo || t >= need) continue;
                  prm.gate[static_cast<int64_t>(r4 + t) * I + nb * kBM + rq + 8 * rho] = float_to_bf16_bits(a[q]);
                }
              }
            continue;
          }
          const int gI = nb - np;  // h-group of the up block
          const int cb = c0 >> 6;  // column block: warps 0-3 (columns 0-63) or 4-7 (64-127)
          uint8_t* stage = smem + CF::kOffFuse;                                               // [NMAX][kStageRow]
          float* xmax = reinterpret_cast<float*>(smem + CF::kOffFuse + NMAX * CF::kStageRow);  // [4][NMAX]
          int* xsum = reinterpret_cast<int*>(xmax + 4 * NMAX);                        // [4][NMAX]
          float hv[4][8][2];
          {
            uint16_t gv[4][8][2];
#pragma unroll
            for (int rho = 0; rho < 4; ++rho)
#pragma unroll
              for (int v = 0; v < 8; ++v)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                  const int t = c0 + 8 * v + cq + q;
                  gv[rho][v][q] = (t >= lo && t < need)
                                      ? prm.gate[static_cast<int64_t>(r4 + t) * I + gI * kBM + rq + 8 * rho]
                                      : uint16_t(0);
                }
#pragma unroll
            for (int rho = 0; rho < 4; ++rho)
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                float a[2];
                asm("mov.b64 {%0, %1}, %2;" : "=f"(a[0]), "=f"(a[1]) : "l"(acc2[v >> 2][rho][v & 3]));
#pragma unroll
                for (int q = 0; q < 2; ++q)
                  hv[rho][v][q] = silu_mul(bf16_bits_to_float(gv[rho][v][q]),
                                           bf16_bits_to_float(float_to_bf16_bits(a[q])));
              }
          }
          // amax of each token column over its 128 h-columns
          float m[8][2];
#pragma unroll
          for (int v = 0; v < 8; ++v)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              float x = fmaxf(fmaxf(fabsf(hv[0][v][q]), fabsf(hv[1][v][q])), fmaxf(fabsf(hv[2][v][q]), fabsf(hv[3][v][q])));
#pragma unroll
              for (int o = 4; o < 32; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
              m[v][q] = x;
            }
          if ((lane >> 2) == 0) {
#pragma unroll
            for (int v = 0; v < 8; ++v) *reinterpret_cast<float2*>(xmax + q4 * NMAX + c0 + 8 * v + cq) = make_float2(m[v][0], m[v][1]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&hx[cb]);
          if (__any_sync(0xffffffffu, !wait_bar(&hx[cb], hx_phase & 1, s_abort))) goto done;
          ++hx_phase;
          float sc[8][2], rc[8][2];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float2 x = *reinterpret_cast<const float2*>(xmax + c0 + 8 * v + cq);
#pragma unroll
            for (int qq = 1; qq < 4; ++qq) {
              const float2 y = *reinterpret_cast<const float2*>(xmax + qq * NMAX + c0 + 8 * v + cq);
              x.x = fmaxf(x.x, y.x);
              x.y = fmaxf(x.y, y.y);
            }
            sc[v][0] = __fdiv_rn(fmaxf(x.x, 1e-12f), 448.0f);
            sc[v][1] = __fdiv_rn(fmaxf(x.y, 1e-12f), 448.0f);
            rc[v][0] = __frcp_rn(sc[v][0]);
            rc[v][1] = __frcp_rn(sc[v][1]);
          }
          // codes (staged as token rows) and each token's exact code sum in units of 2^-9
          int un[8][2];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int rho = 0; rho < 4; ++rho) {
              const uint16_t c2 = e4m3x2(div_by_scale(hv[rho][v][0], sc[v][0], rc[v][0]),
                                         div_by_scale(hv[rho][v][1], sc[v][1], rc[v][1]));
              const int t = c0 + 8 * v + cq;
              stage[t * CF::kStageRow + rq + 8 * rho] = static_cast<uint8_t>(c2 & 0xFF);
              stage[(t + 1) * CF::kStageRow + rq + 8 * rho] = static_cast<uint8_t>(c2 >> 8);
              uint32_t h2;
              asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
              s0 += f.x;
              s1 += f.y;
            }
            un[v][0] = __float2int_rn(s0 * 512.0f);
            un[v][1] = __float2int_rn(s1 * 512.0f);
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int o = 4; o < 32; o <<= 1) un[v][q] += __shfl_xor_sync(0xffffffffu, un[v][q], o);
          }
          if ((lane >> 2) == 0) {
#pragma unroll
            for (int v = 0; v < 8; ++v) *reinterpret_cast<int2*>(xsum + q4 * NMAX + c0 + 8 * v + cq) = make_int2(un[v][0], un[v][1]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&hx[cb]);
          if (__any_sync(0xffffffffu, !wait_bar(&hx[cb], hx_phase & 1, s_abort))) goto done;
          ++hx_phase;
          if (q4 == 0 && (lane >> 2) == 0) {  // the scale and correction of each token
#pragma unroll
            for (int v = 0; v < 8; ++v)
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const int t = c0 + 8 * v + cq + q;
                if (t < lo || t >= need) continue;
                int u = 0;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) u += xsum[qq * NMAX + t];
                prm.hs[gI * prm.h_ld + r4 + t] = sc[v][q];
                if (prm.hc) prm.hc[gI * prm.h_ld + r4 + t] = corr_from_units(u, sc[v][q]);
              }
          }
          // each warp of the column block writes 16 of its 64 token rows of codes, 16 bytes per lane
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int t = c0 + q4 * 16 + 4 * k + (lane >> 3);
            if (t < lo || t >= need) continue;
            const uint4 w = *reinterpret_cast<const uint4*>(stage + t * CF::kStageRow + (lane & 7) * 16);
            *reinterpret_cast<uint4*>(prm.hq + static_cast<int64_t>(r4 + t) * I + gI * kBM + (lane & 7) * 16) = w;
          }
          continue;
        }
        if constexpr (!SPLIT && CF::kEpiStgBytes > 0) {
          // The tile's bf16 values through the warp's staging block, 16 tokens at a time: an 8 x 8
          // fragment (weight rows x tokens) is stored transposed by stmatrix, as 8 token rows of 16
          // bytes, and read back as 16-byte pieces of token rows (8 consecutive output columns), one
          // global store each (C is 16-byte aligned, as the entry points require, and N a multiple of
          // 128).  Chunk c of staging row r sits at 16 * (c ^ ((r >> 1) & 3)): the 8 rows of a matrix
          // and the 8 pieces of a quarter warp's read fall on distinct banks.
          uint8_t* stg = smem + CF::kOffEpiStg + ew * 1024;
          const uint32_t stg_s = smem_u32(stg);
          const int mi = lane >> 3, mk = lane & 7;  // stmatrix row address: matrix mi (= rho), its row mk
          const int rr = lane >> 2, rc = lane & 3;  // read-back: staging rows rr and rr + 8, chunk rc
#pragma unroll
          for (int hb = 0; hb < NB32; ++hb)
#pragma unroll
            for (int vp = 0; vp < 2; ++vp) {
              if (c0 + 32 * hb + 16 * vp >= need) continue;  // warp-uniform: none of these 16 tokens stored
              __syncwarp();  // the previous round's reads are done
#pragma unroll
              for (int vv = 0; vv < 2; ++vv) {
                uint32_t r[4];
#pragma unroll
                for (int rho = 0; rho < 4; ++rho) {
                  float a0, a1;
                  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc2[hb][rho][2 * vp + vv]));
                  r[rho] = bf16x2_bits(a0, a1);
                }
                const int row = 8 * vv + mk;  // token c0 + 32 hb + 16 vp + row
                stmatrix_x4_trans(stg_s + row * 64 + ((mi ^ ((row >> 1) & 3)) << 4), r);
              }
              __syncwarp();
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int row = rr + 8 * h;
                const int t = c0 + 32 * hb + 16 * vp + row;
                const uint4 w = *reinterpret_cast<const uint4*>(stg + row * 64 + ((rc ^ ((row >> 1) & 3)) << 4));
                if (t >= lo && t < need)
                  st_global_na_v4(prm.C + static_cast<int64_t>(r4 + t) * prm.N + nb * kBM + q4 * 32 + 8 * rc, w);
              }
            }
          continue;
        }
#pragma unroll
        for (int hb = 0; hb < NB32; ++hb)
#pragma unroll
          for (int rho = 0; rho < 4; ++rho)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float a[2];
              asm("mov.b64 {%0, %1}, %2;" : "=f"(a[0]), "=f"(a[1]) : "l"(acc2[hb][rho][v]));
              const int n = nb * kBM + rq + 8 * rho;  // output column: weight row of the block
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const int t = c0 + 32 * hb + 8 * v + cq + q;  // tile column: token row r4 + t
                if (t < lo || t >= need) continue;
                const int64_t m = r4 + t;
                if (SPLIT)
                  prm.partial[(static_cast<int64_t>(item % sch.S) * prm.M + m) * prm.N + n] = a[q];
                else
                  st_global_na_u16(prm.C + m * prm.N + n, float_to_bf16_bits(a[q]));
              }
            }
      }
    } else {
      // ---- promotion and epilogue ----
      // Warp w: lane quarter q4 = w & 3, epilogue set `eset` (the groups j of every stage with
      // j % EPIS == eset) and, within the set, column block `half`.
      const int ew = warp - kWarpEpi0;
      const int q4 = warp & 3;
      const int eset = ew / CF::kEpiSetWarps;
      const int half = (ew % CF::kEpiSetWarps) >> 2;
      const int r = q4 * 32 + lane;
      const int c0 = half * NHALF;
      const uint32_t t_lane = static_cast<uint32_t>(q4 * 32) << 16;
      constexpr int CH = NHALF < 16 ? 8 : 16;  // columns per tensor-memory load
      uint32_t st = 0, tile = 0;
      for (int it = 0; it < n_mine; ++it, ++tile) {
        const int item = sch.item_of(it);
        int e, nb, row0, rows;
        sch.tile(it, item, e, nb, row0, rows);
        const int r4 = row0 & ~3;
        const int lo = row0 - r4;   // columns [lo, lo + rows) of the tile are this chunk's rows
        const int need = lo + rows;  // columns past `need` are never stored: skip their promotion
        uint64_t acc2[NHALF / 2];   // packed pairs of fp32 accumulators
#pragma unroll
        for (int q = 0; q < NHALF / 2; ++q) acc2[q] = 0ull;
        int g_beg, g_end;
        sch.krange(item, g_beg, g_end);
        for (int g0 = g_beg; g0 < g_end; g0 += gps, ++st) {
          const int ss = st % SSTAGES;
          const uint32_t sph = (st / SSTAGES) & 1;
          const int pslot = st % NP;
          const uint32_t pph = (st / NP) & 1;
          const float* tsc = reinterpret_cast<const float*>(s_sc + ss * CF::kScBytes);
          const float* tcr = reinterpret_cast<const float*>(s_sc + ss * CF::kScBytes + CF::kTscBytes);
          const float* wsc = reinterpret_cast<const float*>(s_sc + ss * CF::kScBytes + 2 * CF::kTscBytes);
          bool ok = true;
          if (!mbar_try_wait(&sfull[ss], sph) || !mbar_try_wait(&pfull[pslot], pph))
            ok = wait_bar(&sfull[ss], sph, s_abort) && wait_bar(&pfull[pslot], pph, s_abort);
          if (__any_sync(0xffffffffu, !ok)) goto done;  // warp converged below
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < GPS; ++j) {
            if (j >= gps) break;
            if (EPIS > 1 && j % EPIS != eset) continue;
            const float ws = wsc[j * kBM + r];
            uint64_t ws2;
            asm("mov.b64 %0, {%1, %1};" : "=l"(ws2) : "f"(ws));
            const float* ts = tsc + j * NMAX;
            const float* tc = tcr + j * NMAX;
#pragma unroll
            for (int c = 0; c < NHALF; c += CH) {
              if (c0 + c >= need) continue;  // warp-uniform
              uint32_t p[CH];
              tmem_load_cols<CH>(tmem_base + t_lane + (pslot * GPS + j) * NMAX + c0 + c, p);
              tmem_wait_ld();
#pragma unroll
              for (int q = 0; q < CH; q += 4) {
                const float4 t = *reinterpret_cast<const float4*>(ts + c0 + c + q);
                const float4 k = *reinterpret_cast<const float4*>(tc + c0 + c + q);
                promote2(acc2[(c + q) / 2], ws2, t.x, t.y, k.x, k.y, p[q], p[q + 1]);
                promote2(acc2[(c + q) / 2 + 1], ws2, t.z, t.w, k.z, k.w, p[q + 2], p[q + 3]);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&pempty[pslot]);
            mbar_arrive(&sempty[ss]);
          }
        }
        if constexpr (EPIS > 1) {
          // Set 1 hands its partial sums to set 0 through tensor memory (same lane quarter and
          // columns); slot = tile parity, guarded by xfull / xempty.
          const int xs = tile & 1;
          const uint32_t xph = (tile >> 1) & 1;
          const uint32_t xaddr = tmem_base + t_lane + CF::kXColBase + xs * NMAX + c0;
          if (eset != 0) {
            if (__any_sync(0xffffffffu, !wait_bar(&xempty[xs], xph ^ 1, s_abort))) goto done;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < NHALF; c += 8) {
              uint32_t v[8];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                asm("mov.b64 {%0, %1}, %2;" : "=r"(v[2 * q]), "=r"(v[2 * q + 1]) : "l"(acc2[c / 2 + q]));
              tmem_st8(xaddr + c, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&xfull[xs]);
            continue;
          }
          if (__any_sync(0xffffffffu, !wait_bar(&xfull[xs], xph, s_abort))) goto done;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < NHALF; c += 8) {
            uint32_t v[8];
            tmem_ld8(xaddr + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint64_t o;
              asm("mov.b64 %0, {%1, %2};" : "=l"(o) : "r"(v[2 * q]), "r"(v[2 * q + 1]));
              asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc2[c / 2 + q]) : "l"(o));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&xempty[xs]);
        }
        if (SPLIT) {  // split-K: fp32 partial sums of this split, reduced by a second kernel
          float* prow = prm.partial + (static_cast<int64_t>(item % sch.S) * prm.M + r4) * prm.N + nb * kBM + r;
#pragma unroll
          for (int q = 0; q < NHALF / 2; ++q) {
            float a0, a1;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc2[q]));
            const int t = c0 + 2 * q;
            if (t >= lo && t < lo + rows) prow[static_cast<int64_t>(t) * prm.N] = a0;
            if (t + 1 >= lo && t + 1 < lo + rows) prow[static_cast<int64_t>(t + 1) * prm.N] = a1;
          }
          continue;
        }
        uint16_t* crow = prm.C + static_cast<int64_t>(r4) * prm.N + nb * kBM + r;
#pragma unroll
        for (int q = 0; q < NHALF / 2; ++q) {
          float a0, a1;
          asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc2[q]));
          const int t = c0 + 2 * q;
          if (t >= lo && t < lo + rows) crow[static_cast<int64_t>(t) * prm.N] = float_to_bf16_bits(a0);
          if (t + 1 >= lo && t + 1 < lo + rows) crow[static_cast<int64_t>(t + 1) * prm.N] = float_to_bf16_bits(a1);
        }
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

int make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t dims[3],
                const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle sw, const char* name) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(W4A8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides[0], strides[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, dt, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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

// groups per stage: the largest power of two <= Cfg::GPS dividing K/128
template <class CF>
int stage_groups(int64_t K) {
  const int64_t G = K / kGroup;
  int gps = 1;
  while (gps * 2 <= CF::GPS && G % (gps * 2) == 0) gps *= 2;
  return gps;
}

// K splits of a dense GEMM whose tiles leave SMs idle.  A CTA takes ceil(items / SMs) items of
// ceil(stages / S) stages each, so the launch lasts about that many stage times; a split adds the
// partial-sum pass (about two stage times) and may write at most a quarter of the weight bytes in
// fp32 partials.  S = 1 .. 16 minimising that estimate, ties to the smaller S.
template <class CF>
int plan_splits(int64_t M, int64_t N, int64_t K, int sms) {
  const int64_t tiles = ceil_div(M, CF::NMAX) * (N / kBM);
  if (M <= 0 || tiles <= 0 || tiles >= sms) return 1;
  const int64_t stages = K / kGroup / stage_groups<CF>(K);
  int best = 1;
  int64_t best_cost = ceil_div(tiles, sms) * stages;
  for (int S = 2; S <= 16 && S <= stages && S * M * N * 4 <= N * K / 8; ++S) {
    const int64_t cost = ceil_div(tiles * S, sms) * ceil_div(stages, S) + 2;
    if (cost < best_cost) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

// Outputs of the fused SiLU-and-Mul requantisation (a configuration with kFuse).
struct FuseOut {
  uint16_t* gate;  // [M][N/2] bf16 scratch
  uint8_t* hq;
  float* hs;
  float* hc;
  int64_t h_ld;
};

// Upper bound on the shared-memory tile list (tiles per CTA), for tests of the in-place tile decode that
// launches too large for the list fall back to; negative: no bound.
std::atomic<int> g_tile_cap_limit{-1};

template <class CF>
int launch(const uint8_t* A, const float* a_s, const float* a_c, int64_t a_ld, const uint8_t* B, const float* b_s,
           const int64_t* seg, int64_t E, int64_t N, int64_t K, int64_t M, uint16_t* C, float* partial, int splits,
           cudaStream_t st, int min_rows = 1, int max_rows = 0x7fffffff, const FuseOut* fo = nullptr) {
  const int64_t G = K / kGroup;
  const int gps = stage_groups<CF>(K);
  CUtensorMap tA, tAS, tAC, tB, tBS;
  int rc;
  {  // tokens viewed as [group][row][128 B]: one box = gps groups x NMAX rows
    const uint64_t dims[3] = {128, static_cast<uint64_t>(M), static_cast<uint64_t>(G)};
    const uint64_t strides[2] = {static_cast<uint64_t>(K), 128};
    const uint32_t box[3] = {128, static_cast<uint32_t>(CF::NMAX), static_cast<uint32_t>(gps)};
    if ((rc = make_map_3d(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                          "A")))
      return rc;
  }
  {  // packed weights viewed as [group][row][64 B]: one box = gps groups x 128 rows
    const uint64_t dims[3] = {64, static_cast<uint64_t>(E * N), static_cast<uint64_t>(G)};
    const uint64_t strides[2] = {static_cast<uint64_t>(K / 2), 64};
    const uint32_t box[3] = {64, static_cast<uint32_t>(kBM), static_cast<uint32_t>(gps)};
    if ((rc = make_map_3d(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B,
                          "B")))
      return rc;
  }
  if ((rc = make_map_2d(&tAS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a_s, a_ld, G, a_ld * 4, CF::NMAX, gps,
                        CU_TENSOR_MAP_SWIZZLE_NONE, "a_scales")))
    return rc;
  if ((rc = make_map_2d(&tAC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a_c, a_ld, G, a_ld * 4, CF::NMAX, gps,
                        CU_TENSOR_MAP_SWIZZLE_NONE, "a_gcorr")))
    return rc;
  if ((rc = make_map_2d(&tBS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, b_s, N, E * G, N * 4, kBM, gps,
                        CU_TENSOR_MAP_SWIZZLE_NONE, "b_scales")))
    return rc;
  static DeviceOnce attrs;  // per template instance; function attributes are per device
  if (int rc2 = attrs.run([] {
        if (cudaFuncSetAttribute(w4a8_gemm_kernel<CF, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxDynSmem) != cudaSuccess ||
            cudaFuncSetAttribute(w4a8_gemm_kernel<CF, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxDynSmem) != cudaSuccess)
          return check_launch("cudaFuncSetAttribute(gemm)");
        if constexpr (CF::kRegSplit) {
          // setmaxnreg.inc waits until the released registers cover the request: the warpgroups'
          // budgets must fit in what the block is launched with, or the claim would never return.
          for (int sp = 0; sp < 2; ++sp) {
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, sp ? w4a8_gemm_kernel<CF, true> : w4a8_gemm_kernel<CF, false>) !=
                cudaSuccess)
              return check_launch("cudaFuncGetAttributes(gemm)");
            const int need = 128 * CF::kRegsCtl + 32 * CF::kConvSets * kConvWarps * CF::kRegsConv +
                             32 * CF::kEpiWarps * CF::kRegsEpi;
            if (fa.numRegs * CF::kThreads < need)
              return set_error(W4A8_ERR_UNSUPPORTED, "gemm kernel built with %d registers per thread: %d < %d",
                               fa.numRegs, fa.numRegs * CF::kThreads, need);
          }
        }
        return static_cast<int>(W4A8_OK);
      }))
    return rc2;
  GemmParams p;
  p.seg = seg;
  p.C = C;
  p.E = static_cast<int>(E);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.M = static_cast<int>(M);
  p.gps = gps;
  p.partial = partial;
  p.splits = splits;
  p.min_rows = min_rows;
  p.max_rows = max_rows;
  p.gate = fo ? fo->gate : nullptr;
  p.hq = fo ? fo->hq : nullptr;
  p.hs = fo ? fo->hs : nullptr;
  p.hc = fo ? fo->hc : nullptr;
  p.h_ld = fo ? fo->h_ld : 0;
  // tile list: an expert's chunks sit on the NMAX grid from its first row rounded down to 4, so it
  // has at most (3 + rows) / NMAX + 1 of them; tiles = chunks x 128-row blocks x K splits
  const int Ed = seg ? static_cast<int>(E) : 1;
  const int64_t chunks = seg ? (3 * E + M) / CF::NMAX + E + 1 : (M + CF::NMAX - 1) / CF::NMAX + 1;
  const int64_t per_cta = CF::kFuse ? 2 * ceil_div(chunks * (N / kBM) / 2, num_sms())
                                   : ceil_div(chunks * (N / kBM) * std::max(splits, 1), num_sms());
  const int64_t room = (kMaxDynSmem - CF::smem_bytes(Ed, 0)) / 16;
  p.tile_cap = static_cast<int>(std::max<int64_t>(0, std::min(per_cta, room)));
  const int cap_limit = g_tile_cap_limit.load();
  if (cap_limit >= 0 && p.tile_cap > cap_limit) p.tile_cap = cap_limit;
  return launch_pdl("w4a8_gemm_kernel", splits > 1 ? w4a8_gemm_kernel<CF, true> : w4a8_gemm_kernel<CF, false>,
                    dim3(num_sms()), dim3(CF::kThreads), CF::smem_bytes(Ed, p.tile_cap), st, tA, tAS,
                    tAC, tB, tBS, p);
}

// decode: few rows per expert, weight streaming; converted weights in tensor memory
using CfgDecode = Cfg<16, 4, 5, 4, 6, 2, 3, true, 2, 2, 4, 1>;
// the same with 4 MMA-issuing warps, for long K (many stages per tile): a thread stalls ~130 cycles per
// tcgen05.mma, so 2 warps issuing 8 MMAs each per stage sit near the stage period; with short K the
// extra warps cost more at the frequent tile changes than they save (grouped w13 / w2 of the decode
// layer: 0.638 -> 0.624 ms / 0.335 -> 0.342 ms)
using CfgDecodeLongK = Cfg<16, 4, 5, 4, 6, 2, 3, true, 2, 4, 4, 1>;
// prefill: 128-row token tiles, two groups per stage (the stage's fixed costs of waits and hand-overs
// paid once per two groups), so the fp32 partials of 2 slots x 2 groups fill the tensor memory and the
// converted weights go to shared memory (prefill w13 4.378 -> 4.320 ms, w2 2.589 -> 2.504 ms against
// one group per stage with the weights in tensor memory)
using CfgPrefill = Cfg<128, 2, 4, 2, 4, 2, 2, false, 2, 2, 8, 1>;
// the same with the SiLU-and-Mul requantisation fused into the epilogue (w13); one weight stage fewer
// leaves shared memory for the staged codes
using CfgPrefillSilu = Cfg<128, 2, 3, 2, 4, 2, 2, false, 2, 2, 8, 1, true>;

// C[m][n] = bf16(sum over s of partial[s][m][n]), four columns per thread.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ partial,
                                                            uint16_t* __restrict__ C, int64_t MN, int S) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * 4; i < MN;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x * 4) {
    float4 acc = *reinterpret_cast<const float4*>(partial + i);
    for (int s = 1; s < S; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(partial + s * MN + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    uint2 o;
    o.x = static_cast<uint32_t>(float_to_bf16_bits(acc.x)) | (static_cast<uint32_t>(float_to_bf16_bits(acc.y)) << 16);
    o.y = static_cast<uint32_t>(float_to_bf16_bits(acc.z)) | (static_cast<uint32_t>(float_to_bf16_bits(acc.w)) << 16);
    *reinterpret_cast<uint2*>(C + i) = o;
  }
}

// Tile-cost model of the two token-tile widths of the grouped GEMM, the per-expert expected-cost
// choice of the DeepGEMM PR #53 page (Conversation, the cost-model commit: a tile width's cost is
// a * R + b * T with T the tiles and R the rows they pad to, taken in expectation over Poisson row
// counts), restated for these kernels.  Units: one 16-wide tile's time at the same N and K (weight
// streaming dominates it).  A 128-wide tile converts the same weights and promotes up to eight times
// the columns.  cost_W(x) = b_W * T_W(x) + a_W * R_W(x), T_W = ceil(x / W), R_W = rows padded to
// 16 within each tile; fitted to GB300 sweeps of 256 experts with x rows each at (N, K) = (4096,
// 7168) and (7168, 2048), x = 1 ... 256, to within ~10 %: narrow a = 0, b = 1; wide a = 0.004, b = 2.
struct TileCost {
  double a, b;
  int width;
};
constexpr TileCost kNarrowCost{0.0, 1.0, 16};
constexpr TileCost kWideCost{0.004, 2.0, 128};
// The start-up of one more launch (~15 us of the whole GPU) in 16-wide tile times per weight block of
// all E experts: a 16-wide tile takes ~1.8 ns per K on one SM.
double launch_cost_tiles(int64_t E, int64_t K, int sms) {
  const double tile_us = 1.8e-3 * static_cast<double>(K);
  return 15.0 * sms / tile_us / static_cast<double>(E);
}

double tile_cost(int wide, int64_t x) {
  const TileCost& c = wide ? kWideCost : kNarrowCost;
  if (x <= 0) return 0.0;
  const int64_t full = x / c.width, rem = x - full * c.width;
  const int64_t T = full + (rem > 0 ? 1 : 0);
  const int64_t R = full * c.width + (rem + 15) / 16 * 16;
  return c.b * static_cast<double>(T) + c.a * static_cast<double>(R);
}

// The largest row count of one expert for which the narrow tiles cost no more than the wide ones.
int crossover_rows() {
  int x = 1;
  while (x <= 128 && tile_cost(0, x) <= tile_cost(1, x)) ++x;
  return x - 1;
}

// E[cost_W(X) ; lo <= X <= hi] for X ~ Poisson(lambda), summed until the tail is negligible.
double expected_cost(int wide, double lambda, int64_t lo, int64_t hi) {
  if (lambda <= 0.0) return 0.0;
  const int64_t top = static_cast<int64_t>(lambda + 12.0 * std::sqrt(lambda) + 40.0);
  double sum = 0.0, logp = -lambda;  // log P(X = 0)
  for (int64_t x = 1; x <= top && x <= hi; ++x) {
    logp += std::log(lambda) - std::log(static_cast<double>(x));
    if (x >= lo) sum += std::exp(logp) * tile_cost(wide, x);
  }
  return sum;
}

constexpr int kPlanNarrow = 1, kPlanWide = 2, kPlanSplit = 3;

// Launch plan of a grouped GEMM from what the host knows (M rows over E experts, K): the expected
// cost per expert of each plan under Poisson(M / E) row counts, plus one launch start-up for the
// split plan (narrow tiles for experts with at most theta rows, wide ones for the rest, in two
// launches; the device applies the threshold to the realised row counts).  Poisson counts describe
// balanced routing only; when the mean lies between the crossover and the wide tile (theta * E < M <
// 128 * E), a skewed batch has experts on both sides, so the split plan is kept there: it costs at
// most one start-up more than the Poisson optimum (skewed layer 4.13 -> 3.81 ms).
int plan_grouped(int64_t M, int64_t E, int64_t K, int* theta_out) {
  const int theta = crossover_rows();
  if (theta_out) *theta_out = theta;
  const double lambda = static_cast<double>(M) / static_cast<double>(E);
  const double inf = 1e18;
  const double narrow = expected_cost(0, lambda, 1, static_cast<int64_t>(inf));
  const double wide = expected_cost(1, lambda, 1, static_cast<int64_t>(inf));
  const double split = expected_cost(0, lambda, 1, theta) + expected_cost(1, lambda, theta + 1, static_cast<int64_t>(inf)) +
                       launch_cost_tiles(E, K, num_sms());
  int best = narrow <= wide ? kPlanNarrow : kPlanWide;
  if (split < std::min(narrow, wide)) best = kPlanSplit;
  if (best != kPlanSplit && M > static_cast<int64_t>(theta) * E && M < 128 * E) best = kPlanSplit;
  return best;
}

// K splits the dense Linear uses for this shape on the current device (1: none).
int linear_splits(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || N % kBM || K % kGroup) return 1;
  return M <= 32 ? plan_splits<CfgDecode>(M, N, K, num_sms()) : plan_splits<CfgPrefill>(M, N, K, num_sms());
}

int gemm_common(const uint8_t* A, const float* a_s, const float* a_c, int64_t a_ld, const uint8_t* B, const float* b_s,
                const int64_t* seg, int64_t E, int64_t N, int64_t K, int64_t M, uint16_t* C, void* ws,
                size_t ws_bytes, void* stream) {
  W4A8_REQUIRE(K > 0 && K % kGroup == 0, "K=%lld must be a positive multiple of 128", (long long)K);
  W4A8_REQUIRE(N > 0 && N % kBM == 0, "N=%lld must be a positive multiple of 128", (long long)N);
  W4A8_REQUIRE(M >= 0 && M < (1ll << 31), "M=%lld out of range", (long long)M);
  W4A8_REQUIRE(E >= 1 && E <= kMaxExperts, "E=%lld must be in [1, 1024]", (long long)E);
  W4A8_REQUIRE(E * N < (1ll << 31) && K < (1ll << 31), "E*N or K too large");
  W4A8_REQUIRE(a_ld >= M && a_ld % 4 == 0 && a_ld > 0, "a_scale_ld=%lld must be >= M and a multiple of 4",
               (long long)a_ld);
  W4A8_REQUIRE(A && a_s && B && b_s && C, "null pointer");
  W4A8_REQUIRE(aligned16(A) && aligned16(a_s) && aligned16(a_c) && aligned16(B) && aligned16(b_s) && aligned16(C),
               "device pointers must be 16-byte aligned");
  if (M == 0) return W4A8_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // split-K only for the dense GEMM: the grouped GEMM's tile count depends on device-side seg_indptr
  const int S = seg ? 1 : linear_splits(M, N, K);
  // workspace: [split-K partial sums][corrections, when the caller passes none]
  const size_t part_bytes = S > 1 ? static_cast<size_t>(S) * M * N * sizeof(float) : 0;
  const size_t corr_off = (part_bytes + 255) & ~size_t(255);
  const size_t need = a_c ? part_bytes : corr_off + static_cast<size_t>(K / kGroup) * a_ld * sizeof(float);
  W4A8_REQUIRE(need == 0 || (ws != nullptr && ws_bytes >= need && aligned16(ws)),
               "workspace of %zu bytes (16-byte aligned) required for this call, got %zu", need, ws_bytes);
  float* partial = S > 1 ? static_cast<float*>(ws) : nullptr;
  int rc;
  if (!a_c) {  // the activation corrections from the codes, as the quantisation kernels compute them
    float* corr = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + corr_off);
    if ((rc = launch_gcorr(A, M, K, a_s, a_ld, corr, st))) return rc;
    a_c = corr;
  }
  // The dense Linear: 16-wide token tiles (weight streaming) up to 32 rows, 128-wide above.  The grouped
  // GEMM: the cost-model plan (narrow, wide, or both over disjoint experts split at theta rows).
  int theta = 0;
  const int plan = seg ? plan_grouped(M, E, K, &theta) : (M <= 32 ? kPlanNarrow : kPlanWide);
  const int narrow_max = plan == kPlanSplit ? theta : 0x7fffffff;
  if (plan != kPlanWide) {
    rc = K >= 4096 && seg ? launch<CfgDecodeLongK>(A, a_s, a_c, a_ld, B, b_s, seg, E, N, K, M, C, partial, S, st, 1,
                                                   narrow_max)
                          : launch<CfgDecode>(A, a_s, a_c, a_ld, B, b_s, seg, E, N, K, M, C, partial, S, st, 1,
                                              narrow_max);
    if (rc != W4A8_OK) return rc;
  }
  if (plan != kPlanNarrow)
    rc = launch<CfgPrefill>(A, a_s, a_c, a_ld, B, b_s, seg, E, N, K, M, C, partial, S, st,
                            plan == kPlanSplit ? theta + 1 : 1);
  if (rc != W4A8_OK || S == 1) return rc;
  const int64_t MN = M * N;  // N % 128 == 0, so MN % 4 == 0
  const int64_t blocks = ceil_div(MN / 4, 256) < 8 * 152 ? ceil_div(MN / 4, 256) : 8 * 152;
  return launch_pdl("splitk_reduce_kernel", splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                    st, static_cast<const float*>(partial), C, MN, S);
}

// The w13 GEMM followed by SiLU-and-Mul with FP8 requantisation.  When the plan takes the wide tiles only
// (and a tile has at least two stages), the requantisation runs in the GEMM's epilogue and Y13 is never
// written (the gate half passes through the workspace as bf16, read back by the threads that wrote it);
// otherwise the GEMM writes Y13 [M][2I] into the workspace and the SiLU-and-Mul kernel reads it.  Both give
// the same bits: the fused epilogue rounds gate and up to bf16 and uses the kernel's arithmetic.
int gemm_silu(const uint8_t* A, const float* a_s, const float* a_c, int64_t a_ld, const uint8_t* B,
              const float* b_s, const int64_t* seg, int64_t E, int64_t I, int64_t K, int64_t M, uint8_t* q, float* hs,
              float* hc, int64_t h_ld, void* ws, size_t ws_bytes, void* stream, bool allow_fuse) {
  W4A8_REQUIRE(seg != nullptr, "seg_indptr is null");
  W4A8_REQUIRE(I > 0 && I % kGroup == 0, "I=%lld must be a positive multiple of 128", (long long)I);
  W4A8_REQUIRE(K > 0 && K % kGroup == 0, "K=%lld must be a positive multiple of 128", (long long)K);
  W4A8_REQUIRE(M >= 0 && M < (1ll << 31), "M=%lld out of range", (long long)M);
  W4A8_REQUIRE(h_ld >= M && h_ld % 4 == 0 && h_ld > 0, "h_scale_ld=%lld must be >= M and a multiple of 4",
               (long long)h_ld);
  W4A8_REQUIRE(a_ld >= M && a_ld % 4 == 0 && a_ld > 0, "a_scale_ld=%lld must be >= M and a multiple of 4",
               (long long)a_ld);
  W4A8_REQUIRE(q && hs, "null pointer");
  W4A8_REQUIRE(aligned16(q) && (reinterpret_cast<uintptr_t>(hs) & 3) == 0 && (reinterpret_cast<uintptr_t>(hc) & 3) == 0,
               "q must be 16-byte, h_scales and h_gcorr 4-byte aligned");
  const size_t y_bytes = (static_cast<size_t>(M) * 2 * I * 2 + 255) & ~size_t(255);
  const size_t need = y_bytes + (a_c ? 0 : static_cast<size_t>(K / kGroup) * a_ld * sizeof(float));
  W4A8_REQUIRE(ws != nullptr && ws_bytes >= need && aligned16(ws),
               "workspace of %zu bytes (16-byte aligned) required for this call, got %zu", need, ws_bytes);
  if (M == 0) return W4A8_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc;
  if (!a_c) {
    float* corr = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + y_bytes);
    if ((rc = launch_gcorr(A, M, K, a_s, a_ld, corr, st))) return rc;
    a_c = corr;
  }
  int theta = 0;
  const int64_t G = K / kGroup;
  if (allow_fuse && plan_grouped(M, E, K, &theta) == kPlanWide && G / stage_groups<CfgPrefillSilu>(K) >= 2) {
    W4A8_REQUIRE(E >= 1 && E <= kMaxExperts && E * 2 * I < (1ll << 31), "E=%lld out of range", (long long)E);
    W4A8_REQUIRE(A && a_s && B && b_s && aligned16(A) && aligned16(a_s) && aligned16(a_c) && aligned16(B) &&
                     aligned16(b_s),
                 "GEMM operands must be non-null and 16-byte aligned");
    const FuseOut fo{static_cast<uint16_t*>(ws), q, hs, hc, h_ld};
    return launch<CfgPrefillSilu>(A, a_s, a_c, a_ld, B, b_s, seg, E, 2 * I, K, M, nullptr, nullptr, 1, st, 1,
                                  0x7fffffff, &fo);
  }
  uint16_t* y13 = static_cast<uint16_t*>(ws);
  if ((rc = gemm_common(A, a_s, a_c, a_ld, B, b_s, seg, E, 2 * I, K, M, y13, nullptr, 0, stream))) return rc;
  return silu_mul_requant(y13, M, I, q, hs, hc, h_ld, stream);
}

}  // namespace

size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int S = linear_splits(M, N, K);
  return S > 1 ? static_cast<size_t>(S) * M * N * sizeof(float) : 0;
}

size_t gemm_silu_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || K <= 0 || K % kGroup) return 0;
  return ((static_cast<size_t>(M) * N * 2 + 255) & ~size_t(255)) + gemm_workspace_bytes(M, N, K, false);
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, bool dense) {
  if (M <= 0 || K <= 0 || K % kGroup) return 0;
  const size_t part = dense ? linear_workspace_bytes(M, N, K) : 0;
  const int64_t ld = (M + 3) / 4 * 4;
  return ((part + 255) & ~size_t(255)) + static_cast<size_t>(K / kGroup) * ld * sizeof(float);
}

}  // namespace w4a8

extern "C" int w4a8_grouped_gemm(const uint8_t* A, const float* a_scales, const float* a_gcorr, int64_t a_scale_ld,
                                 const uint8_t* B_prepacked, const float* b_scales, const int64_t* seg_indptr,
                                 int64_t E, int64_t N, int64_t K, int64_t M_total, uint16_t* C, void* ws,
                                 size_t ws_bytes, void* stream) {
  W4A8_REQUIRE(seg_indptr != nullptr, "seg_indptr is null");
  return w4a8::gemm_common(A, a_scales, a_gcorr, a_scale_ld, B_prepacked, b_scales, seg_indptr, E, N, K, M_total, C,
                           ws, ws_bytes, stream);
}

extern "C" int w4a8_grouped_gemm_silu(const uint8_t* A, const float* a_scales, const float* a_gcorr,
                                      int64_t a_scale_ld, const uint8_t* B_prepacked, const float* b_scales,
                                      const int64_t* seg_indptr, int64_t E, int64_t I, int64_t K, int64_t M_total,
                                      uint8_t* q, float* h_scales, float* h_gcorr, int64_t h_scale_ld, void* ws,
                                      size_t ws_bytes, void* stream) {
  return w4a8::gemm_silu(A, a_scales, a_gcorr, a_scale_ld, B_prepacked, b_scales, seg_indptr, E, I, K, M_total, q,
                         h_scales, h_gcorr, h_scale_ld, ws, ws_bytes, stream, true);
}

// The same entry point with the fusion switched off (the GEMM then the SiLU-and-Mul kernel): for tests.
extern "C" int w4a8_grouped_gemm_silu_unfused(const uint8_t* A, const float* a_scales, const float* a_gcorr,
                                              int64_t a_scale_ld, const uint8_t* B_prepacked, const float* b_scales,
                                              const int64_t* seg_indptr, int64_t E, int64_t I, int64_t K,
                                              int64_t M_total, uint8_t* q, float* h_scales, float* h_gcorr,
                                              int64_t h_scale_ld, void* ws, size_t ws_bytes, void* stream) {
  return w4a8::gemm_silu(A, a_scales, a_gcorr, a_scale_ld, B_prepacked, b_scales, seg_indptr, E, I, K, M_total, q,
                         h_scales, h_gcorr, h_scale_ld, ws, ws_bytes, stream, false);
}

extern "C" int w4a8_linear(const uint8_t* A, const float* a_scales, const float* a_gcorr, int64_t a_scale_ld,
                           const uint8_t* B_prepacked, const float* b_scales, int64_t M, int64_t N, int64_t K,
                           uint16_t* C, void* ws, size_t ws_bytes, void* stream) {
  return w4a8::gemm_common(A, a_scales, a_gcorr, a_scale_ld, B_prepacked, b_scales, nullptr, 1, N, K, M, C, ws,
                           ws_bytes, stream);
}

extern "C" int w4a8_linear_split_k(int64_t M, int64_t N, int64_t K) { return w4a8::linear_splits(M, N, K); }

extern "C" int w4a8_test_tile_list_limit(int max_tiles) {
  w4a8::g_tile_cap_limit.store(max_tiles < 0 ? -1 : max_tiles);
  return W4A8_OK;
}

extern "C" int w4a8_test_wait_timeout(uint64_t limit_ns, int* gave_up, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(gave_up != nullptr && (reinterpret_cast<uintptr_t>(gave_up) & 3) == 0, "gave_up must be an int");
  W4A8_REQUIRE(limit_ns > 0 && limit_ns <= kTimeoutNs, "limit_ns must be in (0, 2e9]");
  wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, gave_up);
  return check_launch("wait_timeout_probe_kernel");
}

extern "C" double w4a8_tile_cost(int wide, int64_t rows) { return w4a8::tile_cost(wide, rows); }

extern "C" double w4a8_expected_tile_cost(int wide, double mean_rows) {
  return w4a8::expected_cost(wide, mean_rows, 1, 1ll << 40);
}

extern "C" int w4a8_grouped_gemm_plan(int64_t M_total, int64_t E, int64_t K, int* theta) {
  if (M_total <= 0 || E < 1 || K <= 0) return 0;
  return w4a8::plan_grouped(M_total, E, K, theta);
}

extern "C" int w4a8_prepack_weights(const uint8_t* w, int64_t rows, int64_t K, uint8_t* out, void* stream) {
  using namespace w4a8;
  W4A8_REQUIRE(rows >= 0 && K > 0 && K % 8 == 0, "K=%lld must be a positive multiple of 8", (long long)K);
  if (rows == 0) return W4A8_OK;
  W4A8_REQUIRE(w && out, "null pointer");
  W4A8_REQUIRE(((uintptr_t)w & 3) == 0 && ((uintptr_t)out & 3) == 0, "w and out must be 4-byte aligned");
  const int64_t n_words = rows * (K / 8);
  const int64_t blocks = ceil_div(n_words, 256) < 4 * 1184 ? ceil_div(n_words, 256) : 4 * 1184;
  prepack_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint32_t*>(w), reinterpret_cast<uint32_t*>(out), n_words);
  return check_launch("prepack_kernel");
}
