// Persistent tcgen05 GEMMs for sm_103a with the epilogues of fused linear
// cross-entropy.
//
// The three contractions of the FLCE pages' per-chunk schedule ("Fused Linear
// Cross-Entropy: LLM 학습 logits 메모리 병목 없애기", section "FLCE의 핵심
// 아이디어": projection x_c·Wᵀ, dx = dlogits·W, dW += dlogitsᵀ·x_c) run on two
// kernel templates that share their epilogue:
//
//   umma_gemm_kernel   one CTA per SM, 128 x 256 output tiles, 4-stage ring
//                      of 48 KB (A 128x64, B 256x64), tcgen05 cta_group::1
//   umma_pair_kernel   a cluster of two CTAs on two SMs computes a 256 x 256
//                      tile with tcgen05 cta_group::2: each CTA holds its 128
//                      rows of A and its 128 columns of B (6-stage ring of
//                      32 KB), the even CTA issues the MMAs for both, and
//                      each CTA's TMEM receives its 128 rows of the result
//
// Warp roles (both kernels): warp 0 TMA producer; warp 1 allocates 512 TMEM
// columns and (one thread) issues the MMAs into one of two 256-column
// accumulators, so the epilogue of tile i overlaps the main loop of tile i+1;
// warps 2..5 epilogue: tcgen05.ld the accumulator (one token row per thread),
// transform, stage 16 KB sub-tiles in 128-byte-swizzled shared memory and
// write them out with TMA stores.
//
// The logits epilogue (kEpiLse) is the on-chip softmax statistics of the
// Unsloth page ("Unsloth 심층 아키텍처 …", section "스트리밍 청크 기반 Fast
// CrossEntropy 손실 커널"): per token row and 256-wide vocab tile it takes
// the max m and l = sum exp(z - m) from the fp32 accumulator (two passes over
// TMEM), picks up the target logit, and optionally stores the tile as bf16
// logits shifted by m. The row's tiles are combined later by the log-sum-exp
// combine, the online-softmax step across tiles.
//
// Every mbarrier wait is bounded (timeout in UmmaArgs). A wait that runs out
// records FLCE_ERR_TIMEOUT in the control block; the CTA then waits (bounded)
// for its own TMA loads and MMAs in flight, frees its TMEM and returns.
#include <cuda_bf16.h>

#include "flce_internal.h"
#include "ptx.cuh"

namespace flce {
namespace {

constexpr uint32_t kABytes = kBM * kBK * 2;                // 16 KB: 128 rows of A
constexpr uint32_t kBBytes = kBN * kBK * 2;                // 32 KB: 256 columns of B
constexpr uint32_t kBHalfBytes = kBBytes / 2;              // 16 KB: 128 columns of B
constexpr int kStages = 4;                                 // single-CTA ring
#ifndef FLCE_PAIR_STAGES
#define FLCE_PAIR_STAGES 6
#endif
constexpr int kStagesPair = FLCE_PAIR_STAGES;              // CTA-pair ring
constexpr uint32_t kStageBytes = kABytes + kBBytes;        // 48 KB
constexpr uint32_t kStageBytesPair = kABytes + kBHalfBytes;  // 32 KB per CTA
constexpr uint32_t kEpiBytes = 128 * 128;                  // 128 rows x 128 bytes
constexpr uint32_t kSmemBytes =
    1024 + kStages * kStageBytes + 2 * kEpiBytes + (2 * kStages + 5) * 8 + 16;
constexpr uint32_t kSmemBytesPair =
    1024 + kStagesPair * kStageBytesPair + 2 * kEpiBytes + (2 * kStagesPair + 5) * 8 + 16;
// wide CTA-pair tiles: 256 x 512, each CTA holding 128 rows of A and 256
// columns of B per k-block
#ifndef FLCE_WIDE_STAGES
#define FLCE_WIDE_STAGES 4
#endif
#ifndef FLCE_WIDE_EPI_BUFS
#define FLCE_WIDE_EPI_BUFS 1
#endif
constexpr int kStagesWide = FLCE_WIDE_STAGES;
constexpr int kEpiBufsWide = FLCE_WIDE_EPI_BUFS;            // staging buffers per epilogue
constexpr uint32_t kStageBytesWide = kABytes + kBBytes;    // 48 KB per CTA
constexpr uint32_t kSmemBytesWide = 1024 + kStagesWide * kStageBytesWide +
                                    2 * kEpiBufsWide * kEpiBytes + (2 * kStagesWide + 4) * 8 + 16;
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 192;
// wide tiles: warpgroup 0 (TMA producer warp, MMA warp, two idle warps) and
// two epilogue warpgroups; registers move from warpgroup 0 to the epilogues
// (setmaxnreg), whose log-sum-exp pass keeps a row's 256 columns of bf16 in
// registers. The split must fit the launch: 384 threads x kWideLaunchRegs.
constexpr int kThreadsWide = 384;
constexpr uint32_t kWideRegsCtl = 56;    // warpgroup 0
constexpr uint32_t kWideRegsEpi = 224;   // each epilogue warpgroup
constexpr int kWideLaunchRegs = 168;     // what __launch_bounds__(384, 1) leaves a thread
static_assert(128 * kWideRegsCtl + 256 * kWideRegsEpi <= kThreadsWide * kWideLaunchRegs,
              "register split of the wide kernel");
constexpr int kEpiThreads = 128;
constexpr uint32_t kEpiBar = 1;
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kSmemBytes <= 232448 && kSmemBytesPair <= 232448 && kSmemBytesWide <= 232448,
              "shared memory per CTA");

struct Unit {
  int m, n, s;
};

__device__ __forceinline__ Unit unit_coords(const UmmaArgs& a, int u) {
  Unit r;
  const int mn = a.num_m * a.num_n;
  r.s = u / mn;
  const int w = u - r.s * mn;
  if (a.raster == 0) {
    r.m = w % a.num_m;
    r.n = w / a.num_m;
  } else if (a.raster == 2) {
    // a group of group_m tile rows (fewer in the last group) sweeps all the
    // columns, its rows fastest: consecutive units share both operands
    const int per = a.group_m * a.num_n;
    const int g = w / per;
    const int idx = w - g * per;
    const int rows = min(a.group_m, a.num_m - g * a.group_m);
    r.m = g * a.group_m + idx % rows;
    r.n = idx / rows;
  } else {
    r.n = w % a.num_n;
    r.m = w / a.num_n;
  }
  return r;
}

// wait bounded by time only (used while draining after an error)
__device__ __forceinline__ void mbar_drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Row r of a 128-row x 128-byte staging tile, in the 128-byte swizzle that
// the TMA store expects: 16-byte chunk j of row r sits at chunk j ^ (r % 8).
__device__ __forceinline__ void stage_row(uint8_t* buf, int r, const uint32_t (&w)[32]) {
  uint4* rowp = reinterpret_cast<uint4*>(buf + r * 128);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    rowp[j ^ (r & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// The epilogue of one 128-row x 256-column accumulator tile. Runs on the 128
// epilogue threads; thread `row` owns one tile row. `release` is called right
// after the last tcgen05.ld of the tile, handing the accumulator back to the
// MMA issuer.
// NBUF staging buffers of kEpiBytes at sE (2: alternate, 1: reuse one), and
// the named barrier `bar` over this epilogue's 128 threads.
template <int EPI, int NBUF = 2, class Release>
__device__ __forceinline__ void epilogue_tile(const UmmaArgs& a, const CUtensorMap* tmO, uint8_t* sE,
                                              uint32_t& ebuf, int row, bool leader, int m0, int n0,
                                              int s_idx, uint32_t tbase,
                                              Release&& release, uint32_t bar = kEpiBar) {
  static_assert(NBUF == 1 || NBUF == 2, "staging buffers");
  if (n0 >= a.cols) {  // a tile past the last column (uniform): nothing to read
    release();
    return;
  }
  const int grow = m0 + row;
  const bool rvalid = grow < a.rows;

  // stage one 16 KB sub-tile and hand it to the TMA unit
  auto stage_and_store = [&](const uint32_t (&w)[32], auto&& issue) {
    uint8_t* buf = sE + ebuf * kEpiBytes;
    if (leader) bulk_wait_group_read<NBUF - 1>();
    named_bar_sync(bar, kEpiThreads);
    stage_row(buf, row, w);
    fence_proxy_async_smem();
    named_bar_sync(bar, kEpiThreads);
    if (leader) {
      issue(smem_u32(buf));
      bulk_commit_group();
    }
    __syncwarp();
    if (NBUF == 2) ebuf ^= 1u;
  };

  if constexpr (EPI == kEpiLse) {
    // One pass over the accumulator, then the arithmetic. Per 64-column group
    // g: read the group from TMEM, take its row max m_g (and the target logit
    // when it falls in the group), and keep y = z - m_g packed as bf16 in
    // registers. Once the last group is read the accumulator goes back to the
    // MMA issuer; only then come the exponentials (the MUFU-bound part:
    // 16 per clock per SM), s_g = sum of exp(y) over the packed values, and
    // the stores of y. The partial of group g is (m_g, s_g). Stored relative
    // to its group's max, every group's largest entries sit near 0, where
    // bf16 is most precise; the dlogits pass adds m_g back from the partial,
    // and since s_g sums the same bf16 values that pass exponentiates, the
    // softmax it forms sums to one over the row. Columns past the output's
    // last (a ragged vocabulary) enter as -inf: they add nothing.
    constexpr int kGroups = kBN / 64;
    int64_t tg = -1;
    if (rvalid) tg = a.targets[grow];
    const int64_t tl = (rvalid && tg != a.ignore_index) ? tg - a.col_base : -1;
    const int tcol = (tl >= n0 && tl < n0 + kBN) ? static_cast<int>(tl - n0) : -1;
    const int last_g = min(kGroups - 1, (a.cols - n0 - 1) / 64);  // uniform, >= 0
    uint32_t y[kGroups][32];
    float mg[kGroups];
    float zt = 0.f;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      if (g > last_g) break;  // uniform across the epilogue threads
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(tbase + g * 64, r0);
      tmem_ld_32x32b_x32(tbase + g * 64 + 32, r1);
      tmem_ld_wait();
      tmem_regs_ready(r0);
      tmem_regs_ready(r1);
      if (g == last_g) release();
      const int ncv = a.cols - (n0 + g * 64);  // valid columns in the group (uniform)
      if (ncv < 64) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i >= ncv) r0[i] = 0xFF800000u;  // -inf
          if (i + 32 >= ncv) r1[i] = 0xFF800000u;
        }
      }
      float m8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m8[j] = fmaxf(__uint_as_float(r0[j]), __uint_as_float(r1[j]));
#pragma unroll
      for (int i = 8; i < 32; ++i) {
        m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(r0[i]));
        m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(r1[i]));
      }
      const float m = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                            fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      if (tcol >= g * 64 && tcol < g * 64 + 64) {
        const int k = tcol - g * 64;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i == k) zt = __uint_as_float(r0[i]);
          if (i + 32 == k) zt = __uint_as_float(r1[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        y[g][i] = pack_bf16x2(__uint_as_float(r0[2 * i]) - m, __uint_as_float(r0[2 * i + 1]) - m);
        y[g][16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]) - m, __uint_as_float(r1[2 * i + 1]) - m);
      }
      mg[g] = m;
    }
    // the accumulator is free: sums of exp and stores
    const size_t prow = static_cast<size_t>(grow) * a.vocab_tiles + static_cast<size_t>(n0 / 64);
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      if (g > last_g) break;
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s4[i & 3] += ex2_approx(__uint_as_float(y[g][i] << 16) * kLog2e);
        s4[(i + 2) & 3] += ex2_approx(__uint_as_float(y[g][i] & 0xFFFF0000u) * kLog2e);
      }
      if (rvalid) a.partials[prow + g] = make_float2(mg[g], (s4[0] + s4[1]) + (s4[2] + s4[3]));
      if (a.store_logits) {
        const int c0 = n0 + g * 64;
        stage_and_store(y[g], [&](uint32_t src) { tma_store_2d(tmO, src, c0, m0); });
      }
    }
    if (rvalid && tcol >= 0) a.zt[grow] = zt;
  } else if constexpr (EPI == kEpiDlogits) {
    // d = (exp(z - lse) - onehot) * scale, one pass over the accumulator; the
    // fp32 rounding error of the target entry goes to dcorr for the dx
    // reduction
    int64_t tg = -1;
    if (rvalid) tg = a.targets[grow];
    const bool tvalid = rvalid && tg != a.ignore_index;
    const int64_t tl = tg - a.col_base;  // target column in this GEMM's output
    const int tcol = (tvalid && tl >= n0 && tl < n0 + kBN) ? static_cast<int>(tl - n0) : -1;
    const uint32_t nv = a.ctrl[kCtrlNValid];
    const float scale = (tvalid && nv > 0) ? 1.0f / static_cast<float>(nv) : 0.f;
    const float lse_l2 = rvalid ? a.lse[grow] * kLog2e : 0.f;
    // last 64-column group holding valid columns (uniform)
    const int last_g = min(kBN / 64 - 1, (a.cols - n0 - 1) / 64);
#pragma unroll 1
    for (int g = 0; g <= last_g; ++g) {
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(tbase + g * 64, r0);
      tmem_ld_32x32b_x32(tbase + g * 64 + 32, r1);
      tmem_ld_wait();
      tmem_regs_ready(r0);
      tmem_regs_ready(r1);
      if (g == last_g) release();
      const int c0 = n0 + g * 64;
      const int k = (tcol >= g * 64 && tcol < g * 64 + 64) ? tcol - g * 64 : -1;
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float v[4] = {__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]),
                      __uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1])};
        const int ci[4] = {2 * i, 2 * i + 1, 32 + 2 * i, 33 + 2 * i};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float p = ex2_approx(fmaf(v[q], kLog2e, -lse_l2));
          if (ci[q] == k) p -= 1.0f;
          v[q] = p * scale;
        }
        w[i] = pack_bf16x2(v[0], v[1]);
        w[16 + i] = pack_bf16x2(v[2], v[3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (ci[q] == k) {
            const uint32_t word = q < 2 ? w[i] : w[16 + i];
            const uint32_t bits = (q & 1) ? (word >> 16) : (word & 0xFFFFu);
            a.dcorr[grow] = v[q] - __uint_as_float(bits << 16);
          }
        }
      }
      stage_and_store(w, [&](uint32_t src) { tma_store_2d(tmO, src, c0, m0); });
    }
  } else if constexpr (EPI == kEpiBf16) {
#pragma unroll 1
    for (int g = 0; g < kBN / 64; ++g) {
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(tbase + g * 64, r0);
      tmem_ld_32x32b_x32(tbase + g * 64 + 32, r1);
      tmem_ld_wait();
      if (g == kBN / 64 - 1) release();
      const int c0 = n0 + g * 64;
      if (c0 >= a.cols) continue;
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        w[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
        w[16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
      }
      stage_and_store(w, [&](uint32_t src) { tma_store_2d(tmO, src, c0, m0); });
    }
  } else {  // kEpiF32
    // The TMEM reads run kAhead 32-column groups ahead of the stores, in
    // registers. The stores are paced by the TMA unit draining the staging
    // buffer, so the accumulator goes back to the MMA issuer after
    // kG - kAhead store rounds rather than kG - 1, and the last rounds' stores
    // overlap the next tile's MMAs.
    constexpr int kG = kBN / 32;
    constexpr int kAhead = 6;   // 192 registers of look-ahead: the wide kernel's
                                // epilogue warpgroups hold 224 (setmaxnreg)
    static_assert(kAhead <= kG, "look-ahead");
    uint32_t r[kAhead][32];
#pragma unroll
    for (int g = 0; g < kAhead; ++g) tmem_ld_32x32b_x32(tbase + g * 32, r[g]);
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      uint32_t (&cur)[32] = r[g % kAhead];
      tmem_ld_wait();
      tmem_regs_ready(cur);
      if (g == kG - kAhead) release();  // every column of the tile is in registers
      const int c0 = n0 + g * 32;
      if (c0 < a.cols) {  // uniform across the epilogue threads
        if (a.reduce_add)
          stage_and_store(cur, [&](uint32_t src) { tma_reduce_add_3d(tmO, src, c0, m0, s_idx); });
        else
          stage_and_store(cur, [&](uint32_t src) { tma_store_3d(tmO, src, c0, m0, s_idx); });
      }
      if (g + kAhead < kG) tmem_ld_32x32b_x32(tbase + (g + kAhead) * 32, cur);
    }
  }
}

// The log-sum-exp epilogue of a wide tile (256 x 512 on the pair, 128 rows x
// 512 columns of TMEM per CTA), for one of its two epilogue warpgroups (grp):
// the warpgroup reads its 64-column groups of the accumulator's first half
// (columns grp*128 .. grp*128+127) and hands that half back (release0), then
// its groups of the second half (256 + grp*128 ..) and hands that back
// (release1). With both warpgroups done with the first half, the MMA issuer
// starts the next tile's first-half MMAs while the second half is still
// being read. The arithmetic per group is that of epilogue_tile<kEpiLse>:
// max m_g, the target logit, y = z - m_g packed as bf16 in registers; the
// sums of exp and the stores of y follow the second release. tbase is the
// accumulator's column 0 at this thread's TMEM lane; n0 the tile's first
// output column.
template <class Release0, class Release1>
__device__ __forceinline__ void epilogue_lse_wide(const UmmaArgs& a, const CUtensorMap* tmO, uint8_t* sE,
                                                  uint32_t& ebuf, int row, bool leader, int m0, int n0,
                                                  int grp, uint32_t tbase, Release0&& release0,
                                                  Release1&& release1, uint32_t bar) {
  constexpr int kGroups = 4;
  const int grow = m0 + row;
  const bool rvalid = grow < a.rows;
  int64_t tg = -1;
  if (rvalid) tg = a.targets[grow];
  const int64_t tl = (rvalid && tg != a.ignore_index) ? tg - a.col_base : -1;
  // tile column of group q: two groups in each half
  auto col_of = [&](int q) { return (q < 2 ? 0 : kBN) + grp * 128 + (q & 1) * 64; };
  uint32_t y[kGroups][32];
  float mg[kGroups];
  float zt = 0.f;
  bool zt_here = false;
#pragma unroll
  for (int q = 0; q < kGroups; ++q) {
    const int c = n0 + col_of(q);  // output column of the group's first entry (uniform)
    if (c < a.cols) {
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(tbase + col_of(q), r0);
      tmem_ld_32x32b_x32(tbase + col_of(q) + 32, r1);
      tmem_ld_wait();
      tmem_regs_ready(r0);
      tmem_regs_ready(r1);
      if (q == 1) release0();
      if (q == 3) release1();
      const int ncv = a.cols - c;  // valid columns in the group (uniform)
      if (ncv < 64) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i >= ncv) r0[i] = 0xFF800000u;  // -inf
          if (i + 32 >= ncv) r1[i] = 0xFF800000u;
        }
      }
      float m8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m8[j] = fmaxf(__uint_as_float(r0[j]), __uint_as_float(r1[j]));
#pragma unroll
      for (int i = 8; i < 32; ++i) {
        m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(r0[i]));
        m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(r1[i]));
      }
      const float m = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                            fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      if (tl >= c && tl < c + 64) {
        const int k = static_cast<int>(tl - c);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i == k) zt = __uint_as_float(r0[i]);
          if (i + 32 == k) zt = __uint_as_float(r1[i]);
        }
        zt_here = true;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        y[q][i] = pack_bf16x2(__uint_as_float(r0[2 * i]) - m, __uint_as_float(r0[2 * i + 1]) - m);
        y[q][16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]) - m, __uint_as_float(r1[2 * i + 1]) - m);
      }
      mg[q] = m;
    } else {
      // a group past the last column: nothing to read
      if (q == 1) release0();
      if (q == 3) release1();
    }
  }
  // both halves are free: sums of exp and stores
  const size_t prow = static_cast<size_t>(grow) * a.vocab_tiles;
#pragma unroll
  for (int q = 0; q < kGroups; ++q) {
    const int c = n0 + col_of(q);
    if (c >= a.cols) continue;  // uniform
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      s4[i & 3] += ex2_approx(__uint_as_float(y[q][i] << 16) * kLog2e);
      s4[(i + 2) & 3] += ex2_approx(__uint_as_float(y[q][i] & 0xFFFF0000u) * kLog2e);
    }
    if (rvalid) a.partials[prow + c / 64] = make_float2(mg[q], (s4[0] + s4[1]) + (s4[2] + s4[3]));
    if (a.store_logits) {
      // stage one 16 KB sub-tile and hand it to the TMA unit
      uint8_t* buf = sE + ebuf * kEpiBytes;
      if (leader) bulk_wait_group_read<kEpiBufsWide - 1>();
      named_bar_sync(bar, kEpiThreads);
      stage_row(buf, row, y[q]);
      fence_proxy_async_smem();
      named_bar_sync(bar, kEpiThreads);
      if (leader) {
        tma_store_2d(tmO, smem_u32(buf), c, m0);
        bulk_commit_group();
      }
      __syncwarp();
      if (kEpiBufsWide == 2) ebuf ^= 1u;
    }
  }
  if (rvalid && zt_here) a.zt[grow] = zt;
}

// ===================================================== single-CTA kernel

template <int AMN, int BMN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, const UmmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sE = sB + kStages * kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + 2 * kEpiBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int acc) { return bar0 + 8u * (2 * kStages + acc); };
  auto tempty_bar = [&](int acc) { return bar0 + 8u * (2 * kStages + 2 + acc); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int acc = 0; acc < 2; ++acc) {
      mbar_init(tfull_bar(acc), 1);
      mbar_init(tempty_bar(acc), kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    tma_prefetch_map(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_units = a.num_m * a.num_n * a.num_s;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      uint32_t n_issued = 0;
      bool failed = false;
      for (int u = blockIdx.x; u < num_units && !failed; u += gridDim.x) {
        const Unit t = unit_coords(a, u);
        const int kb0 = t.s * a.kb_per_split;
        const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int stage = n_issued % kStages;
          const uint32_t phase = (n_issued / kStages) & 1u;
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, a.ctrl, a.timeout_ns)) {
            failed = true;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, kStageBytes);
          const uint32_t sa = smem_u32(sA + stage * kABytes);
          const uint32_t sb = smem_u32(sB + stage * kBBytes);
          const int k0 = kb * kBK;
          if (AMN == 0) {
            tma_load_2d(sa, &tmA, fb, k0, t.m * kBM);
          } else {
            tma_load_2d(sa, &tmA, fb, t.m * kBM, k0);
            tma_load_2d(sa + 8192, &tmA, fb, t.m * kBM + 64, k0);
          }
          if (BMN == 0) {
            tma_load_2d(sb, &tmB, fb, k0, t.n * kBN);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(sb + 8192 * j, &tmB, fb, t.n * kBN + 64 * j, k0);
          }
          ++n_issued;
        }
      }
      if (failed) {
        // let the loads already in flight land before the CTA goes away
        const uint32_t first = n_issued > kStages ? n_issued - kStages : 0;
        for (uint32_t i = first; i < n_issued; ++i)
          mbar_drain_wait(full_bar(i % kStages), (i / kStages) & 1u, a.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, AMN, BMN);
      uint32_t n_consumed = 0;
      bool issued = false, failed = false;
      int it = 0;
      for (int u = blockIdx.x; u < num_units && !failed; u += gridDim.x, ++it) {
        const Unit t = unit_coords(a, u);
        const int kb0 = t.s * a.kb_per_split;
        const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, a.ctrl, a.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        for (int kb = kb0; kb < kb1; ++kb) {
          const int stage = n_consumed % kStages;
          const uint32_t phase = (n_consumed / kStages) & 1u;
          if (!mbar_wait_bounded(full_bar(stage), phase, a.ctrl, a.timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sA + stage * kABytes);
          const uint32_t sb = smem_u32(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // K-major: the 16-deep slice starts 32 bytes further along the
            // swizzled 128-byte row. MN-major: 16 k-rows of 128 bytes further.
            const uint64_t ad = AMN ? smem_desc_sw128(sa + 2048u * k, 8192u, 1024u)
                                    : smem_desc_sw128(sa + 32u * k, 16u, 1024u);
            const uint64_t bd = BMN ? smem_desc_sw128(sb + 2048u * k, 8192u, 1024u)
                                    : smem_desc_sw128(sb + 32u * k, 16u, 1024u);
            tc_mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          tc_commit(empty_bar(stage));
          ++n_consumed;
        }
        if (failed) break;
        tc_commit(tfull_bar(acc));
      }
      if (failed && issued) {
        tc_commit(drain_bar);
        mbar_drain_wait(drain_bar, 0, a.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;               // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;        // tile row owned by this thread
    const bool leader = threadIdx.x == 64; // issues the TMA stores
    uint32_t ebuf = 0;
    int it = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, a.ctrl, a.timeout_ns);
      if (named_bar_or(kEpiBar, kEpiThreads, !ok)) break;
      tc_fence_after();
      const Unit t = unit_coords(a, u);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wq * 32) << 16) + acc * kBN;
      epilogue_tile<EPI>(a, &tmO, sE, ebuf, row, leader, t.m * kBM, t.n * kBN, t.s, tbase, [&] {
        tc_fence_before();
        mbar_arrive(tempty_bar(acc));
      });
    }
    if (leader) bulk_wait_group<0>();
  }

  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ======================================================= CTA-pair kernel

template <int AMN, int BMN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    umma_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, const UmmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStagesPair * kABytes;
  uint8_t* sE = sB + kStagesPair * kBHalfBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + 2 * kEpiBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStagesPair + 5);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStagesPair + s); };
  auto tfull_bar = [&](int acc) { return bar0 + 8u * (2 * kStagesPair + acc); };
  auto tempty_bar = [&](int acc) { return bar0 + 8u * (2 * kStagesPair + 2 + acc); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStagesPair + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: the CTA that issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesPair; ++s) {
      mbar_init(full_bar(s), 1);     // used in CTA 0 only: both CTAs' loads land here
      mbar_init(empty_bar(s), 1);    // each CTA's own, released by the pair's MMA commit
    }
    for (int acc = 0; acc < 2; ++acc) {
      mbar_init(tfull_bar(acc), 1);
      mbar_init(tempty_bar(acc), 2 * kEpiThreads);  // used in CTA 0: both epilogues arrive
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    tma_prefetch_map(&tmO);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_units = a.num_m * a.num_n * a.num_s;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      uint32_t n_issued = 0;
      bool failed = false;
      for (int u = pair; u < num_units && !failed; u += npairs) {
        const Unit t = unit_coords(a, u);
        const int kb0 = t.s * a.kb_per_split;
        const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
        const int mA = t.m * 2 * kBM + static_cast<int>(rank) * kBM;   // this CTA's rows of A
        const int nB = t.n * kBN + static_cast<int>(rank) * (kBN / 2);  // this CTA's columns of B
        for (int kb = kb0; kb < kb1; ++kb) {
          const int stage = n_issued % kStagesPair;
          const uint32_t phase = (n_issued / kStagesPair) & 1u;
          if (!mbar_wait_bounded_cluster(empty_bar(stage), phase ^ 1u, a.ctrl, a.timeout_ns)) {
            failed = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * kStageBytesPair);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t sa = smem_u32(sA + stage * kABytes);
          const uint32_t sb = smem_u32(sB + stage * kBHalfBytes);
          const int k0 = kb * kBK;
          if (AMN == 0) {
            tma_load_2d_pair(sa, &tmA, fb, k0, mA);
          } else {
            tma_load_2d_pair(sa, &tmA, fb, mA, k0);
            tma_load_2d_pair(sa + 8192, &tmA, fb, mA + 64, k0);
          }
          if (BMN == 0) {
            tma_load_2d_pair(sb, &tmB, fb, k0, nB);
          } else {
            tma_load_2d_pair(sb, &tmB, fb, nB, k0);
            tma_load_2d_pair(sb + 8192, &tmB, fb, nB + 64, k0);
          }
          ++n_issued;
        }
      }
      if (failed && rank == 0) {
        const uint32_t first = n_issued > kStagesPair ? n_issued - kStagesPair : 0;
        for (uint32_t i = first; i < n_issued; ++i)
          mbar_drain_wait(full_bar(i % kStagesPair), (i / kStagesPair) & 1u, a.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------- MMA issuer (CTA 0 of the pair)
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, kBN, AMN, BMN);
      uint32_t n_consumed = 0;
      bool issued = false, failed = false;
      int it = 0;
      for (int u = pair; u < num_units && !failed; u += npairs, ++it) {
        const Unit t = unit_coords(a, u);
        const int kb0 = t.s * a.kb_per_split;
        const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded_cluster(tempty_bar(acc), acc_phase ^ 1u, a.ctrl, a.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        for (int kb = kb0; kb < kb1; ++kb) {
          const int stage = n_consumed % kStagesPair;
          const uint32_t phase = (n_consumed / kStagesPair) & 1u;
          if (!mbar_wait_bounded_cluster(full_bar(stage), phase, a.ctrl, a.timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sA + stage * kABytes);
          const uint32_t sb = smem_u32(sB + stage * kBHalfBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = AMN ? smem_desc_sw128(sa + 2048u * k, 8192u, 1024u)
                                    : smem_desc_sw128(sa + 32u * k, 16u, 1024u);
            const uint64_t bd = BMN ? smem_desc_sw128(sb + 2048u * k, 8192u, 1024u)
                                    : smem_desc_sw128(sb + 32u * k, 16u, 1024u);
            tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          tc_commit_pair_multicast(empty_bar(stage), 0x3);
          ++n_consumed;
        }
        if (failed) break;
        tc_commit_pair_multicast(tfull_bar(acc), 0x3);
      }
      if (failed && issued) {
        tc_commit_pair(drain_bar);
        mbar_drain_wait(drain_bar, 0, a.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const bool leader = threadIdx.x == 64;
    uint32_t ebuf = 0;
    int it = 0;
    for (int u = pair; u < num_units; u += npairs, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool ok = mbar_wait_bounded_cluster(tfull_bar(acc), acc_phase, a.ctrl, a.timeout_ns);
      if (named_bar_or(kEpiBar, kEpiThreads, !ok)) break;
      tc_fence_after();
      const Unit t = unit_coords(a, u);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wq * 32) << 16) + acc * kBN;
      const int m0 = t.m * 2 * kBM + static_cast<int>(rank) * kBM;
      epilogue_tile<EPI>(a, &tmO, sE, ebuf, row, leader, m0, t.n * kBN, t.s, tbase, [&] {
        tc_fence_before();
        if (rank == 0)
          mbar_arrive(tempty_bar(acc));
        else
          mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      });
    }
    if (leader) bulk_wait_group<0>();
  }

  __syncwarp();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs may touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ============================================ wide CTA-pair tiles (256 x 512)
//
// The pair kernel's shared memory is the limit: per k-block a CTA takes
// 32 KB of TMA writes and serves 32 KB of MMA reads for 8.4 MFLOP, about the
// 128 bytes per clock its shared memory moves at the tensor cores' full rate.
// Here a pair computes a 256 x 512 tile as two 256 x 256 MMAs per k-step that
// share their A operand through the tensor core's collector buffer
// (collector::a::fill, then ::lastuse), so A is read from shared memory once
// for twice the work: 48 KB written and 48 KB read per 16.8 MFLOP. The 512
// accumulator columns fill TMEM, so the accumulator is single-buffered: the
// next tile's MMAs wait until the epilogue has read it out (the fp32
// epilogue's last stores run after that). Its two 256-column halves are
// handed back on separate barriers: the log-sum-exp epilogue frees the first
// half before reading the second, and meanwhile the MMA issuer runs the next
// tile's first-half MMAs on the k-blocks already staged. The shape pays most
// where K per tile is long.
// The TMA loads of one wide-tile work unit, k-blocks kb0 .. kb1: this CTA's
// 128 rows of A (from row mA) and its 256 columns of B (two 128-column halves,
// one per MMA, from column nB0 and nB0 + 256), into the ring after the
// n_issued stages already filled. Both CTAs' loads complete on the even CTA's
// full barrier (full0: stage 0's; empty0: this CTA's stage-0 empty barrier).
// Returns false once a wait for a free stage has run out.
template <int AMN, int BMN>
__device__ __forceinline__ bool load_wide_unit(const CUtensorMap* tmA, const CUtensorMap* tmB, int kb0, int kb1,
                                               int mA, int nB0, uint32_t rank, const uint8_t* sA,
                                               const uint8_t* sB, uint32_t full0, uint32_t empty0,
                                               uint32_t& n_issued, uint32_t* ctrl, uint64_t timeout_ns) {
  const int nB1 = nB0 + kBN;
  for (int kb = kb0; kb < kb1; ++kb) {
    const uint32_t stage = n_issued % kStagesWide;
    const uint32_t phase = (n_issued / kStagesWide) & 1u;
    if (!mbar_wait_bounded_cluster(empty0 + 8u * stage, phase ^ 1u, ctrl, timeout_ns)) return false;
    const uint32_t full = full0 + 8u * stage;
    if (rank == 0) mbar_arrive_expect_tx(full, 2 * kStageBytesWide);
    const uint32_t fb = mapa_shared(full, 0);
    const uint32_t sa = smem_u32(sA + stage * kABytes);
    const uint32_t sb = smem_u32(sB + stage * kBBytes);
    const int k0 = kb * kBK;
    if (AMN == 0) {
      tma_load_2d_pair(sa, tmA, fb, k0, mA);
    } else {
      tma_load_2d_pair(sa, tmA, fb, mA, k0);
      tma_load_2d_pair(sa + 8192, tmA, fb, mA + 64, k0);
    }
    if (BMN == 0) {
      tma_load_2d_pair(sb, tmB, fb, k0, nB0);
      tma_load_2d_pair(sb + kBHalfBytes, tmB, fb, k0, nB1);
    } else {
      tma_load_2d_pair(sb, tmB, fb, nB0, k0);
      tma_load_2d_pair(sb + 8192, tmB, fb, nB0 + 64, k0);
      tma_load_2d_pair(sb + kBHalfBytes, tmB, fb, nB1, k0);
      tma_load_2d_pair(sb + kBHalfBytes + 8192, tmB, fb, nB1 + 64, k0);
    }
    ++n_issued;
  }
  return true;
}

template <int AMN, int BMN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsWide, 1)
    umma_wide_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, const UmmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStagesWide * kABytes;
  uint8_t* sE = sB + kStagesWide * kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + 2 * kEpiBufsWide * kEpiBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStagesWide + 4);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStagesWide + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * kStagesWide);
  // the accumulator's two 256-column halves are handed back separately
  const uint32_t tempty0_bar = bar0 + 8u * (2 * kStagesWide + 1);
  const uint32_t drain_bar = bar0 + 8u * (2 * kStagesWide + 2);
  const uint32_t tempty1_bar = bar0 + 8u * (2 * kStagesWide + 3);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: the CTA that issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesWide; ++s) {
      mbar_init(full_bar(s), 1);     // used in CTA 0 only: both CTAs' loads land here
      mbar_init(empty_bar(s), 1);    // each CTA's own, released by the pair's MMA commit
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty0_bar, 2 * 2 * kEpiThreads);  // used in CTA 0: both CTAs' two epilogues arrive
    mbar_init(tempty1_bar, 2 * 2 * kEpiThreads);
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    tma_prefetch_map(&tmO);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_units = a.num_m * a.num_n * a.num_s;
  // each role's code sits inside the branch that sets its register budget
  if (warp < 4) {
    warpgroup_regs_dec<kWideRegsCtl>();
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t n_issued = 0;
        bool failed = false;
        for (int u = pair; u < num_units && !failed; u += npairs) {
          const Unit t = unit_coords(a, u);
          const int kb0 = t.s * a.kb_per_split;
          const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
          const int mA = t.m * 2 * kBM + static_cast<int>(rank) * kBM;      // this CTA's rows of A
          const int nB0 = t.n * 2 * kBN + static_cast<int>(rank) * (kBN / 2);  // its columns, MMA 0
          if (!load_wide_unit<AMN, BMN>(&tmA, &tmB, kb0, kb1, mA, nB0, rank, sA, sB, full_bar(0), empty_bar(0),
                                        n_issued, a.ctrl, a.timeout_ns))
            failed = true;
        }
        if (failed && rank == 0) {
          const uint32_t first = n_issued > kStagesWide ? n_issued - kStagesWide : 0;
          for (uint32_t i = first; i < n_issued; ++i)
            mbar_drain_wait(full_bar(i % kStagesWide), (i / kStagesWide) & 1u, a.timeout_ns);
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && rank == 0) {
        // ------------------------------------- MMA issuer (CTA 0 of the pair)
        constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, kBN, AMN, BMN);
        uint32_t n_consumed = 0;
        bool issued = false, failed = false;
        int it = 0;
        // the MMAs of one k-block (four k-steps) at ring stage `stage`: both
        // halves sharing A through the collector (half < 0), or one half
        // with A read from shared memory
        auto mma_kblock = [&](int stage, int half, bool first) {
          const uint32_t sa = smem_u32(sA + stage * kABytes);
          const uint32_t sb = smem_u32(sB + stage * kBBytes);
  #pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = AMN ? smem_desc_sw128(sa + 2048u * k, 8192u, 1024u)
                                    : smem_desc_sw128(sa + 32u * k, 16u, 1024u);
            const uint32_t ko = BMN ? 2048u * k : 32u * k;
            const uint64_t bd0 = BMN ? smem_desc_sw128(sb + ko, 8192u, 1024u)
                                     : smem_desc_sw128(sb + ko, 16u, 1024u);
            const uint64_t bd1 = BMN ? smem_desc_sw128(sb + kBHalfBytes + ko, 8192u, 1024u)
                                     : smem_desc_sw128(sb + kBHalfBytes + ko, 16u, 1024u);
            const uint32_t acc_in = (!first || k > 0) ? 1u : 0u;
            if (half < 0) {
              tc_mma_bf16_pair_a_fill(tmem_base, ad, bd0, idesc, acc_in);
              tc_mma_bf16_pair_a_lastuse(tmem_base + kBN, ad, bd1, idesc, acc_in);
            } else {
              tc_mma_bf16_pair(tmem_base + half * kBN, ad, half ? bd1 : bd0, idesc, acc_in);
            }
          }
        };
        for (int u = pair; u < num_units && !failed; u += npairs, ++it) {
          const Unit t = unit_coords(a, u);
          const int kb0 = t.s * a.kb_per_split;
          const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
          const uint32_t tph = (it & 1) ^ 1u;
          if (!mbar_wait_bounded_cluster(tempty0_bar, tph, a.ctrl, a.timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          // While the epilogue still reads the second half, the first half's
          // MMAs of the tile's first k-blocks run (at most the ring's depth:
          // their stages stay until the second half's MMAs have read them).
          int deferred = 0;
          {
            const uint64_t t0 = globaltimer_ns();
  #pragma unroll 1
            for (uint32_t spin = 0; !mbar_try_wait_cluster(tempty1_bar, tph); ++spin) {
              if (deferred < kStagesWide && kb0 + deferred < kb1) {
                const uint32_t n = n_consumed + static_cast<uint32_t>(deferred);
                if (mbar_try_wait_cluster(full_bar(n % kStagesWide), (n / kStagesWide) & 1u)) {
                  tc_fence_after();
                  mma_kblock(n % kStagesWide, 0, deferred == 0);
                  issued = true;
                  ++deferred;
                  continue;
                }
              }
              if ((spin & 63u) == 0u) {
                if (ld_volatile_u32(a.ctrl) != 0u || globaltimer_ns() - t0 > a.timeout_ns) {
                  atomicCAS(a.ctrl, 0u, kErrTimeout);
                  failed = true;
                  break;
                }
              }
            }
          }
          if (failed) break;
          tc_fence_after();
          // the second half's MMAs of the deferred k-blocks, in k order
          for (int j = 0; j < deferred; ++j) {
            const int stage = (n_consumed + static_cast<uint32_t>(j)) % kStagesWide;
            mma_kblock(stage, 1, j == 0);
            tc_commit_pair_multicast(empty_bar(stage), 0x3);
          }
          n_consumed += static_cast<uint32_t>(deferred);
          for (int kb = kb0 + deferred; kb < kb1; ++kb) {
            const int stage = n_consumed % kStagesWide;
            const uint32_t phase = (n_consumed / kStagesWide) & 1u;
            if (!mbar_wait_bounded_cluster(full_bar(stage), phase, a.ctrl, a.timeout_ns)) {
              failed = true;
              break;
            }
            tc_fence_after();
            mma_kblock(stage, -1, kb == kb0);
            issued = true;
            tc_commit_pair_multicast(empty_bar(stage), 0x3);
            ++n_consumed;
          }
          if (failed) break;
          tc_commit_pair_multicast(tfull_bar, 0x3);
        }
        if (failed && issued) {
          tc_commit_pair(drain_bar);
          mbar_drain_wait(drain_bar, 0, a.timeout_ns);
        }
      }
    }
  } else {
    warpgroup_regs_inc<kWideRegsEpi>();
    // ------------------------------------------------------------ epilogue
    // two epilogue warpgroups, one per 256-column half of the tile, each
    // with its own staging buffer and named barrier; every thread of both
    // hands the accumulator back after its last TMEM read. Warp w reads TMEM
    // lanes 32 (w % 4) .. 32 (w % 4) + 31.
    const int grp = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const bool leader = threadIdx.x == (grp + 1) * kEpiThreads;
    const uint32_t bar = kEpiBar + static_cast<uint32_t>(grp);
    uint8_t* sEg = sE + grp * kEpiBufsWide * kEpiBytes;
    uint32_t ebuf = 0;
    int it = 0;
    for (int u = pair; u < num_units; u += npairs, ++it) {
      const bool ok = mbar_wait_bounded_cluster(tfull_bar, it & 1, a.ctrl, a.timeout_ns);
      if (named_bar_or(bar, kEpiThreads, !ok)) break;
      tc_fence_after();
      const Unit t = unit_coords(a, u);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wq * 32) << 16) + grp * kBN;
      const int m0 = t.m * 2 * kBM + static_cast<int>(rank) * kBM;
      const int n0 = t.n * 2 * kBN + grp * kBN;
      auto release_half = [&](uint32_t b) {
        tc_fence_before();
        if (rank == 0)
          mbar_arrive(b);
        else
          mbar_arrive_cluster(mapa_shared(b, 0));
      };
      if constexpr (EPI == kEpiLse) {
        // both warpgroups read the first half, then the second
        epilogue_lse_wide(a, &tmO, sEg, ebuf, row, leader, m0, t.n * 2 * kBN, grp,
                          tmem_base + (static_cast<uint32_t>(wq * 32) << 16),
                          [&] { release_half(tempty0_bar); }, [&] { release_half(tempty1_bar); }, bar);
      } else {
        // each warpgroup reads its own half and hands back both at once
        auto release = [&] {
          release_half(tempty0_bar);
          release_half(tempty1_bar);
        };
        if (n0 < a.cols)
          epilogue_tile<EPI, kEpiBufsWide>(a, &tmO, sEg, ebuf, row, leader, m0, n0, t.s, tbase,
                                           release, bar);
        else
          release();   // the second half lies beyond the last column
      }
    }
    if (leader) bulk_wait_group<0>();
  }

  __syncwarp();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs may touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ============================================ dx and dW GEMMs in one launch
//
// Both backward contractions of a chunk read the finished dlogits buffer
// and write fp32 (dx split partials; dW stored or added), so they can share
// one persistent launch. Problem 0 is dx (A = dlogits, K-major), problem 1 is
// dW (A = dlogitsᵀ, MN-major); B (W, x_c) is MN-major in both.
//
// The units differ in length (a dx unit runs ~1000 k-blocks, a dW unit 64),
// so they are handed out dynamically: the even CTA's producer claims the next
// unit from a global counter (dx units first; the counter runs on across the
// launches of a call, each launch told where it starts) and publishes its index in a
// 4-deep ring in shared memory, to its own MMA issuer and epilogue and, over
// distributed shared memory, to the odd CTA's producer and epilogue. Each of
// those four consumers releases the slot on an mbarrier of the even CTA. A
// pair that finished early simply claims more of the short units.
constexpr int kSchedDepth = 4;
constexpr uint32_t kSmemBytesDual = kSmemBytesPair + 2 * kSchedDepth * 8 + kSchedDepth * 4 + 16;
static_assert(kSmemBytesDual <= 232448, "shared memory per CTA");

template <int AMN>
__device__ __forceinline__ void load_a_pair(uint32_t sa, const CUtensorMap* m, uint32_t fb, int k0,
                                            int mA) {
  if (AMN == 0) {
    tma_load_2d_pair(sa, m, fb, k0, mA);
  } else {
    tma_load_2d_pair(sa, m, fb, mA, k0);
    tma_load_2d_pair(sa + 8192, m, fb, mA + 64, k0);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    umma_pair_dual_kernel(const __grid_constant__ DualMaps maps, const __grid_constant__ DualArgs d) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStagesPair * kABytes;
  uint8_t* sE = sB + kStagesPair * kBHalfBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + 2 * kEpiBytes);
  uint64_t* sbars = bars + 2 * kStagesPair + 5;  // unit ring: full[kSchedDepth], empty[kSchedDepth]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbars + 2 * kSchedDepth);
  int32_t* sched_u = reinterpret_cast<int32_t*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStagesPair + s); };
  auto tfull_bar = [&](int acc) { return bar0 + 8u * (2 * kStagesPair + acc); };
  auto tempty_bar = [&](int acc) { return bar0 + 8u * (2 * kStagesPair + 2 + acc); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStagesPair + 4);
  const uint32_t sbar0 = smem_u32(sbars);
  auto sfull_bar = [&](int i) { return sbar0 + 8u * i; };
  auto sempty_bar = [&](int i) { return sbar0 + 8u * (kSchedDepth + i); };
  const uint32_t su0 = smem_u32(sched_u);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  uint32_t* ctrl = d.p[0].ctrl;
  const uint64_t timeout_ns = d.p[0].timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesPair; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int acc = 0; acc < 2; ++acc) {
      mbar_init(tfull_bar(acc), 1);
      mbar_init(tempty_bar(acc), 2 * kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(sfull_bar(i), 1);   // the even CTA's producer publishes
      mbar_init(sempty_bar(i), 4);  // even MMA, even epilogue, odd producer, odd epilogue
    }
    fence_mbar_init();
    fence_proxy_async_smem();
    for (int q = 0; q < 2; ++q) {
      tma_prefetch_map(&maps.a[q]);
      tma_prefetch_map(&maps.b[q]);
      tma_prefetch_map(&maps.o[q]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int units1 = d.p[1].num_m * d.p[1].num_n * d.p[1].num_s;
  const int num_units = d.units0 + units1;
  // problem and its own unit index for a unit of the combined schedule
  auto locate = [&](int u, int& q, Unit& t) {
    q = u >= d.units0 ? 1 : 0;
    t = unit_coords(d.p[q], q ? u - d.units0 : u);
  };
  // consumers: the unit of step i (-1 = no more), then release the slot.
  // Returns false if the wait ran out.
  auto next_unit = [&](int i, int& u, bool release) {
    const int slot = i % kSchedDepth;
    if (!mbar_wait_bounded_cluster(sfull_bar(slot), (i / kSchedDepth) & 1u, ctrl, timeout_ns))
      return false;
    u = ld_shared_s32(su0 + 4u * slot);
    if (release) {
      if (rank == 0)
        mbar_arrive(sempty_bar(slot));
      else
        mbar_arrive_cluster(mapa_shared(sempty_bar(slot), 0));
    }
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t n_issued = 0;
      bool failed = false;
      for (int i = 0; !failed; ++i) {
        int u;
        if (rank == 0) {
          // claim the next unit and publish it to both CTAs
          const int slot = i % kSchedDepth;
          if (!mbar_wait_bounded_cluster(sempty_bar(slot), ((i / kSchedDepth) & 1u) ^ 1u, ctrl,
                                         timeout_ns)) {
            failed = true;
            break;
          }
          u = atomicAdd(d.sched_ctr, 1) - d.sched_base;
          if (u < 0 || u >= num_units) u = -1;
          sched_u[slot] = u;
          st_shared_cluster_u32(mapa_shared(su0 + 4u * slot, 1), static_cast<uint32_t>(u));
          mbar_arrive(sfull_bar(slot));
          mbar_arrive_cluster(mapa_shared(sfull_bar(slot), 1));
        } else if (!next_unit(i, u, true)) {
          failed = true;
          break;
        }
        if (u < 0) break;
        int q;
        Unit t;
        locate(u, q, t);
        const UmmaArgs& a = d.p[q];
        const int kb0 = t.s * a.kb_per_split;
        const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
        const int mA = t.m * 2 * kBM + static_cast<int>(rank) * kBM;
        const int nB = t.n * kBN + static_cast<int>(rank) * (kBN / 2);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int stage = n_issued % kStagesPair;
          const uint32_t phase = (n_issued / kStagesPair) & 1u;
          if (!mbar_wait_bounded_cluster(empty_bar(stage), phase ^ 1u, ctrl, timeout_ns)) {
            failed = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * kStageBytesPair);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t sa = smem_u32(sA + stage * kABytes);
          const uint32_t sb = smem_u32(sB + stage * kBHalfBytes);
          const int k0 = kb * kBK;
          if (q == 0)
            load_a_pair<0>(sa, &maps.a[0], fb, k0, mA);
          else
            load_a_pair<1>(sa, &maps.a[1], fb, k0, mA);
          tma_load_2d_pair(sb, &maps.b[q], fb, nB, k0);
          tma_load_2d_pair(sb + 8192, &maps.b[q], fb, nB + 64, k0);
          ++n_issued;
        }
      }
      if (failed && rank == 0) {
        const uint32_t first = n_issued > kStagesPair ? n_issued - kStagesPair : 0;
        for (uint32_t i = first; i < n_issued; ++i)
          mbar_drain_wait(full_bar(i % kStagesPair), (i / kStagesPair) & 1u, timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_k = idesc_bf16_f32(2 * kBM, kBN, 0, 1);
      constexpr uint32_t idesc_mn = idesc_bf16_f32(2 * kBM, kBN, 1, 1);
      uint32_t n_consumed = 0;
      bool issued = false, failed = false;
      for (int it = 0; !failed; ++it) {
        int u;
        if (!next_unit(it, u, true)) {
          failed = true;
          break;
        }
        if (u < 0) break;
        int q;
        Unit t;
        locate(u, q, t);
        const UmmaArgs& a = d.p[q];
        const int kb0 = t.s * a.kb_per_split;
        const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded_cluster(tempty_bar(acc), acc_phase ^ 1u, ctrl, timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        const uint32_t idesc = q ? idesc_mn : idesc_k;
        for (int kb = kb0; kb < kb1; ++kb) {
          const int stage = n_consumed % kStagesPair;
          const uint32_t phase = (n_consumed / kStagesPair) & 1u;
          if (!mbar_wait_bounded_cluster(full_bar(stage), phase, ctrl, timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sA + stage * kABytes);
          const uint32_t sb = smem_u32(sB + stage * kBHalfBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = q ? smem_desc_sw128(sa + 2048u * k, 8192u, 1024u)
                                  : smem_desc_sw128(sa + 32u * k, 16u, 1024u);
            const uint64_t bd = smem_desc_sw128(sb + 2048u * k, 8192u, 1024u);
            tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          tc_commit_pair_multicast(empty_bar(stage), 0x3);
          ++n_consumed;
        }
        if (failed) break;
        tc_commit_pair_multicast(tfull_bar(acc), 0x3);
      }
      if (failed && issued) {
        tc_commit_pair(drain_bar);
        mbar_drain_wait(drain_bar, 0, timeout_ns);
      }
    }
  } else {
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const bool leader = threadIdx.x == 64;
    uint32_t ebuf = 0;
    for (int it = 0;; ++it) {
      int u = -1;
      const bool got = next_unit(it, u, false);
      // all 128 threads have read the slot (or given up) before one releases it
      if (named_bar_or(kEpiBar, kEpiThreads, !got)) break;
      if (leader) {
        const int slot = it % kSchedDepth;
        if (rank == 0)
          mbar_arrive(sempty_bar(slot));
        else
          mbar_arrive_cluster(mapa_shared(sempty_bar(slot), 0));
      }
      if (u < 0) break;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool ok = mbar_wait_bounded_cluster(tfull_bar(acc), acc_phase, ctrl, timeout_ns);
      if (named_bar_or(kEpiBar, kEpiThreads, !ok)) break;
      tc_fence_after();
      int q;
      Unit t;
      locate(u, q, t);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wq * 32) << 16) + acc * kBN;
      const int m0 = t.m * 2 * kBM + static_cast<int>(rank) * kBM;
      epilogue_tile<kEpiF32>(d.p[q], &maps.o[q], sE, ebuf, row, leader, m0, t.n * kBN, t.s, tbase,
                             [&] {
                               tc_fence_before();
                               if (rank == 0)
                                 mbar_arrive(tempty_bar(acc));
                               else
                                 mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                             });
    }
    if (leader) bulk_wait_group<0>();
  }

  __syncwarp();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ================================ dx and dW GEMMs in one launch, wide tiles
//
// The same dynamically scheduled backward on the wide tiles: 256 x 512 output
// tiles, two MMAs per k-step sharing A through the collector, the single-
// buffered 512-column accumulator and the two epilogue warpgroups of
// umma_wide_kernel. Each ring slot now has six consumers: the even CTA's MMA
// issuer, the odd CTA's producer, and the leader of each of the four epilogue
// warpgroups (two per CTA), each after its whole warpgroup has read the slot.
// With separate launches the dx GEMM's last wave of long units leaves pairs
// idle, and a dW launch beside it on another stream only starts its
// statically assigned units once dx units retire; here a pair that runs out
// of dx units takes the next dW unit at once.
constexpr int kSchedConsumersWide = 6;
constexpr uint32_t kSmemBytesWideDual =
    kSmemBytesWide + 2 * kSchedDepth * 8 + kSchedDepth * 4 + 16;
static_assert(kSmemBytesWideDual <= 232448, "shared memory per CTA");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsWide, 1)
    umma_wide_dual_kernel(const __grid_constant__ DualMaps maps, const __grid_constant__ DualArgs d) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStagesWide * kABytes;
  uint8_t* sE = sB + kStagesWide * kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + 2 * kEpiBufsWide * kEpiBytes);
  uint64_t* sbars = bars + 2 * kStagesWide + 3;  // unit ring: full[kSchedDepth], empty[kSchedDepth]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbars + 2 * kSchedDepth);
  int32_t* sched_u = reinterpret_cast<int32_t*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStagesWide + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * kStagesWide);
  const uint32_t tempty_bar = bar0 + 8u * (2 * kStagesWide + 1);
  const uint32_t drain_bar = bar0 + 8u * (2 * kStagesWide + 2);
  const uint32_t sbar0 = smem_u32(sbars);
  auto sfull_bar = [&](int i) { return sbar0 + 8u * i; };
  auto sempty_bar = [&](int i) { return sbar0 + 8u * (kSchedDepth + i); };
  const uint32_t su0 = smem_u32(sched_u);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: the CTA that claims units and issues the MMAs
  uint32_t* ctrl = d.p[0].ctrl;
  const uint64_t timeout_ns = d.p[0].timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesWide; ++s) {
      mbar_init(full_bar(s), 1);     // used in CTA 0 only: both CTAs' loads land here
      mbar_init(empty_bar(s), 1);    // each CTA's own, released by the pair's MMA commit
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * 2 * kEpiThreads);  // used in CTA 0: both CTAs' two epilogues arrive
    mbar_init(drain_bar, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(sfull_bar(i), 1);                     // the even CTA's producer publishes
      mbar_init(sempty_bar(i), kSchedConsumersWide);  // used in CTA 0
    }
    fence_mbar_init();
    fence_proxy_async_smem();
    for (int q = 0; q < 2; ++q) {
      tma_prefetch_map(&maps.a[q]);
      tma_prefetch_map(&maps.b[q]);
      tma_prefetch_map(&maps.o[q]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int units1 = d.p[1].num_m * d.p[1].num_n * d.p[1].num_s;
  const int num_units = d.units0 + units1;
  // problem (0: dx, 1: dW) and its own unit of a unit of the combined schedule
  auto locate = [&](int u, int& q, Unit& t) {
    q = u >= d.units0 ? 1 : 0;
    t = unit_coords(d.p[q], q ? u - d.units0 : u);
  };
  // the unit of step i (-1: no more), optionally releasing the slot; false
  // if the wait ran out
  auto next_unit = [&](int i, int& u, bool release) {
    const int slot = i % kSchedDepth;
    if (!mbar_wait_bounded_cluster(sfull_bar(slot), (i / kSchedDepth) & 1u, ctrl, timeout_ns))
      return false;
    u = ld_shared_s32(su0 + 4u * slot);
    if (release) {
      if (rank == 0)
        mbar_arrive(sempty_bar(slot));
      else
        mbar_arrive_cluster(mapa_shared(sempty_bar(slot), 0));
    }
    return true;
  };

  // each role's code sits inside the branch that sets its register budget
  if (warp < 4) {
    warpgroup_regs_dec<kWideRegsCtl>();
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t n_issued = 0;
        bool failed = false;
        for (int i = 0; !failed; ++i) {
          int u;
          if (rank == 0) {
            // claim the next unit and publish it to both CTAs
            const int slot = i % kSchedDepth;
            if (!mbar_wait_bounded_cluster(sempty_bar(slot), ((i / kSchedDepth) & 1u) ^ 1u, ctrl,
                                           timeout_ns)) {
              failed = true;
              break;
            }
            u = atomicAdd(d.sched_ctr, 1) - d.sched_base;
            if (u < 0 || u >= num_units) u = -1;
            sched_u[slot] = u;
            st_shared_cluster_u32(mapa_shared(su0 + 4u * slot, 1), static_cast<uint32_t>(u));
            mbar_arrive(sfull_bar(slot));
            mbar_arrive_cluster(mapa_shared(sfull_bar(slot), 1));
          } else if (!next_unit(i, u, true)) {
            failed = true;
            break;
          }
          if (u < 0) break;
          int q;
          Unit t;
          locate(u, q, t);
          const UmmaArgs& a = d.p[q];
          const int kb0 = t.s * a.kb_per_split;
          const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
          const int mA = t.m * 2 * kBM + static_cast<int>(rank) * kBM;      // this CTA's rows of A
          const int nB0 = t.n * 2 * kBN + static_cast<int>(rank) * (kBN / 2);  // its columns, MMA 0
          // A is K-major for dx and MN-major for dW; B is MN-major in both
          const bool ok = q ? load_wide_unit<1, 1>(&maps.a[1], &maps.b[1], kb0, kb1, mA, nB0, rank, sA, sB,
                                                   full_bar(0), empty_bar(0), n_issued, ctrl, timeout_ns)
                            : load_wide_unit<0, 1>(&maps.a[0], &maps.b[0], kb0, kb1, mA, nB0, rank, sA, sB,
                                                   full_bar(0), empty_bar(0), n_issued, ctrl, timeout_ns);
          if (!ok) failed = true;
        }
        if (failed && rank == 0) {
          const uint32_t first = n_issued > kStagesWide ? n_issued - kStagesWide : 0;
          for (uint32_t i = first; i < n_issued; ++i)
            mbar_drain_wait(full_bar(i % kStagesWide), (i / kStagesWide) & 1u, timeout_ns);
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && rank == 0) {
        // ------------------------------------- MMA issuer (CTA 0 of the pair)
        constexpr uint32_t idesc_k = idesc_bf16_f32(2 * kBM, kBN, 0, 1);
        constexpr uint32_t idesc_mn = idesc_bf16_f32(2 * kBM, kBN, 1, 1);
        uint32_t n_consumed = 0;
        bool issued = false, failed = false;
        for (int it = 0; !failed; ++it) {
          int u;
          if (!next_unit(it, u, true)) {
            failed = true;
            break;
          }
          if (u < 0) break;
          int q;
          Unit t;
          locate(u, q, t);
          const UmmaArgs& a = d.p[q];
          const int kb0 = t.s * a.kb_per_split;
          const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);
          if (!mbar_wait_bounded_cluster(tempty_bar, (it & 1) ^ 1u, ctrl, timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t idesc = q ? idesc_mn : idesc_k;
          for (int kb = kb0; kb < kb1; ++kb) {
            const int stage = n_consumed % kStagesWide;
            const uint32_t phase = (n_consumed / kStagesWide) & 1u;
            if (!mbar_wait_bounded_cluster(full_bar(stage), phase, ctrl, timeout_ns)) {
              failed = true;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(sA + stage * kABytes);
            const uint32_t sb = smem_u32(sB + stage * kBBytes);
  #pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint64_t ad = q ? smem_desc_sw128(sa + 2048u * k, 8192u, 1024u)
                                    : smem_desc_sw128(sa + 32u * k, 16u, 1024u);
              const uint64_t bd0 = smem_desc_sw128(sb + 2048u * k, 8192u, 1024u);
              const uint64_t bd1 = smem_desc_sw128(sb + kBHalfBytes + 2048u * k, 8192u, 1024u);
              const uint32_t acc_in = (kb > kb0 || k > 0) ? 1u : 0u;
              tc_mma_bf16_pair_a_fill(tmem_base, ad, bd0, idesc, acc_in);
              tc_mma_bf16_pair_a_lastuse(tmem_base + kBN, ad, bd1, idesc, acc_in);
            }
            issued = true;
            tc_commit_pair_multicast(empty_bar(stage), 0x3);
            ++n_consumed;
          }
          if (failed) break;
          tc_commit_pair_multicast(tfull_bar, 0x3);
        }
        if (failed && issued) {
          tc_commit_pair(drain_bar);
          mbar_drain_wait(drain_bar, 0, timeout_ns);
        }
      }
    }
  } else {
    warpgroup_regs_inc<kWideRegsEpi>();
    // ------------------------------------------------------------ epilogue
    // one warpgroup per 256-column half of the tile, as in umma_wide_kernel
    const int grp = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const bool leader = threadIdx.x == (grp + 1) * kEpiThreads;
    const uint32_t bar = kEpiBar + static_cast<uint32_t>(grp);
    uint8_t* sEg = sE + grp * kEpiBufsWide * kEpiBytes;
    uint32_t ebuf = 0;
    for (int it = 0;; ++it) {
      int u = -1;
      const bool got = next_unit(it, u, false);
      // the whole warpgroup has read the slot (or given up) before its leader releases it
      if (named_bar_or(bar, kEpiThreads, !got)) break;
      if (leader) {
        const int slot = it % kSchedDepth;
        if (rank == 0)
          mbar_arrive(sempty_bar(slot));
        else
          mbar_arrive_cluster(mapa_shared(sempty_bar(slot), 0));
      }
      if (u < 0) break;
      const bool ok = mbar_wait_bounded_cluster(tfull_bar, it & 1, ctrl, timeout_ns);
      if (named_bar_or(bar, kEpiThreads, !ok)) break;
      tc_fence_after();
      int q;
      Unit t;
      locate(u, q, t);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wq * 32) << 16) + grp * kBN;
      const int m0 = t.m * 2 * kBM + static_cast<int>(rank) * kBM;
      const int n0 = t.n * 2 * kBN + grp * kBN;
      // a half past the last column only releases the accumulator
      epilogue_tile<kEpiF32, kEpiBufsWide>(d.p[q], &maps.o[q], sEg, ebuf, row, leader, m0, n0, t.s,
                                           tbase,
                                           [&] {
                                             tc_fence_before();
                                             if (rank == 0)
                                               mbar_arrive(tempty_bar);
                                             else
                                               mbar_arrive_cluster(mapa_shared(tempty_bar, 0));
                                           },
                                           bar);
    }
    if (leader) bulk_wait_group<0>();
  }

  __syncwarp();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs may touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// One bounded wait on a barrier that nothing completes: checks that a wait
// which runs out reports FLCE_ERR_TIMEOUT and returns.
__global__ void wait_check_kernel(uint32_t* ctrl, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: nobody arrives
    mbar_wait_bounded(smem_u32(&bar), 0u, ctrl + kCtrlError, timeout_ns);
  }
  __syncthreads();
}

template <int AMN, int BMN, int EPI>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                       const UmmaArgs& args, int grid, cudaStream_t s) {
  auto kern = umma_gemm_kernel<AMN, BMN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, s>>>(ta, tb, to, args);
  return cudaGetLastError();
}

// grid = 2 x pairs (a multiple of the cluster size)
template <int AMN, int BMN, int EPI>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                        const UmmaArgs& args, int pairs, cudaStream_t s) {
  auto kern = umma_pair_kernel<AMN, BMN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytesPair));
  if (e != cudaSuccess) return e;
  kern<<<2 * pairs, kThreads, kSmemBytesPair, s>>>(ta, tb, to, args);
  return cudaGetLastError();
}

// The registers a wide kernel is launched with must cover its warpgroups'
// split (setmaxnreg.inc would otherwise wait forever): checked once per
// instantiation from the compiled register count.
template <class Kernel>
cudaError_t check_wide_regs(Kernel kern) {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  return attr.numRegs * kThreadsWide >= static_cast<int>(128 * kWideRegsCtl + 256 * kWideRegsEpi)
             ? cudaSuccess
             : cudaErrorInvalidConfiguration;
}

template <int AMN, int BMN, int EPI>
cudaError_t launch_wide_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                          const UmmaArgs& args, int pairs, cudaStream_t s) {
  auto kern = umma_wide_kernel<AMN, BMN, EPI>;
  static const cudaError_t regs_ok = check_wide_regs(kern);
  if (regs_ok != cudaSuccess) return regs_ok;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytesWide));
  if (e != cudaSuccess) return e;
  kern<<<2 * pairs, kThreadsWide, kSmemBytesWide, s>>>(ta, tb, to, args);
  return cudaGetLastError();
}

}  // namespace

int umma_smem_bytes() { return static_cast<int>(kSmemBytes > kSmemBytesPair ? kSmemBytes : kSmemBytesPair); }

cudaError_t launch_umma(int kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                        const UmmaArgs& args, int grid, cudaStream_t s) {
  switch (kind) {
    case kUmmaLogits: return launch_one<0, 0, kEpiLse>(a, b, o, args, grid, s);
    case kUmmaDlogits: return launch_one<0, 0, kEpiDlogits>(a, b, o, args, grid, s);
    case kUmmaDxBf16: return launch_one<0, 1, kEpiBf16>(a, b, o, args, grid, s);
    case kUmmaDxF32: return launch_one<0, 1, kEpiF32>(a, b, o, args, grid, s);
    case kUmmaDw: return launch_one<1, 1, kEpiF32>(a, b, o, args, grid, s);
    case kUmmaCheckKK: return launch_one<0, 0, kEpiF32>(a, b, o, args, grid, s);
    case kUmmaCheckMK: return launch_one<1, 0, kEpiF32>(a, b, o, args, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_umma_pair(int kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                             const UmmaArgs& args, int pairs, cudaStream_t s) {
  switch (kind) {
    case kUmmaLogits: return launch_pair<0, 0, kEpiLse>(a, b, o, args, pairs, s);
    case kUmmaDlogits: return launch_pair<0, 0, kEpiDlogits>(a, b, o, args, pairs, s);
    case kUmmaDxF32: return launch_pair<0, 1, kEpiF32>(a, b, o, args, pairs, s);
    case kUmmaDw: return launch_pair<1, 1, kEpiF32>(a, b, o, args, pairs, s);
    case kUmmaCheckKK: return launch_pair<0, 0, kEpiF32>(a, b, o, args, pairs, s);
    case kUmmaCheckMK: return launch_pair<1, 0, kEpiF32>(a, b, o, args, pairs, s);
    default: return cudaErrorInvalidValue;
  }
}

// wide tiles: num_n counts 512-column tiles
cudaError_t launch_umma_wide(int kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                             const UmmaArgs& args, int pairs, cudaStream_t s) {
  switch (kind) {
    case kUmmaLogits: return launch_wide_t<0, 0, kEpiLse>(a, b, o, args, pairs, s);
    case kUmmaDlogits: return launch_wide_t<0, 0, kEpiDlogits>(a, b, o, args, pairs, s);
    case kUmmaDxF32: return launch_wide_t<0, 1, kEpiF32>(a, b, o, args, pairs, s);
    case kUmmaDw: return launch_wide_t<1, 1, kEpiF32>(a, b, o, args, pairs, s);
    case kUmmaCheckKK: return launch_wide_t<0, 0, kEpiF32>(a, b, o, args, pairs, s);
    case kUmmaCheckMK: return launch_wide_t<1, 0, kEpiF32>(a, b, o, args, pairs, s);
    default: return cudaErrorInvalidValue;
  }
}

// Clusters of two that fit on the device at once for the wide kernels
int umma_wide_max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreadsWide, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytesWide;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  auto kern = umma_wide_kernel<1, 1, kEpiF32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytesWide)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_umma_wide_dual(const DualMaps& maps, const DualArgs& args, int pairs,
                                  cudaStream_t s) {
  static const cudaError_t regs_ok = check_wide_regs(umma_wide_dual_kernel);
  if (regs_ok != cudaSuccess) return regs_ok;
  cudaError_t e = cudaFuncSetAttribute(umma_wide_dual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytesWideDual));
  if (e != cudaSuccess) return e;
  umma_wide_dual_kernel<<<2 * pairs, kThreadsWide, kSmemBytesWideDual, s>>>(maps, args);
  return cudaGetLastError();
}

cudaError_t launch_umma_pair_dual(const DualMaps& maps, const DualArgs& args, int pairs,
                                  cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(umma_pair_dual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytesDual));
  if (e != cudaSuccess) return e;
  umma_pair_dual_kernel<<<2 * pairs, kThreads, kSmemBytesDual, s>>>(maps, args);
  return cudaGetLastError();
}

// Clusters of two that fit on the device at once for the pair kernels
int umma_pair_max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytesPair;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  auto kern = umma_pair_kernel<1, 1, kEpiF32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytesPair)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_wait_check(uint32_t* ctrl, uint64_t timeout_ns, cudaStream_t s) {
  wait_check_kernel<<<1, 32, 0, s>>>(ctrl, timeout_ns);
  return cudaGetLastError();
}

}  // namespace flce
