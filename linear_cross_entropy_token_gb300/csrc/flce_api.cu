// Host runtime of the FLCE library: the C ABI of include/flce.h, the token-chunk
// scheduler, the workspace, TMA descriptors, per-kernel timing, and the
// chunk loop that enqueues the kernels on the caller's stream.
//
// The chunk loop is the schedule of the FLCE page ("Fused Linear
// Cross-Entropy: LLM 학습 logits 메모리 병목 없애기", section "FLCE의 핵심
// 아이디어: logits을 오래 들고 있지 않는다"): for each chunk of C tokens,
// project to C x V logits, take the CE loss and turn the same buffer into
// softmax - onehot, compute that chunk's dx at once and add its
// dlogitsᵀ·x_chunk into dW; only one chunk buffer exists at a time. Streams
// follow the pattern of "Unlocking asynchronicity in continuous batching"
// (pogovet.com): all work is ordered on one caller stream and the host blocks
// once per call, on the loss read-back.
#include <cudaTypedefs.h>

#include <algorithm>
#include <array>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/flce.h"
#include "flce_internal.h"

using namespace flce;

namespace {

constexpr uint64_t kDefaultBudget = 5ull << 28;  // 1.25 GiB
constexpr int64_t kMaxChunk = 32768;
// SLABS: the slab buffer (chunk x slab bf16) takes what the budget leaves,
// up to 256 MiB: wider slabs mean fewer, longer GEMM launches (at the
// 128256-vocabulary shape 5 slabs of 29184 columns ran 39.7 ms per step,
// 14 of 9728 41.1 ms and 18 of 7168 41.7 ms). The chunk is capped at 4096
// tokens: the dx accumulator (C x H fp32) grows with it and leaves less room
// for the slab.
#ifndef FLCE_SLAB_MIB
#define FLCE_SLAB_MIB 256
#endif
constexpr uint64_t kSlabBytes = static_cast<uint64_t>(FLCE_SLAB_MIB) << 20;
constexpr int64_t kSlabAlign = 512;
constexpr int64_t kMinSlab = 8192;
constexpr int64_t kSlabMaxChunk = 4096;
constexpr int64_t kMaxDim = (1ll << 31) - 1;
constexpr uint64_t kAlign = 1024;
// in-place and recompute modes run the dW GEMM beside the dx GEMM on a second
// stream when the dx launch has fewer work units than this many waves of CTA
// pairs (small problems, where dx leaves SMs idle)
#ifndef FLCE_OVERLAP_WAVES
#define FLCE_OVERLAP_WAVES 2
#endif
constexpr int kOverlapWaves = FLCE_OVERLAP_WAVES;

uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ driver entry

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// --------------------------------------------------------------- profiling

struct EventPair {
  cudaEvent_t start = nullptr, stop = nullptr;
  int kind = 0;
  double flops = 0, bytes = 0;
};

struct Profiler {
  bool enabled = false;
  std::vector<EventPair> pool;
  size_t used = 0;
  flce_kernel_profile totals[FLCE_K_NUM_KINDS] = {};
};

// ------------------------------------------------------------- workspace

struct Layout {
  uint64_t ctrl = 0, logits = 0, partials = 0, zt = 0, lse = 0, dcorr = 0, token_loss = 0,
           dxpart = 0;
  uint64_t total = 0;
};

Layout make_layout(int64_t N, int64_t H, int64_t C, int64_t ldv, int64_t vt, int64_t splits,
                   int esize) {
  Layout L;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  L.ctrl = take(kCtrlWords * 4);
  L.logits = take(static_cast<uint64_t>(C) * ldv * esize);
  // One region serves two buffers that are never live together: the
  // log-sum-exp partials of the chunk (written by the logits GEMM or the
  // statistics pass, last read by the dlogits pass) and the fp32 partials of
  // the dx GEMM's splits (written by the dx GEMM, read by the dx reduction).
  // On the call's stream every mode finishes with the first before it starts
  // on the second, and the next chunk's logits GEMM comes after the dx
  // reduction.
  const uint64_t part_bytes = static_cast<uint64_t>(C) * vt * 8;
  const uint64_t dxpart_bytes = static_cast<uint64_t>(splits) * C * H * 4;
  L.partials = take(std::max(part_bytes, dxpart_bytes));
  L.dxpart = L.partials;
  L.zt = take(static_cast<uint64_t>(C) * 4);
  L.lse = take(static_cast<uint64_t>(C) * 4);
  L.dcorr = take(static_cast<uint64_t>(C) * 4);
  L.token_loss = take(static_cast<uint64_t>(std::max<int64_t>(N, 1)) * 4);
  L.total = off;
  return L;
}

// Tile shape that FLCE_CTA_AUTO resolves to
constexpr int kAutoCta = FLCE_CTA_WIDE;

// CTAs per GEMM work unit: 1 (single) or 2 (pair, wide)
int cta_group_size(const flce_config* cfg) {
  if (cfg->dtype != FLCE_DTYPE_BF16) return 1;
  const int mode = cfg->cta_pair == FLCE_CTA_AUTO ? kAutoCta : cfg->cta_pair;
  return (mode == FLCE_CTA_PAIR || mode == FLCE_CTA_WIDE) ? 2 : 1;
}

bool valid_cta_mode(int mode) {
  return mode == FLCE_CTA_AUTO || mode == FLCE_CTA_SINGLE || mode == FLCE_CTA_PAIR ||
         mode == FLCE_CTA_WIDE;
}

// Tile shapes of one GEMM launch
enum Shape : int { kShapeSingle = 0, kShapePair = 1, kShapeWide = 2 };

// A time model of one GEMM on CTA pairs, in SM cycles, for choosing between
// wide (256 x 512, single-buffered accumulator) and pair (256 x 256, double-
// buffered) tiles per launch. Fitted to 27 launches timed on GB300 (logits, dx
// and dW GEMMs at N x H x V from 1024 x 1024 x 32000 to 4096 x 4096 x 32768,
// both shapes, run one after the other): a 64-deep k-block of a wide tile
// takes ~1110 cycles and of a pair tile ~720 (the wide tile does twice the MMA
// work per k-block with less shared-memory traffic per FLOP); a wide tile's
// epilogue holds the accumulator ~4000 cycles (log-sum-exp: one pass over
// TMEM, the exponentials after the release) or ~5700 (fp32 stores) before the
// next tile's MMAs may start, while a pair tile's epilogue (~5000 / ~4150
// cycles) overlaps its successor's main loop and only shows when that is
// shorter; each tile also pays ~1500 cycles of pipeline fill. Work units run
// in waves of `slots` pairs. The model gets every measured wide-or-pair
// decision right that differs by more than 3%, its pair/wide ratios within
// about 7% on average.
// One work unit of kb k-blocks in that model: what it occupies its pair for.
double unit_cycles(int shape, int64_t kb, bool lse) {
  const double fill = 1500.0;
  if (shape == kShapeWide) return 1110.0 * kb + (lse ? 4000.0 : 5700.0) + fill;
  return std::max(720.0 * kb, lse ? 5000.0 : 4150.0) + fill;
}

double gemm_cycles(int shape, int64_t M, int64_t N, int64_t K, bool lse, int64_t S, int slots) {
  const int64_t kb = cdiv(cdiv(K, kBK), S);
  const int64_t units = cdiv(M, 2 * kBM) * cdiv(N, shape == kShapeWide ? 2 * kBN : kBN) * S;
  const double waves = static_cast<double>(cdiv(units, std::max(slots, 1)));
  return waves * unit_cycles(shape, kb, lse);
}

// HBM round trip of the dx GEMM's fp32 split partials (written, then read by
// the reduction, which also writes dx), in SM cycles at about 3.6 KB per cycle
double dx_partials_cycles(int64_t S, int64_t C, int64_t H) {
  return (4.0 * S * C * H + 6.0 * C * H) / 3600.0;
}

// Splits of the dx GEMM's V reduction when dx and dW share one dynamically
// scheduled launch on tile shape `shape`: the pairs hand units out until none
// is left, so the launch takes about the longer of its longest unit and its
// whole work spread over the pairs. Fewer splits mean longer dx units but
// less partial traffic; with long dx units the short dW units fill in
// behind them. Measured with one launch on GB300: one split at the Llama-3
// and Qwen3 shapes (29.6 and 35.0 ms per step against 30.2 and 35.4 with four
// and five), two to four at 2048 x 1024 x 32000 (within 1%).
int64_t one_launch_splits(int shape, int64_t C, int64_t H, int64_t V, int slots) {
  const int64_t kb = cdiv(V, kBK);
  const int64_t tiles_dx = cdiv(C, 2 * kBM) * cdiv(H, shape == kShapeWide ? 2 * kBN : kBN);
  const int64_t units_dw = cdiv(V, 2 * kBM) * cdiv(H, shape == kShapeWide ? 2 * kBN : kBN);
  const double dw = static_cast<double>(units_dw) * unit_cycles(shape, cdiv(C, kBK), false);
  int64_t best = 1;
  double best_t = -1;
  for (int64_t sp = 1; sp <= 8; ++sp) {
    if (sp > 1 && kb / sp < 16) break;
    const int64_t kbps = cdiv(kb, sp), S = cdiv(kb, kbps);
    const double unit = unit_cycles(shape, kbps, false);
    const double t = std::max(unit, (static_cast<double>(tiles_dx * S) * unit + dw) / std::max(slots, 1)) +
                     dx_partials_cycles(S, C, H);
    if (best_t < 0 || t < best_t * 0.999) {  // more splits only for a gain
      best_t = t;
      best = sp;
    }
  }
  return best;
}

// Pair tiles replace the wide ones only where the model times them more
// than this much faster (its error against measured launches is 5-7%).
constexpr double kPairMargin = 0.95;

// The tile shape (wide or pair) for one GEMM.
int pick_shape(int64_t M, int64_t N, int64_t K, bool lse, int slots) {
  return gemm_cycles(kShapePair, M, N, K, lse, 1, slots) <
                 kPairMargin * gemm_cycles(kShapeWide, M, N, K, lse, 1, slots)
             ? kShapePair
             : kShapeWide;
}

// Output-tile columns of the handle's GEMMs: 512 for wide CTA-pair tiles
int tile_cols(const flce_config* cfg) {
  const int mode = cfg->cta_pair == FLCE_CTA_AUTO ? kAutoCta : cfg->cta_pair;
  return cfg->dtype == FLCE_DTYPE_BF16 && mode == FLCE_CTA_WIDE ? 2 * kBN : kBN;
}

// Splits of the dx GEMM's V reduction that fill the machine's waves best:
// `slots` work units run at once (SMs, or SM pairs), each tile_m x tile_n.
int pick_dx_splits(int64_t C, int64_t H, int64_t V, int slots, int tile_m, int tile_n) {
  const int64_t tiles = cdiv(C, tile_m) * cdiv(H, tile_n);
  const int64_t kb = cdiv(V, kBK);
  int best = 1;
  double best_score = -1;
  for (int s = 1; s <= 4; ++s) {
    if (s > 1 && kb / s < 16) break;
    const int64_t units = tiles * s;
    const int64_t waves = cdiv(units, slots);
    const double eff = static_cast<double>(units) / static_cast<double>(waves * slots);
    const double score = eff - 0.01 * (s - 1);
    if (score > best_score + 1e-12) {
      best_score = score;
      best = s;
    }
  }
  return best;
}

// Tile order for a GEMM whose operands are both streamed from DRAM: dx,
// whose A (the chunk's dlogits) and B (W) are each far larger than L2. The
// persistent grid runs `slots` units at once, moving along k together, so a
// wave of consecutive units reads the k-slices of each tile row's A slab and
// each tile column's B slab once, whatever the number of units sharing them.
// Returns the group_m of the grouped order (1 = columns fastest, num_m =
// rows fastest) whose waves read the fewest slab bytes in total (a row slab
// weighs tile_m, a column slab tile_n).
int pick_group_m(int num_m, int num_n, int num_s, int slots, int tile_m, int tile_n) {
  const int per_s = num_m * num_n;
  const int units = per_s * num_s;
  std::vector<int> seen_m(static_cast<size_t>(num_m) * num_s), seen_n(static_cast<size_t>(num_n) * num_s);
  int best = num_m;
  int64_t best_cost = -1;
  for (int G = num_m; G >= 1; --G) {
    std::fill(seen_m.begin(), seen_m.end(), -1);
    std::fill(seen_n.begin(), seen_n.end(), -1);
    int64_t cost = 0;
    for (int u = 0; u < units; ++u) {
      const int wave = u / slots;
      const int sp = u / per_s, w = u - sp * per_s;
      const int per = G * num_n, g = w / per, idx = w - g * per;
      const int rows = std::min(G, num_m - g * G);
      const int m = g * G + idx % rows, n = idx / rows;
      int& sm = seen_m[static_cast<size_t>(sp) * num_m + m];
      if (sm != wave) {
        sm = wave;
        cost += tile_m;
      }
      int& sn = seen_n[static_cast<size_t>(sp) * num_n + n];
      if (sn != wave) {
        sn = wave;
        cost += tile_n;
      }
    }
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = G;
    }
  }
  return best;
}

flce_status plan_impl(const flce_config* cfg, int64_t N, int64_t H, int64_t V, int64_t chunk,
                      int num_sms, flce_plan* out, std::string* why) {
  if (!cfg || !out) {
    *why = "null config or plan";
    return FLCE_ERR_INVALID_ARG;
  }
  if (N < 0 || H < 1 || V < 1 || chunk < 0 || N > kMaxDim || H > kMaxDim || V > kMaxDim) {
    *why = "sizes must satisfy N >= 0, H >= 1, V >= 1, chunk >= 0";
    return FLCE_ERR_INVALID_ARG;
  }
  if (cfg->dtype != FLCE_DTYPE_BF16 && cfg->dtype != FLCE_DTYPE_FP32) {
    *why = "dtype must be FLCE_DTYPE_BF16 or FLCE_DTYPE_FP32";
    return FLCE_ERR_UNSUPPORTED;
  }
  if (cfg->dlogits_mode < FLCE_DLOGITS_AUTO || cfg->dlogits_mode > FLCE_DLOGITS_SLABS) {
    *why = "dlogits_mode must be one of FLCE_DLOGITS_*";
    return FLCE_ERR_INVALID_ARG;
  }
  if (!valid_cta_mode(cfg->cta_pair)) {
    *why = "cta_pair must be one of FLCE_CTA_AUTO, _SINGLE, _PAIR, _WIDE";
    return FLCE_ERR_INVALID_ARG;
  }
  if (num_sms <= 0) num_sms = 152;
  const bool bf16 = cfg->dtype == FLCE_DTYPE_BF16;
  const bool slabs = cfg->dlogits_mode == FLCE_DLOGITS_SLABS;
  const int esize = bf16 ? 2 : 4;
  const uint64_t budget = cfg->hbm_budget_bytes ? cfg->hbm_budget_bytes : kDefaultBudget;
  std::memset(out, 0, sizeof(*out));
  out->vocab_tiles = cdiv(V, kVocabTile);
  const int group = cta_group_size(cfg);
  const int slots = num_sms / group;
  const int tile_m = group * kBM, tile_n = tile_cols(cfg);
  // an AUTO bf16 handle picks wide or pair tiles per GEMM (the slab walk
  // keeps the wide tiles its slab sizing assumes)
  const bool mixed = bf16 && !slabs && cfg->cta_pair == FLCE_CTA_AUTO;
  // dx on a mixed plan: the tile shape and split of the V reduction with the
  // lowest modelled GEMM time plus the split partials' HBM round trip (about
  // 3.6 KB per cycle)
  struct DxChoice {
    int shape;
    int64_t splits;
  };
  auto dx_choice = [&](int64_t C) -> DxChoice {
    const int64_t kb = cdiv(V, kBK);
    DxChoice best[2] = {{kShapeWide, 1}, {kShapePair, 1}};
    double best_t[2] = {-1, -1};
    for (int i = 0; i < 2; ++i) {
      for (int64_t sp = 1; sp <= 8; ++sp) {
        if (sp > 1 && kb / sp < 16) break;
        const double t = gemm_cycles(best[i].shape, C, H, V, false, sp, slots) +
                         dx_partials_cycles(sp, C, H);
        if (best_t[i] < 0 || t < best_t[i] * 0.999) {  // more splits only for a gain
          best_t[i] = t;
          best[i].splits = sp;
        }
      }
    }
    return best_t[1] < kPairMargin * best_t[0] ? best[1] : best[0];
  };
  // The backward GEMMs of a chunk of C tokens (bf16 in-place and recompute
  // modes on CTA pairs): their tile shapes, and whether they share one
  // dynamically scheduled launch. A mixed plan picks dW's shape with the time
  // model; by default the two share a launch when dW runs on wide tiles, dx
  // joining it there (with units handed out dynamically, the wave count that
  // can favour pair tiles for a dx launch of its own no longer matters). An
  // explicit one-launch request takes the wide tiles too when dW has them,
  // else dx's own choice. Handles with one tile shape share a launch when
  // asked to, or by default on wide tiles.
  struct Backward {
    int dx_shape, dw_shape;
    bool one_launch;
  };
  const int handle_shape = group == 1 ? kShapeSingle : (tile_n == 2 * kBN ? kShapeWide : kShapePair);
  auto backward_for = [&](int64_t C) -> Backward {
    const int bl = cfg->backward_launch;
    if (!bf16 || slabs || group == 1) return {handle_shape, handle_shape, false};
    if (!mixed) {
      const bool one = bl == FLCE_BACKWARD_ONE_LAUNCH ||
                       (bl == FLCE_BACKWARD_AUTO && handle_shape == kShapeWide);
      return {handle_shape, handle_shape, one};
    }
    const int64_t c = std::max<int64_t>(C, 1);
    const int dws = pick_shape(V, H, c, false, slots);
    if (bl == FLCE_BACKWARD_ONE_LAUNCH) {
      const int sh = dws == kShapeWide ? kShapeWide : dx_choice(c).shape;
      return {sh, sh, true};
    }
    if (bl == FLCE_BACKWARD_AUTO && dws == kShapeWide) return {kShapeWide, kShapeWide, true};
    return {dx_choice(c).shape, dws, false};
  };
  // splits of the dx GEMM's V reduction. fp32: the CUDA-core dx GEMM splits
  // when its C x H output has too few tiles to fill the SMs (the count for the
  // full V bounds that of any slab). bf16: one split for SLABS (dx accumulates
  // over the slabs in one fp32 buffer); the one-launch model when dx and dW
  // share a launch; else the mixed plan's choice, or the count that fills the
  // waves of the handle's tile shape.
  auto splits_for = [&](int64_t C) -> int64_t {
    if (!bf16) {
      // the partials take at most an eighth of the budget
      const uint64_t per_split = static_cast<uint64_t>(std::max<int64_t>(C, 1)) * H * 4;
      const int64_t cap = static_cast<int64_t>(budget / 8 / per_split);
      const int64_t s = std::min<int64_t>(simt_split_k(std::max<int64_t>(C, 1), H, V, num_sms), cap);
      return s > 1 ? s : 0;
    }
    if (slabs) return 1;
    const Backward bw = backward_for(C);
    if (bw.one_launch) return one_launch_splits(bw.dx_shape, std::max<int64_t>(C, 1), H, V, slots);
    if (mixed) return dx_choice(std::max<int64_t>(C, 1)).splits;
    return pick_dx_splits(C, H, V, slots, tile_m, tile_n);
  };
  // SLABS: the widest slab (a multiple of 512 columns) whose C x slab buffer
  // fits both kSlabBytes and what the budget leaves beside the rest of the
  // workspace, narrowed where that fills the waves of the per-slab dlogits
  // GEMM (C x slab tiles) and dW GEMM (slab x H tiles) better; within half a
  // percent the wider slab wins. Below 512 columns the workspace exceeds the
  // budget and the planner tries a smaller chunk.
  auto slab_for = [&](int64_t C) -> int64_t {
    if (!slabs) return V;
    const uint64_t cc = static_cast<uint64_t>(std::max<int64_t>(C, 1));
    const uint64_t rest = make_layout(N, H, C, 0, out->vocab_tiles, splits_for(C), esize).total + kAlign;
    const uint64_t room = budget > rest ? std::min(kSlabBytes, budget - rest) : 0;
    const int64_t cmax =
        std::max<int64_t>(kSlabAlign, static_cast<int64_t>(room / (esize * cc)) / kSlabAlign * kSlabAlign);
    if (cmax >= V) return V;
    auto eff = [&](int64_t units) {
      return static_cast<double>(units) / static_cast<double>(cdiv(units, slots) * slots);
    };
    int64_t best = cmax;
    double best_eff = -1;
    for (int64_t vs = cmax; vs >= kSlabAlign; vs -= kSlabAlign) {
      const double e = 0.5 * (eff(cdiv(std::max<int64_t>(C, 1), tile_m) * cdiv(vs, tile_n)) +
                              eff(cdiv(vs, tile_m) * cdiv(H, tile_n)));
      if (e > best_eff + 0.005) {
        best_eff = e;
        best = vs;
      }
    }
    return best;
  };
  auto ldv_for = [&](int64_t C) {
    return static_cast<int64_t>(align_up(static_cast<uint64_t>(slab_for(C)), 64));
  };
  auto ws = [&](int64_t C) {
    return make_layout(N, H, C, ldv_for(C), out->vocab_tiles, splits_for(C), esize).total;
  };
  const int64_t max_chunk = slabs ? kSlabMaxChunk : kMaxChunk;
  int64_t C;
  if (N == 0) {
    C = 0;
  } else if (chunk > 0) {
    C = std::min<int64_t>(std::min(chunk, N), max_chunk);
    if (ws(C) > budget) {
      char b[200];
      std::snprintf(b, sizeof b, "chunk %lld needs %llu workspace bytes, above the budget %llu",
                    static_cast<long long>(C), static_cast<unsigned long long>(ws(C)),
                    static_cast<unsigned long long>(budget));
      *why = b;
      return FLCE_ERR_BUDGET;
    }
  } else {
    const int64_t cap = std::min<int64_t>(max_chunk, static_cast<int64_t>(align_up(N, kBM)));
    int64_t cmax = 0;
    if (slabs) {
      // the largest chunk that still leaves slabs kMinSlab columns wide: a
      // narrower slab multiplies the launches (chunks x slabs) faster than a
      // shorter chunk does
      for (int64_t c = cap; c >= kBM && cmax == 0; c -= kBM)
        if (ws(c) <= budget && slab_for(c) >= std::min<int64_t>(V, kMinSlab)) cmax = c;
    }
    if (cmax == 0)
      for (int64_t c = kBM; c <= cap; c += kBM)
        if (ws(c) <= budget) cmax = c;
    if (cmax == 0) {
      const int64_t c = std::min<int64_t>(N, kBM);
      if (ws(c) <= budget) cmax = c;
    }
    if (cmax == 0) {
      *why = "not even one 128-token chunk fits the HBM budget";
      return FLCE_ERR_BUDGET;
    }
    // even the chunks out over ceil(N / cmax) of them; a shorter chunk can
    // plan more dx splits than cmax did, so take more chunks until the
    // workspace fits again (cmax itself always does)
    const int64_t k0 = cdiv(N, cmax);
    C = cmax;
    for (int64_t k = k0; k <= 4 * k0; ++k) {
      const int64_t c = std::min(std::min<int64_t>(static_cast<int64_t>(align_up(cdiv(N, k), kBM)), cmax), N);
      if (ws(c) <= budget) {
        C = c;
        break;
      }
    }
  }
  out->chunk = C;
  out->num_chunks = C ? cdiv(N, C) : 0;
  out->vocab_slab = slab_for(C);
  out->ldv = ldv_for(C);
  out->dx_splits = std::max<int64_t>(1, C ? splits_for(C) : 1);
  out->workspace_bytes =
      make_layout(N, H, C, out->ldv, out->vocab_tiles, C ? splits_for(C) : 0, esize).total;
  out->logits_bytes = static_cast<uint64_t>(C) * out->ldv * esize;
  out->tile_m = tile_m;
  out->tile_n = tile_n;
  out->tile_n_dx = tile_n;
  out->tile_n_dw = tile_n;
  auto cols = [](int sh) -> int64_t { return sh == kShapeWide ? 2 * kBN : kBN; };
  if (mixed && C > 0) out->tile_n = cols(pick_shape(C, V, H, true, slots));
  // in-place and recompute modes on CTA pairs: the dx and dW GEMMs of a chunk
  // share one dynamically scheduled launch (measured faster than separate
  // launches at every workload shape on wide tiles), or the dW GEMM runs
  // beside a dx launch that fills less than kOverlapWaves waves
  if (bf16 && !slabs && C > 0 && group == 2) {
    const Backward bw = backward_for(C);
    out->tile_n_dx = cols(bw.dx_shape);
    out->tile_n_dw = cols(bw.dw_shape);
    out->backward_one_launch = bw.one_launch ? 1 : 0;
    if (!bw.one_launch) {
      const int64_t kb = cdiv(V, kBK);
      const int64_t kbps = cdiv(kb, std::max<int64_t>(out->dx_splits, 1));
      const int64_t S = cdiv(kb, kbps);
      const int64_t dx_units = cdiv(C, 2 * kBM) * cdiv(H, out->tile_n_dx) * S;
      out->dw_beside_dx = dx_units < static_cast<int64_t>(kOverlapWaves) * slots ? 1 : 0;
    }
  }
  // fp32 handles run SLABS as asked and every other mode in place
  out->dlogits_mode = slabs ? FLCE_DLOGITS_SLABS
                      : (bf16 && cfg->dlogits_mode == FLCE_DLOGITS_RECOMPUTE) ? FLCE_DLOGITS_RECOMPUTE
                                                                               : FLCE_DLOGITS_INPLACE;
  return FLCE_OK;
}

}  // namespace

// ------------------------------------------------------------------ handle

struct flce_handle_s {
  flce_config cfg{};
  int device = 0;
  int num_sms = 0;
  int pair_clusters = 0;  // clusters of two the pair kernels fit at once
  int wide_clusters = 0;  // clusters of two the wide kernels fit at once
  // tile shape of the handle's GEMMs; an AUTO handle (cfg.cta_pair stays
  // FLCE_CTA_AUTO) runs each GEMM on the shape its plan names, wide or pair
  int shape = kShapeSingle;
  uint64_t timeout_ns = 0;
  std::string err;
  // workspace
  void* ws = nullptr;
  uint64_t ws_bytes = 0;
  bool ws_external = false;
  bool ws_fresh = true;  // the control block, sticky word included, needs zeroing
  // staging for the host-buffer entry point
  void* stage = nullptr;
  uint64_t stage_bytes = 0;
  uint32_t* host_ctrl = nullptr;  // pinned
  // pipelined host-buffer entry: two staging slots, copies on their own stream
  struct Slot {
    void* stage = nullptr;
    uint64_t bytes = 0;
    cudaEvent_t copied = nullptr;  // the slot's inputs have landed (copy stream)
    cudaEvent_t freed = nullptr;   // the call that read the slot has finished with it
    cudaEvent_t done = nullptr;    // the call's control words are in host memory
    uint32_t* host = nullptr;      // pinned copy of the control words
    uint64_t ticket = 0;
    bool pending = false;
  };
  Slot slots[2];
  cudaStream_t copy_stream = nullptr;
  // SLABS: the dW GEMM of a slab runs on a second stream beside the dx GEMM
  // of the same slab, so each fills the other's last wave
  cudaStream_t side_stream = nullptr;
  cudaEvent_t slab_ready = nullptr;  // the slab's dlogits are in the buffer
  cudaEvent_t slab_freed = nullptr;  // the slab's dW GEMM has read the buffer
  uint64_t next_ticket = 1;
  flce_plan last_plan{};
  int64_t last_N = -1;
  uint64_t token_loss_off = 0;
  bool has_plan = false;
  int64_t launches = 0;
  Profiler prof;
  std::map<std::array<int, 5>, int> group_cache;  // pick_group_m by (shape, num_m, num_n, num_s, slots)
  // the plan of the last sizes planned (a training loop repeats them)
  std::array<int64_t, 4> plan_key{-1, -1, -1, -1};
  flce_plan plan_cached{};
};

namespace {

flce_status fail(flce_handle_t h, flce_status st, const char* fmt, ...) {
  if (h) {
    char b[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(b, sizeof b, fmt, ap);
    va_end(ap);
    h->err = b;
  }
  return st;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

void prof_begin(flce_handle_t h, int kind, cudaStream_t s) {
  if (!h->prof.enabled) return;
  Profiler& p = h->prof;
  if (p.used == p.pool.size()) {
    EventPair e;
    cudaEventCreate(&e.start);
    cudaEventCreate(&e.stop);
    p.pool.push_back(e);
  }
  EventPair& e = p.pool[p.used];
  e.kind = kind;
  cudaEventRecord(e.start, s);
}

void prof_end(flce_handle_t h, cudaStream_t s, double flops, double bytes) {
  if (!h->prof.enabled) return;
  Profiler& p = h->prof;
  EventPair& e = p.pool[p.used];
  e.flops = flops;
  e.bytes = bytes;
  cudaEventRecord(e.stop, s);
  ++p.used;
}

void prof_collect(flce_handle_t h) {
  Profiler& p = h->prof;
  for (size_t i = 0; i < p.used; ++i) {
    EventPair& e = p.pool[i];
    float ms = 0.f;
    cudaEventSynchronize(e.stop);
    cudaEventElapsedTime(&ms, e.start, e.stop);
    flce_kernel_profile& t = p.totals[e.kind];
    t.launches += 1;
    t.total_ms += ms;
    t.flops += e.flops;
    t.bytes += e.bytes;
  }
  p.used = 0;
}

// NVTX range over the host-side enqueue of a call, a chunk or a launch, so a
// timeline profiler can attribute the GPU work to the path's steps. Costs a
// few nanoseconds when no profiler is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

#define FLCE_LAUNCH(kind, flops, bytes, expr)                                                \
  do {                                                                                      \
    NvtxRange nvtx_(flce_kernel_name(kind));                                                \
    prof_begin(h, (kind), s);                                                               \
    cudaError_t e_ = (expr);                                                                \
    prof_end(h, s, (flops), (bytes));                                                       \
    ++h->launches;                                                                          \
    if (e_ != cudaSuccess)                                                                  \
      return fail(h, FLCE_ERR_CUDA, "%s: %s", flce_kernel_name(kind), cudaGetErrorString(e_)); \
  } while (0)

flce_status ensure_workspace(flce_handle_t h, uint64_t bytes) {
  if (h->ws_external) {
    if (h->ws_bytes < bytes)
      return fail(h, FLCE_ERR_BUDGET, "caller workspace has %llu bytes, the call needs %llu",
                  static_cast<unsigned long long>(h->ws_bytes), static_cast<unsigned long long>(bytes));
    return FLCE_OK;
  }
  if (h->ws_bytes >= bytes) return FLCE_OK;
  if (h->ws) {
    cudaFree(h->ws);
    h->ws = nullptr;
    h->ws_bytes = 0;
  }
  if (cudaMalloc(&h->ws, bytes) != cudaSuccess) {
    cudaGetLastError();
    h->ws = nullptr;
    return fail(h, FLCE_ERR_BUDGET, "cudaMalloc of %llu workspace bytes failed",
                static_cast<unsigned long long>(bytes));
  }
  h->ws_bytes = bytes;
  h->ws_fresh = true;
  return FLCE_OK;
}

bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int rank,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                std::string* why) {
  if (!get_encode()) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  (void)esize;
  CUresult r = g_encode(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char b[160];
    std::snprintf(b, sizeof b, "cuTensorMapEncodeTiled failed (%d), rank %d, dims %llu x %llu", int(r),
                  rank, static_cast<unsigned long long>(dims[0]),
                  static_cast<unsigned long long>(dims[1]));
    *why = b;
    return false;
  }
  return true;
}

// 2-D bf16 map over a row-major matrix (inner = contiguous extent)
bool map_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                 uint32_t box_inner, uint32_t box_outer, std::string* why) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {row_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, 2, dims, strides, box, why);
}

// 3-D fp32 map (col, row, plane) for the fp32 epilogue; box 32 x 128 x 1
bool map_f32_3d(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, uint64_t planes,
                uint64_t row_bytes, uint64_t plane_bytes, std::string* why) {
  const uint64_t dims[3] = {cols, rows, planes};
  const uint64_t strides[2] = {row_bytes, plane_bytes};
  const uint32_t box[3] = {32, 128, 1};
  return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, 3, dims, strides, box, why);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The status a device error word stands for (0: FLCE_OK).
flce_status device_status(flce_handle_t h, uint32_t code) {
  if (code == FLCE_ERR_BAD_TARGET)
    return fail(h, FLCE_ERR_BAD_TARGET, "a target is outside [0, V) and is not ignore_index");
  if (code == FLCE_ERR_TIMEOUT)
    return fail(h, FLCE_ERR_TIMEOUT, "a device-side wait ran out (limit %llu ns)",
                static_cast<unsigned long long>(h->timeout_ns));
  if (code == FLCE_ERR_INVALID_ARG)
    return fail(h, FLCE_ERR_INVALID_ARG,
                "the token-sharded divisor is negative or below this shard's own n_valid");
  if (code != 0) return fail(h, FLCE_ERR_CUDA, "device error word %u", code);
  return FLCE_OK;
}

// The status and loss of a finished call from its control words in host memory.
flce_status decode_ctrl(flce_handle_t h, const uint32_t* hc, float* loss) {
  const uint32_t code = hc[kCtrlError];
  if (loss) std::memcpy(loss, &hc[kCtrlLoss], 4);
  return device_status(h, code);
}

flce_status read_back(flce_handle_t h, uint32_t* ctrl_dev, cudaStream_t s, float* loss) {
  cudaError_t e = cudaMemcpyAsync(h->host_ctrl, ctrl_dev, 4 * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "read-back: %s", cudaGetErrorString(e));
  return decode_ctrl(h, h->host_ctrl, loss);
}

// One GEMM on the handle's tile shape; sets num_m from the M extent and the
// grid from the work units (persistent CTAs, or CTA pairs).
int group_for(flce_handle_t h, int shape, int num_m, int num_n, int num_s, int slots) {
  const std::array<int, 5> key{shape, num_m, num_n, num_s, slots};
  auto it = h->group_cache.find(key);
  if (it != h->group_cache.end()) return it->second;
  const int tile_m = shape == kShapeSingle ? kBM : 2 * kBM;
  const int g = pick_group_m(num_m, num_n, num_s, slots, tile_m, shape == kShapeWide ? 2 * kBN : kBN);
  h->group_cache.emplace(key, g);
  return g;
}

// The shape a GEMM with tile_n output columns (from its plan) runs on.
int shape_for(flce_handle_t h, int64_t tile_n) {
  if (h->cfg.cta_pair != FLCE_CTA_AUTO || h->shape == kShapeSingle) return h->shape;
  return tile_n == 2 * kBN ? kShapeWide : kShapePair;
}

// One GEMM on tile shape `shape`; sets num_m and num_n from the extents (M
// rows, args.cols columns) and the grid from the work units (persistent
// CTAs, or CTA pairs).
cudaError_t launch_gemm(flce_handle_t h, int shape, int kind, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& o, UmmaArgs args, int64_t M, cudaStream_t s) {
  const int rows_per_unit = shape == kShapeSingle ? kBM : 2 * kBM;
  const int slots_max = shape == kShapeWide ? h->wide_clusters
                        : shape == kShapePair ? h->pair_clusters : h->num_sms;
  args.num_m = static_cast<int>(cdiv(M, rows_per_unit));
  args.num_n = static_cast<int>(cdiv(args.cols, shape == kShapeWide ? 2 * kBN : kBN));
  const int units = args.num_m * args.num_n * args.num_s;
  const int slots = std::min(units, slots_max);
  if (args.raster == 2) args.group_m = group_for(h, shape, args.num_m, args.num_n, args.num_s, slots);
  if (shape == kShapeWide) return launch_umma_wide(kind, a, b, o, args, slots, s);
  if (shape == kShapePair) return launch_umma_pair(kind, a, b, o, args, slots, s);
  return launch_umma(kind, a, b, o, args, slots, s);
}

// Device copies of a call's host inputs, in one buffer (grown as needed).
struct Staged {
  const void* x = nullptr;
  const void* W = nullptr;
  const int64_t* t = nullptr;
};

flce_status stage_inputs(flce_handle_t h, void** buf, uint64_t* buf_bytes, const void* x_host,
                         const void* W_host, const int64_t* t_host, int64_t N, int64_t H, int64_t V,
                         cudaStream_t s, Staged* out) {
  const uint64_t es = h->cfg.dtype == FLCE_DTYPE_BF16 ? 2 : 4;
  const uint64_t xb = static_cast<uint64_t>(N) * H * es, wb = static_cast<uint64_t>(V) * H * es;
  const uint64_t tb = static_cast<uint64_t>(N) * 8;
  const uint64_t ox = 0, ow = align_up(xb, kAlign), ot = ow + align_up(wb, kAlign);
  const uint64_t need = ot + align_up(std::max<uint64_t>(tb, 8), kAlign);
  if (*buf_bytes < need) {
    if (*buf) {
      cudaDeviceSynchronize();
      cudaFree(*buf);
      *buf = nullptr;
      *buf_bytes = 0;
    }
    if (cudaMalloc(buf, need) != cudaSuccess) {
      cudaGetLastError();
      *buf = nullptr;
      return fail(h, FLCE_ERR_BUDGET, "cudaMalloc of %llu staging bytes failed",
                  static_cast<unsigned long long>(need));
    }
    *buf_bytes = need;
  }
  uint8_t* st = static_cast<uint8_t*>(*buf);
  cudaError_t e = cudaSuccess;
  // timed on `s` when profiling is on (a copy, not a launch)
  prof_begin(h, FLCE_K_H2D_COPY, s);
  if (xb) e = cudaMemcpyAsync(st + ox, x_host, xb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + ow, W_host, wb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && tb) e = cudaMemcpyAsync(st + ot, t_host, tb, cudaMemcpyHostToDevice, s);
  prof_end(h, s, 0.0, static_cast<double>(xb + wb + tb));
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "staging copy: %s", cudaGetErrorString(e));
  out->x = st + ox;
  out->W = st + ow;
  out->t = reinterpret_cast<const int64_t*>(st + ot);
  return FLCE_OK;
}

// The SLABS backward of one chunk, after its statistics: per vocabulary
// slab, the slab's dlogits recomputed into the chunk buffer (C x vocab_slab),
// dx (+)= d_s · W_s into one fp32 C x H buffer (stored by the first slab,
// added by the others, in slab order) and, on the side stream, dW_s (+)=
// d_sᵀ · x_c; then the dx reduction. *side_pending is set once work is on
// the side stream (the caller's stream must join it before the call ends).
struct SlabChunk {
  const flce_plan* plan;
  const UmmaArgs* logits_args;  // the chunk's logits-GEMM arguments
  const CUtensorMap* mX_k;      // x_c, K-major and MN-major
  const CUtensorMap* mX_mn;
  const __nv_bfloat16* W;
  float* dW;
  __nv_bfloat16* buf;           // chunk buffer, row stride plan->ldv
  float* dxacc;                 // C x H fp32
  __nv_bfloat16* dx;            // this chunk's rows of dx
  const int64_t* t;             // this chunk's targets
  float* dcorr;
  uint32_t* ctrl;
  int64_t H, V, C, chunk_index, ignore_index;
  int rows;
  int b_box;                    // rows of a K-major B box for the handle's tile shape
};

// The handle's second stream and its two events (created on first use).
flce_status ensure_side_stream(flce_handle_t h) {
  if (h->side_stream) return FLCE_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&h->side_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->slab_ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->slab_freed, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "side stream: %s", cudaGetErrorString(e));
  return FLCE_OK;
}

flce_status slab_backward(flce_handle_t h, const SlabChunk& k, cudaStream_t s, bool* side_pending) {
  std::string why;
  cudaError_t e = cudaSuccess;
  {
    const flce_status st = ensure_side_stream(h);
    if (st != FLCE_OK) return st;
  }
  const cudaStream_t side = h->side_stream;
  const int64_t H = k.H, V = k.V, Vs = k.plan->vocab_slab, ldv = k.plan->ldv;
  const int rows = k.rows;
  const double dr = rows, dH = static_cast<double>(H);
  const int64_t n_slabs = cdiv(V, Vs);
  CUtensorMap mWs_k, mWs_mn, mZs_out, mZs_k, mZs_mn, mDws, mDxs;
  if (!map_f32_3d(&mDxs, k.dxacc, H, rows, 1, H * 4, static_cast<uint64_t>(k.C) * H * 4, &why))
    return fail(h, FLCE_ERR_INVALID_ARG, "%s", why.c_str());
  for (int64_t sl = 0; sl < n_slabs; ++sl) {
    const int64_t v0 = sl * Vs;
    const int64_t vs = std::min(Vs, V - v0);
    const double dvs = static_cast<double>(vs);
    if (!map_bf16_2d(&mWs_k, k.W + v0 * H, H, vs, H * 2, 64, k.b_box, &why) ||
        !map_bf16_2d(&mWs_mn, k.W + v0 * H, H, vs, H * 2, 64, 64, &why) ||
        !map_f32_3d(&mDws, k.dW + v0 * H, H, vs, 1, H * 4, static_cast<uint64_t>(vs) * H * 4, &why) ||
        !map_bf16_2d(&mZs_out, k.buf, vs, rows, ldv * 2, 64, 128, &why) ||
        !map_bf16_2d(&mZs_k, k.buf, vs, rows, ldv * 2, 64, 128, &why) ||
        !map_bf16_2d(&mZs_mn, k.buf, vs, rows, ldv * 2, 64, 64, &why))
      return fail(h, FLCE_ERR_INVALID_ARG, "%s", why.c_str());
    // the slab's dlogits: a logits GEMM over W_s with the dlogits epilogue;
    // the previous slab's dW GEMM (on the side stream) must have read the
    // buffer first (earlier calls' are ordered by the join that ends them)
    UmmaArgs g = *k.logits_args;
    g.num_n = static_cast<int>(cdiv(vs, kBN));
    g.cols = static_cast<int>(vs);
    g.col_base = v0;
    if (*side_pending) {
      e = cudaStreamWaitEvent(s, h->slab_freed, 0);
      if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "slab wait: %s", cudaGetErrorString(e));
    }
    FLCE_LAUNCH(FLCE_K_GEMM_DLOGITS, 2 * dr * dH * dvs, 2 * dr * dH + 2 * dvs * dH + 2 * dr * dvs + 12 * dr,
                launch_gemm(h, h->shape, kUmmaDlogits, *k.mX_k, mWs_k, mZs_out, g, rows, s));
    e = cudaEventRecord(h->slab_ready, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, h->slab_ready, 0);
    if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "slab fork: %s", cudaGetErrorString(e));
    // dx (+)= d_s · W_s
    UmmaArgs b = *k.logits_args;
    b.num_n = static_cast<int>(cdiv(H, kBN));
    b.num_s = 1;
    b.kb_total = static_cast<int>(cdiv(vs, kBK));
    b.kb_per_split = b.kb_total;
    b.raster = 2;
    b.rows = rows;
    b.cols = static_cast<int>(H);
    b.reduce_add = sl > 0 ? 1 : 0;
    FLCE_LAUNCH(FLCE_K_GEMM_DX, 2 * dr * dvs * dH, 2 * dr * dvs + 2 * dvs * dH + (sl > 0 ? 8.0 : 4.0) * dr * dH,
                launch_gemm(h, h->shape, kUmmaDxF32, mZs_k, mWs_mn, mDxs, b, rows, s));
    // dW_s (+)= d_sᵀ · x_c, beside it on the side stream
    UmmaArgs d = *k.logits_args;
    d.num_n = static_cast<int>(cdiv(H, kBN));
    d.num_s = 1;
    d.kb_total = static_cast<int>(cdiv(rows, kBK));
    d.kb_per_split = d.kb_total;
    d.raster = 1;
    d.rows = static_cast<int>(vs);
    d.cols = static_cast<int>(H);
    d.reduce_add = k.chunk_index > 0 ? 1 : 0;
    {
      const cudaStream_t s = side;  // the launch and its timing events go on the side stream
      FLCE_LAUNCH(FLCE_K_GEMM_DW, 2 * dr * dvs * dH,
                  2 * dr * dvs + 2 * dr * dH + (k.chunk_index > 0 ? 8.0 : 4.0) * dvs * dH,
                  launch_gemm(h, h->shape, kUmmaDw, mZs_mn, *k.mX_mn, mDws, d, vs, s));
    }
    e = cudaEventRecord(h->slab_freed, side);
    if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "slab join: %s", cudaGetErrorString(e));
    *side_pending = true;
  }
  FLCE_LAUNCH(FLCE_K_DX_REDUCE, 0.0, 4 * dr * dH + 2 * dr * dH,
              launch_dx_reduce(k.dxacc, 1, k.C * H, rows, H, k.W, V, k.t, k.ignore_index, k.ctrl, k.dcorr,
                               k.dx, s));
  return FLCE_OK;
}

// Everything of one call up to its control words on the device (*ctrl_out):
// the result is read from them once the stream gets there.
// The sync-free entry points' result in caller device memory (either may be
// null): the loss (NaN after a recorded error) and n_valid.
struct DeviceResult {
  float* loss = nullptr;
  int32_t* n_valid = nullptr;
};

// nv_total: the divisor of a token-sharded batch (device, one int32), or
// null to divide by this call's own n_valid. dres: where the loss reduction
// also writes the device result, or null.
flce_status enqueue_fb(flce_handle_t h, const void* x, const void* W, const int64_t* t, int64_t N,
                       int64_t H, int64_t V, int64_t ignore_index, int64_t chunk, void* dx,
                       float* dW, cudaStream_t s, uint32_t** ctrl_out,
                       const int32_t* nv_total = nullptr, const DeviceResult* dres = nullptr) {
  NvtxRange nvtx_call("flce_forward_backward");
  if (!W || !dW || (N > 0 && (!x || !t || !dx)))
    return fail(h, FLCE_ERR_INVALID_ARG, "null pointer argument");
  const bool bf16 = h->cfg.dtype == FLCE_DTYPE_BF16;
  if (N > 0 && (reinterpret_cast<uintptr_t>(t) & 7u))
    return fail(h, FLCE_ERR_INVALID_ARG, "t must be 8-byte aligned");
  if (bf16) {
    if (H % 8 != 0) return fail(h, FLCE_ERR_INVALID_ARG, "bf16 needs H %% 8 == 0 (H = %lld)", (long long)H);
    if (!aligned16(x) || !aligned16(W) || !aligned16(dW) || (N > 0 && !aligned16(dx)))
      return fail(h, FLCE_ERR_INVALID_ARG, "x, W, dx and dW must be 16-byte aligned");
  } else if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(dW) |
              (N > 0 ? reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(dx) : 0)) & 3u) {
    return fail(h, FLCE_ERR_INVALID_ARG, "x, W, dx and dW must be 4-byte aligned");
  }
  flce_plan p;
  flce_status st = FLCE_OK;
  std::string why;
  const std::array<int64_t, 4> key{N, H, V, chunk};
  if (key == h->plan_key) {
    p = h->plan_cached;
  } else {
    st = plan_impl(&h->cfg, N, H, V, chunk, h->num_sms, &p, &why);
    if (st != FLCE_OK) return fail(h, st, "%s", why.c_str());
    h->plan_key = key;
    h->plan_cached = p;
  }
  st = ensure_workspace(h, p.workspace_bytes);
  if (st != FLCE_OK) return st;
  // the same split count the plan sized the workspace with (fp32 plans
  // without a split hold no partials)
  const int64_t part_splits = bf16 ? p.dx_splits : (p.dx_splits > 1 ? p.dx_splits : 0);
  const Layout L = make_layout(N, H, p.chunk, p.ldv, p.vocab_tiles, part_splits, bf16 ? 2 : 4);
  uint8_t* ws = static_cast<uint8_t*>(h->ws);
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(ws + L.ctrl);
  float2* partials = reinterpret_cast<float2*>(ws + L.partials);
  float* zt = reinterpret_cast<float*>(ws + L.zt);
  float* lse = reinterpret_cast<float*>(ws + L.lse);
  float* dcorr = reinterpret_cast<float*>(ws + L.dcorr);
  float* token_loss = reinterpret_cast<float*>(ws + L.token_loss);
  h->last_plan = p;
  h->last_N = N;
  h->token_loss_off = L.token_loss;
  h->has_plan = true;

  // per-call words: count_valid, the call's first kernel, clears them; a
  // memset only for an empty batch (no count_valid) and, once, to clear the
  // sticky error word of a new block
  cudaError_t e = cudaSuccess;
  if (h->ws_fresh || N == 0)
    e = cudaMemsetAsync(ctrl, 0, (h->ws_fresh ? kCtrlWords : kCtrlSticky) * 4, s);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
  h->ws_fresh = false;
  if (N == 0) {
    e = cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * 4, s);
    if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
    if (dres)
      FLCE_LAUNCH(FLCE_K_DEVICE_RESULT, 0.0, 16.0, launch_device_result(ctrl, dres->loss, dres->n_valid, s));
    *ctrl_out = ctrl;
    return FLCE_OK;
  }
  FLCE_LAUNCH(FLCE_K_COUNT_VALID, 0.0, 8.0 * N,
              launch_count_valid(t, N, V, ignore_index, nv_total, ctrl, s));

  const int64_t C = p.chunk, ldv = p.ldv;
  const int vt = static_cast<int>(p.vocab_tiles);
  // SLABS: whether this call has work on the side stream. However the call
  // returns, its stream then waits for that work, so that no later call can
  // overwrite the slab buffer under a dW GEMM still reading it.
  bool side_pending = false;
  struct SideJoin {
    flce_handle_t h;
    cudaStream_t s;
    const bool& pending;
    ~SideJoin() {
      if (pending) cudaStreamWaitEvent(s, h->slab_freed, 0);
    }
  } side_join{h, s, side_pending};
  const double dV = static_cast<double>(V), dH = static_cast<double>(H);
  int32_t sched_claims = 0;  // work-unit claims of this call's dynamically scheduled launches
  bool loss_done = false;    // the last dx reduction has taken the loss reduction

  if (!bf16) {
    // ---------------------------------------------------------- fp32 path
    const float* xf = static_cast<const float*>(x);
    const float* Wf = static_cast<const float*>(W);
    float* dxf = static_cast<float*>(dx);
    float* logits = reinterpret_cast<float*>(ws + L.logits);
    float* dxpart = reinterpret_cast<float*>(ws + L.dxpart);
    const int dx_splits = static_cast<int>(p.dx_splits);
    const bool slabs = h->cfg.dlogits_mode == FLCE_DLOGITS_SLABS;
    for (int64_t c = 0; c < p.num_chunks; ++c) {
      char nvtx_name[40];
      std::snprintf(nvtx_name, sizeof nvtx_name, "flce chunk %lld", static_cast<long long>(c));
      NvtxRange nvtx_chunk(nvtx_name);
      const int64_t off = c * C;
      const int rows = static_cast<int>(std::min(C, N - off));
      const double dr = rows;
      if (slabs) {
        // statistics slab by slab, the combine, then each slab's logits again:
        // dlogits in place, dx (+)= d_s · W_s, dW_s (+)= d_sᵀ · x_c
        const int64_t Vs = p.vocab_slab, n_slabs = cdiv(V, Vs);
        for (int64_t sl = 0; sl < n_slabs; ++sl) {
          const int64_t v0 = sl * Vs, vs = std::min(Vs, V - v0);
          const double dvs = static_cast<double>(vs);
          const int vts = static_cast<int>(cdiv(vs, kVocabTile));
          FLCE_LAUNCH(FLCE_K_SIMT_GEMM, 2 * dr * dH * dvs, 4 * (dr * dH + dvs * dH + dr * dvs),
                      launch_simt_gemm_f32(xf + off * H, H, 1, Wf + v0 * H, 1, H, logits, ldv, rows, vs, H, 0,
                                           1, nullptr, s));
          FLCE_LAUNCH(FLCE_K_SIMT_TILE_STATS, 0.0, 4 * dr * dvs + 12 * dr * vts,
                      launch_simt_tile_stats(logits, ldv, rows, vs, vts, vt, v0, t + off, ignore_index,
                                             partials + v0 / kVocabTile, zt, s));
        }
        FLCE_LAUNCH(FLCE_K_LSE_COMBINE, 0.0, 8 * dr * vt + 24 * dr,
                    launch_lse_combine(partials, vt, zt, t + off, rows, ignore_index, lse, token_loss + off, s));
        for (int64_t sl = 0; sl < n_slabs; ++sl) {
          const int64_t v0 = sl * Vs, vs = std::min(Vs, V - v0);
          const double dvs = static_cast<double>(vs);
          FLCE_LAUNCH(FLCE_K_SIMT_GEMM, 2 * dr * dH * dvs, 4 * (dr * dH + dvs * dH + dr * dvs),
                      launch_simt_gemm_f32(xf + off * H, H, 1, Wf + v0 * H, 1, H, logits, ldv, rows, vs, H, 0,
                                           1, nullptr, s));
          FLCE_LAUNCH(FLCE_K_DLOGITS, 0.0, 8 * dr * dvs,
                      launch_dlogits_f32(logits, ldv, rows, vs, v0, lse, t + off, ignore_index, ctrl, s));
          FLCE_LAUNCH(FLCE_K_SIMT_GEMM, 2 * dr * dvs * dH, 4 * (dr * dvs + dvs * dH + (sl > 0 ? 2 : 1) * dr * dH),
                      launch_simt_gemm_f32(logits, ldv, 1, Wf + v0 * H, H, 1, dxf + off * H, H, rows, H, vs,
                                           sl > 0 ? 1 : 0, dx_splits, dxpart, s));
          FLCE_LAUNCH(FLCE_K_SIMT_GEMM, 2 * dr * dvs * dH, 4 * (dr * dvs + dr * dH + (c > 0 ? 2 : 1) * dvs * dH),
                      launch_simt_gemm_f32(logits, 1, ldv, xf + off * H, H, 1, dW + v0 * H, H, vs, H, rows,
                                           c > 0 ? 1 : 0, 1, nullptr, s));
        }
        continue;
      }
      FLCE_LAUNCH(FLCE_K_SIMT_GEMM, 2 * dr * dH * dV, 4 * (dr * dH + dV * dH + dr * dV),
                  launch_simt_gemm_f32(xf + off * H, H, 1, Wf, 1, H, logits, ldv, rows, V, H, 0, 1, nullptr, s));
      // the row steps in one launch: log-sum-exp, token loss, dlogits in place
      FLCE_LAUNCH(FLCE_K_COMBINE_DLOGITS, 0.0, 12 * dr * dV + 24 * dr,
                  launch_rows_f32(logits, ldv, rows, V, t + off, ignore_index, ctrl, lse, token_loss + off, s));
      FLCE_LAUNCH(FLCE_K_SIMT_GEMM, 2 * dr * dV * dH, 4 * (dr * dV + dV * dH + dr * dH),
                  launch_simt_gemm_f32(logits, ldv, 1, Wf, H, 1, dxf + off * H, H, rows, H, V, 0, dx_splits,
                                       dxpart, s));
      FLCE_LAUNCH(FLCE_K_SIMT_GEMM, 2 * dr * dV * dH, 4 * (dr * dV + dr * dH + 2 * dV * dH),
                  launch_simt_gemm_f32(logits, 1, ldv, xf + off * H, H, 1, dW, H, V, H, rows, c > 0 ? 1 : 0, 1,
                                       nullptr, s));
    }
  } else {
    // ------------------------------------------------- bf16 tcgen05 path
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    __nv_bfloat16* dxb = static_cast<__nv_bfloat16*>(dx);
    __nv_bfloat16* logits = reinterpret_cast<__nv_bfloat16*>(ws + L.logits);
    float* dxpart = reinterpret_cast<float*>(ws + L.dxpart);
    const bool recompute = h->cfg.dlogits_mode == FLCE_DLOGITS_RECOMPUTE;
    const bool slabs = h->cfg.dlogits_mode == FLCE_DLOGITS_SLABS;
    const int64_t zw = slabs ? p.vocab_slab : V;  // columns of the chunk buffer
    const int b_box = h->shape == kShapeSingle ? 256 : 128;
    CUtensorMap mW_k, mW_mn, mX_k, mX_mn, mZ_out, mZ_k, mZ_mn, mDx, mDw;
    // a CTA of a pair loads 128 of the tile's 256 columns of a K-major B
    if (!map_bf16_2d(&mW_k, W, H, V, H * 2, 64, b_box, &why) ||
        !map_bf16_2d(&mW_mn, W, H, V, H * 2, 64, 64, &why) ||
        !map_f32_3d(&mDw, dW, H, V, 1, H * 4, static_cast<uint64_t>(V) * H * 4, &why))
      return fail(h, FLCE_ERR_INVALID_ARG, "%s", why.c_str());
    const int kb_h = static_cast<int>(cdiv(H, kBK));
    const int kb_v = static_cast<int>(cdiv(V, kBK));
    for (int64_t c = 0; c < p.num_chunks; ++c) {
      char nvtx_name[40];
      std::snprintf(nvtx_name, sizeof nvtx_name, "flce chunk %lld", static_cast<long long>(c));
      NvtxRange nvtx_chunk(nvtx_name);
      const int64_t off = c * C;
      const int rows = static_cast<int>(std::min(C, N - off));
      const double dr = rows;
      const void* xc = xb + off * H;
      if (!map_bf16_2d(&mX_k, xc, H, rows, H * 2, 64, 128, &why) ||
          !map_bf16_2d(&mX_mn, xc, H, rows, H * 2, 64, 64, &why) ||
          !map_bf16_2d(&mZ_out, logits, zw, rows, ldv * 2, 64, 128, &why) ||
          !map_bf16_2d(&mZ_k, logits, zw, rows, ldv * 2, 64, 128, &why) ||
          !map_bf16_2d(&mZ_mn, logits, zw, rows, ldv * 2, 64, 64, &why))
        return fail(h, FLCE_ERR_INVALID_ARG, "%s", why.c_str());

      // the previous chunk's dW GEMM, if it ran on the side stream, must have
      // read the buffer before this chunk's logits GEMM overwrites it
      if (side_pending && !slabs) {
        e = cudaStreamWaitEvent(s, h->slab_freed, 0);
        if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "dW wait: %s", cudaGetErrorString(e));
      }
      // 1. projection with the online max / sum-exp epilogue
      UmmaArgs a{};
      a.num_n = static_cast<int>(cdiv(V, kBN));
      a.num_s = 1;
      a.kb_total = kb_h;
      a.kb_per_split = kb_h;
      a.raster = 0;
      a.rows = rows;
      a.cols = static_cast<int>(V);
      a.vocab_tiles = vt;
      a.store_logits = (recompute || slabs) ? 0 : 1;
      a.ignore_index = ignore_index;
      a.targets = t + off;
      a.partials = partials;
      a.zt = zt;
      a.lse = lse;
      a.dcorr = dcorr;
      a.ctrl = ctrl;
      a.timeout_ns = h->timeout_ns;
      FLCE_LAUNCH(FLCE_K_GEMM_LOGITS, 2 * dr * dH * dV,
                  2 * dr * dH + 2 * dV * dH + ((recompute || slabs) ? 0 : 2 * dr * dV) + 8 * dr * vt + 12 * dr,
                  launch_gemm(h, shape_for(h, p.tile_n), kUmmaLogits, mX_k, mW_k, mZ_out, a, rows, s));
      // 2a. cross-tile log-sum-exp and token losses (in in-place mode, for rows
      // of at most combine_dlogits_max_cols() columns, in one launch with the
      // dlogits pass, 2b)
      const bool fused_rows = !recompute && !slabs && ldv <= combine_dlogits_max_cols();
      if (!fused_rows)
        FLCE_LAUNCH(FLCE_K_LSE_COMBINE, 0.0, 8 * dr * vt + 24 * dr,
                    launch_lse_combine(partials, vt, zt, t + off, rows, ignore_index, lse, token_loss + off, s));
      if (slabs) {
        const SlabChunk k{&p, &a, &mX_k, &mX_mn, static_cast<const __nv_bfloat16*>(W), dW, logits,
                          dxpart, dxb + off * H, t + off, dcorr, ctrl, H, V, C, c, ignore_index, rows,
                          b_box};
        st = slab_backward(h, k, s, &side_pending);
        if (st != FLCE_OK) return st;
        continue;
      }
      // 2b. dlogits = (softmax - onehot) / n_valid over the chunk buffer
      if (recompute) {
        FLCE_LAUNCH(FLCE_K_GEMM_DLOGITS, 2 * dr * dH * dV, 2 * dr * dH + 2 * dV * dH + 2 * dr * dV + 12 * dr,
                    launch_gemm(h, shape_for(h, p.tile_n), kUmmaDlogits, mX_k, mW_k, mZ_out, a, rows, s));
      } else if (fused_rows) {
        FLCE_LAUNCH(FLCE_K_COMBINE_DLOGITS, 0.0, 4 * dr * dV + 8 * dr * vt + 24 * dr,
                    launch_combine_dlogits_bf16(logits, ldv, rows, V, partials, vt, zt, t + off, ignore_index,
                                                ctrl, lse, token_loss + off, dcorr, s));
      } else {
        FLCE_LAUNCH(FLCE_K_DLOGITS, 0.0, 4 * dr * dV,
                    launch_dlogits_bf16(logits, ldv, rows, V, partials, vt, lse, t + off, ignore_index,
                                        ctrl, dcorr, s));
      }
      // 3. dx_chunk = dlogits · W
      const int S_req = static_cast<int>(p.dx_splits);
      const int kbps = (kb_v + S_req - 1) / S_req;
      const int S = (kb_v + kbps - 1) / kbps;
      UmmaArgs b = a;
      b.num_n = static_cast<int>(cdiv(H, kBN));
      b.num_s = S;
      b.kb_total = kb_v;
      b.kb_per_split = kbps;
      b.raster = 2;  // grouped: both operands stream from DRAM (group_m set at launch)
      b.rows = rows;
      b.cols = static_cast<int>(H);
      b.reduce_add = 0;
      // fp32 partials of dlogits·W per split; the reduction adds them in split
      // order, adds dcorr·W[t_i] (the target entry's bf16 rounding error) and
      // rounds dx to bf16 once
      if (!map_f32_3d(&mDx, dxpart, H, rows, S, H * 4, static_cast<uint64_t>(C) * H * 4, &why))
        return fail(h, FLCE_ERR_INVALID_ARG, "%s", why.c_str());
      // 4. dW (+)= dlogitsᵀ · x_chunk, fp32 (stored on the first chunk, added after)
      UmmaArgs d = a;
      d.num_n = static_cast<int>(cdiv(H, kBN));
      d.num_s = 1;
      d.kb_total = static_cast<int>(cdiv(rows, kBK));
      d.kb_per_split = d.kb_total;
      d.raster = 1;
      d.rows = static_cast<int>(V);
      d.cols = static_cast<int>(H);
      d.reduce_add = c > 0 ? 1 : 0;
      // dW beside dx when the plan says so (the dx launch is short of
      // kOverlapWaves waves)
      const bool overlap_dw = p.dw_beside_dx != 0;
      if (overlap_dw) {
        st = ensure_side_stream(h);
        if (st != FLCE_OK) return st;
      }
      const double dx_bytes = 2 * dr * dV + 2 * dV * dH + 4.0 * S * dr * dH;
      const double dw_bytes = 2 * dr * dV + 2 * dr * dH + (c > 0 ? 8.0 : 4.0) * dV * dH;
      if (p.backward_one_launch) {
        // both read the finished dlogits buffer: one launch on the dx GEMM's
        // tile shape, dx units first, handed out from a counter in the
        // control block
        const int shape = shape_for(h, p.tile_n_dx);
        const bool wide = shape == kShapeWide;
        const int64_t tile_cols = wide ? 2 * kBN : kBN;
        const int slots_max = wide ? h->wide_clusters : h->pair_clusters;
        DualMaps maps;
        maps.a[0] = mZ_k;
        maps.b[0] = mW_mn;
        maps.o[0] = mDx;
        maps.a[1] = mZ_mn;
        maps.b[1] = mX_mn;
        maps.o[1] = mDw;
        DualArgs da;
        da.p[0] = b;
        da.p[1] = d;
        da.p[0].num_m = static_cast<int>(cdiv(rows, 2 * kBM));
        da.p[1].num_m = static_cast<int>(cdiv(V, 2 * kBM));
        da.p[0].num_n = da.p[1].num_n = static_cast<int>(cdiv(H, tile_cols));
        da.units0 = da.p[0].num_m * da.p[0].num_n * da.p[0].num_s;
        da.p[0].group_m = group_for(h, shape, da.p[0].num_m, da.p[0].num_n, da.p[0].num_s,
                                    std::min(da.units0, slots_max));
        // the counter (cleared by count_valid) runs on across the call's launches
        da.sched_ctr = reinterpret_cast<int32_t*>(ctrl + kCtrlSched);
        da.sched_base = sched_claims;
        const int units = da.units0 + da.p[1].num_m * da.p[1].num_n;
        const int pairs = std::min(units, slots_max);
        FLCE_LAUNCH(FLCE_K_GEMM_DX_DW, 4 * dr * dV * dH, dx_bytes + dw_bytes,
                    wide ? launch_umma_wide_dual(maps, da, pairs, s)
                         : launch_umma_pair_dual(maps, da, pairs, s));
        sched_claims += units + pairs;
      } else if (overlap_dw) {
        // the dx GEMM fills less than kOverlapWaves waves of the GPU: the dW
        // GEMM runs beside it on the side stream (both only read the finished
        // buffer); the next chunk's logits GEMM waits for it before it
        // overwrites the buffer, and the call's end joins the side stream
        e = cudaEventRecord(h->slab_ready, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side_stream, h->slab_ready, 0);
        if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "dW fork: %s", cudaGetErrorString(e));
        {
          const cudaStream_t s = h->side_stream;  // the launch and its timing events go there
          FLCE_LAUNCH(FLCE_K_GEMM_DW, 2 * dr * dV * dH, dw_bytes,
                      launch_gemm(h, shape_for(h, p.tile_n_dw), kUmmaDw, mZ_mn, mX_mn, mDw, d, V, s));
        }
        e = cudaEventRecord(h->slab_freed, h->side_stream);
        if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "dW join: %s", cudaGetErrorString(e));
        side_pending = true;
        FLCE_LAUNCH(FLCE_K_GEMM_DX, 2 * dr * dV * dH, dx_bytes,
                    launch_gemm(h, shape_for(h, p.tile_n_dx), kUmmaDxF32, mZ_k, mW_mn, mDx, b, rows, s));
      } else {
        FLCE_LAUNCH(FLCE_K_GEMM_DX, 2 * dr * dV * dH, dx_bytes,
                    launch_gemm(h, shape_for(h, p.tile_n_dx), kUmmaDxF32, mZ_k, mW_mn, mDx, b, rows, s));
        FLCE_LAUNCH(FLCE_K_GEMM_DW, 2 * dr * dV * dH, dw_bytes,
                    launch_gemm(h, shape_for(h, p.tile_n_dw), kUmmaDw, mZ_mn, mX_mn, mDw, d, V, s));
      }
      // the last chunk's reduction also takes the loss reduction, unless dW
      // work on the side stream (which may record an error) is still to join
      const bool finish = c == p.num_chunks - 1 && !side_pending;
      FLCE_LAUNCH(FLCE_K_DX_REDUCE, 0.0, 4.0 * S * dr * dH + 4 * dr * dH + (finish ? 4.0 * N : 0.0),
                  launch_dx_reduce(dxpart, S, C * H, rows, H, static_cast<const __nv_bfloat16*>(W), V,
                                   t + off, ignore_index, ctrl, dcorr, dxb + off * H, s,
                                   finish ? token_loss : nullptr, N, dres ? 1 : 0,
                                   dres ? dres->loss : nullptr, dres ? dres->n_valid : nullptr));
      loss_done = finish;
    }
  }
  if (side_pending) {
    // the call ends on its stream only once the side stream's dW GEMMs are
    // done; the loss reduction below reads the error word they may have set
    side_pending = false;
    e = cudaStreamWaitEvent(s, h->slab_freed, 0);
    if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "slab join: %s", cudaGetErrorString(e));
  }
  if (!loss_done)
    FLCE_LAUNCH(FLCE_K_LOSS_FINALIZE, 0.0, 4.0 * N,
                launch_loss_finalize(token_loss, N, ctrl, dres ? 1 : 0, dres ? dres->loss : nullptr,
                                     dres ? dres->n_valid : nullptr, s));
  *ctrl_out = ctrl;
  return FLCE_OK;
}

flce_status run_fb(flce_handle_t h, const void* x, const void* W, const int64_t* t, int64_t N,
                   int64_t H, int64_t V, int64_t ignore_index, int64_t chunk, float* loss, void* dx,
                   float* dW, cudaStream_t s) {
  if (!loss) return fail(h, FLCE_ERR_INVALID_ARG, "null pointer argument");
  uint32_t* ctrl = nullptr;
  const flce_status st = enqueue_fb(h, x, W, t, N, H, V, ignore_index, chunk, dx, dW, s, &ctrl);
  if (st != FLCE_OK) return st;
  return read_back(h, ctrl, s, loss);
}

}  // namespace

// ================================================================== C ABI

extern "C" {

int32_t flce_abi_version(void) { return FLCE_ABI_VERSION; }

const char* flce_status_string(flce_status s) {
  switch (s) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED";
    case FLCE_ERR_BUDGET: return "FLCE_ERR_BUDGET";
    case FLCE_ERR_BAD_TARGET: return "FLCE_ERR_BAD_TARGET";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
  }
  return "FLCE_ERR_UNKNOWN";
}

const char* flce_kernel_name(int32_t kind) {
  switch (kind) {
    case FLCE_K_COUNT_VALID: return "count_valid";
    case FLCE_K_GEMM_LOGITS: return "gemm_logits_lse";
    case FLCE_K_LSE_COMBINE: return "lse_combine";
    case FLCE_K_DLOGITS: return "dlogits_inplace";
    case FLCE_K_GEMM_DLOGITS: return "gemm_dlogits_recompute";
    case FLCE_K_GEMM_DX: return "gemm_dx";
    case FLCE_K_DX_REDUCE: return "dx_split_reduce";
    case FLCE_K_GEMM_DW: return "gemm_dw";
    case FLCE_K_LOSS_FINALIZE: return "loss_finalize";
    case FLCE_K_SIMT_GEMM: return "simt_gemm_f32";
    case FLCE_K_SIMT_TILE_STATS: return "simt_tile_stats_f32";
    case FLCE_K_GEMM_DX_DW: return "gemm_dx_dw";
    case FLCE_K_DEVICE_RESULT: return "device_result";
    case FLCE_K_COMBINE_DLOGITS: return "combine_dlogits";
    case FLCE_K_H2D_COPY: return "h2d_copy";
    default: return "?";
  }
}

flce_status flce_make_plan(const flce_config* cfg, int64_t N, int64_t H, int64_t V, int64_t chunk,
                           int32_t num_sms, flce_plan* out) {
  std::string why;
  return plan_impl(cfg, N, H, V, chunk, num_sms, out, &why);
}

flce_status flce_create(flce_handle_t* out, const flce_config* cfg) {
  if (!out || !cfg) return FLCE_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->dtype != FLCE_DTYPE_BF16 && cfg->dtype != FLCE_DTYPE_FP32) return FLCE_ERR_UNSUPPORTED;
  if (cfg->dlogits_mode < FLCE_DLOGITS_AUTO || cfg->dlogits_mode > FLCE_DLOGITS_SLABS ||
      !valid_cta_mode(cfg->cta_pair))
    return FLCE_ERR_INVALID_ARG;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    return FLCE_ERR_UNSUPPORTED;
  }
  if (cfg->device < 0 || cfg->device >= count) return FLCE_ERR_INVALID_ARG;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return FLCE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return FLCE_ERR_UNSUPPORTED;
  if (prop.sharedMemPerBlockOptin < static_cast<size_t>(umma_smem_bytes())) return FLCE_ERR_UNSUPPORTED;
  flce_handle_t h = new flce_handle_s();
  h->cfg = *cfg;
  h->device = cfg->device;
  h->num_sms = prop.multiProcessorCount;
  h->timeout_ns = static_cast<uint64_t>(cfg->timeout_ms > 0 ? cfg->timeout_ms : 2000) * 1000000ull;
  DeviceGuard g(h->device);
  if (cfg->dtype == FLCE_DTYPE_BF16) {
    const int mode = cfg->cta_pair;
    if (mode == FLCE_CTA_AUTO || mode == FLCE_CTA_WIDE) h->wide_clusters = umma_wide_max_clusters();
    if (mode == FLCE_CTA_AUTO || mode == FLCE_CTA_PAIR) h->pair_clusters = umma_pair_max_clusters();
    if ((mode == FLCE_CTA_WIDE && h->wide_clusters <= 0) || (mode == FLCE_CTA_PAIR && h->pair_clusters <= 0)) {
      delete h;
      return FLCE_ERR_UNSUPPORTED;
    }
    if (mode == FLCE_CTA_AUTO && h->wide_clusters > 0 && h->pair_clusters > 0) {
      h->shape = kShapeWide;   // per GEMM, the plan's choice of wide or pair
    } else {
      h->shape = (mode == FLCE_CTA_AUTO || mode == FLCE_CTA_WIDE) && h->wide_clusters > 0 ? kShapeWide
                 : (mode == FLCE_CTA_AUTO || mode == FLCE_CTA_PAIR) && h->pair_clusters > 0 ? kShapePair
                                                                                          : kShapeSingle;
      // the handle's plans follow the one tile shape it actually runs
      h->cfg.cta_pair = h->shape == kShapeWide   ? FLCE_CTA_WIDE
                        : h->shape == kShapePair ? FLCE_CTA_PAIR
                                                 : FLCE_CTA_SINGLE;
    }
  }
  if (cudaMallocHost(&h->host_ctrl, kCtrlWords * 4) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return FLCE_ERR_CUDA;
  }
  *out = h;
  return FLCE_OK;
}

void flce_destroy(flce_handle_t h) {
  if (!h) return;
  {
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    for (auto& e : h->prof.pool) {
      cudaEventDestroy(e.start);
      cudaEventDestroy(e.stop);
    }
    if (h->ws && !h->ws_external) cudaFree(h->ws);
    if (h->stage) cudaFree(h->stage);
    if (h->host_ctrl) cudaFreeHost(h->host_ctrl);
    for (auto& sl : h->slots) {
      if (sl.stage) cudaFree(sl.stage);
      if (sl.host) cudaFreeHost(sl.host);
      if (sl.copied) cudaEventDestroy(sl.copied);
      if (sl.freed) cudaEventDestroy(sl.freed);
      if (sl.done) cudaEventDestroy(sl.done);
    }
    if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
    if (h->side_stream) cudaStreamDestroy(h->side_stream);
    if (h->slab_ready) cudaEventDestroy(h->slab_ready);
    if (h->slab_freed) cudaEventDestroy(h->slab_freed);
  }
  delete h;
}

flce_status flce_set_workspace(flce_handle_t h, void* dev_ptr, uint64_t bytes) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  if (dev_ptr && (reinterpret_cast<uintptr_t>(dev_ptr) & (kAlign - 1)) != 0)
    return fail(h, FLCE_ERR_INVALID_ARG, "workspace must be %llu-byte aligned",
                static_cast<unsigned long long>(kAlign));
  if (h->ws && !h->ws_external) {
    cudaDeviceSynchronize();
    cudaFree(h->ws);
  }
  h->ws = dev_ptr;
  h->ws_bytes = dev_ptr ? bytes : 0;
  h->ws_external = dev_ptr != nullptr;
  h->ws_fresh = true;
  return FLCE_OK;
}

flce_status flce_forward_backward(flce_handle_t h, const void* x, const void* W, const int64_t* t,
                                  int64_t N, int64_t H, int64_t V, int64_t ignore_index,
                                  int64_t chunk, float* loss, void* dx, float* dW, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  DeviceGuard g(h->device);
  return run_fb(h, x, W, t, N, H, V, ignore_index, chunk, loss, dx, dW,
                static_cast<cudaStream_t>(stream));
}

flce_status flce_forward_backward_async(flce_handle_t h, const void* x, const void* W,
                                        const int64_t* t, int64_t N, int64_t H, int64_t V,
                                        int64_t ignore_index, int64_t chunk, float* loss_dev,
                                        int32_t* n_valid_dev, void* dx, float* dW, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  if ((reinterpret_cast<uintptr_t>(loss_dev) & 3u) || (reinterpret_cast<uintptr_t>(n_valid_dev) & 3u))
    return fail(h, FLCE_ERR_INVALID_ARG, "loss_dev and n_valid_dev must be 4-byte aligned");
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* ctrl = nullptr;
  DeviceResult dres;
  dres.loss = loss_dev;
  dres.n_valid = n_valid_dev;
  return enqueue_fb(h, x, W, t, N, H, V, ignore_index, chunk, dx, dW, s, &ctrl, nullptr, &dres);
}

flce_status flce_async_status(flce_handle_t h, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "async status: %s", cudaGetErrorString(e));
  if (!h->ws || h->ws_fresh) return FLCE_OK;
  uint32_t* sticky = static_cast<uint32_t*>(h->ws) + kCtrlSticky;  // the control block leads the workspace
  uint32_t code = 0;
  e = cudaMemcpy(&code, sticky, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && code != 0) e = cudaMemset(sticky, 0, 4);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "async status: %s", cudaGetErrorString(e));
  return device_status(h, code);
}

flce_status flce_count_valid(flce_handle_t h, const int64_t* t, int64_t N, int64_t ignore_index,
                             int32_t* n_valid_dev, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  if (!n_valid_dev || (N > 0 && !t) || N < 0 || N > kMaxDim)
    return fail(h, FLCE_ERR_INVALID_ARG, "null pointer or bad size");
  if ((reinterpret_cast<uintptr_t>(t) & 7u) || (reinterpret_cast<uintptr_t>(n_valid_dev) & 3u))
    return fail(h, FLCE_ERR_INVALID_ARG, "t must be 8-byte and n_valid_dev 4-byte aligned");
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FLCE_LAUNCH(FLCE_K_COUNT_VALID, 0.0, 8.0 * N + 4.0, launch_count_only(t, N, ignore_index, n_valid_dev, s));
  return FLCE_OK;
}

flce_status flce_forward_backward_shard(flce_handle_t h, const void* x, const void* W,
                                        const int64_t* t, int64_t N, int64_t H, int64_t V,
                                        int64_t ignore_index, int64_t chunk,
                                        const int32_t* n_valid_total_dev, float* loss_dev,
                                        void* dx, float* dW, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  if (!n_valid_total_dev || (reinterpret_cast<uintptr_t>(n_valid_total_dev) & 3u) ||
      (reinterpret_cast<uintptr_t>(loss_dev) & 3u))
    return fail(h, FLCE_ERR_INVALID_ARG, "n_valid_total_dev (non-null) and loss_dev must be 4-byte aligned");
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* ctrl = nullptr;
  DeviceResult dres;
  dres.loss = loss_dev;
  return enqueue_fb(h, x, W, t, N, H, V, ignore_index, chunk, dx, dW, s, &ctrl, n_valid_total_dev,
                    &dres);
}

flce_status flce_forward_backward_host(flce_handle_t h, const void* x_host, const void* W_host,
                                       const int64_t* t_host, int64_t N, int64_t H, int64_t V,
                                       int64_t ignore_index, int64_t chunk, float* loss, void* dx,
                                       float* dW, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  if (!x_host || !W_host || !t_host || N < 0 || H < 1 || V < 1)
    return fail(h, FLCE_ERR_INVALID_ARG, "null host pointer or bad size");
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Staged in;
  flce_status st = stage_inputs(h, &h->stage, &h->stage_bytes, x_host, W_host, t_host, N, H, V, s, &in);
  if (st != FLCE_OK) return st;
  return run_fb(h, in.x, in.W, in.t, N, H, V, ignore_index, chunk, loss, dx, dW, s);
}

flce_status flce_submit_host(flce_handle_t h, const void* x_host, const void* W_host,
                             const int64_t* t_host, int64_t N, int64_t H, int64_t V,
                             int64_t ignore_index, int64_t chunk, void* dx, float* dW, void* stream,
                             uint64_t* ticket) {
  if (!h || !ticket) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  *ticket = 0;
  if (!x_host || !W_host || !t_host || N < 0 || H < 1 || V < 1)
    return fail(h, FLCE_ERR_INVALID_ARG, "null host pointer or bad size");
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  flce_handle_s::Slot& sl = h->slots[h->next_ticket & 1];
  if (sl.pending)
    return fail(h, FLCE_ERR_INVALID_ARG, "two submissions are outstanding: wait for ticket %llu first",
                static_cast<unsigned long long>(sl.ticket));
  cudaError_t e = cudaSuccess;
  if (!h->copy_stream) e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess && !sl.copied) e = cudaEventCreateWithFlags(&sl.copied, cudaEventDisableTiming);
  if (e == cudaSuccess && !sl.freed) e = cudaEventCreateWithFlags(&sl.freed, cudaEventDisableTiming);
  if (e == cudaSuccess && !sl.done) e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming);
  if (e == cudaSuccess && !sl.host)
    e = cudaHostAlloc(reinterpret_cast<void**>(&sl.host), kCtrlWords * 4, cudaHostAllocDefault);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "submit set-up: %s", cudaGetErrorString(e));
  // the copies wait only for the call that last read this slot, so they
  // overlap the call running on the other slot
  e = cudaStreamWaitEvent(h->copy_stream, sl.freed, 0);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "submit: %s", cudaGetErrorString(e));
  Staged in;
  flce_status st =
      stage_inputs(h, &sl.stage, &sl.bytes, x_host, W_host, t_host, N, H, V, h->copy_stream, &in);
  if (st != FLCE_OK) return st;
  e = cudaEventRecord(sl.copied, h->copy_stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, sl.copied, 0);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "submit: %s", cudaGetErrorString(e));
  uint32_t* ctrl = nullptr;
  st = enqueue_fb(h, in.x, in.W, in.t, N, H, V, ignore_index, chunk, dx, dW, s, &ctrl);
  if (st != FLCE_OK) return st;
  e = cudaEventRecord(sl.freed, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(sl.host, ctrl, kCtrlWords * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaEventRecord(sl.done, s);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "submit: %s", cudaGetErrorString(e));
  sl.pending = true;
  sl.ticket = h->next_ticket++;
  *ticket = sl.ticket;
  return FLCE_OK;
}

flce_status flce_wait(flce_handle_t h, uint64_t ticket, float* loss) {
  if (!h || !loss) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  flce_handle_s::Slot& sl = h->slots[ticket & 1];
  if (ticket == 0 || !sl.pending || sl.ticket != ticket)
    return fail(h, FLCE_ERR_INVALID_ARG, "ticket %llu is not outstanding",
                static_cast<unsigned long long>(ticket));
  DeviceGuard g(h->device);
  const cudaError_t e = cudaEventSynchronize(sl.done);
  sl.pending = false;
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "wait: %s", cudaGetErrorString(e));
  return decode_ctrl(h, sl.host, loss);
}

flce_status flce_token_losses(flce_handle_t h, float* out, int64_t N, void* stream) {
  if (!h || !out) return FLCE_ERR_INVALID_ARG;
  if (!h->has_plan || N != h->last_N) return fail(h, FLCE_ERR_INVALID_ARG, "N differs from the last call");
  if (N == 0) return FLCE_OK;
  DeviceGuard g(h->device);
  const float* src = reinterpret_cast<const float*>(static_cast<uint8_t*>(h->ws) + h->token_loss_off);
  cudaError_t e = cudaMemcpyAsync(out, src, static_cast<size_t>(N) * 4, cudaMemcpyDeviceToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "%s", cudaGetErrorString(e));
  return FLCE_OK;
}

flce_status flce_last_plan(flce_handle_t h, flce_plan* out) {
  if (!h || !out || !h->has_plan) return FLCE_ERR_INVALID_ARG;
  *out = h->last_plan;
  return FLCE_OK;
}

flce_status flce_set_profiling(flce_handle_t h, int32_t enable) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->prof.enabled = enable != 0;
  return FLCE_OK;
}

flce_status flce_profile_read(flce_handle_t h, int32_t kind, flce_kernel_profile* out) {
  if (!h || !out || kind < 0 || kind >= FLCE_K_NUM_KINDS) return FLCE_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  prof_collect(h);
  *out = h->prof.totals[kind];
  return FLCE_OK;
}

void flce_profile_reset(flce_handle_t h) {
  if (!h) return;
  DeviceGuard g(h->device);
  prof_collect(h);
  std::memset(h->prof.totals, 0, sizeof(h->prof.totals));
}

int64_t flce_launch_count(flce_handle_t h) { return h ? h->launches : 0; }

uint64_t flce_workspace_bytes(flce_handle_t h, int64_t N, int64_t H, int64_t V, int64_t chunk) {
  if (!h) return 0;
  h->err.clear();
  flce_plan p;
  std::string why;
  if (plan_impl(&h->cfg, N, H, V, chunk, h->num_sms, &p, &why) != FLCE_OK) {
    h->err = why;
    return 0;
  }
  return p.workspace_bytes;
}

const char* flce_last_error(flce_handle_t h) { return h ? h->err.c_str() : "null handle"; }

flce_status flce_check_gemm(flce_handle_t h, int32_t a_mn_major, int32_t b_mn_major, const void* A,
                            const void* B, float* C, int64_t M, int64_t N, int64_t K, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  if (!A || !B || !C || M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return fail(h, FLCE_ERR_INVALID_ARG, "null pointer or bad size");
  const int64_t a_inner = a_mn_major ? M : K, b_inner = b_mn_major ? N : K;
  if (a_inner % 8 || b_inner % 8 || N % 4)
    return fail(h, FLCE_ERR_INVALID_ARG, "contiguous extents must be multiples of 8 (N of 4)");
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  flce_status st = ensure_workspace(h, kAlign);
  if (st != FLCE_OK) return st;
  uint32_t* ctrl = static_cast<uint32_t*>(h->ws);
  std::string why;
  CUtensorMap ma, mb, mc;
  bool ok = a_mn_major ? map_bf16_2d(&ma, A, M, K, M * 2, 64, 64, &why)
                       : map_bf16_2d(&ma, A, K, M, K * 2, 64, 128, &why);
  ok = ok && (b_mn_major ? map_bf16_2d(&mb, B, N, K, N * 2, 64, 64, &why)
                         : map_bf16_2d(&mb, B, K, N, K * 2, 64, h->shape == kShapeSingle ? 256 : 128, &why));
  ok = ok && map_f32_3d(&mc, C, N, M, 1, N * 4, static_cast<uint64_t>(M) * N * 4, &why);
  if (!ok) return fail(h, FLCE_ERR_INVALID_ARG, "%s", why.c_str());
  UmmaArgs a{};
  a.num_m = static_cast<int>(cdiv(M, kBM));
  a.num_n = static_cast<int>(cdiv(N, kBN));
  a.num_s = 1;
  a.kb_total = static_cast<int>(cdiv(K, kBK));
  a.kb_per_split = a.kb_total;
  a.rows = static_cast<int>(M);
  a.cols = static_cast<int>(N);
  a.ctrl = ctrl;
  a.timeout_ns = h->timeout_ns;
  const int kind = a_mn_major ? (b_mn_major ? kUmmaDw : kUmmaCheckMK) : (b_mn_major ? kUmmaDxF32 : kUmmaCheckKK);
  cudaError_t e = cudaMemsetAsync(ctrl, 0, kCtrlWords * 4, s);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "%s", cudaGetErrorString(e));
  const double flops = 2.0 * M * N * K;
  const int kkind = a_mn_major ? FLCE_K_GEMM_DW : (b_mn_major ? FLCE_K_GEMM_DX : FLCE_K_GEMM_LOGITS);
  FLCE_LAUNCH(kkind, flops, 2.0 * (M * K + N * K) + 4.0 * M * N,
              launch_gemm(h, h->shape, kind, ma, mb, mc, a, M, s));
  return read_back(h, ctrl, s, nullptr);
}

flce_status flce_check_wait_timeout(flce_handle_t h, uint32_t timeout_us, void* stream) {
  if (!h) return FLCE_ERR_INVALID_ARG;
  h->err.clear();
  DeviceGuard g(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  flce_status st = ensure_workspace(h, kAlign);
  if (st != FLCE_OK) return st;
  uint32_t* ctrl = static_cast<uint32_t*>(h->ws);
  cudaError_t e = cudaMemsetAsync(ctrl, 0, kCtrlWords * 4, s);
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "%s", cudaGetErrorString(e));
  e = launch_wait_check(ctrl, static_cast<uint64_t>(timeout_us) * 1000ull, s);
  ++h->launches;
  if (e != cudaSuccess) return fail(h, FLCE_ERR_CUDA, "%s", cudaGetErrorString(e));
  return read_back(h, ctrl, s, nullptr);
}

}  // extern "C"
