// Internal declarations shared by the kernels and the host runtime.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flce {

// Control block in device memory, one per handle workspace (uint32 words).
enum CtrlWord : int {
  kCtrlError = 0,    // first error recorded by a kernel (flce_status numbering)
  kCtrlNValid = 1,   // number of non-ignored tokens
  kCtrlLoss = 2,     // fp32 bits of the mean loss
  kCtrlSched = 3,    // work-unit counter of a dynamically scheduled launch
  kCtrlNValidLocal = 4,  // this call's own non-ignored tokens (kCtrlNValid may be a
                         // token-sharded batch's total)
  kCtrlSticky = 15,  // first error of the device-result calls, kept across calls
  kCtrlWords = 16
};

// Tile shape of the tcgen05 GEMMs: 128 x 256 output tile per CTA, 64-deep
// k-blocks (one 128-byte swizzle row of bf16), 4-stage TMA pipeline.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
// Vocabulary columns per log-sum-exp partial (running max, sum of exp): one
// 64-column group of an output tile. The bf16 chunk buffer stores each group
// relative to its own max.
constexpr int kVocabTile = 64;

// Epilogues of the tcgen05 GEMM
enum Epilogue : int {
  kEpiLse = 0,       // online max / sum-exp + target gather (+ bf16 logits store)
  kEpiBf16 = 1,      // bf16 store
  kEpiF32 = 2,       // fp32 store or reduce-add (3-D map: col, row, split)
  kEpiDlogits = 3    // (exp(z - lse) - onehot) / n_valid, bf16 store
};

// The kernel instantiations the runtime launches
enum UmmaKind : int {
  kUmmaLogits = 0,     // A = x_c (K-major), B = W (K-major), kEpiLse
  kUmmaDlogits = 1,    // A = x_c, B = W, kEpiDlogits
  kUmmaDxBf16 = 2,     // A = dlogits (K-major), B = W (MN-major), kEpiBf16
  kUmmaDxF32 = 3,      // same operands, fp32 split partials
  kUmmaDw = 4,         // A = dlogitsᵀ (MN-major), B = x_c (MN-major), kEpiF32
  kUmmaCheckKK = 5,    // both K-major, fp32 out (tests)
  kUmmaCheckMK = 6     // A MN-major, B K-major, fp32 out (tests)
};

struct UmmaArgs {
  int32_t num_m, num_n, num_s;   // output tiles along M, N and splits of K
  int32_t kb_total;              // 64-deep k-blocks over the whole K
  int32_t kb_per_split;          // k-blocks per split
  int32_t raster;                // 0: m fastest; 1: n fastest; 2: groups of group_m rows of
                                 // tiles, m fastest inside a group (then the other, then s)
  int32_t rows;                  // valid output rows (M extent)
  int32_t cols;                  // valid output columns (N extent; V for the logits GEMM)
  int32_t vocab_tiles;           // log-sum-exp partials per token
  int32_t reduce_add;            // kEpiF32: 1 = add into the output instead of storing
  int32_t store_logits;          // kEpiLse: 1 = also store bf16 logits
  int32_t group_m;               // raster 2: tile rows per group
  int64_t ignore_index;
  int64_t col_base;              // kEpiLse / kEpiDlogits: vocabulary index of output column 0
  const int64_t* targets;        // targets of this chunk's tokens
  float2* partials;              // [rows][vocab_tiles] (max, sum of exp) per 64-column group
  float* zt;                     // [rows] fp32 target logit
  const float* lse;              // [rows] log-sum-exp (kEpiDlogits)
  float* dcorr;                  // [rows] rounding error of the target entry (kEpiDlogits)
  uint32_t* ctrl;                // control block
  uint64_t timeout_ns;           // limit of every mbarrier wait
};

// flce_umma.cu
int umma_smem_bytes();
cudaError_t launch_umma(int kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                        const UmmaArgs& args, int grid, cudaStream_t s);
// CTA-pair kernels: 256 x 256 tiles; num_m counts 256-row tiles; B maps of
// K-major operands use a 64 x 128 box (each CTA loads half of B)
cudaError_t launch_umma_pair(int kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                             const UmmaArgs& args, int pairs, cudaStream_t s);
int umma_pair_max_clusters();
// Wide CTA-pair kernels: 256 x 512 tiles (two MMAs per k-step sharing A);
// num_m counts 256-row tiles, num_n 512-column tiles; B maps of K-major
// operands use a 64 x 128 box, as for pairs
cudaError_t launch_umma_wide(int kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                             const UmmaArgs& args, int pairs, cudaStream_t s);
int umma_wide_max_clusters();

// The dx and dW GEMMs of one chunk in one CTA-pair launch: problem 0 = dx
// (A K-major), problem 1 = dW (A MN-major); B MN-major, fp32 epilogue in both.
// The dx units come first in the schedule.
struct DualMaps {
  CUtensorMap a[2], b[2], o[2];
};
struct DualArgs {
  UmmaArgs p[2];
  int32_t units0;       // work units of problem 0
  int32_t sched_base;   // the counter's value when this launch starts
  int32_t* sched_ctr;   // claims so far: each pair claims its units and then one
                        // past the last, so a launch of U units on P pairs leaves
                        // it at sched_base + U + P for the next launch of the call
};
cudaError_t launch_umma_pair_dual(const DualMaps& maps, const DualArgs& args, int pairs,
                                  cudaStream_t s);
// The same on wide tiles (256 x 512; num_n counts 512-column tiles), launched
// on at most umma_wide_max_clusters() pairs.
cudaError_t launch_umma_wide_dual(const DualMaps& maps, const DualArgs& args, int pairs,
                                  cudaStream_t s);
cudaError_t launch_wait_check(uint32_t* ctrl, uint64_t timeout_ns, cudaStream_t s);

// flce_rows.cu
// nv_total: device divisor of a token-sharded batch, or null (divide by the
// call's own count)
cudaError_t launch_count_valid(const int64_t* t, int64_t N, int64_t V, int64_t ignore_index,
                               const int32_t* nv_total, uint32_t* ctrl, cudaStream_t s);
cudaError_t launch_count_only(const int64_t* t, int64_t N, int64_t ignore_index, int32_t* out,
                              cudaStream_t s);
cudaError_t launch_lse_combine(const float2* partials, int vocab_tiles, const float* zt,
                               const int64_t* t_chunk, int rows, int64_t ignore_index, float* lse,
                               float* token_loss_chunk, cudaStream_t s);
cudaError_t launch_dlogits_bf16(__nv_bfloat16* buf, int64_t ldv, int rows, int64_t V,
                                const float2* partials, int vocab_tiles, const float* lse,
                                const int64_t* t_chunk, int64_t ignore_index,
                                const uint32_t* ctrl, float* dcorr, cudaStream_t s);
// buf's column 0 is vocabulary column col_base (a slab of the vocabulary)
cudaError_t launch_dlogits_f32(float* buf, int64_t ldv, int rows, int64_t V, int64_t col_base,
                               const float* lse, const int64_t* t_chunk, int64_t ignore_index,
                               const uint32_t* ctrl, cudaStream_t s);
// token_loss non-null: this is the call's last dx reduction, and it also
// runs the loss reduction of launch_loss_finalize (same arguments)
cudaError_t launch_dx_reduce(const float* partials, int splits, int64_t split_stride, int rows,
                             int64_t H, const __nv_bfloat16* W, int64_t V, const int64_t* t_chunk,
                             int64_t ignore_index, uint32_t* ctrl, const float* dcorr,
                             __nv_bfloat16* dx, cudaStream_t s, const float* token_loss = nullptr,
                             int64_t N = 0, int result = 0, float* loss_dev = nullptr,
                             int32_t* n_valid_dev = nullptr);
// The log-sum-exp combine and the in-place dlogits pass in one launch (one
// block per token row), for buffers of at most combine_dlogits_max_cols()
// columns (ldv); arguments as for the two launches it replaces.
cudaError_t launch_combine_dlogits_bf16(__nv_bfloat16* buf, int64_t ldv, int rows, int64_t V,
                                        const float2* partials, int vocab_tiles, const float* zt,
                                        const int64_t* t_chunk, int64_t ignore_index,
                                        const uint32_t* ctrl, float* lse, float* token_loss_chunk,
                                        float* dcorr, cudaStream_t s);
int64_t combine_dlogits_max_cols();
// fp32 path, in place: per token row of the chunk's fp32 logits, the
// log-sum-exp, token loss and (softmax - onehot)/n_valid in one launch (a
// block per row); replaces the tile statistics, combine and dlogits passes
cudaError_t launch_rows_f32(float* buf, int64_t ldv, int rows, int64_t V, const int64_t* t_chunk,
                            int64_t ignore_index, const uint32_t* ctrl, float* lse,
                            float* token_loss_chunk, cudaStream_t s);
cudaError_t launch_device_result(uint32_t* ctrl, float* loss_dev, int32_t* n_valid_dev, cudaStream_t s);
// result != 0: also write the sync-free entry points' device result (loss,
// NaN after a recorded error; n_valid; the sticky error word)
cudaError_t launch_loss_finalize(const float* token_loss, int64_t N, uint32_t* ctrl, int result,
                                 float* loss_dev, int32_t* n_valid_dev, cudaStream_t s);

// flce_simt.cu (fp32 path)
// C (+)= A·B over K with strided operands. splits > 1 with part != null
// splits the reduction over that many blocks along K, writing partials to part
// (splits x M x N fp32), and a second launch adds them in split order.
constexpr int kMaxSimtSplits = 64;
int simt_split_k(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_simt_gemm_f32(const float* A, int64_t sam, int64_t sak, const float* B,
                                 int64_t sbk, int64_t sbn, float* C, int64_t ldc, int64_t M,
                                 int64_t N, int64_t K, int accumulate, int splits, float* part,
                                 cudaStream_t s);
// vocab_tiles tiles of the buffer's V columns; the buffer's column 0 is
// vocabulary column col_base, and partials rows are part_stride apart
cudaError_t launch_simt_tile_stats(const float* logits, int64_t ldv, int rows, int64_t V,
                                   int vocab_tiles, int part_stride, int64_t col_base,
                                   const int64_t* t_chunk, int64_t ignore_index, float2* partials,
                                   float* zt, cudaStream_t s);

}  // namespace flce
