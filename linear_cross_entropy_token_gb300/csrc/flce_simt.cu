// fp32 path of fused linear cross-entropy on the CUDA cores.
//
// TF32 tensor cores cannot hold fp32 inputs to a 1e-5 gradient error, so
// fp32 x and W take these kernels: a strided fp32 GEMM (used for x_c·Wᵀ,
// dlogits·W and dlogitsᵀ·x_c) with a fixed-order split of the reduction, and
// the per-vocab-tile max / sum-exp of the stored fp32 logits. The rest of the
// fp32 path shares the row kernels of the bf16 path, and its chunk schedule is
// the same (the four steps of the FLCE page, "Fused Linear Cross-Entropy: LLM
// 학습 logits 메모리 병목 없애기", section "FLCE의 핵심 아이디어").
#include <algorithm>

#include "flce_internal.h"

namespace flce {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;
constexpr int kSimtThreads = 256;
constexpr int kLoads = kTK * kTM / kSimtThreads;  // operand elements per thread per k-tile (4)
static_assert(kTM == kTN, "the load mapping below assumes square tiles");

// Element e (0..1023) of a 64 x 16 operand tile, mapped so that consecutive
// threads walk the operand's unit-stride dimension: `outer` indexes the 64
// rows (m of A, n of B), `kk` the 16-deep k slice.
__device__ __forceinline__ void tile_coords(int e, bool k_unit, int& outer, int& kk) {
  if (k_unit) {
    kk = e % kTK;
    outer = e / kTK;
  } else {
    outer = e % kTM;
    kk = e / kTM;
  }
}

// C[m, n] (+)= sum_k A(m, k) B(k, n), A(m, k) = A[m*sam + k*sak],
// B(k, n) = B[k*sbk + n*sbn], over the k range of split blockIdx.z
// ([z*kps, min(K, (z+1)*kps))). With part == nullptr the block writes C
// (adding to it if accumulate); otherwise it writes its split's partial sums
// to part[z][m][n] (M x N, row-major) for simt_splitk_reduce_kernel.
// 256 threads, a 4 x 4 output block each; the next k-tile's operands are
// loaded into registers while the current one is multiplied.
__global__ void __launch_bounds__(kSimtThreads) simt_gemm_f32_kernel(
    const float* __restrict__ A, int64_t sam, int64_t sak, const float* __restrict__ B,
    int64_t sbk, int64_t sbn, float* __restrict__ C, int64_t ldc, int64_t M, int64_t N,
    int64_t K, int64_t kps, int accumulate, float* __restrict__ part) {
  __shared__ float As[kTK][kTM + 1];
  __shared__ float Bs[kTK][kTN + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTN;
  const int64_t kbeg = static_cast<int64_t>(blockIdx.z) * kps;
  const int64_t kend = min(K, kbeg + kps);
  const bool a_k_unit = sak == 1;
  const bool b_k_unit = sbk == 1 && sbn != 1;
  float ra[kLoads], rb[kLoads];
  auto fetch = [&](int64_t k0) {
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      int o, kk;
      tile_coords(threadIdx.x + q * kSimtThreads, a_k_unit, o, kk);
      const int64_t m = m0 + o, k = k0 + kk;
      ra[q] = (m < M && k < kend) ? A[m * sam + k * sak] : 0.f;
      tile_coords(threadIdx.x + q * kSimtThreads, b_k_unit, o, kk);
      const int64_t n = n0 + o;
      rb[q] = (n < N && k0 + kk < kend) ? B[(k0 + kk) * sbk + n * sbn] : 0.f;
    }
  };
  float acc[4][4] = {};
  if (kbeg < kend) fetch(kbeg);
  for (int64_t k0 = kbeg; k0 < kend; k0 += kTK) {
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      int o, kk;
      tile_coords(threadIdx.x + q * kSimtThreads, a_k_unit, o, kk);
      As[kk][o] = ra[q];
      tile_coords(threadIdx.x + q * kSimtThreads, b_k_unit, o, kk);
      Bs[kk][o] = rb[q];
    }
    __syncthreads();
    if (k0 + kTK < kend) fetch(k0 + kTK);
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  // thread (tx, ty) holds rows ty*4 + i and columns tx + 16*j: a warp's stores
  // of one (i, j) cover 16 consecutive columns of two rows
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx + 16 * j;
      if (n >= N) continue;
      if (part) {
        part[(static_cast<int64_t>(blockIdx.z) * M + m) * N + n] = acc[i][j];
      } else {
        float* c = C + m * ldc + n;
        *c = accumulate ? (*c + acc[i][j]) : acc[i][j];
      }
    }
  }
}

// C[m, n] (+)= sum over the splits, in split order, of part[s][m][n].
__global__ void __launch_bounds__(256) simt_splitk_reduce_kernel(
    const float* __restrict__ part, int splits, int64_t M, int64_t N, float* __restrict__ C,
    int64_t ldc, int accumulate) {
  const int64_t MN = M * N;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < MN;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    // eight splits' loads in flight at a time, added in split order
    float v = part[e];
    int s = 1;
    for (; s + 8 <= splits; s += 8) {
      float q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = part[(s + j) * MN + e];
#pragma unroll
      for (int j = 0; j < 8; ++j) v += q[j];
    }
    for (; s < splits; ++s) v += part[s * MN + e];
    const int64_t m = e / N, n = e - m * N;
    float* c = C + m * ldc + n;
    *c = accumulate ? (*c + v) : v;
  }
}

// One warp per (token row, vocab tile of kVocabTile columns): m = max z,
// l = sum exp(z - m), and z_t when the target falls in the tile; each lane
// takes kVocabTile / 32 columns. The
// buffer's column 0 is vocabulary column col_base; partials rows are
// part_stride apart.
__global__ void __launch_bounds__(256) simt_tile_stats_kernel(
    const float* __restrict__ logits, int64_t ldv, int rows, int64_t V, int vocab_tiles,
    int part_stride, int64_t col_base, const int64_t* __restrict__ t, int64_t ignore_index,
    float2* __restrict__ partials, float* __restrict__ zt) {
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= rows * vocab_tiles) return;
  const int r = w / vocab_tiles, vt = w - r * vocab_tiles;
  const float* row = logits + static_cast<size_t>(r) * ldv;
  const int64_t tg = t[r];
  constexpr int kPerLane = kVocabTile / 32;
  float z[kPerLane];
  float m = -INFINITY;
#pragma unroll
  for (int q = 0; q < kPerLane; ++q) {
    const int64_t j = static_cast<int64_t>(vt) * kVocabTile + q * 32 + lane;
    z[q] = j < V ? row[j] : -INFINITY;
    m = fmaxf(m, z[q]);
    if (j < V && tg != ignore_index && tg - col_base == j) zt[r] = z[q];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
#pragma unroll
  for (int q = 0; q < kPerLane; ++q) l += z[q] == -INFINITY ? 0.f : expf(z[q] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) partials[static_cast<size_t>(r) * part_stride + vt] = make_float2(m, l);
}

}  // namespace

int simt_split_k(int64_t M, int64_t N, int64_t K, int num_sms) {
  // enough blocks for about two per SM, each split at least 128 deep
  const int64_t tiles = ((M + kTM - 1) / kTM) * ((N + kTN - 1) / kTN);
  int64_t s = (2 * static_cast<int64_t>(num_sms) + tiles - 1) / tiles;
  s = std::min<int64_t>(s, std::max<int64_t>(1, K / 128));
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(s, kMaxSimtSplits)));
}

cudaError_t launch_simt_gemm_f32(const float* A, int64_t sam, int64_t sak, const float* B,
                                 int64_t sbk, int64_t sbn, float* C, int64_t ldc, int64_t M,
                                 int64_t N, int64_t K, int accumulate, int splits, float* part,
                                 cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  // k per split, a multiple of the k-tile; the last split may be shorter
  int64_t kps = (K + splits - 1) / std::max(1, splits);
  kps = std::max<int64_t>(kTK, (kps + kTK - 1) / kTK * kTK);
  const int S = static_cast<int>(std::max<int64_t>(1, (K + kps - 1) / kps));
  dim3 grid(static_cast<unsigned>((N + kTN - 1) / kTN), static_cast<unsigned>((M + kTM - 1) / kTM),
            static_cast<unsigned>(S));
  if (S == 1 || !part) {
    grid.z = 1;
    simt_gemm_f32_kernel<<<grid, kSimtThreads, 0, s>>>(A, sam, sak, B, sbk, sbn, C, ldc, M, N, K,
                                                       std::max<int64_t>(K, 1), accumulate, nullptr);
    return cudaGetLastError();
  }
  simt_gemm_f32_kernel<<<grid, kSimtThreads, 0, s>>>(A, sam, sak, B, sbk, sbn, C, ldc, M, N, K, kps,
                                                     accumulate, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t MN = M * N;
  const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((MN + 255) / 256, 4096));
  simt_splitk_reduce_kernel<<<blocks, 256, 0, s>>>(part, S, M, N, C, ldc, accumulate);
  return cudaGetLastError();
}

cudaError_t launch_simt_tile_stats(const float* logits, int64_t ldv, int rows, int64_t V,
                                   int vocab_tiles, int part_stride, int64_t col_base,
                                   const int64_t* t_chunk, int64_t ignore_index, float2* partials,
                                   float* zt, cudaStream_t s) {
  const int64_t warps = static_cast<int64_t>(rows) * vocab_tiles;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  simt_tile_stats_kernel<<<blocks, 256, 0, s>>>(logits, ldv, rows, V, vocab_tiles, part_stride,
                                                col_base, t_chunk, ignore_index, partials, zt);
  return cudaGetLastError();
}

}  // namespace flce
