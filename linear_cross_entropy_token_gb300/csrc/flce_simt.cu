// fp32 path of fused linear cross-entropy on the CUDA cores.
//
// TF32 tensor cores cannot hold fp32 inputs to a 1e-5 gradient error, so
// fp32 x and W take these kernels: a strided fp32 GEMM (used for x_c·Wᵀ,
// dlogits·W and dlogitsᵀ·x_c) and the per-vocab-tile max / sum-exp of the
// stored fp32 logits. The rest of the fp32 path shares the row kernels of the
// bf16 path, and its chunk schedule is the same (the four steps of the FLCE
// page, "Fused Linear Cross-Entropy: LLM 학습 logits 메모리 병목 없애기",
// section "FLCE의 핵심 아이디어").
#include "flce_internal.h"

namespace flce {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;

// C[m, n] (+)= sum_k A(m, k) B(k, n), A(m, k) = A[m*sam + k*sak],
// B(k, n) = B[k*sbk + n*sbn]; 256 threads, 4 x 4 outputs each.
__global__ void __launch_bounds__(256) simt_gemm_f32_kernel(
    const float* __restrict__ A, int64_t sam, int64_t sak, const float* __restrict__ B,
    int64_t sbk, int64_t sbn, float* __restrict__ C, int64_t ldc, int64_t M, int64_t N,
    int64_t K, int accumulate) {
  __shared__ float As[kTK][kTM + 1];
  __shared__ float Bs[kTK][kTN + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTN;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += kTK) {
    for (int i = threadIdx.x; i < kTK * kTM; i += 256) {
      const int kk = i / kTM, mm = i % kTM;
      const int64_t m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < K) ? A[m * sam + k * sak] : 0.f;
    }
    for (int i = threadIdx.x; i < kTK * kTN; i += 256) {
      const int kk = i / kTN, nn = i % kTN;
      const int64_t n = n0 + nn, k = k0 + kk;
      Bs[kk][nn] = (n < N && k < K) ? B[k * sbk + n * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float* c = C + m * ldc + n;
      *c = accumulate ? (*c + acc[i][j]) : acc[i][j];
    }
  }
}

// One block per (token row, vocab tile of 256): m = max z, l = sum exp(z - m),
// and z_t when the target falls in the tile. The buffer's column 0 is
// vocabulary column col_base; partials rows are part_stride apart.
__global__ void __launch_bounds__(256) simt_tile_stats_kernel(
    const float* __restrict__ logits, int64_t ldv, int64_t V, int part_stride, int64_t col_base,
    const int64_t* __restrict__ t, int64_t ignore_index, float2* __restrict__ partials,
    float* __restrict__ zt) {
  __shared__ float red[256];
  const int r = blockIdx.y, vt = blockIdx.x;
  const int64_t j = static_cast<int64_t>(vt) * kVocabTile + threadIdx.x;
  const bool in = j < V;
  const float z = in ? logits[static_cast<size_t>(r) * ldv + j] : -INFINITY;
  red[threadIdx.x] = z;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + w]);
    __syncthreads();
  }
  const float m = red[0];
  __syncthreads();
  red[threadIdx.x] = in ? expf(z - m) : 0.f;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) partials[static_cast<size_t>(r) * part_stride + vt] = make_float2(m, red[0]);
  const int64_t tg = t[r];
  if (in && tg != ignore_index && tg - col_base == j) zt[r] = z;
}

}  // namespace

cudaError_t launch_simt_gemm_f32(const float* A, int64_t sam, int64_t sak, const float* B,
                                 int64_t sbk, int64_t sbn, float* C, int64_t ldc, int64_t M,
                                 int64_t N, int64_t K, int accumulate, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((N + kTN - 1) / kTN), static_cast<unsigned>((M + kTM - 1) / kTM));
  simt_gemm_f32_kernel<<<grid, 256, 0, s>>>(A, sam, sak, B, sbk, sbn, C, ldc, M, N, K, accumulate);
  return cudaGetLastError();
}

cudaError_t launch_simt_tile_stats(const float* logits, int64_t ldv, int rows, int64_t V,
                                   int vocab_tiles, int part_stride, int64_t col_base,
                                   const int64_t* t_chunk, int64_t ignore_index, float2* partials,
                                   float* zt, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(vocab_tiles), static_cast<unsigned>(rows));
  simt_tile_stats_kernel<<<grid, 256, 0, s>>>(logits, ldv, V, part_stride, col_base, t_chunk,
                                              ignore_index, partials, zt);
  return cudaGetLastError();
}

}  // namespace flce
