// Row-wise kernels of fused linear cross-entropy: the n_valid count and
// target range check, the cross-tile log-sum-exp combine, the in-place
// dlogits pass (the two also as one launch), the dx split reduction and the
// loss reduction (also run by the call's last dx reduction).
//
// The formulas are those of the Unsloth page ("Unsloth 심층 아키텍처 …",
// section "스트리밍 청크 기반 Fast CrossEntropy 손실 커널"): per token
// L = -z_y + log sum_j exp(z_j) and dL/dz_j = softmax(z)_j - 1(j = y), with the
// sum kept as a running max m and l = sum exp(z - m) per vocab tile. The
// dlogits pass overwrites the chunk's logits buffer in place, as step 2 of
// the FLCE page does ("Fused Linear Cross-Entropy: LLM 학습 logits 메모리 병목
// 없애기", section "FLCE의 핵심 아이디어"). All reductions run in a fixed
// order, so a call is bit-for-bit repeatable.
#include <cuda_bf16.h>

#include "flce_internal.h"
#include "ptx.cuh"

namespace flce {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// n_valid = #{i : t_i != ignore_index}; any other target outside [0, V)
// records FLCE_ERR_BAD_TARGET. One block; fixed-order integer sum. It first
// clears the call's control words, so the call needs no memset of them.
// nv_total (device, may be null) is the divisor of a token-sharded batch:
// the number of non-ignored tokens over every shard. When given, it becomes
// the n_valid word that every later step of the call divides by, and the
// local count goes to kCtrlNValidLocal; a total below the local count is an
// argument error.
__global__ void count_valid_kernel(const int64_t* __restrict__ t, int64_t N, int64_t V,
                                   int64_t ignore_index, const int32_t* __restrict__ nv_total,
                                   uint32_t* ctrl) {
  __shared__ uint32_t warp_cnt[32];
  // the call's first kernel: its control words start at zero here (the
  // sticky error word, kept across calls, excepted)
  if (threadIdx.x < kCtrlSticky) ctrl[threadIdx.x] = 0u;
  __syncthreads();
  uint32_t cnt = 0;
  bool bad = false;
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x) {
    const int64_t v = t[i];
    if (v == ignore_index) continue;
    if (v < 0 || v >= V) bad = true;
    ++cnt;
  }
  if (bad) atomicCAS(ctrl + kCtrlError, 0u, kErrBadTarget);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) warp_cnt[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t c = threadIdx.x < (blockDim.x >> 5) ? warp_cnt[threadIdx.x] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (threadIdx.x == 0) {
      ctrl[kCtrlNValidLocal] = c;
      if (nv_total) {
        const int32_t tot = *nv_total;
        if (tot < 0 || static_cast<uint32_t>(tot) < c) {
          atomicCAS(ctrl + kCtrlError, 0u, kErrInvalidArg);
          ctrl[kCtrlNValid] = c;
        } else {
          ctrl[kCtrlNValid] = static_cast<uint32_t>(tot);
        }
      } else {
        ctrl[kCtrlNValid] = c;
      }
    }
  }
}

// The count alone, into caller device memory: #{i : t_i != ignore_index}.
// One block; fixed-order integer sum.
__global__ void count_only_kernel(const int64_t* __restrict__ t, int64_t N, int64_t ignore_index,
                                  int32_t* __restrict__ out) {
  __shared__ uint32_t warp_cnt[32];
  uint32_t cnt = 0;
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x) cnt += t[i] != ignore_index ? 1u : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) warp_cnt[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t c = threadIdx.x < (blockDim.x >> 5) ? warp_cnt[threadIdx.x] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (threadIdx.x == 0) *out = static_cast<int32_t>(c);
  }
}

// Per token row: lse = M + log sum_s l_s exp(m_s - M) over the vocab tiles'
// (m_s, l_s); token loss = lse - z_t (0 for an ignored token). One pass over
// the partials: each thread keeps a running (max, sum) and rescales its sum
// when the max grows; the threads' pairs then merge the same way, in a fixed
// order.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * ex2_approx((m - m2) * kLog2e) + s2;
    m = m2;
  } else {
    s += s2 * ex2_approx((m2 - m) * kLog2e);
  }
}

// The log-sum-exp of one token row from its partials, on a block of
// THREADS threads: each thread merges a strided share of the row's partials
// (four loads in flight), then the warps and the block merge their pairs in
// a fixed order. The result is valid in thread 0; warp_ms holds THREADS / 32
// entries of shared memory.
template <int THREADS>
__device__ __forceinline__ float row_lse(const float2* __restrict__ p, int vocab_tiles, float2* warp_ms) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float M = -INFINITY, S = 0.f;
  int s = threadIdx.x;
  for (; s + 3 * THREADS < vocab_tiles; s += 4 * THREADS) {
    float2 q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = p[s + j * THREADS];
#pragma unroll
    for (int j = 0; j < 4; ++j) lse_merge(M, S, q[j].x, q[j].y);
  }
  for (; s < vocab_tiles; s += THREADS) {
    const float2 q = p[s];
    lse_merge(M, S, q.x, q.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
    lse_merge(M, S, m2, s2);
  }
  if (lane == 0) warp_ms[warp] = make_float2(M, S);
  __syncthreads();
  if (threadIdx.x == 0) {
    M = warp_ms[0].x;
    S = warp_ms[0].y;
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) lse_merge(M, S, warp_ms[w].x, warp_ms[w].y);
  }
  return M + logf(S);
}

constexpr int kCombineThreads = 128;

// One block of kCombineThreads per token row.
__global__ void __launch_bounds__(kCombineThreads) lse_combine_kernel(
    const float2* __restrict__ partials, int vocab_tiles, const float* __restrict__ zt,
    const int64_t* __restrict__ t, int rows, int64_t ignore_index, float* __restrict__ lse,
    float* __restrict__ token_loss) {
  __shared__ float2 warp_ms[kCombineThreads / 32];
  const int r = blockIdx.x;
  const float l = row_lse<kCombineThreads>(partials + static_cast<size_t>(r) * vocab_tiles, vocab_tiles,
                                           warp_ms);
  if (threadIdx.x == 0) {
    lse[r] = l;
    const int64_t tg = t[r];
    token_loss[r] = (tg == ignore_index) ? 0.f : (l - zt[r]);
  }
}

// dlogits in place over a bf16 chunk buffer: d = (softmax - onehot) / n_valid.
// The buffer holds y = z - m_s, the logits shifted by their vocab tile's max
// m_s (partials[.].x), so softmax = exp(y + m_s - lse). One block covers 8192
// columns of one token row (blockIdx.y); each thread loads its four 16-byte
// vectors before computing, to keep more bytes in flight.
//
// Almost every vector holds neither the target column nor the end of the
// vocabulary; those take a short path that folds 1/n_valid into the exponent,
// d = 2^(y·log2 e - (lse - m_s)·log2 e - log2 n_valid). Ignored rows are
// written as zeros without being read.
//
// The target column's entry, about -1/n_valid, is stored in bf16 with a 2^-9
// relative error; dx = dlogits·W would multiply that error by the part of W
// common to all rows. Its exact fp32 rounding error goes to dcorr[row] so the
// dx reduction can add dcorr·W[t] back. Ignored rows and padding columns get 0.
constexpr int kDlogitsVecs = 4;
constexpr int kDlogitsThreads = 256;
constexpr int kDlogitsCols = kDlogitsThreads * 8 * kDlogitsVecs;  // columns per block

// A dead row (ignored token, or no valid token in the batch): zeros, the
// buffer not read.
__device__ __forceinline__ void zero_cols(__nv_bfloat16* __restrict__ row, int64_t base, int64_t ldv) {
#pragma unroll
  for (int i = 0; i < kDlogitsVecs; ++i) {
    const int64_t c0 = base + (static_cast<int64_t>(i) * blockDim.x + threadIdx.x) * 8;
    if (c0 < ldv) *reinterpret_cast<uint4*>(row + c0) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// The pass over kDlogitsCols columns of a live row from column `base`. l is
// the row's log-sum-exp, tg its target, scale = 1/n_valid and lg_nv =
// log2 n_valid; s_ll is shared scratch of kDlogitsCols / kVocabTile floats
// (a caller that reuses it waits for the block between calls).
__device__ __forceinline__ void dlogits_cols(__nv_bfloat16* __restrict__ row, int64_t base, int64_t ldv,
                                             int64_t V, const float2* __restrict__ prow, int vocab_tiles,
                                             float l, int64_t tg, float scale, float lg_nv,
                                             float* __restrict__ dcorr_r, float* s_ll) {
  uint4 v[kDlogitsVecs];
#pragma unroll
  for (int i = 0; i < kDlogitsVecs; ++i) {
    const int64_t c0 = base + (static_cast<int64_t>(i) * blockDim.x + threadIdx.x) * 8;
    if (c0 < ldv) v[i] = *reinterpret_cast<const uint4*>(row + c0);
  }
  // the block's per-group exponent offsets (lse - m_g)·log2 e, staged once in
  // shared memory while the vectors above are in flight
  {
    const int64_t g0 = base / kVocabTile;
    for (int q = threadIdx.x; q < kDlogitsCols / kVocabTile; q += blockDim.x)
      if (g0 + q < vocab_tiles) s_ll[q] = (l - prow[g0 + q].x) * kLog2e;
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kDlogitsVecs; ++i) {
    const int64_t c0 = base + (static_cast<int64_t>(i) * blockDim.x + threadIdx.x) * 8;
    if (c0 >= ldv) continue;
    // 8 columns never straddle a vocab tile
    const float ll = s_ll[(c0 - base) / kVocabTile];
    uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    if (c0 + 8 <= V && (tg < c0 || tg >= c0 + 8)) {
      const float nl = ll + lg_nv;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float f0 = __uint_as_float(w[q] << 16);
        const float f1 = __uint_as_float(w[q] & 0xFFFF0000u);
        const __nv_bfloat162 h = __floats2bfloat162_rn(ex2_approx(fmaf(f0, kLog2e, -nl)),
                                                       ex2_approx(fmaf(f1, kLog2e, -nl)));
        w[q] = *reinterpret_cast<const uint32_t*>(&h);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w[q]);
        const float2 f = __bfloat1622float2(h);
        const int64_t j0 = c0 + 2 * q;
        float d0 = ex2_approx(fmaf(f.x, kLog2e, -ll));
        float d1 = ex2_approx(fmaf(f.y, kLog2e, -ll));
        if (j0 == tg) d0 -= 1.f;
        if (j0 + 1 == tg) d1 -= 1.f;
        d0 = (j0 < V) ? d0 * scale : 0.f;
        d1 = (j0 + 1 < V) ? d1 * scale : 0.f;
        h = __floats2bfloat162_rn(d0, d1);
        if (j0 == tg) *dcorr_r = d0 - __low2float(h);
        if (j0 + 1 == tg) *dcorr_r = d1 - __high2float(h);
        w[q] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    *reinterpret_cast<uint4*>(row + c0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void __launch_bounds__(kDlogitsThreads) dlogits_bf16_kernel(
    __nv_bfloat16* __restrict__ buf, int64_t ldv, int64_t V, const float2* __restrict__ partials,
    int vocab_tiles, const float* __restrict__ lse, const int64_t* __restrict__ t,
    int64_t ignore_index, const uint32_t* __restrict__ ctrl, float* __restrict__ dcorr) {
  __shared__ float s_ll[kDlogitsCols / kVocabTile];
  const int r = blockIdx.y;
  const int64_t tg = t[r];
  const uint32_t nv = ctrl[kCtrlNValid];
  __nv_bfloat16* row = buf + static_cast<size_t>(r) * ldv;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kDlogitsCols;
  if (tg == ignore_index || nv == 0) {
    zero_cols(row, base, ldv);
    return;
  }
  dlogits_cols(row, base, ldv, V, partials + static_cast<size_t>(r) * vocab_tiles, vocab_tiles, lse[r], tg,
               1.0f / static_cast<float>(nv), __log2f(static_cast<float>(nv)), dcorr + r, s_ll);
}

// The log-sum-exp combine and the dlogits pass of one token row in one block,
// for chunk buffers of at most kFusedSteps x kDlogitsCols columns (262144):
// the row's log-sum-exp and token loss from its partials, then the row's
// columns kDlogitsCols at a time. One launch per chunk does the work of two,
// at the dlogits pass's bandwidth (one block per row leaves thousands of
// blocks, each keeping its loads in flight); beyond that width the two
// launches remain.
constexpr int kFusedSteps = 32;

__global__ void __launch_bounds__(kDlogitsThreads) combine_dlogits_bf16_kernel(
    __nv_bfloat16* __restrict__ buf, int64_t ldv, int64_t V, const float2* __restrict__ partials,
    int vocab_tiles, const float* __restrict__ zt, const int64_t* __restrict__ t, int64_t ignore_index,
    const uint32_t* __restrict__ ctrl, float* __restrict__ lse, float* __restrict__ token_loss,
    float* __restrict__ dcorr) {
  __shared__ float2 warp_ms[kDlogitsThreads / 32];
  __shared__ float s_ll[kDlogitsCols / kVocabTile];
  __shared__ float s_l;
  const int r = blockIdx.x;
  const float2* prow = partials + static_cast<size_t>(r) * vocab_tiles;
  const int64_t tg = t[r];
  const float lr = row_lse<kDlogitsThreads>(prow, vocab_tiles, warp_ms);
  if (threadIdx.x == 0) {
    lse[r] = lr;
    token_loss[r] = (tg == ignore_index) ? 0.f : (lr - zt[r]);
    s_l = lr;
  }
  __syncthreads();
  const float l = s_l;
  const uint32_t nv = ctrl[kCtrlNValid];
  const bool live = tg != ignore_index && nv > 0;  // uniform across the block
  const float scale = live ? 1.0f / static_cast<float>(nv) : 0.f;
  const float lg_nv = live ? __log2f(static_cast<float>(nv)) : 0.f;
  __nv_bfloat16* row = buf + static_cast<size_t>(r) * ldv;
  for (int64_t base = 0; base < ldv; base += kDlogitsCols) {
    if (!live) {
      zero_cols(row, base, ldv);
      continue;
    }
    dlogits_cols(row, base, ldv, V, prow, vocab_tiles, l, tg, scale, lg_nv, dcorr + r, s_ll);
    __syncthreads();  // s_ll is staged again for the next columns
  }
}

// fp32 version: 4 columns per thread
__global__ void dlogits_f32_kernel(float* __restrict__ buf, int64_t ldv, int64_t V, int64_t col_base,
                                   const float* __restrict__ lse, const int64_t* __restrict__ t,
                                   int64_t ignore_index, const uint32_t* __restrict__ ctrl) {
  const int r = blockIdx.y;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (c0 >= ldv) return;
  const int64_t tg = t[r];
  const uint32_t nv = ctrl[kCtrlNValid];
  const bool valid = tg != ignore_index;
  const float scale = (valid && nv > 0) ? 1.0f / static_cast<float>(nv) : 0.f;
  const float l = lse[r];
  float4* ptr = reinterpret_cast<float4*>(buf + static_cast<size_t>(r) * ldv + c0);
  float4 v = *ptr;
  float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int64_t j = c0 + q;
    float d = expf(f[q] - l);
    if (j + col_base == tg) d -= 1.f;
    f[q] = (j < V) ? d * scale : 0.f;
  }
  *ptr = make_float4(f[0], f[1], f[2], f[3]);
}

// loss = (sum of token losses) / n_valid, the sum in float64 and fixed order
// on a block of THREADS threads: each thread sums a fixed strided set, then
// warp shuffles and one warp merge the partial sums in a fixed tree. With
// `result` set it also writes the device result of the sync-free entry
// points (as device_result_kernel). Every thread of the block calls it.
template <int THREADS>
__device__ __forceinline__ void loss_reduce(const float* __restrict__ token_loss, int64_t N, uint32_t* ctrl,
                                            int result, float* loss_dev, int32_t* n_valid_dev) {
  __shared__ double warp_sum[THREADS / 32];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < N; i += THREADS) s += static_cast<double>(token_loss[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    double w = threadIdx.x < THREADS / 32 ? warp_sum[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_down_sync(0xffffffffu, w, o);
    if (threadIdx.x == 0) {
      const uint32_t nv = ctrl[kCtrlNValid];
      const float loss = nv > 0 ? static_cast<float>(w / static_cast<double>(nv)) : 0.f;
      ctrl[kCtrlLoss] = __float_as_uint(loss);
      if (result) {
        const uint32_t err = ctrl[kCtrlError];
        if (loss_dev) *loss_dev = err ? __uint_as_float(0x7fc00000u) : loss;
        if (n_valid_dev) *n_valid_dev = static_cast<int32_t>(nv);
        if (err && ctrl[kCtrlSticky] == 0u) ctrl[kCtrlSticky] = err;
      }
    }
  }
}

constexpr int kReduceThreads = 128;

// The fp32 path's row steps of one chunk in one block per token row: the
// row's log-sum-exp over its V fp32 logits (a running max and rescaled sum
// per thread, with expf, merged across the block in a fixed order), its
// token loss, then the row overwritten in place with (softmax - onehot) /
// n_valid (zeros for an ignored row, and for the row's padding columns past
// V). It replaces the per-tile statistics, the combine and the dlogits pass
// of that path: one launch instead of three, the row read twice.
constexpr int kRowsF32Threads = 1024;

__device__ __forceinline__ void online_add(float& m, float& s, float z) {
  if (z > m) {
    s = (m == -INFINITY ? 0.f : s * expf(m - z)) + 1.f;
    m = z;
  } else {
    s += expf(z - m);
  }
}

__device__ __forceinline__ void online_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
  } else if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * expf(m2 - m);
  }
}

__global__ void __launch_bounds__(kRowsF32Threads) rows_f32_kernel(
    float* __restrict__ buf, int64_t ldv, int64_t V, const int64_t* __restrict__ t, int64_t ignore_index,
    const uint32_t* __restrict__ ctrl, float* __restrict__ lse, float* __restrict__ token_loss) {
  __shared__ float2 warp_ms[kRowsF32Threads / 32];
  __shared__ float s_l, s_zt;
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* row = buf + static_cast<size_t>(r) * ldv;
  const int64_t tg = t[r];
  float m = -INFINITY, sum = 0.f;
  for (int64_t j = threadIdx.x; j < V; j += kRowsF32Threads) {
    const float z = row[j];
    online_add(m, sum, z);
    if (j == tg) s_zt = z;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
    online_merge(m, sum, m2, s2);
  }
  if (lane == 0) warp_ms[warp] = make_float2(m, sum);
  __syncthreads();
  if (threadIdx.x == 0) {
    m = warp_ms[0].x;
    sum = warp_ms[0].y;
#pragma unroll
    for (int w = 1; w < kRowsF32Threads / 32; ++w) online_merge(m, sum, warp_ms[w].x, warp_ms[w].y);
    const float l = m + logf(sum);
    lse[r] = l;
    token_loss[r] = (tg == ignore_index) ? 0.f : (l - s_zt);
    s_l = l;
  }
  __syncthreads();
  const float l = s_l;
  const uint32_t nv = ctrl[kCtrlNValid];
  const bool live = tg != ignore_index && nv > 0;
  const float scale = live ? 1.0f / static_cast<float>(nv) : 0.f;
  for (int64_t j = threadIdx.x; j < ldv; j += kRowsF32Threads) {
    float d = 0.f;
    if (live && j < V) {
      d = expf(row[j] - l);
      if (j == tg) d -= 1.f;
      d *= scale;
    }
    row[j] = d;
  }
}

// dx row i = sum over splits of the fp32 partials of dlogits·W (in split
// order) + dcorr[i]·W[t_i], rounded once to bf16. dcorr[i] is the fp32
// rounding error of the bf16 dlogits entry at the target column, so the sum
// is dx as if that entry, the largest of the row, had been stored exactly.
// blockIdx.y = token row, 4 columns per thread.
//
// The call's last dx reduction can also take the loss reduction (fin.on):
// block (0, 0) runs it beside its dx columns. It reads only the token losses
// and control words of earlier launches, so no block waits for another; the
// call saves the launch of loss_finalize_kernel.
struct LossFinish {
  int on;
  int result;
  const float* token_loss;
  int64_t N;
  float* loss_dev;
  int32_t* n_valid_dev;
};

__global__ void __launch_bounds__(kReduceThreads) dx_reduce_kernel(
    const float* __restrict__ part, int splits, int64_t split_stride, int64_t H,
    const __nv_bfloat16* __restrict__ W, int64_t V, const int64_t* __restrict__ t, int64_t ignore_index,
    uint32_t* ctrl, const float* __restrict__ dcorr, __nv_bfloat16* __restrict__ dx, LossFinish fin) {
  const int r = blockIdx.y;
  const int64_t h = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (h < H) {
    const int64_t tg = t[r];
    const bool corr = tg != ignore_index && tg >= 0 && tg < V && ctrl[kCtrlNValid] > 0;
    const int64_t i = static_cast<int64_t>(r) * H + h;
    float4 acc = *reinterpret_cast<const float4*>(part + i);
    for (int s = 1; s < splits; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(part + s * split_stride + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (corr) {
      const float c = dcorr[r];
      const uint2 wv = *reinterpret_cast<const uint2*>(W + tg * H + h);
      const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.x));
      const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.y));
      acc.x = fmaf(w01.x, c, acc.x);
      acc.y = fmaf(w01.y, c, acc.y);
      acc.z = fmaf(w23.x, c, acc.z);
      acc.w = fmaf(w23.y, c, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dx + i) = o;
  }
  if (fin.on && blockIdx.x == 0 && blockIdx.y == 0)
    loss_reduce<kReduceThreads>(fin.token_loss, fin.N, ctrl, fin.result, fin.loss_dev, fin.n_valid_dev);
}

__global__ void __launch_bounds__(1024) loss_finalize_kernel(const float* __restrict__ token_loss,
                                                             int64_t N, uint32_t* ctrl, int result,
                                                             float* loss_dev, int32_t* n_valid_dev) {
  loss_reduce<1024>(token_loss, N, ctrl, result, loss_dev, n_valid_dev);
}

// The call's result into caller device memory, for the entry point that
// never synchronises: the loss (NaN when a kernel recorded an error) and
// n_valid; the first such error is also kept in the sticky word.
__global__ void device_result_kernel(uint32_t* ctrl, float* loss_dev, int32_t* n_valid_dev) {
  const uint32_t err = ctrl[kCtrlError];
  if (loss_dev) *loss_dev = err ? __uint_as_float(0x7fc00000u) : __uint_as_float(ctrl[kCtrlLoss]);
  if (n_valid_dev) *n_valid_dev = static_cast<int32_t>(ctrl[kCtrlNValid]);
  if (err && ctrl[kCtrlSticky] == 0u) ctrl[kCtrlSticky] = err;
}

}  // namespace

cudaError_t launch_device_result(uint32_t* ctrl, float* loss_dev, int32_t* n_valid_dev, cudaStream_t s) {
  device_result_kernel<<<1, 1, 0, s>>>(ctrl, loss_dev, n_valid_dev);
  return cudaGetLastError();
}

cudaError_t launch_count_valid(const int64_t* t, int64_t N, int64_t V, int64_t ignore_index,
                               const int32_t* nv_total, uint32_t* ctrl, cudaStream_t s) {
  count_valid_kernel<<<1, 1024, 0, s>>>(t, N, V, ignore_index, nv_total, ctrl);
  return cudaGetLastError();
}

cudaError_t launch_count_only(const int64_t* t, int64_t N, int64_t ignore_index, int32_t* out,
                              cudaStream_t s) {
  count_only_kernel<<<1, 1024, 0, s>>>(t, N, ignore_index, out);
  return cudaGetLastError();
}

cudaError_t launch_lse_combine(const float2* partials, int vocab_tiles, const float* zt,
                               const int64_t* t_chunk, int rows, int64_t ignore_index, float* lse,
                               float* token_loss_chunk, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  lse_combine_kernel<<<rows, kCombineThreads, 0, s>>>(partials, vocab_tiles, zt, t_chunk, rows,
                                                      ignore_index, lse, token_loss_chunk);
  return cudaGetLastError();
}

cudaError_t launch_dlogits_bf16(__nv_bfloat16* buf, int64_t ldv, int rows, int64_t V,
                                const float2* partials, int vocab_tiles, const float* lse,
                                const int64_t* t_chunk, int64_t ignore_index,
                                const uint32_t* ctrl, float* dcorr, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((ldv + kDlogitsCols - 1) / kDlogitsCols), static_cast<unsigned>(rows));
  dlogits_bf16_kernel<<<grid, kDlogitsThreads, 0, s>>>(buf, ldv, V, partials, vocab_tiles, lse, t_chunk,
                                               ignore_index, ctrl, dcorr);
  return cudaGetLastError();
}

cudaError_t launch_dlogits_f32(float* buf, int64_t ldv, int rows, int64_t V, int64_t col_base,
                               const float* lse, const int64_t* t_chunk, int64_t ignore_index,
                               const uint32_t* ctrl, cudaStream_t s) {
  const int threads = 256;
  const int64_t per_block = threads * 4;
  dim3 grid(static_cast<unsigned>((ldv + per_block - 1) / per_block), static_cast<unsigned>(rows));
  dlogits_f32_kernel<<<grid, threads, 0, s>>>(buf, ldv, V, col_base, lse, t_chunk, ignore_index, ctrl);
  return cudaGetLastError();
}

cudaError_t launch_dx_reduce(const float* partials, int splits, int64_t split_stride, int rows,
                             int64_t H, const __nv_bfloat16* W, int64_t V, const int64_t* t_chunk,
                             int64_t ignore_index, uint32_t* ctrl, const float* dcorr,
                             __nv_bfloat16* dx, cudaStream_t s, const float* token_loss, int64_t N,
                             int result, float* loss_dev, int32_t* n_valid_dev) {
  // H % 8 == 0: 4 columns per thread, no partial vectors
  dim3 grid(static_cast<unsigned>((H / 4 + kReduceThreads - 1) / kReduceThreads), static_cast<unsigned>(rows));
  const LossFinish fin{token_loss ? 1 : 0, result, token_loss, N, loss_dev, n_valid_dev};
  dx_reduce_kernel<<<grid, kReduceThreads, 0, s>>>(partials, splits, split_stride, H, W, V, t_chunk,
                                                   ignore_index, ctrl, dcorr, dx, fin);
  return cudaGetLastError();
}

cudaError_t launch_combine_dlogits_bf16(__nv_bfloat16* buf, int64_t ldv, int rows, int64_t V,
                                        const float2* partials, int vocab_tiles, const float* zt,
                                        const int64_t* t_chunk, int64_t ignore_index,
                                        const uint32_t* ctrl, float* lse, float* token_loss_chunk,
                                        float* dcorr, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (ldv > static_cast<int64_t>(kFusedSteps) * kDlogitsCols) return cudaErrorInvalidValue;
  combine_dlogits_bf16_kernel<<<rows, kDlogitsThreads, 0, s>>>(buf, ldv, V, partials, vocab_tiles, zt,
                                                               t_chunk, ignore_index, ctrl, lse,
                                                               token_loss_chunk, dcorr);
  return cudaGetLastError();
}

cudaError_t launch_rows_f32(float* buf, int64_t ldv, int rows, int64_t V, const int64_t* t_chunk,
                            int64_t ignore_index, const uint32_t* ctrl, float* lse,
                            float* token_loss_chunk, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  rows_f32_kernel<<<rows, kRowsF32Threads, 0, s>>>(buf, ldv, V, t_chunk, ignore_index, ctrl, lse,
                                                  token_loss_chunk);
  return cudaGetLastError();
}

int64_t combine_dlogits_max_cols() { return static_cast<int64_t>(kFusedSteps) * kDlogitsCols; }

cudaError_t launch_loss_finalize(const float* token_loss, int64_t N, uint32_t* ctrl, int result,
                                 float* loss_dev, int32_t* n_valid_dev, cudaStream_t s) {
  loss_finalize_kernel<<<1, 1024, 0, s>>>(token_loss, N, ctrl, result, loss_dev, n_valid_dev);
  return cudaGetLastError();
}

}  // namespace flce
