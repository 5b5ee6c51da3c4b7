// Loss-only fused linear cross-entropy that allocates no memory.
//
// Some callers cannot let a library call cudaMalloc: a framework whose pool
// allocator must account for every byte of device memory, a runtime that runs
// on a fixed memory plan decided ahead of time, or code that must not pay the
// device-wide synchronisation cudaFree implies. flce_loss_static serves them.
// It needs no handle and no workspace. Its scratch (the control word, the
// per-vocab-tile max / sum-exp partials of one chunk, the chunk's target
// logits and log-sum-exps) lives in the file-scope device array below, which
// every GPU that loads this library holds until the process exits.
//
// It runs the stats-only logits GEMM (no logits are stored), the log-sum-exp
// combine and the loss reduction; it returns the mean loss and the per-token
// losses, not dx or dW.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/flce.h"
#include "flce_internal.h"

namespace flce {
namespace {

constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB
constexpr int kMaxDevices = 64;
constexpr size_t kCtrlBytes = 256;

// One scratch area per device, shared by every call on that device. Host
// code must not pass this name to a kernel: on the host it is only a stand-in
// for the symbol. The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_dev[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Once per device, with that device current: look up the device address of
// the scratch array and the SM count.
cudaError_t setup_device(int dev, void** scratch, int* sms) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = n;
    g_scratch_dev[dev] = p;
  }
  *scratch = g_scratch_dev[dev];
  *sms = g_num_sms[dev];
  return cudaSuccess;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// scratch bytes for a chunk of C tokens: control block, partials, z_t, lse
size_t chunk_scratch(int64_t C, int64_t vocab_tiles) {
  return kCtrlBytes + align256(static_cast<size_t>(C) * vocab_tiles * 8) +
         align256(static_cast<size_t>(C) * 4) + align256(static_cast<size_t>(C) * 4);
}

bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return false;
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return reinterpret_cast<Encode>(fn)(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                      dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace flce

using namespace flce;

extern "C" flce_status flce_loss_static(const void* x, const void* W, const int64_t* t, int64_t N,
                                        int64_t H, int64_t V, int64_t ignore_index, float* loss,
                                        float* token_loss, void* stream) {
  if (!W || !loss || (N > 0 && (!x || !t || !token_loss))) return FLCE_ERR_INVALID_ARG;
  if (N < 0 || H < 8 || V < 1 || H % 8 != 0 || N > (1ll << 31) - 1 || V > (1ll << 31) - 1)
    return FLCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W)) & 15u) return FLCE_ERR_INVALID_ARG;
  if (N > 0 && ((reinterpret_cast<uintptr_t>(t) & 7u) || (reinterpret_cast<uintptr_t>(token_loss) & 3u)))
    return FLCE_ERR_INVALID_ARG;
  const int64_t vt = (V + kVocabTile - 1) / kVocabTile;
  // tokens per chunk: up to 4096, a multiple of 128, whatever fits the scratch
  int64_t C = 0;
  for (int64_t c = kBM; c <= 4096; c += kBM)
    if (chunk_scratch(c, vt) <= kStaticScratchBytes) C = c;
  if (C == 0) return FLCE_ERR_INVALID_ARG;  // V beyond what 64 MiB of scratch can serve
  if (N > 0 && N < C) C = N;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  void* base = nullptr;
  int sms = 0;
  if (setup_device(dev, &base, &sms) != cudaSuccess) return FLCE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* sc = static_cast<unsigned char*>(base);
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(sc);
  float2* partials = reinterpret_cast<float2*>(sc + kCtrlBytes);
  float* zt = reinterpret_cast<float*>(sc + kCtrlBytes + align256(static_cast<size_t>(C) * vt * 8));
  float* lse = zt + align256(static_cast<size_t>(C) * 4) / 4;

  // the array keeps the last call's contents: clear the control block
  if (cudaMemsetAsync(ctrl, 0, kCtrlBytes, s) != cudaSuccess) return FLCE_ERR_CUDA;
  if (N > 0) {
    if (launch_count_valid(t, N, V, ignore_index, nullptr, ctrl, s) != cudaSuccess) return FLCE_ERR_CUDA;
    CUtensorMap mW, mX;
    if (!encode_bf16_2d(&mW, W, H, V, H * 2, 64, 256)) return FLCE_ERR_INVALID_ARG;
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    for (int64_t off = 0; off < N; off += C) {
      const int rows = static_cast<int>(std::min<int64_t>(C, N - off));
      if (!encode_bf16_2d(&mX, xb + off * H, H, rows, H * 2, 64, 128)) return FLCE_ERR_INVALID_ARG;
      UmmaArgs a{};
      a.num_m = (rows + kBM - 1) / kBM;
      a.num_n = static_cast<int>((V + kBN - 1) / kBN);
      a.num_s = 1;
      a.kb_total = static_cast<int>((H + kBK - 1) / kBK);
      a.kb_per_split = a.kb_total;
      a.rows = rows;
      a.cols = static_cast<int>(V);
      a.vocab_tiles = static_cast<int>(vt);
      a.store_logits = 0;  // statistics only: no logits buffer
      a.ignore_index = ignore_index;
      a.targets = t + off;
      a.partials = partials;
      a.zt = zt;
      a.lse = lse;
      a.ctrl = ctrl;
      a.timeout_ns = 2000000000ull;
      const int units = a.num_m * a.num_n;
      // the output map is never written in statistics-only mode; x's map stands in
      if (launch_umma(kUmmaLogits, mX, mW, mX, a, std::min(units, sms), s) != cudaSuccess)
        return FLCE_ERR_CUDA;
      if (launch_lse_combine(partials, static_cast<int>(vt), zt, t + off, rows, ignore_index, lse,
                             token_loss + off, s) != cudaSuccess)
        return FLCE_ERR_CUDA;
    }
    if (launch_loss_finalize(token_loss, N, ctrl, 0, nullptr, nullptr, s) != cudaSuccess)
      return FLCE_ERR_CUDA;
  }
  uint32_t host_ctrl[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(host_ctrl, ctrl, sizeof host_ctrl, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FLCE_ERR_CUDA;
  std::memcpy(loss, &host_ctrl[kCtrlLoss], 4);
  if (host_ctrl[kCtrlError] == FLCE_ERR_BAD_TARGET) return FLCE_ERR_BAD_TARGET;
  if (host_ctrl[kCtrlError] == FLCE_ERR_TIMEOUT) return FLCE_ERR_TIMEOUT;
  if (host_ctrl[kCtrlError] != 0) return FLCE_ERR_CUDA;
  return FLCE_OK;
}
