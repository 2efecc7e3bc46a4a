// msa_index_select_noalloc: the Index Branch (table path: block-max table +
// warp top-K) for callers that cannot allocate device memory themselves --
// for example code running inside another framework's allocator or plugin
// hooks, where a raw cudaMalloc is forbidden or would break that framework's
// memory accounting, or a host process whose device memory budget is fixed
// up front. Its scratch lives in a file-scope __device__ array that every GPU
// loading this library reserves until the process exits.
#include <mutex>

#include "msa_internal.cuh"

namespace msa {
namespace {

// 32 MiB: a 256-byte header (status word) followed by the block-max table.
// Enough for decode at batch 64 over 1M-token contexts with block 128
// (64 x 8 groups x 8192 blocks x 4 B = 16 MiB) and for small prefills.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 256;
void* g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of the static scratch on the current device. The host-side
// symbol is only a stand-in, so the address is looked up once per device
// (with that device current) and cached for the life of the process; a
// cudaDeviceReset after the first call would leave the cached address stale,
// so the entry point does not support one.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status_t msa_index_select_noalloc(const void* iq, const void* ik, const int32_t* q_offset,
                                                 const int32_t* kv_len, int B, int Nq, int Nk, int G, int di, int Bs,
                                                 int K, int dtype, int32_t* sel, float* block_max,
                                                 cudaStream_t stream) {
  // an empty batch: nothing to read or compute, the same checks as msa_index_select
  if (B >= 0 && Nq >= 0 && (B == 0 || Nq == 0)) return index_select_empty_status(Nk, G, di, Bs, K, dtype);
  if (!iq || !ik || !sel) return MSA_ERR_INVALID_ARG;
  if (B < 1 || Nq < 1 || Nk < 1 || G < 1 || di < 1 || Bs < 1 || K < 1 || Nq > Nk) return MSA_ERR_INVALID_ARG;
  if (dtype != MSA_BF16 && dtype != MSA_FP32) return MSA_ERR_INVALID_ARG;
  if ((di != 32 && di != 64) || Bs > kMaxBs || K > kMaxK) return MSA_ERR_UNSUPPORTED;
  const size_t nblk = (size_t(Nk) + Bs - 1) / Bs;
  const size_t table_bytes = block_max ? 0 : size_t(B) * Nq * G * nblk * sizeof(float);
  if (table_bytes > kNoAllocScratchBytes - kWsHeader) return MSA_ERR_WORKSPACE;  // beyond the static scratch

  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return MSA_ERR_CUDA;
  uint32_t* status = static_cast<uint32_t*>(scratch);
  // the array keeps the previous call's contents: the status word must start at zero
  if (cudaMemsetAsync(scratch, 0, kWsHeader, stream) != cudaSuccess) return MSA_ERR_CUDA;
  float* table = block_max ? block_max : reinterpret_cast<float*>(static_cast<char*>(scratch) + kWsHeader);
  if (launch_index_blockmax_table(dtype, iq, ik, q_offset, kv_len, B, Nq, Nk, G, di, Bs, table, status, stream) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  if (launch_topk_from_table(table, q_offset, kv_len, B, Nq, Nk, G, Bs, K, 0, sel, status, stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}
