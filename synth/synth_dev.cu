// Seeded synthetic inputs, device side: the same counter-based SplitMix64
// draws as synth_host.c (see there for the definition), written straight into
// device buffers so full-size workloads never cross the host. Input generation
// only; nothing of the method is computed here.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__host__ __device__ inline uint64_t sm64(uint64_t x) {
  uint64_t z = x + kGamma;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ inline void store(void* out, int kind, uint64_t e, float v) {
  if (kind == 0)
    static_cast<float*>(out)[e] = v;
  else
    static_cast<uint16_t*>(out)[e] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
}

__global__ void fill_normal_kernel(void* out, int kind, uint64_t n, uint64_t start, uint64_t key,
                                   const float* __restrict__ table) {
  uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t e = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += stride) {
    uint64_t u = sm64(key + (start + e) * kGamma);
    store(out, kind, e, table[u >> 48]);
  }
}

__global__ void fill_int_kernel(void* out, int kind, uint64_t n, uint64_t start, uint64_t key, int a,
                                const uint8_t* __restrict__ row_mult, uint64_t row_len, uint64_t rows_per_batch) {
  uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  uint64_t range = uint64_t(2 * a + 1);
  for (uint64_t e = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += stride) {
    uint64_t idx = start + e;
    uint64_t u = sm64(key + idx * kGamma);
    int64_t iv = int64_t(((u >> 32) * range) >> 32) - a;
    if (row_mult) iv *= int64_t(row_mult[(idx / row_len) % rows_per_batch]);
    store(out, kind, e, float(iv));
  }
}

inline int grid_for(uint64_t n) {
  uint64_t blocks = (n + 255) / 256;
  return int(blocks > 152ull * 64 ? 152ull * 64 : (blocks ? blocks : 1));
}

}  // namespace

extern "C" int synth_dev_fill_normal(void* out, int out_kind, uint64_t n, uint64_t start, uint64_t seed, uint32_t tid,
                                     const float* table_dev, void* stream) {
  if (n == 0) return 0;
  uint64_t key = sm64((seed << 8) | uint64_t(tid & 0xFF));
  fill_normal_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(out, out_kind, n, start, key,
                                                                                 table_dev);
  return int(cudaGetLastError());
}

extern "C" int synth_dev_fill_int(void* out, int out_kind, uint64_t n, uint64_t start, uint64_t seed, uint32_t tid,
                                  int a, const uint8_t* row_mult_dev, uint64_t row_len, uint64_t rows_per_batch,
                                  void* stream) {
  if (n == 0) return 0;
  uint64_t key = sm64((seed << 8) | uint64_t(tid & 0xFF));
  fill_int_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      out, out_kind, n, start, key, a, row_mult_dev, row_len ? row_len : 1, rows_per_batch ? rows_per_batch : 1);
  return int(cudaGetLastError());
}
