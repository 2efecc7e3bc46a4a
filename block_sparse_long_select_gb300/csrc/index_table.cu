// Index Branch, table path (CUDA cores):
//   index_blockmax_table  token scores q_idx . k_idx for every visible key,
//                         max-pooled per key block into a [rows, nblk] table
//   topk_from_table       exact exp-free top-K over each table row, the
//                         query's own block always kept
// (hyper.ai summary of paper 2606.13392, section "方法": dot-product index
//  scores over visible keys, Block Max Pooling, Top-K per GQA group with the
//  local block included; quant_prune_distill post 751, "Метод".)
//
// This path serves fp32 inputs, the optional block-max diagnostic output and
// short query counts (decode), where the key stream dominates and a table of
// a few MB is cheap. Long bf16 prefill uses the fused tensor-core kernel.
#include <cfloat>
#include <cmath>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kTabWarps = 8;   // one key block per warp
constexpr int kTabRows = 16;   // (query row, group) rows per CTA

template <typename T, int DI>
__device__ __forceinline__ void load_row(const T* p, float (&r)[DI]);

template <>
__device__ __forceinline__ void load_row<__nv_bfloat16, 64>(const __nv_bfloat16* p, float (&r)[64]) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 w = __ldg(v + c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __bfloat1622float2(h[e]);
      r[c * 8 + 2 * e] = f.x;
      r[c * 8 + 2 * e + 1] = f.y;
    }
  }
}
template <>
__device__ __forceinline__ void load_row<__nv_bfloat16, 32>(const __nv_bfloat16* p, float (&r)[32]) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w = __ldg(v + c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __bfloat1622float2(h[e]);
      r[c * 8 + 2 * e] = f.x;
      r[c * 8 + 2 * e + 1] = f.y;
    }
  }
}
template <int DI>
__device__ __forceinline__ void load_row_f32(const float* p, float (&r)[DI]) {
  const float4* v = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int c = 0; c < DI / 4; ++c) {
    float4 w = __ldg(v + c);
    r[4 * c] = w.x;
    r[4 * c + 1] = w.y;
    r[4 * c + 2] = w.z;
    r[4 * c + 3] = w.w;
  }
}
template <>
__device__ __forceinline__ void load_row<float, 64>(const float* p, float (&r)[64]) {
  load_row_f32<64>(p, r);
}
template <>
__device__ __forceinline__ void load_row<float, 32>(const float* p, float (&r)[32]) {
  load_row_f32<32>(p, r);
}

// grid (row chunks, key-block chunks, B); 8 warps, warp w owns key block
// blockIdx.y * 8 + w for the CTA's 16 rows.
template <typename T, int DI>
__global__ void __launch_bounds__(kTabWarps * 32) index_blockmax_table_kernel(
    const T* __restrict__ iq, const T* __restrict__ ik, const int32_t* __restrict__ q_offset,
    const int32_t* __restrict__ kv_len, int Nq, int Nk, int G, int Bs, int nblk, float* __restrict__ table,
    uint32_t* status) {
  __shared__ __align__(16) float iq_s[kTabRows][DI];
  __shared__ int pos_s[kTabRows];
  __shared__ int maxpos_s;
  const int b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t rows = int64_t(Nq) * G;
  const int64_t row0 = int64_t(blockIdx.x) * kTabRows;
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  if (!sv.ok && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_status(status, MSA_ERR_BOUNDS);

  for (int e = threadIdx.x; e < kTabRows * DI; e += blockDim.x) {
    const int r = e / DI, c = e % DI;
    const int64_t row = row0 + r;
    iq_s[r][c] = row < rows ? to_f(iq[(int64_t(b) * rows + row) * DI + c]) : 0.f;
  }
  if (threadIdx.x < kTabRows) {
    const int64_t row = row0 + threadIdx.x;
    pos_s[threadIdx.x] = (row < rows && sv.ok) ? sv.q0 + int(row / G) : -1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = -1;
    for (int r = 0; r < kTabRows; ++r) m = max(m, pos_s[r]);
    maxpos_s = m;
  }
  __syncthreads();

  const int t = blockIdx.y * kTabWarps + warp;
  if (t >= nblk) return;
  const int tstart = t * Bs;
  float runmax[kTabRows];
#pragma unroll
  for (int r = 0; r < kTabRows; ++r) runmax[r] = -INFINITY;

  if (tstart <= maxpos_s) {
    const T* ikb = ik + int64_t(b) * Nk * DI;
    for (int jj = lane; jj < Bs; jj += 32) {
      const int j = tstart + jj;
      if (j > maxpos_s || j >= sv.L) break;
      float kr[DI];
      load_row<T, DI>(ikb + int64_t(j) * DI, kr);
#pragma unroll
      for (int r = 0; r < kTabRows; ++r) {
        if (j <= pos_s[r]) {
          float s = 0.f;
#pragma unroll
          for (int c = 0; c < DI; c += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(&iq_s[r][c]);
            s = fmaf(qv.x, kr[c], s);
            s = fmaf(qv.y, kr[c + 1], s);
            s = fmaf(qv.z, kr[c + 2], s);
            s = fmaf(qv.w, kr[c + 3], s);
          }
          runmax[r] = fmaxf(runmax[r], s);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kTabRows; ++r) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) runmax[r] = fmaxf(runmax[r], __shfl_xor_sync(0xffffffffu, runmax[r], off));
  }
#pragma unroll
  for (int r = 0; r < kTabRows; ++r) {
    if (lane == r) {
      const int64_t row = row0 + r;
      if (row < rows) {
        const bool vis = pos_s[r] >= 0 && tstart <= pos_s[r];
        table[(int64_t(b) * rows + row) * nblk + t] = vis ? runmax[r] : NAN;
      }
    }
  }
}

// Warp per (b, i, g) row. Each lane keeps a descending list of its best
// candidates (strided over blocks fs <= t < loc) in shared memory; the 32
// lists are then merged by K-1-fs rounds of a warp-wide maximum. fs = 1 keeps
// block 0 outright, like the local block.
constexpr int kTopkWarps = 4;

__global__ void __launch_bounds__(kTopkWarps * 32) topk_from_table_kernel(
    const float* __restrict__ table, const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len, int B,
    int Nq, int Nk, int G, int Bs, int K, int nblk, int fs, int32_t* __restrict__ sel, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Kc = K - 1 > 0 ? K - 1 : 1;
  uint64_t* lists = reinterpret_cast<uint64_t*>(smem_raw) + size_t(warp) * Kc * 32;  // [Kc][32]
  int* chosen = reinterpret_cast<int*>(reinterpret_cast<uint64_t*>(smem_raw) + size_t(kTopkWarps) * Kc * 32) +
                warp * kMaxK;

  const int64_t row = int64_t(blockIdx.x) * kTopkWarps + warp;
  const int64_t rows = int64_t(B) * Nq * G;
  if (row >= rows) return;
  const int b = int(row / (int64_t(Nq) * G));
  const int i = int((row / G) % Nq);
  int32_t* out = sel + row * K;
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  if (!sv.ok) {
    for (int k = lane; k < K; k += 32) out[k] = -1;
    if (lane == 0) set_status(status, MSA_ERR_BOUNDS);
    return;
  }
  const int pos = sv.q0 + i;
  const int loc = pos / Bs;
  if (loc + 1 <= K) {
    for (int k = lane; k < K; k += 32) out[k] = k <= loc ? k : -1;
    return;
  }
  const float* M = table + row * nblk;
  int n = 0;  // entries in this lane's list
  for (int t = fs + lane; t < loc; t += 32) {  // fs = 1: block 0 is kept outright
    const uint64_t key = rank_key(M[t], t);
    if (n == Kc && key <= lists[(Kc - 1) * 32 + lane]) continue;
    int p = n < Kc ? n++ : Kc - 1;
    while (p > 0 && lists[(p - 1) * 32 + lane] < key) {
      lists[p * 32 + lane] = lists[(p - 1) * 32 + lane];
      --p;
    }
    lists[p * 32 + lane] = key;
  }
  int head = 0;
  for (int k = 0; k < K - 1 - fs; ++k) {
    const uint64_t mine = head < n ? lists[head * 32 + lane] : 0ull;
    uint64_t best = mine;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, off);
      best = other > best ? other : best;
    }
    if (mine == best) ++head;  // keys are unique: exactly one lane advances
    if (lane == 0) chosen[k] = rank_key_block(best);
  }
  if (lane == 0) {
    chosen[K - 1 - fs] = loc;
    if (fs) chosen[K - 1] = 0;
  }
  __syncwarp();
  // ascending order by rank (all entries distinct)
  for (int e = lane; e < K; e += 32) {
    const int v = chosen[e];
    int rank = 0;
    for (int e2 = 0; e2 < K; ++e2) rank += chosen[e2] < v;
    out[rank] = v;
  }
}

}  // namespace

cudaError_t launch_index_blockmax_table(int dtype, const void* iq, const void* ik, const int32_t* q_offset,
                                        const int32_t* kv_len, int B, int Nq, int Nk, int G, int di, int Bs,
                                        float* table, uint32_t* status, cudaStream_t stream) {
  const int nblk = (Nk + Bs - 1) / Bs;
  const int64_t rows = int64_t(Nq) * G;
  dim3 grid(unsigned((rows + kTabRows - 1) / kTabRows), unsigned((nblk + kTabWarps - 1) / kTabWarps), unsigned(B));
  dim3 block(kTabWarps * 32);
  ProfScope prof("index_blockmax_table", stream);
#define MSA_TAB(T, DI)                                                                                            \
  index_blockmax_table_kernel<T, DI><<<grid, block, 0, stream>>>(static_cast<const T*>(iq), static_cast<const T*>(ik), \
                                                                 q_offset, kv_len, Nq, Nk, G, Bs, nblk, table, status)
  if (dtype == MSA_BF16 && di == 64)
    MSA_TAB(__nv_bfloat16, 64);
  else if (dtype == MSA_BF16 && di == 32)
    MSA_TAB(__nv_bfloat16, 32);
  else if (dtype == MSA_FP32 && di == 64)
    MSA_TAB(float, 64);
  else if (dtype == MSA_FP32 && di == 32)
    MSA_TAB(float, 32);
  else
    return cudaErrorInvalidValue;
#undef MSA_TAB
  return cudaGetLastError();
}

cudaError_t launch_topk_from_table(const float* table, const int32_t* q_offset, const int32_t* kv_len, int B, int Nq,
                                   int Nk, int G, int Bs, int K, int fs, int32_t* sel, uint32_t* status,
                                   cudaStream_t stream) {
  const int nblk = (Nk + Bs - 1) / Bs;
  const int64_t rows = int64_t(B) * Nq * G;
  const int Kc = K - 1 > 0 ? K - 1 : 1;
  const size_t smem = size_t(kTopkWarps) * Kc * 32 * sizeof(uint64_t) + size_t(kTopkWarps) * kMaxK * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_from_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = unsigned((rows + kTopkWarps - 1) / kTopkWarps);
  ProfScope prof("topk_from_table", stream);
  topk_from_table_kernel<<<grid, kTopkWarps * 32, smem, stream>>>(table, q_offset, kv_len, B, Nq, Nk, G, Bs, K, nblk,
                                                                  fs, sel, status);
  return cudaGetLastError();
}

}  // namespace msa
