// Main Branch, query-outer CUDA-core kernel: for one (query row, group) a CTA
// walks the group's selected blocks, gathers their keys/values and runs an
// exact online softmax for each of the group's query heads.
// (hyper.ai summary of paper 2606.13392, section "方法": softmax attention
//  restricted to the tokens of the selected blocks, K/V gathered per block.)
//
// This is the fp32 path (tensor cores have no fp32 multiply) and the generic
// path for shapes the tensor-core kernels do not cover. Warp per query head;
// lane per key inside 32-key chunks; the output row is spread over lanes.
#include <cmath>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kQoWarps = 4;

template <typename T, int D>
__device__ __forceinline__ float dot_row(const float* q_s, const T* krow) {
  float s = 0.f;
  if constexpr (sizeof(T) == 2) {
    const uint4* kv = reinterpret_cast<const uint4*>(krow);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 w = __ldg(kv + c);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h[e]);
        s = fmaf(q_s[c * 8 + 2 * e], f.x, s);
        s = fmaf(q_s[c * 8 + 2 * e + 1], f.y, s);
      }
    }
  } else {
    const float4* kv = reinterpret_cast<const float4*>(krow);
#pragma unroll
    for (int c = 0; c < D / 4; ++c) {
      float4 w = __ldg(kv + c);
      s = fmaf(q_s[4 * c], w.x, s);
      s = fmaf(q_s[4 * c + 1], w.y, s);
      s = fmaf(q_s[4 * c + 2], w.z, s);
      s = fmaf(q_s[4 * c + 3], w.w, s);
    }
  }
  return s;
}

// grid.x = B * Nq * Hkv (one CTA per (row, group)); kQoWarps warps stride over
// the group's Hq/Hkv heads.
template <typename T, int D>
__global__ void __launch_bounds__(kQoWarps * 32) attn_query_outer_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const int32_t* __restrict__ sel,
    const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len, int decode, int Nq, int Nk, int Hq,
    int Hkv, int Bs, int K, float scale, T* __restrict__ out, float* __restrict__ lse, uint32_t* status) {
  __shared__ __align__(16) float q_s[kQoWarps][D];
  constexpr int U = D / 32;  // output coordinates per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t rg = blockIdx.x;  // (b, i, g)
  const int g = int(rg % Hkv);
  const int64_t bi = rg / Hkv;  // b * Nq + i
  const int i = int(bi % Nq);
  const int b = int(bi / Nq);
  const int hpg = Hq / Hkv;
  const int nblk = (Nk + Bs - 1) / Bs;
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, decode != 0);
  const int pos = sv.q0 + i;
  const int32_t* srow = sel + rg * K;

  for (int hl = warp; hl < hpg; hl += kQoWarps) {
    const int h = g * hpg + hl;
    const int64_t qrow = (bi * Hq + h) * D;
    for (int c = lane; c < D; c += 32) q_s[warp][c] = to_f(q[qrow + c]);
    __syncwarp();
    float m = -INFINITY, l = 0.f;
    float o[U];
#pragma unroll
    for (int u = 0; u < U; ++u) o[u] = 0.f;
    if (sv.ok) {
      for (int kk = 0; kk < K; ++kk) {
        const int t = srow[kk];
        if (t == -1) continue;
        if (t < -1 || t >= nblk) {
          if (lane == 0) set_status(status, MSA_ERR_BOUNDS);
          continue;
        }
        const int jend = min(min((t + 1) * Bs, pos + 1), sv.L);
        for (int j0 = t * Bs; j0 < jend; j0 += 32) {
          const int j = j0 + lane;
          const bool valid = j < jend;
          const T* krow = k + ((int64_t(b) * Nk + (valid ? j : j0)) * Hkv + g) * D;
          const float s = valid ? dot_row<T, D>(q_s[warp], krow) * scale : -INFINITY;
          float cmax = s;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));
          const float m_new = fmaxf(m, cmax);
          const float corr = expf(m - m_new);  // m = -inf on the first chunk: corr = 0
          const float p = valid ? expf(s - m_new) : 0.f;
          float psum = p;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
          l = l * corr + psum;
#pragma unroll
          for (int u = 0; u < U; ++u) o[u] *= corr;
          const int nvalid = min(32, jend - j0);
          for (int jj = 0; jj < nvalid; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const T* vrow = v + ((int64_t(b) * Nk + j0 + jj) * Hkv + g) * D;
#pragma unroll
            for (int u = 0; u < U; ++u) o[u] = fmaf(pj, to_f(vrow[lane + 32 * u]), o[u]);
          }
          m = m_new;
        }
      }
    } else if (lane == 0 && hl == warp) {
      set_status(status, MSA_ERR_BOUNDS);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) out[qrow + lane + 32 * u] = from_f<T>(o[u] * inv);
    if (lse && lane == 0) lse[bi * Hq + h] = l > 0.f ? m + logf(l) : -INFINITY;
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_attn_query_outer(int dtype, const void* q, const void* k, const void* v, const int32_t* sel,
                                    const int32_t* q_offset, const int32_t* kv_len, bool decode, int B, int Nq,
                                    int Nk, int Hq, int Hkv, int d, int Bs, int K, float scale, void* out, float* lse,
                                    uint32_t* status, cudaStream_t stream) {
  const int64_t grid = int64_t(B) * Nq * Hkv;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  ProfScope prof("attn_query_outer", stream);
#define MSA_QO(T, D)                                                                                         \
  attn_query_outer_kernel<T, D><<<unsigned(grid), kQoWarps * 32, 0, stream>>>(                             \
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), sel, q_offset, kv_len, \
      decode ? 1 : 0, Nq, Nk, Hq, Hkv, Bs, K, scale, static_cast<T*>(out), lse, status)
  if (dtype == MSA_BF16 && d == 128)
    MSA_QO(__nv_bfloat16, 128);
  else if (dtype == MSA_BF16 && d == 64)
    MSA_QO(__nv_bfloat16, 64);
  else if (dtype == MSA_FP32 && d == 128)
    MSA_QO(float, 128);
  else if (dtype == MSA_FP32 && d == 64)
    MSA_QO(float, 64);
  else
    return cudaErrorInvalidValue;
#undef MSA_QO
  return cudaGetLastError();
}

}  // namespace msa
