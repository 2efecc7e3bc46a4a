// Main Branch, decode: one new token per sequence attends to its KV cache
// through the K selected blocks of each group (hyper.ai summary of paper
// 2606.13392, "方法": softmax attention over the selected blocks' keys and
// values; "一句话总结": the decode half of the prefill / decode speedups).
//
//  decode_index    Index Branch for one query per sequence: the index-key
//                  cache streamed once by TMA in 128-key tiles, scores on
//                  tcgen05 (keys along M, the G index-query heads along N),
//                  block maxima straight from TMEM into a small
//                  [B, G, nblk] table
//  decode_topk     exact top-K per (sequence, group) over that table, the
//                  query's own block forced, ascending output
//  decode_attn     one CTA per (sequence, group, selected block): the block's
//                  K and V rows of that group are TMA-loaded (128B-swizzled,
//                  so a thread reading "its" key row is bank-conflict free),
//                  scores for the group's query heads, a block-local softmax,
//                  P.V in fp32 -> per-slot partial (O unnormalised, max, sum)
//  decode_combine  per (sequence, query head): log-sum-exp merge of the K
//                  slot partials in slot order -> bf16 output row (+ lse)
//
// The step streams each selected K/V block from HBM exactly once; partials
// are small (B x G x K x hpg x (d + 2) fp32) and stay in L2.
#include <cmath>

#include "msa_internal.cuh"
#include "tc_utils.cuh"

namespace msa {
namespace {

constexpr int kDecThreads = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2eD = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// smem: K [NH][BS][128 B] | V [NH][BS][128 B] (128B swizzle) | q [hpg][D] f32 | p [hpg][BS] f32 | ml [hpg][2]
template <int D, int BS, int HPG>
__global__ void __launch_bounds__(kDecThreads) decode_attn_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const __nv_bfloat16* __restrict__ q,
    const int32_t* __restrict__ sel, const int32_t* __restrict__ kv_len, int Lmax, int Hq, int G, int K, int nblk,
    float scale_log2, float* __restrict__ part_o, float* __restrict__ part_ml, uint32_t* status) {
  constexpr int NH = D / 64;
  constexpr uint32_t kHalf = BS * 128;
  constexpr uint32_t kTile = BS * D * 2;
  constexpr int OPT = HPG * D / kDecThreads;  // output elements per thread
  static_assert(OPT >= 1 && OPT <= 8 && (HPG * D) % kDecThreads == 0, "decode output mapping");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* kt = smem;
  uint8_t* vt = kt + kTile;
  float* qs = reinterpret_cast<float*>(vt + kTile);  // [HPG][D]
  float* ps = qs + HPG * D;                          // [HPG][BS]
  float* ml = ps + HPG * BS;                         // [HPG][2]
  uint64_t* bar = reinterpret_cast<uint64_t*>(ml + 2 * HPG);  // HPG*(D+BS+2) floats: 8-byte aligned
  __shared__ int abort_s;

  const int item = blockIdx.x;  // (b, g, k)
  const int k = item % K;
  const int g = (item / K) % G;
  const int b = item / (K * G);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = kv_len[b];
  const int pos = L - 1;
  const int t = sel[(int64_t(b) * G + g) * K + k];
  const bool seq_ok = L >= 1 && L <= Lmax;
  const bool valid = seq_ok && t >= 0 && t < nblk && t * BS <= pos;
  if (tid == 0 && (!seq_ok || t < -1 || t >= nblk)) set_status(status, MSA_ERR_BOUNDS);
  float* out_o = part_o + int64_t(item) * HPG * D;
  float* out_ml = part_ml + int64_t(item) * HPG * 2;
  if (!valid) {  // empty slot: contributes nothing to the combine
    for (int x = tid; x < HPG * D; x += kDecThreads) out_o[x] = 0.f;
    if (tid < HPG) {
      out_ml[2 * tid] = -INFINITY;
      out_ml[2 * tid + 1] = 0.f;
    }
    return;
  }
  if (tid == 0) {
    abort_s = 0;
    tc::mbar_init(bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(bar, 2 * kTile);
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      tc::tma_load_4d(kt + h * kHalf, &tmK, bar, h * 64, g, t * BS, b);
      tc::tma_load_4d(vt + h * kHalf, &tmV, bar, h * 64, g, t * BS, b);
    }
  }
  // the group's query heads, pre-scaled so that exp2 gives the softmax
  for (int x = tid; x < HPG * D; x += kDecThreads) {
    const int hh = x / D, c = x % D;
    qs[x] = __bfloat162float(q[(int64_t(b) * Hq + g * HPG + hh) * D + c]) * scale_log2;
  }
  __syncthreads();
  if (!tc::mbar_wait(bar, 0, &abort_s)) {
    set_status(status, MSA_ERR_TIMEOUT);
    // a copy may still land: wait (bounded) before the CTA gives up its smem
    int zero = 0;
    tc::mbar_wait(bar, 0, &zero);
    return;
  }
  const int nvalid = min(BS, pos - t * BS + 1);  // keys j <= pos in this block

  // scores: thread j owns key j (its K row: 16-byte chunks, swizzle-permuted)
  for (int j = tid; j < BS; j += kDecThreads) {
    float s[HPG];
#pragma unroll
    for (int hh = 0; hh < HPG; ++hh) s[hh] = 0.f;
#pragma unroll
    for (int ch = 0; ch < D / 8; ++ch) {
      const int hf = ch >> 3, cc = ch & 7;
      const uint4 raw = *reinterpret_cast<const uint4*>(kt + hf * kHalf + j * 128 + ((cc ^ (j & 7)) << 4));
      const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
      float kf[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(k2[e]);
        kf[2 * e] = f.x;
        kf[2 * e + 1] = f.y;
      }
#pragma unroll
      for (int hh = 0; hh < HPG; ++hh) {
        const float4 qa = *reinterpret_cast<const float4*>(qs + hh * D + ch * 8);
        const float4 qb = *reinterpret_cast<const float4*>(qs + hh * D + ch * 8 + 4);
        s[hh] = fmaf(qa.x, kf[0], s[hh]);
        s[hh] = fmaf(qa.y, kf[1], s[hh]);
        s[hh] = fmaf(qa.z, kf[2], s[hh]);
        s[hh] = fmaf(qa.w, kf[3], s[hh]);
        s[hh] = fmaf(qb.x, kf[4], s[hh]);
        s[hh] = fmaf(qb.y, kf[5], s[hh]);
        s[hh] = fmaf(qb.z, kf[6], s[hh]);
        s[hh] = fmaf(qb.w, kf[7], s[hh]);
      }
    }
#pragma unroll
    for (int hh = 0; hh < HPG; ++hh) ps[hh * BS + j] = j < nvalid ? s[hh] : -INFINITY;
  }
  __syncthreads();
  // block-local softmax per head (warp per head)
  for (int hh = warp; hh < HPG; hh += kDecThreads / 32) {
    float m = -INFINITY;
    for (int j = lane; j < BS; j += 32) m = fmaxf(m, ps[hh * BS + j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int j = lane; j < BS; j += 32) {
      const float e = j < nvalid ? ex2f(ps[hh * BS + j] - m) : 0.f;
      ps[hh * BS + j] = e;
      l += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) {
      ml[2 * hh] = m;
      ml[2 * hh + 1] = l;
    }
  }
  __syncthreads();
  // O[h][c] = sum_j P[h][j] V[j][c]: thread -> (head, OPT consecutive columns)
  {
    const int o0 = tid * OPT;
    const int hh = o0 / D, c0 = o0 % D;
    const int ch = c0 >> 3, hf = ch >> 3, cc = ch & 7, within = (c0 & 7) * 2;
    float acc[OPT];
#pragma unroll
    for (int x = 0; x < OPT; ++x) acc[x] = 0.f;
    const float* prow = ps + hh * BS;
    for (int j = 0; j < nvalid; ++j) {
      const float pj = prow[j];
      const uint8_t* src = vt + hf * kHalf + j * 128 + ((cc ^ (j & 7)) << 4) + within;
      if constexpr (OPT == 4) {
        const uint2 raw = *reinterpret_cast<const uint2*>(src);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        acc[0] = fmaf(pj, a.x, acc[0]);
        acc[1] = fmaf(pj, a.y, acc[1]);
        acc[2] = fmaf(pj, c.x, acc[2]);
        acc[3] = fmaf(pj, c.y, acc[3]);
      } else {
        const __nv_bfloat16* v16 = reinterpret_cast<const __nv_bfloat16*>(src);
#pragma unroll
        for (int x = 0; x < OPT; ++x) acc[x] = fmaf(pj, __bfloat162float(v16[x]), acc[x]);
      }
    }
#pragma unroll
    for (int x = 0; x < OPT; ++x) out_o[o0 + x] = acc[x];
  }
  if (tid < HPG) {
    out_ml[2 * tid] = ml[2 * tid];
    out_ml[2 * tid + 1] = ml[2 * tid + 1];
  }
}

// one warp per (sequence, query head); lanes own D/32 output columns
template <int D>
__global__ void decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml, int B,
                                      int Hq, int G, int K, __nv_bfloat16* __restrict__ out,
                                      float* __restrict__ lse) {
  constexpr int U = D / 32;
  const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= int64_t(B) * Hq) return;
  const int b = int(wid / Hq), h = int(wid % Hq);
  const int hpg = Hq / G, g = h / hpg, hh = h % hpg;
  const int64_t item0 = (int64_t(b) * G + g) * K;
  float M = -INFINITY;
  for (int k = 0; k < K; ++k) M = fmaxf(M, part_ml[((item0 + k) * hpg + hh) * 2]);
  float acc[U], den = 0.f;
#pragma unroll
  for (int u = 0; u < U; ++u) acc[u] = 0.f;
  if (M > -INFINITY) {
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
      const float* mlk = part_ml + ((item0 + k) * hpg + hh) * 2;
      const float w = ex2f(mlk[0] - M);  // 0 for empty slots (max -inf)
      den = fmaf(w, mlk[1], den);
      const float* ok = part_o + ((item0 + k) * hpg + hh) * D;
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = fmaf(w, ok[lane + 32 * u], acc[u]);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat16* dst = out + (int64_t(b) * Hq + h) * D;
#pragma unroll
  for (int u = 0; u < U; ++u) dst[lane + 32 * u] = __float2bfloat16_rn(acc[u] * inv);
  if (lse && lane == 0) lse[int64_t(b) * Hq + h] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------------------
// decode_index: persistent; tiles = (sequence, 128-key tile) in sequence order
// ---------------------------------------------------------------------------
constexpr int kDiThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kDiStages = 8;
constexpr int kDiMaxB = 4096;
constexpr uint32_t kDiA = 128 * 64 * 2;  // 128 keys x 64 (bf16)
constexpr uint32_t kDiB = 16 * 64 * 2;   // 16 index-query rows (G <= 16, padded)
constexpr uint32_t kDiStage = kDiA + kDiB;

template <int BS>
__global__ void __launch_bounds__(kDiThreads, 1)
    decode_index_kernel(const __grid_constant__ CUtensorMap tmIK, const __grid_constant__ CUtensorMap tmIQ,
                        const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len, int B, int Lmax,
                        int G, int nblk, float* __restrict__ table, uint32_t* status) {
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(128, 16);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* stages = smem;                                              // kDiStages x (A | B)
  int* prefix = reinterpret_cast<int*>(stages + kDiStages * kDiStage);  // [B + 1] tile prefix
  float* red = reinterpret_cast<float*>(prefix + kDiMaxB + 1);          // [2][4][16]
  // mbarriers need 8-byte alignment (the prefix array has an odd length): round up
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(red + 2 * 4 * 16) + 15) & ~uintptr_t(15));
  uint64_t* full = bars;
  uint64_t* empty = full + kDiStages;
  uint64_t* acc_full = empty + kDiStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile prefix over sequences (every CTA builds its own copy)
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {  // tiles cover keys 0..pos of each sequence
      prefix[b] = acc;
      const SeqView sv = seq_view(q_offset, kv_len, b, 1, Lmax, false);
      if (!sv.ok) set_status(status, MSA_ERR_BOUNDS);
      acc += sv.ok ? sv.q0 / 128 + 1 : 0;
    }
    prefix[B] = acc;
    for (int s = 0; s < kDiStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 4);
    }
    tc::mbar_init(done_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 64);
    tc::tmem_relinquish();
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int T = prefix[B];
  const int x0 = int((int64_t(T) * blockIdx.x) / gridDim.x);
  const int x1 = int((int64_t(T) * (blockIdx.x + 1)) / gridDim.x);
  auto locate = [&](int x, int& b, int& kt) {  // tile -> (sequence, key tile)
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
    }
    b = lo;
    kt = x - prefix[lo];
  };
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(status, MSA_ERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int x = x0; x < x1; ++x, ++issued) {
        int b, kt;
        locate(x, b, kt);
        const int s = issued % kDiStages;
        if (!tc::mbar_wait(&empty[s], ((issued / kDiStages) & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        tc::mbar_arrive_expect_tx(&full[s], kDiStage);
        tc::tma_load_3d(stages + s * kDiStage, &tmIK, &full[s], 0, kt * 128, b);
        tc::tma_load_3d(stages + s * kDiStage + kDiA, &tmIQ, &full[s], 0, b * G, 0);
      }
      int zero = 0;
      for (int s = 0; s < kDiStages && s < issued; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % kDiStages);
        tc::mbar_wait(&full[s], (last / kDiStages) & 1, &zero);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int n = 0;
      for (int x = x0; x < x1; ++x, ++n) {
        const int s = n % kDiStages, a = n & 1;
        if (!tc::mbar_wait(&full[s], (n / kDiStages) & 1, abort_flag) ||
            !tc::mbar_wait(&acc_empty[a], ((n >> 1) & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const uint32_t sa = tc::smem_u32(stages + s * kDiStage);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = tc::smem_desc(sa + kk * 32, 16, 1024, 2);
          const uint64_t bd = tc::smem_desc(sa + kDiA + kk * 32, 16, 1024, 2);
          tc::mma_f16_ss(tmem + uint32_t(a) * 32u, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&acc_full[a]);
      }
      int zero = 0;
      tc::mma_commit(done_bar);
      tc::mbar_wait(done_bar, 0, &zero);
    }
  } else {
    // epilogue: thread = key row of the tile (TMEM lane)
    const int q = warp & 3;  // lane quarter
    const int etid = (warp - 2) * 32 + lane;
    int n = 0;
    for (int x = x0; x < x1; ++x, ++n) {
      int b, kt;
      locate(x, b, kt);
      const int a = n & 1;
      if (!tc::mbar_wait(&acc_full[a], (n >> 1) & 1, abort_flag)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      uint32_t v[16];
      tc::tmem_ld_32x32b_x16(tmem + (uint32_t(q * 32) << 16) + uint32_t(a) * 32u, v);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[a]);
      const int j = kt * 128 + q * 32 + lane;
      const bool vis = j <= (q_offset ? q_offset[b] : 0);  // causal: keys up to the query's position
      float* rbuf = red + (n & 1) * 64;
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        if (g < G) {
          const float m = tc::warp_max_f32(vis ? __uint_as_float(v[g]) : -INFINITY);
          if (lane == g) rbuf[q * 16 + g] = m;
        }
      }
      tc::named_bar_sync(1, 128);
      constexpr int kWarpsPerBlock = BS / 32, kBlocksPerTile = 128 / BS;
      if (etid < G * kBlocksPerTile) {
        const int bi = etid / G, g = etid % G;
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarpsPerBlock; ++w) m = fmaxf(m, rbuf[(bi * kWarpsPerBlock + w) * 16 + g]);
        const int t = kt * kBlocksPerTile + bi;
        if (t < nblk) table[(int64_t(b) * G + g) * nblk + t] = m;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 64);
  }
}

// ---------------------------------------------------------------------------
// decode_topk: one CTA per (sequence, group). Candidates are blocks t < loc
// keyed by (block max, -t) as one unsigned 64-bit value; the (K-1)-th largest
// key is found bit by bit with block-wide counts, the selected blocks are
// compacted in ascending t, and loc is appended.
// ---------------------------------------------------------------------------
constexpr int kTkThreads = 256;

__global__ void __launch_bounds__(kTkThreads) decode_topk_kernel(const float* __restrict__ table,
                                                                 const int32_t* __restrict__ q_offset,
                                                                 const int32_t* __restrict__ kv_len, int Lmax, int G,
                                                                 int Bs, int K, int nblk, int32_t* __restrict__ sel,
                                                                 uint32_t* status) {
  __shared__ int wsum[2][kTkThreads / 32];
  __shared__ int scan_s[kTkThreads];
  const int row = blockIdx.x;  // b * G + g
  const int b = row / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* out = sel + int64_t(row) * K;
  const SeqView sv = seq_view(q_offset, kv_len, b, 1, Lmax, false);
  if (!sv.ok) {
    for (int k = tid; k < K; k += kTkThreads) out[k] = -1;
    if (tid == 0) set_status(status, MSA_ERR_BOUNDS);
    return;
  }
  const int loc = sv.q0 / Bs;
  if (loc + 1 <= K) {
    for (int k = tid; k < K; k += kTkThreads) out[k] = k <= loc ? k : -1;
    return;
  }
  const float* M = table + int64_t(row) * nblk;
  const int per = (loc + kTkThreads - 1) / kTkThreads;  // contiguous candidates per thread
  const int t0 = min(loc, tid * per), t1 = min(loc, t0 + per);
  const int need = K - 1;
  uint64_t prefix = 0;
  for (int bit = 63; bit >= 0; --bit) {
    const uint64_t cand = prefix | (uint64_t(1) << bit);
    int c = 0;
    for (int t = t0; t < t1; ++t) c += rank_key(M[t], t) >= cand;
    c = __reduce_add_sync(0xffffffffu, c);
    const int par = bit & 1;
    if (lane == 0) wsum[par][warp] = c;
    __syncthreads();
    int total = 0;
#pragma unroll
    for (int w = 0; w < kTkThreads / 32; ++w) total += wsum[par][w];
    if (total >= need) prefix = cand;  // the need-th largest key is >= cand
  }
  // keys >= prefix are exactly the top K-1 (keys are unique)
  int c = 0;
  for (int t = t0; t < t1; ++t) c += rank_key(M[t], t) >= prefix;
  scan_s[tid] = c;
  __syncthreads();
  for (int off = 1; off < kTkThreads; off <<= 1) {
    const int v = tid >= off ? scan_s[tid - off] : 0;
    __syncthreads();
    scan_s[tid] += v;
    __syncthreads();
  }
  int o = scan_s[tid] - c;
  for (int t = t0; t < t1; ++t)
    if (rank_key(M[t], t) >= prefix) out[o++] = t;
  if (tid == 0) out[K - 1] = loc;
}

size_t dec_smem_bytes(int d, int Bs, int hpg) {
  return 1024 + size_t(2) * Bs * d * 2 + size_t(hpg) * d * 4 + size_t(hpg) * Bs * 4 + size_t(hpg) * 8 + 64;
}

}  // namespace

bool decode_attn_supported(int dtype, int Hq, int Hkv, int d, int Bs, int K) {
  if (dtype != MSA_BF16 || (d != 64 && d != 128)) return false;
  if (Bs != 32 && Bs != 64 && Bs != 128) return false;
  if (K < 1 || K > kMaxK || Hq % Hkv != 0) return false;
  const int hpg = Hq / Hkv;
  if (hpg != 1 && hpg != 2 && hpg != 4 && hpg != 8) return false;
  if ((hpg * d) % kDecThreads != 0 || hpg * d / kDecThreads > 8) return false;
  return dec_smem_bytes(d, Bs, hpg) <= 227 * 1024;
}

size_t decode_ws_bytes(int B, int Hq, int Hkv, int d, int K) {
  const size_t items = size_t(B) * Hkv * K, hpg = size_t(Hq / Hkv);
  const size_t o = (items * hpg * d * 4 + 255) & ~size_t(255);
  const size_t m = (items * hpg * 2 * 4 + 255) & ~size_t(255);
  return o + m;
}

cudaError_t launch_decode_attn(const void* q, const void* k_cache, const void* v_cache, const int32_t* sel,
                               const int32_t* kv_len, int B, int Lmax, int Hq, int Hkv, int d, int Bs, int K,
                               float scale, void* out, float* lse, void* scratch, uint32_t* status,
                               cudaStream_t stream) {
  const int G = Hkv, hpg = Hq / Hkv, nblk = (Lmax + Bs - 1) / Bs;
  const size_t items = size_t(B) * G * K;
  float* part_o = static_cast<float*>(scratch);
  float* part_ml =
      reinterpret_cast<float*>(static_cast<char*>(scratch) + ((items * hpg * d * 4 + 255) & ~size_t(255)));
  CUtensorMap tmK, tmV;
  const uint64_t dims[4] = {uint64_t(d), uint64_t(Hkv), uint64_t(Lmax), uint64_t(B)};
  const uint64_t strides[3] = {uint64_t(d) * 2, uint64_t(Hkv) * d * 2, uint64_t(Lmax) * Hkv * d * 2};
  const uint32_t box[4] = {64, 1, uint32_t(Bs), 1};
  if (!make_tmap_bf16(&tmK, k_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tmV, v_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const size_t smem = dec_smem_bytes(d, Bs, hpg);
  const float scale_log2 = scale * kLog2eD;
  cudaError_t e;
  {
    ProfScope pf("decode_attn", stream);
#define MSA_DEC(D_, BS_, HPG_)                                                                                   \
  do {                                                                                                           \
    auto kern = decode_attn_kernel<D_, BS_, HPG_>;                                                              \
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess) \
      return e;                                                                                                  \
    kern<<<unsigned(items), kDecThreads, smem, stream>>>(tmK, tmV, static_cast<const __nv_bfloat16*>(q), sel,     \
                                                         kv_len, Lmax, Hq, G, K, nblk, scale_log2, part_o,        \
                                                         part_ml, status);                                        \
  } while (0)
#define MSA_DEC_BS(D_, HPG_)      \
  do {                            \
    if (Bs == 128)                \
      MSA_DEC(D_, 128, HPG_);     \
    else if (Bs == 64)            \
      MSA_DEC(D_, 64, HPG_);      \
    else                          \
      MSA_DEC(D_, 32, HPG_);      \
  } while (0)
    if (d == 128) {
      if (hpg == 4)
        MSA_DEC_BS(128, 4);
      else if (hpg == 8)
        MSA_DEC_BS(128, 8);
      else if (hpg == 2)
        MSA_DEC_BS(128, 2);
      else
        MSA_DEC_BS(128, 1);
    } else {
      if (hpg == 4)
        MSA_DEC_BS(64, 4);
      else if (hpg == 8)
        MSA_DEC_BS(64, 8);
      else
        MSA_DEC_BS(64, 2);
    }
#undef MSA_DEC_BS
#undef MSA_DEC
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    ProfScope pf("decode_combine", stream);
    const int64_t warps = int64_t(B) * Hq;
    const unsigned grid = unsigned((warps * 32 + 255) / 256);
    if (d == 128)
      decode_combine_kernel<128><<<grid, 256, 0, stream>>>(part_o, part_ml, B, Hq, G, K,
                                                          static_cast<__nv_bfloat16*>(out), lse);
    else
      decode_combine_kernel<64><<<grid, 256, 0, stream>>>(part_o, part_ml, B, Hq, G, K,
                                                         static_cast<__nv_bfloat16*>(out), lse);
  }
  return cudaGetLastError();
}

bool decode_index_supported(int dtype, int B, int Nq, int G, int di, int Bs, int K) {
  return dtype == MSA_BF16 && Nq == 1 && di == 64 && G >= 1 && G <= 16 && B >= 1 && B <= kDiMaxB &&
         (Bs == 32 || Bs == 64 || Bs == 128) && K >= 1 && K <= kMaxK;
}

size_t decode_index_ws_bytes(int B, int G, int Nk, int Bs) {
  return size_t(B) * G * ((Nk + Bs - 1) / Bs) * sizeof(float);
}

cudaError_t launch_decode_index(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len, int B,
                                int Lmax, int G, int Bs, int K, int32_t* sel, float* table, uint32_t* status,
                                cudaStream_t stream) {
  const int nblk = (Lmax + Bs - 1) / Bs;
  CUtensorMap tmIK, tmIQ;
  {
    const uint64_t dims[3] = {64, uint64_t(Lmax), uint64_t(B)};
    const uint64_t strides[2] = {128, uint64_t(Lmax) * 128};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_tmap_bf16(&tmIK, ik, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {64, uint64_t(B) * G, 1};
    const uint64_t strides[2] = {128, uint64_t(B) * G * 128};
    const uint32_t box[3] = {64, 16, 1};
    if (!make_tmap_bf16(&tmIQ, iq, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  const size_t smem = 1024 + size_t(kDiStages) * kDiStage + (kDiMaxB + 1) * 4 + 2 * 4 * 16 * 4 + 16 +
                      (2 * kDiStages + 5) * 8 + 16;
  int dev = 0, sms = kNumSMs;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e;
  {
    ProfScope pf("decode_index", stream);
#define MSA_DI(BS_)                                                                                              \
  do {                                                                                                           \
    auto kern = decode_index_kernel<BS_>;                                                                       \
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess) \
      return e;                                                                                                  \
    kern<<<sms, kDiThreads, smem, stream>>>(tmIK, tmIQ, q_offset, kv_len, B, Lmax, G, nblk, table, status);     \
  } while (0)
    if (Bs == 128)
      MSA_DI(128);
    else if (Bs == 64)
      MSA_DI(64);
    else
      MSA_DI(32);
#undef MSA_DI
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    ProfScope pf("decode_topk", stream);
    decode_topk_kernel<<<B * G, kTkThreads, 0, stream>>>(table, q_offset, kv_len, Lmax, G, Bs, K, nblk, sel, status);
  }
  return cudaGetLastError();
}

}  // namespace msa
