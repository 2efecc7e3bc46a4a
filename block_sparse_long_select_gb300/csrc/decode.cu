// Main Branch, decode: one new token per sequence attends to its KV cache
// through the K selected blocks of each group (hyper.ai summary of paper
// 2606.13392, "方法": softmax attention over the selected blocks' keys and
// values; "一句话总结": the decode half of the prefill / decode speedups).
//
//  decode_index    Index Branch for one query per sequence: the index-key
//                  cache streamed once by TMA in 128-key tiles, scores on
//                  tcgen05 (keys along M, the G index-query heads along N),
//                  32-key sub-block maxima straight from TMEM (one warp
//                  redux each) into a small [B, G, Lmax/32] table
//  decode_topk     exact top-K per (sequence, group): block maxima assembled
//                  from the sub-block maxima, the query's own block forced,
//                  ascending output
//  decode_attn     one CTA per (sequence, group, selected block): the block's
//                  K and V rows of that group are TMA-loaded (128B-swizzled,
//                  so a thread reading "its" key row is bank-conflict free),
//                  scores for the group's query heads, a block-local softmax,
//                  P.V in fp32 -> per-slot partial (O unnormalised, max, sum)
//                  The last of the K slot CTAs of a (sequence, group) (an
//                  arrival counter, not an output atomic) merges the slot
//                  partials in slot order by log-sum-exp -> bf16 rows (+ lse)
//
// The step streams each selected K/V block from HBM exactly once; partials
// are small (B x G x K x hpg x (d + 2) fp32) and stay in L2.
#include <cmath>

#include "msa_internal.cuh"
#include "tc_utils.cuh"

namespace msa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2eD = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// decode_attn (+ combine by the last CTA of each (sequence, group))
// smem: K [NH][BS][128 B] | V [NH][BS][128 B] (TMA, 128B swizzle) |
//       S [HPG][BS] f32 | P [HPG][BS + 8] bf16 | ml [HPG][2] | 2 mbarriers
// Both products run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate): S^T = K q^T with keys along M and the group's heads along N
// (padded to 8), O^T = V^T P^T with head dims along M; operands come straight
// from the swizzled K/V tiles through ldmatrix (.trans for V).
// ---------------------------------------------------------------------------
constexpr int kDecThreads = 256;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// address of 16-byte chunk `ch` (8 columns) of row `row` in a 128B-swizzled [NH][rows][128 B] tile
__device__ __forceinline__ uint32_t swz_addr(uint32_t base, uint32_t half_bytes, int row, int ch) {
  return base + uint32_t(ch >> 3) * half_bytes + uint32_t(row) * 128u + ((uint32_t(ch & 7) ^ uint32_t(row & 7)) << 4);
}

template <int D, int BS, int HPG>
__global__ void __launch_bounds__(kDecThreads) decode_attn_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const __nv_bfloat16* __restrict__ q,
    const int32_t* __restrict__ sel, const int32_t* __restrict__ kv_len, int Lmax, int Hq, int G, int K, int nblk,
    float scale_log2, float* __restrict__ part_o, float* __restrict__ part_ml, int* __restrict__ arrivals,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, uint32_t* status, int inject_timeout) {
  constexpr int NH = D / 64;
  constexpr uint32_t kHalf = BS * 128;
  constexpr uint32_t kTile = BS * D * 2;
  constexpr int kOut = HPG * D;  // outputs per (sequence, group)
  constexpr int kPS = BS + 8;    // padded P row (bf16)
  static_assert(HPG <= 8, "heads of a group must fit the N = 8 of one MMA");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* kt = smem;
  uint8_t* vt = kt + kTile;
  float* ss = reinterpret_cast<float*>(vt + kTile);                          // [HPG][BS] scores (log2 units)
  __nv_bfloat16* pb = reinterpret_cast<__nv_bfloat16*>(ss + HPG * BS);       // [HPG][kPS] probabilities
  float* ml = reinterpret_cast<float*>(pb + HPG * kPS);                      // [HPG][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(ml + 2 * HPG) + 15) & ~uintptr_t(15));
  __shared__ int abort_s, last_s;

  const int item = blockIdx.x;  // (b, g, k)
  const int k = item % K;
  const int bg = item / K;
  const int g = bg % G;
  const int b = bg / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment coordinates
  const int L = kv_len[b];
  const int pos = L - 1;
  tc::griddep_launch_dependents();
  tc::griddep_wait();  // launched early behind the top-K: sel is its output
  const int t = sel[int64_t(bg) * K + k];
  const bool seq_ok = L >= 1 && L <= Lmax;
  const bool valid = seq_ok && t >= 0 && t < nblk && t * BS <= pos;
  if (tid == 0 && (!seq_ok || t < -1 || t >= nblk)) set_status(status, MSA_ERR_BOUNDS);
  float* out_o = part_o + int64_t(item) * kOut;
  float* out_ml = part_ml + int64_t(item) * HPG * 2;

  if (valid) {
    if (tid == 0) {
      abort_s = 0;
      tc::mbar_init(&bars[0], 1);
      tc::mbar_init(&bars[1], 1);
      tc::mbar_init(&bars[2], 1);  // nothing arrives on it (timeout injection)
      tc::fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {  // K and V on separate barriers: scores start while V is in flight
      tc::mbar_arrive_expect_tx(&bars[0], kTile);
      tc::mbar_arrive_expect_tx(&bars[1], kTile);
#pragma unroll
      for (int h = 0; h < NH; ++h) tc::tma_load_4d(kt + h * kHalf, &tmK, &bars[0], h * 64, g, t * BS, b);
#pragma unroll
      for (int h = 0; h < NH; ++h) tc::tma_load_4d(vt + h * kHalf, &tmV, &bars[1], h * 64, g, t * BS, b);
    }
    // q^T fragments (B operand of S^T = K q^T): column n = head gq, rows = head dims
    uint32_t qf[D / 16][2];
    {
      const __nv_bfloat16* qh = q + (int64_t(b) * Hq + g * HPG + gq) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        if (gq < HPG) {
          qf[ks][0] = *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 2 * tq);
          qf[ks][1] = *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 2 * tq + 8);
        } else {
          qf[ks][0] = qf[ks][1] = 0u;
        }
      }
    }
    const int nvalid = min(BS, pos - t * BS + 1);  // keys j <= pos in this block
    if (inject_timeout && tid == 0 && !tc::mbar_wait_for(&bars[2], 0, &abort_s, tc::kInjectedWaitCycles))
      abort_s = 1;
    __syncthreads();
    // every thread of the CTA takes the same branch below (the MMAs are warp-wide)
    bool ok = __syncthreads_and(!abort_s && tc::mbar_wait(&bars[0], 0, &abort_s));
    if (ok && warp < BS / 16) {
      // S^T tile: keys [16 warp, 16 warp + 16) x heads
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t kbase = tc::smem_u32(kt);
      const int row = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(swz_addr(kbase, kHalf, row, ks * 2 + (lane >> 4)), a0, a1, a2, a3);
        mma_bf16_16816(acc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
      }
      // acc: keys (gq, gq + 8) x heads (2 tq, 2 tq + 1)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = warp * 16 + gq + 8 * (e >> 1);
        const int hh = 2 * tq + (e & 1);
        if (hh < HPG) ss[hh * BS + key] = key < nvalid ? acc[e] * scale_log2 : -INFINITY;
      }
    }
    __syncthreads();
    if (ok) {
      // block-local softmax per head (warp per head); P as bf16
      for (int hh = warp; hh < HPG; hh += kDecThreads / 32) {
        float m = -INFINITY;
        for (int j = lane; j < BS; j += 32) m = fmaxf(m, ss[hh * BS + j]);
        m = tc::warp_max_f32(m);
        float l = 0.f;
        for (int j = lane; j < BS; j += 32) {
          const float e = j < nvalid ? ex2f(ss[hh * BS + j] - m) : 0.f;
          pb[hh * kPS + j] = __float2bfloat16_rn(e);
          l += e;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) {
          ml[2 * hh] = m;
          ml[2 * hh + 1] = l;
        }
      }
    }
    __syncthreads();
    ok = __syncthreads_and(ok && tc::mbar_wait(&bars[1], 0, &abort_s));
    if (ok) {
      // O^T tile: head dims [16 warp, 16 warp + 16) x heads, over all keys
      if (warp < D / 16) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t vbase = tc::smem_u32(vt);
        const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
        for (int ks = 0; ks < BS / 16; ++ks) {
          uint32_t a0, a1, a2, a3;
          const int key = ks * 16 + r8 + 8 * (mi >> 1);
          ldsm_x4_t(swz_addr(vbase, kHalf, key, warp * 2 + (mi & 1)), a0, a1, a2, a3);
          uint32_t b0 = 0u, b1 = 0u;
          if (gq < HPG) {
            b0 = *reinterpret_cast<const uint32_t*>(pb + gq * kPS + ks * 16 + 2 * tq);
            b1 = *reinterpret_cast<const uint32_t*>(pb + gq * kPS + ks * 16 + 2 * tq + 8);
          }
          mma_bf16_16816(acc, a0, a1, a2, a3, b0, b1);
        }
        // acc: head dims (gq, gq + 8) x heads (2 tq, 2 tq + 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = warp * 16 + gq + 8 * (e >> 1);
          const int hh = 2 * tq + (e & 1);
          if (hh < HPG) out_o[hh * D + c] = acc[e];
        }
      }
      if (tid < HPG) {
        out_ml[2 * tid] = ml[2 * tid];
        out_ml[2 * tid + 1] = ml[2 * tid + 1];
      }
    } else {
      // gave up: record it, let the copies land (bounded) before the CTA
      // releases its shared memory, and leave an empty slot for the merge. The
      // CTA still counts its arrival below, so the (sequence, group) counter
      // returns to zero and the workspace stays usable.
      if (tid == 0) set_status(status, MSA_ERR_TIMEOUT);
      int zero = 0;
      tc::mbar_wait(&bars[0], 0, &zero);
      tc::mbar_wait(&bars[1], 0, &zero);
      for (int x = tid; x < kOut; x += kDecThreads) out_o[x] = 0.f;
      if (tid < HPG) {
        out_ml[2 * tid] = -INFINITY;
        out_ml[2 * tid + 1] = 0.f;
      }
    }
  } else {  // empty slot: contributes nothing to the merge
    for (int x = tid; x < kOut; x += kDecThreads) out_o[x] = 0.f;
    if (tid < HPG) {
      out_ml[2 * tid] = -INFINITY;
      out_ml[2 * tid + 1] = 0.f;
    }
  }
  // ---- the last of the K slot CTAs of (b, g) merges the partials ----
  // The barrier orders every thread's partial stores before thread 0's
  // device-scope fence, which (being cumulative) publishes them all before
  // its arrival; one fence instead of one per thread.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(&arrivals[bg], 1);
    last_s = old == K - 1;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  if (tid == 0) arrivals[bg] = 0;  // ready for the next call
  const float* po = part_o + int64_t(bg) * K * kOut;
  const float* pm = part_ml + int64_t(bg) * K * HPG * 2;
  // Weights first, one warp per head: every slot's (max, sum) in one round of
  // loads, the head's maximum M and denominator, and each slot's normalised
  // weight exp(m - M) / den into shared memory (the K tile's space, which
  // this CTA no longer reads). Then every output sums its slots with all of
  // a thread's loads of a round in flight at once.
  float* wts = reinterpret_cast<float*>(kt);  // [K][HPG]
  float* hstat = wts + K * HPG;               // [HPG][2]: M, den
  static_assert(kMaxK <= 64 && HPG <= kDecThreads / 32, "two slots per lane, one warp per head");
  if (warp < HPG) {
    const int hh = warp;
    float mv[2], lv[2], M = -INFINITY;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int kk = lane + 32 * x;
      mv[x] = kk < K ? __ldcg(pm + (kk * HPG + hh) * 2) : -INFINITY;
      lv[x] = kk < K ? __ldcg(pm + (kk * HPG + hh) * 2 + 1) : 0.f;
      M = fmaxf(M, mv[x]);
    }
    M = tc::warp_max_f32(M);
    float w[2], den = 0.f;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      w[x] = M > -INFINITY ? ex2f(mv[x] - M) : 0.f;  // 0 for empty slots
      den = fmaf(w[x], lv[x], den);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (lane + 32 * x < K) wts[(lane + 32 * x) * HPG + hh] = w[x] * inv;
    if (lane == 0) {
      hstat[2 * hh] = M;
      hstat[2 * hh + 1] = den;
    }
  }
  __syncthreads();
  constexpr int kPer = (kOut + kDecThreads - 1) / kDecThreads;  // outputs per thread
  float acc[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < K; ++kk) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int o = tid + j * kDecThreads;
      if (kPer * kDecThreads == kOut || o < kOut)
        acc[j] = fmaf(wts[kk * HPG + o / D], __ldcg(po + int64_t(kk) * kOut + o), acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int o = tid + j * kDecThreads;
    if (kPer * kDecThreads != kOut && o >= kOut) continue;
    const int hh = o / D, c = o % D;
    const int h = g * HPG + hh;
    out[(int64_t(b) * Hq + h) * D + c] = __float2bfloat16_rn(acc[j]);  // weights are 0 when den = 0
    if (lse && c == 0) {
      const float den = hstat[2 * hh + 1];
      lse[int64_t(b) * Hq + h] = den > 0.f ? (hstat[2 * hh] + log2f(den)) * kLn2 : -INFINITY;
    }
  }
}

size_t dec_smem_bytes(int d, int Bs, int hpg) {
  return 1024 + size_t(2) * Bs * d * 2 + size_t(hpg) * Bs * 4 + size_t(hpg) * (Bs + 8) * 2 + size_t(hpg) * 8 + 16 +
         32;
}

// ---------------------------------------------------------------------------
// decode_index: persistent; tiles = (sequence, 128-key tile) in sequence order.
// Warps: 0 TMA, 1 MMA + TMEM owner, 2-9 two epilogue warpgroups that take
// alternate tiles (4 TMEM accumulators of 32 columns). Each warp reduces its
// 32 keys per index-query head with one redux and writes the 32-key sub-block
// maximum; the top-K pass assembles block maxima from those.
// ---------------------------------------------------------------------------
constexpr int kDiThreads = 320;
constexpr int kDiStages = 12;
constexpr int kDiMaxB = 1024;
constexpr int kDiAcc = 4;
constexpr uint32_t kDiA = 128 * 64 * 2;  // 128 keys x 64 (bf16)
constexpr uint32_t kDiB = 16 * 64 * 2;   // 16 index-query rows (G <= 16, padded)
constexpr uint32_t kDiStage = kDiA + kDiB;

__global__ void __launch_bounds__(kDiThreads, 1)
    decode_index_kernel(const __grid_constant__ CUtensorMap tmIK, const __grid_constant__ CUtensorMap tmIQ,
                        const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len, int B, int Lmax,
                        int G, int nsub, float* __restrict__ sub_max, uint32_t* status) {
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(128, 16);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* stages = smem;                                              // kDiStages x (A | B)
  int* prefix = reinterpret_cast<int*>(stages + kDiStages * kDiStage);  // [B + 1] tile prefix
  int* qpos = prefix + kDiMaxB + 1;                                     // [B] query position
  // mbarriers need 8-byte alignment: round up past the int arrays
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(qpos + kDiMaxB) + 15) & ~uintptr_t(15));
  uint64_t* full = bars;
  uint64_t* empty = full + kDiStages;
  uint64_t* acc_full = empty + kDiStages;
  uint64_t* acc_empty = acc_full + kDiAcc;
  uint64_t* done_bar = acc_empty + kDiAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tc::griddep_launch_dependents();  // the top-K may launch now; it waits for this grid's maxima

  __shared__ int scan_part[kDiThreads];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDiStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kDiAcc; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 4);
    }
    tc::mbar_init(done_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  // per-sequence tile counts (tiles cover keys 0..pos), then their prefix
  for (int b = threadIdx.x; b < B; b += kDiThreads) {
    const SeqView sv = seq_view(q_offset, kv_len, b, 1, Lmax, false);
    if (!sv.ok) set_status(status, MSA_ERR_BOUNDS);
    qpos[b] = sv.ok ? sv.q0 : -1;
    prefix[b] = sv.ok ? sv.q0 / 128 + 1 : 0;
  }
  __syncthreads();
  {
    const int per = (B + kDiThreads - 1) / kDiThreads;
    const int lo = min(B, int(threadIdx.x) * per), hi = min(B, lo + per);
    int local = 0;
    for (int b = lo; b < hi; ++b) local += prefix[b];
    scan_part[threadIdx.x] = local;
    __syncthreads();
    if (threadIdx.x == 0) {
      int run = 0;
      for (int i = 0; i < kDiThreads; ++i) {
        const int v = scan_part[i];
        scan_part[i] = run;
        run += v;
      }
      prefix[B] = run;
    }
    __syncthreads();
    int base = scan_part[threadIdx.x];
    for (int b = lo; b < hi; ++b) {
      const int c = prefix[b];
      prefix[b] = base;
      base += c;
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 128);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tmIK);
    tc::tma_prefetch(&tmIQ);
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
  // tiles are visited in increasing order: advance the sequence cursor instead of searching
  auto advance = [&](int x, int& b, int& kt) {
    while (b + 1 < B && prefix[b + 1] <= x) ++b;
    kt = x - prefix[b];
  };
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(status, MSA_ERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0, b = 0, kt = 0;
      if (x0 < x1) locate(x0, b, kt);
      for (int x = x0; x < x1; ++x, ++issued) {
        advance(x, b, kt);
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
      constexpr uint32_t kDescHi = tc::smem_desc_hi(1024, 2);  // 128B swizzle, 8-row groups 1024 B apart
      const uint32_t stage_lo0 = tc::smem_desc_lo(tc::smem_u32(stages), 16);
      int n = 0;
      for (int x = x0; x < x1; ++x, ++n) {
        const int s = n % kDiStages, a = n % kDiAcc;
        if (!tc::mbar_wait(&full[s], (n / kDiStages) & 1, abort_flag) ||
            !tc::mbar_wait(&acc_empty[a], ((n / kDiAcc) & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        // descriptors from low words: the stage's first 16-column slice plus 32 bytes per slice
        const uint32_t a_lo = stage_lo0 + uint32_t(s) * (kDiStage >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f16_ss_lo<kDescHi>(tmem + uint32_t(a) * 32u, a_lo + uint32_t(kk * 2), a_lo + (kDiA >> 4) + uint32_t(kk * 2),
                                     kIdesc, kk > 0 ? 1u : 0u);
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&acc_full[a]);
      }
      int zero = 0;
      tc::mma_commit(done_bar);
      tc::mbar_wait(done_bar, 0, &zero);
    }
  } else {
    // epilogue: warpgroup w takes tiles n = w, w + 2, ...; thread = key row
    const int w = (warp - 2) >> 2;
    const int q = warp & 3;  // TMEM lane quarter
    int b = 0, kt = 0;
    if (x0 + w < x1) locate(x0 + w, b, kt);
    for (int n = w; x0 + n < x1; n += 2) {
      advance(x0 + n, b, kt);
      const int a = n % kDiAcc;
      if (!tc::mbar_wait(&acc_full[a], (n / kDiAcc) & 1, abort_flag)) {
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
      const int sblk = kt * 4 + q;           // 32-key sub-block of this warp
      const bool vis = sblk * 32 + lane <= qpos[b];
      float* dst = sub_max + int64_t(b) * G * nsub + sblk;
      // all warp reductions first (independent), then one store per lane
      float mine = -INFINITY;
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        if (g < G) {  // uniform: the padding columns are skipped
          const float m = tc::warp_max_f32(vis ? __uint_as_float(v[g]) : -INFINITY);
          mine = lane == g ? m : mine;
        }
      }
      if (lane < G && sblk < nsub) dst[int64_t(lane) * nsub] = mine;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 128);
  }
}


// Exact top-K of one (sequence, group) row by one warp, from the row's 32-key
// sub-block maxima. Candidates are the blocks t < loc; their maxima become
// order-preserving 32-bit values in registers (block t = lane + 32 j). The
// (K-1)-th largest value v* is found two bits per round with warp sums; then
// every candidate above v* is taken, plus the lowest-t candidates equal to v*
// (ties go to the lower block), compacted in ascending t by ballots; the
// local block loc closes the row. A row that sees at most K blocks takes them
// all.
constexpr int kWarpTopkPer = 32;  // candidates per lane: rows of up to 1024 blocks
// R = sub-blocks per block (Bs / 32). The row's loc * R sub-block maxima are
// first staged in the warp's shared-memory buffer (16-byte cp.async, all in
// flight together), then each lane takes the maxima of its blocks.
template <int R>
__device__ void warp_topk_row(const float* __restrict__ sm, int loc, int K, int fs, int32_t* __restrict__ out,
                              int lane, float* buf) {
  if (loc + 1 <= K) {
    for (int k = lane; k < K; k += 32) out[k] = k <= loc ? k : -1;
    return;
  }
  const int n = loc * R;  // floats; the row starts on 16 bytes
  const uint32_t sbuf = tc::smem_u32(buf);
  for (int i = lane * 4; i < n; i += 128) {
    const uint32_t bytes = uint32_t(min(4, n - i)) * 4u;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sbuf + uint32_t(i) * 4u), "l"(sm + i),
                 "r"(bytes)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncwarp();
  // Candidate values are >= 1 (an order-preserving key of 0 is raised to 1;
  // only a NaN pattern has it) and padding is 0. Every threshold tested below
  // is >= 1, so padding is never counted or taken and no loop needs a branch.
  uint32_t v[kWarpTopkPer];
#pragma unroll
  for (int j = 0; j < kWarpTopkPer; ++j) {
    const int t = lane + 32 * j;
    float m = -INFINITY;
#pragma unroll
    for (int r = 0; r < R; ++r) m = fmaxf(m, buf[(t < loc ? t : 0) * R + r]);
    v[j] = (t < loc && t >= fs) ? max(ord_f32(m), 1u) : 0u;  // fs = 1: block 0 is kept outright
  }
  const int need = K - 1 - fs;
  if (fs && lane == 0) out[0] = 0;
  out += fs;  // the ranked blocks follow block 0
  if (need == 0) {
    if (lane == 0) out[0] = loc;
    return;
  }
  const unsigned lt_mask = (1u << lane) - 1u;
  if (need <= 32) {
    // The need-th largest lane maximum T bounds v* from below (need lanes
    // hold a value >= T), so only candidates >= T can be selected. They are
    // gathered in ascending t and ranked exactly by (value desc, t asc).
    uint32_t lm = v[0];
#pragma unroll
    for (int j = 1; j < kWarpTopkPer; ++j) lm = max(lm, v[j]);
    int lrank = 0;  // rank of this lane's maximum among the lanes' (ties to the lower lane)
#pragma unroll
    for (int o = 0; o < 32; ++o) {
      const uint32_t x = __shfl_sync(0xffffffffu, lm, o);
      lrank += (x > lm) || (x == lm && o < lane);
    }
    const unsigned at = __ballot_sync(0xffffffffu, lrank == need - 1);
    const uint32_t T = max(__shfl_sync(0xffffffffu, lm, __ffs(at) - 1), 1u);
    int c = 0;
#pragma unroll
    for (int j = 0; j < kWarpTopkPer; ++j) c += v[j] >= T;
    const int C = __reduce_add_sync(0xffffffffu, c);
    if (C <= 64) {
      uint32_t* cv = reinterpret_cast<uint32_t*>(buf);  // the staged row is no longer needed
      int* ct = reinterpret_cast<int*>(buf) + 64;
      __syncwarp();
      int base = 0;
#pragma unroll
      for (int j = 0; j < kWarpTopkPer; ++j) {
        const bool f = v[j] >= T;
        const unsigned fm = __ballot_sync(0xffffffffu, f);
        if (f) {
          const int q = base + __popc(fm & lt_mask);
          cv[q] = v[j];
          ct[q] = lane + 32 * j;
        }
        base += __popc(fm);
      }
      __syncwarp();
      bool take[2];
      int tt[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        const uint32_t vi = i < C ? cv[i] : 0u;
        tt[h] = i < C ? ct[i] : 0;
        int rank = 0;
        for (int x = 0; x < C; ++x) rank += (cv[x] > vi) || (cv[x] == vi && x < i);  // candidate x has the lower t
        take[h] = i < C && rank < need;
      }
      int o = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // candidates are in ascending t: compact the taken ones
        const unsigned tm = __ballot_sync(0xffffffffu, take[h]);
        if (take[h]) out[o + __popc(tm & lt_mask)] = tt[h];
        o += __popc(tm);
      }
      if (lane == 0) out[need] = loc;
      return;
    }
  }
  uint32_t prefix = 0;
  for (int round = 0; round < 16; ++round) {
    const int sh = 30 - 2 * round;
    const uint32_t c1 = prefix | (1u << sh), c2 = prefix | (2u << sh), c3 = prefix | (3u << sh);
    int n1 = 0, n2 = 0, n3 = 0;
#pragma unroll
    for (int j = 0; j < kWarpTopkPer; ++j) {
      n1 += v[j] >= c1;
      n2 += v[j] >= c2;
      n3 += v[j] >= c3;
    }
    n1 = __reduce_add_sync(0xffffffffu, n1);
    n2 = __reduce_add_sync(0xffffffffu, n2);
    n3 = __reduce_add_sync(0xffffffffu, n3);
    const uint32_t best = n3 >= need ? 3u : (n2 >= need ? 2u : (n1 >= need ? 1u : 0u));  // counts fall as the value grows
    prefix |= best << sh;
  }
  // prefix = v* >= 1, the need-th largest value
  int gt = 0;
#pragma unroll
  for (int j = 0; j < kWarpTopkPer; ++j) gt += v[j] > prefix;
  const int ties = need - __reduce_add_sync(0xffffffffu, gt);
  int base = 0, eq_seen = 0;
#pragma unroll
  for (int j = 0; j < kWarpTopkPer; ++j) {
    const int t = lane + 32 * j;
    const bool eqf = v[j] == prefix;
    const unsigned eqm = __ballot_sync(0xffffffffu, eqf);
    const bool take = v[j] > prefix || (eqf && eq_seen + __popc(eqm & lt_mask) < ties);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) out[base + __popc(tm & lt_mask)] = t;
    base += __popc(tm);
    eq_seen += __popc(eqm);
  }
  if (lane == 0) out[need] = loc;
}

// ---------------------------------------------------------------------------
// decode_topk: one CTA per (sequence, group). Block maxima of the candidates
// t < loc are assembled from the 32-key sub-block maxima and cached in shared
// memory as order-preserving 32-bit values. The (K-1)-th largest value v* is
// found two bits per round with block-wide counts; then every candidate above
// v* is selected, plus the lowest-t candidates equal to v* until K-1 are
// chosen (ties go to the lower block). Selected blocks are compacted in
// ascending t and the local block is appended.
// ---------------------------------------------------------------------------
constexpr int kTkThreads = 256;
constexpr int kTkMaxCand = 16384;


// exclusive block-wide scan of one int per thread (kTkThreads threads)
__device__ __forceinline__ int block_exclusive_scan(int v, int* buf) {
  const int tid = threadIdx.x;
  buf[tid] = v;
  __syncthreads();
  for (int off = 1; off < kTkThreads; off <<= 1) {
    const int x = tid >= off ? buf[tid - off] : 0;
    __syncthreads();
    buf[tid] += x;
    __syncthreads();
  }
  const int incl = buf[tid];
  __syncthreads();
  return incl - v;
}

__global__ void __launch_bounds__(kTkThreads) decode_topk_kernel(const float* __restrict__ sub_max,
                                                                 const int32_t* __restrict__ q_offset,
                                                                 const int32_t* __restrict__ kv_len, int Lmax, int G,
                                                                 int Bs, int K, int fs, int nsub,
                                                                 int32_t* __restrict__ sel, uint32_t* status) {
  extern __shared__ uint32_t vals[];  // [loc] order-preserving block maxima
  __shared__ int wsum[2][kTkThreads / 32][3];
  __shared__ int scan_buf[kTkThreads];
  const int row = blockIdx.x;  // b * G + g
  const int b = row / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  tc::griddep_launch_dependents();  // attention may launch now; it waits for the selection
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
  const int R = Bs / 32;  // sub-blocks per block
  const float* sm = sub_max + int64_t(row) * nsub;
  const int need = K - 1 - fs;  // fs = 1: block 0 is kept outright, like the local block
  if (need == 0) {
    if (tid == 0) {
      out[0] = 0;
      out[1] = loc;
    }
    return;
  }
  tc::griddep_wait();  // the sub-block maxima come from the index kernel
  const int per = (loc + kTkThreads - 1) / kTkThreads;  // contiguous candidates per thread
  const int t0 = min(loc, tid * per), t1 = min(loc, t0 + per);
  for (int t = t0; t < t1; ++t) {
    float m = sm[t * R];
    for (int r = 1; r < R; ++r) m = fmaxf(m, sm[t * R + r]);
    vals[t] = t >= fs ? max(ord_f32(m), 1u) : 0u;  // candidates >= 1; every threshold below is >= 1
  }
  uint32_t prefix = 0;
  for (int round = 0; round < 16; ++round) {
    const int sh = 30 - 2 * round;
    int c[3] = {0, 0, 0};
    for (int t = t0; t < t1; ++t) {
      const uint32_t v = vals[t];
#pragma unroll
      for (int x = 0; x < 3; ++x) c[x] += v >= (prefix | (uint32_t(x + 1) << sh));
    }
    const int par = round & 1;
#pragma unroll
    for (int x = 0; x < 3; ++x) {
      const int w = __reduce_add_sync(0xffffffffu, c[x]);
      if (lane == 0) wsum[par][warp][x] = w;
    }
    __syncthreads();
    int best = 0;
#pragma unroll
    for (int x = 0; x < 3; ++x) {
      int total = 0;
#pragma unroll
      for (int w = 0; w < kTkThreads / 32; ++w) total += wsum[par][w][x];
      if (total >= need) best = x + 1;  // counts fall as the candidate grows
    }
    prefix |= uint32_t(best) << sh;
  }
  // prefix = v*, the need-th largest value
  int gt = 0, eq = 0;
  for (int t = t0; t < t1; ++t) {
    gt += vals[t] > prefix;
    eq += vals[t] == prefix;
  }
  const int gt_total = block_exclusive_scan(gt, scan_buf) + gt;  // inclusive for the last thread only
  __shared__ int gt_all;
  if (tid == kTkThreads - 1) gt_all = gt_total;
  const int eq_before = block_exclusive_scan(eq, scan_buf);
  const int ties = need - gt_all;
  const int take_eq = max(0, min(eq, ties - eq_before));  // the lowest-t equals go first
  const int my = gt + take_eq;
  int o = fs + block_exclusive_scan(my, scan_buf);
  int eq_seen = 0;
  for (int t = t0; t < t1; ++t) {
    const uint32_t v = vals[t];
    if (v > prefix || (v == prefix && eq_seen++ < take_eq)) out[o++] = t;
  }
  if (tid == 0) {
    if (fs) out[0] = 0;
    out[K - 1] = loc;
  }
}

// decode_topk for rows of at most 1024 blocks: one warp per (sequence,
// group) row, eight rows per CTA, each warp staging its row's sub-block maxima
// in its own 16 KB of shared memory (warp_topk_row).
constexpr int kTkwRows = 8;
constexpr uint32_t kTkwRowBytes = kWarpTopkPer * 32 * 4 * 4;  // 1024 blocks x 4 sub-blocks
__global__ void __launch_bounds__(kTkwRows * 32) decode_topk_warp_kernel(
    const float* __restrict__ sub_max, const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len,
    int Lmax, int G, int Bs, int K, int fs, int nsub, int rows, int32_t* __restrict__ sel, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t tkw_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tc::griddep_launch_dependents();  // attention may launch now; it waits for the selection
  const int row = blockIdx.x * kTkwRows + warp;  // b * G + g
  if (row >= rows) return;
  const int b = row / G;
  int32_t* out = sel + int64_t(row) * K;
  const SeqView sv = seq_view(q_offset, kv_len, b, 1, Lmax, false);
  if (!sv.ok) {
    for (int k = lane; k < K; k += 32) out[k] = -1;
    if (lane == 0) set_status(status, MSA_ERR_BOUNDS);
    return;
  }
  const int loc = sv.q0 / Bs;
  const float* sm = sub_max + int64_t(row) * nsub;
  float* buf = reinterpret_cast<float*>(tkw_smem + size_t(warp) * kTkwRowBytes);
  tc::griddep_wait();  // the sub-block maxima come from the index kernel
  if (Bs == 128)
    warp_topk_row<4>(sm, loc, K, fs, out, lane, buf);
  else if (Bs == 64)
    warp_topk_row<2>(sm, loc, K, fs, out, lane, buf);
  else
    warp_topk_row<1>(sm, loc, K, fs, out, lane, buf);
}

// Launches `kern` with programmatic stream serialization: it may begin while
// the previous kernel of the stream finishes, and waits (griddep_wait) before
// it reads that kernel's output.
template <typename... Params, typename... Args>
cudaError_t launch_after_prev(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Streaming decode: append one token per sequence to its caches. Block b
// copies the token's key and value rows (all kv heads) and its index-key row
// to position L = kv_len[b], then advances kv_len[b] to L + 1 and records L as
// the token's position for the selection. A sequence whose cache is full (or
// whose length is out of range) is left unchanged; its position becomes -1,
// so its selection row comes back -1, and the status becomes MSA_ERR_BOUNDS.
__global__ void __launch_bounds__(256) decode_append_kernel(const uint4* __restrict__ k_new,
                                                            const uint4* __restrict__ v_new,
                                                            const uint4* __restrict__ ik_new, uint4* __restrict__ k_cache,
                                                            uint4* __restrict__ v_cache, uint4* __restrict__ ik_cache,
                                                            int32_t* __restrict__ kv_len, int32_t* __restrict__ q_pos,
                                                            int Lmax, int kv_vec, int ik_vec, uint32_t* status) {
  const int b = blockIdx.x;
  const int L = kv_len[b];
  const bool ok = L >= 0 && L < Lmax;
  __syncthreads();  // every thread has read kv_len[b] before it advances
  if (ok) {
    const int64_t row = int64_t(b) * Lmax + L;
    for (int x = threadIdx.x; x < kv_vec; x += blockDim.x) {
      k_cache[row * kv_vec + x] = k_new[int64_t(b) * kv_vec + x];
      v_cache[row * kv_vec + x] = v_new[int64_t(b) * kv_vec + x];
    }
    for (int x = threadIdx.x; x < ik_vec; x += blockDim.x) ik_cache[row * ik_vec + x] = ik_new[int64_t(b) * ik_vec + x];
  }
  if (threadIdx.x == 0) {
    if (ok) {
      kv_len[b] = L + 1;
      q_pos[b] = L;
    } else {
      q_pos[b] = -1;
      set_status(status, MSA_ERR_BOUNDS);
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
bool decode_attn_supported(int dtype, int Hq, int Hkv, int d, int Bs, int K) {
  if (dtype != MSA_BF16 || (d != 64 && d != 128)) return false;
  if (Bs != 32 && Bs != 64 && Bs != 128) return false;
  if (K < 1 || K > kMaxK || Hq % Hkv != 0) return false;
  const int hpg = Hq / Hkv;
  if (hpg != 1 && hpg != 2 && hpg != 4 && hpg != 8) return false;
  return dec_smem_bytes(d, Bs, hpg) <= 227 * 1024;
}

static size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

size_t decode_ws_bytes(int B, int Hq, int Hkv, int d, int K) {
  const size_t items = size_t(B) * Hkv * K, hpg = size_t(Hq / Hkv);
  return a256(items * hpg * d * 4) + a256(items * hpg * 2 * 4) + a256(size_t(B) * Hkv * 4);
}

cudaError_t launch_decode_attn(const void* q, const void* k_cache, const void* v_cache, const int32_t* sel,
                               const int32_t* kv_len, int B, int Lmax, int Hq, int Hkv, int d, int Bs, int K,
                               float scale, void* out, float* lse, void* scratch, uint32_t* status,
                               cudaStream_t stream) {
  const int G = Hkv, hpg = Hq / Hkv, nblk = (Lmax + Bs - 1) / Bs;
  const size_t items = size_t(B) * G * K;
  char* sc = static_cast<char*>(scratch);
  float* part_o = reinterpret_cast<float*>(sc);
  float* part_ml = reinterpret_cast<float*>(sc + a256(items * hpg * d * 4));
  int* arrivals = reinterpret_cast<int*>(sc + a256(items * hpg * d * 4) + a256(items * hpg * 2 * 4));
  CUtensorMap tmK, tmV;
  const uint64_t dims[4] = {uint64_t(d), uint64_t(Hkv), uint64_t(Lmax), uint64_t(B)};
  const uint64_t strides[3] = {uint64_t(d) * 2, uint64_t(Hkv) * d * 2, uint64_t(Lmax) * Hkv * d * 2};
  const uint32_t box[4] = {64, 1, uint32_t(Bs), 1};
  if (!make_tmap_bf16(&tmK, k_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tmV, v_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const size_t smem = dec_smem_bytes(d, Bs, hpg);
  const float scale_log2 = scale * kLog2eD;
  const int inject = debug_inject_timeout() ? 1 : 0;
  cudaError_t e;
  ProfScope pf("decode_attn", stream);
#define MSA_DEC(D_, BS_, HPG_)                                                                                   \
  do {                                                                                                           \
    auto kern = decode_attn_kernel<D_, BS_, HPG_>;                                                              \
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess) \
      return e;                                                                                                  \
    if ((e = launch_after_prev(kern, dim3(unsigned(items)), dim3(kDecThreads), smem, stream, tmK, tmV,              \
                               static_cast<const __nv_bfloat16*>(q), sel, kv_len, Lmax, Hq, G, K, nblk, scale_log2,   \
                               part_o, part_ml, arrivals, static_cast<__nv_bfloat16*>(out), lse, status,            \
                               inject)) != cudaSuccess)                                                          \
      return e;                                                                                                  \
  } while (0)
#define MSA_DEC_BS(D_, HPG_)  \
  do {                        \
    if (Bs == 128)            \
      MSA_DEC(D_, 128, HPG_); \
    else if (Bs == 64)        \
      MSA_DEC(D_, 64, HPG_);  \
    else                      \
      MSA_DEC(D_, 32, HPG_);  \
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
    else if (hpg == 2)
      MSA_DEC_BS(64, 2);
    else
      MSA_DEC_BS(64, 1);
  }
#undef MSA_DEC_BS
#undef MSA_DEC
  return cudaGetLastError();
}

bool decode_index_supported(int dtype, int B, int Nq, int G, int di, int Bs, int K) {
  return dtype == MSA_BF16 && Nq == 1 && di == 64 && G >= 1 && G <= 16 && B >= 1 && B <= kDiMaxB &&
         (Bs == 32 || Bs == 64 || Bs == 128) && K >= 1 && K <= kMaxK;
}

// row stride of the sub-block maxima table: ceil(Lmax / 32) rounded up to 4
// floats, so that every row starts on 16 bytes (16-byte copies of a row)
static int decode_sub_stride(int Lmax) { return (((Lmax + 31) / 32) + 3) & ~3; }
size_t decode_index_ws_bytes(int B, int G, int Nk) { return size_t(B) * G * decode_sub_stride(Nk) * sizeof(float); }

cudaError_t launch_decode_index(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len, int B,
                                int Lmax, int G, int Bs, int K, int fs, int32_t* sel, float* table, uint32_t* status,
                                cudaStream_t stream) {
  const int nsub = decode_sub_stride(Lmax);  // table row stride (>= sub-blocks per row)
  const int nblk = (Lmax + Bs - 1) / Bs;
  if (nblk > kTkMaxCand) return cudaErrorInvalidValue;
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
  const size_t smem = 1024 + size_t(kDiStages) * kDiStage + (2 * kDiMaxB + 1) * 4 + 16 +
                      (2 * kDiStages + 2 * kDiAcc + 1) * 8 + 16;
  int dev = 0, sms = kNumSMs;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e;
  {
    ProfScope pf("decode_index", stream);
    if ((e = cudaFuncSetAttribute(decode_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) !=
        cudaSuccess)
      return e;
    decode_index_kernel<<<sms, kDiThreads, smem, stream>>>(tmIK, tmIQ, q_offset, kv_len, B, Lmax, G, nsub, table,
                                                           status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (nblk <= kWarpTopkPer * 32) {
    ProfScope pf("decode_topk", stream);
    const int rows = B * G;
    const size_t tkw_smem = size_t(kTkwRows) * kTkwRowBytes;
    if ((e = cudaFuncSetAttribute(decode_topk_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(tkw_smem))) != cudaSuccess)
      return e;
    if ((e = launch_after_prev(decode_topk_warp_kernel, dim3((rows + kTkwRows - 1) / kTkwRows), dim3(kTkwRows * 32),
                               tkw_smem, stream, static_cast<const float*>(table), q_offset, kv_len, Lmax, G, Bs, K,
                               fs, nsub, rows, sel, status)) != cudaSuccess)
      return e;
    return cudaGetLastError();
  }
  {
    ProfScope pf("decode_topk", stream);
    const size_t tk_smem = size_t(nblk) * 4;
    if (tk_smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(decode_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(tk_smem))) !=
            cudaSuccess)
      return e;
    if ((e = launch_after_prev(decode_topk_kernel, dim3(B * G), dim3(kTkThreads), tk_smem, stream,
                               static_cast<const float*>(table), q_offset, kv_len, Lmax, G, Bs, K, fs, nsub, sel,
                               status)) !=
        cudaSuccess)
      return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_append(const void* k_new, const void* v_new, const void* ik_new, void* k_cache,
                                 void* v_cache, void* ik_cache, int32_t* kv_len, int32_t* q_pos, int B, int Lmax,
                                 int Hkv, int d, int di, int elem_bytes, uint32_t* status, cudaStream_t stream) {
  const size_t kv_row = size_t(Hkv) * d * elem_bytes, ik_row = size_t(di) * elem_bytes;
  if (kv_row % 16 || ik_row % 16) return cudaErrorInvalidValue;
  ProfScope pf("decode_append", stream);
  decode_append_kernel<<<B, 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<const uint4*>(ik_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), static_cast<uint4*>(ik_cache), kv_len, q_pos, Lmax,
      int(kv_row / 16), int(ik_row / 16), status);
  return cudaGetLastError();
}

}  // namespace msa
