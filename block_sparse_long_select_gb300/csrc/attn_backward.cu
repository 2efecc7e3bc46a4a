// Main Branch backward, prefill, KV-outer (bf16, sm_103a): dq, dk, dv of the
// sparse attention over the selected blocks, with the selection held fixed.
// (hyper.ai summary of paper 2606.13392, "方法": the Main Branch is standard
//  scaled-dot-product softmax attention over the selected blocks' keys and
//  values; "一句话总结" and "实验": the model is trained through it (MSA-PT,
//  CPT), so its gradient is the textbook softmax-attention gradient.)
//
// Per (query row, head), with the forward's lse and delta = dout . out:
//   P_j = exp(scale q.k_j - lse);  dP_j = dout . v_j;  dS_j = P_j (dP_j - delta)
//   dv_j += P_j dout;  dk_j += scale dS_j q;  dq = scale sum_j dS_j k_j
//
// The work follows the forward's inversion: per-(group, key block) bins of
// (query, slot) entries in 128-row tiles (128 / hpg entries x hpg heads), on
// the same cost-balanced contiguous runs of a persistent grid. Per tile, with
// the block's K and V resident in shared memory for the run of its bin:
//   1. S^T = K Q^T and dP^T = V dO^T on mma.sync (keys along M); P^T and dS^T
//      are formed in registers and written to shared memory as bf16;
//   2. dV += P^T dO and dK += dS^T Q, accumulated in registers over the run's
//      tiles of one bin (each warp a 16-key strip x a slice of d);
//   3. dQ = dS K for the tile's rows, stored as an fp32 partial per (entry,
//      head) row, while the next tile's rows are already being gathered.
// When a bin's run ends, dK and dV are added into per-sequence fp32
// accumulators: plainly when this CTA holds every tile of the bin, atomically
// when the bin is split over CTAs. bwd_dq_combine then sums each row's slot
// partials in slot order (deterministic) and bwd_kv_store rounds dk and dv.
#include <cmath>

#include "msa_internal.cuh"
#include "tc_utils.cuh"

namespace msa {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdRows = kKvoRows;  // 128 rows per tile
constexpr float kLog2eBwd = 1.4426950408889634f;

__device__ __forceinline__ float bwd_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t bwd_pack(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// four 8x8 b16 matrices; lane l gives the row address of matrix l / 8
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp16(void* dst, const void* src, bool in) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
               "r"(in ? 16u : 0u)
               : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src, bool in) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(tc::smem_u32(dst)), "l"(src), "r"(in ? 4u : 0u)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ bool bwd_entry_valid(int t, int pos, int Bs, int nblk) {
  return t >= 0 && t < nblk && t * Bs <= pos;
}

// ---------------------------------------------------------------------------
// delta = dout . out per (row, head): TPR threads per row, 8 elements each
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ out,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, int64_t rows) {
  constexpr int TPR = D / 8;
  const int64_t stride = int64_t(gridDim.x) * (256 / TPR);
  const int sub = threadIdx.x % TPR;
  // the loop bound is uniform over the block, so every lane reaches the shuffles
  for (int64_t r0 = int64_t(blockIdx.x) * (256 / TPR); r0 < rows; r0 += stride) {
    const int64_t r = r0 + threadIdx.x / TPR;
    const bool in = r < rows;
    const uint4 a = in ? *reinterpret_cast<const uint4*>(out + r * D + sub * 8) : make_uint4(0, 0, 0, 0);
    const uint4 g = in ? *reinterpret_cast<const uint4*>(dout + r * D + sub * 8) : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
    float s = 0.f;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 af = __bfloat1622float2(a2[x]), gf = __bfloat1622float2(g2[x]);
      s = fmaf(af.x, gf.x, s);
      s = fmaf(af.y, gf.y, s);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (in && sub == 0) delta[r] = s;
  }
}

// ---------------------------------------------------------------------------
// the tile kernel
// ---------------------------------------------------------------------------
struct BwdParams {
  const __nv_bfloat16 *q, *k, *v, *dout;  // q, dout [B, Nq, Hq, D]; k, v [B, Nk, G, D]
  const float *lse, *delta;               // [B, Nq, Hq]: forward log-sum-exp (natural log), dout . out
  const int* entries;                     // chunk entries (local query * 64 + slot), bins padded to tiles
  const int4* tiles;                      // (bin, first entry position, entries)
  const int* tile_off;                    // [nbins + 1] first tile of each bin
  const int* cta_start;                   // [grid + 1]
  const int32_t* q_offset;
  const int32_t* kv_len;
  float* part_dq;  // [entry position * hpg + head][D] fp32, unscaled
  float* dk_acc;   // [Nk, G, D] fp32 of sequence b, unscaled
  float* dv_acc;   // [Nk, G, D] fp32 of sequence b
  int b, Nq, Nk, Hq, G, hpg, hpg_log2, nblk, c0;
  float scale;
};

template <int D, int BS>
struct BwdSmem {
  static constexpr int KP = D + 8;         // K, V, Q, dO row pitch (bf16): 16-byte rows, no bank conflicts
  static constexpr int RP = kBwdRows + 8;  // P^T, dS^T row pitch
  static constexpr size_t kKV = size_t(BS) * KP * 2;
  static constexpr size_t kQ = size_t(kBwdRows) * KP * 2;
  static constexpr size_t kP = size_t(BS) * RP * 2;
  static constexpr size_t kRow = size_t(kBwdRows) * 4;
  static constexpr size_t kTotal = 2 * kKV + 2 * kQ + 2 * kP + 6 * kRow;  // + lse, delta, row query (x2 buffers)
};

template <int D, int BS>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_tile_kernel(const BwdParams p) {
  using SM = BwdSmem<D, BS>;
  constexpr int KP = SM::KP, RP = SM::RP;
  constexpr int MT = BS / 16;            // 16-key strips
  constexpr int WS = 8 / MT;             // warps per strip
  constexpr int RW = kBwdRows / WS;      // phase 1: rows per warp
  constexpr int DW = D / WS;             // phase 2: d columns per warp
  constexpr int NTD = DW / 8;            // phase 2: 8-column tiles per warp
  constexpr int QC = D < 64 ? D : 64;    // phase 3: dq columns per pass
  static_assert(MT >= 1 && MT <= 8 && NTD % 2 == 0 && RW % 32 == 0, "tile split");
  extern __shared__ __align__(16) uint8_t bwd_smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(bwd_smem);
  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(bwd_smem + SM::kKV);
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(bwd_smem + 2 * SM::kKV);
  __nv_bfloat16* Os = reinterpret_cast<__nv_bfloat16*>(bwd_smem + 2 * SM::kKV + SM::kQ);
  __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(bwd_smem + 2 * SM::kKV + 2 * SM::kQ);
  __nv_bfloat16* Ss = reinterpret_cast<__nv_bfloat16*>(bwd_smem + 2 * SM::kKV + 2 * SM::kQ + SM::kP);
  float* rows_f = reinterpret_cast<float*>(bwd_smem + 2 * SM::kKV + 2 * SM::kQ + 2 * SM::kP);
  float* lse_s = rows_f;                                  // [2][128]
  float* dlt_s = rows_f + 2 * kBwdRows;                   // [2][128]
  int* rq_s = reinterpret_cast<int*>(rows_f + 4 * kBwdRows);  // [2][128] local query of the row, -1 = padding

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int mt = warp % MT, wp = warp / MT;
  const int z0 = p.cta_start[blockIdx.x], z1 = p.cta_start[blockIdx.x + 1];
  if (z0 >= z1) return;
  const SeqView sv = seq_view(p.q_offset, p.kv_len, p.b, p.Nq, p.Nk, false);
  const int hmask = p.hpg - 1;
  const float sl2 = p.scale * kLog2eBwd;

  // tile z's query and dout rows (zero rows for padding entries), their lse and delta
  auto load_rows = [&](int z, int nb) {
    const int4 tl = p.tiles[z];
    const int g = tl.x / p.nblk;
#pragma unroll 2
    for (int x = tid; x < kBwdRows * (D / 8); x += kBwdThreads) {
      const int r = x / (D / 8), c = x % (D / 8);
      const int e = r >> p.hpg_log2;
      const int ent = e < tl.z ? p.entries[tl.y + e] : -1;
      const int il = ent >= 0 ? (ent >> 6) : 0;
      const int64_t row = (int64_t(p.b) * p.Nq + p.c0 + il) * p.Hq + g * p.hpg + (r & hmask);
      cp16(Qs + r * KP + c * 8, p.q + row * D + c * 8, ent >= 0);
      cp16(Os + r * KP + c * 8, p.dout + row * D + c * 8, ent >= 0);
    }
    if (tid < kBwdRows) {
      const int r = tid, e = r >> p.hpg_log2;
      const int ent = e < tl.z ? p.entries[tl.y + e] : -1;
      const int il = ent >= 0 ? (ent >> 6) : 0;
      const int64_t row = (int64_t(p.b) * p.Nq + p.c0 + il) * p.Hq + g * p.hpg + (r & hmask);
      cp4(lse_s + nb * kBwdRows + r, p.lse + row, ent >= 0);
      cp4(dlt_s + nb * kBwdRows + r, p.delta + row, ent >= 0);
      rq_s[nb * kBwdRows + r] = ent >= 0 ? il : -1;
    }
    cp_commit();
  };
  // the block's keys and values, rows past the sequence zero-filled
  auto load_kv = [&](int bin) {
    const int g = bin / p.nblk, t = bin % p.nblk;
#pragma unroll 2
    for (int x = tid; x < BS * (D / 8); x += kBwdThreads) {
      const int r = x / (D / 8), c = x % (D / 8), j = t * BS + r;
      const bool in = j < p.Nk;
      const int64_t off = ((int64_t(p.b) * p.Nk + (in ? j : 0)) * p.G + g) * D + c * 8;
      cp16(Ks + r * KP + c * 8, p.k + off, in);
      cp16(Vs + r * KP + c * 8, p.v + off, in);
    }
    cp_commit();
  };

  int bin = p.tiles[z0].x;
  int bin_first = z0;
  load_kv(bin);
  load_rows(z0, 0);
  float dk[NTD][4], dv[NTD][4];
#pragma unroll
  for (int n = 0; n < NTD; ++n)
#pragma unroll
    for (int x = 0; x < 4; ++x) dk[n][x] = dv[n][x] = 0.f;

  int nb = 0;
  for (int z = z0; z < z1; ++z) {
    const int4 tl = p.tiles[z];
    const int g = bin / p.nblk, t = bin % p.nblk;
    cp_wait_all();
    __syncthreads();
    // ---- 1. S^T, dP^T for keys [16 mt, +16) x rows [RW wp, +RW); P^T, dS^T to shared memory
    {
      const float* lse_b = lse_s + nb * kBwdRows;
      const float* dlt_b = dlt_s + nb * kBwdRows;
      const int* rq_b = rq_s + nb * kBwdRows;
      const int arow = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1), acol = 8 * (lane >> 4);
      const int brow = (lane & 7) + 8 * (lane >> 4), bcol = 8 * ((lane >> 3) & 1);
#pragma unroll 1
      for (int rc = wp * RW; rc < (wp + 1) * RW; rc += 32) {
        float s[4][4], dp[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) s[n][x] = dp[n][x] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t ak[4], av[4];
          ldsm4(tc::smem_u32(Ks + arow * KP + ks * 16 + acol), ak);
          ldsm4(tc::smem_u32(Vs + arow * KP + ks * 16 + acol), av);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t bq[4], bo[4];
            const int r0 = rc + h2 * 16 + brow;
            ldsm4(tc::smem_u32(Qs + r0 * KP + ks * 16 + bcol), bq);
            ldsm4(tc::smem_u32(Os + r0 * KP + ks * 16 + bcol), bo);
            mma_bf16(s[2 * h2], ak, bq[0], bq[1]);
            mma_bf16(s[2 * h2 + 1], ak, bq[2], bq[3]);
            mma_bf16(dp[2 * h2], av, bo[0], bo[1]);
            mma_bf16(dp[2 * h2 + 1], av, bo[2], bo[3]);
          }
        }
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const int r0 = rc + n * 8 + 2 * tq;  // this lane's two rows (fragment columns)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int kl = mt * 16 + gq + 8 * hr;
            const int j = t * BS + kl;
            float pv[2], dsv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = r0 + e;
              const int il = rq_b[r];
              const bool vis = il >= 0 && j <= sv.q0 + p.c0 + il && j < sv.L;
              const float pr = vis ? bwd_ex2(s[n][2 * hr + e] * sl2 - lse_b[r] * kLog2eBwd) : 0.f;
              pv[e] = pr;
              dsv[e] = pr * (dp[n][2 * hr + e] - dlt_b[r]);
            }
            *reinterpret_cast<uint32_t*>(Ps + kl * RP + r0) = bwd_pack(pv[0], pv[1]);
            *reinterpret_cast<uint32_t*>(Ss + kl * RP + r0) = bwd_pack(dsv[0], dsv[1]);
          }
        }
      }
    }
    __syncthreads();
    // ---- 2. dV += P^T dO, dK += dS^T Q: keys [16 mt, +16) x d [DW wp, +DW), rows reduced
    {
      const int arow = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1), acol = 8 * (lane >> 4);
      const int brow = (lane & 7) + 8 * ((lane >> 3) & 1), bcol = wp * DW + 8 * (lane >> 4);
#pragma unroll 2
      for (int ks = 0; ks < kBwdRows / 16; ++ks) {
        uint32_t ap[4], as[4];
        ldsm4(tc::smem_u32(Ps + arow * RP + ks * 16 + acol), ap);
        ldsm4(tc::smem_u32(Ss + arow * RP + ks * 16 + acol), as);
#pragma unroll
        for (int n2 = 0; n2 < NTD / 2; ++n2) {
          uint32_t bo[4], bq[4];
          ldsm4t(tc::smem_u32(Os + (ks * 16 + brow) * KP + bcol + n2 * 16), bo);
          ldsm4t(tc::smem_u32(Qs + (ks * 16 + brow) * KP + bcol + n2 * 16), bq);
          mma_bf16(dv[2 * n2], ap, bo[0], bo[1]);
          mma_bf16(dv[2 * n2 + 1], ap, bo[2], bo[3]);
          mma_bf16(dk[2 * n2], as, bq[0], bq[1]);
          mma_bf16(dk[2 * n2 + 1], as, bq[2], bq[3]);
        }
      }
    }
    __syncthreads();  // Q and dO are free: gather the next tile's rows under phase 3
    const bool more = z + 1 < z1;
    if (more) load_rows(z + 1, nb ^ 1);
    // ---- 3. dQ rows [16 warp, +16) = dS K, keys reduced; fp32 partial rows
    {
      const int m0 = warp * 16;
      const int arow = (lane & 7) + 8 * (lane >> 4), acol = m0 + 8 * ((lane >> 3) & 1);
      const int brow = (lane & 7) + 8 * ((lane >> 3) & 1), bcol = 8 * (lane >> 4);
#pragma unroll 1
      for (int cq = 0; cq < D; cq += QC) {
        float acc[QC / 8][4];
#pragma unroll
        for (int n = 0; n < QC / 8; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) acc[n][x] = 0.f;
#pragma unroll
        for (int ks = 0; ks < BS / 16; ++ks) {
          uint32_t a[4];
          ldsm4t(tc::smem_u32(Ss + (ks * 16 + arow) * RP + acol), a);
#pragma unroll
          for (int n2 = 0; n2 < QC / 16; ++n2) {
            uint32_t bk[4];
            ldsm4t(tc::smem_u32(Ks + (ks * 16 + brow) * KP + cq + n2 * 16 + bcol), bk);
            mma_bf16(acc[2 * n2], a, bk[0], bk[1]);
            mma_bf16(acc[2 * n2 + 1], a, bk[2], bk[3]);
          }
        }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = m0 + gq + 8 * hr;
          const int e = r >> p.hpg_log2;
          if (e < tl.z) {
            float* dst = p.part_dq + (int64_t(tl.y + e) * p.hpg + (r & hmask)) * D + cq + 2 * tq;
#pragma unroll
            for (int n = 0; n < QC / 8; ++n)
              *reinterpret_cast<float2*>(dst + n * 8) = make_float2(acc[n][2 * hr], acc[n][2 * hr + 1]);
          }
        }
      }
    }
    // ---- end of the bin's run: add dK, dV into the sequence's accumulators
    const int next_bin = more ? p.tiles[z + 1].x : -1;
    if (next_bin != bin) {
      const bool whole = bin_first == p.tile_off[bin] && z + 1 == p.tile_off[bin + 1];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int j = t * BS + mt * 16 + gq + 8 * hr;
        if (j < p.Nk) {
          const int64_t base = (int64_t(j) * p.G + g) * D + wp * DW + 2 * tq;
#pragma unroll
          for (int n = 0; n < NTD; ++n) {
            float* pk = p.dk_acc + base + n * 8;
            float* pv = p.dv_acc + base + n * 8;
            if (whole) {
              float2 a = *reinterpret_cast<float2*>(pk), c = *reinterpret_cast<float2*>(pv);
              a.x += dk[n][2 * hr];
              a.y += dk[n][2 * hr + 1];
              c.x += dv[n][2 * hr];
              c.y += dv[n][2 * hr + 1];
              *reinterpret_cast<float2*>(pk) = a;
              *reinterpret_cast<float2*>(pv) = c;
            } else {
              atomicAdd(pk, dk[n][2 * hr]);
              atomicAdd(pk + 1, dk[n][2 * hr + 1]);
              atomicAdd(pv, dv[n][2 * hr]);
              atomicAdd(pv + 1, dv[n][2 * hr + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int n = 0; n < NTD; ++n)
#pragma unroll
        for (int x = 0; x < 4; ++x) dk[n][x] = dv[n][x] = 0.f;
      if (more) {
        __syncthreads();  // every warp is done with this block's K
        bin = next_bin;
        bin_first = z + 1;
        load_kv(bin);
      }
    }
    nb ^= 1;
  }
}

// ---------------------------------------------------------------------------
// dq: one warp per (query, group) sums its valid slots' partial rows in slot
// order; NU float4 of the group's hpg x D row block per lane
// ---------------------------------------------------------------------------
template <int NU>
__global__ void __launch_bounds__(256) bwd_dq_combine_kernel(
    const int32_t* __restrict__ sel, const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len,
    const float4* __restrict__ part_dq, const int* __restrict__ rev, int b, int Nq, int Nk, int Hq, int G, int K,
    int Bs, int nblk, int D, int c0, int cq, float scale, __nv_bfloat16* __restrict__ dq) {
  constexpr int kWarps = 256 / 32;
  constexpr int kBatch = NU <= 2 ? 8 : (NU == 4 ? 4 : 2);  // slots whose loads are in flight together
  __shared__ int slot_e[kWarps][kMaxK];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int hpg = Hq / G;
  const int nvec = hpg * D / 4;  // float4 per slot
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  const int64_t nitems = int64_t(cq) * G;
  for (int64_t item = int64_t(blockIdx.x) * kWarps + wl; item < nitems; item += int64_t(gridDim.x) * kWarps) {
    const int il = int(item / G), g = int(item % G);
    const int i = c0 + il, pos = sv.q0 + i;
    const int32_t* srow = sel + ((int64_t(b) * Nq + i) * G + g) * K;
    const int* rv = rev + (int64_t(il) * G + g) * K;
    int nv = 0;
    for (int k0 = 0; k0 < K; k0 += 32) {
      const int k = k0 + lane;
      const bool ok = k < K && sv.ok && bwd_entry_valid(srow[k], pos, Bs, nblk);
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (ok) slot_e[wl][nv + __popc(bal & ((1u << lane) - 1u))] = rv[k];
      nv += __popc(bal);
    }
    __syncwarp();
    float4 acc[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < nv; j0 += kBatch) {
      float4 x[kBatch][NU];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const bool in = j0 + jj < nv;
        const int64_t base = in ? int64_t(slot_e[wl][j0 + jj]) * nvec : 0;
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const int vi = lane + 32 * u;
          x[jj][u] = (in && vi < nvec) ? part_dq[base + vi] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj)
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          acc[u].x += x[jj][u].x;
          acc[u].y += x[jj][u].y;
          acc[u].z += x[jj][u].z;
          acc[u].w += x[jj][u].w;
        }
    }
    __nv_bfloat16* drow = dq + ((int64_t(b) * Nq + i) * Hq + int64_t(g) * hpg) * D;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int vi = lane + 32 * u;
      if (vi < nvec) {
        uint2 o;
        o.x = bwd_pack(acc[u].x * scale, acc[u].y * scale);
        o.y = bwd_pack(acc[u].z * scale, acc[u].w * scale);
        *reinterpret_cast<uint2*>(drow + vi * 4) = o;
      }
    }
    __syncwarp();
  }
}

// dk = scale * dk_acc, dv = dv_acc, rounded to bf16 (n = Nk * G * D, multiple of 4)
__global__ void __launch_bounds__(256) bwd_kv_store_kernel(const float4* __restrict__ dk_acc,
                                                           const float4* __restrict__ dv_acc, float scale,
                                                           int64_t n4, uint2* __restrict__ dk, uint2* __restrict__ dv) {
  for (int64_t x = int64_t(blockIdx.x) * 256 + threadIdx.x; x < n4; x += int64_t(gridDim.x) * 256) {
    const float4 a = dk_acc[x], c = dv_acc[x];
    dk[x] = make_uint2(bwd_pack(a.x * scale, a.y * scale), bwd_pack(a.z * scale, a.w * scale));
    dv[x] = make_uint2(bwd_pack(c.x, c.y), bwd_pack(c.z, c.w));
  }
}

inline size_t a256b(size_t x) { return (x + 255) & ~size_t(255); }

struct BwdLayout {
  KvoLayout L;  // inversion; its partial area (sized for 2d bf16 = d fp32 per row) holds the dq partials
  size_t delta, dk_acc, dv_acc, end;
};

BwdLayout bwd_layout(int B, int Nq, int Nk, int Hq, int G, int d, int Bs, int K) {
  BwdLayout W;
  W.L = kvo_layout(Nq, Hq, G, 2 * d, Bs, K, Nk);
  size_t o = W.L.end;
  W.delta = o;
  o += a256b(size_t(B) * Nq * Hq * 4);
  W.dk_acc = o;
  o += a256b(size_t(Nk) * G * d * 4);
  W.dv_acc = o;
  o += a256b(size_t(Nk) * G * d * 4);
  W.end = o;
  return W;
}

}  // namespace

bool attn_backward_supported(int dtype, int Hq, int Hkv, int d, int Bs, int K) {
  if (dtype != MSA_BF16 || Hkv < 1 || Hq % Hkv != 0) return false;
  if (d != 64 && d != 128) return false;
  if (Bs != 32 && Bs != 64 && Bs != 128) return false;
  if (K < 1 || K > kMaxK) return false;
  const int hpg = Hq / Hkv;
  return hpg >= 1 && hpg <= 8 && (hpg & (hpg - 1)) == 0;
}

size_t attn_backward_ws_bytes(int B, int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K) {
  return bwd_layout(B, Nq, Nk, Hq, Hkv, d, Bs, K).end;
}

cudaError_t launch_attn_backward(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                 const float* lse, const int32_t* sel, const int32_t* q_offset,
                                 const int32_t* kv_len, int B, int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K,
                                 float scale, void* dq, void* dk, void* dv, void* ws, cudaStream_t stream) {
  const int G = Hkv, hpg = Hq / Hkv, nblk = (Nk + Bs - 1) / Bs;
  const int per_tile = kBwdRows / hpg;
  const BwdLayout W = bwd_layout(B, Nq, Nk, Hq, G, d, Bs, K);
  const KvoLayout& L = W.L;
  char* w = static_cast<char*>(ws);
  uint32_t* status = &static_cast<WsHeader*>(ws)->status;
  float* delta = reinterpret_cast<float*>(w + W.delta);
  const int grid = sm_count() < kKvoMaxGrid ? sm_count() : kKvoMaxGrid;
  const int cq_max = chunk_tokens(Nq, Hq, K, 2 * d);
  cudaError_t e;
  {
    ProfScope pf("bwd_delta", stream);
    const int64_t rows = int64_t(B) * Nq * Hq;
    const int64_t need = (rows * (d / 8) + 255) / 256;
    const int dgrid = int(need < int64_t(grid) * 8 ? need : int64_t(grid) * 8);
    if (d == 128)
      bwd_delta_kernel<128><<<dgrid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(out),
                                                        static_cast<const __nv_bfloat16*>(dout), delta, rows);
    else
      bwd_delta_kernel<64><<<dgrid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(out),
                                                       static_cast<const __nv_bfloat16*>(dout), delta, rows);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  BwdParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.dout = static_cast<const __nv_bfloat16*>(dout);
  prm.lse = lse;
  prm.delta = delta;
  prm.entries = reinterpret_cast<const int*>(w + L.entries);
  prm.tiles = reinterpret_cast<const int4*>(w + L.tiles);
  prm.tile_off = reinterpret_cast<const int*>(w + L.tile_off);
  prm.cta_start = reinterpret_cast<const int*>(w + L.cta_start);
  prm.q_offset = q_offset;
  prm.kv_len = kv_len;
  prm.part_dq = reinterpret_cast<float*>(w + L.part_o);
  prm.dk_acc = reinterpret_cast<float*>(w + W.dk_acc);
  prm.dv_acc = reinterpret_cast<float*>(w + W.dv_acc);
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.Hq = Hq;
  prm.G = G;
  prm.hpg = hpg;
  prm.hpg_log2 = __builtin_ctz(unsigned(hpg));
  prm.nblk = nblk;
  prm.scale = scale;
  const int* rev = reinterpret_cast<const int*>(w + L.rev);
  const int64_t kv_elems = int64_t(Nk) * G * d;

  for (int b = 0; b < B; ++b) {
    if ((e = cudaMemsetAsync(w + W.dk_acc, 0, W.end - W.dk_acc, stream)) != cudaSuccess) return e;
    for (int c0 = 0; c0 < Nq; c0 += cq_max) {
      const int cq = Nq - c0 < cq_max ? Nq - c0 : cq_max;
      if ((e = invert_chunk(sel, q_offset, kv_len, b, Nq, Nk, G, K, Bs, per_tile, c0, cq, grid, w, L, status,
                            stream)) != cudaSuccess)
        return e;
      prm.b = b;
      prm.c0 = c0;
      {
        ProfScope pf("bwd_tile", stream);
#define MSA_BWD(D_, BS_)                                                                              \
  do {                                                                                                \
    auto kern = bwd_tile_kernel<D_, BS_>;                                                             \
    const size_t smem = BwdSmem<D_, BS_>::kTotal;                                                     \
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) !=  \
        cudaSuccess)                                                                                  \
      return e;                                                                                       \
    kern<<<grid, kBwdThreads, smem, stream>>>(prm);                                                   \
  } while (0)
        if (d == 128) {
          if (Bs == 128)
            MSA_BWD(128, 128);
          else if (Bs == 64)
            MSA_BWD(128, 64);
          else
            MSA_BWD(128, 32);
        } else {
          if (Bs == 128)
            MSA_BWD(64, 128);
          else if (Bs == 64)
            MSA_BWD(64, 64);
          else
            MSA_BWD(64, 32);
        }
#undef MSA_BWD
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      {
        ProfScope pf("bwd_dq_combine", stream);
        const int64_t items = int64_t(cq) * G;
        const int nvec = hpg * d / 4;
        const int64_t need = (items + 7) / 8;
        const int cgrid = int(need < int64_t(grid) * 8 ? need : int64_t(grid) * 8);
        const float4* pd = reinterpret_cast<const float4*>(w + L.part_o);
        __nv_bfloat16* dq16 = static_cast<__nv_bfloat16*>(dq);
#define MSA_DQC(NU_)                                                                                             \
  bwd_dq_combine_kernel<NU_><<<cgrid, 256, 0, stream>>>(sel, q_offset, kv_len, pd, rev, b, Nq, Nk, Hq, G, K, Bs, \
                                                        nblk, d, c0, cq, scale, dq16)
        if (nvec <= 32)
          MSA_DQC(1);
        else if (nvec <= 64)
          MSA_DQC(2);
        else if (nvec <= 128)
          MSA_DQC(4);
        else
          MSA_DQC(8);
#undef MSA_DQC
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
    }
    {
      ProfScope pf("bwd_kv_store", stream);
      const int64_t n4 = kv_elems / 4;
      const int64_t need = (n4 + 255) / 256;
      const int sgrid = int(need < int64_t(grid) * 8 ? need : int64_t(grid) * 8);
      bwd_kv_store_kernel<<<sgrid, 256, 0, stream>>>(
          reinterpret_cast<const float4*>(w + W.dk_acc), reinterpret_cast<const float4*>(w + W.dv_acc), scale, n4,
          reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dk) + int64_t(b) * kv_elems),
          reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dv) + int64_t(b) * kv_elems));
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace msa
