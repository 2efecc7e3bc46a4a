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
// the same cost-balanced contiguous runs of a persistent grid, with the
// block's K and V resident in shared memory for the run of its bin. Two tile
// kernels:
//   bwd_tc_kernel (blocks of 128 keys, tcgen05): keys along M; S^T, dP^T in
//     TMEM; P^T, dS^T written back over them (A operands of dV, dK); dQ from
//     dS in shared memory; dV, dK accumulated in TMEM over the bin's run (see
//     the kernel's own notes below).
//   bwd_tile_kernel (blocks of 32 or 64 keys, mma.sync): per tile
//     1. S^T = K Q^T and dP^T = V dO^T (keys along M); P^T and dS^T formed in
//        registers and written to shared memory as bf16;
//     2. dV += P^T dO and dK += dS^T Q, accumulated in registers over the run's
//        tiles of one bin (each warp a 16-key strip x a slice of d);
//     3. dQ = dS K for the tile's rows while the next tile's rows are gathered.
// dQ leaves both kernels as a bf16 partial per (entry, head) row. When a bin's
// run ends, dK and dV are added into per-sequence fp32 accumulators with
// fire-and-forget vector atomics (a bin held whole by one CTA gets one add per
// query chunk; a bin split over CTAs gets one per CTA). bwd_dq_combine then
// sums each row's slot partials in slot order (deterministic) and
// bwd_kv_store rounds dk and dv.
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
__device__ __forceinline__ void cp16_addr(uint32_t dst, const void* src, bool in) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(in ? 16u : 0u) : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src, bool in) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(tc::smem_u32(dst)), "l"(src), "r"(in ? 4u : 0u)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// 8 registers -> 32 TMEM lanes x 8 columns
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

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
  const int* cta_start;                   // [grid + 1]
  const int32_t* q_offset;
  const int32_t* kv_len;
  uint4* part_dq;  // per tile, chunk-major bf16: 8-column chunk c of tile row r at (z * D/8 + c) * 128 + r; unscaled
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
  static_assert(MT >= 1 && MT <= 4 && NTD % 2 == 0 && RW % 32 == 0, "tile split (blocks of 32 or 64 keys)");
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
    // ---- 3. dQ rows [16 warp, +16) = dS K, keys reduced; bf16 partial rows
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
          if ((r >> p.hpg_log2) < tl.z) {
            // columns cq + n * 8 + 2 tq (+1): bf16 pair tq of 8-column chunk (cq + n * 8) / 8
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.part_dq + (int64_t(z) * (D / 8) + (cq >> 3)) * kBwdRows + r) + tq;
#pragma unroll
            for (int n = 0; n < QC / 8; ++n) dst[n * kBwdRows * 4] = bwd_pack(acc[n][2 * hr], acc[n][2 * hr + 1]);
          }
        }
      }
    }
    // ---- end of the bin's run: add dK, dV into the sequence's accumulators
    const int next_bin = more ? p.tiles[z + 1].x : -1;
    if (next_bin != bin) {  // fire-and-forget vector adds (see the tcgen05 kernel's flush)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int j = t * BS + mt * 16 + gq + 8 * hr;
        if (j < p.Nk) {
          const int64_t base = (int64_t(j) * p.G + g) * D + wp * DW + 2 * tq;
#pragma unroll
          for (int n = 0; n < NTD; ++n) {
            float* pk = p.dk_acc + base + n * 8;
            float* pv = p.dv_acc + base + n * 8;
            asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(pk), "f"(dk[n][2 * hr]), "f"(dk[n][2 * hr + 1])
                         : "memory");
            asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(pv), "f"(dv[n][2 * hr]), "f"(dv[n][2 * hr + 1])
                         : "memory");
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
        load_kv(bin);
      }
    }
    nb ^= 1;
  }
}


// ---------------------------------------------------------------------------
// tcgen05 tile kernel for blocks of 128 keys (keys along M = 128 TMEM lanes).
// Per tile: S^T = K Q^T and dP^T = V dO^T into TMEM; the epilogue warpgroup
// (one thread per key) forms P^T and dS^T, writes them back over S^T and dP^T
// as bf16 pairs and dS^T to shared memory (MN-major, 128B-swizzled); then
// dV += P^T dO and dK += dS^T Q take their A operand from TMEM (dO and Q are
// read MN-major from the gathered tile) and dQ = dS K takes dS from shared
// memory into the TMEM columns that P^T and dS^T left free (bf16 partials,
// summed in fp32 by the combine). dV and dK stay
// in TMEM for the run of the bin's tiles.
// TMEM columns: S^T [0, 128) (P^T packed into [0, 64), dQ half 0 at [64, 128)),
// dP^T [128, 256) (dS^T packed into [128, 192), dQ half 1 at [192, 256)),
// dV [256, 256 + D), dK [256 + D, 256 + 2 D).
// Warps 0-3 gather the tile's q and dout rows (cp.async, 128B-swizzled K-major,
// two ring slots) and its row data (lse, delta, last visible key); warps 4-7
// are the epilogue; warp 8 loads K and V by TMA; warp 9 owns TMEM and issues
// the MMAs. Every wait is bounded.
// ---------------------------------------------------------------------------
constexpr int kTcThreads = 320;
constexpr int kTcBs = 128;

__host__ __device__ constexpr uint32_t bwd_idesc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | (uint32_t(a_mn) << 15)       // A major-ness (1 = MN-major)
         | (uint32_t(b_mn) << 16)       // B major-ness (1 = MN-major)
         | (uint32_t(N >> 3) << 17)     // N / 8
         | (uint32_t(M >> 4) << 24);    // M / 16
}

template <int D>
struct TcSmem {
  static constexpr uint32_t kHalf = kTcBs * 128;           // one 64-wide half of a 128-row operand
  static constexpr uint32_t kKV = D * kTcBs * 2;           // K or V block
  static constexpr uint32_t kRowsT = kBwdRows * D * 2;     // q or dout tile
  static constexpr uint32_t kSlot = 2 * kRowsT;            // q + dout
  static constexpr uint32_t kDs = kBwdRows * kTcBs * 2;    // dS (MN-major)
  static constexpr uint32_t oK = 0, oV = kKV, oRing = 2 * kKV, oDs = oRing + 2 * kSlot;
  static constexpr uint32_t oRowF = oDs + kDs;             // [2][2][128] float: lse * log2(e), delta
  static constexpr uint32_t oLim = oRowF + 2 * kBwdRows * 8;  // [2][128] int8: last visible key of the row - t*128
  static constexpr uint32_t oBar = oLim + 2 * kBwdRows;     // 8-byte aligned
  static constexpr uint32_t kBars = 13;
  static constexpr uint32_t kTotal = oBar + kBars * 8 + 16;
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const BwdParams p,
                  uint32_t* status) {
  using SM = TcSmem<D>;
  constexpr int NH = D / 64;
  constexpr uint32_t kIdS = bwd_idesc(128, 128, false, false);  // S^T, dP^T: K and V x q / dout rows
  constexpr uint32_t kIdKV = bwd_idesc(128, D, false, true);    // dV, dK: A from TMEM, B = dout / q MN-major
  constexpr uint32_t kIdQ = bwd_idesc(128, 64, true, true);     // dQ half: A = dS MN-major, B = K half MN-major
  constexpr uint32_t kColDv = 256, kColDk = 256 + D;
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  if (tc::smem_u32(tc_smem) & 1023u) {  // the swizzled operands need 1024-byte alignment
    if (threadIdx.x == 0) set_status(status, MSA_ERR_CUDA);
    return;
  }
  uint8_t* k_buf = tc_smem + SM::oK;
  uint8_t* v_buf = tc_smem + SM::oV;
  uint8_t* ring = tc_smem + SM::oRing;
  uint8_t* ds_buf = tc_smem + SM::oDs;
  float* rowf = reinterpret_cast<float*>(tc_smem + SM::oRowF);  // slot s: lse at [2 s][r], delta at [2 s + 1][r]
  int8_t* lim_s = reinterpret_cast<int8_t*>(tc_smem + SM::oLim);
  uint64_t* bars = reinterpret_cast<uint64_t*>(tc_smem + SM::oBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;   // [2]
  uint64_t* q_empty = bars + 4;  // [2]
  uint64_t* s_full = bars + 6;
  uint64_t* p_full = bars + 7;
  uint64_t* dq_full = bars + 8;
  uint64_t* tm_empty = bars + 9;
  uint64_t* acc_full = bars + 10;
  uint64_t* acc_empty = bars + 11;
  uint64_t* done_bar = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + SM::kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kGather0 = 0, kEpi0 = 4, kTmaWarp = 8, kMmaWarp = 9;
  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    tc::mbar_init(kv_empty, 1);
    for (int r = 0; r < 2; ++r) {
      tc::mbar_init(&q_full[r], 4);
      tc::mbar_init(&q_empty[r], 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, 4);
    tc::mbar_init(dq_full, 1);
    tc::mbar_init(tm_empty, 4);
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(acc_empty, 4);
    tc::mbar_init(done_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tc::tma_prefetch(&tmK);
    tc::tma_prefetch(&tmV);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int z0 = p.cta_start[blockIdx.x], z1 = p.cta_start[blockIdx.x + 1];
  const int n = z1 - z0;
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(status, MSA_ERR_TIMEOUT);
  };
  const SeqView sv = seq_view(p.q_offset, p.kv_len, p.b, p.Nq, p.Nk, false);

  if (warp < kEpi0) {
    // ------------------- q / dout row gather + row data -------------------
    // Warp gw fills rows [32 gw, 32 gw + 32) of every tile; a warp
    // instruction covers two whole 256-byte rows (16-byte chunks, swizzled).
    const int gw = warp - kGather0;
    constexpr int kCpr = D / 8, kRpi = 32 / kCpr;
    const int chunk = lane % kCpr, sub = lane / kCpr;
    const uint32_t hf = uint32_t(chunk) >> 3, cc = uint32_t(chunk) & 7u;
    const int hmask = p.hpg - 1;
    const int r = gw * 32 + lane;  // this lane's row (row data)
    const int e = r >> p.hpg_log2;
    // tile records and entries are fetched one tile ahead, off the critical path
    int4 tl_n = make_int4(0, 0, 0, 0);
    int ent_n = -1;
    auto fetch = [&](int z) {
      tl_n = p.tiles[z0 + z];
      ent_n = e < tl_n.z ? p.entries[tl_n.y + e] : -1;
    };
    if (n > 0) fetch(0);
    for (int z = 0; z < n; ++z) {
      const int slot = z & 1;
      const int4 tl = tl_n;
      const int ent = ent_n;
      if (z + 1 < n) fetch(z + 1);
      if (!tc::mbar_wait(&q_empty[slot], ((z >> 1) & 1) ^ 1, abort_flag)) {
        fail();
        break;
      }
      const int g = tl.x / p.nblk, t = tl.x % p.nblk;
      const int il = ent >= 0 ? (ent >> 6) : 0;
      const int64_t qrow = (int64_t(p.b) * p.Nq + p.c0 + il) * p.Hq + g * p.hpg + (r & hmask);
      const uint32_t qs = tc::smem_u32(ring + slot * SM::kSlot), os = qs + SM::kRowsT;
#pragma unroll 4
      for (int it = 0; it < 32 / kRpi; ++it) {
        const int rr = it * kRpi + sub;  // row within this warp's 32
        const int row = gw * 32 + rr;
        const int ent_r = __shfl_sync(0xffffffffu, ent, rr);
        const int64_t qr = __shfl_sync(0xffffffffu, qrow, rr);
        const uint32_t dst = hf * (kBwdRows * 128) + row * 128 + ((cc ^ uint32_t(row & 7)) << 4);
        cp16_addr(qs + dst, p.q + qr * D + chunk * 8, ent_r >= 0);
        cp16_addr(os + dst, p.dout + qr * D + chunk * 8, ent_r >= 0);
      }
      // the row's lse and delta by 4-byte copies (zero for padding rows)
      cp4(rowf + (2 * slot) * kBwdRows + r, p.lse + qrow, ent >= 0);
      cp4(rowf + (2 * slot + 1) * kBwdRows + r, p.delta + qrow, ent >= 0);
      cp_commit();
      int lim = -1;
      if (ent >= 0 && sv.ok) lim = min(min(sv.q0 + p.c0 + il, sv.L - 1) - t * kTcBs, kTcBs - 1);
      lim_s[slot * kBwdRows + r] = int8_t(lim);
      cp_wait_all();
      rowf[(2 * slot) * kBwdRows + r] *= kLog2eBwd;  // the epilogue wants lse in log2 units
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&q_full[slot]);
    }
    cp_wait_all();
  } else if (warp < kTmaWarp) {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;
    const int key = quarter * 32 + lane;  // TMEM lane: key of S^T, dP^T, dV, dK; row of dQ
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    int nbins = 0;
    int4 tl_n = n > 0 ? p.tiles[z0] : make_int4(0, 0, 0, 0);
    // tile z's dQ row (bf16 pairs) waits in registers and is stored while the
    // MMAs of tile z + 1 run (the epilogue would otherwise idle there)
    uint32_t dq_pk[D / 2];
    uint4* dq_dst = nullptr;
    auto store_dq = [&]() {
      if (dq_dst != nullptr) {
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8)
          dq_dst[c8 * kBwdRows] = make_uint4(dq_pk[4 * c8], dq_pk[4 * c8 + 1], dq_pk[4 * c8 + 2], dq_pk[4 * c8 + 3]);
        dq_dst = nullptr;
      }
    };
    for (int z = 0; z < n; ++z) {
      const int slot = z & 1;
      const int4 tl = tl_n;
      if (z + 1 < n) tl_n = p.tiles[z0 + z + 1];  // in flight while this tile is processed
      const int bin = tl.x;
      // the slot's row data come from the gather warps: observe their phase
      // directly (it has completed: the MMA read the slot before s_full)
      if (!tc::mbar_wait(s_full, z & 1, abort_flag) || !tc::mbar_wait(&q_full[slot], (z >> 1) & 1, abort_flag)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      const float* lse_r = rowf + (2 * slot) * kBwdRows;  // lse * log2(e)
      const float* dlt_r = rowf + (2 * slot + 1) * kBwdRows;
      const int8_t* lm = lim_s + slot * kBwdRows;
      const uint32_t ds_row = tc::smem_u32(ds_buf) + uint32_t(key) * 128u;
      const float sl2 = p.scale * kLog2eBwd;
#pragma unroll 1
      for (int c = 0; c < kBwdRows / 16; ++c) {  // 16 tile rows at a time
        uint32_t sv16[16], dv16[16];
        tc::tmem_ld_32x32b_x16(tmem + lane_base + uint32_t(c * 16), sv16);
        tc::tmem_ld_32x32b_x16(tmem + lane_base + 128u + uint32_t(c * 16), dv16);
        // the 16 rows' data in four vector loads (all threads read the same words: broadcast)
        float lse16[16], dlt16[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 a4 = reinterpret_cast<const float4*>(lse_r + c * 16)[q4];
          const float4 b4 = reinterpret_cast<const float4*>(dlt_r + c * 16)[q4];
          lse16[4 * q4] = a4.x; lse16[4 * q4 + 1] = a4.y; lse16[4 * q4 + 2] = a4.z; lse16[4 * q4 + 3] = a4.w;
          dlt16[4 * q4] = b4.x; dlt16[4 * q4 + 1] = b4.y; dlt16[4 * q4 + 2] = b4.z; dlt16[4 * q4 + 3] = b4.w;
        }
        const uint4 lim16 = reinterpret_cast<const uint4*>(lm)[c];
        const uint32_t limw[4] = {lim16.x, lim16.y, lim16.z, lim16.w};
        tc::tmem_ld_wait();
        uint32_t pk[8], dk2[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float pp[2], dd[2];
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int jr = j + e2;
            const int lim_r = int(int8_t((limw[jr >> 2] >> (8 * (jr & 3))) & 0xffu));
            const float pr = key <= lim_r ? bwd_ex2(fmaf(__uint_as_float(sv16[jr]), sl2, -lse16[jr])) : 0.f;
            pp[e2] = pr;
            dd[e2] = pr * (__uint_as_float(dv16[jr]) - dlt16[jr]);
          }
          pk[j >> 1] = bwd_pack(pp[0], pp[1]);
          dk2[j >> 1] = bwd_pack(dd[0], dd[1]);
        }
        tmem_st_x8(tmem + lane_base + uint32_t(c * 8), pk);  // P^T rows 16 c.. packed over S^T already read
        tmem_st_x8(tmem + lane_base + 128u + uint32_t(c * 8), dk2);
        // dS^T row of this key: rows [16 c, 16 c + 16) = two 16-byte chunks of half (16 c) / 64
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const uint32_t half = uint32_t(c >> 2), ch = uint32_t((c & 3) * 2 + q2);
          const uint32_t addr = ds_row + half * SM::kHalf + ((ch ^ uint32_t(key & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(dk2[q2 * 4]), "r"(dk2[q2 * 4 + 1]),
                       "r"(dk2[q2 * 4 + 2]), "r"(dk2[q2 * 4 + 3])
                       : "memory");
        }
      }
      tc::tmem_st_wait();
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(p_full);
      store_dq();  // the previous tile's dQ, under this tile's dV/dK/dQ MMAs
      // dQ rows of this tile (lane = row) out of TMEM, packed to the bf16 partial
      if (!tc::mbar_wait(dq_full, z & 1, abort_flag)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      uint32_t qv[D];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        tc::tmem_ld_32x32b_x32(tmem + lane_base + (h == 0 ? 64u : 192u), qv + h * 64);
        tc::tmem_ld_32x32b_x32(tmem + lane_base + (h == 0 ? 64u : 192u) + 32u, qv + h * 64 + 32);
      }
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tm_empty);
#pragma unroll
      for (int x = 0; x < D / 2; ++x) dq_pk[x] = bwd_pack(__uint_as_float(qv[2 * x]), __uint_as_float(qv[2 * x + 1]));
      // bf16 partial, chunk-major: a warp store covers 512 contiguous bytes
      if ((key >> p.hpg_log2) < tl.z) dq_dst = p.part_dq + int64_t(z0 + z) * (D / 8) * kBwdRows + key;
      if (z + 1 == n || tl_n.x != bin) {  // last tile of the bin's run
        // dV and dK of the bin's run (lane = key) into the sequence's accumulators
        if (!tc::mbar_wait(acc_full, nbins & 1, abort_flag)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        // fire-and-forget vector adds (no load on the epilogue's path): a bin
        // that this CTA holds whole has this one flush per query chunk, so its
        // sum is deterministic; a split bin's CTAs add in any order
        const int g = bin / p.nblk, t = bin % p.nblk;
        const int j = t * kTcBs + key;
        float* dkr = p.dk_acc + (int64_t(j) * p.G + g) * D;
        float* dvr = p.dv_acc + (int64_t(j) * p.G + g) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t a[32], b2[32];
          tc::tmem_ld_32x32b_x32(tmem + lane_base + kColDv + uint32_t(c * 32), a);
          tc::tmem_ld_32x32b_x32(tmem + lane_base + kColDk + uint32_t(c * 32), b2);
          tc::tmem_ld_wait();
          if (j < p.Nk) {
#pragma unroll
            for (int x = 0; x < 32; x += 4) {
              float4* pv = reinterpret_cast<float4*>(dvr + c * 32 + x);
              float4* pk4 = reinterpret_cast<float4*>(dkr + c * 32 + x);
              const float4 av = make_float4(__uint_as_float(a[x]), __uint_as_float(a[x + 1]), __uint_as_float(a[x + 2]),
                                            __uint_as_float(a[x + 3]));
              const float4 bk = make_float4(__uint_as_float(b2[x]), __uint_as_float(b2[x + 1]),
                                            __uint_as_float(b2[x + 2]), __uint_as_float(b2[x + 3]));
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(pv), "f"(av.x), "f"(av.y), "f"(av.z),
                           "f"(av.w)
                           : "memory");
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(pk4), "f"(bk.x), "f"(bk.y), "f"(bk.z),
                           "f"(bk.w)
                           : "memory");
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(acc_empty);
        ++nbins;
      }
    }
    store_dq();  // the last tile's dQ
  } else if (warp == kTmaWarp) {
    // ------------------------------ K/V producer ------------------------------
    if (lane == 0) {
      int prev_bin = -1, loads = 0;
      for (int z = 0; z < n; ++z) {
        const int bin = p.tiles[z0 + z].x;
        if (bin == prev_bin) continue;
        prev_bin = bin;
        if (!tc::mbar_wait(kv_empty, (loads & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        const int g = bin / p.nblk, t = bin % p.nblk;
        tc::mbar_arrive_expect_tx(kv_full, 2 * SM::kKV);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          tc::tma_load_4d(k_buf + h * SM::kHalf, &tmK, kv_full, h * 64, g, t * kTcBs, p.b);
          tc::tma_load_4d(v_buf + h * SM::kHalf, &tmV, kv_full, h * 64, g, t * kTcBs, p.b);
        }
        ++loads;
      }
      int zero = 0;
      if (loads > 0) tc::mbar_wait(kv_full, (loads - 1) & 1, &zero);  // drain the last copy
    }
  } else {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      int kv_uses = 0, nbins = 0, prev_bin = -1;
      const uint32_t ka = tc::smem_u32(k_buf), va = tc::smem_u32(v_buf), dsa = tc::smem_u32(ds_buf);
      // Descriptors from 32-bit low words (start address, leading offset) with
      // one constant high word (8-row groups 1024 B apart, 128B swizzle): one
      // add per operand and MMA instead of building two 64-bit descriptors
      constexpr uint32_t kDescHi = tc::smem_desc_hi(1024, 2);
      const uint32_t ka16 = tc::smem_desc_lo(ka, 16), va16 = tc::smem_desc_lo(va, 16);
      const uint32_t kaH = tc::smem_desc_lo(ka, SM::kHalf), dsaH = tc::smem_desc_lo(dsa, SM::kHalf);
      int bin_n = n > 0 ? p.tiles[z0].x : -1;
      for (int z = 0; z < n; ++z) {
        const int slot = z & 1;
        const int bin = bin_n;
        bin_n = z + 1 < n ? p.tiles[z0 + z + 1].x : -1;  // one tile ahead
        const bool first = bin != prev_bin;
        prev_bin = bin;
        if (first) {
          if (!tc::mbar_wait(kv_full, kv_uses & 1, abort_flag)) {
            fail();
            break;
          }
          ++kv_uses;
        }
        if (!tc::mbar_wait(&q_full[slot], (z >> 1) & 1, abort_flag) ||
            (z > 0 && !tc::mbar_wait(tm_empty, (z - 1) & 1, abort_flag))) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const uint32_t qa = tc::smem_u32(ring + slot * SM::kSlot), oa = qa + SM::kRowsT;
        const uint32_t qa16 = tc::smem_desc_lo(qa, 16), oa16 = tc::smem_desc_lo(oa, 16);
        const uint32_t qaL = tc::smem_desc_lo(qa, kBwdRows * 128), oaL = tc::smem_desc_lo(oa, kBwdRows * 128);
        // S^T = K Q^T, dP^T = V dO^T (both operands K-major along d)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          tc::mma_f16_ss_lo<kDescHi>(tmem, ka16 + (((kk >> 2) * SM::kHalf + off) >> 4),
                                     qa16 + (((kk >> 2) * (kBwdRows * 128) + off) >> 4), kIdS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          tc::mma_f16_ss_lo<kDescHi>(tmem + 128u, va16 + (((kk >> 2) * SM::kHalf + off) >> 4),
                                     oa16 + (((kk >> 2) * (kBwdRows * 128) + off) >> 4), kIdS, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(s_full);
        if (!tc::mbar_wait(p_full, z & 1, abort_flag) ||
            (first && nbins > 0 && !tc::mbar_wait(acc_empty, (nbins - 1) & 1, abort_flag))) {
          fail();
          break;
        }
        tc::fence_after_sync();
        // dV += P^T dO, dK += dS^T Q: A from TMEM (16 rows = 8 packed columns per step), B MN-major
#pragma unroll
        for (int kk = 0; kk < kBwdRows / 16; ++kk)
          tc::mma_f16_ts_lo<kDescHi>(tmem + kColDv, tmem + uint32_t(kk) * 8u, oaL + ((kk * 16 * 128) >> 4), kIdKV,
                                     (first && kk == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < kBwdRows / 16; ++kk)
          tc::mma_f16_ts_lo<kDescHi>(tmem + kColDk, tmem + 128u + uint32_t(kk) * 8u, qaL + ((kk * 16 * 128) >> 4),
                                     kIdKV, (first && kk == 0) ? 0u : 1u);
        // dQ = dS K, one 64-column half of d at a time (A = dS MN-major over the tile rows)
#pragma unroll
        for (int h = 0; h < NH; ++h) {
#pragma unroll
          for (int kk = 0; kk < kTcBs / 16; ++kk)
            tc::mma_f16_ss_lo<kDescHi>(tmem + (h == 0 ? 64u : 192u), dsaH + ((kk * 16 * 128) >> 4),
                                       kaH + ((h * SM::kHalf + kk * 16 * 128) >> 4), kIdQ, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(dq_full);
        tc::mma_commit(&q_empty[slot]);
        if (bin_n != bin) {  // last tile of the bin's run
          tc::mma_commit(acc_full);
          tc::mma_commit(kv_empty);
          ++nbins;
        }
      }
      int zero = 0;
      tc::mma_commit(done_bar);
      tc::mbar_wait(done_bar, 0, &zero);
    }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dq: one warp per (query, group) sums its valid slots' partial rows in slot
// order; NU 8-column bf16 chunks of the group's hpg x D row block per lane
// ---------------------------------------------------------------------------
template <int NU>
__global__ void __launch_bounds__(256) bwd_dq_combine_kernel(
    const int32_t* __restrict__ sel, const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len,
    const uint4* __restrict__ part_dq, const int* __restrict__ rev, int b, int Nq, int Nk, int Hq, int G, int K,
    int Bs, int nblk, int D, int c0, int cq, float scale, __nv_bfloat16* __restrict__ dq) {
  // partial rows of an entry at position e: tile e / per_tile, rows (e % per_tile) * hpg + head,
  // 8-column chunk c of row r of tile z at (z * D/8 + c) * 128 + r; lane vector vi = chunk * hpg + head
  constexpr int kWarps = 256 / 32;
  constexpr int kBatch = NU <= 2 ? 8 : 4;  // slots whose loads are in flight together
  __shared__ int slot_e[kWarps][kMaxK];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int hpg = Hq / G;
  const int nvec = hpg * D / 8;  // 16-byte chunks per slot
  const int per_tile = kBwdRows / hpg;
  int voff[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const int vi = lane + 32 * u;
    voff[u] = vi < nvec ? (vi / hpg) * kBwdRows + vi % hpg : 0;
  }
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
    float acc[NU][8];
#pragma unroll
    for (int u = 0; u < NU; ++u)
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[u][x] = 0.f;
    for (int j0 = 0; j0 < nv; j0 += kBatch) {
      uint4 x[kBatch][NU];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const bool in = j0 + jj < nv;
        const int e = in ? slot_e[wl][j0 + jj] : 0;
        const int64_t base = int64_t(e / per_tile) * (D / 8) * kBwdRows + (e % per_tile) * hpg;
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const int vi = lane + 32 * u;
          x[jj][u] = (in && vi < nvec) ? part_dq[base + voff[u]] : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj)
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const uint32_t w4[4] = {x[jj][u].x, x[jj][u].y, x[jj][u].z, x[jj][u].w};
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {  // bf16 -> fp32 is a 16-bit shift (low half = even column)
            acc[u][2 * q2] += __uint_as_float(w4[q2] << 16);
            acc[u][2 * q2 + 1] += __uint_as_float(w4[q2] & 0xffff0000u);
          }
        }
    }
    __nv_bfloat16* drow = dq + ((int64_t(b) * Nq + i) * Hq + int64_t(g) * hpg) * D;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int vi = lane + 32 * u;
      if (vi < nvec)
        *reinterpret_cast<uint4*>(drow + (vi % hpg) * D + (vi / hpg) * 8) =
            make_uint4(bwd_pack(acc[u][0] * scale, acc[u][1] * scale), bwd_pack(acc[u][2] * scale, acc[u][3] * scale),
                       bwd_pack(acc[u][4] * scale, acc[u][5] * scale), bwd_pack(acc[u][6] * scale, acc[u][7] * scale));
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
  KvoLayout L;  // inversion; its partial area (bf16 rows of d) holds the dq partials
  size_t delta, dk_acc, dv_acc, end;
};

BwdLayout bwd_layout(int B, int Nq, int Nk, int Hq, int G, int d, int Bs, int K) {
  BwdLayout W;
  W.L = kvo_layout(Nq, Hq, G, d, Bs, K, Nk);
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
  const int cq_max = chunk_tokens(Nq, Hq, K, d);
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
  prm.cta_start = reinterpret_cast<const int*>(w + L.cta_start);
  prm.q_offset = q_offset;
  prm.kv_len = kv_len;
  prm.part_dq = reinterpret_cast<uint4*>(w + L.part_o);
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
  CUtensorMap tmK, tmV;  // blocks of 128 keys, 64-column halves, 128B swizzle (the tcgen05 path)
  if (Bs == kTcBs) {
    const uint64_t dims[4] = {uint64_t(d), uint64_t(Hkv), uint64_t(Nk), uint64_t(B)};
    const uint64_t strides[3] = {uint64_t(d) * 2, uint64_t(Hkv) * d * 2, uint64_t(Nk) * Hkv * d * 2};
    const uint32_t box[4] = {64, 1, uint32_t(kTcBs), 1};
    if (!make_tmap_bf16(&tmK, k, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_bf16(&tmV, v, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }

  for (int b = 0; b < B; ++b) {
    if ((e = cudaMemsetAsync(w + W.dk_acc, 0, W.end - W.dk_acc, stream)) != cudaSuccess) return e;
    for (int c0 = 0; c0 < Nq; c0 += cq_max) {
      const int cq = Nq - c0 < cq_max ? Nq - c0 : cq_max;
      if ((e = invert_chunk(sel, q_offset, kv_len, b, Nq, Nk, G, K, Bs, per_tile, c0, cq, grid, w, L, status,
                            stream)) != cudaSuccess)
        return e;
      prm.b = b;
      prm.c0 = c0;
      if (Bs == kTcBs) {
        ProfScope pf("bwd_tile_tc", stream);
        if (d == 128) {
          auto kern = bwd_tc_kernel<128>;
          if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(TcSmem<128>::kTotal))) != cudaSuccess)
            return e;
          kern<<<grid, kTcThreads, TcSmem<128>::kTotal, stream>>>(tmK, tmV, prm, status);
        } else {
          auto kern = bwd_tc_kernel<64>;
          if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(TcSmem<64>::kTotal))) != cudaSuccess)
            return e;
          kern<<<grid, kTcThreads, TcSmem<64>::kTotal, stream>>>(tmK, tmV, prm, status);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      } else {
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
        if (d == 128) {  // blocks of 32 or 64 keys (128 takes the tcgen05 kernel)
          if (Bs == 64)
            MSA_BWD(128, 64);
          else
            MSA_BWD(128, 32);
        } else {
          if (Bs == 64)
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
        const int nvec = hpg * d / 8;
        const int64_t need = (items + 7) / 8;
        const int cgrid = int(need < int64_t(grid) * 8 ? need : int64_t(grid) * 8);
        const uint4* pd = reinterpret_cast<const uint4*>(w + L.part_o);
        __nv_bfloat16* dq16 = static_cast<__nv_bfloat16*>(dq);
#define MSA_DQC(NU_)                                                                                             \
  bwd_dq_combine_kernel<NU_><<<cgrid, 256, 0, stream>>>(sel, q_offset, kv_len, pd, rev, b, Nq, Nk, Hq, G, K, Bs, \
                                                        nblk, d, c0, cq, scale, dq16)
        if (nvec <= 32)
          MSA_DQC(1);
        else if (nvec <= 64)
          MSA_DQC(2);
        else
          MSA_DQC(4);
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
