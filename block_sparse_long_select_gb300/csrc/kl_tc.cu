// KL auxiliary forward, tile pass on tcgen05 (bf16, d = 128, di = 64, blocks of
// 128 keys). (quant_prune_distill post 751, "Метод": the index branch is
// trained with the KL divergence to the head-averaged main-branch
// distribution; hyper.ai summary, "方法": the two are aligned over the selected
// tokens.) For each (group, key block) tile of the KV-outer inversion
// (128 / hpg entries x hpg heads), per entry e over the block's visible keys j:
//   pbar_j = (1 / hpg) sum_h exp(scale q_h.k_j - lse_h)     (main branch, head mean)
//   s_j    = iq_e . ik_j                                     (index score)
//   partial = (sum_j pbar_j log pbar_j, sum_j pbar_j s_j, max_j s_j, sum_j exp(s_j - max))
// which the combine merges over the entry's selected blocks into
//   KL = sum pbar log pbar - sum pbar s + logsumexp s.
//
// Keys lie along M (the 128 TMEM lanes): S^T = K q^T (128 x 128 rows) and
// I^T = IK iq^T (128 x entries) land in TMEM, so the epilogue thread of key j
// holds all heads of every entry in neighbouring columns (the head mean is
// in-thread). The sums over keys are a reduce-scatter across the warp's lanes
// (lanes l and l + 16 end with entry l of a group of 16) and a four-warp
// merge in shared memory. NS epilogue warpgroups (NS = 3 when three TMEM sets of
// 128 + E columns fit, else 2) take tiles in turn, each with its own TMEM set,
// so the MMAs of the next tiles run under the epilogues. The gathered rows and
// a tile's row data (lse, visibility limits) sit in separate rings: a row slot
// is free once the MMA has read it, a row-data slot once the epilogue has, so
// the copies of tile z start as soon as the MMA of tile z - NR is done, well
// before the epilogue of tile z - NS releases the TMEM set tile z needs.
// Warps 0..4 NS - 1 epilogue (warpgroup z % NS takes tile z), then two warps
// gathering q rows, index-query rows and row data (cp.async, 128B-swizzled
// K-major; tile records and entries fetched a tile ahead), one TMA warp for K
// and IK per bin, one TMEM owner and MMA issuer. Every wait is bounded.
#include <cmath>

#include "msa_internal.cuh"
#include "tc_utils.cuh"

namespace msa {
namespace {

constexpr int kKtEG = 16;  // entries per reduce-scatter group
constexpr int kKtD = 128, kKtDI = 64, kKtBs = 128, kKtRows = kKvoRows;
constexpr float kKtLog2e = 1.4426950408889634f;
constexpr float kKtLn2 = 0.6931471805599453f;

__device__ __forceinline__ float kt_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float kt_lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void kt_cp16(uint32_t dst, const void* src, bool in) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(in ? 16u : 0u) : "memory");
}

__device__ __forceinline__ void cp_async_commit_kt() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_kt() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// all but the most recently committed group have landed
__device__ __forceinline__ void cp_async_wait_but_one_kt() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__host__ __device__ constexpr uint32_t kt_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// reduce-scatter of 16 per-lane values: four levels within each 16-lane half,
// then one exchange across the halves; afterwards v[0] of lane l is the sum
// over all 32 lanes of the original v[l & 15]
__device__ __forceinline__ void kt_rs_sum(float (&v)[kKtEG], int lane) {
#pragma unroll
  for (int o = kKtEG / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16);
}
// merge of two (max, exp-sum) pairs (natural-log units; -inf = empty)
__device__ __forceinline__ void kt_lse_merge(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  const float a = m == -INFINITY ? 0.f : l * kt_ex2((m - M) * kKtLog2e);
  const float b = m2 == -INFINITY ? 0.f : l2 * kt_ex2((m2 - M) * kKtLog2e);
  m = M;
  l = a + b;
}
template <int HPG>
struct KtSmem {
  static constexpr int E = kKtRows / HPG;                  // entries per tile
  static constexpr int NS = 512 / (128 + E) >= 3 ? 3 : 2;  // TMEM sets = epilogue warpgroups
  static constexpr int NR = NS + 1;                         // gathered-row ring slots
  static constexpr int ND = 8;                              // row-data ring slots
  static constexpr int kThreads = (4 * NS + 4) * 32;
  static constexpr uint32_t kHalf = kKtRows * 128;         // one 64-wide half of a 128-row operand
  static constexpr uint32_t kK = kKtBs * kKtD * 2;         // K block (two halves)
  static constexpr uint32_t kIK = kKtBs * kKtDI * 2;       // IK block (one half)
  static constexpr uint32_t kQ = kKtRows * kKtD * 2;       // gathered q rows
  static constexpr uint32_t kIQ = E * kKtDI * 2;           // gathered index-query rows (E x 128 B)
  static constexpr uint32_t kSlot = kQ + kIQ;              // multiple of 1024
  static constexpr uint32_t oK = 0, oIK = kK, oRing = kK + kIK;
  static constexpr uint32_t oLse = oRing + NR * kSlot;     // [ND][128] lse * log2(e)
  static constexpr uint32_t oLim = oLse + ND * kKtRows * 4;  // [ND][E] last visible key - t * 128 (-1: none)
  static constexpr uint32_t oRed = oLim + ND * E * 4;       // [NS warpgroups][2][4 warps][16] float4 per-warp sums
  static constexpr uint32_t oBar = oRed + NS * 2 * 4 * kKtEG * 16;
  static constexpr uint32_t kBars = 3 + 2 * NR + 2 * ND + 6 * NS;
  static constexpr uint32_t kTotal = oBar + kBars * 8 + 16;
  static_assert(kTotal <= 227u * 1024u && kSlot % 1024 == 0, "shared memory window; 1024-byte aligned slots");
};

template <int HPG>
__global__ void __launch_bounds__(KtSmem<HPG>::kThreads, 1)
    kl_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmIK,
                 const KlTcArgs p) {
  using SM = KtSmem<HPG>;
  constexpr int E = SM::E, NS = SM::NS, NR = SM::NR, ND = SM::ND;
  constexpr uint32_t kSet = 128 + E;  // TMEM columns per set: S^T, then I^T
  constexpr int EG = kKtEG;    // entries per reduce-scatter group
  constexpr int NG = E / EG;
  constexpr int RG = EG * HPG;  // tile rows (S^T columns) per group
  static_assert(RG % 32 == 0 && E % EG == 0, "entry groups");
  constexpr uint32_t kIdS = kt_idesc(128, 128), kIdI = kt_idesc(128, E);
  extern __shared__ __align__(1024) uint8_t kt_smem[];
  if (tc::smem_u32(kt_smem) & 1023u) {  // the swizzled operands need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, MSA_ERR_CUDA);
    return;
  }
  uint8_t* k_buf = kt_smem + SM::oK;
  uint8_t* ik_buf = kt_smem + SM::oIK;
  uint8_t* ring = kt_smem + SM::oRing;
  float* lse_s = reinterpret_cast<float*>(kt_smem + SM::oLse);
  int* lim_s = reinterpret_cast<int*>(kt_smem + SM::oLim);
  float4* red = reinterpret_cast<float4*>(kt_smem + SM::oRed);
  uint64_t* bars = reinterpret_cast<uint64_t*>(kt_smem + SM::oBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* done_bar = bars + 2;
  uint64_t* q_full = bars + 3;               // [NR] row slots: the rows have landed
  uint64_t* q_empty = q_full + NR;           // [NR]: the MMA has read them
  uint64_t* rd_full = q_empty + NR;          // [ND] row-data slots: written
  uint64_t* rd_empty = rd_full + ND;         // [ND]: the epilogue has read them
  uint64_t* s_full = rd_empty + ND;          // [NS] TMEM sets
  uint64_t* tm_empty = s_full + NS;          // [NS]
  uint64_t* red_full = tm_empty + NS;        // [NS][2]: a warpgroup's four warps' sums of a group are in red
  uint64_t* red_empty = red_full + 2 * NS;   // [NS][2]: its warp 0 has merged them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + SM::kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kGather0 = 4 * NS, kTmaWarp = 4 * NS + 2, kMmaWarp = 4 * NS + 3;
  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    tc::mbar_init(kv_empty, 1);
    for (int r = 0; r < NR; ++r) {
      tc::mbar_init(&q_full[r], 2);
      tc::mbar_init(&q_empty[r], 1);
    }
    for (int r = 0; r < ND; ++r) {
      tc::mbar_init(&rd_full[r], 2);
      tc::mbar_init(&rd_empty[r], 4);
    }
    for (int r = 0; r < NS; ++r) {
      tc::mbar_init(&s_full[r], 1);
      tc::mbar_init(&tm_empty[r], 4);
    }
    for (int r = 0; r < 2 * NS; ++r) {
      tc::mbar_init(&red_full[r], 4);
      tc::mbar_init(&red_empty[r], 1);
    }
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
    tc::tma_prefetch(&tmIK);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int z0 = p.cta_start[blockIdx.x], z1 = p.cta_start[blockIdx.x + 1];
  const int n = z1 - z0;
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(p.status, MSA_ERR_TIMEOUT);
  };
  const SeqView sv = seq_view(p.q_offset, p.kv_len, p.b, p.Nq, p.Nk, false);

  if (warp < kGather0) {
    // ------------------------------ epilogue ------------------------------
    const int wg = warp >> 2;  // takes tiles z with z % NS == wg (TMEM set wg, row-data slot z % ND)
    const int quarter = warp & 3;
    const int key = quarter * 32 + lane;  // TMEM lane = key of the block
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const float sl2 = p.scale * kKtLog2e;
    int gc = 0;  // this warpgroup's groups merged so far (red buffer gc & 1)
    bool alive = true;
    int4 tl_n = wg < n ? p.tiles[z0 + wg] : make_int4(0, 0, 0, 0);
    for (int z = wg; z < n && alive; z += NS) {
      const int set = wg, ph = (z / NS) & 1;
      const int slot = z % ND, phr = (z / ND) & 1;
      const int4 tl = tl_n;
      if (z + NS < n) tl_n = p.tiles[z0 + z + NS];  // in flight during this tile
      if (!tc::mbar_wait(&s_full[set], ph, abort_flag) ||
          !tc::mbar_wait(&rd_full[slot], phr, abort_flag)) {  // the tile's row data (already complete)
        fail();
        break;
      }
      tc::fence_after_sync();
      const float* lse_r = lse_s + slot * kKtRows;
      const int* lim = lim_s + slot * E;
      const uint32_t s_col = tmem + lane_base + uint32_t(set) * kSet;
#pragma unroll 1
      for (int eg = 0; eg < NG; ++eg) {
        float va[EG], vb[EG], vm[EG], vl[EG];
        // index scores of the group's entries
        uint32_t sc[EG];
        tc::tmem_ld_32x32b_x16(s_col + 128u + uint32_t(eg * EG), sc);
        tc::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < EG; ++x) {
          va[x] = vb[x] = 0.f;
          vm[x] = -INFINITY;
          vl[x] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < RG / 32; ++c) {
          uint32_t sv32[32];
          tc::tmem_ld_32x32b_x32(s_col + uint32_t(eg * RG + c * 32), sv32);
          // the chunk's 32 rows of lse * log2(e) and its 32 / HPG entries' visibility
          // limits in vector loads (the same words for every thread: broadcast)
          constexpr int EC = 32 / HPG;
          float l32[32];
          int lm[EC];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 v = reinterpret_cast<const float4*>(lse_r + eg * RG + c * 32)[q4];
            l32[4 * q4] = v.x; l32[4 * q4 + 1] = v.y; l32[4 * q4 + 2] = v.z; l32[4 * q4 + 3] = v.w;
          }
#pragma unroll
          for (int q4 = 0; q4 < EC / 4; ++q4) {
            const int4 v = reinterpret_cast<const int4*>(lim + eg * EG + c * EC)[q4];
            lm[4 * q4] = v.x; lm[4 * q4 + 1] = v.y; lm[4 * q4 + 2] = v.z; lm[4 * q4 + 3] = v.w;
          }
          tc::tmem_ld_wait();
#pragma unroll
          for (int ee = 0; ee < EC; ++ee) {
            const int el = c * EC + ee;  // entry within the group
            const bool vis = key <= lm[ee];
            float ps = 0.f;
#pragma unroll
            for (int h = 0; h < HPG; ++h) {
              const int col = ee * HPG + h;
              ps += kt_ex2(fmaf(__uint_as_float(sv32[col]), sl2, -l32[col]));
            }
            const float pb = vis ? ps * (1.f / HPG) : 0.f;
            const float s = __uint_as_float(sc[el]);
            va[el] = pb > 0.f ? pb * (kt_lg2(pb) * kKtLn2) : 0.f;
            vb[el] = pb * s;
            vm[el] = vis ? s : -INFINITY;
            vl[el] = vis ? 1.f : 0.f;
          }
        }
        if (eg + 1 == NG) {  // every TMEM column of this tile is in registers
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            tc::mbar_arrive(&tm_empty[set]);
            tc::mbar_arrive(&rd_empty[slot]);  // its row data has been read too
          }
        }
        kt_rs_sum(va, lane);
        kt_rs_sum(vb, lane);
        // the index scores' log-sum-exp over this warp's 32 keys: the warp
        // maximum per entry (one redux each, the same value in every lane),
        // then a plain sum of exp(s - max); warp 0 merges the warps' pairs
        float mw = -INFINITY;
#pragma unroll
        for (int x = 0; x < EG; ++x) {
          const float m = tc::warp_max_f32(vm[x]);
          vl[x] = vl[x] > 0.f ? kt_ex2((vm[x] - m) * kKtLog2e) : 0.f;
          if ((lane & (EG - 1)) == x) mw = m;  // lane l ends with entry l mod 16
        }
        kt_rs_sum(vl, lane);
        vm[0] = mw;
        // the four warps' sums meet in red[buf]; warp 0 merges them (bounded waits, no bar.sync)
        const int buf = gc & 1, rb = wg * 2 + buf;
        if (!tc::mbar_wait(&red_empty[rb], ((gc >> 1) & 1) ^ 1, abort_flag)) {
          fail();
          alive = false;
          break;
        }
        if (lane < EG) red[(rb * 4 + quarter) * EG + lane] = make_float4(va[0], vb[0], vm[0], vl[0]);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&red_full[rb]);
        if (quarter == 0) {
          if (!tc::mbar_wait(&red_full[rb], (gc >> 1) & 1, abort_flag)) {
            fail();
            alive = false;
            break;
          }
          if (lane < EG) {
            float4 a = red[(rb * 4) * EG + lane];
#pragma unroll
            for (int w = 1; w < 4; ++w) {
              const float4 o = red[(rb * 4 + w) * EG + lane];
              a.x += o.x;
              a.y += o.y;
              kt_lse_merge(a.z, a.w, o.z, o.w);
            }
            const int e = eg * EG + lane;
            if (e < tl.z) p.part[int64_t(z0 + z) * E + e] = a;
          }
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&red_empty[rb]);
        }
        ++gc;
      }
    }
  } else if (warp < kTmaWarp) {
    // -------------- q rows, index-query rows and row data (gather) --------------
    const int gw = warp - kGather0;  // rows [64 gw, 64 gw + 64), entries [E/2 gw, E/2 (gw + 1))
    constexpr int kCpr = kKtD / 8, kRpi = 32 / kCpr;         // q: 16 chunks per row, 2 rows per instruction
    constexpr int kCprI = kKtDI / 8, kRpiI = 32 / kCprI;    // iq: 8 chunks per row, 4 rows per instruction
    const int chunk = lane % kCpr, sub = lane / kCpr;
    const int chunkI = lane % kCprI, subI = lane / kCprI;
    constexpr int kItI = (E / 2) / kRpiI;  // index-query copy rounds per tile
    // tile records and the entries this lane needs, fetched one tile ahead
    int4 tl_n = make_int4(0, 0, 0, 0);
    int ent2_n[2], entI_n[kItI], entL_n;
    auto fetch = [&](int z) {
      tl_n = p.tiles[z0 + z];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int e = (gw * 64 + x * 32 + lane) / HPG;
        ent2_n[x] = e < tl_n.z ? p.entries[tl_n.y + e] : -1;
      }
#pragma unroll
      for (int it = 0; it < kItI; ++it) {
        const int e = gw * (E / 2) + it * kRpiI + subI;
        entI_n[it] = e < tl_n.z ? p.entries[tl_n.y + e] : -1;
      }
      const int eL = gw * (E / 2) + lane;
      entL_n = (lane < E / 2 && eL < tl_n.z) ? p.entries[tl_n.y + eL] : -1;
    };
    // tile z's row slot is free once the MMA of tile z - NR has read it, its
    // row-data slot once the epilogue of tile z - ND has
    auto slot_free = [&](int zz) {
      return tc::mbar_wait(&q_empty[zz % NR], ((zz / NR) & 1) ^ 1, abort_flag) &&
             tc::mbar_wait(&rd_empty[zz % ND], ((zz / ND) & 1) ^ 1, abort_flag);
    };
    auto issue = [&](int z) {  // tile z's copies and row data (its records were fetched one tile ahead)
      const int slot = z % NR, dslot = z % ND;
      const int4 tl = tl_n;
      int ent2[2], entI[kItI];
#pragma unroll
      for (int x = 0; x < 2; ++x) ent2[x] = ent2_n[x];
#pragma unroll
      for (int it = 0; it < kItI; ++it) entI[it] = entI_n[it];
      const int entL = entL_n;
      if (z + 1 < n) fetch(z + 1);
      const int g = tl.x / p.nblk, t = tl.x % p.nblk;
      const uint32_t qs = tc::smem_u32(ring + slot * SM::kSlot), iqs = qs + SM::kQ;
      // this lane's two rows of the warp's 64 (row data)
      int64_t qrow2[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int r = gw * 64 + x * 32 + lane;
        const int il = ent2[x] >= 0 ? (ent2[x] >> 6) : 0;
        qrow2[x] = (int64_t(p.b) * p.Nq + p.c0 + il) * p.Hq + g * HPG + (r % HPG);
      }
#pragma unroll 4
      for (int it = 0; it < 64 / kRpi; ++it) {
        const int rr = it * kRpi + sub;  // row within this warp's 64
        const int row = gw * 64 + rr;
        const int src_lane = rr & 31, x = rr >> 5;
        const int ent_r = __shfl_sync(0xffffffffu, x ? ent2[1] : ent2[0], src_lane);
        const int64_t qr = __shfl_sync(0xffffffffu, x ? qrow2[1] : qrow2[0], src_lane);
        const uint32_t hf = uint32_t(chunk) >> 3, cc = uint32_t(chunk) & 7u;
        kt_cp16(qs + hf * SM::kHalf + row * 128 + ((cc ^ uint32_t(row & 7)) << 4), p.q + qr * kKtD + chunk * 8,
                ent_r >= 0);
      }
      // index-query rows of entries [E/2 gw, E/2 gw + E/2)
#pragma unroll
      for (int it = 0; it < kItI; ++it) {
        const int e = gw * (E / 2) + it * kRpiI + subI;
        const int ent = entI[it];
        const int il = ent >= 0 ? (ent >> 6) : 0;
        const __nv_bfloat16* src = p.iq + ((int64_t(p.b) * p.Nq + p.c0 + il) * p.G + g) * kKtDI + chunkI * 8;
        kt_cp16(iqs + e * 128 + ((uint32_t(chunkI) ^ uint32_t(e & 7)) << 4), src, ent >= 0);
      }
      // lse of the two rows by 4-byte copies (zero for padding rows)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int r = gw * 64 + x * 32 + lane;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(tc::smem_u32(lse_s + dslot * kKtRows + r)),
                     "l"(p.lse + qrow2[x]), "r"(ent2[x] >= 0 ? 4u : 0u)
                     : "memory");
      }
      cp_async_commit_kt();
      if (lane < E / 2) {
        int lm = -1;
        if (entL >= 0 && sv.ok) lm = min(min(sv.q0 + p.c0 + (entL >> 6), sv.L - 1) - t * kKtBs, kKtBs - 1);
        lim_s[dslot * E + gw * (E / 2) + lane] = lm;
      }
    };
    auto finish = [&](int z) {  // tile z's copies have landed: scale its lse, publish both slots
      const int dslot = z % ND;
#pragma unroll
      for (int x = 0; x < 2; ++x) lse_s[dslot * kKtRows + gw * 64 + x * 32 + lane] *= kKtLog2e;  // log2 units
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&q_full[z % NR]);
        tc::mbar_arrive(&rd_full[dslot]);
      }
    };
    // Two tiles in flight: tile z + 1's copies go out before tile z's are
    // waited for. Its slots free when the MMA of tile z + 1 - NR and the
    // epilogue of tile z + 1 - ND are done, both of which precede tile z's
    // MMA, so publishing tile z after that wait delays no MMA.
    bool ok = true;
    if (n > 0) {
      fetch(0);
      ok = slot_free(0);
      if (ok)
        issue(0);
      else
        fail();
    }
    for (int z = 0; ok && z < n; ++z) {
      if (z + 1 < n) {
        if (!slot_free(z + 1)) {
          fail();
          break;
        }
        issue(z + 1);
        cp_async_wait_but_one_kt();  // tile z's group
      } else {
        cp_async_wait_all_kt();
      }
      finish(z);
    }
    cp_async_wait_all_kt();
  } else if (warp == kTmaWarp) {
    // ------------------------------ K / IK producer ------------------------------
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
        tc::mbar_arrive_expect_tx(kv_full, SM::kK + SM::kIK);
#pragma unroll
        for (int h = 0; h < kKtD / 64; ++h)
          tc::tma_load_4d(k_buf + h * SM::kHalf, &tmK, kv_full, h * 64, g, t * kKtBs, p.b);
        tc::tma_load_3d(ik_buf, &tmIK, kv_full, 0, t * kKtBs, p.b);
        ++loads;
      }
      int zero = 0;
      if (loads > 0) tc::mbar_wait(kv_full, (loads - 1) & 1, &zero);  // drain the last copy
    }
  } else {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      int kv_uses = 0, prev_bin = -1;
      const uint32_t ka = tc::smem_u32(k_buf), ika = tc::smem_u32(ik_buf);
      // descriptors from 32-bit low words with one constant high word (8-row
      // groups 1024 B apart, 128B swizzle): one add per operand and MMA
      constexpr uint32_t kDescHi = tc::smem_desc_hi(1024, 2);
      const uint32_t ka16 = tc::smem_desc_lo(ka, 16), ika16 = tc::smem_desc_lo(ika, 16);
      int bin_n = n > 0 ? p.tiles[z0].x : -1;
      for (int z = 0; z < n; ++z) {
        const int set = z % NS, ph = (z / NS) & 1;
        const int slot = z % NR, phr = (z / NR) & 1;
        const int bin = bin_n;
        bin_n = z + 1 < n ? p.tiles[z0 + z + 1].x : -1;  // one tile ahead
        const bool first = bin != prev_bin;
        const bool last = bin_n != bin;
        prev_bin = bin;
        if (first) {
          if (!tc::mbar_wait(kv_full, kv_uses & 1, abort_flag)) {
            fail();
            break;
          }
          ++kv_uses;
        }
        if (!tc::mbar_wait(&q_full[slot], phr, abort_flag) || !tc::mbar_wait(&tm_empty[set], ph ^ 1, abort_flag)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const uint32_t qa = tc::smem_u32(ring + slot * SM::kSlot), iqa = qa + SM::kQ;
        const uint32_t qa16 = tc::smem_desc_lo(qa, 16), iqa16 = tc::smem_desc_lo(iqa, 16);
        const uint32_t d_s = tmem + uint32_t(set) * kSet;
#pragma unroll
        for (int kk = 0; kk < kKtD / 16; ++kk) {  // S^T = K q^T
          const uint32_t off = ((kk >> 2) * SM::kHalf + (kk & 3) * 32) >> 4;
          tc::mma_f16_ss_lo<kDescHi>(d_s, ka16 + off, qa16 + off, kIdS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kKtDI / 16; ++kk) {  // I^T = IK iq^T
          const uint32_t off = (kk * 32) >> 4;
          tc::mma_f16_ss_lo<kDescHi>(d_s + 128u, ika16 + off, iqa16 + off, kIdI, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&s_full[set]);
        tc::mma_commit(&q_empty[slot]);
        if (last) tc::mma_commit(kv_empty);
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

}  // namespace

bool kl_tc_supported(int d, int di, int Bs, int hpg) {
  return d == kKtD && di == kKtDI && Bs == kKtBs && (hpg == 2 || hpg == 4 || hpg == 8);
}

cudaError_t launch_kl_tile_tc(const KlTcArgs& a, const void* k, const void* ik, int B, int Nk, int Hkv, int hpg,
                              int grid, cudaStream_t stream) {
  CUtensorMap tmK, tmIK;
  {
    const uint64_t dims[4] = {uint64_t(kKtD), uint64_t(Hkv), uint64_t(Nk), uint64_t(B)};
    const uint64_t strides[3] = {uint64_t(kKtD) * 2, uint64_t(Hkv) * kKtD * 2, uint64_t(Nk) * Hkv * kKtD * 2};
    const uint32_t box[4] = {64, 1, uint32_t(kKtBs), 1};
    if (!make_tmap_bf16(&tmK, k, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {uint64_t(kKtDI), uint64_t(Nk), uint64_t(B)};
    const uint64_t strides[2] = {uint64_t(kKtDI) * 2, uint64_t(Nk) * kKtDI * 2};
    const uint32_t box[3] = {64, uint32_t(kKtBs), 1};
    if (!make_tmap_bf16(&tmIK, ik, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  cudaError_t e;
#define MSA_KT(H_)                                                                                               \
  do {                                                                                                           \
    auto kern = kl_tc_kernel<H_>;                                                                                \
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(KtSmem<H_>::kTotal))) != \
        cudaSuccess)                                                                                             \
      return e;                                                                                                  \
    kern<<<grid, KtSmem<H_>::kThreads, KtSmem<H_>::kTotal, stream>>>(tmK, tmIK, a);                              \
  } while (0)
  if (hpg == 2)
    MSA_KT(2);
  else if (hpg == 4)
    MSA_KT(4);
  else
    MSA_KT(8);
#undef MSA_KT
  return cudaGetLastError();
}

}  // namespace msa
