// Index Branch, fused tensor-core kernel (bf16, sm_103a):
//   index scores  S = iq . ik^T on tcgen05 (TMA-fed shared-memory operands,
//                 fp32 accumulators in TMEM),
//   block max     pooled straight out of TMEM in the epilogue,
//   top-K         exact top-(K-1) per row over the candidate blocks t < loc,
//                 then the local block appended (with the sequence start
//                 forced as well: top-(K-2) over 1 <= t < loc, plus block 0).
// For K - 1 <= 15 the top-K is a running list in registers inside the kernel,
// so neither the token-score matrix nor the block-max table reaches HBM. For
// larger K (many blocks per row at small block sizes) the kernel writes the
// candidate block maxima of a chunk of rows to a workspace table, and
// index_topk_table selects from it, one warp per row; the token scores still
// never leave the chip.
// (hyper.ai summary of paper 2606.13392, section "方法": per GQA group, dot-
//  product scores of the index query against every visible key, Block Max
//  Pooling, Top-K blocks, the block holding the query always included;
//  quant_prune_distill post 751, "Метод": one index query head per group, one
//  index key head for the layer.)
//
// Layout: the G index-query heads of a token are stacked along M, so one GEMM
// of (Nq*G) x Nk per sequence serves every group (the index key is shared by
// all groups). A work unit is 256 stacked rows (two 128-row MMA tiles that
// share each key tile, which halves the key traffic per flop); it sweeps key
// tiles of 256 keys over the blocks before its local block. Units are handed
// out in a static serpentine order, longest first, over a persistent grid of
// one CTA per SM.
//
// Warp roles (384 threads): warps 0-7 epilogue (warpgroup m reads TMEM lanes
// of MMA tile m), warp 8 TMA producer, warp 9 TMEM owner + MMA issuer.
// Pipelines: key tiles in an S-stage shared-memory ring; index-query tiles in
// nA buffers; two TMEM accumulators of 256 columns (one per 128-row MMA tile,
// 512 columns), drained by their warpgroups in turn.
// Every wait is bounded; on expiry the kernel records MSA_ERR_TIMEOUT, stops
// issuing work, drains its copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "msa_internal.cuh"
#include "tc_utils.cuh"

namespace msa {
namespace {

constexpr int kUnitRows = 256;  // stacked (token, group) rows per work unit
constexpr int kTileN = 256;     // keys per key tile (N of each MMA)
constexpr int kThreads = 384;
constexpr int kEpiWarps = 8;       // warps 0-7 (warpgroups 0 and 1)
constexpr int kProducerWarp = 8;   // warpgroup 2: TMA producer, MMA issuer, two idle warps
constexpr int kMmaWarp = 9;
constexpr int kLaunchRegs = 168;   // registers per thread at launch (checked on the host)
constexpr int kProdRegs = 72, kEpiRegs = 216;
static_assert(128 * kProdRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kRegList = 15;       // candidates kept in registers when K - 1 <= 15

struct Unit {
  int gu, b, row0, nrows, q0, nt;
  bool ok;
};

// u-th unit of the launch's range [unit_lo, unit_lo + nunits) of the flat
// (sequence, row block) units
__device__ __forceinline__ Unit get_unit(int u, int unit_lo, int nunits, int nrb, int NqG, int G, int Nq, int Nk,
                                         int Bs, int K, int fs, const int32_t* q_offset, const int32_t* kv_len) {
  Unit U;
  const int gu = unit_lo + nunits - 1 - u;  // longest units (latest rows) first
  U.gu = gu;
  U.b = gu / nrb;
  const int rb = gu % nrb;
  U.row0 = rb * kUnitRows;
  U.nrows = min(kUnitRows, NqG - U.row0);
  const SeqView sv = seq_view(q_offset, kv_len, U.b, Nq, Nk, false);
  U.ok = sv.ok;
  U.q0 = sv.q0;
  const int maxloc = sv.ok ? (sv.q0 + (U.row0 + U.nrows - 1) / G) / Bs : 0;
  // key tiles are needed only if some row has more visible blocks than K and
  // at least one block is ranked (K - 1 - fs of them)
  U.nt = (sv.ok && K - fs > 1 && maxloc + 1 > K) ? (maxloc * Bs + kTileN - 1) / kTileN : 0;
  return U;
}

// serpentine static schedule over the persistent grid
__device__ __forceinline__ int unit_at(int round, int cta, int ncta) {
  return round * ncta + ((round & 1) ? (ncta - 1 - cta) : cta);
}

template <int BS>
__device__ __forceinline__ float block_max(const uint32_t* v) {
  // four independent chains of 3-input max for instruction-level parallelism
  static_assert(BS % 8 == 0, "block size must be a multiple of 8");
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < BS; c += 8) {
    m0 = tc::fmax3(m0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
    m1 = tc::fmax3(m1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
    m2 = tc::fmax3(m2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
    m3 = tc::fmax3(m3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// Table rows are written by TMA tensor stores from shared memory where a
// tile's blocks of one row fill at least 16 bytes (blocks of 32 / 64 keys):
// each epilogue warp stages its 32 rows x (256 / Bs) maxima, double-buffered.
template <int BS>
constexpr bool table_tma() { return (kTileN / BS) * 4 >= 16; }
template <int BS>
constexpr size_t table_stage_bytes() { return table_tma<BS>() ? size_t(kEpiWarps) * 2 * 32 * (kTileN / BS) * 4 : 0; }

// REG: top-K in a register list (K - 1 <= 15); TABLE: the candidate block
// maxima of rows of units [unit_lo, unit_lo + nunits) go to table[row - first
// row of unit_lo][t] (row stride tstride floats; tmT maps that chunk table),
// and no selection is written.
template <int DI, int BS, bool REG, bool TABLE>
__global__ void __launch_bounds__(kThreads, 1)
    index_fused_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmT, const int32_t* __restrict__ q_offset,
                          const int32_t* __restrict__ kv_len, int Nq, int Nk, int G, int K, int fs, int nA, int S,
                          int unit_lo, int nunits, int32_t* __restrict__ sel, float* __restrict__ table, int tstride,
                          uint32_t* status) {
  static_assert(REG != TABLE, "one top-K form");
  constexpr bool kTmaTable = TABLE && table_tma<BS>();
  constexpr uint32_t kABytes = kUnitRows * DI * 2;   // one unit of index queries
  constexpr uint32_t kATile = 128 * DI * 2;          // one 128-row MMA tile
  constexpr uint32_t kBBytes = kTileN * DI * 2;      // one key tile
  constexpr uint32_t kSbo = DI == 64 ? 1024 : 512;   // 8-row swizzle atom
  constexpr uint32_t kSwz = DI == 64 ? 2 : 4;        // 128B / 64B swizzle
  constexpr int kKSteps = DI / 16;
  constexpr int kChunk = 128;  // TMEM columns read per epilogue step (one load round)
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(128, kTileN);
  constexpr uint32_t kDescHi = tc::smem_desc_hi(kSbo, kSwz);  // the descriptors' constant high word

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* a_buf = smem;                                       // nA x kABytes
  uint8_t* b_buf = a_buf + size_t(nA) * kABytes;               // S x kBBytes
  const int Kl = K - 1;  // list slots per row (the host sizes shared memory for K - 1)
  const int Kc = K - 1 - fs;  // blocks ranked per row: fs = 1 keeps block 0 outright, like the local block
  float* stage = reinterpret_cast<float*>(b_buf + size_t(S) * kBBytes);  // [8 warps][2][32 rows][256 / BS]
  uint64_t* lists = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(stage) + (TABLE ? table_stage_bytes<BS>() : 0));  // [Kl][256]
  uint64_t* bars = lists + size_t(TABLE ? 0 : (Kl > 0 ? Kl : 1)) * kUnitRows;
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* a_full = empty + S;
  uint64_t* a_empty = a_full + nA;
  uint64_t* acc_full = a_empty + nA;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NqG = Nq * G;
  const int nrb = (NqG + kUnitRows - 1) / kUnitRows;
  const int ncta = gridDim.x, cta = blockIdx.x;
  const int rounds = (nunits + ncta - 1) / ncta;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int x = 0; x < nA; ++x) {
      tc::mbar_init(&a_full[x], 1);
      tc::mbar_init(&a_empty[x], 1);
    }
    for (int m = 0; m < 2; ++m) {  // one accumulator per MMA tile of the unit
      tc::mbar_init(&acc_full[m], 1);
      tc::mbar_init(&acc_empty[m], kEpiWarps / 2);
    }
    tc::mbar_init(done_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tc::tma_prefetch(&tmA);
    tc::tma_prefetch(&tmB);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&](void) {
    *abort_flag = 1;
    set_status(status, MSA_ERR_TIMEOUT);
  };

  // Each register re-allocation sits at the top of its warpgroups' branch so
  // that the compiler budgets each branch with its own register count.
  if (warp >= kEpiWarps) {
  tc::regs_dec<kProdRegs>();
  if (warp == kProducerWarp) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int kB = 0, jA = 0;
      bool alive = true;
      for (int r = 0; r < rounds && alive; ++r) {
        const int u = unit_at(r, cta, ncta);
        if (u >= nunits) continue;
        const Unit U = get_unit(u, unit_lo, nunits, nrb, NqG, G, Nq, Nk, BS, K, fs, q_offset, kv_len);
        if (U.nt == 0) continue;
        const int x = jA % nA;
        if (!tc::mbar_wait(&a_empty[x], ((jA / nA) & 1) ^ 1, abort_flag)) {
          fail();
          break;
        }
        tc::mbar_arrive_expect_tx(&a_full[x], kABytes);
        tc::tma_load_3d(a_buf + size_t(x) * kABytes, &tmA, &a_full[x], 0, U.row0, U.b);
        ++jA;
        for (int n = 0; n < U.nt; ++n, ++kB) {
          const int s = kB % S;
          if (!tc::mbar_wait(&empty[s], ((kB / S) & 1) ^ 1, abort_flag)) {
            fail();
            alive = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&full[s], kBBytes);
          tc::tma_load_3d(b_buf + size_t(s) * kBBytes, &tmB, &full[s], 0, n * kTileN, U.b);
        }
      }
      // drain: every issued copy must land before the CTA exits
      int zero = 0;
      for (int s = 0; s < S && s < kB; ++s) {
        const int last = kB - 1 - ((kB - 1 - s) % S);  // last tile index that used stage s
        tc::mbar_wait(&full[s], (last / S) & 1, &zero);
      }
      for (int x = 0; x < nA && x < jA; ++x) {
        const int last = jA - 1 - ((jA - 1 - x) % nA);
        tc::mbar_wait(&a_full[x], (last / nA) & 1, &zero);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      int kB = 0, jA = 0, kAcc = 0;
      bool alive = true;
      for (int r = 0; r < rounds && alive; ++r) {
        const int u = unit_at(r, cta, ncta);
        if (u >= nunits) continue;
        const Unit U = get_unit(u, unit_lo, nunits, nrb, NqG, G, Nq, Nk, BS, K, fs, q_offset, kv_len);
        if (U.nt == 0) continue;
        const int x = jA % nA;
        if (!tc::mbar_wait(&a_full[x], (jA / nA) & 1, abort_flag)) {
          fail();
          break;
        }
        ++jA;
        // descriptor low words (start address, leading offset): one add per operand and MMA
        const uint32_t a_lo = tc::smem_desc_lo(tc::smem_u32(a_buf + size_t(x) * kABytes), 16);
        for (int n = 0; n < U.nt; ++n, ++kB, ++kAcc) {
          const int s = kB % S;
          if (!tc::mbar_wait(&full[s], (kB / S) & 1, abort_flag)) {
            fail();
            alive = false;
            break;
          }
          const uint32_t b_lo = tc::smem_desc_lo(tc::smem_u32(b_buf + size_t(s) * kBBytes), 16);
          // ping-pong: tile m's accumulator is drained by warpgroup m while the
          // tensor core works on the other tile
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            if (!tc::mbar_wait(&acc_empty[m], (kAcc & 1) ^ 1, abort_flag)) {
              fail();
              alive = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t d = tmem + uint32_t(m * kTileN);
#pragma unroll
            for (int kk = 0; kk < kKSteps; ++kk)
              tc::mma_f16_ss_lo<kDescHi>(d, a_lo + ((m * kATile + kk * 32) >> 4), b_lo + ((kk * 32) >> 4), kIdesc,
                                         kk > 0 ? 1u : 0u);
            tc::mma_commit(&acc_full[m]);
          }
          if (!alive) break;
          tc::mma_commit(&empty[s]);
          if (n == U.nt - 1) tc::mma_commit(&a_empty[x]);
        }
      }
      // all issued MMAs complete before TMEM is released
      int zero = 0;
      tc::mma_commit(done_bar);
      tc::mbar_wait(done_bar, 0, &zero);
    }
  }  // warps 10-11: idle
  } else {
    tc::regs_inc<kEpiRegs>();
    // -------------------------------- epilogue --------------------------------
    const int m = warp >> 2, quarter = warp & 3;
    const int urow = m * 128 + quarter * 32 + lane;  // row within the unit = TMEM lane of tile m
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    int kAcc = 0;
    bool alive = true;
    uint64_t* my_list = lists + urow;  // entry k at my_list[k * 256]
    int nstore = 0;  // this warp's staged table stores so far (buffer = parity)
    for (int r = 0; r < rounds && alive; ++r) {
      const int u = unit_at(r, cta, ncta);
      if (u >= nunits) continue;
      const Unit U = get_unit(u, unit_lo, nunits, nrb, NqG, G, Nq, Nk, BS, K, fs, q_offset, kv_len);
      const bool active = urow < U.nrows;
      const int row = U.row0 + urow;
      const int pos = U.q0 + row / G;
      const int loc = pos / BS;
      const bool dense = loc + 1 <= K;
      const bool cand_row = active && U.ok && !dense;
      // REG (K - 1 <= 15): the best candidates so far in registers, sorted
      // descending and padded with key 0 (below every real key); an insertion
      // is a branch-free compare-and-shift over the list, taken by the whole
      // warp whenever one of its rows accepts (the others' lists stay as
      // they are: their key is below every slot).
      uint64_t L[kRegList];
      int ncand = 0;
#pragma unroll
      for (int k = 0; k < kRegList; ++k) L[k] = 0;
      // Blocks are offered in ascending t, so a candidate ranks above a kept
      // key exactly when its score word (the key's high 32 bits) is larger:
      // on equal scores the earlier (lower) block ranks higher. The compares
      // take 32-bit words; invalid candidates (key 0) rank above nothing.
      auto offer_reg = [&](int t, float mx) {
        const bool valid = cand_row && unsigned(t - fs) < unsigned(loc - fs);  // fs <= t < loc
        const uint64_t x = valid ? rank_key(mx, t) : 0ull;
        const uint32_t xh = uint32_t(x >> 32);
        ncand += valid ? 1 : 0;
        if (__any_sync(0xffffffffu, xh > uint32_t(L[kRegList - 1] >> 32))) {
          bool c[kRegList];  // the candidate ranks above L[k]
#pragma unroll
          for (int k = 0; k < kRegList; ++k) c[k] = xh > uint32_t(L[k] >> 32);
#pragma unroll
          for (int k = kRegList - 1; k > 0; --k) L[k] = c[k - 1] ? L[k - 1] : (c[k] ? x : L[k]);
          L[0] = c[0] ? x : L[0];
        }
      };
      for (int n = 0; n < U.nt; ++n, ++kAcc) {
        if (!tc::mbar_wait(&acc_full[m], kAcc & 1, abort_flag)) {
          fail();
          alive = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t taddr = tmem + lane_base + uint32_t(m * kTileN);
        // block maxima of the whole tile first (the accumulator is released
        // as soon as its last columns are in registers), offers afterwards
        float bm[kTileN / BS];
        if constexpr (TABLE || BS == 128) {
          // each 32-column load returns the maximum of its columns as well
#pragma unroll
          for (int c = 0; c < kTileN / kChunk; ++c) {
            float m32[kChunk / 32];
#pragma unroll
            for (int q = 0; q < kChunk / 32; ++q) {
              uint32_t v[32];  // the values themselves are not needed
              m32[q] = tc::tmem_ld_max_32x32b_x32(taddr + c * kChunk + q * 32, v);
            }
            tc::tmem_ld_wait();
            if (c == kTileN / kChunk - 1) {  // the whole accumulator has been read: release it
              tc::fence_before_sync();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&acc_empty[m]);
            }
#pragma unroll
            for (int bi = 0; bi < kChunk / BS; ++bi) {
              float mx = m32[bi * (BS / 32)];
#pragma unroll
              for (int q = 1; q < BS / 32; ++q) mx = fmaxf(mx, m32[bi * (BS / 32) + q]);
              bm[c * (kChunk / BS) + bi] = mx;
            }
          }
        } else {
          // many block maxima per tile next to the register list: loaded
          // values reduced by 3-input max chains keep the registers in bounds
#pragma unroll
          for (int c = 0; c < kTileN / kChunk; ++c) {
            uint32_t v[kChunk];
#pragma unroll
            for (int q = 0; q < kChunk / 32; ++q) tc::tmem_ld_32x32b_x32(taddr + c * kChunk + q * 32, v + q * 32);
            tc::tmem_ld_wait();
            if (c == kTileN / kChunk - 1) {  // the whole accumulator is in registers: release it
              tc::fence_before_sync();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&acc_empty[m]);
            }
#pragma unroll
            for (int bi = 0; bi < kChunk / BS; ++bi) bm[c * (kChunk / BS) + bi] = block_max<BS>(v + bi * BS);
          }
        }
        if constexpr (TABLE) {
          // this tile's blocks t < loc, as one full-sector vector store per row
          // where the whole tile is visible
          constexpr int kPer = kTileN / BS;
          const int t0 = n * kPer;
          if constexpr (kTmaTable) {
            // all 32 rows of the warp (rows that rank nothing hold values no
            // one reads; columns past loc likewise, inside the padded row)
            float* buf = stage + size_t(warp * 2 + (nstore & 1)) * 32 * kPer;
            if (lane == 0) tc::bulk_wait_read_but_one();  // the store of two tiles ago has read this buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kPer; j += 4)
              *reinterpret_cast<float4*>(buf + lane * kPer + j) = make_float4(bm[j], bm[j + 1], bm[j + 2], bm[j + 3]);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tc::tma_store_2d(&tmT, buf, t0, (U.gu - unit_lo) * kUnitRows + m * 128 + quarter * 32);
              tc::bulk_commit();
            }
            ++nstore;
          } else if (cand_row) {
            float* dst = table + (int64_t(U.gu - unit_lo) * kUnitRows + urow) * tstride + t0;
            if (t0 + kPer <= loc) {
              if constexpr (kPer >= 4) {
#pragma unroll
                for (int j = 0; j < kPer; j += 4)
                  *reinterpret_cast<float4*>(dst + j) = make_float4(bm[j], bm[j + 1], bm[j + 2], bm[j + 3]);
              } else {
                *reinterpret_cast<float2*>(dst) = make_float2(bm[0], bm[1]);
              }
            } else {
#pragma unroll
              for (int j = 0; j < kPer; ++j)
                if (t0 + j < loc) dst[j] = bm[j];
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < kTileN / BS; ++j) offer_reg(n * (kTileN / BS) + j, bm[j]);
        }
      }
      if constexpr (TABLE) continue;  // the selection kernel writes this chunk's rows
      // the best min(candidates, Kc) keys go to the row's slots
      const int cnt = ncand < Kc ? ncand : Kc;
#pragma unroll
      for (int k = 0; k < kRegList; ++k)
        if (k < cnt) my_list[k * kUnitRows] = L[k];
      if (!alive || !active) continue;
      int32_t* out = sel + (int64_t(U.b) * NqG + row) * K;
      if (!U.ok) {
        for (int k = 0; k < K; ++k) out[k] = -1;
        if (urow == 0) set_status(status, MSA_ERR_BOUNDS);
      } else if (dense) {
        for (int k = 0; k < K; ++k) out[k] = k <= loc ? k : -1;
      } else {
        // candidates -> block ids, ascending (insertion sort in this row's slots)
        for (int k = 0; k < cnt; ++k) my_list[k * kUnitRows] = uint64_t(rank_key_block(my_list[k * kUnitRows]));
        for (int k = 1; k < cnt; ++k) {
          const uint64_t x = my_list[k * kUnitRows];
          int p = k;
          while (p > 0 && my_list[(p - 1) * kUnitRows] > x) {
            my_list[p * kUnitRows] = my_list[(p - 1) * kUnitRows];
            --p;
          }
          my_list[p * kUnitRows] = x;
        }
        // [0 if fs], the ranked blocks ascending, the local block, -1 padding
        if (fs) out[0] = 0;
        for (int k = fs; k < K; ++k)
          out[k] = k - fs < cnt ? int32_t(my_list[(k - fs) * kUnitRows]) : (k - fs == cnt ? loc : -1);
      }
    }
    // the staged table stores are complete before the shared memory goes away
    if constexpr (kTmaTable) {
      if (lane == 0) tc::bulk_wait_all();
      __syncwarp();
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// index_topk_table: the exact top-K of every row of a table chunk, one warp
// per (token, group) row (the same selection rule as the fused top-K: the
// K - 1 - fs best blocks fs <= t < loc by maximum, ties to the lower block,
// then ascending, the local block after them and block 0 first if fs).
//  1. Each lane keeps the NS largest of its candidates t = fs + lane + 32 j.
//     Among those 32 NS sample values, T = the largest one with at least
//     `need` sample values >= T: then at least `need` candidates are >= T, so
//     the need-th largest candidate v* is >= T, and only candidates >= T can
//     be chosen. (T is the sample's (32 NS - need + 1)-th smallest value:
//     found by repeated minimum extraction when that is one of the four
//     smallest, else by ranking the sample with shuffles.)
//  2. The candidates >= T are compacted in ascending t into the warp's list
//     (a second pass over the row, from L2).
//  3. v* by bisection over the list's order-preserving 32-bit values (two bits
//     per round, starting below the bits that T and the list maximum share;
//     the three counts of a round are summed as one packed word) until the
//     bucket holding v* has at most 32 values, which a warp bitonic sort
//     puts in order; then every value above v* and the lowest-t values equal
//     to v*, compacted in list order.
// The two passes compare floats (the order of the 32-bit values, with -0 and
// +0 equal); only listed candidates are converted. A list that overflows
// gives a tighter bound (the need-th largest of its kSelCap entries) and the
// compaction runs again; ties at the bound that make no progress bisect over
// the row itself.
// NS = 1 serves need <= 32, NS = 2 need <= 64.
// ---------------------------------------------------------------------------
constexpr int kSelWarps = 8;
constexpr int kSelCap = 256;  // list entries per warp
constexpr int kSelBatch = 8;  // row loads in flight per lane

__device__ __forceinline__ uint32_t cand_value(const float* __restrict__ M, int t) {
  const uint32_t v = ord_f32(__ldg(M + t));
  return v > 1u ? v : 1u;  // 0 is kept for "no candidate"
}
__device__ __forceinline__ float ord_inv(uint32_t u) {  // the float of an order-preserving value
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

template <int NS>
__global__ void __launch_bounds__(kSelWarps * 32) index_topk_table_kernel(
    const float* __restrict__ table, int tstride, int unit_lo, int nrows, int nrb, int NqG, int G, int Nq, int Nk,
    int Bs, int K, int fs, const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len,
    int32_t* __restrict__ sel, uint32_t* status) {
  __shared__ uint32_t list_v[kSelWarps][kSelCap];
  __shared__ int list_t[kSelWarps][kSelCap];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const int r = blockIdx.x * kSelWarps + warp;  // row of the chunk
  if (r >= nrows) return;
  const int gu = unit_lo + r / kUnitRows;
  const int b = gu / nrb;
  const int row = (gu % nrb) * kUnitRows + r % kUnitRows;
  if (row >= NqG) return;  // past the last row of a sequence
  int32_t* out = sel + (int64_t(b) * NqG + row) * K;
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  if (!sv.ok) {
    for (int k = lane; k < K; k += 32) out[k] = -1;
    if (lane == 0 && row % kUnitRows == 0) set_status(status, MSA_ERR_BOUNDS);
    return;
  }
  const int loc = (sv.q0 + row / G) / Bs;
  if (loc + 1 <= K) {  // every visible block
    for (int k = lane; k < K; k += 32) out[k] = k <= loc ? k : -1;
    return;
  }
  const int need = K - 1 - fs;
  if (lane == 0) {
    if (fs) out[0] = 0;
    out[K - 1] = loc;
  }
  if (need == 0) return;
  out += fs;
  const float* M = table + int64_t(r) * tstride;
  // 1. per-lane sample (kSelBatch loads in flight per lane; -inf past the row)
  float s0 = -INFINITY, s1 = -INFINITY;
  for (int t0 = fs; t0 < loc; t0 += 32 * kSelBatch) {
    float v[kSelBatch];
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u) {
      const int t = t0 + 32 * u + lane;
      v[u] = t < loc ? __ldg(M + t) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u) {
      if constexpr (NS == 1) {
        s0 = fmaxf(s0, v[u]);
      } else {
        s1 = fmaxf(s1, fminf(s0, v[u]));
        s0 = fmaxf(s0, v[u]);
      }
    }
  }
  // T is the (32 NS - need + 1)-th smallest sample value. When that is one
  // of the few smallest, take it by repeated minimum extraction (a lane's
  // values are in ascending order: lo, then hi2); otherwise rank the sample
  // values by shuffles.
  uint32_t T;
  const int below = 32 * NS - need;  // sample values below T in the sorted order
  if (below <= 3) {
    uint32_t lo = ord_f32(NS == 1 ? s0 : s1), hi2 = NS == 1 ? 0xFFFFFFFFu : ord_f32(s0);
    for (int x = 0; x < below; ++x) {
      const uint32_t m = __reduce_min_sync(0xffffffffu, lo);
      const unsigned who = __ballot_sync(0xffffffffu, lo == m);
      if (lane == __ffs(who) - 1) {
        lo = hi2;
        hi2 = 0xFFFFFFFFu;
      }
    }
    T = __reduce_min_sync(0xffffffffu, lo);
  } else {
    int c0 = 0, c1 = 0;
#pragma unroll 8
    for (int o = 0; o < 32; ++o) {
      const float x0 = __shfl_sync(0xffffffffu, s0, o);
      c0 += x0 >= s0;
      if constexpr (NS == 2) {
        const float x1 = __shfl_sync(0xffffffffu, s1, o);
        c0 += x1 >= s0;
        c1 += (x0 >= s1) + (x1 >= s1);
      }
    }
    uint32_t mine = c0 >= need ? ord_f32(s0) : 0u;
    if constexpr (NS == 2) mine = max(mine, c1 >= need ? ord_f32(s1) : 0u);
    T = __reduce_max_sync(0xffffffffu, mine);
  }
  T = max(T, 1u);
  const uint32_t hi = __reduce_max_sync(0xffffffffu, max(ord_f32(s0), 1u));  // the row maximum
  // 2. candidates >= T in ascending t (a list of the first kSelCap; C counts all)
  uint32_t* lv = list_v[warp];
  int* ltb = list_t[warp];
  int C = 0;
  auto compact = [&](float Tf) {
    C = 0;
    for (int t0 = fs; t0 < loc; t0 += 32 * kSelBatch) {
      float v[kSelBatch];
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        const int t = t0 + 32 * u + lane;
        v[u] = t < loc ? __ldg(M + t) : -INFINITY;
      }
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {  // ascending t: batch by batch, then lane by lane
        const bool f = v[u] >= Tf;
        const unsigned fm = __ballot_sync(0xffffffffu, f);
        if (fm) {
          if (f) {
            const int q = C + __popc(fm & lt);
            if (q < kSelCap) {  // the float's bits; converted when loaded below
              lv[q] = __float_as_uint(v[u]);
              ltb[q] = t0 + 32 * u + lane;
            }
          }
          C += __popc(fm);
        }
      }
    }
    __syncwarp();
  };
  constexpr int kPerLane = kSelCap / 32;
  uint32_t e[kPerLane];  // list entry lane + 32 k, order-preserving (0 past the list)
  auto load_list = [&](int n) {
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) {
      const int i = lane + 32 * k;
      e[k] = i < n ? max(ord_f32(__uint_as_float(lv[i])), 1u) : 0u;
    }
  };
  // The need-th largest of the n list values (all >= lo, n >= need): bisection
  // (two bits per round, from below the bits that lo and the list maximum
  // share; the three counts of a round summed as one packed word) while the
  // bucket [v, v + 2^w) holding it has more than 32 values, then those values
  // ranked among themselves. ge = values >= v, above = values >= v + 2^w.
  auto list_kth = [&](int n, uint32_t lo) -> uint32_t {
    uint32_t hl = 0;
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) hl = max(hl, e[k]);
    hl = __reduce_max_sync(0xffffffffu, hl);
    const uint32_t diff = lo ^ hl;
    int w = diff ? ((32 - __clz(int(diff))) + 1) & ~1 : 0;  // low bits to resolve (even)
    uint32_t v = w >= 32 ? 0u : (lo & ~((1u << w) - 1u));
    int ge = n, above = 0;
    while (w > 0 && ge - above > 32) {
      const int sh = w - 2;
      const uint32_t c1v = v | (1u << sh), c2v = v | (2u << sh), c3v = v | (3u << sh);
      uint32_t cnt = 0;  // counts of at most kSelCap in 10-bit fields
#pragma unroll
      for (int k = 0; k < kPerLane; ++k)
        if (32 * k < n) cnt += uint32_t(e[k] >= c1v) + (uint32_t(e[k] >= c2v) << 10) + (uint32_t(e[k] >= c3v) << 20);
      cnt = __reduce_add_sync(0xffffffffu, cnt);
      const int n1 = int(cnt & 1023u), n2 = int((cnt >> 10) & 1023u), n3 = int(cnt >> 20);
      const uint32_t best = n3 >= need ? 3u : (n2 >= need ? 2u : (n1 >= need ? 1u : 0u));
      above = best == 3u ? above : (best == 2u ? n3 : (best == 1u ? n2 : n1));
      ge = best == 3u ? n3 : (best == 2u ? n2 : (best == 1u ? n1 : ge));
      v |= best << sh;
      w = sh;
    }
    if (w == 0) return v;
    const uint64_t vend = uint64_t(v) + (uint64_t(1) << w);
    int nbk = 0;
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) {
      if (32 * k >= n) break;
      const bool in = e[k] >= v && uint64_t(e[k]) < vend;
      const unsigned im = __ballot_sync(0xffffffffu, in);
      if (in) lv[nbk + __popc(im & lt)] = e[k];  // the list's float bits are in e[] by now
      nbk += __popc(im);
    }
    __syncwarp();
    // v* is the m-th largest bucket value: a descending bitonic sort across
    // the lanes (lanes past the bucket hold 0, below every value), then lane m - 1
    uint32_t x = lane < nbk ? lv[lane] : 0u;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
        const bool keep_max = ((lane & k) == 0) == ((lane & j) == 0);
        x = keep_max ? max(x, y) : min(x, y);
      }
    }
    const int m = need - above;
    const uint32_t r = __shfl_sync(0xffffffffu, x, m - 1);
    __syncwarp();
    return r;
  };
  // 3. A list that overflows still holds kSelCap candidates: their need-th
  // largest value is a tighter bound, and the compaction runs again. Ties at
  // the bound that make no progress bisect over the row itself.
  bool listed = false;
  for (int attempt = 0; attempt < 3; ++attempt) {
    compact(ord_inv(T));
    load_list(min(C, kSelCap));
    if (C <= kSelCap) {
      listed = true;
      break;
    }
    const uint32_t T2 = list_kth(kSelCap, T);
    if (T2 <= T) break;
    T = T2;
  }
  uint32_t v;
  if (listed) {
    v = list_kth(C, T);
  } else {
    const uint32_t diff = T ^ hi;
    const int nb = diff ? ((32 - __clz(int(diff))) + 1) & ~1 : 0;
    v = nb >= 32 ? 0u : (T & ~((1u << nb) - 1u));
    for (int sh = nb - 2; sh >= 0; sh -= 2) {
      const uint32_t c1v = v | (1u << sh), c2v = v | (2u << sh), c3v = v | (3u << sh);
      int a1 = 0, a2 = 0, a3 = 0;
      for (int t = fs + lane; t < loc; t += 32) {
        const uint32_t x = cand_value(M, t);
        a1 += x >= c1v;
        a2 += x >= c2v;
        a3 += x >= c3v;
      }
      const int n1 = __reduce_add_sync(0xffffffffu, a1);
      const int n2 = __reduce_add_sync(0xffffffffu, a2);
      const int n3 = __reduce_add_sync(0xffffffffu, a3);
      const uint32_t best = n3 >= need ? 3u : (n2 >= need ? 2u : (n1 >= need ? 1u : 0u));
      v |= best << sh;
    }
  }
  // everything above v*, then the lowest-t values equal to v*
  int gt = 0;
  if (listed) {
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) gt += e[k] > v;
  } else {
    for (int t = fs + lane; t < loc; t += 32) gt += cand_value(M, t) > v;
  }
  const int ties = need - __reduce_add_sync(0xffffffffu, gt);
  int base = 0, eq_seen = 0;
  auto emit = [&](uint32_t x, int t, bool have) {
    const bool eq = have && x == v;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool take = have && (x > v || (eq && eq_seen + __popc(eqm & lt) < ties));
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) out[base + __popc(tm & lt)] = t;
    base += __popc(tm);
    eq_seen += __popc(eqm);
  };
  if (listed) {
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) {
      const int i = lane + 32 * k;
      if (32 * k < C) emit(e[k], i < C ? ltb[i] : 0, i < C);
    }
  } else {
    for (int t0 = fs; t0 < loc; t0 += 32) {
      const int t = t0 + lane;
      emit(t < loc ? cand_value(M, t) : 0u, t, t < loc);
    }
  }
}

int g_num_sms[64] = {0};

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return kNumSMs;
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kNumSMs;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

}  // namespace

namespace {
// Chunk table: rows of whole units, row stride a multiple of 8 floats (32-byte
// rows for the vector stores), at most ~4 GiB unless that leaves fewer than
// four units per SM. MSA_INDEX_TABLE_UNITS (environment, read once per
// process) sets the units per chunk instead.
constexpr size_t kTableBudget = size_t(4) << 30;
int table_stride(int Nk, int Bs) { return (((Nk + Bs - 1) / Bs) + 7) & ~7; }
int table_chunk_units(int B, int Nq, int Nk, int G, int Bs) {
  static int env = -1;
  if (env < 0) {
    const char* e = getenv("MSA_INDEX_TABLE_UNITS");
    env = e ? atoi(e) : 0;
  }
  const int64_t total = int64_t(B) * ((int64_t(Nq) * G + kUnitRows - 1) / kUnitRows);
  const size_t unit_bytes = size_t(kUnitRows) * table_stride(Nk, Bs) * sizeof(float);
  int64_t cu = env > 0 ? env : std::max<int64_t>(4 * kNumSMs, int64_t(kTableBudget / unit_bytes));
  return int(std::min<int64_t>(cu, total));
}
bool uses_table(int K) { return K - 1 > kRegList; }
}  // namespace

size_t index_fused_table_bytes(int B, int Nq, int Nk, int G, int Bs, int K) {
  if (!uses_table(K)) return 0;
  return size_t(table_chunk_units(B, Nq, Nk, G, Bs)) * kUnitRows * table_stride(Nk, Bs) * sizeof(float);
}

bool index_fused_supported(int dtype, int Nq, int G, int di, int Bs, int K) {
  if (dtype != MSA_BF16 || (di != 32 && di != 64)) return false;
  if (Bs != 32 && Bs != 64 && Bs != 128) return false;
  if (K < 1 || K > kMaxK) return false;
  if (int64_t(Nq) * G < 4 * kUnitRows || int64_t(Nq) * G > (int64_t(1) << 30)) return false;
  return true;
}

cudaError_t launch_index_fused_tc(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len,
                                  int B, int Nq, int Nk, int G, int di, int Bs, int K, int fs, int32_t* sel,
                                  float* table, size_t table_bytes, uint32_t* status, cudaStream_t stream) {
  const int NqG = Nq * G;
  const bool tab = uses_table(K);
  if (tab && (!table || table_bytes < index_fused_table_bytes(B, Nq, Nk, G, Bs, K))) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  {
    const uint64_t dims[3] = {uint64_t(di), uint64_t(NqG), uint64_t(B)};
    const uint64_t strides[2] = {uint64_t(di) * 2, uint64_t(NqG) * di * 2};
    const uint32_t box[3] = {uint32_t(di), uint32_t(kUnitRows), 1};
    if (!make_tmap_bf16(&tmA, iq, 3, dims, strides, box,
                        di == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {uint64_t(di), uint64_t(Nk), uint64_t(B)};
    const uint64_t strides[2] = {uint64_t(di) * 2, uint64_t(Nk) * di * 2};
    const uint32_t box[3] = {uint32_t(di), uint32_t(kTileN), 1};
    if (!make_tmap_bf16(&tmB, ik, 3, dims, strides, box,
                        di == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  const size_t a_bytes = size_t(kUnitRows) * di * 2, b_bytes = size_t(kTileN) * di * 2;
  const int Kc = K - 1 > 0 ? K - 1 : 1;
  const size_t lists = tab ? 0 : size_t(Kc) * kUnitRows * 8;
  const size_t stage = !tab ? 0 : Bs == 32 ? table_stage_bytes<32>() : Bs == 64 ? table_stage_bytes<64>() : table_stage_bytes<128>();
  const size_t fixed = 1024 /*alignment slack*/ + lists + stage + 256 /*barriers, flags*/;
  const size_t budget = 227 * 1024;
  int nA = 2, S = 8;
  while (S > 2 && fixed + nA * a_bytes + S * b_bytes > budget) --S;
  if (fixed + nA * a_bytes + S * b_bytes > budget) nA = 1;
  while (S > 2 && fixed + nA * a_bytes + S * b_bytes > budget) --S;
  const size_t smem = fixed + nA * a_bytes + S * b_bytes;
  if (smem > budget) return cudaErrorInvalidValue;
  // barriers must fit in the 256 reserved bytes
  if ((2 * S + 2 * nA + 5) * 8 + 8 > 256) return cudaErrorInvalidValue;

  const int nrb = (NqG + kUnitRows - 1) / kUnitRows;
  const int total = B * nrb;
  const int tstride = table_stride(Nk, Bs);
  const int chunk = tab ? table_chunk_units(B, Nq, Nk, G, Bs) : total;
  // the chunk table for TMA stores: (tstride, chunk rows) fp32, boxes of 32
  // rows x (256 / Bs) blocks (unused by the other forms)
  CUtensorMap tmT;
  std::memset(&tmT, 0, sizeof(tmT));
  if (tab && 256 / Bs * 4 >= 16) {
    const uint64_t dims[2] = {uint64_t(tstride), uint64_t(chunk) * kUnitRows};
    const uint64_t strides[1] = {uint64_t(tstride) * 4};
    const uint32_t box[2] = {uint32_t(256 / Bs), 32};
    if (!make_tmap_f32(&tmT, table, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
  }
  const int need = K - 1 - fs;
  // The register split re-allocates exactly the launch allocation: a build
  // that launches with another register count must not run (the increase
  // would wait for registers that are never released).
#define MSA_FUSED(DI_, BS_, REG_, TAB_)                                                                         \
  do {                                                                                                          \
    auto kern = index_fused_tc_kernel<DI_, BS_, REG_, TAB_>;                                                   \
    cudaFuncAttributes fa;                                                                                      \
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);                                                           \
    if (e != cudaSuccess) return e;                                                                            \
    if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads) return cudaErrorInvalidConfiguration;  \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));                    \
    if (e != cudaSuccess) return e;                                                                            \
    ProfScope prof("index_fused_tc", stream);                                                                  \
    kern<<<grid, kThreads, smem, stream>>>(tmA, tmB, tmT, q_offset, kv_len, Nq, Nk, G, K, fs, nA, S, lo, n,     \
                                           sel, table, tstride, status);                                      \
  } while (0)
#define MSA_FUSED_BS(DI_, REG_, TAB_)  \
  do {                                 \
    if (Bs == 128)                     \
      MSA_FUSED(DI_, 128, REG_, TAB_); \
    else if (Bs == 64)                 \
      MSA_FUSED(DI_, 64, REG_, TAB_);  \
    else                               \
      MSA_FUSED(DI_, 32, REG_, TAB_);  \
  } while (0)
  for (int lo = 0; lo < total; lo += chunk) {
    const int n = std::min(chunk, total - lo);
    const int grid = n < num_sms() ? n : num_sms();
    if (di == 64) {
      if (tab)
        MSA_FUSED_BS(64, false, true);
      else
        MSA_FUSED_BS(64, true, false);
    } else {
      if (tab)
        MSA_FUSED_BS(32, false, true);
      else
        MSA_FUSED_BS(32, true, false);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !tab) return e;
    const int rows = n * kUnitRows;
    const unsigned sgrid = unsigned((rows + kSelWarps - 1) / kSelWarps);
    ProfScope prof("index_topk_table", stream);
    if (need <= 32)
      index_topk_table_kernel<1><<<sgrid, kSelWarps * 32, 0, stream>>>(table, tstride, lo, rows, nrb, NqG, G, Nq, Nk,
                                                                       Bs, K, fs, q_offset, kv_len, sel, status);
    else
      index_topk_table_kernel<2><<<sgrid, kSelWarps * 32, 0, stream>>>(table, tstride, lo, rows, nrb, NqG, G, Nq, Nk,
                                                                       Bs, K, fs, q_offset, kv_len, sel, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
#undef MSA_FUSED_BS
#undef MSA_FUSED
  return cudaSuccess;
}

}  // namespace msa
