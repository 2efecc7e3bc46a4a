// Main Branch, prefill, KV-outer on tcgen05 (bf16, sm_103a).
// (hyper.ai summary of paper 2606.13392, "方法": exact softmax attention over
//  the selected blocks with K/V gathered per block; "核心贡献": KV-outer sparse
//  attention that raises tensor-core use at block granularity and handles
//  skewed block popularity without atomic updates; quant_prune_distill post
//  751, "Метод": a persistent grid for uneven, dynamic load.)
//
// Per query chunk (queries of one sequence, chunked to bound the scratch):
//  1. attn_count    per (group, key block) number of (query, slot) entries that
//                   selected it (shared-memory histograms, one global add per
//                   non-empty bin and CTA)
//  2. attn_scan     exclusive scans: entry offsets and 128-row tile offsets
//  3. attn_tiles    the tile list: (bin, first entry, entry count)
//  4. attn_fill     the inverted lists: bin -> (query, slot) entries
//  5. attn_kv_outer persistent kernel. Each CTA takes a contiguous run of
//                   tiles (ordered by bin, so K/V of a block is loaded once
//                   per run of its tiles). Per tile: gather the 128 query rows
//                   (128/hpg queries x hpg heads of the group), S = Q K^T on
//                   tcgen05 into TMEM, exact softmax in registers (causal mask
//                   only in the local block), P (bf16) written back over S in
//                   TMEM, O = P V on tcgen05 into TMEM, then the per-slot
//                   partial (O / l in bf16, lse in fp32) is stored for the
//                   combine straight from registers (chunk-major rows, so a
//                   warp store covers 512 contiguous bytes).
//  6. attn_combine  per (query, head): log-sum-exp merge of the K slot
//                   partials in slot order -> output row. Deterministic; no
//                   atomics on any output.
//
// attn_kv_outer warp roles (512 threads): warp 0 K/V TMA producer, warps 1-4
// query-row gather (one ring slot each; per tile, four-row TMA gathers for
// rows 80-127 and cp.async for rows 0-79, entries fetched a ring ahead), warp 5
// TMEM owner + MMA issuer, warps 6-7 idle; warps 8-15 two epilogue warpgroups that
// alternate tiles (ping-pong), each owning S (Bs columns) and O (D columns) in
// TMEM. Warpgroups 0-1 hand registers to the epilogue (88 -> 168 per thread)
// so that a whole S row and a whole O row are read from TMEM at once. All
// waits are bounded.
#include <cmath>
#include <algorithm>
#include <cstdlib>

#include "msa_internal.cuh"
#include "tc_utils.cuh"

namespace msa {
namespace {

constexpr int kRows = 128;  // query rows per tile (M of both MMAs)
constexpr int kAttnThreads = 512;
constexpr int kLaunchRegs = 128;  // registers per thread at launch (checked on the host)
// Two designs share this file. The two-issuer design (blocks of 64 and 32
// keys). Warpgroups 0 and 1 (80 registers): warps 0, 1, 2 and 6 gather
// query rows (one ring slot each), warp 3 loads K and V and owns TMEM, warps
// 4 and 5 issue the MMAs of softmax warpgroup 0 and 1, warp 7 is idle.
// Warpgroups 2 and 3 (176 registers: a 128-key row of S in registers): the
// softmax of alternate tiles and the store of their O.
constexpr int kProdRegs = 80, kSoftRegs = 176;
static_assert(128 * (2 * kProdRegs + 2 * kSoftRegs) <= kAttnThreads * kLaunchRegs, "register split");
constexpr int kLoadWarp = 3;   // K/V loads, TMEM allocation
constexpr int kIssueWarp0 = 4;  // warps 4, 5: MMA issuers of softmax warpgroups 0, 1
constexpr int kGatherWarpHi = 6;  // the fourth gather warp (with warps 0, 1, 2)
constexpr int kEpiWarp0 = 8;    // warps 8..15 (warpgroups 2 and 3)
// The single-issuer design (blocks of 128 keys): warpgroup 0 (80 registers):
// warps 0-2 gather query rows, warp 3 issues the MMAs, loads K and V and owns
// TMEM; warpgroup 1 (80) stores the partials; warpgroups 2 and 3 (176) run
// the softmax of alternate tiles.
template <int BS>
struct AttnRegs {
  static constexpr int kStore = BS == 128 ? 80 : 96;
  static constexpr int kSoft = BS == 128 ? 176 : 168;
  static_assert(128 * (kProdRegs + kStore + 2 * kSoft) <= kAttnThreads * kLaunchRegs, "register split");
};
constexpr int kTmaWarp0 = 0;  // warps 0..2: query-row gathers (four-row TMA gathers)
constexpr int kTmaWarps = 3;
constexpr int kMmaWarpA = 3;  // MMA issuer, TMEM owner and K/V loads
constexpr int kStoreWarp0 = 4;  // warps 4..7 (warpgroup 1)
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// inversion
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool entry_valid(int t, int pos, int Bs, int nblk) {
  return t >= 0 && t < nblk && t * Bs <= pos;
}

// grid (row chunks, G); dynamic smem = nblk ints
__global__ void attn_count_kernel(const int32_t* __restrict__ sel, const int32_t* __restrict__ q_offset,
                                  const int32_t* __restrict__ kv_len, int b, int Nq, int Nk, int G, int K, int Bs,
                                  int nblk, int c0, int cq, int rows_per_cta, int* __restrict__ cnt,
                                  int* __restrict__ hist_g, uint32_t* status) {
  extern __shared__ int hist[];
  const int g = blockIdx.y;
  for (int t = threadIdx.x; t < nblk; t += blockDim.x) hist[t] = 0;
  __syncthreads();
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  const int r0 = blockIdx.x * rows_per_cta;
  const int r1 = min(cq, r0 + rows_per_cta);
  if (sv.ok) {
    for (int e = threadIdx.x; e < (r1 - r0) * K; e += blockDim.x) {
      const int il = r0 + e / K, k = e % K;
      const int i = c0 + il;
      const int t = sel[((int64_t(b) * Nq + i) * G + g) * K + k];
      if (t < -1 || t >= nblk) set_status(status, MSA_ERR_BOUNDS);
      if (entry_valid(t, sv.q0 + i, Bs, nblk)) atomicAdd(&hist[t], 1);
    }
  }
  __syncthreads();
  // the CTA's histogram is kept for attn_fill (same CTA decomposition)
  int* keep = hist_g + (int64_t(g) * gridDim.x + blockIdx.x) * nblk;
  for (int t = threadIdx.x; t < nblk; t += blockDim.x) {
    keep[t] = hist[t];
    if (hist[t]) atomicAdd(&cnt[g * nblk + t], hist[t]);
  }
}

// Relative cost of a tile pass's work: a tile, the first tile of a bin (its
// K/V load and the pipeline bubble around it), a tile holding rows whose
// local block this is (masked). The forward attention's weights were fitted
// to per-CTA cycle counts; the KL and backward tile passes (whose epilogues
// bind) were measured faster with a lighter bin weight and no masked weight.
constexpr int kCostTile = 32, kCostBin = 17, kCostMasked = 8;
constexpr int kCostTileT = 32, kCostBinT = 8, kCostMaskedT = 0;
constexpr int kMaxGrid = kKvoMaxGrid;  // persistent grid: one CTA per SM

// The tile where a cost prefix reaches X, searching bins [blo, bhi] (the last
// bin whose cost offset is <= X, then a proportional share of its tiles).
__device__ int split_tile(const int* __restrict__ cost_off, const int* __restrict__ tile_off, int blo, int bhi,
                          int64_t X) {
  while (blo < bhi) {
    const int mid = (blo + bhi + 1) >> 1;
    if (cost_off[mid] <= X)
      blo = mid;
    else
      bhi = mid - 1;
  }
  const int nt = tile_off[blo + 1] - tile_off[blo];
  const int64_t c = int64_t(cost_off[blo + 1]) - cost_off[blo];
  const int64_t kq = c > 0 ? (X - cost_off[blo]) * nt / c : 0;
  return tile_off[blo] + (kq < nt ? int(kq) : nt);
}

// single CTA of 1024 threads: tile offsets, entry offsets (= tile offset x
// entries per tile: every tile owns a full slot range), tile total, and the
// persistent grid's splits:
//  - cta_start: CTA j takes tiles [cta_start[j], cta_start[j+1]), contiguous
//    runs of equal estimated cost under the training passes' weights (the KL
//    and backward passes);
//  - cta_seg [nph][grid + 1]: phase p (the bins of groups
//    [p G / nph, (p+1) G / nph)) split the same way on its own, so that CTA j
//    takes a 1/grid share of every phase, phase after phase (the forward
//    attention: all CTAs gather the query rows of the same groups at a time).
__global__ void __launch_bounds__(1024) attn_scan_kernel(const int* __restrict__ cnt, const int32_t* __restrict__ q_offset,
                                                         int b, int nblk, int nbins, int per_tile, int Bs, int c0,
                                                         int cq, int grid, int G, int nph, int* __restrict__ entry_off,
                                                         int* __restrict__ tile_off, int* __restrict__ cost_off,
                                                         int* __restrict__ cost_off2, int* __restrict__ total_tiles,
                                                         int* __restrict__ cta_start, int* __restrict__ cta_seg) {
  __shared__ int s_e[1024], s_t[1024], s_c[1024], s_c2[1024];
  const int tid = threadIdx.x;
  const int per = (nbins + 1023) / 1024;
  const int lo = min(nbins, tid * per), hi = min(nbins, lo + per);
  const int q0 = q_offset ? q_offset[b] : 0;
  // queries of the chunk whose local block is this bin's block
  auto nloc_of = [&](int x) {
    const int t = x % nblk;
    const int a0 = max(c0, t * Bs - q0), a1 = min(c0 + cq, (t + 1) * Bs - q0);
    return max(0, a1 - a0);
  };
  auto bin_cost = [&](int x, int nt) {  // forward attention
    return nt > 0 ? kCostTile * nt + kCostBin + kCostMasked * min(nt, nloc_of(x)) : 0;
  };
  auto bin_cost2 = [&](int x, int nt) {  // KL and backward tile passes
    return nt > 0 ? kCostTileT * nt + kCostBinT + kCostMaskedT * min(nt, nloc_of(x)) : 0;
  };
  int se = 0, st = 0, sc = 0, sc2 = 0;
  for (int x = lo; x < hi; ++x) {
    const int nt = (cnt[x] + per_tile - 1) / per_tile;
    se += cnt[x];
    st += nt;
    sc += bin_cost(x, nt);
    sc2 += bin_cost2(x, nt);
  }
  s_e[tid] = se;
  s_t[tid] = st;
  s_c[tid] = sc;
  s_c2[tid] = sc2;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive Hillis-Steele scans
    const int ve = tid >= off ? s_e[tid - off] : 0;
    const int vt = tid >= off ? s_t[tid - off] : 0;
    const int vc = tid >= off ? s_c[tid - off] : 0;
    const int vc2 = tid >= off ? s_c2[tid - off] : 0;
    __syncthreads();
    s_e[tid] += ve;
    s_t[tid] += vt;
    s_c[tid] += vc;
    s_c2[tid] += vc2;
    __syncthreads();
  }
  int bt = s_t[tid] - st, bc = s_c[tid] - sc, bc2 = s_c2[tid] - sc2;
  for (int x = lo; x < hi; ++x) {
    const int nt = (cnt[x] + per_tile - 1) / per_tile;
    entry_off[x] = bt * per_tile;  // a bin's entries start on a tile boundary
    tile_off[x] = bt;
    cost_off[x] = bc;
    cost_off2[x] = bc2;
    bt += nt;
    bc += bin_cost(x, nt);
    bc2 += bin_cost2(x, nt);
  }
  if (tid == 1023) {
    entry_off[nbins] = s_t[1023] * per_tile;
    tile_off[nbins] = s_t[1023];
    cost_off[nbins] = s_c[1023];
    cost_off2[nbins] = s_c2[1023];
    *total_tiles = s_t[1023];
  }
  __syncthreads();
  // CTA j starts at the tile where the cost prefix reaches total * j / grid
  const int64_t ctot = s_c2[1023];
  const int ttot = s_t[1023];
  for (int j = tid; j <= grid; j += 1024)
    cta_start[j] = j == grid ? ttot : split_tile(cost_off2, tile_off, 0, nbins - 1, ctot * j / grid);
  for (int x = tid; x < nph * (grid + 1); x += 1024) {
    const int ph = x / (grid + 1), j = x % (grid + 1);
    const int blo = (ph * G / nph) * nblk, bhi = ((ph + 1) * G / nph) * nblk;  // bins [blo, bhi)
    const int64_t c0p = cost_off[blo], c1p = cost_off[bhi];
    cta_seg[x] = j == grid ? tile_off[bhi] : split_tile(cost_off, tile_off, blo, bhi - 1, c0p + (c1p - c0p) * j / grid);
  }
}

// one thread per bin: its tiles (bin, first entry, count, tiles of the bin
// from this one on)
__global__ void attn_tiles_kernel(const int* __restrict__ cnt, const int* __restrict__ entry_off,
                                  const int* __restrict__ tile_off, int nbins, int per_tile, int4* __restrict__ tiles) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= nbins) return;
  const int c = cnt[x], e0 = entry_off[x], t0 = tile_off[x];
  const int nt = (c + per_tile - 1) / per_tile;
  for (int j = 0; j < nt; ++j) tiles[t0 + j] = make_int4(x, e0 + j * per_tile, min(per_tile, c - j * per_tile), nt - j);
}

// grid (row chunks, G); dynamic smem = 2 * nblk ints. Entry = local query * 64 + slot;
// rev[(query, group, slot)] = the entry's index (its partial's row block).
__global__ void attn_fill_kernel(const int32_t* __restrict__ sel, const int32_t* __restrict__ q_offset,
                                 const int32_t* __restrict__ kv_len, int b, int Nq, int Nk, int G, int K, int Bs,
                                 int nblk, int c0, int cq, int rows_per_cta, const int* __restrict__ entry_off,
                                 const int* __restrict__ hist_g, int* __restrict__ cursor, int* __restrict__ entries,
                                 int* __restrict__ rev) {
  extern __shared__ int sm[];
  int* hist = sm;
  int* base = sm + nblk;
  const int g = blockIdx.y;
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  const int r0 = blockIdx.x * rows_per_cta;
  const int r1 = min(cq, r0 + rows_per_cta);
  // this CTA's range of every bin, from the histogram attn_count kept
  const int* keep = hist_g + (int64_t(g) * gridDim.x + blockIdx.x) * nblk;
  for (int t = threadIdx.x; t < nblk; t += blockDim.x) {
    const int h = keep[t];
    base[t] = h ? entry_off[g * nblk + t] + atomicAdd(&cursor[g * nblk + t], h) : 0;
    hist[t] = 0;
  }
  __syncthreads();
  if (sv.ok) {
    for (int e = threadIdx.x; e < (r1 - r0) * K; e += blockDim.x) {
      const int il = r0 + e / K, k = e % K;
      const int t = sel[((int64_t(b) * Nq + c0 + il) * G + g) * K + k];
      if (entry_valid(t, sv.q0 + c0 + il, Bs, nblk)) {
        const int slot = atomicAdd(&hist[t], 1);
        entries[base[t] + slot] = il * 64 + k;
        rev[(int64_t(il) * G + g) * K + k] = base[t] + slot;  // where this (query, slot) partial lands
      }
    }
  }
}

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// paired fp32 arithmetic (one instruction for two lanes of a 64-bit register pair)
__device__ __forceinline__ uint64_t f32x2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_bits(uint32_t a, uint32_t b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(uint64_t r) {
  float a, b;
  unpack_f32x2(r, a, b);
  return pack_bf16(a, b);
}

struct AttnParams {
  const __nv_bfloat16* q;  // [B, Nq, Hq, D]
  uint4* part_o;           // [tiles][D / 8 chunks][128 rows] x 16 bytes (8 bf16)
  const int* entries;      // chunk entries
  const int4* tiles;       // chunk tiles
  const int* cta_seg;      // [nph][grid + 1]: CTA j's tiles of phase p are [cta_seg[p][j], cta_seg[p][j + 1])
  const int32_t* q_offset;
  const int32_t* kv_len;
  float* part_lse;        // [entries, hpg]: row (entry * hpg + head in group)
  uint32_t* status;
  int b, Nq, Nk, Hq, G, Bs, K, nblk, c0, hpg, nph, grid;
  int inject_timeout;  // test hook: the kernel first waits on a barrier nothing completes
  float scale_log2;  // softmax scale * log2(e)
  float scale;
};


constexpr int kRing = 4;  // gathered-query tile ring depth (tile z in slot z % kRing)
// V buffers: two where shared memory has room for them (blocks of up to 64
// keys), so a block's V is loaded ahead like its K; one at 128 keys
constexpr int attn_v_buffers(int bs) { return bs <= 64 ? 2 : 1; }
// Query rows reach the ring by four-row TMA gathers (512 bytes each, 64 per
// tile). Issuing one holds a warp about 70-90 cycles, so the gather rate grows
// with the number of warps that issue them: four warps, one ring slot each.
// Measured alternatives were slower: a cp.async warp issues about a third of
// a TMA warp's rate.


// The single-issuer design, used for blocks of 128 keys: one MMA thread,
// three gather warps and a partial-store warpgroup (the 128-key softmax is
// long enough to hide them); see the constants above.
template <int D, int BS>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kv_outer_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmQ, const AttnParams p) {
  constexpr uint32_t kQBytes = kRows * D * 2;       // one gathered query tile (= one bf16 O tile)
  constexpr uint32_t kSlot = kQBytes;
  constexpr uint32_t kKVHalf = BS * 128;            // one 64-wide half of a K or V block
  constexpr uint32_t kKBytes = BS * D * 2;
  constexpr int NH = D / 64;
  constexpr int NV = attn_v_buffers(BS);
  constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(128, BS, false);
  constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, D, true);  // B = V is MN-major
  constexpr uint32_t kDescHi = tc::smem_desc_hi(1024, 2);           // 128B swizzle, 8-row groups 1024 B apart
  // TMEM columns: warpgroup w owns S at [256 w, 256 w + BS) and O at [256 w + 128, 256 w + 128 + D)
  static_assert(BS <= 128 && D <= 128, "TMEM plan: S <= 128 and O <= 128 columns per warpgroup");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (tc::smem_u32(smem_raw) & 1023u) {  // the swizzled operands need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, MSA_ERR_CUDA);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* k_buf = smem;                    // [2][NH][BS][128 B]: the current key block's K and the next one's
  uint8_t* v_buf = k_buf + 2 * kKBytes;     // [NV][NH][BS][128 B]
  uint8_t* ring = v_buf + NV * kKBytes;     // kRing x kSlot: gathered Q tiles
  float* inv_l = reinterpret_cast<float*>(ring + kRing * kSlot);  // [kRing][128] 1 / row sum of tile z in z % kRing
  int* run_lo = reinterpret_cast<int*>(inv_l + kRing * kRows);    // [kKvoMaxPhases]
  int* run_pref = run_lo + kKvoMaxPhases;                   // [kKvoMaxPhases + 1]
  // mbarriers need 8-byte alignment: round the barrier area up to 16 bytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(run_pref + kKvoMaxPhases + 1) + 15) & ~uintptr_t(15));
  uint64_t* k_full = bars + 0;   // [2] a key block's K has landed in K buffer i
  uint64_t* k_empty = bars + 2;  // [2] the last QK of a block has read K buffer i
  uint64_t* v_full = bars + 4;   // [2] a key block's V has landed in V buffer i (i < NV)
  uint64_t* v_empty = bars + 6;  // [2] the last PV of a block has read V buffer i
  uint64_t* q_full = bars + 8;                // [kRing]
  uint64_t* q_empty = q_full + kRing;         // [kRing]
  uint64_t* s_full = q_empty + kRing;         // [2]
  uint64_t* p_full = s_full + 2;              // [2]
  uint64_t* o_full = p_full + 2;              // [2]
  uint64_t* o_empty = o_full + 2;             // [2]
  uint64_t* done_bar = o_empty + 2;
  uint64_t* never_bar = done_bar + 1;  // no thread arrives on it (timeout injection)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&k_full[i], 1);
      tc::mbar_init(&k_empty[i], 1);
      tc::mbar_init(&v_full[i], 1);
      tc::mbar_init(&v_empty[i], 1);
    }
    for (int r = 0; r < kRing; ++r) {
      tc::mbar_init(&q_full[r], 1);  // the tile's gather warp (arrival with the expected bytes)
      tc::mbar_init(&q_empty[r], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&s_full[s], 1);
      tc::mbar_init(&p_full[s], 4);
      tc::mbar_init(&o_full[s], 1);
      tc::mbar_init(&o_empty[s], 4);  // the four store warps
    }
    tc::mbar_init(done_bar, 1);
    tc::mbar_init(never_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    load_tile_runs(p.cta_seg, p.nph, p.grid, run_lo, run_pref);  // this CTA's share of every phase
  }
  if (warp == kMmaWarpA) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (warp == kMmaWarpA && lane == 0) {
    tc::tma_prefetch(&tmK);
    tc::tma_prefetch(&tmV);
    tc::tma_prefetch(&tmQ);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // this CTA's tiles: local numbers z in [0, n), mapped to the chunk's tiles by TileRuns
  const int n = run_pref[p.nph];
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(p.status, MSA_ERR_TIMEOUT);
  };

  // Each register re-allocation sits at the top of its warpgroups' branch
  // (one instruction for all warps of a warpgroup) so that the compiler
  // budgets each branch with its own register count.
  if (warp < kStoreWarp0) {
  tc::regs_dec<kProdRegs>();
  if (warp >= kTmaWarp0 && warp < kTmaWarp0 + kTmaWarps) {
    // ------------------------------ query-row gather ------------------------------
    // Gather warp gi takes tiles z = gi, gi + kTmaWarps, ... (ring slot z %
    // kRing). Lane l gathers rows [4 l, 4 l + 4) with one four-row TMA
    // gather per 64-column half into the 128B-swizzled K-major layout (the
    // swizzle is address-based); the bytes are counted on the slot's barrier
    // with the warp's arrival. A lane loads its rows' entries itself, one of
    // its tiles ahead (one load when the rows share an entry, as they do
    // when the heads per group are a multiple of 4). Rows of padding entries
    // read the chunk's first query (finite values; their outputs are never
    // read).
    const int gi = warp - kTmaWarp0;
    static_assert(kRows == 32 * 4, "one lane per four rows");
    const int per_tile = kRows / p.hpg;
    const bool one_entry = p.hpg % 4 == 0;  // rows 4 l .. 4 l + 3 belong to one entry
    int4 tl = make_int4(0, 0, 0, 0);
    int ev[4];  // the entries of this lane's four rows (-1 past the tile's count)
    TileRuns runs{run_lo, run_pref};
    const uint64_t pol_q = tc::policy_evict_last();  // the phase's query rows are reused by every CTA
    auto fetch = [&](int z) {  // independent loads: tile zt's entries start at zt * per_tile
      const int zt = runs.at(z);
      tl = p.tiles[zt];
      const int* ent = p.entries + int64_t(zt) * per_tile;
      if (one_entry) {
        const int e = lane * 4 / p.hpg;
        ev[0] = ev[1] = ev[2] = ev[3] = e < per_tile ? ent[e] : -1;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = (lane * 4 + j) / p.hpg;
          ev[j] = e < per_tile ? ent[e] : -1;
        }
      }
    };
    if (gi < n) fetch(gi);
    int issued = 0, last = -1;  // tiles issued by this warp, the last of them
    for (int z = gi; z < n; z += kTmaWarps) {
      const int rs = z % kRing;
      if (!tc::mbar_wait(&q_empty[rs], ((z / kRing) & 1) ^ 1, abort_flag)) {
        fail();
        break;
      }
      const int g = tl.x / p.nblk;
      int rows[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = lane * 4 + j;
        const int il = row / p.hpg < tl.z && ev[j] >= 0 ? (ev[j] >> 6) : 0;
        rows[j] = (p.b * p.Nq + p.c0 + il) * p.Hq + g * p.hpg + row % p.hpg;
      }
      if (lane == 0) tc::mbar_arrive_expect_tx(&q_full[rs], uint32_t(kRows) * D * 2);
      __syncwarp();
      {
        uint8_t* dst = ring + rs * kSlot + lane * 4 * 128;
#pragma unroll
        for (int hf = 0; hf < NH; ++hf)
          tc::tma_gather4_hint(dst + hf * (kRows * 128), &tmQ, &q_full[rs], hf * 64, rows[0], rows[1], rows[2],
                               rows[3], pol_q);
      }
      ++issued;
      last = z;
      if (z + kTmaWarps < n) fetch(z + kTmaWarps);
    }
    // drain after an abort: no gather may still be landing in shared memory
    // when the CTA exits. (In a full run the MMA warp has waited for every
    // tile before the final barrier.) Waits for the last tile this warp issued
    // into each ring slot; one that another warp's later tile has already
    // overtaken ran its course long ago, and its wait ends at the bound.
    int zero = 0;
    if (*abort_flag && lane == 0)
      for (int k = 0; k * kTmaWarps < kRing && k < issued; ++k) {
        const int z = last - k * kTmaWarps;
        tc::mbar_wait(&q_full[z % kRing], (z / kRing) & 1, &zero);
      }
  } else if (warp == kMmaWarpA) {
    // ------------------------------- MMA issuer -------------------------------
    // One thread issues every MMA, so its instructions per tile set the pace
    // when blocks are short: the common path per tile is one wait for the Q
    // tile, QK^T, the previous tile's PV and a few compares; block changes
    // take a separate path. Key blocks are numbered in the order this CTA
    // meets them (bi = 0, 1, ...). Block bi's K goes to K buffer bi & 1 and
    // is loaded during the previous block's second tile (its first tile is
    // known from the tile records, read one tile ahead), into the buffer the
    // block before that has finished with; after a one-tile block it is
    // loaded at the change. With two V buffers V is loaded with K. With one,
    // a block's V is loaded right after the block's first QK, once the
    // previous block's last PV (issued just before) has read the buffer, so
    // the copy overlaps the first tile's softmax.
    if (lane == 0) {
      const uint64_t pol_kv = tc::policy_evict_first();  // each block's K/V is read by one or two CTAs
      // descriptor low words of the first ring slot, K buffer and V buffer
      const uint32_t ring_lo0 = tc::smem_desc_lo(tc::smem_u32(ring), 16);
      const uint32_t k_lo0 = tc::smem_desc_lo(tc::smem_u32(k_buf), 16);
      const uint32_t v_lo0 = tc::smem_desc_lo(tc::smem_u32(v_buf), kKVHalf);
      int kl = 0, vl = 0;  // K / V loads issued: block bi's K is K load bi, its V is V load bi
      int vw = 0;          // blocks whose V has been waited for (once, before the block's first PV)
      bool alive = true;
      auto load_k = [&](int bin, int bi) -> bool {
        const int kb = bi & 1;
        // the buffer's previous block (bi - 2) must be done with it
        if (bi >= 2 && !tc::mbar_wait(&k_empty[kb], ((bi >> 1) - 1) & 1, abort_flag)) return false;
        const int g = bin / p.nblk, t = bin % p.nblk;
        tc::mbar_arrive_expect_tx(&k_full[kb], kKBytes);
#pragma unroll
        for (int h = 0; h < NH; ++h)
          tc::tma_load_4d_hint(k_buf + kb * kKBytes + h * kKVHalf, &tmK, &k_full[kb], h * 64, g, t * BS, p.b,
                               pol_kv);
        kl = bi + 1;
        return true;
      };
      auto load_v = [&](int bin, int bi) -> bool {
        const int vb = bi % NV;
        // the buffer's previous block (bi - NV) must be done with it
        if (bi >= NV && !tc::mbar_wait(&v_empty[vb], ((bi / NV) - 1) & 1, abort_flag)) return false;
        const int g = bin / p.nblk, t = bin % p.nblk;
        tc::mbar_arrive_expect_tx(&v_full[vb], kKBytes);
#pragma unroll
        for (int h = 0; h < NH; ++h)
          tc::tma_load_4d_hint(v_buf + vb * kKBytes + h * kKVHalf, &tmV, &v_full[vb], h * 64, g, t * BS, p.b,
                               pol_kv);
        vl = bi + 1;
        return true;
      };
      // PV of tile z (block bi), the block's last if last_of_bin
      auto issue_pv = [&](int z, int bi, bool last_of_bin) -> bool {
        const int s = z & 1, vb = bi % NV;
        if (vw <= bi) {  // the block's first PV: its V must have landed
          if (!tc::mbar_wait(&v_full[vb], (bi / NV) & 1, abort_flag)) return false;
          vw = bi + 1;
        }
        if (!tc::mbar_wait(&p_full[s], (z >> 1) & 1, abort_flag) ||
            !tc::mbar_wait(&o_empty[s], ((z >> 1) & 1) ^ 1, abort_flag))
          return false;
        tc::fence_after_sync();
        const uint32_t v_lo = v_lo0 + uint32_t(vb) * (kKBytes >> 4);
        const uint32_t t_s = tmem + uint32_t(s) * 256u;
#pragma unroll
        for (int kk = 0; kk < BS / 16; ++kk) {
          // P (bf16 pairs packed per 32-bit column) sits where S was: 16 keys = 8 columns
          tc::mma_f16_ts_lo<kDescHi>(t_s + 128u, t_s + uint32_t(kk) * 8u, v_lo + uint32_t(kk * 16 * 128 >> 4), kIdescPV,
                                     kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&o_full[s]);
        if (last_of_bin) tc::mma_commit(&v_empty[vb]);
        return true;
      };
      if (p.inject_timeout && !tc::mbar_wait_for(never_bar, 0, abort_flag, tc::kInjectedWaitCycles)) {
        fail();
        alive = false;
      }
      // the lookahead cursor: local tile z1 = z + 1 is chunk tile zg1 of run r1 (which ends at local end1)
      int r1 = 0;
      while (r1 < p.nph && run_pref[r1 + 1] == 0) ++r1;
      int zg1 = n > 0 ? run_lo[r1] : 0, end1 = n > 0 ? run_pref[r1 + 1] : 0;
      int4 rec_next = n > 0 ? p.tiles[zg1] : make_int4(-1, 0, 0, 0);
      TileRuns peek{run_lo, run_pref};
      int prev_bin = -1, bi = -1;
      int pend_z = -1, pend_bin = -1;  // at local tile pend_z: load block bi + 1 (from pend_bin)
      if (alive && n > 0 && !(load_k(rec_next.x, 0) && load_v(rec_next.x, 0))) {  // the first block
        fail();
        alive = false;
      }
      for (int z = 0; z < n && alive; ++z) {
        const int s = z & 1, rs = z & (kRing - 1);
        const int4 rec = rec_next;
        const int zg = zg1, end_z = end1;
        if (z + 1 < n) {
          if (z + 1 == end1) {  // the next tile opens the next non-empty run
            do ++r1;
            while (run_pref[r1 + 1] == z + 1);
            zg1 = run_lo[r1];
            end1 = run_pref[r1 + 1];
          } else {
            ++zg1;
          }
          rec_next = p.tiles[zg1];
        }
        const bool first_of_bin = rec.x != prev_bin;
        if (first_of_bin) {
          ++bi;
          // not loaded ahead (the previous block had one tile here): load now
          if ((kl <= bi && !load_k(rec.x, bi)) || (NV == 2 && vl <= bi && !load_v(rec.x, bi)) ||
              !tc::mbar_wait(&k_full[bi & 1], (bi >> 1) & 1, abort_flag)) {
            fail();
            break;
          }
        }
        if (!tc::mbar_wait(&q_full[rs], (z / kRing) & 1, abort_flag)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const uint32_t q_lo = ring_lo0 + uint32_t(rs) * (kSlot >> 4);
        const uint32_t k_lo = k_lo0 + uint32_t(bi & 1) * (kKBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // 16 columns = 32 bytes along the swizzled 128-byte rows
          tc::mma_f16_ss_lo<kDescHi>(tmem + uint32_t(s) * 256u, q_lo + (((kk >> 2) * (kRows * 128) + off) >> 4),
                                     k_lo + (((kk >> 2) * kKVHalf + off) >> 4), kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&s_full[s]);
        tc::mma_commit(&q_empty[rs]);  // the gathered Q tile is consumed
        // the previous tile's PV (the previous block's last at a block change)
        if (z > 0 && !issue_pv(z - 1, first_of_bin ? bi - 1 : bi, first_of_bin)) {
          fail();
          alive = false;
          break;
        }
        if (first_of_bin) {
          // the previous block's K buffer is free once everything issued so
          // far (its last QK among them) has completed
          if (z > 0) tc::mma_commit(&k_empty[(bi - 1) & 1]);
          // the next block: its first tile follows this block's rec.w tiles
          // in this run, or opens the next run; its K (and V) are loaded
          // during this block's second tile
          const int zn = z + rec.w < end_z ? z + rec.w : end_z;
          if (zn < n && zn > z + 1) {
            pend_z = z + 1;
            pend_bin = p.tiles[zn < end_z ? zg + (zn - z) : peek.at(zn)].x;
          }
          // one V buffer: this block's V now. The wait is for the previous
          // block's last PV, issued just above, and ends well before this
          // tile's P is ready
          if (NV == 1 && bi >= 1 && vl == bi && !load_v(rec.x, bi)) {
            fail();
            alive = false;
            break;
          }
        } else if (z == pend_z) {
          if ((kl <= bi + 1 && !load_k(pend_bin, bi + 1)) || (NV == 2 && vl <= bi + 1 && !load_v(pend_bin, bi + 1))) {
            fail();
            alive = false;
            break;
          }
        }
        prev_bin = rec.x;
      }
      if (alive && n > 0 && !*abort_flag) {
        if (!issue_pv(n - 1, bi, true)) fail();
      }
      int zero = 0;  // no K or V copy may still be landing: the last load into each buffer
      for (int b2 = kl - 1; b2 >= 0 && b2 >= kl - 2; --b2) tc::mbar_wait(&k_full[b2 & 1], (b2 >> 1) & 1, &zero);
      for (int b2 = vl - 1; b2 >= 0 && b2 >= vl - NV; --b2) tc::mbar_wait(&v_full[b2 % NV], (b2 / NV) & 1, &zero);
      tc::mma_commit(done_bar);
      tc::mbar_wait(done_bar, 0, &zero);
    }
  }  // other warps of warpgroup 0: none
  } else if (warp < kEpiWarp0) {
    tc::regs_dec<AttnRegs<BS>::kStore>();
    // --------------------------- partial stores ---------------------------
    // Warpgroup 1 reads every tile's O (TMEM lanes of its warp's quarter)
    // and stores it as the tile's bf16 partial rows: 16-byte chunk c of row
    // r of tile zg at part_o[(zg * D/8 + c) * 128 + r], so each warp store
    // instruction writes 32 consecutive rows' chunk (512 contiguous bytes).
    // P is unnormalised: O is scaled by the row's 1 / sum that the softmax
    // left in shared memory (slot z % kRing; the softmax overwrites it only
    // for tile z + kRing, whose QK^T waits for PV(z + 2), which waits for
    // this warpgroup's o_empty arrival below, made after the read).
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    TileRuns runs{run_lo, run_pref};
    const uint64_t pol_part = tc::policy_evict_first();  // partials are read back once, by the combine
    for (int z = 0; z < n; ++z) {
      const int s = z & 1;
      const int zg = runs.at(z);  // the chunk's tile index = its partial row block
      if (!tc::mbar_wait(&o_full[s], (z >> 1) & 1, abort_flag)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      const float inv = inv_l[(z % kRing) * kRows + r];
      const uint64_t inv2 = f32x2(inv, inv);
      const uint32_t o_addr = tmem + lane_base + uint32_t(s) * 256u + 128u;
      uint4* dst = p.part_o + int64_t(zg) * (D / 8) * kRows + r;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tc::tmem_ld_32x32b_x32(o_addr + c0, ov);
        tc::tmem_ld_wait();
        if (c0 + 32 >= D) {  // O is in registers: the next PV may overwrite it
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&o_empty[s]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 o;
          o.x = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 0], ov[c * 8 + 1]), inv2));
          o.y = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 2], ov[c * 8 + 3]), inv2));
          o.z = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 4], ov[c * 8 + 5]), inv2));
          o.w = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 6], ov[c * 8 + 7]), inv2));
          tc::st_v4_hint(dst + (c0 / 8 + c) * kRows, o, pol_part);
        }
      }
    }
  } else {
    tc::regs_inc<AttnRegs<BS>::kSoft>();
    // -------------------------------- softmax --------------------------------
    // Warpgroups 2 and 3 take alternate tiles (TMEM set s = z & 1): the whole
    // S row of a thread's TMEM lane in registers, causal mask in the local
    // block, exact softmax with unnormalised probabilities as P (bf16 pairs
    // written back over S for the PV MMA; the partial-store warps divide O by
    // the row sum), and the row's log-sum-exp stored for the combine. The
    // exponent arguments and the row sum use paired fp32 instructions.
    const int w = (warp - kEpiWarp0) >> 2;         // warpgroup: tiles z with z % 2 == w
    const int quarter = warp & 3;                  // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;             // tile row
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const SeqView sv = seq_view(p.q_offset, p.kv_len, p.b, p.Nq, p.Nk, false);
    TileRuns runs{run_lo, run_pref};
    const uint64_t pol_part = tc::policy_evict_first();
    for (int z = w; z < n; z += 2) {
      const int s = z & 1;  // == w
      // this tile's metadata straight from global memory (the Q ring slot and
      // its staged metadata are recycled as soon as QK^T has consumed them);
      // the loads are in flight while S is being computed
      const int zg = runs.at(z);
      const int4 tl = p.tiles[zg];
      const int e_raw = p.entries[int64_t(zg) * (kRows / p.hpg) + r / p.hpg];
      const int ent = r / p.hpg < tl.z ? e_raw : -1;
      if (!tc::mbar_wait(&s_full[s], (z >> 1) & 1, abort_flag)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      const int bin = tl.x;
      const bool valid = ent >= 0;
      const int t = bin % p.nblk;
      const int il = ent >> 6;
      const int pos = sv.q0 + p.c0 + il;
      const int nvalid = valid ? min(BS, pos - t * BS + 1) : BS;  // keys j <= pos inside the block
      const uint32_t s_addr = tmem + lane_base + uint32_t(s) * 256u;
      const bool full = nvalid >= BS;  // all keys visible (every block but the local one)
      // the whole S row in registers: one TMEM round trip; each 32-column
      // load also returns the maximum of its columns
      uint32_t v[BS];
      float m32[BS / 32];
#pragma unroll
      for (int c = 0; c < BS / 32; ++c) m32[c] = tc::tmem_ld_max_32x32b_x32(s_addr + c * 32, v + c * 32);
      tc::tmem_ld_wait();
      float mx = m32[0];
#pragma unroll
      for (int c = 1; c < BS / 32; ++c) mx = fmaxf(mx, m32[c]);
      if (!full) {  // the local block: the row maximum over its visible keys only
#pragma unroll
        for (int j = 0; j < BS; ++j)
          if (j >= nvalid) v[j] = __float_as_uint(-INFINITY);  // exp2(-inf) = 0 below
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < BS; j += 2)
          m4[(j >> 1) & 3] = tc::fmax3(m4[(j >> 1) & 3], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      // probabilities, 32 keys at a time: packed to bf16 pairs and written
      // back over S in TMEM at once (the PV MMA reads its A operand from
      // there: keys 2c (low half) and 2c+1 (high half) in column c), their
      // sum in fp32, two keys per instruction
      const float mneg = -mx * p.scale_log2;
      uint64_t l2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
      for (int c0 = 0; c0 < BS / 32; ++c0) {
        uint32_t* pk = v + c0 * 32;  // the packed pairs reuse the chunk's first 16 registers
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(v[c0 * 32 + j]), p.scale_log2, mneg));
          const float p1 = ex2(fmaf(__uint_as_float(v[c0 * 32 + j + 1]), p.scale_log2, mneg));
          l2[(j >> 1) & 1] = add_f32x2(l2[(j >> 1) & 1], f32x2(p0, p1));
          pk[j >> 1] = pack_bf16(p0, p1);
        }
        tc::tmem_st_32x32b_x16(s_addr + c0 * 16, pk);
      }
      float la, lb, lc, ld;
      unpack_f32x2(l2[0], la, lb);
      unpack_f32x2(l2[1], lc, ld);
      const float l = (la + lb) + (lc + ld);
      inv_l[(z % kRing) * kRows + r] = l > 0.f ? 1.f / l : 0.f;
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();  // (also orders every lane's 1 / sum before the arrival)
      if (lane == 0) tc::mbar_arrive(&p_full[s]);
      tc::st_f32_hint(p.part_lse + int64_t(zg) * kRows + r, valid ? mx * p.scale + logf(l) : 0.f, pol_part);
    }
  }

  __syncthreads();
  if (warp == kMmaWarpA) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// The two-issuer design, used for blocks of 64 and 32 keys (two to four
// times the tiles per unit of work, each with a short softmax).
template <int D, int BS>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kv_outer2_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmQ, const AttnParams p) {
  constexpr uint32_t kQBytes = kRows * D * 2;       // one gathered query tile (= one bf16 O tile)
  constexpr uint32_t kSlot = kQBytes;
  constexpr uint32_t kKVHalf = BS * 128;            // one 64-wide half of a K or V block
  constexpr uint32_t kKBytes = BS * D * 2;
  constexpr int NH = D / 64;
  constexpr int NV = attn_v_buffers(BS);
  constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(128, BS, false);
  constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, D, true);  // B = V is MN-major
  constexpr uint32_t kDescHi = tc::smem_desc_hi(1024, 2);           // 128B swizzle, 8-row groups 1024 B apart
  // TMEM columns: softmax warpgroup w owns two S buffers at [256 w, 256 w + 2 BS) and O at
  // [256 w + 128, 256 w + 128 + D); tile z uses S buffer (z >> 1) & 1
  static_assert(BS <= 64 && D <= 128, "TMEM plan: 2 BS <= 128 columns of S and O <= 128 columns per warpgroup");
  static_assert(kRing == 4, "four gather warps, one ring slot each");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (tc::smem_u32(smem_raw) & 1023u) {  // the swizzled operands need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, MSA_ERR_CUDA);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* k_buf = smem;                    // [2][NH][BS][128 B]: the current key block's K and the next one's
  uint8_t* v_buf = k_buf + 2 * kKBytes;     // [NV][NH][BS][128 B]
  uint8_t* ring = v_buf + NV * kKBytes;     // kRing x kSlot: gathered Q tiles
  int* run_lo = reinterpret_cast<int*>(ring + kRing * kSlot);  // [kKvoMaxPhases]
  int* run_pref = run_lo + kKvoMaxPhases;                      // [kKvoMaxPhases + 1]
  // mbarriers need 8-byte alignment: round the barrier area up to 16 bytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(run_pref + kKvoMaxPhases + 1) + 15) & ~uintptr_t(15));
  uint64_t* k_full = bars + 0;   // [2] a key block's K has landed in K buffer i
  uint64_t* k_empty = bars + 2;  // [2] both issuers are done with K buffer i (2 arrivals)
  uint64_t* v_full = bars + 4;   // [2] a key block's V has landed in V buffer i (i < NV)
  uint64_t* v_empty = bars + 6;  // [2] both issuers are done with V buffer i (2 arrivals)
  uint64_t* q_full = bars + 8;                // [kRing]
  uint64_t* q_empty = q_full + kRing;         // [kRing]
  uint64_t* s_full = q_empty + kRing;         // [2][2] per softmax warpgroup and S buffer
  uint64_t* p_full = s_full + 4;              // [2]
  uint64_t* o_full = p_full + 2;              // [2]
  uint64_t* done_bar = o_full + 2;            // [2] per issuer
  uint64_t* never_bar = done_bar + 2;  // no thread arrives on it (timeout injection)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&k_full[i], 1);
      tc::mbar_init(&k_empty[i], 2);
      tc::mbar_init(&v_full[i], 1);
      tc::mbar_init(&v_empty[i], 2);
    }
    for (int r = 0; r < kRing; ++r) {
      tc::mbar_init(&q_full[r], 1);  // the slot's gather warp (arrival with the expected bytes)
      tc::mbar_init(&q_empty[r], 1);
    }
    for (int s = 0; s < 4; ++s) tc::mbar_init(&s_full[s], 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&p_full[s], 4);
      tc::mbar_init(&o_full[s], 1);
      tc::mbar_init(&done_bar[s], 1);
    }
    tc::mbar_init(never_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    load_tile_runs(p.cta_seg, p.nph, p.grid, run_lo, run_pref);  // this CTA's share of every phase
  }
  if (warp == kLoadWarp) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tc::tma_prefetch(&tmK);
    tc::tma_prefetch(&tmV);
    tc::tma_prefetch(&tmQ);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // this CTA's tiles: local numbers z in [0, n), mapped to the chunk's tiles by TileRuns
  const int n = run_pref[p.nph];
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(p.status, MSA_ERR_TIMEOUT);
  };

  // Each register re-allocation sits at the top of its warpgroups' branch
  // (one instruction for all warps of a warpgroup) so that the compiler
  // budgets each branch with its own register count.
  if (warp < kEpiWarp0) {
  tc::regs_dec<kProdRegs>();
  if (warp < kLoadWarp || warp == kGatherWarpHi) {
    // ------------------------------ query-row gather ------------------------------
    // Gather warp gw (warps 0, 1, 2, 6) takes tiles z = gw, gw + 4, ... into
    // ring slot gw, so a warp has at most one tile in flight. Lane l gathers
    // rows [4 l, 4 l + 4) with one four-row TMA gather per 64-column half
    // into the 128B-swizzled K-major layout (the swizzle is address-based);
    // the bytes are counted on the slot's barrier with the warp's arrival. A
    // lane loads its rows' entries itself, one of its tiles ahead (one load
    // when the rows share an entry, as they do when the heads per group are a
    // multiple of 4). Rows of padding entries read the chunk's first query
    // (finite values; their outputs are never read).
    const int gw = warp < kLoadWarp ? warp : 3;
    static_assert(kRows == 32 * 4, "one lane per four rows");
    const int per_tile = kRows / p.hpg;
    const bool one_entry = p.hpg % 4 == 0;  // rows 4 l .. 4 l + 3 belong to one entry
    int4 tl = make_int4(0, 0, 0, 0);
    int ev[4];  // the entries of this lane's four rows (-1 past the tile's count)
    TileRuns runs{run_lo, run_pref};
    const uint64_t pol_q = tc::policy_evict_last();  // the phase's query rows are reused by every CTA
    auto fetch = [&](int z) {  // independent loads: tile zt's entries start at zt * per_tile
      const int zt = runs.at(z);
      tl = p.tiles[zt];
      const int* ent = p.entries + int64_t(zt) * per_tile;
      if (one_entry) {
        const int e = lane * 4 / p.hpg;
        ev[0] = ev[1] = ev[2] = ev[3] = e < per_tile ? ent[e] : -1;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = (lane * 4 + j) / p.hpg;
          ev[j] = e < per_tile ? ent[e] : -1;
        }
      }
    };
    if (gw < n) fetch(gw);
    int last = -1;  // the last tile this warp issued
    for (int z = gw; z < n; z += kRing) {
      if (!tc::mbar_wait(&q_empty[gw], ((z / kRing) & 1) ^ 1, abort_flag)) {
        fail();
        break;
      }
      const int g = tl.x / p.nblk;
      int rows[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = lane * 4 + j;
        const int il = row / p.hpg < tl.z && ev[j] >= 0 ? (ev[j] >> 6) : 0;
        rows[j] = (p.b * p.Nq + p.c0 + il) * p.Hq + g * p.hpg + row % p.hpg;
      }
      if (lane == 0) tc::mbar_arrive_expect_tx(&q_full[gw], uint32_t(kRows) * D * 2);
      __syncwarp();
      {
        uint8_t* dst = ring + gw * kSlot + lane * 4 * 128;
#pragma unroll
        for (int hf = 0; hf < NH; ++hf)
          tc::tma_gather4_hint(dst + hf * (kRows * 128), &tmQ, &q_full[gw], hf * 64, rows[0], rows[1], rows[2],
                               rows[3], pol_q);
      }
      last = z;
      if (z + kRing < n) fetch(z + kRing);
    }
    // drain after an abort: no gather may still be landing in shared memory
    // when the CTA exits (the slot's earlier tiles were consumed before this
    // one could be issued; in a full run the issuers consumed every tile)
    int zero = 0;
    if (*abort_flag && lane == 0 && last >= 0) tc::mbar_wait(&q_full[gw], (last / kRing) & 1, &zero);
  } else if (warp == kLoadWarp) {
    // ------------------------------ K/V loads ------------------------------
    // Key blocks are numbered in the order this CTA meets them (bi = 0, 1,
    // ...); block bi's K goes to K buffer bi & 1, its V to V buffer bi % NV.
    // A block is loaded as soon as both issuers have released the block that
    // used its buffers before, so K runs a block ahead (and V too with two V
    // buffers). The walk visits each block's first tile: from there the
    // next block starts rec.w tiles on in the same run, or opens the next run.
    if (lane == 0) {
      const uint64_t pol_kv = tc::policy_evict_first();  // each block's K/V is read by one or two CTAs
      int kl = 0, vl = 0;  // K / V loads issued
      bool alive = true;
      if (p.inject_timeout && !tc::mbar_wait_for(never_bar, 0, abort_flag, tc::kInjectedWaitCycles)) {
        fail();
        alive = false;
      }
      TileRuns runs{run_lo, run_pref};
      for (int z = 0, bi = 0; z < n && alive; ++bi) {
        const int zg = runs.at(z);
        const int e_run = runs.run_end(z);
        const int4 rec = p.tiles[zg];
        const int g = rec.x / p.nblk, t = rec.x % p.nblk;
        const int kb = bi & 1, vb = bi % NV;
        if (bi >= 2 && !tc::mbar_wait(&k_empty[kb], ((bi >> 1) - 1) & 1, abort_flag)) {
          fail();
          break;
        }
        tc::mbar_arrive_expect_tx(&k_full[kb], kKBytes);
#pragma unroll
        for (int h = 0; h < NH; ++h)
          tc::tma_load_4d_hint(k_buf + kb * kKBytes + h * kKVHalf, &tmK, &k_full[kb], h * 64, g, t * BS, p.b,
                               pol_kv);
        kl = bi + 1;
        if (bi >= NV && !tc::mbar_wait(&v_empty[vb], ((bi / NV) - 1) & 1, abort_flag)) {
          fail();
          break;
        }
        tc::mbar_arrive_expect_tx(&v_full[vb], kKBytes);
#pragma unroll
        for (int h = 0; h < NH; ++h)
          tc::tma_load_4d_hint(v_buf + vb * kKBytes + h * kKVHalf, &tmV, &v_full[vb], h * 64, g, t * BS, p.b,
                               pol_kv);
        vl = bi + 1;
        if (rec.w < 1) {  // a malformed tile record: stop rather than walk in place
          set_status(p.status, MSA_ERR_BOUNDS);
          *abort_flag = 1;
          break;
        }
        z = z + rec.w < e_run ? z + rec.w : e_run;
      }
      // no K or V copy may still be landing when the CTA exits: the last load into each buffer
      int zero = 0;
      for (int b2 = kl - 1; b2 >= 0 && b2 >= kl - 2; --b2) tc::mbar_wait(&k_full[b2 & 1], (b2 >> 1) & 1, &zero);
      for (int b2 = vl - 1; b2 >= 0 && b2 >= vl - NV; --b2) tc::mbar_wait(&v_full[b2 % NV], (b2 / NV) & 1, &zero);
    }
  } else if (warp < kIssueWarp0 + 2) {
    // ------------------------------- MMA issuers -------------------------------
    // Issuer w (one thread) issues QK^T and PV of the tiles z = w, w + 2, ...
    // (softmax warpgroup w, TMEM set w): QK(z), then PV(z) once P(z) is
    // ready, then QK(z + 2), which overwrites S(z) = P(z) after PV(z) has
    // read it (one thread's MMAs run in issue order). Both issuers walk every
    // tile record to number the key blocks; at each block change each
    // releases the block it leaves (K and V buffers, two arrivals each: one
    // per issuer, whether or not it had tiles there), after its K and V have
    // landed.
    const int w = warp - kIssueWarp0;
    if (lane == 0) {
      const uint32_t ring_lo0 = tc::smem_desc_lo(tc::smem_u32(ring), 16);
      const uint32_t k_lo0 = tc::smem_desc_lo(tc::smem_u32(k_buf), 16);
      const uint32_t v_lo0 = tc::smem_desc_lo(tc::smem_u32(v_buf), kKVHalf);
      const uint32_t t_s = tmem + uint32_t(w) * 256u;  // this issuer's TMEM set: S at t_s, O at t_s + 128
      int kw = 0, vw = 0;  // blocks whose K / V this issuer has waited for
      // the lookahead cursor: local tile za is chunk tile zga of run ra (which
      // ends at local enda); the bins of tiles z + 1 and z + 2 are in flight
      int ra = 0;
      while (ra < p.nph && run_pref[ra + 1] == 0) ++ra;
      int za = 0, zga = n > 0 ? run_lo[ra] : 0, enda = n > 0 ? run_pref[ra + 1] : 0;
      auto advance = [&]() {  // za -> za + 1 (< n)
        ++za;
        if (za == enda) {  // opens the next non-empty run
          do ++ra;
          while (run_pref[ra + 1] == za);
          zga = run_lo[ra];
          enda = run_pref[ra + 1];
        } else {
          ++zga;
        }
      };
      int bin_n1 = n > 0 ? p.tiles[zga].x : -1, bin_n2 = -1;
      if (n > 1) {
        advance();
        bin_n2 = p.tiles[zga].x;
      }
      // The walk over the tile records numbers the key blocks; blocks left
      // on the way are released once this issuer's MMAs on them are issued.
      int prev_bin = -1, bi = -1;
      int zw = 0;                        // the next tile to walk
      int rel0 = 0, rel1 = 0, nrel = 0;  // blocks left during the walk (at most two), to release
      auto walk_to = [&](int zt) {       // walk up to tile zt: bi is then its block
        while (zw <= zt && zw < n) {
          const int bin = bin_n1;
          bin_n1 = bin_n2;
          if (zw + 2 < n) {
            advance();
            bin_n2 = p.tiles[zga].x;
          }
          if (bin != prev_bin) {  // a new key block
            if (bi >= 0) {
              if (nrel == 0)
                rel0 = bi;
              else
                rel1 = bi;
              ++nrel;
            }
            ++bi;
            prev_bin = bin;
          }
          ++zw;
        }
      };
      // A block is released only once its K and V have been seen to land
      // (waited for here if this issuer had no tile in it): they were loaded
      // after both issuers released the block before it in the same buffers,
      // so one issuer's releases cannot run a buffer phase ahead of the
      // other's.
      auto release = [&]() -> bool {
        for (int i = 0; i < nrel; ++i) {
          const int b = i == 0 ? rel0 : rel1;
          if ((kw <= b && !tc::mbar_wait(&k_full[b & 1], (b >> 1) & 1, abort_flag)) ||
              (vw <= b && !tc::mbar_wait(&v_full[b % NV], (b / NV) & 1, abort_flag)))
            return false;
          if (kw <= b) kw = b + 1;
          if (vw <= b) vw = b + 1;
          tc::mma_commit(&k_empty[b & 1]);
          tc::mma_commit(&v_empty[b % NV]);
        }
        nrel = 0;
        return true;
      };
      // QK^T of tile z (block bz) into S buffer (z >> 1) & 1
      auto issue_qk = [&](int z, int bz) -> bool {
        const int rs = z & (kRing - 1);
        if (kw <= bz) {  // this issuer's first tile in the block: its K must have landed
          if (!tc::mbar_wait(&k_full[bz & 1], (bz >> 1) & 1, abort_flag)) return false;
          kw = bz + 1;
        }
        if (!tc::mbar_wait(&q_full[rs], (z / kRing) & 1, abort_flag)) return false;
        tc::fence_after_sync();
        const uint32_t q_lo = ring_lo0 + uint32_t(rs) * (kSlot >> 4);
        const uint32_t k_lo = k_lo0 + uint32_t(bz & 1) * (kKBytes >> 4);
        const int sb = (z >> 1) & 1;
        const uint32_t d = t_s + uint32_t(sb * BS);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // 16 columns = 32 bytes along the swizzled 128-byte rows
          tc::mma_f16_ss_lo<kDescHi>(d, q_lo + (((kk >> 2) * (kRows * 128) + off) >> 4),
                                     k_lo + (((kk >> 2) * kKVHalf + off) >> 4), kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&s_full[w * 2 + sb]);
        tc::mma_commit(&q_empty[rs]);  // the gathered Q tile is consumed
        return true;
      };
      // PV of tile z (block bz): P(z) in S buffer (z >> 1) & 1, O of this warpgroup
      auto issue_pv = [&](int z, int bz) -> bool {
        const int vb = bz % NV;
        if (vw <= bz) {  // the block's first PV here: its V must have landed
          if (!tc::mbar_wait(&v_full[vb], (bz / NV) & 1, abort_flag)) return false;
          vw = bz + 1;
        }
        if (!tc::mbar_wait(&p_full[w], (z >> 1) & 1, abort_flag)) return false;
        tc::fence_after_sync();
        const uint32_t v_lo = v_lo0 + uint32_t(vb) * (kKBytes >> 4);
        const uint32_t a = t_s + uint32_t(((z >> 1) & 1) * BS);
#pragma unroll
        for (int kk = 0; kk < BS / 16; ++kk) {
          // P (bf16 pairs packed per 32-bit column) sits where S was: 16 keys = 8 columns
          tc::mma_f16_ts_lo<kDescHi>(t_s + 128u, a + uint32_t(kk) * 8u, v_lo + uint32_t(kk * 16 * 128 >> 4), kIdescPV,
                                     kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&o_full[w]);
        return true;
      };
      // Order: QK(z + 2) goes ahead of PV(z) (the other S buffer), so S(z + 2)
      // is ready when the softmax finishes tile z; PV(z) then QK(z + 4)
      // keeps P(z) read before it is overwritten. Tile z + 2's K buffer must
      // not wait on a release that only follows PV(z): a block two or more
      // ahead takes the order PV(z), releases, QK(z + 2).
      bool alive = true;
      walk_to(w);
      int bz = bi;
      if (!release() || (w < n && !issue_qk(w, bz))) {
        fail();
        alive = false;
      }
      for (int z = w; z < n && alive; z += 2) {
        int bz2 = -1;
        bool early = false;
        if (z + 2 < n) {
          walk_to(z + 2);
          bz2 = bi;
          early = bz2 <= bz + 1;
          if (early && !issue_qk(z + 2, bz2)) {
            fail();
            break;
          }
        }
        if (!issue_pv(z, bz) || !release() || (z + 2 < n && !early && !issue_qk(z + 2, bz2))) {
          fail();
          break;
        }
        bz = bz2;
      }
      // every issued MMA completes before TMEM is released
      int zero = 0;
      tc::mma_commit(&done_bar[w]);
      tc::mbar_wait(&done_bar[w], 0, &zero);
    }
  }  // warp 7: idle
  } else {
    tc::regs_inc<kSoftRegs>();
    // --------------------------- softmax and partial store ---------------------------
    // Warpgroups 2 and 3 take alternate tiles (TMEM set w = z & 1): the whole
    // S row of a thread's TMEM lane in registers, causal mask in the local
    // block, exact softmax with unnormalised probabilities as P (bf16 pairs
    // written back over S for the PV MMA), the exponent arguments and the row
    // sum on paired fp32 instructions, and the row's log-sum-exp stored for
    // the combine. Then, while the tensor core computes PV(z) and QK(z + 2),
    // O(z) is read from TMEM, divided by the row sum and stored as the tile's
    // bf16 partial: 16-byte chunk c of row r of tile zg at
    // part_o[(zg * D/8 + c) * 128 + r], so each warp store instruction writes
    // 32 consecutive rows' chunk (512 contiguous bytes). PV(z + 2), which
    // overwrites O, waits for P(z + 2), written after O(z) was read.
    const int w = (warp - kEpiWarp0) >> 2;         // warpgroup: tiles z with z % 2 == w
    const int quarter = warp & 3;                  // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;             // tile row
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const SeqView sv = seq_view(p.q_offset, p.kv_len, p.b, p.Nq, p.Nk, false);
    TileRuns runs{run_lo, run_pref};
    const uint64_t pol_part = tc::policy_evict_first();  // partials are read back once, by the combine
    const uint32_t t_wg = tmem + lane_base + uint32_t(w) * 256u;  // this warpgroup's TMEM set (own lanes)
    // a tile's metadata straight from global memory (the Q ring slot is
    // recycled as soon as QK^T has consumed it), loaded one tile ahead
    int zg_n = 0, e_n = -1;
    int4 tl_n = make_int4(0, 0, 0, 0);
    auto meta = [&](int z) {
      zg_n = runs.at(z);
      tl_n = p.tiles[zg_n];
      e_n = p.entries[int64_t(zg_n) * (kRows / p.hpg) + r / p.hpg];
    };
    if (w < n) meta(w);
    for (int z = w; z < n; z += 2) {
      const int zg = zg_n;
      const int4 tl = tl_n;
      const int ent = r / p.hpg < tl.z ? e_n : -1;
      const int sb = (z >> 1) & 1;  // S buffer of this tile
      const uint32_t s_addr = t_wg + uint32_t(sb * BS);
      if (!tc::mbar_wait(&s_full[w * 2 + sb], (z >> 2) & 1, abort_flag)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      if (z + 2 < n) meta(z + 2);  // in flight during this tile
      const int bin = tl.x;
      const bool valid = ent >= 0;
      const int t = bin % p.nblk;
      const int il = ent >> 6;
      const int pos = sv.q0 + p.c0 + il;
      const int nvalid = valid ? min(BS, pos - t * BS + 1) : BS;  // keys j <= pos inside the block
      const bool full = nvalid >= BS;  // all keys visible (every block but the local one)
      float inv;
      {
        // the whole S row in registers: one TMEM round trip; each 32-column
        // load also returns the maximum of its columns
        uint32_t v[BS];
        float m32[BS / 32];
#pragma unroll
        for (int c = 0; c < BS / 32; ++c) m32[c] = tc::tmem_ld_max_32x32b_x32(s_addr + c * 32, v + c * 32);
        tc::tmem_ld_wait();
        float mx = m32[0];
#pragma unroll
        for (int c = 1; c < BS / 32; ++c) mx = fmaxf(mx, m32[c]);
        if (!full) {  // the local block: the row maximum over its visible keys only
#pragma unroll
          for (int j = 0; j < BS; ++j)
            if (j >= nvalid) v[j] = __float_as_uint(-INFINITY);  // exp2(-inf) = 0 below
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int j = 0; j < BS; j += 2)
            m4[(j >> 1) & 3] = tc::fmax3(m4[(j >> 1) & 3], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        // probabilities, 32 keys at a time: packed to bf16 pairs and written
        // back over S in TMEM at once (the PV MMA reads its A operand from
        // there: keys 2c (low half) and 2c+1 (high half) in column c), their
        // sum in fp32, two keys per instruction
        const float mneg = -mx * p.scale_log2;
        uint64_t l2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
        for (int c0 = 0; c0 < BS / 32; ++c0) {
          uint32_t* pk = v + c0 * 32;  // the packed pairs reuse the chunk's first 16 registers
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float p0 = ex2(fmaf(__uint_as_float(v[c0 * 32 + j]), p.scale_log2, mneg));
            const float p1 = ex2(fmaf(__uint_as_float(v[c0 * 32 + j + 1]), p.scale_log2, mneg));
            l2[(j >> 1) & 1] = add_f32x2(l2[(j >> 1) & 1], f32x2(p0, p1));
            pk[j >> 1] = pack_bf16(p0, p1);
          }
          tc::tmem_st_32x32b_x16(s_addr + c0 * 16, pk);
        }
        float la, lb, lc, ld;
        unpack_f32x2(l2[0], la, lb);
        unpack_f32x2(l2[1], lc, ld);
        const float l = (la + lb) + (lc + ld);
        inv = l > 0.f ? 1.f / l : 0.f;
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&p_full[w]);
        tc::st_f32_hint(p.part_lse + int64_t(zg) * kRows + r, valid ? mx * p.scale + logf(l) : 0.f, pol_part);
      }
      // O(z) = P(z) V as the tile's partial, scaled by 1 / row sum
      if (!tc::mbar_wait(&o_full[w], (z >> 1) & 1, abort_flag)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      const uint64_t inv2 = f32x2(inv, inv);
      uint4* dst = p.part_o + int64_t(zg) * (D / 8) * kRows + r;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tc::tmem_ld_32x32b_x32(t_wg + 128u + c0, ov);
        tc::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 o;
          o.x = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 0], ov[c * 8 + 1]), inv2));
          o.y = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 2], ov[c * 8 + 3]), inv2));
          o.z = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 4], ov[c * 8 + 5]), inv2));
          o.w = pack_bf16x2(mul_f32x2(f32x2_bits(ov[c * 8 + 6], ov[c * 8 + 7]), inv2));
          tc::st_v4_hint(dst + (c0 / 8 + c) * kRows, o, pol_part);
        }
      }
      // (the next tile's P store, which lets PV overwrite O, follows these loads in program order)
      tc::fence_before_sync();
    }
  }

  __syncthreads();
  if (warp == kLoadWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// combine: persistent warps, each taking (query, group) items in a strided
// loop. A slot's partials of the group's heads are hpg consecutive partial
// rows (found through the reverse map), stored chunk-major: 16-byte chunk c
// of row r in tile zg at ((zg * D/8 + c) * 128 + r). Lane vector vi takes
// head vi % hpg and chunk vi / hpg, so neighbouring lanes read neighbouring
// rows of one chunk; hpg divides 32, so every vector of a lane has the head
// h = lane % hpg. Each lane owns NU vectors.
// Items run token-major (item = query * G + group) or, with gmajor, group-
// major (item = group * cq + query): with many slots per item (K > 16) the
// slots of concurrent items then lie in one group's share of the partials,
// which keeps the combine's scattered row reads within fewer memory pages
// (at K 64, 128K tokens: 15.4 -> 12.6 ms per step, and no longer slower
// with larger query chunks). Per item: the valid slots (slot order) and their
// lse values go to the warp's shared-memory area; each lane forms its head's merge weights
// w_s = exp(lse_s - max) / sum_s exp(lse_s - max), then accumulates
// sum_s w_s * partial_s in slot order with a batch of slots' loads in flight.
// Weights known up front need no running rescale, which keeps the register
// count low enough for several CTAs per SM (more loads in flight). The next
// item's selection and reverse-map rows are loaded while the current item's
// partials are in flight. Deterministic; no atomics on any output.
// ---------------------------------------------------------------------------
constexpr int kCmbWarps = 8;
inline size_t combine_smem_bytes(int K, int hpg) { return size_t(kCmbWarps) * (2 * K + K * hpg) * 4; }

template <int NU>
__global__ void __launch_bounds__(256, NU <= 2 ? 2 : 1) attn_combine_kernel(
    const int32_t* __restrict__ sel, const int32_t* __restrict__ q_offset, const int32_t* __restrict__ kv_len,
    const uint4* __restrict__ part_o, const float* __restrict__ part_lse, const int* __restrict__ rev, int b,
    int Nq, int Nk, int Hq, int G, int K, int Bs, int nblk, int D, int c0, int cq, int gmajor,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int kBatch = NU <= 2 ? 8 : (NU == 4 ? 4 : 2);  // slots whose loads are in flight together
  extern __shared__ int cmb_smem[];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int hpg = Hq / G;
  int* slot_e = cmb_smem + wl * (2 * K + K * hpg);                     // [2][K] valid slots' entries
  float* lse_s = reinterpret_cast<float*>(slot_e + 2 * K);             // [K][hpg] their lse values
  const int64_t nitems = int64_t(cq) * G;
  const int64_t stride = int64_t(gridDim.x) * kCmbWarps;
  const int nvec = hpg * D / 8;
  const int h = lane % hpg;  // the head of every vector of this lane
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  int voff[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const int vi = lane + 32 * u;
    voff[u] = vi < nvec ? (vi / hpg) * 128 + h : 0;  // chunk-major offset from the slot's first row
  }
  // an item's selection and reverse-map entries for slots lane and lane + 32
  int s_t[2], s_e[2];
  auto meta_load = [&](int64_t it) {
    const int il = gmajor ? int(it % cq) : int(it / G), g = gmajor ? int(it / cq) : int(it % G);
    const int32_t* srow = sel + ((int64_t(b) * Nq + c0 + il) * G + g) * K;
    const int* rv = rev + (int64_t(il) * G + g) * K;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int k = lane + 32 * x;
      s_t[x] = k < K ? srow[k] : -1;
      s_e[x] = k < K ? rv[k] : 0;
    }
  };
  // valid slots in slot order, as partial-row entries, into slot_e[buf]
  auto meta_finish = [&](int64_t it, int buf) {
    const int pos = sv.q0 + c0 + (gmajor ? int(it % cq) : int(it / G));
    int nv = 0;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int k = lane + 32 * x;
      const bool ok = k < K && sv.ok && entry_valid(s_t[x], pos, Bs, nblk);
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (ok) slot_e[buf * K + nv + __popc(bal & ((1u << lane) - 1u))] = s_e[x];
      nv += __popc(bal);
    }
    __syncwarp();
    return nv;
  };
  int64_t item = int64_t(blockIdx.x) * kCmbWarps + wl;
  int buf = 0, nvalid = 0;
  if (item < nitems) {
    meta_load(item);
    nvalid = meta_finish(item, buf);
  }
  for (; item < nitems; item += stride, buf ^= 1) {
    const int64_t next = item + stride;
    if (next < nitems) meta_load(next);
    const int il = gmajor ? int(item % cq) : int(item / G), g = gmajor ? int(item / cq) : int(item % G);
    const int i = c0 + il;
    const int* se = slot_e + buf * K;
    // the slots' lse values of every head of the group
    for (int x = lane; x < nvalid * hpg; x += 32) lse_s[x] = part_lse[int64_t(se[x / hpg]) * hpg + x % hpg];
    __syncwarp();
    // this lane's head: maximum, then the sum of the weights (slot order)
    float mx = -INFINITY;
    for (int j = 0; j < nvalid; ++j) mx = fmaxf(mx, lse_s[j * hpg + h]);
    float den = 0.f;
    for (int j = 0; j < nvalid; ++j) den += expf(lse_s[j * hpg + h] - mx);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    float acc[NU][8];
#pragma unroll
    for (int u = 0; u < NU; ++u)
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[u][x] = 0.f;
    for (int j0 = 0; j0 < nvalid; j0 += kBatch) {
      uint4 raw[kBatch][NU];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const bool have = j0 + jj < nvalid;
        const int64_t R = have ? int64_t(se[j0 + jj]) * hpg : 0;  // the slot's first partial row
        const uint4* base = part_o + (R >> 7) * (D / 8) * 128 + (R & 127);
#pragma unroll
        for (int u = 0; u < NU; ++u)
          raw[jj][u] = (have && lane + 32 * u < nvec) ? base[voff[u]] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const float w = j0 + jj < nvalid ? expf(lse_s[(j0 + jj) * hpg + h] - mx) * inv : 0.f;
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const uint32_t w4[4] = {raw[jj][u].x, raw[jj][u].y, raw[jj][u].z, raw[jj][u].w};
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {  // bf16 -> fp32 is a 16-bit shift (low half = even column)
            acc[u][2 * q2] = fmaf(w, __uint_as_float(w4[q2] << 16), acc[u][2 * q2]);
            acc[u][2 * q2 + 1] = fmaf(w, __uint_as_float(w4[q2] & 0xffff0000u), acc[u][2 * q2 + 1]);
          }
        }
      }
    }
    __nv_bfloat16* dst = out + ((int64_t(b) * Nq + i) * Hq + g * hpg) * D;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int vi = lane + 32 * u;
      if (vi >= nvec) continue;
      uint4 o;
      o.x = pack_bf16(acc[u][0], acc[u][1]);
      o.y = pack_bf16(acc[u][2], acc[u][3]);
      o.z = pack_bf16(acc[u][4], acc[u][5]);
      o.w = pack_bf16(acc[u][6], acc[u][7]);
      *reinterpret_cast<uint4*>(dst + h * D + (vi / hpg) * 8) = o;
    }
    if (lse_out && lane < hpg)
      lse_out[(int64_t(b) * Nq + i) * Hq + g * hpg + lane] = den > 0.f ? mx + logf(den) : -INFINITY;
    __syncwarp();  // every lane is done with lse_s and slot_e[buf] before they are rewritten
    if (next < nitems) nvalid = meta_finish(next, buf ^ 1);
  }
}

// ---------------------------------------------------------------------------
// KL auxiliary forward (quant_prune_distill post 751, "Метод": the index
// branch is trained with the KL divergence to the head-averaged main-branch
// distribution; hyper.ai summary, "方法": the two are aligned over the selected
// tokens). Per (query, group):
//   KL = sum_j p_j log p_j - sum_j p_j s_j + logsumexp_j s_j
// over the selected tokens j, with p_j the main-branch attention probability
// averaged over the group's heads (exp(scale * q_h.k_j - lse_h), lse_h from
// the forward) and s_j the plain index score. Each selected block contributes
// four partial values per entry (the two sums, the block's index maximum and
// its exp-sum); kl_combine merges a row's slots.
//
// kl_tile: the attention's bins and tiles (one key block of one group, up to
// 128 / hpg entries per tile), on the same cost-balanced contiguous runs. Per
// tile: K and the index keys of the block (once per run of the bin), the
// tile's query rows and index queries, in padded shared-memory rows; both
// products on mma.sync with keys along M: S^T = K . Q^T (the group's heads of
// an entry are adjacent columns, so the head average is a pair sum and one
// shuffle) and I^T = IK . IQ^T.
// ---------------------------------------------------------------------------
struct KlParams {
  const __nv_bfloat16 *q, *k, *iq, *ik;  // q [B, Nq, Hq, D]; k [B, Nk, G, D]; iq [B, Nq, G, DI]; ik [B, Nk, DI]
  const float* lse;                      // [B, Nq, Hq] natural-log softmax normalisers of the forward
  const int* entries;
  const int4* tiles;
  const int* cta_start;
  const int32_t* q_offset;
  const int32_t* kv_len;
  float4* part;  // [tiles * 128 / hpg] (sum p log p, sum p s, index max, index exp-sum)
  int b, Nq, Nk, Hq, G, nblk, c0;
  float scale;
};

__device__ __forceinline__ void kl_ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void kl_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kKlThreads = 256;

template <int D, int DI, int BS, int HPG>
struct KlSmem {
  static constexpr int E = kRows / HPG;        // entries per tile
  static constexpr int KP = D + 8, IP = DI + 8;  // padded row lengths (bf16): 16-byte aligned, bank-conflict free
  static constexpr size_t kK = size_t(BS) * KP * 2, kIK = size_t(BS) * IP * 2, kQ = size_t(kRows) * KP * 2,
                          kIQ = size_t(E) * IP * 2, kLse = kRows * 4, kS = size_t(BS) * (E + 1) * 4, kEnt = E * 4,
                          kAcc = 2 * E * 4;
  static constexpr size_t kTotal = kK + kIK + kQ + kIQ + kLse + kS + kEnt + kAcc;
};

template <int D, int DI, int BS, int HPG>
__global__ void __launch_bounds__(kKlThreads, 1) kl_tile_kernel(const KlParams p) {
  using SM = KlSmem<D, DI, BS, HPG>;
  constexpr int E = SM::E, KP = SM::KP, IP = SM::IP;
  constexpr int MT = BS / 16;      // 16-key tiles of the block
  constexpr int NP = 8 / MT;       // warps sharing one key tile split the columns
  constexpr int NT = 16 / NP;      // 8-column tiles per warp (main product)
  constexpr int NTI = (E / 8 + NP - 1) / NP;  // 8-entry tiles per warp (index product)
  static_assert(HPG >= 2 && HPG <= 8, "head average of adjacent column pairs");
  extern __shared__ __align__(16) uint8_t kl_smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(kl_smem);
  __nv_bfloat16* IKs = reinterpret_cast<__nv_bfloat16*>(kl_smem + SM::kK);
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(kl_smem + SM::kK + SM::kIK);
  __nv_bfloat16* IQs = reinterpret_cast<__nv_bfloat16*>(kl_smem + SM::kK + SM::kIK + SM::kQ);
  float* lse_s = reinterpret_cast<float*>(kl_smem + SM::kK + SM::kIK + SM::kQ + SM::kIQ);
  float* Ss = lse_s + kRows;                                   // [BS][E + 1] index scores
  int* ents = reinterpret_cast<int*>(Ss + BS * (E + 1));        // [E]
  float* accA = reinterpret_cast<float*>(ents + E);             // [E] sum p log p
  float* accB = accA + E;                                       // [E] sum p s
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int mt = warp % MT, np = warp / MT;
  const int z0 = p.cta_start[blockIdx.x], z1 = p.cta_start[blockIdx.x + 1];
  const SeqView sv = seq_view(p.q_offset, p.kv_len, p.b, p.Nq, p.Nk, false);
  constexpr float kLog2eF = 1.4426950408889634f;
  int prev_bin = -1;
  for (int z = z0; z < z1; ++z) {
    const int4 tl = p.tiles[z];
    const int bin = tl.x, g = bin / p.nblk, t = bin % p.nblk;
    if (tid < E) ents[tid] = tid < tl.z ? p.entries[tl.y + tid] : -1;
    if (tid < E) accA[tid] = accB[tid] = 0.f;
    if (bin != prev_bin) {  // the block's keys and index keys, rows past the sequence zero-filled
      for (int x = tid; x < BS * (D / 8); x += kKlThreads) {
        const int r = x / (D / 8), c = x % (D / 8), j = t * BS + r;
        const bool in = j < p.Nk;
        const __nv_bfloat16* src = p.k + ((int64_t(p.b) * p.Nk + (in ? j : 0)) * p.G + g) * D + c * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(Ks + r * KP + c * 8)),
                     "l"(src), "r"(in ? 16u : 0u)
                     : "memory");
      }
      for (int x = tid; x < BS * (DI / 8); x += kKlThreads) {
        const int r = x / (DI / 8), c = x % (DI / 8), j = t * BS + r;
        const bool in = j < p.Nk;
        const __nv_bfloat16* src = p.ik + (int64_t(p.b) * p.Nk + (in ? j : 0)) * DI + c * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(IKs + r * IP + c * 8)),
                     "l"(src), "r"(in ? 16u : 0u)
                     : "memory");
      }
      prev_bin = bin;
    }
    __syncthreads();  // ents
    for (int x = tid; x < kRows * (D / 8); x += kKlThreads) {  // query rows: row = entry * HPG + head
      const int r = x / (D / 8), c = x % (D / 8), ent = ents[r / HPG];
      const int il = ent >= 0 ? (ent >> 6) : 0;
      const __nv_bfloat16* src = p.q + ((int64_t(p.b) * p.Nq + p.c0 + il) * p.Hq + g * HPG + r % HPG) * D + c * 8;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(Qs + r * KP + c * 8)), "l"(src),
                   "r"(ent >= 0 ? 16u : 0u)
                   : "memory");
    }
    for (int x = tid; x < E * (DI / 8); x += kKlThreads) {
      const int e = x / (DI / 8), c = x % (DI / 8), ent = ents[e];
      const int il = ent >= 0 ? (ent >> 6) : 0;
      const __nv_bfloat16* src = p.iq + ((int64_t(p.b) * p.Nq + p.c0 + il) * p.G + g) * DI + c * 8;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(IQs + e * IP + c * 8)), "l"(src),
                   "r"(ent >= 0 ? 16u : 0u)
                   : "memory");
    }
    if (tid < kRows) {
      const int ent = ents[tid / HPG];
      lse_s[tid] = ent >= 0 ? p.lse[(int64_t(p.b) * p.Nq + p.c0 + (ent >> 6)) * p.Hq + g * HPG + tid % HPG] : 0.f;
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // index scores I^T: keys [16 mt, +16) x entries, to shared memory
    {
      const int arow = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int ni = 0; ni < NTI; ++ni) {
        const int nt = np * NTI + ni;
        if (nt * 8 >= E) break;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < DI / 16; ++ks) {
          uint32_t a0, a1, a2, a3;
          kl_ldsm_x4(tc::smem_u32(IKs + arow * IP + ks * 16 + 8 * (lane >> 4)), a0, a1, a2, a3);
          const __nv_bfloat16* bq = IQs + (nt * 8 + gq) * IP + ks * 16 + 2 * tq;
          kl_mma(c, a0, a1, a2, a3, *reinterpret_cast<const uint32_t*>(bq), *reinterpret_cast<const uint32_t*>(bq + 8));
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) Ss[(mt * 16 + gq + 8 * (x >> 1)) * (E + 1) + nt * 8 + 2 * tq + (x & 1)] = c[x];
      }
    }
    // main scores S^T: keys [16 mt, +16) x columns [np * 8 NT, +8 NT)
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    {
      const int arow = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        kl_ldsm_x4(tc::smem_u32(Ks + arow * KP + ks * 16 + 8 * (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const __nv_bfloat16* bq = Qs + ((np * NT + n) * 8 + gq) * KP + ks * 16 + 2 * tq;
          kl_mma(acc[n], a0, a1, a2, a3, *reinterpret_cast<const uint32_t*>(bq),
                 *reinterpret_cast<const uint32_t*>(bq + 8));
        }
      }
    }
    __syncthreads();  // index scores complete
    // p_j per (key, entry): this lane holds heads 2 tq, 2 tq + 1 (mod HPG) of the
    // entries of its columns; the other heads sit in the lanes tq ^ 1, tq ^ 2
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int col = (np * NT + n) * 8 + 2 * tq;  // even column of this lane's pair
      const int e = col / HPG;
      const int ent = ents[e];
      const int pos = sv.q0 + p.c0 + (ent >> 6);
      float pa = 0.f, pb = 0.f;  // sums over the lane's two heads, for keys gq and gq + 8
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int key = t * BS + mt * 16 + gq + 8 * (x >> 1);
        const bool vis = ent >= 0 && sv.ok && key <= pos && key < sv.L;
        const float pr = vis ? ex2((acc[n][x] * p.scale - lse_s[col + (x & 1)]) * kLog2eF) : 0.f;
        if (x >> 1) pb += pr; else pa += pr;
      }
      // the entry's other heads: lanes differing in the low bits of tq
#pragma unroll
      for (int off = 1; off < HPG / 2; off <<= 1) {
        pa += __shfl_xor_sync(0xffffffffu, pa, off);
        pb += __shfl_xor_sync(0xffffffffu, pb, off);
      }
      pa *= 1.f / HPG;
      pb *= 1.f / HPG;
      float A = 0.f, Bv = 0.f;
      const int r0 = mt * 16 + gq;
      if (pa > 0.f) {
        A += pa * __logf(pa);
        Bv += pa * Ss[r0 * (E + 1) + e];
      }
      if (pb > 0.f) {
        A += pb * __logf(pb);
        Bv += pb * Ss[(r0 + 8) * (E + 1) + e];
      }
      // sum over the 8 key rows of this lane group (lanes with equal tq)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        A += __shfl_xor_sync(0xffffffffu, A, off);
        Bv += __shfl_xor_sync(0xffffffffu, Bv, off);
      }
      if (gq == 0 && (2 * tq) % HPG == 0) {  // one lane per entry
        atomicAdd(&accA[e], A);
        atomicAdd(&accB[e], Bv);
      }
    }
    __syncthreads();
    // the block's index log-sum-exp per entry over its visible keys
    if (tid < E && tid < tl.z) {
      const int ent = ents[tid];
      const int pos = sv.q0 + p.c0 + (ent >> 6);
      const int nk = min(BS, min(pos, sv.L - 1) - t * BS + 1);  // visible keys of the block (>= 1)
      float m = -INFINITY;
      for (int r = 0; r < nk; ++r) m = fmaxf(m, Ss[r * (E + 1) + tid]);
      float l = 0.f;
      for (int r = 0; r < nk; ++r) l += ex2((Ss[r * (E + 1) + tid] - m) * kLog2eF);
      p.part[int64_t(z) * E + tid] = make_float4(accA[tid], accB[tid], m, l);
    }
    __syncthreads();  // shared rows and sums are rewritten by the next tile
  }
}

// per (query, group): merge the slot partials of its selected blocks
__global__ void __launch_bounds__(256) kl_combine_kernel(const int32_t* __restrict__ sel,
                                                         const int32_t* __restrict__ q_offset,
                                                         const int32_t* __restrict__ kv_len,
                                                         const float4* __restrict__ part, const int* __restrict__ rev,
                                                         int b, int Nq, int Nk, int G, int K, int Bs, int nblk, int c0,
                                                         int cq, float* __restrict__ kl) {
  const int64_t item = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (item >= int64_t(cq) * G) return;
  const int il = int(item / G), g = int(item % G);
  const int i = c0 + il;
  const SeqView sv = seq_view(q_offset, kv_len, b, Nq, Nk, false);
  const int pos = sv.q0 + i;
  const int32_t* srow = sel + ((int64_t(b) * Nq + i) * G + g) * K;
  const int* rv = rev + (int64_t(il) * G + g) * K;
  float A = 0.f, Bv = 0.f, m = -INFINITY, l = 0.f;
  for (int k = 0; k < K; ++k) {
    if (!sv.ok || !entry_valid(srow[k], pos, Bs, nblk)) continue;
    const float4 v = part[rv[k]];
    A += v.x;
    Bv += v.y;
    const float mn = fmaxf(m, v.z);
    l = l * expf(m - mn) + v.w * expf(v.z - mn);
    m = mn;
  }
  kl[(int64_t(b) * Nq + i) * G + g] = l > 0.f ? A - Bv + m + logf(l) : 0.f;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side of the inversion (shared with the backward's translation unit)
// ---------------------------------------------------------------------------
static int g_sms = 0;
int sm_count() {
  if (g_sms == 0) {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kNumSMs;
    g_sms = n;
  }
  return g_sms;
}

static inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr int kInvRows = 1024;  // query rows per inversion CTA (one group each)

int chunk_tokens(int Nq, int Hq, int K, int d) {
  static int env = -1;
  if (env < 0) {
    const char* s = getenv("MSA_PREFILL_CHUNK");
    env = s ? atoi(s) : 0;
  }
  if (env > 0) return env < Nq ? env : Nq;
  // bound the partial buffers to ~6 GiB per 16 slots, in equal chunks (no
  // short tail chunk); at 128K tokens this gives three chunks at every K,
  // measured faster than five (the per-chunk inversion and grid tails) and
  // than one or two (attention's working set). At K 64 (Bs 32) three chunks
  // instead of eleven took the inversion from 5.1 to 2.0 ms per step.
  const size_t per_tok = size_t(Hq) * K * (size_t(d) * 2 + 4);
  size_t cap = ((size_t(6) << 30) * size_t(K > 16 ? K / 16 : 1)) / per_tok;
  if (cap < 1024) cap = 1024;
  const size_t nchunks = (size_t(Nq) + cap - 1) / cap;
  return int((size_t(Nq) + nchunks - 1) / nchunks);
}

KvoLayout kvo_layout(int Nq, int Hq, int G, int d, int Bs, int K, int Nk) {
  const int nblk = (Nk + Bs - 1) / Bs;
  const int cq = chunk_tokens(Nq, Hq, K, d);
  const size_t nbins = size_t(G) * nblk;
  const size_t max_entries = size_t(cq) * G * K;
  const int hpg = Hq / G;
  const size_t per_tile = size_t(kRows / hpg);
  const size_t max_tiles = max_entries / per_tile + nbins + 1;
  KvoLayout L;
  size_t o = kWsHeader;
  L.cnt = o;
  o += a256(nbins * 4);
  L.cursor = o;
  o += a256(nbins * 4);
  L.entry_off = o;
  o += a256((nbins + 1) * 4);
  L.tile_off = o;
  o += a256((nbins + 1) * 4);
  L.cost_off = o;
  o += a256((nbins + 1) * 4);
  L.cost_off2 = o;
  o += a256((nbins + 1) * 4);
  L.total = o;
  o += 256;
  L.cta_start = o;
  o += a256(size_t(kMaxGrid + 1) * 4);
  L.cta_seg = o;
  o += a256(size_t(kKvoMaxPhases) * (kMaxGrid + 1) * 4);
  L.hist = o;  // [G][count CTAs][nblk]: each inversion CTA's histogram
  o += a256(size_t(G) * ((cq + kInvRows - 1) / kInvRows) * nblk * 4);
  L.max_tiles = max_tiles;
  L.entries = o;
  o += a256(max_tiles * per_tile * 4);  // bins padded to whole tiles
  L.rev = o;
  o += a256(max_entries * 4);
  L.tiles = o;
  o += a256(max_tiles * 16);
  L.part_o = o;  // [tiles][d / 8 chunks][128 rows] x 8 bf16
  o += a256(max_tiles * kRows * size_t(d) * 2);
  L.part_lse = o;  // [tiles * 128 rows] fp32
  o += a256(max_tiles * kRows * 4);
  L.end = o;
  return L;
}

static size_t attn1_smem_bytes(int d, int Bs) {  // the single-issuer design
  const size_t kv = size_t(Bs) * d * 2 * (2 + attn_v_buffers(Bs));  // two K buffers, one or two V buffers
  const size_t slot = size_t(kRows) * d * 2;
  const size_t meta = size_t(kRing) * kRows * 4 + size_t(2 * kKvoMaxPhases + 1) * 4 + 16;
  return kv + kRing * slot + meta + (8 + 2 * kRing + 8 + 2) * 8 + 16;  // the base is 1024-byte aligned
}

static size_t attn2_smem_bytes(int d, int Bs) {  // the two-issuer design
  const size_t kv = size_t(Bs) * d * 2 * (2 + attn_v_buffers(Bs));  // two K buffers, one or two V buffers
  const size_t slot = size_t(kRows) * d * 2;
  const size_t runs = size_t(2 * kKvoMaxPhases + 1) * 4 + 16;  // run arrays, barrier alignment
  return kv + kRing * slot + runs + (8 + 2 * kRing + 10 + 1) * 8 + 16;  // the base is 1024-byte aligned
}

// blocks of 128 keys take the single-issuer design, smaller blocks the two-issuer one
static size_t attn_smem_bytes(int d, int Bs) { return Bs == 128 ? attn1_smem_bytes(d, Bs) : attn2_smem_bytes(d, Bs); }

// selection -> per-(group, block) entry lists, tiles and the persistent
// grid's cost split, for one query chunk [c0, c0 + cq) of sequence b
cudaError_t invert_chunk(const int32_t* sel, const int32_t* q_offset, const int32_t* kv_len, int b, int Nq, int Nk,
                         int G, int K, int Bs, int per_tile, int c0, int cq, int grid, char* w, const KvoLayout& L,
                         uint32_t* status, cudaStream_t stream) {
  const int nblk = (Nk + Bs - 1) / Bs, nbins = G * nblk, rows_per_cta = kInvRows;
  const size_t hist_smem = size_t(nblk) * 4 * 2;
  if (hist_smem > 200 * 1024) return cudaErrorInvalidValue;
  cudaError_t e;
  if (hist_smem > 48 * 1024) {
    e = cudaFuncSetAttribute(attn_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(hist_smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(hist_smem));
    if (e != cudaSuccess) return e;
  }
  int* cnt = reinterpret_cast<int*>(w + L.cnt);
  const dim3 igrid((cq + rows_per_cta - 1) / rows_per_cta, G);
  if ((e = cudaMemsetAsync(w + L.cnt, 0, L.entry_off - L.cnt, stream)) != cudaSuccess) return e;
  ProfScope pf("attn_invert", stream);
  int* hist_g = reinterpret_cast<int*>(w + L.hist);
  attn_count_kernel<<<igrid, 256, size_t(nblk) * 4, stream>>>(sel, q_offset, kv_len, b, Nq, Nk, G, K, Bs, nblk, c0,
                                                              cq, rows_per_cta, cnt, hist_g, status);
  attn_scan_kernel<<<1, 1024, 0, stream>>>(cnt, q_offset, b, nblk, nbins, per_tile, Bs, c0, cq, grid, G,
                                           kvo_phases(G), reinterpret_cast<int*>(w + L.entry_off),
                                           reinterpret_cast<int*>(w + L.tile_off),
                                           reinterpret_cast<int*>(w + L.cost_off),
                                           reinterpret_cast<int*>(w + L.cost_off2), reinterpret_cast<int*>(w + L.total),
                                           reinterpret_cast<int*>(w + L.cta_start),
                                           reinterpret_cast<int*>(w + L.cta_seg));
  attn_tiles_kernel<<<(nbins + 255) / 256, 256, 0, stream>>>(cnt, reinterpret_cast<int*>(w + L.entry_off),
                                                             reinterpret_cast<int*>(w + L.tile_off), nbins, per_tile,
                                                             reinterpret_cast<int4*>(w + L.tiles));
  attn_fill_kernel<<<igrid, 256, hist_smem, stream>>>(sel, q_offset, kv_len, b, Nq, Nk, G, K, Bs, nblk, c0, cq,
                                                      rows_per_cta, reinterpret_cast<int*>(w + L.entry_off), hist_g,
                                                      reinterpret_cast<int*>(w + L.cursor),
                                                      reinterpret_cast<int*>(w + L.entries),
                                                      reinterpret_cast<int*>(w + L.rev));
  return cudaGetLastError();
}

bool attn_kv_outer_supported(int dtype, int Hq, int Hkv, int d, int Bs, int K) {
  if (dtype != MSA_BF16 || (d != 64 && d != 128)) return false;
  if (Bs != 32 && Bs != 64 && Bs != 128) return false;
  if (K < 1 || K > kMaxK) return false;
  const int hpg = Hq / Hkv;
  if (hpg < 1 || hpg > 128 || (hpg & (hpg - 1)) != 0 || hpg * d > 2048) return false;
  return attn_smem_bytes(d, Bs) <= 227 * 1024;
}

size_t attn_kv_outer_ws_bytes(int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K) {
  return kvo_layout(Nq, Hq, Hkv, d, Bs, K, Nk).end;
}

cudaError_t launch_attn_kv_outer(const void* q, const void* k, const void* v, const int32_t* sel,
                                 const int32_t* q_offset, const int32_t* kv_len, int B, int Nq, int Nk, int Hq,
                                 int Hkv, int d, int Bs, int K, float scale, void* out, float* lse, void* ws,
                                 cudaStream_t stream) {
  const int G = Hkv, hpg = Hq / Hkv, nblk = (Nk + Bs - 1) / Bs;
  const int per_tile = kRows / hpg;
  const KvoLayout L = kvo_layout(Nq, Hq, G, d, Bs, K, Nk);
  char* w = static_cast<char*>(ws);
  uint32_t* status = &static_cast<WsHeader*>(ws)->status;
  int* entries = reinterpret_cast<int*>(w + L.entries);
  int* rev = reinterpret_cast<int*>(w + L.rev);
  int4* tiles = reinterpret_cast<int4*>(w + L.tiles);
  uint4* part_o = reinterpret_cast<uint4*>(w + L.part_o);
  float* part_lse = reinterpret_cast<float*>(w + L.part_lse);
  const int cq_max = chunk_tokens(Nq, Hq, K, d);

  CUtensorMap tmK, tmV;
  const uint64_t dims[4] = {uint64_t(d), uint64_t(Hkv), uint64_t(Nk), uint64_t(B)};
  const uint64_t strides[3] = {uint64_t(d) * 2, uint64_t(Hkv) * d * 2, uint64_t(Nk) * Hkv * d * 2};
  const uint32_t box[4] = {64, 1, uint32_t(Bs), 1};
  if (!make_tmap_bf16(&tmK, k, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tmV, v, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  CUtensorMap tmQ;  // query rows (b, i, head) x d, gathered four rows at a time (one-row box)
  {
    const uint64_t qdims[2] = {uint64_t(d), uint64_t(B) * Nq * Hq};
    const uint64_t qstr[1] = {uint64_t(d) * 2};
    const uint32_t qbox[2] = {64, 1};
    if (!make_tmap_bf16(&tmQ, q, 2, qdims, qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }

  const size_t smem = attn_smem_bytes(d, Bs);
  auto set_attr = [&](auto kern) {
    // the register split re-allocates exactly the launch allocation: a build
    // that launches with another register count must not run (the increase
    // would wait for registers that are never released)
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kAttnThreads) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  };
  cudaError_t e = cudaSuccess;

  AttnParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.part_o = part_o;
  prm.entries = entries;
  prm.tiles = tiles;
  prm.cta_seg = reinterpret_cast<const int*>(w + L.cta_seg);
  prm.q_offset = q_offset;
  prm.kv_len = kv_len;
  prm.part_lse = part_lse;
  prm.status = status;
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.Hq = Hq;
  prm.G = G;
  prm.Bs = Bs;
  prm.K = K;
  prm.nblk = nblk;
  prm.hpg = hpg;
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  const int grid = sm_count() < kMaxGrid ? sm_count() : kMaxGrid;
  prm.nph = kvo_phases(G);
  prm.grid = grid;
  prm.inject_timeout = debug_inject_timeout() ? 1 : 0;

  for (int b = 0; b < B; ++b) {
    for (int c0 = 0; c0 < Nq; c0 += cq_max) {
      const int cq = Nq - c0 < cq_max ? Nq - c0 : cq_max;
      if ((e = invert_chunk(sel, q_offset, kv_len, b, Nq, Nk, G, K, Bs, per_tile, c0, cq, grid, w, L, status,
                            stream)) != cudaSuccess)
        return e;
      prm.b = b;
      prm.c0 = c0;
      {
        ProfScope pf("attn_kv_outer_tc", stream);
#define MSA_KVO(KERN)                                                                     \
  do {                                                                                    \
    auto kern = KERN;                                                                     \
    if ((e = set_attr(kern)) != cudaSuccess) return e;                                   \
    kern<<<grid, kAttnThreads, smem, stream>>>(tmK, tmV, tmQ, prm);                      \
  } while (0)
        // blocks of 128 keys: the single-issuer design; 64 and 32: the two-issuer design
        if (d == 128) {
          if (Bs == 128)
            MSA_KVO((attn_kv_outer_kernel<128, 128>));
          else if (Bs == 64)
            MSA_KVO((attn_kv_outer2_kernel<128, 64>));
          else
            MSA_KVO((attn_kv_outer2_kernel<128, 32>));
        } else {
          if (Bs == 128)
            MSA_KVO((attn_kv_outer_kernel<64, 128>));
          else if (Bs == 64)
            MSA_KVO((attn_kv_outer2_kernel<64, 64>));
          else
            MSA_KVO((attn_kv_outer2_kernel<64, 32>));
        }
#undef MSA_KVO
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      {
        ProfScope pf("attn_combine", stream);
        const int64_t items = int64_t(cq) * G;
        const int nvec = hpg * d / 8;
        __nv_bfloat16* o16 = static_cast<__nv_bfloat16*>(out);
        // persistent: as many CTAs as fit at once, each warp striding over items
#define MSA_CMB(NU_)                                                                                           \
  do {                                                                                                         \
    auto kern = attn_combine_kernel<NU_>;                                                                      \
    const size_t csm = combine_smem_bytes(K, hpg);                                                             \
    if (csm > 48 * 1024 &&                                                                                     \
        (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(csm))) != cudaSuccess)  \
      return e;                                                                                                \
    int per_sm = 0;                                                                                            \
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, csm) != cudaSuccess || per_sm < 1)   \
      per_sm = 1;                                                                                              \
    const int64_t need = (items + kCmbWarps - 1) / kCmbWarps;                                                  \
    const unsigned cgrid = unsigned(need < int64_t(per_sm) * grid ? need : int64_t(per_sm) * grid);            \
    kern<<<cgrid, 256, csm, stream>>>(sel, q_offset, kv_len, part_o, part_lse, rev, b, Nq, Nk, Hq, G, K, Bs, nblk, \
                                      d, c0, cq, K > 16 ? 1 : 0, o16, lse);                                    \
  } while (0)
        if (nvec <= 32)
          MSA_CMB(1);
        else if (nvec <= 64)
          MSA_CMB(2);
        else if (nvec <= 128)
          MSA_CMB(4);
        else
          MSA_CMB(8);
#undef MSA_CMB
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
    }
  }
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// KL auxiliary forward (see kl_tile_kernel)
// ---------------------------------------------------------------------------
bool kl_aux_supported(int dtype, int Hq, int Hkv, int d, int di, int Bs, int K) {
  if (dtype != MSA_BF16 || Hkv < 1 || Hq % Hkv != 0) return false;
  if (!((d == 128 && di == 64) || (d == 64 && di == 32))) return false;
  if (Bs != 32 && Bs != 64 && Bs != 128) return false;
  if (K < 1 || K > kMaxK) return false;
  const int hpg = Hq / Hkv;
  return hpg == 2 || hpg == 4 || hpg == 8;
}

size_t kl_aux_ws_bytes(int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K) {
  return kvo_layout(Nq, Hq, Hkv, d, Bs, K, Nk).end;  // the partials fit in the attention's partial area
}

cudaError_t launch_kl_aux(const void* q, const void* k, const void* iq, const void* ik, const int32_t* sel,
                          const float* lse, const int32_t* q_offset, const int32_t* kv_len, int B, int Nq, int Nk,
                          int Hq, int Hkv, int d, int di, int Bs, int K, float scale, float* kl, void* ws,
                          cudaStream_t stream) {
  const int G = Hkv, hpg = Hq / Hkv, nblk = (Nk + Bs - 1) / Bs;
  const int per_tile = kRows / hpg;
  const KvoLayout L = kvo_layout(Nq, Hq, G, d, Bs, K, Nk);
  char* w = static_cast<char*>(ws);
  uint32_t* status = &static_cast<WsHeader*>(ws)->status;
  const int cq_max = chunk_tokens(Nq, Hq, K, d);
  const int grid = sm_count() < kMaxGrid ? sm_count() : kMaxGrid;
  KlParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.iq = static_cast<const __nv_bfloat16*>(iq);
  prm.ik = static_cast<const __nv_bfloat16*>(ik);
  prm.lse = lse;
  prm.entries = reinterpret_cast<const int*>(w + L.entries);
  prm.tiles = reinterpret_cast<const int4*>(w + L.tiles);
  prm.cta_start = reinterpret_cast<const int*>(w + L.cta_start);
  prm.q_offset = q_offset;
  prm.kv_len = kv_len;
  prm.part = reinterpret_cast<float4*>(w + L.part_o);
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.Hq = Hq;
  prm.G = G;
  prm.nblk = nblk;
  prm.scale = scale;
  cudaError_t e;
  for (int b = 0; b < B; ++b) {
    for (int c0 = 0; c0 < Nq; c0 += cq_max) {
      const int cq = Nq - c0 < cq_max ? Nq - c0 : cq_max;
      if ((e = invert_chunk(sel, q_offset, kv_len, b, Nq, Nk, G, K, Bs, per_tile, c0, cq, grid, w, L, status,
                            stream)) != cudaSuccess)
        return e;
      prm.b = b;
      prm.c0 = c0;
      if (kl_tc_supported(d, di, Bs, hpg)) {
        ProfScope pf("kl_tile_tc", stream);
        KlTcArgs ka;
        ka.q = prm.q;
        ka.iq = prm.iq;
        ka.lse = lse;
        ka.entries = prm.entries;
        ka.tiles = prm.tiles;
        ka.cta_start = prm.cta_start;
        ka.q_offset = q_offset;
        ka.kv_len = kv_len;
        ka.part = prm.part;
        ka.status = status;
        ka.b = b;
        ka.Nq = Nq;
        ka.Nk = Nk;
        ka.Hq = Hq;
        ka.G = G;
        ka.nblk = nblk;
        ka.c0 = c0;
        ka.scale = scale;
        if ((e = launch_kl_tile_tc(ka, k, ik, B, Nk, Hkv, hpg, grid, stream)) != cudaSuccess) return e;
      } else {
        ProfScope pf("kl_tile", stream);
#define MSA_KL(D_, DI_, BS_, HPG_)                                                                            \
  do {                                                                                                        \
    auto kern = kl_tile_kernel<D_, DI_, BS_, HPG_>;                                                          \
    const size_t smem = KlSmem<D_, DI_, BS_, HPG_>::kTotal;                                                  \
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess) \
      return e;                                                                                               \
    kern<<<grid, kKlThreads, smem, stream>>>(prm);                                                           \
  } while (0)
#define MSA_KL_HPG(D_, DI_, BS_)  \
  do {                            \
    if (hpg == 2)                 \
      MSA_KL(D_, DI_, BS_, 2);    \
    else if (hpg == 4)            \
      MSA_KL(D_, DI_, BS_, 4);    \
    else                          \
      MSA_KL(D_, DI_, BS_, 8);    \
  } while (0)
#define MSA_KL_BS(D_, DI_)          \
  do {                              \
    if (Bs == 128)                  \
      MSA_KL_HPG(D_, DI_, 128);     \
    else if (Bs == 64)              \
      MSA_KL_HPG(D_, DI_, 64);      \
    else                            \
      MSA_KL_HPG(D_, DI_, 32);      \
  } while (0)
        if (d == 128)
          MSA_KL_BS(128, 64);
        else
          MSA_KL_BS(64, 32);
#undef MSA_KL_BS
#undef MSA_KL_HPG
#undef MSA_KL
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      {
        ProfScope pf("kl_combine", stream);
        const int64_t items = int64_t(cq) * G;
        kl_combine_kernel<<<unsigned((items + 255) / 256), 256, 0, stream>>>(
            sel, q_offset, kv_len, reinterpret_cast<const float4*>(w + L.part_o), reinterpret_cast<const int*>(w + L.rev),
            b, Nq, Nk, G, K, Bs, nblk, c0, cq, kl);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
    }
  }
  return cudaSuccess;
}

}  // namespace msa
