// Internal declarations shared by the MSA CUDA translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"

namespace msa {

constexpr int kNumSMs = 152;       // GB300: 2 dies x 76 SMs
constexpr size_t kWsHeader = 256;  // status word + counters, then op regions
constexpr int kMaxK = 64;
constexpr int kMaxBs = 1024;

// First 256 bytes of every workspace.
struct WsHeader {
  uint32_t status;        // sticky msa_status_t set by kernels
  uint32_t work_counter;  // persistent-grid work queue head (reset per launch)
  uint32_t reserved[62];
};

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
  atomicCAS(status, 0u, code);  // the first error wins
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Order-preserving map of a float to an unsigned 32-bit value (a larger float
// gives a larger value). -0 is folded onto +0 so that the two compare equal,
// as they do in floating point.
__device__ __forceinline__ uint32_t ord_f32(float m) {
  uint32_t u = __float_as_uint(m);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// A block maximum and its block id as one unsigned 64-bit key: a larger key
// means a larger maximum, and among equal maxima the lower block id.
__device__ __forceinline__ uint64_t rank_key(float m, int t) {
  return (uint64_t(ord_f32(m)) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(t));
}
__device__ __forceinline__ int rank_key_block(uint64_t key) { return int(0xFFFFFFFFu - uint32_t(key)); }

// Per-sequence position bounds, validated on the device.
struct SeqView {
  int q0;  // absolute position of query row 0
  int L;   // valid keys
  bool ok;
};
__device__ __forceinline__ SeqView seq_view(const int32_t* q_offset, const int32_t* kv_len, int b, int Nq, int Nk,
                                            bool decode) {
  SeqView s;
  s.L = kv_len ? kv_len[b] : Nk;
  s.q0 = decode ? s.L - 1 : (q_offset ? q_offset[b] : 0);
  s.ok = s.L >= 1 && s.L <= Nk && s.q0 >= 0 && s.q0 + Nq <= s.L;
  return s;
}

// Test hook (msa_debug_inject_timeout): attention kernels first make one
// bounded wait that runs out.
bool debug_inject_timeout();

// RAII bracket of one kernel launch with a CUDA event pair while profiling is
// on (msa_profile_begin / msa_profile_end); a no-op otherwise.
class ProfScope {
 public:
  ProfScope(const char* name, cudaStream_t stream);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  const char* name_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

// ---- KV-outer inversion (host side; kernels in attn_kv_outer_tc.cu) --------
// Per query chunk of one sequence: the selection inverted into per-(group,
// key block) bins of (query, slot) entries, padded to 128-row tiles (128 / hpg
// entries per tile), the tile list, the reverse map (query, group, slot) ->
// entry position, and a cost-balanced split of the tiles over a persistent
// grid. Used by the prefill attention, the KL pass and the backward.
constexpr int kKvoRows = 128;       // rows (entry x head) per tile
constexpr int kKvoMaxGrid = 1024;   // cta_start capacity
constexpr int kKvoMaxPhases = 16;   // forward attention: group ranges processed one after another
inline int kvo_phases(int G) { return G < kKvoMaxPhases ? G : kKvoMaxPhases; }
struct KvoLayout {
  size_t cnt, cursor, entry_off, tile_off, cost_off, cost_off2, total, cta_start, cta_seg, hist, entries, rev, tiles,
      part_o, part_lse, end;
  size_t max_tiles;
};
// A CTA's tiles under the per-phase split (cta_seg [nph][grid + 1]): run r
// holds its local tiles [pref[r], pref[r+1]), which are the chunk's tiles
// lo[r] + (z - pref[r]). A warp role that walks its local tile numbers in
// increasing order keeps its run between lookups.
struct TileRuns {
  const int* lo;
  const int* pref;
  int r = 0;
  __device__ __forceinline__ int at(int z) {
    while (z >= pref[r + 1]) ++r;
    return lo[r] + (z - pref[r]);
  }
  // the first local tile after the run that holds z
  __device__ __forceinline__ int run_end(int z) {
    while (z >= pref[r + 1]) ++r;
    return pref[r + 1];
  }
};
// One thread fills lo[nph] and pref[nph + 1] (shared memory) for this CTA.
__device__ __forceinline__ void load_tile_runs(const int* cta_seg, int nph, int grid, int* lo, int* pref) {
  int acc = 0;
  pref[0] = 0;
  for (int ph = 0; ph < nph; ++ph) {
    const int* seg = cta_seg + ph * (grid + 1);
    const int a = seg[blockIdx.x], b = seg[blockIdx.x + 1];
    lo[ph] = a;
    acc += b - a;
    pref[ph + 1] = acc;
  }
}
// query tokens per chunk (equal chunks; the forward's bf16 partials stay under ~6 GiB)
int chunk_tokens(int Nq, int Hq, int K, int d);
KvoLayout kvo_layout(int Nq, int Hq, int G, int d, int Bs, int K, int Nk);
int sm_count();
// Fills the layout's inversion regions for queries [c0, c0 + cq) of sequence b.
cudaError_t invert_chunk(const int32_t* sel, const int32_t* q_offset, const int32_t* kv_len, int b, int Nq, int Nk,
                         int G, int K, int Bs, int per_tile, int c0, int cq, int grid, char* w, const KvoLayout& L,
                         uint32_t* status, cudaStream_t stream);

// Status of an empty index selection (B == 0 or Nq == 0), shared by the entry
// points that select: the other arguments are checked as for one row.
msa_status_t index_select_empty_status(int Nk, int G, int di, int Bs, int K, int dtype);

// ---- launchers (host) ------------------------------------------------------
// Index Branch, CUDA-core table path: block maxima for every visible block.
cudaError_t launch_index_blockmax_table(int dtype, const void* iq, const void* ik, const int32_t* q_offset,
                                        const int32_t* kv_len, int B, int Nq, int Nk, int G, int di, int Bs,
                                        float* table, uint32_t* status, cudaStream_t stream);
// Index Branch, fused tcgen05 path (bf16): scores + block max on the tensor
// cores. For K - 1 <= 15 the top-K runs in the same persistent kernel (no
// table); for larger K the kernel writes the candidate block maxima of a chunk
// of rows to a workspace table and a warp-per-row selection kernel follows,
// chunk after chunk.
bool index_fused_supported(int dtype, int Nq, int G, int di, int Bs, int K);
// Workspace bytes of the chunk table (0 when the top-K stays in the kernel).
size_t index_fused_table_bytes(int B, int Nq, int Nk, int G, int Bs, int K);
// fs = 1 keeps block 0 as well as the local block (K - 2 blocks ranked);
// table / table_bytes: the chunk table (index_fused_table_bytes of it)
cudaError_t launch_index_fused_tc(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len,
                                  int B, int Nq, int Nk, int G, int di, int Bs, int K, int fs, int32_t* sel,
                                  float* table, size_t table_bytes, uint32_t* status, cudaStream_t stream);
// Exact top-K over a block-max table (warp per row).
cudaError_t launch_topk_from_table(const float* table, const int32_t* q_offset, const int32_t* kv_len, int B, int Nq,
                                   int Nk, int G, int Bs, int K, int fs, int32_t* sel, uint32_t* status,
                                   cudaStream_t stream);
// Main Branch, prefill, KV-outer tcgen05 path (bf16).
bool attn_kv_outer_supported(int dtype, int Hq, int Hkv, int d, int Bs, int K);
size_t attn_kv_outer_ws_bytes(int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K);
cudaError_t launch_attn_kv_outer(const void* q, const void* k, const void* v, const int32_t* sel,
                                 const int32_t* q_offset, const int32_t* kv_len, int B, int Nq, int Nk, int Hq,
                                 int Hkv, int d, int Bs, int K, float scale, void* out, float* lse, void* ws,
                                 cudaStream_t stream);
// Index Branch for one query per sequence (decode): tcgen05 stream of the
// index-key cache into a [B, G, nblk] block-max table, then exact top-K.
bool decode_index_supported(int dtype, int B, int Nq, int G, int di, int Bs, int K);
size_t decode_index_ws_bytes(int B, int G, int Nk);
cudaError_t launch_decode_index(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len, int B,
                                int Lmax, int G, int Bs, int K, int fs, int32_t* sel, float* table, uint32_t* status,
                                cudaStream_t stream);
// Main Branch, decode: split over selected blocks + combine (bf16).
bool decode_attn_supported(int dtype, int Hq, int Hkv, int d, int Bs, int K);
size_t decode_ws_bytes(int B, int Hq, int Hkv, int d, int K);
cudaError_t launch_decode_attn(const void* q, const void* k_cache, const void* v_cache, const int32_t* sel,
                               const int32_t* kv_len, int B, int Lmax, int Hq, int Hkv, int d, int Bs, int K,
                               float scale, void* out, float* lse, void* scratch, uint32_t* status,
                               cudaStream_t stream);
// Main Branch, query-outer CUDA-core path (any dtype; prefill or decode).
// Streaming decode: append one token's k, v and index-key rows per sequence
// at kv_len[b], advance kv_len, write the token's position (or -1) to q_pos.
cudaError_t launch_decode_append(const void* k_new, const void* v_new, const void* ik_new, void* k_cache,
                                 void* v_cache, void* ik_cache, int32_t* kv_len, int32_t* q_pos, int B, int Lmax,
                                 int Hkv, int d, int di, int elem_bytes, uint32_t* status, cudaStream_t stream);
// KL auxiliary forward: KL(head-averaged main-branch distribution || index
// softmax) over each (row, group)'s selected tokens, on the KV-outer bins.
bool kl_aux_supported(int dtype, int Hq, int Hkv, int d, int di, int Bs, int K);
size_t kl_aux_ws_bytes(int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K);
cudaError_t launch_kl_aux(const void* q, const void* k, const void* iq, const void* ik, const int32_t* sel,
                          const float* lse, const int32_t* q_offset, const int32_t* kv_len, int B, int Nq, int Nk,
                          int Hq, int Hkv, int d, int di, int Bs, int K, float scale, float* kl, void* ws,
                          cudaStream_t stream);
// Main Branch backward (bf16): dq, dk, dv over the selected blocks on the
// KV-outer bins, from the forward's out and lse.
bool attn_backward_supported(int dtype, int Hq, int Hkv, int d, int Bs, int K);
size_t attn_backward_ws_bytes(int B, int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K);
cudaError_t launch_attn_backward(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                 const float* lse, const int32_t* sel, const int32_t* q_offset,
                                 const int32_t* kv_len, int B, int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K,
                                 float scale, void* dq, void* dk, void* dv, void* ws, cudaStream_t stream);
// KL auxiliary tile pass on tcgen05 (d 128, di 64, blocks of 128 keys): one
// launch over a chunk's tiles, writing the per-entry partials the combine reads.
struct KlTcArgs {
  const __nv_bfloat16 *q, *iq;  // q [B, Nq, Hq, 128]; iq [B, Nq, G, 64]
  const float* lse;             // [B, Nq, Hq]
  const int* entries;
  const int4* tiles;
  const int* cta_start;
  const int32_t* q_offset;
  const int32_t* kv_len;
  float4* part;  // [entry position] (sum p log p, sum p s, index max, index exp-sum)
  uint32_t* status;
  int b, Nq, Nk, Hq, G, nblk, c0;
  float scale;
};
bool kl_tc_supported(int d, int di, int Bs, int hpg);
cudaError_t launch_kl_tile_tc(const KlTcArgs& a, const void* k, const void* ik, int B, int Nk, int Hkv, int hpg,
                              int grid, cudaStream_t stream);
cudaError_t launch_attn_query_outer(int dtype, const void* q, const void* k, const void* v, const int32_t* sel,
                                    const int32_t* q_offset, const int32_t* kv_len, bool decode, int B, int Nq,
                                    int Nk, int Hq, int Hkv, int d, int Bs, int K, float scale, void* out, float* lse,
                                    uint32_t* status, cudaStream_t stream);

}  // namespace msa
