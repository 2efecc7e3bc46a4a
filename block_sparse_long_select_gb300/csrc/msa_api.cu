// C ABI of the MSA forward path: host-side validation, workspace planning and
// dispatch to the kernels. Every entry point is asynchronous on its stream.
#include <algorithm>
#include <cstring>

#include "msa_internal.cuh"

namespace msa {
namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool dtype_ok(int dtype) { return dtype == MSA_BF16 || dtype == MSA_FP32; }

// ---- Index Branch planning ---------------------------------------------------
struct IndexPlan {
  bool ok = false;
  bool fused = false;  // tcgen05 kernel when no block_max is requested
  msa_status_t err = MSA_ERR_INVALID_ARG;
  size_t table_off = 0, table_bytes = 0;  // table region inside ws (0 if none)
  size_t ws_bytes = 0;
};

IndexPlan plan_index(int B, int Nq, int Nk, int G, int di, int Bs, int K, int dtype, bool have_block_max) {
  IndexPlan p;
  if (B < 1 || Nq < 1 || Nk < 1 || G < 1 || di < 1 || Bs < 1 || K < 1 || !dtype_ok(dtype)) return p;
  if (Nq > Nk) return p;
  if (di != 32 && di != 64) {
    p.err = MSA_ERR_UNSUPPORTED;
    return p;
  }
  if (Bs > kMaxBs || K > kMaxK) {
    p.err = MSA_ERR_UNSUPPORTED;
    return p;
  }
  const int nblk = (Nk + Bs - 1) / Bs;
  size_t table = size_t(B) * Nq * G * nblk * sizeof(float);
  // the one-query (decode) path keeps 32-key sub-block maxima instead
  if (decode_index_supported(dtype, B, Nq, G, di, Bs, K)) table = std::max(table, decode_index_ws_bytes(B, G, Nk));
  p.fused = index_fused_supported(dtype, Nq, G, di, Bs, K);
  // the fused kernel's chunk table (large K only), else the full table
  if (p.fused) table = index_fused_table_bytes(B, Nq, Nk, G, Bs, K);
  p.table_off = kWsHeader;
  p.table_bytes = have_block_max ? 0 : align256(table);
  // size for the call without block_max
  p.ws_bytes = kWsHeader + align256(table);
  p.ok = true;
  p.err = MSA_OK;
  return p;
}

// ---- Main Branch planning ----------------------------------------------------
struct AttnPlan {
  bool ok = false;
  bool kv_outer = false;  // tcgen05 KV-outer kernel (bf16 prefill)
  bool split = false;     // split-over-blocks decode kernel (bf16 decode)
  msa_status_t err = MSA_ERR_INVALID_ARG;
  size_t ws_bytes = 0;
};

AttnPlan plan_attn(int B, int Nq, int Nk, int Hq, int Hkv, int d, int Bs, int K, int dtype, bool prefill) {
  AttnPlan p;
  if (B < 1 || Nq < 1 || Nk < 1 || Hq < 1 || Hkv < 1 || d < 1 || Bs < 1 || K < 1 || !dtype_ok(dtype)) return p;
  if (Hq % Hkv != 0 || Nq > Nk) return p;
  if ((d != 64 && d != 128) || Bs > kMaxBs || K > kMaxK) {
    p.err = MSA_ERR_UNSUPPORTED;
    return p;
  }
  // the KV-outer kernel addresses query rows (b, i, head) with 32-bit TMA coordinates
  p.kv_outer = prefill && attn_kv_outer_supported(dtype, Hq, Hkv, d, Bs, K) &&
               int64_t(B) * Nq * Hq < (int64_t(1) << 31);
  p.split = !prefill && decode_attn_supported(dtype, Hq, Hkv, d, Bs, K);
  p.ws_bytes = p.kv_outer ? attn_kv_outer_ws_bytes(Nq, Nk, Hq, Hkv, d, Bs, K)
                          : (p.split ? kWsHeader + decode_ws_bytes(B, Hq, Hkv, d, K) : kWsHeader);
  p.ok = true;
  p.err = MSA_OK;
  return p;
}

msa_status_t check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need) return MSA_ERR_WORKSPACE;
  return MSA_OK;
}

inline msa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

inline uint32_t* status_word(void* ws) { return &static_cast<WsHeader*>(ws)->status; }

// An empty batch: B == 0, or Nq == 0 for an entry point with query rows.
// Nothing is read or computed; the other arguments are still checked as for a
// batch of one row, so an unsupported configuration fails the same way.
inline bool empty_batch(int B, int Nq) { return B >= 0 && Nq >= 0 && (B == 0 || Nq == 0); }
inline int one_key_min(int Nk) { return Nk < 0 ? Nk : std::max(Nk, 1); }

// Streaming decode step: one workspace holds the status header, the new
// tokens' positions, the index scratch and the attention scratch.
struct StepPlan {
  bool ok = false;
  msa_status_t err = MSA_ERR_INVALID_ARG;
  IndexPlan ip;
  AttnPlan ap;
  size_t off_pos = 0, off_index = 0, off_attn = 0, ws_bytes = 0;
};

StepPlan plan_step(int B, int Lmax, int G, int Hq, int d, int di, int Bs, int K, int dtype) {
  StepPlan p;
  p.ip = plan_index(B, 1, Lmax, G, di, Bs, K, dtype, false);
  if (!p.ip.ok) {
    p.err = p.ip.err;
    return p;
  }
  p.ap = plan_attn(B, 1, Lmax, Hq, G, d, Bs, K, dtype, false);
  if (!p.ap.ok) {
    p.err = p.ap.err;
    return p;
  }
  p.off_pos = kWsHeader;
  p.off_index = p.off_pos + align256(size_t(B) * sizeof(int32_t));
  p.off_attn = p.off_index + align256(p.ip.ws_bytes - kWsHeader);
  p.ws_bytes = p.off_attn + (p.ap.ws_bytes - kWsHeader);
  p.ok = true;
  p.err = MSA_OK;
  return p;
}

}  // namespace

// Status of an empty index selection (B == 0 or Nq == 0): the other arguments
// are checked as for one row of one sequence.
msa_status_t index_select_empty_status(int Nk, int G, int di, int Bs, int K, int dtype) {
  const IndexPlan one = plan_index(1, 1, one_key_min(Nk), G, di, Bs, K, dtype, false);
  return one.ok ? MSA_OK : one.err;
}

}  // namespace msa

using namespace msa;

extern "C" size_t msa_workspace_size(int op, int B, int Nq, int Nk, int G, int Hq, int d, int di, int Bs, int K,
                                     int dtype) {
  const bool rowless = op == MSA_OP_DECODE || op == MSA_OP_DECODE_STEP;  // Nq is ignored
  if (empty_batch(B, rowless ? 1 : Nq)) {
    // only the status header, if the call is valid for one row
    const size_t one = msa_workspace_size(op, 1, 1, one_key_min(Nk), G, Hq, d, di, Bs, K, dtype);
    return one ? kWsHeader : 0;
  }
  switch (op) {
    case MSA_OP_INDEX_SELECT: {
      IndexPlan p = plan_index(B, Nq, Nk, G, di, Bs, K, dtype, false);
      return p.ok ? p.ws_bytes : 0;
    }
    case MSA_OP_PREFILL: {
      AttnPlan p = plan_attn(B, Nq, Nk, Hq, G > 0 ? G : 1, d, Bs, K, dtype, true);
      return p.ok ? p.ws_bytes : 0;
    }
    case MSA_OP_DECODE: {
      AttnPlan p = plan_attn(B, 1, Nk, Hq, G > 0 ? G : 1, d, Bs, K, dtype, false);
      return p.ok ? p.ws_bytes : 0;
    }
    case MSA_OP_DECODE_STEP: {
      StepPlan p = plan_step(B, Nk, G, Hq, d, di, Bs, K, dtype);
      return p.ok ? p.ws_bytes : 0;
    }
    case MSA_OP_KL_AUX: {
      if (B < 1 || Nq < 1 || Nk < 1 || Nq > Nk || G < 1 || Hq < 1 || Hq % G != 0) return 0;
      // the scratch does not depend on di, but a pairing the entry point rejects gets no size
      if (!kl_aux_supported(dtype, Hq, G, d, di, Bs, K)) return 0;
      return kl_aux_ws_bytes(Nq, Nk, Hq, G, d, Bs, K);
    }
    case MSA_OP_BACKWARD: {
      if (B < 1 || Nq < 1 || Nk < 1 || Nq > Nk || G < 1 || Hq < 1 || Hq % G != 0) return 0;
      if (!attn_backward_supported(dtype, Hq, G, d, Bs, K)) return 0;
      return attn_backward_ws_bytes(B, Nq, Nk, Hq, G, d, Bs, K);
    }
    default:
      return 0;
  }
}

extern "C" msa_status_t msa_index_select_v(const void* iq, const void* ik, const int32_t* q_offset,
                                           const int32_t* kv_len, int B, int Nq, int Nk, int G, int di, int Bs, int K,
                                           int dtype, int force, int32_t* sel, float* block_max, void* ws,
                                           size_t ws_bytes, cudaStream_t stream) {
  if (force != MSA_FORCE_LOCAL && force != (MSA_FORCE_LOCAL | MSA_FORCE_START)) return MSA_ERR_INVALID_ARG;
  const int fs = (force & MSA_FORCE_START) ? 1 : 0;  // block 0 kept as well
  if (fs && K < 2) return MSA_ERR_INVALID_ARG;
  if (empty_batch(B, Nq)) return index_select_empty_status(Nk, G, di, Bs, K, dtype);
  if (!iq || !ik || !sel) return MSA_ERR_INVALID_ARG;
  IndexPlan p = plan_index(B, Nq, Nk, G, di, Bs, K, dtype, block_max != nullptr);
  if (!p.ok) return p.err;
  msa_status_t w = check_ws(ws, ws_bytes, block_max ? kWsHeader : p.ws_bytes);
  if (w != MSA_OK) return w;
  uint32_t* status = status_word(ws);
  if (p.fused && !block_max) {
    float* tab = reinterpret_cast<float*>(static_cast<char*>(ws) + p.table_off);
    return cuda_status(launch_index_fused_tc(iq, ik, q_offset, kv_len, B, Nq, Nk, G, di, Bs, K, fs, sel, tab,
                                             p.table_bytes, status, stream));
  }
  if (!block_max && decode_index_supported(dtype, B, Nq, G, di, Bs, K)) {
    float* tab = reinterpret_cast<float*>(static_cast<char*>(ws) + p.table_off);
    return cuda_status(launch_decode_index(iq, ik, q_offset, kv_len, B, Nk, G, Bs, K, fs, sel, tab, status, stream));
  }
  float* table = block_max ? block_max : reinterpret_cast<float*>(static_cast<char*>(ws) + p.table_off);
  cudaError_t e = launch_index_blockmax_table(dtype, iq, ik, q_offset, kv_len, B, Nq, Nk, G, di, Bs, table, status,
                                              stream);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  e = launch_topk_from_table(table, q_offset, kv_len, B, Nq, Nk, G, Bs, K, fs, sel, status, stream);
  return cuda_status(e);
}

extern "C" msa_status_t msa_index_select(const void* iq, const void* ik, const int32_t* q_offset,
                                         const int32_t* kv_len, int B, int Nq, int Nk, int G, int di, int Bs, int K,
                                         int dtype, int32_t* sel, float* block_max, void* ws, size_t ws_bytes,
                                         cudaStream_t stream) {
  return msa_index_select_v(iq, ik, q_offset, kv_len, B, Nq, Nk, G, di, Bs, K, dtype, MSA_FORCE_LOCAL, sel, block_max,
                            ws, ws_bytes, stream);
}

extern "C" msa_status_t msa_sparse_attn_prefill(const void* q, const void* k, const void* v, const int32_t* sel,
                                                const int32_t* q_offset, const int32_t* kv_len, int B, int Nq, int Nk,
                                                int Hq, int Hkv, int d, int Bs, int K, float scale, int dtype,
                                                void* out, float* lse, void* ws, size_t ws_bytes,
                                                cudaStream_t stream) {
  if (empty_batch(B, Nq)) {
    const AttnPlan one = plan_attn(1, 1, one_key_min(Nk), Hq, Hkv, d, Bs, K, dtype, true);
    return one.ok ? MSA_OK : one.err;
  }
  if (!q || !k || !v || !sel || !out) return MSA_ERR_INVALID_ARG;
  AttnPlan p = plan_attn(B, Nq, Nk, Hq, Hkv, d, Bs, K, dtype, true);
  if (!p.ok) return p.err;
  msa_status_t w = check_ws(ws, ws_bytes, p.ws_bytes);
  if (w != MSA_OK) return w;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(float(d));
  if (p.kv_outer)
    return cuda_status(launch_attn_kv_outer(q, k, v, sel, q_offset, kv_len, B, Nq, Nk, Hq, Hkv, d, Bs, K, scale, out,
                                            lse, ws, stream));
  cudaError_t e = launch_attn_query_outer(dtype, q, k, v, sel, q_offset, kv_len, false, B, Nq, Nk, Hq, Hkv, d, Bs,
                                          K, scale, out, lse, status_word(ws), stream);
  return cuda_status(e);
}

extern "C" msa_status_t msa_sparse_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                                               const int32_t* sel, const int32_t* kv_len, int B, int Lmax, int Hq,
                                               int Hkv, int d, int Bs, int K, float scale, int dtype, void* out,
                                               float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (empty_batch(B, 1)) {
    const AttnPlan one = plan_attn(1, 1, Lmax, Hq, Hkv, d, Bs, K, dtype, false);
    return one.ok ? MSA_OK : one.err;
  }
  if (!q || !k_cache || !v_cache || !sel || !kv_len || !out) return MSA_ERR_INVALID_ARG;
  AttnPlan p = plan_attn(B, 1, Lmax, Hq, Hkv, d, Bs, K, dtype, false);
  if (!p.ok) return p.err;
  msa_status_t w = check_ws(ws, ws_bytes, p.ws_bytes);
  if (w != MSA_OK) return w;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(float(d));
  if (p.split)
    return cuda_status(launch_decode_attn(q, k_cache, v_cache, sel, kv_len, B, Lmax, Hq, Hkv, d, Bs, K, scale, out,
                                          lse, static_cast<char*>(ws) + kWsHeader, status_word(ws), stream));
  cudaError_t e = launch_attn_query_outer(dtype, q, k_cache, v_cache, sel, nullptr, kv_len, true, B, 1, Lmax, Hq,
                                          Hkv, d, Bs, K, scale, out, lse, status_word(ws), stream);
  return cuda_status(e);
}

extern "C" msa_status_t msa_decode_step(const void* q, const void* k_new, const void* v_new, const void* iq,
                                        const void* ik_new, void* k_cache, void* v_cache, void* ik_cache,
                                        int32_t* kv_len, int B, int Lmax, int Hq, int Hkv, int d, int di, int Bs,
                                        int K, float scale, int dtype, int32_t* sel, void* out, float* lse, void* ws,
                                        size_t ws_bytes, cudaStream_t stream) {
  if (Hkv < 1 || Hq % Hkv != 0) return MSA_ERR_INVALID_ARG;
  if (empty_batch(B, 1)) {
    const StepPlan one = plan_step(1, Lmax, Hkv, Hq, d, di, Bs, K, dtype);
    return one.ok ? MSA_OK : one.err;
  }
  if (!q || !k_new || !v_new || !iq || !ik_new || !k_cache || !v_cache || !ik_cache || !kv_len || !sel || !out)
    return MSA_ERR_INVALID_ARG;
  StepPlan p = plan_step(B, Lmax, Hkv, Hq, d, di, Bs, K, dtype);
  if (!p.ok) return p.err;
  msa_status_t w = check_ws(ws, ws_bytes, p.ws_bytes);
  if (w != MSA_OK) return w;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(float(d));
  char* base = static_cast<char*>(ws);
  uint32_t* status = status_word(ws);
  int32_t* pos = reinterpret_cast<int32_t*>(base + p.off_pos);
  const int G = Hkv, esize = dtype == MSA_BF16 ? 2 : 4;
  // 1. the new token of every sequence joins its caches
  cudaError_t e = launch_decode_append(k_new, v_new, ik_new, k_cache, v_cache, ik_cache, kv_len, pos, B, Lmax, Hkv, d,
                                       di, esize, status, stream);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  // 2. its selection over the grown index-key cache (position = old length)
  float* table = reinterpret_cast<float*>(base + p.off_index);
  if (decode_index_supported(dtype, B, 1, G, di, Bs, K)) {
    e = launch_decode_index(iq, ik_cache, pos, kv_len, B, Lmax, G, Bs, K, 0, sel, table, status, stream);
  } else {
    e = launch_index_blockmax_table(dtype, iq, ik_cache, pos, kv_len, B, 1, Lmax, G, di, Bs, table, status, stream);
    if (e == cudaSuccess) e = launch_topk_from_table(table, pos, kv_len, B, 1, Lmax, G, Bs, K, 0, sel, status, stream);
  }
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  // 3. attention of the token over its selected blocks (pos = kv_len - 1)
  if (p.ap.split)
    e = launch_decode_attn(q, k_cache, v_cache, sel, kv_len, B, Lmax, Hq, Hkv, d, Bs, K, scale, out, lse,
                           base + p.off_attn, status, stream);
  else
    e = launch_attn_query_outer(dtype, q, k_cache, v_cache, sel, nullptr, kv_len, true, B, 1, Lmax, Hq, Hkv, d, Bs, K,
                                scale, out, lse, status, stream);
  return cuda_status(e);
}

extern "C" msa_status_t msa_kl_aux_forward(const void* q, const void* k, const void* iq, const void* ik,
                                           const int32_t* sel, const float* lse, const int32_t* q_offset,
                                           const int32_t* kv_len, int B, int Nq, int Nk, int Hq, int Hkv, int d, int di,
                                           int Bs, int K, float scale, int dtype, float* kl, void* ws,
                                           size_t ws_bytes, cudaStream_t stream) {
  if (empty_batch(B, Nq)) {
    if (Nk < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || K < 1 || Bs < 1 || !dtype_ok(dtype))
      return MSA_ERR_INVALID_ARG;
    return kl_aux_supported(dtype, Hq, Hkv, d, di, Bs, K) ? MSA_OK : MSA_ERR_UNSUPPORTED;
  }
  if (!q || !k || !iq || !ik || !sel || !lse || !kl) return MSA_ERR_INVALID_ARG;
  if (B < 1 || Nq < 1 || Nk < 1 || Nq > Nk || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || K < 1 || Bs < 1 ||
      !dtype_ok(dtype))
    return MSA_ERR_INVALID_ARG;
  if (!kl_aux_supported(dtype, Hq, Hkv, d, di, Bs, K)) return MSA_ERR_UNSUPPORTED;
  msa_status_t w = check_ws(ws, ws_bytes, kl_aux_ws_bytes(Nq, Nk, Hq, Hkv, d, Bs, K));
  if (w != MSA_OK) return w;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(float(d));
  return cuda_status(launch_kl_aux(q, k, iq, ik, sel, lse, q_offset, kv_len, B, Nq, Nk, Hq, Hkv, d, di, Bs, K, scale,
                                   kl, ws, stream));
}

extern "C" msa_status_t msa_sparse_attn_backward(const void* q, const void* k, const void* v, const void* out,
                                                 const void* dout, const float* lse, const int32_t* sel,
                                                 const int32_t* q_offset, const int32_t* kv_len, int B, int Nq,
                                                 int Nk, int Hq, int Hkv, int d, int Bs, int K, float scale,
                                                 int dtype, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                                                 cudaStream_t stream) {
  if (empty_batch(B, Nq)) {
    if (Nk < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || K < 1 || Bs < 1 || !dtype_ok(dtype))
      return MSA_ERR_INVALID_ARG;
    if (!attn_backward_supported(dtype, Hq, Hkv, d, Bs, K)) return MSA_ERR_UNSUPPORTED;
    const size_t kv_bytes = size_t(B) * Nk * Hkv * d * 2;  // bf16
    if (kv_bytes == 0) return MSA_OK;
    // keys that no query reaches: dk = dv = 0
    if (!dk || !dv) return MSA_ERR_INVALID_ARG;
    if (cudaMemsetAsync(dk, 0, kv_bytes, stream) != cudaSuccess) return MSA_ERR_CUDA;
    return cuda_status(cudaMemsetAsync(dv, 0, kv_bytes, stream));
  }
  if (!q || !k || !v || !out || !dout || !lse || !sel || !dq || !dk || !dv) return MSA_ERR_INVALID_ARG;
  if (B < 1 || Nq < 1 || Nk < 1 || Nq > Nk || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || K < 1 || Bs < 1 ||
      !dtype_ok(dtype))
    return MSA_ERR_INVALID_ARG;
  if (!attn_backward_supported(dtype, Hq, Hkv, d, Bs, K)) return MSA_ERR_UNSUPPORTED;
  msa_status_t w = check_ws(ws, ws_bytes, attn_backward_ws_bytes(B, Nq, Nk, Hq, Hkv, d, Bs, K));
  if (w != MSA_OK) return w;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(float(d));
  return cuda_status(launch_attn_backward(q, k, v, out, dout, lse, sel, q_offset, kv_len, B, Nq, Nk, Hq, Hkv, d, Bs,
                                          K, scale, dq, dk, dv, ws, stream));
}

extern "C" msa_status_t msa_read_status(void* ws, cudaStream_t stream) {
  if (!ws) return MSA_ERR_INVALID_ARG;
  uint32_t host = 0;
  if (cudaMemcpyAsync(&host, status_word(ws), sizeof(host), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_ERR_CUDA;
  if (host != 0) {
    if (cudaMemsetAsync(status_word(ws), 0, sizeof(uint32_t), stream) != cudaSuccess) return MSA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_ERR_CUDA;
  }
  return static_cast<msa_status_t>(host);
}

extern "C" const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK:
      return "MSA_OK";
    case MSA_ERR_INVALID_ARG:
      return "MSA_ERR_INVALID_ARG: invalid argument";
    case MSA_ERR_UNSUPPORTED:
      return "MSA_ERR_UNSUPPORTED: shape or dtype not built";
    case MSA_ERR_WORKSPACE:
      return "MSA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MSA_ERR_CUDA:
      return "MSA_ERR_CUDA: CUDA launch or runtime error";
    case MSA_ERR_TIMEOUT:
      return "MSA_ERR_TIMEOUT: a bounded device wait ran out";
    case MSA_ERR_BOUNDS:
      return "MSA_ERR_BOUNDS: q_offset, kv_len or sel out of range";
    default:
      return "MSA status: unknown code";
  }
}
