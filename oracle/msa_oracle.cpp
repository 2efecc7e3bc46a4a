// MSA oracle: plain, slow, fp64 CPU restatement of what the sparse attention
// path computes (forward, its backward, the KL auxiliary value). TEST INFRASTRUCTURE ONLY: the tests, the smoke check
// and the bench's CPU-baseline / reference leg call it; the product library
// never does. It shares no code, header or helper with the CUDA path.
//
// Sources (MiniMax Sparse Attention; three pages describing one method):
//  * "MiniMax Sparse Attention" summary (hyper.ai, paper 2606.13392), section
//    "方法" (Method): an Index Branch run per GQA group scores every causally
//    visible key with the dot product of an index query and an index key,
//    pools the token scores to blocks by max (Block Max Pooling), keeps the
//    Top-K blocks, and always includes the block that holds the current query;
//    the Main Branch then runs standard scaled-dot-product softmax attention
//    over only the keys/values of the selected blocks.
//  * quant_prune_distill post 751 (tgviewer), section "Метод" (Method): one
//    index query head per query group and a single index key head for the
//    whole layer; pre-softmax score, block maximum, top-K blocks by that
//    maximum; the last block (sliding window) is always added.
//  * same post, section "Эксперименты": 16 blocks of 128 tokens = 2048 tokens,
//    i.e. the forced block counts toward K.
//
// Readings taken where the pages are silent:
//  blocks are aligned to absolute position 0 (block t = keys [t*Bs, (t+1)*Bs));
//  ties in the block maximum go to the lower block index; when a row sees at
//  most K blocks all of them are selected and the list is padded with -1;
//  the index score is the plain dot product (no scale: a positive scale
//  cannot change a ranking); the attention scale is 1/sqrt(d) unless given;
//  the causal mask keeps key j iff j <= pos, pos = q_offset[b] + i.
//
// Variant (same summary, section "实验" (Experiments)): the ablation that
// hard-codes the sequence-start block as well as the local window. With
// force_start, block 0 is kept like the local block and the other K-2 come
// from the ranking of blocks 1..loc-1.
//
// Parity pins for every function here live in tests/test_oracle_pins.py.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

template <class F>
void parallel_rows(int64_t nrows, int nthreads, F&& f) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  if (nthreads == 1 || nrows < 2) {
    for (int64_t r = 0; r < nrows; ++r) f(r);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t)
    pool.emplace_back([&, t] {
      for (int64_t r = t; r < nrows; r += nthreads) f(r);  // interleaved: cost grows with position
    });
  for (auto& th : pool) th.join();
}

// Index Branch for one (row, group): token scores, block maxima, selection.
// Writes K entries of `sel` (ascending block ids, -1 padded) and, if given,
// nblk entries of `bmax` (NaN where a block is not visible).
void index_select_one(const float* iq_g, const float* ik_b, int di, int pos, int L, int Bs, int K, int nblk,
                      bool force_start, int* sel, double* bmax) {
  const int jmax = std::min(pos, L - 1);  // last causally visible key
  const int loc = pos / Bs;               // block holding the query
  std::vector<double> M(loc + 1, -std::numeric_limits<double>::infinity());
  for (int j = 0; j <= jmax; ++j) {
    double s = 0.0;  // pre-softmax index score: plain dot product
    for (int c = 0; c < di; ++c) s += double(iq_g[c]) * double(ik_b[int64_t(j) * di + c]);
    const int t = j / Bs;
    if (s > M[t]) M[t] = s;  // block max pooling
  }
  if (bmax) {
    for (int t = 0; t < nblk; ++t) bmax[t] = t <= loc ? M[t] : std::numeric_limits<double>::quiet_NaN();
  }
  std::vector<int> chosen;
  if (loc + 1 <= K) {
    for (int t = 0; t <= loc; ++t) chosen.push_back(t);  // every visible block
  } else {
    const int first = force_start ? 1 : 0;  // block 0 is kept outright in the variant
    std::vector<int> cand;
    for (int t = first; t < loc; ++t) cand.push_back(t);
    std::sort(cand.begin(), cand.end(), [&](int a, int b) {
      if (M[a] != M[b]) return M[a] > M[b];  // higher block maximum first
      return a < b;                          // tie: lower block index
    });
    const int ranked = K - 1 - first;
    for (int k = 0; k < ranked; ++k) chosen.push_back(cand[k]);
    if (force_start) chosen.push_back(0);
    chosen.push_back(loc);  // the query's own block is always kept
    std::sort(chosen.begin(), chosen.end());
  }
  for (int k = 0; k < K; ++k) sel[k] = k < int(chosen.size()) ? chosen[k] : -1;
}

}  // namespace

extern "C" {

// Index Branch for a list of query rows.
//   iq_rows  [nrows, G, di]    index queries of the listed rows
//   ik       [B, Nk, di]       the layer's single index key head
//   row_b, row_i [nrows]       sequence and query index of each listed row
//   q_offset, kv_len [B]       pos = q_offset[b] + i; keys j < kv_len[b]
//   sel      [nrows, G, K]     out: ascending block ids, -1 padded
//   block_max [nrows, G, nblk] out (optional): fp64 block maxima, NaN if not visible
//   force_start              0: only the local block is forced; 1: block 0 too (K >= 2)
int msa_oracle_index_select_v(const float* iq_rows, const float* ik, const int32_t* row_b, const int32_t* row_i,
                              int64_t nrows, const int32_t* q_offset, const int32_t* kv_len, int B, int Nk, int G,
                              int di, int Bs, int K, int force_start, int32_t* sel, double* block_max, int nthreads) {
  if (!iq_rows || !ik || !row_b || !row_i || !q_offset || !kv_len || !sel) return 1;
  if (B < 1 || Nk < 1 || G < 1 || di < 1 || Bs < 1 || K < 1 || nrows < 0) return 1;
  if (force_start != 0 && (force_start != 1 || K < 2)) return 1;
  const int nblk = (Nk + Bs - 1) / Bs;
  for (int64_t r = 0; r < nrows; ++r) {
    const int b = row_b[r];
    if (b < 0 || b >= B) return 1;
    const int pos = q_offset[b] + row_i[r];
    if (pos < 0 || kv_len[b] < 1 || kv_len[b] > Nk || pos >= kv_len[b]) return 1;
  }
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    const int b = row_b[r];
    const int pos = q_offset[b] + row_i[r];
    for (int g = 0; g < G; ++g) {
      index_select_one(iq_rows + (r * G + g) * di, ik + int64_t(b) * Nk * di, di, pos, kv_len[b], Bs, K, nblk,
                       force_start != 0, sel + (r * G + g) * K, block_max ? block_max + (r * G + g) * nblk : nullptr);
    }
  });
  return 0;
}

int msa_oracle_index_select(const float* iq_rows, const float* ik, const int32_t* row_b, const int32_t* row_i,
                            int64_t nrows, const int32_t* q_offset, const int32_t* kv_len, int B, int Nk, int G,
                            int di, int Bs, int K, int32_t* sel, double* block_max, int nthreads) {
  return msa_oracle_index_select_v(iq_rows, ik, row_b, row_i, nrows, q_offset, kv_len, B, Nk, G, di, Bs, K, 0, sel,
                                   block_max, nthreads);
}

// Main Branch for a list of query rows: exact softmax attention over the
// tokens of the selected blocks, causally masked.
//   q_rows [nrows, Hq, d]; k, v [B, Nk, Hkv, d]; sel_rows [nrows, G=Hkv, K]
//   out [nrows, Hq, d] (fp64); lse [nrows, Hq] (fp64, optional)
//   scale <= 0 selects 1/sqrt(d).
int msa_oracle_sparse_attn(const float* q_rows, const float* k, const float* v, const int32_t* sel_rows,
                           const int32_t* row_b, const int32_t* row_i, int64_t nrows, const int32_t* q_offset,
                           const int32_t* kv_len, int B, int Nk, int Hq, int Hkv, int d, int Bs, int K,
                           double scale, double* out, double* lse, int nthreads) {
  if (!q_rows || !k || !v || !sel_rows || !row_b || !row_i || !q_offset || !kv_len || !out) return 1;
  if (B < 1 || Nk < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || Bs < 1 || K < 1) return 1;
  if (scale <= 0.0) scale = 1.0 / std::sqrt(double(d));
  const int nblk = (Nk + Bs - 1) / Bs;
  const int heads_per_group = Hq / Hkv;
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    const int b = row_b[r];
    const int pos = q_offset[b] + row_i[r];
    const int L = kv_len[b];
    std::vector<int> keys;
    std::vector<double> s;
    for (int h = 0; h < Hq; ++h) {
      const int g = h / heads_per_group;  // GQA: query head h reads key/value head g
      const int32_t* sl = sel_rows + (r * Hkv + g) * K;
      keys.clear();
      for (int kk = 0; kk < K; ++kk) {
        const int t = sl[kk];
        if (t < 0 || t >= nblk) continue;
        for (int j = t * Bs; j < (t + 1) * Bs && j < L && j <= pos; ++j) keys.push_back(j);
      }
      const float* qh = q_rows + (r * Hq + h) * int64_t(d);
      double* oh = out + (r * Hq + h) * int64_t(d);
      for (int c = 0; c < d; ++c) oh[c] = 0.0;
      if (keys.empty()) {
        if (lse) lse[r * Hq + h] = -std::numeric_limits<double>::infinity();
        continue;
      }
      s.assign(keys.size(), 0.0);
      double m = -std::numeric_limits<double>::infinity();
      for (size_t n = 0; n < keys.size(); ++n) {
        const float* kj = k + ((int64_t(b) * Nk + keys[n]) * Hkv + g) * int64_t(d);
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += double(qh[c]) * double(kj[c]);
        s[n] = acc * scale;
        m = std::max(m, s[n]);
      }
      double l = 0.0;
      for (size_t n = 0; n < keys.size(); ++n) {
        const double w = std::exp(s[n] - m);
        l += w;
        const float* vj = v + ((int64_t(b) * Nk + keys[n]) * Hkv + g) * int64_t(d);
        for (int c = 0; c < d; ++c) oh[c] += w * double(vj[c]);
      }
      for (int c = 0; c < d; ++c) oh[c] /= l;
      if (lse) lse[r * Hq + h] = m + std::log(l);
    }
  });
  return 0;
}

// KL auxiliary (forward value only): for each (row, group), the divergence
// KL(p || q) over the tokens T of the group's selected blocks (causally
// visible), where p is the Main Branch's attention distribution averaged over
// the group's query heads and q is the softmax of the Index Branch's scores
// over the same tokens. (quant_prune_distill post 751, "Метод": the loss is the
// KL divergence between the index branch and the head-averaged main branch,
// main-branch probabilities under stop-gradient; hyper.ai summary, "方法":
// the index distribution is aligned with the main branch's on the selected
// tokens.) Index scores enter the softmax as the plain dot products.
//   q_rows [nrows, Hq, d]; k [B, Nk, Hkv, d]; iq_rows [nrows, Hkv, di];
//   ik [B, Nk, di]; sel_rows [nrows, Hkv, K]; kl [nrows, Hkv] (fp64, out)
//   scale <= 0 selects 1/sqrt(d).
int msa_oracle_kl_aux(const float* q_rows, const float* k, const float* iq_rows, const float* ik,
                      const int32_t* sel_rows, const int32_t* row_b, const int32_t* row_i, int64_t nrows,
                      const int32_t* q_offset, const int32_t* kv_len, int B, int Nk, int Hq, int Hkv, int d, int di,
                      int Bs, int K, double scale, double* kl, int nthreads) {
  if (!q_rows || !k || !iq_rows || !ik || !sel_rows || !row_b || !row_i || !q_offset || !kv_len || !kl) return 1;
  if (B < 1 || Nk < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || di < 1 || Bs < 1 || K < 1) return 1;
  if (scale <= 0.0) scale = std::sqrt(1.0 / double(d));  // the attention's default scale
  const int nblk = (Nk + Bs - 1) / Bs;
  const int hpg = Hq / Hkv;
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    const int b = row_b[r];
    const int pos = q_offset[b] + row_i[r];
    const int L = kv_len[b];
    for (int g = 0; g < Hkv; ++g) {
      std::vector<int> keys;
      const int32_t* sl = sel_rows + (r * Hkv + g) * K;
      for (int kk = 0; kk < K; ++kk) {
        const int t = sl[kk];
        if (t < 0 || t >= nblk) continue;
        for (int j = t * Bs; j < (t + 1) * Bs && j <= pos && j < L; ++j) keys.push_back(j);  // causal, diagonal kept
      }
      const size_t n = keys.size();
      if (n == 0) {
        kl[r * Hkv + g] = 0.0;
        continue;
      }
      // p: softmax of the scaled main scores per head, averaged over the group's heads
      std::vector<double> p(n, 0.0), z(n);
      for (int h = g * hpg; h < (g + 1) * hpg; ++h) {
        const float* qh = q_rows + (r * Hq + h) * int64_t(d);
        double m = -std::numeric_limits<double>::infinity();
        for (size_t x = 0; x < n; ++x) {
          const float* kj = k + ((int64_t(b) * Nk + keys[x]) * Hkv + g) * int64_t(d);
          double acc = 0.0;
          for (int c = 0; c < d; ++c) acc += double(qh[c]) * double(kj[c]);
          z[x] = acc * scale;
          m = std::max(m, z[x]);
        }
        double l = 0.0;
        for (size_t x = 0; x < n; ++x) l += std::exp(z[x] - m);
        for (size_t x = 0; x < n; ++x) p[x] += std::exp(z[x] - m) / l / double(hpg);
      }
      // q: softmax of the index scores over the same tokens
      const float* iqg = iq_rows + (r * Hkv + g) * int64_t(di);
      std::vector<double> s(n);
      double ms = -std::numeric_limits<double>::infinity();
      for (size_t x = 0; x < n; ++x) {
        double acc = 0.0;
        for (int c = 0; c < di; ++c) acc += double(iqg[c]) * double(ik[(int64_t(b) * Nk + keys[x]) * di + c]);
        s[x] = acc;
        ms = std::max(ms, s[x]);
      }
      double ls = 0.0;
      for (size_t x = 0; x < n; ++x) ls += std::exp(s[x] - ms);
      const double lse_q = ms + std::log(ls);
      double div = 0.0;  // sum_j p_j (log p_j - log q_j)
      for (size_t x = 0; x < n; ++x)
        if (p[x] > 0.0) div += p[x] * (std::log(p[x]) - (s[x] - lse_q));
      kl[r * Hkv + g] = div;
    }
  });
  return 0;
}

// Main Branch backward for a list of query rows: the gradients of a scalar
// loss with respect to q, k and v, given dout = dLoss/dOut. The selection is
// a discrete choice of the Index Branch and carries no gradient; the Main
// Branch is plain softmax attention over the selected tokens (hyper.ai
// summary, "方法"), so its gradient is the textbook one. The forward is
// recomputed here in fp64 from its definition, then differentiated by the
// chain rule over the attended tokens T of each (row, head):
//   P_j = softmax_j(scale q.k_j),  O = sum_j P_j v_j
//   dv_j += P_j dout;  dP_j = dout.v_j;  delta = dout.O (= sum_j P_j dP_j)
//   dS_j = P_j (dP_j - delta);  dq = scale sum_j dS_j k_j;  dk_j += scale dS_j q
//   q_rows, dout_rows [nrows, Hq, d]; k, v [B, Nk, Hkv, d]; sel_rows [nrows, Hkv, K]
//   dq [nrows, Hq, d] (fp64, out); dk, dv [B, Nk, Hkv, d] (fp64, out): the
//   listed rows' contributions (zero where no listed row attends).
//   scale <= 0 selects 1/sqrt(d).
int msa_oracle_sparse_attn_backward(const float* q_rows, const float* k, const float* v, const float* dout_rows,
                                    const int32_t* sel_rows, const int32_t* row_b, const int32_t* row_i,
                                    int64_t nrows, const int32_t* q_offset, const int32_t* kv_len, int B, int Nk,
                                    int Hq, int Hkv, int d, int Bs, int K, double scale, double* dq, double* dk,
                                    double* dv, int nthreads) {
  if (!q_rows || !k || !v || !dout_rows || !sel_rows || !row_b || !row_i || !q_offset || !kv_len || !dq || !dk ||
      !dv)
    return 1;
  if (B < 1 || Nk < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || Bs < 1 || K < 1) return 1;
  if (scale <= 0.0) scale = 1.0 / std::sqrt(static_cast<double>(d));
  const int nblk = (Nk + Bs - 1) / Bs;
  const int hpg = Hq / Hkv;
  const int64_t kv_elems = int64_t(B) * Nk * Hkv * d;
  for (int64_t x = 0; x < kv_elems; ++x) dk[x] = dv[x] = 0.0;
  // one work unit per (sequence, key/value head): it owns dk, dv of that head
  // and dq of the group's query heads, so units never write the same element
  parallel_rows(int64_t(B) * Hkv, nthreads, [&](int64_t u) {
    const int b = int(u / Hkv), g = int(u % Hkv);
    const int pos_base = q_offset[b], L = kv_len[b];
    std::vector<int> toks;
    std::vector<double> P, o(d);
    for (int64_t r = 0; r < nrows; ++r) {
      if (row_b[r] != b) continue;
      const int pos = pos_base + row_i[r];
      toks.clear();
      const int32_t* blocks = sel_rows + (r * Hkv + g) * K;
      for (int kk = 0; kk < K; ++kk) {
        const int t = blocks[kk];
        if (t < 0 || t >= nblk) continue;
        for (int j = t * Bs; j < (t + 1) * Bs; ++j) {
          if (j > pos || j >= L) break;  // the forward's mask: diagonal kept, nothing at or past kv_len
          toks.push_back(j);
        }
      }
      for (int hh = 0; hh < hpg; ++hh) {
        const int h = g * hpg + hh;
        const float* qh = q_rows + (r * Hq + h) * int64_t(d);
        const float* gh = dout_rows + (r * Hq + h) * int64_t(d);
        double* dqh = dq + (r * Hq + h) * int64_t(d);
        for (int c = 0; c < d; ++c) dqh[c] = 0.0;
        const size_t n = toks.size();
        if (n == 0) continue;
        // forward: probabilities and output
        P.assign(n, 0.0);
        double mx = -std::numeric_limits<double>::infinity();
        for (size_t x = 0; x < n; ++x) {
          const float* kj = k + ((int64_t(b) * Nk + toks[x]) * Hkv + g) * int64_t(d);
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += double(qh[c]) * double(kj[c]);
          P[x] = scale * dot;
          if (P[x] > mx) mx = P[x];
        }
        double den = 0.0;
        for (size_t x = 0; x < n; ++x) {
          P[x] = std::exp(P[x] - mx);
          den += P[x];
        }
        for (size_t x = 0; x < n; ++x) P[x] /= den;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (size_t x = 0; x < n; ++x) {
          const float* vj = v + ((int64_t(b) * Nk + toks[x]) * Hkv + g) * int64_t(d);
          for (int c = 0; c < d; ++c) o[c] += P[x] * double(vj[c]);
        }
        double delta = 0.0;
        for (int c = 0; c < d; ++c) delta += double(gh[c]) * o[c];
        // backward
        for (size_t x = 0; x < n; ++x) {
          const int64_t kvrow = ((int64_t(b) * Nk + toks[x]) * Hkv + g) * int64_t(d);
          const float* kj = k + kvrow;
          const float* vj = v + kvrow;
          double dP = 0.0;
          for (int c = 0; c < d; ++c) dP += double(gh[c]) * double(vj[c]);
          const double dS = P[x] * (dP - delta);
          for (int c = 0; c < d; ++c) {
            dqh[c] += scale * dS * double(kj[c]);
            dk[kvrow + c] += scale * dS * double(qh[c]);
            dv[kvrow + c] += P[x] * double(gh[c]);
          }
        }
      }
    }
  });
  return 0;
}

}  // extern "C"
