/*
 * msa.h -- C ABI of the MiniMax Sparse Attention (MSA) forward path on GB300.
 *
 * MSA is block-sparse attention layered on grouped-query attention (GQA). It
 * has two branches (hyper.ai summary of paper 2606.13392, section "方法";
 * quant_prune_distill post 751, section "Метод"):
 *
 *   Index Branch  one index query head per GQA group and one index key head
 *                 for the whole layer; a pre-softmax dot-product score for
 *                 every causally visible key, max-pooled per key block, then
 *                 the Top-K blocks by that maximum, the block that holds the
 *                 query always included            -> msa_index_select
 *   Main Branch   exact softmax attention restricted to the keys/values of
 *                 the selected blocks               -> msa_sparse_attn_prefill
 *                                                     msa_sparse_attn_decode
 *
 * Notation: B sequences; Nq query rows per sequence; Nk key rows (capacity)
 * per sequence; Hq query heads; Hkv key/value heads = G GQA groups (query
 * head h belongs to group h / (Hq / Hkv)); d head dim; di index head dim;
 * Bs key block size; K selected blocks per (query row, group), the forced
 * local block included. Key block t holds keys [t*Bs, (t+1)*Bs). Query row i
 * of sequence b sits at absolute position pos = q_offset[b] + i and sees keys
 * j <= pos with j < kv_len[b]; its local block is loc = pos / Bs.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays
 *    owned by the caller; the library allocates nothing and keeps no pointer
 *    after the call returns. Work is enqueued on `stream` (0 = legacy default
 *    stream) and runs asynchronously; nothing is synchronised.
 *  - `dtype` (msa_dtype_t) is the element type of q, k, v, iq, ik and of the
 *    attention output: MSA_BF16 (tensor-core path, fp32 accumulation) or
 *    MSA_FP32 (CUDA-core path).
 *  - `ws` is caller-owned DEVICE scratch of at least msa_workspace_size(...)
 *    bytes, 256-byte aligned, zero-filled once before its first use. Its
 *    first word is a sticky device status that kernels set when they detect a
 *    bad index or a wait that ran out; msa_read_status() reads and clears it.
 *    Calls that share one workspace must be ordered on one stream.
 *  - Every device wait is bounded (about a second). A kernel whose wait runs
 *    out records MSA_ERR_TIMEOUT, lets its copies and matrix products finish
 *    and returns; the outputs of that call are unspecified. Nothing the next
 *    call depends on is left behind in the workspace: once msa_read_status()
 *    has cleared the status, the same workspace can be used again.
 *  - Argument errors found on the host return before anything is enqueued.
 *    Per-sequence values (q_offset, kv_len, sel entries) live on the device
 *    and are checked there: an offending row is skipped (its sel row is -1,
 *    its output row zero) and the status becomes MSA_ERR_BOUNDS.
 *  - An empty batch (B == 0, or Nq == 0 for an entry point with query rows)
 *    is valid. The other arguments are checked as for a batch of one row,
 *    pointers (ws included) may be NULL and are not read, nothing is
 *    enqueued, and the call returns MSA_OK. The one exception:
 *    msa_sparse_attn_backward with B * Nk > 0 and Nq == 0 zero-fills dk and
 *    dv (no query reaches any key), so those two must be given.
 *    msa_workspace_size returns 256 for an empty batch.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1, /* a null pointer, a non-positive size, Hq % Hkv != 0, ... */
  MSA_ERR_UNSUPPORTED = 2, /* a shape or dtype this build has no kernel for */
  MSA_ERR_WORKSPACE = 3,   /* ws is NULL, misaligned or smaller than msa_workspace_size() */
  MSA_ERR_CUDA = 4,        /* a launch or CUDA runtime call failed */
  MSA_ERR_TIMEOUT = 5,     /* device: a bounded wait ran out (the kernel returned early) */
  MSA_ERR_BOUNDS = 6       /* device: a q_offset / kv_len / sel value was out of range */
} msa_status_t;

typedef enum { MSA_BF16 = 0, MSA_FP32 = 1 } msa_dtype_t;

typedef enum {
  MSA_OP_INDEX_SELECT = 0,
  MSA_OP_PREFILL = 1,
  MSA_OP_DECODE = 2,
  MSA_OP_DECODE_STEP = 3,
  MSA_OP_KL_AUX = 4,
  MSA_OP_BACKWARD = 5
} msa_op_t;

/* Bytes of scratch `ws` the entry point `op` needs for these sizes (the same
 * argument meanings as the entry points; unused ones may be 0: G and di for
 * the attention ops, Hq and d for MSA_OP_INDEX_SELECT; for MSA_OP_DECODE and
 * MSA_OP_DECODE_STEP, Nq is ignored and Nk is Lmax; MSA_OP_DECODE_STEP and
 * MSA_OP_KL_AUX use every other argument, with G = Hkv; MSA_OP_BACKWARD uses
 * all but di, with G = Hkv). Returns 0 when the arguments are invalid or not
 * supported, and 256 for a valid empty batch. */
size_t msa_workspace_size(int op, int B, int Nq, int Nk, int G, int Hq, int d, int di, int Bs, int K, int dtype);

/* Index Branch: block selection for every (query row, group).
 * (hyper.ai summary, "方法": dot-product index scores over visible keys, Block
 *  Max Pooling, Top-K per group, the query's own block always included;
 *  quant_prune_distill post 751, "Метод"/"Эксперименты": one index query head
 *  per group, one index key head per layer, 16 blocks x 128 = 2048 tokens.)
 *
 *  iq        [B, Nq, G, di]  index queries, one head per group (dtype)
 *  ik        [B, Nk, di]     the layer's single index key head (dtype)
 *  q_offset  [B] int32 or NULL (all 0): absolute position of query row 0
 *  kv_len    [B] int32 or NULL (all Nk): valid keys per sequence;
 *            need 0 <= q_offset[b], q_offset[b] + Nq <= kv_len[b] <= Nk
 *  sel       [B, Nq, G, K] int32, out: selected block ids in ascending order.
 *            Row (b,i,g) holds loc and the K-1 blocks t < loc with the highest
 *            block maximum, ties to the lower t; if loc + 1 <= K it holds
 *            0..loc and is padded with -1.
 *  block_max [B, Nq, G, ceil(Nk/Bs)] fp32 or NULL, out (diagnostic): the
 *            block maxima of the visible keys, NaN for blocks t > loc.
 *  ws        msa_workspace_size(MSA_OP_INDEX_SELECT, ...) bytes. For bf16
 *            prefill on the tensor cores it is the 256-byte status header
 *            when K <= 16; for K > 16 it also holds the block-max table of
 *            one chunk of rows (whole units of 256 (row, group) rows, about
 *            4 GiB at most unless that leaves fewer than 608 units;
 *            MSA_INDEX_TABLE_UNITS in the environment, read once per process,
 *            sets the units per chunk, and the size follows it).
 *  Supported: dtype BF16 or FP32; di in {32, 64}; 1 <= Bs <= 1024; 1 <= K <= 64.
 *  Selection is exact when the index scores are exact in fp32 (for example
 *  integer-valued index q/k with |score| < 2^24). */
msa_status_t msa_index_select(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len, int B,
                              int Nq, int Nk, int G, int di, int Bs, int K, int dtype, int32_t* sel, float* block_max,
                              void* ws, size_t ws_bytes, cudaStream_t stream);

/* Forced blocks of a selection (msa_index_select_v). */
typedef enum { MSA_FORCE_LOCAL = 1, MSA_FORCE_START = 2 } msa_force_t;

/* msa_index_select with a choice of forced blocks. force = MSA_FORCE_LOCAL is
 * msa_index_select. force = MSA_FORCE_LOCAL | MSA_FORCE_START also keeps
 * block 0 (hyper.ai summary of paper 2606.13392, section "实验": the ablation
 * that hard-codes the sequence-start block besides the local window): a row
 * with loc + 1 > K holds 0, loc and the K-2 blocks 1 <= t < loc with the
 * highest block maximum (ties to the lower t), ascending; rows with
 * loc + 1 <= K hold 0..loc as before. MSA_FORCE_START needs K >= 2. Any other
 * force value returns MSA_ERR_INVALID_ARG before anything is enqueued. Other
 * arguments, workspace and errors as msa_index_select. */
msa_status_t msa_index_select_v(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len, int B,
                                int Nq, int Nk, int G, int di, int Bs, int K, int dtype, int force, int32_t* sel,
                                float* block_max, void* ws, size_t ws_bytes, cudaStream_t stream);

/* msa_index_select without a workspace argument: the same selection (and the
 * same optional block_max output) for callers that cannot allocate device
 * memory -- code that runs under another framework's allocator or inside its
 * plugin hooks, where a raw cudaMalloc is forbidden or would bypass that
 * framework's memory accounting, or a process whose device memory is fixed up
 * front. The paper has no counterpart of this entry point.
 *
 * It allocates nothing. Its scratch (a status word and the block-max table)
 * is a file-scope static __device__ array of 32 MiB that every GPU which loads
 * this library reserves until the process exits. The table needs
 * B*Nq*G*ceil(Nk/Bs)*4 bytes (0 when block_max is given); a call needing more
 * than 32 MiB - 256 B returns MSA_ERR_WORKSPACE before anything is enqueued.
 * The first call on each device looks up the array's device address with that
 * device current and keeps it for the life of the process; make that first call
 * before any stream capture, and do not reset the device (cudaDeviceReset)
 * after it while this library stays loaded. Every call
 * shares the one array and clears its status word first: calls whose work
 * overlaps on the GPU (other streams, or other host threads) race on it. Rows
 * that fail the device-side range checks come back as -1 rows; the status
 * word is not reported. Arguments and errors otherwise as msa_index_select. */
msa_status_t msa_index_select_noalloc(const void* iq, const void* ik, const int32_t* q_offset, const int32_t* kv_len,
                                      int B, int Nq, int Nk, int G, int di, int Bs, int K, int dtype, int32_t* sel,
                                      float* block_max, cudaStream_t stream);

/* Main Branch, prefill: exact softmax attention of every query row over the
 * keys of its group's selected blocks, causally masked (j <= pos, j < kv_len).
 * (hyper.ai summary, "方法": the Main Branch gathers the Key/Value vectors of
 *  the selected blocks and computes standard scaled dot-product attention.)
 *
 *  q    [B, Nq, Hq, d] (dtype); k, v [B, Nk, Hkv, d] (dtype)
 *  sel  [B, Nq, Hkv, K] int32: block ids per (row, group) as produced by
 *       msa_index_select (ascending, -1 padded; -1 entries are skipped)
 *  q_offset, kv_len: as for msa_index_select
 *  scale  softmax scale; <= 0 selects 1/sqrt(d)
 *  out  [B, Nq, Hq, d] (dtype), out; lse [B, Nq, Hq] fp32 or NULL, out:
 *       natural-log sum of exp of the scaled scores over the attended keys.
 *       Both are deterministic: each row merges its per-block partials in slot
 *       order, with no atomic update of any output.
 *  Supported: d in {64, 128}; BF16 or FP32; Bs and K as for msa_index_select. */
msa_status_t msa_sparse_attn_prefill(const void* q, const void* k, const void* v, const int32_t* sel,
                                     const int32_t* q_offset, const int32_t* kv_len, int B, int Nq, int Nk, int Hq,
                                     int Hkv, int d, int Bs, int K, float scale, int dtype, void* out, float* lse,
                                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* Main Branch, decode: one new query token per sequence attending to its KV
 * cache through the selected blocks (the decode half of the pages' prefill /
 * decode speedups, hyper.ai summary "一句话总结"). Same operation as
 * msa_sparse_attn_prefill with Nq = 1 and pos = kv_len[b] - 1.
 *
 *  q        [B, Hq, d] (dtype)
 *  k_cache, v_cache [B, Lmax, Hkv, d] (dtype); rows >= kv_len[b] are ignored
 *  sel      [B, Hkv, K] int32: msa_index_select output for Nq = 1 and
 *           q_offset[b] = kv_len[b] - 1
 *  kv_len   [B] int32 (required): 1 <= kv_len[b] <= Lmax
 *  out [B, Hq, d] (dtype); lse [B, Hq] fp32 or NULL */
msa_status_t msa_sparse_attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* sel,
                                    const int32_t* kv_len, int B, int Lmax, int Hq, int Hkv, int d, int Bs, int K,
                                    float scale, int dtype, void* out, float* lse, void* ws, size_t ws_bytes,
                                    cudaStream_t stream);

/* Streaming decode: one step of a serving loop. For every sequence b the new
 * token's key, value and index-key rows are appended to the caches at
 * position L = kv_len[b], kv_len[b] becomes L + 1, and the token is then
 * selected for (msa_index_select with Nq = 1, q_offset = L) and attended
 * (msa_sparse_attn_decode) over the grown caches. (hyper.ai summary of paper
 * 2606.13392, "一句话总结": the decode side of the reported speedups, where each
 * new token re-selects its blocks over the cache.)
 *
 *  q [B, Hq, d]; k_new, v_new [B, Hkv, d]; iq [B, Hkv, di]; ik_new [B, di]  (dtype)
 *  k_cache, v_cache [B, Lmax, Hkv, d]; ik_cache [B, Lmax, di] (dtype): in/out
 *  kv_len [B] int32, in/out: current lengths, advanced by one
 *  sel [B, Hkv, K] int32, out: the token's selection (as msa_index_select)
 *  out [B, Hq, d] (dtype), lse [B, Hq] fp32 or NULL, out (as msa_sparse_attn_decode)
 *  ws: msa_workspace_size(MSA_OP_DECODE_STEP, B, 0, Lmax, Hkv, Hq, d, di, Bs, K, dtype)
 * A sequence whose cache is already full (kv_len[b] == Lmax) or whose length
 * is out of range is left unchanged: its sel row is -1, its output row zero,
 * and the status word becomes MSA_ERR_BOUNDS. Supported sizes as for
 * msa_index_select and msa_sparse_attn_decode; the k/v and index-key rows must
 * be multiples of 16 bytes. */
msa_status_t msa_decode_step(const void* q, const void* k_new, const void* v_new, const void* iq, const void* ik_new,
                             void* k_cache, void* v_cache, void* ik_cache, int32_t* kv_len, int B, int Lmax, int Hq,
                             int Hkv, int d, int di, int Bs, int K, float scale, int dtype, int32_t* sel, void* out,
                             float* lse, void* ws, size_t ws_bytes, cudaStream_t stream);

/* KL auxiliary forward: for every (query row, group) the divergence
 *   KL(p || q) = sum_j p_j (log p_j - log q_j)
 * over the tokens j of the group's selected blocks (causally visible), where
 * p is the Main Branch's attention distribution averaged over the group's
 * query heads and q the softmax of the Index Branch's plain dot-product
 * scores over the same tokens (quant_prune_distill post 751, "Метод": the
 * index branch is trained with the KL divergence to the head-averaged main
 * branch, main-branch probabilities under stop-gradient; hyper.ai summary of
 * paper 2606.13392, "方法": the two distributions are aligned over the selected
 * tokens). Forward value only.
 *
 *  q [B, Nq, Hq, d], k [B, Nk, Hkv, d], iq [B, Nq, Hkv, di], ik [B, Nk, di] (dtype)
 *  sel [B, Nq, Hkv, K] int32: the selection (msa_index_select)
 *  lse [B, Nq, Hq] fp32: the forward's lse (msa_sparse_attn_prefill), which
 *       normalises p; scale must be the forward's (<= 0 selects 1/sqrt(d))
 *  q_offset, kv_len: as for msa_index_select
 *  kl [B, Nq, Hkv] fp32, out (0 for a row without attended tokens)
 *  ws: msa_workspace_size(MSA_OP_KL_AUX, B, Nq, Nk, Hkv, Hq, d, di, Bs, K, dtype)
 *  Supported: BF16; (d, di) in {(128, 64), (64, 32)}; Bs in {32, 64, 128};
 *  Hq / Hkv in {2, 4, 8}; other sizes return MSA_ERR_UNSUPPORTED.
 *  Determinism: for d 128, di 64 and Bs 128 (tensor-core pass) every sum is
 *  taken in a fixed order and repeated calls give identical bits; the other
 *  built shapes add the per-entry sums of a tile with shared-memory atomics,
 *  so their values can differ in the last bits from run to run. */
msa_status_t msa_kl_aux_forward(const void* q, const void* k, const void* iq, const void* ik, const int32_t* sel,
                                const float* lse, const int32_t* q_offset, const int32_t* kv_len, int B, int Nq,
                                int Nk, int Hq, int Hkv, int d, int di, int Bs, int K, float scale, int dtype,
                                float* kl, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Main Branch backward: the gradients of a loss with respect to q, k and v
 * through the sparse attention of msa_sparse_attn_prefill, given the
 * gradient dout of its output. The selection is held fixed (the Index Branch's
 * choice carries no gradient).
 * (hyper.ai summary, "方法": the Main Branch is standard scaled-dot-product
 *  softmax attention over the selected blocks; "一句话总结"/"实验": the model
 *  is trained through it. Per (row, head), over the attended keys j:
 *  P_j = exp(scale q.k_j - lse), delta = dout . out, dS_j = P_j (dout.v_j - delta),
 *  dq = scale sum_j dS_j k_j, dk_j = scale sum dS_j q, dv_j = sum P_j dout.)
 *
 *  q, out, dout [B, Nq, Hq, d]; k, v [B, Nk, Hkv, d] (dtype), as in the forward
 *  lse       [B, Nq, Hq] fp32: the forward's log-sum-exp output
 *  sel       [B, Nq, Hkv, K] int32: the forward's selection
 *  q_offset, kv_len, scale: as for msa_sparse_attn_prefill
 *  dq [B, Nq, Hq, d], dk, dv [B, Nk, Hkv, d] (dtype), out: fp32 accumulation,
 *            rounded once; keys no row attends get 0
 *  ws: msa_workspace_size(MSA_OP_BACKWARD, B, Nq, Nk, Hkv, Hq, d, 0, Bs, K, dtype)
 *  Supported: BF16; d in {64, 128}; Bs in {32, 64, 128}; Hq / Hkv in
 *  {1, 2, 4, 8}; 1 <= K <= 64. Other sizes return MSA_ERR_UNSUPPORTED.
 *  Out-of-range sel entries set MSA_ERR_BOUNDS in the workspace status and
 *  are skipped.
 *  Determinism: dq is a fixed-order sum (per-slot partials merged in slot
 *  order) and repeats bit for bit. dk and dv sum contributions of every query
 *  row that attends a key; they are accumulated in fp32 with atomic adds whose
 *  order varies from run to run, so they can differ in the last bits between
 *  runs (the forward's outputs, sel, out and lse, are deterministic). */
msa_status_t msa_sparse_attn_backward(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                      const float* lse, const int32_t* sel, const int32_t* q_offset,
                                      const int32_t* kv_len, int B, int Nq, int Nk, int Hq, int Hkv, int d, int Bs,
                                      int K, float scale, int dtype, void* dq, void* dk, void* dv, void* ws,
                                      size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, returns the sticky device status of workspace `ws`
 * (MSA_OK, MSA_ERR_TIMEOUT or MSA_ERR_BOUNDS) and clears it. Returns
 * MSA_ERR_CUDA if the stream reports an error. */
msa_status_t msa_read_status(void* ws, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* msa_status_string(msa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
