"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
on synth inputs generated on the device, run the oracle on the same inputs
regenerated on the host, compare."""
from __future__ import annotations

import numpy as np
import torch

import block_sparse_long_select_gb300 as msa
import oracle
import synth

# tolerances (fp64 oracle vs kernel output)
TOL = {"bf16": dict(max_abs=2e-2, mean_abs=2e-3, lse_abs=2e-3), "fp32": dict(max_abs=1e-4, mean_abs=1e-4,
                                                                                lse_abs=1e-4)}


def device_inputs(w, dev, names=("q", "k", "v", "iq", "ik")):
    return {n: synth.device_tensor(w, n, dev) for n in names}


def gpu_prefill(w, t, dev, q_offset=None, kv_len=None, with_lse=True):
    qo = torch.from_numpy(synth.q_offsets(w) if q_offset is None else np.asarray(q_offset, np.int32)).to(dev)
    kl = torch.from_numpy(synth.kv_lens(w) if kv_len is None else np.asarray(kv_len, np.int32)).to(dev)
    sel = msa.msa_index_select(t["iq"], t["ik"], qo, kl, w.Bs, w.K)
    lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device=dev) if with_lse else None
    out = msa.msa_sparse_attn_prefill(t["q"], t["k"], t["v"], sel, qo, kl, w.Bs, w.K, lse=lse)
    torch.cuda.synchronize()
    return sel, out, lse


def gpu_decode(w, t, dev):
    kl = torch.from_numpy(synth.kv_lens(w)).to(dev)
    sel = msa.msa_index_select(t["iq"], t["ik"], kl - 1, kl, w.Bs, w.K)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    out = msa.msa_sparse_attn_decode(t["q"][:, 0], t["k"], t["v"], sel, kl, w.Bs, w.K, lse=lse)
    torch.cuda.synchronize()
    return sel, out, lse


def host_inputs(w):
    return {n: synth.host_tensor(w, n) for n in ("q", "k", "v", "iq", "ik")}


def oracle_full(w, h, q_offset=None, kv_len=None):
    qo = synth.q_offsets(w) if q_offset is None else np.asarray(q_offset, np.int32)
    kl = synth.kv_lens(w) if kv_len is None else np.asarray(kv_len, np.int32)
    return oracle.msa_forward(h["q"], h["k"], h["v"], h["iq"], h["ik"], w.Bs, w.K, q_offset=qo, kv_len=kl)


def oracle_selection_rows(w, rows_b, rows_i, ik_full=None):
    """Oracle selection for listed rows, regenerating iq rows on the host."""
    rows_b, rows_i = np.asarray(rows_b, np.int32), np.asarray(rows_i, np.int32)
    iq = np.stack([synth.host_rows(w, "iq", int(b), [int(i)])[0] for b, i in zip(rows_b, rows_i)])
    ik = synth.host_tensor(w, "ik") if ik_full is None else ik_full
    return oracle.index_select(iq, ik, rows_b, rows_i, synth.q_offsets(w), synth.kv_lens(w), w.Bs, w.K)


def sparse_kv(w, b, blocks):
    """Host K/V of one sequence with only ``blocks`` filled (others never read)."""
    k = np.zeros((1, w.Nk, w.Hkv, w.d), np.float32)
    v = np.zeros((1, w.Nk, w.Hkv, w.d), np.float32)
    row = w.Hkv * w.d
    for t in sorted(set(int(x) for x in blocks if x >= 0)):
        j0, j1 = t * w.Bs, min((t + 1) * w.Bs, w.Nk)
        start = (b * w.Nk + j0) * row
        k[0, j0:j1] = synth.host_range(w, "k", start, (j1 - j0) * row).reshape(j1 - j0, w.Hkv, w.d)
        v[0, j0:j1] = synth.host_range(w, "v", start, (j1 - j0) * row).reshape(j1 - j0, w.Hkv, w.d)
    return k, v


def oracle_attention_rows(w, rows_b, rows_i, sel_rows):
    """Oracle attention for listed rows given the oracle's own selection."""
    rows_b, rows_i = np.asarray(rows_b, np.int32), np.asarray(rows_i, np.int32)
    qo, kl = synth.q_offsets(w), synth.kv_lens(w)
    out = np.empty((len(rows_b), w.Hq, w.d))
    lse = np.empty((len(rows_b), w.Hq))
    for b in np.unique(rows_b):
        idx = np.nonzero(rows_b == b)[0]
        k, v = sparse_kv(w, int(b), sel_rows[idx].reshape(-1))
        q = np.stack([synth.host_rows(w, "q", int(b), [int(rows_i[n])])[0] for n in idx])
        o, l = oracle.sparse_attn(q, k, v, sel_rows[idx], np.zeros(len(idx), np.int32), rows_i[idx],
                                  qo[b:b + 1], kl[b:b + 1], w.Bs, w.K)
        out[idx], lse[idx] = o, l
    return out, lse


def assert_close(got, want, dtype, what, lse=False):
    tol = TOL[dtype]
    err = np.abs(np.asarray(got, np.float64) - want)
    if lse:
        assert err.max() <= tol["lse_abs"], f"{what}: lse max err {err.max():.3g}"
        return
    assert err.max() <= tol["max_abs"], f"{what}: max abs err {err.max():.3g} > {tol['max_abs']}"
    assert err.mean() <= tol["mean_abs"], f"{what}: mean abs err {err.mean():.3g} > {tol['mean_abs']}"


def check_structure(sel, q_offset, kv_len, Bs, K):
    """Properties of a selection that hold at any size: ascending, unique, in
    range, local block present, count = min(K, loc + 1), -1 padding last."""
    sel = sel.astype(np.int64)
    B, Nq, G, _ = sel.shape
    pos = np.asarray(q_offset)[:, None] + np.arange(Nq)[None, :]
    loc = (pos // Bs)[:, :, None, None]  # [B, Nq, 1, 1]
    valid = sel >= 0
    cnt = valid.sum(-1)
    assert np.array_equal(cnt, np.broadcast_to(np.minimum(K, loc[..., 0] + 1), cnt.shape)), "selection count"
    # -1 only at the tail
    assert np.all(np.diff(valid.astype(np.int8), axis=-1) <= 0), "padding not at the tail"
    s = np.where(valid, sel, np.iinfo(np.int64).max)
    d = np.diff(s, axis=-1)
    assert np.all((d > 0) | ~valid[..., 1:]), "not strictly ascending"
    assert np.all(np.where(valid, sel <= loc, True)), "block after the local block"
    assert np.all((sel == loc).any(-1)), "local block missing"
