"""GPU parity of the Main Branch backward (msa_sparse_attn_backward through the
C ABI) against the oracle's fp64 backward on the same bf16 inputs. The GPU
takes the selection, output and lse of the library's own forward (the
selection is first checked bit for bit against the oracle's); the oracle
recomputes the forward in fp64 from the definition.

Tolerance per gradient tensor (the pages give none; derived): the kernels
round P and dS to bf16 before the dV, dK and dQ products (relative 2^-9
each), take delta = dout . out from the bf16 forward output, accumulate in
fp32 and round each result to bf16 once (2^-9); dq is also rounded to bf16
once per selected block (its slot partials) before the fp32 sum. The gradients are sums of
terms of both signs, so the error is bounded relative to the magnitudes
summed, not to the (possibly cancelling) result: max |err| <= 2e-2 max |ref|
and mean |err| <= 1e-2 mean |ref| over each of dq, dk, dv.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import block_sparse_long_select_gb300 as msa
import oracle
import synth
from parity import device_inputs, gpu_prefill, sparse_kv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BASE = synth.WORKLOADS["prefill_8k"]
HERE = os.path.dirname(os.path.abspath(__file__))
MAX_REL, MEAN_REL = 2e-2, 1e-2


def _assert_grad(got, want, what, scale_floor=0.0):
    """scale_floor: a magnitude of the whole gradient tensor, for checks on a
    few rows whose own values may cancel to zero (a row attending only to
    itself has dq = 0 exactly)."""
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    ref_max = max(np.abs(want).max(), scale_floor)
    ref_mean = max(np.abs(want).mean(), scale_floor)
    assert err.max() <= MAX_REL * ref_max, f"{what}: max err {err.max():.3g} vs max |ref| {ref_max:.3g}"
    assert err.mean() <= MEAN_REL * ref_mean, f"{what}: mean err {err.mean():.3g} vs mean |ref| {ref_mean:.3g}"


def _dout_workload(w):
    return synth.scaled(w, seed=w.seed + 1000)  # the output gradient: a q-shaped tensor of another seed


def _gpu_backward(w, t, qo=None, kl=None):
    sel, out, lse = gpu_prefill(w, t, DEV, qo, kl)
    dout = synth.device_tensor(_dout_workload(w), "q", DEV)
    qo_t = torch.from_numpy(synth.q_offsets(w) if qo is None else np.asarray(qo, np.int32)).to(DEV)
    kl_t = torch.from_numpy(synth.kv_lens(w) if kl is None else np.asarray(kl, np.int32)).to(DEV)
    ws = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_BACKWARD, w.B, w.Nq, w.Nk, w.Hkv, w.Hq, w.d, 0, w.Bs, w.K,
                                              msa.MSA_BF16), DEV)
    dq, dk, dv = msa.msa_sparse_attn_backward(t["q"], t["k"], t["v"], out, dout, lse, sel, qo_t, kl_t, w.Bs, w.K,
                                              ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_status(ws) == 0
    return sel, dout, dq, dk, dv


def check_case(w, qo=None, kl=None):
    """Full parity of dq, dk, dv for one workload (all rows)."""
    torch.cuda.set_device(DEV)
    t = device_inputs(w, DEV)
    qo_ = synth.q_offsets(w) if qo is None else np.asarray(qo, np.int32)
    kl_ = synth.kv_lens(w) if kl is None else np.asarray(kl, np.int32)
    sel, dout, dq, dk, dv = _gpu_backward(w, t, qo, kl)
    h = {n: synth.host_tensor(w, n) for n in ("q", "k", "v", "iq", "ik")}
    g = synth.host_tensor(_dout_workload(w), "q")
    rb, ri = oracle.all_rows(w.B, w.Nq)
    osel = oracle.index_select(h["iq"].reshape(-1, w.G, w.di), h["ik"], rb, ri, qo_, kl_, w.Bs, w.K)
    assert np.array_equal(sel.cpu().numpy().reshape(osel.shape), osel), "selection differs from the oracle"
    odq, odk, odv = oracle.sparse_attn_backward(h["q"].reshape(-1, w.Hq, w.d), h["k"], h["v"],
                                                g.reshape(-1, w.Hq, w.d), osel, rb, ri, qo_, kl_, w.Bs, w.K)
    _assert_grad(dq.float().cpu().numpy().reshape(odq.shape), odq, "dq")
    _assert_grad(dk.float().cpu().numpy(), odk, "dk")
    _assert_grad(dv.float().cpu().numpy(), odv, "dv")


CASES = {  # every (d, Bs) build, head ratios 1..8, hot blocks (bins split over CTAs)
    "d128_bs128_hpg4": synth.scaled(BASE, B=2, Nq=1100, Nk=1100, Bs=128, K=5),
    "d128_bs64_hpg4_hot": synth.scaled(BASE, B=1, Nq=1000, Nk=1000, Bs=64, K=6, hot="first4"),
    "d128_bs32_hpg4": synth.scaled(BASE, B=1, Nq=900, Nk=900, Bs=32, K=12),
    "d64_bs64_hpg2": synth.scaled(BASE, B=2, Nq=700, Nk=700, Hq=8, Hkv=4, d=64, di=32, Bs=64, K=5),
    "d64_bs32_hpg8": synth.scaled(BASE, B=1, Nq=800, Nk=800, Hq=16, Hkv=2, d=64, di=32, Bs=32, K=9),
    "d64_bs128_hpg1": synth.scaled(BASE, B=1, Nq=600, Nk=600, Hq=4, Hkv=4, d=64, di=32, Bs=128, K=3),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_small(name):
    check_case(CASES[name])


def test_backward_chunked_offsets():
    """Queries are the last Nq keys of ragged sequences (q_offset > 0, kv_len < Nk)."""
    w = synth.scaled(BASE, B=3, Nq=300, Nk=1100, Bs=64, K=6)
    kl = np.array([1100, 900, 301], np.int32)
    check_case(w, (kl - 300).astype(np.int32), kl)


def test_backward_query_chunks_accumulate():
    """A small query chunk (MSA_PREFILL_CHUNK, read once per process) makes dk,
    dv accumulate over several chunks: run in a child process."""
    code = ("import sys; sys.path[:0] = [%r, %r]; import test_gpu_backward as t; "
            "t.check_case(t.CASES['d128_bs64_hpg4_hot']); t.check_case(t.CASES['d64_bs32_hpg8']); print('ok')"
            % (HERE, os.path.dirname(HERE)))
    env = dict(os.environ, MSA_PREFILL_CHUNK="256")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]


@pytest.mark.slow
def test_backward_128k_properties_and_sampled_rows():
    """The bench workload (128K, Bs 128, K 16): closed forms of the sums
    (sum_j dk_j = 0, sum_j dv_j = the group's summed dout, sum q.dq = sum k.dk
    per kv head) over the whole sequence, and dq of a stratified row sample
    against the oracle."""
    torch.cuda.set_device(DEV)
    w = synth.WORKLOADS["prefill_128k_bs128"]
    t = device_inputs(w, DEV)
    sel, dout, dq, dk, dv = _gpu_backward(w, t)
    hpg = w.Hq // w.Hkv
    for x in (dq, dk, dv):
        assert bool(torch.isfinite(x.float()).all())
    sum_dk = dk[0].double().sum(0)                      # [Hkv, d]
    abs_dk = dk[0].double().abs().sum(0)
    assert bool((sum_dk.abs() <= 1e-2 * abs_dk + 1e-3).all()), float((sum_dk.abs() / abs_dk).max())
    want_dv = dout[0].double().view(w.Nq, w.Hkv, hpg, w.d).sum((0, 2))
    got_dv = dv[0].double().sum(0)
    scale_dv = dv[0].double().abs().sum(0)
    assert bool(((got_dv - want_dv).abs() <= 1e-2 * scale_dv + 1e-3).all())
    qdq = (t["q"][0].double() * dq[0].double()).view(w.Nq, w.Hkv, hpg, w.d).sum((0, 2, 3))
    kdk = (t["k"][0].double() * dk[0].double()).sum((0, 2))
    mag = (t["k"][0].double() * dk[0].double()).abs().sum((0, 2))
    assert bool(((qdq - kdk).abs() <= 2e-2 * mag).all())
    sel_h = sel.cpu().numpy()
    dq_h = dq.float().cpu().numpy()
    dq_scale = float(np.abs(dq_h).mean())
    del t, dk, dv
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 3), np.arange(2046, 2050), np.arange(w.Nq - 3, w.Nq),
                                     rng.choice(w.Nq, 24, replace=False)])).astype(np.int32)
    ik = synth.host_tensor(w, "ik")
    qo, kl_ = synth.q_offsets(w), synth.kv_lens(w)
    wg = _dout_workload(w)
    for r in rows:
        srow = sel_h[0, r]
        iq = synth.host_rows(w, "iq", 0, [int(r)])
        osel = oracle.index_select(iq, ik, np.zeros(1, np.int32), np.array([r], np.int32), qo, kl_, w.Bs, w.K)
        assert np.array_equal(osel[0], srow), f"row {r}: selection"
        k, v = sparse_kv(w, 0, srow.reshape(-1))
        q = synth.host_rows(w, "q", 0, [int(r)])
        g = synth.host_rows(wg, "q", 0, [int(r)])
        odq, _, _ = oracle.sparse_attn_backward(q, k, v, g, srow[None], np.zeros(1, np.int32), np.array([r], np.int32),
                                                qo, kl_, w.Bs, w.K)
        _assert_grad(dq_h[0, r][None], odq, f"dq row {r}", scale_floor=dq_scale)


@pytest.mark.parametrize("Bs", [128, 32])
def test_backward_few_queries(Bs):
    """Three queries at the end of ragged sequences: a handful of tiles, most
    CTAs of the persistent grid without work."""
    w = synth.scaled(BASE, B=2, Nq=3, Nk=260, Bs=Bs, K=4)
    kl = np.array([260, 200], np.int32)
    check_case(w, (kl - 3).astype(np.int32), kl)
