"""GPU parity of the KL auxiliary forward (msa_kl_aux_forward through the C
ABI) against the oracle: the selection and lse come from the library's own
index select and prefill attention, the oracle recomputes the divergence from
the definition in fp64 on the same selection.

Tolerance: |kl - oracle| <= 5e-3 + 1e-3 |oracle|. The kernel's head-averaged
probabilities carry a relative error of about 1e-5 (bf16 inputs multiply
exactly, fp32 sums, the forward's fp32 lse, hardware exp2); the largest term
is sum_j p_j s_j with integer index scores |s_j| up to a few hundred, so the
absolute error stays near 1e-3.
"""
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


def _assert_kl(got, want, what):
    err = np.abs(np.asarray(got, np.float64) - want)
    bound = 5e-3 + 1e-3 * np.abs(want)
    assert (err <= bound).all(), f"{what}: worst excess {(err - bound).max():.3g} (max err {err.max():.3g})"


def _gpu_kl(w, t, sel, lse, qo, kl_):
    kl = msa.msa_kl_aux_forward(t["q"], t["k"], t["iq"], t["ik"], sel, lse, torch.from_numpy(qo).to(DEV),
                                torch.from_numpy(kl_).to(DEV), w.Bs, w.K)
    torch.cuda.synchronize()
    return kl.cpu().numpy()


CASES = {
    "bs64_hpg4": synth.scaled(BASE, B=1, Nq=1000, Nk=1000, Bs=64, K=6),
    "bs128_hpg4": synth.scaled(BASE, B=2, Nq=1100, Nk=1100, Bs=128, K=5),
    "bs32_hpg4_hot": synth.scaled(BASE, B=1, Nq=900, Nk=900, Bs=32, K=12, hot="first4"),
    "d64_di32_hpg2": synth.scaled(BASE, B=2, Nq=700, Nk=700, Hq=8, Hkv=4, d=64, di=32, Bs=64, K=5),
    "d64_di32_hpg8": synth.scaled(BASE, B=1, Nq=800, Nk=800, Hq=16, Hkv=2, d=64, di=32, Bs=32, K=9),
    # blocks of 128 keys with d 128 / di 64 take the tcgen05 tile pass: head ratios 2 and 8, hot blocks
    "bs128_hpg2": synth.scaled(BASE, B=1, Nq=1200, Nk=1200, Hq=16, Hkv=8, Bs=128, K=5),
    "bs128_hpg8_hot": synth.scaled(BASE, B=1, Nq=1300, Nk=1300, Hq=32, Hkv=4, Bs=128, K=6, hot="first4"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_kl_aux_small(name):
    torch.cuda.set_device(DEV)
    w = CASES[name]
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV)
    qo, kl_ = synth.q_offsets(w), synth.kv_lens(w)
    got = _gpu_kl(w, t, sel, lse, qo, kl_)
    h = {n: synth.host_tensor(w, n) for n in ("q", "k", "iq", "ik")}
    rb, ri = oracle.all_rows(w.B, w.Nq)
    osel = oracle.index_select(h["iq"].reshape(-1, w.G, w.di), h["ik"], rb, ri, qo, kl_, w.Bs, w.K)
    assert np.array_equal(sel.cpu().numpy().reshape(osel.shape), osel)
    want = oracle.kl_aux(h["q"].reshape(-1, w.Hq, w.d), h["k"], h["iq"].reshape(-1, w.G, w.di), h["ik"], osel, rb, ri,
                         qo, kl_, w.Bs, w.K)
    _assert_kl(got.reshape(want.shape), want, name)


def test_kl_aux_chunked_offsets():
    """Queries are the last Nq keys of ragged sequences (q_offset > 0, kv_len < Nk)."""
    torch.cuda.set_device(DEV)
    w = synth.scaled(BASE, B=3, Nq=300, Nk=1100, Bs=64, K=6)
    kl_ = np.array([1100, 900, 301], np.int32)
    qo = (kl_ - 300).astype(np.int32)
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV, qo, kl_)
    got = _gpu_kl(w, t, sel, lse, qo, kl_)
    h = {n: synth.host_tensor(w, n) for n in ("q", "k", "iq", "ik")}
    rb, ri = oracle.all_rows(w.B, w.Nq)
    osel = oracle.index_select(h["iq"].reshape(-1, w.G, w.di), h["ik"], rb, ri, qo, kl_, w.Bs, w.K)
    want = oracle.kl_aux(h["q"].reshape(-1, w.Hq, w.d), h["k"], h["iq"].reshape(-1, w.G, w.di), h["ik"], osel, rb, ri,
                         qo, kl_, w.Bs, w.K)
    _assert_kl(got.reshape(want.shape), want, "chunked")


@pytest.mark.slow
def test_kl_aux_128k_sampled_rows():
    """The bench workload (128K, Bs 128, K 16): every row finite and >= 0, a stratified sample against the oracle."""
    torch.cuda.set_device(DEV)
    w = synth.WORKLOADS["prefill_128k_bs128"]
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV)
    qo, kl_ = synth.q_offsets(w), synth.kv_lens(w)
    got = _gpu_kl(w, t, sel, lse, qo, kl_)
    sel_h = sel.cpu().numpy()
    del t, out
    assert np.isfinite(got).all() and got.min() > -1e-3
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 4), np.arange(2044, 2052), np.arange(w.Nq - 4, w.Nq),
                                     rng.choice(w.Nq, 48, replace=False)])).astype(np.int32)
    ik = synth.host_tensor(w, "ik")
    for r in rows:
        srow = sel_h[0, r]
        k, _ = sparse_kv(w, 0, srow.reshape(-1))
        q = synth.host_rows(w, "q", 0, [int(r)])
        iq = synth.host_rows(w, "iq", 0, [int(r)])
        want = oracle.kl_aux(q, k, iq, ik, srow[None], np.zeros(1, np.int32), np.array([r], np.int32), qo, kl_, w.Bs,
                             w.K)
        _assert_kl(got[0, r][None], want, f"row {r}")


@pytest.mark.parametrize("Bs", [128, 32])
def test_kl_aux_few_queries(Bs):
    """Three queries at the end of ragged sequences (most CTAs without tiles)."""
    torch.cuda.set_device(DEV)
    w = synth.scaled(BASE, B=2, Nq=3, Nk=260, Bs=Bs, K=4)
    kl_ = np.array([260, 200], np.int32)
    qo = (kl_ - 3).astype(np.int32)
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV, qo, kl_)
    got = _gpu_kl(w, t, sel, lse, qo, kl_)
    h = {n: synth.host_tensor(w, n) for n in ("q", "k", "iq", "ik")}
    rb, ri = oracle.all_rows(w.B, w.Nq)
    osel = oracle.index_select(h["iq"].reshape(-1, w.G, w.di), h["ik"], rb, ri, qo, kl_, w.Bs, w.K)
    assert np.array_equal(sel.cpu().numpy().reshape(osel.shape), osel)
    want = oracle.kl_aux(h["q"].reshape(-1, w.Hq, w.d), h["k"], h["iq"].reshape(-1, w.G, w.di), h["ik"], osel, rb, ri,
                         qo, kl_, w.Bs, w.K)
    _assert_kl(got.reshape(want.shape), want, f"few queries Bs {Bs}")
