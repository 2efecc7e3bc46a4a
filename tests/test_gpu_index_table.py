"""GPU parity of the Index Branch at large K (K - 1 > 15): the tensor-core
kernel writes the candidate block maxima of a chunk of rows to a workspace
table and a warp-per-row kernel selects from it. Selections must equal the
oracle's bit for bit (hyper.ai summary of 2606.13392, "方法": block max
pooling, top-K with the local block; ties go to the lower block).

Covered: both per-lane sample sizes (K - 1 - fs <= 32 and above), the
table's float2 and float4 row stores (blocks of 128 and of 64 / 32 keys),
index heads of 32 and 64, ragged sequences with chunked-prefill offsets,
hot blocks, the forced start block, rows whose candidates all tie and rows
whose per-lane sample bounds nothing (the selection list overflows and the
kernel bisects over the row itself; both closed forms), heavy integer ties
below the list bound, and several table chunks per call (a child process
with MSA_INDEX_TABLE_UNITS).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
HERE = os.path.dirname(os.path.abspath(__file__))

BASE = synth.WORKLOADS["prefill_8k"]
# (workload, kv_len per sequence or None for Nk); queries are the last Nq keys
CASES = {
    "bs64_k32_ragged": (synth.scaled(BASE, B=3, Nq=1500, Nk=3000, Bs=64, K=32), [3000, 1700, 2345]),
    "bs32_k64": (synth.scaled(BASE, B=1, Nq=3000, Nk=3000, Bs=32, K=64), None),
    "bs32_k33_sample1": (synth.scaled(BASE, B=1, Nq=2600, Nk=2600, Bs=32, K=33), None),
    "bs32_k34_sample2": (synth.scaled(BASE, B=2, Nq=1900, Nk=2100, Bs=32, K=34), [2100, 1999]),
    "bs128_k20_pairs": (synth.scaled(BASE, B=1, Nq=4100, Nk=4100, Bs=128, K=20), None),
    "bs64_k17_smallest": (synth.scaled(BASE, B=1, Nq=2000, Nk=2000, Bs=64, K=17), None),
    "di32_bs32_k40": (synth.scaled(BASE, B=2, Nq=1300, Nk=1300, Hq=8, Hkv=2, d=64, di=32, Bs=32, K=40), None),
    "bs32_k64_hot": (synth.scaled(BASE, B=1, Nq=2500, Nk=2500, Bs=32, K=64, hot="first4"), None),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    torch.cuda.set_device(DEV)


def _offsets(w, kv):
    kl = np.full(w.B, w.Nk, np.int32) if kv is None else np.asarray(kv, np.int32)
    return (kl - w.Nq).astype(np.int32), kl


def _select(iq, ik, qo, kl, Bs, K, force_start=False):
    import block_sparse_long_select_gb300 as msa

    force = msa.MSA_FORCE_LOCAL | (msa.MSA_FORCE_START if force_start else 0)
    sel = msa.msa_index_select_v(iq, ik, torch.from_numpy(qo).to(DEV), torch.from_numpy(kl).to(DEV), Bs, K, force)
    torch.cuda.synchronize()
    return sel.cpu().numpy()


def _oracle(iq_h, ik_h, qo, kl, Bs, K, force_start=False):
    import oracle

    B, Nq, G, di = iq_h.shape
    rb, ri = oracle.all_rows(B, Nq)
    return oracle.index_select(iq_h.reshape(-1, G, di), ik_h, rb, ri, qo, kl, Bs, K,
                               force_start=force_start).reshape(B, Nq, G, K)


def check_case(name, force_start=False):
    w, kv = CASES[name]
    qo, kl = _offsets(w, kv)
    iq = synth.device_tensor(w, "iq", DEV)
    ik = synth.device_tensor(w, "ik", DEV)
    got = _select(iq, ik, qo, kl, w.Bs, w.K, force_start)
    want = _oracle(synth.host_tensor(w, "iq"), synth.host_tensor(w, "ik"), qo, kl, w.Bs, w.K, force_start)
    bad = np.argwhere((got != want).any(-1))
    assert bad.size == 0, f"{name}: {len(bad)} rows differ, first {bad[:3].tolist()}"


@pytest.mark.parametrize("name", sorted(CASES))
def test_table_selection(name):
    check_case(name)


@pytest.mark.parametrize("name", ["bs64_k32_ragged", "bs32_k34_sample2"])
def test_table_selection_force_start(name):
    check_case(name, force_start=True)


def _small_int_inputs(B, Nq, Nk, G, di, lo, hi, seed):
    g = np.random.default_rng(seed)
    iq = g.integers(lo, hi + 1, size=(B, Nq, G, di)).astype(np.float32)
    ik = g.integers(lo, hi + 1, size=(B, Nk, di)).astype(np.float32)
    return iq, ik


def test_all_tied_rows_closed_form():
    """Index queries of zeros: every block maximum is 0, so every row with more
    than K visible blocks takes blocks 0 .. K-2 (ties go to the lower block)
    and its local block. With Bs 32 and up to 400 blocks per row the tied
    candidates overflow the selection list."""
    B, Nq, Nk, G, di, Bs, K = 1, 12800, 12800, 8, 64, 32, 64
    iq_h = np.zeros((B, Nq, G, di), np.float32)
    ik_h = np.random.default_rng(7).standard_normal((B, Nk, di)).astype(np.float32)
    qo, kl = np.zeros(B, np.int32), np.full(B, Nk, np.int32)
    iq = torch.from_numpy(iq_h).to(DEV, torch.bfloat16)
    ik = torch.from_numpy(ik_h).to(DEV, torch.bfloat16)
    got = _select(iq, ik, qo, kl, Bs, K)
    loc = np.arange(Nq) // Bs
    want = np.where((np.arange(K)[None, :] <= loc[:, None]), np.arange(K)[None, :], -1)
    ranked = loc + 1 > K
    want[ranked, : K - 1] = np.arange(K - 1)
    want[ranked, K - 1] = loc[ranked]
    assert np.array_equal(got[0], np.broadcast_to(want[:, None, :], (Nq, G, K)))


def test_list_overflow_bisection_closed_form():
    """Scores equal the first index-key component (index queries e_0). Blocks
    t = 0, 32, 64, ... get the distinct maxima t / 32 + 1 and every other block
    0, so each lane's best two values are 0 except lane 0's: the bound T is 0,
    every candidate is kept, the list overflows for rows past 256 blocks, and
    v* comes from a full bisection over the row. Closed form: the blocks
    t = 0 mod 32 below loc, then the lowest other blocks, then loc."""
    B, Nq, Nk, G, di, Bs, K = 1, 12800, 12800, 8, 64, 32, 64
    iq_h = np.zeros((B, Nq, G, di), np.float32)
    iq_h[..., 0] = 1.0
    ik_h = np.zeros((B, Nk, di), np.float32)
    t_of_key = np.arange(Nk) // Bs
    ik_h[0, :, 0] = np.where(t_of_key % 32 == 0, t_of_key // 32 + 1, 0)
    qo, kl = np.zeros(B, np.int32), np.full(B, Nk, np.int32)
    got = _select(torch.from_numpy(iq_h).to(DEV, torch.bfloat16), torch.from_numpy(ik_h).to(DEV, torch.bfloat16),
                  qo, kl, Bs, K)
    loc = np.arange(Nq) // Bs
    for i in range(0, Nq, 37):
        L = loc[i]
        if L + 1 <= K:
            want = [k if k <= L else -1 for k in range(K)]
        else:
            big = [t for t in range(L) if t % 32 == 0]
            rest = [t for t in range(L) if t % 32 != 0][: K - 1 - len(big)]
            want = sorted(big + rest) + [L]
        assert np.array_equal(got[0, i], np.broadcast_to(np.array(want), (G, K))), i


@pytest.mark.parametrize("lo,hi", [(-1, 1), (0, 2)])
def test_integer_ties(lo, hi):
    """Integer scores from a small range: many equal block maxima at the
    selection threshold, compared in exact arithmetic with the oracle."""
    B, Nq, Nk, G, di, Bs, K = 1, 2400, 2400, 8, 64, 32, 48
    iq_h, ik_h = _small_int_inputs(B, Nq, Nk, G, di, lo, hi, seed=11 + lo)
    qo, kl = np.zeros(B, np.int32), np.full(B, Nk, np.int32)
    got = _select(torch.from_numpy(iq_h).to(DEV, torch.bfloat16), torch.from_numpy(ik_h).to(DEV, torch.bfloat16),
                  qo, kl, Bs, K)
    want = _oracle(iq_h, ik_h, qo, kl, Bs, K)
    assert np.array_equal(got, want)


def test_table_chunks():
    """Three units (768 rows) per table chunk instead of the ~4 GiB default, in
    a child process (the setting is read once per process): the rows of every
    chunk, including a short last one, are selected from their own chunk."""
    code = ("import sys; sys.path[:0] = [%r, %r]; import test_gpu_index_table as t; import torch; "
            "torch.cuda.set_device(0); "
            "[t.check_case(n) for n in ('bs64_k32_ragged', 'bs32_k34_sample2', 'bs128_k20_pairs')]; "
            "t.check_case('bs64_k32_ragged', force_start=True); print('ok')" % (HERE, os.path.dirname(HERE)))
    env = dict(os.environ, MSA_INDEX_TABLE_UNITS="3")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
