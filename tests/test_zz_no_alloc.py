"""msa_index_select_noalloc: the selection entry point for callers that cannot
allocate device memory (a plugin running under another framework's allocator,
a process with a fixed device-memory budget). It runs on a static scratch
array inside the library. Its output must equal msa_index_select's and the
oracle's on consecutive calls (different problems, so each call runs over the
previous call's stale scratch), with and without a caller-owned block_max;
rows whose kv_len is out of range must come back as -1 rows; a problem larger
than the static scratch must be refused before anything is enqueued.
Collected last on purpose."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import block_sparse_long_select_gb300 as msa
import oracle
import synth

DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(w, kv_len=None):
    iq = synth.device_tensor(w, "iq", DEV)
    ik = synth.device_tensor(w, "ik", DEV)
    kl_h = synth.kv_lens(w) if kv_len is None else np.asarray(kv_len, np.int32)
    qo_h = synth.q_offsets(w) if kv_len is None else (kl_h - w.Nq).astype(np.int32)
    return iq, ik, torch.from_numpy(qo_h).to(DEV), torch.from_numpy(kl_h).to(DEV), qo_h, kl_h


def _oracle(w, qo_h, kl_h, want_block_max=False):
    iq, ik = synth.host_tensor(w, "iq"), synth.host_tensor(w, "ik")
    rb, ri = oracle.all_rows(w.B, w.Nq)
    return oracle.index_select(iq.reshape(-1, w.G, w.di), ik, rb, ri, qo_h, kl_h, w.Bs, w.K,
                               want_block_max=want_block_max)


CASES = [
    # decode-shaped: 8 sequences, one query each, ragged KV lengths
    synth.scaled(synth.WORKLOADS["decode_b64"], B=8, Nk=8192, kv_len_range=(100, 8192)),
    # prefill-shaped bf16 (the workspace entry point takes its tensor-core path here)
    synth.scaled(synth.WORKLOADS["prefill_8k"], Nq=2048, Nk=2048, Bs=64, K=8, hot="first4"),
    # fp32
    synth.WORKLOADS["tiny_fp32"],
]


@pytest.mark.gpu
def test_noalloc_matches_index_select_and_oracle(cuda_ok):
    torch.cuda.set_device(DEV)
    for w in CASES + CASES[:1]:  # consecutive calls share (and inherit) the static scratch
        iq, ik, qo, kl, qo_h, kl_h = _inputs(w)
        ref = msa.msa_index_select(iq, ik, qo, kl, w.Bs, w.K)
        got = torch.full_like(ref, -7)
        msa.msa_index_select_noalloc(iq, ik, qo, kl, w.Bs, w.K, sel=got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), w.name
        osel = _oracle(w, qo_h, kl_h)
        assert np.array_equal(got.cpu().numpy().reshape(osel.shape), osel), w.name


@pytest.mark.gpu
def test_noalloc_with_block_max(cuda_ok):
    """Caller-owned block_max: the static array then holds only the status
    word; both outputs equal msa_index_select's and the oracle's."""
    torch.cuda.set_device(DEV)
    w = synth.scaled(synth.WORKLOADS["prefill_8k"], B=2, Nq=600, Nk=600, Bs=32, K=6)
    iq, ik, qo, kl, qo_h, kl_h = _inputs(w)
    nblk = (w.Nk + w.Bs - 1) // w.Bs
    bm_ref = torch.full((w.B, w.Nq, w.G, nblk), 7.0, device=DEV)
    ref = msa.msa_index_select(iq, ik, qo, kl, w.Bs, w.K, block_max=bm_ref)
    bm = torch.full_like(bm_ref, -7.0)
    got = torch.full_like(ref, -7)
    for _ in range(2):
        msa.msa_index_select_noalloc(iq, ik, qo, kl, w.Bs, w.K, sel=got, block_max=bm)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        assert torch.equal(torch.isnan(bm), torch.isnan(bm_ref))
        assert torch.equal(torch.nan_to_num(bm, nan=0.0), torch.nan_to_num(bm_ref, nan=0.0))
    osel, obm = _oracle(w, qo_h, kl_h, want_block_max=True)
    assert np.array_equal(got.cpu().numpy().reshape(osel.shape), osel)
    g = bm.cpu().numpy().reshape(obm.shape).astype(np.float64)
    vis = ~np.isnan(obm)
    assert np.array_equal(np.isnan(g), ~vis) and np.array_equal(g[vis], obm[vis])


@pytest.mark.gpu
def test_noalloc_out_of_range_rows(cuda_ok):
    """A sequence whose kv_len exceeds Nk: its rows come back as -1 (the
    device check skips them); the other sequence's rows are the oracle's."""
    torch.cuda.set_device(DEV)
    w = synth.scaled(synth.WORKLOADS["prefill_8k"], B=2, Nq=200, Nk=700, Hq=8, Hkv=2, Bs=64, K=4)
    kv_len = np.array([700, 701], np.int32)  # sequence 1 claims one key more than Nk
    iq, ik, qo, kl, qo_h, kl_h = _inputs(w, kv_len)
    got = torch.full((w.B, w.Nq, w.G, w.K), 9, dtype=torch.int32, device=DEV)
    msa.msa_index_select_noalloc(iq, ik, qo, kl, w.Bs, w.K, sel=got)
    torch.cuda.synchronize()
    g = got.cpu().numpy()
    assert (g[1] == -1).all()
    w0 = synth.scaled(w, B=1)
    osel = _oracle(w0, qo_h[:1], kl_h[:1])
    assert np.array_equal(g[0].reshape(osel.shape), osel)


def test_noalloc_rejects_oversize():
    """The size check runs before any CUDA call. It runs in a child process
    that sees no GPU, so that a check moved after the launches would come back
    as MSA_ERR_CUDA there instead of writing through the fake pointers."""
    code = r"""
import ctypes, sys
sys.path.insert(0, %r)
import block_sparse_long_select_gb300 as msa
lib = msa.load_library()
fake = ctypes.c_void_p(0x1000)
# a table of 1 x 65536 x 8 x 1024 blocks x 4 B = 2 GiB > 32 MiB
print(lib.msa_index_select_noalloc(fake, fake, None, None, 1, 65536, 131072, 8, 64, 128, 16, 0, fake, None, None))
""" % ROOT
    lib_file = msa.lib_path()
    if not os.path.exists(lib_file):
        msa.build()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert int(r.stdout.strip().splitlines()[-1]) == 3  # MSA_ERR_WORKSPACE
