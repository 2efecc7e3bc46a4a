"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Selections must match bit for bit; outputs within the stated tolerances
(bf16: max-abs 2e-2, mean-abs 2e-3; fp32: 1e-4) element by element.
"""
import numpy as np
import pytest
import torch

import synth
from parity import (assert_close, check_structure, device_inputs, gpu_decode, gpu_prefill, host_inputs,
                    oracle_attention_rows, oracle_full, oracle_selection_rows)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# small problems that span several tiles and leave ragged tails
BASE = synth.WORKLOADS["prefill_8k"]
SMALL = {
    "bf16_ragged_bs64": synth.scaled(BASE, B=2, Nq=1000, Nk=1000, Bs=64, K=4),
    "bf16_bs32_k8": synth.scaled(BASE, B=1, Nq=777, Nk=777, Bs=32, K=8),
    "bf16_bs128_k3": synth.scaled(BASE, B=1, Nq=1500, Nk=1500, Bs=128, K=3),
    "bf16_k1_local_only": synth.scaled(BASE, B=1, Nq=300, Nk=300, Bs=32, K=1),
    "bf16_d64_di32": synth.scaled(BASE, B=2, Nq=640, Nk=640, Hq=8, Hkv=2, d=64, di=32, Bs=64, K=5),
    "bf16_hot_blocks": synth.scaled(BASE, B=1, Nq=2048, Nk=2048, Bs=32, K=16, hot="first4"),
    "bf16_single_row": synth.scaled(BASE, B=1, Nq=1, Nk=1, Bs=128, K=16),
    # head ratios beyond 8 (tensor-core attention takes up to hpg * d = 2048)
    "bf16_hpg16": synth.scaled(BASE, B=1, Nq=600, Nk=600, Hq=32, Hkv=2, Bs=64, K=4),
    "bf16_hpg32_d64": synth.scaled(BASE, B=1, Nq=1100, Nk=1100, Hq=32, Hkv=1, d=64, di=32, Bs=128, K=3),
    # block sizes outside the tensor-core builds: the table index path and the CUDA-core attention
    "bf16_bs100_generic": synth.scaled(BASE, B=2, Nq=900, Nk=900, Hq=8, Hkv=2, Bs=100, K=5),
    "bf16_bs1_k64_tokens": synth.scaled(BASE, B=1, Nq=300, Nk=300, Hq=8, Hkv=2, Bs=1, K=64),
    "bf16_bs1024_k2": synth.scaled(BASE, B=1, Nq=2500, Nk=2500, Hq=8, Hkv=2, Bs=1024, K=2),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    torch.cuda.set_device(DEV)


def _compare_full(w, q_offset=None, kv_len=None):
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV, q_offset, kv_len)
    h = host_inputs(w)
    osel, oout, olse = oracle_full(w, h, q_offset, kv_len)
    assert np.array_equal(sel.cpu().numpy(), osel), f"{w.name}: selected blocks differ"
    assert_close(out.float().cpu().numpy(), oout, w.dtype, w.name)
    assert_close(lse.cpu().numpy(), olse, w.dtype, w.name, lse=True)


def test_tiny_fp32_full():
    """Tiny fp32 config: batch 1, seq 512, Hq 8, Hkv 2, d 64, di 32, block 32, K 4."""
    _compare_full(synth.WORKLOADS["tiny_fp32"])


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_bf16_full(name):
    _compare_full(SMALL[name])


def test_chunked_prefill_offsets():
    """Queries are the last Nq keys of ragged sequences (q_offset > 0, kv_len < Nk)."""
    w = synth.scaled(BASE, B=3, Nq=300, Nk=1100, Bs=64, K=6)
    kv_len = np.array([1100, 900, 301], np.int32)
    q_offset = kv_len - 300
    _compare_full(w, q_offset, kv_len)


def test_prefill_8k_bf16():
    """Prefill bf16 config (seq 8192, block 128, K 16), in the bench's launch
    configuration: every selection bit-exact and every output row (all 8192
    rows x 32 heads x 128 dims) and lse within the bf16 tolerances."""
    w = synth.WORKLOADS["prefill_8k"]
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV)
    sel = sel.cpu().numpy()
    h = host_inputs(w)
    osel, oout, olse = oracle_full(w, h)
    assert np.array_equal(sel, osel)
    assert_close(out.float().cpu().numpy(), oout, "bf16", w.name)
    assert_close(lse.cpu().numpy(), olse, "bf16", w.name, lse=True)


# the optional block_max output of msa_index_select (it takes the table path):
# block maxima of the visible keys, NaN past the local block
BLOCK_MAX_CASES = {
    "bf16_bs64": (synth.scaled(BASE, B=2, Nq=700, Nk=700, Bs=64, K=4), None),
    "bf16_bs100_chunked": (synth.scaled(BASE, B=3, Nq=300, Nk=1100, Hq=8, Hkv=2, Bs=100, K=5),
                           np.array([1100, 900, 301], np.int32)),
    "bf16_bs128_hot": (synth.scaled(BASE, B=1, Nq=1000, Nk=1000, Bs=128, K=3, hot="first4"), None),
    "fp32_tiny": (synth.WORKLOADS["tiny_fp32"], None),
    "bf16_one_query_rows": (synth.scaled(synth.WORKLOADS["decode_b64"], B=6, Nk=3000, kv_len_range=(1, 3000),
                                         Bs=64, K=8), None),
}


@pytest.mark.parametrize("name", sorted(BLOCK_MAX_CASES))
def test_block_max_output(name):
    """block_max element by element against the oracle's block maxima: exact
    (integer-valued index inputs make every score exact in fp32), NaN at
    exactly the blocks the oracle leaves out (t > loc); the selection too."""
    import block_sparse_long_select_gb300 as msa
    import oracle

    w, kv_len = BLOCK_MAX_CASES[name]
    kl = synth.kv_lens(w) if kv_len is None else kv_len
    qo = synth.q_offsets(w) if kv_len is None else (kl - w.Nq).astype(np.int32)
    t = device_inputs(w, DEV, names=("iq", "ik"))
    nblk = (w.Nk + w.Bs - 1) // w.Bs
    bm = torch.full((w.B, w.Nq, w.G, nblk), 12345.0, dtype=torch.float32, device=DEV)
    sel = msa.msa_index_select(t["iq"], t["ik"], torch.from_numpy(qo).to(DEV), torch.from_numpy(kl).to(DEV), w.Bs,
                               w.K, block_max=bm)
    torch.cuda.synchronize()
    iq, ik = synth.host_tensor(w, "iq"), synth.host_tensor(w, "ik")
    rb, ri = oracle.all_rows(w.B, w.Nq)
    osel, obm = oracle.index_select(iq.reshape(-1, w.G, w.di), ik, rb, ri, qo, kl, w.Bs, w.K, want_block_max=True)
    got = bm.cpu().numpy().reshape(obm.shape).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(obm)), f"{name}: visible blocks differ"
    vis = ~np.isnan(obm)
    assert np.array_equal(got[vis], obm[vis]), f"{name}: block maxima differ"
    assert np.array_equal(sel.cpu().numpy().reshape(osel.shape), osel), name


def test_decode_small():
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=5, Nk=4096, kv_len_range=(1, 4096))
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_decode(w, t, DEV)
    h = host_inputs(w)
    osel, oout, olse = oracle_full(w, h)
    assert np.array_equal(sel.cpu().numpy(), osel)
    assert_close(out.float().cpu().numpy(), oout[:, 0], "bf16", w.name)
    assert_close(lse.cpu().numpy(), olse[:, 0], "bf16", w.name, lse=True)


def test_decode_b64_full():
    """Decode config: 64 sequences, KV lengths uniform in [32768, 131072]."""
    w = synth.WORKLOADS["decode_b64"]
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_decode(w, t, DEV)
    del t
    sel = sel.cpu().numpy()
    rb = np.arange(w.B, dtype=np.int32)
    ri = np.zeros(w.B, np.int32)
    osel = oracle_selection_rows(w, rb, ri)
    assert np.array_equal(sel[:, 0], osel)
    oout, olse = oracle_attention_rows(w, rb, ri, osel)
    assert_close(out.float().cpu().numpy(), oout, "bf16", w.name)
    assert_close(lse.cpu().numpy(), olse, "bf16", w.name, lse=True)


DECODE_VARIANTS = {
    "bs64_k8": dict(Bs=64, K=8),
    "bs32_hpg8_d64": dict(Bs=32, K=12, Hq=16, Hkv=2, d=64),
    "bs128_hpg1": dict(Bs=128, K=5, Hq=8, Hkv=8),
    "bs128_hpg2_d64_di32": dict(Bs=128, K=6, Hq=8, Hkv=4, d=64, di=32),
    # K - 1 > 32: the warp top-K takes its exact radix path instead of the lane-maximum filter
    "bs32_k40_radix": dict(Bs=32, K=40),
    # a block size outside the decode kernels' builds: table index path, CUDA-core attention
    "bs100_generic": dict(Bs=100, K=5),
}


@pytest.mark.parametrize("name", sorted(DECODE_VARIANTS))
def test_decode_variants(name):
    """Decode with other block sizes, head maps and head dims (ragged lengths, some shorter than one block)."""
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=6, Nk=3000, kv_len_range=(1, 3000), **DECODE_VARIANTS[name])
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_decode(w, t, DEV)
    h = host_inputs(w)
    osel, oout, olse = oracle_full(w, h)
    assert np.array_equal(sel.cpu().numpy(), osel), name
    assert_close(out.float().cpu().numpy(), oout[:, 0], "bf16", name)
    assert_close(lse.cpu().numpy(), olse[:, 0], "bf16", name, lse=True)


def test_decode_batch_beyond_index_kernel():
    """1025 sequences: one more than the decode index kernel's per-CTA sequence table, so the
    selection takes the table path; the split attention kernel serves any batch."""
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=1025, Nk=160, kv_len_range=(1, 160), Hq=8, Hkv=2, d=64,
                     Bs=32, K=4)
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_decode(w, t, DEV)
    h = host_inputs(w)
    osel, oout, olse = oracle_full(w, h)
    assert np.array_equal(sel.cpu().numpy(), osel)
    assert_close(out.float().cpu().numpy(), oout[:, 0], "bf16", w.name)
    assert_close(lse.cpu().numpy(), olse[:, 0], "bf16", w.name, lse=True)


def test_decode_long_rows_cta_topk():
    """Rows of more than 1024 blocks (Bs 32, caches of 40000 keys): the CTA-per-row top-K."""
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=3, Nk=40000, kv_len_range=(33000, 40000), Bs=32, K=16)
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_decode(w, t, DEV)
    h = host_inputs(w)
    osel, oout, olse = oracle_full(w, h)
    assert np.array_equal(sel.cpu().numpy(), osel)
    assert_close(out.float().cpu().numpy(), oout[:, 0], "bf16", w.name)
    assert_close(lse.cpu().numpy(), olse[:, 0], "bf16", w.name, lse=True)


def test_decode_query_offset_not_last():
    """Index selection with one query per sequence at a position before the end of its keys."""
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=4, Nk=4096, kv_len_range=(2000, 4096))
    t = device_inputs(w, DEV)
    kl = synth.kv_lens(w)
    qo = (kl // 2).astype(np.int32)
    sel = msa_index_select_dev(t, w, qo, kl)
    h = host_inputs(w)
    import oracle

    osel = oracle.index_select(h["iq"].reshape(w.B, w.G, w.di), h["ik"], np.arange(w.B, dtype=np.int32),
                               np.zeros(w.B, np.int32), qo, kl, w.Bs, w.K)
    assert np.array_equal(sel[:, 0], osel)


def msa_index_select_dev(t, w, qo, kl):
    import block_sparse_long_select_gb300 as msa

    s = msa.msa_index_select(t["iq"], t["ik"], torch.from_numpy(qo).to(DEV), torch.from_numpy(kl).to(DEV), w.Bs, w.K)
    torch.cuda.synchronize()
    return s.cpu().numpy()


# forced sequence-start variant (block 0 kept with the local block), one case per top-K implementation
FORCE_START_PREFILL = {
    "fused_registers": synth.scaled(BASE, B=1, Nq=1500, Nk=1500, Bs=64, K=8),
    "fused_table": synth.scaled(BASE, B=1, Nq=1200, Nk=1200, Bs=32, K=20),
    "fused_k2_nothing_ranked": synth.scaled(BASE, B=1, Nq=800, Nk=800, Bs=32, K=2),
    "table_fp32": synth.WORKLOADS["tiny_fp32"],
}
FORCE_START_DECODE = {
    "warp_filter": dict(B=6, Nk=4096, kv_len_range=(1, 4096), Bs=128, K=16),
    "warp_radix": dict(B=6, Nk=3000, kv_len_range=(1, 3000), Bs=32, K=40),
    "cta_long_rows": dict(B=3, Nk=40000, kv_len_range=(33000, 40000), Bs=32, K=16),
    "k2": dict(B=6, Nk=3000, kv_len_range=(1, 3000), Bs=64, K=2),
}


def _force_start_check(w, qo, kl):
    import block_sparse_long_select_gb300 as msa
    import oracle

    t = device_inputs(w, DEV, names=("iq", "ik"))
    sel = msa.msa_index_select_v(t["iq"], t["ik"], torch.from_numpy(qo).to(DEV), torch.from_numpy(kl).to(DEV),
                                 w.Bs, w.K, msa.MSA_FORCE_LOCAL | msa.MSA_FORCE_START)
    torch.cuda.synchronize()
    iq, ik = synth.host_tensor(w, "iq"), synth.host_tensor(w, "ik")
    rb, ri = oracle.all_rows(w.B, w.Nq)
    osel = oracle.index_select(iq.reshape(-1, w.G, w.di), ik, rb, ri, qo, kl, w.Bs, w.K, force_start=True)
    assert np.array_equal(sel.cpu().numpy().reshape(osel.shape), osel), w.name


@pytest.mark.parametrize("name", sorted(FORCE_START_PREFILL))
def test_force_start_prefill(name):
    w = FORCE_START_PREFILL[name]
    _force_start_check(w, synth.q_offsets(w), synth.kv_lens(w))


@pytest.mark.parametrize("name", sorted(FORCE_START_DECODE))
def test_force_start_decode(name):
    w = synth.scaled(synth.WORKLOADS["decode_b64"], **FORCE_START_DECODE[name])
    kl = synth.kv_lens(w)
    _force_start_check(w, (kl - 1).astype(np.int32), kl)


def test_empty_batches():
    """An empty batch through every entry point: zero-size outputs, no device
    error; the backward with keys but no queries gives dk = dv = 0 (the
    oracle's gradients of zero listed rows)."""
    import block_sparse_long_select_gb300 as msa
    import oracle

    bf, i32 = torch.bfloat16, torch.int32
    e = lambda *s, dt=bf: torch.empty(s, dtype=dt, device=DEV)  # noqa: E731
    B, Nk, Hq, Hkv, d, di, Bs, K = 2, 300, 8, 2, 128, 64, 128, 2
    kl = torch.full((B,), Nk, dtype=i32, device=DEV)
    qo0 = torch.zeros(B, dtype=i32, device=DEV)
    for b, nq in ((0, 16), (B, 0)):
        sel = msa.msa_index_select(e(b, nq, Hkv, di), e(b, Nk, di), qo0[:b], kl[:b], Bs, K)
        assert tuple(sel.shape) == (b, nq, Hkv, K)
        sel_v = msa.msa_index_select_v(e(b, nq, Hkv, di), e(b, Nk, di), qo0[:b], kl[:b], Bs, K,
                                       msa.MSA_FORCE_LOCAL | msa.MSA_FORCE_START)
        assert sel_v.numel() == 0
        lse = e(b, nq, Hq, dt=torch.float32)
        out = msa.msa_sparse_attn_prefill(e(b, nq, Hq, d), e(b, Nk, Hkv, d), e(b, Nk, Hkv, d), sel, qo0[:b], kl[:b],
                                          Bs, K, lse=lse)
        assert tuple(out.shape) == (b, nq, Hq, d)
        klv = msa.msa_kl_aux_forward(e(b, nq, Hq, d), e(b, Nk, Hkv, d), e(b, nq, Hkv, di), e(b, Nk, di), sel, lse,
                                     qo0[:b], kl[:b], Bs, K)
        assert tuple(klv.shape) == (b, nq, Hkv)
    out = msa.msa_sparse_attn_decode(e(0, Hq, d), e(0, Nk, Hkv, d), e(0, Nk, Hkv, d), e(0, Hkv, K, dt=i32),
                                     kl[:0], Bs, K)
    assert out.numel() == 0
    sel, out = msa.msa_decode_step(e(0, Hq, d), e(0, Hkv, d), e(0, Hkv, d), e(0, Hkv, di), e(0, di),
                                   e(0, Nk, Hkv, d), e(0, Nk, Hkv, d), e(0, Nk, di), kl[:0], Bs, K)
    assert sel.numel() == 0 and out.numel() == 0
    # backward of a batch with keys but no query rows
    k = synth.device_tensor(synth.scaled(BASE, B=B, Nq=1, Nk=Nk, Hq=Hq, Hkv=Hkv, Bs=Bs, K=K), "k", DEV)
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(k, float("nan"))
    dq, dk, dv = msa.msa_sparse_attn_backward(e(B, 0, Hq, d), k, k, e(B, 0, Hq, d), e(B, 0, Hq, d),
                                              e(B, 0, Hq, dt=torch.float32), e(B, 0, Hkv, K, dt=i32), qo0, kl, Bs, K,
                                              dk=dk, dv=dv)
    torch.cuda.synchronize()
    z = np.zeros((0, Hq, d), np.float32)
    kh = k.float().cpu().numpy()
    _, odk, odv = oracle.sparse_attn_backward(z, kh, kh, z, np.zeros((0, Hkv, K), np.int32), np.zeros(0, np.int32),
                                              np.zeros(0, np.int32), np.zeros(B, np.int32), np.full(B, Nk, np.int32),
                                              Bs, K)
    assert dq.numel() == 0
    assert np.array_equal(dk.float().cpu().numpy(), odk) and np.array_equal(dv.float().cpu().numpy(), odv)
