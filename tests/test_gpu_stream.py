"""GPU parity of the streaming decode step (msa_decode_step through the C ABI):
a loop of steps that each append one token per sequence to the caches and
then select and attend for it, checked step by step against the oracle's
decode at the grown length (selection bit for bit, outputs within the bf16
tolerances), plus the cache rows and lengths the step wrote."""
import numpy as np
import pytest
import torch

import block_sparse_long_select_gb300 as msa
import oracle
import synth
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run_stream(w, L0, steps):
    """Caches hold the synthetic sequence up to L0[b]; each step appends the
    token at position L0[b] + s from the same synthetic sequence."""
    torch.cuda.set_device(DEV)
    k_full, v_full = synth.device_tensor(w, "k", DEV), synth.device_tensor(w, "v", DEV)
    ik_full = synth.device_tensor(w, "ik", DEV)
    k_cache, v_cache, ik_cache = k_full.clone(), v_full.clone(), ik_full.clone()
    for b in range(w.B):  # nothing beyond the current length: the step must write what it reads
        k_cache[b, L0[b]:] = 0
        v_cache[b, L0[b]:] = 0
        ik_cache[b, L0[b]:] = 0
    kv_len = torch.from_numpy(L0.astype(np.int32)).to(DEV)
    ws = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_DECODE_STEP, w.B, 0, w.Nk, w.G, w.Hq, w.d, w.di, w.Bs, w.K,
                                              msa.MSA_BF16), DEV)
    k_h, v_h, ik_h = synth.host_tensor(w, "k"), synth.host_tensor(w, "v"), synth.host_tensor(w, "ik")
    ar = torch.arange(w.B, device=DEV)
    for s in range(steps):
        ws_ = synth.scaled(w, seed=100 + s)  # a new query per step
        q, iq = synth.device_tensor(ws_, "q", DEV)[:, 0], synth.device_tensor(ws_, "iq", DEV)[:, 0]
        pos = torch.from_numpy((L0 + s).astype(np.int64)).to(DEV)
        k_new, v_new, ik_new = k_full[ar, pos].contiguous(), v_full[ar, pos].contiguous(), ik_full[ar, pos].contiguous()
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=DEV)
        sel, out = msa.msa_decode_step(q, k_new, v_new, iq, ik_new, k_cache, v_cache, ik_cache, kv_len, w.Bs, w.K,
                                       lse=lse, ws=ws)
        torch.cuda.synchronize()
        assert msa.msa_read_status(ws) == 0
        L = L0 + s + 1
        assert np.array_equal(kv_len.cpu().numpy(), L), f"step {s}: lengths"
        qh, iqh = synth.host_tensor(ws_, "q"), synth.host_tensor(ws_, "iq")
        osel, oout, olse = oracle.msa_forward(qh, k_h, v_h, iqh, ik_h, w.Bs, w.K, q_offset=(L - 1).astype(np.int32),
                                              kv_len=L.astype(np.int32))
        assert np.array_equal(sel.cpu().numpy(), osel[:, 0]), f"step {s}: selection"
        assert_close(out.float().cpu().numpy(), oout[:, 0], "bf16", f"step {s}")
        assert_close(lse.cpu().numpy(), olse[:, 0], "bf16", f"step {s}", lse=True)
    for b in range(w.B):  # the appended rows are the sequence's own rows, bit for bit
        e = L0[b] + steps
        assert torch.equal(k_cache[b, :e], k_full[b, :e]) and torch.equal(v_cache[b, :e], v_full[b, :e])
        assert torch.equal(ik_cache[b, :e], ik_full[b, :e])


def test_stream_decode_bs128():
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=4, Nk=4096, kv_len_range=(1, 4000))
    L0 = np.array([1, 700, 2047, 3990], np.int64)
    _run_stream(w, L0, steps=8)


def test_stream_decode_bs32_crosses_blocks():
    """Block size 32: lengths start just below block boundaries so appends open new blocks."""
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=3, Nk=2048, kv_len_range=(1, 2000), Bs=32, K=10, Hq=16, Hkv=4)
    L0 = np.array([30, 318, 1500], np.int64)
    _run_stream(w, L0, steps=6)


def test_stream_decode_full_cache_row_left_unchanged():
    """A sequence whose cache is full keeps its length; its row is -1 / zero and the status is BOUNDS."""
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=2, Nk=1024, kv_len_range=(1, 1024))
    torch.cuda.set_device(DEV)
    k_cache, v_cache = synth.device_tensor(w, "k", DEV), synth.device_tensor(w, "v", DEV)
    ik_cache = synth.device_tensor(w, "ik", DEV)
    q, iq = synth.device_tensor(w, "q", DEV)[:, 0], synth.device_tensor(w, "iq", DEV)[:, 0]
    k_new, v_new, ik_new = k_cache[:, 0].contiguous(), v_cache[:, 0].contiguous(), ik_cache[:, 0].contiguous()
    kv_len = torch.tensor([500, 1024], dtype=torch.int32, device=DEV)
    before = k_cache[1].clone()
    ws = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_DECODE_STEP, w.B, 0, w.Nk, w.G, w.Hq, w.d, w.di, w.Bs, w.K,
                                              msa.MSA_BF16), DEV)
    sel, out = msa.msa_decode_step(q, k_new, v_new, iq, ik_new, k_cache, v_cache, ik_cache, kv_len, w.Bs, w.K, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_read_status(ws) == 6  # MSA_ERR_BOUNDS
    assert kv_len.tolist() == [501, 1024]
    assert (sel[1] == -1).all() and (out[1] == 0).all()
    assert torch.equal(k_cache[1], before)
    assert (sel[0] >= 0).any()
