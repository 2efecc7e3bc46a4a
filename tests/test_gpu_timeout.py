"""The bounded-wait timeout path on the GPU, exercised without a fault.

With the library's test hook on (msa_debug_inject_timeout), the attention
kernels first wait on a device barrier that nothing completes. That wait runs
out after about a millisecond; the kernel records MSA_ERR_TIMEOUT in the
workspace status, lets its copies and matrix products finish, frees its tensor
memory and returns. The host reads the status; the context stays usable, and
the next call on the SAME workspace (hook off) must match the oracle."""
import numpy as np
import pytest
import torch

import block_sparse_long_select_gb300 as msa
import synth
from parity import assert_close, device_inputs, host_inputs, oracle_full

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
MSA_ERR_TIMEOUT = 5


@pytest.fixture(autouse=True)
def _hook_off(cuda_ok):
    torch.cuda.set_device(DEV)
    yield
    msa.msa_debug_inject_timeout(False)


def test_prefill_attention_timeout_then_recovers():
    # tensor-core KV-outer path (bf16, blocks of 128), several tiles per CTA
    w = synth.scaled(synth.WORKLOADS["prefill_8k"], Nq=1500, Nk=1500, Bs=128, K=4)
    t = device_inputs(w, DEV)
    qo = torch.from_numpy(synth.q_offsets(w)).to(DEV)
    kl = torch.from_numpy(synth.kv_lens(w)).to(DEV)
    sel = msa.msa_index_select(t["iq"], t["ik"], qo, kl, w.Bs, w.K)
    ws = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_PREFILL, w.B, w.Nq, w.Nk, w.G, w.Hq, w.d, 0, w.Bs, w.K,
                                              msa.MSA_BF16), DEV)
    out = torch.empty_like(t["q"])
    assert msa.msa_debug_inject_timeout(True) is False
    msa.msa_sparse_attn_prefill(t["q"], t["k"], t["v"], sel, qo, kl, w.Bs, w.K, out=out, ws=ws)
    st = msa.msa_read_status(ws)  # synchronises: the kernel returned (no hang)
    msa.msa_debug_inject_timeout(False)
    assert st == MSA_ERR_TIMEOUT, msa.msa_status_string(st)
    # the same workspace again, hook off: a correct result and a clean status
    lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device=DEV)
    out.fill_(float("nan"))
    msa.msa_sparse_attn_prefill(t["q"], t["k"], t["v"], sel, qo, kl, w.Bs, w.K, out=out, lse=lse, ws=ws)
    assert msa.msa_read_status(ws) == 0
    osel, oout, olse = oracle_full(w, host_inputs(w))
    assert np.array_equal(sel.cpu().numpy(), osel)
    assert_close(out.float().cpu().numpy(), oout, "bf16", w.name)
    assert_close(lse.cpu().numpy(), olse, "bf16", w.name, lse=True)


def test_decode_attention_timeout_then_recovers():
    # split decode kernel: every CTA that gave up still counts its arrival, so
    # the per-(sequence, group) merge counters are back at zero afterwards
    w = synth.scaled(synth.WORKLOADS["decode_b64"], B=5, Nk=4096, kv_len_range=(300, 4096))
    t = device_inputs(w, DEV)
    kl = torch.from_numpy(synth.kv_lens(w)).to(DEV)
    sel = msa.msa_index_select(t["iq"], t["ik"], kl - 1, kl, w.Bs, w.K)
    ws = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_DECODE, w.B, 1, w.Nk, w.G, w.Hq, w.d, 0, w.Bs, w.K,
                                              msa.MSA_BF16), DEV)
    q = t["q"][:, 0]
    out = torch.empty_like(q)
    msa.msa_debug_inject_timeout(True)
    msa.msa_sparse_attn_decode(q, t["k"], t["v"], sel, kl, w.Bs, w.K, out=out, ws=ws)
    st = msa.msa_read_status(ws)
    msa.msa_debug_inject_timeout(False)
    assert st == MSA_ERR_TIMEOUT, msa.msa_status_string(st)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=DEV)
    for _ in range(2):  # twice: the counters must stay consistent call after call
        out.fill_(float("nan"))
        msa.msa_sparse_attn_decode(q, t["k"], t["v"], sel, kl, w.Bs, w.K, out=out, lse=lse, ws=ws)
        assert msa.msa_read_status(ws) == 0
        osel, oout, olse = oracle_full(w, host_inputs(w))
        assert np.array_equal(sel.cpu().numpy(), osel)
        assert_close(out.float().cpu().numpy(), oout[:, 0], "bf16", w.name)
        assert_close(lse.cpu().numpy(), olse[:, 0], "bf16", w.name, lse=True)
