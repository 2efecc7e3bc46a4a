"""GPU parity at the full workload sizes, in the launch configuration the
bench times (msa_index_select then msa_sparse_attn_prefill, default chunking):
every selection row is checked against the structural properties that hold
at any size, and a stratified sample of rows is compared with the oracle
(selection bit for bit, outputs within the bf16 tolerances): every dense head
row (the first K*Bs rows, which see at most K blocks), the whole last block,
the rows whose local block is one of the hot blocks (and the rows just past
it), and 1024 rows drawn at random; attention on 320 of them."""
import numpy as np
import pytest
import torch

import synth
from parity import (assert_close, check_structure, device_inputs, gpu_prefill, oracle_attention_rows,
                    oracle_selection_rows)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda:0")
N_RANDOM, N_ATTN = 1024, 320


def stratified_rows(w, seed=0):
    """(selection rows, attention rows) of the sample described above."""
    rng = np.random.default_rng(seed)
    dense = np.arange(0, min(w.Nq, w.K * w.Bs))
    boundary = np.arange(w.K * w.Bs - 8, w.K * w.Bs + 8)
    last = np.arange(w.Nq - w.Bs, w.Nq)
    hot = synth.hot_blocks(w)
    hot = hot[np.linspace(0, len(hot) - 1, min(len(hot), 16)).astype(int)] if len(hot) else hot
    around_hot = np.concatenate([np.array([t * w.Bs, t * w.Bs + w.Bs // 2, t * w.Bs + w.Bs - 1, (t + 1) * w.Bs,
                                           (t + 1) * w.Bs + 1]) for t in hot]) if len(hot) else np.zeros(0, int)
    spread = rng.choice(w.Nq, N_RANDOM, replace=False)
    sel_rows = np.unique(np.clip(np.concatenate([dense, boundary, last, around_hot, spread]), 0, w.Nq - 1))
    # attention: some dense rows, the boundary, the last block's ends, the hot rows, the rest from the spread
    fixed = np.unique(np.clip(np.concatenate([dense[:: max(1, len(dense) // 48)], boundary, last[:8], last[-8:],
                                              around_hot]), 0, w.Nq - 1))
    rest = rng.choice(np.setdiff1d(sel_rows, fixed), N_ATTN - len(fixed), replace=False)
    attn_rows = np.unique(np.concatenate([fixed, rest]))
    return sel_rows.astype(np.int32), attn_rows.astype(np.int32)


def run_sampled(w):
    torch.cuda.set_device(DEV)
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV)
    del t
    sel_h = sel.cpu().numpy()
    check_structure(sel_h, synth.q_offsets(w), synth.kv_lens(w), w.Bs, w.K)
    rows, arows = stratified_rows(w)
    assert len(rows) >= N_RANDOM and len(arows) >= 256
    osel = oracle_selection_rows(w, np.zeros(len(rows), np.int32), rows)
    assert np.array_equal(sel_h[0, rows], osel), f"{w.name}: selected blocks differ on sampled rows"
    idx = np.searchsorted(rows, arows)
    oout, olse = oracle_attention_rows(w, np.zeros(len(arows), np.int32), arows, osel[idx])
    assert_close(out[0, arows].float().cpu().numpy(), oout, "bf16", w.name)
    assert_close(lse[0, arows].cpu().numpy(), olse, "bf16", w.name, lse=True)


@pytest.mark.parametrize("name", ["prefill_128k_bs128", "prefill_128k_bs64", "prefill_128k_bs32"])
def test_prefill_128k_sweep(cuda_ok, name):
    """Block-size sweep at 128K with the first four blocks' index keys scaled x3."""
    run_sampled(synth.WORKLOADS[name])


def test_prefill_1m(cuda_ok):
    """1M-token prefill with 1% of the blocks' index keys scaled x3."""
    run_sampled(synth.WORKLOADS["prefill_1m"])
