"""GPU parity at the full workload sizes, in the launch configuration the
bench times (msa_index_select then msa_sparse_attn_prefill, default chunking):
every selection row is checked against the structural properties that hold
at any size, and a stratified sample of rows is compared with the oracle
(selection bit for bit, outputs within the bf16 tolerances)."""
import numpy as np
import pytest
import torch

import synth
from parity import (assert_close, check_structure, device_inputs, gpu_prefill, oracle_attention_rows,
                    oracle_selection_rows)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda:0")


def stratified_rows(w, n_rand, seed=0):
    """The first rows (dense: fewer visible blocks than K), rows around the
    first non-dense block, the last rows, and a random spread."""
    rng = np.random.default_rng(seed)
    first_sparse = w.K * w.Bs
    rows = np.concatenate([np.arange(0, 8), np.arange(first_sparse - 4, first_sparse + 4),
                           np.arange(w.Nq - 8, w.Nq), rng.choice(w.Nq, n_rand, replace=False)])
    return np.unique(np.clip(rows, 0, w.Nq - 1)).astype(np.int32)


def run_sampled(w, n_rand, n_attn):
    torch.cuda.set_device(DEV)
    t = device_inputs(w, DEV)
    sel, out, lse = gpu_prefill(w, t, DEV)
    del t
    sel_h = sel.cpu().numpy()
    check_structure(sel_h, synth.q_offsets(w), synth.kv_lens(w), w.Bs, w.K)
    rows = stratified_rows(w, n_rand)
    osel = oracle_selection_rows(w, np.zeros(len(rows), np.int32), rows)
    assert np.array_equal(sel_h[0, rows], osel), f"{w.name}: selected blocks differ on sampled rows"
    arows = rows[np.linspace(0, len(rows) - 1, n_attn).astype(int)]
    idx = np.searchsorted(rows, arows)
    oout, olse = oracle_attention_rows(w, np.zeros(len(arows), np.int32), arows, osel[idx])
    assert_close(out[0, arows].float().cpu().numpy(), oout, "bf16", w.name)
    assert_close(lse[0, arows].cpu().numpy(), olse, "bf16", w.name, lse=True)


@pytest.mark.parametrize("name", ["prefill_128k_bs128", "prefill_128k_bs64", "prefill_128k_bs32"])
def test_prefill_128k_sweep(cuda_ok, name):
    """Block-size sweep at 128K with the first four blocks' index keys scaled x3."""
    run_sampled(synth.WORKLOADS[name], n_rand=160, n_attn=64)


def test_prefill_1m(cuda_ok):
    """1M-token prefill with 1% of the blocks' index keys scaled x3."""
    run_sampled(synth.WORKLOADS["prefill_1m"], n_rand=24, n_attn=20)
