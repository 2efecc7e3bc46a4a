"""msa_index_select_noalloc: the selection entry point for callers that cannot
allocate device memory (it runs on a static scratch array inside the library).
Its output must equal msa_index_select's on two calls in a row (different
problems, so the second call runs over the first call's stale scratch), and a
problem larger than the static scratch must be refused before any launch.
Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_long_select_gb300 as msa
import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(w):
    iq = synth.device_tensor(w, "iq", DEV)
    ik = synth.device_tensor(w, "ik", DEV)
    kl = torch.from_numpy(synth.kv_lens(w)).to(DEV)
    qo = torch.from_numpy(synth.q_offsets(w)).to(DEV)
    return iq, ik, qo, kl


def test_noalloc_matches_index_select(cuda_ok):
    torch.cuda.set_device(DEV)
    cases = [
        # decode-shaped: 8 sequences, one query each, ragged KV lengths
        synth.scaled(synth.WORKLOADS["decode_b64"], B=8, Nk=8192, kv_len_range=(100, 8192)),
        # prefill-shaped bf16 (the workspace entry point takes its tensor-core path here)
        synth.scaled(synth.WORKLOADS["prefill_8k"], Nq=2048, Nk=2048, Bs=64, K=8, hot="first4"),
        # fp32
        synth.WORKLOADS["tiny_fp32"],
    ]
    for w in cases:  # consecutive calls share (and inherit) the static scratch
        iq, ik, qo, kl = _inputs(w)
        ref = msa.msa_index_select(iq, ik, qo, kl, w.Bs, w.K)
        got = torch.full_like(ref, -7)
        msa.msa_index_select_noalloc(iq, ik, qo, kl, w.Bs, w.K, sel=got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), w.name


def test_noalloc_rejects_oversize(cuda_ok):
    lib = msa.load_library()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the size check refuses first
    # table of 1 x 65536 x 8 x 1024 blocks x 4 B = 2 GiB > 32 MiB
    code = lib.msa_index_select_noalloc(fake, fake, None, None, 1, 65536, 131072, 8, 64, 128, 16, 0, fake, None,
                                        None)
    assert code == 3  # MSA_ERR_WORKSPACE
