"""Input generator checks (host side; the device twin is checked in test_gpu_synth.py)."""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    # SplitMix64 seeded with state 1234567: first five outputs as published with
    # the reference implementation (Vigna, splitmix64.c test values)
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    assert [synth.u64_py(1234567, i) for i in range(5)] == want
    lib = synth._host_lib()
    assert [lib.synth_u64(1234567, i) for i in range(5)] == want


def test_host_generator_matches_scalar_definition():
    w = synth.WORKLOADS["prefill_8k"]
    table = synth.normal_table("bf16")
    for name in ("q", "k"):
        key = synth.key_py(w.seed, synth.TID[name])
        idx = [0, 1, 2, 12345, 33554431]
        got = [synth.host_range(w, name, i, 1)[0] for i in idx]
        want = [table[synth.u64_py(key, i) >> 48] for i in idx]
        assert got == want
    key = synth.key_py(w.seed, synth.TID["iq"])
    for i in [0, 7, 99999]:
        want = ((synth.u64_py(key, i) >> 32) * 17 >> 32) - 8
        assert synth.host_range(w, "iq", i, 1)[0] == want


def test_slices_are_consistent():
    w = synth.WORKLOADS["tiny_fp32"]
    full = synth.host_tensor(w, "v")
    part = synth.host_range(w, "v", 1000, 777)
    assert np.array_equal(full.reshape(-1)[1000:1777], part)
    rows = synth.host_rows(w, "q", 0, [3, 500, 17])
    assert np.array_equal(rows, synth.host_tensor(w, "q")[0, [3, 500, 17]])


def test_value_ranges_and_moments():
    w = synth.WORKLOADS["prefill_8k"]
    ik = synth.host_tensor(w, "ik")
    assert ik.min() == -8 and ik.max() == 8 and np.all(ik == np.round(ik))
    q = synth.host_range(w, "q", 0, 1 << 20)
    assert abs(q.mean()) < 0.01 and abs(q.std() - 1) < 0.01
    # bf16-exact: low 16 bits clear
    assert np.all(q.view(np.uint32) & 0xFFFF == 0)


def test_hot_blocks_scale_index_key():
    w = synth.scaled(synth.WORKLOADS["prefill_128k_bs32"], Nq=4096, Nk=4096)
    ik = synth.host_tensor(w, "ik")
    assert np.abs(ik[0, :128]).max() == 24 and np.abs(ik[0, 128:]).max() == 8
    assert np.all(ik[0, :128] % 3 == 0)
    w1m = synth.WORKLOADS["prefill_1m"]
    hb = synth.hot_blocks(w1m)
    assert len(hb) == 82 and len(set(hb.tolist())) == 82 and hb.max() < 8192


def test_decode_lengths():
    w = synth.WORKLOADS["decode_b64"]
    L = synth.kv_lens(w)
    assert L.shape == (64,) and L.min() >= 32768 and L.max() <= 131072
    assert np.array_equal(synth.q_offsets(w), L - 1)
