"""Host logic of bench.py that its reported numbers rest on (no GPU): the
algorithmic work counts behind every roofline, the roofline arithmetic, and
the source-hash check on committed ncu traffic figures."""
import hashlib

import numpy as np
import pytest
import torch

import bench
import synth


def _attended_brute(sel, qo, kl, Bs):
    """Keys attended by each (b, i, g), summed: for every selected block t >= 0
    the keys j of [t Bs, (t + 1) Bs) with j <= pos and j < kv_len."""
    B, Nq, G, K = sel.shape
    n = 0
    for b in range(B):
        for i in range(Nq):
            pos = int(qo[b]) + i
            for g in range(G):
                for k in range(K):
                    t = int(sel[b, i, g, k])
                    if t < 0:
                        continue
                    n += sum(1 for j in range(t * Bs, (t + 1) * Bs) if j <= pos and j < int(kl[b]))
    return n


@pytest.mark.parametrize("Bs", [4, 8])
def test_attended_keys_brute_force(Bs):
    rng = np.random.default_rng(3)
    B, Nq, G, K = 2, 13, 3, 4
    qo = np.array([0, 7], np.int32)
    kl = qo + Nq + np.array([0, 5], np.int32)  # the second sequence has keys past its last query
    nblk = (int(kl.max()) + Bs - 1) // Bs
    sel = rng.integers(-1, nblk, size=(B, Nq, G, K)).astype(np.int32)
    got = bench.attended_keys(torch.from_numpy(sel), qo, kl, Bs)
    assert got == _attended_brute(sel, qo, kl, Bs)


def test_prefill_and_decode_work_counts():
    w = synth.scaled(synth.WORKLOADS["prefill_8k"], B=2, Nq=10, Nk=20, Hq=8, Hkv=2, d=64, di=32, Bs=4, K=3)
    qo = np.array([0, 10], np.int32)
    kl = np.array([10, 20], np.int32)
    sel = torch.zeros((w.B, w.Nq, w.G, w.K), dtype=torch.int32)  # block 0 three times: 4 keys each when visible
    work = bench.prefill_work(w, sel, qo, kl)
    # visible keys: sequence 0 rows see 1..10 keys, sequence 1 rows see 11..20
    visible = sum(range(1, 11)) + sum(range(11, 21))
    assert work["visible_keys"] == visible
    assert work["index_flops"] == 2.0 * w.di * w.G * visible
    # attended: block 0 (keys 0..3) per slot; sequence 0 row i sees min(i + 1, 4) of them
    att = w.G * w.K * (sum(min(i + 1, 4) for i in range(10)) + 10 * 4)
    assert work["attended_keys"] == att
    assert work["attn_flops"] == 4.0 * w.d * (w.Hq // w.G) * att
    assert bench.kl_work(w, work)["kl_flops"] == 2.0 * w.d * (w.Hq // w.G) * att + 2.0 * w.di * att
    # top-K over a block-max table: rows with more than K visible blocks read
    # their loc candidate maxima (blocks t < loc), every row writes K ids
    cand = 0
    for b in range(w.B):
        for i in range(w.Nq):
            loc = (int(qo[b]) + i) // w.Bs
            cand += loc if loc + 1 > w.K else 0
    assert work["topk_bytes"] == 4.0 * w.G * cand + 4.0 * w.K * w.G * w.B * w.Nq
    assert bench.backward_work(w, work)["bwd_flops"] == 10.0 * w.d * (w.Hq // w.G) * att

    wd = synth.scaled(synth.WORKLOADS["decode_b64"], B=2, Nk=40, Hq=8, Hkv=2, d=64, di=32, Bs=8, K=2)
    kld = np.array([9, 40], np.int32)
    seld = torch.tensor([[[[0, 1]] * 2], [[[3, 4]] * 2]], dtype=torch.int32)  # [B, 1, G, K]
    dw = bench.decode_work(wd, seld, kld)
    # sequence 0 (pos 8): block 0 -> 8 keys, block 1 -> key 8 only; sequence 1 (pos 39): 8 + 8
    att_d = wd.G * (8 + 1) + wd.G * (8 + 8)
    assert dw["attended_keys"] == att_d
    assert dw["index_bytes"] == (9 + 40) * wd.di * 2
    assert dw["attn_bytes"] == att_d * wd.d * 2 * 2 + wd.B * wd.Hq * wd.d * 4


def test_roofline_arithmetic():
    peaks = {"hbm_gbs": 5000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    work = {"index_flops": 8.0e12, "attn_flops": 4.0e12, "index_bytes": 6.0e8, "attn_bytes": 5.0e8}
    # 2 steps, 6 launches of 1.5 ms each: 4e12 x 2 / 6 flop per launch in 1.5 ms
    prof = {"attn_kv_outer_tc": (6, 9.0)}
    r = bench.roofline_for("attn_kv_outer_tc", prof, work, peaks, "measured", "nowhere", 2)
    want = 4.0e12 * 2 / 6 / 1.5e-3 / 1e12
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(want, abs=0.01)
    # kernels timed inside millisecond-scale steps: against the burst bf16 peak
    assert r["frac"] == pytest.approx(want / 2000.0, abs=1e-4) and r["peak"] == 2000.0
    assert r["launches_per_step"] == 3.0 and r["launch_ms"] == pytest.approx(1.5)
    # decode: bytes over time against the copy bandwidth
    r = bench.roofline_for("decode_index", {"decode_index": (10, 1.0)}, work, peaks, "measured", "nowhere", 10,
                           "decode")
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(6.0e8 / 1.0e-4 / 1e9, abs=0.01)
    assert bench.roofline_for("attn_invert", {"attn_invert": (1, 1.0)}, work, peaks, "m", "w", 1) is None
    # the large-K selection pass: table bytes over time against the copy bandwidth
    r = bench.roofline_for("index_topk_table", {"index_topk_table": (4, 2.0)}, dict(work, topk_bytes=8.0e9), peaks,
                           "measured", "nowhere", 1)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(8.0e9 / 4 / 0.5e-3 / 1e9, abs=0.01)


def test_ncu_traffic_needs_the_current_source(tmp_path, monkeypatch):
    csrc = tmp_path / "block_sparse_long_select_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "decode.cu").write_text("// kernel source\n")
    sha = hashlib.sha256(b"// kernel source\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "x.md").write_text(f"ncu-traffic decode_index decode_b64 6.5e8 {sha}\n"
                               f"ncu-traffic decode_attn decode_b64 5.0e8 0123456789abcdef\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("decode_index", "decode_b64") == 6.5e8
    assert bench.ncu_traffic("decode_index", "prefill_128k_bs128") is None  # another workload
    assert bench.ncu_traffic("decode_attn", "decode_b64") is None           # taken on another source
    assert bench.ncu_traffic("no_such_kernel", "decode_b64") is None
