"""Pins for the CPU oracle: each checks it against something other than itself.

* a hand-worked example derived from the method's definition (tests/golden);
* brute-force token scores via a library matmul (block max pooling);
* the top-K optimality / structure invariants of the selection;
* a second, differently written selection (repeated arg-max in pure Python);
* closed forms: all-equal scores select blocks 0..K-2 plus the local block;
  a planted block is selected by every row that can see it;
* the dense special case (K >= visible blocks) equals textbook causal GQA
  attention from torch's scaled_dot_product_attention in fp64;
* the masked-dense restatement (selected blocks as an explicit attention mask)
  equals torch's SDPA for partial selections, with ragged offsets / lengths;
* decode at length L equals the prefill row at position L-1;
* the forced sequence-start variant: structure, a second implementation, and
  its equivalences with the plain selection when block 0 is the strongest or
  the weakest block;
* the KL auxiliary forward: non-negative, zero on matched distributions, the
  closed form for a uniform main distribution, and invariance to shifting a
  row's index scores;
* the Main Branch backward: equal to torch autograd through the masked-dense
  restatement (fp64), to central finite differences of the forward oracle
  (selection held fixed), and to the closed forms sum_j dk_j = 0,
  sum_j dv_j = sum over the group's rows of dout, sum q.dq = sum k.dk;
* planted mistakes in a copy of the oracle source fail at least one pin.
"""
import math
import os
import re
import shutil

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "handworked_msa.txt")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def rand_problem(seed, B=2, Nq=96, Nk=96, Hq=4, Hkv=2, d=16, di=8, a=3, q_offset=None, kv_len=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Nq, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Nk, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((B, Nk, Hkv, d)).astype(np.float32)
    iq = rng.integers(-a, a + 1, (B, Nq, Hkv, di)).astype(np.float32)
    ik = rng.integers(-a, a + 1, (B, Nk, di)).astype(np.float32)
    q_offset = np.zeros(B, np.int32) if q_offset is None else np.asarray(q_offset, np.int32)
    kv_len = np.full(B, Nk, np.int32) if kv_len is None else np.asarray(kv_len, np.int32)
    return q, k, v, iq, ik, q_offset, kv_len


def sdpa_masked(q, k, v, allowed, scale):
    """torch SDPA (fp64, CPU) with an explicit boolean mask.

    q [B,Nq,Hq,d]; k,v [B,Nk,Hkv,d]; allowed [B,Nq,Hkv,Nk] bool (per group).
    """
    B, Nq, Hq, d = q.shape
    Hkv = k.shape[2]
    hpg = Hq // Hkv
    qt = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(hpg, dim=1)
    vt = torch.from_numpy(v.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(hpg, dim=1)
    m = torch.from_numpy(allowed).permute(0, 2, 1, 3).repeat_interleave(hpg, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    s = torch.einsum("bhqc,bhkc->bhqk", qt, kt) * scale
    lse = torch.logsumexp(s.masked_fill(~m, -math.inf), dim=-1)
    return out.permute(0, 2, 1, 3).numpy(), lse.permute(0, 2, 1).numpy()


def causal_allowed(B, Nq, Nk, Hkv, q_offset, kv_len):
    j = np.arange(Nk)
    al = np.zeros((B, Nq, Hkv, Nk), dtype=bool)
    for b in range(B):
        pos = q_offset[b] + np.arange(Nq)
        al[b] = ((j[None, :] <= pos[:, None]) & (j[None, :] < kv_len[b]))[:, None, :]
    return al


def selected_allowed(sel, Bs, B, Nq, Nk, Hkv, q_offset, kv_len):
    al = causal_allowed(B, Nq, Nk, Hkv, q_offset, kv_len)
    blk = np.arange(Nk) // Bs
    keep = np.zeros_like(al)
    for b in range(B):
        for i in range(Nq):
            for g in range(Hkv):
                s = sel[b, i, g]
                keep[b, i, g] = np.isin(blk, s[s >= 0])
    return al & keep


def token_scores(iq, ik):
    """[B,Nq,G,Nk] index scores by a library matmul (fp64)."""
    return np.einsum("bigc,bjc->bigj", iq.astype(np.float64), ik.astype(np.float64))


def argmax_selection(M, loc, K):
    """Second implementation: K-1 rounds of arg-max (first max = lowest index)."""
    if loc + 1 <= K:
        return list(range(loc + 1)) + [-1] * (K - loc - 1)
    avail = list(range(loc))
    chosen = []
    for _ in range(K - 1):
        best = None
        for t in avail:
            if best is None or M[t] > M[best]:
                best = t
        chosen.append(best)
        avail.remove(best)
    return sorted(chosen + [loc])


def argmax_selection_start(M, loc, K):
    """Second implementation of the forced-start variant: blocks 0 and loc,
    plus K-2 rounds of arg-max over blocks 1..loc-1."""
    if loc + 1 <= K:
        return list(range(loc + 1)) + [-1] * (K - loc - 1)
    avail = list(range(1, loc))
    chosen = []
    for _ in range(K - 2):
        best = None
        for t in avail:
            if best is None or M[t] > M[best]:
                best = t
        chosen.append(best)
        avail.remove(best)
    return sorted(chosen + [0, loc])


def oracle_all(q, k, v, iq, ik, Bs, K, q_offset, kv_len, lib=None, scale=0.0):
    return oracle.msa_forward(q, k, v, iq, ik, Bs, K, q_offset=q_offset, kv_len=kv_len, scale=scale, lib=lib)


# ---------------------------------------------------------------------------
# pins (each takes an optional lib so the mutation test can rerun them)
# ---------------------------------------------------------------------------
def pin_golden(lib=None):
    ik = None
    attn_k = attn_v = expect = None
    with open(GOLDEN) as f:
        lines = [ln.split("#")[0].strip() for ln in f]
    lines = [ln for ln in lines if ln]
    ik = np.array([3, 1, 4, 1, 5, 9, 2, 6, 5, 3], np.float32).reshape(1, 10, 1)
    Bs = 2
    for ln in lines:
        head, _, tail = ln.partition(":")
        parts = head.split()
        if parts[0] == "select":
            iqv, pos, K = float(parts[1]), int(parts[2]), int(parts[3])
            want = [int(x) for x in tail.split()]
            sel = oracle.index_select(np.full((1, 1, 1), iqv, np.float32), ik, [0], [pos], [0], [10], Bs, K,
                                      lib=lib)
            assert sel[0, 0].tolist() == want, (ln, sel[0, 0].tolist())
        elif parts[0] == "blockmax":
            iqv, pos = float(parts[1]), int(parts[2])
            want = [float(x) for x in tail.split()]
            _, bm = oracle.index_select(np.full((1, 1, 1), iqv, np.float32), ik, [0], [pos], [0], [10], Bs, 2,
                                        want_block_max=True, lib=lib)
            assert bm[0, 0, :len(want)].tolist() == want, (ln, bm[0, 0].tolist())
        elif parts[0] == "attend":
            vals = [float(x) for x in parts[2:]]
            if parts[1] == "k":
                attn_k = np.array(vals, np.float32).reshape(1, 10, 1, 1)
            elif parts[1] == "v":
                attn_v = np.array(vals, np.float32).reshape(1, 10, 1, 1)
            else:
                expect = vals
    out, lse = oracle.sparse_attn(np.ones((1, 1, 1), np.float32), attn_k, attn_v,
                                  np.array([[[1, 2]]], np.int32), [0], [4], [0], [10], Bs, 2, scale=1.0, lib=lib)
    assert abs(out[0, 0, 0] - expect[0]) < 1e-6 and abs(lse[0, 0] - expect[1]) < 1e-6, (out, lse)


def pin_blockmax_bruteforce(lib=None):
    q, k, v, iq, ik, _, _ = rand_problem(1)
    Nq = 56
    iq = iq[:, :Nq]
    kl = np.array([96, 96], np.int32)
    qo = np.array([0, 40], np.int32)
    Bs, K = 8, 4
    rb, ri = oracle.all_rows(2, Nq)
    sel, bm = oracle.index_select(iq.reshape(-1, 2, 8), ik, rb, ri, qo, kl, Bs, K, want_block_max=True, lib=lib)
    s = token_scores(iq, ik)
    bm = bm.reshape(2, Nq, 2, -1)
    for b in range(2):
        for i in range(Nq):
            pos = qo[b] + i
            loc = pos // Bs
            for g in range(2):
                for t in range(loc + 1):
                    hi = min((t + 1) * Bs, pos + 1)
                    assert bm[b, i, g, t] == s[b, i, g, t * Bs:hi].max()
                assert np.isnan(bm[b, i, g, loc + 1:]).all()


def pin_selection_invariants(lib=None):
    for seed, Bs, K in [(2, 8, 4), (3, 4, 7), (4, 16, 2), (5, 8, 1)]:
        q, k, v, iq, ik, qo, kl = rand_problem(seed, q_offset=[0, 17], kv_len=[96, 96])
        Nq = 79
        iq = iq[:, :Nq]
        rb, ri = oracle.all_rows(2, Nq)
        sel, bm = oracle.index_select(iq.reshape(-1, 2, 8), ik, rb, ri, qo, kl, Bs, K, want_block_max=True,
                                      lib=lib)
        for r in range(len(rb)):
            pos = qo[rb[r]] + ri[r]
            loc = pos // Bs
            for g in range(2):
                s = sel[r, g]
                valid = s[s >= 0]
                assert (s[len(valid):] == -1).all()
                assert len(valid) == min(K, loc + 1)
                assert (np.diff(valid) > 0).all() and valid.min() >= 0 and valid.max() <= loc
                assert loc in valid
                M = bm[r, g]
                others = [t for t in valid if t != loc]
                unsel = [t for t in range(loc) if t not in valid]
                if others and unsel:
                    worst = min((M[t], -t) for t in others)
                    best_out = max((M[t], -t) for t in unsel)
                    assert worst > best_out
                assert list(s) == argmax_selection(M, loc, K)


def pin_closed_forms(lib=None):
    # all-equal scores (index query zero): blocks 0..K-2 plus the local block
    B, Nq, Nk, di, Bs, K = 1, 64, 64, 4, 4, 5
    ik = np.random.default_rng(0).integers(-3, 4, (B, Nk, di)).astype(np.float32)
    iq = np.zeros((B * Nq, 1, di), np.float32)
    rb, ri = oracle.all_rows(B, Nq)
    sel = oracle.index_select(iq, ik, rb, ri, [0], [Nk], Bs, K, lib=lib)
    for i in range(Nq):
        loc = i // Bs
        want = list(range(loc + 1)) + [-1] * (K - loc - 1) if loc + 1 <= K else list(range(K - 1)) + [loc]
        assert sel[i, 0].tolist() == want
    # planted block: index query e0, index key dim 0 large on block t*
    tstar = 6
    ik2 = np.random.default_rng(1).integers(-3, 4, (B, Nk, di)).astype(np.float32)
    ik2[0, tstar * Bs:(tstar + 1) * Bs, 0] = 100.0
    iq2 = np.zeros((B * Nq, 1, di), np.float32)
    iq2[:, 0, 0] = 1.0
    sel2 = oracle.index_select(iq2, ik2, rb, ri, [0], [Nk], Bs, 2, lib=lib)
    for i in range(Nq):
        if i // Bs > tstar:
            assert tstar in sel2[i, 0].tolist()


def pin_dense_equals_sdpa(lib=None):
    # K >= visible blocks: MSA equals dense causal GQA attention
    q, k, v, iq, ik, qo, kl = rand_problem(7, B=2, Nq=40, Nk=96, q_offset=[56, 30], kv_len=[96, 70])
    Bs, K = 8, 12
    sel, out, lse = oracle_all(q, k, v, iq, ik, Bs, K, qo, kl, lib=lib)
    al = causal_allowed(2, 40, 96, 2, qo, kl)
    ref, ref_lse = sdpa_masked(q, k, v, al, 1.0 / math.sqrt(16))
    assert np.abs(out - ref).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


def pin_masked_dense_equals_sdpa(lib=None):
    for seed, Bs, K in [(8, 8, 3), (9, 4, 5), (10, 16, 2)]:
        q, k, v, iq, ik, qo, kl = rand_problem(seed, B=2, Nq=50, Nk=96, q_offset=[46, 20], kv_len=[96, 70])
        sel, out, lse = oracle_all(q, k, v, iq, ik, Bs, K, qo, kl, lib=lib)
        al = selected_allowed(sel, Bs, 2, 50, 96, 2, qo, kl)
        ref, ref_lse = sdpa_masked(q, k, v, al, 1.0 / math.sqrt(16))
        assert np.abs(out - ref).max() < 1e-12
        assert np.abs(lse - ref_lse).max() < 1e-12


def pin_attention_special_cases(lib=None):
    q, k, v, iq, ik, qo, kl = rand_problem(11)
    Bs, K = 8, 3
    # position 0 attends only to key 0: output is v[0] of its group
    sel, out, lse = oracle_all(q, k, v, iq, ik, Bs, K, [0, 0], [96, 96], lib=lib)
    for h in range(4):
        assert np.array_equal(out[:, 0, h], v[:, 0, h // 2].astype(np.float64))
    # constant values: weights sum to one
    ones = np.ones_like(v)
    _, out1, _ = oracle_all(q, k, ones, iq, ik, Bs, K, [0, 0], [96, 96], lib=lib)
    assert np.abs(out1 - 1.0).max() < 1e-12
    # convex combination of the selected values
    for b in range(2):
        for i in range(0, 96, 7):
            for h in range(4):
                g = h // 2
                s = sel[b, i, g]
                keys = [j for t in s[s >= 0] for j in range(t * Bs, (t + 1) * Bs) if j <= i]
                vv = v[b, keys, g].astype(np.float64)
                assert (out[b, i, h] >= vv.min(0) - 1e-12).all() and (out[b, i, h] <= vv.max(0) + 1e-12).all()


def pin_decode_equals_prefill_row(lib=None):
    q, k, v, iq, ik, qo, kl = rand_problem(12, B=2, Nq=96, Nk=96)
    Bs, K = 8, 4
    sel, out, lse = oracle_all(q, k, v, iq, ik, Bs, K, [0, 0], [96, 96], lib=lib)
    for L in (1, 9, 57, 96):
        dsel, dout, dlse = oracle_all(q[:, L - 1:L], k, v, iq[:, L - 1:L], ik, Bs, K, [L - 1, L - 1], [L, L],
                                      lib=lib)
        assert np.array_equal(dsel[:, 0], sel[:, L - 1])
        assert np.abs(dout[:, 0] - out[:, L - 1]).max() < 1e-12


def pin_force_start(lib=None):
    """Forced sequence-start variant: structure, a second implementation, and
    two equivalences with the plain selection that fix its meaning: when block
    0 is the strongest block the two selections agree; when it is the weakest,
    the variant equals {0} plus the plain selection with one slot fewer."""
    for seed, Bs, K in [(11, 8, 4), (12, 4, 7), (13, 16, 3)]:
        q, k, v, iq, ik, qo, kl = rand_problem(seed, q_offset=[0, 17], kv_len=[96, 96])
        Nq = 79
        iq = iq[:, :Nq]
        rb, ri = oracle.all_rows(2, Nq)
        sel, bm = oracle.index_select(iq.reshape(-1, 2, 8), ik, rb, ri, qo, kl, Bs, K, want_block_max=True,
                                      lib=lib, force_start=True)
        for r in range(len(rb)):
            loc = (qo[rb[r]] + ri[r]) // Bs
            for g in range(2):
                s = sel[r, g]
                valid = s[s >= 0]
                assert len(valid) == min(K, loc + 1) and (s[len(valid):] == -1).all()
                assert (np.diff(valid) > 0).all() and 0 in valid and loc in valid
                assert list(s) == argmax_selection_start(bm[r, g], loc, K)
    # block 0 strongest / weakest: index query e0, index key dim 0 = +-100 on block 0
    B, Nq, Nk, di, Bs, K = 1, 64, 64, 4, 4, 5
    rb, ri = oracle.all_rows(B, Nq)
    iq = np.random.default_rng(3).integers(-3, 4, (B * Nq, 1, di)).astype(np.float32)
    iq[:, 0, 0] = 1.0
    for big, rel in [(100.0, "equal"), (-100.0, "one_fewer")]:
        ik = np.random.default_rng(4).integers(-3, 4, (B, Nk, di)).astype(np.float32)
        ik[0, :Bs, 0] = big
        forced = oracle.index_select(iq, ik, rb, ri, [0], [Nk], Bs, K, lib=lib, force_start=True)
        if rel == "equal":
            plain = oracle.index_select(iq, ik, rb, ri, [0], [Nk], Bs, K, lib=lib)
            assert np.array_equal(forced, plain)
        else:
            plain = oracle.index_select(iq, ik, rb, ri, [0], [Nk], Bs, K - 1, lib=lib)
            for i in range(Nq):
                if i // Bs + 1 > K:
                    assert forced[i, 0].tolist() == sorted([0] + plain[i, 0].tolist())


def _kl_inputs(seed, B=2, Nq=40, Nk=96, Hq=4, Hkv=2, d=16, di=8, Bs=8, K=5):
    q, k, v, iq, ik, qo, kl = rand_problem(seed, B=B, Nq=Nq, Nk=Nk, Hq=Hq, Hkv=Hkv, d=d, di=di,
                                           q_offset=[Nk - Nq, 20], kv_len=[Nk, Nq + 20])
    rb, ri = oracle.all_rows(B, Nq)
    sel = oracle.index_select(iq.reshape(-1, Hkv, di), ik, rb, ri, qo, kl, Bs, K)
    return q, k, iq, ik, qo, kl, rb, ri, sel


def pin_kl_aux(lib=None):
    """KL auxiliary forward: non-negative; zero when the index scores equal the
    main scores (one head per group, scale 1); for a uniform main distribution
    it equals the closed form -log n - mean(s) + logsumexp(s) over the selected
    tokens (index scores from a library matmul); unchanged when every index
    score of a row is shifted by the same constant."""
    Bs, K = 8, 5
    q, k, iq, ik, qo, kl_, rb, ri, sel = _kl_inputs(21)
    n, Hq, d, Hkv, di = len(rb), 4, 16, 2, 8
    kl = oracle.kl_aux(q.reshape(n, Hq, d), k, iq.reshape(n, Hkv, di), ik, sel, rb, ri, qo, kl_, Bs, K, lib=lib)
    assert kl.min() > -1e-12 and kl.max() > 0
    # matched distributions: one kv head, Hq = Hkv = 1, index = main scores at scale 1
    rng = np.random.default_rng(5)
    B1, N1 = 1, 48
    q1 = rng.standard_normal((B1, N1, 1, 8)).astype(np.float32)
    k1 = rng.standard_normal((B1, N1, 1, 8)).astype(np.float32)
    rb1, ri1 = oracle.all_rows(B1, N1)
    sel1 = oracle.index_select(q1.reshape(-1, 1, 8), k1[:, :, 0], rb1, ri1, [0], [N1], 4, 3)
    kl1 = oracle.kl_aux(q1.reshape(-1, 1, 8), k1, q1.reshape(-1, 1, 8), k1[:, :, 0], sel1, rb1, ri1, [0], [N1], 4, 3,
                        scale=1.0, lib=lib)
    assert np.abs(kl1).max() < 1e-12
    # uniform main distribution (query zero): closed form over the selected tokens
    qz = np.zeros_like(q)
    klz = oracle.kl_aux(qz.reshape(n, Hq, d), k, iq.reshape(n, Hkv, di), ik, sel, rb, ri, qo, kl_, Bs, K, lib=lib)
    S = token_scores(iq, ik)  # [B, Nq, G, Nk]
    for r in range(n):
        b, i = rb[r], ri[r]
        pos = qo[b] + i
        for g in range(Hkv):
            toks = [j for t in sel[r, g] if t >= 0 for j in range(t * Bs, (t + 1) * Bs) if j <= pos and j < kl_[b]]
            sv = S[b, i, g, toks]
            m = sv.max()
            want = -math.log(len(toks)) - sv.mean() + m + math.log(np.exp(sv - m).sum())
            assert abs(klz[r, g] - want) < 1e-9 * max(1.0, abs(want))
    # a per-row constant added to every index score: an extra index dim, ik = 1, iq = c
    c = np.random.default_rng(6).integers(-5, 6, (iq.shape[0], iq.shape[1], Hkv, 1)).astype(np.float32)
    iq2 = np.concatenate([iq, c], axis=-1)
    ik2 = np.concatenate([ik, np.ones(ik.shape[:2] + (1,), np.float32)], axis=-1)
    kl2 = oracle.kl_aux(q.reshape(n, Hq, d), k, iq2.reshape(n, Hkv, di + 1), ik2, sel, rb, ri, qo, kl_, Bs, K,
                        lib=lib)
    assert np.abs(kl2 - kl).max() < 1e-9 * max(1.0, np.abs(kl).max())


GOLDEN_KL = os.path.join(os.path.dirname(__file__), "golden", "handworked_kl.txt")


def pin_kl_golden(lib=None):
    """The hand-worked KL values of tests/golden/handworked_kl.txt: two heads
    with different distributions (their probabilities averaged), unequal index
    scores, and a row with a single visible token."""
    k = np.array([0.0, math.log(3.0)], np.float32).reshape(1, 2, 1, 1)
    ik = np.array([0.0, 1.0], np.float32).reshape(1, 2, 1)
    n = 0
    with open(GOLDEN_KL) as f:
        for ln in f:
            ln = ln.split("#")[0].strip()
            if not ln:
                continue
            head, _, tail = ln.partition(":")
            parts = head.split()
            assert parts[0] == "kl", ln
            pos, q0, q1, iqv = int(parts[1]), float(parts[2]), float(parts[3]), float(parts[4])
            want = float(tail)
            got = oracle.kl_aux(np.array([[[q0], [q1]]], np.float32), k, np.array([[[iqv]]], np.float32), ik,
                                np.array([[[0]]], np.int32), [0], [pos], [0], [2], 2, 1, scale=1.0, lib=lib)
            assert abs(got[0, 0] - want) < 1e-7, (ln, got[0, 0])
            n += 1
    assert n == 3


def _bwd_inputs(seed, B=2, Nq=40, Nk=96, Hq=4, Hkv=2, d=16, Bs=8, K=5):
    q, k, v, iq, ik, qo, kl = rand_problem(seed, B=B, Nq=Nq, Nk=Nk, Hq=Hq, Hkv=Hkv, d=d, di=8,
                                           q_offset=[Nk - Nq, 20], kv_len=[Nk, Nq + 20])
    rb, ri = oracle.all_rows(B, Nq)
    sel = oracle.index_select(iq.reshape(-1, Hkv, 8), ik, rb, ri, qo, kl, Bs, K)
    dout = np.random.default_rng(seed + 100).standard_normal(q.shape).astype(np.float32)
    return q, k, v, dout, qo, kl, rb, ri, sel


def pin_attn_backward(lib=None):
    """Main Branch backward: torch autograd through the masked-dense
    restatement in fp64; the closed forms of its sums; central finite
    differences of the (separately pinned) forward oracle on a tiny case."""
    Bs, K = 8, 5
    B, Nq, Nk, Hq, Hkv, d = 2, 40, 96, 4, 2, 16
    hpg = Hq // Hkv
    q, k, v, dout, qo, kl_, rb, ri, sel = _bwd_inputs(31)
    dq, dk, dv = oracle.sparse_attn_backward(q.reshape(-1, Hq, d), k, v, dout.reshape(-1, Hq, d), sel, rb, ri, qo,
                                             kl_, Bs, K, lib=lib)
    scale = 1.0 / math.sqrt(d)
    allowed = selected_allowed(sel.reshape(B, Nq, Hkv, K), Bs, B, Nq, Nk, Hkv, qo, kl_)
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    vt = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    s_ = torch.einsum("bihc,bjhc->bhij", qt, kt.repeat_interleave(hpg, dim=2)) * scale
    m = torch.from_numpy(allowed).repeat_interleave(hpg, dim=2).permute(0, 2, 1, 3)
    p_ = torch.softmax(s_.masked_fill(~m, -math.inf), dim=-1)
    o = torch.einsum("bhij,bjhc->bihc", p_, vt.repeat_interleave(hpg, dim=2))
    (o * torch.from_numpy(dout.astype(np.float64))).sum().backward()
    for got, want in ((dq.reshape(B, Nq, Hq, d), qt.grad), (dk, kt.grad), (dv, vt.grad)):
        want = want.numpy()
        assert np.abs(got - want).max() < 1e-10 * max(1.0, np.abs(want).max())
    # closed forms per (sequence, kv head)
    for b in range(B):
        for g in range(Hkv):
            assert np.abs(dk[b, :, g].sum(axis=0)).max() < 1e-9
            want_v = dout[b, :, g * hpg:(g + 1) * hpg].astype(np.float64).sum(axis=(0, 1))
            assert np.abs(dv[b, :, g].sum(axis=0) - want_v).max() < 1e-9
            qdq = (q[b, :, g * hpg:(g + 1) * hpg].astype(np.float64) *
                   dq.reshape(B, Nq, Hq, d)[b, :, g * hpg:(g + 1) * hpg]).sum()
            kdk = (k[b, :, g].astype(np.float64) * dk[b, :, g]).sum()
            assert abs(qdq - kdk) < 1e-9 * max(1.0, abs(qdq))
    # finite differences: dyadic inputs so that x +- h is exact in fp32
    rng = np.random.default_rng(8)
    B1, N1, Hq1, Hkv1, d1, Bs1, K1 = 1, 24, 2, 1, 8, 4, 3
    q1 = (rng.integers(-32, 33, (B1, N1, Hq1, d1)) / 16).astype(np.float32)
    k1 = (rng.integers(-32, 33, (B1, N1, Hkv1, d1)) / 16).astype(np.float32)
    v1 = (rng.integers(-32, 33, (B1, N1, Hkv1, d1)) / 16).astype(np.float32)
    g1 = (rng.integers(-32, 33, (B1, N1, Hq1, d1)) / 16).astype(np.float32)
    iq1 = rng.integers(-3, 4, (B1, N1, Hkv1, 4)).astype(np.float32)
    ik1 = rng.integers(-3, 4, (B1, N1, 4)).astype(np.float32)
    rb1, ri1 = oracle.all_rows(B1, N1)
    qo1, kl1 = np.zeros(1, np.int32), np.full(1, N1, np.int32)
    sel1 = oracle.index_select(iq1.reshape(-1, Hkv1, 4), ik1, rb1, ri1, qo1, kl1, Bs1, K1)
    gq, gk, gv = oracle.sparse_attn_backward(q1.reshape(-1, Hq1, d1), k1, v1, g1.reshape(-1, Hq1, d1), sel1, rb1, ri1,
                                             qo1, kl1, Bs1, K1, lib=lib)
    grads = {"q": gq.reshape(q1.shape), "k": gk, "v": gv}

    def loss(qq, kk, vv):
        out, _ = oracle.sparse_attn(qq.reshape(-1, Hq1, d1), kk, vv, sel1, rb1, ri1, qo1, kl1, Bs1, K1)
        return float((out * g1.reshape(-1, Hq1, d1).astype(np.float64)).sum())

    h = 2.0 ** -10
    for name, arr in (("q", q1), ("k", k1), ("v", v1)):
        for _ in range(5):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            xp, xm = arr.copy(), arr.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q1, "k": k1, "v": v1, name: xp}
            args_m = {"q": q1, "k": k1, "v": v1, name: xm}
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            assert abs(fd - grads[name][idx]) < 1e-5 * max(1.0, abs(fd)), (name, idx, fd, grads[name][idx])


PINS = [pin_golden, pin_blockmax_bruteforce, pin_selection_invariants, pin_closed_forms, pin_dense_equals_sdpa,
        pin_masked_dense_equals_sdpa, pin_attention_special_cases, pin_decode_equals_prefill_row, pin_force_start,
        pin_kl_aux, pin_kl_golden, pin_attn_backward]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: a broken copy of the oracle must fail some pin
# ---------------------------------------------------------------------------
MUTATIONS = {
    "tie_to_higher_block": ("return a < b;", "return a > b;"),
    "local_block_not_forced": ("chosen.push_back(loc);  // the query's own block is always kept",
                               "chosen.push_back(cand[K - 1]);"),
    "causal_excludes_diagonal": ("j < L && j <= pos; ++j", "j < L && j < pos; ++j"),
    "gqa_head_map_modulo": ("const int g = h / heads_per_group;", "const int g = h % Hkv;"),
    "scale_without_sqrt": ("scale = 1.0 / std::sqrt(double(d));", "scale = 1.0 / double(d);"),
    "score_dim_off_by_one": ("for (int c = 0; c < di; ++c) s +=", "for (int c = 1; c < di; ++c) s +="),
    "blockmax_keeps_min": ("if (s > M[t]) M[t] = s;", "if (s < M[t] || M[t] == -std::numeric_limits<double>::infinity()) M[t] = s;"),
    "selects_lowest_maxima": ("if (M[a] != M[b]) return M[a] > M[b];", "if (M[a] != M[b]) return M[a] < M[b];"),
    "start_variant_ranks_one_too_many": ("const int ranked = K - 1 - first;", "const int ranked = K - 1;"),
    "start_variant_ranks_block_zero": ("const int first = force_start ? 1 : 0;", "const int first = 0;"),
    "kl_causal_excludes_diagonal": ("j <= pos && j < L; ++j) keys.push_back(j);  // causal, diagonal kept",
                                    "j < pos && j < L; ++j) keys.push_back(j);"),
    "kl_heads_not_averaged": ("p[x] += std::exp(z[x] - m) / l / double(hpg);", "p[x] += std::exp(z[x] - m) / l;"),
    "kl_index_scores_scaled": ("        s[x] = acc;\n", "        s[x] = acc * scale;\n"),
    "bwd_drops_delta": ("const double dS = P[x] * (dP - delta);", "const double dS = P[x] * dP;"),
    "bwd_dk_unscaled": ("dk[kvrow + c] += scale * dS * double(qh[c]);", "dk[kvrow + c] += dS * double(qh[c]);"),
    "bwd_dv_weighted_by_ds": ("dv[kvrow + c] += P[x] * double(gh[c]);", "dv[kvrow + c] += dS * double(gh[c]);"),
    "bwd_causal_excludes_diagonal": ("if (j > pos || j >= L) break;", "if (j >= pos || j >= L) break;"),
    "bwd_dq_from_values": ("dqh[c] += scale * dS * double(kj[c]);", "dqh[c] += scale * dS * double(vj[c]);"),
    "kl_reversed_direction": ("if (p[x] > 0.0) div += p[x] * (std::log(p[x]) - (s[x] - lse_q));",
                              "div += std::exp(s[x] - lse_q) * ((s[x] - lse_q) - std::log(p[x] + 1e-300));"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = os.path.join(os.path.dirname(oracle.__file__), "msa_oracle.cpp")
    text = open(src).read()
    old, new = MUTATIONS[name]
    assert text.count(old) == 1, name
    mut_src = tmp_path / "mut.cpp"
    mut_src.write_text(text.replace(old, new))
    lib = oracle.load(oracle.build(str(mut_src), str(tmp_path / "libmut.so")))
    failed = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutation {name} passed every pin"


def test_oracle_independent_of_thread_count():
    """Every oracle function gives bit-identical results on 1 and 4 threads
    (rows are independent; the backward's dk / dv sums keep a fixed order), so
    the timed CPU baseline and the parity references are the same computation."""
    q, k, v, iq, ik, qo, kl = rand_problem(7, B=2, Nq=40, Nk=96, q_offset=[56, 20], kv_len=[96, 60])
    rb, ri = oracle.all_rows(2, 40)
    g = np.random.default_rng(1).standard_normal(q.shape).astype(np.float32)
    res = []
    for nt in (1, 4):
        sel = oracle.index_select(iq.reshape(-1, 2, 8), ik, rb, ri, qo, kl, 8, 5, nthreads=nt)
        out, lse = oracle.sparse_attn(q.reshape(-1, 4, 16), k, v, sel, rb, ri, qo, kl, 8, 5, nthreads=nt)
        klv = oracle.kl_aux(q.reshape(-1, 4, 16), k, iq.reshape(-1, 2, 8), ik, sel, rb, ri, qo, kl, 8, 5, nthreads=nt)
        grads = oracle.sparse_attn_backward(q.reshape(-1, 4, 16), k, v, g.reshape(-1, 4, 16), sel, rb, ri, qo, kl, 8,
                                            5, nthreads=nt)
        res.append((sel, out, lse, klv) + tuple(grads))
    for a, b in zip(*res):
        assert np.array_equal(a, b)
