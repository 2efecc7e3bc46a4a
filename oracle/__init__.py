"""CPU oracle for the MSA path (TEST INFRASTRUCTURE ONLY).

Thin ctypes wrapper over ``msa_oracle.cpp``: plain fp64 C++ that restates the
Index Branch (dot-product index scores, block max pooling, top-K with the local
block forced, ties to the lower block), the Main Branch (exact causal softmax
attention over the selected blocks) with its backward, and the KL auxiliary
value. Only ``tests/``, the smoke check
and the bench's CPU-baseline / reference leg may import this package; the
product library never does. It shares no code with the CUDA path: inputs come
from ``synth`` (generation only), everything else is computed here.

Every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from functools import lru_cache

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libmsa_oracle.so")


def build(src=None, out=None) -> str:
    """Compile the oracle with the host C++ compiler (plain -O2, no fast-math)."""
    src = src or os.path.join(_HERE, "msa_oracle.cpp")
    out = out or _SO
    subprocess.run(["g++", "-std=c++17", "-O2", "-fno-fast-math", "-shared", "-fPIC", "-pthread", src,
                    "-o", out], check=True)
    return out


def load(path):
    """Load an oracle build at ``path`` (the tests load deliberately broken copies)."""
    return _load(path)


def _load(path):
    lib = ctypes.CDLL(path)
    vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.msa_oracle_index_select.argtypes = [vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp,
                                            i32]
    lib.msa_oracle_index_select.restype = i32
    lib.msa_oracle_index_select_v.argtypes = [vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp,
                                              vp, i32]
    lib.msa_oracle_index_select_v.restype = i32
    lib.msa_oracle_sparse_attn.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32, i32,
                                           i32, f64, vp, vp, i32]
    lib.msa_oracle_sparse_attn.restype = i32
    lib.msa_oracle_kl_aux.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                      f64, vp, i32]
    lib.msa_oracle_kl_aux.restype = i32
    lib.msa_oracle_sparse_attn_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32,
                                                    i32, i32, i32, f64, vp, vp, vp, i32]
    lib.msa_oracle_sparse_attn_backward.restype = i32
    return lib


@lru_cache(maxsize=None)
def _lib():
    if not os.path.exists(_SO):
        build()
    return _load(_SO)


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def index_select(iq_rows, ik, row_b, row_i, q_offset, kv_len, Bs, K, want_block_max=False, nthreads=None,
                 lib=None, force_start=False):
    """Index Branch for listed rows.

    iq_rows [n, G, di]; ik [B, Nk, di]; row_b/row_i [n]; q_offset/kv_len [B].
    force_start keeps block 0 as well as the local block (the experiments'
    hard-coded sequence-start ablation; needs K >= 2).
    Returns sel [n, G, K] int32 (and block_max [n, G, nblk] fp64 if asked).
    """
    iq_rows = _c(iq_rows, np.float32)
    ik = _c(ik, np.float32)
    n, G, di = iq_rows.shape
    B, Nk, di2 = ik.shape
    assert di == di2
    row_b, row_i = _c(row_b, np.int32), _c(row_i, np.int32)
    q_offset, kv_len = _c(q_offset, np.int32), _c(kv_len, np.int32)
    nblk = (Nk + Bs - 1) // Bs
    sel = np.empty((n, G, K), dtype=np.int32)
    bmax = np.empty((n, G, nblk), dtype=np.float64) if want_block_max else None
    rc = (lib or _lib()).msa_oracle_index_select_v(iq_rows.ctypes.data, ik.ctypes.data, row_b.ctypes.data,
                                                   row_i.ctypes.data, n, q_offset.ctypes.data, kv_len.ctypes.data,
                                                   B, Nk, G, di, Bs, K, 1 if force_start else 0, sel.ctypes.data,
                                                   bmax.ctypes.data if bmax is not None else None,
                                                   nthreads or threads())
    if rc != 0:
        raise ValueError("oracle index_select rejected its arguments")
    return (sel, bmax) if want_block_max else sel


def sparse_attn(q_rows, k, v, sel_rows, row_b, row_i, q_offset, kv_len, Bs, K, scale=0.0, nthreads=None,
                lib=None):
    """Main Branch for listed rows.

    q_rows [n, Hq, d]; k, v [B, Nk, Hkv, d]; sel_rows [n, Hkv, K].
    Returns out [n, Hq, d] fp64 and lse [n, Hq] fp64.
    """
    q_rows = _c(q_rows, np.float32)
    k = k if (k.dtype == np.float32 and k.flags.c_contiguous) else _c(k, np.float32)
    v = v if (v.dtype == np.float32 and v.flags.c_contiguous) else _c(v, np.float32)
    n, Hq, d = q_rows.shape
    B, Nk, Hkv, d2 = k.shape
    assert d == d2 and v.shape == k.shape
    sel_rows = _c(sel_rows, np.int32)
    assert sel_rows.shape == (n, Hkv, K)
    row_b, row_i = _c(row_b, np.int32), _c(row_i, np.int32)
    q_offset, kv_len = _c(q_offset, np.int32), _c(kv_len, np.int32)
    out = np.empty((n, Hq, d), dtype=np.float64)
    lse = np.empty((n, Hq), dtype=np.float64)
    rc = (lib or _lib()).msa_oracle_sparse_attn(q_rows.ctypes.data, k.ctypes.data, v.ctypes.data, sel_rows.ctypes.data,
                                       row_b.ctypes.data, row_i.ctypes.data, n, q_offset.ctypes.data,
                                       kv_len.ctypes.data, B, Nk, Hq, Hkv, d, Bs, K, float(scale),
                                       out.ctypes.data, lse.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError("oracle sparse_attn rejected its arguments")
    return out, lse


def kl_aux(q_rows, k, iq_rows, ik, sel_rows, row_b, row_i, q_offset, kv_len, Bs, K, scale=0.0, nthreads=None,
           lib=None):
    """KL auxiliary forward for listed rows: KL(head-averaged main-branch
    distribution || index softmax) over each (row, group)'s selected tokens.

    q_rows [n, Hq, d]; k [B, Nk, Hkv, d]; iq_rows [n, Hkv, di]; ik [B, Nk, di];
    sel_rows [n, Hkv, K]. Returns kl [n, Hkv] fp64.
    """
    q_rows, iq_rows = _c(q_rows, np.float32), _c(iq_rows, np.float32)
    k = k if (k.dtype == np.float32 and k.flags.c_contiguous) else _c(k, np.float32)
    ik = _c(ik, np.float32)
    n, Hq, d = q_rows.shape
    B, Nk, Hkv, _ = k.shape
    di = iq_rows.shape[2]
    sel_rows = _c(sel_rows, np.int32)
    row_b, row_i = _c(row_b, np.int32), _c(row_i, np.int32)
    q_offset, kv_len = _c(q_offset, np.int32), _c(kv_len, np.int32)
    kl = np.empty((n, Hkv), dtype=np.float64)
    rc = (lib or _lib()).msa_oracle_kl_aux(q_rows.ctypes.data, k.ctypes.data, iq_rows.ctypes.data, ik.ctypes.data,
                                           sel_rows.ctypes.data, row_b.ctypes.data, row_i.ctypes.data, n,
                                           q_offset.ctypes.data, kv_len.ctypes.data, B, Nk, Hq, Hkv, d, di, Bs, K,
                                           float(scale), kl.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError("oracle kl_aux rejected its arguments")
    return kl


def sparse_attn_backward(q_rows, k, v, dout_rows, sel_rows, row_b, row_i, q_offset, kv_len, Bs, K, scale=0.0,
                         nthreads=None, lib=None):
    """Main Branch backward for listed rows (the selection carries no gradient).

    q_rows, dout_rows [n, Hq, d]; k, v [B, Nk, Hkv, d]; sel_rows [n, Hkv, K].
    Returns dq [n, Hq, d] and dk, dv [B, Nk, Hkv, d] (fp64): the listed rows'
    contributions.
    """
    q_rows, dout_rows = _c(q_rows, np.float32), _c(dout_rows, np.float32)
    k = k if (k.dtype == np.float32 and k.flags.c_contiguous) else _c(k, np.float32)
    v = v if (v.dtype == np.float32 and v.flags.c_contiguous) else _c(v, np.float32)
    n, Hq, d = q_rows.shape
    B, Nk, Hkv, d2 = k.shape
    assert d == d2 and v.shape == k.shape and dout_rows.shape == q_rows.shape
    sel_rows = _c(sel_rows, np.int32)
    assert sel_rows.shape == (n, Hkv, K)
    row_b, row_i = _c(row_b, np.int32), _c(row_i, np.int32)
    q_offset, kv_len = _c(q_offset, np.int32), _c(kv_len, np.int32)
    dq = np.empty((n, Hq, d), dtype=np.float64)
    dk = np.empty((B, Nk, Hkv, d), dtype=np.float64)
    dv = np.empty((B, Nk, Hkv, d), dtype=np.float64)
    rc = (lib or _lib()).msa_oracle_sparse_attn_backward(
        q_rows.ctypes.data, k.ctypes.data, v.ctypes.data, dout_rows.ctypes.data, sel_rows.ctypes.data,
        row_b.ctypes.data, row_i.ctypes.data, n, q_offset.ctypes.data, kv_len.ctypes.data, B, Nk, Hq, Hkv, d, Bs, K,
        float(scale), dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError("oracle sparse_attn_backward rejected its arguments")
    return dq, dk, dv


# ---------------------------------------------------------------------------
# whole problems (all rows), used by the pins and small parity cases
# ---------------------------------------------------------------------------
def all_rows(B, Nq):
    rb = np.repeat(np.arange(B, dtype=np.int32), Nq)
    ri = np.tile(np.arange(Nq, dtype=np.int32), B)
    return rb, ri


def msa_forward(q, k, v, iq, ik, Bs, K, q_offset=None, kv_len=None, scale=0.0, nthreads=None, lib=None):
    """Full MSA forward over dense arrays: q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d],
    iq [B,Nq,G,di], ik [B,Nk,di]. Returns (sel [B,Nq,G,K], out, lse)."""
    B, Nq, Hq, d = q.shape
    Nk = k.shape[1]
    G = iq.shape[2]
    q_offset = np.zeros(B, np.int32) if q_offset is None else np.asarray(q_offset, np.int32)
    kv_len = np.full(B, Nk, np.int32) if kv_len is None else np.asarray(kv_len, np.int32)
    rb, ri = all_rows(B, Nq)
    sel = index_select(iq.reshape(B * Nq, G, -1), ik, rb, ri, q_offset, kv_len, Bs, K, nthreads=nthreads,
                       lib=lib)
    out, lse = sparse_attn(q.reshape(B * Nq, Hq, d), k, v, sel, rb, ri, q_offset, kv_len, Bs, K, scale,
                           nthreads=nthreads, lib=lib)
    return sel.reshape(B, Nq, G, K), out.reshape(B, Nq, Hq, d), lse.reshape(B, Nq, Hq)
