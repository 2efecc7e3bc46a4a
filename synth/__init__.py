"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds input generation only: no step of the sparse-attention method
is computed here. Every element is a counter-based draw (SplitMix64, see
``synth_host.c``), so any slice of any tensor can be regenerated on the host at
any size while the full tensor is generated on the device by ``synth_dev.cu``.

Recipe (stated once; the workload table lives in ``synth/workloads.py``):

* ``normal``: inverse-CDF lookup into a 65536-entry table
  ``z_k = Phi^-1((k + 0.5) / 65536)`` (fp64, then rounded to bf16 for bf16
  tensors or to fp32 for fp32 tensors), indexed by the top 16 bits of the draw.
  A quantised N(0, 1) whose tails stop at about +-4.2.
* ``int``: uniform over ``{-a..a}`` by multiply-high range reduction; the index
  key of "hot" blocks is multiplied by an integer factor (3) to skew block
  popularity. Integers up to 24 are exact in bf16.
* tensor ids: q=1, k=2, v=3, iq=4, ik=5, kv_len=6, hot-block pick=7.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from functools import lru_cache

import numpy as np

from .workloads import WORKLOADS, Workload, scaled, shapes  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
TID = {"q": 1, "k": 2, "v": 3, "iq": 4, "ik": 5, "kv_len": 6, "hot": 7}
_GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1


# ---------------------------------------------------------------------------
# build + load
# ---------------------------------------------------------------------------
def build(cuda: bool = True) -> None:
    """Compile the host generator (gcc) and, if requested, the device one (nvcc)."""
    host_src = os.path.join(_HERE, "synth_host.c")
    host_so = os.path.join(_HERE, "libsynth_host.so")
    subprocess.run(["gcc", "-O2", "-shared", "-fPIC", "-pthread", host_src, "-o", host_so], check=True)
    if cuda:
        dev_src = os.path.join(_HERE, "synth_dev.cu")
        dev_so = os.path.join(_HERE, "libsynth_dev.so")
        subprocess.run(["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                        "-Xcompiler", "-fPIC", dev_src, "-o", dev_so], check=True)


@lru_cache(maxsize=None)
def _host_lib():
    path = os.path.join(_HERE, "libsynth_host.so")
    if not os.path.exists(path):
        build(cuda=False)
    lib = ctypes.CDLL(path)
    u64, u32, i32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
    lib.synth_key.argtypes, lib.synth_key.restype = [u64, u32], u64
    lib.synth_u64.argtypes, lib.synth_u64.restype = [u64, u64], u64
    lib.synth_fill_normal.argtypes = [vp, i32, u64, u64, u64, u32, vp, i32]
    lib.synth_fill_normal.restype = None
    lib.synth_fill_int.argtypes = [vp, i32, u64, u64, u64, u32, i32, vp, u64, u64, i32]
    lib.synth_fill_int.restype = None
    return lib


@lru_cache(maxsize=None)
def _dev_lib():
    path = os.path.join(_HERE, "libsynth_dev.so")
    if not os.path.exists(path):
        raise RuntimeError("synth/libsynth_dev.so is not built: run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    u64, u32, i32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
    lib.synth_dev_fill_normal.argtypes = [vp, i32, u64, u64, u64, u32, vp, vp]
    lib.synth_dev_fill_normal.restype = i32
    lib.synth_dev_fill_int.argtypes = [vp, i32, u64, u64, u64, u32, i32, vp, u64, u64, vp]
    lib.synth_dev_fill_int.restype = i32
    return lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# ---------------------------------------------------------------------------
# scalar reference of the counter (pure Python ints; used by the tests)
# ---------------------------------------------------------------------------
def sm64_py(x: int) -> int:
    z = (x + _GAMMA) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def key_py(seed: int, tid: int) -> int:
    return sm64_py(((seed << 8) | (tid & 0xFF)) & _M64)


def u64_py(key: int, idx: int) -> int:
    return sm64_py((key + idx * _GAMMA) & _M64)


# ---------------------------------------------------------------------------
# value maps
# ---------------------------------------------------------------------------
def _round_f32_to_bf16(x: np.ndarray) -> np.ndarray:
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


@lru_cache(maxsize=None)
def normal_table(kind: str) -> np.ndarray:
    """65536 quantiles of N(0,1), rounded to ``kind`` ('bf16' or 'fp32')."""
    from scipy.special import ndtri

    p = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    z = ndtri(p).astype(np.float32)
    if kind == "bf16":
        z = _round_f32_to_bf16(z)
    elif kind != "fp32":
        raise ValueError(kind)
    z.setflags(write=False)
    return z


def _out_kind(kind: str) -> int:
    return {"fp32": 0, "bf16": 1}[kind]


# ---------------------------------------------------------------------------
# per-workload metadata
# ---------------------------------------------------------------------------
def kv_lens(w: Workload) -> np.ndarray:
    """Per-sequence key lengths: fixed Nk for prefill, uniform draws for decode."""
    if w.kv_len_range is None:
        return np.full(w.B, w.Nk, dtype=np.int32)
    lo, hi = w.kv_len_range
    key = key_py(w.seed, TID["kv_len"])
    n = hi - lo + 1
    return np.array([lo + ((u64_py(key, b) >> 32) * n >> 32) for b in range(w.B)], dtype=np.int32)


def q_offsets(w: Workload) -> np.ndarray:
    """Absolute position of query row 0 per sequence (queries are the last Nq keys)."""
    return (kv_lens(w) - w.Nq).astype(np.int32)


def hot_blocks(w: Workload) -> np.ndarray:
    """Indices of the key blocks whose index key is scaled by ``w.hot_mult``."""
    nblk = (w.Nk + w.Bs - 1) // w.Bs
    if w.hot == "none":
        return np.zeros(0, dtype=np.int64)
    if w.hot == "first4":
        return np.arange(min(4, nblk), dtype=np.int64)
    if w.hot == "pct1":
        count = int(round(0.01 * nblk))
        key = key_py(w.seed, TID["hot"])
        u = np.array([u64_py(key, t) for t in range(nblk)], dtype=np.uint64)
        order = np.lexsort((np.arange(nblk), u))  # smallest draws, ties to lower index
        return np.sort(order[:count]).astype(np.int64)
    raise ValueError(w.hot)


def row_mult(w: Workload) -> np.ndarray | None:
    """Per key token multiplier for the index key (1, or hot_mult in hot blocks)."""
    hb = hot_blocks(w)
    if hb.size == 0:
        return None
    m = np.ones(w.Nk, dtype=np.uint8)
    for t in hb:
        m[t * w.Bs:min((t + 1) * w.Bs, w.Nk)] = w.hot_mult
    return m


# ---------------------------------------------------------------------------
# host generation
# ---------------------------------------------------------------------------
def host_range(w: Workload, name: str, start: int, count: int) -> np.ndarray:
    """Flat elements [start, start+count) of tensor ``name`` as float32 (exact values)."""
    out = np.empty(count, dtype=np.float32)
    lib = _host_lib()
    if name in ("q", "k", "v"):
        table = normal_table(w.dtype)
        lib.synth_fill_normal(out.ctypes.data, 0, count, start, w.seed, TID[name], table.ctypes.data, _threads())
    elif name in ("iq", "ik"):
        rm = row_mult(w) if name == "ik" else None
        rm_ptr = rm.ctypes.data if rm is not None else None
        lib.synth_fill_int(out.ctypes.data, 0, count, start, w.seed, TID[name], w.idx_a, rm_ptr,
                           w.di, w.Nk, _threads())
    else:
        raise ValueError(name)
    return out


def host_tensor(w: Workload, name: str) -> np.ndarray:
    shp = shapes(w)[name]
    return host_range(w, name, 0, int(np.prod(shp))).reshape(shp)


def host_rows(w: Workload, name: str, b: int, rows) -> np.ndarray:
    """Rows ``rows`` (token positions) of sequence ``b`` of a [B, L, ...] tensor."""
    shp = shapes(w)[name]
    row_elems = int(np.prod(shp[2:]))
    out = np.empty((len(rows),) + tuple(shp[2:]), dtype=np.float32)
    for n, r in enumerate(rows):
        start = (b * shp[1] + int(r)) * row_elems
        out[n] = host_range(w, name, start, row_elems).reshape(shp[2:])
    return out


# ---------------------------------------------------------------------------
# device generation (torch only allocates)
# ---------------------------------------------------------------------------
def device_tensor(w: Workload, name: str, device="cuda", stream=None):
    import torch

    shp = shapes(w)[name]
    tdt = torch.float32 if w.dtype == "fp32" else torch.bfloat16
    out = torch.empty(shp, dtype=tdt, device=device)
    fill_device(w, name, out, stream=stream)
    return out


def fill_device(w: Workload, name: str, out, start: int = 0, stream=None) -> None:
    import torch

    lib = _dev_lib()
    s = (stream or torch.cuda.current_stream(out.device)).cuda_stream
    kind = _out_kind(w.dtype)
    n = out.numel()
    if name in ("q", "k", "v"):
        table = torch.from_numpy(normal_table(w.dtype).copy()).to(out.device)
        rc = lib.synth_dev_fill_normal(out.data_ptr(), kind, n, start, w.seed, TID[name], table.data_ptr(), s)
        torch.cuda.synchronize(out.device)  # the table is freed on return
        del table
    elif name in ("iq", "ik"):
        rm = row_mult(w) if name == "ik" else None
        rm_t = torch.from_numpy(rm).to(out.device) if rm is not None else None
        rc = lib.synth_dev_fill_int(out.data_ptr(), kind, n, start, w.seed, TID[name], w.idx_a,
                                    rm_t.data_ptr() if rm_t is not None else None, w.di, w.Nk, s)
        torch.cuda.synchronize(out.device)  # the multiplier table is freed on return
        del rm_t
    else:
        raise ValueError(name)
    if rc != 0:
        raise RuntimeError(f"synth device fill failed: cuda error {rc}")
