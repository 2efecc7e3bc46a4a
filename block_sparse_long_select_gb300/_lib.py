"""ctypes binding of libmsa.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import os
from functools import lru_cache

MSA_BF16, MSA_FP32 = 0, 1
MSA_OP_INDEX_SELECT, MSA_OP_PREFILL, MSA_OP_DECODE, MSA_OP_DECODE_STEP, MSA_OP_KL_AUX, MSA_OP_BACKWARD = 0, 1, 2, 3, 4, 5
MSA_FORCE_LOCAL, MSA_FORCE_START = 1, 2
STATUS_NAMES = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_WORKSPACE",
                4: "MSA_ERR_CUDA", 5: "MSA_ERR_TIMEOUT", 6: "MSA_ERR_BOUNDS"}

# (name, restype, argtypes) of every symbol declared in include/msa.h
_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "msa_workspace_size": (_sz, [_i32] * 11),
    "msa_index_select": (_i32, [_vp, _vp, _vp, _vp] + [_i32] * 8 + [_vp, _vp, _vp, _sz, _vp]),
    "msa_index_select_v": (_i32, [_vp, _vp, _vp, _vp] + [_i32] * 9 + [_vp, _vp, _vp, _sz, _vp]),
    "msa_sparse_attn_prefill": (_i32, [_vp] * 6 + [_i32] * 8 + [_f32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "msa_sparse_attn_decode": (_i32, [_vp] * 5 + [_i32] * 7 + [_f32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "msa_decode_step": (_i32, [_vp] * 9 + [_i32] * 8 + [_f32, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "msa_kl_aux_forward": (_i32, [_vp] * 8 + [_i32] * 9 + [_f32, _i32, _vp, _vp, _sz, _vp]),
    "msa_sparse_attn_backward": (_i32, [_vp] * 9 + [_i32] * 8 + [_f32, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "msa_read_status": (_i32, [_vp, _vp]),
    "msa_status_string": (ctypes.c_char_p, [_i32]),
    "msa_index_select_noalloc": (_i32, [_vp, _vp, _vp, _vp] + [_i32] * 8 + [_vp, _vp, _vp]),
    "msa_profile_begin": (_i32, []),
    "msa_profile_end": (_i32, [_vp, _i32]),
    "msa_debug_inject_timeout": (_i32, [_i32]),
}


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


class MsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmsa.so")


@lru_cache(maxsize=None)
def load_library():
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with block_sparse_long_select_gb300.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


# ---------------------------------------------------------------------------
def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return MSA_BF16
    if t.dtype == torch.float32:
        return MSA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, where: str):
    if code != 0:
        raise MsaError(code, where)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _check_select_args(iq, ik, q_offset, kv_len, Bs, K, sel, block_max):
    """Shapes, dtypes and devices of an index selection's tensors (the library
    writes sel and block_max through raw pointers: a short or mistyped buffer
    would be overrun on the device)."""
    import torch

    if iq.dim() != 4 or ik.dim() != 3:
        raise ValueError("iq must be [B, Nq, G, di] and ik [B, Nk, di]")
    B, Nq, G, di = iq.shape
    if ik.shape[0] != B or ik.shape[2] != di or ik.dtype != iq.dtype or ik.device != iq.device:
        raise ValueError("ik must be [B, Nk, di] with iq's dtype and device")
    for name, t in (("q_offset", q_offset), ("kv_len", kv_len)):
        if t is not None and (t.dtype != torch.int32 or t.numel() != B or t.device != iq.device):
            raise ValueError(f"{name} must be int32 of length B on iq's device")
    if sel is not None and (sel.dtype != torch.int32 or sel.numel() != B * Nq * G * K or sel.device != iq.device):
        raise ValueError("sel must be int32 with B * Nq * G * K elements on iq's device")
    nblk = (ik.shape[1] + Bs - 1) // Bs if Bs > 0 else 0
    if block_max is not None and (block_max.dtype != torch.float32 or block_max.numel() != B * Nq * G * nblk or
                                  block_max.device != iq.device):
        raise ValueError("block_max must be float32 with B * Nq * G * ceil(Nk / Bs) elements on iq's device")


def msa_workspace_size(op, B, Nq, Nk, G, Hq, d, di, Bs, K, dtype) -> int:
    return int(load_library().msa_workspace_size(op, B, Nq, Nk, G, Hq, d, di, Bs, K, dtype))


def workspace(nbytes: int, device="cuda"):
    """Zero-filled device scratch of ``nbytes`` (caching-allocator blocks are 512-byte aligned)."""
    import torch

    ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def msa_index_select(iq, ik, q_offset, kv_len, Bs, K, sel=None, block_max=None, ws=None, stream=None):
    """iq [B,Nq,G,di], ik [B,Nk,di] -> sel [B,Nq,G,K] int32 (see include/msa.h)."""
    return msa_index_select_v(iq, ik, q_offset, kv_len, Bs, K, MSA_FORCE_LOCAL, sel, block_max, ws, stream)


def msa_index_select_v(iq, ik, q_offset, kv_len, Bs, K, force, sel=None, block_max=None, ws=None, stream=None):
    """msa_index_select with a choice of forced blocks: force = MSA_FORCE_LOCAL,
    or MSA_FORCE_LOCAL | MSA_FORCE_START to keep block 0 as well (see include/msa.h)."""
    import torch

    _need_cuda(iq, ik, q_offset, kv_len, sel, block_max)
    _check_select_args(iq, ik, q_offset, kv_len, Bs, K, sel, block_max)
    B, Nq, G, di = iq.shape
    Nk = ik.shape[1]
    dt = _dtype_code(iq)
    if sel is None:
        sel = torch.empty((B, Nq, G, K), dtype=torch.int32, device=iq.device)
    if ws is None:
        ws = workspace(msa_workspace_size(MSA_OP_INDEX_SELECT, B, Nq, Nk, G, 0, 0, di, Bs, K, dt), iq.device)
    code = load_library().msa_index_select_v(_ptr(iq), _ptr(ik), _ptr(q_offset), _ptr(kv_len), B, Nq, Nk, G, di,
                                             Bs, K, dt, int(force), _ptr(sel), _ptr(block_max), _ptr(ws), ws.numel(),
                                             _stream(stream, iq.device))
    _check(code, "msa_index_select_v")
    return sel


def msa_index_select_noalloc(iq, ik, q_offset, kv_len, Bs, K, sel, block_max=None, stream=None):
    """msa_index_select on the library's static scratch (no workspace; see include/msa.h).
    ``sel`` must be given: this wrapper allocates nothing either."""
    _need_cuda(iq, ik, q_offset, kv_len, sel, block_max)
    if sel is None:
        raise ValueError("msa_index_select_noalloc needs a caller-owned sel")
    _check_select_args(iq, ik, q_offset, kv_len, Bs, K, sel, block_max)
    B, Nq, G, di = iq.shape
    Nk = ik.shape[1]
    code = load_library().msa_index_select_noalloc(_ptr(iq), _ptr(ik), _ptr(q_offset), _ptr(kv_len), B, Nq, Nk, G,
                                                   di, Bs, K, _dtype_code(iq), _ptr(sel), _ptr(block_max),
                                                   _stream(stream, iq.device))
    _check(code, "msa_index_select_noalloc")
    return sel


def msa_sparse_attn_prefill(q, k, v, sel, q_offset, kv_len, Bs, K, scale=0.0, out=None, lse=None, ws=None,
                            stream=None):
    """q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d], sel [B,Nq,Hkv,K] -> out [B,Nq,Hq,d]."""
    import torch

    _need_cuda(q, k, v, sel, q_offset, kv_len, out, lse)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(msa_workspace_size(MSA_OP_PREFILL, B, Nq, Nk, Hkv, Hq, d, 0, Bs, K, dt), q.device)
    code = load_library().msa_sparse_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(q_offset),
                                                  _ptr(kv_len), B, Nq, Nk, Hq, Hkv, d, Bs, K, float(scale), dt,
                                                  _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                                  _stream(stream, q.device))
    _check(code, "msa_sparse_attn_prefill")
    return out


def msa_sparse_attn_decode(q, k_cache, v_cache, sel, kv_len, Bs, K, scale=0.0, out=None, lse=None, ws=None,
                           stream=None):
    """q [B,Hq,d], caches [B,Lmax,Hkv,d], sel [B,Hkv,K] (or [B,1,Hkv,K]) -> out [B,Hq,d]."""
    import torch

    _need_cuda(q, k_cache, v_cache, sel, kv_len, out, lse)
    B, Hq, d = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(msa_workspace_size(MSA_OP_DECODE, B, 1, Lmax, Hkv, Hq, d, 0, Bs, K, dt), q.device)
    code = load_library().msa_sparse_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(sel), _ptr(kv_len),
                                                 B, Lmax, Hq, Hkv, d, Bs, K, float(scale), dt, _ptr(out), _ptr(lse),
                                                 _ptr(ws), ws.numel(), _stream(stream, q.device))
    _check(code, "msa_sparse_attn_decode")
    return out


def msa_read_status(ws, stream=None) -> int:
    return int(load_library().msa_read_status(_ptr(ws), _stream(stream, ws.device)))


def msa_status_string(code: int) -> str:
    return load_library().msa_status_string(int(code)).decode()


def msa_profile_begin() -> None:
    load_library().msa_profile_begin()


def msa_profile_end() -> dict:
    """{kernel name: (launches, total device ms)} recorded since msa_profile_begin()."""
    buf = (KernelTime * 64)()
    n = load_library().msa_profile_end(ctypes.cast(buf, ctypes.c_void_p), 64)
    if n < 0:
        raise RuntimeError("msa_profile_end: event query failed")
    return {buf[k].name.decode(): (buf[k].launches, buf[k].total_ms) for k in range(min(n, 64))}


def msa_debug_inject_timeout(enable: bool) -> bool:
    """Test hook (see include/msa_profile.h): while on, the attention kernels
    make one bounded wait that runs out and report MSA_ERR_TIMEOUT. Returns the
    previous setting."""
    return bool(load_library().msa_debug_inject_timeout(1 if enable else 0))


def msa_decode_step(q, k_new, v_new, iq, ik_new, k_cache, v_cache, ik_cache, kv_len, Bs, K, sel=None, out=None,
                    lse=None, scale=0.0, ws=None, stream=None):
    """One streaming decode step (see include/msa.h): append the new token's
    k [B,Hkv,d], v, index key [B,di] at kv_len[b] of the caches, advance
    kv_len, then select and attend for q [B,Hq,d], iq [B,Hkv,di].
    Returns (sel [B,Hkv,K], out [B,Hq,d])."""
    import torch

    _need_cuda(q, k_new, v_new, iq, ik_new, k_cache, v_cache, ik_cache, kv_len, sel, out, lse)
    B, Hq, d = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    di = ik_cache.shape[2]
    dt = _dtype_code(q)
    if sel is None:
        sel = torch.empty((B, Hkv, K), dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(msa_workspace_size(MSA_OP_DECODE_STEP, B, 0, Lmax, Hkv, Hq, d, di, Bs, K, dt), q.device)
    code = load_library().msa_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(iq), _ptr(ik_new), _ptr(k_cache),
                                          _ptr(v_cache), _ptr(ik_cache), _ptr(kv_len), B, Lmax, Hq, Hkv, d, di, Bs, K,
                                          float(scale), dt, _ptr(sel), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                          _stream(stream, q.device))
    _check(code, "msa_decode_step")
    return sel, out


def msa_kl_aux_forward(q, k, iq, ik, sel, lse, q_offset, kv_len, Bs, K, kl=None, scale=0.0, ws=None, stream=None):
    """KL auxiliary forward (see include/msa.h): KL(head-averaged main-branch
    distribution || index softmax) per (row, group) -> kl [B, Nq, Hkv] fp32.
    ``lse`` is the forward's [B, Nq, Hq] output of msa_sparse_attn_prefill."""
    import torch

    _need_cuda(q, k, iq, ik, sel, lse, q_offset, kv_len, kl)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    di = iq.shape[3]
    dt = _dtype_code(q)
    if kl is None:
        kl = torch.empty((B, Nq, Hkv), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(msa_workspace_size(MSA_OP_KL_AUX, B, Nq, Nk, Hkv, Hq, d, di, Bs, K, dt), q.device)
    code = load_library().msa_kl_aux_forward(_ptr(q), _ptr(k), _ptr(iq), _ptr(ik), _ptr(sel), _ptr(lse),
                                             _ptr(q_offset), _ptr(kv_len), B, Nq, Nk, Hq, Hkv, d, di, Bs, K,
                                             float(scale), dt, _ptr(kl), _ptr(ws), ws.numel(),
                                             _stream(stream, q.device))
    _check(code, "msa_kl_aux_forward")
    return kl


def msa_sparse_attn_backward(q, k, v, out, dout, lse, sel, q_offset, kv_len, Bs, K, dq=None, dk=None, dv=None,
                             scale=0.0, ws=None, stream=None):
    """Main Branch backward (see include/msa.h): gradients of q [B,Nq,Hq,d],
    k and v [B,Nk,Hkv,d] through msa_sparse_attn_prefill, given its output
    ``out``, lse [B,Nq,Hq] and selection ``sel`` and the output gradient
    ``dout``. Returns (dq, dk, dv) in q's dtype."""
    import torch

    _need_cuda(q, k, v, out, dout, lse, sel, q_offset, kv_len, dq, dk, dv)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if ws is None:
        ws = workspace(msa_workspace_size(MSA_OP_BACKWARD, B, Nq, Nk, Hkv, Hq, d, 0, Bs, K, dt), q.device)
    code = load_library().msa_sparse_attn_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                                   _ptr(sel), _ptr(q_offset), _ptr(kv_len), B, Nq, Nk, Hq, Hkv, d,
                                                   Bs, K, float(scale), dt, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                                   ws.numel(), _stream(stream, q.device))
    _check(code, "msa_sparse_attn_backward")
    return dq, dk, dv
