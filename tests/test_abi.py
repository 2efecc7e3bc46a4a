"""C ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import block_sparse_long_select_gb300 as msa
from block_sparse_long_select_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(msa_[a-z_]+)\s*\(", text, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.lib_path()):
        msa.build()
    return msa.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"msa_index_select", "msa_sparse_attn_prefill", "msa_sparse_attn_decode", "msa_workspace_size",
            "msa_read_status", "msa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert msa.msa_status_string(code).startswith(name)


def test_workspace_size(lib):
    ws = msa.msa_workspace_size(msa.MSA_OP_INDEX_SELECT, 1, 512, 512, 2, 0, 0, 32, 32, 4, msa.MSA_FP32)
    assert ws >= 256 and ws % 256 == 0
    assert msa.msa_workspace_size(msa.MSA_OP_PREFILL, 1, 8192, 8192, 8, 32, 128, 0, 128, 16, msa.MSA_BF16) >= 256
    assert msa.msa_workspace_size(msa.MSA_OP_DECODE, 64, 1, 131072, 8, 32, 128, 0, 128, 16, msa.MSA_BF16) >= 256
    # invalid: negative batch, Hq not a multiple of Hkv, unknown op (an empty batch is valid: 256)
    assert msa.msa_workspace_size(msa.MSA_OP_INDEX_SELECT, -1, 512, 512, 2, 0, 0, 32, 32, 4, 1) == 0
    assert msa.msa_workspace_size(msa.MSA_OP_INDEX_SELECT, 0, 512, 512, 2, 0, 0, 32, 32, 4, 1) == 256
    assert msa.msa_workspace_size(msa.MSA_OP_PREFILL, 1, 64, 64, 3, 8, 64, 0, 32, 4, 1) == 0
    assert msa.msa_workspace_size(7, 1, 64, 64, 2, 8, 64, 32, 32, 4, 1) == 0


def test_index_workspace_holds_the_chunk_table(lib):
    """Tensor-core index path: the top-K for K - 1 <= 15 stays in the kernel
    (status header only); larger K needs the block-max table of one chunk of
    whole 256-row units, rows padded to a multiple of 8 floats, ~4 GiB at most
    unless that leaves fewer than 608 units (four per SM), never more rows
    than the call has."""
    bf16 = msa.MSA_BF16
    idx = msa.MSA_OP_INDEX_SELECT
    assert msa.msa_workspace_size(idx, 1, 131072, 131072, 8, 0, 0, 64, 128, 16, bf16) == 256
    unit = lambda nblk: 256 * ((nblk + 7) // 8 * 8) * 4  # noqa: E731
    # 128K tokens, Bs 32, K 64: 4096 blocks per row, 1024 units of 4 MiB per 4 GiB chunk
    assert msa.msa_workspace_size(idx, 1, 131072, 131072, 8, 0, 0, 64, 32, 64, bf16) == 256 + 1024 * unit(4096)
    # Bs 64, K 32: 2048 units of 2 MiB
    assert msa.msa_workspace_size(idx, 1, 131072, 131072, 8, 0, 0, 64, 64, 32, bf16) == 256 + 2048 * unit(2048)
    # a small call: all of its 40 units (10000 x 1 rows, 313 blocks padded to 320)
    assert msa.msa_workspace_size(idx, 1, 10000, 10000, 1, 0, 0, 32, 32, 20, bf16) == 256 + 40 * unit(313)
    # 1M tokens at Bs 32: 32768 blocks (32 MiB units) -> the four-per-SM floor, 608 units
    ws = msa.msa_workspace_size(idx, 1, 1048576, 1048576, 8, 0, 0, 64, 32, 64, bf16)
    assert ws == 256 + 608 * unit(32768)


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails host validation


def test_host_validation_before_launch(lib):
    P = lambda: FAKE  # noqa: E731
    # null index tensors
    assert lib.msa_index_select(None, P(), None, None, 1, 8, 8, 1, 32, 4, 2, 1, P(), None, P(), 4096, None) == 1
    # unsupported index head dim
    assert lib.msa_index_select(P(), P(), None, None, 1, 8, 8, 1, 48, 4, 2, 1, P(), None, P(), 1 << 20, None) == 2
    # K beyond the built maximum
    assert lib.msa_index_select(P(), P(), None, None, 1, 8, 8, 1, 32, 4, 65, 1, P(), None, P(), 1 << 20, None) == 2
    # workspace too small / misaligned
    assert lib.msa_index_select(P(), P(), None, None, 1, 8, 8, 1, 32, 4, 2, 1, P(), None, P(), 16, None) == 3
    assert lib.msa_index_select(P(), P(), None, None, 1, 8, 8, 1, 32, 4, 2, 1, P(), None,
                                ctypes.c_void_p(0x1010), 1 << 20, None) == 3
    # Hq % Hkv != 0; unsupported head dim; bad dtype
    args = lambda Hq, Hkv, d, dt: (P(), P(), P(), P(), None, None, 1, 8, 8, Hq, Hkv, d, 4, 2, 0.0, dt, P(),  # noqa
                                   None, P(), 1 << 20, None)
    assert lib.msa_sparse_attn_prefill(*args(6, 4, 64, 1)) == 1
    assert lib.msa_sparse_attn_prefill(*args(8, 2, 96, 1)) == 2
    assert lib.msa_sparse_attn_prefill(*args(8, 2, 64, 9)) == 1
    # decode needs kv_len
    assert lib.msa_sparse_attn_decode(P(), P(), P(), P(), None, 1, 8, 8, 2, 64, 4, 2, 0.0, 1, P(), None, P(),
                                      1 << 20, None) == 1
    assert lib.msa_read_status(None, None) == 1
    # forced blocks: only LOCAL or LOCAL|START; START needs K >= 2
    assert lib.msa_index_select_v(P(), P(), None, None, 1, 8, 8, 1, 32, 4, 2, 1, 0, P(), None, P(), 1 << 20, None) == 1
    assert lib.msa_index_select_v(P(), P(), None, None, 1, 8, 8, 1, 32, 4, 2, 1, 2, P(), None, P(), 1 << 20, None) == 1
    assert lib.msa_index_select_v(P(), P(), None, None, 1, 8, 8, 1, 32, 4, 1, 1, 3, P(), None, P(), 1 << 20, None) == 1


def test_kl_and_backward_host_validation(lib):
    P = lambda: FAKE  # noqa: E731
    bf16 = msa.MSA_BF16
    # workspace sizes: supported shapes get one, unsupported ones 0
    assert msa.msa_workspace_size(msa.MSA_OP_KL_AUX, 1, 8192, 8192, 8, 32, 128, 64, 128, 16, bf16) >= 256
    assert msa.msa_workspace_size(msa.MSA_OP_KL_AUX, 1, 8192, 8192, 8, 32, 96, 64, 128, 16, bf16) == 0
    # di is checked as the entry point checks it: (128, 32) is not a built pairing, 0 is no di
    assert msa.msa_workspace_size(msa.MSA_OP_KL_AUX, 1, 8192, 8192, 8, 32, 128, 32, 128, 16, bf16) == 0
    assert msa.msa_workspace_size(msa.MSA_OP_KL_AUX, 1, 8192, 8192, 8, 32, 128, 0, 128, 16, bf16) == 0
    assert msa.msa_workspace_size(msa.MSA_OP_BACKWARD, 1, 8192, 8192, 8, 32, 128, 0, 128, 16, bf16) >= 256
    assert msa.msa_workspace_size(msa.MSA_OP_BACKWARD, 1, 8192, 8192, 2, 32, 128, 0, 128, 16, bf16) == 0  # hpg 16
    assert msa.msa_workspace_size(msa.MSA_OP_BACKWARD, 1, 8192, 8192, 8, 32, 128, 0, 16, 16, bf16) == 0  # Bs 16

    def kl(lse=True, Hq=8, Hkv=2, d=128, di=64, Bs=128, ws_bytes=1 << 30):
        return lib.msa_kl_aux_forward(P(), P(), P(), P(), P(), P() if lse else None, None, None, 1, 8, 8, Hq, Hkv, d,
                                      di, Bs, 2, 0.0, bf16, P(), P(), ws_bytes, None)
    assert kl(lse=False) == 1          # the forward's lse is required
    assert kl(Hq=6, Hkv=4) == 1        # Hq not a multiple of Hkv
    assert kl(d=96) == 2               # head dimension not built
    assert kl(d=128, di=32) == 2       # (d, di) pairing not built
    assert kl(ws_bytes=16) == 3        # workspace too small

    def bwd(dout=True, Hq=8, Hkv=2, d=128, Bs=128, dtype=bf16, ws_bytes=1 << 30):
        return lib.msa_sparse_attn_backward(P(), P(), P(), P(), P() if dout else None, P(), P(), None, None, 1, 8, 8,
                                            Hq, Hkv, d, Bs, 2, 0.0, dtype, P(), P(), P(), P(), ws_bytes, None)
    assert bwd(dout=False) == 1        # the output gradient is required
    assert bwd(Hq=6, Hkv=4) == 1       # Hq not a multiple of Hkv
    assert bwd(d=96) == 2              # head dimension not built
    assert bwd(Bs=16) == 2             # block size not built
    assert bwd(Hq=32, Hkv=2) == 2      # 16 heads per group: beyond the built ratios
    assert bwd(dtype=msa.MSA_FP32) == 2  # bf16 only
    assert bwd(ws_bytes=16) == 3       # workspace too small


def test_empty_batches_on_the_host(lib):
    """B == 0 or Nq == 0: valid, nothing read (NULL pointers), nothing enqueued;
    the other arguments are still checked. Runs without a GPU: no CUDA call is
    made on these paths."""
    bf16 = msa.MSA_BF16
    for op in (msa.MSA_OP_INDEX_SELECT, msa.MSA_OP_PREFILL, msa.MSA_OP_KL_AUX, msa.MSA_OP_BACKWARD):
        assert msa.msa_workspace_size(op, 0, 64, 64, 2, 8, 128, 64, 128, 4, bf16) == 256
        assert msa.msa_workspace_size(op, 2, 0, 64, 2, 8, 128, 64, 128, 4, bf16) == 256
        assert msa.msa_workspace_size(op, -1, 64, 64, 2, 8, 128, 64, 128, 4, bf16) == 0
        assert msa.msa_workspace_size(op, 0, 64, 64, 2, 8, 96, 48, 128, 4, bf16) == 0  # d 96 / di 48 not built
    for op in (msa.MSA_OP_DECODE, msa.MSA_OP_DECODE_STEP):
        assert msa.msa_workspace_size(op, 0, 0, 64, 2, 8, 128, 64, 128, 4, bf16) == 256
    N = None
    # index selection: empty batch, empty rows; unsupported di and bad force still fail
    assert lib.msa_index_select(N, N, N, N, 0, 8, 8, 1, 32, 4, 2, 1, N, N, N, 0, N) == 0
    assert lib.msa_index_select(N, N, N, N, 3, 0, 8, 1, 32, 4, 2, 1, N, N, N, 0, N) == 0
    assert lib.msa_index_select(N, N, N, N, 0, 8, 8, 1, 48, 4, 2, 1, N, N, N, 0, N) == 2
    assert lib.msa_index_select(N, N, N, N, -1, 8, 8, 1, 32, 4, 2, 1, N, N, N, 0, N) == 1
    assert lib.msa_index_select_v(N, N, N, N, 0, 8, 8, 1, 32, 4, 1, 1, 3, N, N, N, 0, N) == 1  # START needs K >= 2
    assert lib.msa_index_select_noalloc(N, N, N, N, 0, 8, 8, 1, 32, 4, 2, 1, N, N, N) == 0
    assert lib.msa_index_select_noalloc(N, N, N, N, 0, 8, 8, 1, 48, 4, 2, 1, N, N, N) == 2
    # attention
    assert lib.msa_sparse_attn_prefill(N, N, N, N, N, N, 0, 8, 8, 8, 2, 64, 4, 2, 0.0, 1, N, N, N, 0, N) == 0
    assert lib.msa_sparse_attn_prefill(N, N, N, N, N, N, 2, 0, 8, 8, 2, 64, 4, 2, 0.0, 1, N, N, N, 0, N) == 0
    assert lib.msa_sparse_attn_prefill(N, N, N, N, N, N, 0, 8, 8, 6, 4, 64, 4, 2, 0.0, 1, N, N, N, 0, N) == 1
    assert lib.msa_sparse_attn_prefill(N, N, N, N, N, N, 0, 8, 8, 8, 2, 96, 4, 2, 0.0, 1, N, N, N, 0, N) == 2
    assert lib.msa_sparse_attn_decode(N, N, N, N, N, 0, 8, 8, 2, 64, 4, 2, 0.0, 1, N, N, N, 0, N) == 0
    assert lib.msa_decode_step(N, N, N, N, N, N, N, N, N, 0, 64, 8, 2, 64, 32, 16, 2, 0.0, 1, N, N, N, N, 0,
                               N) == 0
    # KL and backward (B == 0: nothing at all to write)
    assert lib.msa_kl_aux_forward(N, N, N, N, N, N, N, N, 0, 8, 8, 8, 2, 128, 64, 128, 2, 0.0, bf16, N, N, 0,
                                  N) == 0
    assert lib.msa_kl_aux_forward(N, N, N, N, N, N, N, N, 2, 0, 8, 8, 2, 128, 64, 128, 2, 0.0, bf16, N, N, 0,
                                  N) == 0
    assert lib.msa_kl_aux_forward(N, N, N, N, N, N, N, N, 0, 8, 8, 8, 2, 96, 64, 128, 2, 0.0, bf16, N, N, 0,
                                  N) == 2
    bwd = lambda B, Nq, Nk, d=128, dtype=bf16: lib.msa_sparse_attn_backward(  # noqa: E731
        N, N, N, N, N, N, N, N, N, B, Nq, Nk, 8, 2, d, 128, 2, 0.0, dtype, N, N, N, N, 0, N)
    assert bwd(0, 8, 8) == 0
    assert bwd(2, 0, 0) == 0
    assert bwd(2, 0, 8) == 1            # keys but no queries: dk and dv are zero-filled, so they must be given
    assert bwd(0, 8, 8, d=96) == 2
    assert bwd(0, 8, 8, dtype=msa.MSA_FP32) == 2
