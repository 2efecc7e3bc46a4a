"""MSA (MiniMax Sparse Attention) hot path on GB300: Python binding.

Argument marshalling over the C ABI of ``libmsa.so`` (declared in
``include/msa.h``); every step of the path runs in the library's CUDA kernels.
PyTorch only provides device memory and the current stream. The functions
carry the C names:

    msa_workspace_size, msa_index_select, msa_index_select_v,
    msa_sparse_attn_prefill, msa_sparse_attn_decode, msa_decode_step,
    msa_kl_aux_forward, msa_sparse_attn_backward, msa_read_status,
    msa_status_string

There is no CPU fallback: if ``libmsa.so`` is missing or was not built for
this GPU, every call raises.
"""
from ._lib import (  # noqa: F401
    MSA_BF16,
    MSA_FORCE_LOCAL,
    MSA_FORCE_START,
    MSA_FP32,
    MSA_OP_BACKWARD,
    MSA_OP_DECODE,
    MSA_OP_DECODE_STEP,
    MSA_OP_INDEX_SELECT,
    MSA_OP_KL_AUX,
    MSA_OP_PREFILL,
    MsaError,
    lib_path,
    load_library,
    msa_debug_inject_timeout,
    msa_index_select,
    msa_index_select_noalloc,
    msa_index_select_v,
    msa_kl_aux_forward,
    msa_profile_begin,
    msa_profile_end,
    msa_decode_step,
    msa_read_status,
    msa_sparse_attn_backward,
    msa_sparse_attn_decode,
    msa_sparse_attn_prefill,
    msa_status_string,
    msa_workspace_size,
    workspace,
)


def build(verbose: bool = False) -> str:
    from ._build import build as _b

    return _b(verbose=verbose)
