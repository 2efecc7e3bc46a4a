"""The synthetic workloads: shapes, value ranges and skew of the MSA settings.

Block 128 with 16 selected blocks (2048 attended tokens), block sizes 32/64/128
at a fixed 2048-token budget, contexts up to 1M tokens, batched single-token
decode over ragged KV lengths. Every value distribution is in ``synth``.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int          # sequences
    Nq: int         # query rows per sequence
    Nk: int         # key rows per sequence (cache capacity for decode)
    Hq: int         # query heads
    Hkv: int        # key/value heads = GQA groups G
    d: int          # head dim
    di: int         # index head dim
    Bs: int         # key block size
    K: int          # selected blocks per (query, group), local block included
    dtype: str      # "fp32" | "bf16"
    idx_a: int      # index q/k integers uniform in [-idx_a, idx_a]
    hot: str = "none"   # "none" | "first4" | "pct1": blocks whose index key is scaled
    hot_mult: int = 3
    kv_len_range: tuple | None = None   # decode: per-sequence KV length range (inclusive)
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hkv

    @property
    def decode(self) -> bool:
        return self.kv_len_range is not None

    @property
    def nblk(self) -> int:
        return (self.Nk + self.Bs - 1) // self.Bs


def shapes(w: Workload) -> dict:
    return {
        "q": (w.B, w.Nq, w.Hq, w.d),
        "k": (w.B, w.Nk, w.Hkv, w.d),
        "v": (w.B, w.Nk, w.Hkv, w.d),
        "iq": (w.B, w.Nq, w.G, w.di),
        "ik": (w.B, w.Nk, w.di),
    }


_P = dict(Hq=32, Hkv=8, d=128, di=64, dtype="bf16", idx_a=8)

WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, Nq=512, Nk=512, Hq=8, Hkv=2, d=64, di=32, Bs=32, K=4,
                          dtype="fp32", idx_a=4),
    "prefill_8k": Workload("prefill_8k", B=1, Nq=8192, Nk=8192, Bs=128, K=16, **_P),
    # a 32K-token prefill: inputs well above the L2 size, a few GB on the device (profiling captures)
    "prefill_32k": Workload("prefill_32k", B=1, Nq=32768, Nk=32768, Bs=128, K=16, hot="first4", **_P),
    "prefill_128k_bs128": Workload("prefill_128k_bs128", B=1, Nq=131072, Nk=131072, Bs=128, K=16,
                                   hot="first4", **_P),
    "prefill_128k_bs64": Workload("prefill_128k_bs64", B=1, Nq=131072, Nk=131072, Bs=64, K=32,
                                  hot="first4", **_P),
    "prefill_128k_bs32": Workload("prefill_128k_bs32", B=1, Nq=131072, Nk=131072, Bs=32, K=64,
                                  hot="first4", **_P),
    "decode_b64": Workload("decode_b64", B=64, Nq=1, Nk=131072, Bs=128, K=16,
                           kv_len_range=(32768, 131072), **_P),
    # a reduced decode batch (caches of 32K, ~4 GB on the device) for profiling captures
    "decode_b32_32k": Workload("decode_b32_32k", B=32, Nq=1, Nk=32768, Bs=128, K=16,
                               kv_len_range=(8192, 32768), **_P),
    "prefill_1m": Workload("prefill_1m", B=1, Nq=1048576, Nk=1048576, Bs=128, K=16, hot="pct1", **_P),
}


def scaled(w: Workload, **kw) -> Workload:
    """A variant of a workload with some fields changed (smaller parity cases)."""
    return replace(w, **kw)
