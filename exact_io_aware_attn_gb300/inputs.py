"""Seeded synthetic inputs and the workload table.

This module holds no attention arithmetic: it only draws Q, K and V from a
seeded generator and names the workloads. Both the GPU path (tests, bench)
and the oracle's callers use it, so the two sides see the very same 16-bit
tensors.

Recipe: torch.Generator("cpu").manual_seed(seed); torch.randn in float32 for
q, then k, then v, each of shape [B, h, T, d]; multiplied by `mult`
(0.5 for the very-long workload, 1 elsewhere); then cast to the 16-bit
dtype (round to nearest even). The shapes, dtypes and masks follow the
pages' GPT-2 head geometry (12 heads of width 64, "Attention and Its
Computational Cost", section "What the numbers do not show") and the
sequence lengths they measure (up to 16,384 tokens).
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

F16 = 0
BF16 = 1

_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}
_NAME = {F16: "f16", BF16: "bf16"}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    h: int
    T_q: int
    T_kv: int
    d: int
    dtype: int          # F16 or BF16
    causal: bool
    mult: float = 1.0
    seed: int = 0
    h_kv: int = 0        # key/value heads (grouped-query attention); 0 = h

    @property
    def torch_dtype(self):
        return _TORCH_DTYPE[self.dtype]

    @property
    def dtype_name(self) -> str:
        return _NAME[self.dtype]

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    @property
    def kv_heads(self) -> int:
        return self.h_kv or self.h

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "h": self.h, "h_kv": self.kv_heads,
                "T_q": self.T_q, "T_kv": self.T_kv, "d": self.d,
                "dtype": self.dtype_name, "causal": self.causal,
                "input_scale": self.mult, "seed": self.seed}


# The five workloads (seven runs) the kernels are checked and measured on.
TINY = Workload("tiny_noncausal_B1_h2_T256_d64_f16", 1, 2, 256, 256, 64, F16, False)
GPT2_PREFILL = Workload("gpt2_causal_prefill_B8_h12_T1024_d64_bf16", 8, 12, 1024, 1024, 64, BF16, True)
LONG_4K = Workload("long_causal_prefill_B1_h16_T4096_d64_bf16", 1, 16, 4096, 4096, 64, BF16, True)
LONG_8K = Workload("long_causal_prefill_B1_h16_T8192_d64_bf16", 1, 16, 8192, 8192, 64, BF16, True)
LONG_8K_D128 = Workload("long_causal_prefill_B1_h16_T8192_d128_bf16", 1, 16, 8192, 8192, 128, BF16, True)
VERY_LONG = Workload("very_long_causal_prefill_B1_h12_T16384_d64_f16_x0.5", 1, 12, 16384, 16384, 64, F16, True, mult=0.5)
DECODE = Workload("decode_B32_h12_Tkv16384_d64_bf16", 32, 12, 1, 16384, 64, BF16, False)

WORKLOADS = [TINY, GPT2_PREFILL, LONG_4K, LONG_8K, LONG_8K_D128, VERY_LONG, DECODE]

# Grouped-query decode (a widening beyond the five workloads above): 32 query
# heads share 8 key/value heads, the geometry of common grouped-query models.
DECODE_GQA = Workload("decode_gqa_B32_hq32_hkv8_Tkv16384_d128_bf16", 32, 32, 1, 16384, 128, BF16,
                      False, h_kv=8)
# Chunked prefill (also beyond the five): 256 new query rows of one sequence
# against a 16K-token causal context, the shape where one CTA per query-tile
# pair leaves most SMs idle and the key range is split.
CHUNKED_PREFILL = Workload("chunked_prefill_B1_h8_Tq256_Tkv16384_d128_bf16", 1, 8, 256, 16384, 128,
                           BF16, True)
# The same grouped-query decode at d = 64 (half the bytes per key row).
DECODE_GQA_D64 = Workload("decode_gqa_B32_hq32_hkv8_Tkv16384_d64_bf16", 32, 32, 1, 16384, 64, BF16,
                          False, h_kv=8)
EXTRA_WORKLOADS = [DECODE_GQA, DECODE_GQA_D64, CHUNKED_PREFILL]


def make_qkv(B, h, T_q, T_kv, d, dtype=BF16, mult=1.0, seed=0, device="cpu", h_kv=None):
    """Draw q [B,h,T_q,d], k and v [B,h_kv,T_kv,d] (h_kv defaults to h) as
    16-bit tensors.

    The draw happens on the CPU generator (so every machine gets the same
    values) and the result is then moved to `device`.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    out = []
    hk = h if h_kv is None else h_kv
    for heads, t in ((h, T_q), (hk, T_kv), (hk, T_kv)):
        x = torch.randn((B, heads, t, d), generator=gen, dtype=torch.float32)
        if mult != 1.0:
            x.mul_(mult)
        out.append(x.to(_TORCH_DTYPE[dtype]).to(device))
    return tuple(out)


def make_workload(w: Workload, device="cpu"):
    return make_qkv(w.B, w.h, w.T_q, w.T_kv, w.d, w.dtype, w.mult, w.seed, device, w.kv_heads)


def make_dout(B, h, T_q, d, dtype=BF16, seed=0, device="cpu"):
    """The incoming gradient dO [B, h, T_q, d] for backward tests and
    benchmarks: N(0,1) in float32 from its own seeded CPU generator (seed +
    1000003, so it is independent of q, k, v drawn with `seed`), cast to the
    16-bit dtype."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 1000003)
    x = torch.randn((B, h, T_q, d), generator=gen, dtype=torch.float32)
    return x.to(_TORCH_DTYPE[dtype]).to(device)
