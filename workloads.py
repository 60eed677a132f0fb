"""Seeded synthetic attention workloads.

This module only draws random inputs and describes shapes. It holds none of
the attention arithmetic, so both the fp64 oracle's tests and the CUDA path's
tests and benchmark can take their inputs from here without sharing any of
the method's code.

The five workloads follow the shapes the FlashAttention explainer pages
measure or discuss: a one-head 256-token check ("What is FlashAttention?",
"Worked example"), the 8,192-token, 32-head, d=128 layer ("What is
FlashAttention?", Step 1; "FlashAttention", byte-accounting panel), and the
32,768-token long context of the same panel. Values are N(0, 1) drawn from a
CPU `torch.Generator`, so every host produces bit-identical tensors.

Recipe (per workload index k):
  * Q, K, V, dO ~ N(0, 1) in fp32 from seeds 1000+k, 2000+k, 3000+k, 4000+k,
    then cast to the workload's dtype (round to nearest even for bf16).
  * The large-magnitude workload multiplies Q and K by sqrt(30) in fp32
    before the cast, so the raw dot products reach about +-90 (30 times the
    unit-variance scale), the magnitude at which an unshifted fp32 exp
    overflows ("FlashAttention", "Why it is allowed to be exact").
  * Its additive mask is bf16 [B, 1, N, N]: 0 everywhere except round(0.01 N)
    query rows per batch, chosen by `randperm` from seed 5000+k, which are -inf
    in every column (fully masked rows).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "bf16", "f16", "f32" or "e4m3"
    causal: bool
    mask: bool
    backward: bool
    qk_mult: float = 1.0
    masked_row_frac: float = 0.0

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "f16": torch.float16}.get(self.dtype, torch.float32)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "B": self.B,
            "H": self.H,
            "N": self.N,
            "d": self.d,
            "dtype": self.dtype,
            "causal": self.causal,
            "mask": self.mask,
            "backward": self.backward,
        }


# The benchmark workload with IEEE half storage (an extension beyond the five
# configurations: same shape, values and flags).
F16_WORKLOADS: Dict[int, Workload] = {}

WORKLOADS: Dict[int, Workload] = {
    1: Workload(1, "one_head_n256_d64_f32_fwd", 1, 1, 256, 64, "f32", False, False, False),
    2: Workload(2, "b4_h16_n2048_d64_bf16_causal_fwd_bwd", 4, 16, 2048, 64, "bf16", True, False, True),
    3: Workload(3, "b1_h32_n8192_d128_bf16_fwd", 1, 32, 8192, 128, "bf16", False, False, False),
    4: Workload(4, "b2_h32_n8192_d128_bf16_causal_mask_x30_fwd_bwd", 2, 32, 8192, 128, "bf16", True, True,
                True, qk_mult=math.sqrt(30.0), masked_row_frac=0.01),
    5: Workload(5, "b1_h16_n32768_d128_bf16_causal_fwd_bwd", 1, 16, 32768, 128, "bf16", True, False, True),
}


F16_WORKLOADS[6] = dataclasses.replace(WORKLOADS[2], index=6, name="b4_h16_n2048_d64_f16_causal_fwd_bwd", dtype="f16")

# Head dim 256 (FlashAttention-2 covers head dims up to 256: "What is FlashAttention?",
# "Trade-offs and edge cases"), forward and backward: the 8,192-token layer shape with half the
# heads, so the FLOPs equal the d = 128 layer's.
D256_WORKLOADS: Dict[int, Workload] = {
    7: Workload(7, "b1_h16_n8192_d256_bf16_fwd_bwd", 1, 16, 8192, 256, "bf16", False, False, True),
    8: Workload(8, "b1_h16_n8192_d256_bf16_causal_fwd_bwd", 1, 16, 8192, 256, "bf16", True, False, True),
}


def with_dtype(w: Workload, dtype: str) -> Workload:
    """The same workload (shape, seeds, flags) stored in another dtype."""
    return dataclasses.replace(w, dtype=dtype)


def _normal(shape, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32)


def masked_rows(w: Workload, b: int) -> torch.Tensor:
    """The query rows of batch b that the additive mask blanks entirely."""
    count = int(round(w.masked_row_frac * w.N))
    g = torch.Generator(device="cpu")
    g.manual_seed(5000 + w.index + 7919 * b)
    return torch.randperm(w.N, generator=g)[:count].sort().values


def make_mask(w: Workload) -> Optional[torch.Tensor]:
    if not w.mask:
        return None
    m = torch.zeros(w.B, 1, w.N, w.N, dtype=w.torch_dtype)
    for b in range(w.B):
        m[b, 0, masked_rows(w, b), :] = float("-inf")
    return m


def make_inputs(w: Workload, with_grad: Optional[bool] = None, shape=None) -> Dict[str, torch.Tensor]:
    """CPU tensors q, k, v (and do, mask when the workload has them).

    `shape` overrides (B, H, N, d) for reduced-size parity cases that keep
    the workload's value distribution and flags.
    """
    B, H, N, d = shape if shape is not None else (w.B, w.H, w.N, w.d)
    k_ = w.index
    out = {}
    q = _normal((B, H, N, d), 1000 + k_)
    kk = _normal((B, H, N, d), 2000 + k_)
    if w.qk_mult != 1.0:
        q = q * w.qk_mult
        kk = kk * w.qk_mult
    out["q"] = q.to(w.torch_dtype)
    out["k"] = kk.to(w.torch_dtype)
    out["v"] = _normal((B, H, N, d), 3000 + k_).to(w.torch_dtype)
    if with_grad is None:
        with_grad = w.backward
    if with_grad:
        out["do"] = _normal((B, H, N, d), 4000 + k_).to(w.torch_dtype)
    if w.mask:
        ws = dataclasses.replace(w, B=B, N=N)
        out["mask"] = make_mask(ws)
    return out


# FP8 forward (E4M3 inputs, "What is FlashAttention?", FAQ on FlashAttention-3): the
# d = 128 layer shape and the long causal context, forward only.
FP8_WORKLOADS: Dict[int, Workload] = {
    9: Workload(9, "b1_h32_n8192_d128_e4m3_fwd", 1, 32, 8192, 128, "e4m3", False, False, False),
    10: Workload(10, "b1_h16_n32768_d128_e4m3_causal_fwd", 1, 16, 32768, 128, "e4m3", True, False, False),
    11: Workload(11, "b1_h16_n8192_d256_e4m3_fwd", 1, 16, 8192, 256, "e4m3", False, False, False),
}


# Smaller cases of the d = 128 kernels for profiler captures that replay each launch many
# times: inputs still larger than L2, a few GB on the device at most. The same seeds and
# flags as the configuration named after them (indices 12, 13 reuse 5's and 4's draws'
# recipe with their own seeds).
PROFILE_WORKLOADS: Dict[int, Workload] = {
    12: Workload(12, "b1_h32_n8192_d128_bf16_causal_fwd_bwd", 1, 32, 8192, 128, "bf16", True, False, True),
    13: Workload(13, "b1_h32_n8192_d128_bf16_causal_mask_x30_fwd_bwd", 1, 32, 8192, 128, "bf16", True, True,
                 True, qk_mult=math.sqrt(30.0), masked_row_frac=0.01),
}


def quantize_e4m3(x: torch.Tensor):
    """fp32 tensor -> (E4M3 codes as uint8, descale) with one per-tensor factor,
    descale = max|x| / 448 (448 is E4M3's largest finite value), so code x descale
    approximates x. Rounding is torch's float8_e4m3fn conversion."""
    amax = float(x.abs().max()) if x.numel() else 1.0
    # an fp32 value, as the library takes it
    descale = float(torch.tensor(amax / 448.0 if amax > 0 else 1.0, dtype=torch.float32))
    codes = (x / descale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, descale


def make_fp8_inputs(w: Workload, shape=None) -> Dict[str, object]:
    """E4M3 codes q8, k8, v8 (uint8, CPU) and their descales q_ds, k_ds, v_ds, from the same
    N(0, 1) draws (seeds 1000+k, 2000+k, 3000+k) as make_inputs."""
    B, H, N, d = shape if shape is not None else (w.B, w.H, w.N, w.d)
    out: Dict[str, object] = {}
    for name, seed in (("q", 1000), ("k", 2000), ("v", 3000)):
        x = _normal((B, H, N, d), seed + w.index)
        if name in ("q", "k") and w.qk_mult != 1.0:
            x = x * w.qk_mult
        out[name + "8"], out[name + "_ds"] = quantize_e4m3(x)
    if w.mask:
        out["mask"] = make_mask(dataclasses.replace(w, B=B, N=N, dtype="bf16"))
    return out


def random_tensor(shape, seed: int, dtype=torch.float32, mult: float = 1.0) -> torch.Tensor:
    """A seeded N(0, mult^2) tensor for ad-hoc parity and edge cases."""
    t = _normal(shape, seed)
    if mult != 1.0:
        t = t * mult
    return t.to(dtype)


def attention_flops(B: int, H: int, N: int, d: int, causal: bool, backward: bool = False) -> float:
    """Useful attention FLOPs: 4 N^2 d per head forward, 2.5x that backward,
    halved for causal ("FlashAttention", "Checking it on a real system")."""
    f = 4.0 * B * H * N * N * d
    if causal:
        f *= 0.5
    if backward:
        f *= 2.5
    return f
