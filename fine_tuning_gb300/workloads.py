"""Seeded synthetic workloads for the fused per-token layer ops.

This module only draws numbers: the five workload shapes, packed sequence
lengths and the random tensors.  It holds none of the arithmetic of RMSNorm,
SwiGLU or RoPE, so the CUDA path and the CPU oracle can both be fed from it
without sharing any of the method.

Recipe (the pages print no dataset records; these draws stand in for them):

* sequence lengths come from ``numpy.random.default_rng(seed)`` (PCG64),
  drawn until their running sum reaches T, the last one cut so that the
  lengths sum to exactly T; ``cu_seqlens`` is their int32 prefix sum;
* every tensor is drawn from its own ``torch.Generator`` seeded with
  ``seed * 1000 + k`` (k = the tensor's slot in ``TENSOR_SLOTS``), as fp32
  N(0, 1) on the target device, then rounded to the storage dtype with
  round-to-nearest-even; RMSNorm weights are ``1 + 0.1 * N(0, 1)``.

The shapes follow the packed fine-tuning runs the pages describe: Qwen2.5-0.5B
on one GPU (Chronicals abstract), Llama-3.2-1B / Qwen3-8B / Qwen3-32B layer
shapes with short/long sequence mixes (Unsloth packing news items), and a
single 524,288-token sequence for the 500k-context 64-bit indexing case
(Unsloth auto-packing article, paragraph on ``LONG_INDEXING``).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence

import numpy as np
import torch

TENSOR_SLOTS = ("x", "w", "dy", "g", "u", "dh", "q", "k", "dq", "dk", "res", "dres", "wq",
                "wk")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str               # "f32" or "bf16": storage dtype
    seed: int
    T: int                   # packed tokens
    lengths: Optional[tuple]  # fixed lengths, or None to draw them
    length_mix: tuple        # ((prob, lo, hi), ...) uniform mixes or ("lognormal", mu, sigma, lo, hi)
    H: int                   # RMSNorm hidden size
    eps: float
    I: int                   # SwiGLU intermediate size
    T_swiglu: int            # tokens SwiGLU runs on
    Hq: int
    Hkv: int
    D: int
    theta: float

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS: Dict[str, Workload] = {
    # tiny fp32 case: four sequences {5, 17, 32, 10}
    "tiny_f32": Workload("tiny_f32", "f32", 0, 64, (5, 17, 32, 10), (),
                         64, 1e-6, 176, 64, 4, 2, 16, 1e4),
    # Qwen2.5-0.5B layer shapes, lognormal(5, 1) lengths clipped to [16, 2048]
    "qwen2.5-0.5b": Workload("qwen2.5-0.5b", "bf16", 1, 16384, None,
                             ("lognormal", 5.0, 1.0, 16, 2048),
                             896, 1e-6, 4864, 16384, 14, 2, 64, 1e6),
    # Llama-3.2-1B layer shapes, half short U[16,256], half long U[1024,4096]
    "llama-3.2-1b": Workload("llama-3.2-1b", "bf16", 2, 32768, None,
                             ((0.5, 16, 256), (0.5, 1024, 4096)),
                             2048, 1e-5, 8192, 32768, 32, 8, 64, 5e5),
    # Qwen3-8B layer shapes, 80% short U[16,256], 20% long U[2048,8192]
    "qwen3-8b": Workload("qwen3-8b", "bf16", 3, 65536, None,
                         ((0.8, 16, 256), (0.2, 2048, 8192)),
                         4096, 1e-6, 12288, 65536, 32, 8, 128, 1e6),
    # Qwen3-32B layer shapes on one 524,288-token sequence; SwiGLU on a
    # 65,536-token slice
    "qwen3-32b-524k": Workload("qwen3-32b-524k", "bf16", 4, 524288, (524288,), (),
                               5120, 1e-6, 25600, 65536, 64, 8, 128, 1e6),
}

WORKLOAD_ORDER = ("tiny_f32", "qwen2.5-0.5b", "llama-3.2-1b", "qwen3-8b", "qwen3-32b-524k")


def draw_lengths(wl: Workload) -> np.ndarray:
    """Sequence lengths of one packed batch, summing to exactly ``wl.T``."""
    if wl.lengths is not None:
        lens = np.asarray(wl.lengths, dtype=np.int64)
        assert int(lens.sum()) == wl.T
        return lens
    rng = np.random.default_rng(wl.seed)
    out = []
    total = 0
    while total < wl.T:
        if wl.length_mix[0] == "lognormal":
            _, mu, sigma, lo, hi = wl.length_mix
            n = int(np.clip(np.rint(rng.lognormal(mu, sigma)), lo, hi))
        else:
            r = rng.random()
            acc = 0.0
            for prob, lo, hi in wl.length_mix:
                acc += prob
                if r < acc:
                    break
            n = int(rng.integers(lo, hi, endpoint=True))
        n = min(n, wl.T - total)
        out.append(n)
        total += n
    return np.asarray(out, dtype=np.int64)


def cu_seqlens_from_lengths(lengths: Sequence[int]) -> np.ndarray:
    """int32 boundaries [0, l0, l0+l1, ...] of a packed batch."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    assert cu[-1] < 2**31
    return cu.astype(np.int32)


def tensor_seed(wl: Workload, slot: str) -> int:
    return wl.seed * 1000 + TENSOR_SLOTS.index(slot)


def draw(wl: Workload, slot: str, shape, device="cpu", dtype=None,
         mean: float = 0.0, std: float = 1.0) -> torch.Tensor:
    """One seeded N(mean, std^2) tensor, rounded to the storage dtype."""
    dtype = dtype or wl.torch_dtype
    gen = torch.Generator(device=device)
    gen.manual_seed(tensor_seed(wl, slot))
    t = torch.empty(tuple(shape), dtype=torch.float32, device=device)
    t.normal_(mean=mean, std=std, generator=gen)
    return t.to(dtype)


def rmsnorm_inputs(wl: Workload, device="cpu", T: Optional[int] = None):
    T = wl.T if T is None else T
    return {
        "x": draw(wl, "x", (T, wl.H), device),
        "w": draw(wl, "w", (wl.H,), device, mean=1.0, std=0.1),
        "dy": draw(wl, "dy", (T, wl.H), device),
    }


def rmsnorm_add_inputs(wl: Workload, device="cpu", T: Optional[int] = None):
    """Inputs of the norm with the residual add in front: x (the sublayer's
    output, N(0, 1)), the residual stream res (N(0, 2^2), larger than one
    sublayer's contribution), w, dy, and dh, the gradient the residual stream
    carries back into h (N(0, 1))."""
    T = wl.T if T is None else T
    d = rmsnorm_inputs(wl, device, T)
    d["res"] = draw(wl, "res", (T, wl.H), device, std=2.0)
    d["dh"] = draw(wl, "dres", (T, wl.H), device)
    return d


def qk_norm_rope_inputs(wl: Workload, device="cpu", T: Optional[int] = None):
    """q, k, dq, dk as for RoPE plus the per-head norm weights wq, wk
    (1 + 0.1 N(0,1), D each)."""
    d = rope_inputs(wl, device, T)
    d["wq"] = draw(wl, "wq", (wl.D,), device, mean=1.0, std=0.1)
    d["wk"] = draw(wl, "wk", (wl.D,), device, mean=1.0, std=0.1)
    return d


def swiglu_inputs(wl: Workload, device="cpu", T: Optional[int] = None):
    T = wl.T_swiglu if T is None else T
    return {
        "g": draw(wl, "g", (T, wl.I), device),
        "u": draw(wl, "u", (T, wl.I), device),
        "dh": draw(wl, "dh", (T, wl.I), device),
    }


def rope_inputs(wl: Workload, device="cpu", T: Optional[int] = None):
    T = wl.T if T is None else T
    return {
        "q": draw(wl, "q", (T, wl.Hq, wl.D), device),
        "k": draw(wl, "k", (T, wl.Hkv, wl.D), device),
        "dq": draw(wl, "dq", (T, wl.Hq, wl.D), device),
        "dk": draw(wl, "dk", (T, wl.Hkv, wl.D), device),
    }


def ideal_bytes(wl: Workload) -> Dict[str, int]:
    """Algorithmic minimum HBM bytes of one call of each op: every input read
    once, every output written once (storage dtype; rstd and dw in fp32)."""
    e = wl.elem_bytes
    T, H, I, Ts = wl.T, wl.H, wl.I, wl.T_swiglu
    rope = 2 * e * T * (wl.Hq + wl.Hkv) * wl.D
    return {
        "rmsnorm_fwd": 2 * e * T * H + 4 * T + e * H,
        "rmsnorm_bwd": 3 * e * T * H + 4 * T + e * H + 4 * H,
        "swiglu_fwd": 3 * e * Ts * I,
        "swiglu_bwd": 5 * e * Ts * I,
        "qk_rope_fwd": rope,
        "qk_rope_bwd": rope,
        # the residual-add variant of the norm: x and res in, h and y out;
        # backward: dy, dh and h in, dx out
        "rmsnorm_add_fwd": 4 * e * T * H + 4 * T + e * H,
        "rmsnorm_add_bwd": 4 * e * T * H + 4 * T + e * H + 4 * H,
        # SwiGLU backward that re-emits h: dh, g, u in; dg, du, h out
        "swiglu_bwd_h": 6 * e * Ts * I,
        # RoPE with a caller's (llama3-scaled) frequency table: same bytes
        "qk_rope_freq_fwd": rope,
        # per-head QK-RMSNorm fused into RoPE: q, k in, out written, r per
        # (token, head) saved; backward: output grads and pre-norm q, k in,
        # grads out, r read
        "qk_norm_rope_fwd": rope + 4 * T * (wl.Hq + wl.Hkv) + 2 * e * wl.D,
        "qk_norm_rope_bwd": 3 * rope // 2 + 4 * T * (wl.Hq + wl.Hkv) + 2 * e * wl.D + 8 * wl.D,
    }


def tokens_per_call(wl: Workload) -> Dict[str, int]:
    return {
        "rmsnorm_fwd": wl.T, "rmsnorm_bwd": wl.T,
        "swiglu_fwd": wl.T_swiglu, "swiglu_bwd": wl.T_swiglu,
        "qk_rope_fwd": wl.T, "qk_rope_bwd": wl.T,
        "rmsnorm_add_fwd": wl.T, "rmsnorm_add_bwd": wl.T, "swiglu_bwd_h": wl.T_swiglu,
        "qk_rope_freq_fwd": wl.T, "qk_norm_rope_fwd": wl.T, "qk_norm_rope_bwd": wl.T,
    }


# ------------------------------------------------------------ LM-head loss

@dataclasses.dataclass(frozen=True)
class HeadWorkload:
    """The cross-entropy of an LM head: T tokens of hidden size H against a
    vocabulary of V rows.  h ~ N(0, 1); W ~ N(0, w_std^2) (w_std 0.02, the
    usual LM-head initialisation, keeps the logits near N(0, 0.6^2) at
    H = 896); targets uniform over the vocabulary, a share of them ignored
    (y = -100) as padding would be."""
    name: str
    T: int
    H: int
    V: int
    seed: int
    w_std: float = 0.02
    ignored: float = 0.05


HEAD_WORKLOADS = {w.name: w for w in (
    HeadWorkload("tiny-head", T=300, H=64, V=1000, seed=11, w_std=0.125),
    # Qwen2.5-0.5B's head (hidden 896, vocabulary 151,936) on 8,192 tokens:
    # the run whose fp32 logits the page puts at 5 GB
    HeadWorkload("qwen2.5-0.5b-head", T=8192, H=896, V=151936, seed=12),
)}


def head_inputs(hw: HeadWorkload, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(hw.seed * 1000 + 1)
    h = torch.randn((hw.T, hw.H), generator=g, device=device).to(torch.bfloat16)
    W = (hw.w_std * torch.randn((hw.V, hw.H), generator=g, device=device)).to(torch.bfloat16)
    y = torch.randint(0, hw.V, (hw.T,), generator=g, device=device, dtype=torch.int64)
    drop = torch.rand((hw.T,), generator=g, device=device) < hw.ignored
    y = torch.where(drop, torch.full_like(y, -100), y).to(torch.int32)
    return {"h": h, "W": W, "y": y}

