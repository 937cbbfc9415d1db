"""Seeded synthetic workloads for Longformer-style band attention.

This module only describes shapes and attention patterns and draws seeded
random inputs.  It holds none of the attention arithmetic, so both the CUDA
library's callers and the fp64 oracle's callers can share it.

The pages this follows (velog.io/@lainshower/Longformer) train and evaluate
on text8/enwik8 character LM (section 4.2), QA / classification with global
tokens (section 3-1, Global Attention) and arXiv summarisation with a 16K
encoder (section 7).  Those datasets are not used: i.i.d. N(0, 1) activations
of the same shapes stand in for the projected Q/K/V of those models.

Draw recipe: one ``torch.Generator`` seeded with ``seed`` draws, in order,
q, k, v and then (when the pattern has global tokens) qg, kg, vg, each with
``torch.randn(shape, dtype=float32)``, then casts to the workload dtype.  The
valid lengths of the padded QA pattern come from a separate CPU generator
seeded 1 (``torch.randint(2048, 4097, (B,))``).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple, Union

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, window pattern and element type."""

    name: str
    dtype: str  # "bf16" or "f32"
    B: int
    H: int
    n: int
    d: int
    w: Union[int, Tuple[int, ...]]  # total window, or one per head; w/2 keys on each side (look-back only if causal)
    dilation: Tuple[int, ...]  # one entry per head
    causal: bool = False
    global_idx: Tuple[int, ...] = ()
    pad_len: Optional[Tuple[int, ...]] = None  # trailing pad count per batch row
    seed: int = 0

    @property
    def G(self) -> int:
        return len(self.global_idx)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "f32": torch.float32}[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def valid_len(self, b: int) -> int:
        return self.n - (self.pad_len[b] if self.pad_len else 0)

    def tokens(self) -> int:
        """Valid (non-padding) tokens over the batch (all heads share them)."""
        return sum(self.valid_len(b) for b in range(self.B))

    def describe(self) -> Dict[str, object]:
        return {
            "workload": self.name,
            "dtype": self.dtype,
            "B": self.B,
            "H": self.H,
            "n": self.n,
            "d": self.d,
            "w": self.w,
            "dilation": list(self.dilation),
            "causal": self.causal,
            "n_global": self.G,
            "padded": self.pad_len is not None,
        }


def _qa_pad_len(B: int, n: int) -> Tuple[int, ...]:
    g = torch.Generator(device="cpu").manual_seed(1)
    valid = torch.randint(2048, 4097, (B,), generator=g)
    return tuple(int(n - x) for x in valid.tolist())


def fp32_window64() -> Workload:
    """fp32 sliding window: B1 H1 n512 d64, w=64 (+-32), no globals."""
    return Workload("fp32_window64_n512", "f32", 1, 1, 512, 64, 64, (1,))


def bf16_encoder() -> Workload:
    """bf16 encoder pattern: B2 H12 n4096 d64, w=512, one global token (CLS at 0)."""
    return Workload("bf16_encoder_n4096_w512_g1", "bf16", 2, 12, 4096, 64, 512, (1,) * 12,
                    global_idx=(0,))


def bf16_charlm() -> Workload:
    """bf16 causal character-LM pattern: B1 H8 n23040 d64, causal w=512,
    heads 0-5 undilated, head 6 dilation 2, head 7 dilation 4."""
    return Workload("bf16_charlm_causal_n23040_w512", "bf16", 1, 8, 23040, 64, 512,
                    (1, 1, 1, 1, 1, 1, 2, 4), causal=True)


def bf16_qa_padded() -> Workload:
    """bf16 QA pattern: B4 H16 n4096 d64, w=512, 64 global tokens at 0..63,
    per-batch valid lengths uniform in [2048, 4096]."""
    return Workload("bf16_qa_padded_n4096_w512_g64", "bf16", 4, 16, 4096, 64, 512, (1,) * 16,
                    global_idx=tuple(range(64)), pad_len=_qa_pad_len(4, 4096))


LED_LENGTHS = (8192, 16384, 32768, 65536, 131072)


def bf16_led(n: int) -> Workload:
    """bf16 long-sequence encoder sweep: B1 H16 d128, w=1024, one global at 0."""
    return Workload(f"bf16_led_n{n}_w1024_g1", "bf16", 1, 16, n, 128, 1024, (1,) * 16,
                    global_idx=(0,))


def all_workloads() -> List[Workload]:
    return [fp32_window64(), bf16_encoder(), bf16_charlm(), bf16_qa_padded()] + [
        bf16_led(n) for n in LED_LENGTHS
    ]


def by_name(name: str) -> Workload:
    for wl in all_workloads():
        if wl.name == name:
            return wl
    raise KeyError(name)


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    qg: Optional[torch.Tensor]
    kg: Optional[torch.Tensor]
    vg: Optional[torch.Tensor]

    def tensors(self) -> List[torch.Tensor]:
        return [t for t in (self.q, self.k, self.v, self.qg, self.kg, self.vg) if t is not None]

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.tensors())


def make_inputs(wl: Workload, device: str = "cpu", seed: Optional[int] = None) -> Inputs:
    """Draw the workload's inputs with a generator on ``device``.

    A CPU and a CUDA generator with the same seed give different numbers;
    whoever checks a device result reads the device tensors back, so both
    sides always see the same values.
    """
    gen = torch.Generator(device=device).manual_seed(wl.seed if seed is None else seed)
    shape = (wl.B, wl.H, wl.n, wl.d)

    def draw(s):
        return torch.randn(s, dtype=torch.float32, generator=gen, device=device).to(wl.torch_dtype)

    q, k, v = draw(shape), draw(shape), draw(shape)
    qg = kg = vg = None
    if wl.G > 0:
        qg = draw((wl.B, wl.H, wl.G, wl.d))
        kg, vg = draw(shape), draw(shape)
    return Inputs(q, k, v, qg, kg, vg)


def custom(name: str = "custom", dtype: str = "bf16", B: int = 1, H: int = 1, n: int = 128,
           d: int = 64, w: int = 8, dilation=None, causal: bool = False, global_idx=(),
           pad_len=None, seed: int = 0) -> Workload:
    """A small pattern for tests and sweeps (w: one window, or one per head)."""
    dil = tuple(dilation) if dilation is not None else (1,) * H
    w = tuple(int(x) for x in w) if isinstance(w, (list, tuple)) else w
    return Workload(name, dtype, B, H, n, d, w, dil, causal, tuple(global_idx),
                    tuple(pad_len) if pad_len is not None else None, seed)
