"""Seeded synthetic inputs for the KATA forward and decode workloads.

This module only draws random numbers and shapes them; it holds none of the
attention arithmetic.  The tests feed the same tensors to the CUDA library and
to the CPU oracle, and the benchmark times the CUDA library on them.

Five forward workloads (shapes of the KATA paper's kernel study: one head of
causal normalised linear attention with the rank-one PSD lift, Sec. 4 and
App. E) plus one decode workload:

  name           B   H  T       d   dv  C    dtype  q, k                         v
  small_fp32     1   1  256     16  16  32   f32    N(0,I) on the unit sphere    N(0,1)
  mid_bf16       4   8  4096    32  64  64   bf16   N(0,I) on the unit sphere    N(0,1)
  recall_bf16    16  4  8192    32  64  64   bf16   drawn from 1024 unit keys    N(0,1)
  lm_layer_bf16  8   16 2048    64  64  64   bf16   N(0, I/d), not normalised    N(0,1)
  long_ctx_bf16  1   16 131072  32  64  128  bf16   N(0,I) on the unit sphere    N(0,1)
  decode         256 16 (1)     64  64  -    bf16   N(0, I/d)                    N(0,1)

recall_bf16: one dictionary of 1024 Gaussian keys normalised to the unit sphere;
each position draws its key index uniformly with replacement (so a key recurs
about 8 times per 8192-token sequence, each time with a fresh value, i.e. a
repeated-key overwrite), and its query index independently from the same
dictionary.

Seeds: tensor i of workload j (j in table order, 0..5) comes from a
torch.Generator seeded with 1000*j + i on the device the tensor is made on.

GatedKATA gates (the pages parameterise log gamma_t as the log-sigmoid of a
per-token projection): gamma = sigmoid(x), x ~ N(4, 1) per (b, h, t) (seed
1000*j + 8; per (b, h) for one decode step, seed 1000*j + 9), so most gates lie
in 0.95 .. 0.995 and writes fade over some tens of tokens.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    T: int
    d: int
    dv: int
    C: int
    dtype: torch.dtype
    kind: str  # "sphere", "dictionary", "scaled_gauss"

    def scaled(self, **kw) -> "Workload":
        """Same recipe at other sizes (for parity cases the oracle can finish)."""
        return dataclasses.replace(self, **kw)

    @property
    def n(self) -> int:
        return self.d * (self.d + 1) // 2

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "small_fp32": Workload("small_fp32", 0, 1, 1, 256, 16, 16, 32, torch.float32, "sphere"),
    "mid_bf16": Workload("mid_bf16", 1, 4, 8, 4096, 32, 64, 64, torch.bfloat16, "sphere"),
    "recall_bf16": Workload("recall_bf16", 2, 16, 4, 8192, 32, 64, 64, torch.bfloat16,
                            "dictionary"),
    "lm_layer_bf16": Workload("lm_layer_bf16", 3, 8, 16, 2048, 64, 64, 64, torch.bfloat16,
                              "scaled_gauss"),
    "long_ctx_bf16": Workload("long_ctx_bf16", 4, 1, 16, 131072, 32, 64, 128,
                              torch.bfloat16, "sphere"),
}

DECODE = Workload("decode", 5, 256, 16, 1, 64, 64, 0, torch.bfloat16, "scaled_gauss")

DICTIONARY_SIZE = 1024


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, device, seed):
    return torch.randn(shape, generator=_gen(device, seed), device=device,
                       dtype=torch.float32)


def _to_sphere(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_qkv(w: Workload, device="cpu"):
    """q, k: [B,H,T,d]; v: [B,H,T,dv]; contiguous, in w.dtype, on `device`."""
    base = 1000 * w.index
    B, H, T, d, dv = w.B, w.H, w.T, w.d, w.dv
    if w.kind == "sphere":
        q = _to_sphere(_randn((B, H, T, d), device, base + 0))
        k = _to_sphere(_randn((B, H, T, d), device, base + 1))
    elif w.kind == "scaled_gauss":
        scale = 1.0 / float(d) ** 0.5
        q = _randn((B, H, T, d), device, base + 0) * scale
        k = _randn((B, H, T, d), device, base + 1) * scale
    elif w.kind == "dictionary":
        keys = _to_sphere(_randn((DICTIONARY_SIZE, d), device, base + 0))
        kidx = torch.randint(0, DICTIONARY_SIZE, (B, H, T), generator=_gen(device, base + 1),
                             device=device)
        qidx = torch.randint(0, DICTIONARY_SIZE, (B, H, T), generator=_gen(device, base + 2),
                             device=device)
        k = keys[kidx]
        q = keys[qidx]
    else:
        raise ValueError(w.kind)
    v = _randn((B, H, T, dv), device, base + 3)
    return (q.to(w.dtype).contiguous(), k.to(w.dtype).contiguous(),
            v.to(w.dtype).contiguous())


def make_decode_inputs(w: Workload = DECODE, device="cpu"):
    """One decode token per (b, h): q, k [B,H,d], v [B,H,dv] in w.dtype."""
    base = 1000 * w.index
    scale = 1.0 / float(w.d) ** 0.5
    q = (_randn((w.B, w.H, w.d), device, base + 0) * scale).to(w.dtype).contiguous()
    k = (_randn((w.B, w.H, w.d), device, base + 1) * scale).to(w.dtype).contiguous()
    v = _randn((w.B, w.H, w.dv), device, base + 2).to(w.dtype).contiguous()
    return q, k, v


def make_decode_prefix(w: Workload = DECODE, length: int = 16, device="cpu"):
    """A seeded token prefix (k [B,H,L,d], v [B,H,L,dv]) from which a decode
    state is built by the recurrence; drawn like the decode tokens."""
    base = 1000 * w.index
    scale = 1.0 / float(w.d) ** 0.5
    k = (_randn((w.B, w.H, length, w.d), device, base + 4) * scale).to(w.dtype)
    v = _randn((w.B, w.H, length, w.dv), device, base + 5).to(w.dtype)
    return k.contiguous(), v.contiguous()


def make_decode_state_fill(w: Workload = DECODE, device="cpu"):
    """A seeded fp32 state (S [B,H,n,dv], z [B,H,n]) for timing the decode step
    only: S ~ N(0,1), z ~ |N(0,1)| + 1.  It is not a state any token sequence
    produces (its normaliser can be <= 0); the content does not change the
    cost.  Parity tests build states from make_decode_prefix instead."""
    base = 1000 * w.index
    S = _randn((w.B, w.H, w.n, w.dv), device, base + 6)
    z = _randn((w.B, w.H, w.n), device, base + 7).abs_() + 1.0
    return S.contiguous(), z.contiguous()


def make_gate(w: Workload, device="cpu"):
    """GatedKATA gates gamma [B,H,T] float32 in (0, 1): sigmoid of N(4, 1)."""
    x = _randn((w.B, w.H, w.T), device, 1000 * w.index + 8) + 4.0
    return torch.sigmoid(x).contiguous()


def make_decode_gate(w: Workload = DECODE, device="cpu"):
    """Gates for one decode step, gamma [B,H] float32: sigmoid of N(4, 1)."""
    x = _randn((w.B, w.H), device, 1000 * w.index + 9) + 4.0
    return torch.sigmoid(x).contiguous()
