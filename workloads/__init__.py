"""Seeded synthetic inputs for the sequence-parallel attention step.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It holds only shapes and random draws: none of the step's
arithmetic (no padding, no masking rule, no exchange, no attention) lives here.

The five workloads mirror the video workloads of the LTX-2 sequence-parallel
write-up ("LTX-2 序列并行拆解", intro: a 121-frame video whose per-step
global attention over thousands of tokens is the latency bottleneck):

  c1  W=2, B=1, T=37, H=4, D=32, fp32, key-only padding mask
  c2  W=4, B=2, T=1001, H=8, D=64, bf16, user (B,T,T) mask built from
      64-token diagonal blocks, i.i.d. Bernoulli(0.1) keeps and the diagonal
  c3  W=8, B=1, T=16*24*16+5=6149, H=32, D=128, bf16, inputs N(0,1)/sqrt(D)
  c4  W=8, B=1, cross-attention: Q of 250 audio tokens, K/V of 24576 video
      tokens (32 frames x 768 patches), H=32, D=128, bf16
  c5  W=8, B=1, T=32*1536+3=49155, H=32, D=128, bf16

Draw order is fixed: Q, K, V, then the mask's uniform draws, from
``torch.Generator('cpu').manual_seed(seed)`` with ``seed = 1000 + index``.
Values are fp32 N(0,1); bf16 workloads round those draws to bf16 with
round-to-nearest-even (``Tensor.to(torch.bfloat16)``), and the oracle is fed
the same bf16 values widened exactly to fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

__all__ = ["Workload", "WORKLOADS", "get", "make_inputs", "make_custom", "SEED_BASE"]

SEED_BASE = 1000


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    W: int            # virtual ranks (world size)
    B: int
    T: int            # key/value (and, for self-attention, query) tokens
    H: int
    D: int
    dtype: str        # "f32" | "bf16"
    mask: str         # "key" (key-only padding mask) | "user" ((B,T,T) user mask)
    Tq: int | None = None       # cross-attention query length (None: self-attention)
    input_scale: float = 1.0    # multiply the N(0,1) draws by this before rounding
    block: int = 64             # user-mask diagonal block size
    keep_p: float = 0.1         # user-mask random keep probability
    notes: dict = field(default_factory=dict, compare=False)

    @property
    def cross(self) -> bool:
        return self.Tq is not None

    @property
    def q_len(self) -> int:
        return self.Tq if self.cross else self.T

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def flops(self) -> float:
        """Dense attention FLOPs on the unpadded sequence: 4*B*H*Tq*Tk*D."""
        return 4.0 * self.B * self.H * self.q_len * self.T * self.D


WORKLOADS = {
    "c1": Workload("c1", 0, W=2, B=1, T=37, H=4, D=32, dtype="f32", mask="key"),
    "c2": Workload("c2", 1, W=4, B=2, T=1001, H=8, D=64, dtype="bf16", mask="user"),
    "c3": Workload("c3", 2, W=8, B=1, T=16 * 24 * 16 + 5, H=32, D=128, dtype="bf16",
                   mask="key", input_scale=1.0 / math.sqrt(128.0)),
    "c4": Workload("c4", 3, W=8, B=1, T=32 * 768, H=32, D=128, dtype="bf16", mask="key",
                   Tq=250),
    "c5": Workload("c5", 4, W=8, B=1, T=32 * 1536 + 3, H=32, D=128, dtype="bf16", mask="key"),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def make_custom(name: str = "custom", *, W: int, B: int, T: int, H: int, D: int,
                dtype: str = "bf16", mask: str = "key", Tq: int | None = None,
                input_scale: float = 1.0, index: int = 100) -> Workload:
    """A workload with the same recipe at other sizes (parity-test cases)."""
    return Workload(name, index, W=W, B=B, T=T, H=H, D=D, dtype=dtype, mask=mask, Tq=Tq,
                    input_scale=input_scale)


def _user_mask(wl: Workload, g: torch.Generator) -> torch.Tensor:
    """(B,T,T) uint8, 1 = may attend: 64-token diagonal blocks over the unpadded
    tokens, i.i.d. Bernoulli(keep_p) keeps, and the diagonal always kept."""
    T = wl.T
    idx = torch.arange(T)
    blk = idx // wl.block
    same_block = blk[:, None] == blk[None, :]
    diag = idx[:, None] == idx[None, :]
    u = torch.rand(wl.B, T, T, generator=g)
    keep = u < wl.keep_p
    return (same_block[None] | diag[None] | keep).to(torch.uint8).contiguous()


def make_inputs(wl: Workload | str, seed: int | None = None) -> dict:
    """Returns a dict of CPU tensors:

    q [B,Tq,H,D], k [B,T,H,D], v [B,T,H,D] in the workload's dtype, and
    ``user_mask`` [B,T,T] uint8 for ``mask == "user"`` (else None).
    """
    if isinstance(wl, str):
        wl = get(wl)
    g = torch.Generator("cpu").manual_seed(wl.seed if seed is None else seed)
    shp_q = (wl.B, wl.q_len, wl.H, wl.D)
    shp_kv = (wl.B, wl.T, wl.H, wl.D)
    out = {}
    for name, shp in (("q", shp_q), ("k", shp_kv), ("v", shp_kv)):
        x = torch.randn(*shp, generator=g, dtype=torch.float32)
        if wl.input_scale != 1.0:
            x.mul_(wl.input_scale)
        out[name] = x.to(wl.torch_dtype).contiguous()
    out["user_mask"] = _user_mask(wl, g) if wl.mask == "user" else None
    return out


def shrink(wl: Workload, **kw) -> Workload:
    """Same recipe with some sizes replaced (used for fast parity cases)."""
    return replace(wl, **kw)
