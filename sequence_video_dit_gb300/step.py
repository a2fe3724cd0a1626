"""One sequence-parallel attention step on preallocated buffers.

The call sequence follows "LTX-2 序列并行拆解" (LTX-2 sequence-parallel
breakdown), sections 补齐 -> 切分 -> 换头 -> 还原:

  self-attention                        cross-attention, small query modality
  1 sp_pad(Q,K,V), sp_pad_mask          1 sp_pad(K,V), sp_pad_mask (key mask)
  2 sp_tile(Q,K,V)                      2 sp_tile(K,V)
  3 sp_send_recv_heads(Q,K,V)           3 sp_send_recv_heads(K,V)  (Q is sliced
                                          per rank in place: no exchange)
  4 sp_attention on the local heads     4 sp_attention, each rank writing its
                                          heads of the [B,Tq,H,D] output
  5 sp_gather_heads(O)
  6 sp_gather_output(O) cropped to the caller's length T (each rank's real
    token count), which is the unpad

The small-query case is the pages' video->audio direction: the audio query
stays whole on every rank and only the video K/V go through the exchange.
The opposite direction (``Tkv``: video queries attend a small, replicated
audio K/V) mirrors it: Q is padded, tiled and exchanged like self-attention,
each rank reads its heads of K/V in place, and O returns through
gather_heads / gather_output.  Pad query rows then see every audio key; they
are cropped by the unpad.

Each virtual rank owns separate device allocations.  sp_pad is skipped when T
is already a multiple of W (padding is then the identity).  Host code here
only allocates buffers and issues library calls on the current stream.

``fused=True`` runs the same step with the fused exchange entry points: one
sp_pad_send_heads per tensor (pad + tile + exchange in one pass, no token-shard
buffers) and one sp_gather_heads_output (inverse exchange + gather + unpad).

``grid=(F, Hg, Wg)`` partitions the tokens with the 2-D spatial split of the
LongCat-Video context-parallel page (智能张量拆分) instead of token ranges:
sp_tile_2d gives rank ih*split_w + iw block (ih, iw) of every frame, the
exchange and attention run unchanged on those shards, and sp_gather_2d puts
the output blocks back.  The split must divide the grid, so nothing is padded
and no mask is needed.

``direct=True`` fuses the head exchange into the attention
(sp_attention_shards): the operands that would go through sp_send_recv_heads
are handed over as the W token shards and each attention tile is loaded from
its source shard, O is written into token-shard layout, so no exchange kernel
runs.  It needs the tensor-core kernel (bf16, D = 64 or 128).  With
``fused=False`` the shards are the W rank buffers sp_tile (or sp_tile_2d)
fills and sp_gather_output (sp_gather_2d) assembles the output; with
``fused=True`` they are views of the caller's tensors, the last ones short of
the pad rows when T % W != 0, and nothing is copied or padded at all: pad
keys and pad queries are simply never read (no padding mask is needed; a
user mask is read as the caller's (B, T, T) mask).  When every shard is a
whole number of 128-row tiles the output equals the staged step's bit for
bit; otherwise the attention visits the keys in another order (each shard's
whole tiles, then one tile gathering the shards' leftover rows), which moves
only the rounding of the key sum.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import SP_BF16, check, lib, stream_handle
from . import (SP_MASK_FULL, SP_MASK_KEY, SP_MASK_NONE, SP_SHARD_KV, SP_SHARD_Q, new_workspace, sp_attention_shards, sp_attention, sp_attention_workspace_bytes,
               sp_gather_2d, sp_gather_heads, sp_gather_heads_output, sp_gather_output, sp_optimal_split, sp_pad,
               sp_pad_mask, sp_pad_send_heads, sp_padded_len, sp_partition, sp_send_recv_heads, sp_tile,
               sp_tile_2d, SPValueError)


class _NullTimer:
    def __call__(self, name):
        return self

    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


class StageTimer:
    """Records CUDA events around named stages on the current stream."""

    def __init__(self):
        self.events = {}

    def __call__(self, name):
        self._name = name
        return self

    def __enter__(self):
        s = torch.cuda.Event(enable_timing=True)
        s.record()
        self._start = s
        return self

    def __exit__(self, *a):
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        self.events.setdefault(self._name, []).append((self._start, e))
        return False

    def totals_ms(self):
        return {k: sum(s.elapsed_time(e) for s, e in v) for k, v in self.events.items()}

    def counts(self):
        return {k: len(v) for k, v in self.events.items()}


class SPStep:
    """Buffers and call sequence of one SP attention step.

    ``T`` is always the length of the token-sharded sequence.
    Self-attention: ``Tq=Tkv=None``, inputs q/k/v [B,T,H,D].
    Cross-attention, small query: ``Tq`` query tokens (replicated on every
    rank), q [B,Tq,H,D]; k/v [B,T,H,D] go through the exchange.
    Cross-attention, small K/V: ``Tkv`` key tokens (replicated on every rank),
    q [B,T,H,D] goes through the exchange; k/v [B,Tkv,H,D], every key valid.
    ``mask``: "key" (key-only padding mask) or "user" ((B,T,T) user mask,
    self-attention only).
    ``grid``: (F, Hg, Wg) with F*Hg*Wg = T selects the 2-D spatial split
    (self-attention, staged exchange).
    ``direct``: the exchange fused into the attention (see the module text).
    """

    def __init__(self, W: int, B: int, T: int, H: int, D: int, dtype=torch.bfloat16, mask: str = "key",
                 Tq: int | None = None, device=None, fused: bool = False, Tkv: int | None = None,
                 grid: tuple | None = None, direct: bool = False):
        if H % W:
            raise SPValueError(2, f"H={H} is not divisible by W={W}")
        if mask not in ("key", "user"):
            raise SPValueError(3, f"mask must be 'key' or 'user', got {mask!r}")
        if (Tq is not None or Tkv is not None) and mask == "user":
            raise SPValueError(3, "cross-attention takes the key-only mask")
        if Tq is not None and Tkv is not None:
            raise SPValueError(3, "give Tq (small query) or Tkv (small K/V), not both")
        if Tkv is not None and Tkv < 0:
            raise SPValueError(3, f"Tkv={Tkv} < 0")
        self.grid = tuple(grid) if grid is not None else None
        if self.grid is not None:
            if Tq is not None or Tkv is not None or mask != "key" or fused:
                raise SPValueError(3, "the 2-D split is built for self-attention with the staged exchange")
            F, Hg, Wg = self.grid
            if F * Hg * Wg != T:
                raise SPValueError(3, f"grid {self.grid} does not hold T={T} tokens")
            self.split = sp_optimal_split(W)
            if Hg % self.split[0] or Wg % self.split[1]:
                raise SPValueError(1, f"grid {Hg}x{Wg} is not divisible by the split {self.split[0]}x{self.split[1]}")
        dev = torch.device(device or "cuda")
        self.W, self.B, self.T, self.H, self.D, self.dtype = W, B, T, H, D, dtype
        self.cross = Tq is not None
        self.Tq = Tq if self.cross else None
        self.kv_small = Tkv is not None
        self.Tkv = Tkv
        self.mask_kind = mask
        self.T_pad = sp_padded_len(T, W)
        sp_partition(self.T_pad, W)
        self.Tl = self.T_pad // W
        self.Hl = H // W
        self.need_pad = self.T_pad != T
        self.fused = fused
        self.direct = direct
        if direct and (dtype != torch.bfloat16 or D not in (64, 128)):
            raise SPValueError(6, "direct: the tensor-core attention needs bf16 and D = 64 or 128")
        # shard views of the caller's tensors (direct + fused) need no buffers,
        # no padding and no padding mask
        views = direct and fused
        self.views = views
        names = ("k", "v") if self.cross else (("q",) if self.kv_small else ("q", "k", "v"))
        self.names = names
        emp = lambda *shape: torch.empty(*shape, dtype=dtype, device=dev)  # noqa: E731
        self.xpad = {n: emp(B, self.T_pad, H, D) for n in names} if (self.need_pad and not fused) else {}
        self.shards = {} if (fused and not direct) or views else {n: [emp(B, self.Tl, H, D) for _ in range(W)]
                                                                   for n in names}
        self.heads = {} if direct else {n: [emp(B, self.T_pad, self.Hl, D) for _ in range(W)] for n in names}
        if not self.cross:
            self.o_heads = [] if direct else [emp(B, self.T_pad, self.Hl, D) for _ in range(W)]
            self.o_shards = [] if (fused and not direct) or views else [emp(B, self.Tl, H, D) for _ in range(W)]
            self.out = emp(B, T, H, D)
            Tq_att = self.T_pad
        else:
            self.out = emp(B, Tq, H, D)
            Tq_att = Tq
        if self.kv_small or self.grid is not None or views:
            # every key is valid: replicated K/V, a 2-D split with no padding,
            # or shard views that hold no pad rows (a user mask is read as given)
            self.mask = None
        elif mask == "key":
            self.mask = torch.empty(1, 1, self.T_pad, dtype=torch.uint8, device=dev)
        else:
            self.mask = torch.empty(B, self.T_pad, self.T_pad, dtype=torch.uint8, device=dev)
        Tk_att = Tkv if self.kv_small else (T if views else self.T_pad)
        if views and not self.cross:
            Tq_att = T
        self.ws_exchange = new_workspace(device=dev)
        self.ws_attn = new_workspace(sp_attention_workspace_bytes(W, B, Tq_att, Tk_att, self.Hl, D, dtype), dev)

    # bytes each exchange launch reads + writes
    def exchange_bytes_per_launch(self) -> int:
        return 2 * self.B * self.T_pad * self.H * self.D * torch.empty((), dtype=self.dtype).element_size()

    def n_exchange_launches(self) -> int:
        """Launches of the exchange kernels per step (send per tensor + gather)."""
        if self.direct:
            return 0
        return len(self.names) + (0 if self.cross else 1)

    def _shard_views(self, x):
        """The W token shards of a caller tensor [B, T, H, D] as views: shard s
        holds tokens [s*Tl, min((s+1)*Tl, T)), the last ones short of the pad
        rows (or empty) when T % W != 0."""
        return [x[:, min(s * self.Tl, self.T):min((s + 1) * self.Tl, self.T)] for s in range(self.W)]

    def __call__(self, q, k, v, user_mask=None, timer=None, out=None):
        """Runs the step on the current stream and returns the output tensor
        (``out`` if given, shaped like ``self.out``, else ``self.out``)."""
        t = timer or _NullTimer()
        if out is None:
            out = self.out
        elif tuple(out.shape) != tuple(self.out.shape) or out.dtype != self.out.dtype:
            raise SPValueError(3, "out must match the step's output shape and dtype")
        src = {"q": q, "k": k, "v": v}
        with t("pad"):
            if self.need_pad and not self.fused:
                for n in self.names:
                    sp_pad(src[n], self.xpad[n])
            if self.mask is None:
                if self.views and self.mask_kind == "user" and user_mask is None:
                    raise SPValueError(3, "this step was built for a user mask")
                # no padded keys: replicated K/V, a 2-D split or in-place shard views
            elif self.mask_kind == "key":
                sp_pad_mask(None, self.mask, self.T)
            else:
                if user_mask is None:
                    raise SPValueError(3, "this step was built for a user mask")
                sp_pad_mask(user_mask, self.mask, self.T)
        if self.views:
            return self._direct_inplace(q, k, v, out, t, user_mask)
        if self.direct:
            return self._direct(q, k, v, src, out, t, user_mask)
        if self.fused:
            with t("send_recv_heads"):
                for n in self.names:
                    sp_pad_send_heads(src[n], self.heads[n], self.ws_exchange)
        else:
            with t("tile"):
                for n in self.names:
                    if self.grid is not None:
                        sp_tile_2d(src[n], self.shards[n], self.grid, self.split)
                    else:
                        sp_tile(self.xpad[n] if self.need_pad else src[n], self.shards[n])
            with t("send_recv_heads"):
                for n in self.names:
                    sp_send_recv_heads(self.shards[n], self.heads[n], self.ws_exchange)
        kind, mask = self._mask_arg()
        Hl, D = self.Hl, self.D
        with t("attention"):
            if self.kv_small:
                kv = [(k[:, :, r * Hl:(r + 1) * Hl, :], v[:, :, r * Hl:(r + 1) * Hl, :]) for r in range(self.W)]
                sp_attention(self.heads["q"], [a for a, _ in kv], [b for _, b in kv], self.o_heads, self.ws_attn)
            elif not self.cross:
                sp_attention(self.heads["q"], self.heads["k"], self.heads["v"], self.o_heads, self.ws_attn,
                             kind, mask)
            else:
                qv = [q[:, :, r * Hl:(r + 1) * Hl, :] for r in range(self.W)]
                ov = [out[:, :, r * Hl:(r + 1) * Hl, :] for r in range(self.W)]
                sp_attention(qv, self.heads["k"], self.heads["v"], ov, self.ws_attn, kind, mask)
        if not self.cross:
            if self.fused:
                with t("gather_heads"):
                    sp_gather_heads_output(self.o_heads, out, self.ws_exchange)
            else:
                with t("gather_heads"):
                    sp_gather_heads(self.o_heads, self.o_shards, self.ws_exchange)
                with t("gather_output"):
                    if self.grid is not None:
                        sp_gather_2d(self.o_shards, out, self.grid, self.split)
                    else:
                        sp_gather_output(self.o_shards, out)
        return out

    def capture(self, q, k, v, user_mask=None, out=None) -> "StepGraph":
        """Records the whole step, for these input and output buffers, as one
        CUDA graph (after one eager run that does the host-side first-call
        set-up).  ``StepGraph.replay()`` then runs every kernel of the step
        with a single launch from the host; copy new data into q, k, v (and
        the user mask) in place between replays."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self(q, k, v, user_mask=user_mask, out=out)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            result = self(q, k, v, user_mask=user_mask, out=out)
        return StepGraph(graph, result, (q, k, v, user_mask))

    def _mask_arg(self):
        if self.mask is None:
            return SP_MASK_NONE, None
        if self.mask_kind == "key":
            return SP_MASK_KEY, self.mask.view(-1)
        return SP_MASK_FULL, self.mask

    def _direct(self, q, k, v, src, out, t, user_mask=None):
        """The step with the exchange fused into the attention: token shards in,
        O in token-shard layout out (after pad and mask, which ran already)."""
        W, Hl = self.W, self.Hl
        if self.fused:  # the caller's tensors, in place
            shards = {n: self._shard_views(src[n]) for n in self.names}
            o_sh = None if self.cross else self._shard_views(out)
        else:
            with t("tile"):
                for n in self.names:
                    if self.grid is not None:
                        sp_tile_2d(src[n], self.shards[n], self.grid, self.split)
                    else:
                        sp_tile(self.xpad[n] if self.need_pad else src[n], self.shards[n])
            shards, o_sh = self.shards, (None if self.cross else self.o_shards)
        kind, mask = self._mask_arg()
        if self.views and self.mask_kind == "user":
            kind, mask = SP_MASK_FULL, user_mask  # the caller's (B, T, T) mask: no pad rows exist here
        # the sharded operands' token count: the caller's T (in place) or the padded buffers' T_pad
        T_sh = self.T if self.fused else self.T_pad
        with t("attention"):
            if self.kv_small:
                kv = [(k[:, :, r * Hl:(r + 1) * Hl, :], v[:, :, r * Hl:(r + 1) * Hl, :]) for r in range(W)]
                sp_attention_shards(shards["q"], [a for a, _ in kv], [b for _, b in kv], o_sh, self.ws_attn,
                                    SP_SHARD_Q, Tq=T_sh)
            elif not self.cross:
                sp_attention_shards(shards["q"], shards["k"], shards["v"], o_sh, self.ws_attn,
                                    SP_SHARD_Q | SP_SHARD_KV, kind, mask, Tq=T_sh, Tk=T_sh)
            else:
                qv = [q[:, :, r * Hl:(r + 1) * Hl, :] for r in range(W)]
                ov = [out[:, :, r * Hl:(r + 1) * Hl, :] for r in range(W)]
                sp_attention_shards(qv, shards["k"], shards["v"], ov, self.ws_attn, SP_SHARD_KV, kind, mask, Tk=T_sh)
        if not self.cross and not self.fused:
            with t("gather_output"):
                if self.grid is not None:
                    sp_gather_2d(o_sh, out, self.grid, self.split)
                else:
                    sp_gather_output(o_sh, out)
        return out


    def _direct_inplace(self, q, k, v, out, t, user_mask=None):
        """The direct step on the caller's tensors in place (``direct=True,
        fused=True``): one sp_attention_shards call whose shard and head-slice
        pointers are offsets into q, k, v and out, marshalled into argument
        arrays built once (this keeps the host cost of a short step low)."""
        W, Hl, H, D, B, T = self.W, self.Hl, self.H, self.D, self.B, self.T
        Tq = self.Tq if self.cross else T
        Tk = self.Tkv if self.kv_small else T
        want = {"q": (B, Tq, H, D), "k": (B, Tk, H, D), "v": (B, Tk, H, D), "out": (B, Tq, H, D)}
        for name, x in (("q", q), ("k", k), ("v", v), ("out", out)):
            if tuple(x.shape) != want[name] or x.dtype != self.dtype or not x.is_contiguous() or not x.is_cuda:
                raise SPValueError(3, f"direct step: {name} must be a contiguous CUDA {self.dtype} {want[name]}")
        if not hasattr(self, "_args"):
            P = ctypes.c_void_p * W
            self._args = [P(), P(), P(), P()]
            self._strides = {n: (ctypes.c_int64 * 3)(sh[1] * H * D, H * D, D) for n, sh in want.items()}
        elt, Tl = q.element_size(), self.Tl
        qa, ka, va, oa = self._args

        def shards(arr, x, n_tok):  # token shard s starts at token min(s*Tl, n_tok)
            base = x.data_ptr()
            for s in range(W):
                arr[s] = base + min(s * Tl, n_tok) * H * D * elt

        def heads(arr, x):  # rank r's heads of a replicated tensor, sliced in place
            base = x.data_ptr()
            for r in range(W):
                arr[r] = base + r * Hl * D * elt

        if self.cross:  # small query sliced per rank, K/V sharded
            heads(qa, q), heads(oa, out), shards(ka, k, Tk), shards(va, v, Tk)
            flags = SP_SHARD_KV
        elif self.kv_small:  # Q sharded, small K/V sliced per rank
            shards(qa, q, Tq), shards(oa, out, Tq), heads(ka, k), heads(va, v)
            flags = SP_SHARD_Q
        else:
            shards(qa, q, T), shards(oa, out, T), shards(ka, k, T), shards(va, v, T)
            flags = SP_SHARD_Q | SP_SHARD_KV
        kind, mptr = SP_MASK_NONE, None
        if self.mask_kind == "user" and not self.cross and not self.kv_small:
            if user_mask is None or tuple(user_mask.shape) != (B, T, T) or user_mask.element_size() != 1 \
                    or not user_mask.is_contiguous() or not user_mask.is_cuda:
                raise SPValueError(3, f"direct step: the user mask must be a contiguous uint8 CUDA ({B}, {T}, {T})")
            kind, mptr = SP_MASK_FULL, user_mask.data_ptr()
        ws = self.ws_attn
        with t("attention"):
            check(lib().sp_attention_shards(qa, ka, va, oa, W, B, Tq, Tk, H, D, SP_BF16, flags, self._strides["q"],
                                            self._strides["k"], self._strides["out"], kind, mptr, 0.0,
                                            ws.data_ptr(), ws.numel() * ws.element_size(), stream_handle(None)))
        return out


class StepGraph:
    """A captured SP step: ``replay()`` reruns it on the captured buffers and
    returns the output tensor (the same storage every time)."""

    def __init__(self, graph, out, inputs):
        self.graph = graph
        self.out = out
        self._inputs = inputs  # kept alive: the graph reads them by address

    def replay(self):
        self.graph.replay()
        return self.out
