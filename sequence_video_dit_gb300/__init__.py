"""Sequence-parallel (Ulysses-style) attention step of a video diffusion
transformer, GB300-native: W virtual ranks as W disjoint buffers on one GPU.

Python binding of the C ABI in ``include/sp_api.h`` with the same names.  The
functions take CUDA tensors, check shapes, and pass raw pointers, sizes and
the current stream to the library; all work runs in the library's CUDA
kernels.  Errors: ``ValueError`` (``SPValueError``) for argument problems
including the partition's not-divisible rule, ``RuntimeError`` (``SPError``)
for CUDA and device-status errors.

Stages (after "LTX-2 序列并行拆解"):
  补齐  sp_padded_len, sp_pad, sp_pad_mask
  切分  sp_partition, sp_tile
  换头  sp_send_recv_heads, sp_attention, sp_gather_heads
  还原  sp_gather_output, sp_unpad
Fused forms: sp_pad_send_heads and sp_gather_heads_output (the exchange with
its neighbours), sp_attention_shards (the exchange inside the attention).
Alternative partition: sp_optimal_split, sp_tile_2d, sp_gather_2d.
``SPStep`` runs the whole step on preallocated buffers.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import (SP_BF16, SP_ERR_TIMEOUT, SP_F32, SP_MASK_FULL, SP_MASK_KEY, SP_MASK_NONE, SP_MAX_RANKS,
                   SP_SHARD_KV, SP_SHARD_Q, SP_WORKSPACE_HEADER_BYTES, SP_WORKSPACE_KV_STALL_OFFSET, SPError,
                   SPValueError, check, lib, ptr_array, stream_handle)

__all__ = [
    "sp_padded_len", "sp_partition", "sp_pad", "sp_pad_mask", "sp_tile", "sp_send_recv_heads",
    "sp_gather_heads", "sp_send_recv_heads_noalloc", "sp_pad_send_heads", "sp_gather_heads_output",
    "sp_attention", "sp_attention_workspace_bytes", "sp_gather_output", "sp_unpad",
    "sp_optimal_split", "sp_tile_2d", "sp_gather_2d", "sp_attention_shards", "SP_SHARD_KV", "SP_SHARD_Q",
    "sp_workspace_status", "sp_sm_rotation_counts", "sp_exchange_grid", "new_workspace", "SPError",
    "SPValueError", "SPStep", "StepGraph", "SP_MASK_NONE", "SP_MASK_KEY", "SP_MASK_FULL", "SP_MAX_RANKS", "lib",
]


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SP_F32
    if t == torch.bfloat16:
        return SP_BF16
    raise SPValueError(3, f"unsupported dtype {t}")


def _row_bytes(x: torch.Tensor, lead: int = 2) -> int:
    return math.prod(x.shape[lead:]) * x.element_size()


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise SPValueError(3, "expected CUDA tensors")
        if not t.is_contiguous():
            raise SPValueError(3, "expected contiguous tensors")


def _same(ts, shape, dtype, what):
    """Every tensor of a per-rank list has the given shape and dtype (the
    kernels index each buffer by these sizes)."""
    for i, t in enumerate(ts):
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
            raise SPValueError(3, f"{what}[{i}]: expected {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")


def _split_heads(H, W, what):
    if W < 1 or H % W:
        raise SPValueError(2, f"{what}: H={H} is not divisible by W={W}")
    return H // W


def new_workspace(nbytes: int = SP_WORKSPACE_HEADER_BYTES, device=None) -> torch.Tensor:
    """A zero-filled device workspace (uint8), as the ABI requires."""
    return torch.zeros(max(int(nbytes), SP_WORKSPACE_HEADER_BYTES), dtype=torch.uint8,
                       device=device or torch.device("cuda"))


# ---------------------------------------------------------------- 补齐
def sp_padded_len(T: int, W: int) -> int:
    out = ctypes.c_int(0)
    check(lib().sp_padded_len(T, W, ctypes.byref(out)))
    return out.value


def sp_pad(x: torch.Tensor, x_pad: torch.Tensor, stream=None) -> torch.Tensor:
    """x [B,T,...] -> x_pad [B,T_pad,...] (zero rows appended)."""
    _need_cuda(x, x_pad)
    if x.shape[0] != x_pad.shape[0] or x.shape[2:] != x_pad.shape[2:] or x.dtype != x_pad.dtype:
        raise SPValueError(3, "sp_pad: shape/dtype mismatch")
    check(lib().sp_pad(x.data_ptr(), x_pad.data_ptr(), x.shape[0], x.shape[1], x_pad.shape[1],
                       _row_bytes(x), stream_handle(stream)))
    return x_pad


def sp_pad_mask(user_mask, mask_out: torch.Tensor, T: int, stream=None) -> torch.Tensor:
    """user_mask None: mask_out (1,1,T_pad) key-only mask; else (B,T,T) -> (B,T_pad,T_pad)."""
    _need_cuda(mask_out)
    T_pad = mask_out.shape[-1]
    if user_mask is None:
        B = 1
        up = None
    else:
        _need_cuda(user_mask)
        if user_mask.dtype not in (torch.uint8, torch.bool) or user_mask.shape[1:] != (T, T):
            raise SPValueError(3, "sp_pad_mask: user mask must be uint8/bool (B,T,T)")
        B = user_mask.shape[0]
        up = user_mask.data_ptr()
        if tuple(mask_out.shape) != (B, T_pad, T_pad):
            raise SPValueError(3, "sp_pad_mask: mask_out must be (B,T_pad,T_pad)")
    check(lib().sp_pad_mask(up, mask_out.data_ptr(), B, T, T_pad, stream_handle(stream)))
    return mask_out


# ---------------------------------------------------------------- 切分
def sp_partition(total_tokens: int, W: int):
    """[(start, length)] per rank; ValueError when total_tokens % W != 0."""
    starts = (ctypes.c_int * max(W, 1))()
    lens = (ctypes.c_int * max(W, 1))()
    check(lib().sp_partition(total_tokens, W, starts, lens))
    return [(starts[i], lens[i]) for i in range(W)]


def sp_tile(x_pad: torch.Tensor, shards, stream=None):
    """x_pad [B,T_pad,...] -> shards[r] [B,T_pad/W,...]."""
    _need_cuda(x_pad, *shards)
    W = len(shards)
    if W < 1 or x_pad.shape[1] % W:
        raise SPValueError(1, f"total_tokens={x_pad.shape[1]} is not divisible by world_size={W}")
    _same(shards, (x_pad.shape[0], x_pad.shape[1] // W, *x_pad.shape[2:]), x_pad.dtype, "shards")
    check(lib().sp_tile(x_pad.data_ptr(), ptr_array(shards), W, x_pad.shape[0], x_pad.shape[1],
                        _row_bytes(x_pad), stream_handle(stream)))
    return shards


# ---------------------------------------------------------------- 2-D spatial split
def sp_optimal_split(W: int):
    """(split_h, split_w): the factor pair of W closest to a square, smaller on height."""
    sh = ctypes.c_int(0)
    sw = ctypes.c_int(0)
    check(lib().sp_optimal_split(W, ctypes.byref(sh), ctypes.byref(sw)))
    return sh.value, sw.value


def _split_2d_shapes(x, shards, grid, split, what):
    F, Hg, Wg = grid
    sh, sw = split
    if len(shards) != sh * sw:
        raise SPValueError(3, f"{what}: {len(shards)} shards for a {sh}x{sw} split")
    if x.shape[1] != F * Hg * Wg:
        raise SPValueError(3, f"{what}: {x.shape[1]} tokens for a {F}x{Hg}x{Wg} grid")
    if Hg % sh or Wg % sw:
        raise SPValueError(1, f"{what}: grid {Hg}x{Wg} is not divisible by the split {sh}x{sw}")
    _same(shards, (x.shape[0], F * (Hg // sh) * (Wg // sw), *x.shape[2:]), x.dtype, "shards")


def sp_tile_2d(x: torch.Tensor, shards, grid, split=None, stream=None):
    """x [B, F*Hg*Wg, ...] -> shards[ih*split_w + iw] [B, F*(Hg/split_h)*(Wg/split_w), ...].
    ``grid`` = (F, Hg, Wg); ``split`` defaults to sp_optimal_split(len(shards))."""
    _need_cuda(x, *shards)
    split = tuple(split) if split is not None else sp_optimal_split(len(shards))
    _split_2d_shapes(x, shards, grid, split, "sp_tile_2d")
    check(lib().sp_tile_2d(x.data_ptr(), ptr_array(shards), x.shape[0], *grid, *split, _row_bytes(x),
                           stream_handle(stream)))
    return shards


def sp_gather_2d(shards, out: torch.Tensor, grid, split=None, stream=None) -> torch.Tensor:
    """Inverse of sp_tile_2d: shards -> out [B, F*Hg*Wg, ...]."""
    _need_cuda(out, *shards)
    split = tuple(split) if split is not None else sp_optimal_split(len(shards))
    _split_2d_shapes(out, shards, grid, split, "sp_gather_2d")
    check(lib().sp_gather_2d(ptr_array(shards), out.data_ptr(), out.shape[0], *grid, *split, _row_bytes(out),
                             stream_handle(stream)))
    return out


# ---------------------------------------------------------------- 换头
def sp_send_recv_heads(shards, heads, workspace: torch.Tensor, stream=None):
    """shards[s] [B,Tl,H,D] -> heads[r] [B,W*Tl,H/W,D]."""
    _need_cuda(*shards, *heads, workspace)
    W = len(shards)
    B, Tl, H, D = shards[0].shape
    Hl = _split_heads(H, W, "sp_send_recv_heads")
    _same(shards, (B, Tl, H, D), shards[0].dtype, "shards")
    _same(heads, (B, W * Tl, Hl, D), shards[0].dtype, "heads")
    check(lib().sp_send_recv_heads(ptr_array(shards), ptr_array(heads), W, B, Tl, H, D,
                                   shards[0].element_size(), workspace.data_ptr(), stream_handle(stream)))
    return heads


def sp_send_recv_heads_noalloc(shards, heads, stream=None, read_status: bool = True):
    """sp_send_recv_heads with the library's static scratch instead of a
    caller workspace (for callers that cannot allocate device memory).
    With read_status the call waits for the stream and returns the exchange's
    device status (0 = OK); otherwise it stays asynchronous and returns None."""
    _need_cuda(*shards, *heads)
    W = len(shards)
    B, Tl, H, D = shards[0].shape
    Hl = _split_heads(H, W, "sp_send_recv_heads_noalloc")
    _same(shards, (B, Tl, H, D), shards[0].dtype, "shards")
    _same(heads, (B, W * Tl, Hl, D), shards[0].dtype, "heads")
    st = ctypes.c_int(-1)
    check(lib().sp_send_recv_heads_noalloc(ptr_array(shards), ptr_array(heads), W, B, Tl, H, D,
                                           shards[0].element_size(), ctypes.byref(st) if read_status else None,
                                           stream_handle(stream)))
    return st.value if read_status else None


def sp_pad_send_heads(x, heads, workspace: torch.Tensor, stream=None):
    """Fused pad + tile + exchange: x [B,T,H,D] -> heads[r] [B,T_pad,H/W,D]."""
    _need_cuda(x, *heads, workspace)
    W = len(heads)
    B, T, H, D = x.shape
    T_pad = heads[0].shape[1]
    Hl = _split_heads(H, W, "sp_pad_send_heads")
    if T_pad < T:
        raise SPValueError(3, f"sp_pad_send_heads: T_pad={T_pad} < T={T}")
    _same(heads, (B, T_pad, Hl, D), x.dtype, "heads")
    check(lib().sp_pad_send_heads(x.data_ptr(), ptr_array(heads), W, B, T, T_pad, H, D, x.element_size(),
                                  workspace.data_ptr(), stream_handle(stream)))
    return heads


def sp_gather_heads_output(heads, out, workspace: torch.Tensor, stream=None):
    """Fused inverse exchange + gather_output: heads[r] [B,T_pad,Hl,D] -> out [B,T_out,W*Hl,D]."""
    _need_cuda(out, *heads, workspace)
    W = len(heads)
    B, T_pad, Hl, D = heads[0].shape
    _same(heads, (B, T_pad, Hl, D), heads[0].dtype, "heads")
    if tuple(out.shape) != (B, out.shape[1], W * Hl, D) or out.dtype != heads[0].dtype or out.shape[1] > T_pad:
        raise SPValueError(3, f"sp_gather_heads_output: out must be [B, T_out <= {T_pad}, {W * Hl}, {D}]")
    check(lib().sp_gather_heads_output(ptr_array(heads), out.data_ptr(), W, B, T_pad, out.shape[1], Hl * W, D,
                                       out.element_size(), workspace.data_ptr(), stream_handle(stream)))
    return out


def sp_gather_heads(heads, shards, workspace: torch.Tensor, stream=None):
    """heads[r] [B,W*Tl,Hl,D] -> shards[s] [B,Tl,W*Hl,D] (inverse exchange)."""
    _need_cuda(*shards, *heads, workspace)
    W = len(heads)
    B, T_all, Hl, D = heads[0].shape
    if T_all % W:
        raise SPValueError(1, f"total_tokens={T_all} is not divisible by world_size={W}")
    _same(heads, (B, T_all, Hl, D), heads[0].dtype, "heads")
    _same(shards, (B, T_all // W, W * Hl, D), heads[0].dtype, "shards")
    check(lib().sp_gather_heads(ptr_array(heads), ptr_array(shards), W, B, T_all // W, Hl * W, D,
                                heads[0].element_size(), workspace.data_ptr(), stream_handle(stream)))
    return shards


def sp_workspace_status(workspace: torch.Tensor, clear: bool = False, stream=None):
    """(status, per-rank CTA counts seen by the last exchange, completed exchange launches)."""
    st = ctypes.c_int(0)
    counts = (ctypes.c_int * SP_MAX_RANKS)()
    n = ctypes.c_int(0)
    check(lib().sp_workspace_status(workspace.data_ptr(), ctypes.byref(st), counts, ctypes.byref(n),
                                    1 if clear else 0, stream_handle(stream)))
    return st.value, list(counts), n.value


def sp_sm_rotation_counts(n_ctas: int, W: int):
    counts = (ctypes.c_int * W)()
    check(lib().sp_sm_rotation_counts(n_ctas, W, counts))
    return list(counts)


def sp_exchange_grid() -> int:
    n = ctypes.c_int(0)
    check(lib().sp_exchange_grid(ctypes.byref(n)))
    return n.value


def sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, dtype: torch.dtype) -> int:
    return int(lib().sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, _dtype_code(dtype)))


def _strides3(t: torch.Tensor):
    if t.dim() != 4 or t.stride(3) != 1:
        raise SPValueError(3, "attention tensors must be 4-D [B,T,Hl,D] with contiguous D")
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def sp_attention(q, k, v, o, workspace: torch.Tensor, mask_kind: int = SP_MASK_NONE, mask=None,
                 scale: float = 0.0, stream=None):
    """Attention on each rank's local heads.  q/k/v/o: lists of W tensors (views
    allowed, D contiguous) shaped [B,Tq,Hl,D] / [B,Tk,Hl,D]."""
    W = len(q)
    if not (len(k) == len(v) == len(o) == W):
        raise SPValueError(3, "sp_attention: q/k/v/o lists differ in length")
    for t in (*q, *k, *v, *o):
        if not t.is_cuda:
            raise SPValueError(3, "expected CUDA tensors")
    B, Tq, Hl, D = q[0].shape
    Tk = k[0].shape[1]
    dt = _dtype_code(q[0].dtype)
    for lst, T in ((q, Tq), (k, Tk), (v, Tk), (o, Tq)):
        for t in lst:
            if tuple(t.shape) != (B, T, Hl, D) or t.dtype != q[0].dtype or t.stride() != lst[0].stride():
                raise SPValueError(3, "sp_attention: inconsistent shapes, dtypes or strides")
    if tuple(k[0].stride()) != tuple(v[0].stride()):
        raise SPValueError(3, "sp_attention: k and v must share strides")
    mptr = None
    if mask_kind != SP_MASK_NONE:
        if mask is None or not mask.is_cuda or not mask.is_contiguous() or mask.element_size() != 1:
            raise SPValueError(3, "sp_attention: mask must be a contiguous uint8/bool CUDA tensor")
        want = Tk if mask_kind == SP_MASK_KEY else B * Tq * Tk
        if mask.numel() != want:
            raise SPValueError(3, f"sp_attention: mask has {mask.numel()} elements, expected {want}")
        mptr = mask.data_ptr()
    check(lib().sp_attention(ptr_array(q), ptr_array(k), ptr_array(v), ptr_array(o), W, B, Tq, Tk, Hl, D, dt,
                             _strides3(q[0]), _strides3(k[0]), _strides3(o[0]), mask_kind, mptr, float(scale),
                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                             stream_handle(stream)))
    return o


# ---------------------------------------------------------------- 还原
def sp_attention_shards(q, k, v, o, workspace: torch.Tensor, shard_flags: int, mask_kind: int = SP_MASK_NONE,
                        mask=None, scale: float = 0.0, stream=None, Tq: int | None = None, Tk: int | None = None):
    """The head exchange fused into the attention.  An operand with its flag
    in ``shard_flags`` is the list of the W source-rank token shards of its T
    tokens (views allowed, D contiguous), read -- or for o written -- in
    place: with Tl = ceil(T / W), shard s holds tokens [s*Tl, s*Tl + n_s) in
    its first n_s = clamp(T - s*Tl, 0, Tl) rows, [B, >= n_s, H, D] (views of
    the caller's [B, T, H, D] tensor, or padded [B, Tl, H, D] buffers).
    ``Tq`` / ``Tk`` give T; by default the sum of the shards' lengths.
    An operand without its flag is per rank as in sp_attention
    ([B, T, H/W, D] views)."""
    W = len(q)
    if not (len(k) == len(v) == len(o) == W):
        raise SPValueError(3, "sp_attention_shards: q/k/v/o lists differ in length")
    for t in (*q, *k, *v, *o):
        if not t.is_cuda:
            raise SPValueError(3, "expected CUDA tensors")
    sq, skv = bool(shard_flags & SP_SHARD_Q), bool(shard_flags & SP_SHARD_KV)
    B, _, hq, D = q[0].shape
    hk = k[0].shape[2]
    H = hq if sq else hq * W
    if (hk if skv else hk * W) != H:
        raise SPValueError(3, "sp_attention_shards: q and k disagree on the head count")

    def tokens(lst, sharded, T, name):
        if not sharded:
            T = lst[0].shape[1] if T is None else T
            want = [T] * W
        else:
            T = sum(t.shape[1] for t in lst) if T is None else T
            Tl = -(-T // W)
            want = [min(max(T - s * Tl, 0), Tl) for s in range(W)]
            if T and lst[0].shape[1] != Tl:
                raise SPValueError(3, f"sp_attention_shards: {name} shard 0 must hold ceil({T}/{W}) = {Tl} rows")
        for t, n in zip(lst, want):
            if t.shape[1] < n or (not sharded and t.shape[1] != n):
                raise SPValueError(3, f"sp_attention_shards: a {name} tensor holds {t.shape[1]} rows, needs {n}")
        return T

    Tq = tokens(q, sq, Tq, "q")
    tokens(o, sq, Tq, "o")
    Tk = tokens(k, skv, Tk, "k")
    tokens(v, skv, Tk, "v")
    for lst in (q, o, k, v):
        for t in lst:
            if (t.shape[0], t.shape[2], t.shape[3]) != (lst[0].shape[0], lst[0].shape[2], lst[0].shape[3]) or \
                    t.dtype != q[0].dtype or t.stride() != lst[0].stride() or t.shape[0] != B or t.shape[3] != D:
                raise SPValueError(3, "sp_attention_shards: inconsistent shapes, dtypes or strides")
    if tuple(k[0].stride()) != tuple(v[0].stride()):
        raise SPValueError(3, "sp_attention_shards: k and v must share strides")
    mptr = None
    if mask_kind != SP_MASK_NONE:
        if mask is None or not mask.is_cuda or not mask.is_contiguous() or mask.element_size() != 1:
            raise SPValueError(3, "sp_attention_shards: mask must be a contiguous uint8/bool CUDA tensor")
        want = Tk if mask_kind == SP_MASK_KEY else B * Tq * Tk
        if mask.numel() != want:
            raise SPValueError(3, f"sp_attention_shards: mask has {mask.numel()} elements, expected {want}")
        mptr = mask.data_ptr()
    check(lib().sp_attention_shards(ptr_array(q), ptr_array(k), ptr_array(v), ptr_array(o), W, B, Tq, Tk, H, D,
                                    _dtype_code(q[0].dtype), int(shard_flags), _strides3(q[0]), _strides3(k[0]),
                                    _strides3(o[0]), mask_kind, mptr, float(scale), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(), stream_handle(stream)))
    return o


def sp_gather_output(shards, out: torch.Tensor, stream=None) -> torch.Tensor:
    """shards[r] [B,Tl,...] -> out [B,T_out,...]: each rank's first
    clamp(T_out - r*Tl, 0, Tl) tokens, concatenated."""
    _need_cuda(out, *shards)
    W = len(shards)
    B, Tl = shards[0].shape[:2]
    _same(shards, shards[0].shape, out.dtype, "shards")
    if out.shape[0] != B or out.shape[2:] != shards[0].shape[2:] or out.shape[1] > W * Tl:
        raise SPValueError(3, f"sp_gather_output: out must be [B, T_out <= {W * Tl}, ...] like the shards")
    check(lib().sp_gather_output(ptr_array(shards), out.data_ptr(), W, B, Tl, out.shape[1], _row_bytes(out),
                                 stream_handle(stream)))
    return out


def sp_unpad(x_pad: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    _need_cuda(x_pad, out)
    if (out.shape[0] != x_pad.shape[0] or out.shape[2:] != x_pad.shape[2:] or out.shape[1] > x_pad.shape[1]
            or out.dtype != x_pad.dtype):
        raise SPValueError(3, "sp_unpad: out must be [B, T <= T_pad, ...] like x_pad")
    check(lib().sp_unpad(x_pad.data_ptr(), out.data_ptr(), x_pad.shape[0], x_pad.shape[1], out.shape[1],
                         _row_bytes(x_pad), stream_handle(stream)))
    return out


from .step import SPStep, StepGraph  # noqa: E402
