"""Plain CPU oracle for the Ulysses-style sequence-parallel attention step.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline leg and ``--impl reference``) may import or
run this package.  The product library never calls it and shares no code
with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation, no fused or
reordered loops); this module compiles it with gcc on first use and wraps it
with numpy.  Every routine follows the LTX-2 sequence-parallel write-up
("LTX-2 序列并行拆解"): 补齐 (pad), 切分 (partition), 换头 (head exchange),
还原 (restore) and the correctness paragraph that closes 还原: the sharded
step is an exact redistribution around ordinary softmax attention.

Parity status of each function is stated in its docstring; the pins are the
``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``.

Arrays: activations are numpy arrays shaped [B, T, H, D].  bf16 data is
carried as uint16 bit patterns for the layout routines; attention takes
float32 values (a bf16 value widens to fp32 exactly) and returns float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_NONE, MASK_KEY, MASK_FULL = 0, 1, 2


class PartitionError(ValueError):
    """total_tokens is not a multiple of world_size (切分)."""


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared object with gcc (-O2, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
                           "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, Z, D_ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
            I64 = ctypes.c_int64
            lib.oracle_padded_len.argtypes = [I, I]
            lib.oracle_padded_len.restype = I
            lib.oracle_pad.argtypes = [P, P, I, I, I, Z]
            lib.oracle_pad_mask_key.argtypes = [P, I, I]
            lib.oracle_pad_mask_user.argtypes = [P, P, I, I, I]
            lib.oracle_partition.argtypes = [I, I, P, P]
            lib.oracle_partition.restype = I
            lib.oracle_tile.argtypes = [P, P, I, I, I, Z]
            lib.oracle_send_recv_heads.argtypes = [P, P, I, I, I, I, I, Z]
            lib.oracle_gather_heads.argtypes = [P, P, I, I, I, I, I, Z]
            lib.oracle_gather_output.argtypes = [P, P, I, I, I, I, Z]
            lib.oracle_unpad.argtypes = [P, P, I, I, I, Z]
            lib.oracle_sm_rotation_counts.argtypes = [I, I, P]
            lib.oracle_optimal_split.argtypes = [I, P, P]
            lib.oracle_optimal_split.restype = I
            lib.oracle_tile_2d.argtypes = [P, P, I, I, I, I, I, I, Z]
            lib.oracle_tile_2d.restype = I
            lib.oracle_gather_2d.argtypes = [P, P, I, I, I, I, I, I, Z]
            lib.oracle_gather_2d.restype = I
            lib.oracle_attention.argtypes = [P, P, P, P, I, I, I, I, I, I, P, D_, I]
            lib.oracle_attention.restype = I
            lib.oracle_attention_rows.argtypes = [P, P, P, P, I, I, I, I, I, I, P, D_, P, I64, I]
            lib.oracle_attention_rows.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _row_bytes(x: np.ndarray, lead: int) -> int:
    return int(np.prod(x.shape[lead:], dtype=np.int64)) * x.itemsize


def default_threads() -> int:
    return os.cpu_count() or 1


# ---------------------------------------------------------------- 补齐 (pad)
def padded_len(T: int, W: int) -> int:
    """Smallest multiple of W that is >= T.  Pinned: closed form ceil(T/W)*W."""
    return int(_L().oracle_padded_len(T, W))


def pad(x: np.ndarray, T_pad: int) -> np.ndarray:
    """[B,T,...] -> [B,T_pad,...], zero rows appended.  Pinned: tiny literal cases."""
    x = np.ascontiguousarray(x)
    B, T = x.shape[:2]
    out = np.empty((B, T_pad) + x.shape[2:], dtype=x.dtype)
    _L().oracle_pad(_p(x), _p(out), B, T, T_pad, _row_bytes(x, 2))
    return out


def pad_mask_key(T: int, T_pad: int) -> np.ndarray:
    """(1,1,T_pad) uint8 key-only padding mask.  Pinned: literal cases."""
    out = np.empty((1, 1, T_pad), dtype=np.uint8)
    _L().oracle_pad_mask_key(_p(out), T, T_pad)
    return out


def pad_mask_user(user: np.ndarray, T_pad: int) -> np.ndarray:
    """(B,T,T) user mask -> (B,T_pad,T_pad) with pad rows seeing all real keys.
    Pinned: hand-derived golden fixture."""
    user = np.ascontiguousarray(user.astype(np.uint8))
    B, T, _ = user.shape
    out = np.empty((B, T_pad, T_pad), dtype=np.uint8)
    _L().oracle_pad_mask_user(_p(user), _p(out), B, T, T_pad)
    return out


# ---------------------------------------------------------------- 切分 (partition)
def partition(total_tokens: int, W: int):
    """Per-rank (start, length) of uniform shards; raises PartitionError when
    total_tokens % W != 0.  Pinned: the page's ValueError rule."""
    starts = np.zeros(max(W, 1), dtype=np.int32)
    lens = np.zeros(max(W, 1), dtype=np.int32)
    rc = _L().oracle_partition(total_tokens, W, _p(starts), _p(lens))
    if rc == 1:
        raise PartitionError(f"total_tokens={total_tokens} is not divisible by world_size={W}")
    if rc != 0:
        raise ValueError("invalid partition arguments")
    return [(int(s), int(n)) for s, n in zip(starts[:W], lens[:W])]


def tile(x_pad: np.ndarray, W: int):
    """[B,T_pad,...] -> W shards [B,T_pad/W,...].  Pinned: brute force."""
    x_pad = np.ascontiguousarray(x_pad)
    B, T_pad = x_pad.shape[:2]
    partition(T_pad, W)
    Tl = T_pad // W
    shards = [np.empty((B, Tl) + x_pad.shape[2:], dtype=x_pad.dtype) for _ in range(W)]
    _L().oracle_tile(_p(x_pad), _ptr_array(shards), W, B, T_pad, _row_bytes(x_pad, 2))
    return shards


# ---------------------------------------------------------------- 换头 (head exchange)
def send_recv_heads(shards):
    """W x [B,Tl,H,D] -> W x [B,W*Tl,H/W,D].  Pinned: brute-force index map,
    round trip with gather_heads."""
    W = len(shards)
    B, Tl, H, D = shards[0].shape
    if H % W:
        raise ValueError("H is not divisible by world_size")
    shards = [np.ascontiguousarray(s) for s in shards]
    heads = [np.empty((B, W * Tl, H // W, D), dtype=shards[0].dtype) for _ in range(W)]
    _L().oracle_send_recv_heads(_ptr_array(shards), _ptr_array(heads), W, B, Tl, H, D,
                                shards[0].itemsize)
    return heads


def gather_heads(heads):
    """W x [B,T_all,Hl,D] -> W x [B,T_all/W,Hl*W,D]; inverse of send_recv_heads."""
    W = len(heads)
    B, T_all, Hl, D = heads[0].shape
    Tl = T_all // W
    heads = [np.ascontiguousarray(h) for h in heads]
    shards = [np.empty((B, Tl, Hl * W, D), dtype=heads[0].dtype) for _ in range(W)]
    _L().oracle_gather_heads(_ptr_array(heads), _ptr_array(shards), W, B, Tl, Hl * W, D,
                             heads[0].itemsize)
    return shards


# ---------------------------------------------------------------- 还原 (restore)
def gather_output(shards, T_out: int) -> np.ndarray:
    """Concatenate each rank's first n_r = clamp(T_out - r*Tl, 0, Tl) tokens.
    Pinned: brute force, round trip with tile."""
    W = len(shards)
    B, Tl = shards[0].shape[:2]
    shards = [np.ascontiguousarray(s) for s in shards]
    out = np.empty((B, T_out) + shards[0].shape[2:], dtype=shards[0].dtype)
    _L().oracle_gather_output(_ptr_array(shards), _p(out), W, B, Tl, T_out,
                              _row_bytes(shards[0], 2))
    return out


def unpad(x_pad: np.ndarray, T: int) -> np.ndarray:
    """[B,T_pad,...] -> [B,T,...].  Pinned: round trip with pad."""
    x_pad = np.ascontiguousarray(x_pad)
    B, T_pad = x_pad.shape[:2]
    out = np.empty((B, T) + x_pad.shape[2:], dtype=x_pad.dtype)
    _L().oracle_unpad(_p(x_pad), _p(out), B, T_pad, T, _row_bytes(x_pad, 2))
    return out


# ---------------------------------------------------------------- 2-D spatial split
# LongCat-Video context parallel ("智能张量拆分"): an alternative to the
# token-range partition for the tile step.  The latent tokens of a batch item
# are a [F, Hg, Wg] grid (frames x patch rows x patch columns) in row-major
# order.
class SplitError(ValueError):
    """The grid is not divisible by the 2-D split."""


def optimal_split(W: int):
    """(split_h, split_w): the factor pair of W closest to a square, the
    smaller factor on height.  Pinned: brute force over all factor pairs."""
    sh = ctypes.c_int(0)
    sw = ctypes.c_int(0)
    if _L().oracle_optimal_split(W, ctypes.byref(sh), ctypes.byref(sw)) != 0:
        raise ValueError(f"W={W} < 1")
    return sh.value, sw.value


def tile_2d(x: np.ndarray, grid, split):
    """x [B, F*Hg*Wg, ...] -> split_h*split_w shards [B, F*(Hg/split_h)*(Wg/split_w), ...];
    rank ih*split_w + iw holds block (ih, iw) of every frame.  Pinned:
    hand-enumerated fixtures, reduction to ``tile`` for one-band splits, round
    trip with gather_2d."""
    F, Hg, Wg = grid
    sh, sw = split
    x = np.ascontiguousarray(x)
    B, T = x.shape[:2]
    if T != F * Hg * Wg:
        raise ValueError("token count does not match the grid")
    if Hg % sh or Wg % sw:
        raise SplitError(f"grid {Hg}x{Wg} is not divisible by the split {sh}x{sw}")
    Tl = F * (Hg // sh) * (Wg // sw)
    shards = [np.empty((B, Tl) + x.shape[2:], dtype=x.dtype) for _ in range(sh * sw)]
    rc = _L().oracle_tile_2d(_p(x), _ptr_array(shards), B, F, Hg, Wg, sh, sw, _row_bytes(x, 2))
    if rc:
        raise SplitError("tile_2d failed")
    return shards


def gather_2d(shards, grid, split) -> np.ndarray:
    """Inverse of tile_2d: shards -> [B, F*Hg*Wg, ...]."""
    F, Hg, Wg = grid
    sh, sw = split
    if len(shards) != sh * sw:
        raise ValueError("one shard per rank of the split")
    if Hg % sh or Wg % sw:
        raise SplitError(f"grid {Hg}x{Wg} is not divisible by the split {sh}x{sw}")
    shards = [np.ascontiguousarray(s) for s in shards]
    B = shards[0].shape[0]
    out = np.empty((B, F * Hg * Wg) + shards[0].shape[2:], dtype=shards[0].dtype)
    rc = _L().oracle_gather_2d(_ptr_array(shards), _p(out), B, F, Hg, Wg, sh, sw, _row_bytes(shards[0], 2))
    if rc:
        raise SplitError("gather_2d failed")
    return out


def sm_rotation_counts(n_sm: int, W: int):
    """#SMs serving each rank when SM i writes rank i % W.  Pinned: the page's
    132-SM / 8-GPU example."""
    counts = np.zeros(W, dtype=np.int32)
    _L().oracle_sm_rotation_counts(n_sm, W, _p(counts))
    return [int(c) for c in counts]


# ---------------------------------------------------------------- attention
def _f32(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:  # bf16 bit patterns: widen exactly
        return (x.astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(x, dtype=np.float32)


def attention(q, k, v, mask_kind: int = MASK_NONE, mask=None, scale: float | None = None,
              threads: int | None = None) -> np.ndarray:
    """Plain softmax attention, fp64 accumulation, [B,Tq,H,D] -> float64.

    Pinned: closed-form weights, two-key logistic case, identity mask, constant
    V, pad-row mean, and torch's fp64 scaled_dot_product_attention."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Tq, H, D = q.shape
    Tk = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    m = None
    if mask_kind != MASK_NONE:
        m = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
    o = np.empty((B, Tq, H, D), dtype=np.float64)
    rc = _L().oracle_attention(_p(q), _p(k), _p(v), _p(o), B, Tq, Tk, H, D, mask_kind,
                               _p(m) if m is not None else None, float(scale),
                               threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_attention failed ({rc})")
    return o


def attention_rows(q, k, v, rows, mask_kind: int = MASK_NONE, mask=None,
                   scale: float | None = None, threads: int | None = None) -> np.ndarray:
    """Attention for selected (b, q, h) rows only -> [n_rows, D] float64."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Tq, H, D = q.shape
    Tk = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    m = None
    if mask_kind != MASK_NONE:
        m = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
    o = np.empty((rows.shape[0], D), dtype=np.float64)
    rc = _L().oracle_attention_rows(_p(q), _p(k), _p(v), _p(o), B, Tq, Tk, H, D, mask_kind,
                                    _p(m) if m is not None else None, float(scale), _p(rows),
                                    rows.shape[0], threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_attention_rows failed ({rc})")
    return o


# ---------------------------------------------------------------- the whole step
def sp_step(q, k, v, W: int, user_mask=None, scale: float | None = None,
            threads: int | None = None, return_stages: bool = False):
    """The sharded step built only from the routines above, in the pages' order:
    pad -> mask -> partition/tile -> send_recv_heads -> per-rank attention on the
    local heads -> gather_heads -> gather_output -> unpad.

    Self-attention: q, k, v are [B,T,H,D].  Returns float64 [B,T,H,D].
    Pinned: equals unsharded ``attention`` exactly (the correctness paragraph)."""
    B, T, H, D = q.shape
    if H % W:
        raise ValueError("H is not divisible by world_size")
    T_pad = padded_len(T, W)
    partition(T_pad, W)
    stages = {}
    if user_mask is None:
        mask = pad_mask_key(T, T_pad)
        kind = MASK_KEY
        mask_arg = mask.reshape(T_pad)
    else:
        mask = pad_mask_user(user_mask, T_pad)
        kind = MASK_FULL
        mask_arg = mask
    sharded = {}
    for name, x in (("q", q), ("k", k), ("v", v)):
        xp = pad(x, T_pad)
        shards = tile(xp, W)
        sharded[name] = send_recv_heads(shards)
        stages[name + "_pad"], stages[name + "_shards"] = xp, shards
        stages[name + "_heads"] = sharded[name]
    o_heads = []
    for r in range(W):
        o_heads.append(attention(sharded["q"][r], sharded["k"][r], sharded["v"][r], kind, mask_arg,
                                 scale, threads))
    o_shards = gather_heads(o_heads)
    o = gather_output(o_shards, W * (T_pad // W))
    o = unpad(o, T)
    stages.update(mask=mask, o_heads=o_heads, o_shards=o_shards)
    return (o, stages) if return_stages else o


def sp_step_2d(q, k, v, grid, W: int, scale: float | None = None, threads: int | None = None):
    """The sharded step with the 2-D spatial split in place of pad + tile:
    tile_2d -> send_recv_heads -> per-rank attention -> gather_heads ->
    gather_2d.  No padding (the split must divide the grid), no mask.
    Self-attention on [B, F*Hg*Wg, H, D]; returns float64.  Pinned: equals
    unsharded ``attention`` up to the order of the key sum."""
    B, T, H, D = q.shape
    if H % W:
        raise ValueError("H is not divisible by world_size")
    split = optimal_split(W)
    heads = {n: send_recv_heads(tile_2d(x, grid, split)) for n, x in (("q", q), ("k", k), ("v", v))}
    o_heads = [attention(heads["q"][r], heads["k"][r], heads["v"][r], MASK_NONE, None, scale, threads)
               for r in range(W)]
    return gather_2d(gather_heads(o_heads), grid, split)
