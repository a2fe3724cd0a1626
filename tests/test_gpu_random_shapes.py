"""Seeded sweeps of random shapes through every path, against the oracle:
the layout chain and the fused exchange (bit-exact), the attention on both
kernels (self and cross lengths, every mask kind), the in-place attention
with one sharded operand, and the whole step in its staged, fused and
in-place forms.  The shapes are drawn once from fixed generators, so a
failing case is reproducible from its parameters."""
import numpy as np
import pytest
import torch

import oracle
import sequence_video_dit_gb300 as sp
import test_gpu_attention as attn_tests
import test_gpu_layout as layout_tests
from gpu_helpers import BF16_TOL, f32_np, max_abs

pytestmark = pytest.mark.gpu

KINDS = [sp.SP_MASK_NONE, sp.SP_MASK_KEY, sp.SP_MASK_FULL]


def _shapes(seed, n, draw):
    rng = np.random.default_rng(seed)
    return [draw(rng) for _ in range(n)]


def _layout_shape(rng):
    W = int(rng.choice([1, 2, 3, 4, 8]))
    dtype = [torch.float32, torch.bfloat16][int(rng.integers(0, 2))]
    return (int(rng.integers(1, 4)), int(rng.integers(1, 3000)), W, W * int(rng.integers(1, 5)),
            int(rng.choice([3, 4, 8, 16, 32, 64, 128])), dtype)


LAYOUT = _shapes(11, 10, _layout_shape)


@pytest.mark.parametrize("B,T,W,H,D,dtype", LAYOUT)
def test_layout_chain_random_shapes(B, T, W, H, D, dtype):
    layout_tests.test_layout_chain_bit_exact(B, T, W, H, D, dtype)


@pytest.mark.parametrize("B,T,W,H,D,dtype", LAYOUT)
def test_fused_exchange_random_shapes(B, T, W, H, D, dtype):
    layout_tests.test_fused_exchange_bit_exact(B, T, W, H, D, dtype)


def _attention_shape(rng):
    kind = KINDS[int(rng.integers(0, 3))]
    W, B, Hl = int(rng.choice([1, 2, 4])), int(rng.integers(1, 3)), int(rng.integers(1, 3))
    Tq = int(rng.integers(1, 700))
    Tk = Tq if rng.random() < 0.5 else int(rng.integers(1, 900))
    path = int(rng.integers(0, 3))
    if path == 0:    # tensor cores
        D, dtype = int(rng.choice([64, 128])), torch.bfloat16
    elif path == 1:  # CUDA cores, bf16 at other head dims
        D, dtype = int(rng.choice([32, 96, 160])), torch.bfloat16
    else:            # CUDA cores, fp32
        D, dtype = int(rng.choice([8, 16, 48, 80, 200])), torch.float32
    return (W, B, Tq, Tk, Hl, D, dtype, kind)


@pytest.mark.parametrize("W,B,Tq,Tk,Hl,D,dtype,mask_kind", _shapes(12, 12, _attention_shape))
def test_attention_random_shapes(W, B, Tq, Tk, Hl, D, dtype, mask_kind):
    attn_tests._run(W, B, Tq, Tk, Hl, D, dtype, mask_kind, seed=31 * Tq + Tk)


def _one_operand_shape(rng):
    W = int(rng.choice([2, 4, 8]))
    return (int(rng.choice([sp.SP_SHARD_KV, sp.SP_SHARD_Q])), W, int(rng.integers(1, 3)),
            int(rng.integers(1, 1500)), int(rng.integers(1, 600)), W * int(rng.integers(1, 3)),
            int(rng.choice([64, 128])), KINDS[int(rng.integers(0, 2))])


@pytest.mark.parametrize("flags,W,B,T_sh,T_rep,H,D,mask_kind", _shapes(14, 8, _one_operand_shape))
def test_one_sharded_operand_random_shapes(flags, W, B, T_sh, T_rep, H, D, mask_kind):
    # K/V (or Q and O) as W token shards of the caller's tensor; the other
    # operand per rank, sliced by head
    g = torch.Generator().manual_seed(7 * T_sh + T_rep)
    Tq, Tk = (T_rep, T_sh) if flags == sp.SP_SHARD_KV else (T_sh, T_rep)
    q = torch.randn(B, Tq, H, D, generator=g).bfloat16().cuda()
    k, v = (torch.randn(B, Tk, H, D, generator=g).bfloat16().cuda() for _ in range(2))
    mask = None
    if mask_kind == sp.SP_MASK_KEY:
        mask = (torch.rand(Tk, generator=g) < 0.85).to(torch.uint8)
        mask[0] = 1
    Hl = H // W
    Tl = -(-T_sh // W)
    views = lambda x: [x[:, min(s * Tl, T_sh):min((s + 1) * Tl, T_sh)] for s in range(W)]  # noqa: E731
    heads = lambda x: [x[:, :, r * Hl:(r + 1) * Hl] for r in range(W)]  # noqa: E731
    out = torch.full((B, Tq, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16))
    m = None if mask is None else mask.cuda()
    if flags == sp.SP_SHARD_KV:
        sp.sp_attention_shards(heads(q), views(k), views(v), heads(out), ws, flags, mask_kind, m)
    else:
        sp.sp_attention_shards(views(q), heads(k), heads(v), views(out), ws, flags, mask_kind, m)
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    ref = oracle.attention(f32_np(q), f32_np(k), f32_np(v), mask_kind, None if mask is None else mask.numpy())
    assert max_abs(f32_np(out), ref) <= BF16_TOL


def _step_shape(rng):
    W = int(rng.choice([2, 4, 8]))
    return (W, int(rng.integers(1, 3)), int(rng.integers(1, 900)), W * int(rng.integers(1, 3)),
            int(rng.choice([64, 128])), ["key", "user"][int(rng.integers(0, 2))],
            ["staged", "fused", "direct"][int(rng.integers(0, 3))])


@pytest.mark.parametrize("W,B,T,H,D,mask,variant", _shapes(13, 9, _step_shape))
def test_step_random_shapes(W, B, T, H, D, mask, variant):
    g = torch.Generator().manual_seed(5 * T + W)
    q, k, v = (torch.randn(B, T, H, D, generator=g).bfloat16() for _ in range(3))
    um = None
    if mask == "user":
        um = (torch.rand(B, T, T, generator=g) < 0.3).to(torch.uint8)
        for b in range(B):
            um[b, torch.arange(T), torch.arange(T)] = 1
    step = sp.SPStep(W, B, T, H, D, dtype=torch.bfloat16, mask=mask, fused=variant != "staged",
                     direct=variant == "direct")
    out = f32_np(step(q.cuda(), k.cuda(), v.cuda(), user_mask=None if um is None else um.cuda()))
    torch.cuda.synchronize()
    for ws in (step.ws_exchange, step.ws_attn):
        assert sp.sp_workspace_status(ws)[0] == 0
    if um is None:
        ref = oracle.attention(f32_np(q), f32_np(k), f32_np(v))
    else:
        ref = oracle.attention(f32_np(q), f32_np(k), f32_np(v), oracle.MASK_FULL, um.numpy())
    assert out.shape == ref.shape
    assert max_abs(out, ref) <= BF16_TOL


def _split_shape(rng):
    # shapes that cut work items into key pieces: a short query (fewer items
    # than SMs, >= 8 key tiles) or a long one whose last wave is partial
    kind = KINDS[int(rng.integers(0, 3))]
    D = int(rng.choice([64, 128]))
    if rng.random() < 0.5:
        W, Hl = int(rng.choice([1, 2, 4])), int(rng.integers(1, 3))
        return (W, int(rng.integers(1, 3)), int(rng.integers(1, 400)), int(rng.integers(1024, 5000)), Hl, D, kind)
    return (8, 1, int(rng.integers(2500, 5000)), int(rng.integers(1024, 3000)), 4, D, kind)


@pytest.mark.parametrize("W,B,Tq,Tk,Hl,D,mask_kind", _shapes(15, 8, _split_shape))
def test_split_attention_random_shapes(W, B, Tq, Tk, Hl, D, mask_kind):
    g = torch.Generator().manual_seed(3 * Tq + Tk)
    mk = lambda T: [torch.randn(B, T, Hl, D, generator=g).bfloat16().cuda() for _ in range(W)]  # noqa: E731
    q, k, v = mk(Tq), mk(Tk), mk(Tk)
    o = [torch.full_like(x, float("nan")) for x in q]
    mask = None
    if mask_kind == sp.SP_MASK_KEY:
        mask = (torch.rand(Tk, generator=g) < 0.8).to(torch.uint8)
        mask[0] = 1
    elif mask_kind == sp.SP_MASK_FULL:
        mask = (torch.rand(B, Tq, Tk, generator=g) < 0.3).to(torch.uint8)
        mask[:, :, 0] = 1
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16))
    sp.sp_attention(q, k, v, o, ws, mask_kind, None if mask is None else mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    rng = np.random.default_rng(Tq + Tk)
    m_np = None if mask is None else mask.numpy()
    for r in sorted({0, W - 1}):
        qs = np.unique(np.concatenate([[0, Tq - 1], rng.integers(0, Tq, 24)]))
        rows = np.array([(b, int(t), h) for b in range(B) for h in range(Hl) for t in qs], dtype=np.int64)
        ref = oracle.attention_rows(f32_np(q[r]), f32_np(k[r]), f32_np(v[r]), rows, mask_kind, m_np)
        got = f32_np(o[r])[rows[:, 0], rows[:, 1], rows[:, 2]]
        assert np.isfinite(got).all()
        assert max_abs(got, ref) <= BF16_TOL, f"rank {r}"


def _grid_shape(rng):
    # a latent grid the W-way split (the factor pair closest to a square) divides
    W = int(rng.choice([1, 2, 3, 4, 6, 8]))
    sh, sw = oracle.optimal_split(W)
    grid = (int(rng.integers(1, 5)), sh * int(rng.integers(1, 7)), sw * int(rng.integers(1, 7)))
    dtype = [torch.float32, torch.bfloat16][int(rng.integers(0, 2))]
    return (int(rng.integers(1, 3)), grid, W, W * int(rng.integers(1, 3)), int(rng.choice([4, 8, 16, 64])), dtype)


@pytest.mark.parametrize("B,grid,W,H,D,dtype", _shapes(16, 8, _grid_shape))
def test_2d_split_random_shapes(B, grid, W, H, D, dtype):
    layout_tests.test_tile_2d_and_gather_2d_bit_exact(B, grid, W, H, D, dtype)
