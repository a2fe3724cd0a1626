"""The whole sequence-parallel step (pad -> tile -> send_recv_heads ->
attention -> gather_heads -> gather_output) on the five workloads at their
full sizes, through the C ABI, against the oracle: every output row for the
small workloads, a strided sample of rows (exact per row: rows are
independent) for the large ones.  Plus the correctness paragraph's claim in
its strongest form: the sharded run equals the same kernels on the unpadded,
unsharded tensors bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import sequence_video_dit_gb300 as sp
import workloads
from gpu_helpers import BF16_TOL, f32_np, max_abs, tol_for

pytestmark = pytest.mark.gpu


def _inputs(wl):
    inp = workloads.make_inputs(wl)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v")}
    um = inp["user_mask"]
    return inp, dev, (um.cuda() if um is not None else None)


def _sample_rows(B, Tq, H, n, seed):
    rng = np.random.default_rng(seed)
    qs = np.unique(np.concatenate([[0, Tq - 1], rng.integers(0, Tq, n)]))
    rows = [(b, int(q), int(rng.integers(0, H))) for b in range(B) for q in qs]
    rows += [(0, int(Tq - 1), h) for h in range(H)] + [(B - 1, 0, h) for h in range(H)]
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_step_small_workloads_every_row(name):
    wl = workloads.get(name)
    inp, dev, um = _inputs(wl)
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask)
    out = f32_np(step(dev["q"], dev["k"], dev["v"], user_mask=um))
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(step.ws_exchange)[0] == 0
    assert sp.sp_workspace_status(step.ws_attn)[0] == 0
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    if um is None:
        ref = oracle.attention(q, k, v)
    else:
        ref = oracle.attention(q, k, v, oracle.MASK_FULL, inp["user_mask"].numpy())
    assert out.shape == ref.shape
    assert max_abs(out, ref) <= tol_for(wl.torch_dtype)
    # the device mask equals the oracle's extension of the user mask
    if um is not None:
        assert np.array_equal(step.mask.cpu().numpy(),
                              oracle.pad_mask_user(inp["user_mask"].numpy(), step.T_pad))


@pytest.mark.parametrize("name,nsample", [("c3", 512), ("c4", 256), ("c5", 192)])
def test_step_large_workloads_sampled_rows(name, nsample):
    wl = workloads.get(name)
    inp, dev, _ = _inputs(wl)
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq)
    out = f32_np(step(dev["q"], dev["k"], dev["v"]))
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(step.ws_exchange)[0] == 0
    assert sp.sp_workspace_status(step.ws_attn)[0] == 0
    assert np.isfinite(out).all()
    rows = _sample_rows(wl.B, wl.q_len, wl.H, nsample, wl.seed)
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    ref = oracle.attention_rows(q, k, v, rows)
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert max_abs(got, ref) <= tol_for(wl.torch_dtype)


@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
def test_sharded_equals_unsharded_bitwise(name):
    # Same kernels on the original tensors, one rank, every head, no padding:
    # key tiles start at 0 in both runs and masked keys get p = 0 exactly, so
    # every floating-point operation is the same.
    wl = workloads.get(name)
    inp, dev, um = _inputs(wl)
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask)
    out_sp = step(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    out_1 = torch.empty_like(out_sp)
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(1, wl.B, wl.T, wl.T, wl.H, wl.D, wl.torch_dtype))
    if um is None:
        sp.sp_attention([dev["q"]], [dev["k"]], [dev["v"]], [out_1], ws)
    else:
        sp.sp_attention([dev["q"]], [dev["k"]], [dev["v"]], [out_1], ws, sp.SP_MASK_FULL, um)
    torch.cuda.synchronize()
    assert torch.equal(out_sp.view(torch.int16), out_1.view(torch.int16))


def test_pad_query_rows_are_finite_and_match_the_mean_of_v():
    # Pad rows have a zero query and see every real key, so their output is
    # the mean of V over the real keys (closed form).
    wl = workloads.get("c3")
    inp, dev, _ = _inputs(wl)
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask)
    step(dev["q"], dev["k"], dev["v"])
    torch.cuda.synchronize()
    vbar = inp["v"].double().mean(dim=1).numpy()  # [B,H,D]
    Hl = step.Hl
    for r in range(wl.W):
        pad_rows = f32_np(step.o_heads[r][:, wl.T:])  # [B, T_pad-T, Hl, D]
        assert np.isfinite(pad_rows).all()
        for t in range(pad_rows.shape[1]):
            assert max_abs(pad_rows[:, t], vbar[:, r * Hl:(r + 1) * Hl]) <= 2e-2


def test_step_is_repeatable():
    wl = workloads.get("c2")
    _, dev, um = _inputs(wl)
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask)
    a = step(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    b = step(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_fused_step_equals_staged_step_bitwise(name):
    # The fused exchange entry points move the same bytes to the same places,
    # so the whole step gives the same output bit for bit.
    wl = workloads.get(name)
    inp, dev, um = _inputs(wl)
    staged = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq)
    fused = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq, fused=True)
    a = staged(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    b = fused(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(fused.ws_exchange)[0] == 0
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("W,B,T,Tkv,H,D,dtype,fused", [
    (2, 2, 37, 20, 4, 32, torch.float32, False),     # CUDA-core path, ragged pad
    (8, 1, 6149, 1001, 32, 128, torch.bfloat16, False),  # video 6149 tokens x audio 1001
    (8, 1, 6149, 1001, 32, 128, torch.bfloat16, True),
    (4, 2, 1001, 250, 8, 64, torch.bfloat16, True),
])
def test_small_kv_cross_attention(W, B, T, Tkv, H, D, dtype, fused):
    # Video queries (token-sharded, exchanged) attend a small audio K/V that
    # every rank holds whole and slices by head in place.
    wl = workloads.make_custom("a2v", W=W, B=B, T=Tkv, H=H, D=D, dtype="f32" if dtype == torch.float32 else "bf16",
                               Tq=T, index=200 + T % 97)
    inp = workloads.make_inputs(wl)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v")}
    step = sp.SPStep(W, B, T, H, D, dtype=dtype, Tkv=Tkv, fused=fused)
    out = f32_np(step(dev["q"], dev["k"], dev["v"]))
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(step.ws_exchange)[0] == 0
    assert sp.sp_workspace_status(step.ws_attn)[0] == 0
    assert out.shape == (B, T, H, D) and np.isfinite(out).all()
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    if T * Tkv * H * B <= 1_000_000:
        ref = oracle.attention(q, k, v)
        assert max_abs(out, ref) <= tol_for(dtype)
    else:
        rows = _sample_rows(B, T, H, 256, wl.seed)
        ref = oracle.attention_rows(q, k, v, rows)
        assert max_abs(out[rows[:, 0], rows[:, 1], rows[:, 2]], ref) <= tol_for(dtype)


@pytest.mark.parametrize("W,B,grid,H,D,dtype,nsample", [
    (6, 2, (2, 4, 6), 12, 32, torch.float32, None),      # CUDA-core path, every row
    (8, 1, (16, 24, 16), 32, 128, torch.bfloat16, 384),  # 6144 video tokens, blocks 12x4
])
def test_step_with_2d_spatial_split(W, B, grid, H, D, dtype, nsample):
    # The 2-D split permutes which tokens a rank contributes; after the head
    # exchange every rank still sees every key, so the step is plain attention.
    T = grid[0] * grid[1] * grid[2]
    wl = workloads.make_custom("grid2d", W=W, B=B, T=T, H=H, D=D, dtype="f32" if dtype == torch.float32 else "bf16",
                               index=300 + W)
    inp = workloads.make_inputs(wl)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v")}
    step = sp.SPStep(W, B, T, H, D, dtype=dtype, grid=grid)
    out = f32_np(step(dev["q"], dev["k"], dev["v"]))
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(step.ws_exchange)[0] == 0
    assert sp.sp_workspace_status(step.ws_attn)[0] == 0
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    if nsample is None:
        assert max_abs(out, oracle.attention(q, k, v)) <= tol_for(dtype)
    else:
        rows = _sample_rows(B, T, H, nsample, wl.seed)
        ref = oracle.attention_rows(q, k, v, rows)
        assert max_abs(out[rows[:, 0], rows[:, 1], rows[:, 2]], ref) <= tol_for(dtype)


def test_2d_split_rejects_an_indivisible_grid():
    with pytest.raises(ValueError):
        sp.SPStep(8, 1, 1 * 5 * 8, 8, 64, grid=(1, 5, 8))  # 5 patch rows, split 2x4


def _direct_cases():
    c4 = workloads.get("c4")
    video = workloads.make_custom("video6144", W=8, B=1, T=6144, H=32, D=128, index=400)
    padded = workloads.make_custom("video6140", W=8, B=1, T=6140, H=32, D=128, index=401)
    return [
        ("c4", c4, dict(Tq=c4.Tq), True),
        ("video6144", video, {}, True),
        ("video6140-padded", padded, {}, True),
        ("video6144-audio1001", workloads.make_custom("a2v", W=8, B=1, T=1001, H=32, D=128, Tq=6144, index=402),
         "kv_small", True),
        ("grid16x24x16", video, dict(grid=(16, 24, 16)), False),
    ]


@pytest.mark.parametrize("case", range(5))
@pytest.mark.parametrize("fused", [False, True])
def test_direct_step_equals_staged_step_bitwise(case, fused):
    name, wl, kw, fusable = _direct_cases()[case]
    if fused and not fusable:
        pytest.skip("in-place shards need contiguous token ranges (the 2-D split copies)")
    inp = workloads.make_inputs(wl)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v")}
    if kw == "kv_small":  # the workload's query is the sharded video, its T the audio keys
        T, kw = wl.q_len, dict(Tkv=wl.T)
    else:
        T = wl.T
    staged = sp.SPStep(wl.W, wl.B, T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, **kw)
    direct = sp.SPStep(wl.W, wl.B, T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, direct=True, fused=fused, **kw)
    a = staged(dev["q"], dev["k"], dev["v"]).clone()
    b = direct(dev["q"], dev["k"], dev["v"]).clone()
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(direct.ws_attn)[0] == 0
    assert direct.n_exchange_launches() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
@pytest.mark.parametrize("fused", [False, True])
def test_direct_step_with_ragged_shards(name, fused):
    # Shards that are not whole 128-row tiles (c2: 251 tokens, c3: 769, c5:
    # 6145; T % W != 0, so with fused=True the last shard view is short): the
    # attention visits each shard's whole tiles, then one tile gathering the
    # leftover rows.  Against the oracle (all rows of c2, sampled rows of
    # c3 / c5 over every head) and, at tolerance, against the staged step.
    wl = workloads.get(name)
    inp, dev, um = _inputs(wl)
    direct = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, direct=True, fused=fused)
    got = direct(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(direct.ws_attn)[0] == 0
    assert direct.n_exchange_launches() == 0
    got = f32_np(got)
    assert np.isfinite(got).all()
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    if name == "c2":
        ref = oracle.attention(q, k, v, oracle.MASK_FULL, inp["user_mask"].numpy())
        assert max_abs(got, ref) <= BF16_TOL
    else:
        Tl = -(-wl.T // wl.W)
        rows = np.array([(0, t, h) for s in range(wl.W) for t in (s * Tl, min((s + 1) * Tl, wl.T) - 1)
                         for h in (0, 13, wl.H - 1)] + [(0, wl.T - 1 - i, i) for i in range(4)], dtype=np.int64)
        ref = oracle.attention_rows(q, k, v, rows)
        assert max_abs(got[rows[:, 0], rows[:, 1], rows[:, 2]], ref) <= BF16_TOL
    del direct
    staged = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask)
    ref2 = f32_np(staged(dev["q"], dev["k"], dev["v"], user_mask=um))
    assert max_abs(got, ref2) <= BF16_TOL


@pytest.mark.parametrize("name,kw", [("c1", {}), ("c2", {}), ("c3", {}), ("c3", dict(fused=True)),
                                     ("c4", dict(fused=True, direct=True))])
def test_captured_step_replays_the_eager_step_bitwise(name, kw):
    # The whole step as one CUDA graph: same bytes as the eager step, on the
    # captured inputs and again after new inputs are copied into them.
    wl = workloads.get(name)
    inp, dev, um = _inputs(wl)
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq, **kw)
    eager = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq, **kw)
    g = step.capture(dev["q"], dev["k"], dev["v"], user_mask=um)
    a = g.replay().clone()
    b = eager(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    new = workloads.make_inputs(wl, seed=wl.seed + 77)
    for n in ("q", "k", "v"):
        dev[n].copy_(new[n])
    a = g.replay().clone()
    b = eager(dev["q"], dev["k"], dev["v"], user_mask=um).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert sp.sp_workspace_status(step.ws_exchange)[0] == 0
    assert sp.sp_workspace_status(step.ws_attn)[0] == 0


@pytest.mark.parametrize("B,T,kw", [(1, 0, {}), (0, 37, {}), (2, 0, dict(fused=True)), (1, 0, dict(Tq=5)),
                                     (1, 0, dict(direct=True)), (0, 256, dict(direct=True, fused=True)),
                                     (1, 1, {})])
def test_degenerate_sizes(B, T, kw):
    # Empty batches, empty sequences and a single token pass through every
    # stage without a launch error; a single token equals its own value row.
    W, H, D = 2, 4, 64
    step = sp.SPStep(W, B, T, H, D, dtype=torch.bfloat16, **kw)
    g = torch.Generator().manual_seed(T + B)
    q = torch.randn(B, kw.get("Tq", T), H, D, generator=g).bfloat16().cuda()
    k = torch.randn(B, T, H, D, generator=g).bfloat16().cuda()
    v = torch.randn(B, T, H, D, generator=g).bfloat16().cuda()
    out = step(q, k, v)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (B, kw.get("Tq", T), H, D)
    assert sp.sp_workspace_status(step.ws_exchange)[0] == 0
    if B and T == 1 and "Tq" not in kw:
        assert torch.equal(out.view(torch.int16), v.view(torch.int16))  # softmax over one key is exactly 1
    if B and T == 0 and "Tq" in kw:
        assert (out.float() == 0).all()  # no keys: rows are 0


def test_empty_layout_calls():
    W, H, D = 4, 8, 16
    ws = sp.new_workspace()
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    sp.sp_pad(e(0, 5, H, D), e(0, 8, H, D))
    sp.sp_tile(e(1, 0, H, D), [e(1, 0, H, D) for _ in range(W)])
    sp.sp_send_recv_heads([e(1, 0, H, D) for _ in range(W)], [e(1, 0, H // W, D) for _ in range(W)], ws)
    sp.sp_gather_heads([e(1, 0, H // W, D) for _ in range(W)], [e(1, 0, H, D) for _ in range(W)], ws)
    sp.sp_pad_send_heads(e(1, 0, H, D), [e(1, 0, H // W, D) for _ in range(W)], ws)
    sp.sp_gather_output([e(2, 0, H, D) for _ in range(W)], e(2, 0, H, D))
    sp.sp_unpad(e(0, 4, H, D), e(0, 3, H, D))
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
