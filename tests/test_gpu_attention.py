"""sp_attention vs the oracle (max-abs <= 1e-4 fp32, <= 2e-2 bf16), on the
tensor-core path (bf16, D = 64 / 128) and the CUDA-core path (fp32, other D),
across several tiles with ragged tails, all mask kinds, the strided
cross-attention query, the split-key pass, and the degenerate rows."""
import numpy as np
import pytest
import torch

import oracle
import sequence_video_dit_gb300 as sp
from gpu_helpers import f32_np, max_abs, tol_for

pytestmark = pytest.mark.gpu


def _mk(W, B, T, Hl, D, dtype, g, scale=1.0):
    return [(torch.randn(B, T, Hl, D, generator=g) * scale).to(dtype).cuda() for _ in range(W)]


def _run(W, B, Tq, Tk, Hl, D, dtype, mask_kind, seed=0, key_keep=0.8, full_keep=0.3):
    g = torch.Generator().manual_seed(seed)
    q = _mk(W, B, Tq, Hl, D, dtype, g)
    k = _mk(W, B, Tk, Hl, D, dtype, g)
    v = _mk(W, B, Tk, Hl, D, dtype, g)
    o = [torch.full((B, Tq, Hl, D), float("nan"), dtype=dtype, device="cuda") for _ in range(W)]
    mask = None
    if mask_kind == sp.SP_MASK_KEY:
        mask = (torch.rand(Tk, generator=g) < key_keep).to(torch.uint8)
        mask[0] = 1
    elif mask_kind == sp.SP_MASK_FULL:
        mask = (torch.rand(B, Tq, Tk, generator=g) < full_keep).to(torch.uint8)
        for b in range(B):
            n = min(Tq, Tk)
            mask[b, torch.arange(n), torch.arange(n)] = 1
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, dtype))
    sp.sp_attention(q, k, v, o, ws, mask_kind, None if mask is None else mask.cuda())
    torch.cuda.synchronize()
    st, _, _ = sp.sp_workspace_status(ws)
    assert st == 0
    m_np = None if mask is None else mask.numpy()
    for r in range(W):
        ref = oracle.attention(f32_np(q[r]), f32_np(k[r]), f32_np(v[r]), mask_kind, m_np)
        got = f32_np(o[r])
        assert np.isfinite(got).all()
        err = max_abs(got, ref)
        assert err <= tol_for(dtype), f"rank {r}: max-abs {err}"
    return q, k, v, o, mask


@pytest.mark.parametrize("W,B,Tq,Tk,Hl,D,mask_kind", [
    (2, 1, 300, 300, 2, 128, sp.SP_MASK_KEY),     # 2 query pairs (last ragged), 3 key tiles (ragged)
    (2, 2, 261, 261, 1, 64, sp.SP_MASK_FULL),     # user-mask kind, D = 64
    (1, 1, 1000, 517, 2, 128, sp.SP_MASK_NONE),   # Tq != Tk
    (4, 1, 128, 128, 1, 128, sp.SP_MASK_KEY),     # exactly one tile
    (1, 1, 7, 5, 3, 64, sp.SP_MASK_NONE),         # tiny, mostly out-of-range tile
    (1, 2, 1536, 1536, 1, 128, sp.SP_MASK_KEY),   # many key tiles -> lazy rescale path
])
def test_tensor_core_attention(W, B, Tq, Tk, Hl, D, mask_kind):
    _run(W, B, Tq, Tk, Hl, D, torch.bfloat16, mask_kind)


@pytest.mark.parametrize("W,B,Tq,Tk,Hl,D,dtype,mask_kind", [
    (2, 1, 38, 38, 2, 32, torch.float32, sp.SP_MASK_KEY),   # c1 shape
    (1, 2, 50, 70, 2, 96, torch.bfloat16, sp.SP_MASK_FULL),  # D without a tensor-core kernel
    (2, 1, 33, 40, 1, 256, torch.float32, sp.SP_MASK_NONE),
])
def test_cuda_core_attention(W, B, Tq, Tk, Hl, D, dtype, mask_kind):
    _run(W, B, Tq, Tk, Hl, D, dtype, mask_kind)


def test_misaligned_buffers_take_the_cuda_core_kernel():
    # bf16, D = 128, but every tensor starts 2 bytes past a 16-byte boundary:
    # TMA cannot address them, so the call runs on the CUDA-core kernel and
    # must still match the oracle
    W, B, T, Hl, D = 2, 1, 300, 2, 128
    g = torch.Generator().manual_seed(77)
    n = B * T * Hl * D

    def off(x):
        buf = torch.empty(n + 1, dtype=torch.bfloat16, device="cuda")
        view = buf[1:].view(B, T, Hl, D)
        view.copy_(x)
        return view

    q, k, v = ([off(t.cuda()) for t in _mk(W, B, T, Hl, D, torch.bfloat16, g)] for _ in range(3))
    o = [off(torch.full((B, T, Hl, D), float("nan"), dtype=torch.bfloat16)) for _ in range(W)]
    assert all(x.data_ptr() % 16 == 2 for x in q + k + v + o)
    mask = (torch.rand(T, generator=g) < 0.8).to(torch.uint8)
    mask[0] = 1
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, T, T, Hl, D, torch.bfloat16))
    sp.sp_attention(q, k, v, o, ws, sp.SP_MASK_KEY, mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    for r in range(W):
        ref = oracle.attention(f32_np(q[r]), f32_np(k[r]), f32_np(v[r]), oracle.MASK_KEY, mask.numpy())
        assert max_abs(f32_np(o[r]), ref) <= 2e-2, f"rank {r}"


def test_large_logits_rescale():
    # Scores spread over a wide range force the running max to move by more
    # than the lazy-rescale threshold many times.
    W, B, T, Hl, D = 1, 1, 1024, 1, 128
    g = torch.Generator().manual_seed(3)
    q = [(torch.randn(B, T, Hl, D, generator=g) * 3).bfloat16().cuda()]
    k = [(torch.randn(B, T, Hl, D, generator=g) * torch.linspace(0.1, 3, T).view(1, T, 1, 1)).bfloat16().cuda()]
    v = [torch.randn(B, T, Hl, D, generator=g).bfloat16().cuda()]
    o = [torch.empty_like(q[0])]
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, T, T, Hl, D, torch.bfloat16))
    sp.sp_attention(q, k, v, o, ws)
    ref = oracle.attention(f32_np(q[0]), f32_np(k[0]), f32_np(v[0]))
    assert max_abs(f32_np(o[0]), ref) <= 2e-2


def test_fully_masked_rows_are_zero():
    W, B, T, Hl, D = 1, 1, 200, 2, 128
    g = torch.Generator().manual_seed(4)
    q, k, v = (_mk(W, B, T, Hl, D, torch.bfloat16, g) for _ in range(3))
    mask = (torch.rand(B, T, T, generator=g) < 0.5).to(torch.uint8)
    mask[0, 5] = 0
    mask[0, 150] = 0
    o = [torch.full_like(q[0], float("nan"))]
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, T, T, Hl, D, torch.bfloat16))
    sp.sp_attention(q, k, v, o, ws, sp.SP_MASK_FULL, mask.cuda())
    got = f32_np(o[0])
    assert (got[0, 5] == 0).all() and (got[0, 150] == 0).all()
    ref = oracle.attention(f32_np(q[0]), f32_np(k[0]), f32_np(v[0]), oracle.MASK_FULL, mask.numpy())
    assert max_abs(got, ref) <= 2e-2


@pytest.mark.parametrize("Tq,Tk,H,W", [(250, 3000, 8, 2), (250, 24576 + 5, 32, 8), (17, 900, 4, 4)])
def test_cross_attention_strided_query_and_split(Tq, Tk, H, W):
    # The small query modality stays whole on every rank; rank r reads heads
    # [r*Hl, (r+1)*Hl) in place and writes them into the shared output.
    B, D = 1, 128
    Hl = H // W
    g = torch.Generator().manual_seed(Tq + Tk)
    Q = torch.randn(B, Tq, H, D, generator=g).bfloat16().cuda()
    k = _mk(W, B, Tk, Hl, D, torch.bfloat16, g)
    v = _mk(W, B, Tk, Hl, D, torch.bfloat16, g)
    key = torch.ones(Tk, dtype=torch.uint8)
    key[-5:] = 0  # a key padding tail
    out = torch.full((B, Tq, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    qv = [Q[:, :, r * Hl:(r + 1) * Hl] for r in range(W)]
    ov = [out[:, :, r * Hl:(r + 1) * Hl] for r in range(W)]
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16))
    sp.sp_attention(qv, k, v, ov, ws, sp.SP_MASK_KEY, key.cuda())
    got = f32_np(out)
    Qn = f32_np(Q)
    for r in range(W):
        ref = oracle.attention(np.ascontiguousarray(Qn[:, :, r * Hl:(r + 1) * Hl]), f32_np(k[r]), f32_np(v[r]),
                               oracle.MASK_KEY, key.numpy())
        assert max_abs(got[:, :, r * Hl:(r + 1) * Hl], ref) <= 2e-2


def test_split_and_unsplit_agree():
    # Same problem with and without the split-key workspace: both within tolerance.
    W, B, Tq, Tk, Hl, D = 2, 1, 250, 4096, 2, 128
    g = torch.Generator().manual_seed(9)
    q, k, v = _mk(W, B, Tq, Hl, D, torch.bfloat16, g), _mk(W, B, Tk, Hl, D, torch.bfloat16, g), \
        _mk(W, B, Tk, Hl, D, torch.bfloat16, g)
    o1 = [torch.empty_like(x) for x in q]
    o2 = [torch.empty_like(x) for x in q]
    need = sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16)
    assert need > sp.SP_WORKSPACE_HEADER_BYTES  # this shape splits the keys
    sp.sp_attention(q, k, v, o1, sp.new_workspace(need))
    sp.sp_attention(q, k, v, o2, sp.new_workspace())  # header only: no split
    for r in range(W):
        ref = oracle.attention(f32_np(q[r]), f32_np(k[r]), f32_np(v[r]))
        assert max_abs(f32_np(o1[r]), ref) <= 2e-2
        assert max_abs(f32_np(o2[r]), ref) <= 2e-2


def test_empty_keys_give_zero():
    W, B, Tq, Hl, D = 1, 1, 10, 1, 128
    q = [torch.randn(B, Tq, Hl, D, device="cuda").bfloat16()]
    k = [torch.empty(B, 0, Hl, D, dtype=torch.bfloat16, device="cuda")]
    o = [torch.full_like(q[0], float("nan"))]
    sp.sp_attention(q, k, k, o, sp.new_workspace())
    assert (o[0].float() == 0).all()


def test_attention_argument_errors():
    q = [torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16, device="cuda")]
    with pytest.raises(ValueError):
        sp.sp_attention(q, q, q, q, sp.new_workspace(), sp.SP_MASK_KEY, None)
    with pytest.raises(ValueError):
        sp.sp_attention(q * 9, q * 9, q * 9, q * 9, sp.new_workspace())  # W = 9 > SP_MAX_RANKS


@pytest.mark.parametrize("stall", [1, 4])
def test_bounded_wait_runs_out_and_the_context_survives(stall):
    # Fault made through the workspace's test word, nothing on the device
    # faults: the producer issues only stall - 1 K/V loads (1: none; 4: K0, V0,
    # K1, so the MMAs of the first key tile are in flight when the wait for V1
    # runs out).  The kernel must report SP_ERR_TIMEOUT, drain, free its TMEM
    # and exit; the next call on a cleared workspace must be exact again.
    W, B, Tq, Tk, Hl, D = 1, 1, 256, 512, 1, 128  # one CTA, four key tiles, no split
    g = torch.Generator().manual_seed(21)
    q, k, v = (_mk(W, B, T, Hl, D, torch.bfloat16, g) for T in (Tq, Tk, Tk))
    o = [torch.empty_like(q[0])]
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16))
    word = sp.SP_WORKSPACE_KV_STALL_OFFSET // 4
    ws.view(torch.int32)[word] = stall
    sp.sp_attention(q, k, v, o, ws)
    torch.cuda.synchronize()
    st, _, _ = sp.sp_workspace_status(ws, clear=True)
    assert st == sp.SP_ERR_TIMEOUT
    ws.view(torch.int32)[word] = 0
    sp.sp_attention(q, k, v, o, ws)
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    ref = oracle.attention(f32_np(q[0]), f32_np(k[0]), f32_np(v[0]))
    assert max_abs(f32_np(o[0]), ref) <= 2e-2


@pytest.mark.parametrize("W,B,T,Hl,D", [(8, 1, 3000, 4, 128),   # 384 items: the last 80 run as key pieces
                                        (8, 2, 2500, 4, 64)])   # 640 items: the last 32 run as key pieces
def test_last_wave_key_pieces(W, B, T, Hl, D):
    # With more work items than SMs, the items of the last, partial wave are
    # cut into key pieces and merged.  Work items are ordered (rank, batch,
    # head, query pair), so the pieced ones are the last ranks' last heads:
    # sample rows there and elsewhere against the oracle, per row exactly.
    g = torch.Generator().manual_seed(T + D)
    q, k, v = (_mk(W, B, T, Hl, D, torch.bfloat16, g) for _ in range(3))
    o = [torch.full_like(x, float("nan")) for x in q]
    mask = torch.ones(T, dtype=torch.uint8)
    mask[-9:] = 0
    need = sp.sp_attention_workspace_bytes(W, B, T, T, Hl, D, torch.bfloat16)
    assert need > sp.SP_WORKSPACE_HEADER_BYTES  # this shape pieces its last wave
    ws = sp.new_workspace(need)
    sp.sp_attention(q, k, v, o, ws, sp.SP_MASK_KEY, mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    rng = np.random.default_rng(T)
    for r in (0, W - 2, W - 1):
        qs = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 40)]))
        rows = np.array([(b, int(t), h) for b in range(B) for h in range(Hl) for t in qs], dtype=np.int64)
        ref = oracle.attention_rows(f32_np(q[r]), f32_np(k[r]), f32_np(v[r]), rows, oracle.MASK_KEY, mask.numpy())
        got = f32_np(o[r])[rows[:, 0], rows[:, 1], rows[:, 2]]
        assert np.isfinite(got).all()
        assert max_abs(got, ref) <= 2e-2, f"rank {r}"


@pytest.mark.parametrize("W,B,Tl,H,D,mask_kind", [
    (8, 1, 384, 32, 128, sp.SP_MASK_KEY),   # c4-like K/V shards, a query pair straddles two shards
    (4, 2, 256, 8, 64, sp.SP_MASK_FULL),    # user-mask kind, D = 64
    (2, 1, 128, 4, 128, sp.SP_MASK_NONE),   # one tile per shard
    (8, 1, 768, 32, 128, sp.SP_MASK_KEY),   # the 6144-token video: the last wave runs in key pieces
])
def test_attention_from_shards_is_the_attention_after_the_exchange(W, B, Tl, H, D, mask_kind):
    # The exchange fused into the attention: loading each tile from its source
    # shard must give exactly the bytes of sp_send_recv_heads + sp_attention
    # (+ sp_gather_heads for O in token-shard layout).
    g = torch.Generator().manual_seed(Tl + W)
    T = W * Tl
    mk = lambda: [torch.randn(B, Tl, H, D, generator=g).bfloat16().cuda() for _ in range(W)]  # noqa: E731
    qs, ks, vs = mk(), mk(), mk()
    mask = None
    if mask_kind == sp.SP_MASK_KEY:
        mask = (torch.rand(T, generator=g) < 0.9).to(torch.uint8)
        mask[0] = 1
        mask = mask.cuda()
    elif mask_kind == sp.SP_MASK_FULL:
        mask = (torch.rand(B, T, T, generator=g) < 0.3).to(torch.uint8)
        for b in range(B):
            mask[b, torch.arange(T), torch.arange(T)] = 1
        mask = mask.cuda()
    Hl = H // W
    wx = sp.new_workspace()
    heads = {}
    for n, x in (("q", qs), ("k", ks), ("v", vs)):
        heads[n] = [torch.empty(B, T, Hl, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
        sp.sp_send_recv_heads(x, heads[n], wx)
    o_heads = [torch.empty_like(x) for x in heads["q"]]
    need = sp.sp_attention_workspace_bytes(W, B, T, T, Hl, D, torch.bfloat16)
    sp.sp_attention(heads["q"], heads["k"], heads["v"], o_heads, sp.new_workspace(need), mask_kind, mask)
    o_ref = [torch.empty_like(x) for x in qs]
    sp.sp_gather_heads(o_heads, o_ref, wx)
    # everything from / to token shards
    o_sh = [torch.full_like(x, float("nan")) for x in qs]
    ws = sp.new_workspace(need)
    sp.sp_attention_shards(qs, ks, vs, o_sh, ws, sp.SP_SHARD_Q | sp.SP_SHARD_KV, mask_kind, mask)
    # K/V from shards only; Q and O per rank
    o_kv = [torch.full_like(x, float("nan")) for x in heads["q"]]
    sp.sp_attention_shards(heads["q"], ks, vs, o_kv, sp.new_workspace(need), sp.SP_SHARD_KV, mask_kind, mask)
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    for s in range(W):
        assert torch.equal(o_sh[s].view(torch.int16), o_ref[s].view(torch.int16)), f"shard {s}"
        assert torch.equal(o_kv[s].view(torch.int16), o_heads[s].view(torch.int16)), f"rank {s}"
    # and the values are attention: a few rows of rank 0 against the oracle
    rows = np.array([(0, 0, 0), (0, T - 1, Hl - 1), (B - 1, T // 2, 0)], dtype=np.int64)
    ref = oracle.attention_rows(f32_np(heads["q"][0]), f32_np(heads["k"][0]), f32_np(heads["v"][0]), rows,
                                mask_kind, None if mask is None else mask.cpu().numpy())
    got = f32_np(o_heads[0])[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert max_abs(got, ref) <= 2e-2


def test_attention_from_shards_refuses_what_it_cannot_do():
    W, B, H, D = 4, 1, 8, 128
    ws = sp.new_workspace()
    mk = lambda Tl, dt=torch.bfloat16: [torch.zeros(B, Tl, H, D, dtype=dt, device="cuda") for _ in range(W)]  # noqa
    with pytest.raises(ValueError):  # no tensor-core kernel for fp32
        x = mk(128, torch.float32)
        sp.sp_attention_shards(x, x, x, mk(128, torch.float32), ws, sp.SP_SHARD_Q | sp.SP_SHARD_KV)
    with pytest.raises(ValueError):  # shard 0 must hold ceil(T / W) rows
        x = mk(100)
        sp.sp_attention_shards(x, x, x, mk(100), ws, sp.SP_SHARD_Q | sp.SP_SHARD_KV, Tq=300, Tk=300)


RAGGED = [
    # W, B, T, H, D, mask_kind: shards of ceil(T / W) tokens that are not whole
    # 128-row tiles, the last shards short (T % W != 0) or empty (T < (W-1) Tl)
    (8, 1, 6149, 32, 128, sp.SP_MASK_NONE),   # c3 video: 769-token shards, last 764 (2 tail tiles)
    (8, 1, 6149, 32, 128, sp.SP_MASK_KEY),    # the same with a key mask over the real tokens
    (4, 2, 1001, 8, 64, sp.SP_MASK_FULL),     # c2 shape: 251-token shards, user mask, 4 tail tiles
    (8, 1, 300, 16, 128, sp.SP_MASK_NONE),    # 38-token shards: no whole tile at all
    (8, 2, 5, 8, 64, sp.SP_MASK_NONE),        # 1-token shards, shards 5..7 empty
    (2, 1, 1000, 4, 128, sp.SP_MASK_KEY),     # 500 = 3 whole tiles + 116 per shard
]


@pytest.mark.parametrize("W,B,T,H,D,mask_kind", RAGGED)
def test_attention_from_ragged_shards_matches_the_oracle(W, B, T, H, D, mask_kind):
    # The exchange fused into the attention for any shard length: every
    # operand is given as W views of the caller's [B, T, H, D] tensor (no
    # padding anywhere), each rank's heads are read from every shard and O is
    # written back in place.  Against plain attention on the unsharded tensors.
    g = torch.Generator().manual_seed(T * 7 + W)
    q, k, v = (torch.randn(B, T, H, D, generator=g).bfloat16().cuda() for _ in range(3))
    mask = None
    if mask_kind == sp.SP_MASK_KEY:
        mask = (torch.rand(T, generator=g) < 0.85).to(torch.uint8)
        mask[0] = 1
    elif mask_kind == sp.SP_MASK_FULL:
        mask = (torch.rand(B, T, T, generator=g) < 0.3).to(torch.uint8)
        for b in range(B):
            mask[b, torch.arange(T), torch.arange(T)] = 1
    Tl = -(-T // W)
    views = lambda x: [x[:, min(s * Tl, T):min((s + 1) * Tl, T)] for s in range(W)]  # noqa: E731
    out = torch.full((B, T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, T, T, H // W, D, torch.bfloat16))
    sp.sp_attention_shards(views(q), views(k), views(v), views(out), ws, sp.SP_SHARD_Q | sp.SP_SHARD_KV,
                           mask_kind, None if mask is None else mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    got = f32_np(out)
    assert np.isfinite(got).all()
    m_np = None if mask is None else mask.numpy()
    if T <= 1100:
        ref = oracle.attention(f32_np(q), f32_np(k), f32_np(v), mask_kind, m_np)
        assert max_abs(got, ref) <= 2e-2
    else:
        # every shard's first and last rows and rows in between, over every head
        rows = []
        for s in range(W):
            lo, hi = s * Tl, min((s + 1) * Tl, T) - 1
            for t in (lo, lo + 1, (lo + hi) // 2, hi - 1, hi):
                for h in range(0, H, 5):
                    rows.append((0, t, h))
        rows = np.array(rows, dtype=np.int64)
        ref = oracle.attention_rows(f32_np(q), f32_np(k), f32_np(v), rows, mask_kind, m_np)
        assert max_abs(got[rows[:, 0], rows[:, 1], rows[:, 2]], ref) <= 2e-2


def _random_ragged_shapes(n, seed=2024):
    # W, B, T, H, D, mask_kind drawn once from a fixed generator: shard lengths
    # ceil(T / W) with every mix of whole, partial (>= 64 leftover rows) and
    # gathered (< 64) tiles, short and empty last shards
    rng = np.random.default_rng(seed)
    kinds = [sp.SP_MASK_NONE, sp.SP_MASK_KEY, sp.SP_MASK_FULL]
    out = []
    for _ in range(n):
        W = int(rng.choice([2, 4, 8]))
        out.append((W, int(rng.integers(1, 3)), int(rng.integers(1, 1500)), W * int(rng.integers(1, 3)),
                    int(rng.choice([64, 128])), kinds[int(rng.integers(0, 3))]))
    return out


@pytest.mark.parametrize("W,B,T,H,D,mask_kind", _random_ragged_shapes(12))
def test_attention_from_ragged_shards_random_shapes(W, B, T, H, D, mask_kind):
    # The in-place attention on seeded random shapes, every row against the oracle.
    g = torch.Generator().manual_seed(T * 13 + W * 3 + D)
    q, k, v = (torch.randn(B, T, H, D, generator=g).bfloat16().cuda() for _ in range(3))
    mask = None
    if mask_kind == sp.SP_MASK_KEY:
        mask = (torch.rand(T, generator=g) < 0.8).to(torch.uint8)
        mask[0] = 1
    elif mask_kind == sp.SP_MASK_FULL:
        mask = (torch.rand(B, T, T, generator=g) < 0.4).to(torch.uint8)
        for b in range(B):
            mask[b, torch.arange(T), torch.arange(T)] = 1
    Tl = -(-T // W)
    views = lambda x: [x[:, min(s * Tl, T):min((s + 1) * Tl, T)] for s in range(W)]  # noqa: E731
    out = torch.full((B, T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, T, T, H // W, D, torch.bfloat16))
    sp.sp_attention_shards(views(q), views(k), views(v), views(out), ws, sp.SP_SHARD_Q | sp.SP_SHARD_KV,
                           mask_kind, None if mask is None else mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    got = f32_np(out)
    ref = oracle.attention(f32_np(q), f32_np(k), f32_np(v), mask_kind, None if mask is None else mask.numpy())
    assert max_abs(got, ref) <= 2e-2


@pytest.mark.parametrize("flags", [sp.SP_SHARD_KV, sp.SP_SHARD_Q])
def test_ragged_shards_of_one_operand(flags):
    # Only K/V (the small-query cross-attention) or only Q (a small replicated
    # K/V) comes as ragged shards; the other operand is per rank, sliced by head.
    W, B, H, D = 8, 1, 16, 128
    T_sh, T_rep = 2053, 250  # sharded operand 257-token shards (last 254), replicated one 250 tokens
    g = torch.Generator().manual_seed(flags)
    Tq, Tk = (T_rep, T_sh) if flags == sp.SP_SHARD_KV else (T_sh, T_rep)
    q = torch.randn(B, Tq, H, D, generator=g).bfloat16().cuda()
    k, v = (torch.randn(B, Tk, H, D, generator=g).bfloat16().cuda() for _ in range(2))
    mask = (torch.rand(Tk, generator=g) < 0.9).to(torch.uint8)
    mask[0] = 1
    Hl = H // W
    Tl = -(-T_sh // W)
    views = lambda x: [x[:, min(s * Tl, T_sh):min((s + 1) * Tl, T_sh)] for s in range(W)]  # noqa: E731
    heads = lambda x: [x[:, :, r * Hl:(r + 1) * Hl] for r in range(W)]  # noqa: E731
    out = torch.full((B, Tq, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16))
    if flags == sp.SP_SHARD_KV:
        sp.sp_attention_shards(heads(q), views(k), views(v), heads(out), ws, flags, sp.SP_MASK_KEY, mask.cuda())
    else:
        sp.sp_attention_shards(views(q), heads(k), heads(v), views(out), ws, flags, sp.SP_MASK_KEY, mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    ref = oracle.attention(f32_np(q), f32_np(k), f32_np(v), sp.SP_MASK_KEY, mask.numpy())
    assert max_abs(f32_np(out), ref) <= 2e-2


def test_concurrent_host_threads_give_the_same_bytes():
    # ctypes drops the GIL around each call, so four host threads really enter
    # the library together (first-use caches included: a fresh process
    # would fill them here), each on its own stream and workspace.
    import threading

    W, B, T, Hl, D = 2, 1, 700, 2, 128
    g = torch.Generator().manual_seed(31)
    q, k, v = (_mk(W, B, T, Hl, D, torch.bfloat16, g) for _ in range(3))
    need = sp.sp_attention_workspace_bytes(W, B, T, T, Hl, D, torch.bfloat16)
    ref = [torch.empty_like(x) for x in q]
    sp.sp_attention(q, k, v, ref, sp.new_workspace(need))
    torch.cuda.synchronize()
    outs, errors = [], []

    def work():
        try:
            s = torch.cuda.Stream()
            ws = sp.new_workspace(need)
            o = [torch.empty_like(x) for x in q]
            with torch.cuda.stream(s):
                for _ in range(5):
                    sp.sp_attention(q, k, v, o, ws, stream=s)
            s.synchronize()
            outs.append((o, sp.sp_workspace_status(ws, stream=s)[0]))
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work) for _ in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert len(outs) == 4
    for o, st in outs:
        assert st == 0
        for a, b in zip(o, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# The row maximum of a key tile comes from the TMEM load of S itself; a tile
# with hidden keys must recompute it over the visible ones.  These inputs make
# the hidden keys (masked, or past the end of the keys) the largest scores of
# every row: every query is +3, a visible key -3, a hidden key +3, so the
# scores are -9 D and +9 D (zero for keys the tile loads past the end).  A
# maximum taken over hidden keys would flush every visible probability to
# zero; the right answer is the plain mean of the visible V rows.
def _hidden_max_inputs(B, Tq, Tk, H, D, hidden, g):
    q = torch.full((B, Tq, H, D), 3.0).bfloat16()
    k = torch.full((B, Tk, H, D), -3.0)
    if len(hidden):
        k[:, hidden] = 3.0
    v = torch.randn(B, Tk, H, D, generator=g).bfloat16()
    return q, k.bfloat16(), v


def _mean_of_visible(v, visible, Tq):
    # closed form: uniform softmax over the visible keys, for every query
    m = f32_np(v)[:, visible].astype(np.float64).mean(axis=1, keepdims=True)
    return np.repeat(m, Tq, axis=1)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask_kind", [sp.SP_MASK_KEY, sp.SP_MASK_FULL])
def test_hidden_keys_with_the_largest_scores_leave_the_row_max(mask_kind, D):
    W, B, Tq, Tk, Hl = 2, 1, 256, 300, 2
    hidden = [5, 77, 130, 200, 201, 202, 299]
    visible = [t for t in range(Tk) if t not in hidden]
    g = torch.Generator().manual_seed(41 + D)
    ranks = [_hidden_max_inputs(B, Tq, Tk, Hl, D, hidden, g) for _ in range(W)]
    keep = torch.ones(Tk, dtype=torch.uint8)
    keep[hidden] = 0
    mask = keep if mask_kind == sp.SP_MASK_KEY else keep.view(1, 1, Tk).repeat(B, Tq, 1).contiguous()
    q, k, v = ([x[i].cuda() for x in ranks] for i in range(3))
    o = [torch.full_like(x, float("nan")) for x in q]
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16))
    sp.sp_attention(q, k, v, o, ws, mask_kind, mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    for r in range(W):
        got = f32_np(o[r])
        assert np.isfinite(got).all()
        assert max_abs(got, _mean_of_visible(ranks[r][2], visible, Tq)) <= 2e-2
        ref = oracle.attention(f32_np(ranks[r][0]), f32_np(ranks[r][1]), f32_np(ranks[r][2]), mask_kind, mask.numpy())
        assert max_abs(got, ref) <= 2e-2


def test_keys_past_the_end_leave_the_row_max():
    # no mask, 300 keys: the last key tile's columns past key 299 hold zeros
    # (the load fills them), larger than every real score (-1152)
    W, B, Tq, Tk, Hl, D = 1, 1, 256, 300, 2, 128
    g = torch.Generator().manual_seed(43)
    q, k, v = _hidden_max_inputs(B, Tq, Tk, Hl, D, [], g)
    o = [torch.full_like(q, float("nan")).cuda()]
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, Tq, Tk, Hl, D, torch.bfloat16))
    sp.sp_attention([q.cuda()], [k.cuda()], [v.cuda()], o, ws)
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    got = f32_np(o[0])
    assert max_abs(got, _mean_of_visible(v, list(range(Tk)), Tq)) <= 2e-2


@pytest.mark.parametrize("mask_kind", [sp.SP_MASK_NONE, sp.SP_MASK_KEY])
def test_sharded_tiles_with_hidden_keys_leave_the_row_max(mask_kind):
    # The exchange inside the attention, ragged shards (partial and gathered
    # key tiles whose rows past a shard's end hold zeros or stale keys).
    W, B, T, H, D = 4, 1, 771, 8, 128
    hidden = [3, 190, 194, 400, 770] if mask_kind == sp.SP_MASK_KEY else []
    visible = [t for t in range(T) if t not in hidden]
    g = torch.Generator().manual_seed(44)
    q, k, v = (x.cuda() for x in _hidden_max_inputs(B, T, T, H, D, hidden, g))
    mask = None
    if mask_kind == sp.SP_MASK_KEY:
        mask = torch.ones(T, dtype=torch.uint8)
        mask[hidden] = 0
    Tl = -(-T // W)
    views = lambda x: [x[:, min(s * Tl, T):min((s + 1) * Tl, T)] for s in range(W)]  # noqa: E731
    out = torch.full((B, T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = sp.new_workspace(sp.sp_attention_workspace_bytes(W, B, T, T, H // W, D, torch.bfloat16))
    sp.sp_attention_shards(views(q), views(k), views(v), views(out), ws, sp.SP_SHARD_Q | sp.SP_SHARD_KV,
                           mask_kind, None if mask is None else mask.cuda())
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    got = f32_np(out)
    assert np.isfinite(got).all()
    assert max_abs(got, _mean_of_visible(v.cpu(), visible, T)) <= 2e-2
