"""Layout kernels vs the oracle, bit-exact: pad, padding masks, tile, the
token x head exchange (send_recv_heads / gather_heads) with its SM-rotation
counters, gather_output and unpad.  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import sequence_video_dit_gb300 as sp
from gpu_helpers import bytes_np, random_bytes

pytestmark = pytest.mark.gpu

CASES = [
    # B, T, W, H, D, dtype
    (1, 37, 2, 4, 32, torch.float32),      # c1 shape
    (2, 1001, 4, 8, 64, torch.bfloat16),   # c2 shape
    (1, 6149, 8, 32, 128, torch.bfloat16),  # c3 shape
    (1, 5, 8, 8, 4, torch.float32),        # T < W: ranks 5..7 hold only padding
    (2, 16, 4, 4, 8, torch.bfloat16),      # already divisible
    (2, 10, 1, 2, 16, torch.bfloat16),     # W = 1: identity exchange
    (3, 7, 3, 6, 3, torch.float32),        # odd sizes: 4-byte vectors
    (1, 9, 2, 2, 5, torch.bfloat16),       # 10-byte chunks: 2-byte vectors
]


@pytest.mark.parametrize("B,T,W,H,D,dtype", CASES)
def test_layout_chain_bit_exact(B, T, W, H, D, dtype):
    g = torch.Generator().manual_seed(B * 1000 + T * 10 + W)
    x = random_bytes((B, T, H, D), dtype, g)
    T_pad = sp.sp_padded_len(T, W)
    Tl, Hl = T_pad // W, H // W
    ws = sp.new_workspace()
    x_np = bytes_np(x)  # [B,T,H,D*elt]

    x_pad = torch.empty(B, T_pad, H, D, dtype=dtype, device="cuda")
    sp.sp_pad(x, x_pad)
    o_pad = oracle.pad(x_np, T_pad)
    assert np.array_equal(bytes_np(x_pad), o_pad)

    shards = [torch.empty(B, Tl, H, D, dtype=dtype, device="cuda") for _ in range(W)]
    sp.sp_tile(x_pad, shards)
    o_shards = oracle.tile(o_pad, W)
    for r in range(W):
        assert np.array_equal(bytes_np(shards[r]), o_shards[r])

    heads = [torch.empty(B, T_pad, Hl, D, dtype=dtype, device="cuda") for _ in range(W)]
    sp.sp_send_recv_heads(shards, heads, ws)
    o_heads = oracle.send_recv_heads(o_shards)
    for r in range(W):
        assert np.array_equal(bytes_np(heads[r]), o_heads[r])

    back = [torch.empty_like(s) for s in shards]
    sp.sp_gather_heads(heads, back, ws)
    for r in range(W):
        assert torch.equal(back[r].view(torch.uint8), shards[r].view(torch.uint8))  # gather(send(x)) == x

    full = torch.empty(B, T_pad, H, D, dtype=dtype, device="cuda")
    sp.sp_gather_output(back, full)
    assert np.array_equal(bytes_np(full), oracle.gather_output(o_shards, T_pad))
    cropped = torch.empty(B, T, H, D, dtype=dtype, device="cuda")
    sp.sp_gather_output(back, cropped)
    assert np.array_equal(bytes_np(cropped), oracle.gather_output(o_shards, T))
    un = torch.empty(B, T, H, D, dtype=dtype, device="cuda")
    sp.sp_unpad(full, un)
    assert np.array_equal(bytes_np(un), oracle.unpad(bytes_np(full), T))
    assert torch.equal(un.view(torch.uint8), x.view(torch.uint8))
    torch.cuda.synchronize()
    st, counts, n = sp.sp_workspace_status(ws)
    assert st == 0 and n == 2


@pytest.mark.parametrize("B,T,W", [(2, 1001, 4), (1, 3, 2), (2, 16, 4), (1, 1, 8)])
def test_pad_masks_bit_exact(B, T, W):
    T_pad = sp.sp_padded_len(T, W)
    key = torch.full((1, 1, T_pad), 7, dtype=torch.uint8, device="cuda")
    sp.sp_pad_mask(None, key, T)
    assert np.array_equal(key.cpu().numpy(), oracle.pad_mask_key(T, T_pad))
    g = torch.Generator().manual_seed(T)
    user = (torch.rand(B, T, T, generator=g) < 0.3).to(torch.uint8)
    out = torch.full((B, T_pad, T_pad), 7, dtype=torch.uint8, device="cuda")
    sp.sp_pad_mask(user.cuda(), out, T)
    assert np.array_equal(out.cpu().numpy(), oracle.pad_mask_user(user.numpy(), T_pad))


def test_exchange_counters_follow_sm_rotation():
    W, B, Tl, H, D = 8, 1, 64, 32, 128
    shards = [torch.randn(B, Tl, H, D, device="cuda").bfloat16() for _ in range(W)]
    heads = [torch.empty(B, W * Tl, H // W, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    ws = sp.new_workspace()
    sp.sp_send_recv_heads(shards, heads, ws)
    torch.cuda.synchronize()
    st, counts, n = sp.sp_workspace_status(ws)
    grid = sp.sp_exchange_grid()
    assert st == 0 and n == 1
    assert counts[:W] == sp.sp_sm_rotation_counts(grid, W) == oracle.sm_rotation_counts(grid, W)
    # the counters were reset for the next launch
    hdr = ws[:sp.SP_WORKSPACE_HEADER_BYTES].view(torch.int32).cpu()
    assert hdr[1].item() == 0 and not hdr[2:2 + W].any()


def test_exchange_barrier_reports_a_short_counter():
    # Fault made on the host: one destination counter starts one short, so
    # the last CTA's check must flag SP_ERR_BARRIER (no device wait involved).
    W, B, Tl, H, D = 4, 1, 32, 8, 64
    shards = [torch.randn(B, Tl, H, D, device="cuda").bfloat16() for _ in range(W)]
    heads = [torch.empty(B, W * Tl, H // W, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    ws = sp.new_workspace()
    ws.view(torch.int32)[2 + 1] = -1  # counters[1] = -1
    sp.sp_send_recv_heads(shards, heads, ws)
    torch.cuda.synchronize()
    st, counts, _ = sp.sp_workspace_status(ws, clear=True)
    assert st == 7  # SP_ERR_BARRIER
    assert counts[1] == sp.sp_sm_rotation_counts(sp.sp_exchange_grid(), W)[1] - 1
    sp.sp_send_recv_heads(shards, heads, ws)
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0


def test_misaligned_buffers_still_exact():
    # a 2-byte offset forces the narrow-vector path
    B, T, W, H, D = 1, 13, 4, 4, 8
    g = torch.Generator().manual_seed(5)
    big = random_bytes((B * T * H * D + 1,), torch.bfloat16, g)
    x = big[1:].view(B, T, H, D)
    T_pad = sp.sp_padded_len(T, W)
    big_out = torch.empty(B * T_pad * H * D + 1, dtype=torch.bfloat16, device="cuda")
    xp = big_out[1:].view(B, T_pad, H, D)
    sp.sp_pad(x, xp)
    assert np.array_equal(bytes_np(xp), oracle.pad(bytes_np(x), T_pad))


def test_argument_errors():
    W = 4
    shards = [torch.zeros(1, 2, 6, 8, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    heads = [torch.zeros(1, 8, 1, 8, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    with pytest.raises(ValueError):  # H = 6 is not divisible by W = 4
        sp.sp_send_recv_heads(shards, heads, sp.new_workspace())
    x = torch.zeros(1, 37, 4, 8, device="cuda")
    with pytest.raises(ValueError):  # 37 tokens cannot be tiled over 2 ranks
        sp.sp_tile(x, [torch.zeros(1, 18, 4, 8, device="cuda")] * 2)


@pytest.mark.parametrize("T_pad", [49160, 131072, 524288], ids=["c5-403MB", "sweep-1GB", "sweep-4GB"])
def test_full_size_exchange_round_trip_and_sampled_map(T_pad):
    # [1, T_pad, 32, 128] bf16 (8 KB per token): the c5 tensors (403 MB) and the
    # 1 GB and 4 GB points of the standalone permute sweep, W = 8
    W, B, H, D = 8, 1, 32, 128
    Tl, Hl = T_pad // W, H // W
    g = torch.Generator(device="cuda").manual_seed(11 + T_pad)
    shards = [torch.randint(-32768, 32767, (B, Tl, H, D), dtype=torch.int16, device="cuda", generator=g)
              .view(torch.bfloat16) for _ in range(W)]
    heads = [torch.empty(B, T_pad, Hl, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    ws = sp.new_workspace()
    sp.sp_send_recv_heads(shards, heads, ws)
    back = [torch.empty_like(s) for s in shards]
    sp.sp_gather_heads(heads, back, ws)
    for r in range(W):
        assert torch.equal(back[r].view(torch.int16), shards[r].view(torch.int16))  # gather(send(x)) == x
    del back
    # sampled tokens (the first and last two of every shard, and some in between):
    # the oracle's exchange of those tokens alone must match
    gen = torch.Generator().manual_seed(T_pad)
    mid = torch.randint(2, Tl - 2, (6,), generator=gen)
    t_sel = torch.cat([torch.tensor([0, 1]), mid, torch.tensor([Tl - 2, Tl - 1])])
    mini = [bytes_np(s[:, t_sel]) for s in shards]
    mini_heads = oracle.send_recv_heads(mini)
    for r in range(W):
        rows = torch.cat([s * Tl + t_sel for s in range(W)])
        assert np.array_equal(bytes_np(heads[r][:, rows]), mini_heads[r])
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0
    del shards, heads
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,T,W,H,D,dtype", CASES)
def test_fused_exchange_bit_exact(B, T, W, H, D, dtype):
    # sp_pad_send_heads == pad -> tile -> send_recv_heads, and
    # sp_gather_heads_output == gather_heads -> gather_output (cropped to T).
    g = torch.Generator().manual_seed(7 * T + W)
    x = random_bytes((B, T, H, D), dtype, g)
    T_pad = sp.sp_padded_len(T, W)
    Hl = H // W
    ws = sp.new_workspace()
    heads = [torch.full((B, T_pad, Hl, D), 1.0, dtype=dtype, device="cuda") for _ in range(W)]
    sp.sp_pad_send_heads(x, heads, ws)
    want = oracle.send_recv_heads(oracle.tile(oracle.pad(bytes_np(x), T_pad), W))
    for r in range(W):
        assert np.array_equal(bytes_np(heads[r]), want[r])
    out = torch.empty(B, T, H, D, dtype=dtype, device="cuda")
    sp.sp_gather_heads_output(heads, out, ws)
    want_out = oracle.gather_output(oracle.gather_heads([bytes_np(h) for h in heads]), T)
    assert np.array_equal(bytes_np(out), want_out)
    assert torch.equal(out.view(torch.uint8), x.view(torch.uint8))  # round trip
    torch.cuda.synchronize()
    st, counts, n = sp.sp_workspace_status(ws)
    assert st == 0 and n == 2
    assert counts[:W] == oracle.sm_rotation_counts(sp.sp_exchange_grid(), W)


def test_fused_exchange_argument_errors():
    x = torch.zeros(1, 10, 6, 8, dtype=torch.bfloat16, device="cuda")
    heads = [torch.zeros(1, 12, 1, 8, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    with pytest.raises(ValueError):  # H = 6 not divisible by W = 4
        sp.sp_pad_send_heads(x, heads, sp.new_workspace())
    x = torch.zeros(1, 10, 4, 8, dtype=torch.bfloat16, device="cuda")
    heads = [torch.zeros(1, 11, 1, 8, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    with pytest.raises(ValueError):  # T_pad = 11 is not a multiple of W = 4
        sp.sp_pad_send_heads(x, heads, sp.new_workspace())


def test_mismatched_rank_buffers_are_rejected_before_launch():
    W, B, Tl, H, D = 4, 1, 8, 8, 16
    shards = [torch.zeros(B, Tl, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    heads = [torch.zeros(B, W * Tl, H // W, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    short = heads[:3] + [torch.zeros(B, W * Tl - 1, H // W, D, dtype=torch.bfloat16, device="cuda")]
    with pytest.raises(ValueError):
        sp.sp_send_recv_heads(shards, short, sp.new_workspace())
    with pytest.raises(ValueError):
        sp.sp_gather_heads(short, shards, sp.new_workspace())
    with pytest.raises(ValueError):
        sp.sp_pad_send_heads(torch.zeros(B, 30, H, D, dtype=torch.bfloat16, device="cuda"), short,
                             sp.new_workspace())
    with pytest.raises(ValueError):  # out longer than the padded length
        sp.sp_gather_heads_output(heads, torch.zeros(B, W * Tl + 1, H, D, dtype=torch.bfloat16, device="cuda"),
                                  sp.new_workspace())
    with pytest.raises(ValueError):
        sp.sp_tile(torch.zeros(B, W * Tl, H, D, device="cuda"), [torch.zeros(B, Tl + 1, H, D, device="cuda")] * W)
    with pytest.raises(ValueError):
        sp.sp_unpad(torch.zeros(B, 8, H, D, device="cuda"), torch.zeros(B, 9, H, D, device="cuda"))


@pytest.mark.parametrize("B,grid,W,H,D,dtype", [
    (1, (16, 24, 16), 8, 32, 128, torch.bfloat16),  # 6144 video tokens, split 2x4, blocks 12x4
    (2, (3, 4, 6), 6, 6, 8, torch.float32),          # split 2x3
    (1, (2, 5, 6), 3, 3, 5, torch.bfloat16),         # split 1x3, 30-byte rows: 2-byte vectors
    (2, (2, 3, 3), 1, 2, 4, torch.float32),          # W = 1: identity
])
def test_tile_2d_and_gather_2d_bit_exact(B, grid, W, H, D, dtype):
    g = torch.Generator().manual_seed(sum(grid) + W)
    F, Hg, Wg = grid
    x = random_bytes((B, F * Hg * Wg, H, D), dtype, g)
    split = sp.sp_optimal_split(W)
    assert split == oracle.optimal_split(W)
    Tl = F * (Hg // split[0]) * (Wg // split[1])
    shards = [torch.empty(B, Tl, H, D, dtype=dtype, device="cuda") for _ in range(W)]
    sp.sp_tile_2d(x, shards, grid)
    want = oracle.tile_2d(bytes_np(x), grid, split)
    for r in range(W):
        assert np.array_equal(bytes_np(shards[r]), want[r])
    back = torch.empty_like(x)
    sp.sp_gather_2d(shards, back, grid)
    assert np.array_equal(bytes_np(back), oracle.gather_2d(want, grid, split))
    assert torch.equal(back.view(torch.uint8), x.view(torch.uint8))


def test_tile_2d_argument_errors():
    x = torch.zeros(1, 1 * 5 * 4, 4, 8, dtype=torch.bfloat16, device="cuda")
    shards = [torch.zeros(1, 5, 4, 8, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    with pytest.raises(ValueError):  # 5 patch rows cannot be cut into 2 bands
        sp.sp_tile_2d(x, shards, (1, 5, 4))
    with pytest.raises(ValueError):  # token count does not match the grid
        sp.sp_tile_2d(x, shards, (1, 4, 4), (2, 2))
