"""Pins for the CPU oracle (no GPU).  Each test ties the oracle to something
other than itself: a value the pages print, a hand-enumerated fixture, a closed
form, an invariant, or an independent library routine.

Source: "LTX-2 序列并行拆解" (LTX-2 sequence-parallel breakdown), sections
补齐 / 切分 / 换头 / 还原, the correctness paragraph and the SM-rotation
paragraph.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def _rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ 切分 (partition)
def test_partition_rejects_non_divisible():
    # 切分: compute_sequence_partition requires total_tokens % world_size == 0, else ValueError.
    with pytest.raises(ValueError):
        oracle.partition(37, 2)
    with pytest.raises(oracle.PartitionError):
        oracle.partition(1001, 4)
    assert oracle.partition(38, 2) == [(0, 19), (19, 19)]
    assert oracle.partition(0, 4) == [(0, 0)] * 4


@pytest.mark.parametrize("T,W", [(37, 2), (1001, 4), (6149, 8), (49155, 8), (24576, 8),
                                 (1, 8), (8, 8), (0, 3)])
def test_padded_len_closed_form(T, W):
    # 补齐: padded to a multiple of world_size -> the smallest such multiple.
    tp = oracle.padded_len(T, W)
    assert tp == -(-T // W) * W
    assert tp % W == 0 and T <= tp < T + W


def test_config_padded_lengths_match_workload_table():
    # The workload descriptions state the padded lengths explicitly.
    assert oracle.padded_len(37, 2) == 38
    assert oracle.padded_len(1001, 4) == 1004
    assert oracle.padded_len(6149, 8) == 6152
    assert oracle.padded_len(49155, 8) == 49160


# ------------------------------------------------------------------ SM rotation
def test_sm_rotation_matches_page_example(golden_dir):
    (row,) = read_golden(os.path.join(golden_dir, "sm_rotation_132_8.txt"))
    n_sm, W, *counts = row
    assert oracle.sm_rotation_counts(n_sm, W) == counts


@pytest.mark.parametrize("n_sm,W", [(152, 8), (148, 8), (152, 3), (7, 8), (152, 1)])
def test_sm_rotation_partition_of_sms(n_sm, W):
    c = oracle.sm_rotation_counts(n_sm, W)
    assert sum(c) == n_sm
    assert max(c) - min(c) <= 1
    assert c == sorted(c, reverse=True)


# ------------------------------------------------------------------ 补齐 (pad) and masks
def test_pad_unpad_round_trip_and_zero_fill():
    x = _rng(1).integers(0, 2**16, size=(2, 5, 3, 4), dtype=np.uint16)
    xp = oracle.pad(x, 8)
    assert xp.shape == (2, 8, 3, 4)
    assert np.array_equal(xp[:, :5], x)
    assert not xp[:, 5:].any()
    assert np.array_equal(oracle.unpad(xp, 5), x)


def test_pad_mask_key_literal():
    assert oracle.pad_mask_key(3, 4).tolist() == [[[1, 1, 1, 0]]]
    assert oracle.pad_mask_key(4, 4).tolist() == [[[1, 1, 1, 1]]]
    assert oracle.pad_mask_key(0, 2).tolist() == [[[0, 0]]]


def test_pad_mask_user_golden(golden_dir):
    rows = read_golden(os.path.join(golden_dir, "pad_mask_user_T3_W2.txt"))
    user = np.array(rows[:3], dtype=np.uint8)[None]
    want = np.array(rows[3:], dtype=np.uint8)[None]
    got = oracle.pad_mask_user(user, oracle.padded_len(3, 2))
    assert np.array_equal(got, want)


def test_pad_mask_user_no_pad_is_identity():
    u = (_rng(2).random((2, 6, 6)) < 0.5).astype(np.uint8)
    assert np.array_equal(oracle.pad_mask_user(u, 6), u)


# ------------------------------------------------------------------ 换头 (head exchange)
def test_exchange_hand_enumerated(golden_dir):
    rows = read_golden(os.path.join(golden_dir, "exchange_W2_Tl2_H4.txt"))
    W, Tl, H = 2, 2, 4
    shards = []
    for s in range(W):
        a = np.zeros((1, Tl, H, 1), dtype=np.int32)
        for t in range(Tl):
            for h in range(H):
                a[0, t, h, 0] = 1000 * s + 100 * t + h
        shards.append(a)
    heads = oracle.send_recv_heads(shards)
    for r in range(W):
        assert heads[r].shape == (1, W * Tl, H // W, 1)
        assert heads[r].reshape(-1).tolist() == rows[r]


@pytest.mark.parametrize("W,B,Tl,H,D,dt", [(2, 1, 3, 4, 5, np.uint8), (4, 2, 3, 8, 2, np.uint16),
                                           (8, 1, 2, 8, 3, np.float32), (3, 2, 5, 6, 1, np.float64),
                                           (1, 2, 4, 3, 2, np.uint16)])
def test_exchange_brute_force_and_round_trip(W, B, Tl, H, D, dt):
    rng = _rng(3)
    if np.issubdtype(dt, np.integer):
        shards = [rng.integers(0, np.iinfo(dt).max, size=(B, Tl, H, D), dtype=dt) for _ in range(W)]
    else:
        shards = [rng.standard_normal((B, Tl, H, D)).astype(dt) for _ in range(W)]
    heads = oracle.send_recv_heads(shards)
    Hl = H // W
    # brute force: every destination element named by its definition
    for r in range(W):
        for b in range(B):
            for g in range(W * Tl):
                s, t = divmod(g, Tl)
                for hl in range(Hl):
                    assert np.array_equal(heads[r][b, g, hl], shards[s][b, t, r * Hl + hl])
    # 正确性: gather(send(x)) == x byte for byte
    back = oracle.gather_heads(heads)
    for s in range(W):
        assert back[s].tobytes() == shards[s].tobytes()
    if W == 1:
        assert heads[0].tobytes() == shards[0].tobytes()


def test_exchange_rejects_heads_not_divisible():
    shards = [np.zeros((1, 2, 3, 1), np.float32) for _ in range(2)]
    with pytest.raises(ValueError):
        oracle.send_recv_heads(shards)


# ------------------------------------------------------------------ 还原 (restore)
@pytest.mark.parametrize("T,W", [(37, 2), (5, 8), (8, 8), (13, 4), (1, 3)])
def test_tile_gather_unpad_round_trip(T, W):
    x = _rng(4).integers(0, 255, size=(2, T, 3, 2), dtype=np.uint8)
    tp = oracle.padded_len(T, W)
    shards = oracle.tile(oracle.pad(x, tp), W)
    Tl = tp // W
    for r in range(W):
        lo = r * Tl
        want = np.zeros((2, Tl, 3, 2), np.uint8)
        n = max(0, min(T - lo, Tl))
        want[:, :n] = x[:, lo:lo + n]
        assert np.array_equal(shards[r], want)
    # crop by real counts directly to T, or gather everything then unpad: same bytes
    assert np.array_equal(oracle.gather_output(shards, T), x)
    full = oracle.gather_output(shards, tp)
    assert np.array_equal(oracle.unpad(full, T), x)


def test_gather_output_real_counts_literal():
    # W=2, Tl=2, T_out=3: rank 0 contributes 2 tokens, rank 1 only its first.
    s0 = np.array([[[1], [2]]], np.int32)
    s1 = np.array([[[3], [4]]], np.int32)
    assert oracle.gather_output([s0, s1], 3).reshape(-1).tolist() == [1, 2, 3]
    assert oracle.gather_output([s0, s1], 4).reshape(-1).tolist() == [1, 2, 3, 4]


# ------------------------------------------------------------------ attention
def test_attention_closed_form_weights():
    # Scores s_j = ln(w_j) make the softmax weights proportional to w_j:
    # O = sum_j w_j v_j / sum_j w_j.  Pins scale, sign, exp and normalisation.
    D = 4
    w = np.array([1.0, 2.0, 3.0, 4.0, 0.5])
    q = np.zeros((1, 1, 1, D), np.float32)
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, len(w), 1, D), np.float32)
    k[0, :, 0, 0] = (np.log(w) * math.sqrt(D)).astype(np.float32)  # scale = 1/sqrt(D)
    v = _rng(5).standard_normal((1, len(w), 1, D)).astype(np.float32)
    o = oracle.attention(q, k, v)
    want = (w[:, None] * v[0, :, 0].astype(np.float64)).sum(0) / w.sum()
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-6, atol=1e-7)


def test_attention_two_keys_logistic():
    # Two visible keys: O = v0 + (v1 - v0) * sigmoid(s1 - s0).
    from scipy.special import expit
    D = 8
    a = np.array([0.3, -1.7], dtype=np.float64)
    q = np.zeros((1, 1, 1, D), np.float32)
    q[..., 0] = 1
    k = np.zeros((1, 2, 1, D), np.float32)
    k[0, :, 0, 0] = (a * math.sqrt(D)).astype(np.float32)
    v = _rng(6).standard_normal((1, 2, 1, D)).astype(np.float32)
    o = oracle.attention(q, k, v)[0, 0, 0]
    v0, v1 = v[0, 0, 0].astype(np.float64), v[0, 1, 0].astype(np.float64)
    ds = float(k[0, 1, 0, 0]) - float(k[0, 0, 0, 0])
    want = v0 + (v1 - v0) * expit(ds / math.sqrt(D))
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)


def _sdpa64(q, k, v, bool_mask=None, scale=None):
    """Independent library routine: torch SDPA in fp64 on [B,H,T,D]."""
    tq = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k.astype(np.float64)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(v.astype(np.float64)).permute(0, 2, 1, 3)
    am = None if bool_mask is None else torch.from_numpy(bool_mask.astype(bool))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("B,Tq,Tk,H,D,kind", [(2, 7, 9, 3, 16, 0), (1, 13, 13, 2, 32, 1),
                                             (2, 11, 11, 4, 8, 2), (1, 5, 40, 2, 64, 1)])
def test_attention_matches_torch_sdpa_fp64(B, Tq, Tk, H, D, kind):
    rng = _rng(7)
    q = rng.standard_normal((B, Tq, H, D)).astype(np.float32)
    k = rng.standard_normal((B, Tk, H, D)).astype(np.float32)
    v = rng.standard_normal((B, Tk, H, D)).astype(np.float32)
    if kind == 0:
        o = oracle.attention(q, k, v)
        ref = _sdpa64(q, k, v)
    elif kind == 1:
        m = (rng.random(Tk) < 0.7).astype(np.uint8)
        m[0] = 1
        o = oracle.attention(q, k, v, oracle.MASK_KEY, m)
        ref = _sdpa64(q, k, v, np.broadcast_to(m.astype(bool), (B, 1, Tq, Tk)))
    else:
        m = (rng.random((B, Tq, Tk)) < 0.4).astype(np.uint8)
        for b in range(B):
            np.fill_diagonal(m[b], 1)
        o = oracle.attention(q, k, v, oracle.MASK_FULL, m)
        ref = _sdpa64(q, k, v, m.astype(bool)[:, None])
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_attention_identity_mask_returns_v_exactly():
    rng = _rng(8)
    B, T, H, D = 2, 6, 2, 4
    q, k, v = (rng.standard_normal((B, T, H, D)).astype(np.float32) for _ in range(3))
    m = np.broadcast_to(np.eye(T, dtype=np.uint8), (B, T, T)).copy()
    o = oracle.attention(q, k, v, oracle.MASK_FULL, m)
    assert np.array_equal(o, v.astype(np.float64))


def test_attention_constant_v():
    rng = _rng(9)
    B, T, H, D = 1, 9, 3, 8
    q, k = (rng.standard_normal((B, T, H, D)).astype(np.float32) for _ in range(2))
    v = np.broadcast_to(rng.standard_normal((1, 1, H, D)).astype(np.float32), (B, T, H, D)).copy()
    o = oracle.attention(q, k, v)
    np.testing.assert_allclose(o, v.astype(np.float64), rtol=1e-14, atol=1e-14)


def test_attention_fully_masked_row_is_zero():
    rng = _rng(10)
    q, k, v = (rng.standard_normal((1, 3, 1, 4)).astype(np.float32) for _ in range(3))
    m = np.ones((1, 3, 3), np.uint8)
    m[0, 1] = 0
    o = oracle.attention(q, k, v, oracle.MASK_FULL, m)
    assert not o[0, 1].any()
    assert np.isfinite(o).all()


def test_attention_key_permutation_invariance():
    rng = _rng(11)
    B, Tq, Tk, H, D = 1, 4, 10, 2, 8
    q = rng.standard_normal((B, Tq, H, D)).astype(np.float32)
    k = rng.standard_normal((B, Tk, H, D)).astype(np.float32)
    v = rng.standard_normal((B, Tk, H, D)).astype(np.float32)
    m = (rng.random(Tk) < 0.6).astype(np.uint8)
    m[3] = 1
    perm = rng.permutation(Tk)
    o1 = oracle.attention(q, k, v, oracle.MASK_KEY, m)
    o2 = oracle.attention(q, k[:, perm], v[:, perm], oracle.MASK_KEY, m[perm])
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)


def test_attention_key_mask_all_ones_equals_unmasked():
    rng = _rng(12)
    q, k, v = (rng.standard_normal((2, 8, 2, 16)).astype(np.float32) for _ in range(3))
    o1 = oracle.attention(q, k, v)
    o2 = oracle.attention(q, k, v, oracle.MASK_KEY, np.ones(8, np.uint8))
    assert np.array_equal(o1, o2)


def test_attention_rows_matches_full():
    rng = _rng(13)
    q, k, v = (rng.standard_normal((2, 9, 3, 8)).astype(np.float32) for _ in range(3))
    full = oracle.attention(q, k, v)
    rows = [(0, 0, 0), (1, 8, 2), (0, 4, 1), (1, 3, 0)]
    got = oracle.attention_rows(q, k, v, rows)
    for i, (b, t, h) in enumerate(rows):
        assert np.array_equal(got[i], full[b, t, h])


def test_bf16_widening_is_exact():
    x = torch.randn(1000).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle._f32(bits), x.float().numpy())


# ------------------------------------------------------------------ the whole sharded step
@pytest.mark.parametrize("W,B,T,H,D,user", [(2, 1, 37, 4, 32, False), (4, 2, 23, 8, 8, True),
                                           (8, 1, 5, 8, 4, False), (1, 1, 6, 2, 4, True),
                                           (3, 2, 10, 3, 4, False)])
def test_sp_step_equals_unsharded_attention(W, B, T, H, D, user):
    # 正确性: global attention is unchanged, only its distribution changes.
    rng = _rng(14)
    q, k, v = (rng.standard_normal((B, T, H, D)).astype(np.float32) for _ in range(3))
    um = None
    if user:
        um = (rng.random((B, T, T)) < 0.3).astype(np.uint8)
        for b in range(B):
            np.fill_diagonal(um[b], 1)
    o_sp, st = oracle.sp_step(q, k, v, W, user_mask=um, return_stages=True)
    if um is None:
        o_ref = oracle.attention(q, k, v)
    else:
        o_ref = oracle.attention(q, k, v, oracle.MASK_FULL, um)
    assert np.array_equal(o_sp, o_ref)
    # pad query rows are finite and equal the mean of V over the real keys
    T_pad = oracle.padded_len(T, W)
    Hl = H // W
    vbar = v.astype(np.float64).mean(axis=1)  # [B,H,D]
    for r in range(W):
        oh = st["o_heads"][r]
        assert np.isfinite(oh).all()
        for t in range(T, T_pad):
            np.testing.assert_allclose(oh[:, t], vbar[:, r * Hl:(r + 1) * Hl], rtol=1e-12,
                                       atol=1e-13)


# ------------------------------------------------------------------ 2-D spatial split (LongCat-Video CP)
def _divisor_pairs(W):
    return [(a, W // a) for a in range(1, W + 1) if W % a == 0]


@pytest.mark.parametrize("W", list(range(1, 65)))
def test_optimal_split_brute_force(W):
    # closest to a square: no factor pair has a smaller gap; smaller factor first
    sh, sw = oracle.optimal_split(W)
    assert sh * sw == W and sh <= sw
    assert sw - sh == min(abs(a - b) for a, b in _divisor_pairs(W))


def test_optimal_split_literal():
    assert oracle.optimal_split(8) == (2, 4)
    assert oracle.optimal_split(4) == (2, 2)
    assert oracle.optimal_split(6) == (2, 3)
    assert oracle.optimal_split(7) == (1, 7)
    assert oracle.optimal_split(12) == (3, 4)
    assert oracle.optimal_split(16) == (4, 4)
    assert oracle.optimal_split(1) == (1, 1)
    with pytest.raises(ValueError):
        oracle.optimal_split(0)


@pytest.mark.parametrize("fixture,W,grid", [("tile_2d_F2_H4_W4_W4.txt", 4, (2, 4, 4)),
                                             ("tile_2d_F1_H4_W6_W6.txt", 6, (1, 4, 6))])
def test_tile_2d_hand_enumerated(golden_dir, fixture, W, grid):
    rows = read_golden(os.path.join(golden_dir, fixture))
    F, Hg, Wg = grid
    x = np.arange(F * Hg * Wg, dtype=np.int32).reshape(1, F * Hg * Wg, 1)
    shards = oracle.tile_2d(x, grid, oracle.optimal_split(W))
    assert [s.reshape(-1).tolist() for s in shards] == rows


@pytest.mark.parametrize("B,grid,split,tail", [(1, (1, 1, 12), (1, 4), (3,)), (2, (1, 8, 3), (4, 1), (2, 5)),
                                                (1, (3, 2, 5), (1, 1), (7,))])
def test_tile_2d_reduces_to_the_token_range_tile(B, grid, split, tail):
    # One band of height across a single-row frame, or one piece of width per
    # band in a single frame, makes every block a contiguous token range: the
    # 2-D split is then the 1-D tile.  A 1x1 split is the identity.
    rng = _rng(11)
    F, Hg, Wg = grid
    x = rng.integers(0, 60000, size=(B, F * Hg * Wg) + tail, dtype=np.uint16)
    got = oracle.tile_2d(x, grid, split)
    want = oracle.tile(x, split[0] * split[1])
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


@pytest.mark.parametrize("B,grid,W,tail,dt", [(2, (3, 4, 6), 6, (2, 3), np.uint16), (1, (2, 6, 8), 8, (4,), np.float32),
                                               (3, (1, 3, 5), 1, (1,), np.uint8), (1, (5, 4, 4), 4, (2, 2), np.float64)])
def test_tile_2d_brute_force_and_round_trip(B, grid, W, tail, dt):
    rng = _rng(12)
    F, Hg, Wg = grid
    x = (rng.standard_normal((B, F * Hg * Wg) + tail) * 100).astype(dt)
    sh, sw = oracle.optimal_split(W)
    shards = oracle.tile_2d(x, grid, (sh, sw))
    bh, bw = Hg // sh, Wg // sw
    for r, s in enumerate(shards):
        ih, iw = divmod(r, sw)
        i = 0
        for f in range(F):
            for h in range(bh):
                for w in range(bw):
                    t = (f * Hg + ih * bh + h) * Wg + iw * bw + w
                    assert np.array_equal(s[:, i], x[:, t])
                    i += 1
    assert np.array_equal(oracle.gather_2d(shards, grid, (sh, sw)), x)


def test_tile_2d_rejects_a_grid_the_split_does_not_divide():
    x = np.zeros((1, 1 * 5 * 4, 1), dtype=np.uint8)
    with pytest.raises(oracle.SplitError):
        oracle.tile_2d(x, (1, 5, 4), (2, 2))
    with pytest.raises(oracle.SplitError):
        oracle.gather_2d([x[:, :5]] * 4, (1, 5, 4), (2, 2))


def test_sp_step_2d_equals_unsharded_attention():
    # The 2-D split only permutes the tokens each rank contributes; after the
    # head exchange every rank still sees every key, so the step is plain
    # attention up to the order of the key sum.
    rng = _rng(13)
    B, grid, H, D, W = 2, (2, 4, 6), 12, 8, 6
    T = grid[0] * grid[1] * grid[2]
    q, k, v = (rng.standard_normal((B, T, H, D)).astype(np.float32) for _ in range(3))
    got = oracle.sp_step_2d(q, k, v, grid, W)
    want = oracle.attention(q, k, v)
    assert np.abs(got - want).max() < 1e-12


@pytest.mark.parametrize("W", [1, 2, 4, 8])
@pytest.mark.parametrize("T", list(range(1, 9)))
def test_sp_step_exhaustive_tiny(W, T):
    # Every tiny case: T <= 8 tokens on W in {1, 2, 4, 8} ranks (pure-pad
    # ranks included when T < W), key-only and user masks.  The composition
    # pad -> tile -> exchange -> attention -> gather -> unpad is plain
    # attention exactly: same fp64 sums, the pad keys contribute nothing.
    rng = _rng(100 * W + T)
    B, H, D = 2, 8, 3
    q, k, v = (rng.standard_normal((B, T, H, D)).astype(np.float32) for _ in range(3))
    got = oracle.sp_step(q, k, v, W)
    assert got.shape == (B, T, H, D) and np.isfinite(got).all()
    assert np.array_equal(got, oracle.attention(q, k, v))
    user = (rng.random((B, T, T)) < 0.5).astype(np.uint8)
    user[:, np.arange(T), np.arange(T)] = 1
    got = oracle.sp_step(q, k, v, W, user_mask=user)
    assert np.array_equal(got, oracle.attention(q, k, v, oracle.MASK_FULL, user))
