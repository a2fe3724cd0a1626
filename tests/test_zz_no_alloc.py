"""sp_send_recv_heads_noalloc: the head exchange for callers that cannot
allocate device memory (its scratch lives in a static device array inside the
library).  Called twice in a row through the C ABI, it must produce exactly
what the workspace-taking sp_send_recv_heads produces (layout work is
bit-exact), and report a clean device status each time."""
import pytest
import torch

import sequence_video_dit_gb300 as sp

pytestmark = pytest.mark.gpu


def _shards(W, B, Tl, H, D, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return [torch.randn(B, Tl, H, D, device="cuda", generator=g).to(dtype) for _ in range(W)]


@pytest.mark.parametrize("W,B,Tl,H,D,dtype", [(8, 1, 769, 32, 128, torch.bfloat16),
                                              (2, 1, 19, 4, 32, torch.float32),
                                              (4, 2, 251, 8, 64, torch.bfloat16)])
def test_noalloc_exchange_matches_workspace_exchange_twice(W, B, Tl, H, D, dtype):
    ws = sp.new_workspace()
    for call in range(2):
        shards = _shards(W, B, Tl, H, D, dtype, seed=100 * call + W)
        want = [torch.empty(B, W * Tl, H // W, D, dtype=dtype, device="cuda") for _ in range(W)]
        got = [torch.full((B, W * Tl, H // W, D), float("nan"), dtype=dtype, device="cuda") for _ in range(W)]
        sp.sp_send_recv_heads(shards, want, ws)
        status = sp.sp_send_recv_heads_noalloc(shards, got)
        assert status == 0, f"call {call}: device status {status}"
        for r in range(W):
            assert torch.equal(got[r].view(torch.uint8), want[r].view(torch.uint8)), f"call {call}, rank {r}"
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws)[0] == 0


def test_noalloc_exchange_async_then_status():
    W, B, Tl, H, D = 8, 1, 64, 16, 128
    shards = _shards(W, B, Tl, H, D, torch.bfloat16, seed=7)
    want = [torch.empty(B, W * Tl, H // W, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    got = [torch.empty_like(x) for x in want]
    sp.sp_send_recv_heads(shards, want, sp.new_workspace())
    assert sp.sp_send_recv_heads_noalloc(shards, got, read_status=False) is None
    assert sp.sp_send_recv_heads_noalloc(shards, got) == 0
    for r in range(W):
        assert torch.equal(got[r].view(torch.uint8), want[r].view(torch.uint8))


def test_noalloc_exchange_rejects_more_ranks_than_its_scratch_holds():
    shards = [torch.zeros(1, 2, 9, 8, dtype=torch.bfloat16, device="cuda") for _ in range(9)]
    heads = [torch.zeros(1, 18, 1, 8, dtype=torch.bfloat16, device="cuda") for _ in range(9)]
    with pytest.raises(ValueError, match="static scratch"):
        sp.sp_send_recv_heads_noalloc(shards, heads)


def test_noalloc_rejected_call_leaves_the_scratch_alone():
    # A call rejected by the host-side argument checks returns its error before
    # touching the shared array; the status word of the asynchronous call before
    # it is then still there for the next call that reads it.
    import ctypes
    from sequence_video_dit_gb300._lib import lib, ptr_array
    W, B, Tl, H, D = 4, 1, 96, 8, 64
    shards = _shards(W, B, Tl, H, D, torch.bfloat16, seed=11)
    want = [torch.empty(B, W * Tl, H // W, D, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    got = [torch.empty_like(x) for x in want]
    sp.sp_send_recv_heads(shards, want, sp.new_workspace())
    assert sp.sp_send_recv_heads_noalloc(shards, got, read_status=False) is None
    st = ctypes.c_int(-1)
    rc = lib().sp_send_recv_heads_noalloc(ptr_array(shards), ptr_array(got), W, B, Tl, H, D, 3,
                                          ctypes.byref(st), None)
    assert rc == 3 and st.value == -1  # SP_ERR_INVALID_ARG (elt_bytes = 3); no status was read
    assert sp.sp_send_recv_heads_noalloc(shards, got) == 0
    for r in range(W):
        assert torch.equal(got[r].view(torch.uint8), want[r].view(torch.uint8))
