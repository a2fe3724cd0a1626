"""The two cluster variants of the tensor-core attention kernel -- CTA pairs
sharing K/V tiles by TMA multicast (mode 1), and CTA pairs running one M=256
tcgen05 pass with cta_group::2 (mode 2) -- must give exactly the bytes the
default kernel (mode 0) gives: same tiles, same accumulation order.  Each mode
runs in its own process because the library reads the selector once."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import sequence_video_dit_gb300 as sp
W, B, T, Hl, D = 4, 1, 1300, 2, 128   # 6 query pairs per head (the last one ragged)
g = torch.Generator().manual_seed(5)
mk = lambda: [torch.randn(B, T, Hl, D, generator=g).bfloat16().cuda() for _ in range(W)]
q, k, v = mk(), mk(), mk()
o = [torch.full_like(x, float("nan")) for x in q]
mask = torch.ones(T, dtype=torch.uint8); mask[-7:] = 0
# A header-only workspace: no key split, so the cluster variants are eligible
# (split plans always run the single-CTA kernel).
ws = sp.new_workspace()
sp.sp_attention(q, k, v, o, ws, sp.SP_MASK_KEY, mask.cuda())
torch.cuda.synchronize()
assert sp.sp_workspace_status(ws)[0] == 0
torch.save([x.cpu() for x in o], sys.argv[2])
"""


def _run(mode, tmp_path):
    out = tmp_path / f"o{mode}.pt"
    env = dict(os.environ, SP_ATTN_CLUSTER_MODE=str(mode))
    subprocess.run([sys.executable, "-c", SCRIPT, ROOT, str(out)], env=env, check=True, timeout=300)
    import torch

    return torch.load(out)


def test_cluster_modes_bitwise_equal(tmp_path):
    import torch

    base = _run(0, tmp_path)
    for mode in (1, 2):
        got = _run(mode, tmp_path)
        for a, b in zip(base, got):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"mode {mode} differs"
