"""moe_permute_noalloc: the permute for callers that cannot allocate device
memory (their scratch comes from the library's fixed device array).

Checked through the C ABI against moe_permute with a caller workspace: the
results must be identical (the permute is bit-exact), on two calls in a row so
that the second call runs on scratch the first one left behind.  This file is
collected last on purpose."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m

pytestmark = pytest.mark.gpu


def _ids(T, K, E, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _run(fn, ids, x, T, K, E, H, with_ws):
    dev = "cuda"
    P = T * K
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    sp = torch.full((P,), -7, dtype=torch.int32, device=dev)
    p2r = torch.full((P,), -7, dtype=torch.int32, device=dev)
    xp = torch.zeros((P, H), dtype=torch.bfloat16, device=dev)
    if with_ws:
        wsz = m.moe_permute_workspace_size(T, K, E)
        ws = torch.empty((max(wsz, 16),), dtype=torch.uint8, device=dev)
        fn(ids, x, T, K, E, H, off, sp, p2r, xp, ws, wsz)
    else:
        fn(ids, x, T, K, E, H, off, sp, p2r, xp)
    torch.cuda.synchronize()
    return [t.cpu() for t in (off, sp, p2r, xp)]


# every case but the last has more than 32 chunks of 512 pairs, so it runs the
# multi-kernel permute whose histogram lives in the fixed scratch (32 chunks or
# fewer take the one-block permute, which keeps its histogram in shared memory);
# (16384, 8, 1024) fills the scratch to its last byte
@pytest.mark.parametrize("T,K,E,H", [(8192, 8, 128, 64), (4100, 8, 256, 128),
                                     (16384, 8, 1024, 16), (37, 3, 1000, 16)])
def test_noalloc_permute_matches_workspace_permute(T, K, E, H):
    m.lib()
    ids = torch.from_numpy(_ids(T, K, E, T + E)).cuda()
    x = torch.randn((T, H), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    want = _run(m.moe_permute, ids, x, T, K, E, H, True)
    for _ in range(2):
        got = _run(m.moe_permute_noalloc, ids, x, T, K, E, H, False)
        for g, w in zip(got, want):
            assert torch.equal(g, w)


def test_noalloc_permute_refuses_sizes_beyond_its_scratch():
    m.lib()
    # the limit P <= 512 * floor(2^18 / E): 16384 x 8 = 131072 pairs at E = 1024
    # fill the scratch exactly (accepted above); one more token is refused
    assert m.moe_permute_workspace_size(16384, 8, 1024) == m.PERMUTE_NOALLOC_MAX_SCRATCH
    T, K, E = 16385, 8, 1024
    assert m.moe_permute_workspace_size(T, K, E) > m.PERMUTE_NOALLOC_MAX_SCRATCH
    d = torch.zeros((16,), dtype=torch.int32, device="cuda")
    with pytest.raises(m.MoeError) as ei:
        m.moe_permute_noalloc(d, None, T, K, E, 0, d, d, d, None)
    assert ei.value.code == m.ERR_WORKSPACE and "scratch" in str(ei.value)
