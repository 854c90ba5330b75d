"""moe_permute_noalloc against moe_permute, on the GPU, through the C ABI.

moe_permute_noalloc serves callers that may not allocate device memory (a
runtime that plans every device buffer at start-up, a plugin interface that
passes an operator only its inputs and outputs): its scratch is a fixed array
inside the library instead of a caller workspace.  Its results must equal the
workspace version's bit for bit, and two calls in a row must not see each
other's leftovers in the shared array.  This file is collected last so that a
run stopping at the first failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
from tests._lib import ensure_library

pytestmark = pytest.mark.gpu


def _outputs(T, E, k, D):
    R = T * k
    dev = "cuda"
    return dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                sorted_rows=torch.empty(R, dtype=torch.int32, device=dev),
                dest=torch.empty(R, dtype=torch.int32, device=dev),
                x_perm=torch.empty((R, D), dtype=torch.bfloat16, device=dev))


def _ids(T, E, k, seed, skew):
    rng = np.random.default_rng(seed)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.3
        p /= p.sum()
        rows = [rng.choice(E, k, replace=False, p=p) for _ in range(T)]
    else:
        rows = [rng.permutation(E)[:k] for _ in range(T)]
    return torch.from_numpy(np.stack(rows).astype(np.int32)).cuda()


def test_noalloc_permute_matches_workspace_permute_twice():
    assert torch.cuda.is_available(), "GPU test"
    ensure_library()
    T, E, k, D = 3000, 128, 8, 264
    x = torch.randn((T, D), device="cuda").to(torch.bfloat16)
    cfg = moe.make_config(T, D, E, k, 64)
    ws = moe.alloc_workspace(cfg)
    # two calls in a row with different routings: the second must not see the
    # first call's histogram left in the shared array
    for seed, skew in ((1, False), (2, True)):
        ids = _ids(T, E, k, seed, skew)
        ref = _outputs(T, E, k, D)
        moe.moe_permute(cfg, ids, x, ref["counts"], ref["offsets"], ref["sorted_rows"], ref["dest"],
                        ref["x_perm"], ws)
        got = _outputs(T, E, k, D)
        moe.moe_permute_noalloc(cfg, ids, x, got["counts"], got["offsets"], got["sorted_rows"],
                                got["dest"], got["x_perm"])
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(ws) == 0
        for name in ref:
            assert torch.equal(got[name], ref[name]), f"{name} differs (call with seed {seed})"


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    ensure_library()
    # at most 2^30 expanded rows
    cfg = moe.make_config(1 << 28, 64, 512, 8, 64)  # T*k = 2^31
    d = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_permute_noalloc(cfg, d, None, d, d, d, d, None)
    assert ei.value.status == -1
