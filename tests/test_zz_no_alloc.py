"""moe_permute_noalloc against moe_permute, on the GPU, through the C ABI.

moe_permute_noalloc serves callers that may not allocate device memory (a
runtime that plans every device buffer at start-up, a plugin interface that
passes an operator only its inputs and outputs): its scratch is a fixed array
inside the library instead of a caller workspace.  Its results must equal the
workspace version's bit for bit, and two calls in a row must not see each
other's leftovers in the shared array.  The cases cover the array filled
exactly (512 experts x 128 routing segments), batches of at most 8192
expanded rows (where moe_permute sorts and gathers in one kernel while this
call runs the histogram and scatter kernels), no x (routing only), and an
expert id out of range.  This file is collected last so that a run stopping
at the first failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
from tests._lib import ensure_library

pytestmark = pytest.mark.gpu


def _outputs(T, E, k, D, fill=None):
    R = T * k
    dev = "cuda"
    mk = (lambda n: torch.full((n,), fill, dtype=torch.int32, device=dev)) if fill is not None else \
        (lambda n: torch.empty(n, dtype=torch.int32, device=dev))
    return dict(counts=mk(E), offsets=mk(E + 1), sorted_rows=mk(R), dest=mk(R),
                x_perm=torch.zeros((R, D), dtype=torch.bfloat16, device=dev))


def _ids(T, E, k, seed, skew):
    rng = np.random.default_rng(seed)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.3
        p /= p.sum()
        rows = [rng.choice(E, k, replace=False, p=p) for _ in range(T)]
    else:
        rows = [rng.permutation(E)[:k] for _ in range(T)]
    return torch.from_numpy(np.stack(rows).astype(np.int32)).cuda()


# (T, E, k, D, with x): 47 routing segments; the scratch array exactly full
# (T*k = 65536 -> 128 segments of 512 rows, times 512 experts = 65536 entries);
# T*k <= 8192 (moe_permute's one-launch path); routing only (x = NULL)
CASES = {
    "segments_47": (3000, 128, 8, 264, True),
    "scratch_full_E512": (8192, 512, 8, 64, True),
    "small_batch": (1000, 128, 8, 136, True),
    "no_x": (2500, 64, 6, 64, False),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_permute_matches_workspace_permute_twice(case):
    assert torch.cuda.is_available(), "GPU test"
    ensure_library()
    T, E, k, D, with_x = CASES[case]
    x = torch.randn((T, D), device="cuda").to(torch.bfloat16) if with_x else None
    cfg = moe.make_config(T, D, E, k, 64)
    ws = moe.alloc_workspace(cfg)
    # two calls in a row with different routings: the second must not see the
    # first call's histogram left in the shared array
    for seed, skew in ((1, False), (2, True)):
        ids = _ids(T, E, k, seed, skew)
        ref = _outputs(T, E, k, D)
        moe.moe_permute(cfg, ids, x, ref["counts"], ref["offsets"], ref["sorted_rows"], ref["dest"],
                        ref["x_perm"] if with_x else None, ws)
        got = _outputs(T, E, k, D)
        moe.moe_permute_noalloc(cfg, ids, x, got["counts"], got["offsets"], got["sorted_rows"],
                                got["dest"], got["x_perm"] if with_x else None)
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(ws) == 0
        for name in ref:
            assert torch.equal(got[name], ref[name]), f"{name} differs (call with seed {seed})"


def test_noalloc_permute_out_of_range_id():
    """One id equal to E: that row gets dest = -1 and stays out of sorted_rows;
    the other rows are sorted as if it were absent, offsets[E] = T*k - 1, and
    the valid permuted rows are the copies of x they name."""
    ensure_library()
    T, E, k, D = 2100, 32, 4, 72
    R = T * k
    x = torch.randn((T, D), device="cuda").to(torch.bfloat16)
    ids = _ids(T, E, k, 5, False)
    bad = 1234
    ids.view(-1)[bad] = E
    cfg = moe.make_config(T, D, E, k, 64)
    got = _outputs(T, E, k, D, fill=-7)
    for _ in range(2):
        moe.moe_permute_noalloc(cfg, ids, x, got["counts"], got["offsets"], got["sorted_rows"],
                                got["dest"], got["x_perm"])
        torch.cuda.synchronize()
        flat = ids.view(-1).cpu().numpy().astype(np.int64)
        valid = flat < E
        counts = np.bincount(flat[valid], minlength=E)
        rows = np.arange(R)[valid]
        order = rows[np.argsort(flat[valid], kind="stable")]  # stable sort of the valid rows
        dest = np.full(R, -1, dtype=np.int64)
        dest[order] = np.arange(order.size)
        assert np.array_equal(got["counts"].cpu().numpy(), counts)
        assert np.array_equal(got["offsets"].cpu().numpy(), np.concatenate([[0], np.cumsum(counts)]))
        assert int(got["offsets"][E]) == R - 1
        n = order.size
        assert np.array_equal(got["sorted_rows"].cpu().numpy()[:n], order)
        assert np.array_equal(got["dest"].cpu().numpy(), dest)
        assert torch.equal(got["x_perm"][:n].cpu(), x.cpu()[torch.from_numpy(order // k)])


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    ensure_library()
    # at most 2^30 expanded rows
    cfg = moe.make_config(1 << 28, 64, 512, 8, 64)  # T*k = 2^31
    d = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_permute_noalloc(cfg, d, None, d, d, d, d, None)
    assert ei.value.status == -1
