"""The allocation-free route preparation (moe_route_prepare_noalloc), called through the C ABI,
gives the same routing metadata as moe_route_prepare with a caller workspace -- bit for bit,
the bar every routing test uses -- on two calls in a row that reuse its fixed scratch array.

This file is collected last so that a stop-at-first-failure run has run every other test
first; it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_moe_gb300 import workloads as wl
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

KEYS = ("sorted_idx", "block_expert", "num_blocks", "expert_count", "expert_offset", "route_slot")


def _compare(ops, M, k, E, E_loc, bm, kind, seed):
    ids, _ = wl.routing_topk(M, E, k, seed=seed, kind=kind)
    emap = None if E_loc == E else wl.expert_map_random(E, E_loc, seed=seed + 1)
    ids_d = to_dev(ids)
    emap_d = None if emap is None else to_dev(emap)
    ref = ops.moe_route_prepare(ids_d, E, emap_d, E_loc, bm, path=ops.ROUTE_MULTI_CTA)
    got = ops.moe_route_prepare_noalloc(ids_d, E, emap_d, E_loc, bm)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(got[key], ref[key]), key
    auto = ops.moe_route_prepare(ids_d, E, emap_d, E_loc, bm)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(got[key], auto[key]), key


def test_noalloc_matches_workspace_route_prepare_twice_in_a_row(ops):
    # first call: prefill-shaped Zipf routing, 4096 routes over 512 experts, block_m 64
    _compare(ops, 512, 8, 512, 512, 64, "zipf", seed=11)
    # second call reuses the scratch left by the first: expert-parallel slice, block_m 16
    _compare(ops, 1024, 6, 256, 32, 16, "uniform", seed=12)
    assert ops.device_status() == 0


def test_noalloc_at_its_maximum_size_then_a_smaller_call(ops):
    """Every part of the fixed scratch in use: 65,536 routes (64 chunk histograms) over 1,024
    local experts of 2,048 through an expert map, block_m 128; then a small call that reuses the
    array (its ticket counter and offsets from the large call are still there)."""
    _compare(ops, 8192, 8, 2048, 1024, 128, "uniform", seed=13)
    _compare(ops, 37, 3, 64, 64, 16, "zipf", seed=14)
    assert ops.device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(ops):
    ids = to_dev(np.zeros((8193, 8), np.int32))  # 65,544 routes > 65,536
    with pytest.raises(ops.MoeError, match="at most 65536 routes"):
        ops.moe_route_prepare_noalloc(ids, 16, None, 16, 16)
    ids = to_dev(np.zeros((4, 2), np.int32))
    with pytest.raises(ops.MoeError, match="1024 local experts"):
        ops.moe_route_prepare_noalloc(ids, 2048, None, 2048, 16)
    ids = to_dev(np.zeros((2, 5), np.int32))
    with pytest.raises(ops.MoeError, match="top-k 5 > E 4"):
        ops.moe_route_prepare_noalloc(ids, 4, None, 4, 16)
