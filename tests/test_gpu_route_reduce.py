"""GPU parity of moe_route_prepare (bit-exact routing metadata) and moe_reduce.

Route preparation: lmdeploy PR #4857 "optimize compact blocked FP8 MoE and route preparation"
("Changes", route-preparation table: 512 routes / 256 experts and 2,048 / 512, random top-8).
moe_reduce: lmdeploy PR #4228 "Moe Reduce kernel"."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_fp8_mixture_moe_gb300 import workloads as wl
from tests.gpu_util import bf16_host, bf16_to_dev, to_dev

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def _route_cases():
    with open(os.path.join(HERE, "golden", "page_shapes.json")) as f:
        g = json.load(f)["route_prepare"]
    cases = []
    for routes, experts in g["cases"]:
        cases.append((routes // g["topk"], g["topk"], experts, experts, 16, "uniform", 0.0))
    cases += [
        (1, 8, 256, 256, 16, "uniform", 0.0), (4, 8, 256, 256, 16, "uniform", 0.0),
        (16, 8, 256, 256, 16, "uniform", 0.0), (32, 8, 256, 256, 16, "uniform", 0.0),
        (4, 2, 16, 16, 16, "softmax", 0.0), (1024, 6, 256, 32, 64, "uniform", 0.0),
        (100, 6, 256, 32, 32, "uniform", 0.2), (512, 8, 512, 512, 64, "zipf", 0.0),
        (1024, 8, 4096, 4096, 128, "zipf", 0.05), (1, 1, 1, 1, 16, "uniform", 0.0),
        (1000, 8, 2048, 2048, 16, "uniform", 0.0), (3, 5, 7, 7, 128, "uniform", 0.5),
    ]
    return cases


def _gpu_route(ops, ids, E, emap, E_loc, bm, path):
    res = ops.moe_route_prepare(to_dev(ids), E, None if emap is None else to_dev(emap), E_loc, bm, path=path)
    torch.cuda.synchronize()
    return {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in res.items() if k != "_ws"}


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("M,k,E,E_loc,bm,kind,inv", _route_cases())
def test_route_prepare_bitwise(ops, M, k, E, E_loc, bm, kind, inv, path):
    R = M * k
    if path == 1 and (R > 8192 or E_loc > 2048):
        pytest.skip("outside the single-CTA path's limits")
    ids, _ = wl.routing_topk(M, E, k, seed=M * 7 + E, kind=kind)
    if inv:
        r = np.random.default_rng(M)
        ids = np.where(r.random(ids.shape) < inv, r.choice([-1, E, E + 9], ids.shape), ids).astype(np.int32)
    emap = None if E_loc == E else wl.expert_map_random(E, E_loc, seed=E_loc)
    got = _gpu_route(ops, ids, E, emap, E_loc, bm, path)
    ref = oracle.route_prepare(ids, E, emap, E_loc, bm)
    assert got["num_blocks"][0] == ref["num_blocks"]
    for key in ("sorted_idx", "block_expert", "expert_count", "expert_offset"):
        assert (got[key] == ref[key]).all(), key
    # route_slot is the inverse of sorted_idx
    rs = got["route_slot"]
    si = got["sorted_idx"]
    for r_ in range(R):
        if rs[r_] >= 0:
            assert si[rs[r_]] == r_
    assert (np.sort(rs[rs >= 0]) == np.sort(np.nonzero(si >= 0)[0])).all()
    assert ops.device_status() == 0


def test_route_prepare_flags_bad_map_entries(ops):
    E, E_loc = 16, 4
    ids = np.array([[0, 1], [2, 3], [4, 5]], np.int32)
    emap = np.full(E, -1, np.int32)
    emap[[0, 2, 4]] = [0, 1, 2]
    emap[3] = 9  # outside [-1, E_loc): dropped and flagged
    got = _gpu_route(ops, ids, E, emap, E_loc, 16, 0)
    emap_ok = emap.copy()
    emap_ok[3] = -1
    ref = oracle.route_prepare(ids, E, emap_ok, E_loc, 16)
    assert (got["sorted_idx"] == ref["sorted_idx"]).all()
    assert ops.device_status() & ops.DEV_BAD_EXPERT_MAP


def test_route_prepare_rejects_bad_arguments(ops):
    ids = to_dev(np.zeros((2, 2), np.int32))
    with pytest.raises(ops.MoeError):
        ops.moe_route_prepare(ids, 16, None, 8, 16)      # no map but E_local != E
    with pytest.raises(ops.MoeError):
        ops.moe_route_prepare(ids, 16, None, 16, 24)     # block_m not in {16, 32, 64, 128}
    with pytest.raises(ops.MoeError):
        ops.moe_route_prepare(ids, 16, None, 16, 0)


def test_route_prepare_empty(ops):
    got = _gpu_route(ops, np.zeros((0, 8), np.int32), 256, None, 256, 16, 0)
    assert got["num_blocks"][0] == 0 and (got["expert_count"] == 0).all()


@pytest.mark.parametrize("M,k,E,H,inv,use_map", [
    (1, 8, 256, 7168, 0.0, False), (32, 8, 256, 7168, 0.1, False), (7, 6, 256, 2048, 0.2, True),
    (512, 8, 512, 4096, 0.0, False), (3, 1, 4, 8, 0.0, False), (0, 8, 16, 512, 0.0, False),
    (1024, 6, 256, 2048, 0.0, True),   # expert-parallel shape: most routes dropped
    (5, 32, 64, 264, 0.3, False),      # the largest top-k, a ragged last 256-column chunk
    (9, 17, 40, 136, 0.0, True),
])
def test_moe_reduce_bitwise(ops, M, k, E, H, inv, use_map):
    """fp32 fused multiply-adds in top-k order on both sides: bit-exact."""
    ids, w = wl.routing_topk(M, E, k, seed=M + k)
    if inv:
        r = np.random.default_rng(1)
        ids = np.where(r.random(ids.shape) < inv, -1, ids).astype(np.int32)
    emap = wl.expert_map_random(E, max(1, E // 4), seed=2) if use_map else None
    z = wl.act_rows(M * k, H, 1.0, seed=H)
    out = ops.moe_reduce(bf16_to_dev(z), to_dev(w), to_dev(ids), None if emap is None else to_dev(emap), E, H,
                         E_local=None if emap is None else max(1, E // 4))
    torch.cuda.synchronize()
    ref = oracle.moe_reduce(z, w, ids, emap, E, H)
    assert (bf16_host(out) == ref).all()


def test_moe_reduce_drops_routes_with_out_of_range_map_entries(ops):
    """A map entry outside [0, E_local) drops the route in the reduce exactly as in route
    preparation (which gives such a route no slot, so its expert output is never written): the
    result equals the oracle's for the map with that entry set to -1."""
    M, k, E, E_loc, H = 16, 6, 64, 16, 512
    ids, w = wl.routing_topk(M, E, k, seed=77)
    emap = wl.expert_map_random(E, E_loc, seed=78)
    local_used = [g for g in np.unique(ids) if emap[g] >= 0]
    bad = emap.copy()
    bad[local_used[0]] = E_loc
    bad[local_used[1]] = E_loc + 100
    z = wl.act_rows(M * k, H, 1.0, seed=79)
    out = ops.moe_reduce(bf16_to_dev(z), to_dev(w), to_dev(ids), to_dev(bad), E, H, E_local=E_loc)
    torch.cuda.synchronize()
    ok = emap.copy()
    ok[local_used[0]] = -1
    ok[local_used[1]] = -1
    assert (bf16_host(out) == oracle.moe_reduce(z, w, ids, ok, E, H)).all()
    with pytest.raises(ValueError):
        ops.moe_reduce(bf16_to_dev(z), to_dev(w), to_dev(ids), to_dev(bad), E, H)  # E_local missing
