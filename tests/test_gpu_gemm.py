"""GPU parity of moe_blockfp8_grouped_gemm (tcgen05 kernel) against the oracle's per-route
block-scaled GEMM, within |err| <= 2e-2 + 1e-2*|ref| (fp32 accumulation in a different order
than the oracle's exact K-block sums).

Method: lmdeploy PR #4956 "Perf/pytorch block fp8 moe decode" ("Active-expert block
scheduling") and lmdeploy PR #4857 ("Changes": compact blocks, transposed MMA); W8A8 block
shape [128, 128] (vLLM PR #53875, "Purpose")."""
import numpy as np
import pytest
import torch

import oracle
from block_fp8_mixture_moe_gb300 import workloads as wl
from tests.gpu_util import assert_bf16_close, bf16_host, to_dev

pytestmark = pytest.mark.gpu


def _setup(ops, M, k, E, E_loc, bm, K, N_out, kind="uniform", seed=0, inv=0.0):
    ids, _ = wl.routing_topk(M, E, k, seed=seed, kind=kind)
    if inv:
        r = np.random.default_rng(seed)
        ids = np.where(r.random(ids.shape) < inv, -1, ids).astype(np.int32)
    emap = None if E_loc == E else wl.expert_map_random(E, E_loc, seed=seed + 1)
    route = ops.moe_route_prepare(to_dev(ids), E, None if emap is None else to_dev(emap), E_loc, bm)
    ref_route = oracle.route_prepare(ids, E, emap, E_loc, bm)
    slots = route["B_cap"] * bm
    # activations in slot order: realistic per-128 quantised rows; pad slots hold NaN codes so
    # any leak of a pad column into a real output shows up
    x = wl.act_rows(max(slots, 1), K, 1.0, seed=seed + 2)[:slots]
    aq, a_s = oracle.act_quant(0, x, K)
    si = ref_route["sorted_idx"]
    aq[si < 0] = 0x7F
    a_s[si < 0] = np.nan
    wq, ws = wl.quantized_weights(E_loc, N_out, K, seed=seed + 3, device="cuda")
    return route, ref_route, aq, a_s, wq, ws


def _oracle_rows(ref_route, aq, a_s, wq_h, ws_h, bm):
    si = ref_route["sorted_idx"]
    valid = np.nonzero(si >= 0)[0].astype(np.int32)
    rexp = ref_route["block_expert"][valid // bm].astype(np.int32)
    out = oracle.route_gemm(aq, a_s, wq_h, ws_h, valid, rexp)
    return valid, out


@pytest.mark.parametrize("tiled", [False, True])
@pytest.mark.parametrize("proj", [0, 1])
@pytest.mark.parametrize("M,k,E,E_loc,bm,K,N_out,kind", [
    (1, 8, 256, 256, 16, 7168, 512, "uniform"),     # decode gate/up, one token
    (32, 8, 256, 256, 16, 1024, 512, "uniform"),
    (32, 8, 256, 256, 16, 256, 1024, "uniform"),    # decode-like down (K = N = 256)
    (100, 6, 256, 32, 32, 2048, 512, "uniform"),    # expert-parallel slice
    (64, 8, 512, 512, 64, 1024, 384, "zipf"),       # skewed routing, block_m 64
    (300, 2, 4, 4, 128, 512, 256, "uniform"),       # many tokens per expert, block_m 128
    (5, 3, 7, 7, 16, 128, 128, "uniform"),          # one K-block, one tile
    (128, 4, 4, 4, 16, 1024, 256, "uniform"),       # runs of 8 blocks of one expert
    (600, 2, 2, 2, 16, 256, 384, "uniform"),        # runs longer than 32 blocks
])
def test_gemm_bf16_vs_oracle(ops, proj, M, k, E, E_loc, bm, K, N_out, kind, tiled):
    route, rr, aq, a_s, wq, ws = _setup(ops, M, k, E, E_loc, bm, K, N_out, kind, seed=M + K)
    slots = route["B_cap"] * bm
    R = M * k
    out_rows = slots if proj == 0 else R
    sentinel = torch.full((out_rows, N_out), -7.0, dtype=torch.bfloat16, device="cuda")
    w_used = ops.moe_blockfp8_pack_weights(wq) if tiled else wq
    out = ops.moe_blockfp8_grouped_gemm(proj, to_dev(aq), to_dev(a_s), w_used, ws, route, bm,
                                        out_dtype=ops.DTYPE_BF16, out_rows=out_rows, out=sentinel)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    wq_h, ws_h = wq.cpu().numpy(), ws.cpu().numpy()
    valid, ref = _oracle_rows(rr, aq, a_s, wq_h, ws_h, bm)
    got = bf16_host(out)
    rows = valid if proj == 0 else rr["sorted_idx"][valid]
    assert_bf16_close(got[rows], ref, f"proj {proj}")
    # rows that no route writes keep the sentinel
    untouched = np.setdiff1d(np.arange(out_rows), rows)
    assert (got[untouched] == bf16_host(torch.tensor([-7.0], dtype=torch.bfloat16))[0]).all()


@pytest.mark.parametrize("splits", [1, 3, 7, 56])
def test_gemm_fp32_split_partials(ops, splits):
    """Split p covers K-blocks [p*KB/S, (p+1)*KB/S): each partial equals the oracle GEMM over
    that slice of K, and the partials sum to the full product."""
    M, k, E, bm, K, N_out = 4, 8, 64, 16, 7168, 256
    route, rr, aq, a_s, wq, ws = _setup(ops, M, k, E, E, bm, K, N_out, seed=splits)
    slots = route["B_cap"] * bm
    out = ops.moe_blockfp8_grouped_gemm(0, to_dev(aq), to_dev(a_s), wq, ws, route, bm,
                                        out_dtype=ops.DTYPE_F32, out_rows=slots, splits=splits)
    torch.cuda.synchronize()
    P = out.cpu().numpy()
    wq_h, ws_h = wq.cpu().numpy(), ws.cpu().numpy()
    si = rr["sorted_idx"]
    valid = np.nonzero(si >= 0)[0].astype(np.int32)
    rexp = rr["block_expert"][valid // bm].astype(np.int32)
    KB = K // 128
    for p in range(splits):
        kb0, kb1 = p * KB // splits, (p + 1) * KB // splits
        sl = slice(kb0 * 128, kb1 * 128)
        ref = oracle.route_gemm(np.ascontiguousarray(aq[:, sl]), np.ascontiguousarray(a_s[:, kb0:kb1]),
                                np.ascontiguousarray(wq_h[:, :, sl]), np.ascontiguousarray(ws_h[:, :, kb0:kb1]),
                                valid, rexp)
        got = oracle.bf16_round(P[p][valid])
        assert_bf16_close(got, ref, f"split {p}")
    full = oracle.route_gemm(aq, a_s, wq_h, ws_h, valid, rexp)
    assert_bf16_close(oracle.bf16_round(P.sum(axis=0)[valid]), full, "sum of partials")


def test_gemm_no_active_blocks(ops):
    """Every route dropped: no blocks, nothing is written."""
    M, k, E, bm, K, N_out = 8, 4, 16, 16, 256, 128
    ids = np.full((M, k), -1, np.int32)
    route = ops.moe_route_prepare(to_dev(ids), E, None, E, bm)
    slots = route["B_cap"] * bm
    aq = torch.zeros((slots, K), dtype=torch.uint8, device="cuda")
    a_s = torch.ones((slots, K // 128), dtype=torch.float32, device="cuda")
    wq, ws = wl.quantized_weights(E, N_out, K, seed=1, device="cuda")
    out = torch.full((slots, N_out), 3.0, dtype=torch.bfloat16, device="cuda")
    ops.moe_blockfp8_grouped_gemm(0, aq, a_s, wq, ws, route, bm, out=out, out_rows=slots)
    torch.cuda.synchronize()
    assert route["num_blocks"].item() == 0
    assert (out == 3.0).all()


def test_gemm_rejects_bad_arguments(ops):
    M, k, E, bm = 2, 2, 4, 16
    route = ops.moe_route_prepare(to_dev(np.zeros((M, k), np.int32)), E, None, E, bm)
    slots = route["B_cap"] * bm
    aq = torch.zeros((slots, 200), dtype=torch.uint8, device="cuda")  # K not a multiple of 128
    a_s = torch.ones((slots, 2), dtype=torch.float32, device="cuda")
    wq = torch.zeros((E, 128, 200), dtype=torch.uint8, device="cuda")
    ws = torch.ones((E, 1, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(ops.MoeError):
        ops.moe_blockfp8_grouped_gemm(0, aq, a_s, wq, ws, route, bm)
    aq = torch.zeros((slots, 256), dtype=torch.uint8, device="cuda")
    wq = torch.zeros((E, 128, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.MoeError):  # BF16 output with splits > 1
        ops.moe_blockfp8_grouped_gemm(0, aq, a_s, wq, ws, route, bm, splits=2)


def test_pack_weights_is_the_tile_regrouping(ops):
    """tiled[e, nt, kb, r, c] == w[e, nt*128 + r, kb*128 + c] (a pure data movement, checked
    against torch's view/permute of the same bytes)."""
    wq, _ = wl.quantized_weights(3, 384, 640, seed=4, device="cuda")
    t = ops.moe_blockfp8_pack_weights(wq)
    torch.cuda.synchronize()
    ref = wq.view(3, 3, 128, 5, 128).permute(0, 1, 3, 2, 4).contiguous()
    assert torch.equal(t, ref)


@pytest.mark.parametrize("proj", [0, 1])
@pytest.mark.parametrize("M,k,E,bm,K,N_out,hot", [
    (1, 8, 256, 16, 7168, 512, False),    # decode M=1: 8 active experts, 248 empty blocks
    (32, 8, 256, 16, 7168, 512, False),   # decode M=32: ~165 active experts
    (48, 4, 16, 16, 1024, 256, True),     # hot experts: several blocks per expert, 8 empty
])
def test_padded_grid_arm_vs_oracle(ops, proj, M, k, E, bm, K, N_out, hot):
    """The padded-grid schedule (every expert owns a block, empty ones included), run through
    the same grouped GEMM, computes the rows of the kept routes exactly as the compact schedule
    does (oracle, within the GEMM tolerance) and writes nothing else -- so the active-block
    comparison of the bench times a checked arm (lmdeploy PR #4956, "Motivation")."""
    seed = M + K + (7 if hot else 0)
    if hot:
        r = np.random.default_rng(seed)
        ids = np.stack([r.choice(8, k, replace=False) for _ in range(M)]).astype(np.int32)
    else:
        ids, _ = wl.routing_topk(M, E, k, seed=seed, kind="uniform")
    rr = oracle.route_prepare(ids, E, None, E, bm)
    pg = wl.padded_grid_route(rr["sorted_idx"], rr["block_expert"], rr["num_blocks"], E, bm)
    assert pg["num_blocks"] == sum(max(1, int(np.ceil(c / bm))) for c in rr["expert_count"])
    slots_p = pg["B_cap"] * bm
    # activations in padded-grid slot order; every slot without a route holds NaN codes
    x = wl.act_rows(slots_p, K, 1.0, seed=seed + 2)
    aq, a_s = oracle.act_quant(0, x, K)
    aq[pg["sorted_idx"] < 0] = 0x7F
    a_s[pg["sorted_idx"] < 0] = np.nan
    wq, ws = wl.quantized_weights(E, N_out, K, seed=seed + 3, device="cuda")
    route = dict(sorted_idx=to_dev(pg["sorted_idx"]), block_expert=to_dev(pg["block_expert"]),
                 num_blocks=to_dev(np.array([pg["num_blocks"]], np.int32)), B_cap=pg["B_cap"])
    R = M * k
    out_rows = slots_p if proj == 0 else R
    sentinel = torch.full((out_rows, N_out), -7.0, dtype=torch.bfloat16, device="cuda")
    out = ops.moe_blockfp8_grouped_gemm(proj, to_dev(aq), to_dev(a_s), wq, ws, route, bm,
                                        out_dtype=ops.DTYPE_BF16, out_rows=out_rows, out=sentinel)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    used = np.unique(pg["block_expert"][np.nonzero(pg["sorted_idx"] >= 0)[0] // bm])
    used_d = torch.from_numpy(used.astype(np.int64)).cuda()
    wq_h = np.zeros(tuple(wq.shape), np.uint8)
    ws_h = np.ones(tuple(ws.shape), np.float32)
    wq_h[used] = wq[used_d].cpu().numpy()
    ws_h[used] = ws[used_d].cpu().numpy()
    valid = np.nonzero(pg["sorted_idx"] >= 0)[0].astype(np.int32)
    rexp = pg["block_expert"][valid // bm].astype(np.int32)
    ref = oracle.route_gemm(aq, a_s, wq_h, ws_h, valid, rexp)
    got = bf16_host(out)
    rows = valid if proj == 0 else pg["sorted_idx"][valid]
    assert_bf16_close(got[rows], ref, f"padded grid proj {proj}")
    untouched = np.setdiff1d(np.arange(out_rows), rows)
    assert (got[untouched] == bf16_host(torch.tensor([-7.0], dtype=torch.bfloat16))[0]).all()
    # the compact slots map onto the padded grid one to one, routes unchanged
    cs = np.nonzero(rr["sorted_idx"] >= 0)[0]
    assert (pg["sorted_idx"][pg["slot_map"][cs]] == rr["sorted_idx"][cs]).all()
