"""Whole-layer GPU parity: moe_blockfp8_forward (both paths: the fused persistent kernel and the
stage-by-stage launches) against the CPU oracle, BF16 outputs within |err| <= 2e-2 + 1e-2*|ref|,
on the pages' workload shapes (seeded synthetic inputs).

Full-size decode (H=7168, N=256, E=256, k=8, M=1..32) is compared on every output; the prefill
shape (M=512, H=4096, N=768, E=512, Zipf routing) on a token sample that includes the tokens of
the most loaded expert (each token's output depends only on its own routes, so a sampled
oracle row is exactly the full-run row)."""
import numpy as np
import pytest
import torch

import oracle
from block_fp8_mixture_moe_gb300 import workloads as wl
from tests.gpu_util import assert_bf16_close, bf16_host, bf16_to_dev, to_dev

pytestmark = pytest.mark.gpu
INF = float("inf")


FUSED, STAGED, EPI = 1, 2, 3  # moe_forward_path (EPI: staged, reduce in the down epilogue)


def _run(ops, L, act=1, clamp=INF, fmt=0, block_m=0, tiled=False, path=FUSED):
    emap = L["expert_map"]
    wgu, wd = L["wgu_q"], L["wd_q"]
    if tiled:
        wgu, wd = ops.moe_blockfp8_pack_weights(wgu), ops.moe_blockfp8_pack_weights(wd)
    out = ops.moe_blockfp8_forward(
        bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"]), L["E"],
        None if emap is None else to_dev(emap), wgu, L["wgu_s"], wd, L["wd_s"],
        act=act, clamp_limit=clamp, act_fmt=fmt, block_m=block_m, path=path)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    return bf16_host(out)


def _host(L, tokens=None):
    ids = L["topk_ids"] if tokens is None else L["topk_ids"][tokens]
    emap = L["expert_map"]
    loc = ids[(ids >= 0) & (ids < L["E"])]
    if emap is not None:
        loc = emap[loc]
    return wl.layer_numpy(L, experts=loc[loc >= 0])


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
@pytest.mark.parametrize("tiled", [False, True])
@pytest.mark.parametrize("act,clamp,fmt", [(1, INF, 0), (1, INF, 1), (1, 7.0, 1), (2, 1.0, 0)])
@pytest.mark.parametrize("block_m", [0, 16, 32, 64, 128])
def test_tiny_layer(ops, act, clamp, fmt, block_m, tiled, path):
    L = wl.make_layer(**wl.CONFIGS["tiny"], seed=0, device="cuda")
    got = _run(ops, L, act, clamp, fmt, block_m, tiled, path)
    ref = oracle.moe_forward(_host(L), act=act, clamp_limit=clamp, fmt=fmt)
    assert_bf16_close(got, ref, "tiny")


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
@pytest.mark.parametrize("M", wl.DECODE_M)
def test_decode_full_size(ops, M, path):
    cfg = dict(wl.CONFIGS["decode"], M=M)
    L = wl.make_layer(**cfg, seed=1, device="cuda")
    got = _run(ops, L, tiled=(M % 2 == 0), path=path)
    ref = oracle.moe_forward(_host(L))
    assert_bf16_close(got, ref, f"decode M={M}")


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
@pytest.mark.parametrize("T", wl.EP_TOKENS)
def test_expert_parallel_slice(ops, T, path):
    """k=6 of E=256 with 32 local experts through an expert map; non-local routes are dropped
    in every stage and add nothing to the output (T=1024 tokens = 6144 routed rows is compared
    on a 48-token sample, including tokens with no local route)."""
    cfg = dict(wl.CONFIGS["ep"], M=T)
    L = wl.make_layer(**cfg, seed=2, device="cuda")
    got = _run(ops, L, clamp=7.0, fmt=1, tiled=(T >= 100), path=path)
    if T <= 100:
        ref = oracle.moe_forward(_host(L), clamp_limit=7.0, fmt=1)
        assert_bf16_close(got, ref, f"ep T={T}")
    else:
        toks = np.random.default_rng(T).choice(T, 48, replace=False)
        ref = oracle.moe_forward(_host(L, toks), clamp_limit=7.0, fmt=1, tokens=toks)
        assert_bf16_close(got[toks], ref[toks], f"ep T={T} sample")
        # a token none of whose routes is local gets exactly zero
        emap = L["expert_map"]
        none_local = [t for t in range(T) if (emap[L["topk_ids"][t]] < 0).all()]
        if none_local:
            assert (oracle.bf16_to_f32(got[none_local]) == 0).all()


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
def test_prefill_zipf_sampled(ops, path):
    cfg = wl.CONFIGS["prefill"]
    L = wl.make_layer(**cfg, seed=3, device="cuda")
    got = _run(ops, L, tiled=True, path=path)
    ids = L["topk_ids"]
    hot = np.bincount(ids.reshape(-1), minlength=cfg["E"]).argmax()
    hot_tokens = np.nonzero((ids == hot).any(axis=1))[0]
    r = np.random.default_rng(0)
    toks = np.unique(np.concatenate([hot_tokens[:8], r.choice(cfg["M"], 16, replace=False), [0, cfg["M"] - 1]]))
    ref = oracle.moe_forward(_host(L, toks), tokens=toks)
    assert_bf16_close(got[toks], ref[toks], "prefill sample")


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
def test_invalid_routes_and_empty(ops, path):
    L = wl.make_layer(M=9, H=256, N=128, E=12, k=3, seed=4, device="cuda", invalid_frac=0.3)
    got = _run(ops, L, path=path)
    ref = oracle.moe_forward(_host(L))
    assert_bf16_close(got, ref, "invalid routes")
    # every route dropped: the output is exactly zero
    L2 = dict(L)
    L2["topk_ids"] = np.full_like(L["topk_ids"], -1)
    assert (f32 := oracle.bf16_to_f32(_run(ops, L2, path=path))).max() == 0 and f32.min() == 0
    # no tokens at all
    L3 = dict(L)
    L3["x"] = L["x"][:0]
    L3["topk_ids"] = L["topk_ids"][:0]
    L3["topk_w"] = L["topk_w"][:0]
    emap = None
    out = ops.moe_blockfp8_forward(
        torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"),
        torch.empty((0, 3), dtype=torch.int32, device="cuda"),
        torch.empty((0, 3), dtype=torch.float32, device="cuda"), 12, emap,
        L["wgu_q"], L["wgu_s"], L["wd_q"], L["wd_s"], path=path)
    assert out.shape == (0, 256)


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
def test_forward_is_deterministic_and_graph_capturable(ops, path):
    cfg = dict(wl.CONFIGS["decode"], M=4)
    L = wl.make_layer(**cfg, seed=5, device="cuda")
    x, ids, w = bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"])
    M, H = x.shape
    need = ops.moe_blockfp8_workspace_bytes(M, 8, 256, 256, H, 256)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    args = (x, ids, w, 256, None, L["wgu_q"], L["wgu_s"], L["wd_q"], L["wd_s"])
    ops.moe_blockfp8_forward(*args, out=out, workspace=ws, path=path)
    first = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        ops.moe_blockfp8_forward(*args, out=out, workspace=ws, stream=s, path=path)  # warm up on s
        torch.cuda.synchronize()
        out.zero_()
        with torch.cuda.graph(g, stream=s):
            ops.moe_blockfp8_forward(*args, out=out, workspace=ws, stream=s, path=path)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
@pytest.mark.parametrize("M", (64, 128, 256))
def test_decode_large_m_sampled(ops, M, path):
    """The decode sweep's larger batches (H=7168, N=256, E=256, k=8), compared on a token
    sample: each token's output depends only on its own routes, so a sampled oracle row is
    exactly the full-run row."""
    cfg = dict(wl.CONFIGS["decode"], M=M)
    L = wl.make_layer(**cfg, seed=6, device="cuda")
    got = _run(ops, L, tiled=True, path=path)
    toks = np.unique(np.concatenate([np.random.default_rng(M).choice(M, 12, replace=False), [0, M - 1]]))
    ref = oracle.moe_forward(_host(L, toks), tokens=toks)
    assert_bf16_close(got[toks], ref[toks], f"decode M={M} sample")


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
def test_decode_hot_experts(ops, path):
    """Decode shape with every route on 12 hot experts (64 routes each, so several block_m=16
    blocks per expert and 244 idle experts)."""
    M, E, k = 96, 256, 8
    cfg = dict(wl.CONFIGS["decode"], M=M)
    L = wl.make_layer(**cfg, seed=7, device="cuda")
    r = np.random.default_rng(7)
    hot = r.choice(E, 12, replace=False)
    ids = np.stack([hot[r.permutation(12)[:k]] for _ in range(M)]).astype(np.int32)
    w = r.random((M, k)).astype(np.float32) + 0.05
    L["topk_ids"], L["topk_w"] = ids, (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    got = _run(ops, L, tiled=True, path=path)
    toks = np.unique(np.concatenate([r.choice(M, 16, replace=False), [0, M - 1]]))
    ref = oracle.moe_forward(_host(L, toks), tokens=toks)
    assert_bf16_close(got[toks], ref[toks], "hot experts sample")


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
@pytest.mark.parametrize("M", [16, 3])
def test_graphs_with_different_routings_share_a_workspace(ops, path, M):
    """Three captured forwards with different routings on one workspace, replayed in a mixed
    order: every replay reproduces its own eager output bit for bit, so no state (counters,
    block tables, cleared regions) carries over from the previous call.  M = 3 (24 routes)
    runs the self-routed gate/up GEMM."""
    cfg = dict(wl.CONFIGS["decode"], M=M)
    L = wl.make_layer(**cfg, seed=8, device="cuda")
    H, E, k = cfg["H"], cfg["E"], cfg["k"]
    x = bf16_to_dev(L["x"])
    routes = []
    for s in range(3):
        i, w = wl.routing_topk(M, E, k, seed=100 + s, kind="uniform")
        routes.append((to_dev(i), to_dev(w)))
    need = ops.moe_blockfp8_workspace_bytes(M, k, E, E, H, cfg["N"])
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = [torch.empty((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    eager = []
    for s in range(3):
        ops.moe_blockfp8_forward(x, routes[s][0], routes[s][1], E, None, L["wgu_q"], L["wgu_s"],
                                 L["wd_q"], L["wd_s"], out=outs[s], workspace=ws, path=path)
        eager.append(outs[s].clone())
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    graphs = []
    with torch.cuda.stream(st):
        torch.cuda.synchronize()
        for s in range(3):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                ops.moe_blockfp8_forward(x, routes[s][0], routes[s][1], E, None, L["wgu_q"],
                                         L["wgu_s"], L["wd_q"], L["wd_s"], out=outs[s],
                                         workspace=ws, stream=st, path=path)
            graphs.append(g)
        for s in (0, 1, 2, 0, 2, 1, 1, 0):
            outs[s].zero_()
            graphs[s].replay()
            st.synchronize()
            assert torch.equal(outs[s], eager[s]), f"replay of routing {s} differs"
    assert ops.device_status() == 0
    for s in range(3):
        assert not torch.equal(eager[s], eager[(s + 1) % 3])


@pytest.mark.parametrize("path", [FUSED, STAGED, EPI])
def test_host_activations_zero_copy(ops, path):
    """x, topk_ids, topk_w and out in pinned host memory: the kernels read and write them across
    the host link, bit for bit the result of the same call on device copies (decode M=16, and
    an expert-parallel slice with dropped routes and UE8M0 scales)."""
    cases = [(dict(wl.CONFIGS["decode"], M=16), 9, {}),
             (dict(wl.CONFIGS["decode"], M=4), 11, {}),  # 32 routes: the self-routed gate/up GEMM
             (dict(wl.CONFIGS["ep"], M=10), 10, dict(clamp_limit=7.0, act_fmt=1))]
    for cfg, seed, kw in cases:
        L = wl.make_layer(**cfg, seed=seed, device="cuda")
        emap = None if L["expert_map"] is None else to_dev(L["expert_map"])
        x_d, ids_d, w_d = bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"])
        args = (L["E"], emap, L["wgu_q"], L["wgu_s"], L["wd_q"], L["wd_s"])
        ref = ops.moe_blockfp8_forward(x_d, ids_d, w_d, *args, path=path, **kw)
        x_h, ids_h, w_h = x_d.cpu().pin_memory(), ids_d.cpu().pin_memory(), w_d.cpu().pin_memory()
        out_h = torch.empty(ref.shape, dtype=torch.bfloat16).pin_memory()
        for t in (x_h, ids_h, w_h, out_h):
            assert ops.pointer_device_accessible(t)
        ops.moe_blockfp8_forward(x_h, ids_h, w_h, *args, out=out_h, path=path, **kw)
        torch.cuda.synchronize()
        assert ops.device_status() == 0
        assert torch.equal(out_h, ref.cpu())
    # pageable host memory is refused before anything is launched
    assert not ops.pointer_device_accessible(torch.zeros(4))
    with pytest.raises(AssertionError):
        ops.moe_blockfp8_forward(x_d.cpu(), ids_d, w_d, *args, path=path, **kw)


@pytest.mark.parametrize("case", ["decode1", "decode4", "decode32", "decode64", "ep_t1", "ep_t100",
                                  "dropped", "topk32", "bm32"])
def test_epilogue_reduce_is_bitwise_the_staged_output(ops, case):
    """The weighted top-k sum done in the down GEMM's epilogue (per-token ownership: the arrival
    that completes a token's kept routes sums it, in top-k order) gives bit for bit the separate
    reduce kernel's output, including zero rows for tokens with no kept route."""
    kw, block_m = {}, 0
    if case.startswith("decode"):
        cfg, seed = dict(wl.CONFIGS["decode"], M=int(case[6:])), 40
    elif case.startswith("ep_t"):
        cfg, seed, kw = dict(wl.CONFIGS["ep"], M=int(case[4:])), 41, dict(clamp_limit=7.0, act_fmt=1)
    elif case == "dropped":
        cfg, seed = dict(M=9, H=256, N=128, E=12, k=3, invalid_frac=0.4), 42
    elif case == "topk32":
        cfg, seed = dict(M=5, H=384, N=128, E=40, k=32), 43
    else:
        cfg, seed, block_m = dict(wl.CONFIGS["decode"], M=16), 44, 32
    L = wl.make_layer(**cfg, seed=seed, device="cuda")
    emap = None if L["expert_map"] is None else to_dev(L["expert_map"])
    args = (bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"]), L["E"], emap,
            L["wgu_q"], L["wgu_s"], L["wd_q"], L["wd_s"])
    ref = ops.moe_blockfp8_forward(*args, path=STAGED, block_m=block_m, **kw)
    got = ops.moe_blockfp8_forward(*args, path=EPI, block_m=block_m, **kw)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    assert torch.equal(got, ref)
