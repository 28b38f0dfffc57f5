"""GPU parity of silu_mul_quant_fp8 / silu_and_mul_bf16 against the CPU oracle.

E4M3 codes and scales are integers decided by floating point in the same precision on both
sides, so every comparison here is bit-exact (vLLM PR #53875 "Fuse clamped MoE activation and
UE8M0 FP8 block quantization", "Correctness and validation": output bytes and scales must match
bit for bit; lmdeploy PR #4956 "Perf/pytorch block fp8 moe decode": the fused activation is
bitwise equal to quant_fp8(silu_and_mul(x)))."""
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
INF = float("inf")


def _gpu_quant(ops, act, x_u16, N, **kw):
    q, s = ops.silu_mul_quant_fp8(act, bf16_to_dev(x_u16), N, **kw)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("strategy", [1, 2])
@pytest.mark.parametrize("rows,N", [(1, 128), (8, 256), (37, 512), (300, 1024), (1024, 2048), (5, 7168)])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("act,clamp", [(0, INF), (1, INF), (1, 7.0), (2, 3.0)])
def test_bitwise_vs_oracle(ops, act, clamp, fmt, rows, N, strategy):
    W = N if act == 0 else 2 * N
    x = wl.act_rows(rows, W, 2.0, seed=rows * 31 + N + act)
    q, s = _gpu_quant(ops, act, x, N, clamp_limit=clamp, fmt=fmt, strategy=strategy)
    rq, rs = oracle.act_quant(act, x, N, clamp_limit=clamp, fmt=fmt)
    assert (q == rq).all(), f"{(q != rq).sum()} codes differ"
    assert (s == rs).all(), f"{(s != rs).sum()} scales differ"
    assert ops.device_status() == 0


def _grid():
    with open(os.path.join(HERE, "golden", "page_shapes.json")) as f:
        g = json.load(f)["act_quant_regression_grid"]
    for h in g["hidden"]:
        for r in g["routed_rows"]:
            for flt in g["filter"]:
                for fmt in g["scale_fmt"]:
                    yield h, r, flt, fmt


@pytest.mark.parametrize("hidden,rows,flt,fmt", list(_grid()))
def test_page_regression_grid(ops, hidden, rows, flt, fmt):
    """The page's grid: hidden 512/2048 x routed rows 8/128/1024 x filter none/IDs/expert map x
    scales fp32/UE8M0, clamped SiLU; filtered rows stay untouched."""
    fmt_i = 1 if fmt == "ue8m0" else 0
    E = 288
    x = wl.act_rows(rows, 2 * hidden, 2.0, seed=hidden + rows)
    r = np.random.default_rng(rows)
    ids = emap = None
    if flt != "none":
        ids = r.integers(-3, E + 3, rows).astype(np.int32)
    if flt == "expert_map":
        emap = np.where(r.random(E) < 0.125, np.arange(E), -1).astype(np.int32)
    q0 = np.full((rows, hidden), 0x5A, np.uint8)
    s0 = np.full((rows, hidden // 128), 123.0, np.float32)
    q, s = ops.silu_mul_quant_fp8(1, bf16_to_dev(x), hidden, clamp_limit=7.0, fmt=fmt_i,
                                  row_expert=None if ids is None else to_dev(ids),
                                  expert_map=None if emap is None else to_dev(emap), E=E,
                                  out_q=to_dev(q0.copy()), out_s=to_dev(s0.copy()))
    torch.cuda.synchronize()
    rq, rs = oracle.act_quant(1, x, hidden, clamp_limit=7.0, fmt=fmt_i, row_expert=ids,
                              expert_map=emap, E=E, out_q=q0.copy(), out_s=s0.copy())
    assert (q.cpu().numpy() == rq).all() and (s.cpu().numpy() == rs).all()
    if flt != "none":
        kept = (ids >= 0) & (ids < E)
        if emap is not None:
            kept[kept] &= emap[ids[kept]] >= 0
        assert (q.cpu().numpy()[~kept] == 0x5A).all()


@pytest.mark.parametrize("act,clamp", [(1, INF), (1, 7.0), (2, 1.0)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_fused_equals_two_kernel_path_on_gpu(ops, act, clamp, fmt):
    """The separate-kernel arm (BF16 SiLU*mul written to memory, then quantised) gives the same
    bytes as the fused kernel."""
    x = wl.act_rows(256, 1024, 2.0, seed=5)
    xd = bf16_to_dev(x)
    q, s = ops.silu_mul_quant_fp8(act, xd, 512, clamp_limit=clamp, fmt=fmt)
    mid = ops.silu_and_mul_bf16(act, xd, 512, clamp_limit=clamp)
    q2, s2 = ops.silu_mul_quant_fp8(0, mid, 512, fmt=fmt)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s, s2)
    # and the BF16 intermediate equals the oracle's
    assert (bf16_host(mid) == oracle.silu_and_mul(act, x, 512, clamp_limit=clamp)).all()


def test_silu_sweep_bitwise(ops):
    """A dense sweep of gate values with up = 1: the BF16 SiLU values match the oracle's (the
    exponential and division are the same fp32 operations on both sides)."""
    g = np.linspace(-120, 120, 2 ** 20, dtype=np.float32)
    g = np.concatenate([g, np.linspace(-2, 2, 2 ** 18, dtype=np.float32)])
    n = (g.size // 1024) * 1024
    g = g[:n].reshape(-1, 1024)
    gu = np.concatenate([g, np.ones_like(g)], axis=1)
    x = torch.from_numpy(gu).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out = bf16_host(ops.silu_and_mul_bf16(1, bf16_to_dev(x), 1024))
    assert (out == oracle.silu_and_mul(1, x, 1024)).all()


@pytest.mark.parametrize("splits", [1, 2, 5])
def test_fp32_split_partials_input(ops, splits):
    """Split-K partials: summed in split order in fp32, rounded to BF16, then SiLU*mul + quant.
    The reference sums the same partials in the same order with torch's fp32 adds."""
    rows, N = 40, 256
    r = np.random.default_rng(splits)
    P = r.standard_normal((splits, rows, 2 * N)).astype(np.float32) * 1.5
    acc = torch.from_numpy(P[0].copy())
    for i in range(1, splits):
        acc = acc + torch.from_numpy(P[i])
    gu = acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, s = ops.silu_mul_quant_fp8(1, to_dev(P), N, in_splits=splits, clamp_limit=7.0, fmt=1)
    rq, rs = oracle.act_quant(1, gu, N, clamp_limit=7.0, fmt=1)
    assert (q.cpu().numpy() == rq).all() and (s.cpu().numpy() == rs).all()


def _split_sum_bf16(P):
    """bf16 bits of the split partials summed in split order with fp32 adds (torch)."""
    acc = torch.from_numpy(P[0].copy())
    for i in range(1, P.shape[0]):
        acc = acc + torch.from_numpy(P[i])
    return acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("rows", [40, 700, 1400])
@pytest.mark.parametrize("act,clamp,fmt", [(1, float("inf"), 0), (1, 7.0, 1), (2, 7.0, 0), (2, float("inf"), 1)])
@pytest.mark.parametrize("splits", [1, 3, 4, 6])
def test_persistent_split_partials(ops, splits, act, clamp, fmt, rows):
    """The persistent launch on split-K partials, as the layer runs it.  At most 4 splits with
    at most 16 groups per SM (40 or 700 rows of width 256: 80 or 1400 groups) take one
    128-column group per warp, 4 values a lane; 6 splits or 2800 groups take the group pairs.
    Both bitwise against the oracle."""
    N = 256
    r = np.random.default_rng(1000 * splits + rows + 10 * act + fmt)
    P = (r.standard_normal((splits, rows, 2 * N)) * 1.5).astype(np.float32)
    q, s = ops.silu_mul_quant_fp8(act, to_dev(P), N, in_splits=splits, clamp_limit=clamp, fmt=fmt,
                                  strategy=ops.QUANT_PERSISTENT)
    rq, rs = oracle.act_quant(act, _split_sum_bf16(P), N, clamp_limit=clamp, fmt=fmt)
    assert (q.cpu().numpy() == rq).all() and (s.cpu().numpy() == rs).all()


@pytest.mark.parametrize("splits", [2, 4, 7])
def test_persistent_split_partials_row_map(ops, splits):
    """The layer's route walk on split partials: work row i writes slot row_map[i] from the
    same slot's partials; dropped routes (-1) and slots no route maps to stay untouched."""
    N, slots, R = 512, 96, 60
    r = np.random.default_rng(splits)
    P = (r.standard_normal((splits, slots, 2 * N)) * 1.5).astype(np.float32)
    row_map = r.permutation(slots)[:R].astype(np.int32)
    row_map[[3, 17, 40]] = -1
    q, s = ops.silu_mul_quant_fp8(1, to_dev(P), N, rows=R, row_map=to_dev(row_map), row_div=0,
                                  out_rows=slots, in_splits=splits, clamp_limit=7.0, fmt=1,
                                  strategy=ops.QUANT_PERSISTENT)
    rq, rs = oracle.act_quant(1, _split_sum_bf16(P), N, clamp_limit=7.0, fmt=1)
    q, s = q.cpu().numpy(), s.cpu().numpy()
    kept = np.zeros(slots, dtype=bool)
    kept[row_map[row_map >= 0]] = True
    assert (q[kept] == rq[kept]).all() and (s[kept] == rs[kept]).all()
    assert (q[~kept] == 0).all() and (s[~kept] == 0).all()


def test_row_map_gather_and_mask(ops):
    """Slot-order gathering as the layer uses it: work row = route r, output row = slot of r,
    input row = r // k (gather) or the slot itself (mask)."""
    M, k, H = 12, 3, 512
    x = wl.act_rows(M, H, 1.0, seed=9)
    r = np.random.default_rng(0)
    slots = 64
    route_slot = r.permutation(slots)[: M * k].astype(np.int32)
    route_slot[[2, 7, 20]] = -1
    q, s = ops.silu_mul_quant_fp8(0, bf16_to_dev(x), H, rows=M * k, row_map=to_dev(route_slot),
                                  row_div=k, out_rows=slots)
    rq, rs = oracle.act_quant(0, x, H)
    q = q.cpu().numpy()
    for route, slot in enumerate(route_slot):
        if slot >= 0:
            assert (q[slot] == rq[route // k]).all()
    untouched = np.setdiff1d(np.arange(slots), route_slot[route_slot >= 0])
    assert (q[untouched] == 0).all()
    # mask mode: input row is the slot itself
    gu = wl.act_rows(slots, 2 * 256, 2.0, seed=3)
    q2, s2 = ops.silu_mul_quant_fp8(1, bf16_to_dev(gu), 256, rows=M * k, row_map=to_dev(route_slot),
                                    row_div=0, out_rows=slots)
    rq2, rs2 = oracle.act_quant(1, gu, 256)
    q2 = q2.cpu().numpy()
    valid = route_slot[route_slot >= 0]
    assert (q2[valid] == rq2[valid]).all() and (s2.cpu().numpy()[valid] == rs2[valid]).all()


def test_encoder_edge_values(ops):
    """With the group amax at 448 the fp32 scale is exactly 1, so the codes are the hardware
    encode of the BF16 inputs themselves: ties, subnormals, saturation-free extremes, signed
    zeros -- compared with the oracle's explicit encoder."""
    vals = [448.0, -448.0, 0.0, -0.0, 1.0, 1.0625, 1.125, 1.1875, 0.001953125, 0.0009765625,
            0.0029296875, -0.0029296875, 0.013671875, 0.0146484375, 0.015625, 416.0, 432.0,
            240.0, 232.0, 248.0, 1e-30, -1e-30, 3.0, 3.25, -3.125, 17.0, 18.0, 19.0]
    row = np.zeros(128, np.float32)
    row[: len(vals)] = vals
    r = np.random.default_rng(1)
    rest = r.uniform(-448, 448, 128 - len(vals)).astype(np.float32)
    row[len(vals):] = rest
    x = torch.from_numpy(row[None, :]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, s = _gpu_quant(ops, 0, x, 128)
    assert s[0, 0] == 1.0
    rq, rs = oracle.act_quant(0, x, 128)
    assert (q == rq).all(), np.nonzero(q != rq)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert (q[0] == oracle.e4m3_encode(xf[0])).all()
