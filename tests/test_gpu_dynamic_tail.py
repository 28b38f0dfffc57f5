"""The grouped GEMMs' dynamic tail: on long weight streams the staged forward's GEMMs walk static
shares of three quarters of their work units and hand out the rest from a counter in the
workspace.  Every unit must still be computed exactly once and exactly as in the static split.

At the Zipf prefill shape (lmdeploy PR #4857, "Changes": the multi-CTA route preparation and
hot experts), where both GEMMs take the dynamic tail, the forward's own gate/up partial sums and
down-projection rows, read from its workspace, equal bit for bit the same GEMMs rerun through
moe_blockfp8_grouped_gemm (which always splits statically) on the forward's own operands.  A
unit computed twice would still match, but a skipped one would leave its rows out of the
forward's result; the counter-zeroing is also checked by running the forward twice on one
workspace.
"""
import numpy as np
import pytest
import torch

from block_fp8_mixture_moe_gb300 import workloads as wl
from tests.gpu_util import bf16_to_dev, to_dev

pytestmark = pytest.mark.gpu


def _region(ws, lay, name, dtype, count):
    off = lay[name]
    n = torch.empty((), dtype=dtype).element_size() * count
    return ws[off:off + n].view(dtype)


def test_plan_takes_the_dynamic_tail_only_on_long_streams(ops):
    p = wl.CONFIGS["prefill"]
    assert ops.moe_blockfp8_dynamic_tail(p["M"], p["k"], p["E"], p["E_local"], p["H"], p["N"]) == (True, True)
    d = wl.CONFIGS["decode"]
    # block_m 16 from 2.5 MB of weights per SM: the gate/up GEMM from M=32, the down GEMM from 64
    for M, want in ((1, (False, False)), (16, (False, False)), (32, (True, False)),
                    (64, (True, True)), (256, (True, True))):
        assert ops.moe_blockfp8_dynamic_tail(M, d["k"], d["E"], d["E_local"], d["H"], d["N"]) == want
    e = wl.CONFIGS["ep"]
    assert ops.moe_blockfp8_dynamic_tail(1024, e["k"], e["E"], e["E_local"], e["H"], e["N"]) == (False, False)
    with pytest.raises(ops.MoeError):
        ops.moe_blockfp8_dynamic_tail(4, 2, 16, 16, 100, 256)


def test_dynamic_tail_computes_every_unit_as_the_static_split(ops):
    cfg = wl.CONFIGS["prefill"]
    M, H, N, E, k, El = cfg["M"], cfg["H"], cfg["N"], cfg["E"], cfg["k"], cfg["E_local"]
    R = M * k
    L = wl.make_layer(**cfg, seed=7, device="cuda")
    wgu = ops.moe_blockfp8_pack_weights(L["wgu_q"])
    wd = ops.moe_blockfp8_pack_weights(L["wd_q"])
    del L["wgu_q"], L["wd_q"]
    x, ids, w = bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"])
    ws = torch.empty(ops.moe_blockfp8_workspace_bytes(M, k, E, El, H, N), dtype=torch.uint8, device="cuda")
    args = (x, ids, w, E, None, wgu, L["wgu_s"], wd, L["wd_s"])
    out1 = ops.moe_blockfp8_forward(*args, path=ops.FORWARD_STAGED, workspace=ws)
    # a second forward on the same workspace: route preparation zeroes the counters again
    out2 = ops.moe_blockfp8_forward(*args, path=ops.FORWARD_STAGED, workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    assert torch.equal(out1, out2)

    lay = ops.moe_blockfp8_workspace_layout(M, k, E, El, H, N)
    bm, B_cap, S = ops.moe_blockfp8_plan(M, k, E, El, H, N)
    slots = B_cap * bm
    route = dict(sorted_idx=_region(ws, lay, "sorted_idx", torch.int32, slots),
                 block_expert=_region(ws, lay, "block_expert", torch.int32, B_cap),
                 num_blocks=_region(ws, lay, "num_blocks", torch.int32, 1), B_cap=B_cap)
    sidx = route["sorted_idx"].cpu().numpy()
    kept_slots = torch.from_numpy(np.nonzero(sidx >= 0)[0]).cuda()
    assert kept_slots.numel() == R  # no expert map: every route is kept

    xq = _region(ws, lay, "xq", torch.uint8, slots * H).view(slots, H)
    xs = _region(ws, lay, "xs", torch.float32, slots * (H // 128)).view(slots, H // 128)
    # one split: the layer keeps the BF16-rounded sum; several: the fp32 partials
    gu_t, gu_dt = (torch.bfloat16, ops.DTYPE_BF16) if S == 1 else (torch.float32, ops.DTYPE_F32)
    gu_layer = _region(ws, lay, "gu", gu_t, S * slots * 2 * N).view(S, slots, 2 * N).clone()
    gu_static = ops.moe_blockfp8_grouped_gemm(ops.PROJ_GATE_UP, xq, xs, wgu, L["wgu_s"], route, bm,
                                              out_dtype=gu_dt, out_rows=slots,
                                              splits=S).view(S, slots, 2 * N)
    torch.cuda.synchronize()
    assert torch.equal(gu_layer[:, kept_slots], gu_static[:, kept_slots])

    aq = _region(ws, lay, "aq", torch.uint8, slots * N).view(slots, N)
    as_ = _region(ws, lay, "as", torch.float32, slots * (N // 128)).view(slots, N // 128)
    z_layer = _region(ws, lay, "z", torch.bfloat16, R * H).view(R, H).clone()
    z_static = ops.moe_blockfp8_grouped_gemm(ops.PROJ_DOWN, aq, as_, wd, L["wd_s"], route, bm, out_rows=R)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    assert torch.equal(z_layer, z_static)
