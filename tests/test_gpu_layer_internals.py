"""The whole layer's own intermediate tensors, read back from the forward's workspace after
moe_blockfp8_forward and checked stage by stage against the oracle, on both paths (the fused
persistent kernel and the staged launches):

* routing metadata (sorted indices, block table, block count, counts, offsets): bit for bit;
* A0, the input quantisation the layer itself runs (a per-token kernel in the staged path, phase
  P0 of the fused kernel, neither of which is the silu_mul_quant_fp8 entry point): the E4M3
  codes and the scale of every kept route's slot equal the oracle's identity quantisation of
  the route's token row, bit for bit;
* A3, the fused SiLU*mul + quantisation inside the layer: codes and scales equal the oracle's
  act-quant of the BF16 gate/up value the layer materialises (its fp32 gate/up partial sums,
  read from the workspace and added in the layer's own split or stream-K piece order, rounded
  to BF16 once), bit for bit;
* A2 and A4, the two GEMMs: the layer's gate/up sums and its down-projection rows, each fed the
  layer's own quantised operands, within |err| <= 2e-2 + 1e-2*|ref| of the oracle's GEMM.

The bit-exact contract on FP8 activations and their scales follows vLLM PR #53875, "Correctness
and validation", and lmdeploy PR #4956, "Fused SwiGLU and FP8 quantization"; the per-stage
comparison (each stage fed the GPU's own upstream output, so no accumulation-order difference
upstream can flip a code) is how a bit-exact stage is checked behind a tolerance-checked GEMM.
"""
import numpy as np
import pytest
import torch

import oracle
from block_fp8_mixture_moe_gb300 import workloads as wl
from tests.gpu_util import assert_bf16_close, bf16_to_dev, to_dev

pytestmark = pytest.mark.gpu
INF = float("inf")
FUSED, STAGED = 1, 2

# (name, workload, seed, activation options)
CASES = [
    ("tiny", dict(wl.CONFIGS["tiny"]), 20, dict(act=1, clamp=7.0, fmt=1)),
    ("decode_m1", dict(wl.CONFIGS["decode"], M=1), 21, dict(act=1, clamp=INF, fmt=0)),
    ("decode_m32", dict(wl.CONFIGS["decode"], M=32), 22, dict(act=1, clamp=INF, fmt=0)),
    ("ep_t100", dict(wl.CONFIGS["ep"], M=100), 23, dict(act=1, clamp=7.0, fmt=1)),
    # M=4 takes a single gate/up split: the layer stores the gate/up value in BF16
    ("gate_upper_m4", dict(wl.CONFIGS["decode"], M=4), 24, dict(act=2, clamp=1.0, fmt=1)),
    # two gate/up splits under the gate/up GEMM's dynamic tail
    ("decode_m64", dict(wl.CONFIGS["decode"], M=64), 25, dict(act=1, clamp=7.0, fmt=1)),
]


def _view(host, off, dtype, count):
    n = np.dtype(dtype).itemsize * count
    return host[off:off + n].view(dtype)


def _fused_pieces(nblk, NT1, KB1, G):
    """Stream-K pieces of every gate/up unit (block, 128-column tile) when W1 = nblk*NT1*KB1
    K-blocks are dealt to G1 = min(G, W1) CTAs in equal contiguous ranges [W1*c/G1, W1*(c+1)/G1):
    the CTA of position x is ((x+1)*G1 - 1) // W1, and a unit's pieces are the CTAs its K range
    touches, in K order."""
    W1 = nblk * NT1 * KB1
    G1 = max(1, min(G, W1))

    def cta_of(x):
        return ((x + 1) * G1 - 1) // W1

    return {u: cta_of(u * KB1 + KB1 - 1) - cta_of(u * KB1) + 1 for u in range(nblk * NT1)}


def _gate_up_sum(host, lay, path, slots_kept, S, slots, N, bm, nblk, KB1):
    """The fp32 gate/up value of each kept slot as the layer's act-quant adds it up: partials
    in split (staged) or stream-K piece (fused) order, fp32 additions, starting from the first."""
    W = 2 * N
    if path == STAGED and S == 1:
        # one split: the layer stores the BF16-rounded sum (exact in fp32)
        g16 = _view(host, lay["gu"], np.uint16, slots * W).reshape(slots, W)[slots_kept]
        return (g16.astype(np.uint32) << 16).view(np.float32)
    if path == STAGED:
        gu = _view(host, lay["gu"], np.float32, S * slots * W).reshape(S, slots, W)
        acc = gu[0][slots_kept].copy()
        for p in range(1, S):
            acc = (acc + gu[p][slots_kept]).astype(np.float32)
        return acc
    NT1 = W // 128
    G = torch.cuda.get_device_properties(0).multi_processor_count
    pieces = _fused_pieces(nblk, NT1, KB1, G)
    rows1 = nblk * bm
    npmax = max(pieces.values()) if pieces else 1
    gu = _view(host, lay["gu"], np.float32, npmax * rows1 * W).reshape(npmax, rows1, W)
    acc = np.zeros((len(slots_kept), W), np.float32)
    for i, s in enumerate(slots_kept):
        b = s // bm
        for nt in range(NT1):
            cols = slice(nt * 128, (nt + 1) * 128)
            v = gu[0, s, cols].copy()
            for q in range(1, pieces[b * NT1 + nt]):
                v = (v + gu[q, s, cols]).astype(np.float32)
            acc[i, cols] = v
    return acc


@pytest.mark.parametrize("path", [FUSED, STAGED])
@pytest.mark.parametrize("name,cfg,seed,opt", CASES, ids=[c[0] for c in CASES])
def test_layer_intermediates_vs_oracle(ops, name, cfg, seed, opt, path):
    L = wl.make_layer(**cfg, seed=seed, device="cuda")
    M, H, N, E, k, El = L["M"], L["H"], L["N"], L["E"], L["k"], L["E_local"]
    act, clamp, fmt = opt["act"], opt["clamp"], opt["fmt"]
    emap = L["expert_map"]
    ids = L["topk_ids"]
    need = ops.moe_blockfp8_workspace_bytes(M, k, E, El, H, N)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ops.moe_blockfp8_forward(bf16_to_dev(L["x"]), to_dev(ids), to_dev(L["topk_w"]), E,
                             None if emap is None else to_dev(emap), L["wgu_q"], L["wgu_s"],
                             L["wd_q"], L["wd_s"], act=act, clamp_limit=clamp, act_fmt=fmt,
                             workspace=ws, path=path)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    host = ws.cpu().numpy()
    lay = ops.moe_blockfp8_workspace_layout(M, k, E, El, H, N)
    bm, B_cap, S = ops.moe_blockfp8_plan(M, k, E, El, H, N)
    slots, R, KB1, GN = B_cap * bm, M * k, H // 128, N // 128

    # ---- routing metadata, bit for bit ----
    ref = oracle.route_prepare(ids, E, emap, El, bm)
    nblk = int(_view(host, lay["num_blocks"], np.int32, 1)[0])
    assert nblk == ref["num_blocks"]
    assert (_view(host, lay["sorted_idx"], np.int32, slots) == ref["sorted_idx"]).all()
    assert (_view(host, lay["block_expert"], np.int32, B_cap) == ref["block_expert"]).all()
    assert (_view(host, lay["expert_count"], np.int32, El) == ref["expert_count"]).all()
    assert (_view(host, lay["expert_offset"], np.int32, El + 1) == ref["expert_offset"]).all()
    route_slot = _view(host, lay["route_slot"], np.int32, R)
    kept = np.nonzero(route_slot >= 0)[0]
    s_of = route_slot[kept]
    assert (ref["sorted_idx"][s_of] == kept).all()
    tok = kept // k
    e_loc = ref["block_expert"][s_of // bm].astype(np.int32)

    # ---- A0: the layer's input quantisation, bit for bit ----
    xq = _view(host, lay["xq"], np.uint8, slots * H).reshape(slots, H)
    xs_raw = _view(host, lay["xs"], np.float32, slots * KB1)
    xs = (xs_raw.reshape(KB1, slots).T if path == FUSED else xs_raw.reshape(slots, KB1))
    xs = np.ascontiguousarray(xs)
    ref_xq, ref_xs = oracle.act_quant(oracle.ACT_IDENTITY, L["x"], H, fmt=fmt)
    assert (xq[s_of] == ref_xq[tok]).all(), "input codes"
    assert (xs[s_of].view(np.uint32) == ref_xs[tok].view(np.uint32)).all(), "input scales"

    Ln = wl.layer_numpy(L, experts=e_loc)
    # ---- A2: gate/up GEMM on the layer's own quantised input, within tolerance ----
    gsum = _gate_up_sum(host, lay, path, s_of, S, slots, N, bm, nblk, KB1)
    gu_bf16 = oracle.bf16_round(gsum)
    ref_gu = oracle.route_gemm(xq, xs, Ln["wgu_q"], Ln["wgu_s"], s_of.astype(np.int32), e_loc)
    assert_bf16_close(gu_bf16, ref_gu, f"{name} gate/up")

    # ---- A3: fused SiLU*mul + quantisation of that BF16 value, bit for bit ----
    aq = _view(host, lay["aq"], np.uint8, slots * N).reshape(slots, N)
    as_raw = _view(host, lay["as"], np.float32, slots * GN)
    a_s = np.ascontiguousarray(as_raw.reshape(GN, slots).T if path == FUSED else as_raw.reshape(slots, GN))
    ref_aq, ref_as = oracle.act_quant(act, gu_bf16, N, clamp_limit=clamp, fmt=fmt)
    assert (aq[s_of] == ref_aq).all(), "activation codes"
    assert (a_s[s_of].view(np.uint32) == ref_as.view(np.uint32)).all(), "activation scales"

    # ---- A4: down GEMM on the layer's own quantised activation, within tolerance ----
    z = _view(host, lay["z"], np.uint16, R * H).reshape(R, H)
    ref_z = oracle.route_gemm(aq, a_s, Ln["wd_q"], Ln["wd_s"], s_of.astype(np.int32), e_loc)
    assert_bf16_close(z[kept], ref_z, f"{name} down")


@pytest.mark.parametrize("path", [FUSED, STAGED])
@pytest.mark.parametrize("M", [10, 5])
def test_out_of_range_map_entry_drops_the_route(ops, path, M):
    """An expert map entry outside [-1, E_local) is an invalid slice: route preparation gives
    the route no slot and flags MOE_DEV_BAD_EXPERT_MAP, and every later stage -- the reduce
    included -- drops the route.  Both paths give the oracle's output for the map with that
    entry set to -1 (lmdeploy PR #4857 review: validate the local-expert slice).  M = 5 (30
    routes) runs the self-routed gate/up GEMM, which must drop the route in the same way."""
    cfg = dict(wl.CONFIGS["ep"], M=M)
    L = wl.make_layer(**cfg, seed=25, device="cuda")
    emap = L["expert_map"].copy()
    used = np.unique(L["topk_ids"])
    local_used = [g for g in used if emap[g] >= 0]
    bad = int(local_used[0])
    emap_bad = emap.copy()
    emap_bad[bad] = L["E_local"] + 3
    out = ops.moe_blockfp8_forward(bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"]),
                                   L["E"], to_dev(emap_bad), L["wgu_q"], L["wgu_s"], L["wd_q"],
                                   L["wd_s"], clamp_limit=7.0, act_fmt=1, path=path)
    torch.cuda.synchronize()
    assert ops.device_status() & ops.DEV_BAD_EXPERT_MAP
    emap_ok = emap.copy()
    emap_ok[bad] = -1
    Lr = dict(L, expert_map=emap_ok)
    loc = emap_ok[L["topk_ids"][L["topk_ids"] >= 0]]
    ref = oracle.moe_forward(wl.layer_numpy(Lr, experts=loc[loc >= 0]), clamp_limit=7.0, fmt=1)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_bf16_close(got, ref, "bad map entry")
    assert ops.device_status() == 0


def test_staged_path_refuses_topk_above_32(ops):
    """The staged reduce takes top-k <= 32 (one route per lane): an explicit STAGED call with
    k = 33 is refused before anything is enqueued, and AUTO takes the fused path, which matches
    the oracle; k = 32 runs staged and matches too."""
    L = wl.make_layer(M=3, H=256, N=128, E=40, k=33, seed=26, device="cuda")
    args = (bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"]), L["E"], None,
            L["wgu_q"], L["wgu_s"], L["wd_q"], L["wd_s"])
    with pytest.raises(ops.MoeError, match="top-k <= 32"):
        ops.moe_blockfp8_forward(*args, path=STAGED)
    assert ops.moe_forward_path_for(3, 33, 40, 40, 256, 128) == FUSED
    out = ops.moe_blockfp8_forward(*args)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    ref = oracle.moe_forward(wl.layer_numpy(L))
    assert_bf16_close(out.view(torch.int16).cpu().numpy().view(np.uint16), ref, "top-k 33")
    L32 = wl.make_layer(M=3, H=256, N=128, E=40, k=32, seed=27, device="cuda")
    out = ops.moe_blockfp8_forward(bf16_to_dev(L32["x"]), to_dev(L32["topk_ids"]), to_dev(L32["topk_w"]),
                                   L32["E"], None, L32["wgu_q"], L32["wgu_s"], L32["wd_q"], L32["wd_s"],
                                   path=STAGED)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    ref = oracle.moe_forward(wl.layer_numpy(L32))
    assert_bf16_close(out.view(torch.int16).cpu().numpy().view(np.uint16), ref, "top-k 32")
