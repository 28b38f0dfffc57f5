"""Pins of the oracle's stages against closed forms, library routines and brute force.

activation quantisation -- vLLM PR #53875 "Fuse clamped MoE activation and UE8M0 FP8 block
quantization" ("Purpose", "Correctness and validation") and lmdeploy PR #4956 "Perf/pytorch
block fp8 moe decode" ("Fused SwiGLU and FP8 quantization", "Correctness and validation");
route preparation -- lmdeploy PR #4857 "optimize compact blocked FP8 MoE and route
preparation" ("Changes"); GEMM -- the W8A8 block shape [128, 128]; reduce -- lmdeploy PR #4228
"Moe Reduce kernel"."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_moe_gb300 import workloads as wl


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32(h, orc):
    return orc.bf16_to_f32(h)


# ---------------------------------------------------------------------------------------------
# activation quantisation
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [0, 1])
def test_identity_quant_equals_library_division_and_cast(orc, fmt):
    """Per 128-group: s from the group amax, q = e4m3(x / s): numpy's IEEE fp32 division and
    torch's E4M3 cast (both library routines) give the same bytes as the oracle."""
    x = wl.act_rows(64, 512, 3.0, seed=5)
    q, s = orc.act_quant(orc.ACT_IDENTITY, x, 512, fmt=fmt)
    xf = f32(x, orc).reshape(64, 4, 128)
    amax = np.abs(xf).max(axis=2)
    s_ref = np.maximum(amax, np.float32(1e-10)) / np.float32(448.0)
    if fmt == 1:
        s_ref = np.exp2(np.ceil(np.log2(s_ref.astype(np.float64)))).astype(np.float32)
    assert (s == s_ref).all()
    v = (xf / s_ref[:, :, None]).astype(np.float32)
    v = np.clip(v, -448, 448)  # saturation (torch's cast would give NaN past 464)
    q_ref = torch.from_numpy(v.reshape(64, 512)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (q == q_ref).all()


def test_identity_quant_amax_element_encodes_to_448(orc):
    x = wl.act_rows(32, 1024, 1.0, seed=6)
    q, s = orc.act_quant(orc.ACT_IDENTITY, x, 1024)
    xf = f32(x, orc).reshape(32, 8, 128)
    arg = np.abs(xf).argmax(axis=2)
    qa = np.take_along_axis(q.reshape(32, 8, 128), arg[:, :, None], axis=2)[..., 0]
    assert ((qa & 0x7F) == 0x7E).all()


def test_identity_quant_error_bound(orc):
    """|dequant - x| <= half an E4M3 step at the quotient's magnitude (times the scale)."""
    x = wl.act_rows(16, 2048, 1.0, seed=7)
    for fmt in (0, 1):
        q, s = orc.act_quant(orc.ACT_IDENTITY, x, 2048, fmt=fmt)
        xf = f32(x, orc).astype(np.float64).reshape(16, 16, 128)
        dq = orc.e4m3_decode(q).astype(np.float64).reshape(16, 16, 128) * s[:, :, None]
        v = np.abs(xf) / s[:, :, None]
        step = np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3))
        assert (np.abs(dq - xf) <= 0.5 * step * s[:, :, None] * (1 + 1e-6)).all()


def test_silu_mul_activation_matches_double_reference(orc):
    """a = bf16(SiLU(g) * u): against a double-precision SiLU*mul rounded to BF16, allowing only
    rare one-ulp differences where the fp32 value sits on a BF16 rounding boundary."""
    gu = wl.act_rows(256, 1024, 2.0, seed=8)
    _, _, a = orc.act_quant(orc.ACT_SILU_MUL, gu, 512, want_a=True)
    gf = f32(gu, orc).astype(np.float64)
    g, u = gf[:, :512], gf[:, 512:]
    ref = orc.bf16_round_double(g / (1 + np.exp(-g)) * u)
    diff = np.abs(a.astype(np.int64) - ref.astype(np.int64))
    assert diff.max() <= 1
    assert (diff > 0).mean() < 1e-3


@pytest.mark.parametrize("act", [1, 2])
def test_clamp_equals_preclamped_inputs(orc, act):
    """The clamp acts on the BF16 gate/up inputs before SiLU: clamping the inputs beforehand and
    running unclamped gives the same bytes.  act 1: both halves to [-L, L]; act 2: gate <= L,
    up in [-L, L]."""
    L = 1.5
    gu = wl.act_rows(64, 1024, 2.0, seed=9)
    q, s, a = orc.act_quant(act, gu, 512, clamp_limit=L, fmt=1, want_a=True)
    gf = f32(gu, orc).copy()
    if act == 1:
        gf[:, :512] = np.clip(gf[:, :512], -L, L)
    else:
        gf[:, :512] = np.minimum(gf[:, :512], L)
    gf[:, 512:] = np.clip(gf[:, 512:], -L, L)
    q2, s2, a2 = orc.act_quant(orc.ACT_SILU_MUL, bf16(gf), 512, fmt=1, want_a=True)
    assert (q == q2).all() and (s == s2).all() and (a == a2).all()
    # and the clamp really fired
    q3, _ = orc.act_quant(act, gu, 512, fmt=1)
    assert (q3 != q).any()


def test_infinite_clamp_is_no_clamp(orc):
    gu = wl.act_rows(32, 512, 4.0, seed=10)
    a1 = orc.act_quant(orc.ACT_SILU_MUL, gu, 256, clamp_limit=float("inf"), want_a=True)
    a2 = orc.act_quant(orc.ACT_SILU_MUL, gu, 256, clamp_limit=1e30, want_a=True)
    for u, v in zip(a1, a2):
        assert (u == v).all()


@pytest.mark.parametrize("fmt", [0, 1])
def test_fused_equals_two_step(orc, fmt):
    """The pages' claim: fused SiLU*mul + quant equals quant(silu_and_mul(x)) in values and
    scales (lmdeploy PR #4956 and vLLM PR #53875, 'Correctness and validation')."""
    gu = wl.act_rows(128, 1024, 2.0, seed=11)
    q, s = orc.act_quant(orc.ACT_SILU_MUL, gu, 512, clamp_limit=7.0, fmt=fmt)
    mid = orc.silu_and_mul(orc.ACT_SILU_MUL, gu, 512, clamp_limit=7.0)
    q2, s2 = orc.act_quant(orc.ACT_IDENTITY, mid, 512, fmt=fmt)
    assert (q == q2).all() and (s == s2).all()


def test_filtered_rows_untouched(orc):
    """Invalid and non-local rows keep whatever the output held (vLLM PR #53875)."""
    rows, N, E = 40, 256, 16
    gu = wl.act_rows(rows, 2 * N, 1.0, seed=12)
    r = np.random.default_rng(0)
    ids = r.integers(-2, E + 2, rows).astype(np.int32)
    emap = np.where(r.random(E) < 0.5, -1, np.arange(E)).astype(np.int32)
    q = np.full((rows, N), 0xAB, np.uint8)
    s = np.full((rows, N // 128), -7.0, np.float32)
    orc.act_quant(orc.ACT_SILU_MUL, gu, N, row_expert=ids, expert_map=emap, E=E, out_q=q, out_s=s)
    kept = (ids >= 0) & (ids < E)
    kept[kept] &= emap[ids[kept]] >= 0
    assert (q[~kept] == 0xAB).all() and (s[~kept] == -7.0).all()
    q_all, s_all = orc.act_quant(orc.ACT_SILU_MUL, gu, N)
    assert (q[kept] == q_all[kept]).all() and (s[kept] == s_all[kept]).all()
    assert kept.any() and (~kept).any()


# ---------------------------------------------------------------------------------------------
# route preparation
# ---------------------------------------------------------------------------------------------
def _check_route_invariants(res, ids, E, emap, E_loc, bm):
    R = ids.size
    flat = ids.reshape(-1)
    loc = np.full(R, -1)
    for r in range(R):
        g = flat[r]
        if 0 <= g < E:
            loc[r] = emap[g] if emap is not None else g
    kept = np.where(loc >= 0)[0]
    si, be, nb = res["sorted_idx"], res["block_expert"], res["num_blocks"]
    body = si[: nb * bm]
    # every kept route exactly once, nothing else
    assert sorted(body[body >= 0].tolist()) == kept.tolist()
    assert (si[nb * bm:] == -1).all() and (be[nb:] == -1).all()
    counts = np.bincount(loc[kept], minlength=E_loc) if kept.size else np.zeros(E_loc, int)
    assert (res["expert_count"] == counts).all()
    assert nb == sum((c + bm - 1) // bm for c in counts)
    assert counts.sum() == kept.size
    for b in range(nb):
        e = be[b]
        assert counts[e] > 0, "no block for an expert without routes"
        blk = si[b * bm:(b + 1) * bm]
        v = blk[blk >= 0]
        assert v.size > 0 and (loc[v] == e).all(), "blocks are expert-homogeneous"
        # pads only at the end of the block
        assert (blk[: v.size] >= 0).all() and (blk[v.size:] == -1).all()
    # brute force stable sort by (local expert, route id)
    order = sorted(kept.tolist(), key=lambda r: (loc[r], r))
    assert body[body >= 0].tolist() == order
    off = res["expert_offset"]
    assert off[0] == 0 and (np.diff(off) == [(c + bm - 1) // bm * bm for c in counts]).all()


@pytest.mark.parametrize("M,k,E,E_loc,bm,inv", [
    (4, 2, 16, 16, 16, 0.0), (1, 8, 256, 256, 16, 0.0), (32, 8, 256, 256, 16, 0.0),
    (64, 8, 256, 32, 32, 0.1), (100, 6, 256, 32, 64, 0.0), (512, 8, 512, 512, 64, 0.05),
    (0, 8, 256, 256, 16, 0.0), (7, 3, 5, 5, 128, 0.3),
])
def test_route_prepare_invariants_and_bruteforce(orc, M, k, E, E_loc, bm, inv):
    ids, _ = wl.routing_topk(M, E, k, seed=M + E, kind="zipf" if M == 512 else "uniform")
    if inv:
        r = np.random.default_rng(1)
        ids = np.where(r.random(ids.shape) < inv, r.choice([-1, E, E + 3], ids.shape), ids).astype(np.int32)
    emap = None if E_loc == E else wl.expert_map_random(E, E_loc, seed=3)
    res = orc.route_prepare(ids, E, emap, E_loc, bm)
    _check_route_invariants(res, ids, E, emap, E_loc, bm)


def test_route_prepare_rejects_bad_slice(orc):
    ids = np.zeros((2, 2), np.int32)
    emap = np.array([5, -1, 0, 1], np.int32)  # 5 >= E_loc
    with pytest.raises(ValueError):
        orc.route_prepare(ids, 4, emap, 2, 16)
    with pytest.raises(ValueError):
        orc.route_prepare(ids, 4, None, 2, 16)  # no map needs E_loc == E


# ---------------------------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------------------------
def test_gemm_exact_integers_unit_scales(orc):
    """All scales 1 and small-integer E4M3 operands: every sum is an exact integer, so the
    result equals an integer matmul (numpy int64) rounded to BF16 (torch's cast)."""
    r = np.random.default_rng(0)
    R, K, N_out, E_loc = 12, 384, 256, 3
    ints = np.arange(-8, 9)
    a_int = r.choice(ints, (R, K))
    w_int = r.choice(ints, (E_loc, N_out, K))
    aq = torch.from_numpy(a_int.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    wq = torch.from_numpy(w_int.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    a_s = np.ones((R, K // 128), np.float32)
    w_s = np.ones((E_loc, N_out // 128, K // 128), np.float32)
    rexp = r.integers(0, E_loc, R).astype(np.int32)
    out = orc.route_gemm(aq, a_s, wq, w_s, np.arange(R, dtype=np.int32), rexp)
    ref = np.stack([w_int[rexp[i]] @ a_int[i] for i in range(R)])
    ref_b = torch.from_numpy(ref.astype(np.float64)).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (out == ref_b).all()


def test_gemm_block_scaled_matches_float64_matmul(orc):
    """Random operands and scales: per K-block matmuls in float64 (numpy/BLAS), scaled by the
    token's and the weight block's scales and summed, agree to within one BF16 step."""
    r = np.random.default_rng(1)
    R, K, N_out, E_loc = 10, 512, 384, 2
    aq = r.integers(0, 256, (R, K)).astype(np.uint8)
    aq[(aq & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    wq = r.integers(0, 256, (E_loc, N_out, K)).astype(np.uint8)
    wq[(wq & 0x7F) == 0x7F] = 0x21
    a_s = r.uniform(0.001, 0.1, (R, K // 128)).astype(np.float32)
    w_s = r.uniform(0.0001, 0.01, (E_loc, N_out // 128, K // 128)).astype(np.float32)
    rexp = r.integers(0, E_loc, R).astype(np.int32)
    rows = r.permutation(R).astype(np.int32)
    out = orc.route_gemm(aq, a_s, wq, w_s, rows, rexp)
    A = torch.from_numpy(aq).view(torch.float8_e4m3fn).double().numpy()
    W = torch.from_numpy(wq).view(torch.float8_e4m3fn).double().numpy()
    ref = np.zeros((R, N_out))
    for i in range(R):
        e, row = rexp[i], rows[i]
        for kb in range(K // 128):
            sl = slice(kb * 128, kb * 128 + 128)
            part = W[e][:, sl] @ A[row, sl]
            ref[i] += part * a_s[row, kb] * np.repeat(w_s[e, :, kb], 128)
    ours = orc.bf16_to_f32(out).astype(np.float64)
    step = np.abs(ref) * 2.0 ** -8 + 1e-30
    assert (np.abs(ours - ref) <= step).all()


def test_gemm_power_of_two_scales_is_exact(orc):
    """Power-of-two (UE8M0-style) scales and E4M3 operands of magnitude >= 2^-3 (or zero): every
    product and partial sum of the whole block-scaled GEMM is exact in double (a span of under
    48 bits), so the result is the float64 matmul of the dequantised operands, in any order,
    rounded once to BF16 (the nearest-BF16 rounding of double pinned in the codec tests)."""
    r = np.random.default_rng(3)
    R, K, N_out, E_loc = 9, 512, 256, 3
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ok = np.flatnonzero(np.isfinite(vals) & ((np.abs(vals) >= 0.125) | (vals == 0))).astype(np.uint8)
    aq = r.choice(ok, (R, K))
    wq = r.choice(ok, (E_loc, N_out, K))
    a_s = np.ldexp(1.0, r.integers(-8, -3, (R, K // 128))).astype(np.float32)
    w_s = np.ldexp(1.0, r.integers(-12, -7, (E_loc, N_out // 128, K // 128))).astype(np.float32)
    rexp = r.integers(0, E_loc, R).astype(np.int32)
    rows = r.permutation(R).astype(np.int32)
    out = orc.route_gemm(aq, a_s, wq, w_s, rows, rexp)
    A = vals[aq] * np.repeat(a_s.astype(np.float64), 128, axis=1)
    W = vals[wq] * np.repeat(np.repeat(w_s.astype(np.float64), 128, axis=1), 128, axis=2)
    ref = np.stack([W[rexp[i]] @ A[rows[i]] for i in range(R)])
    assert (out == orc.bf16_round_double(ref)).all()
    # the same operands with one weight block's scale doubled change that block's rows
    w_s2 = w_s.copy()
    w_s2[0, 0, 0] *= 2
    out2 = orc.route_gemm(aq, a_s, wq, w_s2, rows, rexp)
    hit = rexp == 0
    assert (out2[~hit] == out[~hit]).all() and (out2[hit][:, :128] != out[hit][:, :128]).any()


def test_gemm_skips_dropped_routes(orc):
    r = np.random.default_rng(2)
    aq = r.integers(0, 0x70, (4, 128)).astype(np.uint8)
    wq = r.integers(0, 0x70, (1, 128, 128)).astype(np.uint8)
    out = orc.route_gemm(aq, np.ones((4, 1), np.float32), wq, np.ones((1, 1, 1), np.float32),
                         np.array([0, -1, 2, 3], np.int32), np.array([0, 0, -1, 0], np.int32))
    assert (out[1] == 0).all() and (out[2] == 0).all() and (out[0] != 0).any()


# ---------------------------------------------------------------------------------------------
# moe_reduce
# ---------------------------------------------------------------------------------------------
def test_reduce_single_route_unit_weight_is_identity(orc):
    z = wl.act_rows(8, 256, 1.0, seed=13)
    out = orc.moe_reduce(z, np.ones((8, 1), np.float32), np.zeros((8, 1), np.int32), None, 4, 256)
    assert (out == z).all()


def test_reduce_matches_float64_and_drops(orc):
    M, k, H, E = 16, 8, 512, 64
    z = wl.act_rows(M * k, H, 1.0, seed=14)
    ids, w = wl.routing_topk(M, E, k, seed=2)
    ids = ids.copy()
    ids[0, 3] = -1
    ids[5, 0] = E + 1
    emap = np.arange(E, dtype=np.int32)
    emap[ids[2, 2]] = -1
    out = orc.moe_reduce(z, w, ids, emap, E, H)
    zf = orc.bf16_to_f32(z).astype(np.float64).reshape(M, k, H)
    keep = (ids >= 0) & (ids < E)
    keep[keep] &= emap[ids[keep]] >= 0
    ref = np.einsum("mk,mkh->mh", np.where(keep, w, 0).astype(np.float64), zf)
    ours = orc.bf16_to_f32(out).astype(np.float64)
    assert (np.abs(ours - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6).all()
    # dropping a route equals giving it weight zero (finite z)
    w0 = np.where(keep, w, 0).astype(np.float32)
    out0 = orc.moe_reduce(z, w0, np.clip(ids, 0, E - 1), None, E, H)
    assert (out0 == out).all()
