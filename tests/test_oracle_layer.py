"""Whole-layer pins of the oracle.

* Brute force: every token through every local expert, masked by the routing and summed with
  the routing weights, equals the sparse evaluation bit for bit (the per-(token, expert)
  arithmetic is identical, so any routing or reduce mistake shows).
* Quantisation sanity: against an unquantised float64 evaluation on the same decoded weights,
  relative RMSE < 0.06 and cosine > 0.998 -- the quantised-method gates quoted in vLLM PR
  #53875 "Fuse clamped MoE activation and UE8M0 FP8 block quantization" (ROCm correctness
  note).  A swapped gate/up, a dropped scale or a transposed weight fails these gates.
* Sampling: evaluating a subset of tokens reproduces those rows of the full evaluation."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_moe_gb300 import workloads as wl


def _layer(orc, **kw):
    L = wl.make_layer(**kw)
    return wl.layer_numpy(L)


def _unquantized(orc, L, act, clamp):
    """float64 evaluation without activation quantisation, on the decoded weights."""
    x = orc.bf16_to_f32(L["x"]).astype(np.float64)
    dec = lambda q, s: (torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
                        * np.repeat(np.repeat(s.astype(np.float64), 128, axis=1), 128, axis=2))
    Wgu = dec(L["wgu_q"], L["wgu_s"])
    Wd = dec(L["wd_q"], L["wd_s"])
    N = L["N"]
    E, M, k = L["E"], L["M"], L["k"]
    emap = L["expert_map"]
    out = np.zeros((M, L["H"]))
    for t in range(M):
        for j in range(k):
            g_id = L["topk_ids"][t, j]
            if not (0 <= g_id < E):
                continue
            e = emap[g_id] if emap is not None else g_id
            if e < 0:
                continue
            h = Wgu[e] @ x[t]
            g, u = h[:N], h[N:]
            if np.isfinite(clamp):
                g = np.clip(g, -clamp, clamp) if act == 1 else np.minimum(g, clamp)
                u = np.clip(u, -clamp, clamp)
            a = g / (1 + np.exp(-g)) * u
            out[t] += L["topk_w"][t, j] * (Wd[e] @ a)
    return out


@pytest.mark.parametrize("kw", [
    dict(M=4, H=512, N=256, E=16, k=2, routing="softmax"),
    dict(M=6, H=256, N=384, E=12, k=3, E_local=5, routing="uniform", invalid_frac=0.2),
    dict(M=5, H=384, N=128, E=9, k=4, routing="zipf", invalid_frac=0.1),
])
@pytest.mark.parametrize("act,clamp,fmt", [(1, float("inf"), 0), (1, 7.0, 1), (2, 1.0, 0)])
def test_dense_bruteforce_equals_sparse(orc, kw, act, clamp, fmt):
    L = _layer(orc, seed=0, **kw)
    sparse = orc.moe_forward(L, act=act, clamp_limit=clamp, fmt=fmt)
    dense = orc.moe_forward(L, act=act, clamp_limit=clamp, fmt=fmt, dense=True)
    assert (sparse == dense).all()


@pytest.mark.parametrize("act,clamp,fmt", [(1, float("inf"), 0), (1, float("inf"), 1), (1, 7.0, 1)])
def test_quantisation_error_gates(orc, act, clamp, fmt):
    L = _layer(orc, M=4, H=512, N=256, E=16, k=2, routing="softmax", seed=0)
    ours = orc.bf16_to_f32(orc.moe_forward(L, act=act, clamp_limit=clamp, fmt=fmt)).astype(np.float64)
    ref = _unquantized(orc, L, act, clamp)
    rrmse = np.sqrt(np.mean((ours - ref) ** 2) / np.mean(ref ** 2))
    cos = (ours * ref).sum() / np.linalg.norm(ours) / np.linalg.norm(ref)
    assert rrmse < 0.06 and cos > 0.998, (rrmse, cos)


def test_quantisation_gate_catches_swapped_halves(orc):
    """The gates are sensitive to a plausible oracle mistake: swapping gate and up halves of
    the gate/up weight (what a swapped SiLU operand would compute) fails them."""
    L = _layer(orc, M=4, H=512, N=256, E=16, k=2, routing="softmax", seed=0)
    ref = _unquantized(orc, L, 1, float("inf"))
    Ls = dict(L)
    N = L["N"]
    Ls["wgu_q"] = np.ascontiguousarray(np.concatenate([L["wgu_q"][:, N:], L["wgu_q"][:, :N]], axis=1))
    Ls["wgu_s"] = np.ascontiguousarray(np.concatenate([L["wgu_s"][:, N // 128:], L["wgu_s"][:, :N // 128]], axis=1))
    bad = orc.bf16_to_f32(orc.moe_forward(Ls)).astype(np.float64)
    cos = (bad * ref).sum() / np.linalg.norm(bad) / np.linalg.norm(ref)
    assert cos < 0.998


def test_token_sample_equals_full_rows(orc):
    L = _layer(orc, M=9, H=256, N=128, E=8, k=3, routing="uniform", seed=1, invalid_frac=0.1)
    full = orc.moe_forward(L)
    toks = [0, 3, 8]
    part = orc.moe_forward(L, tokens=toks)
    assert (part[toks] == full[toks]).all()
    others = [t for t in range(9) if t not in toks]
    assert (part[others] == 0).all()
