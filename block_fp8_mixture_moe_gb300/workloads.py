"""Seeded synthetic inputs for the block-FP8 MoE layer (shapes of the pages' workloads).

This module only draws inputs: router logits and top-k routing, BF16 activations, and
synthetic expert weights stored as E4M3 codes with one fp32 scale per 128x128 block.  It holds
none of the layer's arithmetic (no activation quantisation, GEMM, SiLU or reduce); both the
CUDA path and the CPU oracle receive the same bytes from here.

Workloads (sizes from the pages; names describe what they are):

* ``tiny``      -- M=4, H=512, N=256, E=16, k=2, softmax top-k routing (correctness case);
* ``decode``    -- M in {1, 4, 16, 32}, H=7168, N=256, E=256, k=8, uniform random routing
                   (lmdeploy PR #4956, "SwiGLU and FP8 quantization microbenchmark": TP8 local
                   routed shape, top-k 8, local intermediate 256);
* ``act_sweep`` -- routed rows 8*T, T in {1,4,16,64,128,256}, activation width 512, inputs
                   ~N(0, 2^2), clamp +-7, UE8M0 (vLLM PR #53875, "Kernel microbenchmarks");
* ``ep``        -- k=6, E=256, 32 local experts through an expert map, H=N=2048, routed rows
                   {6, 60, 600, 6144} (vLLM PR #53875, DeepSeek-V4-style EP8 benchmark);
* ``prefill``   -- M=512, H=4096, N=768, E=512, k=8, Zipf(1.1) expert popularity, block_m 64
                   (the pages' tile; the layer's automatic choice on GB300 is 32).

Weights are drawn ~N(0, 0.02) and stored as E4M3 with fp32 scales per 128x128 block (scale =
block amax / 448, codes from torch's float8_e4m3fn cast); this stands in for the real
checkpoints the pages measured on, which are not available here.
"""
from __future__ import annotations

import numpy as np
import torch

DECODE_M = (1, 4, 16, 32)
ACT_SWEEP_TOKENS = (1, 4, 16, 64, 128, 256)
EP_TOKENS = (1, 10, 100, 1024)

CONFIGS = {
    "tiny": dict(M=4, H=512, N=256, E=16, k=2, E_local=16, routing="softmax", block_m=16),
    "decode": dict(M=32, H=7168, N=256, E=256, k=8, E_local=256, routing="uniform", block_m=16),
    "ep": dict(M=100, H=2048, N=2048, E=256, k=6, E_local=32, routing="uniform", block_m=16),
    "prefill": dict(M=512, H=4096, N=768, E=512, k=8, E_local=512, routing="zipf", block_m=64),
}


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """fp32 tensor -> BF16 (round to nearest even, torch's cast) as int16 bit patterns."""
    return x.to(torch.bfloat16).view(torch.int16)


def bf16_normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """BF16 activations ~N(0, std^2), returned as a torch.bfloat16 tensor."""
    g = torch.Generator(device=device).manual_seed(seed)
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(
        torch.bfloat16)


def routing_topk(M: int, E: int, k: int, seed: int, kind: str = "softmax", zipf_s: float = 1.1):
    """Router logits -> softmax -> top-k (ties to the lower expert id) -> renormalised weights.

    kind="softmax"/"uniform": logits ~N(0, 1), so the chosen expert sets are uniform.
    kind="zipf": logits log p_e + Gumbel noise with p_e proportional to rank(e)^-s and a seeded
    random rank->id permutation (Gumbel top-k draws k distinct experts with Zipf popularity)."""
    r = rng(seed)
    if kind in ("softmax", "uniform"):
        logits = r.standard_normal((M, E))
    elif kind == "zipf":
        perm = r.permutation(E)
        logp = -zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        logits = logp[np.argsort(perm)][None, :] + r.gumbel(size=(M, E))
    else:
        raise ValueError(kind)
    ids = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    top = np.take_along_axis(logits, ids.astype(np.int64), axis=1)
    w = np.exp(top - top.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


def expert_map_random(E: int, E_local: int, seed: int) -> np.ndarray:
    """A seeded random E_local-of-E slice: global id -> local index (ascending) or -1."""
    r = rng(seed)
    local = np.sort(r.choice(E, size=E_local, replace=False))
    m = np.full(E, -1, np.int32)
    m[local] = np.arange(E_local, dtype=np.int32)
    return m


def quantized_weights(E: int, rows: int, cols: int, seed: int, std: float = 0.02, device="cpu",
                      chunk: int = 8):
    """E experts of [rows, cols] weights ~N(0, std^2) as E4M3 codes [E, rows, cols] (uint8) and
    fp32 scales [E, rows/128, cols/128] (block amax / 448).  Generated chunk by chunk of experts
    so the fp32 temporaries stay small."""
    assert rows % 128 == 0 and cols % 128 == 0
    g = torch.Generator(device=device).manual_seed(seed)
    q = torch.empty((E, rows, cols), dtype=torch.uint8, device=device)
    s = torch.empty((E, rows // 128, cols // 128), dtype=torch.float32, device=device)
    for e0 in range(0, E, chunk):
        e1 = min(E, e0 + chunk)
        w = torch.randn((e1 - e0, rows, cols), generator=g, device=device) * std
        wb = w.view(e1 - e0, rows // 128, 128, cols // 128, 128)
        sc = wb.abs().amax(dim=(2, 4)) / 448.0
        sc = torch.where(sc > 0, sc, torch.ones_like(sc))
        qb = (wb / sc[:, :, None, :, None]).to(torch.float8_e4m3fn)
        q[e0:e1] = qb.view(e1 - e0, rows, cols).view(torch.uint8)
        s[e0:e1] = sc
        del w, wb, qb
    return q, s


def make_layer(M: int, H: int, N: int, E: int, k: int, seed: int = 0, E_local: int | None = None,
               routing: str = "softmax", x_std: float = 1.0, w_std: float = 0.02,
               device="cpu", invalid_frac: float = 0.0, **_unused):
    """One layer's inputs.  Routing, the expert map and the activations are numpy arrays
    (BF16 as uint16 bits); weights are torch tensors on ``device``.

    invalid_frac > 0 replaces that fraction of the routing ids with out-of-range ids (-1 or
    >= E) to exercise the drop rule."""
    E_local = E if E_local is None else E_local
    ids, w = routing_topk(M, E, k, seed * 7919 + 1, routing)
    if invalid_frac > 0 and ids.size:
        r = rng(seed * 7919 + 2)
        mask = r.random(ids.shape) < invalid_frac
        bad = np.where(r.random(ids.shape) < 0.5, -1, E + r.integers(0, 5, ids.shape))
        ids = np.where(mask, bad, ids).astype(np.int32)
    emap = None if E_local == E else expert_map_random(E, E_local, seed * 7919 + 3)
    x = bf16_normal((M, H), x_std, seed * 7919 + 4).view(torch.int16).numpy().view(np.uint16)
    wgu_q, wgu_s = quantized_weights(E_local, 2 * N, H, seed * 7919 + 5, w_std, device)
    wd_q, wd_s = quantized_weights(E_local, H, N, seed * 7919 + 6, w_std, device)
    return dict(x=x, topk_ids=ids, topk_w=w, expert_map=emap, wgu_q=wgu_q, wgu_s=wgu_s,
                wd_q=wd_q, wd_s=wd_s, M=M, H=H, N=N, E=E, k=k, E_local=E_local)


def layer_numpy(layer: dict, experts=None) -> dict:
    """Host (numpy) copy of a layer for the oracle; ``experts`` restricts the copied weights to
    those local experts (the others are zero: a sample never routes to them)."""
    out = dict(layer)
    for key in ("wgu_q", "wgu_s", "wd_q", "wd_s"):
        t = layer[key]
        if experts is None:
            out[key] = t.cpu().numpy()
        else:
            host = torch.zeros(t.shape, dtype=t.dtype)
            idx = torch.as_tensor(sorted(set(int(e) for e in experts)), dtype=torch.long)
            if idx.numel():
                host[idx] = t[idx.to(t.device)].cpu()
            out[key] = host.numpy()
    return out


def act_rows(rows: int, width: int, std: float, seed: int) -> np.ndarray:
    """BF16 rows [rows, width] ~N(0, std^2) as uint16 bits (activation-quant inputs)."""
    return bf16_normal((rows, width), std, seed).view(torch.int16).numpy().view(np.uint16)


def act_sweep_rows(tokens: int, k: int = 8, width: int = 1024, seed: int = 0) -> np.ndarray:
    """Fused clamped act-quant sweep: routed rows = tokens * k, gate/up width 2*512."""
    return act_rows(tokens * k, width, 2.0, seed * 7919 + 11 + tokens)


def padded_grid_route(sorted_idx, block_expert, num_blocks: int, E_local: int, bm: int):
    """The schedule that active-expert block scheduling replaces (lmdeploy PR #4956,
    "Motivation": the dense grid covers every expert): every local expert owns at least one
    block, max(1, its compact block count), in expert order, so the GEMM streams the weights of
    every expert whether or not it received routes.  Built on the host from a compact route
    table (numpy int32 arrays as moe_route_prepare returns them); a table transform only, no
    arithmetic of the layer.

    Returns dict(sorted_idx, block_expert, num_blocks, B_cap, slot_map): slot_map[s] is the
    padded-grid slot that holds compact slot s (-1 for slots past the compact blocks)."""
    sorted_idx = np.asarray(sorted_idx, np.int32)
    block_expert = np.asarray(block_expert, np.int32)
    per_expert = [[] for _ in range(E_local)]
    for b in range(int(num_blocks)):
        per_expert[int(block_expert[b])].append(b)
    nb_pad = sum(max(1, len(bl)) for bl in per_expert)
    si = np.full(nb_pad * bm, -1, np.int32)
    be = np.empty(nb_pad, np.int32)
    slot_map = np.full(sorted_idx.size, -1, np.int32)
    nb = 0
    for e, blocks in enumerate(per_expert):
        if not blocks:
            be[nb] = e
            nb += 1
            continue
        for b in blocks:
            be[nb] = e
            si[nb * bm:(nb + 1) * bm] = sorted_idx[b * bm:(b + 1) * bm]
            slot_map[b * bm:(b + 1) * bm] = np.arange(nb * bm, (nb + 1) * bm, dtype=np.int32)
            nb += 1
    return dict(sorted_idx=si, block_expert=be, num_blocks=nb, B_cap=nb, slot_map=slot_map)
