"""The bounded waits of the fused layer kernel, exercised on the GPU without a fault or a hang.

Every wait in the library's kernels gives up after a time limit, records MOE_DEV_TIMEOUT in the
per-device status word, drains the kernel's own copies and tensor-core work, frees its tensor
memory and returns.  Here the test hook makes one block's activation-step wait unreachable (it
waits for one gate/up piece more than exist; every index and address stays valid) with a 1 ms
limit: the call must return, the status word must report the timeout, and the next normal call
on the same workspace must be bit for bit the undisturbed result (no state carries over)."""
import time

import numpy as np
import pytest
import torch

from block_fp8_mixture_moe_gb300 import workloads as wl
from tests.gpu_util import bf16_to_dev, to_dev

pytestmark = pytest.mark.gpu
FUSED = 1


@pytest.mark.parametrize("M", [4, 32])
def test_fused_wait_runs_out_and_the_next_call_is_exact(ops, M):
    cfg = dict(wl.CONFIGS["decode"], M=M)
    L = wl.make_layer(**cfg, seed=30 + M, device="cuda")
    H, N, E, k = cfg["H"], cfg["N"], cfg["E"], cfg["k"]
    ws = torch.zeros(ops.moe_blockfp8_workspace_bytes(M, k, E, E, H, N), dtype=torch.uint8, device="cuda")
    args = (bf16_to_dev(L["x"]), to_dev(L["topk_ids"]), to_dev(L["topk_w"]), E, None,
            L["wgu_q"], L["wgu_s"], L["wd_q"], L["wd_s"])
    ref = ops.moe_blockfp8_forward(*args, workspace=ws, path=FUSED).clone()
    torch.cuda.synchronize()
    assert ops.device_status() == 0

    ops.moe_debug_inject_stall(0, 1_000_000)  # block 0, 1 ms
    t0 = time.perf_counter()
    ops.moe_blockfp8_forward(*args, workspace=ws, path=FUSED)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    status = ops.device_status()
    assert status & ops.DEV_TIMEOUT, f"status {status}"
    assert waited < 1.5, f"the aborted call took {waited:.3f} s"

    out = ops.moe_blockfp8_forward(*args, workspace=ws, path=FUSED)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    assert torch.equal(out, ref)


def test_stall_hook_is_one_shot_and_checked(ops):
    with pytest.raises(ops.MoeError):
        ops.moe_debug_inject_stall(-1, 1_000_000)
    with pytest.raises(ops.MoeError):
        ops.moe_debug_inject_stall(0, 0)
    with pytest.raises(ops.MoeError):
        ops.moe_debug_inject_stall(0, 3_000_000_000)
