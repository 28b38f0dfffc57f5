"""Helpers shared by the GPU parity tests (host <-> device conversions, tolerance checks)."""
import numpy as np
import pytest
import torch

ATOL, RTOL = 2e-2, 1e-2  # BF16 layer-output tolerance: |err| <= 2e-2 + 1e-2*|ref|


def dev():
    return torch.device("cuda:0")


def bf16_to_dev(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(dev())


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(dev()) if dtype is None else t.to(dev(), dtype)


def bf16_host(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_of_bf16(u16):
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def assert_bf16_close(got_u16, ref_u16, what=""):
    g = f32_of_bf16(got_u16).astype(np.float64)
    r = f32_of_bf16(ref_u16).astype(np.float64)
    err = np.abs(g - r)
    tol = ATOL + RTOL * np.abs(r)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside 2e-2+1e-2|ref|; "
                           f"max err {err.max():.4g} at {np.unravel_index(err.argmax(), err.shape)}")
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    return err.max()


@pytest.fixture(scope="session")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_fp8_mixture_moe_gb300 import build, ops as O
    build.build()
    O.load()
    torch.cuda.set_device(0)
    return O
