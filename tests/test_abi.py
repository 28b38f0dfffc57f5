"""The C-ABI library builds for sm_103a, loads, and exports exactly the entry points that
include/moefp8.h declares (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moefp8.h")


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^MOEFP8_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib_path():
    from block_fp8_mixture_moe_gb300 import build
    return build.build()


def test_header_declares_the_five_entry_points():
    names = set(_declared())
    for n in ("moe_route_prepare", "moe_blockfp8_grouped_gemm", "silu_mul_quant_fp8",
              "moe_reduce", "moe_blockfp8_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(_declared()) <= exported
    # nothing of the internal C++ namespace leaks into the ABI
    assert not [s for s in exported if s.startswith("_ZN3moe")]


def test_binding_signatures_cover_the_header(lib_path):
    from block_fp8_mixture_moe_gb300 import ops
    assert set(ops.SIGNATURES) == set(_declared())
    text = open(HEADER).read()
    for name, (_, args) in ops.SIGNATURES.items():
        m = re.search(r"^MOEFP8_API[^;(]*\b" + name + r"\s*\(([^;]*?)\);", text, flags=re.S | re.M)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(args), (name, len(params), len(args))
    ops.load(lib_path)


def test_library_is_built_for_sm103a_only(lib_path):
    """Every translation unit is compiled with exactly one target, sm_103a code (no PTX for
    other architectures); on a GPU the runtime reports the kernels' binary version as 103."""
    from block_fp8_mixture_moe_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    import torch
    if torch.cuda.is_available():
        from block_fp8_mixture_moe_gb300 import ops
        assert ops.load(lib_path).moe_kernel_binary_version() == 103
    else:
        from block_fp8_mixture_moe_gb300 import ops
        assert ops.load(lib_path).moe_kernel_binary_version() == -1


def test_pure_host_helpers(lib_path):
    from block_fp8_mixture_moe_gb300 import ops
    L = ops.load(lib_path)
    import oracle
    for (M, k, E_loc, bm) in [(1, 8, 256, 16), (32, 8, 256, 16), (512, 8, 512, 64), (0, 8, 16, 16), (7, 3, 5, 128)]:
        assert L.moe_block_capacity(M, k, E_loc, bm) == oracle.block_capacity(M * k, E_loc, bm)
    assert L.moe_block_capacity(-1, 8, 16, 16) == -1
    assert L.moe_blockfp8_workspace_bytes(32, 8, 256, 256, 7168, 256, 0) > 0
    assert L.moe_forward_block_m(1, 8, 256, 7168, 256) in (16, 32, 64, 128)


def test_layer_plan_on_152_sms(lib_path):
    """The layer plan for a GB300 (152 SMs), computed on the host: 16-token blocks up to M=256,
    32 above; the gate/up split-K count (at most 4, two under the dynamic tail up to 1024
    routes); and which GEMMs hand out their last units dynamically.  The table is the plan the
    forward takes on the bench's decode, expert-parallel and prefill shapes."""
    from block_fp8_mixture_moe_gb300 import ops
    ops.load(lib_path)
    import oracle
    plan = lambda M, k, E, El, H, N: ops.moe_blockfp8_plan_for_sms(M, k, E, El, H, N, 152)
    decode = {1: (4, False, False), 2: (2, False, False), 4: (1, False, False),
              8: (3, False, False), 16: (4, False, False), 32: (2, True, False),
              64: (2, True, True), 128: (2, True, True), 256: (1, True, True)}
    for M, (splits, gu, dn) in decode.items():
        bm, bc, sp, dgu, ddn = plan(M, 8, 256, 256, 7168, 256)
        assert (bm, sp, dgu, ddn) == (16, splits, gu, dn), M
        assert bc == oracle.block_capacity(M * 8, 256, 16)
    assert plan(1024, 6, 256, 32, 2048, 2048)[0::2] == (32, 1, False)   # expert-parallel T=1024
    assert plan(100, 6, 256, 32, 2048, 2048)[0::2] == (16, 2, False)    # T=100
    assert plan(512, 8, 512, 512, 4096, 768)[0::2] == (32, 1, True)      # Zipf prefill
    assert plan(512, 8, 512, 512, 4096, 768)[4] is True
    for M in (1, 3, 7, 33, 300, 2048):
        sp = plan(M, 8, 256, 256, 7168, 256)[2]
        assert 1 <= sp <= 4
    assert plan(4, 2, 16, 16, 128, 128)[2] == 1                          # one K-block: one split
    with pytest.raises(ops.MoeError):
        ops.moe_blockfp8_plan_for_sms(1, 8, 256, 256, 7168, 256, 0)


def test_calls_without_a_gpu_fail_cleanly(lib_path):
    """On a machine without an sm_103 device every launch entry point refuses with
    MOE_ERR_UNSUPPORTED and launches nothing."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from block_fp8_mixture_moe_gb300 import ops
    L = ops.load(lib_path)
    assert L.moe_device_supported() == 0
    # no device: no pointer is device-accessible (null and plain host memory included)
    import ctypes
    buf = ctypes.create_string_buffer(64)
    assert L.moe_pointer_device_accessible(None) == 0
    assert L.moe_pointer_device_accessible(ctypes.cast(buf, ctypes.c_void_p)) == 0
    rc = L.moe_reduce(None, None, None, None, 1, 1, 1, 1, 8, None, None)
    assert rc == ops.MOE_ERR_UNSUPPORTED
    assert L.moe_last_error_string()
    # every other launching entry point too (sizes 1, null pointers, zero floats): the device
    # check comes before anything is read or launched
    launching = ["moe_route_prepare", "moe_route_prepare_noalloc", "moe_blockfp8_grouped_gemm",
                 "silu_mul_quant_fp8", "silu_and_mul_bf16", "moe_blockfp8_forward",
                 "moe_blockfp8_pack_weights"]
    for name in launching:
        _, argtypes = ops.SIGNATURES[name]
        args = [0.0 if a in (ctypes.c_float, ctypes.c_double) else
                1 if a in (ctypes.c_int, ctypes.c_size_t, ctypes.c_ulonglong) else None
                for a in argtypes]
        assert getattr(L, name)(*args) == ops.MOE_ERR_UNSUPPORTED, name


def test_forward_refuses_pageable_host_activations(lib_path):
    """Host activations must be pinned (device-accessible at their address); a pageable tensor
    is refused in the binding, before the library is called."""
    import torch
    from block_fp8_mixture_moe_gb300 import ops
    ops.load(lib_path)
    M, H, N, E, k = 2, 256, 128, 4, 2
    x = torch.zeros((M, H), dtype=torch.bfloat16)
    ids = torch.zeros((M, k), dtype=torch.int32)
    w = torch.zeros((M, k), dtype=torch.float32)
    wgu_q = torch.zeros((E, 2 * N, H), dtype=torch.uint8)
    wgu_s = torch.ones((E, 2 * N // 128, H // 128), dtype=torch.float32)
    wd_q = torch.zeros((E, H, N), dtype=torch.uint8)
    wd_s = torch.ones((E, H // 128, N // 128), dtype=torch.float32)
    with pytest.raises(AssertionError, match="pinned"):
        ops.moe_blockfp8_forward(x, ids, w, E, None, wgu_q, wgu_s, wd_q, wd_s,
                                 out=torch.zeros((M, H), dtype=torch.bfloat16))
