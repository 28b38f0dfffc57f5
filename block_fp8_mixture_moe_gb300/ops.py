"""Thin ctypes binding of libmoefp8.so (declared in include/moefp8.h).

Each function has the name of the C entry point it calls and does argument marshalling only:
it checks dtypes and shapes, allocates output tensors with torch (device memory), passes raw
device pointers, sizes and the current CUDA stream, and raises on a non-zero return code.  All
arithmetic runs in the library's CUDA kernels; nothing here computes on the host, and a missing
or unloadable library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoefp8.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_EXPERT_SLICE, MOE_ERR_UNSUPPORTED, MOE_ERR_LAUNCH, MOE_ERR_WORKSPACE = range(6)
SCALE_F32, SCALE_UE8M0 = 0, 1
ACT_IDENTITY, ACT_SILU_MUL, ACT_SILU_MUL_GATE_UPPER = 0, 1, 2
PROJ_GATE_UP, PROJ_DOWN = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1
ROUTE_AUTO, ROUTE_SINGLE_CTA, ROUTE_MULTI_CTA = 0, 1, 2
QUANT_AUTO, QUANT_PER_GROUP, QUANT_PERSISTENT = 0, 1, 2
DEV_TIMEOUT, DEV_BAD_EXPERT_MAP, DEV_BAD_INDEX = 1, 2, 4
WEIGHTS_ROW_MAJOR, WEIGHTS_TILED = 0, 1
FORWARD_AUTO, FORWARD_FUSED, FORWARD_STAGED, FORWARD_STAGED_EPILOGUE_REDUCE = 0, 1, 2, 3

# every entry point of include/moefp8.h with its ctypes signature
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "moe_block_capacity": (_I, [_I, _I, _I, _I]),
    "moe_route_prepare_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "moe_route_prepare": (_I, [_P, _I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_route_prepare_noalloc": (_I, [_P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_blockfp8_grouped_gemm": (_I, [_I, _P, _P, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P, _I, _I,
                                       _P, _I, _I, _I, _P]),
    "moe_blockfp8_pack_weights": (_I, [_P, _I, _I, _I, _P, _P]),
    "silu_mul_quant_fp8": (_I, [_I, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _I, _P, _I, _I, _P, _P,
                                _I, _P]),
    "silu_and_mul_bf16": (_I, [_I, _P, _I, _I, _F, _P, _P, _I, _P, _P]),
    "moe_reduce": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_blockfp8_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_blockfp8_forward": (_I, [_P, _P, _P, _I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I,
                                  _F, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_blockfp8_workspace_layout": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "moe_forward_path_for": (_I, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_block_m": (_I, [_I, _I, _I, _I, _I]),
    "moe_blockfp8_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int),
                               ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "moe_blockfp8_dynamic_tail": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_int)]),
    "moe_blockfp8_plan_for_sms": (_I, [_I, _I, _I, _I, _I, _I, _I, _I] + [ctypes.POINTER(ctypes.c_int)] * 5),
    "moe_last_error_string": (ctypes.c_char_p, []),
    "moe_get_device_status": (_I, [ctypes.POINTER(ctypes.c_int), _I]),
    "moe_device_supported": (_I, []),
    "moe_kernel_binary_version": (_I, []),
    "moe_debug_inject_stall": (_I, [_I, ctypes.c_ulonglong]),
    "moe_pointer_device_accessible": (_I, [_P]),
}

_lib = None
_lock = threading.Lock()


class MoeError(RuntimeError):
    pass


def load(path: str | None = None):
    """Loads the library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise MoeError(f"libmoefp8.so is not built ({p}); run __graft_entry__.build()")
            L = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "device tensors must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _io_ptr(t):
    """A forward activation (x, topk_ids, topk_w, out): a CUDA tensor, or a pinned host tensor
    that the device reaches at the same address (the kernels then move its bytes themselves)."""
    if t.is_cuda:
        return _ptr(t)
    assert t.is_contiguous() and t.is_pinned(), "host activations must be contiguous pinned tensors"
    p = ctypes.c_void_p(t.data_ptr())
    if not load().moe_pointer_device_accessible(p):
        raise MoeError("pinned host tensor is not device-accessible at its host address")
    return p


def pointer_device_accessible(t) -> bool:
    return bool(load().moe_pointer_device_accessible(ctypes.c_void_p(t.data_ptr())))


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc, name):
    if rc != MOE_OK:
        msg = load().moe_last_error_string().decode(errors="replace")
        raise MoeError(f"{name} failed with code {rc}: {msg}")


def _i32(t):
    return None if t is None else t.to(torch.int32).contiguous()


def device_status(reset: bool = True) -> int:
    v = ctypes.c_int(0)
    _check(load().moe_get_device_status(ctypes.byref(v), int(reset)), "moe_get_device_status")
    return v.value


def moe_block_capacity(M, k, E_local, block_m) -> int:
    return load().moe_block_capacity(M, k, E_local, block_m)


def moe_route_prepare(topk_ids, E, expert_map, E_local, block_m, path=ROUTE_AUTO, stream=None):
    """Returns dict(sorted_idx, block_expert, num_blocks, expert_count, expert_offset,
    route_slot, B_cap) -- all int32 device tensors except B_cap."""
    L = load()
    ids = _i32(topk_ids)
    M, k = ids.shape
    dev = ids.device
    B_cap = L.moe_block_capacity(M, k, E_local, block_m)
    if B_cap < 0:
        raise MoeError("moe_block_capacity: bad arguments")
    out = dict(
        sorted_idx=torch.empty(max(1, B_cap * block_m), dtype=torch.int32, device=dev)[: B_cap * block_m],
        block_expert=torch.empty(max(1, B_cap), dtype=torch.int32, device=dev)[:B_cap],
        num_blocks=torch.empty(1, dtype=torch.int32, device=dev),
        expert_count=torch.empty(E_local, dtype=torch.int32, device=dev),
        expert_offset=torch.empty(E_local + 1, dtype=torch.int32, device=dev),
        route_slot=torch.empty(max(1, M * k), dtype=torch.int32, device=dev)[: M * k],
    )
    wsb = L.moe_route_prepare_workspace_bytes(M, k, E_local, block_m)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    em = _i32(expert_map)
    rc = L.moe_route_prepare(_ptr(ids), M, k, E, _ptr(em), E_local, block_m, path,
                             _ptr(out["sorted_idx"]), _ptr(out["block_expert"]),
                             _ptr(out["num_blocks"]), _ptr(out["expert_count"]),
                             _ptr(out["expert_offset"]), _ptr(out["route_slot"]), _ptr(ws),
                             ws.numel(), _stream(stream))
    _check(rc, "moe_route_prepare")
    out["B_cap"] = B_cap
    out["_ws"] = ws
    return out


def moe_route_prepare_noalloc(topk_ids, E, expert_map, E_local, block_m, stream=None):
    """Route preparation that allocates nothing inside the library: its scratch is a fixed
    array in the library (for callers that cannot provide device memory).  The output tensors
    below are allocated here by torch only because this is the Python binding; C callers pass
    their own.  Same outputs as moe_route_prepare."""
    L = load()
    ids = _i32(topk_ids)
    M, k = ids.shape
    dev = ids.device
    B_cap = L.moe_block_capacity(M, k, E_local, block_m)
    if B_cap < 0:
        raise MoeError("moe_block_capacity: bad arguments")
    out = dict(
        sorted_idx=torch.empty(max(1, B_cap * block_m), dtype=torch.int32, device=dev)[: B_cap * block_m],
        block_expert=torch.empty(max(1, B_cap), dtype=torch.int32, device=dev)[:B_cap],
        num_blocks=torch.empty(1, dtype=torch.int32, device=dev),
        expert_count=torch.empty(E_local, dtype=torch.int32, device=dev),
        expert_offset=torch.empty(E_local + 1, dtype=torch.int32, device=dev),
        route_slot=torch.empty(max(1, M * k), dtype=torch.int32, device=dev)[: M * k],
    )
    em = _i32(expert_map)
    rc = L.moe_route_prepare_noalloc(_ptr(ids), M, k, E, _ptr(em), E_local, block_m,
                                     _ptr(out["sorted_idx"]), _ptr(out["block_expert"]),
                                     _ptr(out["num_blocks"]), _ptr(out["expert_count"]),
                                     _ptr(out["expert_offset"]), _ptr(out["route_slot"]),
                                     _stream(stream))
    _check(rc, "moe_route_prepare_noalloc")
    out["B_cap"] = B_cap
    return out


def silu_mul_quant_fp8(act, inp, N, rows=None, clamp_limit=float("inf"), fmt=SCALE_F32,
                       row_expert=None, expert_map=None, E=0, row_map=None, row_div=0,
                       out_rows=None, out_q=None, out_s=None, in_splits=1,
                       strategy=QUANT_AUTO, stream=None):
    """Fused (clamped) SiLU*mul + per-128-group E4M3 quantisation, or identity quantisation.

    inp: bf16 [in_rows, W] or float32 [in_splits, in_rows, W]; returns (out_q uint8, out_s f32)."""
    L = load()
    f32 = inp.dtype == torch.float32
    if f32:
        assert inp.dim() == 3 and inp.shape[0] == in_splits
        in_rows = inp.shape[1]
    else:
        assert inp.dtype == torch.bfloat16 and in_splits == 1
        in_rows = inp.shape[0]
    rows = in_rows if rows is None else rows
    out_rows = rows if out_rows is None else out_rows
    dev = inp.device
    if out_q is None:
        out_q = torch.zeros((out_rows, N), dtype=torch.uint8, device=dev)
    if out_s is None:
        out_s = torch.zeros((out_rows, N // 128), dtype=torch.float32, device=dev)
    rc = L.silu_mul_quant_fp8(act, _ptr(inp), DTYPE_F32 if f32 else DTYPE_BF16, in_splits, in_rows,
                              rows, N, float(clamp_limit), fmt, _ptr(_i32(row_expert)),
                              _ptr(_i32(expert_map)), E, _ptr(_i32(row_map)), row_div, out_rows,
                              _ptr(out_q), _ptr(out_s), strategy, _stream(stream))
    _check(rc, "silu_mul_quant_fp8")
    return out_q, out_s


def silu_and_mul_bf16(act, inp, N, clamp_limit=float("inf"), row_expert=None, expert_map=None, E=0,
                      out=None, stream=None):
    L = load()
    if out is None:
        out = torch.empty((inp.shape[0], N), dtype=torch.bfloat16, device=inp.device)
    rc = L.silu_and_mul_bf16(act, _ptr(inp), inp.shape[0], N, float(clamp_limit),
                             _ptr(_i32(row_expert)), _ptr(_i32(expert_map)), E, _ptr(out),
                             _stream(stream))
    _check(rc, "silu_and_mul_bf16")
    return out


def moe_blockfp8_pack_weights(w_q, stream=None):
    """Row-major E4M3 weights [E, N_out, K] -> the tiled layout (every 128x128 block one
    contiguous 16 KB run).  Returns a uint8 tensor of shape [E, N_out/128, K/128, 128, 128]."""
    L = load()
    E, N_out, K = w_q.shape
    out = torch.empty((E, N_out // 128, K // 128, 128, 128), dtype=torch.uint8, device=w_q.device)
    _check(L.moe_blockfp8_pack_weights(_ptr(w_q), E, N_out, K, _ptr(out), _stream(stream)),
           "moe_blockfp8_pack_weights")
    return out


def _weight_dims(w_q):
    """(E_local, N_out, K, layout) of a row-major [E, N_out, K] or tiled [E, NT, KB, 128, 128]
    weight tensor."""
    if w_q.dim() == 5:
        E, NT, KB = w_q.shape[:3]
        return E, NT * 128, KB * 128, WEIGHTS_TILED
    E, N_out, K = w_q.shape
    return E, N_out, K, WEIGHTS_ROW_MAJOR


def moe_blockfp8_grouped_gemm(proj, a_q, a_s, w_q, w_s, route, block_m, out_dtype=DTYPE_BF16,
                              out_rows=None, splits=1, out=None, stream=None):
    """route: the dict returned by moe_route_prepare.  w_q row-major [E, N_out, K] or tiled
    [E, N_out/128, K/128, 128, 128].  Returns the output tensor."""
    L = load()
    a_rows, K = a_q.shape
    E_local, N_out, _, layout = _weight_dims(w_q)
    B_cap = route["B_cap"]
    if out_rows is None:
        out_rows = B_cap * block_m
    if out is None:
        if out_dtype == DTYPE_F32:
            out = torch.zeros((splits, out_rows, N_out), dtype=torch.float32, device=a_q.device)
        else:
            out = torch.zeros((out_rows, N_out), dtype=torch.bfloat16, device=a_q.device)
    rc = L.moe_blockfp8_grouped_gemm(proj, _ptr(a_q), _ptr(a_s), a_rows, K, _ptr(w_q), _ptr(w_s),
                                     E_local, N_out, layout, _ptr(route["sorted_idx"]),
                                     _ptr(route["block_expert"]), _ptr(route["num_blocks"]), B_cap,
                                     block_m, _ptr(out), out_dtype, out_rows, splits,
                                     _stream(stream))
    _check(rc, "moe_blockfp8_grouped_gemm")
    return out


def moe_reduce(z, topk_w, topk_ids, expert_map, E, H, out=None, stream=None, E_local=None):
    """E_local: number of local experts (the range of the expert map's entries); required
    with an expert map, E without one."""
    L = load()
    ids = _i32(topk_ids)
    M, k = ids.shape
    if E_local is None:
        if expert_map is not None:
            raise ValueError("moe_reduce: pass E_local with an expert map")
        E_local = E
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=z.device)
    rc = L.moe_reduce(_ptr(z), _ptr(topk_w.float().contiguous()), _ptr(ids), _ptr(_i32(expert_map)),
                      M, k, E, E_local, H, _ptr(out), _stream(stream))
    _check(rc, "moe_reduce")
    return out


def moe_blockfp8_workspace_bytes(M, k, E, E_local, H, N, block_m=0) -> int:
    return load().moe_blockfp8_workspace_bytes(M, k, E, E_local, H, N, block_m)


WS_REGIONS = ("sorted_idx", "block_expert", "num_blocks", "expert_count", "expert_offset",
              "route_slot", "xq", "xs", "gu", "aq", "as", "z")


def moe_blockfp8_workspace_layout(M, k, E, E_local, H, N, block_m=0) -> dict:
    """Byte offsets of the forward's intermediate tensors inside its workspace, by region name
    (see moe_ws_region in include/moefp8.h for their layouts)."""
    offs = (ctypes.c_size_t * len(WS_REGIONS))()
    _check(load().moe_blockfp8_workspace_layout(M, k, E, E_local, H, N, block_m, offs),
           "moe_blockfp8_workspace_layout")
    return {name: int(offs[i]) for i, name in enumerate(WS_REGIONS)}


def moe_debug_inject_stall(block: int, wait_limit_ns: int) -> None:
    """Test hook: the calling thread's next path-FUSED forward waits for block `block` until
    wait_limit_ns runs out (see include/moefp8.h)."""
    _check(load().moe_debug_inject_stall(block, wait_limit_ns), "moe_debug_inject_stall")


def moe_kernel_binary_version() -> int:
    return load().moe_kernel_binary_version()


def moe_forward_path_for(M, k, E, E_local, H, N) -> int:
    return load().moe_forward_path_for(M, k, E, E_local, H, N)


def moe_forward_block_m(M, k, E_local, H, N) -> int:
    return load().moe_forward_block_m(M, k, E_local, H, N)


def moe_blockfp8_plan(M, k, E, E_local, H, N, block_m=0):
    """(block_m, B_cap, splits) the layer uses for these sizes."""
    bm, bc, sp = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(load().moe_blockfp8_plan(M, k, E, E_local, H, N, block_m, ctypes.byref(bm),
                                    ctypes.byref(bc), ctypes.byref(sp)), "moe_blockfp8_plan")
    return bm.value, bc.value, sp.value


def moe_blockfp8_dynamic_tail(M, k, E, E_local, H, N, block_m=0):
    """(gate_up, down): whether the staged forward's GEMMs take the dynamic tail."""
    gu, dn = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().moe_blockfp8_dynamic_tail(M, k, E, E_local, H, N, block_m, ctypes.byref(gu),
                                            ctypes.byref(dn)), "moe_blockfp8_dynamic_tail")
    return bool(gu.value), bool(dn.value)


def moe_blockfp8_plan_for_sms(M, k, E, E_local, H, N, sms, block_m=0):
    """(block_m, B_cap, splits, dynamic tail on the gate/up GEMM, on the down GEMM) for a device
    with `sms` SMs; host only, no GPU needed."""
    out = [ctypes.c_int(0) for _ in range(5)]
    _check(load().moe_blockfp8_plan_for_sms(M, k, E, E_local, H, N, block_m, sms,
                                            *[ctypes.byref(o) for o in out]),
           "moe_blockfp8_plan_for_sms")
    bm, bc, sp, gu, dn = (o.value for o in out)
    return bm, bc, sp, bool(gu), bool(dn)


def moe_blockfp8_forward(x, topk_ids, topk_w, E, expert_map, wgu_q, wgu_s, wd_q, wd_s,
                         act=ACT_SILU_MUL, clamp_limit=float("inf"), act_fmt=SCALE_F32,
                         block_m=0, out=None, workspace=None, stream=None, path=FORWARD_AUTO):
    """The whole layer.  x: bf16 [M, H]; weights as uint8 E4M3 codes + fp32 block scales.
    x, topk_ids, topk_w and out may be pinned host tensors (read and written by the kernels
    across the host link); the weights, expert_map and workspace are CUDA tensors."""
    L = load()
    assert x.dtype == torch.bfloat16 and topk_ids.dtype == torch.int32 and topk_w.dtype == torch.float32
    assert expert_map is None or expert_map.dtype == torch.int32
    M, H = x.shape
    k = topk_ids.shape[1]
    E_local, _, _, layout = _weight_dims(wgu_q)
    _, H_d, N, layout_d = _weight_dims(wd_q)
    assert layout == layout_d and H_d == H, "both weight tensors must use the same layout"
    need = L.moe_blockfp8_workspace_bytes(M, k, E, E_local, H, N, block_m)
    dev = wgu_q.device
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    rc = L.moe_blockfp8_forward(_io_ptr(x), _io_ptr(topk_ids), _io_ptr(topk_w), M, k, E, _ptr(expert_map),
                                E_local, H, N, _ptr(wgu_q), _ptr(wgu_s), _ptr(wd_q), _ptr(wd_s), layout, act,
                                float(clamp_limit), act_fmt, block_m, path, _io_ptr(out), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc, "moe_blockfp8_forward")
    return out
