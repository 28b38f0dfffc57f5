"""CPU oracle of the block-FP8 mixture-of-experts layer forward (test infrastructure).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg and reference arm
may import this package.  It wraps ``moe_oracle.c`` (plain C, built with gcc) through ctypes
and numpy; it never imports the CUDA package and the CUDA package never imports it.

Every array argument is a numpy array in the layout the C functions document: BF16 values are
carried as their uint16 bit patterns, E4M3 values as uint8 codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

ACT_IDENTITY, ACT_SILU_MUL, ACT_SILU_MUL_GATE_UPPER = 0, 1, 2
SCALE_F32, SCALE_UE8M0 = 0, 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (OpenMP if the compiler has it)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        cmd = base + extra + [_SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _LIB_PATH)
            return _LIB_PATH
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            F = ctypes.c_float
            Ln = ctypes.c_long
            L.orc_e4m3_decode.restype = F
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [F]
            L.orc_exp_f32.restype = F
            L.orc_exp_f32.argtypes = [F]
            L.orc_group_scale.restype = F
            L.orc_group_scale.argtypes = [F, I]
            for name in ("orc_e4m3_encode_array", "orc_e4m3_decode_array", "orc_bf16_round_array",
                         "orc_bf16_round_double_array", "orc_exp_array", "orc_silu_array"):
                getattr(L, name).argtypes = [P, P, Ln]
                getattr(L, name).restype = None
            L.orc_group_scale_array.argtypes = [P, P, Ln, I]
            L.orc_group_scale_array.restype = None
            L.orc_act_quant.argtypes = [I, P, I, I, F, I, P, P, I, P, P, P]
            L.orc_silu_and_mul.argtypes = [I, P, I, I, F, P]
            L.orc_block_capacity.argtypes = [I, I, I]
            L.orc_route_prepare.argtypes = [P, I, I, I, P, I, I, P, P, P, P, P]
            L.orc_route_gemm.argtypes = [P, P, I, I, P, P, I, I, P, P, I, P]
            L.orc_moe_reduce.argtypes = [P, P, P, P, I, I, I, I, P]
            L.orc_moe_forward.argtypes = [P, P, P, I, I, I, P, I, I, I, P, P, P, P, I, F, I, P, I, P]
            L.orc_moe_forward_dense.argtypes = [P, P, P, I, I, I, P, I, I, I, P, P, P, P, I, F, I, P]
            L.orc_set_threads.argtypes = [I]
            _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} returned error {rc}")


def set_threads(n: int) -> int:
    """Set the OpenMP thread count (0 keeps it); returns the count in effect."""
    return lib().orc_set_threads(int(n))


# ---- codecs -------------------------------------------------------------------------------
def e4m3_encode(x):
    x = _c(x, np.float32)
    q = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(x), _p(q), x.size)
    return q


def e4m3_decode(q):
    q = _c(q, np.uint8)
    x = np.empty(q.shape, np.float32)
    lib().orc_e4m3_decode_array(_p(q), _p(x), q.size)
    return x


def bf16_round(x):
    x = _c(x, np.float32)
    h = np.empty(x.shape, np.uint16)
    lib().orc_bf16_round_array(_p(x), _p(h), x.size)
    return h


def bf16_round_double(x):
    x = _c(x, np.float64)
    h = np.empty(x.shape, np.uint16)
    lib().orc_bf16_round_double_array(_p(x), _p(h), x.size)
    return h


def bf16_to_f32(h):
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def exp_f32(x):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.float32)
    lib().orc_exp_array(_p(x), _p(y), x.size)
    return y


def silu_f32(x):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.float32)
    lib().orc_silu_array(_p(x), _p(y), x.size)
    return y


def group_scale(amax, fmt):
    a = _c(amax, np.float32)
    s = np.empty(a.shape, np.float32)
    lib().orc_group_scale_array(_p(a), _p(s), a.size, int(fmt))
    return s


# ---- stages -------------------------------------------------------------------------------
def act_quant(act, inp, N, clamp_limit=float("inf"), fmt=SCALE_F32, row_expert=None,
              expert_map=None, E=0, out_q=None, out_s=None, want_a=False):
    """Per-128-group E4M3 quantisation (identity) or SiLU*mul + quantisation of BF16 rows.

    Rows dropped by the filter keep the contents of out_q / out_s (pass pre-filled arrays)."""
    inp = _c(inp, np.uint16)
    rows = inp.shape[0]
    q = np.zeros((rows, N), np.uint8) if out_q is None else out_q
    s = np.zeros((rows, N // 128), np.float32) if out_s is None else out_s
    a = np.zeros((rows, N), np.uint16) if want_a else None
    re = _c(row_expert, np.int32)
    em = _c(expert_map, np.int32)
    _check(lib().orc_act_quant(int(act), _p(inp), rows, int(N), float(clamp_limit), int(fmt),
                               _p(re), _p(em), int(E), _p(q), _p(s), _p(a)), "act_quant")
    return (q, s, a) if want_a else (q, s)


def silu_and_mul(act, inp, N, clamp_limit=float("inf")):
    inp = _c(inp, np.uint16)
    out = np.zeros((inp.shape[0], N), np.uint16)
    _check(lib().orc_silu_and_mul(int(act), _p(inp), inp.shape[0], int(N), float(clamp_limit),
                                  _p(out)), "silu_and_mul")
    return out


def block_capacity(R, E_loc, bm):
    return lib().orc_block_capacity(int(R), int(E_loc), int(bm))


def route_prepare(topk_ids, E, expert_map, E_loc, bm):
    ids = _c(topk_ids, np.int32)
    M, k = ids.shape
    B_cap = block_capacity(M * k, E_loc, bm)
    sorted_idx = np.empty(B_cap * bm, np.int32)
    block_expert = np.empty(B_cap, np.int32)
    nb = np.zeros(1, np.int32)
    cnt = np.zeros(E_loc, np.int32)
    off = np.zeros(E_loc + 1, np.int32)
    em = _c(expert_map, np.int32)
    _check(lib().orc_route_prepare(_p(ids), M, k, int(E), _p(em), int(E_loc), int(bm),
                                   _p(sorted_idx), _p(block_expert), _p(nb), _p(cnt), _p(off)),
           "route_prepare")
    return dict(sorted_idx=sorted_idx, block_expert=block_expert, num_blocks=int(nb[0]),
                expert_count=cnt, expert_offset=off, B_cap=B_cap)


def route_gemm(aq, a_s, wq, ws, route_row, route_expert):
    """One output row per route: block-scaled FP8 GEMM against that route's expert."""
    aq = _c(aq, np.uint8)
    a_s = _c(a_s, np.float32)
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.float32)
    rr = _c(route_row, np.int32)
    re = _c(route_expert, np.int32)
    a_rows, K = aq.shape
    E_loc, N_out = wq.shape[0], wq.shape[1]
    out = np.zeros((rr.size, N_out), np.uint16)
    _check(lib().orc_route_gemm(_p(aq), _p(a_s), a_rows, K, _p(wq), _p(ws), E_loc, N_out,
                                _p(rr), _p(re), rr.size, _p(out)), "route_gemm")
    return out


def moe_reduce(z, topk_w, topk_ids, expert_map, E, H):
    z = _c(z, np.uint16)
    w = _c(topk_w, np.float32)
    ids = _c(topk_ids, np.int32)
    M, k = ids.shape
    out = np.zeros((M, H), np.uint16)
    em = _c(expert_map, np.int32)
    _check(lib().orc_moe_reduce(_p(z), _p(w), _p(ids), _p(em), M, k, int(E), int(H), _p(out)),
           "moe_reduce")
    return out


def moe_forward(layer, act=ACT_SILU_MUL, clamp_limit=float("inf"), fmt=SCALE_F32,
                tokens=None, dense=False, out=None):
    """Whole layer on a workload dict (see block_fp8_mixture_moe_gb300.workloads).

    tokens: optional list of token indices (sampled evaluation); other rows of ``out`` are left
    as they were (zeros when ``out`` is not given)."""
    x = _c(layer["x"], np.uint16)
    ids = _c(layer["topk_ids"], np.int32)
    w = _c(layer["topk_w"], np.float32)
    em = _c(layer.get("expert_map"), np.int32)
    wgu_q = _c(layer["wgu_q"], np.uint8)
    wgu_s = _c(layer["wgu_s"], np.float32)
    wd_q = _c(layer["wd_q"], np.uint8)
    wd_s = _c(layer["wd_s"], np.float32)
    M, H = x.shape
    k = ids.shape[1]
    E = int(layer["E"])
    E_loc = wgu_q.shape[0]
    N = wd_q.shape[2]
    if out is None:
        out = np.zeros((M, H), np.uint16)
    L = lib()
    if dense:
        assert tokens is None
        rc = L.orc_moe_forward_dense(_p(x), _p(ids), _p(w), M, k, E, _p(em), E_loc, H, N,
                                     _p(wgu_q), _p(wgu_s), _p(wd_q), _p(wd_s), int(act),
                                     float(clamp_limit), int(fmt), _p(out))
    else:
        tl = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        rc = L.orc_moe_forward(_p(x), _p(ids), _p(w), M, k, E, _p(em), E_loc, H, N,
                               _p(wgu_q), _p(wgu_s), _p(wd_q), _p(wd_s), int(act),
                               float(clamp_limit), int(fmt), _p(tl),
                               0 if tl is None else tl.size, _p(out))
    _check(rc, "moe_forward")
    return out


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
