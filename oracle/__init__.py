"""CPU oracle for the fused MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product (``serving_moe_route_gb300``)
never imports it and has no CPU fallback.

The arithmetic lives in ``moe_oracle.c`` (plain C, double accumulation,
OpenMP over tokens); this module compiles it with gcc on first use and
wraps it with ctypes and numpy.  Inputs are numpy arrays in storage form:
fp32 values, bf16 bit patterns (uint16) or e4m3 codes (uint8).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

DTYPE_F32, DTYPE_BF16, DTYPE_FP8 = 0, 1, 2
SOFTMAX, SIGMOID = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmoe_oracle.so`` (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    except subprocess.CalledProcessError as exc:
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{exc.stderr}") from exc
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        _lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        _lib.oracle_bf16_to_f32.restype = ctypes.c_float
        _lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        _lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        _lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        _lib.oracle_e4m3_decode.restype = ctypes.c_float
        _lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        _lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        _lib.oracle_quant_group128.argtypes = [P, i, P, P]
        _lib.oracle_quant_group128.restype = None
        _lib.oracle_estimate.argtypes = [i, i, i]
        _lib.oracle_estimate.restype = i
        _lib.oracle_route.argtypes = [P, i, i, i, i, i, P, P]
        _lib.oracle_route.restype = i
        _lib.oracle_permute.argtypes = [P, i, i, P, P, P, P]
        _lib.oracle_permute.restype = i
        _lib.oracle_moe_forward.argtypes = [i, i, i, i, i, i, i, i, i, i, i, i, P, P, P, P, P, P,
                                            P, i, P, P, P]
        _lib.oracle_route_grouped.argtypes = [P, i, i, i, i, i, i, i, P, P]
        _lib.oracle_route_grouped.restype = i
        _lib.oracle_moe_forward.restype = i
        _lib.oracle_set_threads.argtypes = [i]
        _lib.oracle_set_threads.restype = None
        _lib.oracle_get_threads.argtypes = []
        _lib.oracle_get_threads.restype = i
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- codecs
def bf16_to_f32(bits: int) -> float:
    return float(lib().oracle_bf16_to_f32(int(bits)))


def f32_to_bf16(v: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code)))


def e4m3_encode(v: float) -> int:
    return int(lib().oracle_e4m3_encode(float(v)))


def quant_group128(v: np.ndarray):
    """fp32 row -> (e4m3 codes uint8, fp32 scales per 128-column group)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    n = v.size
    codes = np.empty(n, np.uint8)
    scales = np.empty((n + 127) // 128, np.float32)
    lib().oracle_quant_group128(_ptr(v), n, _ptr(codes), _ptr(scales))
    return codes, scales


# ---------------------------------------------------------------- method
def estimate(T: int, k: int, E: int) -> int:
    return int(lib().oracle_estimate(T, k, E))


def route(logits: np.ndarray, k: int, scoring: int = SOFTMAX, renorm: bool = True):
    """logits [T, E] float32 -> (ids int32 [T, k], w float64 [T, k])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = lib().oracle_route(_ptr(logits), T, E, k, scoring, int(bool(renorm)), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_route: unsupported sizes")
    return ids, w


def route_grouped(logits: np.ndarray, k: int, n_group: int, topk_group: int,
                  scoring: int = SOFTMAX, renorm: bool = True):
    """Group-limited routing: logits [T, E] -> (ids int32 [T, k], w float64)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = lib().oracle_route_grouped(_ptr(logits), T, E, k, n_group, topk_group, scoring,
                                    int(bool(renorm)), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_route_grouped: unsupported sizes")
    return ids, w


def permute(ids: np.ndarray, E: int):
    """flat ids [R] -> (counts [E], offsets [E+1], src [R], pos [R]), all int32."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    R = ids.size
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    src = np.empty(R, np.int32)
    pos = np.empty(R, np.int32)
    rc = lib().oracle_permute(_ptr(ids), R, E, _ptr(counts), _ptr(offsets), _ptr(src), _ptr(pos))
    if rc != 0:
        raise ValueError("oracle_permute: id outside [0, E)")
    return counts, offsets, src, pos


def moe_forward(*, T, H, I, E, k, dtype, scoring, renorm, x, logits, w13, w2, s13=None, s2=None,
                tokens=None, ep_size=1, ep_rank=0, n_group=1, topk_group=1):
    """Fused MoE forward for the listed tokens (default: all).  With
    ep_size > 1, w13/w2/s13/s2 hold rank ep_rank's E/ep_size experts and the
    output is that rank's partial sum.

    Returns (out float64 [n, H], ids int32 [n, k], w float64 [n, k]).
    """
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = T if tok is None else tok.size
    out = np.empty((n, H), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    rc = lib().oracle_moe_forward(
        T, H, I, E, k, dtype, scoring, int(bool(renorm)), n_group, topk_group, ep_size, ep_rank,
        _ptr(x), _ptr(logits), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2),
        _ptr(tok), n, _ptr(out), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_moe_forward: unsupported sizes or token index")
    return out, ids, w


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def threads() -> int:
    return int(lib().oracle_get_threads())
