"""ctypes binding of ``include/moe_route.h``: same names, argument
marshalling only.  Every step of the layer runs in the CUDA library; if the
library is missing this module raises instead of computing anything."""
from __future__ import annotations

import ctypes
import os

from . import _build

c_i32, c_u32, c_u64, c_void_p = ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE = -5
MOE_ERR_TIMEOUT = -6

MOE_DEVERR_BAD_ID = 1
MOE_DEVERR_DUP_ID = 2
MOE_DEVERR_TIMEOUT = 4
MOE_DEVERR_CAPACITY = 8

MOE_DTYPE_F32, MOE_DTYPE_BF16, MOE_DTYPE_FP8_BLOCK128 = 0, 1, 2
MOE_LOGITS_F32, MOE_LOGITS_BF16 = 0, 1
MOE_SCORING_SOFTMAX, MOE_SCORING_SIGMOID = 0, 1

EXPORTED = ("moe_plan", "moe_plan_ep", "moe_forward", "moe_forward_timed", "moe_forward_with_ids",
            "moe_forward_noalloc", "moe_check_noalloc", "moe_route_topk", "moe_route_grouped_topk",
            "moe_plan_set_groups", "moe_check", "moe_plan_describe",
            "moe_ep_dispatch", "moe_ep_pack", "moe_ep_combine",
            "moe_strerror", "moe_abi_version")


class MoePlan(ctypes.Structure):
    """Mirror of ``moe_plan_t``."""
    _fields_ = [(n, c_i32) for n in (
        "abi_version", "T", "H", "I", "E", "k", "dtype", "scoring", "renorm", "est", "force_est",
        "tile_n", "route_tpc", "n_chunks", "max_tiles", "g1_mblocks", "g2_mblocks", "ep_size",
        "ep_rank", "e_local", "n_group", "topk_group", "gemm_pair", "gemm_tm", "gemm_dyn")]
    _fields_ += [(n, c_u64) for n in (
        "workspace_bytes", "off_err", "off_ids", "off_w", "off_chunk_counts", "off_lrank",
        "off_counts", "off_offsets", "off_chunk_base", "off_src", "off_pos", "off_tiles",
        "off_ntiles", "off_xq", "off_xs", "off_act", "off_as", "off_y", "off_tiles2",
        "off_ntiles2", "off_dep")]
    _fields_ += [("reserved1", c_u64 * 1)]

    def describe(self) -> str:
        buf = ctypes.create_string_buffer(512)
        lib().moe_plan_describe(ctypes.byref(self), buf, 512)
        return buf.value.decode()


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} is missing: build it with "
            "serving_moe_route_gb300._build.build() (or __graft_entry__.build())")
    L = ctypes.CDLL(path)
    P = c_void_p
    i = ctypes.c_int
    L.moe_abi_version.argtypes = []
    L.moe_abi_version.restype = i
    L.moe_strerror.argtypes = [i]
    L.moe_strerror.restype = ctypes.c_char_p
    L.moe_plan.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.POINTER(MoePlan)]
    L.moe_plan.restype = i
    L.moe_plan_ep.argtypes = [i, i, i, i, i, i, i, i, i, i, i, ctypes.POINTER(MoePlan)]
    L.moe_plan_ep.restype = i
    L.moe_plan_describe.argtypes = [ctypes.POINTER(MoePlan), ctypes.c_char_p, ctypes.c_size_t]
    L.moe_plan_describe.restype = i
    L.moe_forward.argtypes = [ctypes.POINTER(MoePlan), P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    L.moe_forward.restype = i
    L.moe_forward_timed.argtypes = [ctypes.POINTER(MoePlan), P, P, P, P, P, P, P, P,
                                    ctypes.c_size_t, P, ctypes.POINTER(c_void_p), i]
    L.moe_forward_timed.restype = i
    L.moe_forward_with_ids.argtypes = [ctypes.POINTER(MoePlan), P, P, P, P, P, P, P, P, P,
                                       ctypes.c_size_t, P]
    L.moe_forward_with_ids.restype = i
    L.moe_forward_noalloc.argtypes = [ctypes.POINTER(MoePlan), P, P, P, P, P, P, P, P]
    L.moe_forward_noalloc.restype = i
    L.moe_check_noalloc.argtypes = [ctypes.POINTER(MoePlan), ctypes.POINTER(c_u32), P]
    L.moe_check_noalloc.restype = i
    L.moe_route_topk.argtypes = [P, i, i, i, i, i, i, P, P, P]
    L.moe_route_grouped_topk.argtypes = [P, i, i, i, i, i, i, i, i, P, P, P]
    L.moe_route_grouped_topk.restype = i
    L.moe_plan_set_groups.argtypes = [ctypes.POINTER(MoePlan), i, i]
    L.moe_plan_set_groups.restype = i
    L.moe_route_topk.restype = i
    L.moe_check.argtypes = [ctypes.POINTER(MoePlan), P, ctypes.POINTER(c_u32), P]
    L.moe_check.restype = i
    L.moe_ep_dispatch.argtypes = [P, i, i, i, i, P, P, P, P]
    L.moe_ep_dispatch.restype = i
    L.moe_ep_pack.argtypes = [P, i, P, P, i, i, i, i, P, P, P, P, P, P]
    L.moe_ep_pack.restype = i
    L.moe_ep_combine.argtypes = [P, P, i, i, i, P, P]
    L.moe_ep_combine.restype = i
    if L.moe_abi_version() != 4:
        raise RuntimeError("libmoe_route ABI version mismatch")
    _lib = L
    return L


def strerror(code: int) -> str:
    try:
        return lib().moe_strerror(int(code)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


# --------------------------------------------------------------- raw calls
def moe_plan(T, H, I, E, k, dtype, scoring=MOE_SCORING_SOFTMAX, renorm=True, force_est=0):
    p = MoePlan()
    _check(lib().moe_plan(T, H, I, E, k, dtype, scoring, int(bool(renorm)), force_est,
                          ctypes.byref(p)), "moe_plan")
    return p


def moe_plan_ep(T, H, I, E, k, dtype, scoring=MOE_SCORING_SOFTMAX, renorm=True, force_est=0,
                ep_size=1, ep_rank=0):
    p = MoePlan()
    _check(lib().moe_plan_ep(T, H, I, E, k, dtype, scoring, int(bool(renorm)), force_est,
                             ep_size, ep_rank, ctypes.byref(p)), "moe_plan_ep")
    return p


def moe_forward(plan, x, logits, w13, s13, w2, s2, out, ws, ws_bytes, stream):
    """Pointers are ints (device addresses); stream is a cudaStream_t as int."""
    return lib().moe_forward(ctypes.byref(plan), x, logits, w13, s13, w2, s2, out, ws, ws_bytes,
                             stream)


def moe_forward_timed(plan, x, logits, w13, s13, w2, s2, out, ws, ws_bytes, stream, events):
    """events: 7 cudaEvent_t handles (ints) recorded at the launch boundaries."""
    arr = (c_void_p * 7)(*events)
    return lib().moe_forward_timed(ctypes.byref(plan), x, logits, w13, s13, w2, s2, out, ws,
                                   ws_bytes, stream, arr, len(events))


def moe_forward_with_ids(plan, x, ids, topk_w, w13, s13, w2, s2, out, ws, ws_bytes, stream):
    return lib().moe_forward_with_ids(ctypes.byref(plan), x, ids, topk_w, w13, s13, w2, s2, out,
                                      ws, ws_bytes, stream)


def moe_forward_noalloc(plan, x, logits, w13, s13, w2, s2, out, stream):
    """moe_forward with the library's built-in 16 MiB device workspace (no
    allocation anywhere); for callers that cannot allocate device memory."""
    return lib().moe_forward_noalloc(ctypes.byref(plan), x, logits, w13, s13, w2, s2, out, stream)


def moe_check_noalloc(plan, stream):
    """(rc, error bits) of the built-in workspace after moe_forward_noalloc."""
    bits = c_u32(0)
    rc = lib().moe_check_noalloc(ctypes.byref(plan), ctypes.byref(bits), stream)
    return rc, bits.value


def moe_route_topk(logits, logits_dtype, T, E, k, scoring, renorm, ids, w, stream):
    return lib().moe_route_topk(logits, logits_dtype, T, E, k, scoring, int(bool(renorm)), ids, w,
                                stream)


def moe_route_grouped_topk(logits, logits_dtype, T, E, k, n_group, topk_group, scoring, renorm,
                           ids, w, stream):
    return lib().moe_route_grouped_topk(logits, logits_dtype, T, E, k, n_group, topk_group,
                                        scoring, int(bool(renorm)), ids, w, stream)


def moe_plan_set_groups(plan, n_group, topk_group):
    _check(lib().moe_plan_set_groups(ctypes.byref(plan), n_group, topk_group),
           "moe_plan_set_groups")
    return plan


def moe_check(plan, ws, stream):
    bits = c_u32(0)
    rc = lib().moe_check(ctypes.byref(plan), ws, ctypes.byref(bits), stream)
    return rc, bits.value


def moe_ep_dispatch(ids, T, k, e_local, ep_size, send_counts, send_tokens, row_of, stream):
    return lib().moe_ep_dispatch(ids, T, k, e_local, ep_size, send_counts, send_tokens, row_of,
                                 stream)


def moe_ep_pack(x, x_dtype, ids, w, T, H, k, ep_size, send_counts, send_tokens, x_send, ids_send,
                w_send, stream):
    return lib().moe_ep_pack(x, x_dtype, ids, w, T, H, k, ep_size, send_counts, send_tokens,
                             x_send, ids_send, w_send, stream)


def moe_ep_combine(back, row_of, T, H, ep_size, out, stream):
    return lib().moe_ep_combine(back, row_of, T, H, ep_size, out, stream)
