"""ctypes binding of libmoe_latent.so (declarations in include/latent_moe.h).

Argument marshalling only: every function here forwards to the C entry point of the
same name; all computation runs in the library's CUDA kernels.  Pointers are plain
integers (device addresses from torch tensors' data_ptr(), stream and event handles).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_latent.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

MOE_F32 = 0
MOE_BF16 = 1
MOE_NVFP4 = 2

MOE_FLAG_TEST_TIMEOUT = 0x80000000
MOE_FLAG_WEIGHT_TILES = 0x40000000
MOE_FLAG_NVFP4_PAIR = 0x20000000
MOE_FLAG_NVFP4_ONE_CTA = 0x10000000

PACK_ROUTER, PACK_W13, PACK_W2, PACK_POOL, PACK_UNPOOL, PACK_SF13, PACK_SF2, PACK_GS13, \
    PACK_GS2 = range(9)

# every symbol the header declares
EXPORTS = ("moe_workspace_size", "moe_workspace_init", "moe_packed_bytes", "moe_pack_weights",
           "moe_quantize_nvfp4", "moe_route", "moe_route_noalloc",
           "moe_read_noalloc_status", "moe_forward",
           "moe_boundary", "moe_forward_boundary", "moe_forward_profiled",
           "moe_num_stages",
           "moe_stage_name", "moe_forward_launches", "moe_workspace_offsets",
           "moe_read_status", "moe_status_string")

OFFSET_NAMES = ("h32", "h16", "ids", "w", "pooled", "row_off", "src", "inv", "a_perm", "s",
                "y", "c", "sf_u", "sf_s", "alpha", "row_cnt", "bnd_ssq", "bnd_cnt")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("p", ctypes.c_int32),
                ("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("I", ctypes.c_int32),
                ("eps", ctypes.c_float), ("act", ctypes.c_int32), ("expert", ctypes.c_int32),
                ("out", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class moe_weights_t(ctypes.Structure):
    _fields_ = [("g_in", ctypes.c_void_p), ("w_router", ctypes.c_void_p),
                ("w_pool", ctypes.c_void_p), ("g_pool", ctypes.c_void_p),
                ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("g_exp", ctypes.c_void_p),
                ("w_unpool", ctypes.c_void_p), ("sf13", ctypes.c_void_p),
                ("sf2", ctypes.c_void_p), ("gs13", ctypes.c_void_p), ("gs2", ctypes.c_void_p),
                ("gs_act2", ctypes.c_void_p)]


class moe_canonical_weights_t(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("w_pool", ctypes.c_void_p),
                ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("w_unpool", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "latent_moe_layer_rmsnorm_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    cfgp = ctypes.POINTER(moe_config_t)
    wp = ctypes.POINTER(moe_weights_t)
    L.moe_workspace_size.argtypes = [cfgp]
    L.moe_workspace_size.restype = sz
    L.moe_workspace_init.argtypes = [vp, sz, vp]
    L.moe_workspace_init.restype = i32
    L.moe_packed_bytes.argtypes = [cfgp, i32]
    L.moe_packed_bytes.restype = sz
    L.moe_pack_weights.argtypes = [cfgp, ctypes.POINTER(moe_canonical_weights_t), vp, vp, vp,
                                   vp, vp, vp]
    L.moe_pack_weights.restype = i32
    L.moe_quantize_nvfp4.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_quantize_nvfp4.restype = i32
    L.moe_route.argtypes = [cfgp, wp, vp, vp, vp, vp, sz, vp]
    L.moe_route.restype = i32
    L.moe_route_noalloc.argtypes = [cfgp, wp, vp, vp, vp, vp]
    L.moe_route_noalloc.restype = i32
    L.moe_read_noalloc_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    L.moe_read_noalloc_status.restype = i32
    L.moe_forward.argtypes = [cfgp, wp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_boundary.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_boundary.restype = i32
    L.moe_forward_boundary.argtypes = [cfgp, wp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_forward_boundary.restype = i32
    L.moe_forward.restype = i32
    L.moe_forward_profiled.argtypes = [cfgp, wp, vp, vp, vp, vp, vp, sz, vp,
                                       ctypes.POINTER(vp), i32]
    L.moe_forward_profiled.restype = i32
    L.moe_num_stages.argtypes = []
    L.moe_num_stages.restype = i32
    L.moe_stage_name.argtypes = [i32]
    L.moe_stage_name.restype = ctypes.c_char_p
    L.moe_forward_launches.argtypes = [cfgp, i32]
    L.moe_forward_launches.restype = i32
    L.moe_workspace_offsets.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t), i32]
    L.moe_workspace_offsets.restype = i32
    L.moe_read_status.argtypes = [vp, sz, vp, ctypes.POINTER(ctypes.c_int32)]
    L.moe_read_status.restype = i32
    L.moe_status_string.argtypes = [i32]
    L.moe_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _ref(s):
    return ctypes.byref(s) if s is not None else None


# ---- same-name wrappers --------------------------------------------------------------

def moe_workspace_size(cfg: moe_config_t) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(cfg)))


def moe_workspace_init(ws: int, ws_bytes: int, stream: int) -> int:
    return int(lib().moe_workspace_init(ws, ws_bytes, stream))


def moe_packed_bytes(cfg: moe_config_t, which: int) -> int:
    return int(lib().moe_packed_bytes(ctypes.byref(cfg), which))


def moe_pack_weights(cfg, src: moe_canonical_weights_t, w_router_out, w13_out, w2_out,
                     w_pool_out, w_unpool_out, stream) -> int:
    return int(lib().moe_pack_weights(ctypes.byref(cfg), ctypes.byref(src), w_router_out,
                                      w13_out, w2_out, w_pool_out, w_unpool_out, stream))


def moe_quantize_nvfp4(cfg, w_gate, w_up, w_down, w13_out, sf13_out, gs13_out, w2_out,
                       sf2_out, gs2_out, stream) -> int:
    return int(lib().moe_quantize_nvfp4(ctypes.byref(cfg), w_gate, w_up, w_down, w13_out,
                                        sf13_out, gs13_out, w2_out, sf2_out, gs2_out, stream))


def moe_route(cfg, W: moe_weights_t, x, ids, w, ws, ws_bytes, stream) -> int:
    return int(lib().moe_route(ctypes.byref(cfg), _ref(W), x, ids, w, ws, ws_bytes, stream))


def moe_route_noalloc(cfg, W: moe_weights_t, x, ids, w, stream) -> int:
    return int(lib().moe_route_noalloc(ctypes.byref(cfg), _ref(W), x, ids, w, stream))


def moe_forward(cfg, W: moe_weights_t, x, ids, w, out, ws, ws_bytes, stream) -> int:
    return int(lib().moe_forward(ctypes.byref(cfg), _ref(W), x, ids, w, out, ws, ws_bytes,
                                 stream))


def moe_boundary(cfg, x, y, g_post, gate, g_next, x_out, h_next, stream) -> int:
    return int(lib().moe_boundary(ctypes.byref(cfg), x, y, g_post, gate, g_next, x_out,
                                  h_next, stream))


def moe_forward_boundary(cfg, W: moe_weights_t, x, ids, w, g_post, gate, g_next, y, x_out,
                         h_next, ws, ws_bytes, stream) -> int:
    return int(lib().moe_forward_boundary(ctypes.byref(cfg), _ref(W), x, ids, w, g_post, gate,
                                          g_next, y, x_out, h_next, ws, ws_bytes, stream))


def moe_forward_profiled(cfg, W, x, ids, w, out, ws, ws_bytes, stream, events) -> int:
    arr = (ctypes.c_void_p * len(events))(*events)
    return int(lib().moe_forward_profiled(ctypes.byref(cfg), _ref(W), x, ids, w, out, ws,
                                          ws_bytes, stream, arr, len(events)))


def moe_num_stages() -> int:
    return int(lib().moe_num_stages())


def moe_stage_name(i: int) -> str:
    return lib().moe_stage_name(i).decode()


def moe_forward_launches(cfg, route_internally: bool) -> int:
    return int(lib().moe_forward_launches(ctypes.byref(cfg), 1 if route_internally else 0))


def moe_workspace_offsets(cfg) -> dict:
    arr = (ctypes.c_size_t * len(OFFSET_NAMES))()
    n = int(lib().moe_workspace_offsets(ctypes.byref(cfg), arr, len(OFFSET_NAMES)))
    return {OFFSET_NAMES[i]: int(arr[i]) for i in range(n)}


def moe_read_status(ws, ws_bytes, stream):
    detail = ctypes.c_int32(0)
    st = int(lib().moe_read_status(ws, ws_bytes, stream, ctypes.byref(detail)))
    return st, int(detail.value)


def moe_read_noalloc_status(stream):
    detail = ctypes.c_int32(0)
    st = int(lib().moe_read_noalloc_status(stream, ctypes.byref(detail)))
    return st, int(detail.value)


def status_string(s: int) -> str:
    return lib().moe_status_string(int(s)).decode()


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)
