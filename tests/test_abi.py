"""The C-ABI library: it loads, exports every entry point the header declares, and
rejects bad arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from latent_moe_layer_rmsnorm_gb300 import build
from latent_moe_layer_rmsnorm_gb300 import _lib as L

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "latent_moe.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(L.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = L.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name


def cfg(**kw):
    base = dict(T=64, d=256, p=128, E=8, top_k=2, I=256, eps=1e-6, act=L.MOE_BF16,
                expert=L.MOE_BF16, out=L.MOE_F32, flags=0)
    base.update(kw)
    return L.moe_config_t(**base)


def test_workspace_size_and_validation():
    assert L.moe_workspace_size(cfg()) > 0
    assert L.moe_workspace_size(cfg(T=0)) > 0
    bad = [dict(top_k=9), dict(top_k=0), dict(E=0), dict(E=300), dict(d=200), dict(p=96),
           dict(I=100), dict(act=7), dict(out=2), dict(eps=-1.0), dict(flags=1),
           dict(expert=L.MOE_F32), dict(T=-1), dict(top_k=9, E=8),
           dict(flags=L.MOE_FLAG_NVFP4_PAIR | L.MOE_FLAG_NVFP4_ONE_CTA)]
    for b in bad:
        assert L.moe_workspace_size(cfg(**b)) == 0, b


def test_workspace_grows_with_tokens():
    a = L.moe_workspace_size(cfg(T=64))
    b = L.moe_workspace_size(cfg(T=128))
    assert b > a
    assert L.moe_workspace_size(cfg(act=L.MOE_F32, expert=L.MOE_F32)) > a


def test_packed_sizes():
    c = cfg(T=1)
    assert L.moe_packed_bytes(c, L.PACK_ROUTER) == 8 * 256 * 4
    assert L.moe_packed_bytes(c, L.PACK_W13) == 8 * 2 * 256 * 128 * 2
    assert L.moe_packed_bytes(c, L.PACK_W2) == 8 * 128 * 256 * 2   # BF16: an FP16 copy
    f = cfg(T=1, act=L.MOE_F32, expert=L.MOE_F32)
    assert L.moe_packed_bytes(f, L.PACK_W2) == 8 * 128 * 256 * 4
    assert L.moe_packed_bytes(f, L.PACK_POOL) == 128 * 256 * 4


FAKE = 1 << 20   # an aligned non-null address that is never dereferenced on the host


def weights():
    return L.moe_weights_t(g_in=FAKE, w_router=FAKE, w_pool=FAKE, g_pool=FAKE, w13=FAKE,
                           w2=FAKE, g_exp=FAKE, w_unpool=FAKE)


def test_host_side_errors_before_any_launch():
    c = cfg()
    ws = L.moe_workspace_size(c)
    W = weights()
    # null config / weights / input / output
    assert L.lib().moe_forward(None, ctypes.byref(W), FAKE, None, None, FAKE, FAKE, ws, None) \
        == L.MOE_ERR_INVALID_ARG
    assert L.moe_forward(c, None, FAKE, None, None, FAKE, FAKE, ws, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_forward(c, W, None, None, None, FAKE, FAKE, ws, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_forward(c, W, FAKE, None, None, None, FAKE, ws, None) == L.MOE_ERR_INVALID_ARG
    # ids without weights
    assert L.moe_forward(c, W, FAKE, FAKE, None, FAKE, FAKE, ws, None) == L.MOE_ERR_INVALID_ARG
    # misaligned input
    assert L.moe_forward(c, W, FAKE + 2, None, None, FAKE, FAKE, ws, None) == L.MOE_ERR_INVALID_ARG
    # workspace: missing, misaligned, too small
    assert L.moe_forward(c, W, FAKE, None, None, FAKE, None, ws, None) == L.MOE_ERR_WORKSPACE
    assert L.moe_forward(c, W, FAKE, None, None, FAKE, FAKE + 16, ws, None) == L.MOE_ERR_WORKSPACE
    assert L.moe_forward(c, W, FAKE, None, None, FAKE, FAKE, ws - 1, None) == L.MOE_ERR_WORKSPACE
    # a null weight
    W2 = weights()
    W2.w13 = None
    assert L.moe_forward(c, W2, FAKE, None, None, FAKE, FAKE, ws, None) == L.MOE_ERR_INVALID_ARG
    # unsupported sizes
    assert L.moe_forward(cfg(E=512), W, FAKE, None, None, FAKE, FAKE, ws, None) \
        == L.MOE_ERR_UNSUPPORTED
    # route-only needs ids and weights outputs
    assert L.moe_route(c, W, FAKE, None, FAKE, FAKE, ws, None) == L.MOE_ERR_INVALID_ARG
    # T = 0 is a no-op that launches nothing
    c0 = cfg(T=0)
    assert L.moe_forward(c0, W, FAKE, None, None, FAKE, FAKE, L.moe_workspace_size(c0), None) \
        == L.MOE_OK
    assert L.moe_forward_launches(c0, True) == 0
    big = cfg(T=16384)                       # enough output tiles: no split-K reductions
    assert L.moe_forward_launches(big, True) == 11
    assert L.moe_forward_launches(big, False) == 10
    # few tokens at full widths: the router, pooler and unpooler split K and add one
    # reduction each; 512 (token, slot) pairs are one dispatch chunk, so the histogram,
    # scan and scatter run as one kernel
    dec = cfg(T=64, d=8192, p=4096, E=256, top_k=8, I=4096)
    assert L.moe_forward_launches(dec, True) == 12
    assert L.moe_forward_launches(dec, False) == 10


def test_boundary_host_side_errors():
    """moe_boundary rejects null, misaligned and overlapping buffers before any launch;
    T = 0 is a no-op.  (x_out == x, the in-place update, is allowed.)"""
    c = cfg(T=4, d=256)
    n = 4 * 256 * 2                     # bytes of one [T, d] BF16 buffer
    X, Y, XO, H, G = FAKE, 2 * FAKE, 3 * FAKE, 4 * FAKE, 5 * FAKE
    assert L.moe_boundary(c, None, Y, G, None, G, XO, H, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X, Y, None, None, G, XO, H, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X, Y, G, None, G, XO, None, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X + 2, Y, G, None, G, XO, H, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X, Y, G, G + 4, G, XO, H, None) == L.MOE_ERR_INVALID_ARG
    # h_next overlapping x, y or x_out; x_out overlapping y or part of x
    assert L.moe_boundary(c, X, Y, G, None, G, XO, X + n - 16, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X, Y, G, None, G, XO, Y, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X, Y, G, None, G, XO, XO + 16, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X, Y, G, None, G, Y, H, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(c, X, Y, G, None, G, X + 16, H, None) == L.MOE_ERR_INVALID_ARG
    assert L.lib().moe_boundary(None, X, Y, G, None, G, XO, H, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_boundary(cfg(T=0, d=256), X, Y, G, None, G, XO, H, None) == L.MOE_OK


def test_fused_boundary_host_side_errors():
    """moe_forward_boundary checks the boundary's buffers like moe_boundary (y, written by
    the call, may not overlap x either) and the block's like moe_forward, before any
    launch; T = 0 is a no-op."""
    c = cfg(T=4, d=256)
    ws = L.moe_workspace_size(c)
    W = weights()
    n = 4 * 256 * 2
    X, Y, XO, H, G, WS = FAKE, 2 * FAKE, 3 * FAKE, 4 * FAKE, 5 * FAKE, 6 * FAKE
    fb = L.moe_forward_boundary
    assert fb(c, W, X, None, None, None, None, G, Y, XO, H, WS, ws, None) == L.MOE_ERR_INVALID_ARG
    assert fb(c, W, X, None, None, G, None, G, None, XO, H, WS, ws, None) == L.MOE_ERR_INVALID_ARG
    assert fb(c, W, X, None, None, G, G + 4, G, Y, XO, H, WS, ws, None) == L.MOE_ERR_INVALID_ARG
    assert fb(c, W, X, None, None, G, None, G, X + n - 16, XO, H, WS, ws, None) \
        == L.MOE_ERR_INVALID_ARG
    assert fb(c, W, X, None, None, G, None, G, Y, Y, H, WS, ws, None) == L.MOE_ERR_INVALID_ARG
    assert fb(c, W, X, None, None, G, None, G, Y, XO, XO, WS, ws, None) == L.MOE_ERR_INVALID_ARG
    assert fb(c, None, X, None, None, G, None, G, Y, XO, H, WS, ws, None) == L.MOE_ERR_INVALID_ARG
    assert fb(c, W, X, None, None, G, None, G, Y, XO, H, WS, ws - 1, None) == L.MOE_ERR_WORKSPACE
    assert fb(c, W, X, FAKE, None, G, None, G, Y, XO, H, WS, ws, None) == L.MOE_ERR_INVALID_ARG
    c0 = cfg(T=0, d=256)
    assert fb(c0, W, X, None, None, G, None, G, Y, XO, H, WS, L.moe_workspace_size(c0), None) \
        == L.MOE_OK


def test_stage_names_and_status_strings():
    n = L.moe_num_stages()
    assert n == 8
    names = [L.moe_stage_name(i) for i in range(n)]
    assert names[0] == "norm" and names[-1] == "unpool"
    assert L.moe_stage_name(n) == ""
    assert L.status_string(L.MOE_ERR_TIMEOUT) == "device wait timed out"
    with pytest.raises(L.MoeError):
        L.check(L.MOE_ERR_WORKSPACE, "x")
