"""Torch-facing wrapper of the C ABI: owns the device buffers, marshals pointers.

PyTorch only allocates memory and supplies the stream; every step of the layer runs
in libmoe_latent.so's kernels.  There is no CPU path: without the library or a CUDA
device the constructor raises.
"""
from __future__ import annotations

import torch

from . import _lib as L
from .synth import Shape

_DT = {"bf16": L.MOE_BF16, "f32": L.MOE_F32, "nvfp4": L.MOE_NVFP4}
_TORCH = {"bf16": torch.bfloat16, "f32": torch.float32, "nvfp4": torch.bfloat16}


def make_config(shape: Shape, T: int | None = None, out: str = "bf16",
                flags: int = 0) -> L.moe_config_t:
    return L.moe_config_t(T=shape.T if T is None else T, d=shape.d, p=shape.p, E=shape.E,
                          top_k=shape.top_k, I=shape.I, eps=shape.eps, act=_DT[shape.act],
                          expert=_DT[shape.expert], out=_DT[out], flags=flags)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


class LatentMoE:
    """One latent-MoE layer with packed weights resident on the current CUDA device.

    weights: canonical tensors as produced by synth.make_inputs (x is ignored):
    g_in, w_router, w_pool, g_pool, w_gate, w_up, w_down, g_exp, w_unpool.
    keep_canonical=False releases the gate/up tensors after packing.
    """

    def __init__(self, shape: Shape, weights: dict, out: str = "bf16",
                 keep_canonical: bool = True):
        if not torch.cuda.is_available():
            raise RuntimeError("LatentMoE needs a CUDA device (no CPU path)")
        L.lib()
        self.shape = shape
        self.out = out
        cfg = make_config(shape, out=out)
        dev = weights["w_router"].device
        self.device = dev
        w = {k: v.contiguous() for k, v in weights.items() if isinstance(v, torch.Tensor)}

        def buf(which, dtype):
            n = L.moe_packed_bytes(cfg, which)
            if n == 0:
                return None
            es = torch.tensor([], dtype=dtype).element_size()
            return torch.empty(n // es, dtype=dtype, device=dev)

        # packed operand dtypes: FP16 for BF16 configurations, FP32 (TF32-rounded) else
        op = torch.float32 if shape.act == "f32" else torch.float16
        nvf4 = shape.expert == "nvfp4"
        self.w_router = buf(L.PACK_ROUTER, torch.float32)
        if nvf4:
            self.w13, w2p = buf(L.PACK_W13, torch.uint8), buf(L.PACK_W2, torch.uint8)
            self.sf13, self.sf2 = buf(L.PACK_SF13, torch.uint8), buf(L.PACK_SF2, torch.uint8)
            self.gs13, self.gs2 = buf(L.PACK_GS13, torch.float32), buf(L.PACK_GS2, torch.float32)
            self.gs_act2 = w["gs_act2"].float().contiguous()
        else:
            self.w13, w2p = buf(L.PACK_W13, op), buf(L.PACK_W2, op)
            self.sf13 = self.sf2 = self.gs13 = self.gs2 = self.gs_act2 = None
        poolp, unpoolp = buf(L.PACK_POOL, op), buf(L.PACK_UNPOOL, op)
        src = L.moe_canonical_weights_t(
            w_router=_ptr(w["w_router"]), w_pool=_ptr(w["w_pool"]), w_gate=_ptr(w["w_gate"]),
            w_up=_ptr(w["w_up"]), w_down=_ptr(w["w_down"]), w_unpool=_ptr(w["w_unpool"]))
        L.check(L.moe_pack_weights(cfg, src, _ptr(self.w_router),
                                   None if nvf4 else _ptr(self.w13),
                                   None if nvf4 else _ptr(w2p), _ptr(poolp), _ptr(unpoolp),
                                   _stream()), "moe_pack_weights")
        if nvf4:
            L.check(L.moe_quantize_nvfp4(cfg, _ptr(w["w_gate"]), _ptr(w["w_up"]),
                                         _ptr(w["w_down"]), _ptr(self.w13), _ptr(self.sf13),
                                         _ptr(self.gs13), _ptr(w2p), _ptr(self.sf2),
                                         _ptr(self.gs2), _stream()), "moe_quantize_nvfp4")
        self.w2 = w2p if w2p is not None else w["w_down"]
        self.w_pool = poolp if poolp is not None else w["w_pool"]
        self.w_unpool = unpoolp if unpoolp is not None else w["w_unpool"]
        self.g_in, self.g_pool, self.g_exp = (w["g_in"].float().contiguous(),
                                              w["g_pool"].float().contiguous(),
                                              w["g_exp"].float().contiguous())
        self.W = L.moe_weights_t(g_in=_ptr(self.g_in), w_router=_ptr(self.w_router),
                                 w_pool=_ptr(self.w_pool), g_pool=_ptr(self.g_pool),
                                 w13=_ptr(self.w13), w2=_ptr(self.w2), g_exp=_ptr(self.g_exp),
                                 w_unpool=_ptr(self.w_unpool), sf13=_ptr(self.sf13),
                                 sf2=_ptr(self.sf2), gs13=_ptr(self.gs13), gs2=_ptr(self.gs2),
                                 gs_act2=_ptr(self.gs_act2))
        if keep_canonical:
            self.canonical = w
        self.ws = None
        self.ws_bytes = 0

    # ---- buffers -----------------------------------------------------------------------
    def config(self, T: int, flags: int = 0) -> L.moe_config_t:
        return make_config(self.shape, T=T, out=self.out, flags=flags)

    def workspace(self, T: int) -> tuple[int, int]:
        need = L.moe_workspace_size(self.config(T))
        if need == 0:
            raise L.MoeError(L.MOE_ERR_INVALID_ARG, "moe_workspace_size")
        if self.ws is None or self.ws_bytes < need:
            self.ws = torch.empty(need + 256, dtype=torch.uint8, device=self.device)
            self.ws_off = (-self.ws.data_ptr()) % 256
            self.ws_bytes = need
            L.check(L.moe_workspace_init(self.ws.data_ptr() + self.ws_off, need, _stream()),
                    "moe_workspace_init")
        return self.ws.data_ptr() + self.ws_off, self.ws_bytes

    def out_dtype(self):
        return _TORCH[self.out]

    # ---- calls -----------------------------------------------------------------------
    def forward(self, x: torch.Tensor, ids: torch.Tensor | None = None,
                w: torch.Tensor | None = None, out: torch.Tensor | None = None,
                flags: int = 0, events=None) -> torch.Tensor:
        T = x.shape[0]
        assert x.is_contiguous() and x.dtype == _TORCH[self.shape.act]
        if out is None:
            out = torch.empty((T, self.shape.d), dtype=self.out_dtype(), device=x.device)
        ws, nbytes = self.workspace(T)
        cfg = self.config(T, flags)
        if ids is not None:
            ids = ids.to(torch.int32).contiguous()
            w = w.to(torch.float32).contiguous()
        if events is None:
            st = L.moe_forward(cfg, self.W, x.data_ptr(), _ptr(ids), _ptr(w), out.data_ptr(),
                               ws, nbytes, _stream())
        else:
            st = L.moe_forward_profiled(cfg, self.W, x.data_ptr(), _ptr(ids), _ptr(w),
                                        out.data_ptr(), ws, nbytes, _stream(), events)
        L.check(st, "moe_forward")
        return out

    def route(self, x: torch.Tensor):
        T = x.shape[0]
        k = self.shape.top_k
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
        ws, nbytes = self.workspace(T)
        L.check(L.moe_route(self.config(T), self.W, x.data_ptr(), ids.data_ptr(), w.data_ptr(),
                            ws, nbytes, _stream()), "moe_route")
        return ids, w

    def boundary(self, x: torch.Tensor, y: torch.Tensor, g_post: torch.Tensor,
                 g_next: torch.Tensor, gate=None, x_out=None, h_next=None):
        """Post-norm of the block output y, residual add into x and the next block's
        pre-norm (moe_boundary).  Returns (x_out, h_next); x_out may be x (in place)."""
        T = x.shape[0]
        if x_out is None:
            x_out = torch.empty_like(x)
        if h_next is None:
            h_next = torch.empty_like(x)
        L.check(L.moe_boundary(self.config(T), x.data_ptr(), y.data_ptr(), g_post.data_ptr(),
                               None if gate is None else gate.data_ptr(), g_next.data_ptr(),
                               x_out.data_ptr(), h_next.data_ptr(), _stream()), "moe_boundary")
        return x_out, h_next

    def forward_boundary(self, x: torch.Tensor, g_post: torch.Tensor, g_next: torch.Tensor,
                         gate=None, ids=None, w=None, y=None, x_out=None, h_next=None,
                         flags: int = 0):
        """The block and its boundary in one call (moe_forward_boundary): the row pass
        runs inside the unpooler's kernel.  Returns (y, x_out, h_next); x_out may be x."""
        T = x.shape[0]
        assert x.is_contiguous() and x.dtype == _TORCH[self.shape.act]
        if y is None:
            y = torch.empty((T, self.shape.d), dtype=self.out_dtype(), device=x.device)
        if x_out is None:
            x_out = torch.empty_like(x)
        if h_next is None:
            h_next = torch.empty_like(x)
        if ids is not None:
            ids = ids.to(torch.int32).contiguous()
            w = w.to(torch.float32).contiguous()
        ws, nbytes = self.workspace(T)
        L.check(L.moe_forward_boundary(self.config(T, flags), self.W, x.data_ptr(), _ptr(ids),
                                       _ptr(w), g_post.data_ptr(), _ptr(gate), g_next.data_ptr(),
                                       y.data_ptr(), x_out.data_ptr(), h_next.data_ptr(), ws,
                                       nbytes, _stream()), "moe_forward_boundary")
        return y, x_out, h_next

    def read_status(self):
        ws, nbytes = self.workspace(1) if self.ws is None else (self.ws.data_ptr() + self.ws_off,
                                                                 self.ws_bytes)
        return L.moe_read_status(ws, nbytes, _stream())

    def intermediate(self, name: str, T: int) -> torch.Tensor:
        """Copy of one workspace intermediate after a call with T tokens (for tests)."""
        sh, k = self.shape, self.shape.top_k
        f32 = sh.act == "f32"
        op = torch.float32 if f32 else torch.float16
        R = 128 * ((T * k + 127) // 128 + sh.E)    # every expert's rows start on a 128-row boundary
        if sh.expert == "nvfp4":
            rows = {"src": ((R,), torch.int32), "a_perm": ((R, sh.p // 2), torch.uint8),
                    "s": ((R, sh.I // 2), torch.uint8), "y": ((R, sh.p), torch.float16),
                    "sf_u": ((R * sh.p // 16,), torch.uint8),
                    "sf_s": ((R * sh.I // 16,), torch.uint8), "alpha": ((R,), torch.float32)}
        else:
            rows = {"src": ((R,), torch.int32), "a_perm": ((R, sh.p), op),
                    "s": ((R, sh.I), torch.float32 if f32 else torch.float16),
                    "y": ((R, sh.p),
                          torch.float32 if sh.expert == "f32" else torch.float16)}
        spec = {"h32": ((T, sh.d), torch.float32), "h16": ((T, sh.d), torch.float16),
                "ids": ((T, k), torch.int32), "w": ((T, k), torch.float32),
                "pooled": ((T, sh.p), torch.float32), "row_off": ((sh.E + 1,), torch.int32),
                "row_cnt": ((sh.E + 1,), torch.int32), "inv": ((T * k,), torch.int32),
                "c": ((T, sh.p), op),
                "bnd_ssq": ((T, sh.d // 128), torch.float32),
                "bnd_cnt": ((8 * ((T + 255) // 256) + 1,), torch.int32)}
        spec.update(rows)
        shape, dtype = spec[name]
        off = L.moe_workspace_offsets(self.config(T))[name] + self.ws_off
        n = 1
        for v in shape:
            n *= v
        es = torch.tensor([], dtype=dtype).element_size()
        return self.ws[off: off + n * es].view(dtype).reshape(shape).clone()

    def launches(self, T: int, route_internally: bool = True) -> int:
        return L.moe_forward_launches(self.config(T), route_internally)
