"""Latent mixture-of-experts block (pooler -> routed SwiGLU experts with per-expert
RMSNorm -> unpooler) for one GB300, as hand-written sm_103a CUDA behind a C ABI
(include/latent_moe.h).  `_lib` is the ctypes binding, `layer.LatentMoE` the
torch-facing wrapper, `synth` the seeded input generator."""
from . import synth  # noqa: F401


def __getattr__(name):
    if name in ("LatentMoE", "make_config"):
        from . import layer
        return getattr(layer, name)
    raise AttributeError(name)
