"""Latent mixture-of-experts block (pooler -> routed SwiGLU experts with per-expert
RMSNorm -> unpooler) for one GB300, as hand-written sm_103a CUDA behind a C ABI."""
