"""Runs the oracle's per-expert steps in worker processes, for the full-size parity tests.

The oracle's `moe_forward(..., expert_map=...)` hands the per-expert steps (one task per
routed expert: the expert id, its rows of u and the step's argument) to the map; this
module's map runs them in a pool of spawned processes.  A worker draws expert e's
matrices itself with the generator's per-expert recipe (`synth.make_expert`, on the
CPU, the same draw the GPU copy of the weights was made from), so no weights travel
between processes, and calls the oracle's own step on them: `oracle.chain_expert`
(BF16 / FP32 experts) or `oracle.nvfp4_expert_weights` + `oracle.nvfp4_expert_rows`
(NVFP4).  For NVFP4 it also returns a digest of the quantised weights laid out as the
library stores them, so a test can check the GPU's quantised weights of every routed
expert bit for bit without moving them.

The pool uses the spawn start method (never fork after CUDA has been initialised).
"""
from __future__ import annotations

import atexit
import hashlib
import multiprocessing as mp
import os

import numpy as np

_POOL = None
TASK_TIMEOUT_S = 900.0
_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _init_worker():
    import torch
    torch.set_num_threads(1)


def workers() -> int:
    n = os.cpu_count() or 1
    try:      # leave ~3 GB of host memory per worker
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
        n = min(n, max(1, int(avail // (3 << 30))))
    except (ValueError, OSError, AttributeError):
        pass
    return max(1, min(n, 32))


def pool():
    global _POOL
    if _POOL is None:
        saved = {k: os.environ.get(k) for k in _THREAD_VARS}
        for k in _THREAD_VARS:       # one BLAS thread per worker process
            os.environ[k] = "1"
        try:
            _POOL = mp.get_context("spawn").Pool(workers(), initializer=_init_worker)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        atexit.register(_POOL.terminate)
    return _POOL


# ---- the library's NVFP4 weight layout (declared in include/latent_moe.h) ---------------

def w13_row_map(I: int) -> np.ndarray:
    """Library row of the packed gate/up matrix -> row of [gate; up] (blocks of 64)."""
    r = np.arange(2 * I)
    b, i = r // 128, r % 128
    return np.where(i < 64, b * 64 + i, I + b * 64 + (i - 64))


def pack_codes(q: np.ndarray) -> np.ndarray:
    """[rows, K] E2M1 codes -> [rows, K/2] bytes, even K element in the low nibble."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def chunk_scales(sf: np.ndarray) -> np.ndarray:
    """[rows, K/16] scale codes (rows a multiple of 128) -> the chunked layout: 512-byte
    chunks (row / 128, k / 64), chunk-row-major; byte (r % 32) * 16 + ((r % 128) / 32) * 4
    + g % 4 inside a chunk."""
    rows, G = sf.shape
    r = np.arange(rows)[:, None]
    g = np.arange(G)[None, :]
    off = ((r // 128) * (G // 4) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    out = np.zeros(rows * G, dtype=np.uint8)
    out[off.reshape(-1)] = sf.reshape(-1)
    return out


def nvfp4_digest(parts) -> str:
    """sha256 over codes13, scales13, codes2, scales2, g13, g2 in the library's layout;
    `parts` = (codes13, sf13, codes2, sf2, g13, g2) as bytes-like objects."""
    h = hashlib.sha256()
    for p in parts:
        h.update(np.ascontiguousarray(p).tobytes())
    return h.hexdigest()


def oracle_nvfp4_digest(wq: dict, I: int) -> str:
    rmap = w13_row_map(I)
    return nvfp4_digest((pack_codes(wq["q13"][rmap]), chunk_scales(wq["sf13"][rmap]),
                         pack_codes(wq["q2"]), chunk_scales(wq["sf2"]),
                         np.float32(wq["g13"]), np.float32(wq["g2"])))


# ---- the worker ---------------------------------------------------------------------------

def _work(task):
    import oracle
    from latent_moe_layer_rmsnorm_gb300 import synth
    kind, shape, seed, e, u_rows, arg, digest = task
    m = synth.make_expert(shape, seed, e, "cpu")
    wg, wu, wd = (m[k].float().numpy() for k in ("w_gate", "w_up", "w_down"))
    if kind == "nvfp4":
        wq = oracle.nvfp4_expert_weights(wg, wu, wd)
        r = oracle.nvfp4_expert_rows(u_rows, wq, arg)
        r.pop("s_deq", None)
        if digest:
            r["digest"] = oracle_nvfp4_digest(wq, shape.I)
    else:
        r = oracle.chain_expert(wg, wu, wd, u_rows, arg)
    return r


class ExpertMap:
    """expert_map for oracle.moe_forward: the per-expert steps of the experts drawn with
    (shape, seed) run in the pool.  digests (NVFP4) collects {expert: digest}."""

    def __init__(self, shape, seed: int, digest: bool = False):
        self.shape, self.seed, self.digest = shape, seed, digest
        self.kind = "nvfp4" if shape.expert == "nvfp4" else "chain"
        self.digests = {}

    def __call__(self, tasks):
        jobs = [(self.kind, self.shape, self.seed, int(e), u, a, self.digest and
                 int(e) not in self.digests) for e, u, a in tasks]
        it = pool().imap(_work, jobs, chunksize=1)
        # a worker that dies loses its task: give up with an error instead of waiting
        out = [it.next(timeout=TASK_TIMEOUT_S) for _ in jobs]
        for (e, _, _), r in zip(tasks, out):
            if "digest" in r:
                self.digests[int(e)] = r.pop("digest")
        return out


def gpu_nvfp4_digest(layer, e: int) -> str:
    """The same digest over expert e's slices of a LatentMoE's quantised weights."""
    s = layer.shape
    I, p = s.I, s.p
    n13, n2 = 2 * I * p, p * I

    def sl(t, a, b):
        return t[a:b].cpu().numpy()
    return nvfp4_digest((sl(layer.w13, e * n13 // 2, (e + 1) * n13 // 2),
                         sl(layer.sf13, e * n13 // 16, (e + 1) * n13 // 16),
                         sl(layer.w2, e * n2 // 2, (e + 1) * n2 // 2),
                         sl(layer.sf2, e * n2 // 16, (e + 1) * n2 // 16),
                         layer.gs13[e].cpu().numpy(), layer.gs2[e].cpu().numpy()))
