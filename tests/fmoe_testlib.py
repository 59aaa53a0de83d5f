"""Shared helpers of the GPU parity tests: pools, oracle calls, error metrics.

Inputs come only from ``synth`` (the seeded generator); expected values only
from ``oracle``.  Expert blobs for the oracle are regenerated on the CPU.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import synth

TOL = 2e-3          # max relative error allowed on outputs (fp32 accumulation)


def rel_errors(got, ref, floor=1e-3):
    """(max |g-r| / max |r|, max elementwise |g-r| / max(|r|, floor * max|r|))."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(r))) if r.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(g - r))) if r.size else 0.0, 0.0
    d = np.abs(g - r)
    primary = float(d.max() / scale)
    elem = float(np.max(d / np.maximum(np.abs(r), floor * scale)))
    return primary, elem


# Elementwise floor for a deep stack: after 48 fp32 layers every output
# element carries about the same absolute rounding error (up to ~4e-5 of the
# largest element, measured), so an element far below the largest is held to
# an absolute bound the arithmetic does not give.  For the 48-layer stack the
# elementwise form divides by at least 5e-2 of the largest element: an
# element twenty times below the largest may be off by 1e-4 of the largest.
# The max-normalised form keeps 2e-3.
STACK_FLOOR = 5e-2


def assert_close(got, ref, tol=TOL, what="", floor=1e-3):
    p, e = rel_errors(got, ref, floor)
    assert p <= tol and e <= tol, f"{what}: max rel err {p:.3e}, elementwise {e:.3e} (tol {tol})"
    return p, e


def gpu_pool(shape: synth.BlockShape, layer: int, count: int, first: int = 0, seed=None) -> torch.Tensor:
    nw = synth.blob_bytes(shape.bits, shape.hidden, shape.inter) // 4
    t = torch.empty(count * nw, dtype=torch.int32, device="cuda")
    synth.fill_pool(t, shape, layer, first, count, seed=seed)
    return t


@functools.lru_cache(maxsize=16)
def oracle_expert(shape: synth.BlockShape, layer: int, expert: int, seed=None):
    blob = synth.expert_blob(shape, layer, expert, device="cpu", seed=seed).numpy().view(np.uint8)
    return oracle.expert_weights(blob, shape.bits, shape.hidden, shape.inter)


def make_layer(fm, shape: synth.BlockShape, layer: int = 0, shared_index: int = 0, pool=None, seed=None):
    """A device Layer for `shape`: routed pool (generated unless given) and, if the
    shape has one, the shared expert n_experts + shared_index."""
    if pool is None:
        pool = gpu_pool(shape, layer, shape.n_experts, seed=seed)
    shared = wsg = None
    if shape.has_shared:
        shared = gpu_pool(shape, layer, 1, first=shape.n_experts + shared_index, seed=seed)
        wsg = synth.shared_gate_vector(shape, layer, seed).cuda()
    return fm.Layer(shape.bits, shape.hidden, shape.inter, shape.n_experts, pool, shared, wsg)


def oracle_block(shape, layer, x, logits, residual, K, shared_index=0, seed=None):
    sh = wsg = None
    if shape.has_shared:
        sh = oracle_expert(shape, layer, shape.n_experts + shared_index, seed)
        wsg = synth.shared_gate_vector(shape, layer, seed).numpy().view(np.uint16)
    return oracle.moe_block(lambda e: oracle_expert(shape, layer, e, seed),
                            np.asarray(x, dtype=np.float64), np.asarray(logits, dtype=np.float64),
                            np.asarray(residual, dtype=np.float64), K, sh, wsg)


def oracle_stack_token(shape: synth.BlockShape, h0, logits, K: int, shared: bool = False):
    """One token through shape.n_layers pre-norm blocks by the oracle (each layer
    its own routed pool; shared expert n_experts of the layer if `shared`).
    Top level so that a spawned worker process can run it."""
    h0 = np.asarray(h0, dtype=np.float64)
    logits = np.asarray(logits, dtype=np.float64)
    return oracle.stack_decode(
        lambda l, e: oracle_expert(shape, l, e), h0, logits, K, shape.eps,
        (lambda l: oracle_expert(shape, l, shape.n_experts)) if shared else None,
        (lambda l: synth.shared_gate_vector(shape, l).numpy().view(np.uint16)) if shared else None)


def _one_thread():
    import torch as _torch
    _torch.set_num_threads(1)


def oracle_pool(workers: int = 8):
    """A process pool for oracle work, started with spawn (safe after CUDA
    initialisation in the parent), each worker on one thread (numpy's BLAS and
    torch) so that the workers do not oversubscribe the host's cores."""
    import concurrent.futures
    import multiprocessing
    import os
    n = max(1, min(workers, os.cpu_count() or 1))
    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        pool = concurrent.futures.ProcessPoolExecutor(max_workers=n, mp_context=multiprocessing.get_context("spawn"),
                                                      initializer=_one_thread)
        pool.submit(int, 0).result()        # start the workers while the limits are set
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return pool
