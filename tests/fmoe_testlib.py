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


def rel_errors(got, ref):
    """(max |g-r| / max |r|, max elementwise |g-r| / max(|r|, 1e-3 max|r|))."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(r))) if r.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(g - r))) if r.size else 0.0, 0.0
    d = np.abs(g - r)
    primary = float(d.max() / scale)
    elem = float(np.max(d / np.maximum(np.abs(r), 1e-3 * scale)))
    return primary, elem


def assert_close(got, ref, tol=TOL, what=""):
    p, e = rel_errors(got, ref)
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
