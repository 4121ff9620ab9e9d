"""Test helpers: seeded workloads fed identically to the oracle and the CUDA path.

The oracle side gets float64 parameters widened from the generator's bf16
bits; the CUDA side gets the same bits packed into pinned shards by the C
library.  Nothing here computes any part of the method.
"""
from __future__ import annotations

import numpy as np

import synthetic
from oracle import dit

GATE_PARAM = 1  # ada_b


def spec_tuple(cfg):
    return (cfg.hidden, cfg.heads, cfg.mlp, cfg.cond_dim)


def param_source(seed: int, transform=None):
    """(block, param, shape) -> bf16 bits from the generator (optionally transformed)."""
    def src(b, i, shape):
        bits = synthetic.weight_bits(seed, b, i, shape)
        return transform(b, i, bits) if transform else bits
    return src


def zero_gates(hidden: int):
    """Transform making every block the identity: ada_w = 0, gate entries of ada_b = 0."""
    def t(b, i, bits):
        bits = bits.copy()
        if i == 0:
            bits[:] = 0
        elif i == GATE_PARAM:
            bits[2 * hidden:3 * hidden] = 0
            bits[5 * hidden:6 * hidden] = 0
        return bits
    return t


def oracle_params(specs, src) -> list[dict]:
    out = []
    for b, (h, H, m, C) in enumerate(specs):
        p = {}
        for i, (name, shape) in enumerate(dit.param_shapes(h, m, C)):
            p[name] = dit.bf16_to_f64(src(b, i, shape)).reshape(shape)
        out.append(p)
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    return dit.bf16_to_f64(np.asarray(bits).view(np.uint16))


def assert_close_rel_max(got, ref, frac, what=""):
    """max |got - ref| <= frac * max |ref|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.max(np.abs(got - ref))
    bound = frac * np.max(np.abs(ref))
    assert err <= bound, f"{what}: max|err| = {err:.3e} > {frac} * max|ref| = {bound:.3e}"
    return err / max(np.max(np.abs(ref)), 1e-300)
