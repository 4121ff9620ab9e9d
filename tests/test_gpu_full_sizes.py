"""The three large workloads at their full sizes.

A full-depth float64 oracle pass there costs tens to hundreds of TFLOP, so at
these sizes the checks are:
  * the first block, in the launch configuration the benchmark uses, against
    the oracle on sampled token rows (keys and values from every token);
  * the whole stack streamed through the two slots against the same stack
    with every block resident on the device, bit for bit (placement must not
    change a single output bit);
  * the device weight footprint: two slots of the largest block.
"""
import gc

import numpy as np
import pytest
import torch

import layerwise_weight_offloaded_gb300 as dlo
import synthetic
from layerwise_weight_offloaded_gb300.pinned import PinnedShards
from oracle import dit

from _workload import assert_close_rel_max, oracle_params, param_source, spec_tuple

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _build():
    from layerwise_weight_offloaded_gb300 import build
    build.build()
    torch.cuda.init()
    yield


def _forward(h, x_np, c_np):
    R, T, _ = x_np.shape
    x = torch.from_numpy(x_np).cuda()
    c = torch.from_numpy(c_np).cuda()
    dlo.dlo_forward(h, x, c, R, T, torch.cuda.current_stream())
    dlo.dlo_synchronize(h, 600000)
    out = x.cpu().numpy()
    del x, c
    return out


@pytest.mark.parametrize("name", ["deep", "video", "large"])
def test_full_size_workload(name):
    cfg = synthetic.get_config(name)
    spec = spec_tuple(cfg)
    specs = [spec] * cfg.blocks
    src = param_source(cfg.seed)
    ps = PinnedShards(specs, cfg.dp_size, src)
    x, c = synthetic.tokens(cfg.seed, cfg.requests, cfg.tokens, cfg.hidden), synthetic.cond(cfg.seed, cfg.requests,
                                                                                           cfg.cond_dim)
    try:
        # first block alone (same shapes, same kernels as every block of the stack)
        h1 = dlo.dlo_create(specs[:1], cfg.dp_size, ps.ptrs[:cfg.dp_size], dlo.DLO_FILL_AUTO)
        try:
            one = _forward(h1, x, c)
        finally:
            dlo.dlo_destroy(h1)
        p0 = oracle_params(specs[:1], src)[0]
        rows = np.array([0, 1, 127, 128, cfg.tokens // 2 + 3, cfg.tokens - 1])
        for r in sorted({0, cfg.requests - 1}):
            ref = dit.block_forward_rows(x, c, p0, cfg.heads, r, rows)
            assert_close_rel_max(one[r, rows], ref, TOL, f"{name} block 0 request {r}")
            assert_close_rel_max(one[r, rows] - x[r, rows], ref - x[r, rows], TOL, f"{name} block 0 delta")
        del p0
        gc.collect()

        # whole stack: streamed through two slots == all blocks resident
        hs = dlo.dlo_create(specs, cfg.dp_size, ps.ptrs, dlo.DLO_FILL_AUTO)
        try:
            streamed = _forward(hs, x, c)
            st = dlo.dlo_get_stats(hs)
            n = dlo.dlo_block_numel(spec)
            assert st["slot_bytes"] == dlo.dlo_shard_numel(n, cfg.dp_size) * cfg.dp_size * 2
            assert st["device_weight_high_water"] == 2 * st["slot_bytes"]
        finally:
            dlo.dlo_destroy(hs)
        torch.cuda.empty_cache()
        hr = dlo.dlo_create(specs, cfg.dp_size, ps.ptrs, dlo.DLO_FILL_MEMCPY | dlo.DLO_RESIDENT)
        try:
            resident = _forward(hr, x, c)
        finally:
            dlo.dlo_destroy(hr)
        assert np.isfinite(streamed).all()
        assert np.array_equal(streamed.view(np.uint32), resident.view(np.uint32))
        assert not np.array_equal(streamed, x)
    finally:
        del ps
        gc.collect()
        torch.cuda.empty_cache()
        if hasattr(torch._C, "_host_emptyCache"):
            torch._C._host_emptyCache()
