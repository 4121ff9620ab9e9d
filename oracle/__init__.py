"""CPU oracle for the layerwise weight-streaming DiT forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it, links it or falls back to it, and this package imports
nothing from the CUDA library: the two share no code.  Inputs come from the
``synthetic`` generator module, which both sides use.

Contents:
  shards.py  - flat per-block buffer, ceil-divided zero-padded shards and the
               inverse reassembly (the pages' weight-sharding technique);
  dit.py     - the DiT block stack in float64: adaLN modulation, LayerNorm +
               modulate, QKV projection, softmax attention, gated residual
               out-projection, GELU MLP with gated residual.

Parity status per function is stated in each module header.
"""
from . import shards  # noqa: F401
from . import dit  # noqa: F401
