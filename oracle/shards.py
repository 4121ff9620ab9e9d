"""Oracle: per-block flat weight buffer and its dp_size host shards.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "vLLM-Omni 发布 Distributed Layerwise Offload，支持 200B+ DiT 模型多卡部署"
(aisignalhub.me write-up), section 2 "weight sharding with AllGather
reconstruction", and section 3 "double-buffered prefetch" (parameters are
re-pointed to slices of the gathered buffer using cached metadata).

What the pages fix, restated:
  * every rank keeps 1/dp_size of the weights; the shard length is the
    block's element count divided by dp_size, rounded UP, so all shards have
    the same length (the collective that rebuilds the layer needs that);
  * shards are zero-filled first and rank r receives the part of the flat
    buffer that falls in [r*S, (r+1)*S); whatever lies past the end of the
    flat buffer stays zero;
  * the gather concatenates the shards in rank order; the parameters are
    then views of that concatenation at cached offsets.

Reading taken where the pages are open: the unit that is flattened and
sharded is one DiT block (one flat buffer per block, all its parameters
concatenated in a fixed order, each flattened row-major).

Parity pins: exact invariants (tests/test_oracle_pins.py) - truncated
concatenation reproduces the buffer, padding is zero, shard lengths are equal,
dp*S - n < dp, brute force over all n <= 40 and dp <= 9, and the pages'
worked per-rank sizes (tests/golden/shard_sizes.txt).
"""
from __future__ import annotations

import numpy as np


def shard_numel(numel: int, dp_size: int) -> int:
    """Equal shard length: numel / dp_size rounded up (section 2)."""
    if dp_size < 1 or numel < 0:
        raise ValueError("dp_size must be >= 1 and numel >= 0")
    q, r = divmod(numel, dp_size)
    return q + (1 if r else 0)


def pack(flat: np.ndarray, dp_size: int) -> list[np.ndarray]:
    """Split one block's flat buffer into dp_size zero-padded equal shards.

    Rank r's shard holds flat[r*S + i] for every i with r*S + i < numel and
    zero elsewhere (section 2: zero-filled shard, copy of the in-range part).
    Works elementwise on the raw bits, so any dtype is copied bit-exactly.
    """
    flat = np.ascontiguousarray(flat).reshape(-1)
    n = flat.size
    S = shard_numel(n, dp_size)
    out = []
    for r in range(dp_size):
        shard = np.zeros(S, dtype=flat.dtype)
        lo = min(r * S, n)
        hi = min((r + 1) * S, n)
        shard[: hi - lo] = flat[lo:hi]
        out.append(shard)
    return out


def gather(shards: list[np.ndarray]) -> np.ndarray:
    """Rank-ordered concatenation of the shards (what the AllGather returns)."""
    return np.concatenate([np.asarray(s).reshape(-1) for s in shards])


def unpack(shards: list[np.ndarray], numel: int) -> np.ndarray:
    """The gathered buffer truncated to the block's real element count."""
    return gather(shards)[:numel]


def views(gathered: np.ndarray, table: list[tuple[str, int, tuple[int, ...]]]) -> dict[str, np.ndarray]:
    """Re-point parameters into the gathered buffer from (name, offset, shape)."""
    out = {}
    for name, off, shape in table:
        n = int(np.prod(shape))
        out[name] = gathered[off: off + n].reshape(shape)
    return out
