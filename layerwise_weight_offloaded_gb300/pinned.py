"""Page-locked host shards for dlo_create.

Section 2 of "vLLM-Omni 发布 Distributed Layerwise Offload…" keeps every block
as dp_size equal, zero-padded flat shards in pinned host memory.  This helper
allocates those shards (torch's page-locked allocator, which maps them into
the device address space) and fills them with ``dlo_pack_block`` from the C
library; the packing itself runs in C++.  The caller supplies the parameter
bits through ``param_source``.
"""
from __future__ import annotations

from typing import Callable, Sequence

import numpy as np

from . import _binding as B


def param_shapes(spec) -> list[tuple[int, ...]]:
    s = B._spec(spec)
    h, m, C = s.hidden, s.mlp_hidden, s.cond_dim
    return [(6 * h, C), (6 * h,), (3 * h, h), (3 * h,), (h, h), (h,), (m, h), (m,), (h, m), (h,)]


class PinnedShards:
    """dp_size pinned bf16 shards per block, packed by dlo_pack_block.

    param_source(block, param_index, shape) -> contiguous uint16 numpy array
    (the parameter's bf16 bits).  With ``contiguous=True`` the shards of one
    block share one allocation back to back (the runtime then rebuilds the
    block with one copy); otherwise every shard is its own allocation, as on
    dp_size separate ranks.
    """

    def __init__(self, specs: Sequence, dp_size: int,
                 param_source: Callable[[int, int, tuple], np.ndarray], contiguous: bool = False,
                 pin: bool = True):
        """pin=False allocates ordinary host memory instead (the copy-engine fill
        still streams it; zero-copy needs device-addressable memory)."""
        import torch

        self.specs = [B._spec(s) for s in specs]
        self.dp = dp_size
        self.shards: list[list] = []  # [block][rank] torch int16 pinned tensors
        self._keep = []
        for b, sp in enumerate(self.specs):
            n = B.dlo_block_numel(sp)
            S = B.dlo_shard_numel(n, dp_size)
            if contiguous:
                buf = torch.empty(S * dp_size, dtype=torch.int16, pin_memory=pin)
                self._keep.append(buf)
                shards = [buf[r * S:(r + 1) * S] for r in range(dp_size)]
            else:
                shards = [torch.empty(S, dtype=torch.int16, pin_memory=pin) for _ in range(dp_size)]
            params = [np.ascontiguousarray(param_source(b, i, shape), dtype=np.uint16).reshape(-1)
                      for i, shape in enumerate(param_shapes(sp))]
            for p, shape in zip(params, param_shapes(sp)):
                if p.size != int(np.prod(shape)):
                    raise ValueError(f"param source returned {p.size} elements for shape {shape}")
            B.dlo_pack_block(sp, params, dp_size, shards)
            self.shards.append(shards)

    @property
    def ptrs(self) -> list[int]:
        return [s.data_ptr() for blk in self.shards for s in blk]

    def shard_numpy(self, block: int, rank: int) -> np.ndarray:
        return self.shards[block][rank].numpy().view(np.uint16)

    def nbytes(self) -> int:
        return sum(s.numel() * 2 for blk in self.shards for s in blk)


def block_flat_offsets(specs: Sequence) -> list[int]:
    """Element offset of each block's flat buffer inside a flat weight file
    holding the blocks back to back (block b's buffer is its parameters in
    the DLO_P_* order, as dlo_param_table lays them out)."""
    offs, at = [], 0
    for sp in specs:
        offs.append(at)
        at += B.dlo_block_numel(B._spec(sp))
    return offs


def pack_from_flat_file(path: str, specs: Sequence, dp_size: int, contiguous: bool = False,
                        pin: bool = True) -> "PinnedShards":
    """Pinned shards packed straight from a memory-mapped flat bf16 weight file.

    Section 1 of "vLLM-Omni 发布 Distributed Layerwise Offload…" builds the
    model on the meta device and loads weights through mmap, so the process
    never holds a private copy of the full checkpoint; section 2 then keeps
    only each rank's shard pinned.  Here the file holds every block's flat
    buffer back to back (block_flat_offsets); each block is packed from the
    mapped pages into its pinned shards and the mapping is dropped before
    returning.  The returned object carries ``mapped_bytes`` and
    ``rss_high_water_kb`` (the process's peak resident set after packing).
    """
    import resource

    specs = [B._spec(s) for s in specs]
    offs = block_flat_offsets(specs)
    total = offs[-1] + B.dlo_block_numel(specs[-1]) if specs else 0
    flat = np.memmap(path, dtype=np.uint16, mode="r")
    try:
        if flat.size < total:
            raise ValueError(f"{path}: {flat.size} bf16 elements, the blocks need {total}")

        def source(b, i, shape):
            p_off, p_num = B.dlo_param_table(specs[b])
            start = offs[b] + p_off[i]
            return flat[start:start + p_num[i]]

        ps = PinnedShards(specs, dp_size, source, contiguous=contiguous, pin=pin)
    finally:
        mapped = flat.size * 2
        del flat  # unmaps the file
    ps.mapped_bytes = mapped
    ps.rss_high_water_kb = resource.getrusage(resource.RUSAGE_SELF).ru_maxrss
    return ps
