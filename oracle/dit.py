"""Oracle: the DiT block stack in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages ("vLLM-Omni 发布 Distributed Layerwise Offload…", sections 2-3)
stream whole DiT blocks but never write down a block's arithmetic: streaming
changes where the weights sit, never the math (the "validation" section and
the B300 results section report byte-identical outputs across placement
strategies).  The block below is therefore the plainest adaLN-zero DiT block
the workload definitions name (adaLN-zero modulation from a 256-d
conditioning vector, multi-head attention, GELU MLP), with these readings:

  params, in this order, row-major, [out, in] like a linear layer:
    ada_w[6h, C], ada_b[6h], qkv_w[3h, h], qkv_b[3h], proj_w[h, h], proj_b[h],
    fc1_w[m, h], fc1_b[m], fc2_w[h, m], fc2_b[h]
  mod = ada_w . SiLU(c) + ada_b, split into shift1, scale1, gate1,
        shift2, scale2, gate2 (each h wide, in that order)
  u1  = LN(x) * (1 + scale1) + shift1          LN: no affine, eps 1e-6,
                                               population variance
  q,k,v = columns [0,h), [h,2h), [2h,3h) of u1 . qkv_w^T + qkv_b;
        head j uses columns [j*d, (j+1)*d) of each
  o   = softmax(q k^T / sqrt(d)) v  per request and head, no mask
  x1  = x + gate1 * (o . proj_w^T + proj_b)
  u2  = LN(x1) * (1 + scale2) + shift2
  g   = GELU_tanh(u2 . fc1_w^T + fc1_b)
  x2  = x1 + gate2 * (g . fc2_w^T + fc2_b)

Everything is float64; the bf16 weight bits widen exactly; no intermediate
is rounded to bf16.  Requests never see each other.

Parity: the pages fix none of the block math, so beyond the pins below the
block math is parity UNPINNED by the pages (it rests on the workload text and
the readings above).  Pins (tests/test_oracle_pins.py): LayerNorm and GELU
against torch's library routines, attention against torch's
scaled_dot_product_attention, closed-form special cases (zero gates give the
identity, a single token gives softmax weight 1, constant rows give LN = 0,
zero q/k rows give the mean of v), and a whole block against a block
assembled from torch.nn library modules.
"""
from __future__ import annotations

import numpy as np

PARAM_NAMES = ("ada_w", "ada_b", "qkv_w", "qkv_b", "proj_w", "proj_b",
               "fc1_w", "fc1_b", "fc2_w", "fc2_b")
LN_EPS = 1e-6


def param_shapes(hidden: int, mlp: int, cond_dim: int) -> list[tuple[str, tuple[int, ...]]]:
    h, m, C = hidden, mlp, cond_dim
    return [("ada_w", (6 * h, C)), ("ada_b", (6 * h,)),
            ("qkv_w", (3 * h, h)), ("qkv_b", (3 * h,)),
            ("proj_w", (h, h)), ("proj_b", (h,)),
            ("fc1_w", (m, h)), ("fc1_b", (m,)),
            ("fc2_w", (h, m)), ("fc2_b", (h,))]


def param_table(hidden: int, mlp: int, cond_dim: int) -> list[tuple[str, int, tuple[int, ...]]]:
    """(name, flat offset, shape) for every parameter of one block."""
    out, off = [], 0
    for name, shape in param_shapes(hidden, mlp, cond_dim):
        out.append((name, off, shape))
        off += int(np.prod(shape))
    return out


def block_numel(hidden: int, mlp: int, cond_dim: int) -> int:
    return sum(int(np.prod(s)) for _, s in param_shapes(hidden, mlp, cond_dim))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def params_from_flat(flat_bits: np.ndarray, hidden: int, mlp: int, cond_dim: int) -> dict[str, np.ndarray]:
    """float64 parameters viewed out of one block's flat bf16 buffer."""
    flat = bf16_to_f64(flat_bits)
    return {name: flat[off: off + int(np.prod(shape))].reshape(shape)
            for name, off, shape in param_table(hidden, mlp, cond_dim)}


def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def adaln_modulation(ada_w: np.ndarray, ada_b: np.ndarray, c: np.ndarray) -> np.ndarray:
    """mod[R, 6h] = SiLU(c) . ada_w^T + ada_b."""
    return silu(np.asarray(c, np.float64)) @ np.asarray(ada_w, np.float64).T + ada_b


def split_modulation(mod: np.ndarray, hidden: int):
    """(shift1, scale1, gate1, shift2, scale2, gate2), each [R, h]."""
    return tuple(mod[:, i * hidden:(i + 1) * hidden] for i in range(6))


def layer_norm(x: np.ndarray) -> np.ndarray:
    """Row LayerNorm without affine: (x - mean) / sqrt(var + eps), population var."""
    x = np.asarray(x, np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + LN_EPS)


def modulate(xn: np.ndarray, shift: np.ndarray, scale: np.ndarray) -> np.ndarray:
    return xn * (1.0 + scale) + shift


def linear(u: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """u . w^T + b with w stored [out, in]."""
    return np.asarray(u, np.float64) @ np.asarray(w, np.float64).T + b


def gelu_tanh(v: np.ndarray) -> np.ndarray:
    """0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))."""
    return 0.5 * v * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (v + 0.044715 * v ** 3)))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, heads: int) -> np.ndarray:
    """Non-causal softmax attention of one request, all heads.

    q: [Tq, h] (only the query rows wanted), k, v: [T, h].  Head j uses
    columns [j*d, (j+1)*d).  Each row is a two-pass softmax over all T keys:
    logits s = q k^T / sqrt(d), weights exp(s - max s) / sum, output weights . v.
    Query rows are independent, so they are processed in slices of at most
    2048 to bound memory; every output value is computed the same way.
    """
    Tq, h = q.shape
    d = h // heads
    scale = 1.0 / np.sqrt(d)
    out = np.empty((Tq, h), np.float64)
    for j in range(heads):
        cols = slice(j * d, (j + 1) * d)
        kj, vj = k[:, cols], v[:, cols]
        for r0 in range(0, Tq, 2048):
            qj = q[r0:r0 + 2048, cols]
            s = (qj @ kj.T) * scale
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            out[r0:r0 + 2048, cols] = (p @ vj) / p.sum(axis=1, keepdims=True)
    return out


def block_forward(x: np.ndarray, c: np.ndarray, p: dict[str, np.ndarray], heads: int) -> np.ndarray:
    """One DiT block over R requests: x [R, T, h], c [R, C] -> new x [R, T, h]."""
    x = np.asarray(x, np.float64)
    R, T, h = x.shape
    sh1, sc1, g1, sh2, sc2, g2 = split_modulation(adaln_modulation(p["ada_w"], p["ada_b"], c), h)
    out = np.empty_like(x)
    for r in range(R):
        u1 = modulate(layer_norm(x[r]), sh1[r], sc1[r])
        qkv = linear(u1, p["qkv_w"], p["qkv_b"])
        o = attention(qkv[:, :h], qkv[:, h:2 * h], qkv[:, 2 * h:], heads)
        x1 = x[r] + g1[r] * linear(o, p["proj_w"], p["proj_b"])
        u2 = modulate(layer_norm(x1), sh2[r], sc2[r])
        g = gelu_tanh(linear(u2, p["fc1_w"], p["fc1_b"]))
        out[r] = x1 + g2[r] * linear(g, p["fc2_w"], p["fc2_b"])
    return out


def block_forward_rows(x: np.ndarray, c: np.ndarray, p: dict[str, np.ndarray], heads: int,
                       request: int, rows: np.ndarray) -> np.ndarray:
    """The same block, evaluated only at token rows `rows` of one request.

    Keys and values need every token of the request; queries, the
    out-projection and the MLP are taken at the wanted rows only.  Returns
    [len(rows), h], equal to block_forward(...)[request, rows].
    """
    x = np.asarray(x, np.float64)
    R, T, h = x.shape
    sh1, sc1, g1, sh2, sc2, g2 = split_modulation(adaln_modulation(p["ada_w"], p["ada_b"], c), h)
    r = request
    u1 = modulate(layer_norm(x[r]), sh1[r], sc1[r])
    w, b = p["qkv_w"], p["qkv_b"]
    k = linear(u1, w[h:2 * h], b[h:2 * h])
    v = linear(u1, w[2 * h:], b[2 * h:])
    q = linear(u1[rows], w[:h], b[:h])
    o = attention(q, k, v, heads)
    x1 = x[r, rows] + g1[r] * linear(o, p["proj_w"], p["proj_b"])
    u2 = modulate(layer_norm(x1), sh2[r], sc2[r])
    g = gelu_tanh(linear(u2, p["fc1_w"], p["fc1_b"]))
    return x1 + g2[r] * linear(g, p["fc2_w"], p["fc2_b"])


def forward(x: np.ndarray, c: np.ndarray, blocks: list[dict[str, np.ndarray]], heads: int) -> np.ndarray:
    """The block stack: blocks applied in order, each reading the previous output."""
    y = np.asarray(x, np.float64)
    for p in blocks:
        y = block_forward(y, c, p, heads)
    return y
