"""Float64 CPU oracle of triangle attention (starting node and ending node).

TEST INFRASTRUCTURE, like ``oracle.trimul``: only the tests, the package's smoke check and the CPU
baseline leg of the benchmark may import it; it shares no code with the CUDA library.

What it computes. The BioIR page ("BioIR da Nvidia acelera previsão de proteínas em 2,9x com PyTorch
puro") names triangle operations and pairwise attention among the parts of the Pairformer and Evoformer
stacks that its kernels target, and gives no arithmetic. The arithmetic below is the standard
AlphaFold3 / Boltz triangle attention over the pair representation z [N][N][c_z], with H heads of
dimension c:

    zh_ij     = LayerNorm(z_ij)                                       (over c_z)
    q_ij^h, k_ij^h, v_ij^h = (W_q zh_ij)^h, (W_k zh_ij)^h, (W_v zh_ij)^h   (c each)
    b_jk^h    = (W_b zh_jk)^h                                         (one scalar per head)
    g_ij^h    = sigmoid(W_g zh_ij)^h                                  (c)
    starting node:  s_ijk^h = q_ij^h . k_ik^h / sqrt(c) + b_jk^h,  over keys k with m_i m_k = 1
                    o_ij^h  = g_ij^h * sum_k softmax_k(s_ij.^h)_k v_ik^h
    ending node:    s_ijk^h = q_ij^h . k_kj^h / sqrt(c) + b_ki^h,  over keys k with m_k m_j = 1
                    o_ij^h  = g_ij^h * sum_k softmax_k(s_ij.^h)_k v_kj^h
    out_ij    = W_o [o_ij^1, ..., o_ij^H]                             (H c -> c_z)

Readings where the pages say nothing: H = 4 heads of c = 32 (the AlphaFold3 Pairformer's triangle
attention), Linear layers without bias, LayerNorm with the biased variance and eps = 1e-5; the key mask
excludes pairs whose token mask product is 0, and a query row with no valid key (m_i = 0 for the
starting node, m_j = 0 for the ending node) has o = 0 -- the sum over an empty set -- rather than the
value a large finite negative mask bias would give, which depends on the arithmetic's precision. The
ending node is the starting node applied to the transposed grid and transposed back (the algebra above
shows the two agree).

Every floating-point step is float64; the matrix products are numpy matmul / einsum calls.
"""
from __future__ import annotations

import numpy as np

from . import trimul as T

NODES = ("starting", "ending")


def weight_shapes(c_z: int, heads: int, c: int) -> dict:
    hc = heads * c
    return {"ln_gamma": (c_z,), "ln_beta": (c_z,), "w_q": (hc, c_z), "w_k": (hc, c_z), "w_v": (hc, c_z),
            "w_b": (heads, c_z), "w_g": (hc, c_z), "w_o": (c_z, hc)}


def _check_node(node):
    if node not in NODES:
        raise ValueError(f"node must be one of {NODES}, got {node!r}")


def attention_rows(q, k, v, bias, key_valid):
    """Per row i and head h: softmax_k(q_j . k_k / sqrt(c) + bias_jk) over valid keys, applied to v.

    q, k, v [N][N][H][c] (row i, position, head, channel); bias [H][N][N] (j, k); key_valid [N][N] (i, k)
    booleans. A row without any valid key gives 0. Returns o [N][N][H][c] before the gate.
    """
    c = q.shape[-1]
    s = np.einsum("ijhc,ikhc->ihjk", q, k, optimize=True) / np.sqrt(c) + bias[None, :, :, :]
    valid = key_valid[:, None, None, :]                       # [i][1][1][k]
    s = np.where(valid, s, -np.inf)
    smax = np.max(s, axis=-1, keepdims=True)
    smax = np.where(np.isfinite(smax), smax, 0.0)
    e = np.where(valid, np.exp(s - smax), 0.0)
    den = e.sum(axis=-1, keepdims=True)
    a = np.where(den > 0, e / np.where(den > 0, den, 1.0), 0.0)
    return np.einsum("ihjk,ikhc->ijhc", a, v, optimize=True)


def starting_node(z, mask, W, heads=4, c=32):
    """Triangle attention around the starting node over z [N][N][c_z]; returns float64 [N][N][c_z]."""
    W = T._w64(W)
    z = T._to_f64(z)
    N = z.shape[0]
    m = np.asarray(mask, np.float64)
    zh = T.layer_norm(z, W["ln_gamma"], W["ln_beta"])
    q = (zh @ W["w_q"].T).reshape(N, N, heads, c)
    k = (zh @ W["w_k"].T).reshape(N, N, heads, c)
    v = (zh @ W["w_v"].T).reshape(N, N, heads, c)
    b = np.moveaxis(zh @ W["w_b"].T, -1, 0)                  # [H][j][k] from zh_jk
    g = T.sigmoid(zh @ W["w_g"].T).reshape(N, N, heads, c)
    key_valid = np.outer(m, m) != 0                          # (i, k)
    o = g * attention_rows(q, k, v, b, key_valid)
    return o.reshape(N, N, heads * c) @ W["w_o"].T


def full(z, mask, W, node, heads=4, c=32):
    """Triangle attention of the given node over the whole grid."""
    _check_node(node)
    if node == "starting":
        return starting_node(z, mask, W, heads, c)
    zt = np.swapaxes(T._to_f64(z), 0, 1)
    return np.swapaxes(starting_node(zt, mask, W, heads, c), 0, 1)


def flops(N: int, c_z: int = 128, heads: int = 4, c: int = 32) -> float:
    """Algorithmic FLOPs of one triangle attention: the two per-row attention products (4 N^3 H c) and
    the per-pair projections q, k, v, g, b and the output (2 c_z (4 H c + H) + 2 H c c_z per pair)."""
    hc = heads * c
    return 4.0 * N ** 3 * hc + float(N) ** 2 * (2 * c_z * (4 * hc + heads) + 2 * hc * c_z)


def pair_bias(z, W, heads=4, chunk=32):
    """b[h][j][k] = (W_b LayerNorm(z_jk))^h for every pair, computed in row chunks (float64)."""
    W = T._w64(W)
    N = z.shape[0]
    b = np.empty((heads, N, N))
    for j0 in range(0, N, chunk):
        zh = T.layer_norm(T._to_f64(z[j0:j0 + chunk]), W["ln_gamma"], W["ln_beta"])
        b[:, j0:j0 + chunk, :] = np.moveaxis(zh @ W["w_b"].T, -1, 0)
    return b


def sampled(z, mask, W, node, lines, heads=4, c=32, bias=None):
    """Whole lines of the output, exactly: out[i, :, :] for i in ``lines`` (starting node) or
    out[:, j, :] for j in ``lines`` (ending node), returned as [len(lines)][N][c_z].

    A starting-node row i needs z[i, :] (its q, k, v, g) and the pair bias of every pair (j, k); the
    ending node is the starting node of the transposed grid. ``bias`` may pass in pair_bias of the
    (transposed, for the ending node) grid to share it between calls. ``z`` may be float32 or uint16
    bf16 bits, indexable like [N][N][c_z].
    """
    _check_node(node)
    W = T._w64(W)
    m = np.asarray(mask, np.float64)
    N = z.shape[0]
    lines = np.asarray(lines, np.int64)
    if bias is None:
        bias = pair_bias(z if node == "starting" else np.swapaxes(z, 0, 1), W, heads)
    out = np.empty((len(lines), N, W["w_o"].shape[0]))
    for n, i in enumerate(lines):
        zi = T._to_f64(z[i, :, :] if node == "starting" else z[:, i, :])      # [N][c_z]: pairs (i, .)
        zh = T.layer_norm(zi, W["ln_gamma"], W["ln_beta"])
        q = (zh @ W["w_q"].T).reshape(1, N, heads, c)
        k = (zh @ W["w_k"].T).reshape(1, N, heads, c)
        v = (zh @ W["w_v"].T).reshape(1, N, heads, c)
        g = T.sigmoid(zh @ W["w_g"].T).reshape(1, N, heads, c)
        key_valid = (m[i] * m != 0)[None, :]
        o = g * attention_rows(q, k, v, bias, key_valid)
        out[n] = o.reshape(N, heads * c) @ W["w_o"].T
    return out
