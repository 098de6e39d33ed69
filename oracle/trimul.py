"""Float64 CPU oracle of the triangle multiplicative update.

TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the CPU
baseline leg of the benchmark may import this module. It shares no code with
the CUDA library and never imports it; the two meet only through the seeded
inputs of ``workloads``.

What it computes. The pages name this layer -- ``TriangleMultiplicationOutgoing``
with an ``Outgoing`` direction selector in the code-sample section
("Exemplo de código: triangle multiplication CP-aware") of "NVIDIA BioNeMo
escala modelagem biomolecular com context parallelism e quebra barreira de
memória da GPU", and "the triangle-multiplication module" that the hyper.ai (fr)
story on BioNeMo's parallélisme contextuel says was adapted -- but never write
out its arithmetic. The arithmetic below is the standard AlphaFold3 / Boltz
Pairformer definition of the update over the pair representation z [N][N][c_z]
(the N x N grid of pair vectors of the "2D tiling da pair representation"
section of the same page):

    zh_ij = LayerNorm_in(z_ij)                              (over c_z)
    M_ik  = m_i m_k                                         (token mask -> pair mask)
    a_ik  = sigmoid(W_ga zh_ik) * (W_a zh_ik) * M_ik        (c_h channels)
    b_ik  = sigmoid(W_gb zh_ik) * (W_b zh_ik) * M_ik
    outgoing: x_ij = sum_k a_ik * b_jk
    incoming: x_ij = sum_k a_ki * b_kj
    out_ij = sigmoid(W_g zh_ij) * W_o LayerNorm_out(x_ij)   (LayerNorm over c_h)

Readings taken where the definition is silent: LayerNorm uses the biased
variance and eps = 1e-5 with its own affine gamma/beta; there are no Linear
biases; the gate W_g reads the normalised zh; the mask is a token mask applied
to a and b at their own pair index as M_ik = m_i m_k.

Storage. ``storage="bf16"`` rounds a and b to bf16 (round-to-nearest-even)
after they are computed in float64, because the bf16 path of the update stores
its a and b intermediates in bf16; everything else stays float64.

Every floating-point step is float64. No blocking, fusion or reordering beyond
the definition: per-channel matrix products are numpy matmul calls.
"""
from __future__ import annotations

import numpy as np

LN_EPS = 1e-5
DIRECTIONS = ("outgoing", "incoming")


def sigmoid(v):
    """Logistic function 1 / (1 + exp(-v)), float64, without overflow warnings."""
    v = np.asarray(v, np.float64)
    e = np.exp(-np.abs(v))                   # in (0, 1]: never overflows
    return np.where(v >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def layer_norm(v, gamma, beta, eps=LN_EPS):
    """LayerNorm over the last axis: biased variance, eps inside the square root."""
    v = np.asarray(v, np.float64)
    mu = v.mean(axis=-1, keepdims=True)
    d = v - mu
    var = (d * d).mean(axis=-1, keepdims=True)
    return d / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def round_to_bf16(v):
    """Round float64 values to the nearest bf16 value (8 significant bits), ties to even.

    Normal-range values only (|v| >= 2**-126); zero maps to zero.
    """
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)                       # v = m * 2**e with 0.5 <= |m| < 1
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)   # np.round: half to even


def _w64(W):
    return {k: np.asarray(v, np.float64) for k, v in W.items()}


def _check_direction(direction):
    if direction not in DIRECTIONS:
        raise ValueError(f"direction must be one of {DIRECTIONS}, got {direction!r}")


# --------------------------------------------------------------------------- steps

def normalise_input(z, W):
    """zh = LayerNorm_in(z) over c_z."""
    return layer_norm(z, W["ln_in_gamma"], W["ln_in_beta"])


def gated_projection(zh, pair_mask, w_gate, w_val, storage="exact"):
    """sigmoid(w_gate zh) * (w_val zh) * pair_mask, optionally stored as bf16."""
    v = sigmoid(zh @ w_gate.T) * (zh @ w_val.T) * pair_mask[..., None]
    return round_to_bf16(v) if storage == "bf16" else v


def contract(a, b, direction):
    """Per-channel contraction. outgoing: x_ij = sum_k a_ik b_jk; incoming: x_ij = sum_k a_ki b_kj.

    a, b are [N][N][c]; the sum runs over the shared token k for each channel.
    """
    _check_direction(direction)
    A = np.moveaxis(a, -1, 0)                # [c][N][N]
    B = np.moveaxis(b, -1, 0)
    if direction == "outgoing":
        X = np.matmul(A, np.swapaxes(B, 1, 2))   # X_c = A_c B_c^T
    else:
        X = np.matmul(np.swapaxes(A, 1, 2), B)   # X_c = A_c^T B_c
    return np.moveaxis(X, 0, -1)


def output(x, zh, W):
    """out = sigmoid(W_g zh) * W_o LayerNorm_out(x)."""
    g = sigmoid(zh @ W["w_g"].T)
    y = layer_norm(x, W["ln_out_gamma"], W["ln_out_beta"]) @ W["w_o"].T
    return g * y


# --------------------------------------------------------------------------- whole update

def full(z, mask, W, direction, storage="exact"):
    """The update over the whole N x N grid. z [N][N][c_z] float64-convertible, mask [N]."""
    _check_direction(direction)
    W = _w64(W)
    z = _to_f64(z)
    m = np.asarray(mask, np.float64)
    M = np.outer(m, m)
    zh = normalise_input(z, W)
    a = gated_projection(zh, M, W["w_ga"], W["w_a"], storage)
    b = gated_projection(zh, M, W["w_gb"], W["w_b"], storage)
    x = contract(a, b, direction)
    return output(x, zh, W)


def intermediates(z, mask, W, direction, storage="exact"):
    """(zh, a, b, x) of the update, for checking single steps."""
    W = _w64(W)
    z = _to_f64(z)
    m = np.asarray(mask, np.float64)
    M = np.outer(m, m)
    zh = normalise_input(z, W)
    a = gated_projection(zh, M, W["w_ga"], W["w_a"], storage)
    b = gated_projection(zh, M, W["w_gb"], W["w_b"], storage)
    return zh, a, b, contract(a, b, direction)


def sampled(z, mask, W, direction, rows, cols, storage="exact"):
    """out[i, j, :] for every i in ``rows`` and j in ``cols`` (the product grid), exactly.

    Recomputes only what those entries depend on. Outgoing needs the a rows
    a[i, :, :] and b rows b[j, :, :]; incoming needs the a columns a[:, i, :]
    and b columns b[:, j, :]. ``z`` may be any array indexable like [N][N][c]
    (float32 values or uint16 bf16 bits are converted per slice by ``to_f64``).
    Returns float64 [len(rows)][len(cols)][c_z].
    """
    _check_direction(direction)
    W = _w64(W)
    rows = np.asarray(rows, np.int64)
    cols = np.asarray(cols, np.int64)
    m = np.asarray(mask, np.float64)
    to64 = _to_f64

    if direction == "outgoing":
        z_a = to64(z[rows, :, :])            # pairs (i, k), i in rows
        z_b = to64(z[cols, :, :])            # pairs (j, k), j in cols
        M_a = np.outer(m[rows], m)
        M_b = np.outer(m[cols], m)
    else:
        z_a = to64(z[:, rows, :])            # pairs (k, i), i in rows
        z_b = to64(z[:, cols, :])            # pairs (k, j), j in cols
        M_a = np.outer(m, m[rows])
        M_b = np.outer(m, m[cols])

    a = gated_projection(normalise_input(z_a, W), M_a, W["w_ga"], W["w_a"], storage)
    b = gated_projection(normalise_input(z_b, W), M_b, W["w_gb"], W["w_b"], storage)

    A = np.moveaxis(a, -1, 0)
    B = np.moveaxis(b, -1, 0)
    if direction == "outgoing":
        X = np.matmul(A, np.swapaxes(B, 1, 2))   # [c][rows][cols], sum over k (axis 2)
    else:
        X = np.matmul(np.swapaxes(A, 1, 2), B)   # sum over k (axis 1)
    x = np.moveaxis(X, 0, -1)

    zh_ij = normalise_input(to64(z[np.ix_(rows, cols)]), W)
    return output(x, zh_ij, W)


def _to_f64(arr):
    arr = np.asarray(arr)
    if arr.dtype == np.uint16:               # bf16 bit patterns
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


# --------------------------------------------------------------------------- comparison metrics

def half_ulp_bf16(v):
    """Half the spacing of bf16 values at |v| (the largest round-to-nearest error there)."""
    v = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(np.where(v == 0, 1.0, v))
    return np.where(v == 0, 0.0, np.ldexp(1.0, e - 9))


def errors(got, ref, out_storage=None):
    """Parity metrics of ``got`` against float64 ``ref`` (same shape).

    max_rel  = max|got - ref| / rms(ref)
    rms_rel  = rms(got - ref) / rms(ref)
    excess   = max(|got - ref| - half_ulp(ref), 0) / rms(ref) when the result is
               stored as bf16 (the error beyond the output's own rounding),
               else equal to max_rel.
    """
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    rms = rms if rms > 0 else 1.0
    out = {"max_rel": float(d.max() / rms) if d.size else 0.0,
           "rms_rel": float(np.sqrt(np.mean(d * d)) / rms) if d.size else 0.0,
           "rms_ref": rms}
    if out_storage == "bf16":
        ex = np.maximum(d - half_ulp_bf16(ref), 0.0)
        out["excess"] = float(ex.max() / rms) if ex.size else 0.0
    else:
        out["excess"] = out["max_rel"]
    return out
