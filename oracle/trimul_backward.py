"""Float64 CPU oracle of the gradient of the triangle multiplicative update.

TEST INFRASTRUCTURE, like ``oracle.trimul``: only the tests, the package's
smoke check and the CPU baseline leg of the benchmark may import it; it shares
no code with the CUDA library.

What it computes. For a cotangent dout [N][N][c_z] of the update's output
(the gradient of a scalar loss L with respect to out), the gradient of L with
respect to z and to every weight of the layer. The forward is the standard
AlphaFold3 / Boltz Pairformer update that ``oracle.trimul`` documents; the
pages want the layer trained at larger crops (the section "A pegadinha" of
"NVIDIA BioNeMo escala modelagem biomolecular com context parallelism e quebra
barreira de memória da GPU" calls fine-tuning with larger crops essential, and
the hyper.ai (fr) story on parallélisme contextuel says the same), so its
gradient is the same function's chain rule, taken step by step in reverse:

    out = g * y,  g = sigmoid(gg),  gg = W_g zh,  y = W_o xh,  xh = LN_out(x)
        dy  = dout * g                     dgg = dout * y * g (1 - g)
        dW_o = sum_p dy xh^T               dW_g = sum_p dgg zh^T
        dxh = W_o^T dy                     dzh = W_g^T dgg  (first term)
    xh = LN_out(x): LayerNorm backward over c_h gives dx, d(gamma_out), d(beta_out)
    outgoing x_ij = sum_k a_ik b_jk :  da_ik = sum_j dx_ij b_jk,  db_jk = sum_i dx_ij a_ik
    incoming x_ij = sum_k a_ki b_kj :  da_ki = sum_j dx_ij b_kj,  db_kj = sum_i dx_ij a_ki
    a = sigmoid(ga) * pa * M,  ga = W_ga zh,  pa = W_a zh   (b alike)
        dpa = da * sigmoid(ga) * M         dga = da * pa * M * sigmoid(ga)(1 - sigmoid(ga))
        dW_a = sum_p dpa zh^T              dW_ga = sum_p dga zh^T
        dzh += W_a^T dpa + W_ga^T dga + W_b^T dpb + W_gb^T dgb
    zh = LN_in(z): LayerNorm backward over c_z gives dz, d(gamma_in), d(beta_in)

(sum_p runs over all N^2 pairs.) LayerNorm backward, for n = (v - mu) r with
r = 1/sqrt(var + eps) and out = gamma n + beta: dn = dout * gamma and
dv = r (dn - mean(dn) - n mean(dn n)), d(gamma) = sum dout n, d(beta) = sum dout.

``storage="bf16"`` rounds a and b to bf16 as the forward does and uses the
rounded values in the contraction's gradient; the rounding itself is passed
through as the identity (its derivative is zero almost everywhere, and the bf16
path stores the rounded values, so this is the gradient that path approximates).

Every floating-point step is float64. No blocking, fusion or reordering beyond
the chain rule: per-channel matrix products are numpy matmul calls.
"""
from __future__ import annotations

import numpy as np

from . import trimul as T

WEIGHT_NAMES = ("ln_in_gamma", "ln_in_beta", "w_a", "w_ga", "w_b", "w_gb", "w_g",
                "ln_out_gamma", "ln_out_beta", "w_o")


def layer_norm_backward(v, gamma, dout, eps=T.LN_EPS):
    """Gradient of LayerNorm over the last axis (biased variance, eps in the root).

    Returns (dv, dgamma, dbeta); dgamma and dbeta are summed over every leading axis.
    """
    v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    mu = v.mean(axis=-1, keepdims=True)
    d = v - mu
    r = 1.0 / np.sqrt((d * d).mean(axis=-1, keepdims=True) + eps)
    n = d * r
    dn = dout * np.asarray(gamma, np.float64)
    dv = r * (dn - dn.mean(axis=-1, keepdims=True) - n * (dn * n).mean(axis=-1, keepdims=True))
    lead = tuple(range(v.ndim - 1))
    return dv, (dout * n).sum(axis=lead), dout.sum(axis=lead)


def contract_backward(dx, a, b, direction):
    """(da, db) of the per-channel contraction for the cotangent dx of x.

    outgoing X_c = A_c B_c^T:  dA_c = dX_c B_c,    dB_c = dX_c^T A_c
    incoming X_c = A_c^T B_c:  dA_c = B_c dX_c^T,  dB_c = A_c dX_c
    """
    T._check_direction(direction)
    dX = np.moveaxis(dx, -1, 0)
    A = np.moveaxis(a, -1, 0)
    B = np.moveaxis(b, -1, 0)
    if direction == "outgoing":
        dA = np.matmul(dX, B)
        dB = np.matmul(np.swapaxes(dX, 1, 2), A)
    else:
        dA = np.matmul(B, np.swapaxes(dX, 1, 2))
        dB = np.matmul(A, dX)
    return np.moveaxis(dA, 0, -1), np.moveaxis(dB, 0, -1)


def gated_projection_backward(da, zh, pair_mask, w_gate, w_val):
    """Gradient of a = sigmoid(w_gate zh) * (w_val zh) * M for the cotangent da.

    Returns (dzh, dw_gate, dw_val).
    """
    ga = zh @ w_gate.T
    pa = zh @ w_val.T
    s = T.sigmoid(ga)
    Mc = pair_mask[..., None]
    dpa = da * s * Mc
    dga = da * pa * Mc * s * (1.0 - s)
    dzh = dpa @ w_val + dga @ w_gate
    c_z = zh.shape[-1]
    zf = zh.reshape(-1, c_z)
    return dzh, dga.reshape(-1, dga.shape[-1]).T @ zf, dpa.reshape(-1, dpa.shape[-1]).T @ zf


def output_backward(dout, x, zh, W):
    """Gradient of out = sigmoid(W_g zh) * W_o LayerNorm_out(x) for the cotangent dout.

    Returns (dx, dzh, grads) with grads holding w_g, w_o, ln_out_gamma, ln_out_beta.
    """
    gg = zh @ W["w_g"].T
    g = T.sigmoid(gg)
    xh = T.layer_norm(x, W["ln_out_gamma"], W["ln_out_beta"])
    y = xh @ W["w_o"].T
    dy = dout * g
    dgg = dout * y * g * (1.0 - g)
    dxh = dy @ W["w_o"]
    dzh = dgg @ W["w_g"]
    dx, dgamma, dbeta = layer_norm_backward(x, W["ln_out_gamma"], dxh)
    c_z, c_h = zh.shape[-1], x.shape[-1]
    grads = {"w_g": dgg.reshape(-1, c_z).T @ zh.reshape(-1, c_z),
             "w_o": dy.reshape(-1, c_z).T @ xh.reshape(-1, c_h),
             "ln_out_gamma": dgamma, "ln_out_beta": dbeta}
    return dx, dzh, grads


def full_backward(z, mask, W, direction, dout, storage="exact"):
    """Gradient of sum(dout * update(z)) with respect to z and every weight.

    Returns a dict: "z" -> dz [N][N][c_z], and one entry per weight name with its
    gradient in the weight's own shape. All float64.
    """
    T._check_direction(direction)
    W = T._w64(W)
    z = T._to_f64(z)
    dout = T._to_f64(dout)
    m = np.asarray(mask, np.float64)
    M = np.outer(m, m)
    zh = T.normalise_input(z, W)
    a = T.gated_projection(zh, M, W["w_ga"], W["w_a"], storage)
    b = T.gated_projection(zh, M, W["w_gb"], W["w_b"], storage)
    x = T.contract(a, b, direction)

    dx, dzh, grads = output_backward(dout, x, zh, W)
    da, db = contract_backward(dx, a, b, direction)
    dzh_a, grads["w_ga"], grads["w_a"] = gated_projection_backward(da, zh, M, W["w_ga"], W["w_a"])
    dzh_b, grads["w_gb"], grads["w_b"] = gated_projection_backward(db, zh, M, W["w_gb"], W["w_b"])
    dzh = dzh + dzh_a + dzh_b
    dz, grads["ln_in_gamma"], grads["ln_in_beta"] = layer_norm_backward(z, W["ln_in_gamma"], dzh)
    grads["z"] = dz
    return grads
