"""Storage model of the bf16 backward pass: the float64 gradient with rounding injected at the points
where the path stores an operand, compared with the exact float64 gradient. A diagnostic logged beside
the path's own error; the parity gates are fixed numbers against the float64 oracle.

This is a model of the path's storage, not of its code: every step is the oracle's chain rule
(float64), and each value the path holds as a tensor-core operand is rounded once to fp16 (rh): the
six weights, zh and xh, dy and dgg, dX, and the gate gradients of a and b; a and b are the bf16
values the forward stores (the oracle's storage="bf16"), which fp16 holds exactly; dz is rounded to
bf16 (rb). The path scales each of those operands by a power of two first, which leaves the relative
rounding of normal values unchanged. Float32 accumulation is taken as exact.

Run as a script to print the model's errors for the test cases: python -m tests.backward_storage_model
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads as wl

rb = oracle.round_to_bf16


def rh(v):
    """Round float64 values to the nearest fp16 value (ties to even), through numpy's float16."""
    return np.asarray(v, np.float64).astype(np.float16).astype(np.float64)


def emulated_backward(z, mask, W, direction, dout):
    W = {k: np.asarray(v, np.float64) for k, v in W.items()}
    Wb = {k: (rh(v) if k.startswith("w_") else v) for k, v in W.items()}
    m = np.asarray(mask, np.float64)
    M = np.outer(m, m)
    zh = oracle.normalise_input(z, W)
    a = oracle.gated_projection(zh, M, W["w_ga"], W["w_a"], "bf16")
    b = oracle.gated_projection(zh, M, W["w_gb"], W["w_b"], "bf16")
    x = oracle.contract(a, b, direction)
    zb = rh(zh)
    # output backward
    xh = rh(oracle.layer_norm(x, W["ln_out_gamma"], W["ln_out_beta"]))
    g = oracle.sigmoid(zb @ Wb["w_g"].T)
    y = xh @ Wb["w_o"].T
    dy = rh(dout * g)
    dgg = rh(dout * y * g * (1 - g))
    dxh = dy @ Wb["w_o"]
    dzh = dgg @ Wb["w_g"]
    dx, d_go, d_bo = oracle.layer_norm_backward(x, W["ln_out_gamma"], dxh)
    grads = {"w_g": dgg.reshape(-1, 128).T @ zb.reshape(-1, 128), "w_o": dy.reshape(-1, 128).T @ xh.reshape(-1, 128),
             "ln_out_gamma": d_go, "ln_out_beta": d_bo}
    da, db = oracle.contract_backward(rh(dx), a, b, direction)
    # projection backward, both sides
    for dV, wv, wg in ((da, "w_a", "w_ga"), (db, "w_b", "w_gb")):
        pv = zb @ Wb[wv].T
        s = oracle.sigmoid(zb @ Wb[wg].T)
        dpv = rh(dV * s * M[..., None])
        dpg = rh(dV * pv * M[..., None] * s * (1 - s))
        dzh = dzh + dpv @ Wb[wv] + dpg @ Wb[wg]
        grads[wv] = dpv.reshape(-1, 128).T @ zb.reshape(-1, 128)
        grads[wg] = dpg.reshape(-1, 128).T @ zb.reshape(-1, 128)
    dz, grads["ln_in_gamma"], grads["ln_in_beta"] = oracle.layer_norm_backward(z, W["ln_in_gamma"], dzh)
    grads["z"] = rb(dz)
    return grads


def floor(N, mask, direction, seed_z, seed_d, seed_m=12):
    """Per-gradient max|model - exact| / rms(exact) for the inputs of a GPU test case."""
    W = wl.make_weights(128, 128, 1, ln_random=True)
    z = wl.as_f64(wl.make_z(N, 128, seed_z, "bf16"))
    m = wl.make_mask(N, mask, seed_m)
    d = np.random.default_rng(seed_d).standard_normal((N, N, 128)).astype(np.float32)
    dout = wl.as_f64(wl.f32_to_bf16_bits(d))
    ex = oracle.full_backward(z, m, W, direction, dout, storage="bf16")
    em = emulated_backward(z, m, W, direction, dout)
    return {k: float(np.max(np.abs(em[k] - ex[k])) / np.sqrt(np.mean(ex[k] ** 2))) for k in ex}


if __name__ == "__main__":
    for N, mask in ((64, "scatter"), (129, "last10pct"), (200, "scatter")):
        for d in ("outgoing", "incoming"):
            f = floor(N, mask, d, 11 + N, 13 + N)
            print(N, mask, d, " ".join(f"{k}={v:.4f}" for k, v in f.items()), "max", f"{max(f.values()):.4f}")
