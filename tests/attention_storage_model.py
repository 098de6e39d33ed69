"""Storage model of the triangle attention path: the oracle's arithmetic with rounding at the values
the path stores, against the exact float64 result. A diagnostic that the GPU tests log beside the
path's own error; the parity gates themselves are fixed numbers against the float64 oracle.

A model of the path's storage, not of its code: zh (the operand of the projections), the weights
W_q, W_k, W_v, W_g, W_o, the stored q (times log2(e)/sqrt(c)), k, v, g and pair bias b (times
log2(e): the path's softmax runs in base 2), the softmax numerator's weights P (an operand of the
P V product, whose extra column of ones also gives the denominator, so both sum the rounded weights)
and the gated output o are each rounded once to fp16 (rh), and the result to bf16 (rb); everything
else is exact. The weight images are scaled by powers of two before their rounding, which leaves the
relative rounding of every normal value unchanged.

Run as a script to print the model's error for the test cases: python -m tests.attention_storage_model
"""
from __future__ import annotations

import math

import numpy as np

import oracle
import oracle.triangle_attention as TA
import workloads as wl

rb = oracle.round_to_bf16


def rh(v):
    """Round float64 values to the nearest fp16 value (ties to even), through numpy's float16."""
    return np.asarray(v, np.float64).astype(np.float16).astype(np.float64)


def emulated(z, mask, W, node, heads=4, c=32):
    if node == "ending":
        return np.swapaxes(emulated(np.swapaxes(z, 0, 1), mask, W, "starting", heads, c), 0, 1)
    W = {k: np.asarray(v, np.float64) for k, v in W.items()}
    N = z.shape[0]
    m = np.asarray(mask, np.float64)
    zh = oracle.layer_norm(z, W["ln_gamma"], W["ln_beta"])
    zb = rh(zh)
    log2e = 1.0 / math.log(2.0)
    q = rh((zb @ rh(W["w_q"]).T) * (log2e / math.sqrt(c))).reshape(N, N, heads, c)
    k = rh(zb @ rh(W["w_k"]).T).reshape(N, N, heads, c)
    v = rh(zb @ rh(W["w_v"]).T).reshape(N, N, heads, c)
    g = rh(oracle.sigmoid(zb @ rh(W["w_g"]).T)).reshape(N, N, heads, c)
    b = rh(np.moveaxis(zh @ W["w_b"].T, -1, 0) * log2e)
    s = np.einsum("ijhc,ikhc->ihjk", q, k) + b[None]            # logits in base 2
    valid = (np.outer(m, m) != 0)[:, None, None, :]
    s = np.where(valid, s, -np.inf)
    smax = np.max(s, axis=-1, keepdims=True)
    smax = np.where(np.isfinite(smax), smax, 0.0)
    e = rh(np.where(valid, np.exp2(s - smax), 0.0))
    den = e.sum(axis=-1, keepdims=True)
    num = np.einsum("ihjk,ikhc->ijhc", e, v)
    den = np.moveaxis(den, 1, 2)                               # [i][j][h][1]
    o = rh(g * np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0))
    return rb(o.reshape(N, N, heads * c) @ rh(W["w_o"]).T)


def attention_weights(seed=1):
    """The weights of the GPU tests: N(0, 1/fan_in), random LayerNorm affine."""
    rng = np.random.default_rng(seed)
    W = {k: (rng.standard_normal(s) / math.sqrt(s[-1])).astype(np.float32)
         for k, s in TA.weight_shapes(128, 4, 32).items()}
    W["ln_gamma"] = (1.0 + 0.3 * rng.standard_normal(128)).astype(np.float32)
    W["ln_beta"] = (0.3 * rng.standard_normal(128)).astype(np.float32)
    return W


def floor(N, mask, node, seed_z, seed_m=12, rms=False):
    """max|model - exact| / rms(exact) for the inputs of a GPU test case (with rms=True, also
    rms(model - exact) / rms(exact))."""
    W = attention_weights()
    z = wl.as_f64(wl.make_z(N, 128, seed_z, "bf16"))
    m = wl.make_mask(N, mask, seed_m)
    ex = TA.full(z, m, W, node)
    em = emulated(z, m, W, node)
    r = np.sqrt(np.mean(ex ** 2))
    mx = float(np.max(np.abs(em - ex)) / r)
    return (mx, float(np.sqrt(np.mean((em - ex) ** 2)) / r)) if rms else mx


if __name__ == "__main__":
    for N, mask in ((64, "scatter"), (129, "last10pct"), (200, "scatter")):
        for node in TA.NODES:
            print(N, mask, node, f"{floor(N, mask, node, 31 + N):.4f}")


def emulated_lines(z, mask, W, node, lines, bias, heads=4, c=32):
    """``emulated`` restricted to whole output lines (rows i of the starting node, columns j of the
    ending node), for grids too large to model whole; ``bias`` is the exact pair bias of the
    (transposed, for the ending node) grid, as oracle.triangle_attention.pair_bias gives it. Returns
    [len(lines)][N][c_z]."""
    if node == "ending":
        return emulated_lines(np.swapaxes(z, 0, 1), mask, W, "starting", lines, bias, heads, c)
    W = {k: np.asarray(v, np.float64) for k, v in W.items()}
    N = z.shape[0]
    m = np.asarray(mask, np.float64)
    log2e = 1.0 / math.log(2.0)
    b = rh(bias * log2e)
    out = np.empty((len(lines), N, W["w_o"].shape[0]))
    for n, i in enumerate(lines):
        zh = oracle.layer_norm(wl.as_f64(np.ascontiguousarray(z[i])), W["ln_gamma"], W["ln_beta"])
        zb = rh(zh)
        q = rh((zb @ rh(W["w_q"]).T) * (log2e / math.sqrt(c))).reshape(N, heads, c)
        k = rh(zb @ rh(W["w_k"]).T).reshape(N, heads, c)
        v = rh(zb @ rh(W["w_v"]).T).reshape(N, heads, c)
        g = rh(oracle.sigmoid(zb @ rh(W["w_g"]).T)).reshape(N, heads, c)
        s = np.einsum("jhc,khc->hjk", q, k, optimize=True) + b
        valid = (m[i] * m != 0)[None, None, :]
        s = np.where(valid, s, -np.inf)
        smax = np.max(s, axis=-1, keepdims=True)
        smax = np.where(np.isfinite(smax), smax, 0.0)
        e = rh(np.where(valid, np.exp2(s - smax), 0.0))
        den = np.moveaxis(e.sum(axis=-1, keepdims=True), 0, 1)          # [j][h][1]
        num = np.einsum("hjk,khc->jhc", e, v, optimize=True)
        o = rh(g * np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0))
        out[n] = rb(o.reshape(N, heads * c) @ rh(W["w_o"]).T)
    return out
