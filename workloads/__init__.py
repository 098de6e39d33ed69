"""Seeded synthetic inputs for the triangle multiplicative update.

This module is shared by the float64 oracle tests and by the GPU path. It holds
none of the method's arithmetic: only random draws, the token-mask recipes, the
workload table and the bf16 storage format (bit packing).

Workload sizes follow the pages:
  * N = 768 is the Boltz-2 training crop, N = 3605 the four-chain
    TTC7A/PI4KA/FAM126A/EFR3A complex ("Os números" section of "NVIDIA BioNeMo
    escala modelagem biomolecular com context parallelism e quebra barreira de
    memória da GPU");
  * N = 6500 the largest partner protein-protein interactions ("Quem já tá
    usando" section of the same page);
  * N = 10000 residues, i.e. 10^8 pair entries ("2D tiling da pair
    representation" section of the same page).

Recipe (every draw is seeded, nothing is read from disk):
  * z ~ N(0, 1), drawn in float32 in row blocks of ``ROW_BLOCK`` rows, block r
    seeded with SeedSequence([seed, r]) so any row block can be regenerated
    alone; bf16 workloads round the float32 draw to bf16 with
    round-to-nearest-even.
  * weights ~ N(0, 1/fan_in) in float32 (PyTorch Linear layout [out][in]),
    LayerNorm gamma = 1, beta = 0 unless ``ln_random`` asks for random affine
    parameters.
  * token masks: see ``make_mask``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

ROW_BLOCK = 16


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    c_z: int
    c_h: int
    dtype: str                      # "f32" or "bf16": storage of z and out
    mask: str                       # recipe name for make_mask
    directions: tuple = ("outgoing", "incoming")
    block: int = 0                  # output block edge of the streamed schedule (0 = whole grid)
    seed_z: int = 0
    seed_w: int = 1
    seed_pairs: int = 2
    note: str = ""
    chains: tuple = field(default_factory=tuple)


WORKLOADS = {
    "tiny48": Workload("tiny48", 48, 16, 16, "f32", "last5",
                       note="tiny oracle case, fp32, last 5 tokens masked"),
    "crop768": Workload("crop768", 768, 128, 128, "bf16", "last10pct",
                        note="Boltz-2 training crop, last floor(N/10) tokens masked"),
    "complex3605": Workload("complex3605", 3605, 128, 128, "bf16", "full",
                            note="four-chain complex, outgoing then incoming",
                            chains=(1200, 1200, 603, 602)),
    "ppi6500": Workload("ppi6500", 6500, 128, 128, "bf16", "full",
                        note="large protein-protein interaction"),
    "n10000": Workload("n10000", 10000, 128, 128, "bf16", "full", directions=("outgoing",),
                       block=2500, note="10^8 pair entries, block-streamed 2500x2500 output blocks"),
}


# --------------------------------------------------------------------------- weights

WEIGHT_NAMES = ("ln_in_gamma", "ln_in_beta", "w_a", "w_ga", "w_b", "w_gb", "w_g",
                "ln_out_gamma", "ln_out_beta", "w_o")


def weight_shapes(c_z: int, c_h: int) -> dict:
    """Shapes of the layer's parameters, Linear layout [out][in]."""
    return {
        "ln_in_gamma": (c_z,), "ln_in_beta": (c_z,),
        "w_a": (c_h, c_z), "w_ga": (c_h, c_z), "w_b": (c_h, c_z), "w_gb": (c_h, c_z),
        "w_g": (c_z, c_z),
        "ln_out_gamma": (c_h,), "ln_out_beta": (c_h,),
        "w_o": (c_z, c_h),
    }


def make_weights(c_z: int, c_h: int, seed: int = 1, ln_random: bool = False) -> dict:
    """float32 parameters: W ~ N(0, 1/fan_in); LayerNorm gamma=1, beta=0 (or random)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7919]))
    out = {}
    for name, shp in weight_shapes(c_z, c_h).items():
        if name.startswith("w_"):
            fan_in = shp[1]
            out[name] = (rng.standard_normal(shp) / np.sqrt(fan_in)).astype(np.float32)
        elif name.endswith("gamma"):
            out[name] = (1.0 + 0.2 * rng.standard_normal(shp)).astype(np.float32) if ln_random \
                else np.ones(shp, np.float32)
        else:
            out[name] = (0.2 * rng.standard_normal(shp)).astype(np.float32) if ln_random \
                else np.zeros(shp, np.float32)
    return out


def attention_weight_shapes(c_z: int = 128, heads: int = 4, c: int = 32) -> dict:
    """Shapes of a triangle attention layer's parameters, Linear layout [out][in]."""
    hc = heads * c
    return {"ln_gamma": (c_z,), "ln_beta": (c_z,), "w_q": (hc, c_z), "w_k": (hc, c_z), "w_v": (hc, c_z),
            "w_b": (heads, c_z), "w_g": (hc, c_z), "w_o": (c_z, hc)}


def make_attention_weights(c_z: int = 128, heads: int = 4, c: int = 32, seed: int = 1) -> dict:
    """float32 parameters of a triangle attention layer: W ~ N(0, 1/fan_in); LayerNorm gamma=1, beta=0."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 104729]))
    out = {}
    for name, shp in attention_weight_shapes(c_z, heads, c).items():
        if name.startswith("w_"):
            out[name] = (rng.standard_normal(shp) / np.sqrt(shp[1])).astype(np.float32)
        else:
            out[name] = (np.ones(shp) if name.endswith("gamma") else np.zeros(shp)).astype(np.float32)
    return out


# --------------------------------------------------------------------------- masks

def make_mask(N: int, kind: str, seed: int = 3) -> np.ndarray:
    """Token mask m (float32, 0/1) of length N.

    "full": all ones; "last5": ones except the last 5 tokens; "last10pct": the
    last floor(N/10) tokens zeroed; "scatter": a seeded random 20 % of tokens
    zeroed; "none": every token masked.
    """
    m = np.ones(N, np.float32)
    if kind == "full":
        pass
    elif kind == "last5":
        m[max(N - 5, 0):] = 0
    elif kind == "last10pct":
        k = N // 10
        if k:
            m[N - k:] = 0
    elif kind == "scatter":
        rng = np.random.default_rng(np.random.SeedSequence([seed, 104729]))
        m[rng.random(N) < 0.2] = 0
    elif kind == "none":
        m[:] = 0
    else:
        raise ValueError(f"unknown mask recipe {kind!r}")
    return m


# --------------------------------------------------------------------------- bf16 storage format

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- pair representation z

def _block_draw(N: int, c: int, seed: int, r: int, rows: int) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed, r]))
    return rng.standard_normal((rows, N, c), dtype=np.float32)


def z_row_block(N: int, c: int, seed: int, r: int, dtype: str) -> np.ndarray:
    """Rows [r*ROW_BLOCK, ...) of z: float32 values, or uint16 bf16 bits for "bf16"."""
    lo = r * ROW_BLOCK
    rows = min(ROW_BLOCK, N - lo)
    blk = _block_draw(N, c, seed, r, rows)
    return f32_to_bf16_bits(blk) if dtype == "bf16" else blk


def make_z(N: int, c: int, seed: int = 0, dtype: str = "bf16", threads: int | None = None) -> np.ndarray:
    """The pair representation z [N][N][c].

    Returns float32 values for dtype "f32" and uint16 bf16 bit patterns for "bf16".
    """
    out = np.empty((N, N, c), np.uint16 if dtype == "bf16" else np.float32)
    nblk = (N + ROW_BLOCK - 1) // ROW_BLOCK

    def fill(r):
        lo = r * ROW_BLOCK
        out[lo:lo + ROW_BLOCK] = z_row_block(N, c, seed, r, dtype)

    threads = threads or min(32, os.cpu_count() or 1)
    if nblk == 1 or threads == 1:
        for r in range(nblk):
            fill(r)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def as_f64(z: np.ndarray) -> np.ndarray:
    """Values of a z array (float32, or uint16 bf16 bits) as float64 (exact)."""
    if z.dtype == np.uint16:
        return bf16_bits_to_f32(z).astype(np.float64)
    return np.asarray(z, np.float64)


def make_inputs(w: Workload):
    """(z, mask, weights) of a workload: z as in make_z, mask float32 [N], weights float32 dict."""
    return (make_z(w.N, w.c_z, w.seed_z, w.dtype), make_mask(w.N, w.mask),
            make_weights(w.c_z, w.c_h, w.seed_w))


# --------------------------------------------------------------------------- sampled entries

def sample_grid(N: int, n_rows: int = 64, n_cols: int = 64, seed: int = 2, edges=(128, 256, 2500)):
    """Rows and columns of a sampled (i, j) grid for large-N parity checks.

    ``n_rows`` x ``n_cols`` seeded uniform indices, plus the structured edge
    indices 0, N-1 and every multiple of each entry of ``edges`` and its two
    neighbours (tile and block boundaries), deduplicated and sorted.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 15485863]))
    rows = set(rng.integers(0, N, n_rows).tolist())
    cols = set(rng.integers(0, N, n_cols).tolist())
    # the last entry of `edges` is the block edge: all its boundaries are kept
    keep = {0, N - 1}
    for k in range(edges[-1], N, edges[-1]):
        keep.update((k - 1, k, k + 1))
    special = set()
    for e in edges[:-1]:
        for k in range(e, N, e):
            special.update((k - 1, k, k + 1))
    special = sorted(s for s in special - keep if 0 <= s < N)
    # keep the tile-edge set bounded so the oracle stays cheap
    if len(special) > 48:
        pick = np.random.default_rng(np.random.SeedSequence([seed, 1299709])).choice(
            len(special), 48, replace=False)
        special = [special[k] for k in sorted(pick)]
    keep = {s for s in keep if 0 <= s < N}
    rows.update(special, keep)
    cols.update(special, keep)
    return np.array(sorted(rows), np.int64), np.array(sorted(cols), np.int64)
