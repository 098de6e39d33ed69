"""Helpers shared by the GPU tests: moving seeded inputs to the device and the parity gates."""
import json
import os

import numpy as np

import oracle

# Tolerances on max|delta| / rms(oracle):
#  * float32 path: 1e-5 against the float64 oracle.
#  * bf16 path: 1.5e-2 on the error beyond the bf16 storage the path mandates
#    (a and b stored as bf16, the output stored as bf16): the oracle rounds a
#    and b to bf16, and the half-ulp rounding of each stored output element is
#    not counted ("excess"). The same 1.5e-2 bounds rms|delta|/rms against the
#    plain float64 oracle. The literal max|delta|/rms against the plain oracle
#    sits at the storage floor (about 0.02-0.04 for c = 128; at most 0.035 in
#    every case measured on the GPU); it is bounded by BF16_LITERAL_BOUND, just
#    above that, so a kernel change that doubled the worst error would fail.
F32_TOL = 1e-5
BF16_TOL = 1.5e-2
BF16_LITERAL_BOUND = 0.045


def z_to_device(z):
    import torch
    if z.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(z).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(z, dtype=np.float32)).cuda()


def mask_to_device(m):
    import torch
    return torch.from_numpy(np.ascontiguousarray(m, dtype=np.float32)).cuda()


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_bf16(got, z, m, W, direction, rows=None, cols=None):
    """Apply the bf16 gates; returns the metrics. got: float64 array of the GPU output entries
    (the whole grid, or the rows x cols sub-grid when given)."""
    if rows is None:
        ref_s = oracle.full(z, m, W, direction, storage="bf16")
        ref_e = oracle.full(z, m, W, direction, storage="exact")
    else:
        ref_s = oracle.sampled(z, m, W, direction, rows, cols, storage="bf16")
        ref_e = oracle.sampled(z, m, W, direction, rows, cols, storage="exact")
    es = oracle.errors(got, ref_s, "bf16")
    ee = oracle.errors(got, ref_e, "bf16")
    metrics = {"excess_vs_storage_oracle": es["excess"], "rms_rel_vs_exact": ee["rms_rel"],
               "max_rel_vs_exact": ee["max_rel"], "max_rel_vs_storage_oracle": es["max_rel"]}
    log = os.environ.get("TM_METRICS_LOG")
    if log:     # one JSON line per check, for the record of the measured precision
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "direction": direction, "n_values": int(np.size(got)),
                                **{k: float(v) for k, v in metrics.items()}}) + "\n")
    assert np.all(np.isfinite(got))
    assert es["excess"] <= BF16_TOL, metrics
    assert ee["rms_rel"] <= BF16_TOL, metrics
    assert ee["max_rel"] <= BF16_LITERAL_BOUND, metrics
    return metrics
