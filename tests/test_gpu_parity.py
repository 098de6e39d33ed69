"""Parity of the CUDA path (through the C ABI) against the float64 oracle, element by element."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_util import (BF16_TOL, F32_TOL, check_bf16, mask_to_device, to_f64, z_to_device)

pytestmark = pytest.mark.gpu

DIRS = ("outgoing", "incoming")


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from pair_representation_boltz_b300 import build
    build.build()
    return torch


@pytest.fixture(scope="module")
def tm128(torch_cuda):
    from pair_representation_boltz_b300 import tm
    W = wl.make_weights(128, 128, 1)
    mod = tm.TriMul(128, 128, W)
    yield mod, W
    mod.close()


# --------------------------------------------------------------------------- float32 path

@pytest.mark.parametrize("direction", DIRS)
def test_tiny48_f32(torch_cuda, direction):
    from pair_representation_boltz_b300 import tm
    w = wl.WORKLOADS["tiny48"]
    z, m, W = wl.make_inputs(w)
    mod = tm.TriMul(w.c_z, w.c_h, W)
    out = mod(z_to_device(z), mask_to_device(m), direction)
    torch_cuda.cuda.synchronize()
    ref = oracle.full(z, m, W, direction)
    e = oracle.errors(to_f64(out), ref)
    assert e["max_rel"] <= F32_TOL, e
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    mod.close()


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("shape", [(37, 20, 12), (5, 3, 7), (1, 8, 8), (70, 256, 64)])
def test_f32_general_shapes(torch_cuda, direction, shape):
    from pair_representation_boltz_b300 import tm
    N, c_z, c_h = shape
    z = wl.make_z(N, c_z, 4, "f32")
    m = wl.make_mask(N, "scatter", 5)
    W = wl.make_weights(c_z, c_h, 6, ln_random=True)
    mod = tm.TriMul(c_z, c_h, W)
    out = mod(z_to_device(z), mask_to_device(m), direction)
    ref = oracle.full(z, m, W, direction)
    e = oracle.errors(to_f64(out), ref)
    assert e["max_rel"] <= F32_TOL, e
    mod.close()


def test_f32_block_schedule(torch_cuda):
    from pair_representation_boltz_b300 import tm
    N = 45
    z = z_to_device(wl.make_z(N, 16, 7, "f32"))
    m = mask_to_device(wl.make_mask(N, "last5"))
    mod = tm.TriMul(16, 16, wl.make_weights(16, 16, 8))
    for d in DIRS:
        full = mod(z, m, d)
        blk = mod(z, m, d, block=16)
        assert torch_cuda.equal(full, blk)
    mod.close()


# --------------------------------------------------------------------------- contraction alone

def _bf16_values(shape, seed):
    f = np.random.default_rng(seed).standard_normal(shape).astype(np.float32)
    bits = wl.f32_to_bf16_bits(f)
    return bits, wl.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("N", [1, 7, 64, 127, 128, 129, 255, 257, 300])
def test_contract_bf16_matches_matmul(tm128, torch_cuda, direction, N):
    from pair_representation_boltz_b300 import tm
    torch = torch_cuda
    mod, _ = tm128
    ld = (N + 7) // 8 * 8
    abits, a = _bf16_values((128, N, ld), 100 + N)
    bbits, b = _bf16_values((128, N, ld), 200 + N)
    ad, bd = z_to_device(abits), z_to_device(bbits)
    A, B = a[:, :, :N], b[:, :, :N]
    ref = np.matmul(A, np.swapaxes(B, 1, 2)) if direction == "outgoing" else np.matmul(np.swapaxes(A, 1, 2), B)
    # whole grid, and an interior block with ragged edges
    blocks = [(0, 0, N, N)]
    if N >= 129:
        blocks.append((3, N // 3, N - 3 - 5, N - N // 3 - 1))
    for (i0, j0, bi, bj) in blocks:
        granule = (bj + 3) // 4 * 4          # stores may fill the 16-byte granule holding column bj-1
        ldx = granule + 8
        x = torch.full((128, bi, ldx), float("nan"), device="cuda")
        tm.tm_contract(mod.ctx, ad, bd, N, ld, direction, i0, j0, bi, bj, x, ldx)
        got = to_f64(x)[:, :, :bj]
        exp = ref[:, i0:i0 + bi, j0:j0 + bj]
        rms = np.sqrt(np.mean(exp * exp))
        err = np.max(np.abs(got - exp)) / rms
        assert err <= 2e-5, (direction, N, (i0, j0, bi, bj), err)
        assert np.all(np.isnan(to_f64(x)[:, :, granule:])), "wrote outside the block's row granules"


# --------------------------------------------------------------------------- projection and finish alone

@pytest.mark.parametrize("N", [1, 100, 129, 257])
def test_project_bf16(tm128, torch_cuda, N):
    from pair_representation_boltz_b300 import tm
    torch = torch_cuda
    mod, W = tm128
    z = wl.make_z(N, 128, 11 + N, "bf16")
    m = wl.make_mask(N, "scatter", 12)
    ld = (N + 7) // 8 * 8
    a = torch.zeros((128, N, ld), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros_like(a)
    tm.tm_project(mod.ctx, z_to_device(z), mask_to_device(m), a, b, ld)
    _, ea, eb, _ = oracle.intermediates(z, m, W, "outgoing", "bf16")
    for got_t, exp in ((a, ea), (b, eb)):
        got = to_f64(got_t)[:, :, :N]                    # [c][i][j]
        exp = np.moveaxis(exp, -1, 0)
        diff = np.abs(got - exp)
        ulp = 2 * oracle.half_ulp_bf16(exp)
        # Before its bf16 rounding the kernel's value carries an absolute error of about
        # 2^-18 * sqrt(c_z) * |W| (hi + lo weights) plus the fp32 accumulation: ~1e-5 of rms(a).
        # So an element may land one bf16 step away from the oracle's rounding, and elements
        # much smaller than rms(a) may be many of their own ulps away in absolute terms.
        rms = np.sqrt(np.mean(exp * exp))
        assert np.all(diff <= ulp * 1.0001 + 3e-5 * rms), np.max((diff - ulp) / rms)
        assert np.mean(diff > 0) < 2e-2                   # rounding flips are rare
        assert np.all(got[:, m == 0, :] == 0) and np.all(got[:, :, m == 0] == 0)


@pytest.mark.parametrize("N", [64, 129])
def test_finish_bf16(tm128, torch_cuda, N):
    from pair_representation_boltz_b300 import tm
    torch = torch_cuda
    mod, W = tm128
    z = wl.make_z(N, 128, 21, "bf16")
    x = np.random.default_rng(22).standard_normal((128, N, N)).astype(np.float32) * 3 + 0.5
    ldx = (N + 3) // 4 * 4
    xd = torch.zeros((128, N, ldx), device="cuda")
    xd[:, :, :N] = torch.from_numpy(x).cuda()
    out = torch.zeros((N, N, 128), dtype=torch.bfloat16, device="cuda")
    tm.tm_finish(mod.ctx, xd, ldx, z_to_device(z), 0, 0, N, N, out)
    zh = oracle.normalise_input(wl.as_f64(z), {k: np.asarray(v, np.float64) for k, v in W.items()})
    ref = oracle.output(np.moveaxis(x.astype(np.float64), 0, -1), zh, {k: np.asarray(v, np.float64) for k, v in W.items()})
    e = oracle.errors(to_f64(out), ref, "bf16")
    assert e["excess"] <= BF16_TOL / 2, e


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("N,mask,ld_pad", [(77, "scatter", 8), (300, "last10pct", 64)])
def test_three_steps_reproduce_forward_bit_for_bit(tm128, torch_cuda, direction, N, mask, ld_pad):
    """tm_project_ex -> tm_contract_ex -> tm_finish_ex with the default fp16 x, over the whole grid, is
    tm_forward: the same kernels on the same values, so the outputs agree bit for bit whatever the
    row padding of the caller's buffers."""
    from pair_representation_boltz_b300 import tm
    torch = torch_cuda
    mod, W = tm128
    z = z_to_device(wl.make_z(N, 128, 61 + N, "bf16"))
    m = mask_to_device(wl.make_mask(N, mask, 62))
    ref = mod(z, m, direction)
    ld = (N + ld_pad - 1) // ld_pad * ld_pad
    a = torch.empty((128, N, ld), dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    zstat = torch.empty((N, N, 2), dtype=torch.float32, device="cuda")
    tm.tm_project_ex(mod.ctx, z, m, a, b, ld, zstat)
    ldx = (N + 7) // 8 * 8
    x = torch.empty((128, N, ldx), dtype=torch.float16, device="cuda")
    tm.tm_contract_ex(mod.ctx, a, b, N, ld, direction, 0, 0, N, N, x, ldx, "fp16")
    out = torch.full_like(z, float("nan"))
    tm.tm_finish_ex(mod.ctx, x, ldx, z, 0, 0, N, N, out, "fp16", zstat)
    torch.cuda.synchronize()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK
    assert torch.equal(out, ref)
    # the stored x is the float32 contraction times 2^e, rounded once to fp16
    e = tm.tm_x_exponent(mod.ctx, N)
    x32 = torch.empty((128, N, ldx), dtype=torch.float32, device="cuda")
    tm.tm_contract_ex(mod.ctx, a, b, N, ld, direction, 0, 0, N, N, x32, ldx, "fp32")
    torch.cuda.synchronize()
    assert torch.equal(x[:, :, :N], (x32[:, :, :N] * 2.0 ** e).to(torch.float16))
    # fp16 x without the projection's statistics is refused before any launch
    with pytest.raises(tm.TmError):
        tm.tm_finish_ex(mod.ctx, x, ldx, z, 0, 0, N, N, out, "fp16", None)


# --------------------------------------------------------------------------- whole update, bf16

@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("N,mask", [(48, "last5"), (129, "scatter"), (300, "last10pct"), (1, "full"), (2, "none")])
def test_forward_bf16(tm128, torch_cuda, direction, N, mask):
    mod, W = tm128
    z = wl.make_z(N, 128, 31 + N, "bf16")
    m = wl.make_mask(N, mask, 32)
    out = mod(z_to_device(z), mask_to_device(m), direction)
    check_bf16(to_f64(out), z, m, W, direction)


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("N,mask", [(129, "scatter"), (300, "last10pct")])
def test_forward_bf16_x_fp32(tm128, torch_cuda, direction, N, mask):
    """The float32 storage of x (tm_options.x_storage) meets the same gates."""
    mod, W = tm128
    z = wl.make_z(N, 128, 51 + N, "bf16")
    m = wl.make_mask(N, mask, 52)
    out = mod(z_to_device(z), mask_to_device(m), direction, x_storage="fp32")
    check_bf16(to_f64(out), z, m, W, direction)


@pytest.mark.parametrize("gain", [300.0, 1e-3])
def test_fp16_x_scale_follows_the_magnitude_of_a_and_b(torch_cuda, gain):
    """Projections scaled up (x ~ 1e5 times larger) or down (x ~ 1e-6 times): the power-of-two scale of the
    fp16 x follows, nothing overflows or flushes, and the bf16 gates hold in both directions."""
    from pair_representation_boltz_b300 import tm
    W = wl.make_weights(128, 128, 1)
    for k in ("w_a", "w_b"):
        W[k] = (W[k] * gain).astype(np.float32)
    mod = tm.TriMul(128, 128, W)
    N = 200
    z = wl.make_z(N, 128, 61, "bf16")
    m = wl.make_mask(N, "last10pct", 62)
    for d in DIRS:
        out = mod(z_to_device(z), mask_to_device(m), d)
        o = to_f64(out)
        assert np.isfinite(o).all()
        check_bf16(o, z, m, W, d)
    mod.close()


def test_forward_large_channel_mean_of_x(torch_cuda):
    """x with a channel mean several times its spread (a, b share a positive offset in every channel):
    the output LayerNorm folded into the finish GEMM (W_o' x - mu rowsum W_o') still meets the gates."""
    from pair_representation_boltz_b300 import tm
    W = wl.make_weights(128, 128, 1)
    W["ln_in_beta"] = np.full(128, 3.0, np.float32)
    for k in ("w_a", "w_b"):     # every row sums to 1/2: a and b get a positive offset in every channel
        W[k] = (W[k] - W[k].mean(axis=1, keepdims=True) + 0.5 / 128).astype(np.float32)
    for k in ("w_ga", "w_gb"):   # gates near 1/2 in every channel, so the offset is alike across channels
        W[k] = (W[k] * 0.05).astype(np.float32)
    mod = tm.TriMul(128, 128, W)
    N = 200
    z = wl.make_z(N, 128, 71, "bf16")
    m = wl.make_mask(N, "full")
    zd = z_to_device(z)
    # the premise: the mean over channels of x dominates its spread
    import oracle
    _, _, _, x = oracle.intermediates(wl.as_f64(z), m, W, "outgoing", storage="bf16")
    ratio = np.abs(x.mean(-1)).mean() / x.std(-1).mean()
    assert ratio > 4, ratio
    for d in DIRS:
        check_bf16(to_f64(mod(zd, mask_to_device(m), d)), z, m, W, d)
    mod.close()


@pytest.mark.parametrize("direction", DIRS)
def test_crop768(tm128, torch_cuda, direction):
    """Boltz-2 training crop: N = 768, last 76 tokens masked, whole grid against the full oracle."""
    mod, W = tm128
    w = wl.WORKLOADS["crop768"]
    z, m, _ = wl.make_inputs(w)
    out = mod(z_to_device(z), mask_to_device(m), direction)
    check_bf16(to_f64(out), z, m, W, direction)


@pytest.mark.parametrize("direction", DIRS)
def test_block_schedule_is_bitwise_identical(tm128, torch_cuda, direction):
    mod, _ = tm128
    N = 300
    z = z_to_device(wl.make_z(N, 128, 41, "bf16"))
    m = mask_to_device(wl.make_mask(N, "scatter", 42))
    full = mod(z, m, direction)
    for blk in (128, 100, 257):
        assert torch_cuda.equal(full, mod(z, m, direction, block=blk)), blk


def test_mask_none_equals_all_ones(tm128, torch_cuda):
    mod, _ = tm128
    N = 96
    z = z_to_device(wl.make_z(N, 128, 43, "bf16"))
    ones = mask_to_device(np.ones(N, np.float32))
    for d in DIRS:
        assert torch_cuda.equal(mod(z, None, d), mod(z, ones, d))


# --------------------------------------------------------------------------- errors and watchdog

def test_invalid_arguments(tm128, torch_cuda):
    from pair_representation_boltz_b300 import tm
    torch = torch_cuda
    mod, _ = tm128
    z = z_to_device(wl.make_z(16, 128, 1, "bf16"))
    with pytest.raises(tm.TmError) as e:
        tm.tm_forward(mod.ctx, z, None, "outgoing", z)            # out aliases z
    assert e.value.status == tm.TM_ERR_INVALID
    with pytest.raises(tm.TmError) as e:
        tm.tm_forward(mod.ctx, z, None, 7, torch.empty_like(z))   # bad direction
    assert e.value.status == tm.TM_ERR_INVALID
    with pytest.raises(tm.TmError) as e:
        tm.tm_forward_ex(mod.ctx, z, None, "outgoing", torch.empty_like(z), workspace_limit=1024)
    assert e.value.status == tm.TM_ERR_OOM
    small = tm.TriMul(64, 64, wl.make_weights(64, 64, 2))
    with pytest.raises(tm.TmError) as e:
        small(z_to_device(wl.make_z(8, 64, 1, "bf16")))
    assert e.value.status == tm.TM_ERR_UNSUPPORTED
    small.close()
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK


def test_watchdog_reports_timeout_and_ctx_stays_usable(tm128, torch_cuda):
    from pair_representation_boltz_b300 import tm
    mod, W = tm128
    tm.tm_watchdog_selftest(mod.ctx, 50)
    assert tm.tm_sync_status(mod.ctx) == tm.TM_ERR_TIMEOUT
    assert "kernel 9" in tm.tm_last_error(mod.ctx)
    assert tm.tm_sync_status(mod.ctx) == tm.TM_OK            # cleared once reported
    N = 40
    z = wl.make_z(N, 128, 3, "bf16")
    m = wl.make_mask(N, "full")
    out = mod(z_to_device(z), mask_to_device(m), "outgoing")
    check_bf16(to_f64(out), z, m, W, "outgoing")


def test_timing_and_launch_count(tm128, torch_cuda):
    from pair_representation_boltz_b300 import tm
    mod, _ = tm128
    N = 200
    z = z_to_device(wl.make_z(N, 128, 5, "bf16"))
    before = tm.tm_launch_count(mod.ctx)
    tm.tm_set_timing(mod.ctx, True)
    mod(z, None, "outgoing", block=100)
    t = tm.tm_get_timing(mod.ctx)
    tm.tm_set_timing(mod.ctx, False)
    assert tm.tm_launch_count(mod.ctx) - before == 1 + 2 * 4
    assert t["project"]["launches"] == 1 and t["contract"]["launches"] == 4 and t["finish"]["launches"] == 4
    assert t["contract"]["units"] == 128 * N * N
    assert all(t[k]["ms"] > 0 for k in ("project", "contract", "finish"))
