"""The binding checks every tensor against the sizes a call touches before it hands a pointer to libtm.

libtm's entry points take raw pointers and sizes; they cannot see how large the buffers behind the
pointers are. A tensor of the wrong shape, dtype or size would make a kernel read or write past its
buffer, so the Python wrappers reject it first. Here the ctx's shape query is replaced by a stand-in
(c_z = c_hidden = 16) and every wrapper is given one mismatched CPU tensor at a time: each must raise
before any pointer conversion (which would itself fail on a CPU tensor with a different message).
"""
import pytest
import torch

from pair_representation_boltz_b300 import tm

CZ = CH = 16
N = 6


@pytest.fixture()
def fake_ctx(monkeypatch):
    monkeypatch.setattr(tm, "_ctx_dims", lambda ctx: (CZ, CH, 0))

    def no_pointer(t):
        raise AssertionError("a pointer was taken before the arguments were checked")
    monkeypatch.setattr(tm, "_ptr", no_pointer)
    return object()


def pair(n=N, c=CZ, dtype=torch.float32):
    return torch.zeros(n, n, c, dtype=dtype)


@pytest.mark.parametrize("fn", ["tm_forward", "tm_forward_ex"])
def test_forward_rejects_mismatched_tensors(fake_ctx, fn):
    f = getattr(tm, fn)
    z = pair()
    with pytest.raises(ValueError, match="z must have shape"):
        f(fake_ctx, pair(c=CZ + 1), None, "outgoing", pair(c=CZ + 1))
    with pytest.raises(ValueError, match="z must have shape"):
        f(fake_ctx, torch.zeros(N, N + 1, CZ), None, "outgoing", torch.zeros(N, N + 1, CZ))
    with pytest.raises(ValueError, match="out must match z"):
        f(fake_ctx, z, None, "outgoing", pair(n=N - 1))
    with pytest.raises(ValueError, match="out must match z"):
        f(fake_ctx, z, None, "outgoing", pair(dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="mask"):
        f(fake_ctx, z, torch.ones(N + 1), "outgoing", pair())
    with pytest.raises(ValueError, match="mask"):
        f(fake_ctx, z, torch.ones(N, dtype=torch.float64), "outgoing", pair())


def test_noalloc_and_pair_update_reject_mismatched_tensors(fake_ctx):
    z = pair(dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must match z"):
        tm.tm_forward_noalloc(fake_ctx, z, None, "outgoing", pair(n=N + 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="z must have shape"):
        tm.tm_pair_update(fake_ctx, pair(c=8, dtype=torch.bfloat16), None)


def test_backward_rejects_mismatched_tensors_and_gradients(fake_ctx):
    z = pair()
    ok = {"w_g": torch.zeros(CZ, CZ), "w_a": torch.zeros(CH, CZ), "ln_out_beta": torch.zeros(CH)}
    with pytest.raises(KeyError, match="w_typo"):
        tm.tm_backward(fake_ctx, z, None, "outgoing", z, z, {"w_typo": torch.zeros(CZ, CZ)})
    with pytest.raises(TypeError, match="w_g"):
        tm.tm_backward(fake_ctx, z, None, "outgoing", z, z, {"w_g": torch.zeros(CZ, CZ, dtype=torch.float64)})
    with pytest.raises(ValueError, match="gradient w_a"):
        tm.tm_backward(fake_ctx, z, None, "outgoing", z, z, {**ok, "w_a": torch.zeros(CZ, CZ + 1)})
    with pytest.raises(ValueError, match="gradient ln_out_beta"):
        tm.tm_backward(fake_ctx, z, None, "outgoing", z, z, {**ok, "ln_out_beta": torch.zeros(CH + 1)})
    with pytest.raises(ValueError, match="dout must match z"):
        tm.tm_backward(fake_ctx, z, None, "outgoing", pair(n=N - 1), z, ok)
    with pytest.raises(ValueError, match="dz must match z"):
        tm.tm_backward(fake_ctx, z, None, "outgoing", z, pair(dtype=torch.bfloat16), ok)
    with pytest.raises(ValueError, match="mask"):
        tm.tm_backward(fake_ctx, z, torch.ones(2 * N), "outgoing", z, z, ok)


def test_attention_rejects_mismatched_tensors(fake_ctx):
    z = pair(dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must match z"):
        tm.tm_attn_forward(fake_ctx, z, None, "starting", pair(n=N - 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="z must have shape"):
        tm.tm_attn_forward(fake_ctx, pair(c=2 * CZ, dtype=torch.bfloat16), None, "starting",
                           pair(c=2 * CZ, dtype=torch.bfloat16))


def test_three_steps_reject_buffers_smaller_than_the_call_touches(fake_ctx):
    z = pair()
    ld = N
    ab = torch.zeros(CH * N * ld)
    with pytest.raises(ValueError, match="a holds"):
        tm.tm_project(fake_ctx, z, None, ab[:-1], ab, ld)
    with pytest.raises(ValueError, match="b must be"):
        tm.tm_project(fake_ctx, z, None, ab, ab.to(torch.bfloat16), ld)
    with pytest.raises(ValueError, match="zstat holds"):
        tm.tm_project_ex(fake_ctx, z, None, ab, ab, ld, zstat=torch.zeros(2 * N * N - 1))
    bi, ldx = 4, 8
    with pytest.raises(ValueError, match="x holds"):
        tm.tm_contract(fake_ctx, ab, ab, N, ld, "outgoing", 0, 0, bi, 4, torch.zeros(CH * bi * ldx - 1), ldx)
    with pytest.raises(ValueError, match="x must be"):
        tm.tm_contract_ex(fake_ctx, ab, ab, N, ld, "outgoing", 0, 0, bi, 4, torch.zeros(CH * bi * ldx), ldx,
                          x_storage="fp16")
    with pytest.raises(ValueError, match="a holds"):
        tm.tm_contract(fake_ctx, ab[: CH * N], ab, N, ld, "outgoing", 0, 0, bi, 4, torch.zeros(CH * bi * ldx), ldx)
    with pytest.raises(ValueError, match="x holds"):
        tm.tm_finish(fake_ctx, torch.zeros(CH * bi * ldx - 1), ldx, z, 0, 0, bi, 4, pair())
    with pytest.raises(ValueError, match="out must match z"):
        tm.tm_finish_ex(fake_ctx, torch.zeros(CH * bi * ldx, dtype=torch.float16), ldx, z, 0, 0, bi, 4,
                        pair(n=N + 1), zstat=torch.zeros(2 * N * N))
    with pytest.raises(ValueError, match="zstat holds"):
        tm.tm_finish_ex(fake_ctx, torch.zeros(CH * bi * ldx, dtype=torch.float16), ldx, z, 0, 0, bi, 4,
                        pair(), zstat=torch.zeros(3))


def test_a_missing_ctx_is_refused():
    with pytest.raises(tm.TmError):
        tm.tm_forward(None, pair(), None, "outgoing", pair())
