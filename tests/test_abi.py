"""The C-ABI library loads and exports every function include/tm.h declares (no GPU needed)."""
import ctypes
import os
import subprocess

import pytest

from pair_representation_boltz_b300 import build, tm


@pytest.fixture(scope="module")
def libtm():
    build.build()
    return tm.load_library()


def test_header_declares_the_boundary():
    names = tm.header_functions()
    for required in ("tm_create", "tm_forward", "tm_forward_ex", "tm_destroy", "tm_sync_status",
                     "tm_status_string", "tm_project", "tm_contract", "tm_finish", "tm_project_ex",
                     "tm_contract_ex", "tm_finish_ex", "tm_x_exponent", "tm_ctx_info"):
        assert required in names


def test_library_exports_every_declared_function(libtm):
    out = subprocess.run(["nm", "-D", "--defined-only", tm.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in tm.header_functions():
        assert name in exported, f"{name} declared in tm.h but not exported"
        assert getattr(libtm, name) is not None


def test_binding_mirrors_the_header():
    for name in tm.header_functions():
        assert callable(getattr(tm, name, None)), f"binding lacks {name}"


def test_status_strings(libtm):
    assert tm.tm_status_string(0) == "ok"
    assert tm.tm_status_string(5) == "device wait timed out"
    assert tm.tm_status_string(99) == "unknown status"


def test_create_rejects_bad_arguments_before_touching_cuda(libtm):
    ctx = ctypes.c_void_p()
    w = tm.TmWeights()                      # all NULL pointers
    assert libtm.tm_create(128, 128, ctypes.byref(w), ctypes.byref(ctx)) == tm.TM_ERR_INVALID
    assert libtm.tm_create(0, 128, None, ctypes.byref(ctx)) == tm.TM_ERR_INVALID
    assert not ctx.value
    libtm.tm_destroy(None)                  # no-op
    assert libtm.tm_launch_count(None) == 0
    assert libtm.tm_ctx_info(None, None, None, None) == tm.TM_ERR_INVALID
    assert libtm.tm_x_exponent(None, 100) == 0


def test_options_struct_layout():
    # int block; int timeout_ms; size_t workspace_limit; int x_storage; int residual; int reserved[6]
    assert ctypes.sizeof(tm.TmOptions) == 4 + 4 + 8 + 4 + 4 + 24
    assert tm.TmOptions.workspace_limit.offset == 8
    assert tm.TmOptions.x_storage.offset == 16
    assert tm.TmOptions.residual.offset == 20
    assert ctypes.sizeof(tm.TmTiming) == 48 + 96 + 96
    assert ctypes.sizeof(tm.TmGrads) == 10 * 8


def test_library_is_built_for_sm_103a(libtm):
    # the build command pins the architecture; check the flag list rather than the binary
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)
    assert os.path.getsize(tm.LIB_PATH) > 0
