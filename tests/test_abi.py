"""Host-side checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/flint_moe.h declares, and rejects bad arguments before
touching a GPU."""
import ctypes
import os
import subprocess

import pytest

from bit_quantized_expert_softmax_b300 import build, flint_moe as fm


@pytest.fixture(scope="module")
def library():
    build.build()
    return fm.lib()


def test_header_declares_the_boundary():
    names = fm.header_functions()
    for n in ["flint_moe_create", "flint_moe_load_weights", "flint_moe_forward", "flint_moe_destroy"]:
        assert n in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(library):
    out = subprocess.run(["nm", "-D", "--defined-only", fm.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    declared = set(fm.header_functions())
    assert declared <= exported, declared - exported
    # nothing but the declared API leaks out of the library
    assert {e for e in exported if e.startswith("flint")} == declared


def test_library_is_built_for_sm_103a(library):
    out = subprocess.run(["cuobjdump", "--list-elf", fm.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_status_strings(library):
    assert library.flint_moe_status_string(0) == b"ok"
    assert library.flint_moe_status_string(1) == b"invalid argument"
    assert library.flint_moe_status_string(99) == b"unknown status"


def test_bad_arguments_are_rejected_without_a_device(library):
    # invalid configurations fail validation before any CUDA call
    bad = [dict(d=100, f=512), dict(d=2048, f=500), dict(d=2048, f=512, n_experts=20),
           dict(d=2048, f=512, top_k=0), dict(d=2048, f=512, top_k=9), dict(d=2048, f=512, n_shared=2),
           dict(d=2048, f=512, wfmt=7), dict(d=2048, f=512, max_tokens=0)]
    for kw in bad:
        with pytest.raises(fm.FlintError) as ei:
            fm.flint_moe_create(**kw)
        assert ei.value.code == fm.FLINT_EINVAL, kw
    null = ctypes.c_void_p()
    assert library.flint_moe_create(None, ctypes.byref(null)) == fm.FLINT_EINVAL
    assert library.flint_moe_forward(None, 0, None, 1, None, None) == fm.FLINT_EINVAL
    assert library.flint_moe_forward_stack(None, 0, 1, None, 1, None) == fm.FLINT_EINVAL
    assert library.flint_moe_load_weights(None, 0, None) == fm.FLINT_EINVAL
    assert library.flint_moe_status(None) == fm.FLINT_EINVAL
    assert library.flint_moe_dequant(None, 0, 0, 0, None, None) == fm.FLINT_EINVAL
    assert library.flint_moe_topk(None, 1, 20, 6, None, None, None) == fm.FLINT_EINVAL   # E not a multiple of 32
    assert library.flint_moe_topk(None, 1, 256, 9, None, None, None) == fm.FLINT_EINVAL  # k > 8
    assert library.flint_moe_topk(None, 0, 256, 6, None, None, None) == fm.FLINT_OK      # T == 0: no-op
    assert library.flint_moe_device_bytes(None) == 0
    library.flint_moe_destroy(None)   # NULL-safe
