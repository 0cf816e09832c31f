"""The C-ABI library builds, loads and exports every function include/rar.h
declares; the ctypes mirror of rar_options matches the C layout.  No GPU."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import ring_all_reduce_rar_gb300 as rar
from ring_all_reduce_rar_gb300 import _build
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "rar.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return rar.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(rar_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    for must in ("rar_init", "rar_allreduce", "rar_destroy", "rar_reduce_scatter", "rar_all_gather",
                 "rar_status", "rar_send_counts", "rar_last_error", "rar_set_options", "rar_version",
                 "rar_allreduce_host", "rar_allreduce_range", "rar_allreduce_noalloc", "rar_trace"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version(lib):
    assert rar.rar_version() == 1


def test_options_layout_matches_c():
    """Compile a C probe that prints sizeof/offsetof of rar_options."""
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "rar.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(rar_options),
    offsetof(rar_options, engine), offsetof(rar_options, channels), offsetof(rar_options, slice_elems),
    offsetof(rar_options, block_threads), offsetof(rar_options, timeout_ns),
    offsetof(rar_options, skip_pointer_check), offsetof(rar_options, fault_mode),
    offsetof(rar_options, fault_rank), offsetof(rar_options, fault_delay_ns),
    offsetof(rar_options, fused_path), offsetof(rar_options, hier_group), offsetof(rar_options, protocol),
    offsetof(rar_options, slice_block), offsetof(rar_options, trace));
  return 0;
}'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "probe.c")
        exe = os.path.join(d, "probe")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        vals = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    O = rar.Options
    assert vals == [ctypes.sizeof(O), O.engine.offset, O.channels.offset, O.slice_elems.offset,
                    O.block_threads.offset, O.timeout_ns.offset, O.skip_pointer_check.offset,
                    O.fault_mode.offset, O.fault_rank.offset, O.fault_delay_ns.offset, O.fused_path.offset,
                    O.hier_group.offset, O.protocol.offset, O.slice_block.offset, O.trace.offset]


def test_host_side_errors_without_gpu(lib):
    """Argument errors come back as status codes, never a crash: a NULL out
    pointer, a NULL handle, and (no GPU here) rar_init reporting the missing
    device."""
    assert lib.rar_init(None, 0, None) == 1
    assert lib.rar_status(None) == 1
    assert lib.rar_destroy(None) == 0
    arr = (ctypes.c_void_p * 1)()
    assert lib.rar_allreduce(None, arr, 1, 4, 1, 0, None) == 1
    assert lib.rar_allreduce_range(None, arr, 1, 8, 0, 4, 1, 0, None) == 1
    assert rar.rar_last_error(None) != ""
    h = ctypes.c_void_p()
    rc = lib.rar_init(ctypes.byref(h), 0, None)
    import torch
    if not torch.cuda.is_available():
        assert rc in (1, 4)  # RAR_EINVAL (no such device) or RAR_ECUDA
        assert h.value is None
    else:
        assert rc == 0
        lib.rar_destroy(h)


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        rar._abi._marshal([torch.zeros(4), torch.zeros(4)])
    with pytest.raises(ValueError):
        rar._abi._marshal([])


def test_short_timeouts_are_refused_before_any_device_work(lib):
    """timeout_ns bounds every wait of the ring and tree executors and of the
    fused streaming path; a nonzero bound under 1 ms is refused by rar_init
    (argument checks come before the device is touched, so this holds on a
    machine without a GPU too)."""
    for bad in (1, 999_999):
        o = rar.make_options(engine="fused", timeout_ns=bad)
        h = ctypes.c_void_p()
        assert lib.rar_init(ctypes.byref(h), 0, ctypes.byref(o)) == 1  # RAR_EINVAL
        assert h.value is None
        assert "timeout_ns" in rar.rar_last_error(None)
    o = rar.make_options(engine="ring", timeout_ns=1_000_000)
    h = ctypes.c_void_p()
    rc = lib.rar_init(ctypes.byref(h), 0, ctypes.byref(o))
    import torch
    if torch.cuda.is_available():
        assert rc == 0
        lib.rar_destroy(h)
    else:
        assert rc in (1, 4) and "timeout_ns" not in rar.rar_last_error(None)
