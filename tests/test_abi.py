"""The C-ABI library loads and exports every function include/kv.h declares
(no GPU needed: nothing here launches a kernel)."""
import ctypes
import os
import subprocess

from paged_kv_cache_492_b300 import build, kv


def test_library_builds_for_sm103a():
    path = build.build()
    assert os.path.exists(path)
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


def test_exports_every_declared_symbol():
    path = build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    declared = kv.declared_functions()
    assert len(declared) >= 20
    missing = [n for n in declared if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(path)
    for n in declared:
        getattr(lib, n)


def test_binding_covers_header():
    assert set(kv.declared_functions()) <= set(kv._SIGS)


def test_status_strings_and_sizes():
    assert kv.status_string(kv.KV_OK) == "ok"
    assert "free list" in kv.status_string(kv.KV_ENOSPACE)
    assert kv.kv_status_workspace_size() == 256
    assert kv.kv_select_workspace_size(64, 300) >= 256 + 64 * 4
    assert kv.kv_append_workspace_size(8) >= 256 + 64
    assert kv.kv_compact_workspace_size(4, 10) >= 256 + 4 * 10 * 4
