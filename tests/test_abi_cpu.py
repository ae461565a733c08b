"""The C-ABI library loads and exports every function include/moe_ep.h declares; host-only
argument logic (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_ep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    from combine_routing_count_gb300 import _abi, build
    build.build()
    return _abi.lib()


def test_every_declared_symbol_is_exported(L):
    from combine_routing_count_gb300 import _abi
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_abi.EXPORTED)


def _dims(N=8, T=128, H=7168, E=256, R=8, cap=0, payload=0):
    from combine_routing_count_gb300 import MoeDims
    return MoeDims(N, T, H, E, R, cap, payload)


def test_dims_validation(L):
    ok = _dims()
    assert L.moe_check_dims(ctypes.byref(ok)) == 0
    bad = [_dims(E=255), _dims(N=0), _dims(T=-1), _dims(H=7170), _dims(R=0), _dims(cap=-1),
           _dims(H=200, payload=1), _dims(payload=2), _dims(E=2048, N=8), _dims(N=4096, E=4096)]
    for d in bad:
        assert L.moe_check_dims(ctypes.byref(d)) == 1, (d.N, d.T, d.H, d.E, d.R, d.cap, d.payload)
    assert L.moe_check_dims(None) == 1


def test_sizes(L):
    d = _dims()
    assert L.moe_recv_capacity_rows(ctypes.byref(d)) == 8 * 128 * max(8, 32)
    assert L.moe_row_bytes(ctypes.byref(d)) == 2 * 7168
    assert L.moe_capacity(ctypes.byref(d)) == 8 * 128
    f = _dims(N=64, T=32, E=384, payload=1)
    assert L.moe_row_bytes(ctypes.byref(f)) == 7168 + 4 * 56
    assert L.moe_recv_capacity_rows(ctypes.byref(f)) == 64 * 32 * 8
    s = _dims(N=16, T=512, H=4096, E=128)
    assert L.moe_recv_capacity_rows(ctypes.byref(s)) == 16 * 512 * 8
    ws = L.moe_layout_workspace_bytes(ctypes.byref(d))
    assert ws % 256 == 0 and ws >= 4 * (3 * 8 * 128 * 8 * 2 + 256 * 1024 + 8 * 32768)
    assert L.moe_layout_workspace_bytes(ctypes.byref(_dims(E=255))) == 0


def test_layout_init_rejects_bad_workspace_without_gpu(L):
    from combine_routing_count_gb300 import MoeLayout
    d = _dims()
    lay = MoeLayout()
    need = L.moe_layout_workspace_bytes(ctypes.byref(d))
    assert L.moe_layout_init(ctypes.byref(d), None, need, ctypes.byref(lay), None) == 1
    assert L.moe_layout_init(ctypes.byref(d), 256 * 1000, need - 1, ctypes.byref(lay), None) == 1
    assert L.moe_layout_init(ctypes.byref(d), 256 * 1000 + 16, need, ctypes.byref(lay), None) == 1


def test_status_strings(L):
    from combine_routing_count_gb300 import _abi
    for code in range(7):
        assert _abi.status_string(code)
    assert L.moe_launch_count() == 0   # nothing launched in a CPU-only process


def test_build_targets_sm103a_only():
    from combine_routing_count_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_library_never_calls_exit(L):
    """nvcc turns a host call of a __device__-only function into a call of exit(1); the
    library must contain no such call (it never exits the caller's process)."""
    import subprocess
    from combine_routing_count_gb300 import build
    r = subprocess.run(["nm", "-D", "--undefined-only", build.LIB], capture_output=True, text=True, check=True)
    imported = {line.split()[-1].split("@")[0] for line in r.stdout.splitlines() if line.strip()}
    assert not ({"exit", "abort", "_exit"} & imported), sorted({"exit", "abort", "_exit"} & imported)
