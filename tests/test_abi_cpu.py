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


def test_binding_constants_match_the_header():
    """The binding's kernel names follow the header's moe_kernel_id order, and its flag values
    are the header's."""
    from combine_routing_count_gb300 import _abi
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "moe_ep.h")).read(), flags=re.S)
    ids = {m.group(1): int(m.group(2)) for m in re.finditer(r"\bMOE_K_([A-Z0-9_]+)\s*=\s*(\d+)", src)}
    num = ids.pop("NUM")
    assert sorted(ids.values()) == list(range(num)) and len(_abi.KERNEL_NAMES) == num
    for name, i in ids.items():
        assert _abi.KERNEL_NAMES[i] == name.lower(), (name, i)
    flags = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define\s+(MOE_FLAG_[A-Z_]+)\s+0x([0-9a-fA-F]+)u", src)}
    assert len(flags) >= 8
    for name, v in flags.items():
        assert getattr(_abi, name) == v, name


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


def test_library_exports_only_the_abi(L):
    """Every C-linkage symbol the library defines is one of the header's moe_* entry points
    (internal helpers stay out of the dynamic symbol table)."""
    import subprocess
    from combine_routing_count_gb300 import build
    from combine_routing_count_gb300._abi import EXPORTED
    r = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True)
    c_syms = {line.split()[-1].split("@")[0] for line in r.stdout.splitlines()
              if line.strip() and line.split()[-2] in ("T", "W") and not line.split()[-1].startswith("_Z")}
    assert c_syms == set(EXPORTED), sorted(c_syms ^ set(EXPORTED))


def test_host_batch_count_rule(L):
    """The copy-engine pipeline's token batches: about 2 sqrt(token-row MB) by default, the
    caller's count when set (capped at 24 and at T), one for the one-batch flag and for the
    staged fp8 quantiser; 0 for bad dims. Host only."""
    from combine_routing_count_gb300 import MoeLayout
    def nb(N, T, H, E, R, payload=0, flags=0, batches=0, host=1):
        lay = MoeLayout()
        lay.flags, lay.batches = flags, batches
        return L.moe_batches(ctypes.byref(_dims(N, T, H, E, R, 0, payload)), ctypes.byref(lay), host)
    assert nb(8, 128, 7168, 256, 8) == 8        # 14.7 MB of token rows
    assert nb(32, 128, 7168, 384, 8) == 15      # 58.7 MB
    assert nb(16, 512, 4096, 128, 8) == 16      # 67.1 MB
    assert nb(64, 32, 7168, 384, 8, 1) == 11    # 29.4 MB (fp8 payload, bf16 tokens)
    assert nb(64, 256, 7168, 384, 8) == 24      # 235 MB: capped
    assert nb(2, 16, 128, 8, 2) == 1            # 8 KB: no pipeline
    assert nb(8, 128, 7168, 256, 8, batches=7) == 7
    assert nb(8, 3, 7168, 256, 8, batches=16) == 3
    assert nb(8, 128, 7168, 256, 8, batches=40) == 24
    assert nb(8, 128, 7168, 256, 8, flags=0x40) == 1
    assert nb(64, 32, 7168, 384, 8, 1, flags=0x10) == 1
    assert nb(8, 0, 7168, 256, 8) == 1
    assert nb(8, 128, 7168, 250, 8) == 0        # E not a multiple of N



def test_forward_micro_batch_count_rule(L):
    """moe_forward's micro-batches: about one per 55 MB of dispatch and combine rows for bf16
    (at most 20 and T), one per 60 MB for fp8, direct push or separate kernels (at most 16), the
    caller's count when set (at most 32 and T), one for the one-batch flag and for the staged
    fp8 quantiser. Host only."""
    from combine_routing_count_gb300 import MoeLayout
    def nb(N, T, H, E, R, payload=0, flags=0, batches=0):
        lay = MoeLayout()
        lay.flags, lay.batches = flags, batches
        return L.moe_batches(ctypes.byref(_dims(N, T, H, E, R, 0, payload)), ctypes.byref(lay), 0)
    assert nb(8, 128, 7168, 256, 8) == 4         # 235 MB of rows
    assert nb(64, 32, 7168, 384, 8, 1) == 6      # 356 MB (fp8 rows of 7392 B): one per 60 MB
    assert nb(32, 128, 7168, 384, 8) == 18       # 940 MB: 17, rounded up to an even count
    assert nb(16, 512, 4096, 128, 8) == 20       # 1074 MB: 20
    assert nb(16, 1024, 4096, 128, 8) == 20      # 2147 MB: capped
    assert nb(2, 16, 128, 8, 2) == 1             # 32 tokens
    assert nb(8, 32, 7168, 256, 8) == 1          # 59 MB
    assert nb(8, 64, 7168, 256, 8) == 2          # 117 MB
    assert nb(8, 128, 7168, 256, 8, flags=0x80) == 4    # separate kernels: one per 60 MB
    assert nb(16, 512, 4096, 128, 8, flags=0x8) == 16   # direct push: one per 60 MB, capped at 16
    assert nb(32, 128, 7168, 384, 8, flags=0x80) == 16  # capped at 16
    assert nb(8, 160, 7168, 256, 8, flags=0x80) == 6    # 294 MB: 5 rounded up to an even count
    assert nb(8, 128, 7168, 256, 8, batches=3) == 3
    assert nb(8, 2, 7168, 256, 8, batches=9) == 2
    assert nb(16, 512, 4096, 128, 8, batches=20) == 20
    assert nb(16, 512, 4096, 128, 8, batches=40) == 32
    assert nb(8, 128, 7168, 256, 8, flags=0x40) == 1
    assert nb(64, 32, 7168, 384, 8, 1, flags=0x10) == 1


def test_phase_batch_count_rule(L):
    """moe_dispatch / moe_combine token batches: none up to 2048 tokens of all ranks, about
    T/8 beyond (at most 16), the caller's count when set (at most 32 and T), one with the
    one-batch flag. Host only."""
    from combine_routing_count_gb300 import MoeLayout
    def nb(N, T, H, E, R, payload=0, flags=0, batches=0):
        lay = MoeLayout()
        lay.flags, lay.batches = flags, batches
        return L.moe_batches(ctypes.byref(_dims(N, T, H, E, R, 0, payload)), ctypes.byref(lay), 2)
    assert nb(8, 128, 7168, 256, 8) == 1         # 1024 tokens
    assert nb(64, 32, 7168, 384, 8, 1) == 1      # 2048 tokens
    assert nb(64, 64, 7168, 384, 8, 1) == 8      # 4096 tokens, T = 64
    assert nb(32, 128, 7168, 384, 8) == 16       # T = 128
    assert nb(16, 512, 4096, 128, 8) == 16       # T = 512: capped
    assert nb(8, 128, 7168, 256, 8, batches=5) == 5
    assert nb(16, 512, 4096, 128, 8, flags=0x40) == 1
    assert L.moe_batches(ctypes.byref(_dims()), ctypes.byref(MoeLayout()), 3) == 0


def _fake_layout():
    """A layout whose arrays are non-null placeholders: enough for the host-side argument
    checks, which return before anything touches device memory."""
    from combine_routing_count_gb300 import MoeLayout
    from combine_routing_count_gb300._abi import LAYOUT_FIELDS
    lay = MoeLayout()
    for i, f in enumerate(LAYOUT_FIELDS):
        setattr(lay, f, 0x100000 + 256 * i)
    return lay


def test_batched_entry_points_reject_bad_arguments_without_gpu(L):
    """moe_dispatch, moe_combine and moe_forward check their arguments on the host and
    return MOE_ERR_INVALID_ARG (1) before any CUDA call: missing or misaligned buffers, a
    missing layout. (Runs on a machine without a GPU.)"""
    d = _dims(4, 8, 256, 16, 4)
    lay = _fake_layout()
    A, M = 0x200000, 0x200008            # a 16-byte aligned and a misaligned placeholder
    # moe_dispatch(dims, lay, x, send, recv, expert_x, expert_scale, stream)
    assert L.moe_dispatch(ctypes.byref(d), ctypes.byref(lay), None, A, A, A, None, None) == 1
    assert L.moe_dispatch(ctypes.byref(d), ctypes.byref(lay), M, A, A, A, None, None) == 1
    assert L.moe_dispatch(ctypes.byref(d), ctypes.byref(lay), A, None, A, A, None, None) == 1   # send needed
    assert L.moe_dispatch(ctypes.byref(d), None, A, A, A, A, None, None) == 1
    fp8 = _dims(4, 8, 256, 16, 4, 0, 1)
    assert L.moe_dispatch(ctypes.byref(fp8), ctypes.byref(lay), A, A, A, A, None, None) == 1   # scales needed
    # moe_combine(dims, lay, expert_y, csend, crecv, w, out, stream)
    assert L.moe_combine(ctypes.byref(d), ctypes.byref(lay), A, A, A, None, A, None) == 1
    assert L.moe_combine(ctypes.byref(d), ctypes.byref(lay), A, None, A, A, A, None) == 1     # csend needed
    assert L.moe_combine(ctypes.byref(d), ctypes.byref(lay), A, A, M, A, A, None) == 1
    # moe_forward with a micro-batched pass and a missing receive buffer
    from combine_routing_count_gb300 import MoeBuffers
    b = MoeBuffers()
    for f in ("x", "idx", "w", "send", "expert_x", "expert_y", "csend", "crecv", "out"):
        setattr(b, f, A)
    lay.batches = 3
    assert L.moe_forward(ctypes.byref(d), ctypes.byref(lay), ctypes.byref(b), None) == 1
    assert L.moe_forward(ctypes.byref(d), ctypes.byref(lay), None, None) == 1


def test_forward_in_one_batch_checks_every_buffer_first(L):
    """moe_forward in one batch returns MOE_ERR_INVALID_ARG for a missing buffer before the
    layout is launched (without a GPU, a launch would fail with MOE_ERR_CUDA instead)."""
    from combine_routing_count_gb300 import MoeBuffers
    d = _dims(4, 8, 256, 16, 4)
    lay = _fake_layout()
    lay.flags = 0x40
    A = 0x200000
    b = MoeBuffers()
    for f in ("x", "idx", "w", "send", "recv", "expert_x", "expert_y", "csend", "crecv"):
        setattr(b, f, A)
    assert L.moe_forward(ctypes.byref(d), ctypes.byref(lay), ctypes.byref(b), None) == 1   # out missing
    fp8 = _dims(4, 8, 256, 16, 4, 0, 1)
    b.out, b.expert_scale = A, A
    lay.flags = 0x40 | 0x10                                                                # staged quantiser
    assert L.moe_forward(ctypes.byref(fp8), ctypes.byref(lay), ctypes.byref(b), None) == 1  # xq missing
