"""The C ABI from plain C: tests/c_abi_consumer.c is compiled with gcc against
include/moe_ep.h and libmoe_ep.so (no Python binding, no PyTorch), runs a whole pass on
buffers it allocates itself, and its output must equal the oracle's bit for bit."""
import os
import subprocess

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    from combine_routing_count_gb300 import build
    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_consumer")
    subprocess.check_call(["gcc", "-O2", "-std=c99", os.path.join(ROOT, "tests", "c_abi_consumer.c"),
                           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                           "-L", libdir, "-lmoe_ep", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe])
    return exe


@pytest.mark.parametrize("wl", [workloads.Workload("c-abi-bf16", 4, 19, 2048, 32, 8, "bf16", "zipf", 200),
                                workloads.Workload("c-abi-fp8", 8, 9, 1024, 16, 4, "fp8", "uniform", 201)],
                         ids=lambda w: w.name)
def test_c_program_matches_oracle(orc, consumer, tmp_path, wl):
    inp = workloads.make_inputs(wl)
    files = {}
    for k in ("x", "idx", "w"):
        files[k] = str(tmp_path / f"{k}.bin")
        np.ascontiguousarray(inp[k]).tofile(files[k])
    out_path = str(tmp_path / "out.bin")
    r = subprocess.run([consumer, str(wl.N), str(wl.T), str(wl.H), str(wl.E), str(wl.R),
                        "1" if wl.payload == "fp8" else "0", files["x"], files["idx"], files["w"], out_path],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    got = np.fromfile(out_path, dtype=np.uint16).reshape(wl.N, wl.T, wl.H)
    o = orc.forward(wl.N, wl.T, wl.H, wl.E, wl.R, 0, wl.payload, inp["x"], inp["idx"], inp["w"])
    np.testing.assert_array_equal(got, o["out"])
