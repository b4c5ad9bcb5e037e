"""The C ABI from a plain C99 program (tests/c_abi/mlp_block.c): the header
compiles as C, the program links against libtpmlp.so and the CUDA runtime
alone, and on a GPU its forward and backward outputs equal, bit for bit,
those of the same calls made through the Python binding, and match the fp64
oracle within the block's tolerances ("Megatron-LM: Tensor Model Parallel",
Figure 3(a))."""

import glob
import os
import subprocess

import numpy as np
import pytest
import torch

from tensor_transformer_mlp_forward_gb300 import build, inputs

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c_abi", "mlp_block.c")
OUT_DIR = os.path.join(build.BUILD_DIR, "c_abi")
EXE = os.path.join(OUT_DIR, "mlp_block")


def cuda_root() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(build.nvcc())))


def cuda_lib_dir(root: str) -> str:
    for cand in [os.path.join(root, "lib64")] + sorted(glob.glob(os.path.join(root, "targets", "*", "lib"))):
        if os.path.exists(os.path.join(cand, "libcudart.so")):
            return cand
    raise RuntimeError("libcudart.so not found under " + root)


def build_caller() -> str:
    build.build()
    os.makedirs(OUT_DIR, exist_ok=True)
    root = cuda_root()
    libdir = cuda_lib_dir(root)
    pkg = os.path.dirname(build.LIB)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2", "-I", build.INCLUDE,
           "-I", os.path.join(root, "include"), SRC, "-o", EXE, "-L", pkg, "-ltpmlp",
           "-L", libdir, "-lcudart", f"-Wl,-rpath,{pkg}:{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, " ".join(cmd) + "\n" + r.stdout + r.stderr
    return EXE


@pytest.fixture(scope="module")
def exe():
    return build_caller()


def test_builds_and_rejects_bad_arguments(exe):
    # exits before any CUDA call, so it runs without a GPU
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 2 and "usage" in r.stderr
    r = subprocess.run([exe, "0", "256", "1024", "2", "in", "out"], capture_output=True, text=True)
    assert r.returncode == 2


def bits(x: torch.Tensor) -> bytes:
    return x.contiguous().view(torch.int16).numpy().tobytes()


def run_caller(exe, w, cpu):
    tag = f"{w.T}_{w.h}_{w.F}_{w.t}"
    src, dst = os.path.join(OUT_DIR, f"in_{tag}.bin"), os.path.join(OUT_DIR, f"out_{tag}.bin")
    with open(src, "wb") as f:
        for k in inputs.DRAW_ORDER:
            f.write(bits(cpu[k]))
    r = subprocess.run([exe, str(w.T), str(w.h), str(w.F), str(w.t), src, dst],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    raw = open(dst, "rb").read()
    T, h, F = w.T, w.h, w.F
    shapes = [("Y", (T, h), 2), ("Z", (T, F), 2), ("H", (T, F), 2), ("dX", (T, h), 2),
              ("dA", (h, F), 2), ("dB", (F, h), 2), ("db1", (F,), 4), ("db2", (h,), 4)]
    out, pos = {}, 0
    for name, shape, size in shapes:
        n = int(np.prod(shape)) * size
        a = np.frombuffer(raw[pos:pos + n], dtype=np.int16 if size == 2 else np.float32).reshape(shape)
        t = torch.from_numpy(a.copy())
        out[name] = t.view(torch.bfloat16) if size == 2 else t
        pos += n
    assert pos == len(raw)
    os.remove(src)
    os.remove(dst)
    return out


CASES = [
    inputs.custom(T=257, h=520, F=1600, t=8, seed=41),   # ragged tiles and shard widths
    inputs.custom(T=300, h=256, F=1600, t=8, seed=42),   # MN-major operands as one box a stage
    inputs.custom(T=512, h=512, F=2048, t=2, seed=43),   # a row-parallel split in the workspace
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: f"T{w.T}_h{w.h}_F{w.F}_t{w.t}")
def test_plain_c_caller_matches_binding_and_oracle(exe, w):
    import oracle
    from tests.test_gpu_parity import TOL_BWD, TOL_FWD, np64, rel, run_gpu

    cpu = inputs.make_inputs(w)
    got = run_caller(exe, w, cpu)
    ref = run_gpu(cpu, w.t)
    for name, v in got.items():
        assert torch.equal(v, ref[name].cpu()), name
    Y, Z, H = oracle.forward(cpu["X"], cpu["A"], cpu["b1"], cpu["B"], cpu["b2"], cpu["residual"], w.t)
    dX, dA, dB, db1, db2 = oracle.backward(cpu["dY"], cpu["X"], cpu["A"], cpu["b1"], cpu["B"], w.t)
    for name, r, tol in (("Y", Y, TOL_FWD), ("Z", Z, TOL_FWD), ("H", H, TOL_FWD),
                         ("dX", dX, TOL_BWD), ("dA", dA, TOL_BWD), ("dB", dB, TOL_BWD),
                         ("db1", db1, TOL_BWD), ("db2", db2, TOL_BWD)):
        assert rel(np64(got[name]), r) <= tol, name
