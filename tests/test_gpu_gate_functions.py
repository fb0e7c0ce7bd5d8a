"""Accuracy of every on-device form of the gate log sigmoid(g) (and of
sigmoid itself in the product form), on a dense grid of logits, against the
fp64 definition and beside CUDA's log2f(1 / (1 + expf(-x))).

Bounds (absolute error of log2 sigmoid, or relative error of sigmoid):
  polynomial form (log2(1 + u) by a degree-7 fit)   |err| <= 1e-6 + 3e-7 |ref|
  ex2 + lg2 forms                                   |err| <= 1e-6 + 3e-7 |ref|
  natural-log form log1pf / expf                    |err| <= 1e-6 + 3e-7 |ref|
  sigmoid = 1 / (1 + 2^{-g log2 e}) (product form)  relative <= 5e-7 + 1.5e-7 |g| where sigmoid >= 2^-120
(the |g| term is the fp32 rounding of the exponent g log2 e, which 2^x turns
into a relative error of ln 2 times its size)
A mistake in a fitted coefficient or a dropped term shows up far above these.
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def lib():
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libgate_functions.so")
    src = os.path.join(HERE, "gate_functions.cu")
    subprocess.run([os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc"), "-gencode", "arch=compute_103a,code=sm_103a",
                    "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    lib.lizard_test_eval_gate.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    lib.lizard_test_eval_gate.restype = ctypes.c_int
    return lib


def grid():
    dense = torch.linspace(-90.0, 90.0, 2_000_001, dtype=torch.float32)
    fine = torch.linspace(-4.0, 4.0, 400_001, dtype=torch.float32)
    special = torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e-6, -1e-6, 88.0, -88.0, 1e4, -87.0], dtype=torch.float32)
    return torch.cat([dense, fine, special])


def evaluate(lib, x, which):
    xd = x.cuda()
    out = torch.empty_like(xd)
    assert lib.lizard_test_eval_gate(xd.data_ptr(), out.data_ptr(), xd.numel(), which) == 0
    return out.cpu()


def log2_sigmoid_ref(x):
    xd = x.double()
    return torch.nn.functional.logsigmoid(xd) / torch.log(torch.tensor(2.0, dtype=torch.float64))


@pytest.mark.parametrize("which,name", [(0, "polynomial"), (1, "ex2+lg2 pair"), (3, "natural log")])
def test_log_sigmoid_forms(lib, which, name):
    x = grid()
    got = evaluate(lib, x, which).double()
    ref = log2_sigmoid_ref(x)
    if which == 3:  # natural logarithm
        ref = ref * torch.log(torch.tensor(2.0, dtype=torch.float64))
    err = (got - ref).abs()
    bound = 1e-6 + 3e-7 * ref.abs()
    worst = int(torch.argmax(err - bound))
    assert bool((err <= bound).all()), f"{name}: x={float(x[worst])} got {float(got[worst])} ref {float(ref[worst])}"
    assert bool((got[x == 0] == got[x == 0][0]).all())


def test_sigmoid_product_form(lib):
    x = grid()
    got = evaluate(lib, x, 4).double()
    ref = torch.sigmoid(x.double())
    ok = ref >= 2.0 ** -120
    rel = ((got - ref).abs() / ref)[ok]
    bound = (5e-7 + 1.5e-7 * x.double().abs())[ok]
    worst = int(torch.argmax(rel - bound))
    assert bool((rel <= bound).all()), (float(x[ok][worst]), float(rel[worst]))
    # tokens past the end are read as g = +inf: no decay at all
    assert float(evaluate(lib, torch.tensor([float("inf")]), 4)[0]) == 1.0


def test_forms_agree_with_cuda_log2f(lib):
    """Beside CUDA's log2f(1 / (1 + expf(-x))) on the grid where that
    expression is itself accurate (it loses precision once 1 + e^{-x}
    rounds to 1 or overflows)."""
    x = grid()
    cuda = evaluate(lib, x, 5).double()
    ref = log2_sigmoid_ref(x)
    usable = (x.abs() <= 15) & torch.isfinite(cuda)
    assert float((cuda - ref).abs()[usable].max()) <= 1e-5
    for which in (0, 1):
        got = evaluate(lib, x, which).double()
        assert float((got - cuda).abs()[usable].max()) <= 2e-5, which
