"""The tcgen05 building blocks the prefill kernel relies on, checked in isolation.

A test-only CUDA source (tests/probes/tcgen05_probe.cu, compiled here with nvcc
for sm_103a against the library's own PTX wrappers) runs one CTA that:
  * multiplies a 128x128 bf16 A by a 32x128 B^T with both operands in shared
    memory in the no-swizzle K-major layout (LBO = 128 B, SBO = 2048 B);
  * repeats it with A held in tensor memory as packed bf16 pairs;
  * multiplies A[:, :16] (tensor memory) by a 128x16 B^T laid out with SBO = 256 B;
  * multiplies V^T by a 16x16 B^T with V, a [16][128] tile, stored M-major with the
    128-byte swizzle a TMA load writes (two 64-column boxes; LBO = 2048 B, SBO = 1024 B).
The products are compared with the same products computed on the host.
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "chunked_kda_delta_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = tmp_path_factory.mktemp("probe") / "probe.so"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", CSRC, "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
                    os.path.join(HERE, "probes", "tcgen05_probe.cu"), "-o", str(out)],
                   check=True)
    lib = ctypes.CDLL(str(out))
    lib.tcgen05_probe.argtypes = [ctypes.c_void_p] * 7
    lib.tcgen05_probe.restype = ctypes.c_int
    lib.tcgen05_probe_mn_sw128.argtypes = [ctypes.c_void_p] * 4
    lib.tcgen05_probe_mn_sw128.restype = ctypes.c_int
    return lib


def test_mma_layouts(probe):
    torch.manual_seed(0)
    dev = "cuda:0"
    A = torch.randn(128, 128, device=dev).to(torch.bfloat16)
    B1 = torch.randn(32, 128, device=dev).to(torch.bfloat16)
    B2 = torch.randn(128, 16, device=dev).to(torch.bfloat16)
    D1ss = torch.full((128, 32), float("nan"), device=dev)
    D1ts = torch.full((128, 32), float("nan"), device=dev)
    D2 = torch.full((128, 128), float("nan"), device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    rc = probe.tcgen05_probe(*(ctypes.c_void_p(t.data_ptr()) for t in (A, B1, B2, D1ss, D1ts, D2, err)))
    assert rc == 0
    assert int(err.item()) == 0
    ref1 = A.double() @ B1.double().T
    ref2 = A[:, :16].double() @ B2.double().T
    for name, got, ref in (("smem A", D1ss, ref1), ("tmem A", D1ts, ref1), ("K=16 N=128", D2, ref2)):
        diff = (got.double() - ref).abs().max().item()
        assert diff < 1e-3, f"{name}: max diff {diff}"


def test_mn_major_swizzled_a(probe):
    torch.manual_seed(1)
    dev = "cuda:0"
    V = torch.randn(16, 128, device=dev).to(torch.bfloat16)
    B = torch.randn(16, 16, device=dev).to(torch.bfloat16)
    D = torch.full((128, 16), float("nan"), device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    rc = probe.tcgen05_probe_mn_sw128(*(ctypes.c_void_p(t.data_ptr()) for t in (V, B, D, err)))
    assert rc == 0
    assert int(err.item()) == 0, "9: the operand's shared-memory base is not 1 KiB aligned"
    ref = V.double().T @ B.double().T
    diff = (D.double() - ref).abs().max().item()
    assert diff < 1e-3, f"M-major swizzled A: max diff {diff}"
