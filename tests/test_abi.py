"""The C-ABI library builds, loads and exports every symbol that
include/pcloth.h declares (no GPU needed: nothing here calls into CUDA)."""
import ctypes
import os
import re

from sparse_linear_solve_gb300 import build as B
from sparse_linear_solve_gb300 import pcloth as pc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "pcloth.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pcloth_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert sorted(pc.EXPORTS) == declared_functions()


def test_library_loads_and_exports_every_declared_symbol():
    path = B.build()
    assert os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm_103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.NVCC_FLAGS)


def test_binding_rejects_bad_tensors_before_calling_cuda():
    import pytest
    import torch
    x = torch.zeros(4, 3, dtype=torch.float64)
    with pytest.raises(TypeError):
        pc._check(x, torch.float32, None, None, "x")
    y = torch.zeros(3, 4, dtype=torch.float32).t()
    with pytest.raises(ValueError):
        pc._check(y, torch.float32, None, None, "y")
