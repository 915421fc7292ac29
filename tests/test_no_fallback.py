"""The product has one implementation, the CUDA library: without libaq.so every
call raises, and nothing under the package (Python or CUDA source) imports,
loads or links the oracle."""
import os
import re

import pytest

import affine_bit_quantized_gb300 as aq
from affine_bit_quantized_gb300 import _lib

PKG = os.path.dirname(os.path.abspath(aq.__file__))


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB", str(tmp_path / "libaq.so"))
    for call in (aq.version, lambda: aq.status_string(0), lambda: aq.aq_matmul_workspace_bytes(32, 512)):
        with pytest.raises(RuntimeError, match="not built"):
            call()


def test_package_never_reaches_the_oracle():
    # an import, an attribute of the module, its C symbols or its library
    pattern = re.compile(r"^\s*(import|from)\s+oracle\b|\boracle\.[A-Za-z_]|\baqo_|liboracle|oracle/")
    offenders = []
    for root, _, files in os.walk(PKG):
        if "__pycache__" in root or os.sep + "_build" in root:
            continue
        for name in files:
            if not name.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                continue
            path = os.path.join(root, name)
            for i, line in enumerate(open(path, encoding="utf-8"), 1):
                code = line.split("#", 1)[0] if name.endswith(".py") else line.split("//", 1)[0]
                if pattern.search(code):
                    offenders.append(f"{os.path.relpath(path, PKG)}:{i}: {line.strip()}")
    assert not offenders, offenders
