"""The product path and the oracle stay apart, and a missing CUDA library fails loudly (no CPU
fallback). CPU only."""
import os
import re
import subprocess
import sys

import pytest

from tiled_attention_gb300 import attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "tiled_attention_gb300")


def test_package_sources_never_use_the_oracle():
    """No import of the oracle package and no use of its names anywhere in the library (its
    docstrings may still say what the oracle shares with it: the seeded inputs)."""
    use = re.compile(r"^\s*(import|from)\s+oracle\b|\boracle\.[a-z_]|#include\s+\"[^\"]*oracle",
                     re.M)
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".inc")):
                text = open(os.path.join(dirpath, f)).read()
                assert not use.search(text), os.path.join(dirpath, f)


def test_using_the_package_loads_no_oracle_module():
    code = ("import sys; from tiled_attention_gb300 import attn, inputs, runner; "
            "attn.declared_functions(); "
            "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules), "
            "sorted(m for m in sys.modules if 'oracle' in m)")
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, check=True)


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(attn, "_lib", None)
    monkeypatch.setattr(attn, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libtiled_attn.so"))
    with pytest.raises(RuntimeError, match="missing"):
        attn.lib()
