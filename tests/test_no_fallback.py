"""The library has one compute path, the CUDA one: no CPU fallback, no oracle.

Checked on the host: the package never imports the oracle, a missing shared
library is an error rather than a silent detour, and host tensors are refused
instead of being computed on the CPU.
"""
import ast
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "decode_gemv_sign_gb300")


def _imports(path: str) -> set:
    tree = ast.parse(open(path).read(), path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_package_sources_never_import_the_oracle():
    files = [os.path.join(PKG, f) for f in os.listdir(PKG) if f.endswith(".py")]
    assert files
    for f in files:
        assert "oracle" not in _imports(f), f
    for f in os.listdir(os.path.join(PKG, "csrc")):
        text = open(os.path.join(PKG, "csrc", f)).read()
        assert "wcomp_oracle" not in text and "oracle/" not in text, f


def test_importing_the_package_loads_no_oracle():
    code = ("import sys; sys.path.insert(0, sys.argv[1]); import decode_gemv_sign_gb300, "
            "decode_gemv_sign_gb300.wcomp, decode_gemv_sign_gb300.synth, decode_gemv_sign_gb300.validate; "
            "print(sorted(m for m in sys.modules if m.split('.')[0] == 'oracle'))")
    r = subprocess.run([sys.executable, "-c", code, ROOT], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "[]"


def test_missing_library_is_an_error(tmp_path):
    # point the binding at a library that does not exist: every entry point must raise
    code = r"""
import sys
sys.path.insert(0, sys.argv[1])
from decode_gemv_sign_gb300 import wcomp
wcomp.LIB_PATH = sys.argv[2]
wcomp._lib = None
failed = []
for call in (wcomp.version, wcomp.launch_count, lambda: wcomp.deserialize(b"WCMP" + bytes(92))):
    try:
        call()
    except RuntimeError as e:
        failed.append("not built" in str(e))
print(failed)
"""
    r = subprocess.run([sys.executable, "-c", code, ROOT, str(tmp_path / "libwcomp.so")], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "[True, True, True]"


def test_host_tensors_are_refused():
    from decode_gemv_sign_gb300 import wcomp

    w = torch.zeros(4, 8, dtype=torch.bfloat16)
    x = torch.zeros(1, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="CUDA tensor"):
        wcomp.encode(w, 0)
    with pytest.raises(TypeError, match="CUDA tensor"):
        wcomp.gemv_bf16(w, x)
