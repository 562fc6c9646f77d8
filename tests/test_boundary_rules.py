"""Host-side rules of the boundary, checked without a GPU: the product path has
no CPU fallback (a missing library or host tensors fail loudly before any
compute) and shares nothing with the oracle (no import, include or link)."""
import ast
import os
import subprocess
import sys

import pytest
import torch

import mla_latent_kv_07_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mla_latent_kv_07_gb300")


def test_missing_library_fails_loudly():
    # a fresh interpreter whose library path points nowhere: the first call raises
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import mla_latent_kv_07_gb300 as mla\n"
        "mla.LIB_PATH = '/nonexistent/libmla.so'\n"
        "try:\n"
        "    mla.workspace_size(8, 128, 4096)\n"
        "except RuntimeError as e:\n"
        "    print('raised', 'missing' in str(e))\n"
        "else:\n"
        "    print('no error')\n" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert out.stdout.strip() == "raised True", out.stdout + out.stderr


def test_host_tensors_are_refused_before_any_compute():
    # every entry point takes device tensors only; host ones are refused by the
    # binding's checks (there is no CPU path to fall back on)
    with pytest.raises(ValueError):
        mla.Cache(2, 64, mla.MLA_KV_BF16, device="cpu")
    kv = torch.zeros(2, 512, dtype=torch.bfloat16)
    pe = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises((ValueError, AttributeError)):
        mla.cache_append(object(), kv, pe, [0, 1])


def _imports(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_product_code_never_touches_the_oracle():
    py = [os.path.join(PKG, f) for f in os.listdir(PKG) if f.endswith(".py")]
    assert py
    for path in py:
        mods = list(_imports(path))
        assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), (path, mods)
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f), errors="replace").read()
        assert "mla_oracle" not in text and "orc_" not in text, f
    # and the oracle neither imports the package nor includes or loads its code
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        path = os.path.join(ROOT, "oracle", f)
        if f.endswith(".py"):
            mods = list(_imports(path))
            assert not any(m.startswith("mla_latent_kv_07_gb300") for m in mods), (f, mods)
            assert "libmla" not in open(path).read(), f
        elif f.endswith((".c", ".h")):
            incl = [ln for ln in open(path) if ln.lstrip().startswith("#include")]
            assert not any("csrc" in ln or "mla.h" in ln or ".cuh" in ln for ln in incl), (f, incl)
