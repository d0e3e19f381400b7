"""The C ABI library builds, loads and exports every entry point include/gpt2.h declares;
host-side argument checks (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from step_gpt_train_03_b300 import build
    build.build()
    from step_gpt_train_03_b300 import gpt2lib
    return gpt2lib


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(gpt2_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 25
    cdll = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in names if not hasattr(cdll, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert not [n for n in names if n not in lib.SIGNATURES]


def test_workspace_size_and_validation(lib):
    from step_gpt_train_03_b300 import synth
    n32 = lib.workspace_bytes(synth.TINY, 2, 32, "fp32")
    n16 = lib.workspace_bytes(synth.TINY_HS64, 2, 32, "bf16")
    assert n32 > 0 and n16 > 0
    # bf16 runs attention on the tensor cores, whose kernels take head size 64 only
    with pytest.raises(lib.GPT2Error) as e:
        lib.workspace_bytes(synth.TINY, 2, 32, "bf16")
    assert e.value.status == 8
    big = lib.workspace_bytes(synth.GPT2_124M, 16, 1024, "bf16")
    assert 5e9 < big < 40e9
    bad = synth.ModelShape(32, 512, 500, 2, 4, 64)          # Vp < V
    with pytest.raises(lib.GPT2Error) as e:
        lib.workspace_bytes(bad, 2, 32, "fp32")
    assert e.value.status == 1
    with pytest.raises(lib.GPT2Error):
        lib.workspace_bytes(synth.TINY, 2, 64, "fp32")       # T > max_seq_len
    with pytest.raises(lib.GPT2Error):
        lib.workspace_bytes(synth.ModelShape(32, 512, 512, 2, 3, 64), 2, 32, "fp32")   # C % NH


def test_strerror_names_every_status(lib):
    for st in range(len(lib.STATUS)):
        assert lib.lib.gpt2_strerror(st).decode() != "unknown status"
