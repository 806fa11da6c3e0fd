"""Structural guards on the CPU: the product package and the CUDA library never reach the
oracle (and the oracle never reaches them), and the profiles' validity stamp follows the device
code only."""
import os
import re

from exact_attention_50_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "exact_attention_50_gb300")


def _files(top, exts):
    for dirpath, _, names in os.walk(top):
        if "__pycache__" in dirpath or "_build" in dirpath:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(dirpath, n)


def test_product_does_not_reach_the_oracle():
    for path in _files(PKG, (".py", ".cu", ".cuh", ".h")):
        text = open(path).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), path
        assert "attn_oracle" not in text and "liboracle" not in text, path


def test_oracle_does_not_reach_the_product():
    for path in _files(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")):
        text = open(path).read()
        assert "exact_attention_50_gb300" not in text and "attn_gb300" not in text, path


def test_code_stamp_ignores_comments_and_host_code_but_not_device_code():
    real = lambda path: open(path).read()
    base = B.code_stamp(real)
    fwd = os.path.join(B.CSRC, "fwd_tc.cuh")
    api = os.path.join(B.CSRC, "attn_api.cu")

    def with_change(target, change):
        return lambda path: change(real(path)) if path == target else real(path)

    assert B.code_stamp(with_change(fwd, lambda t: "// a note\n/* another */\n\n" + t)) == base
    assert B.code_stamp(with_change(api, lambda t: t + "\nint attn_host_helper_for_the_test() { return 1; }\n")) == base
    assert B.code_stamp(with_change(fwd, lambda t: t.replace("kRescaleLog2 = 8.0f", "kRescaleLog2 = 7.0f"))) != base
    assert B.code_stamp(with_change(api, lambda t: t + "\n__device__ int g_extra_for_the_test;\n")) != base
