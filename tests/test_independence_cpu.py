"""The oracle and the CUDA path share no code, and the product has no fallback.

* oracle/ includes no header of the library and imports nothing of the package;
  the package and its CUDA sources never import, link or name the oracle;
* without the built library every binding call raises instead of computing
  anything on the CPU.
"""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fsdp_sharded_mixed_flatparameter_gb300")


def _files(top, exts):
    for d, _, fs in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_oracle_uses_nothing_of_the_library():
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    includes = re.findall(r'#include\s*[<"]([^>"]+)[>"]', src)
    assert includes and all(not i.startswith(("zero_", "kernels", "common", "reduce", "table", "adam")) for i in includes), includes
    py = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert "fsdp_sharded_mixed_flatparameter_gb300" not in py and "zero_shard" not in py


def test_library_uses_nothing_of_the_oracle():
    for f in list(_files(PKG, (".py", ".cu", ".cuh", ".h"))) + [os.path.join(ROOT, "include", "zero_shard.h")]:
        text = open(f).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
        assert "orc_" not in text and "liboracle" not in text, f


def test_binding_raises_without_the_built_library():
    code = (
        "import fsdp_sharded_mixed_flatparameter_gb300.build as b\n"
        "b.LIB = '/nonexistent/libzeroshard.so'\n"
        "from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs\n"
        "zs._lib = None\n"
        "try:\n"
        "    zs.zero_shard_range(10, 2, 0)\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    print('computed without the library')\n")
    p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0 and "raised:" in p.stdout and "not built" in p.stdout, p.stdout + p.stderr
