"""The float64 oracle and the CUDA path share no code: no source of the package imports or
includes anything under oracle/, and no oracle source imports the package or includes its
headers.  The seeded input generators (selective_scan_mamba_gb300/synth.py) are the one
module both sides use; they import neither side.  Static checks, no GPU."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "selective_scan_mamba_gb300")
ORACLE = os.path.join(ROOT, "oracle")
SOURCE_EXT = (".py", ".c", ".h", ".cu", ".cuh", ".cpp")


def _sources(top):
    for d, _, files in os.walk(top):
        if "__pycache__" in d:
            continue
        for f in files:
            if f.endswith(SOURCE_EXT):
                yield os.path.join(d, f)


def _imports(path):
    text = open(path, encoding="utf-8").read()
    py = re.findall(r"^\s*(?:from\s+(\S+)\s+import|import\s+([\w.]+))", text, re.M)
    inc = re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', text, re.M)
    return [a or b for a, b in py], inc


def test_package_never_imports_the_oracle():
    for path in _sources(PKG):
        mods, incs = _imports(path)
        assert not [m for m in mods if m.split(".")[0] == "oracle"], path
        assert not [i for i in incs if "oracle" in i], path


def test_oracle_never_imports_the_package():
    for path in _sources(ORACLE):
        mods, incs = _imports(path)
        assert not [m for m in mods if m.split(".")[0] in ("selective_scan_mamba_gb300", "bench")
                    or m.startswith(".")], path
        assert not [i for i in incs if "ssmscan" in i or "csrc" in i or i.endswith(".cuh")], path


def test_input_generators_import_neither_side():
    mods, incs = _imports(os.path.join(PKG, "synth.py"))
    assert not incs
    assert not [m for m in mods if m.split(".")[0] in ("oracle", "selective_scan_mamba_gb300")
                or m.startswith(".")]
