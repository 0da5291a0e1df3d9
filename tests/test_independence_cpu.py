"""The oracle and the product share no code: neither imports the other, and
the seeded input generators (the one module both sides use) import neither.
Also: the product's sources never read anything under oracle/ at build time."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            if node.level:  # relative: stays inside its own package
                continue
            out.add((node.module or "").split(".")[0])
    return out


def _py_files(sub):
    for dp, _, fs in os.walk(os.path.join(ROOT, sub)):
        if "__pycache__" in dp:
            continue
        for f in fs:
            if f.endswith(".py"):
                yield os.path.join(dp, f)


def test_oracle_does_not_import_the_library():
    for p in _py_files("oracle"):
        assert "top_routing_dispatch_gb300" not in _imports(p), p


def test_library_does_not_import_the_oracle():
    for p in _py_files("top_routing_dispatch_gb300"):
        assert "oracle" not in _imports(p), p


def test_input_generators_import_neither():
    for p in _py_files("workloads"):
        imps = _imports(p)
        assert "oracle" not in imps and "top_routing_dispatch_gb300" not in imps, p


def test_cuda_sources_include_nothing_from_the_oracle():
    csrc = os.path.join(ROOT, "top_routing_dispatch_gb300", "csrc")
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h")):
            for line in open(os.path.join(csrc, f)):
                if line.lstrip().startswith("#include"):
                    assert "oracle" not in line, (f, line)


def test_missing_library_fails_loudly(monkeypatch):
    """No CPU fallback: without the built library every entry point raises."""
    import pytest
    from top_routing_dispatch_gb300 import _lib, api
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmoe_gb300.so"))
    monkeypatch.setattr(_lib, "_LIB", None)
    with pytest.raises(ImportError):
        _lib.load()
    desc = _lib.LayerDesc(n=8, H=256, I=128, E=8, K=2, dtype=1, norm_topk_prob=0)
    with pytest.raises(ImportError):
        api.moe_backward_workspace_size(desc)
