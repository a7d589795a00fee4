"""The oracle and the CUDA path share no code and do not import each other."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _imports(path):
    tree = ast.parse(open(path).read())
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def _py_files(d):
    for base, _, files in os.walk(os.path.join(ROOT, d)):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(base, f)


def test_oracle_does_not_import_product_or_workloads():
    for f in _py_files("oracle"):
        bad = _imports(f) & {"fp8_fine_grained_24_b300", "workloads", "torch", "ctypes"}
        assert not bad, (f, bad)


def test_product_does_not_touch_oracle():
    for f in _py_files("fp8_fine_grained_24_b300"):
        assert "oracle" not in _imports(f), f
    for base, _, files in os.walk(os.path.join(ROOT, "fp8_fine_grained_24_b300")):
        for f in files:
            if f.endswith((".cu", ".cuh", ".h", ".cpp", ".py")):
                assert "oracle" not in open(os.path.join(base, f)).read().replace("oracle-free", ""), f


def test_workloads_hold_no_method_arithmetic():
    src = open(os.path.join(ROOT, "workloads", "__init__.py")).read()
    for word in ("448", "e4m3", "float8", "amax", "matmul", "@"):
        assert word not in src.lower().replace("@dataclass", ""), word
