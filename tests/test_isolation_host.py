"""The product path and the oracle stay apart, checked on the source without a
GPU: the package neither imports nor links anything under oracle/; the oracle
uses nothing of the package; in bench.py only the CPU-baseline sampler imports
the oracle, and only the cpu_baseline leg and the reference arm call it; the
input generators hold no arithmetic of the layer; and the binding raises when
the CUDA library is missing instead of computing anything itself."""
import ast
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "transformer_gqa_attention_qkv_gb300")


def _imports(path):
    """Module names a Python file imports, anywhere in it."""
    with open(path) as f:
        tree = ast.parse(f.read(), path)
    names = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names += [a.name for a in node.names]
        elif isinstance(node, ast.ImportFrom) and node.module:
            names.append(node.module)
    return names


def test_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(PKG, "*.py"))
    assert files
    for path in files:
        bad = [m for m in _imports(path) if m == "oracle" or m.startswith("oracle.")]
        assert not bad, f"{os.path.basename(path)} imports {bad}"


def test_cuda_sources_do_not_include_or_name_oracle_files():
    files = glob.glob(os.path.join(PKG, "csrc", "*"))
    assert files
    for path in files:
        with open(path) as f:
            src = f.read()
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', src):
            assert "oracle" not in inc, f"{os.path.basename(path)} includes {inc}"
        assert "gqa_oracle" not in src and "liboracle" not in src, os.path.basename(path)


def test_build_script_compiles_no_oracle_source():
    with open(os.path.join(PKG, "build.py")) as f:
        src = f.read()
    assert "oracle" not in src


def test_oracle_uses_nothing_of_the_package():
    bad = [m for m in _imports(os.path.join(ROOT, "oracle", "__init__.py"))
           if m.startswith("transformer_gqa_attention_qkv_gb300")]
    assert not bad
    with open(os.path.join(ROOT, "oracle", "gqa_oracle.c")) as f:
        src = f.read()
    incs = re.findall(r'#include\s*[<"]([^>"]+)[>"]', src)
    assert all("gqa_attn" not in i and "csrc" not in i and "include/" not in i for i in incs), incs


def test_input_generators_hold_no_layer_arithmetic():
    path = os.path.join(PKG, "inputs.py")
    mods = _imports(path)
    assert not [m for m in mods if "oracle" in m or "binding" in m], mods
    with open(path) as f:
        src = f.read()
    # draws and shapes only: no softmax, normalisation, rotation or products of the layer
    for op in ("softmax", "rsqrt", "matmul", "einsum", ".cos(", ".sin(", "exp("):
        assert op not in src, op
    assert not re.search(r"[\w)\]][ \t]*@[ \t]*[\w(]", src), "matrix product in the input generators"


def _enclosing_functions(tree):
    """Map each node to the name of the innermost top-level or nested def holding it."""
    owner = {}

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            owner[child] = name
            visit(child, name)

    visit(tree, None)
    return owner


def test_bench_touches_the_oracle_only_in_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    with open(path) as f:
        tree = ast.parse(f.read(), path)
    owner = _enclosing_functions(tree)
    importers = {owner[n] for n in ast.walk(tree)
                 if isinstance(n, ast.Import) and any(a.name == "oracle" for a in n.names)}
    importers |= {owner[n] for n in ast.walk(tree)
                  if isinstance(n, ast.ImportFrom) and (n.module or "").startswith("oracle")}
    assert importers == {"cpu_oracle_sample"}, importers
    callers = {owner[n] for n in ast.walk(tree)
               if isinstance(n, ast.Call) and getattr(n.func, "id", None) == "cpu_oracle_sample"}
    # run_ours calls it once, after its GPU lines, for the cpu_baseline key; run_reference is the reference arm
    assert callers == {"run_ours", "run_reference"}, callers


def test_bench_cpu_baseline_leg_is_rank0_only():
    with open(os.path.join(ROOT, "bench.py")) as f:
        src = f.read()
    i = src.index("cpu_oracle_sample(cfg, args.cpu_tokens")
    guard = src.rfind("if ", 0, i)
    assert "rank == 0" in src[guard:i] and "world == 1" in src[guard:i], src[guard:i]


def test_binding_raises_without_the_library(tmp_path, monkeypatch):
    import transformer_gqa_attention_qkv_gb300.binding as b
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "libgqa_attn.so"))
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        b.lib()
