"""Static import rules, checked by parsing the sources (no execution).

* the oracle imports only the standard library and numpy (and itself);
* the library package never imports the oracle, so no product path can
  route through it.
"""
import ast
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name.split(".")[0], 0
        elif isinstance(node, ast.ImportFrom):
            yield (node.module or "").split(".")[0], node.level


def _py_files(folder):
    for dp, _, fns in os.walk(os.path.join(ROOT, folder)):
        for fn in fns:
            if fn.endswith(".py"):
                yield os.path.join(dp, fn)


def test_oracle_imports_only_stdlib_and_numpy():
    allowed = set(sys.stdlib_module_names) | {"numpy", "__future__"}
    files = list(_py_files("oracle"))
    assert files
    for f in files:
        for mod, level in _imports(f):
            if level > 0:
                continue
            assert mod in allowed, f"{f} imports {mod}"


def test_library_never_imports_oracle():
    files = list(_py_files("serving_slot_mapping_gb300"))
    assert files
    for f in files:
        for mod, level in _imports(f):
            assert mod != "oracle", f"{f} imports the oracle"
        src = open(f).read()
        assert "import oracle" not in src and "from oracle" not in src
