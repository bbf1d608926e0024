"""Static checks (CPU) that the oracle and the CUDA path share no code: the
package never imports the oracle, the oracle never imports the package, neither
side's C/CUDA sources include the other's, and the only places outside tests/
that touch the oracle are bench.py's CPU-baseline and reference legs and
__graft_entry__'s build() and smoke()."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp4_sparse_attention_tma_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def imported_modules(path):
    """(module name, enclosing top-level function or None) of every import."""
    tree = ast.parse(open(path).read(), filename=path)
    out = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = func
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) and func is None:
                f = child.name
            if isinstance(child, ast.Import):
                out.extend((a.name, f) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                out.append(((child.module or "") if child.level == 0 else "." + (child.module or ""), f))
            visit(child, f)

    visit(tree, None)
    return out


def top(name):
    return name.split(".")[0]


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        for mod, _ in imported_modules(path):
            assert top(mod) != "oracle", (path, mod)


def test_oracle_never_imports_the_package():
    for path in glob.glob(os.path.join(ORACLE, "*.py")):
        for mod, _ in imported_modules(path):
            assert top(mod) not in ("fp4_sparse_attention_tma_gb300", "bench", "tests"), (path, mod)


def test_c_sources_include_nothing_of_the_other_side():
    for path in glob.glob(os.path.join(ORACLE, "*.c")) + glob.glob(os.path.join(ORACLE, "*.h")):
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert "/" not in inc and not inc.startswith("idx"), (path, inc)
    for path in glob.glob(os.path.join(PKG, "csrc", "*")):
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert "oracle" not in inc, (path, inc)


def test_oracle_users_outside_tests():
    allowed = {"bench.py": {"cpu_baseline", "run_reference"},
               "__graft_entry__.py": {"build", "smoke"}}
    for name, funcs in allowed.items():
        for mod, func in imported_modules(os.path.join(ROOT, name)):
            if top(mod) == "oracle":
                assert func in funcs, (name, func)
