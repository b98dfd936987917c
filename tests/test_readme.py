"""The README's quick starts stay in step with the interfaces: the C example
compiles and links against the library (no GPU needed), the Python example
is valid Python that names only what the binding exports."""
import ast
import os
import re
import shutil
import subprocess

import pytest

import dsa_sparse_attention_score_gb300 as dsa
from dsa_sparse_attention_score_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
README = open(os.path.join(ROOT, "README.md")).read()
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_example_compiles_and_links(tmp_path):
    if not shutil.which("gcc") or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    lib = dsa_build.build()
    (src,) = re.findall(r"```c\n(.*?)```", README, flags=re.S)
    path = tmp_path / "decode.c"
    path.write_text(src)
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", str(path), "-I" + os.path.join(ROOT, "include"),
                        "-I" + os.path.join(CUDA, "include"), "-L" + os.path.dirname(lib), "-ldsa_gb300",
                        "-L" + os.path.join(CUDA, "lib64"), "-lcudart", "-o", str(tmp_path / "decode")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_python_example_names_only_exported_calls():
    (src,) = re.findall(r"```python\n(.*?)```", README, flags=re.S)
    tree = ast.parse(src)
    used = {n.attr for n in ast.walk(tree) if isinstance(n, ast.Attribute)
            and isinstance(n.value, ast.Name) and n.value.id == "dsa"}
    assert used and all(hasattr(dsa, name) for name in used), used
