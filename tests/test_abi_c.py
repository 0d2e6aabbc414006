"""The C ABI from C: `tests/abi_consumer.c` includes `include/topk.h`, links
the built library and checks the host-side contract (workspace sizing, status
strings, validation status codes). It is compiled as strict C99 and once more
as C++17, so the header is checked in both languages. No GPU work."""

from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "abi_consumer.c")


@pytest.fixture(scope="module")
def lib_dir():
    from sparse_attention_top_row_gb300 import build as b
    b.build()
    import sparse_attention_top_row_gb300 as topk
    return os.path.dirname(topk.LIB_PATH)


@pytest.mark.parametrize("lang", ["c99", "c++17"])
def test_c_consumer(lib_dir, tmp_path, lang):
    cc = shutil.which("gcc" if lang == "c99" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    exe = str(tmp_path / f"abi_consumer_{lang.replace('+', 'p')}")
    cmd = [cc, f"-std={lang}", "-Wall", "-Wextra", "-Werror", "-pedantic"]
    if lang != "c99":
        cmd += ["-x", "c++"]
    cmd += [f"-I{os.path.join(ROOT, 'include')}", SRC, "-x", "none", f"-L{lib_dir}", "-ltopk",
            f"-Wl,-rpath,{lib_dir}", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok ")
