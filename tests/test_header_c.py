"""The C ABI header stands on its own: it compiles as C99 (pedantic, warnings as errors) and as C++17,
and a C program that includes it links against libkvq.so and finds every entry point by name."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_compiles(lang, std, tmp_path):
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    r = subprocess.run([cc, "-fsyntax-only", f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-x", lang,
                        HEADER], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_every_entry_point(tmp_path):
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("no host compiler")
    from attention_group_quantized_gb300 import kvq
    lib = kvq.LIB_PATH
    if not os.path.exists(lib):
        pytest.skip("libkvq.so not built")
    names = [n for n in kvq.EXPORTS if n != "kvq_status_str"]
    src = tmp_path / "use.c"
    src.write_text('#include "kvq.h"\n#include <stdio.h>\nint main(void) {\n'
                   '  void* p[] = {' + ", ".join(f"(void*){n}" for n in names) + '};\n'
                   '  printf("%s %d\\n", kvq_status_str(KVQ_ERR_WORKSPACE), (int)(sizeof(p) / sizeof(p[0])));\n'
                   '  return 0;\n}\n')
    exe = tmp_path / "use"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), lib,
                        f"-Wl,-rpath,{os.path.dirname(lib)}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split()[-1] == str(len(names))
