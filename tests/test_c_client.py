"""The C ABI used from plain C (tests/c_client/mosaic_client.c): on the CPU the client must compile
as C11 against include/mosaic.h and link against libmosaic.so; on a GB300 it runs a chunked
mask-only logits call and checks every element against exact integer arithmetic."""
import os
import shutil
import subprocess

import pytest

from masked_token_lm_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "mosaic_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_client(out_dir):
    if not os.path.exists(mbuild.LIB):
        mbuild.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(out_dir, "mosaic_client")
    libdir = os.path.dirname(mbuild.LIB)
    cudalib = os.path.join(CUDA, "lib64")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"), SRC,
           "-o", exe, "-L", libdir, "-lmosaic", "-L", cudalib, "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}:{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(compile_client(str(tmp_path)))


@pytest.mark.gpu
def test_c_client_runs_exact(tmp_path):
    exe = compile_client(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "elements exact over 3 chunks" in r.stdout
    for line in ("csr bf16: 312000 elements exact", "sampling: 300 tokens exact",
                 "noalloc: bit for bit over 3 chunks", "min_chunk_rows: 100 x 3"):
        assert line in r.stdout, r.stdout
