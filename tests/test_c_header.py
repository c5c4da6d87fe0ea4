"""The boundary is a C ABI: include/gma.h compiles as C99 and a C program links
against libgma.so and calls it (host-side paths only, no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from gaussian_mixture_sequence_gb300 import build as gbuild
from gaussian_mixture_sequence_gb300 import gma

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "gma.h"

int main(void)
{
    gma_shape s;
    memset(&s, 0, sizeof s);
    s.B = 2; s.H = 3; s.N = 100; s.d_route = 64; s.d_v = 64; s.K = 128; s.chunk = 0; s.eps = 1e-6f;
    s.x_dtype = GMA_F32; s.v_dtype = GMA_F32; s.gemm_dtype = GMA_F32;
    size_t need = gma_workspace_size(&s, GMA_OP_CAUSAL);
    if (need == 0) return 10;
    if (gma_workspace_size(&s, GMA_OP_CAUSAL_HOST) <= need) return 11;
    gma_params p = {0, 0, 0};
    /* a null shape, null parameters, a short workspace: rejected on the host */
    if (gma_forward_causal(NULL, p, 0, 0, 0, NULL, NULL, NULL, NULL, 0, NULL) != GMA_ERR_INVALID_ARG) return 12;
    if (gma_forward_bidir(&s, p, 0, 0, 0, NULL, NULL, 0, NULL) != GMA_ERR_INVALID_ARG) return 13;
    s.d_route = 48;
    if (gma_workspace_size(&s, GMA_OP_CAUSAL) != 0) return 14;
    if (strcmp(gma_status_string(GMA_OK), gma_status_string(GMA_ERR_CUDA)) == 0) return 15;
    if (strcmp(gma_last_cuda_error(), "cudaSuccess") != 0) return 16;
    printf("ok %zu\n", need);
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    gbuild.build()
    return gma.library_path()


def test_header_is_c99_and_links(tmp_path, lib_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_gma.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_gma"
    libdir = os.path.dirname(lib_path)
    name = os.path.basename(lib_path)[3:-3]   # libgma.so -> gma
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                           "-L", libdir, "-l" + name, "-Wl,-rpath," + libdir])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")
    shape = gma.Shape.make(2, 3, 100, 64, 64, 128)
    assert int(r.stdout.split()[1]) == gma.gma_workspace_size(shape, gma.OP_CAUSAL)
