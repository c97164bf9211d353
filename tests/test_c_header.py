"""The boundary is a C ABI: include/nf4.h compiles as C11 (gcc, -Wall
-Werror) and a C program linked against libnf4.so calls it -- version,
status names, host-side argument checks (fp32 accepted by the linear entry
points), and the workspace rule -- with no GPU and no Python in between."""
import os
import shutil
import subprocess

import pytest

from nf4_weight_quantized_quantize_gb300 import build as nf4_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "nf4.h"

int main(void) {
    int bad = 0;
    void* fake = (void*)(1 << 20);   /* 16-byte aligned, never dereferenced: every call below fails validation */
    size_t ws = 0;
    if (nf4_version() < 100) bad |= 1;
    if (strcmp(nf4_status_string(NF4_ERR_DTYPE), "NF4_ERR_DTYPE") != 0) bad |= 2;
    if (nf4_quantize((const uint16_t*)fake, 127, NF4_BLOCK, (uint8_t*)fake, (float*)fake, 0) != NF4_ERR_SHAPE) bad |= 4;
    if (nf4_dequantize_ex((const uint8_t*)fake, (const float*)fake, 128, NF4_BLOCK, (nf4_dtype)7, fake, 0)
        != NF4_ERR_DTYPE) bad |= 8;
    if (nf4_linear((const uint16_t*)fake, 256, 96, (const uint8_t*)fake, (const float*)fake, 64, NF4_BLOCK,
                   (uint16_t*)fake, NULL, 0, NULL) != NF4_ERR_SHAPE) bad |= 16;
    if (nf4_linear_geglu_ex(fake, NF4_DTYPE_F16, 256, 128, (const uint8_t*)fake, (const float*)fake, 64, 32,
                            fake, NULL, 0, NULL) != NF4_ERR_BLOCKSIZE) bad |= 32;
    if (nf4_linear_workspace_size(16, 3840, 15360, &ws) != NF4_OK || ws == 0) bad |= 64;
    if (nf4_linear_workspace_size(2048, 3840, 15360, &ws) != NF4_OK || ws != 0) bad |= 128;
    /* fp32 is a compute dtype of the linear (tf32 tensor cores): accepted, and
       M = 0 enqueues nothing; a value outside nf4_dtype is refused */
    if (nf4_linear_ex(fake, NF4_DTYPE_F32, 0, 128, (const uint8_t*)fake, (const float*)fake, 64, NF4_BLOCK,
                      fake, NULL, 0, NULL) != NF4_OK) bad |= 256;
    if (nf4_linear_geglu_ex(fake, NF4_DTYPE_F32, 0, 128, (const uint8_t*)fake, (const float*)fake, 32,
                            NF4_BLOCK, fake, NULL, 0, NULL) != NF4_OK) bad |= 512;
    if (nf4_linear_ex(fake, (nf4_dtype)3, 0, 128, (const uint8_t*)fake, (const float*)fake, 64, NF4_BLOCK,
                      fake, NULL, 0, NULL) != NF4_ERR_DTYPE) bad |= 1024;
    /* every skinny workspace carries the counter header */
    if (nf4_linear_workspace_size(1, 64, 64, &ws) != NF4_OK || ws < NF4_WORKSPACE_HEADER_BYTES) bad |= 2048;
    printf("%d\n", bad);
    return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c_and_library_links_from_c(tmp_path):
    lib = nf4_build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), lib, f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "0", out.stdout + out.stderr
