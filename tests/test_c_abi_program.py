"""include/aq.h as a C user sees it: a C99 program (and the same source as
C++) that includes only the header, links libaq.so and calls the entry points
that need no device: version and status strings, the argument validation that
runs before any CUDA call, and the host packing and quantization utilities
checked against values worked out by hand from the format."""
import os
import shutil
import subprocess

import pytest

from affine_bit_quantized_gb300 import _build

PROGRAM = r"""
#include "aq.h"
#include <stdio.h>
#include <string.h>

int main(void) {
    /* a 64 KiB-aligned fake device address: validation never dereferences it */
    void *const fake = (void *)0x10000;
    const uint32_t *const fake_w = (const uint32_t *)0x10000;
    aq_status st;
    uint8_t codes[64];
    uint32_t packed[8];
    float w[64];
    uint32_t wp[8];
    uint16_t s = 0, b = 0;
    int k;

    if (aq_version() <= 0) return 10;
    if (strlen(aq_status_string(AQ_OK)) == 0 || strlen(aq_status_string(AQ_ERR_BAD_INDEX)) == 0) return 11;

    /* rejected before anything is enqueued */
    st = aq_matmul_bf16(fake, fake_w, fake, fake, fake, 1, 8, 64, 32, 4, NULL);
    if (st != AQ_ERR_UNSUPPORTED) return 12;                        /* group size 32 */
    st = aq_matmul_bf16(NULL, NULL, NULL, NULL, fake, 1, 8, 64, 64, 4, NULL);
    if (st != AQ_ERR_INVALID_ARG) return 13;                        /* null inputs */
    st = aq_matmul_bf16(fake, fake_w, fake, fake, fake, 1, 8, 96, 64, 4, NULL);
    if (st != AQ_ERR_INVALID_ARG) return 14;                        /* K not a multiple of 64 */
    st = aq_matmul_bf16((char *)fake + 2, fake_w, fake, fake, fake, 1, 8, 64, 64, 4, NULL);
    if (st != AQ_ERR_ALIGNMENT) return 15;                          /* x not 16-byte aligned */
    st = aq_matmul_bf16_ex(fake, fake_w, fake, fake, fake, 1, 8, 64, 64, 4, 7, 0u, NULL);
    if (st != AQ_ERR_INVALID_ARG) return 16;                        /* unknown kernel */

    /* codes 0..15 twice along k: word 0 holds k = 0..7 lowest nibble first */
    for (k = 0; k < 64; ++k) codes[k] = (uint8_t)(k & 15);
    if (aq_pack_ref(codes, 1, 64, 4, packed) != AQ_OK) return 20;
    if (packed[0] != 0x76543210u || packed[1] != 0xFEDCBA98u || packed[7] != 0xFEDCBA98u) return 21;
    codes[3] = 16;                                                  /* out of range for 4 bits */
    if (aq_pack_ref(codes, 1, 64, 4, packed) == AQ_OK) return 22;

    /* w = k mod 16: min 0, max 15, so scale = 15/15 = 1 (bf16 0x3F80), bias 0, q = w */
    for (k = 0; k < 64; ++k) w[k] = (float)(k % 16);
    if (aq_quantize_ref(w, 1, 64, 64, 4, wp, &s, &b) != AQ_OK) return 30;
    if (s != 0x3F80u || b != 0u) return 31;
    if (wp[0] != 0x76543210u || wp[1] != 0xFEDCBA98u) return 32;

    printf("ok\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    _build.build_library()
    return os.path.dirname(_build.LIB)


@pytest.mark.parametrize("compiler,flags", [
    ("gcc", ["-x", "c", "-std=c99"]),
    ("g++", ["-x", "c++", "-std=c++17"]),
])
def test_header_compiles_links_and_runs(tmp_path, lib_dir, compiler, flags):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    src = tmp_path / "use_aq.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_aq"
    cmd = [compiler, *flags, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", _build.INCLUDE, str(src),
           "-x", "none", "-L", lib_dir, "-laq", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
