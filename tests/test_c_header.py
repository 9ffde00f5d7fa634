"""The C ABI from plain C: include/usp.h compiles as C99 with warnings as
errors, a C program links against the library and gets the documented
host-side answers (version, status strings, head-count and empty-input
rules) without a GPU, and the header's struct size and field offsets equal
those of the Python binding's mirror of it."""
import ctypes
import os
import shutil
import subprocess

import pytest

from ulysses_sequence_attention_usp_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include "usp.h"

int main(void) {
  usp_dims d;
  void* fake = (void*)(uintptr_t)(1u << 20);  /* never dereferenced */
  usp_status s;
  if (usp_abi_version() != USP_ABI_VERSION) return 10;
  memset(&d, 0, sizeof d);
  d.S = 0; d.P = 4; d.Hq = 4; d.Hkv = 1; d.D = 64; d.causal = 1;
  s = usp_attn_fwd(&d, fake, fake, fake, (const int32_t*)fake, fake, (float*)fake, NULL);
  if (s != USP_ERR_HEADS_NOT_DIVISIBLE) return 11;
  d.P = 1;                                   /* one shard: any Hkv dividing Hq */
  s = usp_attn_fwd(&d, fake, fake, fake, (const int32_t*)fake, fake, (float*)fake, NULL);
  if (s != USP_OK) return 12;
  d.D = 96;
  if (usp_attn_fwd(&d, fake, fake, fake, (const int32_t*)fake, fake, (float*)fake, NULL)
      != USP_ERR_UNSUPPORTED) return 13;
  printf("%s\n", usp_status_string(USP_ERR_HEADS_NOT_DIVISIBLE));
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(usp_dims), offsetof(usp_dims, cu_seqlens),
         offsetof(usp_dims, n_docs), offsetof(usp_dims, causal), offsetof(usp_dims, scale),
         offsetof(usp_dims, zigzag));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_is_c99_and_links(tmp_path):
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    lib_dir = os.path.dirname(B.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    B.LIB_PATH, f"-Wl,-rpath,{lib_dir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    lines = out.stdout.strip().splitlines()
    assert "divisible" in lines[0]
    size, *offs = (int(x) for x in lines[1].split())
    T = B.usp_dims
    assert size == ctypes.sizeof(T)
    assert offs == [T.cu_seqlens.offset, T.n_docs.offset, T.causal.offset, T.scale.offset,
                    T.zigzag.offset]
