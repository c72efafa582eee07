"""include/kvc.h is a C header: a C99 translation unit that includes it builds
with warnings as errors, links against libsinkwin.so, and sees the same
struct layout, buffer sizes and argument checks as the library (no GPU
work: only calls that validate and return)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "sink_short_window_sinkwin_b300")

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "kvc.h"

int main(void) {
  kvc_cache c;
  memset(&c, 0, sizeof c);
  c.heads = 12; c.head_dim = 128; c.tokens_per_frame = 1560; c.chunk_frames = 3;
  c.window_chunks = 3; c.dtype = KVC_BF16;
  if (kvc_sizeof_cache() != sizeof(kvc_cache)) { puts("layout"); return 1; }
  if (kvc_cache_bytes(&c, 0) != (size_t)18720 * 12 * 128 * 2) { puts("bytes"); return 2; }
  if (kvc_init(&c) != KVC_EINVAL) { puts("null buffers accepted"); return 3; }
  c.k = (void*)0x10000000; c.v = (void*)0x20000000; c.dev_ws = (int32_t*)0x30000000;
  if (kvc_init(&c) != KVC_OK) { puts("init"); return 4; }
  if (kvc_evict(&c, 0, NULL) != KVC_ESTATE) { puts("sink evict"); return 5; }
  if (sinkwin_attn(&c, NULL, NULL, 0, 0.1f, NULL) != KVC_OK) { puts("tq = 0"); return 6; }
  if (sinkwin_attn(&c, (void*)0x40000000, (void*)0x50000000, 8, 0.1f, NULL) != KVC_ESTATE) {
    puts("empty sink"); return 7;
  }
  printf("ok %s\n", kvc_status_string(KVC_ESTATE));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_compiles_as_c_and_links(tmp_path):
    src = tmp_path / "use_kvc.c"
    src.write_text(C_SRC)
    exe = tmp_path / "use_kvc"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", LIBDIR, "-lsinkwin", f"-Wl,-rpath,{LIBDIR}"],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok ")
