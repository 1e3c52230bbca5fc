"""The C ABI as a plain C program sees it: include/pagedkv.h compiles as
strict C11, every declared entry point links against libpagedkv.so, and the
host block manager works through it (allocate, append, fork with
copy-on-write, tables, refcounts, free list, error status and message).
No GPU: only host calls are made."""
import os
import shutil
import subprocess

import pytest

from tests.libfixture import palib  # noqa: F401
from tests.test_abi import HEADER, declared_functions

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "paged_kv_cache_191_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "pagedkv.h"

typedef void (*any_fn)(void);
static const any_fn every_entry_point[] = {
%(table)s
};

#define CHECK(x) do { if (!(x)) { printf("FAIL line %%d: %%s\n", __LINE__, #x); return 1; } } while (0)

int main(void) {
  pa_alloc* a = NULL;
  int64_t slot, src, dst, n_tok;
  int32_t tab[8], nb, total, nfree, rc[4], fl[4], nfl;
  size_t i;
  for (i = 0; i < sizeof every_entry_point / sizeof every_entry_point[0]; ++i) CHECK(every_entry_point[i] != NULL);
  CHECK(pa_version() == 100);

  CHECK(pa_alloc_create(0, PA_BLOCK_SIZE, NULL, &a) == PA_ERR_INVALID && a == NULL);
  CHECK(pa_alloc_create(4, 15, NULL, &a) == PA_ERR_UNSUPPORTED);   /* only 16-token blocks are built */
  CHECK(strlen(pa_last_error()) > 0);
  CHECK(pa_alloc_create(4, PA_BLOCK_SIZE, NULL, &a) == PA_OK);

  CHECK(pa_alloc_seq(a, 1, 20) == PA_OK);                           /* blocks 0, 1 */
  CHECK(pa_append_slot(a, 1, &slot, &src, &dst) == PA_OK);          /* token 20: block 1, row 4 */
  CHECK(slot == 20 && src == -1 && dst == -1);
  CHECK(pa_fork(a, 1, 2) == PA_OK);                                 /* 2 shares blocks 0, 1 */
  CHECK(pa_append_slot(a, 2, &slot, &src, &dst) == PA_OK);          /* partial shared block: copy 1 -> 2 */
  CHECK(src == 1 && dst == 2 && slot == 2 * 16 + 5);
  CHECK(pa_block_table(a, 2, tab, 8, &nb, &n_tok) == PA_OK);
  CHECK(nb == 2 && tab[0] == 0 && tab[1] == 2 && n_tok == 22);
  CHECK(pa_alloc_stats(a, &total, &nfree, rc) == PA_OK);
  CHECK(total == 4 && nfree == 1 && rc[0] == 2 && rc[1] == 1 && rc[2] == 1 && rc[3] == 0);

  CHECK(pa_alloc_seq(a, 3, 33) == PA_ERR_OOM);                      /* needs 3 blocks, 1 free */
  CHECK(pa_alloc_stats(a, &total, &nfree, NULL) == PA_OK && nfree == 1);   /* unchanged */
  CHECK(pa_append_slot(a, 99, &slot, &src, &dst) == PA_ERR_NOT_FOUND);

  CHECK(pa_free_seq(a, 1) == PA_OK);                                /* block 1 freed, block 0 kept */
  CHECK(pa_free_list(a, fl, 4, &nfl) == PA_OK);
  CHECK(nfl == 2 && fl[0] == 3 && fl[1] == 1);                      /* FIFO: freed blocks go to the back */
  CHECK(pa_free_seq(a, 2) == PA_OK);
  CHECK(pa_alloc_stats(a, &total, &nfree, rc) == PA_OK);
  CHECK(nfree == 4 && rc[0] == 0 && rc[2] == 0);
  pa_alloc_destroy(a);
  printf("ok %%u entry points\n", (unsigned)(sizeof every_entry_point / sizeof every_entry_point[0]));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_plain_c_program_uses_the_abi(palib, tmp_path):
    names = declared_functions()
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM % {"table": ",\n".join(f"  (any_fn){n}" for n in names)})
    exe = tmp_path / "consumer"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER),
           str(src), "-o", str(exe), "-L", LIBDIR, "-lpagedkv", f"-Wl,-rpath,{LIBDIR}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == f"ok {len(names)} entry points"
