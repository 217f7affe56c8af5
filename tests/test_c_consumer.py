"""The C ABI from C: include/moe.h compiles as strict C99 and a C program links
against libmoe.so and gets host-side answers (workspace sizes, validation
errors, names) without touching a GPU."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "tests", "_build")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

static int fails = 0;
#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); ++fails; } } while (0)

int main(void) {
  moe_config_t glm = {6144, 2048, 256, 8, 8, 4, 2.5f, 1, 2048, 32, 512, MOE_W_INT4};
  moe_config_t bad = glm, row8 = glm;
  moe_layer_t* h = (moe_layer_t*)1;
  int32_t flags = 0;
  bad.group_size = 64;
  row8.group_size = 0; /* one scale a row */
  row8.weight_format = MOE_W_INT8;
  /* a valid config has a workspace, an invalid one has none */
  CHECK(moe_workspace_bytes(&glm) > 0);
  CHECK(moe_workspace_bytes(&row8) == moe_workspace_bytes(&glm));
  CHECK(moe_workspace_bytes(&bad) == 0);
  CHECK(moe_workspace_bytes(NULL) == 0);
  /* argument errors come back before any CUDA call */
  CHECK(moe_layer_create(&bad, NULL, &h) == MOE_ERR_UNSUPPORTED && h == NULL);
  CHECK(strlen(moe_last_error(NULL)) > 0);
  CHECK(moe_layer_create(&glm, NULL, &h) == MOE_ERR_INVALID_ARG && h == NULL);
  CHECK(moe_forward(NULL, NULL, MOE_BF16, 1, NULL, NULL, 0.0f, 0, NULL, NULL) ==
        MOE_ERR_INVALID_ARG);
  CHECK(moe_route(NULL, NULL, MOE_F32, 1, NULL, 0.0f, NULL, NULL) == MOE_ERR_INVALID_ARG);
  CHECK(moe_device_status(NULL, &flags) == MOE_ERR_INVALID_ARG);
  CHECK(moe_selftest_bounded_wait(2, &flags) == MOE_ERR_INVALID_ARG);
  CHECK(moe_selftest_desync(NULL) == MOE_ERR_INVALID_ARG);
  CHECK(moe_trace_phase_name(0) != NULL && moe_trace_phase_name(-1) == NULL);
  moe_destroy(NULL);
  {
    /* the expert tier's residency policy is plain host code: 8 experts,
       4 slots, one of them for the hot store, calls of up to 2 experts */
    moe_slot_cache_t* c = NULL;
    moe_slot_cache_stats_t st;
    int32_t a[2] = {3, 5}, b[2] = {6, 7}, d[2] = {5, 1}, slot[2], kind[2], where[8];
    uint64_t uses[8];
    moe_tier_t* t = (moe_tier_t*)1;
    moe_tier_config_t tc = {4, 0};
    CHECK(moe_slot_cache_create(8, 4, 1, 2, &c) == MOE_OK && c != NULL);
    CHECK(moe_slot_cache_admit(c, a, 2, slot, kind) == MOE_OK);
    CHECK(slot[0] == 0 && slot[1] == 1 && kind[0] == 2 && kind[1] == 2);
    CHECK(moe_slot_cache_admit(c, d, 2, slot, kind) == MOE_OK);
    CHECK(slot[0] == 1 && kind[0] == 1 && slot[1] == 2 && kind[1] == 2);
    CHECK(moe_slot_cache_admit(c, b, 2, slot, kind) == MOE_OK);
    CHECK(slot[0] == 3 && slot[1] == 0); /* expert 3 (oldest use) was evicted */
    CHECK(moe_slot_cache_query(c, &st, where, uses) == MOE_OK);
    CHECK(st.misses == 5 && st.hits_lru == 1 && st.evictions == 1 && st.n_resident == 4);
    CHECK(where[3] == -1 && where[7] == 0 && uses[5] == 2);
    a[1] = 3;
    a[0] = 3; /* repeated id: refused, nothing changed */
    CHECK(moe_slot_cache_admit(c, a, 2, slot, kind) == MOE_ERR_INVALID_ARG);
    CHECK(moe_slot_cache_repin(NULL, 1) == -1);
    moe_slot_cache_destroy(c);
    /* the tier's checks come before any CUDA call: NULL weights, and 4
       slots where 512 tokens of top-8 need all 256 experts to fit */
    CHECK(moe_tier_create(&glm, NULL, &tc, &t) == MOE_ERR_INVALID_ARG && t == NULL);
    {
      moe_weights_t w;
      memset(&w, 0, sizeof(w));
      t = (moe_tier_t*)1;
      CHECK(moe_tier_create(&glm, &w, &tc, &t) == MOE_ERR_INVALID_ARG && t == NULL);
      CHECK(strstr(moe_last_error(NULL), "n_slots") != NULL);
    }
    moe_tier_destroy(NULL);
  }
  printf("%s\n", fails ? "failed" : "ok");
  return fails != 0;
}
"""


@pytest.fixture(scope="module")
def lib():
    from int4_routed_expert_gb300 import build as b
    return b.build()


def test_header_is_strict_c99_and_links(lib):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, "consumer.c")
    exe = os.path.join(OUT, "consumer")
    with open(src, "w") as f:
        f.write(PROGRAM)
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), src, "-o", exe, "-L", libdir, "-lmoe",
                    f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
    for p in (src, exe):
        os.remove(p)
