"""The per-context address cache behind moer_topk_signature_noalloc, on the CPU.

The no-alloc entry point keeps the device address of its fixed scratch array
per CUDA context, keyed on the context's unique ID.  This test compiles the
cache (a plain C++ header) with g++ and drives it with made-up context IDs
and a counting fake of the symbol look-up: a context looks up once; a
context created again (a new ID, as after cudaDeviceReset) never receives
the old context's address; a failed look-up is not cached; a full cache
replaces its oldest entry.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "moe_expert_routing_top_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <cstdint>
#include "ctx_cache.h"

static int lookups = 0;
static uintptr_t next_addr = 0x1000;
static bool fail_next = false;

static bool fake_lookup(void** p) {
  ++lookups;
  if (fail_next) { fail_next = false; return false; }
  *p = reinterpret_cast<void*>(next_addr);
  next_addr += 0x1000;
  return true;
}

#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

int main() {
  moer::CtxAddressCache<4> cache;
  // context 7: one look-up, then served from the cache
  void* a = cache.get(7, fake_lookup);
  CHECK(a == reinterpret_cast<void*>(0x1000) && lookups == 1);
  CHECK(cache.get(7, fake_lookup) == a && lookups == 1);
  // context 7 destroyed and created again: the new context has a new ID and
  // gets its own look-up, never the dead context's address
  void* b = cache.get(8, fake_lookup);
  CHECK(b != a && lookups == 2);
  CHECK(cache.get(8, fake_lookup) == b && lookups == 2);
  // a failed look-up returns nullptr and caches nothing
  fail_next = true;
  CHECK(cache.get(9, fake_lookup) == nullptr && lookups == 3);
  void* c = cache.get(9, fake_lookup);
  CHECK(c != nullptr && c != a && c != b && lookups == 4);
  CHECK(cache.size() == 3);
  // full: the oldest entry (context 7) is replaced, the others stay
  void* d = cache.get(10, fake_lookup);
  CHECK(cache.size() == 4 && lookups == 5);
  void* e = cache.get(11, fake_lookup);
  CHECK(e != nullptr && lookups == 6 && cache.size() == 4);
  CHECK(cache.get(8, fake_lookup) == b && cache.get(9, fake_lookup) == c);
  CHECK(cache.get(10, fake_lookup) == d && cache.get(11, fake_lookup) == e && lookups == 6);
  void* a2 = cache.get(7, fake_lookup);
  CHECK(a2 != a && lookups == 7);
  std::printf("OK\n");
  return 0;
}
"""


def test_ctx_cache_keys_on_context_id(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    src = tmp_path / "drv.cpp"
    src.write_text(DRIVER)
    exe = tmp_path / "drv"
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe), "-pthread"],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
