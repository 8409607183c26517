"""Checked mode's range arithmetic and switch, on the CPU.

The extent test behind MOER_EEXTENT (`csrc/extent.h`, plain C++) is compiled
with g++ and driven with a made-up allocation table standing in for the
driver's address-range query: a buffer passes only when [p, p + bytes) lies
inside the one allocation that holds p, with no wrap-around at the top of
the address space; NULL or empty extents are skipped; the first failing
argument is reported.  The process-wide switch is pure host state and is
read back through the C ABI without touching a GPU.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "moe_expert_routing_top_gb300", "csrc")

DRIVER = r"""
#include <cstdint>
#include <cstdio>
#include "extent.h"

struct Alloc { uintptr_t base; size_t size; };
static const Alloc table[] = {{0x10000, 0x1000}, {0x20000, 0x100}, {UINTPTR_MAX - 0xFF, 0x100}};
static int queries = 0;

static bool fake_range(uintptr_t p, uintptr_t* base, size_t* size) {
  ++queries;
  for (const Alloc& a : table)
    if (p >= a.base && p - a.base < a.size) { *base = a.base; *size = a.size; return true; }
  return false;
}

#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)
static const void* P(uintptr_t a) { return reinterpret_cast<const void*>(a); }

int main() {
  using moer::extent_within;
  // the allocation itself, exactly
  CHECK(extent_within(0x10000, 0x1000, 0x10000, 0x1000));
  CHECK(!extent_within(0x10000, 0x1001, 0x10000, 0x1000));
  // a tail piece, up to the last byte
  CHECK(extent_within(0x10FFF, 1, 0x10000, 0x1000));
  CHECK(!extent_within(0x10FFF, 2, 0x10000, 0x1000));
  CHECK(extent_within(0x11000, 0, 0x10000, 0x1000));
  // before the base, past the end
  CHECK(!extent_within(0xFFFF, 1, 0x10000, 0x1000));
  CHECK(!extent_within(0x11001, 0, 0x10000, 0x1000));
  // a huge extent cannot wrap around to pass
  CHECK(!extent_within(0x10010, SIZE_MAX, 0x10000, 0x1000));
  CHECK(!extent_within(UINTPTR_MAX - 0x10, 0x20, UINTPTR_MAX - 0xFF, 0x100));
  CHECK(extent_within(UINTPTR_MAX - 0x10, 0x11, UINTPTR_MAX - 0xFF, 0x100));

  // lists: NULL and empty extents are skipped without a query
  queries = 0;
  CHECK(moer::first_bad_extent({{nullptr, 100}, {P(0x10000), 0}}, fake_range) == -1 && queries == 0);
  CHECK(moer::first_bad_extent({{P(0x10000), 0x1000}, {P(0x20000), 0x100}}, fake_range) == -1);
  // the first failing argument is reported
  CHECK(moer::first_bad_extent({{P(0x10000), 0x1000}, {P(0x20080), 0x81}, {P(0x5), 1}}, fake_range) == 1);
  // a pointer in no allocation fails
  CHECK(moer::first_bad_extent({{P(0x10000), 1}, {nullptr, 8}, {P(0x30000), 1}}, fake_range) == 2);
  // an extent that starts in one allocation and runs into the next one fails
  CHECK(moer::first_bad_extent({{P(0x10F00), 0x10200}}, fake_range) == 0);
  std::printf("ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not available")
def test_extent_arithmetic(tmp_path):
    src = tmp_path / "extent_test.cpp"
    exe = tmp_path / "extent_test"
    src.write_text(DRIVER)
    subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr


def test_switch_round_trip():
    nat = pytest.importorskip("moe_expert_routing_top_gb300._native")
    before = nat.moer_extent_checks()
    try:
        nat.moer_set_extent_checks(True)
        assert nat.moer_extent_checks() is True
        nat.moer_set_extent_checks(False)
        assert nat.moer_extent_checks() is False
    finally:
        nat.moer_set_extent_checks(before)
    assert nat.STATUS[8] == "MOER_EEXTENT"
    assert "checked mode" in nat.moer_status_str(8)


def test_null_is_not_a_buffer():
    nat = pytest.importorskip("moe_expert_routing_top_gb300._native")
    assert nat.moer_buffer_holds(None, 16) is False
