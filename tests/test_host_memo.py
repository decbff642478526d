"""The host-side memos of one-time launch set-up (csrc/host_memo.h), driven by a
plain C++ program on the CPU: a kernel's raised shared-memory limit and a
device array's address are remembered per device and per context, so a
second device, or a new context on the same device (as after
cudaDeviceReset), runs the set-up again, and concurrent host threads agree.
The same program checks the residency rule the fused decode launch applies
before it starts a grid whose blocks wait for one another."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_grouped_expert_moe_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "host_memo.h"
using namespace bgmoe;
#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)
int main() {
  SmemLimitMemo m;
  int calls = 0, last = 0;
  auto set = [&](int b) { ++calls; last = b; return 0; };
  CHECK(m.ensure(0, 7, 1000, set) == 0 && calls == 1 && last == 1000);
  CHECK(m.ensure(0, 7, 900, set) == 0 && calls == 1);      // smaller: already allowed
  CHECK(m.ensure(0, 7, 1000, set) == 0 && calls == 1);
  CHECK(m.ensure(1, 7, 900, set) == 0 && calls == 2);      // second device: set again
  CHECK(m.ensure(1, 7, 900, set) == 0 && calls == 2);
  CHECK(m.ensure(0, 7, 2000, set) == 0 && calls == 3);     // larger: raised
  CHECK(m.ensure(0, 8, 500, set) == 0 && calls == 4);      // new context on device 0
  CHECK(m.ensure(0, 8, 500, set) == 0 && calls == 4);
  CHECK(m.ensure(0, 0, 500, set) == 0 && calls == 5);      // unknown context: never memoised
  CHECK(m.ensure(0, 0, 500, set) == 0 && calls == 6);
  CHECK(m.ensure(99, 7, 500, set) == 0 && calls == 7);     // device index past the table
  int fails = 0;
  auto bad = [&](int) { ++fails; return 3; };
  CHECK(m.ensure(2, 7, 100, bad) == 3 && fails == 1);       // a failed set-up is not remembered
  CHECK(m.ensure(2, 7, 100, bad) == 3 && fails == 2);

  PointerMemo pm;
  int finds = 0;
  char a0, a1, a2;
  void* p = nullptr;
  auto f0 = [&](void** o) { ++finds; *o = &a0; return 0; };
  auto f1 = [&](void** o) { ++finds; *o = &a1; return 0; };
  auto f2 = [&](void** o) { ++finds; *o = &a2; return 0; };
  CHECK(pm.get(0, 7, &p, f0) == 0 && p == &a0 && finds == 1);
  CHECK(pm.get(0, 7, &p, f1) == 0 && p == &a0 && finds == 1);  // memoised
  CHECK(pm.get(1, 7, &p, f1) == 0 && p == &a1 && finds == 2);  // per device
  CHECK(pm.get(0, 9, &p, f2) == 0 && p == &a2 && finds == 3);  // new context: looked up again
  CHECK(pm.get(0, 9, &p, f0) == 0 && p == &a2 && finds == 3);

  // 8 threads racing on one fresh device: the set-up runs once and every
  // thread sees success.
  SmemLimitMemo mt;
  int tcalls = 0;
  std::vector<std::thread> th;
  std::vector<int> rc(8, -1);
  for (int i = 0; i < 8; ++i)
    th.emplace_back([&, i] { rc[i] = mt.ensure(3, 11, 4096, [&](int) { ++tcalls; return 0; }); });
  for (auto& t : th) t.join();
  CHECK(tcalls == 1);
  for (int r : rc) CHECK(r == 0);

  // the fused decode launch's residency rule: one block per SM on every SM
  CHECK(all_blocks_resident(1, 152, 152));
  CHECK(all_blocks_resident(2, 152, 304));
  CHECK(!all_blocks_resident(0, 152, 152));   // the block does not fit on an SM at all
  CHECK(!all_blocks_resident(1, 152, 153));   // more blocks than can be resident
  CHECK(!all_blocks_resident(1, 0, 1));
  CHECK(!all_blocks_resident(1, 152, 0));
  CHECK(all_blocks_resident(1 << 20, 1 << 20, 1 << 30));  // no overflow in the product
  std::printf("ok\n");
  return 0;
}
"""


def test_host_memos_per_device_and_context(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    src = tmp_path / "memo.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "memo"
    r = subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
