"""Host-side bookkeeping of libcpa.so that needs no GPU.

The kernels' shared-memory limit and the static scratch's device address are
per-device facts: a process that drives several GPUs through one library
instance must set up each device, once.  The helper that remembers this
(``csrc/cpa_host.h``) is compiled here with the host C++ compiler alone and
driven with fake device indices and a fake set-up step.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "cascade_paged_attention_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "cpa_host.h"

int main() {
    cpa::PerDevice<int> pd;
    int calls[cpa::kMaxDevices] = {};
    int fail_next = 1;  // the first set-up of device 3 fails
    auto setup = [&](int dev) {
        return [&, dev](int& v) {
            ++calls[dev];
            if (dev == 3 && fail_next) { fail_next = 0; return 7; }
            v = 100 + dev;
            return 0;
        };
    };
    int out = -1;
    // device 0: set up once, remembered
    if (pd.run(0, -9, setup(0), &out) != 0 || out != 100) return 1;
    if (pd.run(0, -9, setup(0), &out) != 0 || out != 100 || calls[0] != 1) return 2;
    // device 1 is independent of device 0
    if (pd.run(1, -9, setup(1), &out) != 0 || out != 101 || calls[1] != 1) return 3;
    // a failed set-up is reported and retried on the next call
    if (pd.run(3, -9, setup(3), &out) != 7) return 4;
    if (pd.run(3, -9, setup(3), &out) != 0 || out != 103 || calls[3] != 2) return 5;
    // device indices outside the table
    if (pd.run(-1, -9, setup(0)) != -9 || pd.run(cpa::kMaxDevices, -9, setup(0)) != -9) return 6;
    // many threads racing on a new device run its set-up exactly once
    std::vector<std::thread> ts;
    for (int i = 0; i < 16; ++i)
        ts.emplace_back([&] { int o = 0; pd.run(5, -9, setup(5), &o); });
    for (auto& t : ts) t.join();
    if (calls[5] != 1) return 7;
    std::printf("ok\n");
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_per_device_setup_runs_once_per_device(tmp_path):
    src = tmp_path / "harness.cpp"
    exe = tmp_path / "harness"
    src.write_text(HARNESS)
    subprocess.run(["g++", "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
