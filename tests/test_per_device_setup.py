"""Per-device set-up of the library's kernels, on the CPU.

Kernel attributes (opt-in shared memory, non-portable cluster sizes) apply to
the device that is current when they are set, so the launchers run their
set-up once per device ordinal (PerDeviceOnce in csrc/bitlin_internal.cuh).
This test compiles that helper with g++ against a stand-in cudaGetDevice and
checks, with several host threads racing, that each of two device ordinals is
set up exactly once, that a failed set-up is retried, and that an ordinal
outside the table is refused.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>
#include "bitlin_internal.cuh"

static thread_local int g_current = 0;
// Stand-in for the runtime call: the calling thread's current device.
extern "C" cudaError_t cudaGetDevice(int* d) { *d = g_current; return cudaSuccess; }

int main()
{
    using bitlin_impl::PerDeviceOnce;
    static PerDeviceOnce once;
    std::atomic<int> calls[2] = {};
    std::vector<std::thread> ts;
    for (int t = 0; t < 8; ++t)
        ts.emplace_back([&, t] {
            g_current = t & 1;
            for (int i = 0; i < 1000; ++i) {
                int dev = -1;
                cudaError_t e = once.run(&dev, [&](int d) { calls[d]++; return cudaSuccess; });
                if (e != cudaSuccess || dev != (t & 1)) std::abort();
            }
        });
    for (auto& th : ts) th.join();
    if (calls[0] != 1 || calls[1] != 1) { std::printf("calls %d %d\n", calls[0].load(), calls[1].load()); return 1; }

    // A failed set-up is not recorded: the next call runs it again.
    static PerDeviceOnce retry;
    int dev = 0, tries = 0;
    g_current = 3;
    cudaError_t e = retry.run(&dev, [&](int) { ++tries; return cudaErrorInvalidValue; });
    if (e != cudaErrorInvalidValue) return 2;
    e = retry.run(&dev, [&](int) { ++tries; return cudaSuccess; });
    if (e != cudaSuccess || tries != 2) return 3;
    e = retry.run(&dev, [&](int) { ++tries; return cudaSuccess; });
    if (e != cudaSuccess || tries != 2) return 4;

    // An ordinal beyond the table is refused without running the set-up.
    g_current = bitlin_impl::kMaxDevices;
    e = retry.run(&dev, [&](int) { ++tries; return cudaSuccess; });
    if (e != cudaErrorInvalidDevice || tries != 2) return 5;
    std::printf("ok\n");
    return 0;
}
"""


def test_set_up_runs_once_per_device(tmp_path):
    gxx = shutil.which("g++")
    if not gxx or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    src = tmp_path / "per_device.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "per_device"
    inc = [f"-I{CUDA_INC}", f"-I{os.path.join(ROOT, 'include')}",
           f"-I{os.path.join(ROOT, 'hadamard_rotated_binary_gb300', 'csrc')}"]
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", *inc, str(src), "-o", str(exe)], check=True,
                   capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
