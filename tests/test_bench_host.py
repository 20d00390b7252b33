"""CPU tests of bench.py's host logic: the restated launch policy that names
the kernel in the roofline object, and the lookup of the committed ncu
traffic figure (tied to the kernel source and the size it was taken at)."""

import json
import os

import bench


def test_kernel_name_follows_the_launch_policy():
    # The decode-sized message: 256-thread blocks would number fewer than
    # the SMs, so 128-thread blocks of the one-vector 8-byte form.
    assert bench.reduce_kernel_name(8, 131072, False) == "reduce_half_kernel<8, 128, 1, 0>"
    assert bench.reduce_kernel_name(8, 131072, True) == "reduce_half_kernel<8, 128, 1, 1>"
    # One pass of the 8-byte grid (152 SMs x 8 blocks x 256 threads, 1/16
    # slack) covers 2^20 elements at W = 8; 2^21 needs a second one, where
    # W = 8 takes the pipelined 16-byte form and W = 5-7 keep the 8-byte one.
    assert bench.reduce_kernel_name(8, 1 << 20, False) == "reduce_half_kernel<8, 256, 1, 0>"
    assert bench.reduce_kernel_name(8, 1 << 21, False) == "reduce_vec_kernel<8, 256, 1, 1, 0>"
    assert bench.reduce_kernel_name(6, 1 << 21, False) == "reduce_half_kernel<6, 256, 1, 0>"
    # Above 2^22 elements: the pipelined 16-byte forms.
    assert bench.reduce_kernel_name(8, 1 << 23, False) == "reduce_vec_kernel<8, 256, 1, 1, 0>"
    assert bench.reduce_kernel_name(4, 1 << 23, True) == "reduce_vec_kernel<4, 256, 1, 1, 1>"
    assert bench.reduce_kernel_name(2, 1 << 23, False) == "reduce_vec_kernel<2, 128, 2, 1, 0>"


def test_stored_traffic_is_tied_to_source_and_size():
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    with open(path) as fh:
        rec = json.load(fh)
    assert bench.stored_traffic("no_such_workload", 131072) is None
    for workload, e in rec.items():
        n = e.get("n", 131072)
        got = bench.stored_traffic(workload, n)
        if e["kernel_hash"] == bench.kernel_source_hash():
            assert got == float(e["dram_bytes_per_launch"])
        else:
            assert got is None      # the kernel changed since the capture
        if "n" in e:
            assert bench.stored_traffic(workload, n + 8) is None   # taken at another size
