"""bench.py's bookkeeping, on the CPU: the DRAM-traffic table is keyed by
workload, element types and path the way the bench looks it up, and every
source file a kernel hash covers exists (a missing file would silently change
the hash)."""
import os

import bench
import workloads


def test_kernel_sources_exist():
    csrc = os.path.join(bench.ROOT, "dense_fp16_tensor_gemm_gb300", "csrc")
    lists = list(bench.KERNEL_SOURCES.values()) + [bench._SMALL_SRC]
    for names in lists:
        for n in names:
            assert os.path.exists(os.path.join(csrc, n)), n
    assert set(bench.KERNEL_SOURCES) <= set(workloads.WORKLOADS)


def test_traffic_keys():
    k = bench.traffic_key
    assert k("square_8192") == "square_8192"
    assert k("square_8192", "e4m3", "f32", True) == "square_8192/mx-e4m3"
    assert k("square_8192", "e2m1") == "square_8192/e2m1"
    assert k("square_8192", "bf16", "bf16") == "square_8192/bf16->bf16"
    assert k("skinny_64x16384x8192", path="TC05_WS") == "skinny_64x16384x8192/TC05_WS"
    for key, (traffic, sha) in bench.TRAFFIC.items():
        assert key.split("/")[0] in workloads.WORKLOADS
        assert traffic > 0 and len(sha) == 16


def test_source_hash_by_path():
    # an explicit path of the other instruction shapes hashes that kernel's sources
    assert bench.kernel_source_sha("skinny_64x16384x8192", "TC05_WS") != \
        bench.kernel_source_sha("skinny_64x16384x8192")
    assert bench.kernel_source_sha("skinny_64x16384x8192", "TC05_M64") == \
        bench.kernel_source_sha("skinny_64x16384x8192", "TC05_WS")
