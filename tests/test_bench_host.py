"""bench.py host-side helpers (no GPU): argument parsing, peaks, byte counts,
clock parsing, the traffic lookup and the memory probe."""
import json

import bench


def test_helpers_exist_and_run():
    assert bench.host_memory_available() > 0
    p = bench.load_peaks()
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0 and p["source"] in ("measured", "fallback")
    assert bench.BYTES_PER_TOKEN_HEAD == 768 + 512 + 4 + 256
    assert bench.FLOPS_PER_TOKEN_HEAD == 180224
    assert bench.decode_bytes_per_unit(128) == 2 * 65536 + 768 + 512 + 4 + 256
    srcs = [f for fs in bench.PREFILL_KERNELS.values() for f in fs]
    assert bench.committed_traffic("no/such_kernel", srcs) is None
    for f in srcs + bench.DECODE_SOURCES:
        assert bench.kernel_source_sha([f])
    # a workspace larger than the work list means the split kernel runs
    assert bench.prefill_kernel_name(512, 1) == "prefill_tc_kernel"
    assert bench.prefill_kernel_name(40 << 20, 1) == "prefill_split_kernel"


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1980, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 2025 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_argument_parsing():
    import argparse
    ns = []
    orig = bench.run_kda
    try:
        bench.run_kda = lambda a: ns.append(a) or 0
        assert bench.main(["--steps", "4", "--warmup", "3", "--only", "decode", "--no-e2e"]) == 0
    finally:
        bench.run_kda = orig
    a = ns[0]
    assert a.steps == 4 and a.only == "decode" and a.no_e2e and not a.no_cpu and a.gpus == 1
