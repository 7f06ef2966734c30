"""bench.py's host-side logic, on the CPU: the raw-ahead policy, the config
object both arms print, and the lookup of the DRAM-traffic rows."""
import argparse
import sys

import pytest

import bench
from lossless_exponent_reuse_gb300 import workloads


def _args(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.parse_args()
    finally:
        sys.argv = old


@pytest.mark.parametrize("argv,expected", [
    ((), False),                                   # exact sender, sequential
    (("--sender", "hash"), True),
    (("--schedule", "pipelined"), True),
    (("--schedule", "graph"), True),
    (("--raw-ahead",), True),
    (("--sender", "hash", "--no-raw-ahead"), False),
    (("--schedule", "graph", "--no-raw-ahead"), False),
])
def test_raw_ahead_policy(argv, expected):
    assert bench.raw_ahead_of(_args(*argv)) is expected


def test_raw_ahead_flags_are_exclusive():
    with pytest.raises(SystemExit):
        _args("--raw-ahead", "--no-raw-ahead")


@pytest.mark.parametrize("argv", [(), ("--config", "2"), ("--config", "4", "--steps", "3"),
                                  ("--sender", "rans", "--variant", "clustered0.1")])
def test_both_arms_name_the_same_config(argv):
    """The reference arm derives the accepted tensors with the oracle's
    predicate, the GPU arm with the library's; the config objects agree."""
    import oracle
    args = _args(*argv)
    wl = workloads.workload(args.config, args.variant)
    acc, declined = bench.accepted_tensors(wl)
    n = sum(k for _, k in acc)
    ours = bench.arm_config(args, wl, n, declined, 1)
    offs = workloads.layer_offsets(wl)
    n_ref = sum(k for _, o, k in offs if oracle.should_compress(k))
    ref = bench.arm_config(args, wl, n_ref, sum(k for _, o, k in offs) - n_ref, 1)
    assert ours == ref
    assert ours["workload"] == wl.name and ours["numel"] == n * wl.layers
    assert ("raw_ahead" in ours) == (args.sender != "rans")


def test_traffic_rows_follow_the_raw_ahead_setting(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("k_compress")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.md").write_text(
        "| kernel | source sha256 prefix | workload | raw-ahead | step | bytes per value |\n"
        "|---|---|---|---|---|---|\n"
        f"| k_compress | {h} | w | off | 0.1 | 5.0 |\n"
        f"| k_compress | {h} | w | on | 0.1 | 4.0 |\n"
        f"| k_compress | {h} | w | off | 0.2 | 7.0 |\n"
        f"| k_compress | {h} | v | - | 0.1 | 3.0 |\n"
        "| k_compress | 0000000000000000 | v | - | 0.2 | 9.0 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: h)
    assert bench.traffic_per_value("k_compress", "w", [0.1, 0.2], False) == 6.0
    assert bench.traffic_per_value("k_compress", "w", [0.1], True) == 4.0
    # a step with no row for the setting: no figure
    assert bench.traffic_per_value("k_compress", "w", [0.1, 0.2], True) is None
    # rows marked "-" serve either setting; rows of other kernel code never
    assert bench.traffic_per_value("k_compress", "v", [0.1], True) == 3.0
    assert bench.traffic_per_value("k_compress", "v", [0.2], False) is None


def test_default_bench_line_has_dram_traffic_for_the_current_kernels():
    """profiles/traffic.md holds rows captured on the current kernel code for
    the default workload's timed iterations, so the default bench line carries
    roofline.traffic and frac_dram."""
    args = _args()
    wl = workloads.workload(args.config, args.variant)
    steps = [wl.step_of(t) for t in range(args.warmup, args.warmup + args.steps)]
    raw_ahead = bench.raw_ahead_of(args)
    assert bench.traffic_per_value("k_compress", wl.name, steps, raw_ahead) is not None
    assert bench.traffic_per_value("k_decompress", wl.name, steps, raw_ahead) is not None
    # 20 steps after 5 warm-ups wrap the rates once: still covered
    steps20 = [wl.step_of(t) for t in range(5, 25)]
    assert bench.traffic_per_value("k_compress", wl.name, steps20, raw_ahead) is not None
