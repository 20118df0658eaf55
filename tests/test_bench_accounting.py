"""Host-side accounting of bench.py (no GPU): the algorithmic bytes behind the roofline
fraction and the lookup of recorded DRAM traffic.

The roofline's numerator counts each distinct value row that an in-level corner touches
once ("unique value bytes").  bench.unique_value_rows computes it with vectorised numpy;
here it is recounted by brute force, one sample and one corner at a time, on small drawn
problems in 2D and 3D with samples straddling and leaving the levels.
"""
import math
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _brute_unique_rows(inp):
    return len(set(_brute_rows(inp)))


def _brute_corner_rows(inp):
    return len(_brute_rows(inp))


def _brute_rows(inp):
    """Every (batch, value row, head) an in-level corner of a sample touches, with
    repeats, one sample and one corner at a time."""
    loc = inp["sampling_locations"].astype(np.float64)
    B, Nq, M, L, P, nd = loc.shape
    rows = []
    for b in range(B):
        for q in range(Nq):
            for m in range(M):
                for l in range(L):
                    ext = [int(e) for e in inp["spatial_shapes"][l][::-1]]   # (W, H[, Z])
                    start = int(inp["level_start_index"][l])
                    for p in range(P):
                        pix = [loc[b, q, m, l, p, k] * ext[k] - 0.5 for k in range(nd)]
                        if not all(math.isfinite(x) and -1 < x < e for x, e in zip(pix, ext)):
                            continue
                        base = [math.floor(x) for x in pix]
                        for c in range(2 ** nd):
                            idx = [base[k] + ((c >> k) & 1) for k in range(nd)]
                            if not all(0 <= i < e for i, e in zip(idx, ext)):
                                continue
                            flat = idx[0] + ext[0] * idx[1]
                            if nd == 3:
                                flat += ext[0] * ext[1] * idx[2]
                            rows.append((b, start + flat, m))
    return rows


@pytest.mark.parametrize("nd,shapes", [(2, [(7, 9), (3, 4)]), (3, [(3, 4, 5), (2, 2, 3)])])
def test_unique_value_rows_matches_brute_force(nd, shapes):
    inp = workloads.random_problem(nd, shapes, B=2, Nq=23, M=3, D=8, P=3, seed=31)
    w = workloads.Workload("t", nd, 2, tuple(tuple(s) for s in shapes), 23, 3, 8, 3, "f32", 31)
    assert bench.unique_value_rows(w, inp) == _brute_unique_rows(inp)


def test_algorithmic_bytes_of_the_encoder_forward():
    """The encoder-shaped forward: locations, weights and output by size, and the unique
    value bytes never above the whole value tensor."""
    w = workloads.WORKLOADS["encoder2d"]
    inp = workloads.make_inputs(w)
    ab = bench.algorithmic_bytes(w, inp)
    parts = ab["parts"]
    samples = w.B * w.Nq * w.M * w.L * w.P
    assert parts["locations"] == samples * 2 * 4 and parts["weights"] == samples * 4
    assert parts["out"] == w.B * w.Nq * w.M * w.D * 4
    assert 0 < parts["unique_value"] <= parts["whole_value_tensor"]
    assert ab["total"] == sum(v for k, v in parts.items() if k != "whole_value_tensor")


def test_recorded_traffic_is_keyed_by_workload_mode_and_source_hash(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("forward")
    (tmp_path / "a.md").write_text(f"bench_workload: encoder2d\nkernel_source_sha256: {h}\n"
                                   "dram_bytes_per_launch: 123\n")
    (tmp_path / "b.md").write_text(f"bench_workload: encoder2d+order\nkernel_source_sha256: {h}\n"
                                   "dram_bytes_per_launch: 456\n")
    (tmp_path / "c.md").write_text("bench_workload: decoder2d\nkernel_source_sha256: "
                                   + "0" * 64 + "\ndram_bytes_per_launch: 789\n")
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    assert bench.recorded_traffic("encoder2d") == 123
    assert bench.recorded_traffic("encoder2d", "+order") == 456
    assert bench.recorded_traffic("decoder2d") is None      # taken on other sources
    assert bench.recorded_traffic("volume3d") is None       # no summary


def _run_bench(args, env_extra=None):
    import json
    import subprocess
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    return [json.loads(l) for l in lines]


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the CPU oracle, no GPU) prints one JSON line with the
    contract's keys, on the same metric and workload keys as the GPU arm."""
    flags = ["--workload", "tiny2d", "--steps", "3", "--warmup", "3"]
    (line,) = _run_bench(["--impl", "reference", *flags])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "impl", "cpu_baseline", "e2e", "gpu_launches"):
        assert k in line, k
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["steps"] == 3 and line["gpu_launches"] == 0
    # the same config dict as the GPU arm prints for the same flags
    args = bench.build_parser().parse_args(flags)
    assert line["config"] == bench.run_config(workloads.WORKLOADS["tiny2d"], args, 1)
    # the forward oracle runs on every host thread
    import oracle
    oracle.build()
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["cores"] == oracle.default_threads()


def test_corner_row_count_and_l1_ceiling():
    """The L1 ceiling counts every in-level corner row of every sample (brute force on a
    small problem) and turns rows into microseconds at one 128-B wavefront per SM clock."""
    nd, shapes = 2, [(5, 7), (2, 3)]
    inp = workloads.random_problem(nd, shapes, B=2, Nq=9, M=3, D=8, P=2, seed=5,
                                   backward=False)
    w = workloads.Workload("t", nd, 2, tuple(shapes), 9, 3, 8, 2, "f32", 5)
    uniq, total = bench.value_row_counts(w, inp)
    assert uniq == _brute_unique_rows(inp)
    assert total == _brute_corner_rows(inp)
    c = bench.l1_ceiling(w, 148 * 2000 * 10, None, 148, 2000.0, 20e-6, 6.4e6, 6400.0)
    assert abs(c["rows_floor_us"] - 10.0) < 1e-9 and abs(c["rows_frac"] - 0.5) < 1e-12
    assert c["frac"] is None and abs(c["hbm_frac_ceiling"] - 0.1) < 1e-12
    c = bench.l1_ceiling(w, 1, 148 * 2000 * 15, 148, 2000.0, 20e-6, 6.4e6, 6400.0)
    assert abs(c["floor_us"] - 15.0) < 1e-9 and abs(c["frac"] - 0.75) < 1e-12


def test_l2_reduction_ceiling():
    """The backward's L2 ceiling: D * 4 / 32 sector updates per in-level corner row (fp32
    grad_value rows, reductions in runs of whole sectors) at the probe's measured rate."""
    w = workloads.WORKLOADS["volume3d_bwd"]                 # D = 32: four sectors per row
    rows = 1_000_000
    c = bench.l2_reduction_ceiling(w, rows, 40e-6)
    assert c["sector_updates_per_launch"] == 4 * rows
    want_us = 4 * rows / bench.L2_RED_SECTORS_PER_S * 1e6
    assert abs(c["floor_us"] - want_us) < 1e-9
    assert abs(c["frac"] - want_us / 40.0) < 1e-12
    w8 = workloads.Workload("t", 2, 1, ((4, 4),), 3, 1, 8, 1, "bf16", 1, backward=True)
    assert bench.l2_reduction_ceiling(w8, 10, 1e-6)["sector_updates_per_launch"] == 10


def test_reference_arm_other_ranks_stay_silent():
    """Under torchrun only rank 0 runs the reference arm; another rank prints nothing."""
    assert _run_bench(["--impl", "reference", "--workload", "tiny2d", "--steps", "3",
                       "--warmup", "3"], {"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_config_names_the_query_order_mode():
    """`--order` (each step) and `--order once` (outside the timed region) are different
    measurements; the config says which."""
    w = workloads.WORKLOADS["volume3d"]
    p = bench.build_parser()
    assert "each step" in bench.run_config(w, p.parse_args(["--order"]), 1)["query_order"]
    assert "once per input set" in bench.run_config(w, p.parse_args(["--order", "once"]),
                                                    1)["query_order"]
    assert bench.run_config(w, p.parse_args([]), 1)["query_order"] == "as given"
