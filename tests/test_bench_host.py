"""Host-side logic of bench.py on the CPU: max-over-ranks timing with two
gloo ranks, and the oracle (reference) arm on a small sample."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    d = bench.Dist(world)
    d.barrier()
    got = d.max(1.5 + rank)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"rank": d.rank, "world": d.world, "max": got}, f)
    d.close()


def test_max_over_ranks_with_gloo(tmp_path):
    if torch.cuda.is_available():
        pytest.skip("exercises the CPU (gloo) path")
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    assert [r["rank"] for r in res] == [0, 1]
    assert all(r["world"] == 2 and r["max"] == 2.5 for r in res)


class _FakeDist:
    def __init__(self, rank):
        self.rank, self.world = rank, 2


def test_reference_arm_only_rank0_prints(capsys):
    ns = type("A", (), {"steps": 2, "warmup": 1, "gpus": 2})()
    assert bench.run_reference(ns, _FakeDist(1)) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_small_inputs(capsys):
    from dense_gemm_14_gb300 import inputs
    data = {"f32_3072": inputs.make(64, 48, 40, "f32", "uniform", 1.0, 1),
            "bf16_8192": inputs.make(32, 40, 48, "bf16", "normal", 0.1, 2)}
    ns = type("A", (), {"steps": 2, "warmup": 1, "gpus": 1})()
    line = bench.run_reference(ns, _FakeDist(0), data=data)
    printed = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert printed == json.loads(json.dumps(line))
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True
    assert line["metric"] == bench.METRIC


def test_source_hash_and_traffic_gate(tmp_path, monkeypatch):
    sha = bench.source_sha("sgemm_simt.cu")
    assert len(sha) == 16
    t = bench.traffic_for("sgemm_simt_kernel", "sgemm_simt.cu", "f32_3072")
    assert t is None or t > 0
    assert bench.traffic_for("sgemm_simt_kernel", "sgemm_simt.cu", "other_workload") is None


def test_accuracy_of_reports_the_oracle_comparison():
    """The bench's accuracy entry (computed in its oracle leg): a correctly
    rounded product is within the bound with a tiny relative RMSE; one wrong
    element in the sampled rows is reported."""
    from dense_gemm_14_gb300 import inputs
    A, B = inputs.make_workload("f32_256")
    C = (A.double() @ B.double()).float()
    _, _, rows, _, ref_rows = bench.time_oracle_sample("f32_256", 0.01, A, B, want_rows=True)
    assert ref_rows.shape == (rows, 256)
    acc = bench.accuracy_of("f32_256", A, B, C, ref_rows)
    assert acc["within"] and acc["rel_rmse"] < 1e-7 and acc["bound"] == 1e-5
    assert acc["max_err_over_abs"] < 1e-7 and acc["rows_bound"] == min(16, rows)
    bad = C.clone()
    bad[0, 3] += 1.0
    acc = bench.accuracy_of("f32_256", A, B, bad, ref_rows)
    assert not acc["within"] and acc["max_err_over_abs"] > 1e-5 and acc["rel_rmse"] > 1e-4


def test_clock_summary_counts_reasons_per_sample():
    """The clock record's summary: median and range of the SM clock, the
    highest power, and how many samples carried each clock-event reason
    (bits of NVML's public header: 0x4 sw_power_cap, 0x8 hw_slowdown, 0x20
    sw_thermal_slowdown, 0x40 hw_thermal_slowdown)."""
    c = bench.ClockSampler(0, period_s=0.002)
    assert c.summary()["samples"] == 0 and c.summary()["reasons"] == ["no samples"]
    c.samples = [(2070.0, 900.0, 0x0), (1900.0, 1390.0, 0x4), (1700.0, 1400.0, 0x4 | 0x8),
                 (2070.0, 700.0, 0x1)]
    s = c.summary()
    assert s["samples"] == 4 and s["sm_mhz"] == 1985.0 and s["sm_min_mhz"] == 1700.0
    assert s["power_w_max"] == 1400.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["reason_samples"] == {"sw_power_cap": 2, "hw_slowdown": 1}
    assert s["period_ms"] == 2.0


def test_one_thread_oracle_sample():
    """The cpu_baseline's one-thread leg: the oracle on one thread, a bounded
    number of rows, the whole product when it fits."""
    f, t, rows, threads = bench.time_oracle_sample("f32_256", 0.5, threads=1)
    assert threads == 1 and rows == 256 and f == 2 * 256 ** 3 and t > 0


def test_software_loader_table_shapes_break_tma_rules():
    """Every shape of the software-loader table gives at least one operand a
    pitch that is not a multiple of 8 elements or a base off 16 bytes, so the
    plain call cannot use TMA; the reference run rounds both pitches up to 8."""
    for name, M, N, K, ta, tb, xa, xb, off in bench.SOFT_SHAPES:
        ac = M if ta else K
        bc = K if tb else N
        assert (ac + xa) % 8 or (bc + xb) % 8 or (2 * off) % 16, name
        assert min(M, N, K) > 0


def test_tf32_table_options_parse(monkeypatch):
    """--table-tf32 with one shape and mode, without a workspace (the plain
    entry points), is the command the converter kernel's profile names."""
    monkeypatch.setattr(sys, "argv", ["bench.py", "--table-tf32", "--tf32-only", "f32_3072:tf32",
                                      "--tf32-plain", "--steps", "5", "--warmup", "1"])
    a = bench.parse_args()
    assert a.table_tf32 and a.tf32_plain and a.tf32_only == "f32_3072:tf32"
    assert (a.steps, a.warmup) == (5, 1)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--table-tf32"])
    assert not bench.parse_args().tf32_plain
