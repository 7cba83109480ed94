"""Host-side logic of bench.py (no GPU): the max/sum-over-ranks reductions on
2 gloo ranks, the reference (oracle) arm's JSON line, rank handling, and the
clock-sample parser."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

from mxcheck import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cpu = torch.device("cpu")
    m = bench.max_over_ranks(1.5 * (rank + 1), world, cpu)
    s = bench.sum_over_ranks(float(rank + 1), world, cpu)
    q.put((rank, m, s))
    dist.barrier()
    dist.destroy_process_group()


def test_step_time_is_max_and_units_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 3.0, 3.0), (1, 3.0, 3.0)]


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         env=env, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["metric"] == bench.METRIC


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1"]) == 0
    assert capsys.readouterr().out == ""


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1965, 2070, 900.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "0, 1980, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 345, 2070, 120.0, 0x1, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["sm_mhz"] == 1972.5
    assert s["reasons"] == ["sw_power_cap"]


def test_peaks_file_is_read_or_falls_back():
    d, src = bench.read_peaks()
    assert src in ("measured", "fallback")
    assert d["hbm_gbs"] > 1000 and d["bf16_tflops"] > 100


def test_moe_roofline_bounds():
    """The MoE roofline: one large expert is tensor-bound with time = FLOP /
    peak; experts without tokens cost nothing in the forward but their FP32
    zero outputs in the weight gradient; the per-expert sum of maxima is
    never below the overall bound."""
    n, k, peak, bw = 2048, 7168, 4000.0, 8000.0
    r = bench.moe_roofline([65536], n, k, "forward", peak, bw)
    assert r["bound"] == "tensor"
    assert abs(r["time_ms"] - 2 * 65536 * n * k / (peak * 1e12) * 1e3) < 1e-3
    assert bench.moe_roofline([0, 0, 0], n, k, "forward", peak, bw)["time_ms"] == 0.0
    w = bench.moe_roofline([0] * 64, n, k, "wgrad", peak, bw)
    assert w["bound"] == "hbm" and w["bytes"] == 64 * n * k * 4
    assert abs(w["time_ms"] - 64 * n * k * 4 / (bw * 1e9) * 1e3) < 1e-3
    for kind in ("forward", "dgrad", "wgrad"):
        m = bench.moe_roofline([0, 1, 31, 500, 20000, 45004], n, k, kind, peak, bw)
        assert m["per_expert_ms"] >= m["time_ms"] - 1e-9
        row = bench.with_roofline({"ms": 2 * m["time_ms"]}, m)
        assert row["roofline"]["frac"] == 0.5


def test_gemm_row_reports_loop_and_burst_against_both_peaks():
    fl = 2 * 16384 * 18432 * 7168
    row = bench._gemm_row(fl, 1.30, 1.14, 3781.4, 3393.4)
    assert row["ms"] == 1.3 and row["burst"]["ms"] == 1.14
    assert abs(row["TFLOP/s"] - fl / 1.30e-3 / 1e12) < 0.1
    assert abs(row["frac_fp8_peak"] - row["TFLOP/s"] / 3781.4) < 1e-3
    assert abs(row["frac_fp8_sustained_peak"] - row["TFLOP/s"] / 3393.4) < 1e-3
    assert abs(row["burst"]["frac_fp8_peak"] - row["burst"]["TFLOP/s"] / 3781.4) < 1e-3
    roof = {"time_ms": 0.5, "per_expert_ms": 0.6}
    bench.with_roofline(row, roof)
    assert row["roofline"]["frac"] == round(0.5 / 1.30, 3)
    assert row["burst"]["roofline_frac"] == round(0.5 / 1.14, 3)


def test_row_clocks_record_the_sampled_median_only():
    class Sampler:
        def summary(self, t0, t1):
            return {"sm_mhz": 1500.0, "samples": 4}
    rc = bench.RowClocks()
    row = {"TFLOP/s": 3000.0}
    rc.mark(row, (0.0, 1.0), "TFLOP/s")
    rc.fill(Sampler())
    assert row["sm_mhz_median"] == 1500.0 and row["clock_samples"] == 4
    assert "clock_normalized" not in row
