"""bench.py's host logic on the CPU: the reference arm's JSON line, the replicas' aggregation over ranks
(world size 2 over gloo), the clock sampler's reading of nvidia-smi lines, the kernel-source hash and
the peak lookup. No GPU and no oracle run."""
import io
import json
import os
import socket
import types
from contextlib import redirect_stdout

import pytest

import bench


def ref_args(**kw):
    a = dict(workload="decode_b1", steps=3, warmup=1, ref_budget_s=150.0)
    a.update(kw)
    return types.SimpleNamespace(**a)


def test_reference_arm_line(monkeypatch):
    calls = []

    def fake_sample(shape, seed, zipf_s, x_dtype, n_tokens):
        calls.append(n_tokens)
        return 2.0  # seconds per oracle call
    monkeypatch.setattr(bench, "oracle_sample", fake_sample)
    monkeypatch.setattr(bench, "cpu_cores", lambda: 8)
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(ref_args(), rank=0, world=1)
    lines = [ln for ln in out.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert calls == [1, 8, 8, 8]  # one warm-up call of one token, then `steps` samples of 8 tokens
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] == pytest.approx(8 / 2.0) and d["ms_per_step"] == pytest.approx(2000.0)
    assert d["steps"] == 3 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "decode_b1" and d["config"]["tokens_per_layer_call"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 8 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_stops_at_its_budget(monkeypatch):
    monkeypatch.setattr(bench, "oracle_sample", lambda *a: 0.01)
    monkeypatch.setattr(bench, "cpu_cores", lambda: 4)
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(ref_args(steps=10**9, ref_budget_s=0.0), rank=0, world=1)
    d = json.loads(out.getvalue())
    assert d["steps"] == 1  # the first sample already exceeds a zero budget


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    def fail(*a):
        raise AssertionError("rank 1 must not run the oracle")
    monkeypatch.setattr(bench, "oracle_sample", fail)
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(ref_args(), rank=1, world=2)
    assert out.getvalue() == ""


def test_job_rate_is_whole_job_throughput():
    # 2 replicas x 64 tokens x 10 steps in 20 ms of the slowest rank
    assert bench.job_rate(2, 64, 10, 20.0) == pytest.approx(2 * 64 * 10 / 0.020)
    assert bench.job_rate(1, 1, 2000, 152.4) == pytest.approx(2000 / 0.1524)
    assert bench.max_over_ranks(3.5, 1) == 3.5  # one rank: its own time, no collective


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    import datetime

    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        q.put((rank, ms, bench.job_rate(world, 16, 5, ms)))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_over_gloo():
    """World size 2: each rank times its own replica; both end with the larger time, and the job's
    value counts both ranks' tokens over it."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [12.5, 17.25]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q), daemon=True) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
    finally:
        for p in procs:
            if p.is_alive():
                p.kill()
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, v in res:
        assert ms == 17.25
        assert v == pytest.approx(2 * 16 * 5 / 0.01725)


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_reads_reasons_and_median():
    cs = bench.ClockSampler(0)
    cs.proc = _FakeProc()
    cs.lines = [
        "2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1300.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",  # unreadable: skipped
        "garbage",
    ]
    clk = cs.stop()
    assert clk["sm_mhz"] == 2070.0 and clk["sm_max_mhz"] == 2070.0 and clk["samples"] == 3
    assert clk["reasons"] == ["sw_power_cap"]
    cs = bench.ClockSampler(0)
    cs.proc = _FakeProc()
    cs.lines = ["1200, 2070, 700, 0x0, Active, Not Active, Active, Not Active"]
    assert cs.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]


def _copy_kernel_sources(dst):
    src = os.path.join(bench.ROOT, "mxfp4_routed_expert_k3moe_gb300", "csrc")
    os.makedirs(os.path.join(dst, "mxfp4_routed_expert_k3moe_gb300", "csrc"))
    for f in ("k3moe_tc.cu", "k3moe_ptx.cuh", "k3moe_common.cuh"):
        with open(os.path.join(src, f)) as fi, open(os.path.join(dst, "mxfp4_routed_expert_k3moe_gb300", "csrc", f),
                                                    "w") as fo:
            fo.write(fi.read())
    return os.path.join(dst, "mxfp4_routed_expert_k3moe_gb300", "csrc", "k3moe_tc.cu")


def test_kernel_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    tc = _copy_kernel_sources(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_hash()
    assert h0 == bench.kernel_hash() and len(h0) == 16
    with open(tc, "a") as fh:
        fh.write("\n// a new comment line\n    \n")
    assert bench.kernel_hash() == h0
    with open(tc, "a") as fh:
        fh.write("static int k3moe_new_symbol = 1;\n")
    assert bench.kernel_hash() != h0


def test_hbm_peak_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6781.1}))
    assert bench.hbm_peak() == (6781.1, "measured")
