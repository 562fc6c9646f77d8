"""The benchmark's multi-rank harness logic on CPU: two gloo ranks, each with
its own timing; every rank must see the slowest rank's time, and the
whole-job rate must count the units of all ranks (weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 7.5][rank]
    slow = bench.slowest(ms, "cpu")
    rate = bench.whole_job_rate(100.0, world, slow / 1e3)
    results[rank] = (slow, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert results[0] == results[1]
        slow, rate = results[0]
        assert slow == 7.5
        assert rate == pytest.approx(2 * 100.0 / 7.5e-3)


def test_single_process_is_identity():
    import bench
    assert bench.slowest(4.25, "cpu") == 4.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_e2e_packing_round_trips_and_aligns():
    # the end-to-end leg moves a step's inputs in one copy: every tensor gets a
    # 256-byte-aligned, non-overlapping slice and reads back unchanged
    import torch
    import bench
    named = {"a": torch.arange(7, dtype=torch.int32), "b": torch.randn(3, 5).to(torch.bfloat16),
             "c": torch.randn(2, 2, 3)}
    offs, total = bench._pack(named)
    spans = sorted((offs[k], offs[k] + t.numel() * t.element_size()) for k, t in named.items())
    assert all(o % 256 == 0 for o, _ in spans) and spans[-1][1] <= total
    assert all(spans[i][1] <= spans[i + 1][0] for i in range(len(spans) - 1))
    buf = torch.zeros(total, dtype=torch.uint8)
    for k, v in bench._views(buf, offs, named).items():
        v.copy_(named[k])
    for k, v in bench._views(buf.clone(), offs, named).items():
        assert v.dtype == named[k].dtype and v.shape == named[k].shape and torch.equal(v, named[k])


def test_roofline_peaks_from_the_measured_file(tmp_path):
    # each denominator is the measured one when the file gives it, else the fallback
    import json as _json
    import bench
    fb = bench.FALLBACK_PEAKS
    missing = tmp_path / "none.json"
    assert bench.peaks(str(missing)) == (fb, "fallback")
    full = tmp_path / "full.json"
    full.write_text(_json.dumps({"hbm_gbs": 7400.5, "bf16_tflops": {"value": 2100}, "bf16_tflops_sustained": 1800,
                                 "clocks": {"sm": 2070}}))
    assert bench.peaks(str(full)) == ({"hbm_gbs": 7400.5, "bf16_tflops": 2100.0, "bf16_tflops_sustained": 1800.0},
                                      "measured")
    part = tmp_path / "part.json"
    part.write_text(_json.dumps({"hbm_gbs": 7000, "bf16_tflops": "n/a"}))
    pk, src = bench.peaks(str(part))
    assert src == "measured and fallback" and pk["hbm_gbs"] == 7000.0
    assert pk["bf16_tflops"] == fb["bf16_tflops"] and pk["bf16_tflops_sustained"] == fb["bf16_tflops_sustained"]
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    assert bench.peaks(str(bad)) == (fb, "fallback")


def test_reference_arm_prints_one_json_line():
    # the oracle timed on the host cores, on the tiny workload: one JSON line
    # with the contract's keys (the arm runs without a GPU)
    import json as _json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "1",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = _json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["config"]["workload"] == "tiny_b1_h16_t256_bf16"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
