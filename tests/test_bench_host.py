"""Host-side logic of bench.py, without a GPU: the max-over-ranks timing and
whole-job aggregation across 2 gloo ranks, the clock-sample parser, the peak
file reader and the traffic record's staleness check."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    slow = bench.max_over_ranks(1.0 + r, dist)          # rank 1 is the slow one
    rate = bench.aggregate_rate(3.0e9, w, slow)
    bench.barrier(dist)
    q.put((r, slow, rate))
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _r, slow, rate in res:
        assert slow == 2.0                      # max over ranks
        assert rate == pytest.approx(3.0e9)     # 2 ranks x 3 GB / 2 s


def test_single_process_needs_no_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(1.5, None) == 1.5
    assert bench.aggregate_rate(10.0, 1, 2.0) == 5.0


def test_clock_summary_keeps_the_timed_window():
    """Samples (time, SM MHz, max MHz, power W, active reasons) outside
    [t0, t1] are dropped; the median clock, the maximum and the union of the
    reasons inside are reported."""
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.source = "nvml"
    c.rows = [(10.0, 1900.0, 2070.0, 900.1, set()),
              (10.5, 1800.0, 2070.0, 1200.5, {"sw_power_cap"}),
              (11.0, 1700.0, 2070.0, 1300.0, {"sw_power_cap"}),
              (20.0, 300.0, 2070.0, 100.0, {"hw_slowdown"})]
    c.t0, c.t1 = 9.9, 11.0
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1800
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 1300.0
    # a region between two samples: the samples just before and after it
    c.t0, c.t1 = 10.6, 10.9
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1750 and "before and after" in s["window"]
    c.rows = []
    assert c.summary()["samples"] == 0


def test_clock_reason_bits():
    """NVML clock-event reason bits of the four reasons the timing rules name."""
    assert bench.ClockSampler.REASON_BITS == {"sw_power_cap": 0x4, "hw_slowdown": 0x8,
                                              "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}


def test_peaks_and_traffic(tmp_path, monkeypatch):
    p = bench.load_peaks()
    assert p["hbm_gbs"] > 1000 and p["source"] in ("measured", "fallback")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks()["source"] == "fallback"
    assert bench.kernel_traffic("k") is None
    src = tmp_path / "a.cu"
    src.write_text("kernel v1")
    import hashlib
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"sources": ["a.cu"], "sha256": hashlib.sha256(b"kernel v1").hexdigest(),
                 "bytes_per_launch": 123.0}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.kernel_traffic("k") == 123.0
    src.write_text("kernel v2")               # the kernel changed since the capture
    assert bench.kernel_traffic("k") is None
