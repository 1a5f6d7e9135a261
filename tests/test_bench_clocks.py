"""CPU tests of the bench's clock record and of its graph-replay loop: samples
outside the load window are dropped (with a fallback when none is inside),
throttle reasons are parsed, the sampler reads a live nvidia-smi-like
process, and the replay loop holds the load for the sampler."""
import contextlib
import os
import stat
import sys
import time
import types

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

IDLE = "0, 1005, 2070, 120.5, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active"
BUSY = "0, 2070, 2070, 980.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
CAPPED = "0, 1890, 2070, 1400.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active"


def test_only_samples_inside_the_load_window_count():
    lines = [(0.0, IDLE), (0.2, IDLE), (1.0, BUSY), (1.2, CAPPED), (1.4, BUSY), (2.5, IDLE)]
    c = bench.summarise_clocks(lines, (0.9, 1.3))
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                 "window_s": 0.4}
    whole = bench.summarise_clocks(lines)
    assert whole["samples"] == 6 and whole["sm_mhz"] == pytest.approx((1005 + 1890) / 2)
    assert "window_s" not in whole


def test_no_sample_inside_the_window_falls_back_to_all():
    lines = [(5.0, BUSY), (5.0, BUSY), (5.0, IDLE)]
    c = bench.summarise_clocks(lines, (1.0, 2.0))
    assert c["samples"] == 3 and c["window_s"] is None and c["sm_mhz"] == 2070.0


def test_malformed_lines_are_skipped_and_all_reasons_parsed():
    hot = "0, 1500, 2070, 900, 0x68, Active, Active, Active, Not Active"
    lines = [(0.0, "garbage"), (0.1, "0, [N/A], 2070, 1, 0x0, a, b, c, d"), (0.2, hot)]
    c = bench.summarise_clocks(lines)
    assert c["samples"] == 1 and c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert bench.summarise_clocks([(0.0, "garbage")]) is None


def test_sampler_reads_a_live_process(tmp_path, monkeypatch):
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!" + sys.executable + "\n"
                    "import sys, time\n"
                    "for _ in range(200):\n"
                    f"    print({BUSY!r}, flush=True)\n"
                    "    time.sleep(0.02)\n")
    fake.chmod(fake.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(0.3)
    t0 = time.time()
    time.sleep(0.3)
    c = s.stop((t0, time.time()))
    assert c is not None and c["sm_mhz"] == 2070.0 and c["samples"] >= 5 and c["window_s"] >= 0.3


class _Event:
    def __init__(self, enable_timing=False):
        self.t = None

    def record(self, stream=None):
        self.t = time.perf_counter()

    def synchronize(self):
        pass

    def elapsed_time(self, other):
        return (other.t - self.t) * 1e3


def _fake_torch(log):
    class Graph:
        def replay(self):
            log.append("replay")

    cuda = types.SimpleNamespace(
        Event=_Event, Stream=lambda: object(), CUDAGraph=Graph,
        synchronize=lambda: log.append("sync"),
        stream=lambda s: contextlib.nullcontext(),
        graph=lambda g, stream=None: contextlib.nullcontext())
    return types.SimpleNamespace(cuda=cuda)


def test_graph_loop_times_steps_and_holds_the_load():
    log = []
    torch = _fake_torch(log)
    flush = types.SimpleNamespace(zero_=lambda: log.append("flush"))
    calls = []
    d = {k: k for k in ("q", "kv_pool", "qo_indptr", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask",
                        "mask_indptr", "out")}
    inp = types.SimpleNamespace(sm_scale=0.1)

    def runner(*args, events=None):
        calls.append(len(events))

    call_ms, split_ms, comb_ms, (t0, t1) = bench.measure_graph(inp, d, runner, 4, 3, flush, torch, hold_s=0.2)
    assert calls == [4]                                     # one captured call with four phase events
    assert len(call_ms) == len(split_ms) == len(comb_ms) == 4
    assert t1 - t0 >= 0.2
    replays = log.count("replay")
    assert replays > 7 and log.count("flush") == replays    # every replay after a flush
    # two device syncs around the capture, then one after every untimed replay
    # (they synchronise one by one, so no queue of replays builds up)
    assert log.count("sync") == 2 + (replays - 7)
    assert log[-1] == "sync"
    _, _, _, (u0, u1) = bench.measure_graph(inp, d, runner, 2, 0, flush, torch)
    assert u1 - u0 < 0.2                                    # hold_s = 0: no extra load
