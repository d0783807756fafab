"""bench.py's JSON line on the host (no GPU): torch's CUDA calls are replaced by
host no-ops (events that report 0.25 ms, graphs that call the captured
function, streams as plain contexts) and the library by a stand-in whose calls
do nothing, so that the timing, roofline, end-to-end, clocks, launch count and
CPU-baseline legs run and print their line.  Only the line's shape and its
arithmetic are checked here; the kernels' results are the parity tests'."""
import contextlib
import io
import json

import pytest
import torch

import bench
from paged_kv_cache_240_gb300 import inputs as I

STEP_MS = 0.25


class _Event:
    def __init__(self, **kw):
        pass

    def record(self, stream=None):
        pass

    def elapsed_time(self, other):
        return STEP_MS


class _Graph:
    def replay(self):
        self.fn()


class _Stream:
    cuda_stream = 0


class _Library:
    """Stand-in for the CUDA library's binding: every call does nothing."""

    class PagedCache:
        def __init__(self, num_blocks, num_kv_heads, head_dim, dtype):
            self.k = torch.zeros(1)

    @staticmethod
    def pa_write_kv(*args):
        pass

    @staticmethod
    def pa_decode(*args):
        pass

    @staticmethod
    def pa_decode_append(*args):
        pass

    @staticmethod
    def pa_prefill_chunk(*args):
        pass

    @staticmethod
    def pa_decode_workspace_bytes(*args):
        return 0


@pytest.fixture
def host_cuda(monkeypatch):
    @contextlib.contextmanager
    def as_context(*args, **kw):
        yield

    def capture(torch_, fn, stream):
        g = _Graph()
        g.fn = fn
        fn()
        return g

    def no_device(*args):
        raise RuntimeError("no device")

    zeros, empty, to = torch.zeros, torch.empty, torch.Tensor.to
    device_normal = I.device_normal
    monkeypatch.setattr(torch.cuda, "Event", _Event)
    monkeypatch.setattr(torch.cuda, "Stream", _Stream)
    monkeypatch.setattr(torch.cuda, "stream", as_context)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "set_device", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "get_device_properties", no_device)
    monkeypatch.setattr(torch, "zeros", lambda *a, device=None, **k: zeros(*a, **k))
    monkeypatch.setattr(torch, "empty", lambda *a, device=None, **k: empty(*a, **k))
    monkeypatch.setattr(torch.Tensor, "to",
                        lambda self, *a, **k: self if a and a[0] == "cuda" else to(self, *a, **k))
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    monkeypatch.setattr(I, "device_normal",
                        lambda shape, dtype, seed, stream, device="cuda":
                        device_normal(shape, dtype, seed, stream, "cpu"))
    monkeypatch.setattr(bench, "capture", capture)
    import __graft_entry__
    import paged_kv_cache_240_gb300 as pa
    monkeypatch.setattr(__graft_entry__, "build", lambda: None)
    for name in ("PagedCache", "pa_write_kv", "pa_decode", "pa_decode_append", "pa_prefill_chunk",
                 "pa_decode_workspace_bytes"):
        monkeypatch.setattr(pa, name, getattr(_Library, name))


def _run(monkeypatch, argv):
    monkeypatch.setattr("sys.argv", ["bench.py"] + argv)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main()
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_json_line(host_cuda, monkeypatch):
    steps = 4
    line = _run(monkeypatch, ["--workload", "qwen2.5-1.5b", "--steps", str(steps), "--warmup",
                              "3", "--cpu-budget", "0.5"])
    w = I.make_workload("qwen2.5-1.5b", seed=0)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "clocks", "e2e", "gpu_launches", "roofline", "cpu_baseline"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == steps and line["warmup"] == 3
    assert line["scaling"] == "weak" and line["higher_is_better"] is True
    assert line["vs_baseline"] is None and line["dtype"] == "bf16"
    assert line["config"]["workload"] == "qwen2.5-1.5b"
    assert abs(line["ms_per_step"] - STEP_MS) < 1e-12
    assert abs(line["value"] - w.kv_bytes() / (STEP_MS * 1e-3) / 1e9) < 1e-9
    assert line["gpu_launches"] == steps  # one pa_decode_append launch, no merge kernel here
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    e = line["e2e"]
    assert e["unit"] == "GB/s" and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] == 1 and c["value"] > 0 and c["unit"] == "GB/s"
    assert "value" in c["all_cores"] or "unavailable" in c["all_cores"]


def test_json_line_int8_linear(host_cuda, monkeypatch):
    from paged_kv_cache_240_gb300 import linear as L
    gen_cls = torch.Generator
    randint, rand, randn = torch.randint, torch.rand, torch.randn
    monkeypatch.setattr(torch, "Generator", lambda device=None: gen_cls())
    monkeypatch.setattr(torch, "randint", lambda *a, device=None, **k: randint(*a, **k))
    monkeypatch.setattr(torch, "rand", lambda *a, device=None, **k: rand(*a, **k))
    monkeypatch.setattr(torch, "randn", lambda *a, device=None, **k: randn(*a, **k))
    monkeypatch.setattr(L, "int8_linear_grouped", lambda mats, x, outs=None, **k: outs)
    steps = 3
    line = _run(monkeypatch, ["--workload", "int8-linear", "--layers", "1", "--num-seqs", "2",
                              "--steps", str(steps), "--warmup", "3", "--cpu-budget", "0.3"])
    groups = bench.LINEAR_GROUPS
    assert line["config"]["workload"] == "int8-linear" and line["config"]["tokens"] == 2
    assert abs(line["value"] - bench.linear_bytes(2, groups) / (STEP_MS * 1e-3) / 1e9) < 1e-9
    # one grouped launch per group: the k splits are merged inside it
    assert line["gpu_launches"] == steps * len(groups)
    assert line["roofline"]["traffic"] is None  # recorded for the four-layer, 8-token stack
    assert line["e2e"]["h2d_bytes_per_step"] == sum(2 * 2 * grp[0][1] for grp in groups)
    assert line["e2e"]["d2h_bytes_per_step"] == sum(2 * 2 * n for grp in groups for n, _ in grp)
    assert line["cpu_baseline"]["kind"] == "oracle"
