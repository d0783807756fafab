"""Benchmark of the paged-KV decode step on GB300.

One step = pa_write_kv of the step's new tokens (one per decoding sequence, plus
the prefill chunks' tokens in the mixed workload) + pa_decode over the batch (+
pa_prefill_chunk for the chunks), one layer.  The headline workload is the
7B-shaped MHA decode (64 sequences, 32/32 heads, head_dim 128, fp16, contexts
U[1024, 4096], 16-token blocks, shuffled pool 1.25x the tokens): its ~2.6 GB of
KV per step is far larger than the 129 MB L2, so every timed step reads HBM.

Printed: one JSON line (rank 0).  ``value`` = algorithmic KV bytes per step /
device time per step (CUDA events on the launching stream, inputs resident);
``e2e`` = the same through the C ABI with the step's inputs copied from pinned
host memory and its output copied back inside the timed region; ``roofline`` =
the decode call's achieved KV GB/s against the measured HBM copy bandwidth;
``cpu_baseline`` = the CPU oracle on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle (the only reference this repo has)
on the same workload and prints the same line with ``impl: reference``.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV-read GB/s (% of GB300 HBM peak); decode steps/sec"
DEFAULT_WORKLOAD = "mha-7b"
L2_BYTES = 129 * 2 ** 20
FILL_CHUNK = 1 << 15  # history rows per pa_write_kv while a pool is filled
# GB300 datasheet figures, reported beside the measured peaks for context only:
# HBM3e 7.9 TB/s, dense bf16 tensor 2.25 PFLOP/s
NOMINAL = {"GB/s": 7900.0, "TFLOP/s": 2250.0}
TRAFFIC_FILES = {"decode": os.path.join(ROOT, "profiles", "decode_traffic.json"),
                 "prefill": os.path.join(ROOT, "profiles", "prefill_traffic.json"),
                 "linear": os.path.join(ROOT, "profiles", "linear_traffic.json")}


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_240_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, call="decode"):
    """DRAM bytes per pa_decode (or pa_prefill_chunk) call from the committed ncu
    record, or None when the kernel sources changed since it was taken."""
    try:
        with open(TRAFFIC_FILES[call]) as f:
            tr = json.load(f)
    except (OSError, ValueError):
        return None
    if tr.get("kernel_source_hash") != kernel_source_hash(tr.get("kernel_sources", [])):
        return None
    return tr.get("traffic_bytes_per_launch", {}).get(workload)


def max_over_ranks(torch, values, world, device="cuda"):
    """Each rank's timings -> their maximum over the ranks (every rank gets it):
    the job runs as long as its slowest rank.  One process: the values as given."""
    if world <= 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def measured_peaks(path=os.path.join(ROOT, "MEASURED_PEAKS.json")):
    """(peaks, "measured") from the measured-peaks file, or the earlier GB300
    measurement (6.8 TB/s copy, 1.9 PFLOP/s bf16 burst, 1.7 sustained) and
    "fallback" when the file is missing, unreadable or lacks a figure."""
    fallback = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    try:
        with open(path) as f:
            got = json.load(f)
    except (OSError, ValueError):
        return fallback, "fallback"
    if not isinstance(got, dict) or not all(
            isinstance(got.get(k), (int, float)) and got[k] > 0 for k in fallback):
        return fallback, "fallback"
    return got, "measured"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid, self.proc = uuid, None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


# ------------------------------------------------------------------ device workload

def pack_tensors(torch, tensors, dev):
    """One uint8 device buffer holding the tensors back to back, each at a
    256-byte boundary (the library wants 16), and views of it shaped and typed
    like them with their values copied in: a step's inputs (or outputs) then move
    between host and device in one copy."""
    sizes = [t.numel() * t.element_size() for t in tensors]
    offs, off = [], 0
    for nb in sizes:
        offs.append(off)
        off += (nb + 255) // 256 * 256
    buf = torch.empty(max(off, 256), dtype=torch.uint8, device=dev)
    views = []
    for t, o, nb in zip(tensors, offs, sizes):
        v = buf[o:o + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class DeviceStep:
    """Everything one step needs, resident on the device ``dev`` (the host serves only
    checks of this bookkeeping that stand host functions in for the library's calls)."""

    def __init__(self, w, torch, pa, I, seed, dev="cuda"):
        self.w, self.torch, self.pa = w, torch, pa
        src = I.source_dtype(w)
        self.cache = pa.PagedCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.cache_dtype)
        self.err = torch.zeros(4, dtype=torch.int32, device=dev)
        # history = every position before the step's new tokens
        new = w.new_slot_mapping()
        hist = []
        for b in range(w.num_seqs):
            L, C = int(w.context_lens[b]), int(w.q_lens[b])
            hist.append(w.slots(b, np.arange(0, L - C)))
        hist = np.concatenate(hist).astype(np.int32)
        chunk = FILL_CHUNK
        for i in range(0, hist.size, chunk):
            s = torch.from_numpy(hist[i:i + chunk]).to(dev)
            shape = (s.shape[0], w.num_kv_heads, w.head_dim)
            k = I.device_normal(shape, src, seed, 2 * i + 1, dev)
            v = I.device_normal(shape, src, seed, 2 * i + 2, dev)
            pa.pa_write_kv(self.cache, k, v, s, self.err)
        T = w.num_q_tokens
        self.k_new = I.device_normal((T, w.num_kv_heads, w.head_dim), src, seed, 10 ** 7, dev)
        self.v_new = I.device_normal((T, w.num_kv_heads, w.head_dim), src, seed, 10 ** 7 + 1,
                                     dev)
        self.slots = torch.from_numpy(new).to(dev)
        nd = w.num_decode
        self.nd = nd
        nq = int(w.cu_q_lens[nd])
        q = I.device_normal((T, w.num_q_heads, w.head_dim), w.q_dtype, seed, 10 ** 7 + 2, dev)
        # decode and prefill parts as separate (aligned, contiguous) tensors
        self.q_dec, self.q_pre = q[:nq].clone(), q[nq:].clone()
        self.out_dec, self.out_pre = torch.empty_like(self.q_dec), torch.empty_like(self.q_pre)
        self.tables_dec = torch.from_numpy(w.block_tables[:nd].copy()).to(dev)
        self.tables_pre = torch.from_numpy(w.block_tables[nd:].copy()).to(dev)
        self.lens_dec = torch.from_numpy(w.context_lens[:nd].copy()).to(dev)
        self.lens_pre = torch.from_numpy(w.context_lens[nd:].copy()).to(dev)
        self.cu = torch.from_numpy(w.cu_q_lens[nd:] - w.cu_q_lens[nd]).to(dev)
        self.max_q = int(w.q_lens[nd:].max()) if w.num_seqs > nd else 0
        self.sm = 1.0 / float(np.sqrt(w.head_dim))
        nbytes = pa.pa_decode_workspace_bytes(nd, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                              w.max_blocks_per_seq, w.window)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        self.reduce_launched = nbytes > 0 and nd > 0
        # the step's inputs, and its outputs, each packed into one device buffer so
        # that the end-to-end run moves them with one copy each way
        self.inputs_buf = self._pack(self.INPUTS, dev)
        self.outputs_buf = self._pack(self.OUTPUTS, dev)
        if torch.device(dev).type == "cuda":
            torch.cuda.synchronize()
        if int(self.err[0]) != 0:
            raise RuntimeError("device flags %d while filling the cache" % int(self.err[0]))

    # tensors the end-to-end run copies in from the host every step / out after it
    INPUTS = ("q_dec", "q_pre", "k_new", "v_new", "slots", "tables_dec", "tables_pre",
              "lens_dec", "lens_pre", "cu")
    OUTPUTS = ("out_dec", "out_pre")

    def _pack(self, names, dev):
        """Pack the named tensors into one buffer (pack_tensors); they become its views."""
        buf, views = pack_tensors(self.torch, [getattr(self, n) for n in names], dev)
        for n, v in zip(names, views):
            setattr(self, n, v)
        return buf

    def launches_per_step(self):
        if self.nd and not self.max_q:  # pa_decode_append (+ its merge kernel)
            return 1 + (1 if self.reduce_launched else 0)
        n = 1 + (1 if self.nd else 0) + (1 if self.reduce_launched else 0)
        return n + (1 if self.max_q else 0)

    def write(self):
        self.pa.pa_write_kv(self.cache, self.k_new, self.v_new, self.slots, self.err)

    def decode(self):
        if not self.nd:  # a step with no decoding sequence (spec-verify)
            return
        self.pa.pa_decode(self.cache, self.out_dec, self.q_dec, self.tables_dec, self.lens_dec,
                          self.sm, self.w.window, self.ws, self.err)

    def prefill(self):
        if self.max_q:
            self.pa.pa_prefill_chunk(self.cache, self.out_pre, self.q_pre, self.cu, self.max_q,
                                     self.tables_pre, self.lens_pre, self.sm, self.w.window,
                                     self.err)

    def run(self, side=None):
        """One step as the benchmark times it: decoding sequences alone in one
        launch (pa_decode_append: each new token written at its position, then
        the attention); otherwise the write, then the attention calls (side by
        side when a second stream is given, see attend)."""
        if self.nd and not self.max_q:
            self.pa.pa_decode_append(self.cache, self.k_new, self.v_new, self.out_dec, self.q_dec,
                                     self.tables_dec, self.lens_dec, self.sm, self.w.window,
                                     self.ws, self.err)
            return
        self.write()
        self.attend(side)

    def attend(self, side=None):
        """The two attention calls.  Given a second stream ``side`` (and both calls
        having work), the prefill call is enqueued there first and the decode call
        after it on the current stream, joined before returning: both only read
        the cache the write filled, and the decode's CTAs take the SMs that the
        persistent prefill launch gives up as its CTAs finish their items."""
        if side is None or not (self.nd and self.max_q):
            self.decode()
            self.prefill()
            return
        cur = self.torch.cuda.current_stream()
        side.wait_stream(cur)
        with self.torch.cuda.stream(side):
            self.prefill()
        self.decode()
        cur.wait_stream(side)


def prefill_flops(w):
    """Tensor-core work of the prefill chunks: 2*D flops for q.k and 2*D for p*v
    per (query, head, visible key)."""
    total = 0
    for b in range(w.num_decode, w.num_seqs):
        L, C = int(w.context_lens[b]), int(w.q_lens[b])
        pos = np.arange(L - C, L, dtype=np.int64)
        keys = np.minimum(pos + 1, w.window) if w.window > 0 else pos + 1
        total += int(keys.sum()) * w.num_q_heads * 4 * w.head_dim
    return total


def prefill_kv_bytes(w):
    """Algorithmic KV bytes of the prefill call: each chunk's visible keys once per
    kv head (the chunk's last query sees the most)."""
    el = 1 if w.cache_dtype == "i8" else 2
    per_tok = 2 * w.head_dim * el + (8 if w.cache_dtype == "i8" else 0)
    total = 0
    for b in range(w.num_decode, w.num_seqs):
        L, C = int(w.context_lens[b]), int(w.q_lens[b])
        lo = max(0, L - C - w.window + 1) if w.window > 0 else 0
        total += (L - lo) * per_tok * w.num_kv_heads
    return total


def decode_kv_bytes(w):
    """Algorithmic KV bytes of the decode call (the decoding sequences only)."""
    el = 1 if w.cache_dtype == "i8" else 2
    per_tok = 2 * w.head_dim * el + (8 if w.cache_dtype == "i8" else 0)
    L = w.context_lens[:w.num_decode].astype(np.int64)
    eff = np.minimum(L, w.window) if w.window > 0 else L
    return int(eff.sum()) * per_tok * w.num_kv_heads


def roofline(w, dec_ms, pre_ms, peaks, src, full_size=True):
    """The roofline object of the call that takes longer: the prefill call against
    the bf16 tensor peak when its flop per algorithmic byte exceeds the machine
    balance, else against HBM; otherwise the decode call against HBM.  ``achieved``
    = the call's algorithmic flops or bytes / its mean CUDA-event time (ms).  The
    recorded ncu traffic is of the full-size workloads only (else null)."""
    pre_flops, pre_bytes = prefill_flops(w), prefill_kv_bytes(w)
    balance = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flop per byte
    if pre_ms > dec_ms and pre_flops > balance * pre_bytes:
        # the prefill kernel dominates and is a dense contraction: tensor-core roofline
        achieved = pre_flops / (pre_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": recorded_traffic(w.name, "prefill"),
                "kernel": ("pa_prefill_chunk (tcgen05.mma kind::f16, TMEM accumulators)"
                           if w.cache_dtype != "i8" else "pa_prefill_chunk (mma.sync m16n8k16)"),
                "peak_source": src + " bf16_tflops (burst)"}
    elif pre_ms > dec_ms:
        # the prefill kernel dominates with few queries per key (verification of a
        # few drafted tokens): it streams the cache, HBM roofline
        achieved = pre_bytes / (pre_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(w.name, "prefill"),
                "kernel": "pa_prefill_chunk (%d queries per sequence)" % int(w.q_lens.max()),
                "peak_source": src + " hbm_gbs"}
    else:
        achieved = decode_kv_bytes(w) / (dec_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(w.name),
                "kernel": "pa_decode (split-K attention and its merge)",
                "peak_source": src + " hbm_gbs"}
    if not full_size:
        roof["traffic"] = None
    roof["frac_of_nominal"] = roof["achieved"] / NOMINAL[roof["unit"]]
    return roof


def needs_l2_flush(w):
    """Whether a step's KV is small enough (under four L2s) to be partly served
    from L2 by the step before; such workloads flush L2 between timed runs."""
    return w.kv_bytes() <= 4 * L2_BYTES


def capture(torch, fn, stream):
    """CUDA graph of fn's launches (the library's kernels enqueue on the current
    stream, so they are captured like any other work)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm the lazily-set kernel attributes outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def time_replays(torch, stream, run, n, flush=None):
    """CUDA-event time (ms) of each of n runs on ``stream``; ``flush``, when given,
    is enqueued before each run, outside its events."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in ev:
        if flush is not None:
            flush()
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_ours(args, w, torch, pa, I, rank, world, steps=None, warmup=None):
    """Time K graph replays of the step (after W warm-ups) on this rank, then the
    two attention calls on their own, the step launched call by call, and the
    step end to end through pinned host memory."""
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    st = DeviceStep(w, torch, pa, I, seed=args.seed + 1000 * rank)
    stream = torch.cuda.Stream()
    side = torch.cuda.Stream() if st.nd and st.max_q else None

    def step():
        st.run(side)

    if args.no_graph:
        run_step, run_dec, run_pre = step, st.decode, st.prefill
    else:
        g_step = capture(torch, step, stream)
        # a call with nothing to do (no decoding sequence, or no chunk) is not captured
        g_dec = capture(torch, st.decode, stream) if st.nd else None
        g_pre = capture(torch, st.prefill, stream) if st.max_q else None
        run_step = g_step.replay
        run_dec = g_dec.replay if g_dec else (lambda: None)
        run_pre = g_pre.replay if g_pre else (lambda: None)
    try:
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    flush = None
    if needs_l2_flush(w):
        # a step's KV could stay in L2 from the one before: write a buffer twice
        # the L2's size before every timed run so that each one reads cold
        scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        flush = scratch.zero_
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run_step()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        clocks.start()
        time.sleep(0.3)
        step_ms = time_replays(torch, stream, run_step, steps, flush)
        if world > 1:
            torch.distributed.barrier()
        clk = clocks.stop()
        # the two attention calls on their own, for the per-kernel roofline
        nk = max(3, min(steps, 500))
        dec_ms = time_replays(torch, stream, run_dec, nk, flush) if st.nd else [0.0]
        pre_ms = time_replays(torch, stream, run_pre, nk, flush) if st.max_q else [0.0]
        # the same step launched call by call from Python, for comparison with the
        # graph replays above
        eager_ms = time_replays(torch, stream, step, nk, flush) if not args.no_graph else step_ms
        torch.cuda.synchronize()
        if int(st.err[0]) != 0:
            raise RuntimeError("device flags %d during the timed steps" % int(st.err[0]))

        # end to end: the step's inputs from pinned host memory, its outputs back,
        # each direction one copy of the packed buffer
        host_in = st.inputs_buf.cpu().pin_memory()
        host_out = torch.empty(st.outputs_buf.shape, dtype=torch.uint8).pin_memory()
        h2d = host_in.numel()
        d2h = host_out.numel()
        e2e_steps = max(3, min(steps, 200))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(e2e_steps):
            st.inputs_buf.copy_(host_in, non_blocking=True)
            run_step()
            host_out.copy_(st.outputs_buf, non_blocking=True)
        s1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1) / e2e_steps
    return dict(step_ms=step_ms, dec_ms=dec_ms, pre_ms=pre_ms, eager_ms=eager_ms,
                total_ms=sum(step_ms),
                clocks=clk, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h,
                launches=st.launches_per_step() * steps, reduce=st.reduce_launched,
                flushed=flush is not None)


# ------------------------------------------------------------------ CPU oracle timing

class OracleSample:
    """The CPU oracle as it stands (single-threaded C) on a bounded sample of the
    workload: the first few sequences, each in its own small pool.  One run =
    the write of the sequence's new tokens + fp64 attention of its queries, on
    the first ``heads`` kv heads (and their GQA query heads)."""

    def __init__(self, w, I, nseq, first=0):
        import oracle
        self.oracle, self.lib, self.w = oracle, oracle.load(), w
        self.per_tok = 2 * w.head_dim * (1 if w.cache_dtype == "i8" else 2) + (
            8 if w.cache_dtype == "i8" else 0)
        self.seqs = []
        for b in range(first, min(first + nseq, w.num_seqs)):
            L, C = int(w.context_lens[b]), int(w.q_lens[b])
            nblk = -(-L // w.block_size)
            c = oracle.Cache(w.cache_dtype, nblk, w.num_kv_heads, w.head_dim)
            kh, vh = I.history_rows(w, [b])
            slots = np.arange(L, dtype=np.int32)
            oracle.write_kv(c, kh[:L - C], vh[:L - C], I.source_dtype(w), slots[:L - C],
                            lib=self.lib)
            self.seqs.append(dict(L=L, C=C, nblk=nblk, cache=c, k=kh[L - C:], v=vh[L - C:],
                                  slot=slots[L - C:], q=I.query_rows(w, [b]), subs={}))
        self.src = I.source_dtype(w)

    def run(self, i, heads=None):
        w, o, sq = self.w, self.oracle, self.seqs[i % len(self.seqs)]
        heads = heads or w.num_kv_heads
        if heads not in sq["subs"]:
            c = sq["cache"]
            sub = o.Cache(w.cache_dtype, sq["nblk"], heads, w.head_dim, k=c.k[:, :heads],
                          v=c.v[:, :heads],
                          k_scale=None if c.k_scale is None else c.k_scale[:, :heads],
                          v_scale=None if c.v_scale is None else c.v_scale[:, :heads])
            sq["subs"][heads] = (sub, np.ascontiguousarray(sq["k"][:, :heads]),
                                 np.ascontiguousarray(sq["v"][:, :heads]),
                                 np.ascontiguousarray(sq["q"][:, :heads * w.group]))
        c, k, v, q = sq["subs"][heads]
        table = np.full((1, w.max_blocks_per_seq), -1, np.int32)
        table[0, :sq["nblk"]] = np.arange(sq["nblk"])
        L, C = sq["L"], sq["C"]
        t0 = time.perf_counter()
        o.write_kv(c, k, v, self.src, sq["slot"], lib=self.lib)
        o.attention(c, q, w.q_dtype, np.array([0, C], np.int32), table,
                    np.array([L], np.int32), window=w.window, lib=self.lib)
        dt = time.perf_counter() - t0
        lo = max(0, L - C - w.window + 1) if w.window > 0 else 0
        return (L - lo) * self.per_tok * heads, dt


def cpu_baseline(w, I, budget_s, nseq=8):
    """Repeat runs over the sample until ``budget_s`` seconds of oracle time."""
    smp = OracleSample(w, I, nseq)
    nbytes, spent, runs = 0, 0.0, 0
    while spent < budget_s:
        b, dt = smp.run(runs)
        nbytes, spent, runs = nbytes + b, spent + dt, runs + 1
    return nbytes / spent, len(smp.seqs), runs, spent


def _oracle_core_worker(name, seed, num_seqs, b, budget_s, barrier, results):
    """One process of the all-cores baseline: sequence ``b``'s sample, timed for
    ``budget_s`` seconds after every process has built its own."""
    try:
        from paged_kv_cache_240_gb300 import inputs as I
        w = I.make_workload(name, seed=seed, num_seqs=num_seqs)
        smp = OracleSample(w, I, 1, first=b % w.num_seqs)
        smp.run(0)                                        # untimed: first touch
        barrier.wait(timeout=300)
        nbytes, t0 = 0, time.time()
        while time.time() - t0 < budget_s:
            nbytes += smp.run(0)[0]
        results.put((b, nbytes, t0, time.time(), None))
    except Exception as e:  # reported by the parent, which then leaves the field out
        results.put((b, 0, 0.0, 0.0, repr(e)))


def cpu_baseline_all_cores(w, budget_s, seed=0, num_seqs=None, procs=None):
    """The same oracle, one process per host core (spawned, so that no process
    forks after the GPU is in use), each on its own sequence: bytes of all of
    them / the wall-clock window from the first start to the last end.
    Returns (GB/s, processes) or raises."""
    import multiprocessing as mp
    import queue as q
    n = procs or (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                  else os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(n), ctx.Queue()
    ps = [ctx.Process(target=_oracle_core_worker,
                      args=(w.name, seed, num_seqs, b, budget_s, barrier, results), daemon=True)
          for b in range(n)]
    for p in ps:
        p.start()
    got, deadline = [], time.time() + budget_s + 300
    try:
        while len(got) < n:
            try:
                got.append(results.get(timeout=1.0))
                if got[-1][4]:                    # failed: release the others too
                    barrier.abort()
                    raise RuntimeError(got[-1][4])
                continue
            except q.Empty:
                pass
            # a process that failed before reporting exits non-zero; the others
            # would wait for it at the barrier
            if any(p.exitcode not in (None, 0) for p in ps) or time.time() > deadline:
                barrier.abort()
                raise RuntimeError("%d of %d oracle processes reported" % (len(got), n))
    finally:
        for p in ps:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
    nbytes = sum(g[1] for g in got)
    window = max(g[3] for g in got) - min(g[2] for g in got)
    return nbytes / window / 1e9, n


# ------------------------------------------------------------------ INT8 linear

# Four 7B-shaped decoder layers' projections (n output channels, k inputs):
# q, k, v, o 4096x4096, gate and up 11008x4096, down 4096x11008 -- 810 MB of int8
# codes, over six times the L2, so every step streams the weights from HBM.  The
# projections that read the same activations run as one grouped launch: (q, k,
# v), (o), (gate, up), (down) -- four launches per layer.
LINEAR_LAYERS = 4
LINEAR_GROUPS = [[(4096, 4096)] * 3, [(4096, 4096)], [(11008, 4096)] * 2, [(4096, 11008)]]
LINEAR_SHAPES = [shape for grp in LINEAR_GROUPS for shape in grp]
LINEAR_METRIC = "weight-only INT8 linear: weight-read GB/s (% of GB300 HBM peak)"


def linear_bytes(m, groups):
    """Algorithmic bytes of one pass: every code and scale once, each group's
    activations in once and every output out (16-bit)."""
    return sum(sum(n * k + 4 * n + 2 * m * n for n, k in grp) + 2 * m * grp[0][1]
               for grp in groups)


class OracleLinearSample:
    """The oracle's INT8 linear (single-threaded C, fp64) on one 4096x4096 layer
    with the same token count: a bounded sample of the workload."""

    def __init__(self, m, I):
        import oracle
        self.oracle, self.lib, self.m = oracle, oracle.load(), m
        n = k = 4096
        rng = np.random.default_rng(7)
        self.codes = rng.integers(-127, 128, size=(n, k), dtype=np.int8)
        self.scales = (rng.random(n, dtype=np.float32) * 0.01 + 0.001).astype(np.float32)
        self.x = I.normal_bits((m, k), "bf16", 7, 1)
        self.bytes = linear_bytes(m, [[(n, k)]])

    def run(self):
        t0 = time.perf_counter()
        self.oracle.linear_int8(self.codes, self.scales, self.x, "bf16", lib=self.lib)
        return self.bytes, time.perf_counter() - t0


def linear_layers(torch, groups, m, seed, dev="cuda"):
    """Per group (x, [(codes, scales, y)]), drawn in order from one seeded
    generator on ``dev``: codes uniform in [-127, 127], scales uniform in
    [0.001, 0.011], m activation rows ~N(0, 1) in bf16 shared by the group, y the
    bf16 outputs."""
    gen = torch.Generator(device=dev).manual_seed(seed)
    out = []
    for grp in groups:
        k = grp[0][1]
        x = torch.randn((m, k), device=dev, generator=gen).to(torch.bfloat16)
        mats = []
        for n, _ in grp:
            codes = torch.randint(-127, 128, (n, k), dtype=torch.int8, device=dev, generator=gen)
            scales = torch.rand(n, device=dev, generator=gen) * 0.01 + 0.001
            y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            mats.append((codes, scales, y))
        out.append((x, mats))
    return out


def bench_linear(args):
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    m = args.num_seqs or 8
    layers = args.layers or LINEAR_LAYERS
    groups = LINEAR_GROUPS * layers
    step_bytes = linear_bytes(m, groups)
    cfg = {"workload": "int8-linear", "tokens": m, "layers": layers,
           "groups_n_k": LINEAR_GROUPS,
           "weight_bytes": sum(n * k for grp in groups for n, k in grp),
           "activation_dtype": "bf16", "l2": "inputs larger than L2"}
    from paged_kv_cache_240_gb300 import inputs as I
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        smp = OracleLinearSample(m, I)
        nbytes, secs = 0, 0.0
        for i in range(args.warmup + args.steps):
            b, dt = smp.run()
            if i >= args.warmup:
                nbytes, secs = nbytes + b, secs + dt
        value = nbytes / secs / 1e9
        print(json.dumps({
            "impl": "reference", "metric": LINEAR_METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(cfg, sample_bytes_per_step=nbytes / args.steps),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "per step: one 4096x4096 layer, %d tokens" % m},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return
    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    from __graft_entry__ import build
    build()
    from paged_kv_cache_240_gb300 import linear as L
    layers_dev = linear_layers(torch, groups, m, args.seed + 1000 * rank)
    # every group's activations in one device buffer, every output in another, so
    # that the end-to-end run moves each direction in one copy
    x_buf, xs = pack_tensors(torch, [x for x, _ in layers_dev], "cuda")
    y_buf, ys = pack_tensors(torch, [y for _, mats in layers_dev for _, _, y in mats], "cuda")
    it = iter(ys)
    layers_dev = [(x, [(c, sc, next(it)) for c, sc, _ in mats])
                  for x, (_, mats) in zip(xs, layers_dev)]
    launches = len(groups)  # one grouped launch per group, splits merged in the launch
    stream = torch.cuda.Stream()

    def step():
        for x, mats in layers_dev:
            L.int8_linear_grouped([(c, sc, None) for c, sc, _ in mats], x,
                                  outs=[y for _, _, y in mats])

    run = capture(torch, step, stream).replay if not args.no_graph else step
    try:
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        clocks.start()
        time.sleep(0.3)
        step_ms = time_replays(torch, stream, run, args.steps)
        if world > 1:
            torch.distributed.barrier()
        clk = clocks.stop()
        # end to end: every group's activations in from pinned memory, the outputs
        # back, each direction one copy of the packed buffer
        hx = x_buf.cpu().pin_memory()
        hy = torch.empty(y_buf.shape, dtype=torch.uint8).pin_memory()
        h2d, d2h = hx.numel(), hy.numel()
        e2e_steps = max(3, min(args.steps, 100))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(e2e_steps):
            x_buf.copy_(hx, non_blocking=True)
            run()
            hy.copy_(y_buf, non_blocking=True)
        s1.record(stream)
        torch.cuda.synchronize()
    total_ms, e2e_ms = max_over_ranks(torch, [sum(step_ms), s0.elapsed_time(s1) / e2e_steps],
                                      world)
    ms_per_step = total_ms / args.steps
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    peaks, peak_kind = measured_peaks()
    src = peak_kind + " (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    achieved = step_bytes / (statistics.median(step_ms) * 1e-3) / 1e9
    line = {"metric": LINEAR_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i8xbf16",
            "data": "synthetic (random int8 codes and bf16 activations)", "config": cfg,
            "clocks": clk,
            "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         # the record is of the default stack (four layers, 8 tokens)
                         "traffic": (recorded_traffic("int8-linear", "linear")
                                     if (layers, m) == (LINEAR_LAYERS, 8) else None),
                         "kernel": "pa_linear_int8_grouped (int8 codes -> exact f16, mma.sync "
                                   "m16n8k16; k splits merged over distributed shared memory)",
                         "peak_source": src + " hbm_gbs",
                         "frac_of_nominal": achieved / NOMINAL["GB/s"]},
            "p10_p50_p90_step_ms": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleLinearSample(m, I)
        nb, spent, runs = 0, 0.0, 0
        while spent < args.cpu_budget:
            b, dt = smp.run()
            nb, spent, runs = nb + b, spent + dt, runs + 1
        line["cpu_baseline"] = {"value": nb / spent / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle",
                                "sample": "%d runs of one 4096x4096 layer with %d tokens, %.1f s"
                                          % (runs, m, spent)}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ main

# The other configurations of the method's workloads, measured after the headline
# in the default single-GPU run and reported under "workloads".
EXTRA_WORKLOADS = ("int8-kv", "qwen2.5-1.5b", "mixed", "spec-verify")
EXTRA_MIN_STEPS = 200  # the small steps (16 us - 0.3 ms) need more than a handful


def workload_config(w):
    """The ``config`` object of a paged-attention workload's line."""
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_decode": w.num_decode,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "cache_dtype": w.cache_dtype,
            "q_dtype": w.q_dtype, "window": w.window, "num_blocks": w.num_blocks,
            "mean_context": float(w.context_lens[:w.num_decode].mean() if w.num_decode
                                  else w.context_lens.mean()),
            "kv_bytes_per_step": w.kv_bytes(),
            "l2": ("L2 flushed before every timed run (a %d MB buffer written); the e2e "
                   "loop is not flushed" % (2 * L2_BYTES >> 20)) if needs_l2_flush(w) else
                  "inputs larger than L2 (%d MB of KV per step)" % (w.kv_bytes() >> 20)}


def measure(args, w, torch, pa, I, rank, world, steps, warmup, peaks, src):
    """One workload's timed steps -> the fields of its JSON line (value, timing,
    roofline of the dominant call, clocks, end to end, launch count)."""
    r = time_ours(args, w, torch, pa, I, rank, world, steps, warmup)
    total_ms, e2e_ms = max_over_ranks(torch, [r["total_ms"], r["e2e_ms"]], world)
    kv_step = w.kv_bytes()
    ms_per_step = total_ms / steps
    value = world * kv_step / (ms_per_step * 1e-3) / 1e9
    dec_ms, pre_ms = statistics.mean(r["dec_ms"]), statistics.mean(r["pre_ms"])
    # recorded DRAM traffic belongs to the workload as defined: none for variants
    roof = roofline(w, dec_ms, pre_ms, peaks, src,
                    full_size=args.num_seqs is None and not getattr(args, "cache_dtype", None))
    cfg = workload_config(w)
    cfg["launch"] = "python calls" if args.no_graph else "CUDA graph replay of the step"
    if w.num_decode and w.num_decode < w.num_seqs:
        cfg["streams"] = "prefill call on a second stream, launched before the decode call"
    fields = {"value": value, "unit": "GB/s", "steps": steps, "warmup": warmup,
              "ms_per_step": ms_per_step, "steps_per_s": 1e3 / ms_per_step * world,
              "hbm_frac": value / peaks["hbm_gbs"], "config": cfg, "clocks": r["clocks"],
              "l2_flushed": r["flushed"],
              "e2e": {"value": world * kv_step / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                      "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
              "gpu_launches": r["launches"], "roofline": roof,
              "decode_call_ms": dec_ms, "prefill_call_ms": pre_ms,
              "p10_p50_p90_step_ms": [float(np.percentile(r["step_ms"], p)) for p in (10, 50, 90)],
              "median_step_ms_python_launches": float(np.median(r["eager_ms"]))}
    if roof["bound"] == "tensor" and dec_ms > 0:
        # the decode half of a mixed step, against HBM
        achieved = decode_kv_bytes(w) / (dec_ms * 1e-3) / 1e9
        fields["decode_roofline"] = {"bound": "hbm", "achieved": achieved,
                                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                     "frac": achieved / peaks["hbm_gbs"],
                                     "kernel": "pa_decode", "peak_source": src + " hbm_gbs"}
    return fields


def reference_line(args, w, I):
    """The oracle (single-threaded C, fp64) timed on a bounded sample of the
    workload per step: the line reports what was measured -- the sample's bytes
    over the sample's time -- and says what the sample was."""
    import oracle
    oracle.build()
    smp = OracleSample(w, I, nseq=4)
    # size each step's sample so that the whole run stays near two minutes
    per_step_s = min(args.cpu_budget, 120.0 / max(1, args.warmup + args.steps))
    b, dt = smp.run(0)
    heads = max(1, min(w.num_kv_heads, int(w.num_kv_heads * per_step_s / max(dt, 1e-6))))
    nbytes, secs = 0, 0.0
    for i in range(args.warmup + args.steps):
        b, dt = smp.run(i, heads)
        if i >= args.warmup:
            nbytes, secs = nbytes + b, secs + dt
    value = nbytes / secs / 1e9
    sample = ("per step: one of the first %d sequences (whole context), %d of %d kv heads: "
              "write of its new tokens + fp64 attention of its queries; %.3f MB and %.3f s per "
              "step on average" % (len(smp.seqs), heads, w.num_kv_heads,
                                   nbytes / args.steps / 1e6, secs / args.steps))
    cfg = workload_config(w)
    cfg["sample_bytes_per_step"] = nbytes / args.steps
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every call from Python instead of replaying a CUDA graph")
    ap.add_argument("--layers", type=int, default=None,
                    help="int8-linear only: layers per step (default %d)" % LINEAR_LAYERS)
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="fewer decoding sequences (small profiling captures)")
    ap.add_argument("--cache-dtype", choices=["f16", "bf16", "i8"], default=None,
                    help="the workload's shapes over a cache of this type (a 16-bit cache "
                         "takes queries of its own type; an int8 one keeps the workload's)")
    ap.add_argument("--extra-workloads", default="auto",
                    help="comma-separated workloads measured after the headline and reported "
                         "under 'workloads'; 'auto' = %s on one GPU with the default workload, "
                         "'none' = no others" % ",".join(EXTRA_WORKLOADS))
    args = ap.parse_args()

    if args.workload == "int8-linear":
        bench_linear(args)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    from paged_kv_cache_240_gb300 import inputs as I
    w = I.make_workload(args.workload, seed=args.seed, num_seqs=args.num_seqs)
    if args.cache_dtype:
        w.cache_dtype = args.cache_dtype
        if args.cache_dtype != "i8":
            w.q_dtype = args.cache_dtype

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_line(args, w, I)))
        return

    if args.extra_workloads == "auto":
        extras = list(EXTRA_WORKLOADS) if (world == 1 and args.workload == DEFAULT_WORKLOAD) \
            else []
    elif args.extra_workloads in ("", "none"):
        extras = []
    else:
        extras = [x for x in args.extra_workloads.split(",") if x and x != args.workload]

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    from __graft_entry__ import build
    build()
    import paged_kv_cache_240_gb300 as pa
    peaks, peak_kind = measured_peaks()
    src = peak_kind + " (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    f = measure(args, w, torch, pa, I, rank, world, args.steps, args.warmup, peaks, src)
    line = {"metric": METRIC, "value": f["value"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": f["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.cache_dtype, "data": "synthetic", "config": f["config"]}
    line.update({k: v for k, v in f.items() if k not in line and k not in ("steps", "warmup")})
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, nseq, runs, spent = cpu_baseline(w, I, args.cpu_budget)
        line["cpu_baseline"] = {
            "value": v / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d runs over the first %d of %d sequences (whole contexts, all heads): "
                      "write of each one's new tokens + fp64 attention of its queries, "
                      "%.1f s of CPU time" % (runs, nseq, w.num_seqs, spent)}
        try:
            va, procs = cpu_baseline_all_cores(w, args.cpu_budget, args.seed, args.num_seqs)
            line["cpu_baseline"]["all_cores"] = {
                "value": va, "unit": "GB/s", "cores": procs,
                "sample": "%d concurrent processes, process i on sequence i (whole context, "
                          "all heads), %.0f s each; bytes of all / wall-clock window"
                          % (procs, args.cpu_budget)}
        except Exception as e:  # the single-thread figure above stands alone
            line["cpu_baseline"]["all_cores"] = {"unavailable": str(e)[:200]}
    if extras:
        # the other configurations, one at a time, each pool freed before the next
        line["workloads"] = {}
        for name in extras:
            torch.cuda.empty_cache()
            wx = I.make_workload(name, seed=args.seed, num_seqs=args.num_seqs)
            line["workloads"][name] = measure(
                args, wx, torch, pa, I, rank, world, max(args.steps, EXTRA_MIN_STEPS),
                max(args.warmup, 3), peaks, src)
        torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
