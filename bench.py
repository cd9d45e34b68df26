"""Benchmark of the GDN hot path on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]
                    [--workload all|decode|verify|prefill_kda|prefill_varlen|...]

Headline workload: batched decode, 64 sequences x 1 token, H=16,
D_k=D_v=128, GDA gate, bf16 q/k/v, fp32 state ~N(0, 0.05); one step is one
decode step (64 tokens) through gdn_forward. The default run (--workload
all) then measures speculative verify, the KDA chunked prefill and the varlen
GDA chunked prefill the same way (K timed steps after W warm-up steps each),
and reports them under "workloads" in the same JSON line. Prints ONE JSON
line on rank 0. Inputs are resident in HBM when the timed region starts; the
inputs of every workload are larger than the L2 (decode rotates over enough
state banks that every step reads its state from HBM). The "e2e" figure
repeats the measurement with each step's inputs copied from pinned host
memory and the outputs copied back, inside the timed region. Decode takes
its host buffers through gdn_forward_host (the kernel reads the pinned host
inputs and writes the pinned host outputs over the host link itself, all on
the launch stream), with the copy-engine pipeline (copies on their own
streams, overlapping neighbouring calls) reported beside it; the other
workloads use the copy-engine pipeline.

--impl reference times the fp64 CPU oracle (a deliberately slow baseline) on
the same workload, on this host's cores, on a bounded sample per step.
Under torchrun every rank runs its own replica (weak scaling); the time is the
max over ranks.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_net_02_gb300 import inputs  # noqa: E402

METRIC = "GDN tokens/s (decode, verify, prefill); % of HBM GB/s or tensor peak"
FALLBACK_HBM_GBS = 6800.0
E2E_HOST_PATH = ("gdn_forward_host: each call reads its step's inputs from pinned host "
                 "memory and writes its output to pinned host memory over the host link "
                 "itself, one stream, no copy engine")
E2E_COPY_PATH = ("gdn_forward(_chunked) on device buffers: one pinned host-to-device copy "
                 "per step on a copy-in stream, one device-to-host copy of the output on a "
                 "copy-out stream, overlapping the neighbouring steps' calls")
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------- utilities

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(ms, ms_e2e, tokens_per_step, K, ws, device):
    """Whole-job figures of a replicated run: each rank timed K steps of its
    own replica (ms, ms_e2e); the job's time is the slowest rank's, and its
    tokens are every rank's. Uses a MAX all-reduce when ws > 1 (any backend).
    Returns (ms_max, ms_e2e_max, tokens/s, e2e tokens/s)."""
    t = torch.tensor([ms, ms_e2e], dtype=torch.float64, device=device)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max, ms_e2e_max = t.tolist()
    tokens_all = tokens_per_step * K * ws
    return ms_max, ms_e2e_max, tokens_all / (ms_max / 1e3), tokens_all / (ms_e2e_max / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_delta_net_02_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, sha):
    """Per-launch DRAM bytes of `kernel_key` from the committed ncu summary,
    if it was taken on the current kernel source (same hash)."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        with open(path) as f:
            for line in f:
                parts = line.strip().strip("|").split("|")
                parts = [p.strip() for p in parts]
                if len(parts) >= 3 and parts[0] == kernel_key and parts[1] == sha:
                    return float(parts[2])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        self.f.close()
        os.unlink(self.f.name)
        return rows


def summarize_clocks(rows, t0, t1):
    """Median SM clock and active throttle reasons of the samples taken while
    the timed region ran (wall-clock window [t0, t1])."""
    import datetime
    picked = []
    for r in rows:
        if len(r) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            continue
        picked.append((ts, r))
    inside = [r for ts, r in picked if t0 <= ts <= t1]
    note = "samples inside the timed region"
    if not inside and picked:
        # region shorter than the sampling period: nearest samples around it
        near = sorted(picked, key=lambda x: min(abs(x[0] - t0), abs(x[0] - t1)))[:3]
        inside = [r for _, r in near]
        note = "timed region shorter than the sampling period; nearest samples"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"],
                "samples": 0}
    sm = [float(r[2]) for r in inside if r[2].strip().replace(".", "").isdigit()]
    smax = [float(r[3]) for r in inside if r[3].strip().replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in inside for i in range(4)
                      if r[6 + i].strip().lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": reasons, "samples": len(inside), "note": note}


def timed_graph_steps(graphs, K, stream):
    """Replays `graphs` (list of (graph, n_steps)) to cover exactly K steps;
    returns elapsed ms from CUDA events on `stream`."""
    plan = []
    left = K
    full, full_n = graphs[0]
    while left >= full_n:
        plan.append(full)
        left -= full_n
    for g, n in graphs[1:]:
        if left >= n:
            plan.append(g)
            left -= n
    assert left == 0, "graph plan does not cover K"
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        start.record(stream)
        for g in plan:
            g.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def capture(fn_steps, stream, steps, pre=None, post=None):
    """CUDA graph of `steps` consecutive calls fn_steps(i) for i in steps
    (with pre() before and post() after them, inside the capture)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        if pre:
            pre()
        for i in steps:
            fn_steps(i)
        if post:
            post()
    return g


# ----------------------------------------------------------------- workloads

class PackedInputs:
    """End-to-end staging: a step's host inputs (q, k, v, g, beta) packed at
    256-byte offsets in one pinned buffer per step, copied with one
    host-to-device copy into one of two device buffers of the same layout
    (double-buffered, so that the next step's copy can run during this step),
    whose typed views are what the API call receives."""

    def __init__(self, host, dev):
        # host: tensors with a leading step dimension [P, ...] (P may be 1)
        P = host[0].shape[0]
        self.offs, self.nbytes = [], []
        off = 0
        for t in host:
            nb = t[0].numel() * t.element_size()
            self.offs.append(off)
            self.nbytes.append(nb)
            off = (off + nb + 255) // 256 * 256
        self.step_bytes = off
        self.host = torch.zeros(P, off, dtype=torch.uint8).pin_memory()
        for t, o, nb in zip(host, self.offs, self.nbytes):
            self.host[:, o:o + nb].copy_(t.reshape(P, -1).view(torch.uint8))
        self.stage = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.views = [[st[o:o + nb].view(t.dtype).view(t.shape[1:])
                       for t, o, nb in zip(host, self.offs, self.nbytes)] for st in self.stage]

    def copy_in(self, p, b):
        """Host step p into device buffer b (on the current stream)."""
        self.stage[b].copy_(self.host[p], non_blocking=True)
        return self.views[b]

    def host_views(self, p):
        """Typed views of host step p itself (pinned, for gdn_forward_host)."""
        return [self.host[p, o:o + nb].view(v.dtype).view(v.shape)
                for v, o, nb in zip(self.views[0], self.offs, self.nbytes)]


class E2EPipeline:
    """End-to-end steps with the copies of neighbouring steps overlapping:
    step i's inputs go host -> device buffer i % 2 on a copy-in stream, the
    API call runs on the launch stream once they have landed (and once the
    output buffer i % 2 has been read back by step i - 2), and step i's output
    goes device -> pinned host on a copy-out stream after the call. Every
    step's two copies stay inside the timed region; captured into the same
    CUDA graph as the calls (event edges between the three streams)."""

    def __init__(self, wl, dev):
        self.wl = wl
        self.cs_in = torch.cuda.Stream(device=dev)
        self.cs_out = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]

    def begin(self, stream):
        ev = torch.cuda.Event()
        ev.record(stream)
        self.cs_in.wait_event(ev)
        self.cs_out.wait_event(ev)
        self.used = [False, False]

    def step(self, i, stream):
        wl, b = self.wl, i % 2
        with torch.cuda.stream(self.cs_in):
            if self.used[b]:   # buffer b was last read by the call of step i - 2
                self.cs_in.wait_event(self.ev_done[b])
            views = wl.packed.copy_in(wl.e2e_host_index(i), b)
            self.ev_in[b].record(self.cs_in)
        stream.wait_event(self.ev_in[b])
        if self.used[b]:       # output b of step i - 2 has been read back
            stream.wait_event(self.ev_out[b])
        wl.e2e_call(i, views, wl.out2[b], stream)
        self.ev_done[b].record(stream)
        with torch.cuda.stream(self.cs_out):
            self.cs_out.wait_event(self.ev_done[b])
            wl.out_host2[b].copy_(wl.out2[b], non_blocking=True)
            self.ev_out[b].record(self.cs_out)
        self.used[b] = True

    def end(self, stream):
        for b in range(2):
            if self.used[b]:
                stream.wait_event(self.ev_out[b])
                stream.wait_event(self.ev_in[b])


class HostIOPipeline:
    """End-to-end steps through gdn_forward_host: the call of step i reads
    that step's inputs straight from its slice of the pinned host pool and
    writes its output into pinned host buffer i % 2, over the host link, on
    the launch stream; no copy-engine transfer and no cross-stream event
    between consecutive calls."""

    def __init__(self, wl, dev):
        self.wl = wl
        self.views = [wl.packed.host_views(p) for p in range(wl.packed.host.shape[0])]

    def begin(self, stream):
        pass

    def step(self, i, stream):
        wl = self.wl
        wl.e2e_call_host(i, self.views[wl.e2e_host_index(i)], wl.out_host2[i % 2], stream)

    def end(self, stream):
        pass


class Decode:
    """64 sequences x 1 token, H=16, D=128, GDA, bf16 q/k/v, fp32 state.

    Cold-L2 protocol: SETS independent decode batches, each with its own
    double-buffered state; step i advances batch i % SETS, so between two
    steps of one batch the other batches move (SETS-1) x 128 MiB through
    the memory system and its state is read from HBM, not L2."""
    compute_dtype = "f32"   # fp32 state arithmetic on CUDA cores (bf16 inputs widened)
    N, H, D = 64, 16, 128
    POOL = 256      # distinct token steps resident on the device
    SETS = 8        # independent batches (8 x 2 x 64 MiB = 1 GiB)
    name = "decode"

    @property
    def tokens_per_step(self):
        return self.N

    def config(self):
        return {"workload": "batched decode: 64 sequences x 1 token, H=16, D_k=D_v=128, GDA "
                            "scalar gate, bf16 q/k/v, fp32 state ~N(0,0.05), K=1 slot",
                "n_seqs": self.N, "heads": self.H, "D_k": self.D, "D_v": self.D,
                "tokens_per_step": self.N, "input_dtype": "bf16", "state_dtype": "f32",
                "l2": f"inputs larger than L2: {self.SETS} independent 64-sequence decode "
                      f"batches advance in turn (each step's 64 MiB state was last written "
                      f"{self.SETS - 1} steps earlier), {self.POOL} distinct token steps",
                "timing": "CUDA graphs of consecutive steps, CUDA events on the launch stream"}

    def launches_per_step(self):
        return 1   # recurrent_kernel

    def alg_bytes_per_step(self):
        D = self.D
        per = 8 * D * D + (2 * D + D) * 2 + 4 + 4 + 4 * D   # 132,360 B per token-head
        return per * self.N * self.H

    def setup(self, gdn, dev):
        N, H, D = self.N, self.H, self.D
        self.gdn = gdn
        s0 = inputs.decode_state(1, N, H, D).to(dev)
        self.bufs = [[s0.clone(), torch.empty_like(s0)] for _ in range(self.SETS)]
        del s0
        self.buf_ptrs = [[gdn.state_ptr_array(gdn.per_seq_state_ptrs(b, N), dev) for b in pair]
                         for pair in self.bufs]
        toks = [inputs.decode_tokens(1, s, N, H, D) for s in range(self.POOL)]
        self.host = [torch.stack([t[i] for t in toks]) for i in range(5)]  # q,k,v,g,beta
        self.dev = [h.to(dev) for h in self.host]
        self.out = torch.empty(N, H, D, device=dev)
        self.shape = gdn.gdn_shape(N, 1, H, D, D, gdn.GDN_BF16, D ** -0.5)
        # e2e: packed pinned host pool, one device staging buffer, pinned output
        self.packed = PackedInputs(self.host, dev)
        self.out2 = [self.out, torch.empty_like(self.out)]
        self.out_host2 = [torch.empty(N, H, D, dtype=torch.float32).pin_memory()
                          for _ in range(2)]
        self.h2d_bytes = self.packed.step_bytes
        self.d2h_bytes = self.out.numel() * 4

    def _bufs(self, i):
        """(state_in pointer array, slot buffer) of step i: batch i % SETS,
        ping-ponging between its two state buffers."""
        b = i % self.SETS
        parity = (i // self.SETS) % 2
        return self.buf_ptrs[b][parity], self.bufs[b][1 - parity]

    def step(self, i, stream):
        p = i % self.POOL
        src, dst = self._bufs(i)
        q, k, v, g, beta = (t[p] for t in self.dev)
        self.gdn.gdn_forward(self.shape, q, k, v, g, beta, src, dst, self.out, 1, "gda",
                             stream)

    def e2e_host_index(self, i):
        return i % self.POOL

    def e2e_call(self, i, views, out, stream):
        q, k, v, g, beta = views
        src, dst = self._bufs(i)
        self.gdn.gdn_forward(self.shape, q, k, v, g, beta, src, dst, out, 1, "gda", stream)

    def e2e_call_host(self, i, views, out, stream):
        q, k, v, g, beta = views
        src, dst = self._bufs(i)
        self.gdn.gdn_forward_host(self.shape, q, k, v, g, beta, src, dst, out, 1, "gda",
                                  stream)

    def graph_len(self):
        return self.POOL  # a multiple of 2 x SETS: replays continue every chain

    def step_in_place(self, i, stream):
        """One batch stepping in place (its 64 MiB state ping-pongs between two
        buffers and stays largely in L2): reported beside the headline,
        labelled, never as it."""
        p = i % self.POOL
        src, dst = self.buf_ptrs[0][i % 2], self.bufs[0][1 - i % 2]
        q, k, v, g, beta = (t[p] for t in self.dev)
        self.gdn.gdn_forward(self.shape, q, k, v, g, beta, src, dst, self.out, 1, "gda",
                             stream)

    # ---- CPU oracle on a bounded sample of the same workload
    def oracle_step_fn(self, n_seqs, threads=0):
        import oracle
        N, H, D = self.N, self.H, self.D
        st = inputs.to_f64(inputs.decode_state(1, N, H, D)[:n_seqs])
        pool = [inputs.decode_tokens(1, s, N, H, D) for s in range(4)]
        pool = [[inputs.to_f64(t[:n_seqs]) for t in toks] for toks in pool]
        state = {"S": st, "i": 0}

        def run():
            q, k, v, g, beta = pool[state["i"] % len(pool)]
            _, S, _ = oracle.forward(q, k, v, g, beta, state["S"], scale=D ** -0.5,
                                     threads=threads)
            state["S"] = S
            state["i"] += 1
            return n_seqs  # tokens processed
        return run


class Verify(Decode):
    """32 sequences x T=8 tokens (draft_max 7), K=8 slots, H=16, D=128, GDA."""
    N, T, K, H, D = 32, 8, 8, 16, 128
    POOL = 64
    BANKS = 4
    name = "verify"

    @property
    def tokens_per_step(self):
        return self.N * self.T

    def config(self):
        return {"workload": "speculative verify: 32 sequences x T=8 tokens, K=8 snapshot slots, "
                            "H=16, D_k=D_v=128, GDA, bf16 q/k/v, fp32 state",
                "n_seqs": self.N, "T": self.T, "n_slots": self.K, "heads": self.H,
                "tokens_per_step": self.N * self.T, "input_dtype": "bf16",
                "l2": "inputs larger than L2: 256 MiB of slots written per call, "
                      f"{self.BANKS} rotating input-state banks",
                "timing": "CUDA graphs of consecutive calls, CUDA events on the launch stream"}

    def alg_bytes_per_step(self):
        D = self.D
        per_seq_head = 4 * D * D * (1 + self.K) + self.T * ((2 * D + D) * 2 + 8 + 4 * D)
        return per_seq_head * self.N * self.H

    def setup(self, gdn, dev):
        N, T, H, D, K = self.N, self.T, self.H, self.D, self.K
        self.gdn = gdn
        base = inputs.verify_batch(2, N, T, H, D, K)
        self.banks = [base.state.to(dev)] + [
            (base.state + 0.001 * j).to(dev) for j in range(1, self.BANKS)]
        self.bank_ptrs = [gdn.state_ptr_array(gdn.per_seq_state_ptrs(b, N), dev)
                          for b in self.banks]
        pool = [inputs.make_batch(1000 + s, [T] * N, H, D, D, n_slots=K, state_std=0.0)
                for s in range(self.POOL)]
        self.host = [torch.stack([getattr(b, n) for b in pool])
                     for n in ("q", "k", "v", "g", "beta")]
        self.dev = [h.to(dev) for h in self.host]
        self.slots = torch.empty(N, K, H, D, D, device=dev)
        self.out = torch.empty(N * T, H, D, device=dev)
        self.shape = gdn.gdn_shape(N, T, H, D, D, gdn.GDN_BF16, D ** -0.5)
        self.packed = PackedInputs(self.host, dev)
        self.out2 = [self.out, torch.empty_like(self.out)]
        self.out_host2 = [torch.empty(N * T, H, D, dtype=torch.float32).pin_memory()
                          for _ in range(2)]
        self.h2d_bytes = self.packed.step_bytes
        self.d2h_bytes = self.out.numel() * 4

    def step(self, i, stream):
        p = i % self.POOL
        q, k, v, g, beta = (t[p] for t in self.dev)
        self.gdn.gdn_forward(self.shape, q, k, v, g, beta, self.bank_ptrs[i % self.BANKS],
                             self.slots, self.out, self.K, "gda", stream)

    def e2e_call(self, i, views, out, stream):
        q, k, v, g, beta = views
        self.gdn.gdn_forward(self.shape, q, k, v, g, beta, self.bank_ptrs[i % self.BANKS],
                             self.slots, out, self.K, "gda", stream)

    # No e2e_call_host: a verify call's 3.2 MB of tokens would cross the host
    # link at the start of every CTA, ahead of its compute (4.07 M tokens/s
    # end to end, measured), while copy-engine transfers of the next call's
    # tokens overlap this call (4.64 M tokens/s).
    e2e_call_host = None

    def graph_len(self):
        return self.POOL

    def oracle_step_fn(self, n_seqs, threads=0):
        import oracle
        b = inputs.verify_batch(2, self.N, self.T, self.H, self.D, self.K)
        sl = slice(0, n_seqs * self.T)
        args = [inputs.to_f64(getattr(b, n)[sl]) for n in ("q", "k", "v", "g", "beta")]
        S0 = inputs.to_f64(b.state[:n_seqs])

        def run():
            oracle.forward(*args, S0, scale=self.D ** -0.5, n_slots=self.K, threads=threads)
            return n_seqs * self.T
        return run


class Prefill:
    """Chunked prefill through gdn_forward_chunked; one step = one call."""
    name = "prefill"
    SETS = 2        # rotating input sets, each larger than half the L2
    mode = "gda"

    def batch(self, j):
        raise NotImplementedError

    def setup(self, gdn, dev):
        self.gdn = gdn
        self.sets = []
        for j in range(self.SETS):
            b = self.batch(j)
            d = {n: getattr(b, n).to(dev) for n in ("q", "k", "v", "g", "beta", "state")}
            d["cu"] = b.cu_seqlens.to(torch.int32).to(dev)
            d["ptrs"] = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], b.n_seqs), dev)
            self.sets.append((b, d))
        b0 = self.sets[0][0]
        self.b0 = b0
        self.N, self.H = b0.n_seqs, b0.q.shape[1]
        self.ntok = b0.q.shape[0]
        self.K = b0.n_slots
        self.shape = gdn.gdn_varlen_shape(self.N, self.ntok, self.H, 128, 128,
                                          gdn.dtype_code(b0.q.dtype), b0.scale)
        self.ws_bytes = gdn.gdn_chunked_workspace_size(self.shape, self.K)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.slots = torch.empty(self.N, self.K, self.H, 128, 128, device=dev)
        self.out = torch.empty(self.ntok, self.H, 128, device=dev)
        self.packed = PackedInputs([getattr(b0, n).unsqueeze(0)
                                    for n in ("q", "k", "v", "g", "beta")], dev)
        self.out2 = [self.out, torch.empty_like(self.out)]
        self.out_host2 = [torch.empty(self.ntok, self.H, 128).pin_memory() for _ in range(2)]
        self.h2d_bytes = self.packed.step_bytes
        self.d2h_bytes = self.out.numel() * 4

    @property
    def tokens_per_step(self):
        return self.ntok

    in_bytes = 2    # q, k, v element size
    # tensor-core products of bf16 operands, fp32 accumulation and state
    compute_dtype = "bf16"

    def launches_per_step(self):
        if self.in_bytes == 4:
            return 2   # work list, recurrent kernel (token-loop route)
        return 4       # work list, chunk prep, chunk scan, recurrent tail

    def alg_bytes_per_step(self):
        g_bytes = 4 * 128 if self.mode == "kda" else 4
        per_tok_head = 3 * 128 * self.in_bytes + g_bytes + 4 + 4 * 128
        state = 2 * self.N * self.H * 128 * 128 * 4 + self.N * self.K * self.H * 128 * 128 * 4
        return per_tok_head * self.ntok * self.H + state

    def alg_flops_per_step(self):
        C, D = 64, 128
        return (2 * C * (3 * D + 2 * D) + 6 * D * D) * self.ntok * self.H

    def _call(self, d, q, k, v, g, beta, stream, out=None):
        self.gdn.gdn_forward_chunked(self.shape, d["cu"], q, k, v, g, beta, d["ptrs"],
                                     self.slots, self.out if out is None else out, self.K,
                                     self.mode, self.ws, self.ws_bytes, stream)

    def step(self, i, stream):
        _, d = self.sets[i % self.SETS]
        self._call(d, d["q"], d["k"], d["v"], d["g"], d["beta"], stream)

    def e2e_host_index(self, i):
        return 0

    def e2e_call(self, i, views, out, stream):
        q, k, v, g, beta = views
        _, d = self.sets[0]
        self._call(d, q, k, v, g, beta, stream, out)

    def graph_len(self):
        return 4

    def oracle_step_fn(self, n_seqs, threads=0):
        import oracle
        b = self.batch(0)
        cu = b.cu_seqlens
        self.ntok, self.H, self.K = b.q.shape[0], b.q.shape[1], b.n_slots
        H = max(1, min(self.H, n_seqs))   # bounded sample: a subset of the heads
        args = [inputs.to_f64(getattr(b, n)[:, :H]) for n in ("q", "k", "v", "g", "beta")]
        S0 = inputs.to_f64(b.state[:, :H])

        def run():
            oracle.forward(*args, S0, mode=self.mode, scale=b.scale, n_slots=self.K,
                           seq_start=cu[:-1].numpy(), seq_len=b.seq_len.numpy(),
                           threads=threads)
            return self.ntok * H / self.H
        return run


class PrefillKDA(Prefill):
    name = "prefill_kda"
    mode = "kda"
    N = 1

    def batch(self, j):
        return inputs.kda_prefill(3 + 100 * j)

    def config(self):
        return {"workload": "KDA per-row-gate chunked prefill: 1 sequence x T=4096, H=32, "
                            "D_k=D_v=128, bf16 q/k/v, fp32 g [T,H,D_k] and state, K=1",
                "tokens_per_step": 4096, "heads": 32, "chunk": 64,
                "l2": "inputs larger than L2: 2 rotating input sets of 240 MB",
                "timing": "CUDA graphs of consecutive calls, CUDA events on the launch stream"}


class PrefillVarlen(Prefill):
    name = "prefill_varlen"
    mode = "gda"
    N = 8

    def batch(self, j):
        # every set keeps the lengths drawn with seed 4; values differ per set
        lens = inputs.varlen_lengths(4)
        return inputs.make_batch(5 + 100 * j, lens, 16, 128, 128, mode="gda",
                                 state_std=0.05, n_slots=8)

    def config(self):
        return {"workload": "varlen GDA chunked prefill: 8 sequences, lengths ~U[512,8192] "
                            "(seed 4), H=16, D_k=D_v=128, bf16 q/k/v, fp32 state, K=8 slots",
                "tokens_per_step": int(inputs.varlen_lengths(4).sum()), "heads": 16,
                "chunk": 64,
                "l2": "inputs larger than L2: 2 rotating input sets",
                "timing": "CUDA graphs of consecutive calls, CUDA events on the launch stream"}


class PrefillVarlenF32(PrefillVarlen):
    """The varlen batch with fp32 q/k/v: gdn_forward_chunked takes the token
    loop (the recurrent kernel) for every token."""
    name = "prefill_varlen_fp32"
    in_bytes = 4
    compute_dtype = "f32"   # token loop on CUDA cores

    def batch(self, j):
        lens = inputs.varlen_lengths(4)
        return inputs.make_batch(5 + 100 * j, lens, 16, 128, 128, dtype=torch.float32,
                                 mode="gda", state_std=0.05, n_slots=8)

    def config(self):
        c = super().config()
        c["workload"] = ("varlen GDA prefill with fp32 q/k/v (token-loop route of "
                         "gdn_forward_chunked): 8 sequences, lengths ~U[512,8192] (seed 4), "
                         "H=16, D_k=D_v=128, fp32 state, K=8 slots")
        c.pop("chunk", None)
        return c


class DecodeGQA(Decode):
    """The decode step with grouped-query heads: 4 q/k heads read by the 16
    value heads (grouped map)."""
    H_QK = 4
    name = "decode_gqa"

    def config(self):
        c = super().config()
        c["workload"] = ("batched decode with grouped-query heads: 64 sequences x 1 token, "
                         "H=16 value heads reading H_qk=4 q/k heads (grouped), D_k=D_v=128, "
                         "GDA, bf16 q/k/v, fp32 state, K=1 slot")
        c["H_qk"] = self.H_QK
        return c

    def alg_bytes_per_step(self):
        D = self.D
        per_head = 8 * D * D + D * 2 + 4 + 4 + 4 * D       # state r+w, v, g, beta, out
        return self.N * (self.H * per_head + self.H_QK * 2 * D * 2)

    def setup(self, gdn, dev):
        super().setup(gdn, dev)
        hq = self.H_QK
        for lst in (self.host, self.dev):
            for i in (0, 1):  # q, k keep their first H_qk heads
                lst[i] = lst[i][:, :, :hq].contiguous()
        self.packed = PackedInputs(self.host, dev)
        self.h2d_bytes = self.packed.step_bytes
        self.shape = gdn.gdn_shape(self.N, 1, self.H, self.D, self.D, gdn.GDN_BF16,
                                   self.D ** -0.5, hq, gdn.GDN_QK_GROUPED)

    def oracle_step_fn(self, n_seqs, threads=0):
        import oracle
        N, H, D, hq = self.N, self.H, self.D, self.H_QK
        st = inputs.to_f64(inputs.decode_state(1, N, H, D)[:n_seqs])
        pool = []
        for s_ in range(4):
            q, k, v, g, beta = (inputs.to_f64(t[:n_seqs]) for t in inputs.decode_tokens(1, s_, N, H, D))
            pool.append((q[:, :hq].copy(), k[:, :hq].copy(), v, g, beta))
        state = {"S": st, "i": 0}

        def run():
            q, k, v, g, beta = pool[state["i"] % len(pool)]
            _, S, _ = oracle.forward(q, k, v, g, beta, state["S"], scale=D ** -0.5,
                                     threads=threads, qk_map="grouped")
            state["S"] = S
            state["i"] += 1
            return n_seqs
        return run
class PrefillVarlenCkpt(PrefillVarlen):
    """The varlen batch through gdn_forward_chunked_checkpointed, with a
    checkpoint every 1024 tokens of each sequence (up to 8 per sequence)."""
    name = "prefill_varlen_ckpt"
    EVERY, MAX_CKPTS = 1024, 8

    def setup(self, gdn, dev):
        super().setup(gdn, dev)
        self.ckpts = torch.empty(self.N, self.MAX_CKPTS, self.H, 128, 128, device=dev)

    def n_ckpts(self):
        return int(sum(min(int(L) // self.EVERY, self.MAX_CKPTS) for L in self.b0.seq_len))

    def alg_bytes_per_step(self):
        return super().alg_bytes_per_step() + self.n_ckpts() * self.H * 128 * 128 * 4

    def _call(self, d, q, k, v, g, beta, stream, out=None):
        self.gdn.gdn_forward_chunked_checkpointed(
            self.shape, d["cu"], q, k, v, g, beta, d["ptrs"], self.slots,
            self.out if out is None else out, self.K, self.mode, self.ckpts, self.EVERY,
            self.MAX_CKPTS, self.ws, self.ws_bytes, stream)

    def config(self):
        c = super().config()
        c["workload"] = ("varlen GDA chunked prefill with state checkpoints every 1024 tokens "
                         "(gdn_forward_chunked_checkpointed, up to 8 per sequence): "
                         "8 sequences, lengths ~U[512,8192] (seed 4), H=16, D_k=D_v=128, "
                         "bf16 q/k/v, fp32 state, K=8 slots")
        c["checkpoints_per_step"] = sum(min(int(L) // self.EVERY, self.MAX_CKPTS)
                                        for L in inputs.varlen_lengths(4))
        return c


# the default run: the headline first, then the other workloads of the metric
ALL_WORKLOADS = ["decode", "verify", "prefill_kda", "prefill_varlen"]

WORKLOADS = {"decode": Decode, "verify": Verify, "prefill_kda": PrefillKDA,
             "decode_gqa": DecodeGQA, "prefill_varlen_fp32": PrefillVarlenF32,
             "prefill_varlen": PrefillVarlen, "prefill_varlen_ckpt": PrefillVarlenCkpt}


# ----------------------------------------------------------------- arms

def run_cpu_baseline(wl, budget_s=10.0):
    """The oracle, as it stands, on this host's cores, on a bounded sample
    (about budget_s seconds of work on all cores, a third of that on one)."""
    import oracle
    cores = oracle.max_threads()
    n_seqs = wl.N
    fn = wl.oracle_step_fn(n_seqs)
    t = time.perf_counter()
    fn()
    one = time.perf_counter() - t
    reps = max(1, min(20000, int(budget_s / max(one, 1e-6))))
    tok = 0
    t = time.perf_counter()
    for _ in range(reps):
        tok += fn()
    el = time.perf_counter() - t
    # the same sample on one core
    fn1 = wl.oracle_step_fn(n_seqs, threads=1)
    t = time.perf_counter()
    fn1()
    one1 = time.perf_counter() - t
    reps1 = max(1, min(5000, int(budget_s / 3 / max(one1, 1e-6))))
    tok1 = 0
    t = time.perf_counter()
    for _ in range(reps1):
        tok1 += fn1()
    el1 = time.perf_counter() - t
    return {"value": tok / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} full steps of the same workload ({n_seqs} sequences each), "
                      f"fp64, {el:.1f} s",
            "value_1core": tok1 / el1,
            "sample_1core": f"{reps1} steps on 1 core, {el1:.1f} s"}


def reference_arm(args, wl_cls):
    ws, rank, local = dist_env()
    wl = wl_cls()
    if rank != 0:
        return 0
    import oracle
    cores = oracle.max_threads()
    # size each step's sample so that warmup + steps take about a minute
    probe = wl.oracle_step_fn(1)
    t = time.perf_counter()
    probe()
    per_seq = time.perf_counter() - t
    budget = 60.0 / max(1, args.steps + args.warmup)
    n_seqs = int(max(1, min(wl.N, budget / max(per_seq, 1e-6))))
    fn = wl.oracle_step_fn(n_seqs)
    for _ in range(args.warmup):
        fn()
    tok = 0
    t = time.perf_counter()
    for _ in range(args.steps):
        tok += fn()
    el = time.perf_counter() - t
    val = tok / el
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wl.config(),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: {n_seqs} of {wl.N} sequences of the "
                                       f"workload, fp64 oracle on host cores"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def measure(wl, args, gdn, dev, stream, ws, rank, local):
    """Times K steps of workload `wl` (CUDA graphs of consecutive steps,
    events on the launch stream), then K end-to-end steps; returns this
    rank's figures and the clock record of the timed region."""
    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    L = wl.graph_len()
    K, W = args.steps, args.warmup

    def graphs_for(step_fn, L=L, pre=None, post=None):
        gs = []
        with torch.cuda.stream(stream):
            gs.append((capture(lambda i: step_fn(i, stream), stream, range(L), pre, post), L))
            rem = K % L
            if rem:
                gs.append((capture(lambda i: step_fn(i, stream), stream, range(rem), pre, post),
                           rem))
        return gs

    # warm-up: W eager steps (also initialises per-device state before capture)
    with torch.cuda.stream(stream):
        for i in range(W):
            wl.step(i, stream)
    stream.synchronize()
    gdn.gdn_check_device_error(stream)
    graphs = graphs_for(wl.step)
    with torch.cuda.stream(stream):
        for g, _ in graphs:  # one untimed replay uploads each graph
            g.replay()
    stream.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3)
    barrier()
    t_wall0 = time.time()
    ms = timed_graph_steps(graphs, K, stream)
    t_wall1 = time.time()
    barrier()
    time.sleep(0.15)
    clock_rows = sampler.stop() if sampler else []
    gdn.gdn_check_device_error(stream)
    del graphs

    # e2e: host inputs in, host outputs back, every step, same K, within
    # graphs of at least 16 steps: through gdn_forward_host where the
    # workload has it (HostIOPipeline), and with copy-engine transfers whose
    # neighbouring steps overlap each call (E2EPipeline)
    def time_e2e(pipe):
        graphs_e2e = graphs_for(pipe.step, max(L, min(K, 16)), lambda: pipe.begin(stream),
                                lambda: pipe.end(stream))
        with torch.cuda.stream(stream):
            for g, _ in graphs_e2e:
                g.replay()
        stream.synchronize()
        barrier()
        t = timed_graph_steps(graphs_e2e, K, stream)
        barrier()
        gdn.gdn_check_device_error(stream)
        del graphs_e2e
        return t

    ms_e2e_copy = time_e2e(E2EPipeline(wl, dev))
    ms_e2e = time_e2e(HostIOPipeline(wl, dev)) if getattr(wl, "e2e_call_host", None) else None

    in_place = None
    if wl.name == "decode" and K >= L:
        K2 = min(K, 2 * L * max(1, 1024 // L))
        gs = []
        with torch.cuda.stream(stream):
            gs.append((capture(lambda i: wl.step_in_place(i, stream), stream, range(L)), L))
            for g, _ in gs:
                g.replay()
        stream.synchronize()
        ms_ip = timed_graph_steps(gs, K2 - K2 % L, stream)
        gdn.gdn_check_device_error(stream)
        steps_ip = K2 - K2 % L
        in_place = {"value": wl.tokens_per_step * steps_ip / (ms_ip / 1e3), "unit": "tokens/s",
                    "ms_per_step": ms_ip / steps_ip,
                    "note": "one 64-sequence batch stepping in place: its 64 MiB state "
                            "ping-pongs between two buffers and largely stays in L2; an L2 "
                            "figure beside the cold-L2 headline, not the headline"}
    return ms, ms_e2e, ms_e2e_copy, in_place, summarize_clocks(clock_rows, t_wall0, t_wall1)


def roofline(wl, kern_s):
    """Roofline object of one workload from its average step duration."""
    peaks, src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = wl.alg_bytes_per_step() / kern_s / 1e9
    if isinstance(wl, Prefill):
        sha = source_sha("chunked.cu", "recurrent.cu", "umma.cuh", "common.cuh")
        tflops = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
        flops = wl.alg_flops_per_step() / kern_s / 1e12
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm,
                "traffic": ncu_traffic("gdn_chunked_" + wl.name, sha),
                "kernel": "whole gdn_forward_chunked call (work list, chunk prep, "
                          "chunk scan, recurrent tail)",
                "algorithmic_bytes_per_launch": wl.alg_bytes_per_step(),
                "tensor": {"achieved": flops, "peak": tflops, "unit": "TFLOP/s",
                           "frac": flops / tflops,
                           "algorithmic_flops_per_launch": wl.alg_flops_per_step()},
                # ideal time of the binding roofline / measured time
                "binding_frac": max(achieved / hbm, flops / tflops),
                "peak_source": f"{src} hbm_gbs and bf16_tflops (burst)"}
        if wl.in_bytes == 4:  # token-loop route: fp32 CUDA-core work, HBM-bound
            roof["tensor"] = None
            roof["binding_frac"] = achieved / hbm
            roof["kernel"] = "whole gdn_forward_chunked call (token-loop route: work list, " \
                             "recurrent kernel)"
        return roof
    sha = source_sha("recurrent.cu", "common.cuh")
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": ncu_traffic("gdn_recurrent_" + wl.name, sha),
            "kernel": "recurrent_kernel (gdn_forward)",
            "algorithmic_bytes_per_launch": wl.alg_bytes_per_step(),
            "peak_source": f"{src} hbm_gbs"}


def gdn_arm(args, names):
    """Measures the workloads `names` in order; the first is the headline
    (top-level keys of the JSON line), the others go under "workloads"."""
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn

    stream = torch.cuda.Stream(device=dev)
    K, W = args.steps, args.warmup
    lines = []
    for name in names:
        wl = WORKLOADS[name]()
        wl.setup(gdn, dev)
        torch.cuda.synchronize()
        ms, ms_e2e, ms_e2e_copy, in_place, clocks = measure(wl, args, gdn, dev, stream, ws,
                                                            rank, local)
        host_io = ms_e2e is not None
        ms_max, ms_e2e_max, value, e2e_value = aggregate_over_ranks(
            ms, ms_e2e if host_io else ms_e2e_copy, wl.tokens_per_step, K, ws, dev)
        _, _, _, e2e_copy_value = aggregate_over_ranks(
            ms, ms_e2e_copy, wl.tokens_per_step, K, ws, dev)
        line = None
        if rank == 0:
            kern_s = ms / K / 1e3  # this rank's average launch duration
            line = {
                "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
                "steps": K, "warmup": W, "ms_per_step": ms_max / K,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": wl.compute_dtype, "data": "synthetic", "config": wl.config(),
                "roofline": roofline(wl, kern_s),
                "e2e": {"value": e2e_value, "unit": "tokens/s",
                        "h2d_bytes_per_step": wl.h2d_bytes,
                        "d2h_bytes_per_step": wl.d2h_bytes,
                        "ms_per_step": ms_e2e_max / K,
                        "path": E2E_HOST_PATH if host_io else E2E_COPY_PATH,
                        **({"copy_engine": {"value": e2e_copy_value, "unit": "tokens/s",
                                            "path": E2E_COPY_PATH}} if host_io else {})},
                "gpu_launches": K * wl.launches_per_step(),
                **({"l2_warm_in_place": in_place} if in_place else {}),
                "clocks": clocks,
            }
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = run_cpu_baseline(wl)
        lines.append(line)
        del wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    if rank == 0:
        head = lines[0]
        if len(lines) > 1:
            head["gpu_launches_all_workloads"] = sum(x["gpu_launches"] for x in lines)
            head["workloads"] = {n: {k: v for k, v in x.items()
                                     if k not in ("metric", "n_gpus", "higher_is_better",
                                                  "scaling", "vs_baseline", "data")}
                                 for n, x in zip(names[1:], lines[1:])}
        print(json.dumps(head), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def ncu_range(args, name):
    """W eager warm-up steps, then `--ncu-range N` eager steps between
    cudaProfilerStart/Stop, for an ncu range-replay capture of the DRAM bytes
    of N consecutive steps (the write-back of one step's state counts even
    when it leaves L2 during the next). Prints the step count only."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn
    wl = WORKLOADS[name]()
    wl.setup(gdn, dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            wl.step(i, stream)
    stream.synchronize()
    gdn.gdn_check_device_error(stream)
    n = args.ncu_range
    torch.cuda.profiler.start()
    with torch.cuda.stream(stream):
        for i in range(args.warmup, args.warmup + n):
            wl.step(i, stream)
    stream.synchronize()
    torch.cuda.profiler.stop()
    gdn.gdn_check_device_error(stream)
    print(json.dumps({"ncu_range": name, "steps_in_range": n,
                      "launches_per_step": wl.launches_per_step()}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--workload", choices=["all"] + sorted(WORKLOADS), default="all",
                    help="all (default): decode as the headline, then verify, KDA prefill "
                         "and varlen prefill under 'workloads'")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-range", type=int, default=0,
                    help="profiling aid: run N eager steps between cudaProfilerStart/Stop "
                         "(for ncu --replay-mode range) and print no bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    names = ALL_WORKLOADS if args.workload == "all" else [args.workload]
    if args.ncu_range:
        return ncu_range(args, names[0])
    if args.impl == "reference":
        return reference_arm(args, WORKLOADS[names[0]])
    return gdn_arm(args, names)


if __name__ == "__main__":
    sys.exit(main())
