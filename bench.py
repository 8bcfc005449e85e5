"""Benchmark of the Gated DeltaNet state path on one GB300 (or N replicas).

One step = one pass of the whole path over one batch of synthetic input:
  1. chunked prefill of a 27B-shaped GDN layer (16 qk / 48 v heads, d = 128,
     bf16 x and o, fp32 state), 4 sequences x 8192 tokens, block 896 with a
     checkpoint written into the paged pool at every crossed boundary
     (block table = seeded permutation of the pages);
  2. batched decode of a 4B-shaped layer (16 qk / 32 v heads), 256 sequences
     at seeded random pages, 24 layers back to back (separate pools);
  3. replay verify on the same 4B-shaped layer: 16 requests x 16 rows
     appended to a 32-slot bf16 log, rollback to an accepted length uniform on
     [0, 16], then the flush of the kept rows into the checkpoint, 24 layers.

`value` is prefill tokens/s per layer (device-timed, inputs resident in HBM);
decode and flush are reported as microseconds per layer.  Every input is
larger than L2 (x alone is 671 MB; decode touches 15 GiB of pages; the replay
pools of 24 layers are 960 MiB), so no L2 flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       (N > 1: launch with torch.distributed.run; each rank runs a replica).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gated_deltanet_state_gb300 as gdn  # noqa: E402
from gated_deltanet_state_gb300 import inputs  # noqa: E402

METRIC = "GDN prefill tokens/s/layer; decode & replay-flush µs/layer; % of TC/HBM roofline"
HBM_NOMINAL_GBS = 7900.0    # nominal HBM3e rate of the part (fractions use the measured copy rate first)
PREFILL = inputs.QWEN27B
SMALL = inputs.QWEN4B
N_SEQ, SEQ_LEN = 4, 8192
# DRAM bytes (read + write) of one 4 x 8,192 prefill call on each tensor-core
# path (every launch of the call summed), from an ncu capture of the current
# kernels on this workload (profiles/prefill_traffic_27b_4x8192.md); None
# once a kernel of the path changes.  fused: 4 tc_prefill_kernel launches +
# the window pass; two kernels: 1 tc_chunk_kernel + 4 tc_chain_kernel
# launches + the window pass.
PREFILL_TRAFFIC_PER_CALL = {"fused": 713.26e6 + 366.86e6, "two_kernels": 3025.54e6 + 2545.82e6}
# Algorithmic flops of the chunk form per token and value head (chunk C = 64,
# d = 128): 2 [C (3 dk + 2 dv) + 3 dk dv]; the kernel runs every product as
# three bf16 passes (hi*hi + hi*lo + lo*hi) over the shapes it issues per
# chunk (M = 128 throughout): [K^;Q^]K^T 128x64x128, S0[K^;Q^]^T 128x128x128,
# R T^T 128x64x64, U^T (K^T dec)^T 128x128x64, U^T P^T 128x64x64.
CHUNK_FLOPS_PER_TOKEN_HEAD = 2 * (64 * (3 * 128 + 2 * 128) + 3 * 128 * 128)
EXECUTED_FLOPS_PER_TOKEN_HEAD = 3 * 2 * (128 * 64 * 128 + 128 * 128 * 128 + 128 * 64 * 64 + 128 * 128 * 64
                                         + 128 * 64 * 64) / 64
DEC_SEQS, DEC_LAYERS = 256, 24
REP_REQS, REP_ROWS, REP_LAYERS = 16, 16, 24


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}, "fallback"


def _smi_id(local: int) -> str:
    """nvidia-smi's id of this process's device: its UUID (nvidia-smi numbers
    the GPUs of the machine, not the ones this process sees)."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


def _bind_near_gpu(local: int):
    """Run this process on the CPUs next to its GPU (the sysfs local_cpulist
    of the device), so that the pinned host buffers of the end-to-end
    measurement are allocated in that node's memory.  Returns the CPU count,
    or None where the list is not available (the affinity is then left as
    it is)."""
    try:
        pr = torch.cuda.get_device_properties(local)
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/local_cpulist" % (
            pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        cpus = set()
        with open(path) as f:
            for part in f.read().strip().split(","):
                a, _, b = part.partition("-")
                cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return len(cpus)
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = _smi_id(index)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.index, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- replicas

def max_over_ranks(values, dist=None, device="cpu"):
    """Each timing's maximum over the ranks: the slowest replica sets the
    job's time.  Without an initialised process group: the local values."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job units per second: every replica processes units_per_rank
    units (weak scaling) in the max-over-ranks time ms."""
    return world * units_per_rank / (ms * 1e-3)


# ----------------------------------------------------------------------------- workloads

class PrefillWork:
    """4 x 8192 tokens of the 27B-shaped layer, checkpoints every 896 tokens
    (other batch shapes and a forced path for profiling)."""

    def __init__(self, seed: int, seq_len: int = SEQ_LEN, num_seqs: int = N_SEQ, path: int = gdn.PREFILL_AUTO):
        sh = PREFILL
        self.sh = sh
        self.n = num_seqs
        self.path = path
        T = num_seqs * seq_len
        # a2: the scheduler's chunk for this call; the whole prompt fits the budget
        self.chunk_end = gdn.gdn_chunk_end(0, seq_len, seq_len, sh.block_size)
        assert self.chunk_end == seq_len
        ti = inputs.token_inputs(sh, T, seed)
        self.host = {k: v.pin_memory() for k, v in ti.items()}
        self.x = ti["x"].cuda()
        self.g = ti["g"].cuda()
        self.beta = ti["beta"].cuda()
        self.w = inputs.conv_weights(sh, seed).cuda()
        nck = max(1, seq_len // sh.block_size)    # 9 boundaries per sequence at 8192
        self.num_pages = self.n * (nck + 1)
        perm = inputs.permutation(self.num_pages, seed).tolist()
        self.block_table = torch.tensor([perm[s * nck:(s + 1) * nck] for s in range(self.n)],
                                        dtype=torch.int32).cuda()
        self.out_slot = torch.tensor(perm[self.n * nck:], dtype=torch.int32).cuda()
        self.pool = gdn.StatePool(sh, self.num_pages, fill=0)
        self.cu = torch.arange(0, T + 1, seq_len, dtype=torch.int32).cuda()
        self.seq_len = seq_len
        self.start = torch.zeros(self.n, dtype=torch.int64).cuda()
        self.init = torch.full((self.n,), -1, dtype=torch.int32).cuda()
        self.o = torch.empty(T, sh.num_v_heads, sh.head_dim_v, dtype=torch.bfloat16, device="cuda")
        self.o_host = torch.empty_like(self.o, device="cpu").pin_memory()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.tokens = T
        self.ws = gdn.workspace_for(gdn.gdn_prefill_workspace_size(sh, self.n, T))

    def run(self, x=None, g=None, beta=None, o=None):
        gdn.gdn_prefill_chunked(self.sh, self.pool, cu_seqlens=self.cu, start_pos=self.start,
                                init_page=self.init, block_table=self.block_table, out_slot=self.out_slot,
                                x=self.x if x is None else x, g=self.g if g is None else g,
                                beta=self.beta if beta is None else beta, conv_w=self.w,
                                o=self.o if o is None else o, dev_error=self.err,
                                start_pos_host=[0] * self.n, init_page_host=[-1] * self.n,
                                workspace=self.ws, max_seq_len=self.seq_len, path=self.path)

    def e2e_pipelined_ms(self, steps: int, warmup: int = 6, nbuf: int = 3) -> float:
        """Streaming end to end: every step copies its inputs from pinned host
        memory to the device, runs the prefill, and copies its outputs back,
        with later steps' input copies and earlier steps' output copies
        running on their own streams while a step computes (nbuf device
        buffer sets).  Returns ms per step from the first input copy to the
        last output copy.  The warm-up runs every buffer set twice: the first
        streamed steps of a process run well below the link's rate."""
        comp = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        bufs = [{k: torch.empty_like(v, device="cuda") for k, v in self.host.items()} for _ in range(nbuf)]
        outs = [torch.empty_like(self.o) for _ in range(nbuf)]
        ev = lambda: torch.cuda.Event(enable_timing=True)
        in_ready = [torch.cuda.Event() for _ in range(nbuf)]
        in_free = [torch.cuda.Event() for _ in range(nbuf)]
        out_ready = [torch.cuda.Event() for _ in range(nbuf)]
        out_free = [torch.cuda.Event() for _ in range(nbuf)]
        for e in in_free + out_free:
            e.record(comp)

        def step(k):
            b = k % nbuf
            with torch.cuda.stream(h2d):
                h2d.wait_event(in_free[b])
                for name, t in bufs[b].items():
                    t.copy_(self.host[name], non_blocking=True)
                in_ready[b].record(h2d)
            comp.wait_event(in_ready[b])
            comp.wait_event(out_free[b])
            self.run(bufs[b]["x"], bufs[b]["g"], bufs[b]["beta"], outs[b])
            in_free[b].record(comp)
            out_ready[b].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(out_ready[b])
                self.o_host.copy_(outs[b], non_blocking=True)
                out_free[b].record(d2h)

        for k in range(warmup):
            step(k)
        torch.cuda.synchronize()
        t0, t1 = ev(), ev()
        t0.record(h2d)
        for k in range(steps):
            step(warmup + k)
        t1.record(d2h)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps

    def link_gbs(self, reps: int = 3) -> dict:
        """The host link on its own, with the same pinned buffers: GB/s of the
        step's input copies alone, of its output copy alone, and of both at
        once on two streams (the floor of the streamed step)."""
        xd = torch.empty_like(self.host["x"], device="cuda")
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event(enable_timing=True)

        def timed(streams):
            torch.cuda.synchronize()
            e0 = [ev() for _ in streams]
            e1 = [ev() for _ in streams]
            for i, st in enumerate(streams):
                e0[i].record(st)
            for _ in range(reps):
                if s_in in streams:
                    with torch.cuda.stream(s_in):
                        xd.copy_(self.host["x"], non_blocking=True)
                if s_out in streams:
                    with torch.cuda.stream(s_out):
                        self.o_host.copy_(self.o, non_blocking=True)
            for i, st in enumerate(streams):
                e1[i].record(st)
            torch.cuda.synchronize()
            return max(a.elapsed_time(b) for a, b in zip(e0, e1)) / reps

        xb = self.host["x"].numel() * self.host["x"].element_size()
        ob = self.o_host.numel() * self.o_host.element_size()
        # best of three trials of each (a trial can read far below the link)
        t_in = min(timed([s_in]) for _ in range(3))
        t_out = min(timed([s_out]) for _ in range(3))
        t_both = min(timed([s_in, s_out]) for _ in range(3))
        del xd
        return {"h2d_gbs": round(xb / t_in / 1e6, 1), "d2h_gbs": round(ob / t_out / 1e6, 1),
                "both_gbs": round((xb + ob) / t_both / 1e6, 1)}

    @property
    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.host.values())

    @property
    def d2h_bytes(self):
        return self.o_host.numel() * self.o_host.element_size()

    # roofline inputs for the prefill kernel
    def algorithmic_flops(self):
        """The chunk form's flops for every token of every value head."""
        return float(CHUNK_FLOPS_PER_TOKEN_HEAD) * self.sh.num_v_heads * self.tokens

    def algorithmic_bytes(self):
        sh = self.sh
        per_tok = sh.conv_dim * 2 + 2 * sh.num_v_heads * 4 + sh.num_v_heads * sh.head_dim_v * 2
        ck = (self.seq_len // sh.block_size + 1) * self.n * sh.payload_bytes
        return per_tok * self.tokens + ck


def prefill_paths_ms(pre, runs: int = 5) -> dict:
    """The same prefill call forced onto each tensor-core path (both give the
    same bits), outside the timed step: ms per call, CUDA events."""
    out = {}
    for name, path in (("fused", gdn.PREFILL_FUSED), ("two_kernels", gdn.PREFILL_TWO_KERNELS)):
        keep = pre.path
        pre.path = path
        for _ in range(2):
            pre.run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(runs):
            pre.run()
        e1.record()
        torch.cuda.synchronize()
        pre.path = keep
        out[name + "_ms"] = round(e0.elapsed_time(e1) / runs, 4)
    if int(pre.err.item()):
        raise RuntimeError("device error word set while timing the prefill paths")
    return out


class DecodeWork:
    """256 sequences x 24 layers of the 4B-shaped layer, one token each."""

    def __init__(self, seed: int, layers: int = DEC_LAYERS):
        sh = SMALL
        self.sh = sh
        self.nlayers = layers
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        self.pools, self.slots, self.x, self.g, self.beta = [], [], [], [], []
        for layer in range(layers):
            pool = gdn.StatePool(sh, DEC_SEQS, fill=0)
            for p in range(0, DEC_SEQS, 64):
                n = min(64, DEC_SEQS - p)
                blk = pool.buf[p * sh.page:(p + n) * sh.page].view(n, sh.page)
                st = blk[:, :sh.state_bytes].view(torch.float32)
                st.copy_(0.3 * torch.randn(st.shape, generator=gen, device="cuda"))
            self.pools.append(pool)
            self.slots.append(inputs.permutation(DEC_SEQS, seed + layer).cuda())
            ti = inputs.token_inputs(sh, DEC_SEQS, seed + 1000 + layer)
            self.x.append(ti["x"].cuda())
            self.g.append(ti["g"].cuda())
            self.beta.append(ti["beta"].cuda())
        self.w = inputs.conv_weights(sh, seed).cuda()
        self.o = torch.empty(DEC_SEQS, sh.num_v_heads, sh.head_dim_v, dtype=torch.bfloat16, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self):
        for L in range(self.nlayers):
            gdn.gdn_decode_step(self.sh, self.pools[L], x=self.x[L], g=self.g[L], beta=self.beta[L],
                                conv_w=self.w, slot=self.slots[L], o=self.o, dev_error=self.err)

    def bytes_per_layer(self):
        sh = self.sh
        per_seq = 2 * sh.state_bytes + 2 * sh.window_bytes + sh.conv_dim * 2 + 2 * sh.num_v_heads * 4 \
            + sh.num_v_heads * sh.head_dim_v * 2
        return per_seq * DEC_SEQS


class ReplayWork:
    """16 requests x 16 rows per layer, 24 layers: append, rollback, flush."""

    def __init__(self, seed: int, layers: int = REP_LAYERS):
        sh = SMALL
        self.sh = sh
        self.nlayers = layers
        L = gdn.REPLAY_LOG_SLOTS
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        self.layers = []
        for layer in range(layers):
            pool = gdn.StatePool(sh, REP_REQS, fill=0)
            st = pool.buf.view(REP_REQS, sh.page)[:, :sh.state_bytes].view(torch.float32)
            st.copy_(0.3 * torch.randn(st.shape, generator=gen, device="cuda"))
            ti = inputs.token_inputs(sh, REP_REQS * REP_ROWS, seed + 2000 + layer)
            self.layers.append({
                "pool": pool,
                "ckpt": inputs.permutation(REP_REQS, seed + layer).cuda(),
                "log_x": torch.zeros(REP_REQS, L, sh.conv_dim, dtype=torch.bfloat16, device="cuda"),
                "log_g": torch.zeros(REP_REQS, L, sh.num_v_heads, device="cuda"),
                "log_b": torch.zeros(REP_REQS, L, sh.num_v_heads, device="cuda"),
                "log_len": torch.zeros(REP_REQS, dtype=torch.int32, device="cuda"),
                "x": ti["x"].cuda().view(REP_REQS, REP_ROWS, -1),
                "g": ti["g"].cuda().view(REP_REQS, REP_ROWS, -1),
                "beta": ti["beta"].cuda().view(REP_REQS, REP_ROWS, -1),
                "acc": inputs.accept_lengths(REP_REQS, REP_ROWS, seed + layer).cuda(),
            })
        self.w = inputs.conv_weights(sh, seed).cuda()
        self.o = torch.empty(REP_REQS, REP_ROWS, sh.num_v_heads, sh.head_dim_v, dtype=torch.bfloat16,
                             device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.kept_rows = float(sum(int(l["acc"].sum()) for l in self.layers)) / layers
        self.ws = gdn.workspace_for(gdn.gdn_replay_workspace_size(sh, REP_REQS))

    def _kw(self, l):
        return dict(ckpt_slot=l["ckpt"], log_x=l["log_x"], log_g=l["log_g"], log_beta=l["log_b"],
                    log_len=l["log_len"], conv_w=self.w, dev_error=self.err, workspace=self.ws)

    def verify(self):
        for l in self.layers:
            gdn.gdn_replay_append(self.sh, l["pool"], x_new=l["x"], g_new=l["g"], beta_new=l["beta"],
                                  o=self.o, **self._kw(l))
            gdn.gdn_replay_rollback(l["log_len"], l["acc"], REP_ROWS, self.err)

    def flush(self):
        for l in self.layers:
            gdn.gdn_replay_flush(self.sh, l["pool"], **self._kw(l))

    def verify_bytes_per_layer(self):
        """Append: the checkpoint state read once per request and head, the
        new rows read and copied into the log, the outputs written."""
        sh = self.sh
        row = sh.conv_dim * 2 + 2 * sh.num_v_heads * 4
        return REP_REQS * (sh.payload_bytes + REP_ROWS * (2 * row + sh.num_v_heads * sh.head_dim_v * 2))

    def flush_bytes_per_layer(self):
        sh = self.sh
        return REP_REQS * (2 * sh.payload_bytes) + self.kept_rows * (sh.conv_dim * 2 + 2 * sh.num_v_heads * 4)


class FlushSweep:
    """The flush alone at R kept rows for each of N requests (the log holds
    exactly R rows), over a few layers whose pools together exceed L2; one
    CUDA graph flushes every layer, log_len is restored before each replay
    outside the timed events."""

    def __init__(self, seed: int, n_req: int, rows: int, layers: int, boundary: int = 0):
        sh = SMALL
        self.sh, self.n, self.rows, self.nlayers = sh, n_req, rows, layers
        # boundary > 0: every request's kept rows cross a block boundary after
        # that many rows (the state there also goes to a boundary page)
        self.boundary = boundary
        L = gdn.REPLAY_LOG_SLOTS
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        self.lens = torch.full((layers, n_req), rows, dtype=torch.int32, device="cuda")
        self.w = inputs.conv_weights(sh, seed).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.layers = []
        for layer in range(layers):
            pool = gdn.StatePool(sh, 2 * n_req if boundary else n_req, fill=0)
            st = pool.buf.view(-1, sh.page)[:, :sh.state_bytes].view(torch.float32)
            st.copy_(0.3 * torch.randn(st.shape, generator=gen, device="cuda"))
            self.layers.append(dict(
                pool=pool, ckpt=inputs.permutation(n_req, seed + layer).cuda(),
                bpage=torch.arange(n_req, 2 * n_req, dtype=torch.int32, device="cuda") if boundary else None,
                brows=torch.full((n_req,), boundary, dtype=torch.int32, device="cuda") if boundary else None,
                log_x=torch.randn(n_req, L, sh.conv_dim, generator=gen, device="cuda").to(torch.bfloat16),
                log_g=-0.1 * torch.nn.functional.softplus(torch.randn(n_req, L, sh.num_v_heads, generator=gen,
                                                                      device="cuda")),
                log_b=torch.sigmoid(torch.randn(n_req, L, sh.num_v_heads, generator=gen, device="cuda")),
                log_len=self.lens[layer]))

    def flush(self):
        for l in self.layers:
            gdn.gdn_replay_flush(self.sh, l["pool"], ckpt_slot=l["ckpt"], log_x=l["log_x"], log_g=l["log_g"],
                                 log_beta=l["log_b"], log_len=l["log_len"], conv_w=self.w, dev_error=self.err,
                                 boundary_rows=l["brows"], boundary_page=l["bpage"])

    def bytes_per_layer(self):
        sh = self.sh
        pages = 3 if self.boundary else 2          # + the boundary checkpoint written
        return self.n * (pages * sh.payload_bytes + self.rows * (sh.conv_dim * 2 + 2 * sh.num_v_heads * 4))

    def time_us_per_layer(self, reps: int = 5) -> float:
        self.flush()
        self.lens.fill_(self.rows)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.flush()
        total = 0.0
        for _ in range(reps + 1):
            self.lens.fill_(self.rows)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1) if _ else 0.0
        if int(self.err.item()):
            raise RuntimeError("device error word set in the flush sweep")
        return 1000.0 * total / reps / self.nlayers


def flush_sweep(seed: int, hbm_gbs: float):
    """Flush time per layer: every log length R = 1..32 at N = 16 requests,
    R = 16 at N = 64 and 256, and R = 16 at N = 16 with every request's kept
    rows crossing a block boundary after 8 rows (4B-shaped layer)."""
    out = []
    cases = [(16, r, 0) for r in range(1, 33)] + [(64, 16, 0), (256, 16, 0), (16, 16, 8)]
    for n_req, rows, bnd in cases:
        layers = max(2, 128 // n_req)          # 2.5 MiB pages: >= 320 MB of pools per replay
        fs = FlushSweep(seed + 31 * rows + n_req, n_req, rows, layers, boundary=bnd)
        us = fs.time_us_per_layer()
        gbs = fs.bytes_per_layer() / (us * 1e-6) / 1e9
        case = {"N": n_req, "R": rows, "us_per_layer": round(us, 2), "hbm_gbs": round(gbs, 1),
                "hbm_frac": round(gbs / hbm_gbs, 3)}
        if bnd:
            case["boundary_after"] = bnd
        out.append(case)
        del fs
    torch.cuda.empty_cache()
    return out


def checkpoint_copy(seed: int, hbm_gbs: float, n: int = 256, reps: int = 5):
    """Checkpoint saves of the 27B-shaped layer (`gdn_checkpoint_save`): n
    working slots copied to n block pages in a permuted order, state and conv
    window as 16-byte words, each byte read and written once; the pool (2n
    pages, 1.9 GB at n = 256) is larger than L2."""
    sh = PREFILL
    pool = gdn.StatePool(sh, 2 * n, fill=0)
    src = torch.arange(n, dtype=torch.int32, device="cuda")
    dst = (n + inputs.permutation(n, seed)).cuda()
    nch = torch.full((n,), 4 * sh.block_size, dtype=torch.int64)     # at a block boundary
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        gdn.gdn_checkpoint_save(sh, pool, src, dst, nch, err)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        gdn.gdn_checkpoint_save(sh, pool, src, dst, nch, err)
    e1.record()
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError("device error word set in the checkpoint copies")
    us = 1000.0 * e0.elapsed_time(e1) / reps
    gbs = 2 * n * sh.payload_bytes / (us * 1e-6) / 1e9
    del pool
    torch.cuda.empty_cache()
    return {"pages": n, "payload_bytes": sh.payload_bytes, "us": round(us, 1), "hbm_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / hbm_gbs, 3), "hbm_frac_nominal": round(gbs / HBM_NOMINAL_GBS, 3)}


def long_context(seed: int, reps: int = 3):
    """The long-context prefix hit on one 27B-shaped layer: a cold prefill of
    a 229,376-token request (256 blocks of 896, a checkpoint at every
    boundary), then the same request resumed from block 222 (the state after
    199,808 tokens, the last full block of a 200,000-token shared prefix) over
    its 29,568-token suffix.  One sequence gives 48 (sequence, v head) chains,
    so 48 of the SMs work.  Inputs are drawn on the device (timing only)."""
    sh = PREFILL
    T, B = 256 * sh.block_size, sh.block_size
    hit = (200_000 // B) * B
    resume_block = gdn.gdn_resume_block(hit, B)
    start = (resume_block + 1) * B
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = torch.empty(T, sh.conv_dim, dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, T, 16384):
        r1 = min(T, r0 + 16384)
        x[r0:r1] = torch.randn(r1 - r0, sh.conv_dim, generator=gen, device="cuda").to(torch.bfloat16)
    g = -0.1 * torch.nn.functional.softplus(torch.randn(T, sh.num_v_heads, generator=gen, device="cuda"))
    beta = torch.sigmoid(torch.randn(T, sh.num_v_heads, generator=gen, device="cuda"))
    w = inputs.conv_weights(sh, seed).cuda()
    pool = gdn.StatePool(sh, 258, fill=0)
    bt = inputs.permutation(258, seed)[:256].view(1, 256).cuda()
    used = set(bt.flatten().tolist())
    slot = torch.tensor([next(p for p in range(258) if p not in used)], dtype=torch.int32).cuda()
    o = torch.empty(T, sh.num_v_heads, sh.head_dim_v, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = gdn.workspace_for(gdn.gdn_prefill_workspace_size(sh, 1, T))

    def run(t0, init):
        n = T - t0
        gdn.gdn_prefill_chunked(sh, pool, cu_seqlens=torch.tensor([0, n], dtype=torch.int32, device="cuda"),
                                start_pos=torch.tensor([t0], dtype=torch.int64, device="cuda"),
                                init_page=torch.tensor([init], dtype=torch.int32, device="cuda"),
                                block_table=bt, out_slot=slot, x=x[t0:], g=g[t0:], beta=beta[t0:], conv_w=w,
                                o=o[t0:], dev_error=err, start_pos_host=[t0], init_page_host=[init],
                                workspace=ws, max_seq_len=n)

    def timed(t0, init):
        run(t0, init)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            run(t0, init)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    cold_ms = timed(0, -1)
    resume_ms = timed(start, int(bt[0, resume_block]))
    if int(err.item()):
        raise RuntimeError("device error word set in the long-context prefill")
    del x, o, pool, ws
    torch.cuda.empty_cache()
    return {"tokens": T, "cold_ms": round(cold_ms, 2), "cold_tokens_per_s_per_layer": round(T / cold_ms * 1e3),
            "resume_block": resume_block, "resume_from_tokens": start, "suffix_tokens": T - start,
            "resume_ms": round(resume_ms, 2),
            "resume_tokens_per_s_per_layer": round((T - start) / resume_ms * 1e3), "chains": sh.num_v_heads}


# ----------------------------------------------------------------------------- cpu baseline

def _oracle_setup(seed: int):
    import oracle
    sh = PREFILL
    d = oracle.Dims(sh.num_qk_heads, sh.num_v_heads, sh.head_dim_k, sh.head_dim_v, sh.q_scale, sh.norm_eps)
    ti = inputs.token_inputs(sh, N_SEQ * SEQ_LEN, seed)
    w = inputs.conv_weights(sh, seed)
    oracle.build()

    def run(n):
        # n tokens of the workload: whole 8192-token sequences plus a prefix
        cu = list(range(0, n, SEQ_LEN)) + [n]
        t0 = time.perf_counter()
        oracle.prefill(d, cu, [0] * (len(cu) - 1), sh.block_size, ti["x"][:n], ti["g"][:n],
                       ti["beta"][:n], w)
        return time.perf_counter() - t0

    return run, oracle.num_threads()


def _calibrate(run, seconds: float) -> int:
    """Tokens of one 27B-shaped sequence the oracle prefills in about `seconds`."""
    n, dt = 32, run(32)
    while dt < min(2.0, seconds / 2) and n < N_SEQ * SEQ_LEN:
        n = min(N_SEQ * SEQ_LEN, n * 4)
        dt = run(n)
    return max(16, min(N_SEQ * SEQ_LEN, int(n * seconds / max(dt, 1e-6))))


def cpu_baseline(seconds: float = 12.0, seed: int = 0):
    """The fp64 oracle on the host cores, on a bounded sample of the prefill
    workload (one sequence of the 27B-shaped layer, all 48 heads, a prefix of
    its tokens), scaled to tokens/s per layer."""
    run, cores = _oracle_setup(seed)
    n = _calibrate(run, seconds)
    dt = run(n)
    return {"value": n / dt, "unit": "tokens/s/layer", "cores": cores, "kind": "oracle",
            "sample": f"27B-shaped layer, first {n} of the 4 x 8192 tokens, all 48 heads, fp64, "
                      f"{dt:.1f} s wall"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: W warm-up and K timed steps, each a
    bounded sample of the prefill workload on the host cores (rank 0 only)."""
    if rank != 0:
        return
    run, cores = _oracle_setup(args.seed)
    per_step = max(2.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    n = _calibrate(run, per_step)
    for _ in range(args.warmup):
        run(n)
    times = [run(n) for _ in range(args.steps)]
    value = n / statistics.mean(times)
    sample = (f"27B-shaped layer, first {n} of the 4 x 8192 tokens per step, all 48 heads, fp64, "
              f"{statistics.mean(times):.1f} s per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s/layer",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill 27B-shaped GDN layer (16 qk / 48 v heads, d 128), 4 x 8192 "
                                   "tokens, block 896 (bounded sample per step)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s/layer", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main

def run_part(args):
    """One part of the step alone (for profiling): W warm-up and K timed runs,
    one JSON line with the part's device time."""
    if args.only == "prefill":
        path = {"auto": gdn.PREFILL_AUTO, "fused": gdn.PREFILL_FUSED, "two": gdn.PREFILL_TWO_KERNELS}[args.path]
        w = PrefillWork(args.seed, args.seq_len, args.num_seqs, path)
        fn, unit_ms = w.run, None
    elif args.only == "decode":
        w = DecodeWork(args.seed, args.layers)
        fn = w.run
    elif args.only == "flush":
        w = FlushSweep(args.seed, args.requests, args.rows, args.layers, boundary=args.boundary)

        def fn():
            w.lens.fill_(w.rows)      # the flush clears log_len: every run flushes R rows
            w.flush()
    else:
        w = ReplayWork(args.seed, args.layers)
        fn = lambda: (w.verify(), w.flush())
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    line = {"part": args.only, "ms_per_run": ms, "steps": args.steps, "warmup": args.warmup}
    if args.only == "prefill":
        line["tokens_per_s_per_layer"] = w.tokens / (ms * 1e-3)
        line["seq_len"] = args.seq_len
        line["num_seqs"] = args.num_seqs
        line["plan"] = gdn.gdn_prefill_plan_for(PREFILL, args.num_seqs, args.seq_len, 0, w.path)
    if args.only == "flush":
        line.update(requests=args.requests, rows=args.rows, boundary_after=args.boundary,
                    us_per_layer_incl_log_len_reset=1000.0 * ms / args.layers)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-flush-sweep", action="store_true",
                    help="skip the flush sweep over kept rows and requests")
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode", "replay", "flush"],
                    help="time one part only (profiling); the default times the whole step")
    ap.add_argument("--requests", type=int, default=16, help="flush requests with --only flush")
    ap.add_argument("--rows", type=int, default=16, help="kept rows per request with --only flush")
    ap.add_argument("--boundary", type=int, default=0,
                    help="with --only flush: every request's kept rows cross a block boundary after this many rows")
    ap.add_argument("--seq-len", type=int, default=SEQ_LEN,
                    help="prefill tokens per sequence (profiling of smaller cases)")
    ap.add_argument("--num-seqs", type=int, default=N_SEQ,
                    help="prefill sequences with --only prefill (profiling of other batch shapes)")
    ap.add_argument("--path", default="auto", choices=["auto", "fused", "two"],
                    help="tensor-core prefill path with --only prefill (both give the same bits)")
    ap.add_argument("--layers", type=int, default=DEC_LAYERS,
                    help="decode / replay layers with --only (profiling of smaller cases)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    args.warmup = max(args.warmup, 3)
    torch.cuda.set_device(local)
    all_cpus = os.sched_getaffinity(0)
    near_cpus = _bind_near_gpu(local) if args.only == "all" else None
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    gdn.load_library()

    if args.only != "all":
        return run_part(args)
    pre = PrefillWork(args.seed + rank, args.seq_len)
    dec = DecodeWork(args.seed + 10 + rank)
    rep = ReplayWork(args.seed + 20 + rank)
    stream = torch.cuda.current_stream()

    ev = lambda: torch.cuda.Event(enable_timing=True)

    # Warm up eagerly, then capture the launch-bound 24-layer loops of decode
    # and replay into CUDA graphs (the prefill is one call).
    for _ in range(args.warmup):
        pre.run(); dec.run(); rep.verify(); rep.flush()
    torch.cuda.synchronize()
    errs = [int(pre.err.item()), int(dec.err.item()), int(rep.err.item())]
    if any(errs):
        raise RuntimeError(f"device error words after warm-up: {errs}")
    graphs = {}
    for name, fn in (("dec", dec.run), ("ver", rep.verify), ("fl", rep.flush)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    for _ in range(2):
        for g in graphs.values():
            g.replay()
    torch.cuda.synchronize()

    def step(record=None):
        e = [ev() for _ in range(5)] if record is not None else None
        if e: e[0].record(stream)
        pre.run()
        if e: e[1].record(stream)
        graphs["dec"].replay()
        if e: e[2].record(stream)
        graphs["ver"].replay()
        if e: e[3].record(stream)
        graphs["fl"].replay()
        if e: e[4].record(stream)
        if record is not None:
            record.append(e)

    step()
    torch.cuda.synchronize()
    if int(rep.err.item()) or int(dec.err.item()) or int(pre.err.item()):
        raise RuntimeError("device error word set during graph replay")

    recs = []
    with ClockSampler(local) as clk:
        if dist: dist.barrier()
        torch.cuda.synchronize()
        t_start = ev(); t_end = ev()
        t_start.record(stream)
        for _ in range(args.steps):
            step(recs)
        t_end.record(stream)
        torch.cuda.synchronize()
        if dist: dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = sum(r[0].elapsed_time(r[1]) for r in recs) / args.steps
    dec_ms = sum(r[1].elapsed_time(r[2]) for r in recs) / args.steps
    ver_ms = sum(r[2].elapsed_time(r[3]) for r in recs) / args.steps
    fl_ms = sum(r[3].elapsed_time(r[4]) for r in recs) / args.steps
    total_ms, pre_ms, dec_ms, ver_ms, fl_ms = max_over_ranks([total_ms, pre_ms, dec_ms, ver_ms, fl_ms],
                                                            dist, "cuda")

    # end to end through the same call with host buffers (prefill part):
    # every step copies its inputs in and its outputs out; the copies of
    # neighbouring steps overlap the prefill on their own streams
    # (at least 32 steps: the timed region also fills and drains the pipeline
    # once, about one prefill and one output copy beyond the steps' copies).
    # Three trials, the median reported and every trial listed: now and then
    # a whole trial runs far below the host link's rate while the link,
    # measured alone in the same process, runs at its full rate.
    e2e_steps = max(args.steps, 32)
    e2e_trials = [pre.e2e_pipelined_ms(e2e_steps) for _ in range(3)]
    e2e_ms = statistics.median(e2e_trials)
    link = pre.link_gbs()
    (e2e_ms,) = max_over_ranks([e2e_ms], dist, "cuda")

    peaks, peak_kind = _peaks()
    clocks = clk.summary()
    tc_peak = peaks["bf16_tflops"]                          # dense bf16, measured (burst)
    achieved = pre.algorithmic_flops() / (pre_ms * 1e-3) / 1e12
    dec_gbs = dec.bytes_per_layer() / (dec_ms / DEC_LAYERS * 1e-3) / 1e9
    fl_gbs = rep.flush_bytes_per_layer() / (fl_ms / REP_LAYERS * 1e-3) / 1e9
    ver_gbs = rep.verify_bytes_per_layer() / (ver_ms / REP_LAYERS * 1e-3) / 1e9
    value = job_throughput(pre.tokens, world, pre_ms)
    pre_plan = gdn.gdn_prefill_plan_for(PREFILL, N_SEQ, args.seq_len)
    # the call's own path (both give the same bits): its chain (or fused)
    # launches and, on the two-kernel path, the chunk kernel's launches
    pre_launches = pre_plan["launches"] + pre_plan["chunk_launches"]
    path_key = "two_kernels" if pre_plan["two_kernels"] else "fused"

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s/layer", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16x3", "data": "synthetic",
        "config": {"workload": "prefill 27B-shaped GDN layer (16 qk / 48 v heads, d 128), 4 x 8192 tokens, "
                               "block 896, checkpoints every block; + decode 4B-shaped 256 seqs x 24 layers; "
                               "+ replay 16 req x 16 rows x 24 layers",
                   "io_dtype": "bf16 x/o, fp32 state",
                   "arithmetic": "tensor-core products as three bf16 passes (hi*hi + hi*lo + lo*hi of fp32 "
                                 "operands split into bf16 hi + lo) with fp32 accumulation; the rest fp32",
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (no flush)"},
        "prefill_ms": pre_ms, "decode_us_per_layer": 1000.0 * dec_ms / DEC_LAYERS,
        "replay_verify_us_per_layer": 1000.0 * ver_ms / REP_LAYERS,
        "flush_us_per_layer": 1000.0 * fl_ms / REP_LAYERS,
        "decode_hbm_gbs": dec_gbs, "flush_hbm_gbs": fl_gbs, "verify_hbm_gbs": ver_gbs,
        "decode_hbm_frac": dec_gbs / peaks["hbm_gbs"], "flush_hbm_frac": fl_gbs / peaks["hbm_gbs"],
        "verify_hbm_frac": ver_gbs / peaks["hbm_gbs"],
        # the same against the nominal HBM3e rate (a second denominator)
        "hbm_nominal_gbs": HBM_NOMINAL_GBS,
        "decode_hbm_frac_nominal": dec_gbs / HBM_NOMINAL_GBS, "flush_hbm_frac_nominal": fl_gbs / HBM_NOMINAL_GBS,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak,
                     "traffic": PREFILL_TRAFFIC_PER_CALL[path_key] if (args.seq_len == SEQ_LEN and args.num_seqs == N_SEQ) else None,
                     "traffic_note": "DRAM bytes per prefill call (every launch of the call summed; achieved "
                                     "is the call's work over its time), ncu capture of this workload",
                     "kernel": ("tc_chunk_kernel + tc_chain_kernel (the call)" if pre_plan["two_kernels"]
                                else "tc_prefill_kernel"),
                     "work": "chunk-form flops (C 64) per token and v-head x tokens x heads; "
                             "executed as 3 bf16 passes",
                     "executed_tflops": achieved * EXECUTED_FLOPS_PER_TOKEN_HEAD / CHUNK_FLOPS_PER_TOKEN_HEAD,
                     "executed_frac": achieved * EXECUTED_FLOPS_PER_TOKEN_HEAD / CHUNK_FLOPS_PER_TOKEN_HEAD / tc_peak,
                     # the algorithmic fraction with the tensor pipe busy all the time: three passes per
                     # product over M = 128 tiles execute this many times the algorithmic flops
                     "pass_ceiling": CHUNK_FLOPS_PER_TOKEN_HEAD / EXECUTED_FLOPS_PER_TOKEN_HEAD,
                     "peak_kind": f"dense bf16 {peak_kind} (burst)",
                     "algorithmic_bytes_per_call": pre.algorithmic_bytes(),
                     "hbm_gbs_achieved": pre.algorithmic_bytes() / (pre_ms * 1e-3) / 1e9,
                     # the call's measured DRAM traffic over its time: how close the path runs to HBM
                     "traffic_gbs": (PREFILL_TRAFFIC_PER_CALL[path_key] / (pre_ms * 1e-3) / 1e9
                                     if args.seq_len == SEQ_LEN and PREFILL_TRAFFIC_PER_CALL[path_key] else None),
                     "traffic_hbm_frac": (PREFILL_TRAFFIC_PER_CALL[path_key] / (pre_ms * 1e-3) / 1e9
                                          / peaks["hbm_gbs"]
                                          if args.seq_len == SEQ_LEN and PREFILL_TRAFFIC_PER_CALL[path_key]
                                          else None),
                     "hbm_peak_kind": peak_kind},
        "e2e": {"value": job_throughput(pre.tokens, world, e2e_ms), "unit": "tokens/s/layer",
                "h2d_bytes_per_step": pre.h2d_bytes, "d2h_bytes_per_step": pre.d2h_bytes, "steps": e2e_steps,
                "trials_ms_per_step": [round(t, 3) for t in e2e_trials], "reported": "median of the trials",
                "scope": "prefill part of the step; each step's input and output copies run on their own "
                         "streams, overlapping the neighbouring steps' prefill (three device buffer sets); "
                         "timed from the first input copy to the last output copy of `steps` steps",
                "link_measured": link,
                "copies_floor_ms": (pre.h2d_bytes + pre.d2h_bytes) / link["both_gbs"] / 1e6,
                "link_note": "the host link bounds the streamed step (copies_floor_ms: the step's bytes at the "
                             "link's measured both-ways rate on this box); it has measured ~295 GB/s both ways on "
                             "some boxes of the pool and well under 200 GB/s on others"},
        # per step: prefill (the launches of the path the library takes on
        # this GPU, + the window pass); decode 1 per layer; replay per layer:
        # append 2 (tensor-core append, log_len), rollback 1, flush 2
        "gpu_launches": args.steps * (pre_launches + 1 + DEC_LAYERS + 5 * REP_LAYERS),
        "prefill_path": "chunk + chain kernels" if pre_plan["two_kernels"] else "fused kernel",
        "prefill_paths": prefill_paths_ms(pre),
        "prefill_launches": pre_launches,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"]},
    }
    if not args.no_flush_sweep:
        line["flush_sweep"] = flush_sweep(args.seed + 40 + rank, peaks["hbm_gbs"])
    line["checkpoint_copy"] = checkpoint_copy(args.seed + 50 + rank, peaks["hbm_gbs"])
    if not args.no_flush_sweep:
        line["long_context"] = long_context(args.seed + 60 + rank)
    line["config"]["host_cpus"] = (f"{near_cpus} next to the GPU (end-to-end buffers)" if near_cpus
                                   else "not bound")
    os.sched_setaffinity(0, all_cpus)          # the oracle baseline uses every host core
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    # last key: a compact summary, so that the end of the line (what a log's
    # tail keeps of a long line) carries every headline figure
    line["summary"] = {
        "prefill_ms": round(pre_ms, 4), "prefill_tokens_per_s_layer": round(value),
        "prefill_tc_frac": round(achieved / tc_peak, 4),
        "decode_us_per_layer": round(1000.0 * dec_ms / DEC_LAYERS, 2), "decode_hbm_frac": round(dec_gbs / peaks["hbm_gbs"], 3),
        "verify_us_per_layer": round(1000.0 * ver_ms / REP_LAYERS, 2), "verify_hbm_frac": round(ver_gbs / peaks["hbm_gbs"], 3),
        "flush_us_per_layer": round(1000.0 * fl_ms / REP_LAYERS, 2), "flush_hbm_frac": round(fl_gbs / peaks["hbm_gbs"], 3),
        "e2e_tokens_per_s_layer": round(line["e2e"]["value"]),
        "e2e_ms_per_step": round(e2e_ms, 3), "e2e_copies_floor_ms": round(line["e2e"]["copies_floor_ms"], 3),
        "prefill_path": line["prefill_path"],
    }
    lc = line.get("long_context")
    if isinstance(lc, dict):
        line["summary"]["long_context"] = {k: lc[k] for k in lc if k.endswith("_ms")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
