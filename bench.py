"""Benchmark of one verify round of tree-speculative verification on a GDN hybrid.

One step is one pass of every step of the hot path over one batch of synthetic inputs:

  * tree prepare for the batch's draft trees;
  * the 24-layer gated-DeltaNet stack at batch 64 (B=64 sequences, 40-node k=3 d=3 trees,
    H=16, d=128, bf16) in fork/checkpoint mode -- verify all 24 layers, then commit all 24 --
    and in TreeWY mode -- verify all 24, then commit all 24 (separate S_0 buffers per mode).
    Fork mode runs in two passes per layer: the TreeWY pass (outputs and w) on the main stream
    and the snapshot pass on a side stream, overlapping the next layer's TreeWY pass;
  * one tree-masked attention layer at batch 32 (B=32, 16q/4kv, hd 256, bf16, paged prefixes
    P ~ U[2048, 32768], 40-node trees) followed by the KV compaction of its accepted paths.

``value`` = GDN node-layer verifications per second over the whole step (64 x 40 nodes x 24
layers x 2 modes per step, divided by the step time, attention rows included).  Every row is
also timed on its own with CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica (weak scaling, no collective on the data path).
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS = 24
# w scratch slots of the fork mode's two passes: the TreeWY passes run up to this many layers
# ahead of the snapshot passes (6 hides as much as 24 did in a sweep; 2 hid 15 us less per layer)
FORK_SLOTS = 6
METRIC = "tree-verified draft nodes/s per GDN layer; HBM GB/s & tensor util vs roofline"
WORKLOAD = ("GDN stack: 24 GDN layers, B=64, N=40 (k=3 d=3), H=16, dk=dv=128, bf16, fork+commit and "
            "TreeWY+commit; paged attention: tree attention B=32, 16q/4kv, hd=256, paged P~U[2048,32768], N=40, "
            "+ KV compaction")


# ----------------------------------------------------------------------------- accounting
def checkpoint_bytes(layers: int, heads: int, dk: int, dv: int, elem_bytes: int) -> int:
    """Bytes of one GDN checkpoint of a whole stack (qwen35-tree-spec §六: 24 x 16 x 128 x 128 x 2
    bytes ~ 12 MB)."""
    return layers * heads * dk * dv * elem_bytes


def gdn_bytes(B, N, H, dk, dv, e_io, e_state, mode, L_sum=0):
    """Algorithmic HBM bytes of one GDN layer call (inputs read once, outputs written once)."""
    inputs = B * (H * dv * dk * e_state + N * H * (2 * dk + dv) * e_io + N * H * 8 + N * 4)
    if mode == "fork":
        return inputs + B * N * H * dv * e_io + B * N * H * dv * dk * e_state
    if mode == "wy":
        return inputs + B * N * H * dv * e_io + B * N * H * dv * 4 + B * N * H * 4
    if mode == "materialize":  # the snapshot pass alone: S_0, k, w and alpha in, every snapshot out
        return (B * (H * dv * dk * e_state + N * H * (dk * e_io + dv * 4 + 4) + N * 4)
                + B * N * H * dv * dk * e_state)
    if mode == "commit_fork":
        return 2 * B * H * dv * dk * e_state + B * N * 4
    if mode == "commit_wy":
        return 2 * B * H * dv * dk * e_state + L_sum * H * (dv * 4 + dk * e_io + 4) + B * N * 4
    raise ValueError(mode)


def attn_bytes(prefix_lens, N, Hq, Hkv, hd, e=2):
    kv = sum(prefix_lens) * Hkv * hd * 2 * e
    nodes = len(prefix_lens) * N * (Hq + 2 * Hkv) * hd * e      # q, k_new, v_new
    writes = len(prefix_lens) * N * (2 * Hkv + Hq) * hd * e     # cache node slots + out
    return kv + nodes + writes


def attn_flops(prefix_lens, depths_per_seq, Hq, hd):
    """QK^T and PV over the visible keys of every node: 4 * hd flops per (query head, key)."""
    total = 0
    for P, dep in zip(prefix_lens, depths_per_seq):
        total += sum(4 * Hq * hd * (P + d + 1) for d in dep)
    return total


def _depths(parents):
    d = []
    for p in parents:
        d.append(0 if p < 0 else d[p] + 1)
    return d


def compact_bytes(path_lens, Hkv, hd, e=2):
    return sum(path_lens) * Hkv * hd * e * 2 * 2   # K and V, read + write


# ----------------------------------------------------------------------------- multi-rank
def max_over_ranks(dist, ms: float, device: str) -> float:
    """The slowest rank's time (every rank gets it); ``dist`` None means a single process."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank (weak scaling)."""
    return units_per_rank * world / (ms * 1e-3)


# ----------------------------------------------------------------------------- helpers
def kernel_traffic(row: str):
    """dram read+write bytes per launch of a row's main kernel from ``profiles/traffic.txt``, a
    summary of an ncu capture; null when the kernel's source changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for ln in f:
            parts = ln.split()
            if len(parts) >= 4 and parts[0] == row:
                src = os.path.join(ROOT, "tree_speculative_verification_gdn_gb300", "csrc", parts[2])
                if not os.path.exists(src):
                    return None
                with open(src, "rb") as g:
                    digest = hashlib.sha256(g.read()).hexdigest()[:16]
                return float(parts[1]) if digest == parts[3] else None
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- our arm
class Round:
    """Device buffers of one verify round and the sequence of ABI calls that run it."""

    def __init__(self, rank: int, layers: int, torch, tv, W):
        self.torch, self.tv = torch, tv
        dev = torch.device("cuda", torch.cuda.current_device())
        self.dev = dev
        seed = 1000 * rank
        self.seed = seed
        self.layers = layers
        self.gdn_host = [W.stack_b64_layer(layer=l, seed=seed) for l in range(layers)]
        c0 = self.gdn_host[0]
        self.B, self.N, self.H, self.dk, self.dv = c0.shape
        B, N, H, dk, dv = self.B, self.N, self.H, self.dk, self.dv
        self.attn_host = W.paged_attn_b32_case(seed=seed)
        a = self.attn_host
        self.aB, self.aN, self.Hq, self.Hkv, self.hd = a.shape

        def d(t):
            return t.contiguous().to(dev)

        # per-round inputs (copied from host in the end-to-end measurement); every layer's keys lie
        # in one [layers, B, N, H, dk] tensor, which the stack's TreeWY commit reads in one launch
        self.k_all = torch.stack([c.k for c in self.gdn_host]).contiguous().to(dev)
        self.in_gdn = [dict(q=d(c.q), k=self.k_all[l], v=d(c.v), alpha=d(c.alpha), beta=d(c.beta))
                       for l, c in enumerate(self.gdn_host)]
        self.parents = d(c0.parents)
        # draft and target tokens under which the on-device accept walk takes the sampled paths
        draft, target = W.walk_tokens(c0.trees, c0.path.numpy(), c0.path_len.numpy(), seed=seed + 1)
        self.tokens = dict(draft=d(draft), target=d(target))
        self.in_attn = dict(q=d(a.q), k_new=d(a.k_new), v_new=d(a.v_new), block_table=d(a.block_table),
                            prefix_len=d(a.prefix_len), parents=d(a.parents))
        draft, target = W.walk_tokens(a.trees, a.path.numpy(), a.path_len.numpy(), seed=seed + 2)
        self.a_tokens = dict(draft=d(draft), target=d(target))
        # resident state, each mode's layers back to back ([layers, B, H, dv, dk]) so that one launch
        # commits the stack; S0_fork[l] / S0_wy[l] are views of layer l
        self.S0_fork_all = torch.stack([c.S0 for c in self.gdn_host]).contiguous().to(dev)
        self.S0_wy_all = self.S0_fork_all.clone()
        self.S0_fork = [self.S0_fork_all[l] for l in range(layers)]
        self.S0_wy = [self.S0_wy_all[l] for l in range(layers)]
        self.k_cache, self.v_cache = d(a.k_cache), d(a.v_cache)
        # outputs
        bf = torch.bfloat16
        self.o_fork = [torch.empty((B, N, H, dv), dtype=bf, device=dev) for _ in range(layers)]
        self.o_wy = [torch.empty((B, N, H, dv), dtype=bf, device=dev) for _ in range(layers)]
        mem0 = torch.cuda.memory_allocated()
        self.states_all = torch.empty((layers, B, N, H, dv, dk), dtype=bf, device=dev)
        self.states = [self.states_all[l] for l in range(layers)]
        self.fork_state_bytes = torch.cuda.memory_allocated() - mem0
        mem0 = torch.cuda.memory_allocated()
        self.pv_all = torch.empty((layers, B, N, H, dv), dtype=torch.float32, device=dev)
        self.lg_all = torch.empty((layers, B, N, H), dtype=torch.float32, device=dev)
        self.pv = [self.pv_all[l] for l in range(layers)]
        self.lg = [self.lg_all[l] for l in range(layers)]
        self.wy_state_bytes = torch.cuda.memory_allocated() - mem0
        i32 = torch.int32
        # accepted paths: written by the accept walk each round, read by the commits / compaction
        self.path = torch.empty(c0.path.shape, dtype=i32, device=dev)
        self.path_len = torch.empty((B,), dtype=i32, device=dev)
        self.next_tok = torch.empty((B,), dtype=i32, device=dev)
        self.a_path = torch.empty(a.path.shape, dtype=i32, device=dev)
        self.a_path_len = torch.empty((self.aB,), dtype=i32, device=dev)
        self.a_next_tok = torch.empty((self.aB,), dtype=i32, device=dev)
        self.depth = torch.empty((B, N), dtype=i32, device=dev)
        self.mask = torch.empty((B, N, (N + 31) // 32), dtype=i32, device=dev)
        # rows 0..15: one per call site; row 16 + l: fork-mode layer l (its two passes overlap
        # the next layer's on two streams, so every layer has a status row of its own)
        self.err = torch.zeros((16 + layers, max(B, self.aB)), dtype=i32, device=dev)
        self.a_out = torch.empty((self.aB, self.aN, self.Hq, self.hd), dtype=bf, device=dev)
        ws = tv.tv_tree_attn_workspace_size(self.aB, self.aN, self.Hq, self.Hkv, self.hd, a.block_table.shape[1])
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.slot_map = torch.empty(a.path.shape, dtype=i32, device=dev)
        # fork mode: the TreeWY pass of layer l writes w into slot l % FORK_SLOTS, the snapshot
        # pass of layer l reads it on the side stream while the next layers' TreeWY passes run
        self.side = torch.cuda.Stream()
        self.fork_pv = [torch.empty((B, N, H, dv), dtype=torch.float32, device=dev) for _ in range(FORK_SLOTS)]
        self.fork_lg = [torch.empty((B, N, H), dtype=torch.float32, device=dev) for _ in range(FORK_SLOTS)]
        self.w_ready = [torch.cuda.Event() for _ in range(layers)]
        self.slot_free = [torch.cuda.Event() for _ in range(FORK_SLOTS)]
        self.new_len = torch.empty((self.aB,), dtype=i32, device=dev)
        self.rows = ["tree_prepare", "fork_verify", "fork_materialize", "accept_walk", "fork_commit", "wy_verify",
                     "wy_commit", "tree_attn", "kv_compact"]
        # tree prepare; per layer the fork's two passes and the TreeWY verify; one commit launch per
        # mode for the whole stack; two accept walks; three attention kernels; the compaction
        self.launches_per_step = 1 + layers * 3 + 2 + 2 + 3 + 1

    def step(self, ev=None, io=None):
        """One verify round.  ``ev``: optional dict row -> list of (start, end, calls) entries.
        ``io``: optional ``HostIO`` whose hooks order the step against its host copies."""
        torch, tv = self.torch, self.tv
        B = self.B
        err = self.err
        main = torch.cuda.current_stream()
        if io is not None:
            io.start(main)

        def timing_event(stream):
            if ev is None:
                return None
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            return e

        def mark(row, fn, stream=None, calls=1):
            st = main if stream is None else stream
            s = timing_event(st)
            fn()
            if ev is not None:
                ev[row].append((s, timing_event(st), calls))

        mark("tree_prepare", lambda: tv.tv_tree_prepare(self.parents, self.depth, self.mask, err[0, :B]))
        # Fork mode in two passes: the TreeWY pass (every output, and w) on this stream, then the
        # snapshot pass on the side stream, which the next layer's TreeWY pass overlaps -- the
        # next layer needs the outputs, not the snapshots.  The row spans all layers.
        f0 = timing_event(main)
        for l in range(self.layers):
            x = self.in_gdn[l]
            slot = l % FORK_SLOTS
            if l >= FORK_SLOTS:
                main.wait_event(self.slot_free[slot])   # the snapshot pass that used it has read it
            if io is not None:
                io.layer_inputs(main, l)
            tv.tv_gdn_tree_verify_wy(x["q"], x["k"], x["v"], x["alpha"], x["beta"], self.S0_fork[l], self.parents,
                                     self.o_fork[l], self.fork_pv[slot], self.fork_lg[slot], err[16 + l, :B])
            if io is not None:
                io.output(main, "fork", l)
            self.w_ready[l].record(main)
            self.side.wait_event(self.w_ready[l])
            mark("fork_materialize", lambda: tv.tv_gdn_fork_materialize(
                x["k"], x["alpha"], self.S0_fork[l], self.parents, self.fork_pv[slot], self.states[l],
                err[16 + l, :B], stream=self.side), stream=self.side)
            self.slot_free[slot].record(self.side)
        main.wait_stream(self.side)
        if ev is not None:
            ev["fork_verify"].append((f0, timing_event(main), self.layers))
        # the target's tokens pick the accepted path on the device (one walk feeds both modes' commits)
        mark("accept_walk", lambda: tv.tv_accept_walk(
            self.parents, self.tokens["draft"], self.tokens["target"], self.path, self.path_len, self.next_tok,
            err[7, :B]))
        # every layer commits the accepted paths at once: one launch for the stack
        mark("fork_commit", lambda: tv.tv_gdn_commit_layers(
            tv.TV_MODE_FORK, self.path, self.path_len, self.parents, self.S0_fork_all, err[2, :B],
            node_states=self.states_all), calls=self.layers)
        for l in range(self.layers):
            x = self.in_gdn[l]
            mark("wy_verify", lambda: tv.tv_gdn_tree_verify_wy(
                x["q"], x["k"], x["v"], x["alpha"], x["beta"], self.S0_wy[l], self.parents, self.o_wy[l],
                self.pv[l], self.lg[l], err[3, :B]))
            if io is not None:
                io.output(main, "wy", l)
        mark("wy_commit", lambda: tv.tv_gdn_commit_layers(
            tv.TV_MODE_WY, self.path, self.path_len, self.parents, self.S0_wy_all, err[4, :B],
            pseudo_v=self.pv_all, log_gamma=self.lg_all, k=self.k_all), calls=self.layers)
        if io is not None:
            for l in range(self.layers):
                io.layer_done(main, l)   # the last reader of the layers' inputs has been issued
        a = self.in_attn
        aB = self.aB
        if io is not None:
            io.attn_inputs(main)
        mark("tree_attn", lambda: tv.tv_tree_attn(
            a["q"], a["k_new"], a["v_new"], self.k_cache, self.v_cache, a["block_table"], a["prefix_len"],
            a["parents"], self.a_out, self.ws, err[5, :aB], rope_theta=1e6))
        mark("accept_walk", lambda: tv.tv_accept_walk(
            a["parents"], self.a_tokens["draft"], self.a_tokens["target"], self.a_path, self.a_path_len,
            self.a_next_tok, err[8, :aB]))
        if io is not None:
            io.output(main, "attn", 0)
        mark("kv_compact", lambda: tv.tv_kv_compact(
            self.k_cache, self.v_cache, a["block_table"], a["prefix_len"], a["parents"], self.a_path,
            self.a_path_len, self.slot_map, self.new_len, err[6, :aB]))
        if io is not None:
            io.finish(main)

    # end-to-end: per-round inputs from pinned host memory, outputs back to pinned host memory
    def host_buffers(self):
        # a second set of per-layer input buffers: a step's uploads go into the set the step
        # before did not use, so they need not wait for that step's readers
        torch = self.torch
        k2 = torch.empty_like(self.k_all)
        in2 = [dict(q=torch.empty_like(x["q"]), k=k2[l], v=torch.empty_like(x["v"]),
                    alpha=torch.empty_like(x["alpha"]), beta=torch.empty_like(x["beta"]))
               for l, x in enumerate(self.in_gdn)]
        self.in_sets = [(self.in_gdn, self.k_all), (in2, k2)]
        self.e2e_steps = 0
        self.io = HostIO(self)
        return self.io.h2d_bytes, self.io.d2h_bytes

    def step_e2e(self):
        parity = self.e2e_steps % 2
        self.in_gdn, self.k_all = self.in_sets[parity]
        self.io.upload(parity)
        self.step(io=self.io)
        self.e2e_steps += 1

    def end_e2e(self):
        self.in_gdn, self.k_all = self.in_sets[0]


class HostIO:
    """Pinned host buffers and two copy streams for the end-to-end measurement.  Each layer's
    inputs go up on one stream ahead of their first use, into the input set the previous step
    did not use, as soon as the last reader of that set (two steps back) has been issued; each
    output comes back on the other stream as soon as its kernel has written it.  Both overlap
    the kernels.  The step ends only after every download, so the timed region holds all of
    them."""

    def __init__(self, rnd):
        torch = rnd.torch
        self.torch, self.rnd = torch, rnd
        pin = lambda t: t.detach().cpu().pin_memory()  # noqa: E731
        self.h_in = [{k: pin(v) for k, v in x.items()} for x in rnd.in_gdn]
        self.h_attn = {k: pin(v) for k, v in rnd.in_attn.items()}
        self.h_parents = pin(rnd.parents)
        self.h_tokens = [{k: pin(v) for k, v in x.items()} for x in (rnd.tokens, rnd.a_tokens)]
        self.h_o_fork = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in rnd.o_fork]
        self.h_o_wy = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in rnd.o_wy]
        self.h_a_out = torch.empty(rnd.a_out.shape, dtype=rnd.a_out.dtype).pin_memory()
        self.h_err = torch.empty(rnd.err.shape, dtype=rnd.err.dtype).pin_memory()
        self.small = (rnd.slot_map, rnd.new_len, rnd.next_tok, rnd.a_next_tok)
        self.h_small = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in self.small]
        h2d = sum(t.numel() * t.element_size() for x in self.h_in for t in x.values())
        h2d += sum(t.numel() * t.element_size() for t in self.h_attn.values())
        h2d += self.h_parents.numel() * 4 + sum(t.numel() * 4 for x in self.h_tokens for t in x.values())
        d2h = sum(t.numel() * t.element_size() for t in self.h_o_fork + self.h_o_wy)
        d2h += self.h_a_out.numel() * 2 + self.h_err.numel() * 4 + sum(t.numel() * 4 for t in self.h_small)
        self.h2d_bytes, self.d2h_bytes = h2d, d2h
        self.up, self.down = torch.cuda.Stream(), torch.cuda.Stream()
        L = rnd.layers
        ev = torch.cuda.Event
        self.in_ready = [[ev() for _ in range(L)] for _ in range(2)]
        self.in_free = [[ev() for _ in range(L)] for _ in range(2)]
        self.parity = 0
        self.out_ev = {"fork": [ev() for _ in range(L)], "wy": [ev() for _ in range(L)], "attn": [ev()]}
        self.pre_ready, self.pre_free = ev(), ev()
        self.attn_ready, self.attn_free = ev(), ev()
        self.end = ev()

    def upload(self, parity):
        """Every input copy of one step into input set `parity`, on the upload stream, each
        behind the event that frees its device buffer (never recorded before its first use: no
        wait)."""
        torch, rnd, up = self.torch, self.rnd, self.up
        self.parity = parity
        with torch.cuda.stream(up):
            up.wait_event(self.pre_free)
            rnd.parents.copy_(self.h_parents, non_blocking=True)
            for dst, src in zip((rnd.tokens, rnd.a_tokens), self.h_tokens):
                for k in dst:
                    dst[k].copy_(src[k], non_blocking=True)
            self.pre_ready.record(up)
            for l, (dst, src) in enumerate(zip(rnd.in_sets[parity][0], self.h_in)):
                up.wait_event(self.in_free[parity][l])
                for k in dst:
                    dst[k].copy_(src[k], non_blocking=True)
                self.in_ready[parity][l].record(up)
            up.wait_event(self.attn_free)
            for k in rnd.in_attn:
                rnd.in_attn[k].copy_(self.h_attn[k], non_blocking=True)
            self.attn_ready.record(up)

    # hooks called by Round.step on the main stream
    def start(self, main):
        main.wait_event(self.pre_ready)

    def layer_inputs(self, main, l):
        main.wait_event(self.in_ready[self.parity][l])

    def layer_done(self, main, l):
        self.in_free[self.parity][l].record(main)

    def attn_inputs(self, main):
        main.wait_event(self.attn_ready)

    def output(self, main, kind, l):
        torch, rnd, down = self.torch, self.rnd, self.down
        e = self.out_ev[kind][l]
        e.record(main)
        down.wait_event(e)
        with torch.cuda.stream(down):
            if kind == "fork":
                self.h_o_fork[l].copy_(rnd.o_fork[l], non_blocking=True)
            elif kind == "wy":
                self.h_o_wy[l].copy_(rnd.o_wy[l], non_blocking=True)
            else:
                self.h_a_out.copy_(rnd.a_out, non_blocking=True)

    def finish(self, main):
        torch, rnd, down = self.torch, self.rnd, self.down
        self.attn_free.record(main)
        self.pre_free.record(main)
        self.end.record(main)
        down.wait_event(self.end)
        with torch.cuda.stream(down):
            self.h_err.copy_(rnd.err, non_blocking=True)
            for h, d in zip(self.h_small, self.small):
                h.copy_(d, non_blocking=True)
        main.wait_stream(down)


class OraclePool:
    """The fp64 oracle, as it stands, on every host core: one sequence of the batch-64 GDN stack (40 nodes,
    16 heads, one GDN layer) per task through ``oracle.gdn.verify_by_depth``, in spawned worker
    processes with single-threaded BLAS.  Started before any GPU work."""

    def __init__(self, cores: int | None = None):
        import concurrent.futures as cf
        import multiprocessing as mp
        self.cores = cores or os.cpu_count() or 1
        env_keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
        old = {k: os.environ.get(k) for k in env_keys}
        for k in env_keys:
            os.environ[k] = "1"
        try:
            self.ex = cf.ProcessPoolExecutor(max_workers=self.cores, mp_context=mp.get_context("spawn"),
                                             initializer=_oracle_init)
            list(self.ex.map(_oracle_sequence, [0] * self.cores))   # imports + input generation
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.next_b = 0

    def sample(self, seconds: float) -> dict:
        t0 = time.perf_counter()
        done = 0
        while True:
            list(self.ex.map(_oracle_sequence, [(self.next_b + j) % 64 for j in range(self.cores)]))
            self.next_b += self.cores
            done += self.cores
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
        return {"value": done * 40 / dt, "unit": "nodes/s", "cores": self.cores, "kind": "oracle",
                "sample": f"{done} sequences of the batch-64 GDN stack (40 nodes x 16 heads, one GDN layer, bf16 inputs in fp64) "
                          f"through the oracle's depth-by-depth schedule in {dt:.1f} s"}

    def close(self):
        self.ex.shutdown()


_ORACLE_CACHE = {}


def _oracle_init():
    import workloads as W
    _ORACLE_CACHE["inp"] = W.stack_b64_layer(layer=0).oracle_inputs()


def _oracle_sequence(b):
    import numpy as np
    from oracle import gdn as G
    inp = _ORACLE_CACHE["inp"]
    sub = {k: (v[b:b + 1] if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    G.verify_by_depth(sub)
    return b


def selective_fork_report(rnd, torch, tv, iters: int = 3) -> dict:
    """Fork mode with selective snapshots (qwen35-tree-spec §六, 选择性 Fork) on the same 24-layer
    stack, timed apart from the step: nodes with draft confidence above 0.95 keep no snapshot
    (synthetic confidences, about half of the nodes above the threshold), and the commit
    replays from the deepest kept snapshot of the accepted path.  Verify runs in the step's
    two-pass schedule (TreeWY passes on this stream, selective snapshot passes on the side
    stream, six w slots); the one-pass selective kernel is timed too."""
    import numpy as np
    B, N, H, dk, dv, L = rnd.B, rnd.N, rnd.H, rnd.dk, rnd.dv, rnd.layers
    rng = np.random.default_rng(99)
    high = rng.random((B, N)) < 0.5
    conf_np = np.where(high, rng.uniform(0.951, 1.0, (B, N)), rng.uniform(0.0, 0.95, (B, N))).astype(np.float32)
    kept = int((conf_np <= 0.95).sum(axis=1).max())
    conf = torch.from_numpy(conf_np).to(rnd.dev)
    states = [torch.empty((B, kept, H, dv, dk), dtype=torch.bfloat16, device=rnd.dev) for _ in range(L)]
    slot = [torch.empty((B, N), dtype=torch.int32, device=rnd.dev) for _ in range(L)]
    S0 = [s.clone() for s in rnd.S0_fork]
    out = torch.empty_like(rnd.o_fork[0])
    err = torch.zeros((L + 2, B), dtype=torch.int32, device=rnd.dev)
    main, side = torch.cuda.current_stream(), rnd.side
    ev = torch.cuda.Event

    def two_pass():
        for l in range(L):
            x = rnd.in_gdn[l]
            k = l % FORK_SLOTS
            if l >= FORK_SLOTS:
                main.wait_event(rnd.slot_free[k])
            tv.tv_gdn_tree_verify_wy(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0[l], rnd.parents, out,
                                     rnd.fork_pv[k], rnd.fork_lg[k], err[l])
            rnd.w_ready[l].record(main)
            side.wait_event(rnd.w_ready[l])
            tv.tv_gdn_fork_materialize_selective(x["k"], x["alpha"], S0[l], rnd.parents, rnd.fork_pv[k], conf, 0.95,
                                                 states[l], slot[l], err[l], stream=side)
            rnd.slot_free[k].record(side)
        main.wait_stream(side)

    def commits():
        for l in range(L):
            x = rnd.in_gdn[l]
            tv.tv_gdn_commit_selective(rnd.path, rnd.path_len, rnd.parents, states[l], slot[l], x["k"], x["v"],
                                       x["alpha"], x["beta"], S0[l], err[L])

    def one_pass():
        for l in range(L):
            x = rnd.in_gdn[l]
            tv.tv_gdn_tree_verify_fork_selective(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0[l], rnd.parents,
                                                 conf, 0.95, out, states[l], slot[l], err[L + 1])

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(iters):
            s_, e_ = ev(enable_timing=True), ev(enable_timing=True)
            s_.record(main)
            fn()
            e_.record(main)
            torch.cuda.synchronize()
            t.append(s_.elapsed_time(e_) / L)
        return sum(t) / len(t)

    v_ms = timed(two_pass)
    c_ms = timed(commits)       # after a verify: its snapshots and slots are in place
    p_ms = timed(one_pass)
    assert int(err.abs().sum()) == 0, err
    full = B * N * H * dv * dk * 2
    return {"threshold": 0.95, "kept_fraction": round(float((conf_np <= 0.95).mean()), 4),
            "snapshot_bytes_per_layer": B * kept * H * dv * dk * 2, "full_checkpoint_bytes_per_layer": full,
            "verify_ms_per_layer": round(v_ms, 5), "commit_ms_per_layer": round(c_ms, 5),
            "one_pass_verify_ms_per_layer": round(p_ms, 5)}


def one_pass_fork_report(rnd, torch, tv, iters: int = 3) -> dict:
    """The one-pass fork verify (each row's dot products computed along the walk) on the same
    24-layer stack, timed apart from the step, which uses the two-pass form."""
    err = torch.zeros((rnd.B,), dtype=torch.int32, device=rnd.dev)
    S0 = [s.clone() for s in rnd.S0_fork]

    def once(ev=None):
        for l in range(rnd.layers):
            x = rnd.in_gdn[l]
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            tv.tv_gdn_tree_verify_fork(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0[l], rnd.parents,
                                       rnd.o_fork[l], rnd.states[l], err)
            e.record()
            if ev is not None:
                ev.append((s, e))
    once()
    torch.cuda.synchronize()
    ev = []
    for _ in range(iters):
        once(ev)
    torch.cuda.synchronize()
    assert int(err.abs().sum()) == 0, err
    return {"ms_per_layer": round(sum(s.elapsed_time(e) for s, e in ev) / len(ev), 5)}


def lazy_commit_report(rnd, torch, tv, iters: int = 3) -> dict:
    """TreeWY with the previous round's commit fused into this round's verify, on the same
    24-layer stack, timed apart from the step: each layer's last W, log(gamma), keys and the
    accepted paths stand for the previous round."""
    B, N, H, dv, L = rnd.B, rnd.N, rnd.H, rnd.dv, rnd.layers
    S0 = [s.clone() for s in rnd.S0_wy]
    out = torch.empty_like(rnd.o_wy[0])
    pv = [torch.empty_like(p) for p in rnd.pv]
    lg = [torch.empty_like(g) for g in rnd.lg]
    err = torch.zeros((B,), dtype=torch.int32, device=rnd.dev)

    def once(ev=None):
        for l in range(L):
            x = rnd.in_gdn[l]
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            tv.tv_gdn_tree_verify_wy_lazy(rnd.path, rnd.path_len, rnd.parents, rnd.pv[l], rnd.lg[l], x["k"], x["q"],
                                          x["k"], x["v"], x["alpha"], x["beta"], S0[l], rnd.parents, out, pv[l], lg[l],
                                          err)
            e.record()
            if ev is not None:
                ev.append((s, e))
    once()
    torch.cuda.synchronize()
    ev = []
    for _ in range(iters):
        once(ev)
    torch.cuda.synchronize()
    assert int(err.abs().sum()) == 0, err
    return {"fused_ms_per_layer": round(sum(s.elapsed_time(e) for s, e in ev) / len(ev), 5),
            "bytes_saved_per_layer": B * H * dv * dv * 2}


def block_table_compaction_report(rnd, torch, tv, W, iters: int = 20) -> dict:
    """Compaction of accepted paths that run down long draft chains, on the step's paged cache
    (batch 32, 4 KV heads, hd 256): a root with chains of 16, 16 and 7 nodes (40 nodes, as the
    step's trees), each path down one chain.  Moving every kept entry (``tv_kv_compact``)
    against exchanging whole blocks of the table where it can (``tv_kv_compact_remap``)."""
    import numpy as np
    aB, aN = rnd.aB, rnd.aN
    assert aN == 1 + sum(W.CHAIN_LENGTHS)
    parents = torch.tensor([W.candidate_chains(W.CHAIN_LENGTHS)] * aB, dtype=torch.int32, device=rnd.dev)
    paths = W.candidate_chain_paths(W.CHAIN_LENGTHS, aB, np.random.default_rng(rnd.seed + 21))
    lens = [len(p) for p in paths]
    Lmax = max(lens)
    path = torch.tensor([p + [-1] * (Lmax - len(p)) for p in paths], dtype=torch.int32, device=rnd.dev)
    path_len = torch.tensor(lens, dtype=torch.int32, device=rnd.dev)
    table, plen = rnd.in_attn["block_table"], rnd.in_attn["prefix_len"]
    table_out = torch.empty_like(table)
    i32 = dict(dtype=torch.int32, device=rnd.dev)
    slot_map, new_len = torch.empty((aB, Lmax), **i32), torch.empty((aB,), **i32)
    remapped, err = torch.zeros((aB,), **i32), torch.zeros((2, aB), **i32)

    def copy_form():
        tv.tv_kv_compact(rnd.k_cache, rnd.v_cache, table, plen, parents, path, path_len, slot_map, new_len, err[0])

    def remap_form():
        tv.tv_kv_compact_remap(rnd.k_cache, rnd.v_cache, table, table_out, plen, parents, path, path_len,
                               slot_map, new_len, remapped, err[1])

    def timed(fn):
        # a call takes microseconds on the device and longer to issue from Python: the calls are
        # queued behind a device-side sleep so that the events bracket device time only
        fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(4_000_000)
        s.record()
        for _ in range(iters):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / iters

    ms_copy = timed(copy_form)
    ms_remap = timed(remap_form)
    assert int(err.abs().sum()) == 0, err
    return {"tree": "root + chains of 16, 16, 7 nodes", "kept_entries": sum(lens),
            "blocks_exchanged": int(remapped.sum()),
            "copy_form_bytes": compact_bytes(lens, rnd.Hkv, rnd.hd),
            "copy_form_ms": round(ms_copy, 5), "block_table_form_ms": round(ms_remap, 5)}


# ----------------------------------------------------------------------------- wide-tree sweep
HYBRID_GDN_LAYERS, HYBRID_ATTN_LAYERS, HYBRID_PREFIX = 24, 8, 8192
GRID_N = (15, 40, 64, 128, 256)
GRID_B = (1, 8, 32, 128)


def device_timed(torch, fn, iters: int, launches: int) -> float:
    """Mean device time of ``fn`` (ms) over ``iters`` calls issued behind a device-side sleep,
    so that the events bracket device time even where issuing the launches from Python takes
    longer than running them (the small trees are launch-latency-bound)."""
    fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2e6 + 4e4 * launches * iters))
    s.record()
    for _ in range(iters):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def hybrid_point(torch, tv, W, peaks, B: int, N: int, trees, gdn_layers: int, attn_layers: int, prefix: int,
                 seed: int, iters: int = 3) -> dict:
    """One verify round of a synthetic hybrid stack (``attn_layers`` groups of gdn_layers /
    attn_layers GDN layers and one attention layer; 3:1 at 24 + 8) over B sequences of N-node
    trees, in fork mode and in TreeWY mode, each followed by the accept walk, the stacked GDN
    commit and the compaction of every attention layer's cache.  Per mode: the round's device
    time, the GDN part alone (verify + commit per layer), and the measured peak of device memory
    the mode adds (torch.cuda.max_memory_allocated over the mode's buffers and its rounds; the
    library allocates nothing).  Fork mode is run only where its snapshots fit the free device
    memory; otherwise the point reports the bytes it would need."""
    import numpy as np
    dev = torch.device("cuda", torch.cuda.current_device())
    H, d, Hq, Hkv, hd = 16, 128, 16, 4, 128
    L = gdn_layers
    i32 = dict(dtype=torch.int32, device=dev)
    parents = torch.tensor(np.array(trees, dtype=np.int32), device=dev)
    rng = np.random.default_rng(seed + 17)
    paths = [W.random_accepted_path(t, rng, 4) for t in trees]
    Lmax = max(len(p) for p in paths)
    p_np = np.array([p + [-1] * (Lmax - len(p)) for p in paths], dtype=np.int32)
    l_np = np.array([len(p) for p in paths], dtype=np.int32)
    draft, target = W.walk_tokens(trees, p_np, l_np, seed=seed + 18)
    draft, target = draft.to(dev), target.to(dev)
    g = W.device_gdn_stack(L, B, N, H, d, seed=seed + 19, device=dev)
    attn = [W.device_attn_layer(B, N, prefix, Hq, Hkv, hd, seed=seed + 100 + j, device=dev) for j in range(attn_layers)]
    ws = None
    if attn_layers:
        ws = torch.empty(tv.tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, attn[0]["block_table"].shape[1]),
                         dtype=torch.uint8, device=dev)
    a_out = torch.empty((B, N, Hq, hd), dtype=torch.bfloat16, device=dev)
    path, plen, nxt = torch.empty((B, Lmax), **i32), torch.empty((B,), **i32), torch.empty((B,), **i32)
    smap, new_len = torch.empty((B, Lmax), **i32), torch.empty((B,), **i32)
    err = torch.zeros((8 + L, B), **i32)
    o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=dev)
    per_group = L // attn_layers if attn_layers else L
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    max_depth = max(max(_depths(t)) for t in trees)

    def attn_layer(j):
        x = attn[j]
        tv.tv_tree_attn(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["block_table"],
                        x["prefix_len"], parents, a_out, ws, err[4], rope_theta=1e6)

    def compactions():
        for x in attn:
            tv.tv_kv_compact(x["k_cache"], x["v_cache"], x["block_table"], x["prefix_len"], parents, path, plen,
                             smap, new_len, err[5])

    def attn_only():
        for j in range(attn_layers):
            attn_layer(j)
        compactions()

    tv.tv_accept_walk(parents, draft, target, path, plen, nxt, err[1])   # the paths the compactions read
    torch.cuda.synchronize()
    out = {"B": B, "N": N, "max_depth": max_depth}
    if attn_layers:
        a_ms = device_timed(torch, attn_only, iters, 5 * attn_layers)
        ab = attn_bytes([prefix] * B, N, Hq, Hkv, hd)
        af = attn_flops([prefix] * B, [_depths(t) for t in trees], Hq, hd)
        out["attention"] = {"ms_per_layer_with_compaction": round(a_ms / attn_layers, 5),
                            "frac_hbm": round(ab / (a_ms / attn_layers * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                            "tflops": round(af / (a_ms / attn_layers * 1e-3) / 1e12, 2)}
    for mode in ("fork", "wy"):
        state_bytes = (L * B * N * H * d * d * 2 if mode == "fork" else L * B * N * H * (d + 1) * 4)
        torch.cuda.synchronize()
        free, total = torch.cuda.mem_get_info()
        reserve_free = torch.cuda.memory_reserved() - torch.cuda.memory_allocated()
        slots = min(FORK_SLOTS, L)
        extra = B * N * H * (d + 1) * 4 * slots + L * B * H * d * d * 2 if mode == "fork" else L * B * H * d * d * 2
        if state_bytes + extra > free + reserve_free - (2 << 30):
            out[mode] = {"exceeds_hbm": True, "state_bytes_predicted": state_bytes,
                         "free_bytes": free + reserve_free}
            continue
        S0 = g["S0"].clone()            # the mode's resident state, an input of both modes
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        if mode == "fork":
            states = torch.empty((L, B, N, H, d, d), dtype=torch.bfloat16, device=dev)
            w = [torch.empty((B, N, H, d), dtype=torch.float32, device=dev) for _ in range(slots)]
            lgs = [torch.empty((B, N, H), dtype=torch.float32, device=dev) for _ in range(slots)]
            w_ready = [torch.cuda.Event() for _ in range(L)]
            slot_free = [torch.cuda.Event() for _ in range(slots)]
        else:
            pv = torch.empty((L, B, N, H, d), dtype=torch.float32, device=dev)
            lg = torch.empty((L, B, N, H), dtype=torch.float32, device=dev)

        def gdn_layer(l):
            if mode == "wy":
                tv.tv_gdn_tree_verify_wy(g["q"][l], g["k"][l], g["v"][l], g["alpha"][l], g["beta"][l], S0[l], parents,
                                         o, pv[l], lg[l], err[0])
                return
            k = l % slots
            if l >= slots:
                main.wait_event(slot_free[k])
            tv.tv_gdn_tree_verify_wy(g["q"][l], g["k"][l], g["v"][l], g["alpha"][l], g["beta"][l], S0[l], parents,
                                     o, w[k], lgs[k], err[8 + l])
            w_ready[l].record(main)
            side.wait_event(w_ready[l])
            tv.tv_gdn_fork_materialize(g["k"][l], g["alpha"][l], S0[l], parents, w[k], states[l], err[8 + l],
                                       stream=side)
            slot_free[k].record(side)

        def commit():
            tv.tv_accept_walk(parents, draft, target, path, plen, nxt, err[1])
            if mode == "fork":
                tv.tv_gdn_commit_layers(tv.TV_MODE_FORK, path, plen, parents, S0, err[2], node_states=states)
            else:
                tv.tv_gdn_commit_layers(tv.TV_MODE_WY, path, plen, parents, S0, err[3], pseudo_v=pv, log_gamma=lg,
                                        k=g["k"])

        def gdn_only():
            for l in range(L):
                gdn_layer(l)
            main.wait_stream(side)
            commit()

        def hybrid():
            for l in range(L):
                gdn_layer(l)
                if attn_layers and (l + 1) % per_group == 0:
                    attn_layer((l + 1) // per_group - 1)
            main.wait_stream(side)
            commit()
            if attn_layers:
                compactions()

        nl = L * (2 if mode == "fork" else 1)
        g_ms = device_timed(torch, gdn_only, iters, nl + 2)
        r_ms = device_timed(torch, hybrid, iters, nl + 2 + 5 * attn_layers) if attn_layers else g_ms
        peak = torch.cuda.max_memory_allocated() - base
        assert int(err.abs().sum()) == 0, (mode, B, N, err.cpu().tolist())
        gb = gdn_bytes(B, N, H, d, d, 2, 2, "fork" if mode == "fork" else "wy")
        per_layer = g_ms / L
        out[mode] = {"round_ms": round(r_ms, 4), "round_nodes_per_s": round(B * N / (r_ms * 1e-3)),
                     "gdn_ms_per_layer": round(per_layer, 5),
                     "gdn_nodes_per_s_per_layer": round(B * N / (per_layer * 1e-3)),
                     "gdn_frac_hbm": round(gb / (per_layer * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "state_bytes": state_bytes, "peak_bytes_measured": int(peak)}
        if mode == "fork":
            del states, w, lgs
        else:
            del pv, lg
        del S0
        torch.cuda.synchronize()
    del g, attn, ws
    torch.cuda.empty_cache()
    return out


def wide_tree_sweep(torch, tv, W, peaks, Bs=GRID_B, Ns=GRID_N, iters: int = 3) -> dict:
    """The wide-tree sweep on the synthetic 3:1 hybrid stack: 24 GDN layers (H=16, d=128) and 8
    tree-attention layers (16q/4kv, hd 128, prefix 8192), bf16, random dynamic trees (1..4
    children per node, depth <= 8) of N nodes at batch B, fork vs TreeWY."""
    torch.cuda.empty_cache()
    rows = []
    for B in Bs:
        for N in Ns:
            trees = W.sweep_trees(N, B)
            rows.append(hybrid_point(torch, tv, W, peaks, B, N, trees, HYBRID_GDN_LAYERS, HYBRID_ATTN_LAYERS,
                                     HYBRID_PREFIX, seed=10 * N + B, iters=iters))
    return {"workload": "3:1 hybrid stack, 24 GDN layers (H=16, d=128) + 8 tree-attention layers (16q/4kv, hd 128, "
                        "prefix 8192), bf16, random dynamic trees (1..4 children, depth <= 8), inputs drawn on the device",
            "pages_bytes_per_checkpoint": checkpoint_bytes(24, 16, 128, 128, 2),
            "timing": "device time of whole rounds issued behind a device-side sleep, mean of 3",
            "rows": rows}


def small_config_lines(torch, tv, W, peaks) -> dict:
    """Timed lines for the two launch-latency-bound single-sequence workloads: the small fp32
    layer (B=1, H=2, d=64, the 7-node tree) and the single bf16 layer (B=1, H=16, d=128: a chain
    of 5 nodes vs the 15-node k=2 d=3 tree, plus its attention layer, 16q/4kv, hd 128, prefix
    4096), each mode's verify and commit queued behind a device-side sleep."""
    dev = torch.device("cuda", torch.cuda.current_device())
    lines = {}

    def gdn_modes(case):
        x = {k: getattr(case, k).contiguous().to(dev) for k in ("q", "k", "v", "alpha", "beta", "S0", "parents")}
        B, N, H, dk, dv = case.shape
        path, plen = case.path.to(dev), case.path_len.to(dev)
        out = torch.empty((B, N, H, dv), dtype=x["q"].dtype, device=dev)
        st = torch.empty((B, N, H, dv, dk), dtype=x["S0"].dtype, device=dev)
        pv = torch.empty((B, N, H, dv), dtype=torch.float32, device=dev)
        lg = torch.empty((B, N, H), dtype=torch.float32, device=dev)
        err = torch.zeros((4, B), dtype=torch.int32, device=dev)
        S0f, S0w = x["S0"].clone(), x["S0"].clone()

        def fork():
            tv.tv_gdn_tree_verify_fork(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0f, x["parents"], out, st,
                                       err[0], q_scale=case.q_scale)
            tv.tv_gdn_commit(tv.TV_MODE_FORK, path, plen, x["parents"], S0f, err[1], node_states=st)

        def wy():
            tv.tv_gdn_tree_verify_wy(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0w, x["parents"], out, pv, lg,
                                     err[2], q_scale=case.q_scale)
            tv.tv_gdn_commit(tv.TV_MODE_WY, path, plen, x["parents"], S0w, err[3], pseudo_v=pv, log_gamma=lg,
                             k=x["k"])

        r = {}
        for name, fn in (("fork", fork), ("wy", wy)):
            ms = device_timed(torch, fn, 50, 2)
            r[name] = {"verify_commit_ms": round(ms, 5), "nodes_per_s": round(B * N / (ms * 1e-3))}
        assert int(err.abs().sum()) == 0, err
        return r

    lines["small_fp32_layer"] = dict(workload="1 GDN layer, B=1, H=2, d=64, fp32, 7-node k=2 d=2 tree",
                                     bound="launch latency", **gdn_modes(W.small_fp32_case()))
    for tree in ("chain", "tree"):
        case = W.single_layer_gdn_case(tree)
        a = W.single_layer_attn_case(tree)
        B, N, Hq, Hkv, hd = a.shape
        x = {k: getattr(a, k).contiguous().to(dev) for k in
             ("q", "k_new", "v_new", "k_cache", "v_cache", "block_table", "prefix_len", "parents")}
        out = torch.empty((B, N, Hq, hd), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(tv.tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, x["block_table"].shape[1]),
                         dtype=torch.uint8, device=dev)
        err = torch.zeros((B,), dtype=torch.int32, device=dev)
        a_ms = device_timed(torch, lambda: tv.tv_tree_attn(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                                           x["block_table"], x["prefix_len"], x["parents"], out, ws,
                                                           err, rope_theta=1e6), 50, 4)
        assert int(err.abs().sum()) == 0, err
        name = "single_bf16_layer_chain5" if tree == "chain" else "single_bf16_layer_k2d3"
        lines[name] = dict(workload=f"1 GDN layer, B=1, H=16, d=128, bf16, {N}-node "
                                    f"{'chain' if tree == 'chain' else 'k=2 d=3 tree'}; attention 16q/4kv hd 128 "
                                    f"prefix 4096", bound="launch latency", **gdn_modes(case),
                           attention={"ms": round(a_ms, 5), "nodes_per_s": round(N / (a_ms * 1e-3))})
    return lines


def run_ours(args) -> None:
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = OraclePool()                         # spawned before any GPU work
        cpu_base = pool.sample(args.cpu_seconds)
        pool.close()

    import __graft_entry__
    __graft_entry__.build()
    import tree_speculative_verification_gdn_gb300 as tv
    import workloads as W

    rnd = Round(rank, args.layers, torch, tv, W)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        rnd.step()
    barrier()
    assert int(rnd.err.abs().sum()) == 0, f"verify errors: {rnd.err.cpu().tolist()}"

    ev = {r: [] for r in rnd.rows}
    steps_ev = []
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        s = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        rnd.step(ev)
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        steps_ev.append((s, e))
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(dist, t_start.elapsed_time(t_end), "cuda")
    ms_per_step = total_ms / args.steps
    step_ms = sorted(s.elapsed_time(e) for s, e in steps_ev)
    row_ms = {r: sum(s.elapsed_time(e) for s, e, _ in ev[r]) / args.steps for r in rnd.rows}
    row_calls = {r: sum(n for _, _, n in ev[r]) // args.steps for r in rnd.rows}

    # end-to-end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        h2d, d2h = rnd.host_buffers()
        for _ in range(max(2, args.warmup)):
            rnd.step_e2e()
        barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(args.steps):
            rnd.step_e2e()
        e.record(stream)
        barrier()
        rnd.end_e2e()
        e2e_ms = max_over_ranks(dist, s.elapsed_time(e) / args.steps, "cuda")
        e2e = {"value": whole_job_rate(rnd.B * rnd.N * rnd.layers * 2, world, e2e_ms), "unit": "nodes/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "copies": "pinned host memory, per layer on an upload and a download stream overlapping the kernels, "
                         "uploads into two alternating input sets; the step ends after the last download"}

    selective = lazy = one_pass = remap = None
    if not args.no_reports:
        selective = selective_fork_report(rnd, torch, tv)
        lazy = lazy_commit_report(rnd, torch, tv)
        one_pass = one_pass_fork_report(rnd, torch, tv)
        remap = block_table_compaction_report(rnd, torch, tv, W)
    peaks = load_peaks()
    step_peak = torch.cuda.max_memory_allocated()
    B, N, H, dk, dv = rnd.B, rnd.N, rnd.H, rnd.dk, rnd.dv
    L_sum = int(rnd.gdn_host[0].path_len.sum())
    a = rnd.attn_host
    plens = [int(x) for x in a.prefix_len]
    row_bytes = {
        "tree_prepare": B * N * 4 * 3,
        "fork_verify": gdn_bytes(B, N, H, dk, dv, 2, 2, "fork"),
        "fork_materialize": gdn_bytes(B, N, H, dk, dv, 2, 2, "materialize"),
        "fork_commit": gdn_bytes(B, N, H, dk, dv, 2, 2, "commit_fork"),
        "wy_verify": gdn_bytes(B, N, H, dk, dv, 2, 2, "wy"),
        "wy_commit": gdn_bytes(B, N, H, dk, dv, 2, 2, "commit_wy", L_sum),
        "tree_attn": attn_bytes(plens, rnd.aN, rnd.Hq, rnd.Hkv, rnd.hd),
        "kv_compact": compact_bytes([int(x) for x in a.path_len], rnd.Hkv, rnd.hd),
        # per call, the two calls averaged: parents, draft and target tokens in; path, length, next out
        "accept_walk": ((B + rnd.aB) * N * 12 + (B + rnd.aB) * (a.path.shape[1] + 2) * 4) // 2,
    }
    a_flops = attn_flops(plens, [_depths(t) for t in a.trees], rnd.Hq, rnd.hd)
    rows = {}
    for r in rnd.rows:
        per_call_ms = row_ms[r] / max(1, row_calls[r])
        gbs = row_bytes[r] / (per_call_ms * 1e-3) / 1e9 if per_call_ms > 0 else 0.0
        rows[r] = {"ms_per_call": round(per_call_ms, 5), "calls_per_step": row_calls[r],
                   "algorithmic_bytes_per_call": row_bytes[r], "achieved_gbs": round(gbs, 1),
                   "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    rows["tree_attn"]["achieved_tflops"] = round(a_flops / (row_ms["tree_attn"] * 1e-3) / 1e12, 2)
    rows["fork_verify"]["nodes_per_s_per_layer"] = round(B * N / (rows["fork_verify"]["ms_per_call"] * 1e-3))
    rows["wy_verify"]["nodes_per_s_per_layer"] = round(B * N / (rows["wy_verify"]["ms_per_call"] * 1e-3))
    # the dominant kernel: fork_verify spans two kernels on two streams, every other row is one
    dom = max((r for r in rnd.rows if r != "fork_verify"), key=lambda r: row_ms[r])
    roof = {"kernel": dom, "bound": "hbm", "achieved": rows[dom]["achieved_gbs"], "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": rows[dom]["frac_hbm"], "traffic": kernel_traffic(dom),
            "peak_source": peaks["source"] + " (copy, burst)"}
    value = whole_job_rate(B * N * rnd.layers * 2, world, ms_per_step)
    # accepted tokens per round (the device accept walk's path lengths) over the stack's verify
    # and commit time, per mode
    l_sum = int(rnd.path_len.sum())
    stack_ms = {m: rnd.layers * (rows[f"{m}_verify"]["ms_per_call"] + rows[f"{m}_commit"]["ms_per_call"])
                for m in ("fork", "wy")}
    accepted = {"tokens_per_round": l_sum, "batch": B,
                "fork_tokens_per_s": round(l_sum / (stack_ms["fork"] * 1e-3), 1),
                "wy_tokens_per_s": round(l_sum / (stack_ms["wy"] * 1e-3), 1),
                "stack_verify_commit_ms": {m: round(v, 4) for m, v in stack_ms.items()}}
    mem = {"fork_checkpoint_bytes": rnd.fork_state_bytes, "wy_pseudo_value_bytes": rnd.wy_state_bytes,
           "pages_bytes_per_checkpoint": checkpoint_bytes(24, 16, 128, 128, 2),
           "pages_accounting_fork_bytes": checkpoint_bytes(24, 16, 128, 128, 2) * B * N,
           "peak_allocated_bytes": step_peak}
    # The per-mode figures below run on a clean device: the step's buffers are freed first.
    trees_b64 = [list(t) for t in rnd.gdn_host[0].trees]
    fork_rate = rows["fork_verify"]["nodes_per_s_per_layer"]
    wy_rate = rows["wy_verify"]["nodes_per_s_per_layer"]
    layers, aB, launches_per_step = rnd.layers, rnd.aB, rnd.launches_per_step
    del rnd
    import gc
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    per_mode = sweep = small = None
    if not args.no_grid and world == 1:
        # measured peak device memory per mode on the batch-64 GDN stack alone (24 layers, verify +
        # accept walk + stacked commit; the library allocates nothing, so this is every buffer the
        # mode adds to the inputs)
        pm = hybrid_point(torch, tv, W, peaks, B, N, trees_b64, LAYERS, 0, 0, seed=64)
        per_mode = {m: {"peak_bytes_measured": pm[m]["peak_bytes_measured"], "state_bytes": pm[m]["state_bytes"],
                        "gdn_ms_per_layer_alone": pm[m]["gdn_ms_per_layer"]} for m in ("fork", "wy")}
        per_mode["pages_accounting_fork_bytes"] = checkpoint_bytes(24, 16, 128, 128, 2) * B * N
        small = small_config_lines(torch, tv, W, peaks)
        sweep = wide_tree_sweep(torch, tv, W, peaks)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "nodes/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "ms_per_step_min": round(step_ms[0], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": layers, "global_batch": B * world,
                       "nodes_per_tree": N, "attn_batch": aB * world,
                       "l2": "working set >> 129 MB L2 (fork checkpoints 1.3 GB per layer)",
                       "parallelism": f"replicas x{world}"},
            "gpu_launches": launches_per_step * args.steps, "clocks": clk, "roofline": roof,
            "fork_nodes_per_s_per_layer": fork_rate, "wy_nodes_per_s_per_layer": wy_rate,
            "peak_memory_per_mode": per_mode,
            "rows": rows, "accepted_tokens": accepted, "state_memory": mem, "selective_fork": selective,
            "lazy_commit": lazy,
            "one_pass_fork": one_pass, "block_table_compaction": remap, "e2e": e2e,
            "small_workloads": small, "wide_tree_sweep": sweep,
            "cpu_baseline": cpu_base}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args) -> None:
    """The fp64 oracle on the host cores, each step a bounded sample of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    pool = OraclePool()
    seconds = max(2.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        pool.sample(seconds=0.0)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(pool.sample(seconds=seconds))
    dt = time.perf_counter() - t0
    pool.close()
    value = statistics.mean(v["value"] for v in vals)
    base = dict(vals[-1])
    base["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "nodes/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": base["sample"]},
            "cpu_baseline": base,
            "e2e": {"value": round(value, 2), "unit": "nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_sweep(args) -> None:
    """Per-layer GDN verify times across tree sizes: random dynamic trees (1..4 children per
    node, depth <= 8), N in {15, 40, 64, 128, 256}, B in {8, 32}, H=16, d=128, bf16.  Fork mode
    runs its two passes on one stream (tv_gdn_tree_verify_fork_ws), TreeWY one launch.  One
    JSON line, apart from the benchmark's."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import tree_speculative_verification_gdn_gb300 as tv
    import workloads as W
    torch.cuda.set_device(0)
    peaks = load_peaks()
    ev = torch.cuda.Event

    def timed(fn, iters=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        s, e = ev(enable_timing=True), ev(enable_timing=True)
        # queued behind a device-side sleep: the events bracket device time even where a call
        # takes less time on the device than to issue from Python
        torch.cuda._sleep(4_000_000)
        s.record()
        for _ in range(iters):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / iters

    rows = []
    for B in (8, 32):
        for N in (15, 40, 64, 128, 256):
            c = W.sweep_gdn_layer(N, B)
            x = {k: getattr(c, k).contiguous().to("cuda") for k in ("q", "k", "v", "alpha", "beta", "S0", "parents")}
            _, _, H, dk, dv = c.shape
            out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device="cuda")
            pv = torch.empty((B, N, H, dv), dtype=torch.float32, device="cuda")
            lg = torch.empty((B, N, H), dtype=torch.float32, device="cuda")
            states = torch.empty((B, N, H, dv, dk), dtype=torch.bfloat16, device="cuda")
            ws = torch.empty(tv.tv_gdn_fork_workspace_size(B, N, H, dv), dtype=torch.uint8, device="cuda")
            err = torch.zeros((B,), dtype=torch.int32, device="cuda")
            wy_ms = timed(lambda: tv.tv_gdn_tree_verify_wy(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                                           x["parents"], out, pv, lg, err))
            fork_ms = timed(lambda: tv.tv_gdn_tree_verify_fork_ws(x["q"], x["k"], x["v"], x["alpha"], x["beta"],
                                                                  x["S0"], x["parents"], out, states, ws, err))
            assert int(err.abs().sum()) == 0, (N, B, err.tolist())
            fb, wb = gdn_bytes(B, N, H, dk, dv, 2, 2, "fork"), gdn_bytes(B, N, H, dk, dv, 2, 2, "wy")
            rows.append({"B": B, "N": N, "max_depth": max(max(_depths(t)) for t in c.trees),
                         "wy_ms": round(wy_ms, 4), "wy_nodes_per_s": round(B * N / (wy_ms * 1e-3)),
                         "wy_frac_hbm": round(wb / (wy_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                         "fork_ms": round(fork_ms, 4), "fork_nodes_per_s": round(B * N / (fork_ms * 1e-3)),
                         "fork_frac_hbm": round(fb / (fork_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)})
            del states, ws
    print(json.dumps({"sweep": "GDN verify per layer, random dynamic trees, H=16, d=128, bf16", "rows": rows}),
          flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=LAYERS, help="GDN layers per step (24 = the config)")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-reports", action="store_true",
                    help="skip the selective-fork, lazy-commit and one-pass-fork reports after the timed steps")
    ap.add_argument("--no-grid", action="store_true",
                    help="skip the per-mode memory, the small workloads and the wide-tree sweep after the step")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark: per-layer GDN verify times across tree sizes (one JSON line)")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
