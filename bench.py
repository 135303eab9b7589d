#!/usr/bin/env python3
"""Benchmark of the TokenSwift per-step decode hot path on one GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
for every layer, tree verification attention with fused importance
(ts_verify_attention) and the partial-KV top-B refresh (ts_partial_kv_select_gather);
then the penalised sampling + tree acceptance of the step
(ts_penalized_sample_accept) and the KV commit of the accepted path in every
layer (ts_kv_commit_batched).  Every layer has its own K/V buffers, so one step streams
~13 GB (LLaMA3.1-8B shape, 102,400 cached tokens) -- far more than L2.

metric: algorithmic HBM bytes of the step / step time (GB/s), with decode
steps/s beside it.  `--impl reference` times the CPU oracle instead.

Run:  python bench.py [--gpus N --steps K --warmup W --workload NAME]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

# the CPU oracle legs run single-threaded; set before numpy is imported
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import ts_synth as syn  # noqa: E402

METRIC = "verify-attn+KV-select HBM GB/s (% of GB300 peak); decode steps/s @100K ctx"
UNIT = "GB/s"


# ---------------------------------------------------------------------------
# algorithmic bytes (the minimum traffic each call must move)
# ---------------------------------------------------------------------------
def verify_bytes(w: syn.Workload) -> int:
    kv = 2 * 2 * (w.L + w.T) * w.Hkv * w.d          # K and V read once, bf16
    q = 2 * w.T * w.Hq * w.d                         # queries
    out = 4 * w.T * w.Hq * w.d + 4 * w.T * w.Hq      # o + lse, fp32
    imp = 4 * w.L * w.Hkv                            # importance written
    return kv + q + out + imp


def verify_flops(w: syn.Workload) -> int:
    """Contraction work of one call: S = Q K^T and O += P V, 2 flops per
    multiply-add, over the L+T keys of every KV head for its T*G query rows."""
    return 4 * w.T * (w.Hq // w.Hkv) * w.d * (w.L + w.T) * w.Hkv


def select_bytes(w: syn.Workload) -> int:
    imp = 4 * w.L * w.Hkv                            # importance read
    gather = 2 * 2 * 2 * w.N * w.Hkv * w.d           # K,V rows read + written
    idx = 4 * w.N * w.Hkv
    return imp + gather + idx


def sample_bytes(w: syn.Workload) -> int:
    return 4 * w.T * w.V + 4 * w.W + 16 * w.T


def commit_bytes(w: syn.Workload, n_moved: int = 3) -> int:
    # every layer: n_moved accepted rows of K and V read and written
    return w.layers * 2 * 2 * 2 * n_moved * w.Hkv * w.d


def step_bytes(w: syn.Workload) -> int:
    return w.layers * (verify_bytes(w) + select_bytes(w)) + sample_bytes(w) + commit_bytes(w)


# Storage of the V caches: "fp16" (the precision of the P.V product; the
# model's bf16 V rows are rounded once, when appended) or "bf16" (the kernel
# converts every V tile it reads).  Same values either way.
V_CACHE = "fp16"


def v_cache_dtype():
    import torch
    return torch.float16 if V_CACHE == "fp16" else torch.bfloat16


def config_dict(w: syn.Workload, world: int = 1) -> dict:
    """The workload's description, shared by the GPU arm and the oracle arm."""
    sb = step_bytes(w)
    return {"workload": w.name, "layers": w.layers, "Hq": w.Hq, "Hkv": w.Hkv, "v_cache": V_CACHE,
            "d": w.d, "L": w.L, "tree_nodes": w.T, "budget_B": w.B, "sinks": w.S,
            "recent": w.R, "vocab": w.V, "penalty_window": w.W,
            "bytes_per_step": sb,
            "l2": (f"inputs larger than L2 (distinct K/V per layer, {sb / 1e9:.1f} GB per step)"
                   if sb > 129e6 else "inputs fit in L2 (parity-size case)"),
            "parallelism": f"replicas x{world}"}


# ---------------------------------------------------------------------------
# measured peaks and profile-derived traffic
# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_tensor_peak():
    """Dense bf16 TFLOP/s for a kernel inside a long step (the sustained
    figure), measured when available."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    return 1700.0, "fallback (sustained)"


def code_of(src: str) -> str:
    """C++/CUDA source without comments and with whitespace runs collapsed:
    what the compiler sees, so that a comment edit keeps the hash."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif src[i] == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return " ".join("".join(out).split())


def verify_source_sha1() -> str:
    """Hash of the verification kernels' code (comments and layout ignored)."""
    h = hashlib.sha1()
    for name in ("verify_tc.cu", "tc_ptx.cuh", "verify_attn.cu", "ts_common.cuh"):
        with open(os.path.join(ROOT, "self_speculative_ultra_gb300", "csrc", name)) as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:12]


def profiled_traffic(workload: str):
    """dram bytes per verify launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", f"verify_attention_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"traffic_bytes_per_call:\s*([0-9.eE+]+)\s+source_sha1:\s*([0-9a-f]+)", txt)
    if not m or m.group(2) != verify_source_sha1():
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Step:
    """Device-resident state of one benchmark replica and its step()."""

    def __init__(self, w: syn.Workload, device, seed: int = 0, e2e: bool = True):
        import torch
        import self_speculative_ultra_gb300 as ts
        self.ts, self.torch, self.w = ts, torch, w
        dev = self.dev = device
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        T, Hq, Hkv, d, L = w.T, w.Hq, w.Hkv, w.d, w.L
        L_cap = L + T
        self.L, self.L_cap = L, L_cap
        tree = syn.make_tree(w, np.random.default_rng(seed))
        self.parents = torch.from_numpy(tree[0]).to(dev)
        self.tokens = torch.from_numpy(tree[1]).to(dev)
        self.q, self.k, self.v = [], [], []
        n_pl = w.planted
        for layer in range(w.layers):
            q = torch.randn((T, Hq, d), generator=g, device=dev, dtype=torch.float32)
            k = torch.randn((Hkv, L_cap, d), generator=g, device=dev, dtype=torch.float32)
            v = torch.randn((Hkv, L_cap, d), generator=g, device=dev, dtype=torch.float32)
            # heavy hitters: keys aligned with the group's summed importance queries
            G = w.G
            qs = q[T - w.n_imp:].reshape(w.n_imp, Hkv, G, d).sum(dim=(0, 2))
            qhat = qs / qs.norm(dim=-1, keepdim=True)
            pos = torch.randint(w.S, L - w.R, (Hkv, n_pl), generator=g, device=dev)
            xi = torch.randn((Hkv, n_pl, d), generator=g, device=dev)
            xi = xi / xi.norm(dim=-1, keepdim=True)
            kk = 0.9 * qhat[:, None, :] + 0.1 * xi
            kk = (d ** 0.5) * kk / kk.norm(dim=-1, keepdim=True)
            k.scatter_(1, pos[..., None].expand(-1, -1, d), kk)
            self.q.append(q.to(torch.bfloat16))
            self.k.append(k.to(torch.bfloat16))
            self.v.append(v.to(torch.bfloat16).to(v_cache_dtype()))
            del q, k, v
        N = w.N
        self.imp = [torch.empty((Hkv, L), dtype=torch.float32, device=dev) for _ in range(w.layers)]
        self.o = [torch.empty((T, Hq, d), dtype=torch.float32, device=dev) for _ in range(w.layers)]
        self.lse = [torch.empty((T, Hq), dtype=torch.float32, device=dev) for _ in range(w.layers)]
        self.idx = [torch.empty((Hkv, N), dtype=torch.int32, device=dev) for _ in range(w.layers)]
        self.kd = [torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=dev) for _ in range(w.layers)]
        self.vd = [torch.empty((Hkv, N, d), dtype=v_cache_dtype(), device=dev) for _ in range(w.layers)]
        sin = syn.sampling_inputs(w, step=0, tree=tree)
        self.logits = torch.from_numpy(sin["logits"]).to(dev)
        self.prior = torch.from_numpy(sin["prior"]).to(dev)
        self.uniforms = torch.from_numpy(sin["uniforms"]).to(dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.sampled = torch.empty(T, **i32)
        # path | n_path | bonus in one buffer, so the per-step readback is one copy
        self.result = torch.empty(T + 2, **i32)
        self.path, self.n_path, self.bonus = (self.result[:T], self.result[T:T + 1],
                                              self.result[T + 1:T + 2])
        self.status = torch.zeros(1, **i32)
        u8 = dict(dtype=torch.uint8, device=dev)
        self.ws_v = torch.empty(max(ts.ts_verify_workspace_bytes(T, Hq, Hkv, d, L), 256), **u8)
        self.ws_s = torch.empty(max(ts.ts_select_batched_workspace_bytes(w.layers, Hkv, L), 256), **u8)
        self.sel_table = ts.layer_pointer_table(self.imp, self.k, self.v, self.idx, self.kd, self.vd)
        self.commit_table = ts.commit_pointer_table(self.k, self.v)
        self.ws_p = torch.empty(max(ts.ts_sample_workspace_bytes(T, w.V), 256), **u8)
        self.v_events = None
        if e2e:
            self._init_e2e()
        torch.cuda.synchronize()

    def _init_e2e(self):
        torch, w, dev = self.torch, self.w, self.dev
        T, Hq, Hkv, d, L = w.T, w.Hq, w.Hkv, w.d, self.L
        # end-to-end leg: the per-step inputs live in one pinned host buffer,
        # uploaded with a single copy into one of two device staging buffers.
        # The step reads queries, logits, tree, window and uniforms in place
        # there; only the tree's K/V rows move, into every layer's cache, by
        # one batched append.
        nl = w.layers
        spec = [("q", (nl, T, Hq, d), torch.bfloat16), ("k_rows", (nl, Hkv, T, d), torch.bfloat16),
                ("v_rows", (nl, Hkv, T, d), torch.bfloat16), ("logits", (T, w.V), torch.float32),
                ("parents", (T,), torch.int32), ("tokens", (T,), torch.int32),
                ("prior", tuple(self.prior.shape), torch.int32), ("uniforms", (T,), torch.float32)]
        offs, off = {}, 0
        for name, shape, dt in spec:
            offs[name] = off
            off += (int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size() + 255) // 256 * 256
        self.h_stage = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.d_stage = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.staged = [torch.cuda.Event() for _ in range(2)]
        self.consumed = [torch.cuda.Event() for _ in range(2)]

        def views(buf):
            out = {}
            for name, shape, dt in spec:
                n = int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size()
                out[name] = buf[offs[name]:offs[name] + n].view(dt).view(shape)
            return out
        self.stage_views = [views(b) for b in self.d_stage]
        hv = views(self.h_stage)
        hv["q"].copy_(torch.stack(self.q).cpu())
        hv["k_rows"].copy_(torch.stack([x[:, L:L + T] for x in self.k]).cpu())
        hv["v_rows"].copy_(torch.stack([x[:, L:L + T] for x in self.v]).cpu())
        for name in ("logits", "parents", "tokens", "prior", "uniforms"):
            hv[name].copy_(getattr(self, name).cpu())
        self.h_bytes = sum(int(np.prod(sh)) * torch.empty(0, dtype=dt).element_size()
                           for _, sh, dt in spec)
        self.h_out = torch.empty(T + 2, dtype=torch.int32).pin_memory()

    def h2d_bytes(self) -> int:
        return self.h_bytes

    def d2h_bytes(self) -> int:
        return self.h_out.numel() * 4

    def stage_inputs(self, s: int, after=None):
        """Upload step s's inputs from pinned host memory into staging
        buffer s % 2 on the copy stream (after `after`, and after the step
        that last read that buffer)."""
        torch, b = self.torch, s % 2
        with torch.cuda.stream(self.copy_stream):
            if after is not None:
                self.copy_stream.wait_event(after)
            if s >= 2:
                self.copy_stream.wait_event(self.consumed[b])
            self.d_stage[b].copy_(self.h_stage, non_blocking=True)
            self.staged[b].record(self.copy_stream)

    def unpack_inputs(self, s: int):
        """Wait for step s's upload and append its tree K/V rows to every
        layer's cache; returns the step's input views."""
        b = s % 2
        self.torch.cuda.current_stream().wait_event(self.staged[b])
        v = self.stage_views[b]
        self.ts.ts_kv_append_batched(self.k, self.v, v["k_rows"], v["v_rows"], self.L,
                                     table=self.commit_table, status=self.status)
        return v

    def release_inputs(self, s: int):
        self.consumed[s % 2].record()

    def upload_inputs(self, s: int = 0):
        self.stage_inputs(s)
        return self.unpack_inputs(s)

    def download_result(self):
        self.h_out.copy_(self.result, non_blocking=True)

    def step(self, events=None, inp=None):
        """One pass of the hot path.  `inp` holds the step's inputs (q per
        layer, logits, parents, tokens, prior, uniforms); default: the
        resident copies."""
        ts, w = self.ts, self.w
        if inp is None:
            q, logits, parents, tokens, prior, uniforms = (self.q, self.logits, self.parents,
                                                           self.tokens, self.prior, self.uniforms)
        else:
            q, logits, parents, tokens, prior, uniforms = (inp["q"], inp["logits"], inp["parents"],
                                                           inp["tokens"], inp["prior"],
                                                           inp["uniforms"])
        if events is not None:
            events[0].record()
        for layer in range(w.layers):
            ts.ts_verify_attention(q[layer], self.k[layer], self.v[layer], self.L, parents,
                                   n_imp=w.n_imp, o=self.o[layer], lse=self.lse[layer],
                                   imp=self.imp[layer], workspace=self.ws_v, status=self.status)
        if events is not None:
            events[1].record()
        # partial-cache refresh of every layer in one batched pipeline (read by
        # the next step's drafting only)
        ts.ts_partial_kv_select_gather_batched(self.imp, self.k, self.v, self.L, w.B, w.S, w.R,
                                               self.idx, self.kd, self.vd, table=self.sel_table,
                                               workspace=self.ws_s, status=self.status)
        ts.ts_penalized_sample_accept(logits, tokens, parents, prior, w.W,
                                      w.penalty, w.temperature, w.top_p, w.min_p, uniforms,
                                      sampled=self.sampled, path=self.path, n_path=self.n_path,
                                      bonus=self.bonus, workspace=self.ws_p, status=self.status)
        ts.ts_kv_commit_batched(self.k, self.v, self.L, w.T, self.path, self.n_path,
                                table=self.commit_table, status=self.status)

    def capture(self, n_ev: int = 3, e2e: bool = False):
        """CUDA graphs of the step (the step's launches replay without host
        issue cost): the resident-input step; n_ev copies that also record an
        event pair around the step's block of verify calls (event record
        nodes); and, for the end-to-end leg, one step per staging buffer."""
        torch, w = self.torch, self.w
        self.step()                       # first calls set kernel attributes
        torch.cuda.synchronize()
        w = self.w

        def cap(fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            return g
        self.g_main = cap(self.step)
        self.ev, self.g_ev = [], []
        for _ in range(n_ev):
            e = [timing_event(external=True) for _ in range(2)]
            if e[0] is None:
                break
            self.g_ev.append(cap(lambda e=e: self.step(events=e)))
            self.ev.append(e)
        if not self.g_ev:
            # event record nodes unavailable: a graph of the verify calls alone
            self.g_ver = cap(self.verify_only)
        if e2e:
            self.g_in = [cap(lambda b=b: self.step(inp=self.stage_views[b])) for b in range(2)]
        torch.cuda.synchronize()

    def verify_only(self):
        w = self.w
        for layer in range(w.layers):
            self.ts.ts_verify_attention(self.q[layer], self.k[layer], self.v[layer], self.L,
                                        self.parents, n_imp=w.n_imp, o=self.o[layer],
                                        lse=self.lse[layer], imp=self.imp[layer],
                                        workspace=self.ws_v, status=self.status)

    def launches_per_step(self) -> int:
        # verify: split kernel + merge per layer; batched select: histogram,
        # collect, gather; sample; commit
        return self.w.layers * 2 + 3 + 2


def timing_event(external: bool = False):
    """A timing CUDA event; with external=True one that stream capture turns
    into an event record node (None where this torch cannot)."""
    import torch
    if not external:
        return torch.cuda.Event(enable_timing=True)
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


def time_steps(st: Step, steps: int, warmup: int, barrier=None, clocks=None):
    """Device time of `steps` hot-path steps (graph replays) after `warmup`
    untimed ones, CUDA events on the launching stream; the last len(st.g_ev)
    timed steps also carry an event pair around their block of verify calls.
    Returns (ms per step, list of mean verify-call ms per event-carrying step,
    clock record)."""
    torch, w = st.torch, st.w
    sync = barrier or torch.cuda.synchronize
    for _ in range(warmup):
        st.g_main.replay()
    sync()
    n_ev = min(len(st.g_ev), steps)
    if clocks is not None:
        clocks.start()
    t0, t1 = timing_event(), timing_event()
    sync()
    t0.record()
    for s_ in range(steps):
        k_ev = s_ - (steps - n_ev)
        (st.g_ev[k_ev] if k_ev >= 0 else st.g_main).replay()
    t1.record()
    sync()
    clk = clocks.stop() if clocks is not None else None
    ms_step = t0.elapsed_time(t1) / steps
    if n_ev:
        # per step: the block of verify calls (programmatic overlap between
        # calls intact) / layers
        ver_ms = [e[0].elapsed_time(e[1]) / w.layers for e in st.ev[:n_ev]]
    else:
        # one replay of the verify calls alone, timed around the graph
        v0, v1 = timing_event(), timing_event()
        v0.record()
        st.g_ver.replay()
        v1.record()
        torch.cuda.synchronize()
        ver_ms = [v0.elapsed_time(v1) / w.layers]
    return ms_step, ver_ms, clk


def per_config_line(w: syn.Workload, ms_step: float, ver_ms, peak: float, tf_peak: float,
                    steps: int) -> dict:
    v_ms = statistics.mean(ver_ms)
    gbs = step_bytes(w) / (ms_step * 1e-3) / 1e9
    vgbs = verify_bytes(w) / (v_ms * 1e-3) / 1e9
    return {"ms_per_step": round(ms_step, 4), "steps_per_s": round(1e3 / ms_step, 2),
            "GB_per_s": round(gbs, 1), "hbm_frac": round(gbs / peak, 4),
            "bytes_per_step": step_bytes(w), "verify_avg_call_ms": round(v_ms, 4),
            "verify_GB_per_s": round(vgbs, 1), "verify_hbm_frac": round(vgbs / peak, 4),
            "verify_tensor_frac": round(verify_flops(w) / (v_ms * 1e-3) / 1e12 / tf_peak, 4),
            "timed_steps": steps}


def measure_other_configs(dev, skip: str, steps: int, warmup: int, peak: float,
                          tf_peak: float) -> dict:
    """Every other workload of the suite, one after the other, each with its
    own device-resident inputs (freed before the next)."""
    import torch
    out = {}
    for name in ("tiny", "qwen2.5-1.5b", "llama3.1-8b", "mha-7b", "qwen2.5-14b"):
        if name == skip:
            continue
        w = syn.WORKLOADS[name]
        st = Step(w, dev, seed=0, e2e=False)
        st.capture()
        ms_step, ver_ms, _ = time_steps(st, steps, warmup)
        line = per_config_line(w, ms_step, ver_ms, peak, tf_peak, steps)
        line["device_status"] = int(st.status.item())
        out[name] = line
        del st
        torch.cuda.empty_cache()
    return out


def run_gpu(args, w: syn.Workload):
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import self_speculative_ultra_gb300 as ts
    ts.build()
    st = Step(w, dev, seed=rank)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # the step is replayed from CUDA graphs; the device-timed region has its
    # inputs resident in HBM.  Per-call verify events are recorded in the last
    # three timed steps only: an event between two programmatic-dependent
    # launches holds the next one back.
    st.capture(n_ev=3, e2e=True)
    clocks = ClockSampler(local)
    ms_step, ver_ms, clk = time_steps(st, args.steps, args.warmup, barrier=barrier, clocks=clocks)
    ms = torch.tensor([ms_step], device=dev)
    if world > 1:
        dist.all_reduce(ms, op=dist.ReduceOp.MAX)
    ms_step = float(ms.item())

    # end-to-end leg: pinned host inputs in, result out, every step
    for i in range(2):
        st.upload_inputs(i)
        st.g_in[i].replay()
        st.release_inputs(i)
        st.download_result()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # per-step phase events on the compute stream: unpack | step | readback
    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    e0.record()
    st.stage_inputs(0, after=e0)
    for s_ in range(args.steps):
        if s_ + 1 < args.steps:
            st.stage_inputs(s_ + 1)
        ph[s_][0].record()
        st.unpack_inputs(s_)
        ph[s_][1].record()
        st.g_in[s_ % 2].replay()
        st.release_inputs(s_)
        ph[s_][2].record()
        st.download_result()
        ph[s_][3].record()
    e1.record()
    barrier()
    e2e_ms = torch.tensor([e0.elapsed_time(e1) / args.steps], device=dev)
    phase_ms = [sum(ph[i][k].elapsed_time(ph[i][k + 1]) for i in range(args.steps)) / args.steps
                for k in range(3)]
    if world > 1:
        dist.all_reduce(e2e_ms, op=dist.ReduceOp.MAX)
    e2e_ms = float(e2e_ms.item())
    status = int(st.status.item())

    if rank == 0:
        peak, peak_kind = load_peaks()
        sb = step_bytes(w)
        value = world * sb / (ms_step * 1e-3) / 1e9
        vb = verify_bytes(w)
        v_avg_ms = statistics.mean(ver_ms)
        achieved = vb / (v_avg_ms * 1e-3) / 1e9
        tf_peak, tf_kind = load_tensor_peak()
        tf_achieved = verify_flops(w) / (v_avg_ms * 1e-3) / 1e12
        traffic = profiled_traffic(w.name)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 K/V with planted heavy hitters, "
                    "N(0,9) fp32 logits)",
            "config": config_dict(w, world),
            "steps_per_s": round(world / (ms_step * 1e-3), 2),
            "pct_of_hbm_peak": round(100 * value / world / peak, 2),
            "roofline": {"bound": "hbm", "kernel": "ts_verify_attention (split + merge)",
                         "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_source": peak_kind,
                         "bytes_per_call": vb, "avg_call_ms": round(v_avg_ms, 4),
                         "tensor": {"achieved": round(tf_achieved, 1), "peak": tf_peak,
                                    "unit": "TFLOP/s", "frac": round(tf_achieved / tf_peak, 4),
                                    "flops_per_call": verify_flops(w), "peak_source": tf_kind}},
            "e2e": {"value": round(world * sb / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                    "h2d_bytes_per_step": st.h2d_bytes(), "d2h_bytes_per_step": st.d2h_bytes(),
                    "ms_per_step": round(e2e_ms, 4),
                    "phase_ms": {"unpack": round(phase_ms[0], 4), "step": round(phase_ms[1], 4),
                                 "readback": round(phase_ms[2], 4)}},
            "gpu_launches": st.launches_per_step() * args.steps,
            "clocks": clk,
            "device_status": status,
        }
        per = {w.name: per_config_line(w, ms_step, ver_ms, peak, tf_peak, args.steps)}
        if world == 1 and not args.no_per_config:
            del st
            torch.cuda.empty_cache()
            per.update(measure_other_configs(dev, w.name, max(20, min(args.steps, 50)),
                                             max(3, args.warmup), peak, tf_peak))
        line["per_config"] = per
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------
def _oracle_layer_unit(w: syn.Workload, heads: int, sample_nodes: int, seed: int = 0,
                       barrier=None):
    """Time the oracle on `heads` KV heads of one layer (verify + select +
    gather) and `sample_nodes` tree nodes of the sampling step.  The inputs
    are generated first; with a barrier, every worker starts timing together.
    Returns (start, end) perf_counter stamps and the algorithmic bytes
    processed."""
    from oracle import ts_oracle as orc
    sub = syn.scaled(w, Hkv=heads, Hq=heads * w.G)
    inp = syn.attention_inputs(sub, layer=seed)
    sin = syn.sampling_inputs(w, step=seed)
    q, k, v = (orc.bf16_to_f64(inp[n]) for n in ("q", "k", "v"))
    if barrier is not None:
        barrier.wait()
    t = time.perf_counter()
    _, _, imp = orc.verify_attention(q, k, v, sub.L, inp["parents"], sub.n_imp)
    for h in range(heads):
        idx = orc.select_partial(imp[h].astype(np.float32), sub.L, sub.B, sub.S, sub.R)
        orc.gather_rows(inp["k"][h], idx)
        orc.gather_rows(inp["v"][h], idx)
    paths = orc.root_paths(sin["parents"])
    for i in range(sample_nodes):
        drafted = [int(sin["tokens"][a]) for a in paths[i][1:]]
        orc.sample_node(sin["logits"][i], sin["prior"], drafted, w.W, w.penalty, w.temperature,
                        w.top_p, w.min_p, float(sin["uniforms"][i]))
    t1 = time.perf_counter()
    nbytes = verify_bytes(sub) + select_bytes(sub) + sample_nodes * 4 * w.V
    return t, t1, nbytes


_POOL_BARRIER = None


def _pool_init(barrier):
    global _POOL_BARRIER
    _POOL_BARRIER = barrier


def _pool_unit(args):
    name, heads, nodes, seed = args
    return _oracle_layer_unit(syn.WORKLOADS[name], heads, nodes, seed, _POOL_BARRIER)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """One oracle worker process per host core (spawned: no state is
    inherited from a process that already used the GPU).  A round gives
    every worker one unit -- one KV head of one layer, verify + select +
    gather, plus `nodes` node draws -- started together behind a barrier;
    its throughput is the units' algorithmic bytes over the round's wall
    time (first start to last end)."""

    def __init__(self, cores: int):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.cores = cores
        self.barrier = ctx.Barrier(cores)
        self.pool = ctx.Pool(cores, initializer=_pool_init, initargs=(self.barrier,))

    def round(self, w: syn.Workload, nodes: int, seed0: int):
        units = [(w.name, 1, nodes, seed0 + i) for i in range(self.cores)]
        res = self.pool.map(_pool_unit, units, chunksize=1)
        wall = max(r[1] for r in res) - min(r[0] for r in res)
        return wall, sum(r[2] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(w: syn.Workload):
    """The oracle as it stands, on the host cores: two rounds of the pool
    (each: one KV head of one layer per core plus 2 node draws each), and one
    such unit on one core for the single-thread figure."""
    cores = host_cores()
    t0, t1, b1 = _oracle_layer_unit(w, heads=1, sample_nodes=2, seed=0)
    single = b1 / (t1 - t0) / 1e9
    pool = OraclePool(cores)
    try:
        wall, nbytes = 0.0, 0
        for r in range(2):
            s_, b_ = pool.round(w, 2, seed0=r * cores)
            wall += s_
            nbytes += b_
    finally:
        pool.close()
    return {"value": round(nbytes / wall / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"fp64 numpy oracle, {cores} processes (one per host core), two rounds "
                      f"of one unit each: verify+select+gather of 1 of {w.Hkv} KV heads of one "
                      f"layer + 2 of {w.T} node draws ({nbytes / 1e6:.1f} MB of algorithmic "
                      f"traffic in {wall:.2f} s wall)",
            "single_thread": {"value": round(single, 4), "unit": UNIT, "cores": 1,
                              "sample": f"one such unit on one core ({b1 / 1e6:.1f} MB in "
                                        f"{t1 - t0:.2f} s)"}}


def run_reference(args, w: syn.Workload):
    """The oracle arm: each step is one round of the oracle pool over the
    host cores (a bounded sample of the workload: one KV head of one layer
    per core plus 2 node draws each), timed by the host clock."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    cores = host_cores()
    pool = OraclePool(cores)
    try:
        for i in range(args.warmup):
            pool.round(w, 2, seed0=1000 + i * cores)
        tot_s, tot_b = 0.0, 0
        for i in range(args.steps):
            s, b = pool.round(w, 2, seed0=i * cores)
            tot_s += s
            tot_b += b
    finally:
        pool.close()
    value = tot_b / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / max(args.steps, 1), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 K/V with planted heavy hitters, N(0,9) fp32 "
                "logits)",
        "config": config_dict(w, world),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: {cores} processes (one per host core), each "
                                   f"verify+select+gather of 1 of {w.Hkv} KV heads of one layer "
                                   f"+ 2 node draws, fp64 numpy"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_case(kind: str, w: syn.Workload):
    """Small, fixed cases for ncu captures (a few GB on the device):
    verify -- 2 layers of the workload's K/V, 3 + 5*2 ts_verify_attention calls
    (split kernel and merge);
    select -- 4 layers through the batched partial-KV refresh and the sampling
    step, 3 rounds;
    imp -- 2 layers of K, 3 + 2*2 ts_importance_softmax calls;
    commit -- 4 layers: 3 rounds of the batched append and commit;
    eta -- 5 eta-sampling calls;
    reject, ngram, draft, refresh -- the timing modes of those calls with
    3 timed and 1 warm-up call, draft on 2 layers and refresh on 4."""
    import torch
    import self_speculative_ultra_gb300 as ts
    ts.build()
    if kind == "reject":
        return run_reject_case(w, 3, 1)
    if kind == "ngram":
        return run_ngram_case(w, 3, 1)
    if kind == "draft":
        return run_draft_case(syn.scaled(w, layers=2), 3, 1)
    if kind == "refresh":
        return run_refresh_case(syn.scaled(w, layers=4), 3, 1)
    if kind == "eta":
        sin = syn.sampling_inputs(w)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        args = (t(sin["logits"]), t(sin["tokens"]), t(sin["parents"]), t(sin["prior"]), w.W,
                w.penalty, w.temperature, 0.0009, 0.03, t(sin["uniforms"]))
        for _ in range(5):
            ts.ts_penalized_sample_accept_eta(*args)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": kind, "workload": w.name}))
        return
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    T, Hq, Hkv, d, L = w.T, w.Hq, w.Hkv, w.d, w.L
    nl = 4 if kind in ("select", "commit") else 2
    ks = [torch.randn((Hkv, L + T, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(nl)]
    if kind == "imp":
        q = torch.randn((T, Hq, d), generator=g, device=dev).to(torch.bfloat16)
        lse = torch.full((T, Hq), 12.0, dtype=torch.float32, device=dev)
        for i in range(3 + 2 * nl):
            ts.ts_importance_softmax(q, ks[i % nl], L, lse, n_imp=w.n_imp)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": kind, "workload": w.name, "layers": nl}))
        return
    vs = [torch.randn((Hkv, L + T, d), generator=g, device=dev).to(torch.bfloat16).to(v_cache_dtype())
          for _ in range(nl)]
    tree = syn.make_tree(w, np.random.default_rng(0))
    parents = torch.from_numpy(tree[0]).to(dev)
    if kind == "commit":
        table = ts.commit_pointer_table(ks, vs)
        rows = [torch.randn((nl, Hkv, T, d), generator=g, device=dev).to(torch.bfloat16)
                for _ in range(2)]
        path = torch.tensor([0, 1, 2, 3] + [0] * (T - 4), dtype=torch.int32, device=dev)
        n_path = torch.tensor([4], dtype=torch.int32, device=dev)
        for _ in range(3):
            ts.ts_kv_append_batched(ks, vs, rows[0], rows[1], L, table=table)
            ts.ts_kv_commit_batched(ks, vs, L, T, path, n_path, table=table)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": kind, "workload": w.name, "layers": nl}))
        return
    if kind == "verify":
        q = torch.randn((T, Hq, d), generator=g, device=dev).to(torch.bfloat16)
        ws = torch.empty(ts.ts_verify_workspace_bytes(T, Hq, Hkv, d, L), dtype=torch.uint8, device=dev)
        for i in range(3 + 5 * nl):
            ts.ts_verify_attention(q, ks[i % nl], vs[i % nl], L, parents, n_imp=w.n_imp, workspace=ws)
    else:
        imps = [torch.randn((Hkv, L), generator=g, device=dev) * 16 for _ in range(nl)]
        N = w.N
        idx = [torch.empty((Hkv, N), dtype=torch.int32, device=dev) for _ in range(nl)]
        kd = [torch.empty((Hkv, N, d), dtype=torch.bfloat16, device=dev) for _ in range(nl)]
        vd = [torch.empty((Hkv, N, d), dtype=v_cache_dtype(), device=dev) for _ in range(nl)]
        sin = syn.sampling_inputs(w, tree=tree)
        logits = torch.from_numpy(sin["logits"]).to(dev)
        toks = torch.from_numpy(sin["tokens"]).to(dev)
        prior = torch.from_numpy(sin["prior"]).to(dev)
        u = torch.from_numpy(sin["uniforms"]).to(dev)
        for _ in range(3):
            ts.ts_partial_kv_select_gather_batched(imps, ks, vs, L, w.B, w.S, w.R, idx, kd, vd)
            ts.ts_penalized_sample_accept(logits, toks, parents, prior, w.W, w.penalty,
                                          w.temperature, w.top_p, w.min_p, u)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": kind, "workload": w.name, "layers": nl}))


def run_draft_case(w: syn.Workload, steps: int, warmup: int):
    """Draft-side attention over the compact cache (the partial-cache half of a
    step): ts_verify_attention with a 4-token draft chain over the S+B+R
    gathered rows plus the draft rows, one call per layer, distinct buffers
    per layer (inputs larger than L2).  Prints one JSON line."""
    import torch
    import self_speculative_ultra_gb300 as ts
    ts.build()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    T_d, Hq, Hkv, d = 4, w.Hq, w.Hkv, w.d
    N = min(w.L, w.S + w.B + w.R)
    layers = w.layers
    ks = [torch.randn((Hkv, N + T_d, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(layers)]
    vs = [torch.randn((Hkv, N + T_d, d), generator=g, device=dev).to(torch.bfloat16).to(v_cache_dtype())
          for _ in range(layers)]
    q = torch.randn((T_d, Hq, d), generator=g, device=dev).to(torch.bfloat16)
    par = torch.tensor([-1] + list(range(T_d - 1)), dtype=torch.int32, device=dev)
    ws = torch.empty(ts.ts_verify_workspace_bytes(T_d, Hq, Hkv, d, N), dtype=torch.uint8, device=dev)
    o = torch.empty((T_d, Hq, d), device=dev)
    lse = torch.empty((T_d, Hq), device=dev)
    def one_pass():
        for i in range(layers):
            ts.ts_verify_attention(q, ks[i], vs[i], N, par, n_imp=T_d, o=o, lse=lse,
                                   want_imp=False, workspace=ws)
    for _ in range(warmup):
        one_pass()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one_pass()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (steps * layers)
    nbytes = 2 * Hkv * (N + T_d) * d * 2 + T_d * Hq * d * 2 + T_d * Hq * (d + 1) * 4
    peak, peak_src = load_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    print(json.dumps({"metric": "draft attention over the compact cache (GB/s)", "value": round(gbs, 1),
                      "unit": "GB/s", "us_per_call": round(us, 2), "calls": steps * layers,
                      "config": {"workload": w.name, "draft_tokens": T_d, "compact_rows": N,
                                 "Hq": Hq, "Hkv": Hkv, "d": d, "bytes_per_call": nbytes,
                                 "l2": f"{layers} distinct per-layer caches, {layers * 2 * Hkv * (N + T_d) * d * 2 / 1e6:.0f} MB"},
                      "frac_of_peak": round(gbs / peak, 3), "peak_source": peak_src}))


def run_imp_softmax_case(w: syn.Workload, steps: int, warmup: int):
    """Softmax-weighted importance pass (ts_importance_softmax) at the
    workload's full cache length: one call per layer over distinct per-layer
    K caches (inputs larger than L2), timed with CUDA events.  Algorithmic
    bytes per call: K rows [0, L) once + imp written + q and lse read.
    Prints one JSON line."""
    import torch
    import self_speculative_ultra_gb300 as ts
    ts.build()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    T, Hq, Hkv, d, L, layers = w.T, w.Hq, w.Hkv, w.d, w.L, w.layers
    n_imp = w.n_imp if w.n_imp > 0 else T
    ks = [torch.empty((Hkv, L + T, d), dtype=torch.bfloat16, device=dev).normal_(generator=g)
          for _ in range(layers)]
    q = torch.randn((T, Hq, d), generator=g, device=dev).to(torch.bfloat16)
    lse = torch.full((T, Hq), 12.0, dtype=torch.float32, device=dev)
    imp = torch.empty((Hkv, L), dtype=torch.float32, device=dev)

    def one_pass():
        for i in range(layers):
            ts.ts_importance_softmax(q, ks[i], L, lse, n_imp=n_imp, imp=imp)
    for _ in range(max(warmup, 3)):
        one_pass()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one_pass()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (steps * layers)
    nbytes = Hkv * L * d * 2 + Hkv * L * 4 + T * Hq * d * 2 + T * Hq * 4
    flops = 2 * n_imp * (Hq // Hkv) * d * L * Hkv
    peak, peak_src = load_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    print(json.dumps({"metric": "softmax-weighted importance pass (GB/s)", "value": round(gbs, 1),
                      "unit": "GB/s", "us_per_call": round(us, 2), "calls": steps * layers,
                      "tflops": round(flops / (us * 1e-6) / 1e12, 1),
                      "frac_of_peak": round(gbs / peak, 3), "peak_source": peak_src,
                      "config": {"workload": w.name, "L": L, "Hq": Hq, "Hkv": Hkv, "d": d,
                                 "importance_rows": n_imp * (Hq // Hkv), "bytes_per_call": nbytes,
                                 "l2": f"{layers} distinct per-layer K caches, "
                                       f"{layers * Hkv * (L + T) * d * 2 / 1e9:.1f} GB"}}))


def run_refresh_case(w: syn.Workload, steps: int, warmup: int, drift: float = 0.3):
    """Partial-cache refresh of all layers per step, full rewrite
    (ts_partial_kv_select_gather_batched) against the incremental update
    (ts_partial_kv_refresh_incremental_batched), on the same sequence of
    importance rows: a fixed per-layer base score ~ N(0, 4^2) plus fresh
    N(0, drift^2) noise each step (importance that drifts between steps), the
    cache growing by 2 tokens per step.  Each call is timed with CUDA events;
    drawing the importance is outside the timed region.  Prints one JSON
    line."""
    import torch
    import self_speculative_ultra_gb300 as ts
    ts.build()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    Hkv, d, nl, B, S, R = w.Hkv, w.d, w.layers, w.B, w.S, w.R
    n_all = max(warmup, 3) + steps
    L0 = w.L - 2 * n_all
    L_cap = w.L + w.T
    N_cap = S + B + R
    ks = [torch.empty((Hkv, L_cap, d), dtype=torch.bfloat16, device=dev).normal_(generator=g)
          for _ in range(nl)]
    vs = [torch.empty((Hkv, L_cap, d), dtype=torch.bfloat16, device=dev).normal_(generator=g)
          .to(v_cache_dtype()) for _ in range(nl)]
    base = [torch.randn((Hkv, w.L), generator=g, device=dev) * 4.0 for _ in range(nl)]
    imp_buf = [torch.empty(Hkv * w.L, device=dev) for _ in range(nl)]
    mk = lambda shape, dt: [torch.empty(shape, dtype=dt, device=dev) for _ in range(nl)]  # noqa: E731
    f_idx, f_kd, f_vd = mk((Hkv, N_cap), torch.int32), mk((Hkv, N_cap, d), torch.bfloat16), \
        mk((Hkv, N_cap, d), v_cache_dtype())
    i_idx, i_kd, i_vd = mk((Hkv, N_cap), torch.int32), mk((Hkv, N_cap, d), torch.bfloat16), \
        mk((Hkv, N_cap, d), v_cache_dtype())
    ws_f = torch.empty(ts.ts_select_batched_workspace_bytes(nl, Hkv, w.L), dtype=torch.uint8,
                       device=dev)
    ws_i = torch.empty(ts.ts_refresh_workspace_bytes(nl, Hkv, w.L, N_cap), dtype=torch.uint8,
                       device=dev)
    written = torch.zeros(nl * Hkv, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_all)]
    w_sum, N_prev = 0, 0
    for s_ in range(n_all):
        L = L0 + 2 * s_
        imps = [x[:Hkv * L].view(Hkv, L) for x in imp_buf]
        for x, b_ in zip(imps, base):
            torch.randn((Hkv, L), generator=g, device=dev, out=x)
            x.mul_(drift).add_(b_[:, :L])
        ev[s_][0].record()
        ts.ts_partial_kv_select_gather_batched(imps, ks, vs, L, B, S, R, f_idx, f_kd, f_vd,
                                               workspace=ws_f, status=status)
        ev[s_][1].record()
        N_prev = ts.ts_partial_kv_refresh_incremental_batched(
            imps, ks, vs, L, B, S, R, i_idx, i_kd, i_vd, N_prev, n_written=written,
            workspace=ws_i, status=status)
        ev[s_][2].record()
        if s_ >= n_all - steps:
            w_sum += int(written.sum().item())
    torch.cuda.synchronize()
    timed = range(n_all - steps, n_all)
    full_us = sum(ev[i][0].elapsed_time(ev[i][1]) for i in timed) * 1e3 / steps
    inc_us = sum(ev[i][1].elapsed_time(ev[i][2]) for i in timed) * 1e3 / steps
    rows_full = nl * Hkv * N_cap
    print(json.dumps({
        "metric": "partial-cache refresh of all layers per step (us)", "unit": "us",
        "full_rewrite_us": round(full_us, 1), "incremental_us": round(inc_us, 1),
        "speedup": round(full_us / inc_us, 3),
        "rows_written_frac": round(w_sum / (steps * rows_full), 4),
        "device_status": int(status.item()), "steps": steps,
        "config": {"workload": w.name, "layers": nl, "Hkv": Hkv, "L": w.L, "B": B, "S": S, "R": R,
                   "importance": f"fixed base N(0,16) + N(0,{drift}^2) per step",
                   "growth": "2 tokens per step"}}))


def run_reject_case(w: syn.Workload, steps: int, warmup: int):
    """Rejection-sampling acceptance (ts_rejection_sample_accept) on the
    workload's tree, logits and penalty settings, with a draft distribution
    per node correlated with the target (softmax of half the logits plus
    N(0,1) noise).  Device time per call with CUDA events.  Prints one JSON
    line."""
    import torch
    import self_speculative_ultra_gb300 as ts
    ts.build()
    dev = torch.device("cuda", 0)
    inp = syn.sampling_inputs(w, step=0)
    rng = np.random.default_rng(0)
    z = 0.5 * inp["logits"].astype(np.float64) + rng.standard_normal(inp["logits"].shape)
    q = np.exp(z - z.max(axis=1, keepdims=True))
    q = (q / q.sum(axis=1, keepdims=True)).astype(np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    logits, qd, toks, par, prior = t(inp["logits"]), t(q), t(inp["tokens"]), t(inp["parents"]), \
        t(inp["prior"])
    ua, ud = t(syn.node_uniforms(w.seed, 0, w.T)), t(syn.node_uniforms(w.seed, 7919, w.T))
    ws = torch.empty(ts.ts_reject_workspace_bytes(w.V), dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    path, n_path, bonus = torch.empty(w.T, **i32), torch.empty(1, **i32), torch.empty(1, **i32)

    def call():
        ts.ts_rejection_sample_accept(logits, qd, toks, par, prior, w.W, w.penalty, w.temperature,
                                      w.top_p, w.min_p, ua, ud, path=path, n_path=n_path,
                                      bonus=bonus, workspace=ws)
    for _ in range(max(warmup, 3)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    n = int(n_path.item())
    print(json.dumps({"metric": "rejection-sampling acceptance per step (us)", "value": round(us, 1),
                      "unit": "us", "higher_is_better": False, "calls": steps,
                      "accepted_path_nodes": n,
                      "config": {"workload": w.name, "tree_nodes": w.T, "V": w.V,
                                 "top_p": w.top_p, "min_p": w.min_p, "penalty_window": w.W}}))


def run_ngram_case(w: syn.Workload, steps: int, warmup: int):
    """Token reutilization per decode step: insert the 4-grams of the newly
    committed tokens (4 per step), then build the next draft tree (heads'
    [1,3,3,3] tree + up to k=20 retrieved 4-gram continuations, T <= 64),
    on a table prefilled from an 8K-token synthetic history.  Prints one
    JSON line with the device time per step."""
    import torch
    import self_speculative_ultra_gb300 as ts
    ts.build()
    dev = torch.device("cuda", 0)
    V, cap, k, T_max = w.V, 64, 20, min(64, w.T)
    rng = np.random.default_rng(0)
    # a Zipf-like token stream: frequent tokens repeat, as in text
    n_hist = 8192 + 4 * (steps + warmup)
    toks = np.minimum(rng.zipf(1.2, size=n_hist), V) - 1
    hist = torch.from_numpy(toks.astype(np.int32)).to(dev)
    table = ts.ngram_table(V, cap)
    e_pre0, e_pre1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_pre0.record()
    ts.ts_ngram_insert(table, V, cap, hist, 0, n_tokens=8192)
    e_pre1.record()
    heads = torch.from_numpy(rng.integers(0, V, size=(3, 3)).astype(np.int32)).to(dev)
    keys = [torch.from_numpy(syn.ngram_rand_keys(1, s_, cap)).to(dev) for s_ in range(steps + warmup)]
    par = torch.empty(T_max, dtype=torch.int32, device=dev)
    tok = torch.empty(T_max, dtype=torch.int32, device=dev)
    nn = torch.empty(1, dtype=torch.int32, device=dev)
    n = 8192

    def step(i, n):
        ts.ts_ngram_insert(table, V, cap, hist, n, n_tokens=n + 4)
        ts.ts_ngram_build_tree(table, V, cap, hist[n + 3:n + 4], heads, k, keys[i], T_max,
                               parents=par, tokens=tok, n_nodes=nn)
        return n + 4
    for i in range(warmup):
        n = step(i, n)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(warmup, warmup + steps):
        n = step(i, n)
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"metric": "token reutilization per decode step (us)",
                      "value": round(e0.elapsed_time(e1) * 1e3 / steps, 2), "unit": "us",
                      "higher_is_better": False, "steps": steps,
                      "prefill_8192_tokens_us": round(e_pre0.elapsed_time(e_pre1) * 1e3, 1),
                      "mean_tree_nodes": int(nn.item()),
                      "config": {"workload": w.name, "V": V, "cap": cap, "k": k, "T_max": T_max,
                                 "new_tokens_per_step": 4}}))


def run_loop_case(w: syn.Workload, until: int, L0: int = 2048):
    """A whole generation loop on synthetic tokens: from a prefix of L0
    cached tokens until the cache holds `until` tokens.  Every step draws the
    draft tree's fresh N(0,1) K/V rows, appends them to every layer's cache
    (one batched launch), verifies
    every layer (importance on), refreshes every layer's partial cache,
    draws fresh N(0, 3^2) logits in which each node's first child's token is
    raised by 30 with probability 0.7 (about 2.5 committed tokens per step),
    samples and accepts, commits the accepted rows in every layer and
    advances by the accepted length, which is read back to the host each
    step.  Prints one JSON line."""
    import torch
    import self_speculative_ultra_gb300 as ts
    ts.build()
    lib, P = ts.lib(), ts._ptr
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    T, Hq, Hkv, d, V, nl = w.T, w.Hq, w.Hkv, w.d, w.V, w.layers
    L_cap = until + T
    bf = dict(dtype=torch.bfloat16, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    ks = [torch.empty((Hkv, L_cap, d), **bf).normal_(generator=g) for _ in range(nl)]
    vs = [torch.empty((Hkv, L_cap, d), **bf).normal_(generator=g).to(v_cache_dtype())
          for _ in range(nl)]
    qs = [torch.empty((T, Hq, d), **bf).normal_(generator=g) for _ in range(nl)]
    # fresh N(0,1) tree K/V rows every step, drawn on the device and written
    # into every layer's cache by one batched append
    tree_kv_f32 = torch.empty((2, nl, Hkv, T, d), dtype=torch.float32, device=dev)
    tree_kv = torch.empty((2, nl, Hkv, T, d), **bf)
    parents_np, tokens_np = syn.make_tree(w, np.random.default_rng(w.seed))
    parents = torch.from_numpy(np.asarray(parents_np, np.int32)).to(dev)
    tokens = torch.from_numpy(np.asarray(tokens_np, np.int32)).to(dev)
    first_child = np.full(T, -1, dtype=np.int64)
    for i in range(T - 1, 0, -1):
        first_child[parents_np[i]] = i
    has_fc = torch.from_numpy(first_child >= 0).to(dev)
    fc_tok = torch.from_numpy(np.asarray(tokens_np, np.int64)[np.maximum(first_child, 0)]).to(dev)
    rows = torch.arange(T, device=dev)
    prior_np = np.random.default_rng(w.seed + 1).integers(0, V, size=w.W).astype(np.int32)
    prior_np[-1] = tokens_np[0]
    prior = torch.from_numpy(prior_np).to(dev)
    logits = torch.empty((T, V), dtype=torch.float32, device=dev)
    uniforms = torch.empty(T, dtype=torch.float32, device=dev)
    o = [torch.empty((T, Hq, d), dtype=torch.float32, device=dev) for _ in range(nl)]
    lse = [torch.empty((T, Hq), dtype=torch.float32, device=dev) for _ in range(nl)]
    imp = [torch.empty(Hkv * until, dtype=torch.float32, device=dev) for _ in range(nl)]
    N = w.S + w.B + w.R
    idx = [torch.empty((Hkv, N), **i32) for _ in range(nl)]
    kd = [torch.empty((Hkv, N, d), **bf) for _ in range(nl)]
    vd = [torch.empty((Hkv, N, d), dtype=v_cache_dtype(), device=dev) for _ in range(nl)]
    vflag = 1 if V_CACHE == "fp16" else 0     # TS_VERIFY_V_FP16 / TS_KV_V_FP16
    u8 = dict(dtype=torch.uint8, device=dev)
    ws_v = torch.empty(max(ts.ts_verify_workspace_bytes(T, Hq, Hkv, d, Lx)
                           for Lx in range(L0, until + 256, 256)), **u8)
    ws_s = torch.empty(max(ts.ts_select_batched_workspace_bytes(nl, Hkv, Lx)
                           for Lx in range(L0, until + 256, 256)), **u8)
    ws_p = torch.empty(ts.ts_sample_workspace_bytes(T, V), **u8)
    sampled, path, n_path, bonus = (torch.empty(T, **i32), torch.empty(T, **i32),
                                    torch.empty(1, **i32), torch.empty(1, **i32))
    status = torch.zeros(1, **i32)
    n_path_h = torch.empty(1, dtype=torch.int32).pin_memory()
    table = ts.layer_pointer_table(imp, ks, vs, idx, kd, vd)
    trow = [ctypes.c_void_p(table[r].data_ptr()) for r in range(6)]
    ctable = ts.commit_pointer_table(ks, vs)
    crow = [ctypes.c_void_p(ctable[r].data_ptr()) for r in range(2)]
    stream = ts._stream(None)
    n_out = ctypes.c_int64(0)
    lay = [(P(qs[i]), P(ks[i]), P(vs[i]), P(o[i]), P(lse[i]), P(imp[i])) for i in range(nl)]
    nb_v, nb_s, nb_p = ws_v.numel(), ws_s.numel(), ws_p.numel()
    torch.cuda.synchronize()

    t_issue = [0.0]

    def step(s_, L):
        t_s = time.perf_counter()
        torch.randn(tree_kv_f32.shape, generator=g, device=dev, out=tree_kv_f32)
        tree_kv.copy_(tree_kv_f32)
        ts._check(lib.ts_kv_append_batched_flags(nl, crow[0], crow[1], P(tree_kv[0]),
                                                 P(tree_kv[1]), L, L_cap, Hkv, d, T, vflag,
                                                 P(status), stream))
        torch.randn((T, V), generator=g, device=dev, out=logits)
        logits.mul_(3.0)
        plant = (torch.rand(T, generator=g, device=dev) < 0.7) & has_fc
        logits.index_put_((rows, fc_tok), plant.float() * 30.0, accumulate=True)
        torch.rand(T, generator=g, device=dev, out=uniforms)
        for (q_, k_, v_, o_, lse_, imp_) in lay:
            ts._check(lib.ts_verify_attention_flags(q_, k_, v_, L, L_cap, P(parents), T, Hq, Hkv,
                                                    d, w.n_imp, o_, lse_, imp_, P(ws_v), nb_v,
                                                    vflag, P(status), stream))
        ts._check(lib.ts_partial_kv_select_gather_batched(
            nl, trow[0], trow[1], trow[2], L, L_cap, Hkv, d, w.B, w.S, w.R, trow[3], trow[4],
            trow[5], ctypes.byref(n_out), P(ws_s), nb_s, P(status), stream))
        ts._check(lib.ts_penalized_sample_accept(
            P(logits), P(tokens), P(parents), T, P(prior), prior.numel(), w.W, V, w.penalty,
            w.temperature, w.top_p, w.min_p, P(uniforms), P(sampled), P(path), P(n_path),
            P(bonus), P(ws_p), nb_p, P(status), stream))
        ts._check(lib.ts_kv_commit_batched(nl, crow[0], crow[1], L, L_cap, Hkv, d, T, P(path),
                                           P(n_path), P(status), stream))
        n_path_h.copy_(n_path, non_blocking=True)
        t_issue[0] += time.perf_counter() - t_s
        torch.cuda.current_stream().synchronize()
        return int(n_path_h.item())

    for s_ in range(3):                     # warm-up at the prefix length
        step(s_, L0)
    torch.cuda.synchronize()
    L, steps, committed, hist = L0, 0, 0, [0] * (T + 1)
    t_issue[0] = 0.0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    while L < until:
        n = step(steps, L)
        if not 1 <= n <= T:
            raise RuntimeError(f"accepted length {n} at L={L} (device status "
                               f"{int(status.item())})")
        hist[n] += 1
        L += n
        committed += n
        steps += 1
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    print(json.dumps({
        "metric": "generation loop wall time", "value": round(wall, 3), "unit": "s",
        "higher_is_better": False, "steps": steps, "tokens_committed": committed,
        "tokens_per_s": round(committed / wall, 1),
        "mean_accepted_per_step": round(committed / max(steps, 1), 4),
        "accepted_length_histogram": {str(i): c for i, c in enumerate(hist) if c},
        "ms_per_step": round(1e3 * wall / max(steps, 1), 4),
        "host_issue_ms_per_step": round(1e3 * t_issue[0] / max(steps, 1), 4),
        "device_status": int(status.item()), "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "layers": nl, "Hq": Hq, "Hkv": Hkv, "d": d,
                   "prefix_L0": L0, "until_L": until, "tree_nodes": T, "B": w.B, "S": w.S,
                   "R": w.R, "V": V, "acceptance": "first child's token +30 with p=0.7",
                   "per_step": f"{nl} verify + 1 batched select/gather over {nl} layers + "
                               f"1 sample/accept + 1 batched commit over {nl} layers"}}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--workload", default="llama3.1-8b", choices=sorted(syn.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the timing of the other workloads")
    ap.add_argument("--profile", choices=["verify", "select", "imp", "commit", "eta", "reject",
                                          "ngram", "draft", "refresh"],
                    help="run a small fixed case for ncu captures and exit")
    ap.add_argument("--draft", action="store_true",
                    help="time draft-side attention over the compact cache and exit")
    ap.add_argument("--loop", type=int, default=0, metavar="L_END",
                    help="time a whole generation loop from a 2048-token prefix to L_END "
                         "cached tokens and exit")
    ap.add_argument("--imp-softmax", action="store_true",
                    help="time the softmax-weighted importance pass and exit")
    ap.add_argument("--refresh", action="store_true",
                    help="time the full against the incremental partial-cache refresh and exit")
    ap.add_argument("--reject", action="store_true",
                    help="time the rejection-sampling acceptance and exit")
    ap.add_argument("--ngram", action="store_true",
                    help="time the token-reutilization step (4-gram table + tree) and exit")
    ap.add_argument("--v-cache", default="fp16", choices=["fp16", "bf16"],
                    help="storage of the V caches (same values; fp16 skips the per-tile "
                         "conversion in the verification kernel)")
    args = ap.parse_args()
    global V_CACHE
    V_CACHE = args.v_cache
    w = syn.WORKLOADS[args.workload]
    if args.reject:
        run_reject_case(w, args.steps, args.warmup)
    elif args.refresh:
        run_refresh_case(w, args.steps, args.warmup)
    elif args.imp_softmax:
        run_imp_softmax_case(w, args.steps, args.warmup)
    elif args.loop:
        run_loop_case(w, args.loop)
    elif args.draft:
        run_draft_case(w, args.steps, args.warmup)
    elif args.ngram:
        run_ngram_case(w, args.steps, args.warmup)
    elif args.profile:
        run_profile_case(args.profile, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
