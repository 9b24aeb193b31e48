#!/usr/bin/env python
"""Decode layer-step benchmark of the GB300 decode-step library.

One step = one decode layer step of the Llama-3.2-3B-shaped layer over one
batch of rows: QKV GEMV, RoPE + KV store, split-KV attention, merge, O GEMV,
gate/up GEMV, down GEMV (Q8_0 weights, f16 KV mirror, f32 activations).  The
headline workload is 8 rows of one session at positions 5120..5127 over 5120
cached keys; 1 row and 12 independent streams (6 + 6 rows) are measured beside
it.  Eight distinct layers (weights and caches, about 1 GB) are cycled, so the
inputs of consecutive steps are larger than L2.  Steps are replayed from CUDA
graphs and timed with CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica (independent sessions, no data
exchange); the value is all ranks' layer-steps over the slowest rank's time.
`--impl reference` times the CPU oracle on a bounded sample of the same step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode layer-steps/sec and achieved HBM GB/s (% of GB300 peak) at 1/8/12 rows"
UNIT = "layer-steps/s"
FALLBACK_HBM_GBS = 6800.0
L2_CYCLE_BYTES = 260_000_000          # about twice the 129 MB L2: bytes one pass over cycled inputs exceeds


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=8)
    p.add_argument("--repeats", type=int, default=5,
                   help="timed regions of --steps steps each; the line reports the median region")
    p.add_argument("--workload", default="3b-8", choices=["3b-8", "3b-1", "3b-2", "3b-4", "3b-12", "1b-1", "3b-8-32k"])
    p.add_argument("--no-extras", action="store_true", help="skip the 1-row and 12-stream side measurements")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--breakdown", action="store_true",
                   help="only the step breakdown: each launch timed alone and the step without it (3B, 8 and 1 rows)")
    p.add_argument("--side-only", action="store_true",
                   help="only the side measurements (f16-weight GEMV, attention on each KV mirror), a few "
                        "repetitions each: a small program for profilers")
    p.add_argument("--gemv-path", type=int, default=0, choices=[0, 1, 2],
                   help="inner product of the GEMVs: 0 library choice, 1 CUDA cores (<= 2 rows), 2 tensor cores")
    p.add_argument("--attn-path", type=int, default=0, choices=[0, 1, 2],
                   help="inner product of the attention: 0 library choice, 1 CUDA cores, 2 tensor cores")
    p.add_argument("--gemv-chain", type=int, default=0, choices=[0, 1],
                   help="1: the O, gate/up and down projections as the phases of one persistent launch")
    p.add_argument("--cluster-merge", type=int, default=0, choices=[0, 1],
                   help="1: the pieces of a KV head merge inside their thread-block cluster (no merge launch)")
    p.add_argument("--kv", default="f16", choices=["f16", "f32", "q8_0"],
                   help="the KV mirror of the measured step (f16: the path's; q8_0: the block-codec mirror)")
    p.add_argument("--tail-merge", type=int, default=0, choices=[0, 1],
                   help="1: commands of at most 8 queries per KV head merge in the attention launch "
                        "(dl_decode_attn_merged: the last piece of each KV head merges)")
    p.add_argument("--concurrent-commands", type=int, default=1, choices=[0, 1],
                   help="1: the commands of a step (independent sessions) run on streams of their own, "
                        "forked and joined inside the step's graph (twelve streams: two 6-row commands)")
    p.add_argument("--l2-prefetch", type=int, default=0, choices=[0, 1],
                   help="1: each launch asks L2 for the weights or keys of a later kernel while it runs "
                        "(dl_l2_prefetch_next)")
    p.add_argument("--one-launch", type=int, default=0, choices=[0, 1],
                   help="1: each command's whole layer step as one persistent launch (dl_layer_step)")
    p.add_argument("--fused-rope", type=int, default=1, choices=[0, 1],
                   help="1: the rope/store runs inside the attention launch (dl_decode_attn_rope); "
                        "0: separate dl_rope_kv_store and dl_decode_attn launches")
    return p.parse_args()


# ----------------------------------------------------------------------------- workloads

def workload(name):
    import synth
    if name == "3b-8":
        return dict(shape=synth.LLAMA_3B, positions=list(range(5120, 5128)), regions=[0] * 8, n_regions=1,
                    capacity=5128, desc="Llama-3.2-3B-shaped layer step, 8 rows of one session at "
                    "positions 5120-5127 over 5120 cached keys")
    if name == "3b-1":
        return dict(shape=synth.LLAMA_3B, positions=[5120], regions=[0], n_regions=1, capacity=5128,
                    desc="Llama-3.2-3B-shaped layer step, 1 row at position 5120 over 5120 cached keys")
    if name in ("3b-2", "3b-4"):
        n = int(name[3:])
        return dict(shape=synth.LLAMA_3B, positions=list(range(5120, 5120 + n)), regions=[0] * n, n_regions=1,
                    capacity=5128, desc="Llama-3.2-3B-shaped layer step, %d rows of one session at positions "
                    "5120-%d over 5120 cached keys" % (n, 5119 + n))
    if name == "3b-12":
        lens = synth.twelve_stream_lengths(0)
        return dict(shape=synth.LLAMA_3B, positions=lens, regions=list(range(12)), n_regions=12,
                    capacity=max(lens) + 1, desc="Llama-3.2-3B-shaped layer step, 12 one-row streams "
                    "(cache lengths U{512..8192}, seed 0) run as 6+6-row commands")
    if name == "1b-1":
        return dict(shape=synth.LLAMA_1B, positions=[4096], regions=[0], n_regions=1, capacity=4097,
                    desc="Llama-3.2-1B-shaped layer step, 1 row at position 4096 over 4096 cached keys")
    if name == "3b-8-32k":
        return dict(shape=synth.LLAMA_3B, positions=list(range(32760, 32768)), regions=[0] * 8, n_regions=1,
                    capacity=32768, desc="Llama-3.2-3B-shaped layer step, 8 rows at 32760-32767 over "
                    "32760 cached keys")
    raise ValueError(name)


def step_bytes(wl, step, kv="f16", weights_once=False):
    """Algorithmic HBM bytes of one layer step: weights once per command (once per step with
    `weights_once`: commands that run at the same time can share one pass through L2), each
    session's keys once, the new K/V rows (at the mirror's bytes per value), and every call's
    activation rows in and out (f32)."""
    eb = KV_ELEM_BYTES[kv]
    S = wl["shape"]
    D, n_q, n_kv, H, F = S.head_dim, S.n_q, S.n_kv, S.hidden, S.ffn
    w_bytes = sum(no * ni // 32 * 34 for no, ni in S.projections().values())
    total = w_bytes if weights_once else 0
    for c in step.commands:
        n = c.n
        if not weights_once:
            total += w_bytes
        p = c.plan
        keys = 0
        for s in range(p.n_sessions):
            rows = [p.sess_rows[i] for i in range(p.sess_begin[s], p.sess_begin[s + 1])]
            keys += max(c.seqlen_host[r] for r in rows)
        total += int(keys * n_kv * D * 2 * eb)           # K and V read
        total += int(n * n_kv * D * 2 * eb)              # new K and V rows
        qkv = (n_q + 2 * n_kv) * D
        act = n * (H + qkv) + n * (qkv + n_q * D)         # QKV GEMV in/out; rope q in/out, k, v in
        act += n * n_q * D * 2 + n * n_q                  # attention q in, merge out + lse
        act += n * (n_q * D + H)                          # O GEMV
        if F:
            act += n * (H + 2 * F) + n * (F + H)          # gate/up, down
        total += act * 4
    return total


def gu_bytes(wl, rows):
    S = wl["shape"]
    return 2 * S.ffn * S.hidden // 32 * 34 + rows * (S.hidden + 2 * S.ffn) * 4


# ----------------------------------------------------------------------------- peaks, clocks, traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs_sustained", "hbm_gbs"):
            if isinstance(d.get(key), (int, float)) and d[key] > 0:
                return float(d[key]), "measured (%s)" % key
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.rows = []
        self.proc = None
        self.err = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu_index)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.err = str(e)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 9:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.err or not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": self.err or "no samples"}
        sel = [p for (t, p) in self.rows if t0 <= t <= t1] or [p for (_, p) in self.rows]
        sm = [float(p[1]) for p in sel if p[1].replace(".", "", 1).isdigit()]
        mx = [float(p[2]) for p in sel if p[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in sel for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel)}


def traffic_for(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    src = os.path.join(ROOT, "row_decode_step_gb300", "csrc", "gemv_q8.cu")
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for line in open(path):
            parts = line.split("#", 1)[0].split()
            if len(parts) == 3 and parts[0] == kernel_tag and parts[1] == digest:
                return float(parts[2])
    except OSError:
        pass
    return None


# ----------------------------------------------------------------------------- our arm

KV_ELEM_BYTES = {"f16": 2.0, "f32": 4.0, "q8_0": 34 / 32}     # HBM bytes per cached value


def build_layers(wl, L, dev, seed=0, kv="f16"):
    import synth
    import torch
    import row_decode_step_gb300 as dl
    from row_decode_step_gb300.step import LayerWeights
    S = wl["shape"]
    layers, caches = [], []
    for l in range(L):
        packed = {}
        for name, (n_out, n_in) in S.projections().items():
            blocks = synth.q8_0_blocks_from_normal(seed, "%s/L%d/%s" % (S.name, l, name), n_out, n_in, device=dev)
            packed[name] = dl.dl_q8_pack(blocks, n_out, n_in)
            del blocks
        layers.append(LayerWeights(packed["wqkv"], packed["wo"], packed.get("wgu"), packed.get("wdown")))
        shape = (wl["n_regions"], S.n_kv, wl["capacity"], S.head_dim)
        if kv == "q8_0":
            shape = shape[:2] + ((wl["capacity"] + 3) // 4 * 4,) + shape[3:]    # the mirror's capacity rule
            kc, ks = synth.kv_q8_random_planes(seed, "%s/L%d/K" % (S.name, l), *shape, device=dev)
            vc, vs = synth.kv_q8_random_planes(seed, "%s/L%d/V" % (S.name, l), *shape, device=dev)
            caches.append(dl.KVCache.q8(kc, ks, vc, vs))
            continue
        if kv == "f32":
            k = synth.normal_f32(seed, "%s/L%d/K32" % (S.name, l), shape, device=dev)
            v = synth.normal_f32(seed, "%s/L%d/V32" % (S.name, l), shape, device=dev)
        else:
            k = synth.kv_cache_normal(seed, "%s/L%d/K" % (S.name, l), *shape, device=dev)
            v = synth.kv_cache_normal(seed, "%s/L%d/V" % (S.name, l), *shape, device=dev)
        caches.append(dl.KVCache(k, v))
    torch.cuda.synchronize()
    return layers, caches


def measure(wl, L, steps, warmup, dev, rank, world, want_clocks=True, want_e2e=True, paths=(0, 0), fused=False,
            cluster=False, chain=False, prefetch=False, concurrent=False, tail=False, kv="f16", one=False,
            repeats=5):
    import synth
    import torch
    import row_decode_step_gb300 as dl
    from row_decode_step_gb300.step import LayerStep
    S = wl["shape"]
    layers, caches = build_layers(wl, L, dev, kv=kv)
    rope = dl.make_rope(S.rope_theta, S.head_dim, wl["capacity"], device=dev)
    step = LayerStep(wl["positions"], wl["regions"], S.n_q, S.n_kv, S.head_dim, S.hidden, S.ffn, dev,
                     gemv_path=paths[0], attn_path=paths[1], fused_rope=fused, cluster_merge=cluster,
                     gemv_chain=chain, l2_prefetch=prefetch, concurrent=concurrent and not one, tail_merge=tail,
                     one_launch=one)
    for i, c in enumerate(step.commands):
        c.x.copy_(synth.normal_f32(0, "bench/x%d" % i, tuple(c.x.shape), device=dev))
        if c.x_ffn is not None:
            c.x_ffn.copy_(synth.normal_f32(0, "bench/xf%d" % i, tuple(c.x_ffn.shape), device=dev))
            c.h.copy_(synth.normal_f32(0, "bench/h%d" % i, tuple(c.h.shape), device=dev))
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for l in range(L):                      # eager pass: sets kernel attributes, checks the path
            step.run(layers[l], rope, caches[l])
    stream.synchronize()
    # one graph holds the L layer steps back to back (launch gaps overlapped by PDL); K steps
    # replay it K // L times, then single-layer graphs for the remainder
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        for l in range(L):
            step.run(layers[l], rope, caches[l])
    g_one = []
    for l in range(L):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step.run(layers[l], rope, caches[l])
        g_one.append(g)
    torch.cuda.synchronize()

    def replay(n):
        for _ in range(n // L):
            g_all.replay()
        for l in range(n % L):
            g_one[l].replay()

    with torch.cuda.stream(stream):
        replay(max(3, warmup))
    stream.synchronize()

    sampler = ClockSampler(torch.cuda.current_device()).start() if want_clocks else None
    # soak so that the clock sampler sees the GPU under this load before the timed region
    t_soak = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t_soak < 1.0:
            replay(4 * L)
            stream.synchronize()
    # `repeats` timed regions of exactly `steps` layer steps, each bracketed by a barrier and a
    # device synchronisation; the median region is the result
    region_ms = []
    t0 = time.time()
    for _ in range(max(1, repeats)):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            replay(steps)
            e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        region_ms.append(e0.elapsed_time(e1))
    t1 = time.time()
    ms = statistics.median(region_ms)
    clocks = None
    if sampler:
        time.sleep(0.25)
        sampler.stop()
        clocks = sampler.summary(t0 - 0.2, t1 + 0.2)
    status = sum(int(c.status.item()) for c in step.commands)

    # the dominant kernel on its own: the gate/up GEMV of every layer, back to back, timed on its stream
    gu_ms = None
    if S.ffn and not one:
        c0 = step.commands[0]
        g_gu = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_gu, stream=stream):
            for l in range(L):
                dl.dl_gemv_q8(layers[l].wgu, c0.x_ffn, c0.gu, path=paths[0])
        reps = max(4, min(200, steps // L))
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_gu.replay()
            k0 = torch.cuda.Event(enable_timing=True)
            k1 = torch.cuda.Event(enable_timing=True)
            k0.record(stream)
            for _ in range(reps):
                g_gu.replay()
            k1.record(stream)
        torch.cuda.synchronize()
        gu_ms = k0.elapsed_time(k1) / (reps * L)
        del g_gu
    graphs = g_one

    e2e = None
    if want_e2e:
        e2e = measure_e2e(step, graphs, L, max(10, min(steps, 500)), stream, dev)
    return dict(ms_total=ms, ms_per_step=ms / steps, status=status, gu_ms=gu_ms, clocks=clocks, step=step,
                launches_per_step=step.launches, e2e=e2e, region_ms=region_ms)


def measure_f16w(dev, peak, n_out=16384, n_in=3072, mats=4, reps=50):
    """The f16-weight lane on the 3B gate/up shape: `mats` distinct matrices (> L2 together)
    multiplied back to back in one CUDA graph, per row count; bytes = the f16 weights + x + y."""
    import synth
    import torch
    import row_decode_step_gb300 as dl
    stream = torch.cuda.Stream(device=dev)
    Ws = []
    for m in range(mats):
        w = synth.f16_weights_from_normal(0, "bench/f16w/%d" % m, n_out, n_in, device=dev)
        Ws.append(dl.dl_f16w_pack(w))
        del w
    out = {"shape": [n_out, n_in], "matrices_cycled": mats}
    for rows in (1, 8):
        x = synth.normal_f32(0, "bench/f16w/x/%d" % rows, (rows, n_in), device=dev)
        y = torch.empty(rows, n_out, device=dev)
        with torch.cuda.stream(stream):
            for W in Ws:
                dl.dl_gemv_f16w(W, x, y, stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for W in Ws:
                dl.dl_gemv_f16w(W, x, y, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            k0 = torch.cuda.Event(enable_timing=True)
            k1 = torch.cuda.Event(enable_timing=True)
            k0.record(stream)
            for _ in range(reps):
                g.replay()
            k1.record(stream)
        torch.cuda.synchronize()
        ms = k0.elapsed_time(k1) / (reps * mats)
        b = n_out * n_in * 2 + rows * (n_in + n_out) * 4
        out["rows_%d" % rows] = {"launch_us": ms * 1e3, "achieved_gbs": b / (ms / 1e3) / 1e9,
                                 "frac": b / (ms / 1e3) / 1e9 / peak}
        del g
    return out


def measure_attn_mirrors(dev, peak, caches=4, reps=30, path=0):
    """The attention alone (work items + merge) of the 3B shape at 1 and 8 rows on the f16, f32 and
    q8_0 mirrors: `caches` distinct caches (> L2 together) cycled in one CUDA graph; bytes = the
    keys and values read + queries + outputs."""
    import synth
    import torch
    import row_decode_step_gb300 as dl
    S = synth.LLAMA_3B
    cap, D = 5128, S.head_dim
    stream = torch.cuda.Stream(device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for name, dt in (("f16", torch.float16), ("f32", torch.float32), ("q8_0", torch.int8)):
        eb = 4 if dt == torch.float32 else 34 / 32 if dt == torch.int8 else 2    # q8_0: codes + a scale per 32
        # enough distinct caches that one pass over them exceeds L2 about twice
        n_caches = max(caches, -(-L2_CYCLE_BYTES // int(S.n_kv * cap * D * 2 * eb)))
        kvs = []
        for c in range(n_caches):
            if dt == torch.int8:
                kc, ks = synth.kv_q8_random_planes(0, "bench/mir/k%d" % c, 1, S.n_kv, cap, D, device=dev)
                vc, vs = synth.kv_q8_random_planes(0, "bench/mir/v%d" % c, 1, S.n_kv, cap, D, device=dev)
                kvs.append(dl.KVCache.q8(kc, ks, vc, vs))
                continue
            k = synth.normal_f32(0, "bench/mir/k%d" % c, (1, S.n_kv, cap, D), device=dev).to(dt)
            v = synth.normal_f32(0, "bench/mir/v%d" % c, (1, S.n_kv, cap, D), device=dev).to(dt)
            kvs.append(dl.KVCache(k, v))
        for rows in (1, 8):
            seqlen = list(range(5121, 5121 + rows))
            # the f32 mirror's ring holds one CTA per SM at D = 128: half the SMs' worth of pieces
            plan = dl.dl_attn_plan_build(seqlen, S.n_q, S.n_kv, D,
                                         sm_count=sms // 2 if dt == torch.float32 and D == 128 else 0)
            ws = dl.workspace_for(plan, dev)
            q = synth.normal_f32(0, "bench/mir/q%d" % rows, (rows, S.n_q * D), device=dev)
            sl = torch.tensor(seqlen, dtype=torch.int32, device=dev)
            o = torch.empty(rows, S.n_q * D, device=dev)
            lse = torch.empty(rows, S.n_q, device=dev)

            def run():
                for kv in kvs:
                    dl.dl_decode_attn(q, kv, sl, plan, ws, stream=stream, path=path)
                    dl.dl_attn_merge(ws, plan, sl, o, lse, stream=stream)
            with torch.cuda.stream(stream):
                run()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
                k0 = torch.cuda.Event(enable_timing=True)
                k1 = torch.cuda.Event(enable_timing=True)
                k0.record(stream)
                for _ in range(reps):
                    g.replay()
                k1.record(stream)
            torch.cuda.synchronize()
            ms = k0.elapsed_time(k1) / (reps * n_caches)
            b = int(max(seqlen) * S.n_kv * D * 2 * eb) + rows * S.n_q * D * 4 * 2
            out["%s_rows_%d" % (name, rows)] = {"attention_us": ms * 1e3, "achieved_gbs": b / (ms / 1e3) / 1e9,
                                                 "frac": b / (ms / 1e3) / 1e9 / peak, "caches_cycled": n_caches,
                                                 "work_items": plan.n_work}
            del g
        del kvs
        torch.cuda.empty_cache()
    return out


def measure_e2e(step, graphs, L, steps, stream, dev):
    """Same steps through host buffers: per step, the activation rows and positions are copied
    from pinned host memory, the graph runs, and the step's outputs are read back."""
    import torch
    host_in, host_out = [], []
    h2d = d2h = 0
    for c in step.commands:
        ins = [c.x, c.pos, c.seqlen] + ([c.x_ffn, c.h] if c.x_ffn is not None else [])
        outs = [c.y_o] + ([c.y_down] if c.y_down is not None else [])
        hi = [t.detach().cpu().pin_memory() for t in ins]
        ho = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        host_in.append(list(zip(hi, ins)))
        host_out.append(list(zip(outs, ho)))
        h2d += sum(t.numel() * t.element_size() for t in ins)
        d2h += sum(t.numel() * t.element_size() for t in outs)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(steps):
            for pairs in host_in:
                for h, d in pairs:
                    d.copy_(h, non_blocking=True)
            graphs[i % L].replay()
            for pairs in host_out:
                for d, h in pairs:
                    h.copy_(d, non_blocking=True)
            stream.synchronize()
    dt = time.perf_counter() - t0
    return {"value": steps / dt, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps}


def host_info():
    """The host's core count (all of them and those this process may use) and CPU model."""
    import platform
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.split(":", 1)[0].strip() in ("model name", "CPU part"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "usable_cores": cores, "model": model, "machine": platform.machine()}


def oracle_step_inputs(wl):
    """Layer 0 of the workload for the oracle: Q8_0 blocks, caches and activation rows (seeded)."""
    import numpy as np
    import synth
    S = wl["shape"]
    D = S.head_dim
    blocks = {}
    for name, (n_out, n_in) in S.projections().items():
        blocks[name] = synth.q8_0_blocks_from_normal(0, "%s/L0/%s" % (S.name, name), n_out, n_in).numpy()
    k = synth.kv_cache_normal(0, "%s/L0/K" % S.name, wl["n_regions"], S.n_kv, wl["capacity"], D).numpy().view(np.uint16)
    v = synth.kv_cache_normal(0, "%s/L0/V" % S.name, wl["n_regions"], S.n_kv, wl["capacity"], D).numpy().view(np.uint16)
    n = len(wl["positions"])
    x = synth.normal_f32(0, "bench/x0", (n, S.hidden)).numpy()
    xf = synth.normal_f32(0, "bench/xf0", (n, S.hidden)).numpy()
    h = synth.normal_f32(0, "bench/h0", (n, S.ffn)).numpy()
    return blocks, k, v, x, xf, h


def oracle_step_seconds(wl, inp):
    """One full layer step of the workload in the oracle (the caches restored first, untimed)."""
    import numpy as np
    import oracle
    S = wl["shape"]
    blocks, k, v, x, xf, h = inp
    n = len(wl["positions"])
    kc, vc = k.copy(), v.copy()
    t0 = time.perf_counter()
    for g0 in range(0, n, 8):
        sl = slice(g0, min(n, g0 + 8))
        pos = np.array(wl["positions"][sl], np.int32)
        oracle.layer_step(blocks, x[sl], kc, vc, pos, n_q=S.n_q, n_kv=S.n_kv, head_dim=S.head_dim,
                          theta=S.rope_theta, chunk=256, n_splits=-(-int(pos.max() + 1) // 256),
                          regions=np.array(wl["regions"][sl], np.int32), x_ffn=xf[sl], h=h[sl])
    return time.perf_counter() - t0


def cpu_baseline_sample(wl, threads=1, budget_s=12.0, max_reps=5, inp=None):
    """The oracle, as it stands, on full layer steps of the workload on the host's cores: `threads`
    threads over its (row, output) and (row, head) loops (OpenMP), up to `max_reps` steps within
    about `budget_s` seconds."""
    import oracle
    inp = inp if inp is not None else oracle_step_inputs(wl)
    used = oracle.set_threads(threads)
    reps, t_total = 0, 0.0
    while reps < max_reps and (reps == 0 or t_total < budget_s):
        t_total += oracle_step_seconds(wl, inp)
        reps += 1
    oracle.set_threads(1)
    return {"value": reps / t_total, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": "%d full layer step(s) of the workload on layer 0, C oracle (double), %d thread(s)"
                      % (reps, used)}


def cpu_baselines(wl):
    """The oracle on all the host's usable cores (the reported baseline) and on one core."""
    host = host_info()
    inp = oracle_step_inputs(wl)
    allc = cpu_baseline_sample(wl, threads=host["usable_cores"], budget_s=8.0, max_reps=5, inp=inp)
    one = cpu_baseline_sample(wl, threads=1, budget_s=4.0, max_reps=2, inp=inp)
    allc.update({"host_cores": host["usable_cores"], "host": host, "single_thread": one})
    return allc


def combine_ranks(ms_local, steps, world, device):
    """Whole-job time and throughput of `world` replicas that each ran `steps` layer steps.

    The job takes as long as its slowest rank (max over ranks); every rank did the same
    fixed work, so the job's throughput is world * steps over that time.  Returns
    (ms, layer_steps_per_s) on every rank.
    """
    import torch
    ms = float(ms_local)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * steps / (ms / 1e3)


def measure_breakdown(wl, L, dev, reps=50):
    """Where the step's time goes: each launch of the default step form timed alone (its L
    layers back to back in one CUDA graph) and the step timed without it, us per layer."""
    import synth
    import torch
    import row_decode_step_gb300 as dl
    from row_decode_step_gb300.step import LayerStep
    S = wl["shape"]
    layers, caches = build_layers(wl, L, dev)
    rope = dl.make_rope(S.rope_theta, S.head_dim, wl["capacity"], device=dev)
    c = LayerStep(wl["positions"], wl["regions"], S.n_q, S.n_kv, S.head_dim, S.hidden, S.ffn, dev).commands[0]
    c.x.copy_(synth.normal_f32(0, "bench/x0", tuple(c.x.shape), device=dev))
    c.x_ffn.copy_(synth.normal_f32(0, "bench/xf0", tuple(c.x_ffn.shape), device=dev))
    c.h.copy_(synth.normal_f32(0, "bench/h0", tuple(c.h.shape), device=dev))
    launch = {
        "qkv": lambda l: dl.dl_gemv_q8(layers[l].wqkv, c.x, c.qkv),
        "attention+rope": lambda l: dl.dl_decode_attn_rope(c.q, c.k, c.v, c.pos, rope, caches[l], c.seqlen, c.plan,
                                                           c.workspace, status=c.status),
        "merge": lambda l: dl.dl_attn_merge(c.workspace, c.plan, c.seqlen, c.attn, c.lse),
        "o": lambda l: dl.dl_gemv_q8(layers[l].wo, c.attn, c.y_o),
        "gate/up": lambda l: dl.dl_gemv_q8(layers[l].wgu, c.x_ffn, c.gu),
        "down": lambda l: dl.dl_gemv_q8(layers[l].wdown, c.h, c.y_down),
    }
    order = list(launch)
    stream = torch.cuda.Stream(device=dev)

    def timed(names):
        with torch.cuda.stream(stream):
            for l in range(L):
                for n in names:
                    launch[n](l)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                for n in names:
                    launch[n](l)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (reps * L)

    full = timed(order)
    out = {"workload": wl["desc"], "step_us": full, "launches": {}}
    for n in order:
        alone, without = timed([n]), timed([o for o in order if o != n])
        out["launches"][n] = {"alone_us": alone, "step_without_us": without, "share_of_step_us": full - without}
    return out


def run_ours(args):
    import torch
    import row_decode_step_gb300 as dl
    from row_decode_step_gb300 import _build
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(dl.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    dl.lib()
    if args.breakdown:
        if rank == 0:
            for name in ("3b-8", "3b-1"):
                print(json.dumps({"breakdown": measure_breakdown(workload(name), args.layers, dev)}))
        return
    if args.side_only:
        peak, _ = hbm_peak()
        side = {"f16w_gemv": measure_f16w(dev, peak, mats=2, reps=2),
                "attention_kv_mirrors": measure_attn_mirrors(dev, peak, caches=2, reps=2, path=args.attn_path)}
        if rank == 0:
            print(json.dumps({"side_only": True, "side_workloads": side}))
        return

    wl = workload(args.workload)
    res = measure(wl, args.layers, args.steps, args.warmup, dev, rank, world, paths=(args.gemv_path, args.attn_path),
                  fused=bool(args.fused_rope), cluster=bool(args.cluster_merge), chain=bool(args.gemv_chain),
                  prefetch=bool(args.l2_prefetch), concurrent=bool(args.concurrent_commands),
                  tail=bool(args.tail_merge), kv=args.kv, one=bool(args.one_launch), repeats=args.repeats)
    steps = args.steps
    ms, value = combine_ranks(res["ms_total"], steps, world, dev)
    step = res["step"]
    rows = len(wl["positions"])
    sb = step_bytes(wl, step, args.kv)
    peak, peak_src = hbm_peak()
    step_gbs = sb / (ms / steps / 1e3) / 1e9
    gu_avg_ms = res["gu_ms"]
    gu_gbs = gu_bytes(wl, step.commands[0].n) / (gu_avg_ms / 1e3) / 1e9 if gu_avg_ms else None
    extras = {}
    if not args.no_extras and args.workload == "3b-8":
        # the other configurations, each its own line: median of the repeated timed regions
        for name in ("3b-1", "3b-2", "3b-4", "1b-1", "3b-8-32k", "3b-12"):
            w2 = workload(name)
            st2 = max(20, min(args.steps, 2000))
            r2 = measure(w2, args.layers, st2, args.warmup, dev, rank, world,
                         want_clocks=False, want_e2e=False, paths=(args.gemv_path, args.attn_path),
                         fused=bool(args.fused_rope), cluster=bool(args.cluster_merge),
                         chain=bool(args.gemv_chain), prefetch=bool(args.l2_prefetch),
                         concurrent=bool(args.concurrent_commands), tail=bool(args.tail_merge), kv=args.kv,
                         one=bool(args.one_launch), repeats=args.repeats)
            sb2 = step_bytes(w2, r2["step"], args.kv)
            sec = r2["ms_per_step"] / 1e3
            line2 = {"workload": w2["desc"], "rows": len(w2["positions"]), "layer_steps_per_s": 1 / sec,
                     "ms_per_step": r2["ms_per_step"], "tokens_per_s": len(w2["positions"]) / sec,
                     "algorithmic_bytes": sb2, "algorithmic_gbs": sb2 / sec / 1e9, "hbm_frac": sb2 / sec / 1e9 / peak,
                     "commands": [c.n for c in r2["step"].commands], "status": r2["status"],
                     "timed_regions_ms_per_step": [m / st2 for m in r2["region_ms"]], "steps_per_region": st2}
            if len(r2["step"].commands) > 1 and bool(args.concurrent_commands):
                # commands that run at the same time may share the weights' pass through L2: the
                # fraction with the weights counted once is the one to hold against the peak
                sb1 = step_bytes(w2, r2["step"], args.kv, weights_once=True)
                line2.update({"algorithmic_bytes_weights_per_command": sb2, "algorithmic_bytes": sb1,
                              "algorithmic_gbs": sb1 / sec / 1e9, "hbm_frac": sb1 / sec / 1e9 / peak,
                              "hbm_frac_weights_per_command": sb2 / sec / 1e9 / peak})
            extras[name] = line2
            del r2
            torch.cuda.empty_cache()
    if not args.no_extras and args.workload == "3b-8" and args.kv == "f16":
        # the same step over the block-codec (q8_0) mirror: half the key and value bytes
        r2 = measure(wl, args.layers, max(20, min(args.steps, 2000)), args.warmup, dev, rank, world,
                     want_clocks=False, want_e2e=False, paths=(args.gemv_path, args.attn_path),
                     fused=bool(args.fused_rope), prefetch=bool(args.l2_prefetch), kv="q8_0")
        sbq = step_bytes(wl, r2["step"], "q8_0")
        extras["3b-8 q8_0 KV"] = {
            "layer_steps_per_s": 1e3 / r2["ms_per_step"], "ms_per_step": r2["ms_per_step"],
            "algorithmic_bytes": sbq, "algorithmic_gbs": sbq / (r2["ms_per_step"] / 1e3) / 1e9,
            "hbm_frac": sbq / (r2["ms_per_step"] / 1e3) / 1e9 / peak, "status": r2["status"]}
        del r2
        torch.cuda.empty_cache()
    if not args.no_extras and args.workload == "3b-8":
        # the same step with the rope/store as its own launch (the other form of the path)
        r2 = measure(wl, args.layers, max(20, min(args.steps, 2000)), args.warmup, dev, rank, world,
                     want_clocks=False, want_e2e=False, paths=(args.gemv_path, args.attn_path),
                     fused=not args.fused_rope, prefetch=bool(args.l2_prefetch))
        extras["3b-8 rope %s" % ("separate" if args.fused_rope else "in attention")] = {
            "layer_steps_per_s": 1e3 / r2["ms_per_step"], "ms_per_step": r2["ms_per_step"],
            "algorithmic_gbs": sb / (r2["ms_per_step"] / 1e3) / 1e9,
            "hbm_frac": sb / (r2["ms_per_step"] / 1e3) / 1e9 / peak, "status": r2["status"]}
        del r2
        torch.cuda.empty_cache()
        extras["f16w_gemv"] = measure_f16w(dev, peak)
        torch.cuda.empty_cache()
        extras["attention_kv_mirrors"] = measure_attn_mirrors(dev, peak, path=args.attn_path)
        torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baselines(wl)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "timing": {"timed_regions": len(res["region_ms"]), "steps_per_region": steps,
                   "ms_per_step_each": [m / steps for m in res["region_ms"]], "reported": "median region"},
        "operands": "q8_0 weights, f32 activations, f16 KV mirror; f32 accumulation (tensor-core operands f16)",
        "data": "synthetic (seeded N(0,0.02) Q8_0 weights, N(0,1) activations and f16 KV; no trained weights)",
        "config": {"workload": wl["desc"], "rows": rows, "layers_cycled": args.layers,
                   "l2": "inputs larger than L2: %d distinct layers cycled (%.2f GB)" % (
                       args.layers, args.layers * sb / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "commands": [c.n for c in step.commands],
                   "attn_chunk": [c.plan.chunk for c in step.commands],
                   "attn_work_items": [c.plan.n_work for c in step.commands],
                   "gemv_path": args.gemv_path, "attn_path": args.attn_path,
                   "rope_in_attention": bool(args.fused_rope), "merge_in_cluster": bool(args.cluster_merge),
                   "l2_prefetch": bool(args.l2_prefetch), "concurrent_commands": bool(args.concurrent_commands),
                   "tail_merge": bool(args.tail_merge), "kv_mirror": args.kv,
                   "gemv_chain": bool(args.gemv_chain)},
        "tokens_per_s": rows * value,
        "step": {"algorithmic_bytes": sb, "algorithmic_gbs": step_gbs, "hbm_frac": step_gbs / peak,
                 "peak_gbs": peak, "peak_source": peak_src},
        "roofline": {"kernel": "gemv_q8 gate/up projection (16384 x 3072, %d rows), timed back to back "
                               "over the %d layers" % (step.commands[0].n, args.layers),
                     "bound": "hbm", "achieved": gu_gbs, "peak": peak, "unit": "GB/s",
                     "frac": (gu_gbs / peak) if gu_gbs else None,
                     "traffic": traffic_for("gemv_gu_%drows" % step.commands[0].n),
                     "traffic_source": "stored: ncu --set full capture of this kernel (profiles/ncu_traffic.txt), "
                                       "null when gemv_q8.cu changed since",
                     "launch_ms": gu_avg_ms, "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": res["e2e"],
        "gpu_launches": res["launches_per_step"] * steps,
        "gpu_launches_note": "per timed region (%d regions timed)" % len(res["region_ms"]),
        "clocks": res["clocks"],
        "device_status": res["status"],
        "side_workloads": extras,
    }
    print(json.dumps(line))


# ----------------------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args):
    """The oracle as it stands on the host's cores: whole layer steps of the workload, each timed.
    Warm-up and timed steps stop early once they pass a time budget (the line then reports the
    steps it timed)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    wl = workload(args.workload)
    host = host_info()
    inp = oracle_step_inputs(wl)
    used = oracle.set_threads(host["usable_cores"])
    t_w = 0.0
    for _ in range(min(args.warmup, 3)):
        t_w += oracle_step_seconds(wl, inp)
        if t_w > 20.0:
            break
    times = []
    while len(times) < args.steps and (not times or sum(times) < 90.0):
        times.append(oracle_step_seconds(wl, inp))
    oracle.set_threads(1)
    sec = sum(times) / len(times)
    value = 1.0 / sec
    sample = ("%d whole layer steps of the workload on layer 0, each timed; C oracle (double) on %d threads "
              "(OpenMP over (row, output) and (row, head))" % (len(times), used))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": len(times),
        "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": wl["desc"], "rows": len(wl["positions"])},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample,
                         "host_cores": host["usable_cores"], "host": host},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    a = parse_args()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
