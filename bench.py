#!/usr/bin/env python
"""Decode-step benchmark of the compressed KV cache on one GB300.

Workload (the metric's 128K configuration): a Llama-3.1-8B-shaped decode step
-- 32 layers, 32 q / 8 kv heads, head_dim 128, batch 1, a 131072-token prompt
of synthetic fp16 K/V ~ N(0,1) with four outlier K channels (x10) per layer and
kv head, 16-token pages through a shuffled block table.  Layer 0 is 1-bit
quantized (K per channel, V per token, groups of 64); layers 1-31 are sparse:
8 critical channels, top-K with K = floor(0.03 T), 4 sinks + 128 window, exact
attention over the selection.  One step = append one token to every layer +
attention of a fresh random query in every layer, captured in one CUDA graph.

Metric: decode steps/s (higher is better) and achieved HBM GB/s of the step's
algorithmic bytes (packed K/V + scales of layer 0, critical-channel keys,
score writes and selected fp16 rows of layers 1-31).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference]
                  [--prompt T0] [--layers L] [--no-e2e] [--no-cpu-baseline]

For N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the path has no cross-GPU exchange); value = all ranks' steps / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HQ, HKV, D = 32, 8, 128
N_CRIT, N_SINK, WINDOW, RATIO = 8, 4, 128, 0.03
CONFIG_ID = 1
WORKLOAD = "llama31-8b-128k-decode"


# ------------------------------------------------------------------------ helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_bytes(T, n_layers=32):
    """Algorithmic HBM bytes of one decode step at context T (after append):
    layer 0 reads its 1-bit K/V codes and (scale, zero) pairs, 48 B per token
    and kv head; every sparse layer reads the critical-channel keys (8 fp16 per
    token and q head) and the selected fp16 K and V rows (512 B per row)."""
    sel = N_SINK + WINDOW + math.floor(RATIO * T)
    l0 = HKV * T * (16 + 16 + 8 + 8)
    crit = HQ * N_CRIT * T * 2
    rows = HQ * sel * 2 * D * 2
    return l0 + (n_layers - 1) * (crit + rows), crit, rows, l0


class Clocks:
    """Samples nvidia-smi clocks during the timed region (best effort)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc, self.path = None, None
        try:
            out = os.path.join(ROOT, "gpurun_out")
            os.makedirs(out, exist_ok=True)
            self.path = os.path.join(out, f"clocks_bench_{os.getpid()}.csv")
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        load = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------ the GPU workload

class Workload:
    def __init__(self, T0, n_layers, max_steps, device, seed):
        import torch

        from compressed_kv_cache_quant_gb300 import kvq, synth
        self.torch, self.kvq, self.synth = torch, kvq, synth
        self.T0, self.L = T0, n_layers
        self.cap = T0 + max(512, max_steps + 16)
        self.cap = (self.cap + 63) // 64 * 64
        self.n_pages = self.cap // 16
        alloc = kvq.Allocator(self.n_pages, seed=synth.mix(seed, 17) or 1)
        pages = alloc.alloc(self.n_pages)
        bt = torch.tensor([pages], dtype=torch.int32, device=device)
        self.batch = kvq.Batch(bt, torch.tensor([T0], dtype=torch.int32, device=device), self.cap)
        self.layers = []
        for l in range(n_layers):
            if l == 0:
                c = kvq.LayerCache(HQ, HKV, 1, self.n_pages, 1, v_group_dims=64, device=device)
            else:
                c = kvq.LayerCache(HQ, HKV, 16, self.n_pages, 1, t_cap=self.cap, device=device)
            K, V = synth.kv_rows(T0, HKV, synth.mix(seed, 100 + l), device=device)
            kvq.kv_quant_pack(c, self.batch, 0, 0, T0, K, V)
            del K, V
            self.layers.append(c)
        torch.cuda.synchronize()
        self.stride = (self.cap + 7) // 8 * 8
        self.sel_cap = N_SINK + WINDOW + math.floor(RATIO * self.cap)
        self.scores = torch.zeros((1, HQ, self.stride), device=device)
        self.sel = torch.zeros((1, HQ, self.sel_cap), dtype=torch.int32, device=device)
        self.cnt = torch.zeros((1, HQ), dtype=torch.int32, device=device)
        self.in_q = torch.zeros((n_layers, 1, HQ, D), dtype=torch.float16, device=device)
        self.in_k = torch.zeros((n_layers, 1, HKV, D), dtype=torch.float16, device=device)
        self.in_v = torch.zeros((n_layers, 1, HKV, D), dtype=torch.float16, device=device)
        self.out = torch.zeros((n_layers, 1, HQ, D), device=device)
        self.ws_app = kvq.Workspace(kvq.kv_page_append_ws())
        self.ws_q = kvq.Workspace(kvq.kv_decode_attn_quant_ws(self.layers[0], self.batch))
        self.ws_sx = kvq.Workspace(kvq.kv_sparse_layer_decode_ws())
        self.launches_per_step = 1 + 2 + (n_layers - 1)

    def step(self, stream):
        """One decode step: append + attention in every layer.  Layer 0: page
        append and fused dequant attention; sparse layers: the fused append +
        critical score (+ key histogram), then the fused top-K + attention."""
        kvq, b = self.kvq, self.batch
        kvq.kvq_seq_lens_add(b.seq_lens, 1, stream)
        for l, c in enumerate(self.layers):
            if l == 0:
                kvq.kv_page_append(c, b, self.in_k[l], self.in_v[l], self.ws_app, stream)
                kvq.kv_decode_attn_quant(c, b, self.in_q[l], self.out[l], self.ws_q, stream)
            else:
                self.sparse_layer(l, stream)

    def sparse_layer(self, l, stream):
        """Sparse layer: append + critical scores + top-K + attention in one launch."""
        self.kvq.kv_sparse_layer_decode(self.layers[l], self.batch, self.in_k[l], self.in_v[l], self.in_q[l], N_CRIT,
                                        -1, RATIO, N_SINK, WINDOW, self.out[l], self.ws_sx, stream=stream)

    def capture(self, fn, stream):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                fn(stream.cuda_stream)
        return g


def _gen_inputs(torch, synth, n_layers, n_sets, seed, device):
    q = synth.normal((n_sets, n_layers, 1, HQ, D), synth.mix(seed, 1), device)
    k = synth.normal((n_sets, n_layers, 1, HKV, D), synth.mix(seed, 2), device)
    v = synth.normal((n_sets, n_layers, 1, HKV, D), synth.mix(seed, 3), device)
    return q, k, v


# ------------------------------------------------------------------------ CPU oracle baseline

_ATTACHED = {}


def _views(meta):
    """numpy views of the shared-memory arrays described by `meta` (worker side)."""
    import numpy as np
    from multiprocessing import shared_memory
    out = {}
    for name, (shm_name, shape, dt) in meta.items():
        if shm_name not in _ATTACHED:
            _ATTACHED[shm_name] = shared_memory.SharedMemory(name=shm_name)
        out[name] = np.ndarray(shape, dtype=np.dtype(dt), buffer=_ATTACHED[shm_name].buf)
    return out


def _oracle_task(args):
    """One (layer, kv head) of a decode step on the CPU oracle; returns seconds."""
    from oracle import kvq_oracle as O
    kind, g, q, meta = args
    a = _views(meta)
    t = time.perf_counter()
    if kind == "quant":
        n_packed = a["k_codes"].shape[1]
        pk = dict(codes=a["k_codes"][g], scale16=a["k_scale16"][g], zero16=a["k_zero16"][g],
                  tail=a["k_tail"][g], n_packed=n_packed, bits=1, group_tokens=64)
        pv = dict(codes=a["v_codes"][g], scale16=a["v_scale16"][g], zero16=a["v_zero16"][g], bits=1,
                  group_dims=64)
        O.decode_attn_quant(q, [pk], [pv])
    else:
        K, V = a["k1"][g], a["v1"][g]
        k = O.ratio_k(K.shape[0], RATIO)
        for h in range(q.shape[0]):
            C = O.critical_channels(q[h], O.key_absmax(K), N_CRIT)
            s = O.critical_scores(q[h], K, C)
            ids = O.topk_select(s, k, N_SINK, WINDOW)
            O.sparse_attn(q[h], K, V, ids)
    return time.perf_counter() - t


class OracleSample:
    """Layer 0 (packed by the oracle) and one sparse layer of the workload in
    shared memory, so that a process pool runs the oracle without copies."""

    def __init__(self, K0, V0, K1, V1):
        import numpy as np
        from multiprocessing import shared_memory
        from oracle import kvq_oracle as O
        arrs = {"k1": np.ascontiguousarray(K1.transpose(1, 0, 2)), "v1": np.ascontiguousarray(V1.transpose(1, 0, 2))}
        pks = [O.pack_k(K0[:, g], 1) for g in range(HKV)]
        pvs = [O.pack_v(V0[:, g], 1, 64) for g in range(HKV)]
        arrs["k_codes"] = np.stack([p["codes"].astype(np.uint8) for p in pks])
        arrs["k_scale16"] = np.stack([p["scale16"] for p in pks])
        arrs["k_zero16"] = np.stack([p["zero16"] for p in pks])
        arrs["k_tail"] = np.stack([p["tail"] for p in pks])
        arrs["v_codes"] = np.stack([p["codes"].astype(np.uint8) for p in pvs])
        arrs["v_scale16"] = np.stack([p["scale16"] for p in pvs])
        arrs["v_zero16"] = np.stack([p["zero16"] for p in pvs])
        self.shm, self.meta = [], {}
        for name, a in arrs.items():
            m = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=a.dtype, buffer=m.buf)[...] = a
            self.shm.append(m)
            self.meta[name] = (m.name, a.shape, a.dtype.str)

    def step_time(self, pool, q0, q1, n_layers):
        """Oracle time of one decode step: layer 0 and one sparse layer on the
        pool (8 kv-head tasks each), t_step = t0 + (n_layers - 1) * t1."""
        G = HQ // HKV
        t = time.perf_counter()
        pool.map(_oracle_task, [("quant", g, q0[g * G:(g + 1) * G], self.meta) for g in range(HKV)])
        t0 = time.perf_counter() - t
        t = time.perf_counter()
        pool.map(_oracle_task, [("sparse", g, q1[g * G:(g + 1) * G], self.meta) for g in range(HKV)])
        t1 = time.perf_counter() - t
        return t0 + (n_layers - 1) * t1, t0, t1

    def close(self):
        for m in self.shm:
            m.close()
            m.unlink()


def make_pool(n):
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    return mp.get_context("spawn").Pool(n)


# ------------------------------------------------------------------------ main

def traffic_record(kernel):
    """ncu DRAM bytes per launch for `kernel`, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, "compressed_kv_cache_quant_gb300", "csrc", rec["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if h != rec["sha256_16"] or rec.get("prompt") is None:
        return None
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)  # ~0.6 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--prompt", type=int, default=131072)
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-workers", type=int, default=0)
    args = ap.parse_args()
    assert args.warmup >= 1 and args.steps >= 1 and args.layers >= 2

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    n_workers = args.cpu_workers or min(16, os.cpu_count() or 1)

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, n_workers)
        return

    # the oracle's process pool is spawned before the first GPU call
    pool = None
    if rank == 0 and not args.no_cpu_baseline:
        pool = make_pool(n_workers)

    import torch
    import torch.distributed as dist

    from compressed_kv_cache_quant_gb300 import synth
    from compressed_kv_cache_quant_gb300.build import build
    build()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    seed = synth.BASE_SEED + CONFIG_ID
    total_steps = args.warmup + args.steps
    W = Workload(args.prompt, args.layers, 2 * total_steps + 8, device, seed)
    n_sets = min(64, total_steps)
    qs, ks, vs = _gen_inputs(torch, synth, args.layers, n_sets, seed, device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()

    # ---- one eager step (first launches set kernel attributes), then capture one full step
    with torch.cuda.stream(stream):
        W.step(stream.cuda_stream)
    stream.synchronize()
    g_step = W.capture(W.step, stream)

    def feed(i):
        W.in_q.copy_(qs[i % n_sets], non_blocking=True)
        W.in_k.copy_(ks[i % n_sets], non_blocking=True)
        W.in_v.copy_(vs[i % n_sets], non_blocking=True)

    step_i = 0
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            feed(step_i)
            g_step.replay()
            step_i += 1
    stream.synchronize()

    # ---- timed region: K steps, inputs resident in HBM (each step streams > L2)
    clocks = Clocks(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            feed(step_i)
            g_step.replay()
            step_i += 1
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    if world > 1:
        t = torch.tensor([ms], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
        dist.barrier()
    ms_per_step = ms / args.steps
    T_mid = args.prompt + step_i - args.steps // 2
    step_bytes, crit_bytes, rows_bytes, l0_bytes = algorithmic_bytes(T_mid, args.layers)

    # ---- per-kernel durations (CUDA events around graphs of one kernel kind, 31 launches each)
    kern = {}
    g = W.capture(lambda s: [W.sparse_layer(l, s) for l in range(1, args.layers)], stream)
    with torch.cuda.stream(stream):
        g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            g.replay()
        b.record(stream)
    stream.synchronize()
    kern["kv_sparse_layer_decode"] = a.elapsed_time(b) / (args.steps * (args.layers - 1))
    step_i += args.steps + 1   # each replay appended one token to the sparse layers
    del g
    g0 = W.capture(lambda s: W.kvq.kv_decode_attn_quant(W.layers[0], W.batch, W.in_q[0], W.out[0], W.ws_q, s),
                   stream)
    with torch.cuda.stream(stream):
        g0.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            g0.replay()
        b.record(stream)
    stream.synchronize()
    kern["kv_decode_attn_quant"] = a.elapsed_time(b) / args.steps
    peak, peak_src = measured_peaks()
    Tk = args.prompt + step_i
    kb = {"kv_sparse_layer_decode": HQ * N_CRIT * Tk * 2 + HQ * (N_SINK + WINDOW + math.floor(RATIO * Tk)) * 2 * D * 2,
          "kv_decode_attn_quant": HKV * Tk * 48}
    per_kernel = {k: {"ms": kern[k], "GBps": (kb[k] / (kern[k] * 1e-3) / 1e9) if k in kb else None}
                  for k in kern}
    dom = "kv_sparse_layer_decode"
    achieved = kb[dom] / (kern[dom] * 1e-3) / 1e9
    tr = traffic_record(dom)

    # ---- end to end through the C ABI: pinned host inputs in, outputs out, every step
    e2e = None
    if not args.no_e2e:
        hq = qs.cpu().pin_memory()
        hk = ks.cpu().pin_memory()
        hv = vs.cpu().pin_memory()
        hout = torch.empty(W.out.shape, dtype=W.out.dtype).pin_memory()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                j = (step_i + i) % n_sets
                W.in_q.copy_(hq[j], non_blocking=True)
                W.in_k.copy_(hk[j], non_blocking=True)
                W.in_v.copy_(hv[j], non_blocking=True)
                g_step.replay()
                hout.copy_(W.out, non_blocking=True)
        stream.synchronize()
        t_e2e = time.perf_counter() - t0
        step_i += args.steps
        bi = (W.in_q.numel() + W.in_k.numel() + W.in_v.numel()) * 2
        e2e = {"value": world * args.steps / t_e2e, "unit": "steps/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": W.out.numel() * 4}

    # ---- CPU oracle baseline (rank 0, bounded sample of the same workload)
    cpu = None
    if pool is not None:
        K0, V0 = synth.kv_rows(args.prompt, HKV, synth.mix(seed, 100 + 0), device=device)
        K1, V1 = synth.kv_rows(args.prompt, HKV, synth.mix(seed, 100 + 1), device=device)
        sample = OracleSample(K0.cpu().numpy(), V0.cpu().numpy(), K1.cpu().numpy(), V1.cpu().numpy())
        del K0, V0, K1, V1
        t_step, t0c, t1c = sample.step_time(pool, qs[0, 0, 0].cpu().numpy(), qs[0, 1, 0].cpu().numpy(), args.layers)
        sample.close()
        pool.close()
        cpu = {"value": 1.0 / t_step, "unit": "steps/s", "cores": n_workers, "kind": "oracle",
               "sample": f"layer 0 (1-bit quantized) and one sparse layer, 8 kv-head tasks each, of a "
                         f"{args.prompt}-token step on a {n_workers}-process pool; step time = t0 + "
                         f"{args.layers - 1} x t_sparse = {t0c:.2f} s + {args.layers - 1} x {t1c:.2f} s"}

    if rank == 0:
        value = world * args.steps / (ms * 1e-3)
        line = {
            "metric": "decode-attention steps/s (compressed KV, 128K context)",
            "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp16 in / fp32 accumulate (1-bit codes in layer 0)", "data": "synthetic",
            "config": workload_config(args, world),
            "hbm_GBps_step": step_bytes * value / world / 1e9,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": tr["bytes_per_launch_scaled"] if tr else None,
                         "algorithmic_bytes_per_launch": kb[dom]},
            "kernels": per_kernel,
            "e2e": e2e, "gpu_launches": W.launches_per_step * args.steps,
            "clocks": clk, "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def workload_config(args, world):
    """The workload description both arms print."""
    step_bytes = algorithmic_bytes(args.prompt, args.layers)[0]
    return {"workload": WORKLOAD, "layers": args.layers, "q_heads": HQ, "kv_heads": HKV,
            "head_dim": D, "batch": 1, "prompt_tokens": args.prompt, "page_tokens": 16,
            "layer0": "1-bit K per-channel g64, V per-token g64",
            "sparse_layers": f"8 critical channels, top-K floor({RATIO} T), {N_SINK} sinks + {WINDOW} window",
            "l2": f"inputs larger than L2: each step streams {step_bytes / 1e9:.2f} GB",
            "parallelism": f"replicas x{world}", "cuda_graph": "one graph per step"}


def run_reference(args, n_workers):
    """The reference arm: the CPU oracle on the same workload and metric."""
    pool = make_pool(n_workers)
    from compressed_kv_cache_quant_gb300 import synth
    seed = synth.BASE_SEED + CONFIG_ID
    K0, V0 = synth.kv_rows(args.prompt, HKV, synth.mix(seed, 100), device="cpu")
    K1, V1 = synth.kv_rows(args.prompt, HKV, synth.mix(seed, 101), device="cpu")
    # every step is a bounded sample (~0.5 s of oracle work); at most 24 steps are timed so that
    # any --steps finishes within minutes; the metric is 1 / (mean step time)
    n_warm, n_time = min(args.warmup, 2), min(args.steps, 24)
    qs = synth.normal((n_warm + n_time, 2, HQ, D), synth.mix(seed, 1), "cpu")
    sample = OracleSample(K0.numpy(), V0.numpy(), K1.numpy(), V1.numpy())
    del K0, V0, K1, V1
    times = []
    for i in range(n_warm + n_time):
        t_step, _, _ = sample.step_time(pool, qs[i, 0].numpy(), qs[i, 1].numpy(), args.layers)
        if i >= n_warm:
            times.append(t_step)
    sample.close()
    pool.close()
    total = sum(times) * args.steps / n_time  # the K steps at the measured mean step time
    value = args.steps / total
    line = {"impl": "reference", "metric": "decode-attention steps/s (compressed KV, 128K context)",
            "value": value, "unit": "steps/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp64 attention / fp32 quantizer (oracle)", "data": "synthetic",
            "config": workload_config(args, args.gpus),
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": n_workers, "kind": "oracle",
                             "sample": "per step: layer 0 and one sparse layer timed on the process pool, "
                                       f"extrapolated to {args.layers} layers; {n_time} steps timed "
                                       f"after {n_warm} warm-up steps"},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
