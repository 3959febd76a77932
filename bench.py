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
                  [--prompt T0] [--layers L] [--no-e2e] [--no-cpu-baseline] [--no-rows]
  python bench.py --rows [--only NAME...]   # the other rows alone

After the decode step, the same line carries under "rows" the other rows of
the hot path, each timed on its own configuration with its own clock samples:
the 40-layer 1-bit prefill pack (GB/s), the INT4 serving batch (steps/s), the
H2O eviction run (steps/s), the offload gather pipeline (host-link GB/s and
overlap fraction), block pruning, and the tiny-configuration kernels.

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
import tempfile
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


def measured_tensor_peak():
    """Dense bf16 TFLOP/s (burst) of this GPU: the measured figure, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


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
            out = os.environ.get("KVQ_CLOCKS_DIR") or tempfile.gettempdir()  # the samples, summarised below
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
    """One kv head of layer 0, or one q head of a sparse layer, of a decode step on the
    CPU oracle; returns seconds."""
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
    else:  # q is one q head of kv head g
        K, V = a["k1"][g], a["v1"][g]
        k = O.ratio_k(K.shape[0], RATIO)
        C = O.critical_channels(q, O.key_absmax(K), N_CRIT)
        s = O.critical_scores(q, K, C)
        ids = O.topk_select(s, k, N_SINK, WINDOW)
        O.sparse_attn(q, K, V, ids)
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
        """Oracle time of one decode step: layer 0 (8 kv-head tasks) and one sparse
        layer (32 q-head tasks) on the pool, t_step = t0 + (n_layers - 1) * t1."""
        G = HQ // HKV
        t = time.perf_counter()
        pool.map(_oracle_task, [("quant", g, q0[g * G:(g + 1) * G], self.meta) for g in range(HKV)])
        t0 = time.perf_counter() - t
        t = time.perf_counter()
        pool.map(_oracle_task, [("sparse", h // G, q1[h], self.meta) for h in range(HQ)], chunksize=1)
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

def rank_max_ms(ms, world, device):
    """The job's time for one timed region: the slowest rank's (an all-reduce MAX over the ranks of
    the process group); with one rank, its own."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_steps_per_s(world, steps, ms):
    """Whole-job throughput of replicas: the steps every rank ran, over the slowest rank's time."""
    return world * steps / (ms * 1e-3)


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
    ap.add_argument("--rows", action="store_true",
                    help="instead of the step: time the other hot-path rows on their configurations (one JSON line)")
    ap.add_argument("--only", nargs="*", default=None, help="with --rows: the rows whose names start with these")
    ap.add_argument("--no-rows", action="store_true", help="the decode step only, without the other rows")
    ap.add_argument("--row-layers", type=int, default=0,
                    help="with --rows: layers of the H2O run and of the pack (default: 32 and 40; fewer for a "
                         "profiler capture)")
    args = ap.parse_args()
    if args.rows:
        import torch

        from compressed_kv_cache_quant_gb300.build import build
        build()
        dev = torch.device("cuda", 0)
        global ROW_LAYERS
        ROW_LAYERS = args.row_layers
        print(json.dumps({"rows": run_rows(dev, torch.cuda.Stream(dev), args.only)}))
        return
    assert args.warmup >= 1 and args.steps >= 1 and args.layers >= 2

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    n_workers = args.cpu_workers or (os.cpu_count() or 1)

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
    ms = rank_max_ms(ms, world, device)
    if world > 1:
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
        t_e2e = rank_max_ms(1e3 * (time.perf_counter() - t0), world, device) * 1e-3
        step_i += args.steps
        bi = (W.in_q.numel() + W.in_k.numel() + W.in_v.numel()) * 2
        e2e = {"value": job_steps_per_s(world, args.steps, t_e2e * 1e3), "unit": "steps/s", "h2d_bytes_per_step": bi,
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
               "sample": f"layer 0 (1-bit quantized, 8 kv-head tasks) and one sparse layer (32 q-head "
                         f"tasks) of a {args.prompt}-token step on a {n_workers}-process pool (the host's "
                         f"{os.cpu_count()} cores); step time = t0 + {args.layers - 1} x t_sparse = "
                         f"{t0c:.2f} s + {args.layers - 1} x {t1c:.2f} s"}

    # ---- the other rows of the hot path, each on its own configuration (rank 0, after the step)
    rows = None
    launches = W.launches_per_step * args.steps
    if rank == 0 and not args.no_rows:
        del W, g0, g_step, qs, ks, vs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        rows = run_rows(device, stream)

    if rank == 0:
        value = job_steps_per_s(world, args.steps, ms)
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
            "e2e": e2e, "gpu_launches": launches,
            "clocks": clk, "cpu_baseline": cpu,
            "rows": rows,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------------ the other rows
#
# Every other row of the hot path on its configuration: CUDA events on the launching stream
# around enough calls to fill a fraction of a second (inputs larger than L2 wherever a row
# streams memory), nvidia-smi clocks sampled during that region, and a bounded single-threaded
# sample of the oracle doing the same work.  Each row's inputs are built first and freed
# after it, so that the rows run one after another in the same process as the decode step.

def _timed(torch, fn, stream, min_ms=250.0, warm=2):
    """(ms per call, calls, clocks) of fn(), which launches on `stream`: CUDA events on that
    stream around enough calls to fill about min_ms of device time."""
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        a.record(stream)
        fn()
        b.record(stream)
    stream.synchronize()
    reps = max(3, min(2000, int(math.ceil(min_ms / max(a.elapsed_time(b), 1e-3)))))
    clocks = Clocks(torch.cuda.current_device())
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    return a.elapsed_time(b) / reps, reps, clk


def _wall(fn):
    t = time.perf_counter()
    fn()
    return time.perf_counter() - t


def _hbm(peak, peak_src):
    def f(achieved):
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": peak_src}
    return f


def _capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def row_pack(torch, np, kvq, synth, O, device, stream, hbm):
    """a1 kv_quant_pack, the Qwen-1.5-14B-shaped prefill: 40 layers x 40 kv heads x 131072 tokens
    to 1 bit (K per channel g64, V per token G64), one call per layer."""
    T, H, L = 131072, 40, ROW_LAYERS or 40
    n_in = min(8, L)
    seed = synth.BASE_SEED + 4
    n_pages = T // 16
    seqs = kvq.Batch(torch.arange(n_pages, dtype=torch.int32, device=device)[None],
                     torch.tensor([T], dtype=torch.int32, device=device), T)
    ins = [synth.kv_rows(T, H, synth.mix(seed, 200 + j), device=device) for j in range(n_in)]
    caches = [kvq.LayerCache(H, H, 1, n_pages, 1, v_group_dims=64, device=device) for _ in range(L)]
    sh = stream.cuda_stream

    def all_layers():
        for l in range(L):
            K, V = ins[l % n_in]
            kvq.kv_quant_pack(caches[l], seqs, 0, 0, T, K, V, stream=sh)
    ms, reps, clk = _timed(torch, all_layers, stream)
    nbytes = L * (2 * T * H * D * 2 + T * H * 48)
    gbs = nbytes / (ms * 1e-3) / 1e9
    k1, v1 = ins[0][0][:, 0].cpu().numpy(), ins[0][1][:, 0].cpu().numpy()
    del ins, caches
    t = _wall(lambda: (O.pack_k(k1, 1), O.pack_v(v1, 1, 64)))
    return {"config": "Qwen-1.5-14B-shaped prefill: 40 layers x 40 kv heads x 131072 tokens to 1 bit (K per channel "
                      "g64, V per token G64), one call per layer; 8 distinct 2.68 GB fp16 inputs cycled over the layers",
            "value": gbs, "unit": "GB/s (pack of all layers)", "ms_all_layers": ms, "bytes": nbytes, "calls": reps,
            "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": (T * D * 2 * 2 + T * 48) / t / 1e9, "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": f"one kv head of one layer ({T} tokens), numpy"}}


def row_int4(torch, np, kvq, synth, O, device, stream, hbm):
    """a3 kv_decode_attn_quant, the Llama-2-7B-shaped INT4 serving batch: 16 sequences with
    lengths U[4096, 32768], 32 heads MHA, K 4-bit g64, V 4-bit G32, sequences 0-7 sharing a
    2048-token prefix (128 reference-counted pages), shuffled page ids; a step is 32 layers."""
    B, H, L, n_c, pre = 16, 32, 32, 4, 2048
    seed = synth.BASE_SEED + 2
    lens = [int(x) for x in synth.lengths_uniform(B, 4096, 32768, seed)]
    pages = [-(-T // 16) for T in lens]
    alloc = kvq.Allocator(sum(pages) + 4, seed=7)
    bt = np.full((B, max(pages)), -1, dtype=np.int32)
    for b in range(B):
        start = 0
        if 0 < b < 8:
            bt[b, :pre // 16] = bt[0, :pre // 16]
            for pg in bt[0, :pre // 16]:
                alloc.ref(int(pg))
            start = pre // 16
        bt[b, start:pages[b]] = alloc.alloc(pages[b] - start)
    seqs = kvq.Batch(torch.from_numpy(bt).to(device), torch.tensor(lens, dtype=torch.int32, device=device), max(lens))
    caches = []
    for c in range(n_c):
        cache = kvq.LayerCache(H, H, 4, sum(pages) + 4, B, v_group_dims=32, device=device)
        prefix = None
        for b, T in enumerate(lens):
            K, V = synth.kv_rows(T, H, synth.mix(seed, 10 + b, c), device=device)
            if b == 0:
                prefix = (K[:pre].clone(), V[:pre].clone())
            elif b < 8:
                K[:pre], V[:pre] = prefix
            t0 = pre if 0 < b < 8 else 0
            kvq.kv_quant_pack(cache, seqs, b, t0, T - t0, K[t0:], V[t0:])
            if c == 0 and b == 0:
                k0, v0 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
            del K, V
        caches.append(cache)
        del prefix
    torch.cuda.synchronize()
    q = synth.normal((L, B, H, D), synth.mix(seed, 99), device)
    out = torch.empty((L, B, H, D), device=device)
    ws = kvq.Workspace(kvq.kv_decode_attn_quant_ws(caches[0], seqs))
    plan = kvq.kv_decode_attn_quant_plan(caches[0], seqs)
    g = _capture(torch, lambda: [kvq.kv_decode_attn_quant(caches[l % n_c], seqs, q[l], out[l], ws,
                                                         stream=stream.cuda_stream) for l in range(L)], stream)
    ms, reps, clk = _timed(torch, g.replay, stream)
    kvq.kvq_check(ws, stream=stream.cuda_stream)
    tails = sum(T % 64 for T in lens) * H * D * 2
    unique = (sum(lens) - 7 * pre) * H * 152 + tails
    per_request = sum(lens) * H * 152 + tails
    gbs = L * unique / (ms * 1e-3) / 1e9
    q0 = q[0, 0, :1].cpu().numpy()
    del caches, g
    pk, pv = O.pack_k(k0, 4), O.pack_v(v0, 4, 32)
    t = _wall(lambda: O.decode_attn_quant(q0, [pk], [pv]))
    return {"config": f"Llama-2-7B-shaped INT4 serving batch: 16 sequences, T ~ U[4096, 32768] (sum {sum(lens)}), "
                      "32 heads MHA, K 4-bit g64, V 4-bit G32, sequences 0-7 sharing 128 prefix pages, shuffled "
                      "page ids; one step = 32 layers (4 distinct 1.7 GB layer caches cycled, each larger than L2)",
            "value": 1e3 / ms, "unit": "steps/s", "ms_per_step": ms, "GBps_unique": gbs,
            "bytes_per_step_unique": L * unique, "bytes_per_step_per_request": L * per_request,
            "split_plan": {"n_splits": plan[0], "groups_per_split": plan[1]}, "steps": reps,
            "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": (lens[0] * 152) / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"one (sequence, head) of {lens[0]} tokens, numpy fp64"}}


def row_outlier(torch, np, kvq, synth, O, device, stream, hbm):
    """f3 kv_decode_attn_quant_outlier: the INT4 serving batch shape (16 sequences, lengths
    U[4096, 32768], 32 heads MHA, K 4-bit g64, V 4-bit G32; no shared prefix, since the outlier
    channels are chosen per sequence) with the top-0.5 % key channel of every (sequence, head)
    isolated in fp16 (n_out = ceil(0.005 * 128) = 1), chosen from the prompt; a step is 32
    layers.  The plain attention over the same main caches is timed beside it (the fp16 outlier
    term is then missing: the cost of the isolation, not a second answer)."""
    B, H, L, n_c, n_out = 16, 32, 32, 4, 1
    seed = synth.BASE_SEED + 2
    lens = [int(x) for x in synth.lengths_uniform(B, 4096, 32768, seed)]
    pages = [-(-T // 16) for T in lens]
    alloc = kvq.Allocator(sum(pages) + 4, seed=7)
    bt = np.full((B, max(pages)), -1, dtype=np.int32)
    for b in range(B):
        bt[b, :pages[b]] = alloc.alloc(pages[b])
    seqs = kvq.Batch(torch.from_numpy(bt).to(device), torch.tensor(lens, dtype=torch.int32, device=device), max(lens))
    caches, chs, kos = [], [], []
    wc = kvq.Workspace(kvq.kv_outlier_channels_ws(kvq.make_layout(H, H, 4, 32)))
    keys0 = []  # layer cache 0's prompt keys, kept to time the prefill isolation again below
    for c in range(n_c):
        cache = kvq.LayerCache(H, H, 4, sum(pages) + 4, B, v_group_dims=32, device=device)
        och = torch.zeros((B, H, n_out), dtype=torch.int32, device=device)
        k_out = torch.zeros((sum(pages) + 4, H, 16, n_out), dtype=torch.float16, device=device)
        for b, T in enumerate(lens):
            K, V = synth.kv_rows(T, H, synth.mix(seed, 10 + b, c), device=device)
            kvq.kv_quant_pack(cache, seqs, b, 0, T, K, V)
            kvq.kv_outlier_channels(cache, K, T, n_out, och[b], wc)
            kvq.kv_outlier_isolate(cache, seqs, b, 0, T, K, n_out, och, k_out)
            if c == 0:
                keys0.append(K)
                if b == 0:
                    k0, v0 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
            del K, V
        caches.append(cache)
        chs.append(och)
        kos.append(k_out)
    torch.cuda.synchronize()
    # the prefill side of one layer: channel statistics and isolation of every sequence (repeating it
    # on the isolated cache rewrites the same values), as one graph: device time without host gaps
    sh = stream.cuda_stream
    gi = _capture(torch, lambda: [(kvq.kv_outlier_channels(caches[0], keys0[b], T, n_out, chs[0][b], wc, stream=sh),
                                   kvq.kv_outlier_isolate(caches[0], seqs, b, 0, T, keys0[b], n_out, chs[0], kos[0],
                                                          stream=sh))
                                  for b, T in enumerate(lens)], stream)
    ms_iso, _, _ = _timed(torch, gi.replay, stream, min_ms=50.0)
    del gi, keys0
    q = synth.normal((L, B, H, D), synth.mix(seed, 99), device)
    out = torch.empty((L, B, H, D), device=device)
    ws = kvq.Workspace(kvq.kv_decode_attn_quant_ws(caches[0], seqs))
    g = _capture(torch, lambda: [kvq.kv_decode_attn_quant_outlier(caches[l % n_c], seqs, q[l], n_out, chs[l % n_c],
                                                                  kos[l % n_c], out[l], ws, stream=stream.cuda_stream)
                                 for l in range(L)], stream)
    ms, reps, clk = _timed(torch, g.replay, stream)
    kvq.kvq_check(ws, stream=stream.cuda_stream)
    gp = _capture(torch, lambda: [kvq.kv_decode_attn_quant(caches[l % n_c], seqs, q[l], out[l], ws,
                                                          stream=stream.cuda_stream) for l in range(L)], stream)
    ms_plain, _, _ = _timed(torch, gp.replay, stream)
    tails = sum(T % 64 for T in lens) * H * D * 2
    per_tok = 152 + 2 * n_out
    unique = sum(lens) * H * per_tok + tails
    gbs = L * unique / (ms * 1e-3) / 1e9
    q0 = q[0, 0, :1].cpu().numpy()
    del caches, kos, g, gp
    ch0 = O.outlier_channels(k0, n_out)
    t = _wall(lambda: O.decode_attn_quant(q0, [O.pack_k_outlier(k0, 4, ch0)], [O.pack_v(v0, 4, 32)]))
    return {"config": f"INT4 serving batch with isolated outlier channels: 16 sequences, T ~ U[4096, 32768] "
                      f"(sum {sum(lens)}), 32 heads MHA, K 4-bit g64 + {n_out} fp16 outlier channel per (sequence, "
                      "head), V 4-bit G32, shuffled page ids; one step = 32 layers (4 distinct layer caches cycled)",
            "value": 1e3 / ms, "unit": "steps/s", "ms_per_step": ms, "GBps": gbs,
            "bytes_per_step": L * unique, "plain_attention_ms_per_step": ms_plain,
            "isolation_overhead": ms / ms_plain - 1.0,
            "prefill_channels_and_isolate_ms_per_layer": ms_iso,
            "prefill_channels_GBps": sum(lens) * H * D * 2 / (ms_iso * 1e-3) / 1e9, "steps": reps,
            "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": (lens[0] * per_tok) / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"one (sequence, head) of {lens[0]} tokens, numpy fp64"}}


def row_h2o(torch, np, kvq, synth, O, device, stream, hbm, steps=256):
    """a2 + a6 + a7, the Llama-3-8B-shaped H2O eviction run: 8 sequences, 32 layers of 32 q / 8 kv
    heads, 32768-token prompts, budget 6553 = 4 sinks + 2048 window + 4501 heavy hitters; step 0
    picks the initial heavy hitters from one full-context attention, then every decode step
    appends a token, attends the retained set (one list per kv head, probabilities out), adds the
    group's probabilities to the cumulative scores, evicts down to budget - 1 and admits the
    next token.  Queries prefer 64 hot keys per (layer, sequence, kv head) with Zipf(1.2) weights."""
    B, Hq, Hkv, L, T0, budget, ns, w = 8, 32, 8, ROW_LAYERS or 32, 32768, 6553, 4, 2048
    G, n_hot = Hq // Hkv, 64
    seed = synth.BASE_SEED + 3
    cap_tok = T0 + steps + 16
    per = -(-cap_tok // 16)
    alloc = kvq.Allocator(B * per, seed=11)
    bt = torch.tensor([alloc.alloc(per) for _ in range(B)], dtype=torch.int32, device=device)
    seqs = kvq.Batch(bt, torch.full((B,), T0, dtype=torch.int32, device=device), cap_tok)
    caches = []
    kn = torch.empty((L, steps, B, Hkv, D), dtype=torch.float16, device=device)
    vn = torch.empty_like(kn)
    qb = torch.empty((L, steps, B, Hq, D), dtype=torch.float16, device=device)
    for l in range(L):
        cache = kvq.LayerCache(Hq, Hkv, 16, B * per, B, device=device)
        hot = torch.empty((B, Hkv, n_hot, D), dtype=torch.float16, device=device)
        for b in range(B):
            K, V = synth.kv_rows(T0 + steps, Hkv, synth.mix(seed, l, b), device=device)
            kvq.kv_quant_pack(cache, seqs, b, 0, T0, K[:T0], V[:T0])
            kn[l, :, b], vn[l, :, b] = K[T0:], V[T0:]
            pos, _ = synth.h2o_hot_positions(synth.mix(seed, l, b), T0, n_hot)
            hot[b] = K[pos.to(device)].permute(1, 0, 2)
            if l == 0 and b == 0:
                k00, v00 = K[:T0, 0].cpu().numpy(), V[:T0, 0].cpu().numpy()
            del K, V
        bank = synth.h2o_query_bank(hot.reshape(B * Hkv, n_hot, D), steps * G, synth.mix(seed, 900, l))
        qb[l] = bank.view(B, Hkv, steps, G, D).permute(2, 0, 1, 3, 4).reshape(steps, B, Hq, D)
        caches.append(cache)
    cap = T0 + 2
    retained = torch.zeros((L, B, Hkv, cap), dtype=torch.int32, device=device)
    retained[..., :T0] = torch.arange(T0, dtype=torch.int32, device=device)
    counts = torch.full((L, B, Hkv), T0, dtype=torch.int32, device=device)
    cum = torch.zeros((L, B, Hkv, cap), device=device)
    probs = torch.zeros((B, Hq, cap), device=device)
    out = torch.empty((L, B, Hq, D), device=device)
    in_q = torch.empty((L, B, Hq, D), dtype=torch.float16, device=device)
    in_k = torch.empty((L, B, Hkv, D), dtype=torch.float16, device=device)
    in_v = torch.empty_like(in_k)
    wsa = kvq.Workspace(kvq.kv_sparse_attn_ws(caches[0], seqs, cap))
    wsh = kvq.Workspace(kvq.kv_h2o_accumulate_ws())
    wsp = kvq.Workspace(kvq.kv_page_append_ws())
    sh = stream.cuda_stream
    torch.cuda.synchronize()
    # step 0: the initial heavy hitters from one full-context attention per layer (not timed)
    with torch.cuda.stream(stream):
        for l in range(L):
            kvq.kv_sparse_attn(caches[l], seqs, qb[l, 0], retained[l], counts[l], 1, out[l], probs, wsa, stream=sh)
            kvq.kv_h2o_accumulate(caches[l], seqs, probs, retained[l], counts[l], cum[l], budget, ns, w,
                                  seqs.seq_lens, None, wsh, stream=sh)
    stream.synchronize()

    def one_step():
        kvq.kvq_seq_lens_add(seqs.seq_lens, 1, stream=sh)
        for l in range(L):
            kvq.kv_page_append(caches[l], seqs, in_k[l], in_v[l], wsp, stream=sh)
            kvq.kv_sparse_attn(caches[l], seqs, in_q[l], retained[l], counts[l], 1, out[l], probs, wsa, stream=sh)
            kvq.kv_h2o_accumulate(caches[l], seqs, probs, retained[l], counts[l], cum[l], budget, ns, w,
                                  seqs.seq_lens, None, wsh, stream=sh)
    g = _capture(torch, one_step, stream)

    def feed(s):
        in_q.copy_(qb[:, s], non_blocking=True)
        in_k.copy_(kn[:, s - 1], non_blocking=True)
        in_v.copy_(vn[:, s - 1], non_blocking=True)
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for s in range(1, steps):
            feed(s)
            g.replay()
        e.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    for x in (wsa, wsh, wsp):
        kvq.kvq_check(x, stream=sh)
    ms = a.elapsed_time(e) / (steps - 1)
    n_ret = int(counts.sum().item()) // (L * B * Hkv)
    rows = B * Hkv * budget * 2 * D * 2
    book = B * Hkv * budget * 12 + B * Hq * budget * 8   # ids + cum read/write, probabilities write + read
    nbytes = L * (rows + book)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del caches, g, kn, vn, qb
    r0 = np.concatenate([np.arange(ns), np.sort(np.random.default_rng(5).choice(np.arange(ns, T0 - w), budget - ns - w,
                                                                                   replace=False)),
                         np.arange(T0 - w, T0)])
    qg = synth.normal((G, D), 17, "cpu").numpy()
    t = _wall(lambda: O.h2o_step(qg, k00, v00, r0, np.zeros(budget), T0 - 1, budget, ns, w))
    return {"config": "Llama-3-8B-shaped H2O eviction: 8 sequences, 32 layers of 32 q / 8 kv heads (GQA 4), 32768-token "
                      "prompts, budget 6553 = 4 sinks + 2048 window + 4501 heavy hitters, power-law queries; one step = "
                      "append + attention over the retained set + accumulate / evict / admit in every layer",
            "value": 1e3 / ms, "unit": "steps/s", "ms_per_step": ms, "steps": steps - 1,
            "retained_per_kv_head": n_ret, "GBps": gbs, "bytes_per_step": nbytes,
            "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": 1.0 / (t * L * B * Hkv), "unit": "steps/s", "cores": 1, "kind": "oracle",
                             "sample": "one (sequence, kv head, layer) step of the oracle, numpy fp64, times 2048"}}


def row_offload(torch, np, kvq, synth, O, device, stream):
    """a9, the Qwen-1.5-14B-shaped offload: 40 layers of 40 MHA heads at 131072 tokens, fp16 K/V in
    pinned host memory; per layer the top-K (K = 3932) rows of every head are gathered over the
    host link into an HBM double buffer while the previous layer attends."""
    from compressed_kv_cache_quant_gb300.offload import OffloadLayers
    H, T, L, n_res = 40, 131072, 40, 2
    seed = synth.BASE_SEED + 4
    KV = [synth.kv_rows(T, H, synth.mix(seed, 300 + j), device=device) for j in range(n_res)]
    off = OffloadLayers(H, T, KV, [l % n_res for l in range(L)], device=device)
    k0 = KV[0][0][:, 0].cpu().numpy()
    del KV
    torch.cuda.empty_cache()
    qs = synth.normal((L, 1, H, D), synth.mix(seed, 301), device)
    outs = torch.empty((L, 1, H, D), device=device)
    copy_s = torch.cuda.Stream(device, priority=0)
    attn_s = torch.cuda.Stream(device, priority=-1)   # the attention's CTAs go first when SMs free up

    def pipelined():
        off.step(qs, outs, copy_s, attn_s)

    def gathers():            # the host-link side alone
        for l in range(L):
            off.gather(l, l % 2, attn_s)

    def compute():            # the GPU side alone: selection and attention of every layer
        for l in range(L):
            off.select(l, qs[l], l % 2, attn_s)
            off.attend(l, qs[l], outs[l], l % 2, attn_s)

    def attention():
        for l in range(L):
            off.attend(l, qs[l], outs[l], l % 2, attn_s)
    t_pipe, reps, clk = _timed(torch, pipelined, attn_s)
    t_g = _timed(torch, gathers, attn_s, min_ms=150.0)[0]
    t_c = _timed(torch, compute, attn_s, min_ms=150.0)[0]
    t_attn = _timed(torch, attention, attn_s, min_ms=150.0)[0]
    off.check()
    link_bytes = L * off.gather_bytes_per_layer
    hsrc = torch.empty(off.gather_bytes_per_layer, dtype=torch.uint8).pin_memory()
    ddst = torch.empty(off.gather_bytes_per_layer, dtype=torch.uint8, device=device)
    ms_copy = _timed(torch, lambda: ddst.copy_(hsrc, non_blocking=True), attn_s, min_ms=100.0)[0]
    peak = off.gather_bytes_per_layer / (ms_copy * 1e-3) / 1e9
    link = link_bytes / (t_g * 1e-3) / 1e9
    overlap = (t_g + t_c - t_pipe) / min(t_g, t_c)
    rng = np.random.default_rng(9)
    ids = np.sort(rng.choice(T, size=off.K, replace=False))
    t = _wall(lambda: O.offload_gather(k0, ids))
    del off, hsrc, ddst
    return {"config": "Qwen-1.5-14B-shaped offload: 40 layers of 40 MHA heads, T = 131072, fp16 K/V in pinned host memory "
                      f"(2 distinct layers cycled), top-K = {math.floor(RATIO * T)} rows per head gathered into an HBM "
                      "double buffer; critical keys, 4 sinks and the 128-token window in HBM",
            "value": link, "unit": "GB/s over the host link (gathers alone)",
            "overlap": overlap, "overlap_definition": "(t_gather + t_compute - t_pipelined) / min(t_gather, t_compute); "
                                                      "gather = the host-link gathers alone, compute = selection + "
                                                      "attention of every layer alone",
            "ms_step_pipelined": t_pipe, "ms_gather": t_g, "ms_compute": t_c, "ms_attention": t_attn,
            "bytes_per_step": link_bytes, "calls": reps,
            "roofline": {"bound": "host link", "achieved": link, "peak": peak, "unit": "GB/s", "frac": link / peak,
                         "peak_source": "measured pinned->device cudaMemcpyAsync of one layer's gather bytes"},
            "clocks": clk,
            "cpu_baseline": {"value": len(ids) * D * 2 / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "one head's K rows, numpy (host to host)"}}


def row_block(torch, np, kvq, synth, O, device, stream, hbm, T=131072):
    """f1 block pruning (64-token blocks) next to the token top-K on one Llama-3.1-8B-shaped
    sparse layer: selection over the critical-channel scores + exact attention."""
    Hq, Hkv, ns, w, blk = 32, 8, 4, 128, 64
    seed = synth.BASE_SEED + 6
    n_pages = -(-T // 16)
    alloc = kvq.Allocator(n_pages, seed=13)
    seqs = kvq.Batch(torch.tensor([alloc.alloc(n_pages)], dtype=torch.int32, device=device),
                     torch.tensor([T], dtype=torch.int32, device=device), T)
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, 1, t_cap=(T + 7) // 8 * 8, device=device)
    K, V = synth.kv_rows(T, Hkv, synth.mix(seed, 0), device=device)
    kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)
    del K, V
    sh = stream.cuda_stream
    q = synth.normal((1, Hq, D), synth.mix(seed, 1), device)
    sc = torch.empty((1, Hq, (T + 7) // 8 * 8), device=device)
    kvq.kv_critical_score(cache, seqs, q, 8, None, sc)
    kt, nb = O.ratio_k(T, RATIO), O.block_count(T, RATIO, blk)
    cap = max(O.topk_count(T, kt, ns, w), ns + w + nb * blk)
    sel_t = torch.empty((1, Hq, cap), dtype=torch.int32, device=device)
    sel_b = torch.empty((1, Hq, cap), dtype=torch.int32, device=device)
    cnt_t = torch.empty((1, Hq), dtype=torch.int32, device=device)
    cnt_b = torch.empty((1, Hq), dtype=torch.int32, device=device)
    out = torch.empty((1, Hq, D), device=device)
    wt = kvq.Workspace(kvq.kv_topk_select_ws())
    wb = kvq.Workspace(kvq.kv_block_select_ws(seqs, Hq, blk))
    wa = kvq.Workspace(kvq.kv_sparse_attn_ws(cache, seqs, cap))

    def tok():
        kvq.kv_topk_select(seqs, Hq, sc, -1, RATIO, ns, w, sel_t, cnt_t, wt, stream=sh)
        kvq.kv_sparse_attn(cache, seqs, q, sel_t, cnt_t, 0, out, None, wa, stream=sh)

    def blkp():
        kvq.kv_block_select(seqs, Hq, sc, -1, RATIO, ns, w, blk, sel_b, cnt_b, wb, stream=sh)
        kvq.kv_sparse_attn(cache, seqs, q, sel_b, cnt_b, 0, out, None, wa, stream=sh)
    ms_tok = _timed(torch, tok, stream, min_ms=100.0)[0]
    ms_blk, reps, clk = _timed(torch, blkp, stream, min_ms=150.0)
    for x in (wt, wb, wa):
        kvq.kvq_check(x, stream=sh)
    rows_t, rows_b = int(cnt_t.sum().item()), int(cnt_b.sum().item())
    by_t, by_b = Hq * T * 4 + rows_t * 2 * D * 2, Hq * T * 4 + rows_b * 2 * D * 2
    s0 = sc[0, 0, :T].cpu().numpy()
    del cache
    t = _wall(lambda: O.block_select(s0, nb, ns, w, blk))
    gbs = by_b / (ms_blk * 1e-3) / 1e9
    return {"config": f"32 q / 8 kv heads, T = {T}, ratio {RATIO}: {nb} blocks of {blk} + {ns} sinks + {w} window per "
                      f"q head (token top-K: {kt}); selection over precomputed critical scores + exact attention",
            "value": gbs, "unit": "GB/s", "ms_block_path": ms_blk, "ms_token_path": ms_tok,
            "token_path_GBps": by_t / (ms_tok * 1e-3) / 1e9, "rows_block": rows_b, "rows_token": rows_t,
            "bytes": by_b, "calls": reps, "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": t * 1e3 * Hq, "unit": "ms per layer (selection only)", "cores": 1,
                             "kind": "oracle", "sample": "block selection of one q head, numpy, times 32"}}


def row_group(torch, np, kvq, synth, O, device, stream, hbm, T=131072):
    """f1 selection shared by the q heads of a kv head (GQA) on one Llama-3.1-8B-shaped sparse
    layer: critical scores per kv head (the group's |q| summed), top-K per kv head, exact
    attention of the 4 q heads over their kv head's list -- three launches -- next to the
    per-q-head layer kernel of the decode step on the same cache."""
    Hq, Hkv, ns, w = 32, 8, 4, 128
    seed = synth.BASE_SEED + 7
    n_pages = -(-(T + 64) // 16)
    alloc = kvq.Allocator(n_pages, seed=19)
    seqs = kvq.Batch(torch.tensor([alloc.alloc(n_pages)], dtype=torch.int32, device=device),
                     torch.tensor([T], dtype=torch.int32, device=device), 16 * n_pages)
    t_cap = 16 * n_pages
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, 1, t_cap=t_cap, device=device)
    K, V = synth.kv_rows(T, Hkv, synth.mix(seed, 0), device=device)
    kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)
    k_new, v_new = K[-1:].clone(), V[-1:].clone()
    K0, V0 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
    del K, V
    sh = stream.cuda_stream
    q = synth.normal((1, Hq, D), synth.mix(seed, 1), device)
    sc = torch.empty((1, Hkv, t_cap), device=device)
    kt = O.ratio_k(T, RATIO)
    cap = O.topk_count(T, kt, ns, w)
    sel = torch.empty((1, Hkv, cap), dtype=torch.int32, device=device)
    cnt = torch.empty((1, Hkv), dtype=torch.int32, device=device)
    out = torch.empty((1, Hq, D), device=device)
    wt = kvq.Workspace(kvq.kv_topk_select_ws())
    wa = kvq.Workspace(kvq.kv_sparse_attn_ws(cache, seqs, cap))
    wl = kvq.Workspace(kvq.kv_sparse_layer_decode_ws())

    def grouped():
        kvq.kv_group_critical_score(cache, seqs, q, N_CRIT, None, sc, stream=sh)
        kvq.kv_topk_select(seqs, Hkv, sc, -1, RATIO, ns, w, sel, cnt, wt, stream=sh)
        kvq.kv_sparse_attn(cache, seqs, q, sel, cnt, 1, out, None, wa, stream=sh)
    g = _capture(torch, grouped, stream)
    ms, reps, clk = _timed(torch, g.replay, stream, min_ms=150.0)
    # the per-q-head layer kernel on the same cache (it also appends the newest token, rewriting
    # the same position each call: the sequence length does not change)
    g1 = _capture(torch, lambda: kvq.kv_sparse_layer_decode(cache, seqs, k_new, v_new, q, N_CRIT, -1, RATIO, ns, w,
                                                            out, wl, stream=sh), stream)
    ms_head = _timed(torch, g1.replay, stream, min_ms=100.0)[0]
    for x in (wt, wa, wl):
        kvq.kvq_check(x, stream=sh)
    nbytes = Hkv * N_CRIT * T * 2 + 2 * Hkv * T * 4 + Hkv * cap * 2 * D * 2
    head_bytes = Hq * N_CRIT * T * 2 + Hq * cap * 2 * D * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    del cache, g, g1
    qg = q[0, :Hq // Hkv].cpu().numpy()

    def oracle_kv_head():
        C = O.group_critical_channels(qg, O.key_absmax(K0), N_CRIT)
        ids = O.topk_select(O.group_critical_scores(qg, K0, C), kt, ns, w)
        for j in range(Hq // Hkv):
            O.sparse_attn(qg[j], K0, V0, ids)
    t = _wall(oracle_kv_head)
    return {"config": f"32 q / 8 kv heads, T = {T}: per kv head 8 critical channels (|q| summed over its 4 q heads), "
                      f"top-K = {kt} + 4 sinks + 128 window, the 4 q heads attend the shared list (3 launches); "
                      "per-q-head layer kernel on the same cache for comparison",
            "value": 1e3 / ms, "unit": "layers/s", "ms_per_layer": ms, "ms_per_layer_per_q_head_selection": ms_head,
            "bytes_per_layer": nbytes, "bytes_per_layer_per_q_head_selection": head_bytes, "GBps": gbs,
            "calls": reps, "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": 1.0 / (t * Hkv), "unit": "layers/s", "cores": 1, "kind": "oracle",
                             "sample": "one kv head's selection and its 4 heads' attention, numpy, times 8"}}


def row_fp8(torch, np, kvq, synth, O, device, stream, hbm, T=131072):
    """f4 an FP8 E4M3 layer of the Llama-3.1-8B shape (32 q / 8 kv heads, 131072 tokens): decode
    attention over the E4M3 cache (pages staged by bulk asynchronous copies, tensor cores)."""
    Hq, Hkv = 32, 8
    seed = synth.BASE_SEED + 8
    n_pages = T // 16
    alloc = kvq.Allocator(n_pages, seed=23)
    seqs = kvq.Batch(torch.tensor([alloc.alloc(n_pages)], dtype=torch.int32, device=device),
                     torch.tensor([T], dtype=torch.int32, device=device), T)
    cache = kvq.LayerCache(Hq, Hkv, kvq.BITS_E4M3, n_pages, 1, device=device)
    K, V = synth.kv_rows(T, Hkv, synth.mix(seed, 0), device=device)
    kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)
    K0, V0 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
    del K, V
    q = synth.normal((1, Hq, D), synth.mix(seed, 1), device)
    out = torch.empty((1, Hq, D), device=device)
    ws = kvq.Workspace(kvq.kv_decode_attn_quant_ws(cache, seqs))
    sh = stream.cuda_stream
    g = _capture(torch, lambda: kvq.kv_decode_attn_quant(cache, seqs, q, out, ws, stream=sh), stream)
    ms, reps, clk = _timed(torch, g.replay, stream, min_ms=150.0)
    kvq.kvq_check(ws, stream=sh)
    plan = kvq.kv_decode_attn_quant_plan(cache, seqs)
    nbytes = Hkv * T * 2 * D
    gbs = nbytes / (ms * 1e-3) / 1e9
    q0 = q[0, 0].cpu().numpy()
    del cache, g
    t = _wall(lambda: O.fp8_attention(q0, K0, V0))
    return {"config": f"FP8 E4M3 layer, 32 q / 8 kv heads (GQA 4), T = {T}: K and V rows as E4M3 bytes (256 B per token "
                      "and kv head), decode attention of all 32 heads",
            "value": gbs, "unit": "GB/s", "us_per_launch": ms * 1e3, "bytes_per_launch": nbytes,
            "split_plan": {"n_splits": plan[0], "groups_per_split": plan[1]}, "calls": reps,
            "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": T * 2 * D / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "one q head over one kv head's E4M3 cache, numpy fp64"}}


def row_mixed(torch, np, kvq, synth, O, device, stream, hbm, T=131072):
    """f2 + f4 head-level: one Llama-3.1-8B-shaped layer (32 q / 8 kv heads, T = 131072) whose kv
    heads were classified one by one; 2 of the 8 dense (their q heads attend every token), 6 sparse
    (critical scores + top-K + attention); classes dispatched on the device (the cluster launch for
    the sparse heads and every append, then the dense kv heads' GQA-shared attention).  Algorithmic
    bytes: a dense kv head's K and V once (its q heads share them), a sparse q head's critical
    channels and selected rows."""
    Hq, Hkv, ns, w = 32, 8, 4, 128
    dense = [1, 0, 0, 0, 0, 1, 0, 0]
    seed = synth.BASE_SEED + 9
    n_pages = -(-(T + 64) // 16)
    alloc = kvq.Allocator(n_pages, seed=29)
    seqs = kvq.Batch(torch.tensor([alloc.alloc(n_pages)], dtype=torch.int32, device=device),
                     torch.tensor([T], dtype=torch.int32, device=device), 16 * n_pages)
    cache = kvq.LayerCache(Hq, Hkv, 16, n_pages, 1, t_cap=16 * n_pages, device=device)
    K, V = synth.kv_rows(T, Hkv, synth.mix(seed, 0), device=device)
    kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)
    k_new, v_new = K[-1:].clone(), V[-1:].clone()
    K0, V0 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
    del K, V
    q = synth.normal((1, Hq, D), synth.mix(seed, 1), device)
    out = torch.empty((1, Hq, D), device=device)
    dn = torch.tensor([dense], dtype=torch.int32, device=device)
    wk = kvq.Workspace(kvq.kv_mixed_layer_decode_ws(cache, seqs))
    sh = stream.cuda_stream
    g = _capture(torch, lambda: kvq.kv_mixed_layer_decode(cache, seqs, k_new, v_new, q, N_CRIT, -1, RATIO, ns, w, dn,
                                                          out, wk, stream=sh), stream)
    ms, reps, clk = _timed(torch, g.replay, stream, min_ms=150.0)
    kvq.kvq_check(wk, stream=sh)
    n_d = sum(dense) * (Hq // Hkv)
    sel = ns + w + math.floor(RATIO * T)
    nbytes = sum(dense) * T * 2 * D * 2 + (Hq - n_d) * (N_CRIT * T * 2 + sel * 2 * D * 2)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del cache, g
    q0 = q[0, 0].cpu().numpy()
    t_d = _wall(lambda: O.sparse_attn(q0, K0, V0, np.arange(T)))

    def one_sparse():
        C = O.critical_channels(q0, O.key_absmax(K0), N_CRIT)
        O.sparse_attn(q0, K0, V0, O.topk_select(O.critical_scores(q0, K0, C), O.ratio_k(T, RATIO), ns, w))
    t_s = _wall(one_sparse)
    return {"config": f"32 q / 8 kv heads, T = {T}: kv heads {[i for i, x in enumerate(dense) if x]} classified dense "
                      "(their 8 q heads attend all tokens), the other 24 q heads sparse (8 critical channels, top-K = "
                      "floor(0.03 T) + 4 sinks + 128 window); classes dispatched on the device (cluster launch + the dense kv heads' GQA-shared attention)",
            "value": gbs, "unit": "GB/s", "us_per_layer": ms * 1e3, "bytes_per_layer": nbytes, "calls": reps,
            "roofline": hbm(gbs), "clocks": clk,
            "cpu_baseline": {"value": 1.0 / (n_d * t_d + (Hq - n_d) * t_s), "unit": "layers/s", "cores": 1,
                             "kind": "oracle", "sample": "one dense and one sparse q head, numpy, scaled to 8 + 24"}}


def row_densepref(torch, np, kvq, synth, O, device, stream, tensor_peak):
    """a8 kv_dense_pref_score at the 128K layer shape: 32 q / 8 kv heads, T = 131072, the
    n_q = 32 most recent queries, top-k = floor(0.03 T) = 3932 (the sparse layers' K).  One call
    = the tensor-core scores of 8 kv heads x 128 query rows x 131072 keys (34.4 GFLOP, K read
    once per kv head) + per-row reductions of 1024 rows of up to 131072 scores."""
    Hq, Hkv, T, n_q = 32, 8, 131072, 32
    topk = int(0.03 * T)
    seed = synth.BASE_SEED + 1
    alloc = kvq.Allocator(T // 16, seed=21)
    seqs = kvq.Batch(torch.tensor([alloc.alloc(T // 16)], dtype=torch.int32, device=device),
                     torch.tensor([T], dtype=torch.int32, device=device), T)
    cache = kvq.LayerCache(Hq, Hkv, 16, T // 16, 1, t_cap=T, device=device)
    K, V = synth.kv_rows(T, Hkv, synth.mix(seed, 60), device=device)
    kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)
    Q = synth.queries((1, Hq, n_q, D), synth.mix(seed, 61)).to(device)
    P = torch.empty((1, Hq), device=device)
    wd = kvq.Workspace(kvq.kv_dense_pref_score_ws(cache, seqs, n_q))
    sh = stream.cuda_stream
    ms, reps, clk = _timed(torch, lambda: kvq.kv_dense_pref_score(cache, seqs, Q, n_q, topk, P, wd, stream=sh),
                           stream, min_ms=100.0)
    kvq.kvq_check(wd, stream=sh)
    flops = 2.0 * Hkv * (Hq // Hkv) * n_q * T * D
    kh, qh = K[:, 0].cpu().numpy(), Q[0, 0].cpu().numpy()
    del cache, wd, K, V
    t = _wall(lambda: O.dense_pref_score(qh, kh, topk))
    return {"config": f"32 q / 8 kv heads, T = {T}, n_q = {n_q} recent queries, top-k = {topk}; one call over "
                      "all heads", "value": ms, "unit": "ms per call", "steps": reps,
            "scores_tflops_if_alone": flops / (ms * 1e-3) / 1e12,
            "roofline": {"bound": "latency", "note": "one call per layer at prefill (classification); the score "
                         f"product is {flops / 1e9:.1f} GFLOP, the per-row reductions read 1024 rows of "
                         f"{T} fp32 scores; reported as time, with the contraction rate it implies as a lower "
                         f"bound against the measured bf16 peak {tensor_peak} TFLOP/s"},
            "clocks": clk,
            "cpu_baseline": {"value": t * 1e3 * Hq, "unit": "ms per call", "cores": 1, "kind": "oracle",
                             "sample": "one q head with numpy fp64, scaled to 32 heads"}}


def row_tiny(torch, np, kvq, synth, O, device, stream):
    """a1, a3, a4, a5, a6, a8 at the tiny single-layer configuration: 8 q / 2 kv heads, T = 4096;
    a1/a3 on a 1-bit cache (K per channel g64, V per token G64) of the same keys and values
    (latency-bound: microseconds, no roofline target)."""
    Hq, Hkv, T, ncrit, kk, ns, w = 8, 2, 4096, 8, 128, 4, 64
    seed = synth.BASE_SEED
    alloc = kvq.Allocator(T // 16, seed=13)
    seqs = kvq.Batch(torch.tensor([alloc.alloc(T // 16)], dtype=torch.int32, device=device),
                     torch.tensor([T], dtype=torch.int32, device=device), T)
    cache = kvq.LayerCache(Hq, Hkv, 16, T // 16, 1, t_cap=T, device=device)
    K, V = synth.kv_rows(T, Hkv, synth.mix(seed, 1), device=device)
    kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)
    sh = stream.cuda_stream
    q = synth.queries((1, Hq, D), synth.mix(seed, 2)).to(device)
    crit = torch.empty((1, Hq, ncrit), dtype=torch.int32, device=device)
    scores = torch.empty((1, Hq, T), device=device)
    sel = torch.empty((1, Hq, ns + w + kk), dtype=torch.int32, device=device)
    cnt = torch.empty((1, Hq), dtype=torch.int32, device=device)
    out = torch.empty((1, Hq, D), device=device)
    probs = torch.empty((1, Hq, ns + w + kk), device=device)
    wt = kvq.Workspace(kvq.kv_topk_select_ws())
    wa = kvq.Workspace(kvq.kv_sparse_attn_ws(cache, seqs, ns + w + kk))
    Q = synth.queries((1, Hq, 32, D), synth.mix(seed, 41)).to(device)
    P = torch.empty((1, Hq), device=device)
    wd = kvq.Workspace(kvq.kv_dense_pref_score_ws(cache, seqs, 32))
    qc = kvq.LayerCache(Hq, Hkv, 1, T // 16, 1, v_group_dims=64, device=device)
    kvq.kv_quant_pack(qc, seqs, 0, 0, T, K, V)
    oq = torch.empty((1, Hq, D), device=device)
    wq = kvq.Workspace(kvq.kv_decode_attn_quant_ws(qc, seqs))
    calls = {
        "a1 kv_quant_pack": lambda: kvq.kv_quant_pack(qc, seqs, 0, 0, T, K, V, stream=sh),
        "a3 kv_decode_attn_quant": lambda: kvq.kv_decode_attn_quant(qc, seqs, q, oq, wq, stream=sh),
        "a4 kv_critical_score": lambda: kvq.kv_critical_score(cache, seqs, q, ncrit, crit, scores, stream=sh),
        "a5 kv_topk_select": lambda: kvq.kv_topk_select(seqs, Hq, scores, kk, 0.0, ns, w, sel, cnt, wt, stream=sh),
        "a6 kv_sparse_attn": lambda: kvq.kv_sparse_attn(cache, seqs, q, sel, cnt, 0, out, probs, wa, stream=sh),
        "a8 kv_dense_pref_score": lambda: kvq.kv_dense_pref_score(cache, seqs, Q, 32, 128, P, wd, stream=sh),
    }
    us = {n: 1e3 * _timed(torch, f, stream, min_ms=30.0)[0] for n, f in calls.items()}
    for x in (wt, wa, wd, wq):
        kvq.kvq_check(x, stream=sh)
    Kc, Vc = K.cpu().numpy(), V.cpu().numpy()
    qn, Qn = q.cpu().numpy()[0], Q.cpu().numpy()[0]
    am = [O.key_absmax(Kc[:, g]) for g in range(Hkv)]
    chans = [O.critical_channels(qn[h], am[O.kv_head_of(h, Hq, Hkv)], ncrit) for h in range(Hq)]
    sc = []
    pk, pv = [], []
    cpu = {
        "a1 kv_quant_pack": _wall(lambda: (pk.extend(O.pack_k(Kc[:, g], 1) for g in range(Hkv)),
                                           pv.extend(O.pack_v(Vc[:, g], 1, 64) for g in range(Hkv)))),
        "a3 kv_decode_attn_quant": _wall(lambda: O.decode_attn_quant(qn, pk, pv)),
        "a4 kv_critical_score": _wall(lambda: sc.extend(O.critical_scores(qn[h], Kc[:, O.kv_head_of(h, Hq, Hkv)],
                                                                          chans[h]) for h in range(Hq))),
        "a5 kv_topk_select": _wall(lambda: [O.topk_select(sc[h], kk, ns, w) for h in range(Hq)]),
        "a6 kv_sparse_attn": _wall(lambda: [O.sparse_attn(qn[h], Kc[:, O.kv_head_of(h, Hq, Hkv)],
                                                          Vc[:, O.kv_head_of(h, Hq, Hkv)],
                                                          O.topk_select(sc[h], kk, ns, w)) for h in range(Hq)]),
        "a8 kv_dense_pref_score": _wall(lambda: [O.dense_pref_score(Qn[h], Kc[:, O.kv_head_of(h, Hq, Hkv)], 128)
                                                 for h in range(Hq)]),
    }
    return {n: {"config": "8 q / 2 kv heads, T = 4096 (1-bit cache: K per channel g64, V per token G64; 8 critical "
                          "channels, K = 128 + 4 sinks + 64 window; dense preference over 32 recent queries, "
                          "top-128)", "value": v, "unit": "us",
                "roofline": {"bound": "latency", "note": "tiny parity configuration: microseconds, no roofline target"},
                "cpu_baseline": {"value": cpu[n] * 1e6, "unit": "us", "cores": 1, "kind": "oracle",
                                 "sample": "the same call on the CPU oracle, numpy"}}
            for n, v in us.items()}


ROW_LAYERS = 0  # layers of the H2O run and of the pack when set (a smaller case for a profiler capture)

ROWS = [
    ("a1 kv_quant_pack (40-layer prefill)", row_pack),
    ("a3 kv_decode_attn_quant (INT4 serving batch)", row_int4),
    ("a2+a6+a7 H2O decode (append, attention, accumulate / evict / admit)", row_h2o),
    ("a9 offload gather pipeline", row_offload),
    ("f1 kv_block_select + kv_sparse_attn (block-sparse layer)", row_block),
    ("f1 kv_group_critical_score + shared top-K + shared-list attention (GQA-shared selection)", row_group),
    ("f4 kv_decode_attn_quant on an FP8 E4M3 layer", row_fp8),
    ("f3 kv_decode_attn_quant_outlier (isolated outlier key channels, INT4 batch)", row_outlier),
    ("f2 kv_mixed_layer_decode (head-level classes dispatched on the device)", row_mixed),
    ("a8 kv_dense_pref_score (128K layer classification)", row_densepref),
    ("tiny", row_tiny),
]


def run_rows(device, stream, only=None):
    """Every row in turn (`only`: a list of name prefixes); returns {name: result}."""
    import numpy as np
    import torch

    from compressed_kv_cache_quant_gb300 import kvq, synth
    from oracle import kvq_oracle as O
    peak, src = measured_peaks()
    out = {}
    for name, fn in ROWS:
        if only and not any(name.startswith(o) for o in only):
            continue
        t0 = time.perf_counter()
        try:
            if fn in (row_offload, row_tiny):
                r = fn(torch, np, kvq, synth, O, device, stream)
            elif fn is row_densepref:
                r = fn(torch, np, kvq, synth, O, device, stream, measured_tensor_peak())
            else:
                r = fn(torch, np, kvq, synth, O, device, stream, _hbm(peak, src))
            if fn is row_tiny:
                out.update(r)
            else:
                r["wall_s"] = time.perf_counter() - t0
                out[name] = r
        except Exception as e:  # report the row's failure and go on with the others
            out[name] = {"error": repr(e)}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


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
                             "sample": "per step: layer 0 and one sparse layer timed on the process pool "
                                       f"({n_workers} processes, the host's {os.cpu_count()} cores), "
                                       f"extrapolated to {args.layers} layers; {n_time} steps timed "
                                       f"after {n_warm} warm-up steps"},
            "extrapolated": f"ms_per_step is the mean of {n_time} sampled steps (each one layer 0 plus one "
                            f"sparse layer scaled to {args.layers} layers); the wall time of this run is "
                            f"shorter than steps x ms_per_step",
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
