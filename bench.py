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
  python bench.py --rows    # the other rows (pack, INT4 batch attention, H2O step, offload
                            # gather, tiny-config kernels), one JSON line each

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
                    help="instead of the step: time the other hot-path rows on their configurations, one JSON line each")
    args = ap.parse_args()
    if args.rows:
        run_rows(args)
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
               "sample": f"layer 0 (1-bit quantized, 8 kv-head tasks) and one sparse layer (32 q-head "
                         f"tasks) of a {args.prompt}-token step on a {n_workers}-process pool (the host's "
                         f"{os.cpu_count()} cores); step time = t0 + {args.layers - 1} x t_sparse = "
                         f"{t0c:.2f} s + {args.layers - 1} x {t1c:.2f} s"}

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


# ------------------------------------------------------------------------ per-row measurements (--rows)
#
# The hot-path rows outside the headline step, each timed on its configuration with CUDA
# events on the launching stream (inputs larger than L2 where the row streams memory), next
# to a bounded single-threaded sample of the oracle doing the same work.

def _ev_ms(torch, fn, stream, reps, warm=2):
    torch.cuda.synchronize()  # inputs made on other streams are complete
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / reps


def _wall(fn):
    t = time.perf_counter()
    fn()
    return time.perf_counter() - t


def _paged(torch, kvq, lengths, device, seed):
    """Block table over a shuffled allocator, one row per sequence."""
    pages = [-(-int(T) // 16) for T in lengths]
    alloc = kvq.Allocator(sum(pages) + 4, seed=seed)
    mb = max(pages)
    bt = torch.full((len(lengths), mb), -1, dtype=torch.int32)
    for b, n in enumerate(pages):
        bt[b, :n] = torch.tensor(alloc.alloc(n), dtype=torch.int32)
    seqs = kvq.Batch(bt.to(device), torch.tensor([int(T) for T in lengths], dtype=torch.int32, device=device),
                     max(int(T) for T in lengths))
    return seqs, sum(pages) + 4, alloc


def _row_line(row, config, value, unit, roof, cpu, extra=None):
    line = {"row": row, "config": config, "value": value, "unit": unit, "roofline": roof, "cpu_baseline": cpu}
    if extra:
        line.update(extra)
    print(json.dumps(line), flush=True)


def run_rows(args):
    import numpy as np
    import torch

    from compressed_kv_cache_quant_gb300 import kvq, synth
    from compressed_kv_cache_quant_gb300.build import build
    from oracle import kvq_oracle as O
    build()
    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device)
    sh = stream.cuda_stream
    peak, peak_src = measured_peaks()
    seed = synth.BASE_SEED

    def hbm(achieved):
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": peak_src}

    # a1 kv_quant_pack: one Qwen-1.5-14B-shaped layer, 40 kv heads x 131072 tokens, 1-bit, G 64
    try:
        T, H = args.prompt, 40
        seqs, npg, _ = _paged(torch, kvq, [T], device, 3)
        cache = kvq.LayerCache(H, H, 1, npg, 1, v_group_dims=64)
        K, V = synth.kv_rows(T, H, synth.mix(seed + 5, 1), device=device)
        ms = _ev_ms(torch, lambda: kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V, stream=sh), stream, 5)
        nbytes = 2 * T * H * D * 2 + T * H * 48
        k1, v1 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
        del K, V, cache
        t = _wall(lambda: (O.pack_k(k1, 1), O.pack_v(v1, 1, 64)))
        cpu_gbs = (T * D * 2 * 2 + T * 48) / t / 1e9
        _row_line("a1 kv_quant_pack", f"40 kv heads x {T} tokens, 1-bit, K g64 / V G64 (one layer)",
                  nbytes / (ms * 1e-3) / 1e9, "GB/s", hbm(nbytes / (ms * 1e-3) / 1e9),
                  {"value": cpu_gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": f"one kv head of the layer ({T} tokens), numpy"}, {"ms": ms, "bytes": nbytes})
    except Exception as e:  # report and go on with the other rows
        print(json.dumps({"row": "a1 kv_quant_pack", "error": repr(e)}), flush=True)
    torch.cuda.empty_cache()

    # a3 kv_decode_attn_quant, INT4 serving batch: 16 sequences, lengths U[4096, 32768], 32 heads MHA,
    # K 4-bit g64, V 4-bit G 32; one layer
    try:
        B, H = 16, 32
        lens = [int(x) for x in synth.lengths_uniform(B, 4096, 32768, seed + 2)]
        seqs, npg, _ = _paged(torch, kvq, lens, device, 7)
        cache = kvq.LayerCache(H, H, 4, npg, B, v_group_dims=32)
        for b, T in enumerate(lens):
            K, V = synth.kv_rows(T, H, synth.mix(seed + 2, 10 + b), device=device)
            kvq.kv_quant_pack(cache, seqs, b, 0, T, K, V)  # same stream as K, V
            if b == 0:
                k0, v0 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
            del K, V
        stream.synchronize()
        q = synth.normal((B, H, D), synth.mix(seed + 2, 99), device)
        out = torch.empty((B, H, D), device=device)
        wsq = kvq.Workspace(kvq.kv_decode_attn_quant_ws(cache, seqs))
        ms = _ev_ms(torch, lambda: kvq.kv_decode_attn_quant(cache, seqs, q, out, wsq, stream=sh), stream, 20)
        kvq.kvq_check(wsq, stream=sh)
        nbytes = sum(lens) * H * 152
        pk, pv = O.pack_k(k0, 4), O.pack_v(v0, 4, 32)
        q0 = q[0, :1].cpu().numpy()
        t = _wall(lambda: O.decode_attn_quant(q0, [pk], [pv]))
        cpu_gbs = lens[0] * 152 / t / 1e9
        _row_line("a3 kv_decode_attn_quant (INT4 batch)",
                  f"16 sequences, T ~ U[4096, 32768] (sum {sum(lens)}), 32 heads MHA, K 4-bit g64, V 4-bit G32",
                  nbytes / (ms * 1e-3) / 1e9, "GB/s", hbm(nbytes / (ms * 1e-3) / 1e9),
                  {"value": cpu_gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": f"one (sequence, head) of {lens[0]} tokens, numpy fp64"}, {"ms": ms, "bytes": nbytes})
        del cache
    except Exception as e:
        print(json.dumps({"row": "a3 kv_decode_attn_quant (INT4 batch)", "error": repr(e)}), flush=True)
    torch.cuda.empty_cache()

    # a6 + a7: H2O layer step: attention over the retained set (shared per kv head, probabilities
    # out), then accumulate and evict; 8 sequences x 8 kv heads, T = 32768, budget 6553
    try:
        B, Hq, Hkv, T, budget, ns, w = 8, 32, 8, 32768, 6553, 4, 2048
        G = Hq // Hkv
        seqs, npg, _ = _paged(torch, kvq, [T] * B, device, 11)
        cache = kvq.LayerCache(Hq, Hkv, 16, npg, B, t_cap=T)
        rng = np.random.default_rng(5)
        cap = budget + 2
        ret = np.zeros((B, Hkv, cap), np.int32)
        for b in range(B):
            K, V = synth.kv_rows(T, Hkv, synth.mix(seed + 4, b), device=device)
            kvq.kv_quant_pack(cache, seqs, b, 0, T, K, V)  # same stream as K, V
            if b == 0:
                k0, v0 = K[:, 0].cpu().numpy(), V[:, 0].cpu().numpy()
            del K, V
            for g in range(Hkv):
                mid = rng.choice(np.arange(ns, T - w), size=budget - ns - w, replace=False)
                ret[b, g, :budget] = rng.permutation(np.concatenate([np.arange(ns), mid, np.arange(T - w, T)]))
        stream.synchronize()
        retained = torch.from_numpy(ret).to(device)
        counts = torch.full((B, Hkv), budget, dtype=torch.int32, device=device)
        cum = torch.from_numpy(rng.random((B, Hkv, cap)).astype(np.float32)).to(device)
        probs = torch.zeros((B, Hq, cap), device=device)
        q = synth.normal((B, Hq, D), synth.mix(seed + 4, 99), device)
        out = torch.empty((B, Hq, D), device=device)
        wsa = kvq.Workspace(kvq.kv_sparse_attn_ws(cache, seqs, cap))
        wsh = kvq.Workspace(kvq.kv_h2o_accumulate_ws())

        def h2o_step():
            kvq.kv_sparse_attn(cache, seqs, q, retained, counts, 1, out, probs, wsa, stream=sh)
            kvq.kv_h2o_accumulate(cache, seqs, probs, retained, counts, cum, budget, ns, w, None, None, wsh,
                                  stream=sh)
        ms = _ev_ms(torch, h2o_step, stream, 20)
        ms_attn = _ev_ms(torch, lambda: kvq.kv_sparse_attn(cache, seqs, q, retained, counts, 1, out, probs, wsa,
                                                           stream=sh), stream, 20)
        kvq.kvq_check(wsa, stream=sh)
        kvq.kvq_check(wsh, stream=sh)
        nbytes = B * Hkv * budget * 2 * D * 2 + B * Hkv * cap * 8 + B * Hq * cap * 4
        r0 = ret[0, 0, :budget].copy()
        qg = q[0, :G].cpu().numpy()
        t = _wall(lambda: O.h2o_step(qg, k0, v0, r0, np.zeros(budget), T - 1, budget, ns, w))
        cpu_ms = t * 1e3 * B * Hkv
        _row_line("a6+a7 kv_sparse_attn + kv_h2o_accumulate (H2O layer step)",
                  f"8 sequences x 8 kv heads (GQA 4), T = {T}, budget {budget} = {ns} + {w} + {budget - ns - w}",
                  nbytes / (ms * 1e-3) / 1e9, "GB/s", hbm(nbytes / (ms * 1e-3) / 1e9),
                  {"value": cpu_ms, "unit": "ms per layer step", "cores": 1, "kind": "oracle",
                   "sample": "one (sequence, kv head) of the step, numpy fp64, times 64"},
                  {"ms": ms, "ms_sparse_attn_only": ms_attn, "bytes": nbytes})
        del cache
    except Exception as e:
        print(json.dumps({"row": "a6+a7 H2O layer step", "error": repr(e)}), flush=True)
    torch.cuda.empty_cache()

    # f1 block-granular selection (block pruning in 64-token blocks) next to the token top-K on one
    # Llama-3.1-8B-shaped sparse layer: selection over the critical-channel scores + exact attention
    try:
        Hq, Hkv, T, ns, w, blk = 32, 8, args.prompt, 4, 128, 64
        seqs, npg, _ = _paged(torch, kvq, [T], device, 13)
        cache = kvq.LayerCache(Hq, Hkv, 16, npg, 1, t_cap=(T + 7) // 8 * 8)
        K, V = synth.kv_rows(T, Hkv, synth.mix(seed + 6, 0), device=device)
        kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)  # same stream as K, V
        del K, V
        q = synth.normal((1, Hq, D), synth.mix(seed + 6, 1), device)
        sc = torch.empty((1, Hq, (T + 7) // 8 * 8), device=device)
        crit = torch.empty((1, Hq, 8), dtype=torch.int32, device=device)
        kvq.kv_critical_score(cache, seqs, q, 8, crit, sc)
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
        sel_tok = lambda: kvq.kv_topk_select(seqs, Hq, sc, -1, RATIO, ns, w, sel_t, cnt_t, wt, stream=sh)
        sel_blk = lambda: kvq.kv_block_select(seqs, Hq, sc, -1, RATIO, ns, w, blk, sel_b, cnt_b, wb, stream=sh)
        att_tok = lambda: kvq.kv_sparse_attn(cache, seqs, q, sel_t, cnt_t, 0, out, None, wa, stream=sh)
        att_blk = lambda: kvq.kv_sparse_attn(cache, seqs, q, sel_b, cnt_b, 0, out, None, wa, stream=sh)
        ms_tok = _ev_ms(torch, lambda: (sel_tok(), att_tok()), stream, 20)
        ms_blk = _ev_ms(torch, lambda: (sel_blk(), att_blk()), stream, 20)
        ms_att_tok = _ev_ms(torch, att_tok, stream, 20)
        ms_att_blk = _ev_ms(torch, att_blk, stream, 20)
        for wk in (wt, wb, wa):
            kvq.kvq_check(wk, stream=sh)
        rows_t, rows_b = int(cnt_t.sum().item()), int(cnt_b.sum().item())
        by_t, by_b = Hq * T * 4 + rows_t * 2 * D * 2, Hq * T * 4 + rows_b * 2 * D * 2
        s0 = sc[0, 0, :T].cpu().numpy()
        t = _wall(lambda: O.block_select(s0, nb, ns, w, blk))
        _row_line("f1 kv_block_select + kv_sparse_attn (block-sparse layer)",
                  f"32 q / 8 kv heads, T = {T}, ratio {RATIO}: {nb} blocks of {blk} + {ns} sinks + {w} window "
                  f"per q head (token top-K: {kt})",
                  by_b / (ms_blk * 1e-3) / 1e9, "GB/s", hbm(by_b / (ms_blk * 1e-3) / 1e9),
                  {"value": t * 1e3 * Hq, "unit": "ms per layer (selection only)", "cores": 1, "kind": "oracle",
                   "sample": "block selection of one q head, numpy, times 32"},
                  {"ms_block_path": ms_blk, "ms_token_path": ms_tok, "ms_attn_block_lists": ms_att_blk,
                   "ms_attn_token_lists": ms_att_tok, "token_path_GBps": by_t / (ms_tok * 1e-3) / 1e9,
                   "rows_block": rows_b, "rows_token": rows_t, "bytes": by_b})
        del cache
    except Exception as e:
        print(json.dumps({"row": "f1 block-sparse layer", "error": repr(e)}), flush=True)
    torch.cuda.empty_cache()

    # a9 kv_offload_gather: 40 heads x 3932 selected rows of 131072 from pinned host memory
    try:
        T, H, sel_n = args.prompt, 40, math.floor(RATIO * args.prompt)
        K, V = synth.kv_rows(T, H, synth.mix(seed + 5, 2), n_out=0)
        src_k = K.permute(1, 0, 2).contiguous().pin_memory()
        src_v = V.permute(1, 0, 2).contiguous().pin_memory()
        del K, V
        rng = np.random.default_rng(9)
        sel = np.stack([np.sort(rng.choice(T, size=sel_n, replace=False)) for _ in range(H)]).astype(np.int32)
        sel_t = torch.from_numpy(sel).to(device)
        cnt = torch.full((H,), sel_n, dtype=torch.int32, device=device)
        npg = -(-sel_n // 16)
        dk = torch.empty((npg, H, 16, D), dtype=torch.float16, device=device)
        dv = torch.empty_like(dk)
        wg = kvq.Workspace(kvq.kv_offload_gather_ws())
        ms = _ev_ms(torch, lambda: kvq.kv_offload_gather(src_k.data_ptr(), src_v.data_ptr(), T * D, T, H, sel_t, cnt,
                                                        dk, dv, wg, stream=sh), stream, 10)
        kvq.kvq_check(wg, stream=sh)
        nbytes = H * sel_n * 2 * D * 2
        # the link's roofline: one contiguous pinned -> device copy of the same size
        hsrc = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        ddst = torch.empty(nbytes, dtype=torch.uint8, device=device)
        ms_copy = _ev_ms(torch, lambda: ddst.copy_(hsrc, non_blocking=True), stream, 10)
        link = nbytes / (ms_copy * 1e-3) / 1e9
        k0 = src_k[0].numpy()
        t = _wall(lambda: O.offload_gather(k0, sel[0]))
        cpu_gbs = sel_n * D * 2 / t / 1e9
        ach = nbytes / (ms * 1e-3) / 1e9
        _row_line("a9 kv_offload_gather", f"40 heads x {sel_n} of {T} fp16 K and V rows from pinned host memory",
                  ach, "GB/s", {"bound": "host link", "achieved": ach, "peak": link, "unit": "GB/s",
                                "frac": ach / link, "peak_source": "measured pinned->device cudaMemcpyAsync, same bytes"},
                  {"value": cpu_gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": "one head's K rows, numpy fancy indexing (host to host)"}, {"ms": ms, "bytes": nbytes})
        del src_k, src_v, hsrc, ddst
    except Exception as e:
        print(json.dumps({"row": "a9 kv_offload_gather", "error": repr(e)}), flush=True)
    torch.cuda.empty_cache()

    # a4, a5, a6, a8 at the tiny configuration: 8 q / 2 kv heads, T = 4096 (latency-bound; microseconds)
    try:
        Hq, Hkv, T, ncrit, kk, ns, w = 8, 2, 4096, 8, 128, 4, 64
        seqs, npg, _ = _paged(torch, kvq, [T], device, 13)
        cache = kvq.LayerCache(Hq, Hkv, 16, npg, 1, t_cap=T)
        K, V = synth.kv_rows(T, Hkv, synth.mix(seed, 1), device=device)
        kvq.kv_quant_pack(cache, seqs, 0, 0, T, K, V)
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
        us = {
            "a4 kv_critical_score": 1e3 * _ev_ms(torch, lambda: kvq.kv_critical_score(cache, seqs, q, ncrit, crit, scores,
                                                                                     stream=sh), stream, 50),
            "a5 kv_topk_select": 1e3 * _ev_ms(torch, lambda: kvq.kv_topk_select(seqs, Hq, scores, kk, 0.0, ns, w, sel,
                                                                               cnt, wt, stream=sh), stream, 50),
            "a6 kv_sparse_attn": 1e3 * _ev_ms(torch, lambda: kvq.kv_sparse_attn(cache, seqs, q, sel, cnt, 0, out, probs,
                                                                               wa, stream=sh), stream, 50),
            "a8 kv_dense_pref_score": 1e3 * _ev_ms(torch, lambda: kvq.kv_dense_pref_score(cache, seqs, Q, 32, 128, P, wd,
                                                                                         stream=sh), stream, 20),
        }
        for wsx in (wt, wa, wd):
            kvq.kvq_check(wsx, stream=sh)
        Kc, Vc = K.cpu().numpy(), V.cpu().numpy()
        qn, Qn = q.cpu().numpy()[0], Q.cpu().numpy()[0]
        am = [O.key_absmax(Kc[:, g]) for g in range(Hkv)]
        chans = [O.critical_channels(qn[h], am[O.kv_head_of(h, Hq, Hkv)], ncrit) for h in range(Hq)]
        sc = []
        cpu = {
            "a4 kv_critical_score": _wall(lambda: sc.extend(O.critical_scores(qn[h], Kc[:, O.kv_head_of(h, Hq, Hkv)],
                                                                              chans[h]) for h in range(Hq))),
            "a5 kv_topk_select": _wall(lambda: [O.topk_select(sc[h], kk, ns, w) for h in range(Hq)]),
            "a6 kv_sparse_attn": _wall(lambda: [O.sparse_attn(qn[h], Kc[:, O.kv_head_of(h, Hq, Hkv)],
                                                              Vc[:, O.kv_head_of(h, Hq, Hkv)],
                                                              O.topk_select(sc[h], kk, ns, w)) for h in range(Hq)]),
            "a8 kv_dense_pref_score": _wall(lambda: [O.dense_pref_score(Qn[h], Kc[:, O.kv_head_of(h, Hq, Hkv)], 128)
                                                     for h in range(Hq)]),
        }
        for name, v in us.items():
            _row_line(name, "8 q / 2 kv heads, T = 4096 (8 critical channels, K = 128 + 4 sinks + 64 window; "
                            "dense preference over 32 recent queries, top-128)", v, "us",
                      {"bound": "latency", "note": "tiny parity configuration: microseconds, no roofline target"},
                      {"value": cpu[name] * 1e6, "unit": "us", "cores": 1, "kind": "oracle",
                       "sample": "the same call on the CPU oracle, numpy"})
    except Exception as e:
        print(json.dumps({"row": "a4/a5/a6/a8 tiny", "error": repr(e)}), flush=True)


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
