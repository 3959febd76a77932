"""Offloaded sparse layers with a double-buffered host-link gather.

The fp16 K and V of every offloaded layer live in pinned host memory
([heads][tokens][d], read by the GPU in place over the host link).  HBM keeps,
per layer, what selection needs -- the channel-major key copy and the running
max |K| per channel, the critical-key buffer of the TailorKV article (§2.3) --
and the rows that are always attended: the attention sinks and the recent
window (a ring of window/16 pages, token t in slot t mod window).  Each decode
step, per layer and head, the critical-channel scores pick the top-K tokens,
their K and V rows are gathered from host memory into one of two HBM staging
buffers, and exact attention runs over sinks + staged rows + window.  The
gather of layer l + 1 (into buffer B) overlaps the attention of layer l (on
buffer A), with an event handoff and the buffers flipped every layer: the
double buffer of the meeting article (§4.2: buffer A holds the current step,
buffer B is in flight), the prefetch while the previous layer computes of
TailorKV (§2.3, §3.2).

Host-side plumbing only: every step runs in libkvq's kernels (kv_critical_score,
kv_topk_select, kv_offload_gather, kv_sparse_attn); this module allocates the
buffers, builds the block tables and lists, and orders the launches on two
streams with events.  The attention reads the staged rows through a virtual
sequence: page 0 holds the sinks, pages 1 .. P the staged rows (list entry i in
page 1 + i / 16, slot i % 16), the last window/16 pages the window ring; its
list holds those positions, so the staged rows are attended in place.
"""
from __future__ import annotations

import math

import torch

from . import kvq
from ._abi import HEAD_DIM, Pool, check, lib

D = HEAD_DIM


class _View:
    """A kvq_layout + kvq_pool pair (what the binding's calls read as `cache`)."""

    def __init__(self, layout, pool):
        self.layout, self.c = layout, pool


class OffloadLayers:
    """Offloaded fp16 layers of one sequence (H heads, MHA) at context T, and the
    double-buffered decode step over them.

    layer_kv: one (K, V) pair of device fp16 [T][H][d] tensors per distinct
    layer; layer_of[l] names the distinct layer that layer l uses (several layers
    may share one, each with its own query).  The prompt is packed once (the
    channel-major key copy and max |K| in HBM, sinks and window into their
    resident pages) and copied to pinned host memory."""

    def __init__(self, H, T, layer_kv, layer_of, ratio=0.03, n_sink=4, window=128, n_crit=8, device="cuda"):
        assert window % 16 == 0 and window > 0 and 0 <= n_sink <= 16
        self.H, self.T, self.ratio, self.n_sink, self.window, self.n_crit = H, T, ratio, n_sink, window, n_crit
        self.layer_of = list(layer_of)
        self.L = len(self.layer_of)
        self.K = math.floor(ratio * T)
        assert T > n_sink + window + self.K, "the offloaded context must exceed sinks + window + top-K"
        self.sel_cap = n_sink + window + self.K
        self.P = -(-self.K // 16)                      # staging pages per buffer
        self.W = window // 16                          # window ring pages
        nres = len(layer_kv)
        self.res0 = 2 * self.P                         # first resident page
        n_pages = 2 * self.P + nres * (1 + self.W)
        self.layout = kvq.make_layout(H, H, 16)
        self.k16 = torch.zeros((n_pages, H, 16, D), dtype=torch.float16, device=device)
        self.v16 = torch.zeros_like(self.k16)
        self.t_cap = (T + 7) // 8 * 8
        self.host_k, self.host_v, self.kT, self.absmax = [], [], [], []
        n_tp = -(-T // 16)
        tmp = kvq.LayerCache(H, H, 16, n_tp, 1, t_cap=self.t_cap, device=device)  # prompt pages, reused
        ident = torch.arange(n_tp, dtype=torch.int32, device=device)[None]
        full = kvq.Batch(ident, torch.tensor([T], dtype=torch.int32, device=device), T)
        for j, (Kd, Vd) in enumerate(layer_kv):
            assert Kd.shape == (T, H, D) and Vd.shape == (T, H, D)
            tmp.kT.zero_()
            tmp.k_absmax.zero_()
            kvq.kv_quant_pack(tmp, full, 0, 0, T, Kd, Vd)
            torch.cuda.synchronize()
            self.kT.append(tmp.kT.clone())
            self.absmax.append(tmp.k_absmax.clone())
            # resident rows: sinks (page res + 0) and the window ring (token t at ring slot t mod window)
            base = self.res0 + j * (1 + self.W)
            self.k16[base, :, :16] = tmp.k16[0]
            self.v16[base, :, :16] = tmp.v16[0]
            t = torch.arange(T - window, T, device=device)
            ring = t % window
            self.k16[base + 1 + ring // 16, :, ring % 16] = tmp.k16[t // 16, :, t % 16]
            self.v16[base + 1 + ring // 16, :, ring % 16] = tmp.v16[t // 16, :, t % 16]
            self.host_k.append(Kd.permute(1, 0, 2).contiguous().cpu().pin_memory())
            self.host_v.append(Vd.permute(1, 0, 2).contiguous().cpu().pin_memory())
        del tmp
        # selection descriptors (the real sequence; its block table is not read by selection)
        self.sel_seqs = kvq.Batch(ident, torch.tensor([T], dtype=torch.int32, device=device), T)
        self.sel_views = [_View(self.layout, Pool(n_tp, 1, self.t_cap, None, None, None, None, None, None, None,
                                                  self.kT[j].data_ptr(), self.absmax[j].data_ptr()))
                          for j in range(nres)]
        # attention descriptors: one virtual sequence per (distinct layer, buffer)
        self.att_view = _View(self.layout, Pool(n_pages, 1, 0, None, None, None, None, None, self.k16.data_ptr(),
                                                self.v16.data_ptr(), None, None))
        vlen = 16 * (1 + self.P + self.W)
        self.att_seqs = {}
        for j in range(nres):
            base = self.res0 + j * (1 + self.W)
            for b in range(2):
                row = [base] + list(range(b * self.P, (b + 1) * self.P)) + list(range(base + 1, base + 1 + self.W))
                self.att_seqs[j, b] = kvq.Batch(torch.tensor([row], dtype=torch.int32, device=device),
                                                torch.tensor([vlen], dtype=torch.int32, device=device), vlen)
        ids = list(range(n_sink)) + [16 + i for i in range(self.K)] + \
            [16 * (1 + self.P) + r for r in range(window)]
        self.vlist = torch.tensor(ids, dtype=torch.int32, device=device).repeat(1, H, 1).contiguous()
        self.vcount = torch.full((1, H), len(ids), dtype=torch.int32, device=device)
        self.gcount = torch.full((H,), self.K, dtype=torch.int32, device=device)
        # per-buffer selection state (the selection of a layer feeds only its own gather)
        self.scores = [torch.empty((1, H, self.t_cap), device=device) for _ in range(2)]
        self.sel = [torch.empty((1, H, self.sel_cap), dtype=torch.int32, device=device) for _ in range(2)]
        self.cnt = [torch.empty((1, H), dtype=torch.int32, device=device) for _ in range(2)]
        self.ws_sel = [kvq.Workspace(kvq.kv_topk_select_ws(), device) for _ in range(2)]
        self.ws_g = [kvq.Workspace(kvq.kv_offload_gather_ws(), device) for _ in range(2)]
        self.ws_a = kvq.Workspace(kvq.kv_sparse_attn_ws(self.att_view, self.att_seqs[0, 0], self.sel_cap), device)
        self.ev_selected = [torch.cuda.Event() for _ in range(2)]
        self.ev_gathered = [torch.cuda.Event() for _ in range(2)]
        self.ev_attended = [torch.cuda.Event() for _ in range(2)]

    # ---- the three stages of one layer

    def select(self, l, q, b, stream):
        """Critical-channel scores and top-K of layer l (query q [1][H][d]) into buffer b's list."""
        j = self.layer_of[l]
        kvq.kv_critical_score(self.sel_views[j], self.sel_seqs, q, self.n_crit, None, self.scores[b], stream=stream)
        kvq.kv_topk_select(self.sel_seqs, self.H, self.scores[b], -1, self.ratio, self.n_sink, self.window,
                           self.sel[b], self.cnt[b], self.ws_sel[b], stream=stream)

    def gather(self, l, b, stream):
        """The listed top-K rows of layer l (the list entries after the sinks, before the
        window: the selection is ascending) from host memory into staging buffer b."""
        j = self.layer_of[l]
        page = self.H * 16 * D * 2
        off = b * self.P * page
        check(lib().kv_offload_gather(self.host_k[j].data_ptr(), self.host_v[j].data_ptr(), self.T * D, self.T,
                                      self.H, self.sel[b].data_ptr() + 4 * self.n_sink, self.sel_cap,
                                      self.gcount.data_ptr(), self.k16.data_ptr() + off, self.v16.data_ptr() + off,
                                      self.ws_g[b].ptr, self.ws_g[b].nbytes, kvq._s(stream)), "kv_offload_gather")

    def attend(self, l, q, out, b, stream):
        """Exact attention of layer l over sinks + staged rows (buffer b) + window."""
        kvq.kv_sparse_attn(self.att_view, self.att_seqs[self.layer_of[l], b], q, self.vlist, self.vcount, 0, out,
                           None, self.ws_a, stream=stream)

    # ---- one decode step over all layers

    def step(self, qs, outs, copy_stream, attn_stream):
        """Layers 0 .. L-1 with queries qs[l] into outs[l].  The host-link gathers run back to
        back on copy_stream (layer l into buffer l % 2); the GPU work runs on attn_stream, the
        selection of layer l + 1 ahead of the attention of layer l, so that neither waits on
        the other's stream more than the data requires: gather l needs selection l, and
        buffer l % 2 is refilled (gather l + 2) only after attention l has read it.  Waits
        are stream/event ordering only.  Both streams start after the work already queued on
        attn_stream; attn_stream ends after the last attention."""
        start = torch.cuda.Event()
        start.record(attn_stream)
        copy_stream.wait_event(start)

        def select_and_gather(l):
            b = l % 2
            # sel[b] was last read by gather l - 2, which attention l - 2 (earlier on attn_stream) waited for
            self.select(l, qs[l], b, attn_stream)
            self.ev_selected[b].record(attn_stream)
            copy_stream.wait_event(self.ev_selected[b])
            if l >= 2:
                copy_stream.wait_event(self.ev_attended[b])
            self.gather(l, b, copy_stream)
            self.ev_gathered[b].record(copy_stream)
        select_and_gather(0)
        for l in range(self.L):
            b = l % 2
            if l + 1 < self.L:
                select_and_gather(l + 1)
            attn_stream.wait_event(self.ev_gathered[b])
            self.attend(l, qs[l], outs[l], b, attn_stream)
            self.ev_attended[b].record(attn_stream)
        copy_stream.wait_stream(attn_stream)

    def check(self):
        for w in self.ws_sel + self.ws_g + [self.ws_a]:
            kvq.kvq_check(w)

    @property
    def gather_bytes_per_layer(self):
        """Bytes one layer moves over the host link: K and V rows of the top-K per head."""
        return self.H * self.K * 2 * D * 2
