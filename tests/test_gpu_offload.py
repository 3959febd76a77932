"""GPU parity of the offloaded sparse layers (the Qwen-1.5-14B-shaped offload
configuration at reduced size): fp16 K/V in pinned host memory, critical keys,
sinks and window in HBM, a double-buffered decode step that gathers layer
l + 1's top-K rows over the host link while layer l attends.  The staged rows
equal the host rows byte for byte, and every layer's attention equals the
oracle's exact attention over sinks + top-K + window.
Sources: meeting article §4.2 (double buffer); TailorKV §2.3, §3.2, §5.1."""
import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import synth
from compressed_kv_cache_quant_gb300.offload import OffloadLayers
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,T,layer_of", [(4, 4096 + 37, [0, 1, 0, 1, 0]),   # two distinct layers, five steps
                                          (40, 6000, [0, 1, 2])])             # 40 MHA heads
def test_offload_pipeline_matches_oracle(H, T, layer_of):
    require_gpu()
    seed = synth.mix(synth.BASE_SEED + 4, 500, H, T)
    n_res = max(layer_of) + 1
    KV = [synth.kv_rows(T, H, synth.mix(seed, j), device="cuda") for j in range(n_res)]
    off = OffloadLayers(H, T, KV, layer_of)
    L = len(layer_of)
    qs = synth.queries((L, 1, H, 128), synth.mix(seed, 99)).cuda()
    outs = torch.full((L, 1, H, 128), float("nan"), device="cuda")
    cs, at = torch.cuda.Stream(), torch.cuda.Stream()
    at.wait_stream(torch.cuda.current_stream())
    off.step(qs, outs, cs, at)
    at.synchronize()
    cs.synchronize()
    off.check()
    o = outs.cpu().numpy()
    Kh = [k.cpu().numpy() for k, _ in KV]
    Vh = [v.cpu().numpy() for _, v in KV]
    k = O.ratio_k(T, 0.03)
    ids_of = {}
    for l, j in enumerate(layer_of):
        for h in range(H):
            q = qs[l, 0, h].cpu().numpy()
            C = O.critical_channels(q, O.key_absmax(Kh[j][:, h]), 8)
            ids = O.topk_select(O.critical_scores(q, Kh[j][:, h], C), k, 4, 128)
            ids_of[l, h] = ids
            ref, _ = O.sparse_attn(q, Kh[j][:, h], Vh[j][:, h], ids)
            e = attn_err(o[l, 0, h], ref)
            assert e <= ATTN_TOL, (l, h, e)
    # the two staging buffers hold the last two layers' top-K rows, byte for byte
    k16, v16 = off.k16.cpu().numpy(), off.v16.cpu().numpy()
    for l in (L - 2, L - 1):
        b, j = l % 2, layer_of[l]
        for h in range(H):
            top = ids_of[l, h][4:4 + k]
            staged_k = np.stack([k16[b * off.P + i // 16, h, i % 16] for i in range(k)])
            staged_v = np.stack([v16[b * off.P + i // 16, h, i % 16] for i in range(k)])
            assert np.array_equal(staged_k.view(np.uint16), O.offload_gather(Kh[j][:, h], top).view(np.uint16))
            assert np.array_equal(staged_v.view(np.uint16), O.offload_gather(Vh[j][:, h], top).view(np.uint16))
