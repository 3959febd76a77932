"""GPU parity of f3, outlier-channel isolation of the keys [meeting article §8.2],
against the oracle:
  - channel variances bit-exact (exact integer sums on both sides) and the chosen
    channels exact, including ties, mixed magnitudes and a strided input;
  - the isolated cache after prefill and after appends across 64-token group
    boundaries: codes (bit-exact up to the documented rounding near-ties), scales
    and zeros bit-exact, outlier channels zero in the main cache, their fp16 keys
    exact in the side cache;
  - the outlier attention within the attention tolerance of the oracle's attention
    over the isolated cache, and visibly different from attending the main cache
    alone (the outlier term is really added)."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws
from kvq_format import quant_logical
from test_gpu_pack import assert_codes

pytestmark = pytest.mark.gpu


def _gpu_channels(layout, K, n_out, stride_pad=0):
    """kv_outlier_channels of fp16 K [T][H][d] (CPU tensor): (channels [H][n_out], var [H][d])."""
    T, H, d = K.shape
    buf = torch.zeros((max(T, 1), H * d + stride_pad), dtype=torch.float16)
    buf[:T, :H * d] = K.reshape(T, H * d)
    kd = buf.cuda()
    ch = torch.full((H, n_out), -1, dtype=torch.int32, device="cuda")
    var = torch.full((H, d), float("nan"), dtype=torch.float64, device="cuda")
    w = ws(kvq.kv_outlier_channels_ws(layout))
    kvq.kv_outlier_channels(layout, kd, T, n_out, ch, w, var=var, stride_t=H * d + stride_pad)
    # the workspace is left zeroed: a second call gives the same answer
    ch2 = torch.empty_like(ch)
    kvq.kv_outlier_channels(layout, kd, T, n_out, ch2, w, stride_t=H * d + stride_pad)
    torch.cuda.synchronize()
    assert torch.equal(ch, ch2)
    return ch.cpu().numpy(), var.cpu().numpy()


@pytest.mark.parametrize("T,n_out,pad", [(0, 1, 0), (1, 2, 0), (1000, 1, 64), (4133, 4, 0), (70001, 8, 8)])
def test_outlier_channels_bitexact(T, n_out, pad):
    require_gpu()
    H = 4
    K, _ = synth.kv_rows(max(T, 1), H, synth.mix(synth.BASE_SEED, 501, T))
    K = K[:T].clone()
    if T > 7:
        K[::7, 0, 5] = 300.0                 # tiny and large values in one channel
        K[:, 1, 11] = K[:, 1, 9]             # equal variances: the lower channel ranks first
        K[:, 2, 3] = 1e-4                    # constant channel: variance 0
    layout = kvq.make_layout(H, H, 4)
    ch, var = _gpu_channels(layout, K, n_out, pad)
    Kn = K.numpy()
    for h in range(H):
        ref = O.channel_variance(Kn[:, h]) if T else np.zeros(128)
        assert np.array_equal(var[h].view(np.uint64), ref.view(np.uint64)), h
        want = O.outlier_channels(Kn[:, h], n_out) if T else np.arange(n_out)
        assert ch[h].tolist() == list(want), (h, ch[h], want)


def _isolated_batch(bits, G, Hq, Hkv, prompt, total, n_out, seed):
    """Sequences with `prompt[b]` tokens packed, channels chosen from the prompt and isolated, then
    appended one token at a time up to `total[b]` (each append followed by kv_outlier_append).
    Returns (cache, batch, bt, KV, out_ch, k_out)."""
    B = len(prompt)
    KV = [synth.kv_rows(max(total[b], 1), Hkv, synth.mix(seed, b)) for b in range(B)]
    n_pages = sum(math.ceil(max(t, 1) / 16) for t in total) + 4
    alloc = kvq.Allocator(n_pages, seed=seed % 997 + 1)
    batch, bt = paged_batch([max(t, 1) for t in total], alloc, lengths=prompt)
    cache = kvq.LayerCache(Hq, Hkv, bits, n_pages, B, v_group_dims=G)
    out_ch = torch.zeros((B, Hkv, n_out), dtype=torch.int32, device="cuda")
    k_out = torch.full((n_pages, Hkv, 16, n_out), float("nan"), dtype=torch.float16, device="cuda")
    wc = ws(kvq.kv_outlier_channels_ws(cache))
    for b in range(B):
        T0 = prompt[b]
        if T0 == 0:
            continue
        kd = KV[b][0][:T0].cuda()
        kvq.kv_quant_pack(cache, batch, b, 0, T0, kd, KV[b][1][:T0].cuda())
        kvq.kv_outlier_channels(cache, kd, T0, n_out, out_ch[b], wc)
        kvq.kv_outlier_isolate(cache, batch, b, 0, T0, kd, n_out, out_ch, k_out)
    n_app = max(t - p for t, p in zip(total, prompt))
    if n_app:
        assert all(t - p == n_app for t, p in zip(total, prompt))
        wa, wo = ws(kvq.kv_page_append_ws()), ws(kvq.kv_outlier_append_ws())
        for i in range(n_app):
            kvq.kvq_seq_lens_add(batch.seq_lens, 1)
            kn = torch.stack([KV[b][0][prompt[b] + i] for b in range(B)]).cuda()
            vn = torch.stack([KV[b][1][prompt[b] + i] for b in range(B)]).cuda()
            kvq.kv_page_append(cache, batch, kn, vn, wa)
            kvq.kv_outlier_append(cache, batch, n_out, out_ch, k_out, wo)
        kvq.kvq_check(wa)
        kvq.kvq_check(wo)
    torch.cuda.synchronize()
    return cache, batch, bt, KV, out_ch.cpu().numpy(), k_out


@pytest.mark.parametrize("bits,G,n_out", [(4, 32, 1), (8, 128, 4), (4, 64, 8)])
def test_isolated_cache_prefill_and_append(bits, G, n_out):
    require_gpu()
    H = 2
    prompt, n_app = [1000, 64, 37, 128], 100
    total = [p + n_app for p in prompt]
    cache, batch, bt, KV, out_ch, k_out = _isolated_batch(bits, G, 4, H, prompt, total, n_out,
                                                          synth.mix(synth.BASE_SEED, 502, bits, n_out))
    cnp = {n: getattr(cache, n).cpu().numpy() for n in ("k_codes", "v_codes", "k_sz", "v_sz", "k_tail")}
    ko = k_out.cpu().numpy()
    for b, T in enumerate(total):
        K = KV[b][0].numpy()
        sub = dict(cnp)
        sub["k_tail"] = cnp["k_tail"][b:b + 1]
        for h in range(H):
            ch = O.outlier_channels(K[:prompt[b], h], n_out)
            assert out_ch[b, h].tolist() == ch.tolist()
            po = O.pack_k_outlier(K[:, h], bits, ch)
            lg = quant_logical(sub, bt[b], T, h, bits, G)
            n = po["n_packed"]
            assert np.all(lg["k_codes"][:, ch] == 0)
            assert_codes(lg["k_codes"], po["codes"], K[:n, h], np.where(po["scale32"] > 0, po["scale32"], 1),
                         po["zero16"].astype(np.float32), lambda i: (i[0] // 64, i[1]))
            assert np.array_equal(lg["k_scale16"].view(np.uint16), po["scale16"].view(np.uint16))
            assert np.array_equal(lg["k_zero16"].view(np.uint16), po["zero16"].view(np.uint16))
            side = np.stack([ko[int(bt[b][t // 16]), h, t % 16] for t in range(n)]) if n else np.zeros((0, n_out))
            assert np.array_equal(side.view(np.uint16), po["outlier_values"].view(np.uint16))
            nt = T - n
            assert np.array_equal(sub["k_tail"][0, h, :nt].view(np.uint16), po["tail"].view(np.uint16))


def _attend(bits, G, Hq, Hkv, prompt, total, n_out, seed):
    cache, batch, bt, KV, out_ch, k_out = _isolated_batch(bits, G, Hq, Hkv, prompt, total, n_out, seed)
    B = len(total)
    q = synth.queries((B, Hq, 128), synth.mix(seed, 99))
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    w = ws(kvq.kv_decode_attn_quant_ws(cache, batch))
    och = torch.from_numpy(out_ch).cuda()
    kvq.kv_decode_attn_quant_outlier(cache, batch, q.cuda(), n_out, och, k_out, out, w)
    kvq.kvq_check(w)
    plain = torch.empty_like(out)
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), plain, w)
    torch.cuda.synchronize()
    o, o_plain = out.cpu().numpy(), plain.cpu().numpy()
    worst_plain = 0.0
    for b, T in enumerate(total):
        if T == 0:
            assert np.all(o[b] == 0)
            continue
        K, V = KV[b][0][:T].numpy(), KV[b][1][:T].numpy()
        pk = [O.pack_k_outlier(K[:, g], bits, O.outlier_channels(K[:prompt[b], g], n_out)) for g in range(Hkv)]
        pv = [O.pack_v(V[:, g], bits, G) for g in range(Hkv)]
        ref = O.decode_attn_quant(q[b].numpy(), pk, pv)
        for h in range(Hq):
            e = attn_err(o[b, h], ref[h])
            assert e <= ATTN_TOL, (b, h, T, e)
            if T >= 64:
                worst_plain = max(worst_plain, attn_err(o_plain[b, h], ref[h]))
    return worst_plain


@pytest.mark.parametrize("bits,G,Hq,Hkv,n_out", [(4, 32, 8, 2, 1), (4, 64, 8, 8, 4), (8, 128, 16, 2, 8),
                                                  (4, 128, 32, 4, 2)])
def test_outlier_attention_matches_oracle(bits, G, Hq, Hkv, n_out):
    require_gpu()
    prompt = [1, 63, 64, 65, 1000, 4096 + 37, 0]
    worst_plain = _attend(bits, G, Hq, Hkv, prompt, prompt, n_out, synth.mix(synth.BASE_SEED, 503, bits, Hq, n_out))
    assert worst_plain > 10 * ATTN_TOL      # the main cache alone misses the outlier channels


def test_outlier_attention_after_appends():
    """Prompt, then 100 decode appends with isolation per completed group, then attention."""
    require_gpu()
    prompt = [1000, 64, 37, 2048]
    _attend(4, 32, 8, 2, prompt, [p + 100 for p in prompt], 1, synth.mix(synth.BASE_SEED, 504))


def test_outlier_argument_errors():
    require_gpu()
    H = 2
    cache2 = kvq.LayerCache(4, H, 2, 8, 1, v_group_dims=64)
    alloc = kvq.Allocator(8, seed=1)
    batch, _ = paged_batch([64], alloc)
    k_out = torch.zeros((8, H, 16, 1), dtype=torch.float16, device="cuda")
    och = torch.zeros((1, H, 1), dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 4, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((1, 4, 128), device="cuda")
    w = ws(kvq.kv_decode_attn_quant_ws(cache2, batch))
    with pytest.raises(kvq.KvqError) as e:          # 2-bit codes: not supported
        kvq.kv_decode_attn_quant_outlier(cache2, batch, q, 1, och, k_out, out, w)
    assert e.value.code == -2
    cache4 = kvq.LayerCache(4, H, 4, 8, 1, v_group_dims=64)
    for n_out in (0, 9):
        with pytest.raises(kvq.KvqError) as e:
            kvq.kv_decode_attn_quant_outlier(cache4, batch, q, n_out, och, k_out, out, w)
        assert e.value.code == -1
    with pytest.raises(kvq.KvqError):
        kvq.kv_outlier_isolate(cache2, batch, 0, 0, 64, torch.zeros((64, H, 128), dtype=torch.float16,
                                                                      device="cuda"), 1, och, k_out)
