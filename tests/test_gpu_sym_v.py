"""GPU parity of symmetric V quantization (on-device article, section 3.1: V INT4
symmetric with group quantization): the pack and the append store, per token and V
group, the code + L (L = 2^(b-1) - 1) and (scale16, fp16(-L * scale16)); codes and
scales equal the oracle's bit for bit (a code may differ only at a documented
near-tie of the fp32 quotient), and the quantized decode attention over such a
cache is within 2e-3 of the oracle's attention over code * scale16."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import ATTN_TOL, attn_err, paged_batch, require_gpu, ws
from kvq_format import quant_logical

pytestmark = pytest.mark.gpu


def _check_v(cache, bt_row, T, V, h, bits, G):
    cnp = {n: getattr(cache, n).cpu().numpy() for n in ("k_codes", "v_codes", "k_sz", "v_sz", "k_tail")}
    lg = quant_logical(cnp, bt_row, T, h, bits, G)
    L = 2 ** (bits - 1) - 1
    pv = O.pack_v_sym(V[:T, h], bits, G)
    got = lg["v_codes"] - L
    bad = np.argwhere(got != pv["codes"])
    for t, d in bad:   # only near-ties of the quotient x / scale32
        u = float(V[t, h, d]) / float(pv["scale32"][t, d // G])
        assert abs(abs(u - math.floor(u)) - 0.5) < 1e-6, (t, d, got[t, d], pv["codes"][t, d])
    assert np.array_equal(lg["v_scale16"].view(np.uint16), pv["scale16"].view(np.uint16))
    zero = (np.float32(-L) * pv["scale16"].astype(np.float32)).astype(np.float16)
    assert np.array_equal(lg["v_zero16"].view(np.uint16), zero.view(np.uint16))
    return pv


@pytest.mark.parametrize("bits,G", [(2, 32), (4, 32), (4, 64), (8, 128)])
def test_symmetric_pack_append_and_attention(bits, G):
    require_gpu()
    Hq, Hkv, T0, n_app = 8, 2, 1000, 70
    T = T0 + n_app
    seed = synth.mix(synth.BASE_SEED, 800, bits, G)
    K, V = synth.kv_rows(T, Hkv, seed)
    V[5, 0] = 0.0                                   # an all-zero token: scale 0, codes 0
    n_pages = math.ceil(T / 16) + 2
    alloc = kvq.Allocator(n_pages, seed=7)
    batch, bt = paged_batch([T], alloc, lengths=[T0])
    cache = kvq.LayerCache(Hq, Hkv, bits | kvq.V_SYMMETRIC, n_pages, 1, v_group_dims=G)
    kvq.kv_quant_pack(cache, batch, 0, 0, T0, K[:T0].cuda(), V[:T0].cuda())
    w = ws(kvq.kv_page_append_ws())
    for i in range(n_app):
        kvq.kvq_seq_lens_add(batch.seq_lens, 1)
        kvq.kv_page_append(cache, batch, K[T0 + i][None].cuda(), V[T0 + i][None].cuda(), w)
    kvq.kvq_check(w)
    Kn, Vn = K.numpy(), V.numpy()
    pvs = [_check_v(cache, bt[0], T, Vn, h, bits, G) for h in range(Hkv)]
    q = synth.queries((1, Hq, 128), synth.mix(seed, 2))
    out = torch.full((1, Hq, 128), float("nan"), device="cuda")
    wq = ws(kvq.kv_decode_attn_quant_ws(cache, batch))
    kvq.kv_decode_attn_quant(cache, batch, q.cuda(), out, wq)
    kvq.kvq_check(wq)
    pk = [O.pack_k(Kn[:, g], bits) for g in range(Hkv)]
    ref = O.decode_attn_quant(q[0].numpy(), pk, pvs)
    o = out.cpu().numpy()
    for h in range(Hq):
        assert attn_err(o[0, h], ref[h]) <= ATTN_TOL, h


def test_symmetric_rejects_one_bit():
    require_gpu()
    cache = kvq.LayerCache(8, 2, 2, 4, 1, v_group_dims=64)
    cache.layout.bits = 1 | kvq.V_SYMMETRIC
    batch = kvq.Batch(torch.zeros((1, 4), dtype=torch.int32, device="cuda"),
                      torch.tensor([0], dtype=torch.int32, device="cuda"), 64)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_quant_pack(cache, batch, 0, 0, 64, torch.zeros((64, 2, 128), dtype=torch.float16, device="cuda"),
                          torch.zeros((64, 2, 128), dtype=torch.float16, device="cuda"))
    assert e.value.code == -2
