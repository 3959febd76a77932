"""GPU parity of a1 kv_quant_pack and a2 kv_page_append against the oracle:
codes, scales, zeros and fp16 tails bit-exact (quantizer arithmetic is IEEE
fp32 on both sides), paged through shuffled block tables."""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_quant_gb300 import kvq, synth
from oracle import kvq_oracle as O
from gpu_helpers import paged_batch, require_gpu, ws
from kvq_format import quant_logical, fp16_logical

pytestmark = pytest.mark.gpu


def _np(t):
    return t.cpu().numpy()


def _cache_np(cache):
    return {n: _np(getattr(cache, n)) for n in ("k_codes", "v_codes", "k_sz", "v_sz", "k_tail")}


def assert_codes(gpu, ref, x16, scale32, mn, axis_group):
    """Bit-exact codes; a mismatch is allowed only at a documented near-tie
    (exact quotient within 1e-6 of a half-integer)."""
    if np.array_equal(gpu, ref):
        return
    bad = np.argwhere(gpu != ref)
    for idx in bad:
        idx = tuple(idx)
        g = axis_group(idx)
        u = (float(x16[idx]) - float(mn[g])) / float(scale32[g])
        assert abs(u - math.floor(u) - 0.5) < 1e-6, f"code mismatch at {idx}: gpu {gpu[idx]} ref {ref[idx]} u={u}"


def _check_quant(cache, bt_row, T, K, V, bits, G, strict=False):
    cnp = _cache_np(cache)
    H = K.shape[1]
    for h in range(H):
        lg = quant_logical(cnp, bt_row, T, h, bits, G)
        pk = O.pack_k(K[:, h], bits)
        pv = O.pack_v(V[:, h], bits, G)
        n_full = pk["n_packed"]
        kx = K[:n_full, h]
        k_mn = pk["zero16"].astype(np.float32)
        if strict:
            assert np.array_equal(lg["k_codes"], pk["codes"])
        assert_codes(lg["k_codes"], pk["codes"], kx, pk["scale32"], k_mn, lambda i: (i[0] // 64, i[1]))
        assert np.array_equal(lg["k_scale16"].view(np.uint16), pk["scale16"].view(np.uint16))
        assert np.array_equal(lg["k_zero16"].view(np.uint16), pk["zero16"].view(np.uint16))
        v_mn = pv["zero16"].astype(np.float32)
        if strict:
            assert np.array_equal(lg["v_codes"], pv["codes"])
        assert_codes(lg["v_codes"], pv["codes"], V[:, h], pv["scale32"], v_mn, lambda i: (i[0], i[1] // G))
        assert np.array_equal(lg["v_scale16"].view(np.uint16), pv["scale16"].view(np.uint16))
        assert np.array_equal(lg["v_zero16"].view(np.uint16), pv["zero16"].view(np.uint16))
        tail = cnp["k_tail"][0, h, : T - n_full]
        assert np.array_equal(tail.view(np.uint16), pk["tail"].view(np.uint16))


@pytest.mark.parametrize("bits,G,T", [(1, 64, 4096 + 37), (2, 32, 1000), (4, 32, 2048 + 63), (8, 128, 640),
                                      (1, 32, 64), (4, 64, 17), (8, 64, 4096)])
def test_pack_quant_bitexact(bits, G, T):
    require_gpu()
    H = 2
    K, V = synth.kv_rows(T, H, synth.mix(synth.BASE_SEED, bits, G, T))
    n_pages = math.ceil(T / 16)
    alloc = kvq.Allocator(n_pages + 7, seed=11)
    batch, bt = paged_batch([T], alloc)
    cache = kvq.LayerCache(8, H, bits, n_pages + 7, 1, v_group_dims=G)
    kvq.kv_quant_pack(cache, batch, 0, 0, T, K.cuda(), V.cuda())
    torch.cuda.synchronize()
    _check_quant(cache, bt[0], T, K.numpy(), V.numpy(), bits, G)


def _grid_rows(T, H, bits, G, seed):
    """K, V fp16 on half-steps of a quantization grid: x = offset + span * k / (2L),
    k uniform in [0, 2L]; each K group of 64 tokens and each V group of G channels
    holds k = 0 and k = 2L, so its zero and scale come from offset and span.  With
    span = L, L/2 or L/4 the quotients of odd k are exact ties (x - zero = (k/2)
    scale); the other spans put quotients a few ulps from a half-integer."""
    L = 2 ** bits - 1
    rng = np.random.default_rng(seed)
    spans = np.array([L, L / 2, L / 4, 1.0, 0.7, 100.0])
    offs = np.array([-1.5, 0.0, 0.25, -3.0])

    kk = rng.integers(0, 2 * L + 1, size=(T, H, 128))
    kk[0::64] = 0
    kk[1::64] = 2 * L
    ks = spans[rng.integers(0, len(spans), size=(1, H, 128))]
    ko = offs[rng.integers(0, len(offs), size=(1, H, 128))]
    K = (ko + ks * kk / (2 * L)).astype(np.float16)
    vk = rng.integers(0, 2 * L + 1, size=(T, H, 128))
    vk[:, :, 0::G] = 0
    vk[:, :, 1::G] = 2 * L
    vs = np.repeat(spans[rng.integers(0, len(spans), size=(T, H, 128 // G))], G, axis=2)
    vo = np.repeat(offs[rng.integers(0, len(offs), size=(T, H, 128 // G))], G, axis=2)
    V = (vo + vs * vk / (2 * L)).astype(np.float16)
    return torch.from_numpy(K), torch.from_numpy(V)


@pytest.mark.parametrize("bits,G", [(1, 64), (2, 32), (4, 128), (8, 64)])
def test_pack_rounding_ties_bitexact(bits, G):
    """Codes whose quotient is an exact tie or within a few ulps of one: the
    quantizer takes the IEEE fp32 quotient and rounds half to even on both sides,
    so every code matches bit for bit (no near-tie allowance here)."""
    require_gpu()
    H, T = 2, 640 + 23
    K, V = _grid_rows(T, H, bits, G, synth.mix(synth.BASE_SEED, 91, bits, G))
    n_pages = math.ceil(T / 16)
    alloc = kvq.Allocator(n_pages + 3, seed=5)
    batch, bt = paged_batch([T], alloc)
    cache = kvq.LayerCache(8, H, bits, n_pages + 3, 1, v_group_dims=G)
    kvq.kv_quant_pack(cache, batch, 0, 0, T, K.cuda(), V.cuda())
    torch.cuda.synchronize()
    _check_quant(cache, bt[0], T, K.numpy(), V.numpy(), bits, G, strict=True)


@pytest.mark.parametrize("bits,G", [(1, 64), (4, 32), (2, 128)])
def test_append_matches_pack_of_whole_sequence(bits, G):
    """Prefill T0 tokens, append 150 one at a time (crossing 64-token group
    boundaries): the cache must equal the oracle's packing of all tokens."""
    require_gpu()
    H, T0, n_app, B = 2, 1000, 150, 2
    T = T0 + n_app
    seeds = [synth.mix(synth.BASE_SEED, 77, bits, b) for b in range(B)]
    KV = [synth.kv_rows(T, H, s) for s in seeds]
    n_pages = B * math.ceil(T / 16)
    alloc = kvq.Allocator(n_pages, seed=3)
    batch, bt = paged_batch([T] * B, alloc, lengths=[T0] * B)
    cache = kvq.LayerCache(4, H, bits, n_pages, B, v_group_dims=G)
    for b in range(B):
        kvq.kv_quant_pack(cache, batch, b, 0, T0, KV[b][0][:T0].cuda(), KV[b][1][:T0].cuda())
    w = ws(kvq.kv_page_append_ws())
    for i in range(n_app):
        kvq.kvq_seq_lens_add(batch.seq_lens, 1)
        kn = torch.stack([KV[b][0][T0 + i] for b in range(B)]).cuda()
        vn = torch.stack([KV[b][1][T0 + i] for b in range(B)]).cuda()
        kvq.kv_page_append(cache, batch, kn, vn, w)
    kvq.kvq_check(w)
    assert _np(batch.seq_lens).tolist() == [T] * B
    cnp = _cache_np(cache)
    for b in range(B):
        K, V = KV[b][0].numpy(), KV[b][1].numpy()
        sub = {k: v for k, v in cnp.items()}
        sub["k_tail"] = cnp["k_tail"][b:b + 1]
        for h in range(H):
            lg = quant_logical(sub, bt[b], T, h, bits, G)
            pk = O.pack_k(K[:, h], bits)
            pv = O.pack_v(V[:, h], bits, G)
            assert np.array_equal(lg["k_codes"], pk["codes"])
            assert np.array_equal(lg["k_scale16"].view(np.uint16), pk["scale16"].view(np.uint16))
            assert np.array_equal(lg["v_codes"], pv["codes"])
            assert np.array_equal(lg["v_zero16"].view(np.uint16), pv["zero16"].view(np.uint16))
            nt = T - pk["n_packed"]
            assert np.array_equal(sub["k_tail"][0, h, :nt].view(np.uint16), pk["tail"].view(np.uint16))


def test_pack_and_append_fp16_layer():
    require_gpu()
    H, T0, n_app = 2, 777, 40
    T = T0 + n_app
    t_cap = 1024
    K, V = synth.kv_rows(T, H, synth.mix(synth.BASE_SEED, 5))
    n_pages = math.ceil(T / 16) + 3
    alloc = kvq.Allocator(n_pages, seed=9)
    batch, bt = paged_batch([T], alloc, lengths=[T0])
    cache = kvq.LayerCache(8, H, 16, n_pages, 1, t_cap=t_cap)
    kvq.kv_quant_pack(cache, batch, 0, 0, T0, K[:T0].cuda(), V[:T0].cuda())
    w = ws(kvq.kv_page_append_ws())
    for i in range(n_app):
        kvq.kvq_seq_lens_add(batch.seq_lens, 1)
        kvq.kv_page_append(cache, batch, K[T0 + i][None].cuda(), V[T0 + i][None].cuda(), w)
    kvq.kvq_check(w)
    k16, v16, kT, am = _np(cache.k16), _np(cache.v16), _np(cache.kT), _np(cache.k_absmax)
    for h in range(H):
        assert np.array_equal(fp16_logical(k16, bt[0], T, h).view(np.uint16), K[:, h].numpy().view(np.uint16))
        assert np.array_equal(fp16_logical(v16, bt[0], T, h).view(np.uint16), V[:, h].numpy().view(np.uint16))
        assert np.array_equal(kT[0, h, :, :T].T.view(np.uint16), K[:, h].numpy().view(np.uint16))
        assert np.array_equal(am[0, h], O.key_absmax(K[:, h].numpy()).astype(np.float32))


def test_page_copy_and_shared_prefix_refcounts():
    """Copy-on-write support: a shared page is copied before a write."""
    require_gpu()
    alloc = kvq.Allocator(16, seed=0)
    a, b_ = alloc.alloc(2)
    alloc.ref(a)
    assert alloc.refcount(a) == 2
    cache = kvq.LayerCache(4, 2, 4, 16, 1, v_group_dims=32)
    cache.k_codes[a].random_(0, 255)
    cache.v_sz[a].normal_()
    kvq.kv_page_copy(cache, a, b_)
    torch.cuda.synchronize()
    assert torch.equal(cache.k_codes[a], cache.k_codes[b_])
    assert torch.equal(cache.v_sz[a], cache.v_sz[b_])
    alloc.free(a)
    assert alloc.refcount(a) == 1


def test_append_flags_bad_page():
    """A block table entry outside the pool is skipped and reported by kvq_check."""
    require_gpu()
    cache = kvq.LayerCache(4, 2, 1, 4, 1, v_group_dims=64)
    bt = torch.tensor([[99, 0]], dtype=torch.int32, device="cuda")
    batch = kvq.Batch(bt, torch.tensor([1], dtype=torch.int32, device="cuda"), 32)
    w = ws(kvq.kv_page_append_ws())
    kn = torch.zeros((1, 2, 128), dtype=torch.float16, device="cuda")
    kvq.kv_page_append(cache, batch, kn, kn, w)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_check(w)
    assert e.value.code == -6
    kvq.kvq_check(w)  # cleared
