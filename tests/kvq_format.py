"""Test-side knowledge of libkvq's storage format (include/kvq.h): turns the
paged device arrays back into logical per-(sequence, kv head) arrays that
can be compared with the oracle.  Pure numpy; no method arithmetic."""
import numpy as np


def k_code_pos(c, bits):
    """(word, bit) of channel c in a K token row: the channel pair (2p, 2p+1),
    p = 8s + r + 4e, is pair m = 2s + e of column r, stored in word
    r*bits + m // (16//bits) at offset (m % (16//bits))*bits, the odd channel
    in the high half word."""
    p = c // 2
    s, r, e = p // 8, p % 4, (p // 4) % 2
    m, per = 2 * s + e, 16 // bits
    return r * bits + m // per, (m % per) * bits + 16 * (c % 2)


def v_code_pos(tok, d, bits):
    """(word, bit) of token tok (of the page) and channel d in a V page block:
    d = 16t + 8u + x, token pair y = tok // 2 = r + 4e -> pair m = 4r + 2e + u of
    row 8t + x, word (8t + x)*bits + m // (16//bits), offset (m % (16//bits))*bits,
    the odd token in the high half word."""
    t, x, u = d // 16, d % 8, (d // 8) % 2
    y = tok // 2
    r, e = y % 4, y // 4
    m, per = 4 * r + 2 * e + u, 16 // bits
    return (8 * t + x) * bits + m // per, (m % per) * bits + 16 * (tok % 2)


def k_row_codes(rows_u8, bits):
    """[..., 16*bits] bytes of K token rows -> [..., 128] codes."""
    words = np.ascontiguousarray(rows_u8).view("<u4").astype(np.int64)
    out = np.zeros(words.shape[:-1] + (128,), np.int64)
    for c in range(128):
        w, b = k_code_pos(c, bits)
        out[..., c] = (words[..., w] >> b) & ((1 << bits) - 1)
    return out


def v_page_codes(block_u8, bits):
    """[..., 16, 16*bits] bytes (one page block per leading index) -> [..., 16, 128] codes."""
    blk = np.ascontiguousarray(block_u8)
    words = blk.reshape(blk.shape[:-2] + (-1,)).view("<u4").astype(np.int64)
    out = np.zeros(words.shape[:-1] + (16, 128), np.int64)
    for tok in range(16):
        for d in range(128):
            w, b = v_code_pos(tok, d, bits)
            out[..., tok, d] = (words[..., w] >> b) & ((1 << bits) - 1)
    return out


def quant_logical(cache_np, bt_row, T, h, bits, G):
    """Logical view of sequence (block table row bt_row, length T), kv head h."""
    n_full = T // 64
    pages = [int(bt_row[t // 16]) for t in range(T)]
    slots = [t % 16 for t in range(T)]
    kc = np.stack([cache_np["k_codes"][pages[t], h, slots[t]] for t in range(n_full * 64)]) if n_full else \
        np.zeros((0, 16 * bits), np.uint8)
    vpages = {}
    for t in range(T):
        if pages[t] not in vpages:
            vpages[pages[t]] = v_page_codes(cache_np["v_codes"][pages[t], h], bits)
    vc = np.stack([vpages[pages[t]][slots[t]] for t in range(T)]) if T else np.zeros((0, 128), np.int64)
    ksz = np.stack([cache_np["k_sz"][int(bt_row[4 * g]), h] for g in range(n_full)]) if n_full else \
        np.zeros((0, 128, 2), np.float16)
    vsz = np.stack([cache_np["v_sz"][pages[t], h, slots[t]] for t in range(T)])
    return dict(k_codes=k_row_codes(kc, bits), k_scale16=ksz[..., 0], k_zero16=ksz[..., 1],
                v_codes=vc, v_scale16=vsz[..., 0], v_zero16=vsz[..., 1])


def fp16_logical(k16_np, bt_row, T, h):
    return np.stack([k16_np[int(bt_row[t // 16]), h, t % 16] for t in range(T)])
