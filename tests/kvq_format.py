"""Test-side knowledge of libkvq's storage format (include/kvq.h): turns the
paged device arrays back into logical per-(sequence, kv head) arrays that
can be compared with the oracle.  Pure numpy; no method arithmetic."""
import numpy as np


def unpack_codes(rows_u8, bits):
    """[..., R] bytes -> [..., 128] codes; channel c at bits [c*bits, (c+1)*bits)
    of the row read little-endian."""
    rows_u8 = np.ascontiguousarray(rows_u8)
    bitarr = np.unpackbits(rows_u8, axis=-1, bitorder="little")
    bitarr = bitarr.reshape(rows_u8.shape[:-1] + (128, bits)).astype(np.int64)
    return (bitarr << np.arange(bits)).sum(axis=-1)


def quant_logical(cache_np, bt_row, T, h, bits, G):
    """Logical view of sequence (block table row bt_row, length T), kv head h."""
    n_full = T // 64
    pages = [int(bt_row[t // 16]) for t in range(T)]
    slots = [t % 16 for t in range(T)]
    kc = np.stack([cache_np["k_codes"][pages[t], h, slots[t]] for t in range(n_full * 64)]) if n_full else \
        np.zeros((0, 16 * bits), np.uint8)
    vc = np.stack([cache_np["v_codes"][pages[t], h, slots[t]] for t in range(T)])
    ksz = np.stack([cache_np["k_sz"][int(bt_row[4 * g]), h] for g in range(n_full)]) if n_full else \
        np.zeros((0, 128, 2), np.float16)
    vsz = np.stack([cache_np["v_sz"][pages[t], h, slots[t]] for t in range(T)])
    return dict(k_codes=unpack_codes(kc, bits), k_scale16=ksz[..., 0], k_zero16=ksz[..., 1],
                v_codes=unpack_codes(vc, bits), v_scale16=vsz[..., 0], v_zero16=vsz[..., 1])


def fp16_logical(k16_np, bt_row, T, h):
    return np.stack([k16_np[int(bt_row[t // 16]), h, t % 16] for t in range(T)])
