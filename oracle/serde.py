"""Storage-layer serialise / deserialise of a KV tensor (oracle side; test
infrastructure).

Restates "lmcache.v1.distributed.serde.turboquant": Configuration
(skip_first_layers / skip_last_layers and the compressed range
quant_start = min(skip_first, L), quant_end = max(quant_start, L - skip_last))
and Tensor Layout (input [2, L, T, hidden]; output = raw first layers |
compressed middle layers | raw last layers; compressed layers laid out
[L_c, ceil(T / block_size), block_size, H, slot]; H = hidden / head_dim;
slot = key bytes + value bytes).

Readings: a raw group keeps the [2, layers, T, hidden] order (all keys of the
group, then all values); the slot is the key block followed by the value
block with no padding (slot_size_aligned = slot, 4-byte aligned for 66+66);
token slots past T in the last token block are zero bytes; the codec of the
middle layers is this package's codec for both K and V.
"""

import numpy as np

from .codec import block_bytes, encode, pack_block, unpack_block, decode


def serde_ranges(num_layers, skip_first, skip_last):
    qs = min(skip_first, num_layers)
    qe = max(qs, num_layers - skip_last)
    return qs, qe


def serde_size(num_layers, num_tokens, hidden, head_dim, block_size,
               skip_first, skip_last, kbits, vbits, elem_bytes=2):
    qs, qe = serde_ranges(num_layers, skip_first, skip_last)
    heads = hidden // head_dim
    nblk = -(-num_tokens // block_size)
    slot = block_bytes(kbits) + block_bytes(vbits)
    raw_layers = num_layers - (qe - qs)
    return (2 * raw_layers * num_tokens * hidden * elem_bytes
            + (qe - qs) * nblk * block_size * heads * slot)


def serialize(src, block_size, skip_first, skip_last, kbits, vbits,
              signs, kb32, vb32, head_dim=128):
    """Serialise one KV object.

    ``src`` is a pair (values, raw): values are the exact element values
    [2, L, T, hidden] as float64, raw the same tensor's bytes as uint8
    [2, L, T, hidden * elem_bytes].  Returns the serialised uint8 buffer.
    """
    values, raw = src
    _, L, T, hidden = values.shape
    qs, qe = serde_ranges(L, skip_first, skip_last)
    H = hidden // head_dim
    nblk = -(-T // block_size)
    kbb, vbb = block_bytes(kbits), block_bytes(vbits)
    slot = kbb + vbb
    parts = [raw[:, :qs].reshape(-1)]
    comp = np.zeros((qe - qs, nblk * block_size, H, slot), np.uint8)
    for li, l in enumerate(range(qs, qe)):
        for kv, (bb32, bits, off) in enumerate(((kb32, kbits, 0), (vb32, vbits, kbb))):
            x = values[kv, l].reshape(T * H, head_dim)
            idx, n16, _ = encode(x, signs, bb32)
            blk = pack_block(idx, n16, bits).reshape(T, H, -1)
            comp[li, :T, :, off:off + blk.shape[-1]] = blk
    parts.append(comp.reshape(-1))
    parts.append(raw[:, qe:].reshape(-1))
    return np.concatenate(parts)


def deserialize(buf, num_layers, num_tokens, hidden, block_size, skip_first,
                skip_last, kbits, vbits, signs, kc, vc, elem_dtype, head_dim=128):
    """Inverse of serialize.  Returns (raw layer bytes as uint8
    [2, L, T, hidden*elem_bytes] for raw layers, float64 reconstructions
    [2, L, T, hidden] for compressed layers, (qs, qe))."""
    L, T = num_layers, num_tokens
    qs, qe = serde_ranges(L, skip_first, skip_last)
    H = hidden // head_dim
    eb = np.dtype(elem_dtype).itemsize
    nblk = -(-T // block_size)
    kbb, vbb = block_bytes(kbits), block_bytes(vbits)
    slot = kbb + vbb
    buf = np.asarray(buf, np.uint8)
    n_first = 2 * qs * T * hidden * eb
    n_comp = (qe - qs) * nblk * block_size * H * slot
    first = buf[:n_first].reshape(2, qs, T, hidden * eb)
    comp = buf[n_first:n_first + n_comp].reshape(qe - qs, nblk * block_size, H, slot)
    last = buf[n_first + n_comp:].reshape(2, L - qe, T, hidden * eb)
    raw = np.zeros((2, L, T, hidden * eb), np.uint8)
    raw[:, :qs] = first
    raw[:, qe:] = last
    rec = np.zeros((2, L, T, hidden))
    for li, l in enumerate(range(qs, qe)):
        for kv, (c, bits, off, bb) in enumerate(((kc, kbits, 0, kbb), (vc, vbits, kbb, vbb))):
            blk = comp[li, :T, :, off:off + bb].reshape(T * H, bb)
            idx, n16 = unpack_block(blk, bits)
            rec[kv, l] = decode(idx, n16, c, signs).reshape(T, hidden)
    return raw, rec, (qs, qe)
