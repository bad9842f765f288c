"""Thin ctypes binding over libtq (include/tq.h).  Argument marshalling only:
every step of the path runs in the library's CUDA kernels.  There is no
fallback: if libtq.so is missing the import of a compute function raises.

Functions keep the C names.  Device buffers are torch tensors (their data
pointers are passed); streams default to torch's current CUDA stream.
Every non-zero status raises ``TQError``.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")

TQ_OK, TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN, TQ_ERR_WORKSPACE, TQ_ERR_CUDA, TQ_ERR_TIMEOUT = \
    0, -1, -2, -3, -4, -5, -6
TQ_F32, TQ_BF16, TQ_F16 = 0, 1, 2
_DT = {torch.float32: TQ_F32, torch.bfloat16: TQ_BF16, torch.float16: TQ_F16}


class tq_codebook(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int), ("bits", ctypes.c_int), ("levels", ctypes.c_int),
                ("centroids", ctypes.c_float * 16), ("boundaries", ctypes.c_float * 15)]


class tq_signs(ctypes.Structure):
    _fields_ = [("w", ctypes.c_uint32 * 4)]


class TQError(RuntimeError):
    def __init__(self, status, what):
        super().__init__("%s: %s (status %d)" % (what, tq_status_string(status), status))
        self.status = status


_lib = None


def lib():
    """Load libtq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libtq.so not built at %s; run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, c_int, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        cbp = ctypes.POINTER(tq_codebook)
        L.tq_codebook_load.argtypes = [c_int, c_int, cbp]
        L.tq_signs_from_seed.argtypes = [ctypes.c_uint64, c_int, ctypes.POINTER(tq_signs)]
        L.tq_block_bytes.argtypes = [c_int]
        L.tq_block_bytes.restype = sz
        L.tq_encode_kv.argtypes = [vp, c_int, i64, i64, cbp, tq_signs, vp, i64, vp, vp]
        L.tq_decode_kv.argtypes = [vp, i64, i64, cbp, tq_signs, vp, c_int, i64, vp]
        L.tq_qjl_encode.argtypes = [vp, c_int, i64, i64, vp, i64, cbp, tq_signs, vp, vp, vp, vp]
        L.tq_attn_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int]
        L.tq_attn_workspace_bytes.restype = sz
        L.tq_attn_plan.argtypes = [c_int] * 8 + [ctypes.POINTER(i64)]
        L.tq_attn_plan_d.argtypes = [c_int] * 5 + [ctypes.POINTER(ctypes.c_int32)]
        L.tq_attn_decode.argtypes = [vp, c_int, vp, cbp, vp, cbp, vp, c_int, c_int, c_int, c_int, c_int,
                                     ctypes.c_float, tq_signs, vp, vp, vp, vp, vp, sz, vp]
        L.tq_serde_size.argtypes = [c_int] * 10
        L.tq_serde_size.restype = sz
        ser = [vp, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, cbp, cbp, tq_signs, vp, vp]
        L.tq_serde_serialize.argtypes = ser
        L.tq_serde_deserialize.argtypes = ser
        L.tq_attn_prefill.argtypes = [vp, c_int, vp, cbp, vp, cbp, vp, c_int, c_int, c_int, c_int, c_int, c_int,
                                      ctypes.c_float, tq_signs, vp, vp]
        L.tq_block_bytes_ex.argtypes = [c_int, c_int]
        L.tq_block_bytes_ex.restype = sz
        L.tq_encode_kv_ex.argtypes = [vp, c_int, i64, i64, cbp, tq_signs, vp, i64, vp, c_int, vp]
        L.tq_decode_kv_ex.argtypes = [vp, i64, i64, cbp, tq_signs, vp, c_int, i64, c_int, vp]
        L.tq_attn_prefill_paged.argtypes = [vp, c_int, vp, cbp, vp, cbp, vp, c_int, c_int, vp, c_int, c_int, c_int,
                                            c_int, c_int, ctypes.c_float, tq_signs, vp, vp]
        L.tq_attn_decode_paged.argtypes = [vp, c_int, vp, cbp, vp, cbp, vp, c_int, c_int, vp, c_int, c_int, c_int,
                                           c_int, ctypes.c_float, tq_signs, vp, vp, sz, vp]
        L.tq_device_status.argtypes = [c_int, vp]
        L.tq_debug_drop_copies.argtypes = [c_int]
        L.tq_attn_workspace_bytes_sms.argtypes = [c_int] * 5
        L.tq_attn_workspace_bytes_sms.restype = sz
        L.tq_status_string.argtypes = [c_int]
        L.tq_status_string.restype = ctypes.c_char_p
        L.tq_block_bytes_d.argtypes = [c_int, c_int]
        L.tq_block_bytes_d.restype = sz
        L.tq_rotation_hadamard.argtypes = [c_int, tq_signs, vp]
        L.tq_encode_kv_d.argtypes = [vp, c_int, i64, c_int, cbp, vp, vp, vp]
        L.tq_decode_kv_d.argtypes = [vp, i64, c_int, cbp, vp, vp, c_int, vp]
        L.tq_attn_workspace_bytes_d.argtypes = [c_int] * 5
        L.tq_attn_workspace_bytes_d.restype = sz
        L.tq_attn_decode_d.argtypes = [vp, c_int, vp, cbp, vp, cbp, vp, c_int, c_int, c_int, c_int, c_int, c_int,
                                       ctypes.c_float, vp, vp, vp, sz, vp]
        _lib = L
    return _lib


def _check(status, what):
    if status != TQ_OK:
        raise TQError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype(t):
    if t.dtype not in _DT:
        raise TypeError("unsupported dtype %s" % t.dtype)
    return _DT[t.dtype]


def _row_stride(x):
    if x.dim() < 1 or x.shape[-1] != 128 or x.stride(-1) != 1:
        raise ValueError("rows of 128 contiguous elements expected")
    if x.dim() == 1:
        return 128
    # rows may be strided along one flattened leading axis
    return x.stride(-2)


def tq_status_string(status):
    return lib().tq_status_string(int(status)).decode()


def tq_codebook_load(head_dim=128, bits=4):
    cb = tq_codebook()
    _check(lib().tq_codebook_load(head_dim, bits, ctypes.byref(cb)), "tq_codebook_load")
    return cb


def tq_signs_from_seed(seed, head_dim=128):
    s = tq_signs()
    _check(lib().tq_signs_from_seed(ctypes.c_uint64(seed), head_dim, ctypes.byref(s)), "tq_signs_from_seed")
    return s


def tq_block_bytes(bits):
    return int(lib().tq_block_bytes(bits))


def _nvec_rows(x):
    """Number of 128-element rows of x and their stride (leading dims must
    flatten to one uniformly strided axis)."""
    if x.dim() == 1:
        return 1, 128
    lead = x.shape[:-1]
    n = 1
    for s in lead:
        n *= s
    if n == 0:
        return 0, 128
    stride = x.stride(-2)
    expect = stride
    for i in range(x.dim() - 2, -1, -1):
        if x.shape[i] != 1 and x.stride(i) != expect:
            raise ValueError("leading dims of x must flatten to one strided axis")
        expect *= x.shape[i]
    return n, stride


def tq_encode_kv(x, cb, signs, blocks, block_stride_bytes=None, dst_index=None, block_offset=0, stream=None):
    """Encode the 128-element rows of ``x`` into ``blocks`` (uint8 tensor).

    Block of row i is written at byte ``block_offset + dst(i) * block_stride_bytes``
    of ``blocks``; dst(i) = i, or ``dst_index[i]`` (int64 device tensor)."""
    n, stride = _nvec_rows(x)
    bs = block_stride_bytes or tq_block_bytes(cb.bits)
    base = ctypes.c_void_p(blocks.data_ptr() + block_offset)
    _check(lib().tq_encode_kv(_ptr(x), _dtype(x), n, stride, ctypes.byref(cb), signs, base, bs,
                              _ptr(dst_index), _stream(stream)), "tq_encode_kv")
    return blocks


def tq_decode_kv(blocks, n_vec, cb, signs, out, block_stride_bytes=None, block_offset=0, stream=None):
    """Dequantise ``n_vec`` blocks into the 128-element rows of ``out``."""
    _, stride = _nvec_rows(out)
    bs = block_stride_bytes or tq_block_bytes(cb.bits)
    base = ctypes.c_void_p(blocks.data_ptr() + block_offset)
    _check(lib().tq_decode_kv(base, bs, n_vec, ctypes.byref(cb), signs, _ptr(out), _dtype(out), stride,
                              _stream(stream)), "tq_decode_kv")
    return out


def tq_qjl_encode(k, k_blocks, cb, signs, S, qjl_bits, res_norm_f16, block_stride_bytes=None, stream=None):
    n, stride = _nvec_rows(k)
    bs = block_stride_bytes or tq_block_bytes(cb.bits)
    _check(lib().tq_qjl_encode(_ptr(k), _dtype(k), n, stride, _ptr(k_blocks), bs, ctypes.byref(cb), signs,
                               _ptr(S), _ptr(qjl_bits), _ptr(res_norm_f16), _stream(stream)), "tq_qjl_encode")


def tq_attn_plan(B, Hq, Hkv, T, key_bits, value_bits, qjl=False, sms=0):
    """The tensor-core attention path's work partition for a shape, as a dict
    (C, Ctot, P, W, Smax, combine_groups, warps); raises TQError when the shape
    takes the split path or is invalid."""
    out = (ctypes.c_int64 * 7)()
    _check(lib().tq_attn_plan(B, Hq, Hkv, T, key_bits, value_bits, 1 if qjl else 0, sms, out), "tq_attn_plan")
    return dict(zip(("C", "Ctot", "P", "W", "Smax", "combine_groups", "warps"), (int(x) for x in out)))


def tq_attn_plan_d(B, Hkv, T, ctas_resident, warps_per_cta=4):
    """Host-only split plan of tq_attn_decode_d: (splits, tokens per split, most splits)."""
    out = (ctypes.c_int32 * 3)()
    _check(lib().tq_attn_plan_d(B, Hkv, T, ctas_resident, warps_per_cta, out), "tq_attn_plan_d")
    return int(out[0]), int(out[1]), int(out[2])


def tq_attn_workspace_bytes(B, Hq, Hkv, T_cap):
    return int(lib().tq_attn_workspace_bytes(B, Hq, Hkv, T_cap))


def tq_attn_decode(q, k_blocks, kcb, v, vcb, out, workspace, T, scale, signs, seq_lens=None,
                   qjl_bits=None, res_norm_f16=None, S=None, stream=None):
    """Decode attention.  q [B, Hq, 128]; k_blocks uint8 [B, Hkv, T_cap, kbytes];
    v uint8 blocks [B, Hkv, T_cap, vbytes] (vcb given) or fp16 [B, Hkv, T_cap, 128]
    (vcb None); out float32 [B, Hq, 128]; workspace uint8 device tensor."""
    B, Hq, _ = q.shape
    Hkv, T_cap = k_blocks.shape[1], k_blocks.shape[2]
    _check(lib().tq_attn_decode(_ptr(q), _dtype(q), _ptr(k_blocks), ctypes.byref(kcb), _ptr(v),
                                ctypes.byref(vcb) if vcb is not None else None, _ptr(seq_lens), B, Hq, Hkv,
                                T_cap, T, ctypes.c_float(scale), signs, _ptr(qjl_bits), _ptr(res_norm_f16),
                                _ptr(S), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)), "tq_attn_decode")
    return out


def tq_serde_size(num_layers, num_tokens, hidden_dim, block_size, skip_first, skip_last, key_bits,
                  value_bits, head_dim=128, elem_bytes=2):
    return int(lib().tq_serde_size(num_layers, num_tokens, hidden_dim, head_dim, block_size, skip_first,
                                   skip_last, key_bits, value_bits, elem_bytes))


def tq_serde_serialize(src, kcb, vcb, signs, dst, block_size=16, skip_first=2, skip_last=2, stream=None):
    """src: [2, L, T, hidden] bf16/fp16 device tensor; dst: uint8 device tensor."""
    _, L, T, hidden = src.shape
    _check(lib().tq_serde_serialize(_ptr(src), _dtype(src), L, T, hidden, 128, block_size, skip_first,
                                    skip_last, ctypes.byref(kcb), ctypes.byref(vcb), signs, _ptr(dst),
                                    _stream(stream)), "tq_serde_serialize")
    return dst


def tq_serde_deserialize(src, kcb, vcb, signs, dst, block_size=16, skip_first=2, skip_last=2, stream=None):
    """src: serialised uint8 device tensor; dst: [2, L, T, hidden] bf16/fp16 device tensor."""
    _, L, T, hidden = dst.shape
    _check(lib().tq_serde_deserialize(_ptr(src), _dtype(dst), L, T, hidden, 128, block_size, skip_first,
                                      skip_last, ctypes.byref(kcb), ctypes.byref(vcb), signs, _ptr(dst),
                                      _stream(stream)), "tq_serde_deserialize")
    return dst


def tq_device_status(clear=False, stream=None):
    """Sticky status of the kernels' bounded waits on the current device
    (TQ_OK or TQ_ERR_TIMEOUT; returned, not raised).  Synchronises the stream."""
    return int(lib().tq_device_status(1 if clear else 0, _stream(stream)))


def tq_debug_drop_copies(on):
    """Test hook: while on, kernels with bounded waits issue no copies, so
    their waits run out (include/tq.h)."""
    _check(lib().tq_debug_drop_copies(1 if on else 0), "tq_debug_drop_copies")


def tq_attn_workspace_bytes_sms(B, Hq, Hkv, T_cap, sms):
    return int(lib().tq_attn_workspace_bytes_sms(B, Hq, Hkv, T_cap, sms))


def tq_attn_prefill(q, k_blocks, kcb, v_blocks, vcb, out, T, scale, signs, seq_lens=None, stream=None):
    """Causal attention of M query tokens per sequence.  q [B, M, Hq, 128];
    k_blocks / v_blocks uint8 [B, Hkv, T_cap, bytes]; out float32 [B, M, Hq, 128]."""
    B, M, Hq, _ = q.shape
    Hkv, T_cap = k_blocks.shape[1], k_blocks.shape[2]
    _check(lib().tq_attn_prefill(_ptr(q), _dtype(q), _ptr(k_blocks), ctypes.byref(kcb), _ptr(v_blocks),
                                 ctypes.byref(vcb), _ptr(seq_lens), B, M, Hq, Hkv, T_cap, T, ctypes.c_float(scale),
                                 signs, _ptr(out), _stream(stream)), "tq_attn_prefill")
    return out


TQ_FMT_NORM_CORRECT, TQ_FMT_DENSE3 = 1, 2


def tq_block_bytes_ex(bits, flags=0):
    return int(lib().tq_block_bytes_ex(bits, flags))


def tq_encode_kv_ex(x, cb, signs, blocks, flags=0, block_stride_bytes=None, dst_index=None, block_offset=0,
                    stream=None):
    """tq_encode_kv with format flags (TQ_FMT_NORM_CORRECT, TQ_FMT_DENSE3); an
    8-bit codebook selects turboq8."""
    n, stride = _nvec_rows(x)
    bs = block_stride_bytes or tq_block_bytes_ex(cb.bits, flags)
    base = ctypes.c_void_p(blocks.data_ptr() + block_offset)
    _check(lib().tq_encode_kv_ex(_ptr(x), _dtype(x), n, stride, ctypes.byref(cb), signs, base, bs, _ptr(dst_index),
                                 flags, _stream(stream)), "tq_encode_kv_ex")


def tq_decode_kv_ex(blocks, n_vec, cb, signs, out, flags=0, block_stride_bytes=None, block_offset=0, stream=None):
    bs = block_stride_bytes or tq_block_bytes_ex(cb.bits, flags)
    n, stride = _nvec_rows(out)
    base = ctypes.c_void_p(blocks.data_ptr() + block_offset)
    _check(lib().tq_decode_kv_ex(base, bs, n_vec, ctypes.byref(cb), signs, _ptr(out), _dtype(out), stride, flags,
                                 _stream(stream)), "tq_decode_kv_ex")


def tq_attn_prefill_paged(q, k_pool, kcb, v_pool, vcb, block_table, page_tokens, out, T, scale, signs,
                          seq_lens=None, stream=None):
    """Causal attention over a paged cache: q [B, M, Hq, 128]; k_pool / v_pool
    uint8 [pages, Hkv, page_tokens, bytes]; block_table int32 [B, max_pages]."""
    B, M, Hq, _ = q.shape
    Hkv = k_pool.shape[1]
    _check(lib().tq_attn_prefill_paged(_ptr(q), _dtype(q), _ptr(k_pool), ctypes.byref(kcb), _ptr(v_pool),
                                       ctypes.byref(vcb), _ptr(block_table), block_table.shape[1], page_tokens,
                                       _ptr(seq_lens), B, M, Hq, Hkv, T, ctypes.c_float(scale), signs, _ptr(out),
                                       _stream(stream)), "tq_attn_prefill_paged")
    return out


def tq_attn_decode_paged(q, k_pool, kcb, v_pool, vcb, block_table, page_tokens, out, T, scale, signs,
                         seq_lens=None, workspace=None, stream=None):
    """Decode attention over a paged cache: q [B, Hq, 128], out [B, Hq, 128];
    with a workspace (uint8 device tensor) the split-K decode kernels run."""
    B, Hq, _ = q.shape
    Hkv = k_pool.shape[1]
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tq_attn_decode_paged(_ptr(q), _dtype(q), _ptr(k_pool), ctypes.byref(kcb), _ptr(v_pool),
                                      ctypes.byref(vcb), _ptr(block_table), block_table.shape[1], page_tokens,
                                      _ptr(seq_lens), B, Hq, Hkv, T, ctypes.c_float(scale), signs, _ptr(out),
                                      _ptr(workspace), nbytes, _stream(stream)), "tq_attn_decode_paged")
    return out


# ---- head dims 64 / 96 / 128 / 160 (the rotation R is a device float32 [d, d] orthogonal matrix)

def tq_block_bytes_d(head_dim, bits):
    return int(lib().tq_block_bytes_d(head_dim, bits))


def tq_rotation_hadamard(head_dim, signs):
    """R = H D / sqrt(head_dim) (head_dim 64 or 128) as a CPU float32 tensor [d, d]."""
    R = torch.empty((head_dim, head_dim), dtype=torch.float32)
    _check(lib().tq_rotation_hadamard(head_dim, signs, ctypes.c_void_p(R.data_ptr())), "tq_rotation_hadamard")
    return R


def tq_encode_kv_d(x, cb, R, blocks, stream=None):
    """Encode contiguous rows x [n, d] into blocks [n, tq_block_bytes_d(d, bits)]."""
    d = x.shape[-1]
    n = x.numel() // d if d else 0
    _check(lib().tq_encode_kv_d(_ptr(x), _dtype(x), n, d, ctypes.byref(cb), _ptr(R), _ptr(blocks), _stream(stream)),
           "tq_encode_kv_d")
    return blocks


def tq_decode_kv_d(blocks, n_vec, cb, R, out, stream=None):
    """Decode n_vec blocks into contiguous rows out [n_vec, d]."""
    _check(lib().tq_decode_kv_d(_ptr(blocks), n_vec, out.shape[-1], ctypes.byref(cb), _ptr(R), _ptr(out),
                                _dtype(out), _stream(stream)), "tq_decode_kv_d")
    return out


def tq_attn_workspace_bytes_d(B, Hq, Hkv, T_cap, head_dim):
    return int(lib().tq_attn_workspace_bytes_d(B, Hq, Hkv, T_cap, head_dim))


def tq_attn_decode_d(q, k_blocks, kcb, v_blocks, vcb, R, out, workspace, T, scale, seq_lens=None, stream=None):
    """Decode attention at head dim d = q.shape[-1]: q [B, Hq, d]; k/v blocks
    [B, Hkv, T_cap, bytes]; out float32 [B, Hq, d]."""
    B, Hq, d = q.shape
    Hkv, T_cap = k_blocks.shape[1], k_blocks.shape[2]
    _check(lib().tq_attn_decode_d(_ptr(q), _dtype(q), _ptr(k_blocks), ctypes.byref(kcb), _ptr(v_blocks),
                                  ctypes.byref(vcb), _ptr(seq_lens), B, Hq, Hkv, T_cap, T, d, ctypes.c_float(scale),
                                  _ptr(R), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "tq_attn_decode_d")
    return out
