"""Python binding of libpkv: paged-KV grouped-query attention for GB300 (sm_103a).

Argument marshalling only: every function here has the name of a ``pkv_*``
entry point of ``include/pkv.h`` and forwards to it through ctypes.  Device
arrays are torch CUDA tensors (f32, contiguous); host arrays are numpy arrays
or CPU tensors; streams are ``torch.cuda.Stream`` objects, raw ``cudaStream_t``
integers or None.  Constructors return an opaque handle or None (check
``pkv_last_error()``); the rest return the library's status code.

The library must be built first (``python paged_kv_gqa_nx_gb300/build.py`` or
``__graft_entry__.build()``); importing this package without it raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_ERR_BAD_DIM = 1
PKV_ERR_BAD_GQA = 2
PKV_ERR_SEQ = 3
PKV_ERR_EXHAUSTED = 4
PKV_ERR_CAPACITY = 5
PKV_ERR_ARG = 6
PKV_ERR_CUDA = 7
PKV_ERR_DEVICE_BOUNDS = 8
PKV_ERR_DEVICE_TIMEOUT = 9

PKV_DEVERR_BOUNDS = 1
PKV_DEVERR_TIMEOUT = 2
PKV_ERRWORD_POOL = 0
PKV_ERRWORD_CONTIGUOUS = 1
PKV_ERRWORD_NOALLOC = 2

PKV_POOL_HOST_ONLY = 1
PKV_POOL_BF16 = 2
PKV_POOL_FP8 = 4
PKV_NOALLOC_SCRATCH_BYTES = 16 << 20

PKV_KERNEL_APPEND = 0
PKV_KERNEL_DECODE = 1
PKV_KERNEL_MERGE = 2
PKV_KERNEL_PREFILL = 3
PKV_KERNEL_COPY = 4
PKV_KERNEL_PAGETABLE = 5
PKV_KERNEL_SPLIT = 6
PKV_KERNEL_KINDS = 7
KERNEL_NAMES = ["append", "decode", "merge", "prefill", "copy", "pagetable", "split"]


class PkvError(RuntimeError):
    def __init__(self, rc: int, what: str = ""):
        super().__init__("pkv error %d: %s" % (rc, what or pkv_last_error()))
        self.rc = rc


if not os.path.exists(LIB_PATH):
    raise ImportError("libpkv.so is not built (%s); run `python paged_kv_gqa_nx_gb300/build.py`"
                      % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_f32 = ctypes.c_float
_int = ctypes.c_int
_pi32 = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "pkv_pool_new": (_vp, [_i32, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _u32]),
    "pkv_pool_free": (None, [_vp]),
    "pkv_pool_set_stream": (_int, [_vp, _vp]),
    "pkv_pool_k_data": (_vp, [_vp]),
    "pkv_pool_v_data": (_vp, [_vp]),
    "pkv_pool_free_blocks": (_i32, [_vp]),
    "pkv_alloc_block": (_i64, [_vp]),
    "pkv_unref_block": (_int, [_vp, _i64]),
    "pkv_refcnt": (_i32, [_vp, _i64]),
    "pkv_seq_new": (_vp, [_vp, _i32]),
    "pkv_seq_fork": (_vp, [_vp]),
    "pkv_seq_free": (_int, [_vp]),
    "pkv_seq_truncate": (_int, [_vp, _i32]),
    "pkv_seq_truncate_batch": (_int, [_vp, _i32, _pi32]),
    "pkv_seq_len": (_i32, [_vp]),
    "pkv_seq_page_table": (_i32, [_vp, _pi32, _i32]),
    "pkv_seq_slot": (_i32, [_vp]),
    "pkv_ensure_append": (_int, [_vp, _i32]),
    "pkv_ensure_append_batch": (_int, [_vp, _i32, _pi32]),
    "pkv_advance": (_int, [_vp, _i32]),
    "pkv_advance_batch": (_int, [_vp, _i32, _pi32]),
    "pkv_append_layer": (_int, [_vp, _i32, _vp, _vp, _i32]),
    "pkv_attn_with_paged": (_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _i32, _f32, _vp]),
    "pkv_attn_batch": (_int, [_vp, _i32, _pi32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp]),
    "pkv_attn_batch_host": (_int, [_vp, _i32, _pi32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp]),
    "pkv_attn_batch_rope": (_int, [_vp, _i32, _pi32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32,
                                   ctypes.c_double, _vp]),
    "pkv_attn_contiguous": (_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp]),
    "pkv_attn_contiguous_noalloc": (_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp]),
    "pkv_sync_error": (_int, [_vp]),
    "pkv_contiguous_sync_error": (_int, [_vp]),
    "pkv_debug_or_error_bits": (_int, [_vp, _i32, _u32]),
    "pkv_pool_flush": (_int, [_vp]),
    "pkv_set_split_keys": (_int, [_i32]),
    "pkv_get_split_keys": (_i32, []),
    "pkv_set_fused_append": (_int, [_i32]),
    "pkv_get_fused_append": (_i32, []),
    "pkv_set_cascade": (_int, [_i32]),
    "pkv_pool_last_work": (_int, [_vp, ctypes.POINTER(ctypes.c_int64), _i32]),
    "pkv_pool_set_image_cache": (_int, [_vp, ctypes.c_int64]),
    "pkv_pool_set_kv_scale": (_int, [_vp, _f32]),
    "pkv_get_cascade": (_i32, []),
    "pkv_set_prefill_pairing": (_int, [_i32]),
    "pkv_get_prefill_pairing": (_i32, []),
    "pkv_launch_count": (_i64, []),
    "pkv_profile_enable": (_int, [_i32]),
    "pkv_profile_reset": (_int, []),
    "pkv_profile_read": (_int, [_i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]),
    "pkv_probe_tf32_mma": (_int, [_i32, _i32, _i32, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)]),
    "pkv_probe_f16_mma": (_int, [_i32, _i32, _i32, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)]),
    "pkv_last_error": (ctypes.c_char_p, []),
}

for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


# ------------------------------------------------------------ marshalling ----

def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _dev(t, name="tensor", dtypes=("float32",)):
    """Device address of a contiguous CUDA tensor of one of `dtypes` (default
    f32), or a raw int address."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if str(t.dtype).replace("torch.", "") not in dtypes or not t.is_contiguous():
        raise TypeError("%s must be a contiguous %s tensor" % (name, " or ".join(dtypes)))
    return t.data_ptr()


def _host(a, name="array"):
    """Host address of a contiguous f32 numpy array or CPU tensor."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.is_cuda or a.dtype != torch.float32 or not a.is_contiguous():
                raise TypeError("%s must be a contiguous float32 CPU tensor" % name)
            return a.data_ptr()
    except ImportError:
        pass
    import numpy as np
    if not isinstance(a, np.ndarray) or a.dtype != np.float32 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError("%s must be a contiguous float32 array" % name)
    return a.ctypes.data


def _seq_array(seqs):
    if isinstance(seqs, ctypes.Array):
        return seqs
    return (_vp * len(seqs))(*seqs)


def _i32_array(vals):
    if isinstance(vals, ctypes.Array):
        return vals
    vals = [int(v) for v in vals]
    return (_i32 * max(1, len(vals)))(*vals)


def seq_array(seqs):
    """A reusable ctypes array of sequence handles (saves re-marshalling a
    batch on every call)."""
    return (_vp * len(seqs))(*seqs)


def i32_array(vals):
    """A reusable ctypes int32 array (per-row counts or lengths)."""
    return (_i32 * max(1, len(vals)))(*[int(v) for v in vals])


# ------------------------------------------------------------ entry points ----

def pkv_last_error() -> str:
    return (_lib.pkv_last_error() or b"").decode()


def pkv_pool_new(n_blocks, n_layers, kv_dim, block_size, k_pool=None, v_pool=None,
                 max_seqs=1024, max_blocks_per_seq=4096, stream=None, flags=0):
    """k_pool / v_pool: float32 tensors, bfloat16 with flags |= PKV_POOL_BF16,
    float8_e4m3fn (or uint8) with flags |= PKV_POOL_FP8."""
    want = (("bfloat16",) if flags & PKV_POOL_BF16 else
            ("float8_e4m3fn", "uint8") if flags & PKV_POOL_FP8 else ("float32",))
    return _lib.pkv_pool_new(n_blocks, n_layers, kv_dim, block_size, _dev(k_pool, "k_pool", want),
                             _dev(v_pool, "v_pool", want), max_seqs, max_blocks_per_seq,
                             _stream(stream), flags)


def pkv_pool_free(pool):
    _lib.pkv_pool_free(pool)


def pkv_pool_set_stream(pool, stream):
    return _lib.pkv_pool_set_stream(pool, _stream(stream))


def pkv_pool_k_data(pool):
    return _lib.pkv_pool_k_data(pool)


def pkv_pool_v_data(pool):
    return _lib.pkv_pool_v_data(pool)


def pkv_pool_free_blocks(pool):
    return _lib.pkv_pool_free_blocks(pool)


def pkv_alloc_block(pool):
    return _lib.pkv_alloc_block(pool)


def pkv_unref_block(pool, block_id):
    return _lib.pkv_unref_block(pool, block_id)


def pkv_refcnt(pool, block_id):
    return _lib.pkv_refcnt(pool, block_id)


def pkv_seq_new(pool, max_tokens):
    return _lib.pkv_seq_new(pool, max_tokens)


def pkv_seq_fork(seq):
    return _lib.pkv_seq_fork(seq)


def pkv_seq_free(seq):
    return _lib.pkv_seq_free(seq)


def pkv_seq_truncate(seq, new_len):
    return _lib.pkv_seq_truncate(seq, new_len)


def pkv_seq_truncate_batch(seqs, new_len):
    return _lib.pkv_seq_truncate_batch(_seq_array(seqs), len(seqs), _i32_array(new_len))


def pkv_seq_len(seq):
    return _lib.pkv_seq_len(seq)


def pkv_seq_slot(seq):
    return _lib.pkv_seq_slot(seq)


def pkv_seq_page_table(seq):
    """The page table as a list of block ids."""
    n = _lib.pkv_seq_page_table(seq, None, 0)
    if n < 0:
        return None
    buf = (_i32 * max(1, n))()
    _lib.pkv_seq_page_table(seq, buf, n)
    return list(buf[:n])


def pkv_ensure_append(seq, n):
    return _lib.pkv_ensure_append(seq, n)


def pkv_ensure_append_batch(seqs, n):
    return _lib.pkv_ensure_append_batch(_seq_array(seqs), len(seqs), _i32_array(n))


def pkv_advance(seq, n):
    return _lib.pkv_advance(seq, n)


def pkv_advance_batch(seqs, n):
    return _lib.pkv_advance_batch(_seq_array(seqs), len(seqs), _i32_array(n))


def pkv_append_layer(seq, layer, K_new, V_new, n_tokens):
    return _lib.pkv_append_layer(seq, layer, _dev(K_new, "K_new"), _dev(V_new, "V_new"), n_tokens)


def pkv_attn_with_paged(Q, K_new, V_new, n_tokens, n_heads, n_kv_heads, head_dim, seq, layer,
                        causal, scale, out):
    return _lib.pkv_attn_with_paged(_dev(Q, "Q"), _dev(K_new, "K_new"), _dev(V_new, "V_new"),
                                    n_tokens, n_heads, n_kv_heads, head_dim, seq, layer, causal,
                                    scale, _dev(out, "out"))


def pkv_attn_batch(seqs, n_q, Q, K_new, V_new, n_heads, n_kv_heads, head_dim, layer, causal,
                   scale, out):
    return _lib.pkv_attn_batch(_seq_array(seqs), len(seqs), _i32_array(n_q), _dev(Q, "Q"),
                               _dev(K_new, "K_new"), _dev(V_new, "V_new"), n_heads, n_kv_heads,
                               head_dim, layer, causal, scale, _dev(out, "out"))


def pkv_attn_batch_rope(seqs, n_q, Q, K_new, V_new, n_heads, n_kv_heads, head_dim, layer, causal,
                        scale, rope_base, out):
    return _lib.pkv_attn_batch_rope(_seq_array(seqs), len(seqs), _i32_array(n_q), _dev(Q, "Q"),
                                    _dev(K_new, "K_new"), _dev(V_new, "V_new"), n_heads,
                                    n_kv_heads, head_dim, layer, causal, scale, float(rope_base),
                                    _dev(out, "out"))


def pkv_attn_batch_host(seqs, n_q, Q, K_new, V_new, n_heads, n_kv_heads, head_dim, layer, causal,
                        scale, out):
    return _lib.pkv_attn_batch_host(_seq_array(seqs), len(seqs), _i32_array(n_q), _host(Q, "Q"),
                                    _host(K_new, "K_new"), _host(V_new, "V_new"), n_heads,
                                    n_kv_heads, head_dim, layer, causal, scale, _host(out, "out"))


def pkv_attn_contiguous(Q, Kc, Vc, n_q, total_k, n_heads, n_kv_heads, head_dim, causal, scale,
                        out, stream=None):
    return _lib.pkv_attn_contiguous(_dev(Q, "Q"), _dev(Kc, "Kc"), _dev(Vc, "Vc"), n_q, total_k,
                                    n_heads, n_kv_heads, head_dim, causal, scale, _dev(out, "out"),
                                    _stream(stream))


def pkv_attn_contiguous_noalloc(Q, Kc, Vc, n_q, total_k, n_heads, n_kv_heads, head_dim, causal,
                                scale, out, stream=None):
    """pkv_attn_contiguous without any device allocation (static scratch of
    PKV_NOALLOC_SCRATCH_BYTES; see include/pkv.h)."""
    return _lib.pkv_attn_contiguous_noalloc(_dev(Q, "Q"), _dev(Kc, "Kc"), _dev(Vc, "Vc"), n_q,
                                            total_k, n_heads, n_kv_heads, head_dim, causal, scale,
                                            _dev(out, "out"), _stream(stream))


def pkv_sync_error(pool):
    return _lib.pkv_sync_error(pool)


def pkv_contiguous_sync_error(stream=None):
    return _lib.pkv_contiguous_sync_error(_stream(stream))


def pkv_debug_or_error_bits(pool, which, bits):
    return _lib.pkv_debug_or_error_bits(pool, which, bits)


def pkv_pool_flush(pool):
    return _lib.pkv_pool_flush(pool)


def pkv_set_split_keys(keys):
    return _lib.pkv_set_split_keys(keys)


def pkv_get_split_keys():
    return _lib.pkv_get_split_keys()


def pkv_set_fused_append(on):
    return _lib.pkv_set_fused_append(1 if on else 0)


def pkv_get_fused_append():
    return bool(_lib.pkv_get_fused_append())


PKV_WORK_FIELDS = 11
WORK_FIELD_NAMES = ("decode_units", "prefill_tiles", "prefix_tiles", "merge_items",
                    "prefill_pairs", "prefix_pairs", "fused_append", "image_hits", "image_builds",
                    "prefix_split_keys", "prefill_ctas")


def pkv_pool_last_work(pool):
    """The pool's last attend call's work list as a dict (see WORK_FIELD_NAMES)."""
    buf = (ctypes.c_int64 * PKV_WORK_FIELDS)()
    check(_lib.pkv_pool_last_work(pool, buf, PKV_WORK_FIELDS))
    return dict(zip(WORK_FIELD_NAMES, list(buf)))


def pkv_pool_set_image_cache(pool, max_bytes):
    return _lib.pkv_pool_set_image_cache(pool, int(max_bytes))


def pkv_pool_set_kv_scale(pool, scale):
    return _lib.pkv_pool_set_kv_scale(pool, float(scale))


def pkv_set_cascade(on):
    return _lib.pkv_set_cascade(1 if on else 0)


def pkv_get_cascade():
    return bool(_lib.pkv_get_cascade())


def pkv_set_prefill_pairing(mode):
    return _lib.pkv_set_prefill_pairing(int(mode))


def pkv_get_prefill_pairing():
    return _lib.pkv_get_prefill_pairing()


def pkv_launch_count():
    return _lib.pkv_launch_count()


def pkv_profile_enable(on):
    return _lib.pkv_profile_enable(1 if on else 0)


def pkv_profile_reset():
    return _lib.pkv_profile_reset()


def pkv_profile_read(kind):
    """(total device ms, launches) of kernel kind ``kind`` since the last reset."""
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    rc = _lib.pkv_profile_read(kind, ctypes.byref(ms), ctypes.byref(n))
    if rc != PKV_OK:
        raise PkvError(rc)
    return ms.value, n.value


def pkv_probe_tf32_mma(n_cols, a_in_tmem=True, iters=4096):
    """(SM clocks per MMA, TFLOP/s) of back-to-back tcgen05.mma kind::tf32,
    M = 128, N = n_cols (see include/pkv.h)."""
    clk = ctypes.c_double()
    tf = ctypes.c_double()
    check(_lib.pkv_probe_tf32_mma(int(n_cols), 1 if a_in_tmem else 0, int(iters), ctypes.byref(clk),
                                  ctypes.byref(tf)))
    return clk.value, tf.value


def pkv_probe_f16_mma(n_cols, a_in_tmem=True, iters=4096):
    """(SM clocks per MMA, TFLOP/s) of back-to-back tcgen05.mma kind::f16,
    M = 128, N = n_cols, K = 16 (see include/pkv.h)."""
    clk = ctypes.c_double()
    tf = ctypes.c_double()
    check(_lib.pkv_probe_f16_mma(int(n_cols), 1 if a_in_tmem else 0, int(iters), ctypes.byref(clk),
                                 ctypes.byref(tf)))
    return clk.value, tf.value


def check(rc: int, what: str = "") -> None:
    """Raise PkvError unless rc is PKV_OK."""
    if rc != PKV_OK:
        raise PkvError(rc, what)


def exported_symbols():
    return sorted(_SIGS)
