"""CPU oracle for the 4-bit / fp8 quantized KV store (test infrastructure only).

This package wraps ``kvq_oracle.c``: a plain, slow, single-threaded C
implementation of what the attention-over-a-quantized-KV-cache path computes.
It is the independent reference that the CUDA library is compared with.  It
shares no code with the library, and only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it.  The product path never does.

Everything here is argument marshalling around the C functions; the
arithmetic lives in the C file, whose header lists the passages it follows
and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
# KVQ_SANITIZE=1: a separate build with AddressSanitizer and UndefinedBehaviorSanitizer
# (run the process with the ASan runtime preloaded; the sanitizer test does).
_SANITIZE = os.environ.get("KVQ_SANITIZE") == "1"
_LIB_PATH = os.path.join(_HERE, "_build", "libkvq_oracle_san.so" if _SANITIZE else "libkvq_oracle.so")
_SAN_FLAGS = ["-O1", "-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined"]
_lock = threading.Lock()
_lib = None

# Formats and input dtypes, mirrored from the C enums of the oracle.  Q4_0: the
# 4-bit rows without the rotation; TQ4: randomized-Hadamard rows with the
# Lloyd-Max codebook.
Q4, BF16, FP8, Q4_0, TQ4 = 0, 1, 2, 3, 4
IN_F32, IN_BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (single-threaded, no fp contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        opt = _SAN_FLAGS if _SANITIZE else ["-O2"]
        # (the compiler runs without a sanitizer runtime a test process may preload)
        env = {k: v for k, v in os.environ.items() if k != "LD_PRELOAD"}
        subprocess.check_call(["gcc", *opt, "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"], env=env)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


class _Cache(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int), ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("rope_dim", ctypes.c_int), ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("k", _P), ("k_scale", _P), ("v", _P), ("v_scale", _P), ("signs", _P)]


def _declare(lib):
    sig = {
        "kvo_f32_to_f16_n": (None, [_P, _P, _I64]),
        "kvo_f32_to_f16_sat_n": (None, [_P, _P, _I64]),
        "kvo_f16_to_f64_n": (None, [_P, _P, _I64]),
        "kvo_f32_to_bf16_n": (None, [_P, _P, _I64]),
        "kvo_f32_to_e4m3_n": (None, [_P, _P, _I64]),
        "kvo_e4m3_to_f64_n": (None, [_P, _P, _I64]),
        "kvo_fwht32_f32_n": (None, [_P, _I64]),
        "kvo_hadamard32_f64_n": (None, [_P, _P, _I64]),
        "kvo_rotation_constant": (ctypes.c_float, []),
        "kvo_q4_quantize_row": (None, [_P, _I32, _P, _P]),
        "kvo_q4_0_quantize_row": (None, [_P, _I32, _P, _P]),
        "kvo_q4_dequant_row": (None, [_P, _P, _I32, _P]),
        "kvo_fp8_encode_row": (ctypes.c_float, [_P, _I32, _P]),
        "kvo_tq4_level": (ctypes.c_double, [_I32]),
        "kvo_tq4_rotate_f32": (None, [_P, _I32, _P, _P]),
        "kvo_tq4_rotate_f64": (None, [_P, _I32, _P, _I32, _P]),
        "kvo_tq4_quantize_row": (ctypes.c_uint16, [_P, _I32, _P, _P]),
        "kvo_tq4_dequant_row": (None, [_P, ctypes.c_uint16, _I32, _P]),
        "kvo_store": (_I32, [ctypes.POINTER(_Cache), _P, _P, _I32, _I64, _P]),
        "kvo_decode": (_I32, [ctypes.POINTER(_Cache), _P, _I32, _I32, _I32, _P, _P, _I32, _P, _I32,
                              ctypes.c_double, _I32, _P]),
        "kvo_prefill": (_I32, [ctypes.POINTER(_Cache), _P, _I32, _I32, _I32, _I64, _P, _P, _I32,
                               ctypes.c_double, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- scalar formats

def f32_to_f16_bits(x, saturate=False):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint16)
    (_L().kvo_f32_to_f16_sat_n if saturate else _L().kvo_f32_to_f16_n)(_ptr(x), _ptr(y), x.size)
    return y


def f16_bits_to_f64(h):
    h = _c(h, np.uint16)
    y = np.empty(h.shape, np.float64)
    _L().kvo_f16_to_f64_n(_ptr(h), _ptr(y), h.size)
    return y


def f32_to_bf16_bits(x):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint16)
    _L().kvo_f32_to_bf16_n(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_e4m3(x):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint8)
    _L().kvo_f32_to_e4m3_n(_ptr(x), _ptr(y), x.size)
    return y


def e4m3_to_f64(c):
    c = _c(c, np.uint8)
    y = np.empty(c.shape, np.float64)
    _L().kvo_e4m3_to_f64_n(_ptr(c), _ptr(y), c.size)
    return y


def fwht32_f32(x):
    """fp32 butterfly rotation of every 32-group (the store's rotation)."""
    y = _c(x, np.float32).copy()
    assert y.size % 32 == 0
    _L().kvo_fwht32_f32_n(_ptr(y), y.size // 32)
    return y


def hadamard32_f64(x):
    """fp64 y = H x of every 32-group by the matrix definition."""
    x = _c(x, np.float64)
    y = np.empty_like(x)
    _L().kvo_hadamard32_f64_n(_ptr(x), _ptr(y), x.size // 32)
    return y


def rotation_constant():
    return _L().kvo_rotation_constant()


def q4_quantize_row(x, rotate=True):
    """One row of D fp32 values -> (stored codes [D/2] u8: group G at bytes 16G ..,
    element 2b / 2b+1 in the low / high nibble of byte b of its group; scales [D/32]
    fp16 bits); rotate=False: the unrotated Q4_0 form."""
    x = _c(x, np.float32)
    D = x.size
    codes = np.empty(D // 2, np.uint8)
    sc = np.empty(D // 32, np.uint16)
    (_L().kvo_q4_quantize_row if rotate else _L().kvo_q4_0_quantize_row)(_ptr(x), D, _ptr(codes), _ptr(sc))
    return codes, sc


def q4_dequant_row(stored, scales):
    stored = _c(stored, np.uint8)
    scales = _c(scales, np.uint16)
    D = stored.size * 2
    out = np.empty(D, np.float64)
    _L().kvo_q4_dequant_row(_ptr(stored), _ptr(scales), D, _ptr(out))
    return out


def tq4_levels():
    """The 16 TQ4 levels, indexed by code (code & 8: negative)."""
    return np.array([_L().kvo_tq4_level(c) for c in range(16)])


def tq4_rotate_f32(x, signs):
    """The store's fp32 signed butterfly of one row."""
    x = _c(x, np.float32)
    y = np.empty_like(x)
    _L().kvo_tq4_rotate_f32(_ptr(x), x.size, _ptr(_c(signs, np.uint32)), _ptr(y))
    return y


def tq4_rotate_f64(x, signs, inverse=False):
    """The signed transform by its matrix definition (fp64), forward or inverse."""
    x = _c(x, np.float64)
    y = np.empty_like(x)
    _L().kvo_tq4_rotate_f64(_ptr(x), x.size, _ptr(_c(signs, np.uint32)), int(inverse), _ptr(y))
    return y


def tq4_quantize_row(x, signs):
    """One row -> (codes [n/2] u8, fp16 scale bits)."""
    x = _c(x, np.float32)
    codes = np.empty(x.size // 2, np.uint8)
    sc = _L().kvo_tq4_quantize_row(_ptr(x), x.size, _ptr(_c(signs, np.uint32)), _ptr(codes))
    return codes, np.uint16(sc)


def tq4_dequant_row(codes, scale):
    """Rotated-space values of a stored TQ4 row (fp64)."""
    codes = _c(codes, np.uint8)
    out = np.empty(codes.size * 2, np.float64)
    _L().kvo_tq4_dequant_row(_ptr(codes), int(scale), codes.size * 2, _ptr(out))
    return out


def fp8_encode_row(x):
    x = _c(x, np.float32)
    codes = np.empty(x.size, np.uint8)
    s = _L().kvo_fp8_encode_row(_ptr(x), x.size, _ptr(codes))
    return codes, np.float32(s)


# --------------------------------------------------------------------------- cache

class Cache:
    """A paged KV cache held in numpy arrays, laid out as the library's planes.

    Q4, Q4_0: k/v codes [num_pages, Hk, page_size, D/2] u8, scales [.., D/32] fp16 bits
    BF16: k/v [num_pages, Hk, page_size, D] bf16 bits, no scales
    FP8:  latent codes [num_pages, page_size, D] u8, rope codes [.., rope] u8,
          latent / rope scales [num_pages, page_size] f32
    TQ4:  k/v codes [num_pages, Hk, page_size, D/2] u8, one scale per row
          [num_pages, Hk, page_size] fp16 bits; `signs` the rotation's sign mask
          [D/32] u32 (bit i set: element i negated)
    """

    def __init__(self, fmt, num_kv_heads, head_dim, page_size, num_pages, rope_dim=0, signs=None):
        self.fmt, self.Hk, self.D, self.page_size, self.num_pages = fmt, num_kv_heads, head_dim, page_size, num_pages
        self.rope = rope_dim
        self.signs = None if signs is None else _c(signs, np.uint32)
        rows = (num_pages, num_kv_heads, page_size)
        if fmt == TQ4:
            assert self.signs is not None and self.signs.size == head_dim // 32
            self.k = np.zeros(rows + (head_dim // 2,), np.uint8)
            self.v = np.zeros_like(self.k)
            self.k_scale = np.zeros(rows, np.uint16)
            self.v_scale = np.zeros_like(self.k_scale)
        elif fmt in (Q4, Q4_0):
            self.k = np.zeros(rows + (head_dim // 2,), np.uint8)
            self.v = np.zeros_like(self.k)
            self.k_scale = np.zeros(rows + (head_dim // 32,), np.uint16)
            self.v_scale = np.zeros_like(self.k_scale)
        elif fmt == BF16:
            self.k = np.zeros(rows + (head_dim,), np.uint16)
            self.v = np.zeros_like(self.k)
            self.k_scale = self.v_scale = None
        else:
            assert num_kv_heads == 1
            self.k = np.zeros(rows + (head_dim,), np.uint8)
            self.v = np.zeros(rows + (rope_dim,), np.uint8)
            self.k_scale = np.zeros(rows, np.float32)
            self.v_scale = np.zeros(rows, np.float32)

    def _struct(self):
        return _Cache(self.fmt, self.Hk, self.D, self.rope, self.page_size, self.num_pages,
                      _ptr(self.k), _ptr(self.k_scale), _ptr(self.v), _ptr(self.v_scale), _ptr(self.signs))


def _in(x):
    """Input tensor -> (contiguous array, dtype code).  bf16 inputs come as uint16 bits."""
    if x.dtype == np.uint16:
        return _c(x, np.uint16), IN_BF16
    return _c(x, np.float32), IN_F32


def store(cache: Cache, k, v, slot_mapping):
    """Quantise and write n_tok tokens; returns the number of out-of-range slots."""
    k, dt = _in(k)
    if v is not None:
        v, dt2 = _in(v)
        assert dt2 == dt
    sm = _c(slot_mapping, np.int32)
    s = cache._struct()
    return _L().kvo_store(ctypes.byref(s), _ptr(k), _ptr(v), dt, sm.size, _ptr(sm))


def decode(cache: Cache, q, seq_lens, block_tables, sm_scale, sel=None, split=False):
    """Decode attention, fp64 output [B, Hq, value width]."""
    q, dt = _in(q)
    B, Hq = q.shape[0], q.shape[1]
    sl = _c(seq_lens, np.int32)
    bt = _c(block_tables, np.int32)
    n_sel = 0
    if sel is not None:
        sel = _c(sel, np.int32)
        n_sel = sel.shape[1]
    out = np.zeros((B, Hq, cache.D), np.float64)
    s = cache._struct()
    ok = _L().kvo_decode(ctypes.byref(s), _ptr(q), dt, B, Hq, _ptr(sl), _ptr(bt), bt.shape[1],
                         _ptr(sel), n_sel, float(sm_scale), int(split), _ptr(out))
    if not ok:
        raise ValueError("oracle: block table points outside the pool")
    return out


def prefill(cache: Cache, q, q_start, block_table, sm_scale, rows=None):
    """Causal prefill over decoded slots, fp64 output [n_rows or n_q, Hq, D]."""
    q, dt = _in(q)
    n_q, Hq = q.shape[0], q.shape[1]
    bt = _c(block_table, np.int32).reshape(-1)
    r = None if rows is None else _c(rows, np.int32)
    n_rows = n_q if r is None else r.size
    out = np.zeros((n_rows, Hq, cache.D), np.float64)
    s = cache._struct()
    ok = _L().kvo_prefill(ctypes.byref(s), _ptr(q), dt, n_q, Hq, int(q_start), _ptr(bt), _ptr(r),
                          n_rows, float(sm_scale), _ptr(out))
    if not ok:
        raise ValueError("oracle: block table points outside the pool")
    return out
