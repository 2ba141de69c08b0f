"""ctypes binding of libkvq (include/kvq.h).

Argument marshalling only: every step of the path runs in the CUDA kernels of
libkvq.so.  Tensors are torch tensors on a CUDA device; their ``data_ptr()`` and
the current torch stream are passed straight to the C entry points.  If the
library has not been built, loading raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# KVQ_SANITIZE=1: the host-sanitizer build (argument validation checked on the CPU)
LIB_PATH = os.path.join(_PKG, "_build_san" if os.environ.get("KVQ_SANITIZE") == "1" else "_build", "libkvq.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE_TOO_SMALL = 0, -1, -2, -3, -4
DEV_BAD_SLOT, DEV_BAD_PAGE, DEV_BAD_LENGTH, DEV_BAD_INDEX, DEV_TIMEOUT = 1, 2, 4, 8, 16
DT_F32, DT_BF16 = 0, 1
# Q4_0: the 4-bit rows without the rotation; TQ4: randomized-Hadamard rows with the Lloyd-Max codebook
FMT_Q4_HAD32, FMT_BF16, FMT_FP8_ROW, FMT_Q4_0, FMT_TQ4 = 0, 1, 2, 3, 4

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float


class CacheDesc(ctypes.Structure):
    _fields_ = [("format", _I32), ("num_kv_heads", _I32), ("head_dim", _I32), ("rope_dim", _I32),
                ("page_size", _I32), ("num_pages", _I32), ("k", _P), ("k_scale", _P), ("v", _P), ("v_scale", _P),
                ("signs", _P)]


# name -> (restype, argtypes); mirrors include/kvq.h
SIGNATURES = {
    "kvq_version": (_I32, []),
    "kvq_status_string": (ctypes.c_char_p, [_I32]),
    "kvq_last_cuda_error": (_I32, []),
    "kvq_plane_bytes": (_SZ, [ctypes.POINTER(CacheDesc), _I32]),
    "kvq_store": (_I32, [ctypes.POINTER(CacheDesc), _P, _P, _I32, _I64, _P, _P, _P]),
    "kvq_rotate_query": (_I32, [_P, _I32, _P, _I64, _I32, _P]),
    "kvq_tq4_rotate": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _P, _I64, _I32, _P]),
    "kvq_store_rotate": (_I32, [ctypes.POINTER(CacheDesc), _P, _P, _I32, _I64, _P, _P, _P, _I32, _P, _I64, _P]),
    "kvq_decode_workspace_size": (_SZ, [ctypes.POINTER(CacheDesc), _I32, _I32, _I32, _I32]),
    "kvq_decode_attn": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _I32, _P, _P, _I32, _I32, _P, _I32, _F, _P,
                               _SZ, _P]),
    "kvq_decode_window": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _I32, _P, _P, _I32, _I32, _F, _P, _SZ, _P]),
    "kvq_decode_merged": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _I32, _P, _P, _I32, _I32, _F, _P, _SZ, _P,
                                 _P]),
    "kvq_decode_attn_unrotated": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _I32, _I32, _P, _P, _I32, _I32, _P,
                                         _I32, _F, _P, _SZ, _P]),
    "kvq_decode_step": (_I32, [ctypes.POINTER(CacheDesc), _P, _P, _I32, _P, _I32, _I32, _I32, _P, _P, _I32, _I32, _F,
                               _P, _SZ, _P]),
    "kvq_merge": (_I32, [ctypes.POINTER(CacheDesc), _P, _SZ, _I32, _I32, _P, _I32, _I32, _I32, _P, _P]),
    "kvq_prefill_attn": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _I32, _I32, _I32, _P, _I32, _F, _P, _P, _P]),
    "kvq_read_status": (_I32, [_P, _P, _P]),
    "kvq_prefill_fp8_workspace_size": (_SZ, [ctypes.POINTER(CacheDesc), _I32, _I32]),
    "kvq_selftest_wait_timeout": (_I32, [_P, _P]),
    "kvq_prefill_attn_fp8": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _I32, _I32, _P, _I32, _F, _P, _SZ, _P, _P]),
    "kvq_noalloc_scratch_bytes": (_SZ, []),
    "kvq_decode_noalloc": (_I32, [ctypes.POINTER(CacheDesc), _P, _I32, _I32, _P, _P, _I32, _I32, _P, _I32, _F, _I32,
                                  _P, _P, _P]),
}

_lib = None


def lib():
    """Load libkvq.so (raises if it is missing: the CUDA path has no substitute)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvq.so is not built ({LIB_PATH}); run bit_quantized_kv_store_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class KvqError(RuntimeError):
    def __init__(self, status, where):
        msg = lib().kvq_status_string(status).decode()
        if status == ERR_CUDA:
            msg += f" (cudaError {lib().kvq_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{status}]")
        self.status = status


def _check(status, where):
    if status != OK:
        raise KvqError(status, where)


def _ptr(t):
    """Device address of a tensor for the C ABI (None -> NULL).  The kernels read
    plain row-major device memory, so a host tensor (whose address the GPU would
    fault on) or a strided view (read with the wrong layout) is refused here."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"kvq: expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError("kvq: expected a contiguous tensor (call .contiguous())")
    return t.data_ptr()


# The current stream's handle without building a torch Stream object (the
# accessor torch's own compiler uses; the public route is the fallback).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None):
    """The CUDA stream handle to launch on: `stream`'s, else the current
    device's current torch stream."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dtype_code(t):
    if t.dtype == torch.float32:
        return DT_F32
    if t.dtype == torch.bfloat16:
        return DT_BF16
    raise TypeError(f"unsupported activation dtype {t.dtype}")


class Cache:
    """A paged KV cache: the planes are caller-owned torch tensors on one device.

    Q4:   k, v codes [num_pages, Hk, page_size, D/2] uint8; k_scale, v_scale
          [num_pages, Hk, page_size, D/32] float16.
    BF16: k, v [num_pages, Hk, page_size, D] bfloat16.
    FP8:  k (latent codes) [num_pages, page_size, D] uint8, v (rope codes)
          [num_pages, page_size, R] uint8, k_scale / v_scale [num_pages, page_size] f32.
    TQ4:  k, v codes [num_pages, Hk, page_size, D/2] uint8; k_scale, v_scale
          [num_pages, Hk, page_size] float16; `signs` the rotation's sign mask,
          int32 [D/32] (bit i set: element i negated), given by the caller.
    """

    def __init__(self, fmt, num_kv_heads, head_dim, page_size, num_pages, device="cuda", rope_dim=0, signs=None):
        if torch.device(device).type != "cuda":
            raise ValueError(f"kvq: the cache planes live in device memory, not on {device}")
        self.fmt, self.Hk, self.D, self.page_size, self.num_pages = fmt, num_kv_heads, head_dim, page_size, num_pages
        self.rope = rope_dim
        self.signs = None
        rows = (num_pages, num_kv_heads, page_size)
        if fmt == FMT_TQ4:
            if signs is None or signs.numel() != head_dim // 32:
                raise ValueError("TQ4 needs a sign mask of head_dim / 32 words")
            self.signs = signs.to(device=device, dtype=torch.int32).contiguous()
            self.k = torch.zeros(rows + (head_dim // 2,), dtype=torch.uint8, device=device)
            self.v = torch.zeros_like(self.k)
            self.k_scale = torch.zeros(rows, dtype=torch.float16, device=device)
            self.v_scale = torch.zeros_like(self.k_scale)
        elif fmt in (FMT_Q4_HAD32, FMT_Q4_0):
            self.k = torch.zeros(rows + (head_dim // 2,), dtype=torch.uint8, device=device)
            self.v = torch.zeros_like(self.k)
            self.k_scale = torch.zeros(rows + (head_dim // 32,), dtype=torch.float16, device=device)
            self.v_scale = torch.zeros_like(self.k_scale)
        elif fmt == FMT_BF16:
            self.k = torch.zeros(rows + (head_dim,), dtype=torch.bfloat16, device=device)
            self.v = torch.zeros_like(self.k)
            self.k_scale = self.v_scale = None
        elif fmt == FMT_FP8_ROW:
            assert num_kv_heads == 1
            self.k = torch.zeros(rows + (head_dim,), dtype=torch.uint8, device=device)
            self.v = torch.zeros(rows + (rope_dim,), dtype=torch.uint8, device=device)
            self.k_scale = torch.zeros(rows, dtype=torch.float32, device=device)
            self.v_scale = torch.zeros(rows, dtype=torch.float32, device=device)
        else:
            raise ValueError(fmt)
        self.refresh()

    def refresh(self):
        for t in (self.k, self.v, self.k_scale, self.v_scale, self.signs):
            if t is not None and not (t.is_cuda and t.is_contiguous()):
                raise ValueError("kvq: cache planes must be contiguous CUDA tensors")
        self.desc = CacheDesc(self.fmt, self.Hk, self.D, self.rope, self.page_size, self.num_pages,
                              self.k.data_ptr(), 0 if self.k_scale is None else self.k_scale.data_ptr(),
                              self.v.data_ptr(), 0 if self.v_scale is None else self.v_scale.data_ptr(),
                              0 if self.signs is None else self.signs.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self.desc)

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in (self.k, self.v, self.k_scale, self.v_scale) if t is not None)


def store(cache: Cache, k, v, slot_mapping, status=None, stream=None):
    n_tok = k.shape[0]
    _check(lib().kvq_store(cache.ref, _ptr(k), _ptr(v), _dtype_code(k), n_tok, _ptr(slot_mapping), _ptr(status),
                           _stream(stream)), "kvq_store")


def rotate_query(x, out=None, stream=None):
    D = x.shape[-1]
    rows = x.numel() // D
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    _check(lib().kvq_rotate_query(_ptr(x), _dtype_code(x), _ptr(out), rows, D, _stream(stream)), "kvq_rotate_query")
    return out


def tq4_rotate(cache: Cache, x, inverse=False, out=None, stream=None):
    """The TQ4 cache's signed row transform (queries in; inverse: outputs back)."""
    rows = x.numel() // cache.D
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    _check(lib().kvq_tq4_rotate(cache.ref, _ptr(x), _dtype_code(x), _ptr(out), rows, int(inverse), _stream(stream)),
           "kvq_tq4_rotate")
    return out


def store_rotate(cache: Cache, k, v, slot_mapping, q, out=None, status=None, stream=None):
    """store(cache, k, v, slot_mapping) and rotate_query(q, out) in one launch
    (4-bit format, a few tokens); returns the rotated queries."""
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    rows = q.numel() // q.shape[-1]
    _check(lib().kvq_store_rotate(cache.ref, _ptr(k), _ptr(v), _dtype_code(k), k.shape[0], _ptr(slot_mapping),
                                  _ptr(status), _ptr(q), _dtype_code(q), _ptr(out), rows, _stream(stream)),
           "kvq_store_rotate")
    return out


def workspace_size(cache: Cache, num_seqs, num_q_heads, max_seq_len, n_sel=0):
    return lib().kvq_decode_workspace_size(cache.ref, num_seqs, num_q_heads, max_seq_len, n_sel)


def alloc_workspace(cache: Cache, num_seqs, num_q_heads, max_seq_len, n_sel=0, device="cuda"):
    n = workspace_size(cache, num_seqs, num_q_heads, max_seq_len, n_sel)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_attn(cache: Cache, q, seq_lens, block_tables, max_seq_len, sm_scale, workspace, sel=None, stream=None):
    B, Hq = q.shape[0], q.shape[1]
    n_sel = 0 if sel is None else sel.shape[1]
    _check(lib().kvq_decode_attn(cache.ref, _ptr(q), B, Hq, _ptr(seq_lens), _ptr(block_tables),
                                 block_tables.shape[1], max_seq_len, _ptr(sel), n_sel, float(sm_scale),
                                 _ptr(workspace), workspace.numel(), _stream(stream)), "kvq_decode_attn")


def decode_step(cache: Cache, k_new, v_new, q, seq_lens, block_tables, max_seq_len, sm_scale, workspace,
                stream=None):
    """Store each sequence's new K/V rows at position seq_lens[b] - 1, rotate the
    (unrotated) queries and write the split-T partials, in one launch (4-bit
    formats); merge with merge()."""
    B, Hq = q.shape[0], q.shape[1]
    _check(lib().kvq_decode_step(cache.ref, _ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(q), _dtype_code(q), B,
                                 Hq, _ptr(seq_lens), _ptr(block_tables), block_tables.shape[1], max_seq_len,
                                 float(sm_scale), _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvq_decode_step")


def decode_merged(cache: Cache, q_rot, seq_lens, block_tables, max_seq_len, sm_scale, workspace, out=None,
                  stream=None):
    """Decode partials and their merge in one launch (4-bit formats); q_rot as for
    decode_attn.  Returns out [B, Hq, 256]."""
    B, Hq = q_rot.shape[0], q_rot.shape[1]
    if out is None:
        out = torch.empty((B, Hq, cache.D), dtype=torch.float32, device=q_rot.device)
    _check(lib().kvq_decode_merged(cache.ref, _ptr(q_rot), B, Hq, _ptr(seq_lens), _ptr(block_tables),
                                   block_tables.shape[1], max_seq_len, float(sm_scale), _ptr(workspace),
                                   workspace.numel(), _ptr(out), _stream(stream)), "kvq_decode_merged")
    return out


def decode_window(cache: Cache, q_rot, row_lens, block_table, max_seq_len, sm_scale, workspace, stream=None):
    """Partials for a window of rows of one sequence sharing its block table
    (row i attends keys 0 .. row_lens[i] - 1); merge with merge(num_seqs=rows)."""
    R, Hq = q_rot.shape[0], q_rot.shape[1]
    bt = block_table.reshape(-1)
    _check(lib().kvq_decode_window(cache.ref, _ptr(q_rot), R, Hq, _ptr(row_lens), _ptr(bt), bt.numel(), max_seq_len,
                                   float(sm_scale), _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvq_decode_window")


def decode_window_causal(cache: Cache, q, prefix_len, block_table, sm_scale, workspace, out=None, stream=None):
    """One speculative-decoding verify step: the R rows of q sit at positions
    prefix_len .. prefix_len + R - 1 (their keys already stored) and row i attends
    keys 0 .. prefix_len + i.  Rotates the queries (Hadamard format), decodes the
    window, merges; returns the outputs [R, Hq, D]."""
    R, Hq = q.shape[0], q.shape[1]
    row_lens = torch.arange(prefix_len + 1, prefix_len + R + 1, dtype=torch.int32, device=q.device)
    qq = rotate_query(q, stream=stream) if cache.fmt == FMT_Q4_HAD32 else q.float()
    decode_window(cache, qq, row_lens, block_table, prefix_len + R, sm_scale, workspace, stream=stream)
    if out is None:
        out = torch.empty((R, Hq, cache.D), dtype=torch.float32, device=q.device)
    return merge(cache, workspace, R, Hq, row_lens, prefix_len + R, out, stream=stream)


def decode_attn_unrotated(cache: Cache, q, seq_lens, block_tables, max_seq_len, sm_scale, workspace, sel=None,
                          stream=None):
    """Decode partials from an unrotated query (4-bit format): the rotation runs in the decode kernel."""
    B, Hq = q.shape[0], q.shape[1]
    n_sel = 0 if sel is None else sel.shape[1]
    _check(lib().kvq_decode_attn_unrotated(cache.ref, _ptr(q), _dtype_code(q), B, Hq, _ptr(seq_lens), _ptr(block_tables),
                                           block_tables.shape[1], max_seq_len, _ptr(sel), n_sel, float(sm_scale),
                                           _ptr(workspace), workspace.numel(), _stream(stream)),
           "kvq_decode_attn_unrotated")


def merge(cache: Cache, workspace, num_seqs, num_q_heads, seq_lens, max_seq_len, out, n_sel=0, rotate_back=None,
          stream=None):
    if rotate_back is None:
        rotate_back = cache.fmt in (FMT_Q4_HAD32, FMT_TQ4)
    _check(lib().kvq_merge(cache.ref, _ptr(workspace), workspace.numel(), num_seqs, num_q_heads, _ptr(seq_lens),
                           max_seq_len, n_sel, int(rotate_back), _ptr(out), _stream(stream)), "kvq_merge")
    return out


def decode(cache: Cache, q, seq_lens, block_tables, max_seq_len, sm_scale, workspace, out=None, sel=None,
           stream=None):
    """Rotate the query (4-bit formats), decode partials, merge: one decode step."""
    B, Hq = q.shape[0], q.shape[1]
    qq = q
    if cache.fmt == FMT_Q4_HAD32:
        qq = rotate_query(q, stream=stream)
    elif cache.fmt == FMT_TQ4:
        qq = tq4_rotate(cache, q, stream=stream)
    elif q.dtype != torch.float32:
        qq = q.float()
    decode_attn(cache, qq, seq_lens, block_tables, max_seq_len, sm_scale, workspace, sel=sel, stream=stream)
    if out is None:
        out = torch.empty((B, Hq, cache.D), dtype=torch.float32, device=q.device)
    return merge(cache, workspace, B, Hq, seq_lens, max_seq_len, out, n_sel=0 if sel is None else sel.shape[1],
                 stream=stream)


def prefill_attn(cache: Cache, q, q_start, block_table, sm_scale, out=None, status=None, stream=None):
    n_q, Hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((n_q, Hq, cache.D), dtype=torch.float32, device=q.device)
    bt = block_table.reshape(-1)
    _check(lib().kvq_prefill_attn(cache.ref, _ptr(q), _dtype_code(q), n_q, Hq, int(q_start), _ptr(bt), bt.numel(),
                                  float(sm_scale), _ptr(out), _ptr(status), _stream(stream)), "kvq_prefill_attn")
    return out


def decode_noalloc(cache: Cache, q_rot, seq_lens, block_tables, max_seq_len, sm_scale, out, sel=None,
                   rotate_back=None, status=None, stream=None):
    """Decode partials + merge without a caller workspace (the library's fixed
    device scratch array is used instead; see kvq_decode_noalloc in kvq.h)."""
    B, Hq = q_rot.shape[0], q_rot.shape[1]
    n_sel = 0 if sel is None else sel.shape[1]
    if rotate_back is None:
        rotate_back = cache.fmt in (FMT_Q4_HAD32, FMT_TQ4)
    _check(lib().kvq_decode_noalloc(cache.ref, _ptr(q_rot), B, Hq, _ptr(seq_lens), _ptr(block_tables),
                                    block_tables.shape[1], max_seq_len, _ptr(sel), n_sel, float(sm_scale),
                                    int(rotate_back), _ptr(out), _ptr(status), _stream(stream)), "kvq_decode_noalloc")
    return out


def prefill_attn_fp8(cache: Cache, q, q_start, block_table, sm_scale, workspace=None, out=None, stream=None):
    """Causal prefill of q [n_q, Hq, 576] (positions q_start ..) over the fp8
    latent cache; returns out [n_q, Hq, 512] (the workspace's first word is the
    status)."""
    n_q, Hq = q.shape[0], q.shape[1]
    if workspace is None:
        workspace = torch.zeros(lib().kvq_prefill_fp8_workspace_size(cache.ref, n_q, Hq), dtype=torch.uint8,
                                device=q.device)
    if out is None:
        out = torch.empty((n_q, Hq, cache.D), dtype=torch.float32, device=q.device)
    bt = block_table.reshape(-1)
    _check(lib().kvq_prefill_attn_fp8(cache.ref, _ptr(q), n_q, Hq, int(q_start), _ptr(bt), bt.numel(),
                                      float(sm_scale), _ptr(workspace), workspace.numel(), _ptr(out),
                                      _stream(stream)), "kvq_prefill_attn_fp8")
    return out


def selftest_wait_timeout(d_status, stream=None):
    """Run the bounded-wait diagnostic (about 2 s); KVQ_DEV_TIMEOUT lands in d_status."""
    _check(lib().kvq_selftest_wait_timeout(_ptr(d_status), _stream(stream)), "kvq_selftest_wait_timeout")


def read_status(d_status, stream=None):
    v = ctypes.c_int32(0)
    _check(lib().kvq_read_status(_ptr(d_status), ctypes.byref(v), _stream(stream)), "kvq_read_status")
    return v.value
