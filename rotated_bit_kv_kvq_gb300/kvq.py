"""Thin Python binding of the kvq C ABI (include/kvq.h).

Argument marshalling only: every step of the write and read paths runs in the
CUDA library.  PyTorch provides device memory and streams.  The functions keep
the C names; ``KVCache`` allocates the planes of one cache with torch and
builds the C descriptor.  Loading fails loudly when the library cannot be
built or loaded -- there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

# ---- constants mirrored from include/kvq.h ---------------------------------
KVQ_OK = 0
KVQ_ERR_INVALID_ARG = -1
KVQ_ERR_UNSUPPORTED = -2
KVQ_ERR_WORKSPACE = -3
KVQ_ERR_CUDA = -4
KVQ_ERR_TIMEOUT = -5
KVQ_ERR_DEVICE_RANGE = -6

KVQ_TYPE_Q4_0, KVQ_TYPE_Q5_0, KVQ_TYPE_Q8_0, KVQ_TYPE_Q4_1, KVQ_TYPE_Q5_1 = 0, 1, 2, 3, 4
TYPE_IDS = {"q4_0": KVQ_TYPE_Q4_0, "q5_0": KVQ_TYPE_Q5_0, "q8_0": KVQ_TYPE_Q8_0,
            "q4_1": KVQ_TYPE_Q4_1, "q5_1": KVQ_TYPE_Q5_1}
KVQ_F32, KVQ_BF16, KVQ_F16 = 0, 1, 2
KVQ_ROT_AUTO, KVQ_ROT_K_OFF, KVQ_ROT_V_OFF = 1, 2, 4
KVQ_INPUT_PREROTATED = 1
(KVQ_PLANE_K_QS, KVQ_PLANE_K_QH, KVQ_PLANE_K_D, KVQ_PLANE_V_QS, KVQ_PLANE_V_QH, KVQ_PLANE_V_D,
 KVQ_PLANE_K_TAIL, KVQ_PLANE_V_TAIL, KVQ_PLANE_SEQ_LEN, KVQ_PLANE_STATUS, KVQ_PLANE_OUTLIER,
 KVQ_PLANE_OUTLIER_IDX) = range(12)
KVQ_NUM_PLANES = 12
KVQ_DEV_ERR_APPEND_RANGE, KVQ_DEV_ERR_PREFILL_RANGE, KVQ_DEV_ERR_TIMEOUT, KVQ_DEV_ERR_PAGE = 1, 2, 4, 8
KVQ_DEV_ERR_OUTLIER = 16


class kvq_cache(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("max_ctx", ctypes.c_int32), ("tail_len", ctypes.c_int32), ("k_type", ctypes.c_int32),
        ("v_type", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("k_qs", ctypes.c_void_p), ("k_qh", ctypes.c_void_p), ("k_d", ctypes.c_void_p),
        ("v_qs", ctypes.c_void_p), ("v_qh", ctypes.c_void_p), ("v_d", ctypes.c_void_p),
        ("k_tail", ctypes.c_void_p), ("v_tail", ctypes.c_void_p),
        ("seq_len", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("page_tokens", ctypes.c_int32), ("n_pages", ctypes.c_int32), ("page_table", ctypes.c_void_p),
        ("n_outlier", ctypes.c_int32), ("outlier_idx", ctypes.c_void_p),
        ("outl", ctypes.c_void_p),
    ]


# every symbol include/kvq.h declares, with its C signature
_P = ctypes.POINTER(kvq_cache)
SIGNATURES = {
    "kvq_version": (ctypes.c_int32, []),
    "kvq_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "kvq_plane_bytes": (ctypes.c_size_t, [_P, ctypes.c_int32]),
    "kvq_cache_check": (ctypes.c_int32, [_P]),
    "kvq_resolve_rotation": (ctypes.c_int32, [_P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "kvq_rotate_quantize_append": (ctypes.c_int32, [_P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                    ctypes.c_int32, ctypes.c_void_p, ctypes.c_uint32,
                                                    ctypes.c_void_p]),
    "kvq_decode_workspace_bytes": (ctypes.c_size_t, [_P, ctypes.c_int32]),
    "kvq_decode_attention": (ctypes.c_int32, [_P, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                              ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_void_p]),
    "kvq_decode_attention_noalloc": (ctypes.c_int32, [_P, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                      ctypes.c_float, ctypes.c_void_p, ctypes.c_int32,
                                                      ctypes.c_void_p]),
    "kvq_append_decode": (ctypes.c_int32, [_P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "kvq_prefill_workspace_bytes": (ctypes.c_size_t, [_P, ctypes.c_int32, ctypes.c_int32]),
    "kvq_prefill_attention": (ctypes.c_int32, [_P, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                               ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                               ctypes.c_void_p]),
    "kvq_dequant_debug": (ctypes.c_int32, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p]),
    "kvq_sync_status": (ctypes.c_int32, [_P, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "kvq_selftest_wait_timeout": (ctypes.c_int32, [_P, ctypes.c_int64, ctypes.c_void_p]),
}

_lib = None


def lib():
    """The loaded C library (built in-tree on first use if stale)."""
    global _lib
    if _lib is None:
        path = _build.ensure_built()
        if not os.path.exists(path):
            raise RuntimeError(f"kvq CUDA library missing at {path}")
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {lib().kvq_status_string(status).decode()} ({status})")
        self.status = status


def _check(status: int, what: str) -> None:
    if status != KVQ_OK:
        raise KvqError(status, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_id(t) -> int:
    import torch
    return {torch.float32: KVQ_F32, torch.bfloat16: KVQ_BF16, torch.float16: KVQ_F16}[t.dtype]


# ---- the C entry points, same names -----------------------------------------

def kvq_rotate_quantize_append(cache: kvq_cache, k, v, n_new_per_seq=None, prerotated=False, stream=None,
                               in_dtype=None, n_new=None):
    """k, v: [batch][n_new][kv_heads][head_dim] device tensors (or raw pointers with in_dtype/n_new)."""
    dt = _dtype_id(k) if in_dtype is None else in_dtype
    n = k.shape[1] if n_new is None else n_new
    _check(lib().kvq_rotate_quantize_append(ctypes.byref(cache), _ptr(k), _ptr(v), dt, n, _ptr(n_new_per_seq),
                                            KVQ_INPUT_PREROTATED if prerotated else 0, _stream(stream)),
           "kvq_rotate_quantize_append")


def kvq_decode_workspace_bytes(cache: kvq_cache, n_q_heads: int) -> int:
    return lib().kvq_decode_workspace_bytes(ctypes.byref(cache), n_q_heads)


def kvq_decode_attention(cache: kvq_cache, q, out, workspace, scale: float = 0.0, stream=None,
                         n_q_heads=None, q_dtype=None, out_dtype=None, ws_bytes=None):
    """q, out: [batch][n_q_heads][head_dim] device tensors; workspace: device byte tensor."""
    nq = q.shape[1] if n_q_heads is None else n_q_heads
    wsb = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib().kvq_decode_attention(ctypes.byref(cache), _ptr(q), _dtype_id(q) if q_dtype is None else q_dtype,
                                      nq, float(scale), _ptr(out),
                                      _dtype_id(out) if out_dtype is None else out_dtype,
                                      _ptr(workspace), wsb, _stream(stream)),
           "kvq_decode_attention")


KVQ_NOALLOC_SCRATCH_BYTES = 16 << 20


def kvq_append_decode(cache: kvq_cache, k, v, q, out, workspace, n_new_per_seq=None, prerotated=False,
                      scale: float = 0.0, stream=None):
    """One decode step: append k, v ([batch][n_new][kv_heads][head_dim]) then decode q
    ([batch][n_q_heads][head_dim]) into out; fused into the decode launch when possible."""
    wsb = workspace.numel() * workspace.element_size()
    _check(lib().kvq_append_decode(ctypes.byref(cache), _ptr(k), _ptr(v), _dtype_id(k), k.shape[1],
                                   _ptr(n_new_per_seq), KVQ_INPUT_PREROTATED if prerotated else 0,
                                   _ptr(q), _dtype_id(q), q.shape[1], float(scale), _ptr(out), _dtype_id(out),
                                   _ptr(workspace), wsb, _stream(stream)),
           "kvq_append_decode")


def kvq_decode_attention_noalloc(cache: kvq_cache, q, out, scale: float = 0.0, stream=None):
    """Decode attention with the library's fixed device scratch instead of a caller workspace."""
    _check(lib().kvq_decode_attention_noalloc(ctypes.byref(cache), _ptr(q), _dtype_id(q), q.shape[1], float(scale),
                                              _ptr(out), _dtype_id(out), _stream(stream)),
           "kvq_decode_attention_noalloc")


def kvq_prefill_workspace_bytes(cache: kvq_cache, n_q_heads: int, n_tokens: int) -> int:
    return lib().kvq_prefill_workspace_bytes(ctypes.byref(cache), n_q_heads, n_tokens)


def kvq_prefill_attention(cache: kvq_cache, q, out, workspace, q_pos0=None, causal=True, chunk=0, scale=0.0,
                          stream=None):
    """q, out: [batch][n_tokens][n_q_heads][head_dim] device tensors."""
    wsb = workspace.numel() * workspace.element_size()
    _check(lib().kvq_prefill_attention(ctypes.byref(cache), _ptr(q), _dtype_id(q), q.shape[2], q.shape[1],
                                       _ptr(q_pos0), 1 if causal else 0, chunk, float(scale), _ptr(out),
                                       _dtype_id(out), _ptr(workspace), wsb, _stream(stream)),
           "kvq_prefill_attention")


def kvq_dequant_debug(cache: kvq_cache, seq, kv_head, which, t0, count, out=None, blocks=None,
                      original_basis=False, stream=None):
    _check(lib().kvq_dequant_debug(ctypes.byref(cache), seq, kv_head, which, t0, count, 1 if original_basis else 0,
                                   _ptr(out), _ptr(blocks), _stream(stream)),
           "kvq_dequant_debug")


def kvq_selftest_wait_timeout(cache: kvq_cache, limit_cycles: int = 1 << 20, stream=None):
    """Launches the bounded wait that nothing completes (sets KVQ_DEV_ERR_TIMEOUT)."""
    _check(lib().kvq_selftest_wait_timeout(ctypes.byref(cache), int(limit_cycles), _stream(stream)),
           "kvq_selftest_wait_timeout")


def kvq_sync_status(cache: kvq_cache, stream=None):
    """Synchronizes; returns (status, raw device bits)."""
    bits = ctypes.c_uint32(0)
    st = lib().kvq_sync_status(ctypes.byref(cache), _stream(stream), ctypes.byref(bits))
    return st, bits.value


def kvq_plane_bytes(cache: kvq_cache, plane: int) -> int:
    return lib().kvq_plane_bytes(ctypes.byref(cache), plane)


def kvq_resolve_rotation(cache: kvq_cache):
    rk, rv = ctypes.c_int32(0), ctypes.c_int32(0)
    st = lib().kvq_resolve_rotation(ctypes.byref(cache), ctypes.byref(rk), ctypes.byref(rv))
    return st, rk.value, rv.value


def default_flags(env=None) -> int:
    """Cache flags when the caller gives none: the automatic enable rule, with K and
    V rotation switched off by the environment variables KVQ_ROT_K_DISABLE /
    KVQ_ROT_V_DISABLE (any value other than empty or "0"), as the patch's own
    per-side switches allow (velog "fix-kv-cache-quantization-outliers", section
    적용 및 배경 기술)."""
    env = os.environ if env is None else env
    on = lambda name: env.get(name, "") not in ("", "0")
    f = KVQ_ROT_AUTO
    if on("KVQ_ROT_K_DISABLE"):
        f |= KVQ_ROT_K_OFF
    if on("KVQ_ROT_V_DISABLE"):
        f |= KVQ_ROT_V_OFF
    return f


def descriptor(batch, n_kv_heads, head_dim, max_ctx, tail_len, k_type, v_type, flags=KVQ_ROT_AUTO,
               page_tokens=0, n_pages=0, n_outlier=0) -> kvq_cache:
    """A descriptor with sizes and types only (pointers NULL)."""
    c = kvq_cache()
    c.batch, c.n_kv_heads, c.head_dim, c.max_ctx, c.tail_len = batch, n_kv_heads, head_dim, max_ctx, tail_len
    c.k_type = TYPE_IDS.get(k_type, k_type)
    c.v_type = TYPE_IDS.get(v_type, v_type)
    c.flags = flags
    c.page_tokens, c.n_pages = page_tokens, n_pages
    c.n_outlier = n_outlier
    return c


class KVCache:
    """The planes of one cache, allocated with torch on the current device."""

    def __init__(self, batch, n_kv_heads, head_dim, max_ctx, tail_len, k_type, v_type,
                 flags=None, device="cuda", page_tokens=0, n_pages=0, page_table=None,
                 outliers=None):
        """flags None: default_flags() (the automatic rule, unless the environment
        switches K or V rotation off).  page_tokens > 0: paged body planes, a pool of n_pages pages (default: batch *
        max_ctx / page_tokens) and a page table (device int32 [batch][max_ctx / page_tokens];
        default: sequence b owns pages b * per_seq ...).  outliers: int [n_kv_heads][32],
        each row the strictly increasing channels kept at 8 bits (None: off)."""
        import torch
        if flags is None:
            flags = default_flags()
        if page_tokens and not n_pages:
            n_pages = batch * (max_ctx // page_tokens)
        n_outlier = 0 if outliers is None else len(outliers[0])
        self.desc = descriptor(batch, n_kv_heads, head_dim, max_ctx, tail_len, k_type, v_type, flags,
                               page_tokens, n_pages, n_outlier)
        if page_tokens:
            per_seq = max_ctx // page_tokens
            if page_table is None:
                page_table = torch.arange(batch * per_seq, dtype=torch.int32, device=device)
            self.page_table = page_table.to(device=device, dtype=torch.int32).contiguous()
            self.desc.page_table = self.page_table.data_ptr()
        self.planes = {}
        names = ["k_qs", "k_qh", "k_d", "v_qs", "v_qh", "v_d", "k_tail", "v_tail", "seq_len", "status",
                 "outl"]
        if n_outlier:
            self.outlier_idx = torch.as_tensor(outliers, dtype=torch.int32).to(device).contiguous()
            if tuple(self.outlier_idx.shape) != (n_kv_heads, n_outlier):
                raise ValueError("outliers: [n_kv_heads][n_outlier]")
            self.desc.outlier_idx = self.outlier_idx.data_ptr()
        for idx, name in enumerate(names):
            nbytes = kvq_plane_bytes(self.desc, idx)
            if nbytes == 0:
                if name in ("k_qs", "v_qs", "k_d", "v_d", "seq_len", "status"):
                    raise ValueError("invalid cache sizes")
                continue
            t = torch.zeros(nbytes, dtype=torch.uint8, device=device)
            self.planes[name] = t
            setattr(self.desc, name, t.data_ptr())
        _check(lib().kvq_cache_check(ctypes.byref(self.desc)), "kvq_cache_check")

    @property
    def seq_len(self):
        import torch
        return self.planes["seq_len"].view(torch.int32)

    def plane(self, name):
        return self.planes[name]

    def reset(self):
        for t in self.planes.values():
            t.zero_()
