"""Host-only checks of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every symbol include/kvq.h declares, and rejects bad arguments on
the host before any launch.  No compute call is made."""

import ctypes
import os
import re

import pytest

from rotated_bit_kv_kvq_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(built_lib_path):
    names = _declared_functions()
    assert len(names) >= 12
    assert set(names) == set(kvq.SIGNATURES), "binding signatures out of sync with include/kvq.h"
    handle = ctypes.CDLL(built_lib_path)
    for n in names:
        assert hasattr(handle, n), n
    assert kvq.lib().kvq_version() == 1


def _header_defines():
    """Integer #defines of include/kvq.h (name -> value): plain integers and
    shifted ones of the form (Nu << M)."""
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    out = {}
    for name, val in re.findall(r"^#define\s+(KVQ_[A-Z0-9_]+)\s+(-?\d+)u?\b", src, flags=re.M):
        out[name] = int(val)
    for name, a, sh in re.findall(r"^#define\s+(KVQ_[A-Z0-9_]+)\s+\(\s*(\d+)u?\s*<<\s*(\d+)\s*\)", src, flags=re.M):
        out[name] = int(a) << int(sh)
    return out


def test_binding_constants_match_header():
    """Every integer constant of the header that the binding mirrors has the same value."""
    defs = _header_defines()
    assert len(defs) >= 30
    mirrored = [n for n in defs if hasattr(kvq, n)]
    assert len(mirrored) >= 30, sorted(set(defs) - set(mirrored))
    for n in mirrored:
        assert getattr(kvq, n) == defs[n], n
    # the scratch size of the allocation-free entry point is written as a shift
    assert defs["KVQ_NOALLOC_SCRATCH_BYTES"] == kvq.KVQ_NOALLOC_SCRATCH_BYTES == 16 << 20
    # the binding's kvq_cache has the header's fields in the header's order
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    body = re.search(r"typedef struct kvq_cache \{(.*?)\} kvq_cache;", src, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b([a-z_][a-z0-9_]*)\s*[;,]", body)
    assert fields == [f for f, _ in kvq.kvq_cache._fields_]


def test_status_strings(built_lib_path):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert kvq.lib().kvq_status_string(s)
    assert kvq.lib().kvq_status_string(-99) == b"unknown status"


def _desc(**kw):
    base = dict(batch=2, n_kv_heads=4, head_dim=128, max_ctx=256, tail_len=32, k_type="q8_0", v_type="q4_0")
    base.update(kw)
    return kvq.descriptor(**base)


def test_plane_bytes(built_lib_path):
    c = _desc()
    rows = 2 * 4 * 256
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_K_QS) == rows * 128
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_V_QS) == rows * 64
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_K_QH) == 0
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_K_D) == rows * 4 * 2
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_K_TAIL) == 2 * 4 * 32 * 128 * 2
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_SEQ_LEN) == 8
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_STATUS) == 16
    c5 = _desc(k_type="q5_0", v_type="q5_0")
    assert kvq.kvq_plane_bytes(c5, kvq.KVQ_PLANE_V_QH) == rows * 4 * 4
    # packed bytes per token-head equal the GGUF block sizes (18 / 22 / 34 per 32 values)
    for qt, blk in (("q4_0", 18), ("q5_0", 22), ("q8_0", 34), ("q4_1", 20), ("q5_1", 24)):
        c = _desc(k_type=qt, v_type=qt)
        per = sum(kvq.kvq_plane_bytes(c, p) for p in (kvq.KVQ_PLANE_K_QS, kvq.KVQ_PLANE_K_QH, kvq.KVQ_PLANE_K_D))
        assert per == rows * (128 // 32) * blk
    # paged: a pool of n_pages pages of page_tokens rows per KV head
    cp = kvq.descriptor(2, 4, 128, 256, 32, "q8_0", "q4_0", page_tokens=64, n_pages=11)
    assert kvq.kvq_plane_bytes(cp, kvq.KVQ_PLANE_K_QS) == 11 * 4 * 64 * 128
    assert kvq.kvq_plane_bytes(cp, kvq.KVQ_PLANE_V_D) == 11 * 4 * 64 * 4 * 2
    assert kvq.kvq_plane_bytes(cp, kvq.KVQ_PLANE_K_TAIL) == 2 * 4 * 32 * 128 * 2   # the tail is not paged
    for bad in (dict(page_tokens=32, n_pages=4), dict(page_tokens=192, n_pages=4), dict(page_tokens=64, n_pages=0),
                dict(page_tokens=0, n_pages=3)):
        assert kvq.kvq_plane_bytes(kvq.descriptor(2, 4, 128, 256, 32, "q8_0", "q4_0", **bad), 0) == 0, bad
    assert kvq.kvq_plane_bytes(_desc(head_dim=100), 0) == 0
    assert kvq.kvq_plane_bytes(_desc(max_ctx=100), 0) == 0


@pytest.mark.parametrize("d,flags,expect", [
    (64, kvq.KVQ_ROT_AUTO, (0, 1, 1)),
    (128, kvq.KVQ_ROT_AUTO, (0, 1, 1)),
    (192, kvq.KVQ_ROT_AUTO, (0, 1, 1)),
    (96, kvq.KVQ_ROT_AUTO, (0, 0, 0)),
    (32, kvq.KVQ_ROT_AUTO, (0, 0, 0)),
    (96, 0, (kvq.KVQ_ERR_UNSUPPORTED, 0, 0)),
    (96, kvq.KVQ_ROT_K_OFF | kvq.KVQ_ROT_V_OFF, (0, 0, 0)),
    (128, 0, (0, 1, 1)),
    (128, kvq.KVQ_ROT_AUTO | kvq.KVQ_ROT_K_OFF, (0, 0, 1)),
    (128, kvq.KVQ_ROT_AUTO | kvq.KVQ_ROT_V_OFF, (0, 1, 0)),
])
def test_enable_rule(built_lib_path, d, flags, expect):
    """velog 적용 및 배경 기술: automatic for head_dim >= 64 and %64 == 0; K / V switches."""
    st, rk, rv = kvq.kvq_resolve_rotation(_desc(head_dim=d, flags=flags))
    assert (st, rk, rv) == expect


FAKE = 0x7f0000000000  # an aligned address; never dereferenced by the rejected calls


def _full_desc(**kw):
    c = _desc(**kw)
    for name in ("k_qs", "k_d", "v_qs", "v_d", "seq_len", "status", "k_tail", "v_tail"):
        setattr(c, name, FAKE)
    if c.k_type in (kvq.KVQ_TYPE_Q5_0, kvq.KVQ_TYPE_Q5_1):
        c.k_qh = FAKE
    if c.v_type in (kvq.KVQ_TYPE_Q5_0, kvq.KVQ_TYPE_Q5_1):
        c.v_qh = FAKE
    if c.tail_len == 0:
        c.k_tail = None
        c.v_tail = None
    return c


def test_cache_check_rejections(built_lib_path):
    L = kvq.lib()
    assert L.kvq_cache_check(ctypes.byref(_full_desc())) == 0
    assert L.kvq_cache_check(None) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(); c.k_qs = None
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(); c.v_d = FAKE + 8
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(); c.k_qh = FAKE                      # qh given for a q8_0 plane
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(k_type="q5_0"); c.k_qh = None          # q5_0 without its qh plane
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(v_type="q5_1"); c.v_qh = None          # q5_1 without its qh plane
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(k_type="q4_1"); c.k_qh = FAKE          # qh given for a q4_1 plane
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(tail_len=0); c.k_tail = FAKE
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c = _full_desc(); c.page_tokens, c.n_pages = 64, 8          # paged without a page table
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    c.page_table = FAKE
    assert L.kvq_cache_check(ctypes.byref(c)) == 0
    c = _full_desc(); c.page_table = FAKE                        # a page table without pages
    assert L.kvq_cache_check(ctypes.byref(c)) == kvq.KVQ_ERR_INVALID_ARG
    for bad in (dict(head_dim=48), dict(head_dim=544), dict(max_ctx=100), dict(max_ctx=(1 << 30) + 64),
                dict(batch=0), dict(tail_len=-1),
                dict(k_type=7), dict(v_type=5), dict(flags=8)):
        assert L.kvq_cache_check(ctypes.byref(_full_desc(**bad))) == kvq.KVQ_ERR_INVALID_ARG, bad


def test_call_rejections_before_launch(built_lib_path):
    L = kvq.lib()
    c = _full_desc()
    ref = ctypes.byref(c)
    # append: bad dtype, negative count, null / misaligned inputs, unknown flag
    assert L.kvq_rotate_quantize_append(ref, FAKE, FAKE, 7, 1, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_rotate_quantize_append(ref, FAKE, FAKE, 0, -1, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_rotate_quantize_append(ref, None, FAKE, 0, 1, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_rotate_quantize_append(ref, FAKE + 4, FAKE, 0, 1, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_rotate_quantize_append(ref, FAKE, FAKE, 0, 1, None, 2, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_rotate_quantize_append(ref, FAKE, FAKE, 0, 0, None, 0, None) == 0   # n_new = 0: no-op
    # explicit rotation on an ineligible head_dim
    c96 = _full_desc(head_dim=96, flags=0)
    assert L.kvq_rotate_quantize_append(ctypes.byref(c96), FAKE, FAKE, 0, 1, None, 0, None) == kvq.KVQ_ERR_UNSUPPORTED
    # decode: heads not a multiple of kv heads, bad dtype, null out, workspace
    assert L.kvq_decode_attention(ref, FAKE, 0, 6, 0.0, FAKE, 0, FAKE, 1 << 30, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attention(ref, FAKE, 5, 8, 0.0, FAKE, 0, FAKE, 1 << 30, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attention(ref, FAKE, 0, 8, 0.0, None, 0, FAKE, 1 << 30, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attention(ref, FAKE, 0, 8, -1.0, FAKE, 0, FAKE, 1 << 30, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attention(ref, FAKE, 0, 8, 0.0, FAKE, 0, None, 1 << 30, None) == kvq.KVQ_ERR_WORKSPACE
    assert L.kvq_decode_attention(ref, FAKE, 0, 8, 0.0, FAKE, 0, FAKE, 16, None) == kvq.KVQ_ERR_WORKSPACE
    for dd in (160, 384, 512):  # head dims with no decode kernel
        cdd = _full_desc(head_dim=dd)
        assert L.kvq_cache_check(ctypes.byref(cdd)) == 0
        assert L.kvq_decode_attention(ctypes.byref(cdd), FAKE, 0, 8, 0.0, FAKE, 0, FAKE, 1 << 30, None) == \
            kvq.KVQ_ERR_UNSUPPORTED
    # debug: out-of-range sequence / head / which / positions
    assert L.kvq_dequant_debug(ref, 2, 0, 0, 0, 1, 0, FAKE, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequant_debug(ref, 0, 4, 0, 0, 1, 0, FAKE, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequant_debug(ref, 0, 0, 4, 0, 1, 0, FAKE, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequant_debug(ref, 0, 0, 0, 250, 10, 0, FAKE, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequant_debug(ref, 0, 0, 2, 0, 1, 0, FAKE, FAKE, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequant_debug(ref, 0, 0, 0, 0, 1, 0, None, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_sync_status(None, None, None) == kvq.KVQ_ERR_INVALID_ARG


def test_decode_workspace_bytes_is_a_pure_size_query(built_lib_path):
    c = _desc()
    n = kvq.kvq_decode_workspace_bytes(c, 8)
    assert n > 0 and n % 4 == 0
    assert kvq.kvq_decode_workspace_bytes(c, 6) == 0     # not a multiple of kv heads


def test_outlier_planes_and_checks(built_lib_path):
    """Outlier channels: 32 per KV head, planes sized per body row (paged like the
    body), every pointer required together; prerotated input refused."""
    c = kvq.descriptor(2, 4, 128, 256, 16, "q4_0", "q8_0", n_outlier=32)
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_OUTLIER) == 2 * 4 * 256 // 16 * 1088   # 2 x 34 B per row
    assert kvq.kvq_plane_bytes(c, kvq.KVQ_PLANE_OUTLIER_IDX) == 4 * 32 * 4
    cp = kvq.descriptor(2, 4, 128, 256, 16, "q4_0", "q8_0", page_tokens=64, n_pages=5, n_outlier=32)
    assert kvq.kvq_plane_bytes(cp, kvq.KVQ_PLANE_OUTLIER) == 5 * 4 * 64 * 68
    assert kvq.kvq_plane_bytes(_desc(), kvq.KVQ_PLANE_OUTLIER) == 0        # off: absent plane
    for bad in (dict(n_outlier=16), dict(n_outlier=64), dict(n_outlier=32, head_dim=32)):
        assert kvq.kvq_plane_bytes(_desc(**bad), 0) == 0, bad
    L = kvq.lib()
    full = _full_desc()
    full.n_outlier = 32
    assert L.kvq_cache_check(ctypes.byref(full)) == kvq.KVQ_ERR_INVALID_ARG   # pointers missing
    full.outlier_idx, full.outl = FAKE, FAKE
    assert L.kvq_cache_check(ctypes.byref(full)) == 0
    full.outl = FAKE + 8
    assert L.kvq_cache_check(ctypes.byref(full)) == kvq.KVQ_ERR_INVALID_ARG   # misaligned
    off = _full_desc()
    off.outl = FAKE
    assert L.kvq_cache_check(ctypes.byref(off)) == kvq.KVQ_ERR_INVALID_ARG    # plane without n_outlier
    full.outl = FAKE
    ref = ctypes.byref(full)
    assert L.kvq_rotate_quantize_append(ref, FAKE, FAKE, 0, 1, None, kvq.KVQ_INPUT_PREROTATED, None) == \
        kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_prefill_workspace_bytes(ref, 8, 64) == L.kvq_prefill_workspace_bytes(ctypes.byref(_full_desc()), 8, 64)
    # decode: the q4_0 / q5_0 / q8_0 pairs only; the workspace holds the outlier partials too
    assert L.kvq_decode_workspace_bytes(ref, 8) > L.kvq_decode_workspace_bytes(ctypes.byref(_full_desc()), 8)
    q41 = _full_desc(k_type=kvq.KVQ_TYPE_Q4_1)
    q41.n_outlier, q41.outlier_idx, q41.outl = 32, FAKE, FAKE
    assert L.kvq_decode_attention(ctypes.byref(q41), FAKE, 0, 8, 0.0, FAKE, 0, FAKE, 1 << 40, None) == \
        kvq.KVQ_ERR_UNSUPPORTED


def test_selftest_wait_timeout_argument_checks(built_lib_path):
    L = kvq.lib()
    c = _full_desc()
    assert L.kvq_selftest_wait_timeout(ctypes.byref(c), 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_selftest_wait_timeout(ctypes.byref(c), (1 << 31) + 1, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_selftest_wait_timeout(None, 1000, None) == kvq.KVQ_ERR_INVALID_ARG
    c.status = FAKE + 4
    assert L.kvq_selftest_wait_timeout(ctypes.byref(c), 1000, None) == kvq.KVQ_ERR_INVALID_ARG


def test_rotation_switches_from_the_environment(built_lib_path):
    """KVQ_ROT_K_DISABLE / KVQ_ROT_V_DISABLE switch each side off in the default flags;
    the enable rule then reports that side off (and leaves the other on)."""
    assert kvq.default_flags({}) == kvq.KVQ_ROT_AUTO
    assert kvq.default_flags({"KVQ_ROT_K_DISABLE": "0", "KVQ_ROT_V_DISABLE": ""}) == kvq.KVQ_ROT_AUTO
    fk = kvq.default_flags({"KVQ_ROT_K_DISABLE": "1"})
    fv = kvq.default_flags({"KVQ_ROT_V_DISABLE": "yes"})
    fb = kvq.default_flags({"KVQ_ROT_K_DISABLE": "1", "KVQ_ROT_V_DISABLE": "1"})
    assert fk == kvq.KVQ_ROT_AUTO | kvq.KVQ_ROT_K_OFF and fv == kvq.KVQ_ROT_AUTO | kvq.KVQ_ROT_V_OFF
    for f, want in ((kvq.default_flags({}), (1, 1)), (fk, (0, 1)), (fv, (1, 0)), (fb, (0, 0))):
        st, rk, rv = kvq.kvq_resolve_rotation(kvq.descriptor(1, 1, 128, 64, 0, "q4_0", "q4_0", flags=f))
        assert st == 0 and (rk, rv) == want, (f, rk, rv)
