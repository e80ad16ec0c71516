"""GPU write path vs the oracle: packed blocks bit-exact, tail bf16 exact, seq_len,
ragged counts, ring wrap-around, range errors, and the GPU's own rotation."""

import json

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from conftest import golden_path
from kvq_testlib import append_both, gpu_blocks, gpu_values, require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _edge_blocks():
    """The hand-worked golden blocks (ties, halves, clamp, zeros, subnormal scale)."""
    g = json.load(open(golden_path("quant_blocks.json")))
    out = []
    for blk in g["blocks"]:
        x = np.zeros(32, np.float32)
        for k, v in blk["x"].items():
            x[int(k)] = v
        out.append(x)
    return out


def _inputs(rng, B, n, H, d, scale=1.0):
    x = rng.standard_normal((B, n, H, d)).astype(np.float32) * scale
    x[:, :, :, 3 % d] *= 20
    x[:, ::5] *= np.float32(1e-3)
    edges = _edge_blocks()
    # plant the golden blocks in the first positions of sequence 0, head 0
    for i, blk in enumerate(edges):
        t, j = divmod(i, d // 32)
        if t < n:
            x[0, t, 0, 32 * j:32 * j + 32] = blk
    x[1 % B, 0, 0, :] = 0.0                        # an all-zero vector
    x[0, n - 1, H - 1, :] = -0.0
    return x


@pytest.mark.parametrize("qt", ["q4_0", "q5_0", "q8_0", "q4_1", "q5_1"])
@pytest.mark.parametrize("d", [32, 64, 96, 128, 192, 256, 320, 384, 512])
def test_blocks_bit_exact_prerotated(qt, d):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(100 + d)
    B, H, n, T = 2, 3, 37, 8
    other = {"q4_0": "q8_0", "q5_0": "q4_1", "q8_0": "q5_1", "q4_1": "q5_0", "q5_1": "q4_0"}[qt]
    gc = kvq.KVCache(B, H, d, 64, T, qt, other)
    oc = ko.OracleCache(B, H, d, 64, T, qt, other, ko.rotation_enabled(d), ko.rotation_enabled(d))
    k = _inputs(rng, B, n, H, d)
    v = _inputs(rng, B, n, H, d, scale=3.0)
    append_both(gc, oc, k, v, torch=torch)
    assert np.array_equal(gc.seq_len.cpu().numpy(), [n, n])
    for b in range(B):
        for h in range(H):
            for which, w, t in ((0, "k", qt), (1, "v", other)):
                got = gpu_blocks(gc, b, h, which, 0, n, t, d, torch)
                exp = oc.ggml_blocks(w, b, h, 0, n)
                assert np.array_equal(got, exp), (qt, d, b, h, w)
                # the values the body holds equal the oracle's dequantization exactly
                vals = gpu_values(gc, b, h, which, 0, n, d, torch)
                assert np.array_equal(vals, oc.body_values(w, b, h, 0, n))
            for which, w in ((2, "k"), (3, "v")):
                pos = np.arange(n - T, n)
                got = gpu_values(gc, b, h, which, n - T, T, d, torch)
                assert np.array_equal(got, oc.tail_values(w, b, h, pos))


def test_ragged_counts_ring_wrap_and_many_appends():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(7)
    B, H, d, T = 3, 2, 128, 16
    gc = kvq.KVCache(B, H, d, 256, T, "q5_0", "q8_0")
    oc = ko.OracleCache(B, H, d, 256, T, "q5_0", "q8_0", True, True)
    for step in range(30):
        nn = [int(x) for x in rng.integers(0, 9, B)]
        k = _inputs(rng, B, 8, H, d)
        v = _inputs(rng, B, 8, H, d)
        append_both(gc, oc, k, v, n_new_per_seq=nn, torch=torch)
    lens = gc.seq_len.cpu().numpy()
    assert np.array_equal(lens, oc.seq_len)
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            assert np.array_equal(gpu_blocks(gc, b, h, 0, 0, n, "q5_0", d, torch), oc.ggml_blocks("k", b, h, 0, n))
            assert np.array_equal(gpu_blocks(gc, b, h, 1, 0, n, "q8_0", d, torch), oc.ggml_blocks("v", b, h, 0, n))
            lo = max(0, n - T)
            got = gpu_values(gc, b, h, 2, lo, n - lo, d, torch)
            assert np.array_equal(got, oc.tail_values("k", b, h, np.arange(lo, n)))


def test_single_call_longer_than_tail_keeps_last_tokens():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(8)
    B, H, d, T, n = 2, 2, 64, 16, 150
    gc = kvq.KVCache(B, H, d, 192, T, "q4_0", "q4_0")
    oc = ko.OracleCache(B, H, d, 192, T, "q4_0", "q4_0", True, True)
    append_both(gc, oc, _inputs(rng, B, n, H, d), _inputs(rng, B, n, H, d), torch=torch)
    for b in range(B):
        for h in range(H):
            got = gpu_values(gc, b, h, 3, n - T, T, d, torch)
            assert np.array_equal(got, oc.tail_values("v", b, h, np.arange(n - T, n)))


def test_overflow_sets_status_and_leaves_sequence_untouched():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(9)
    gc = kvq.KVCache(2, 1, 64, 64, 0, "q8_0", "q8_0")
    k = to_dev(rng.standard_normal((2, 40, 1, 64)).astype(np.float32), "f32", torch)
    kvq.kvq_rotate_quantize_append(gc.desc, k, k)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == 0 and bits == 0
    nps = torch.tensor([30, 10], dtype=torch.int32, device="cuda")   # sequence 0 would pass 64
    kvq.kvq_rotate_quantize_append(gc.desc, k, k, n_new_per_seq=nps)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == kvq.KVQ_ERR_DEVICE_RANGE and bits == kvq.KVQ_DEV_ERR_APPEND_RANGE
    assert gc.seq_len.cpu().numpy().tolist() == [40, 50]
    st, bits = kvq.kvq_sync_status(gc.desc)            # cleared after being reported
    assert st == 0 and bits == 0


@pytest.mark.parametrize("in_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("d,n", [(64, 64), (128, 64), (256, 64), (192, 64), (64, 320), (128, 320), (256, 320),
                                 (320, 64), (384, 64), (512, 64)])
def test_gpu_rotation_against_oracle(in_dtype, d, n):
    """The GPU rotates in fp32 (warp FWHT); the oracle in fp64.  Codes may flip
    only where the rotated value sits within float rounding of a code boundary:
    at most 1 in 1000 elements, each by one level, and bf16 tail values agree
    to one bf16 unit.  n = 320 (5,120 vectors) takes the bulk, block-per-lane
    kernel; n = 64 the vector-per-warp one."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(11)
    B, H, T = 2, 4, 16
    x = rng.standard_normal((B, n, H, d)).astype(np.float32)
    x[..., 5] *= 20
    xd = to_dev(x, in_dtype, torch)
    xin = xd.float().cpu().numpy()            # the values the GPU actually received
    for qt in ("q4_0", "q5_0", "q8_0", "q4_1", "q5_1"):
        gc = kvq.KVCache(B, H, d, n, T, qt, qt)
        oc = ko.OracleCache(B, H, d, n, T, qt, qt, True, True)
        kvq.kvq_rotate_quantize_append(gc.desc, xd, xd)
        oc.append(xin, xin)
        flips = 0
        total = 0
        for b in range(B):
            for h in range(H):
                got = gpu_values(gc, b, h, 0, 0, n, d, torch)
                exp = oc.body_values("k", b, h, 0, n)
                dq = ko.scale_and_min(qt, oc.dbits["k"][b, h, :n])[0].repeat(32, axis=-1).reshape(n, d)
                diff = got != exp
                flips += int(diff.sum())
                total += got.size
                # a flipped element moves by one quantization level of its block
                # (the block scale itself can differ in its last fp16 bit)
                lvl = np.abs(dq[diff]) * 1.01 + 1e-30
                assert np.all(np.abs(got[diff] - exp[diff]) <= lvl)
                tg = gpu_values(gc, b, h, 2, n - T, T, d, torch)
                te = oc.tail_values("k", b, h, np.arange(n - T, n))
                # one bf16 unit, plus the fp32 rounding of the transform itself for
                # values that nearly cancel (absolute, relative to the row's largest)
                tol = np.abs(te) * 2.0 ** -7 + np.abs(te).max(axis=-1, keepdims=True) * 2.0 ** -16
                assert np.all(np.abs(tg - te) <= tol)
        assert flips <= total // 1000 + 2, (qt, flips, total)
        # back in the original basis the values are x up to the quantization error
        back = gpu_values(gc, 0, 0, 0, 0, n, d, torch, original_basis=True)
        amax = np.abs(ko.rotate(xin[0, :, 0])).reshape(n, d // 32, 32).max(-1)
        # quantization step relative to the block's largest magnitude (range / levels for the _1 types)
        step = {"q4_0": 1 / 8, "q5_0": 1 / 16, "q8_0": 1 / 127, "q4_1": 2 / 15, "q5_1": 2 / 31}[qt]
        err = np.linalg.norm(back - xin[0, :, 0], axis=-1)
        assert np.all(err <= np.sqrt(d) * (amax.max(-1) * step) * 1.01 + 1e-6)


@pytest.mark.parametrize("qt", ["q4_0", "q5_0", "q8_0", "q4_1", "q5_1"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bulk_blocks_bit_exact_prerotated(qt, d):
    """Appends of at least 2,048 vectors (the block-per-lane kernel): blocks,
    dequantized values and tail rows bit-exact, ragged counts, two calls."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(200 + d)
    B, H, T = 2, 4, 16
    other = {"q4_0": "q8_0", "q5_0": "q4_1", "q8_0": "q5_1", "q4_1": "q5_0", "q5_1": "q4_0"}[qt]
    gc = kvq.KVCache(B, H, d, 640, T, qt, other)
    oc = ko.OracleCache(B, H, d, 640, T, qt, other, True, True)
    for n, nps in ((300, [300, 261]), (290, [250, 290])):
        k = _inputs(rng, B, n, H, d)
        v = _inputs(rng, B, n, H, d, scale=3.0)
        append_both(gc, oc, k, v, n_new_per_seq=nps, torch=torch)
    lens = gc.seq_len.cpu().numpy()
    assert np.array_equal(lens, oc.seq_len)
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            for which, w, t in ((0, "k", qt), (1, "v", other)):
                assert np.array_equal(gpu_blocks(gc, b, h, which, 0, n, t, d, torch), oc.ggml_blocks(w, b, h, 0, n))
            for which, w in ((2, "k"), (3, "v")):
                got = gpu_values(gc, b, h, which, n - T, T, d, torch)
                assert np.array_equal(got, oc.tail_values(w, b, h, np.arange(n - T, n)))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bulk_partial_last_task(d):
    """Bulk appends whose vector count (batch x tokens x KV heads = 3 x 229 x 3) is
    no multiple of the vectors a warp task holds (32 / (d / 32)): the last K task
    and the last V task each have lanes past the end, which must store nothing,
    and the first V task follows a partly filled K task.  Mixed K/V formats,
    ragged counts, two calls; blocks and tail rows bit-exact."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(300 + d)
    B, H, T = 3, 3, 8
    gc = kvq.KVCache(B, H, d, 512, T, "q8_0", "q5_0")
    oc = ko.OracleCache(B, H, d, 512, T, "q8_0", "q5_0", True, True)
    for n, nps in ((229, [229, 200, 3]), (229, [1, 229, 228])):
        assert (B * n * H) % (32 // (d // 32)) != 0
        k = _inputs(rng, B, n, H, d)
        v = _inputs(rng, B, n, H, d, scale=2.0)
        append_both(gc, oc, k, v, n_new_per_seq=nps, torch=torch)
    lens = gc.seq_len.cpu().numpy()
    assert np.array_equal(lens, oc.seq_len)
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            for which, w, t in ((0, "k", "q8_0"), (1, "v", "q5_0")):
                assert np.array_equal(gpu_blocks(gc, b, h, which, 0, n, t, d, torch), oc.ggml_blocks(w, b, h, 0, n))
            for which, w in ((2, "k"), (3, "v")):
                got = gpu_values(gc, b, h, which, n - T, T, d, torch)
                assert np.array_equal(got, oc.tail_values(w, b, h, np.arange(n - T, n)))


def test_bulk_k_rotated_v_not():
    """K rotated in the kernel, V stored as given (KVQ_ROT_V_OFF), through the
    bulk kernel (its warp tasks hold K vectors or V vectors, each side with its
    own switch).  V blocks are bit-exact; K within the rotation tolerance (exact
    here: dyadic inputs at head_dim 64)."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(203)
    B, H, d, n, T = 2, 4, 64, 300, 8
    gc = kvq.KVCache(B, H, d, 320, T, "q4_0", "q8_0", flags=kvq.KVQ_ROT_AUTO | kvq.KVQ_ROT_V_OFF)
    oc = ko.OracleCache(B, H, d, 320, T, "q4_0", "q8_0", True, False)
    k = rng.integers(-64, 65, (B, n, H, d)).astype(np.float32) * np.float32(0.125)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    kvq.kvq_rotate_quantize_append(gc.desc, to_dev(k, "f32", torch), to_dev(v, "f32", torch))
    oc.append(k, v)
    for b in range(B):
        for h in range(H):
            for which, w, t in ((0, "k", "q4_0"), (1, "v", "q8_0")):
                assert np.array_equal(gpu_blocks(gc, b, h, which, 0, n, t, d, torch), oc.ggml_blocks(w, b, h, 0, n))
            for which, w in ((2, "k"), (3, "v")):
                got = gpu_values(gc, b, h, which, n - T, T, d, torch)
                assert np.array_equal(got, oc.tail_values(w, b, h, np.arange(n - T, n)))
