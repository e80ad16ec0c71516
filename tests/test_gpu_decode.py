"""GPU decode attention vs the float64 oracle on the same (bit-identical) cache.

Bar: max-abs 2e-3 and rel-L2 1e-3 on the outputs, fp32 accumulation on the GPU.
Covers the five workload shapes (the large ones reduced, plus sampled heads at
full size), every K/V format pair, head_dim 64/128/192/256, GQA groups 1..16,
tails longer / shorter than the sequence, empty sequences, rotation switches,
q / out dtypes, and repeated steps with appends in between."""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from rotated_bit_kv_kvq_gb300 import workloads as wl
from kvq_testlib import append_both, assert_close, gpu_decode, require_gpu

pytestmark = pytest.mark.gpu


def _run_workload(w, seed=0):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    inp = wl.make_inputs(w, seed)
    rot = ko.rotation_enabled(w.head_dim)
    max_ctx = w.max_ctx()
    gc = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, max_ctx, w.tail_len, w.k_type, w.v_type)
    oc = ko.OracleCache(w.batch, w.n_kv_heads, w.head_dim, max_ctx, w.tail_len, w.k_type, w.v_type, rot, rot)
    append_both(gc, oc, inp.k_hist, inp.v_hist, n_new_per_seq=inp.lengths, torch=torch)
    got = gpu_decode(gc, inp.q, w.dtype, torch)
    qin = inp.q
    ref = ko.decode_attention(oc, qin)
    return assert_close(got, ref, what=w.name)


def test_decode_d64_ctx256():
    _run_workload(wl.WORKLOADS["decode_d64_ctx256"])


def test_decode_gqa16x8_ctx4k():
    _run_workload(wl.WORKLOADS["decode_gqa16x8_ctx4k"])


def test_decode_b32_ragged_reduced():
    _run_workload(wl.WORKLOADS["decode_b32_ragged8k"].scaled(batch=6, ctx=2048, ragged_min=300))


def test_decode_b4_ctx64k_reduced():
    _run_workload(wl.WORKLOADS["decode_b4_ctx64k"].scaled(batch=2, ctx=4096))


def _cache_pair(B, H, d, max_ctx, T, kt, vt, flags=None, rot_k=None, rot_v=None):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    fl = kvq.KVQ_ROT_AUTO if flags is None else flags
    gc = kvq.KVCache(B, H, d, max_ctx, T, kt, vt, flags=fl)
    st, rk, rv = kvq.kvq_resolve_rotation(gc.desc)
    assert st == 0
    oc = ko.OracleCache(B, H, d, max_ctx, T, kt, vt, bool(rk), bool(rv))
    return torch, gc, oc


def _kv(rng, B, n, H, d):
    k = rng.standard_normal((B, n, H, d)).astype(np.float32)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    k[..., 7] *= 20
    v[..., 11 % d] *= 20
    return k, v


@pytest.mark.parametrize("kt", ["q4_0", "q5_0", "q8_0", "q4_1", "q5_1"])
@pytest.mark.parametrize("vt", ["q4_0", "q5_0", "q8_0", "q4_1", "q5_1"])
def test_every_format_pair(kt, vt):
    rng = np.random.default_rng(21)
    B, H, g, d, T = 2, 2, 4, 128, 48
    torch, gc, oc = _cache_pair(B, H, d, 640, T, kt, vt)
    k, v = _kv(rng, B, 600, H, d)
    append_both(gc, oc, k, v, n_new_per_seq=[600, 333], torch=torch)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=f"{kt}/{vt}")


@pytest.mark.parametrize("d,kt,vt", [(64, "q8_0", "q4_0"), (64, "q5_0", "q5_0"), (256, "q8_0", "q4_0"),
                                     (256, "q4_0", "q5_0"), (256, "q8_0", "q8_0"), (192, "q4_0", "q4_0"),
                                     (64, "q4_1", "q5_1"), (256, "q5_1", "q4_1"), (256, "q8_0", "q5_1"),
                                     (256, "q5_0", "q4_1"),
                                     # block-diagonal H_64 head dims, every format on each side
                                     (192, "q8_0", "q4_0"), (192, "q5_0", "q5_1"), (192, "q4_1", "q8_0"),
                                     (320, "q8_0", "q4_0"), (320, "q4_0", "q4_0"), (320, "q5_0", "q5_1"),
                                     (320, "q4_1", "q8_0"), (320, "q5_1", "q5_0")])
def test_head_dims(d, kt, vt):
    rng = np.random.default_rng(22)
    B, H, g, T = 2, 2, 3, 40
    torch, gc, oc = _cache_pair(B, H, d, 1024, T, kt, vt)
    k, v = _kv(rng, B, 1000, H, d)
    append_both(gc, oc, k, v, n_new_per_seq=[1000, 517], torch=torch)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=f"d={d}")


@pytest.mark.parametrize("g", [1, 2, 3, 6, 8, 12, 16])
def test_gqa_groups(g):
    rng = np.random.default_rng(23)
    B, H, d, T = 1, 2, 128, 32
    torch, gc, oc = _cache_pair(B, H, d, 512, T, "q8_0", "q4_0")
    k, v = _kv(rng, B, 450, H, d)
    append_both(gc, oc, k, v, torch=torch)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=f"g={g}")


@pytest.mark.parametrize("lens,T", [([0, 5], 8), ([3, 17], 32), ([100, 1], 0), ([16, 64], 16), ([700, 699], 13),
                                    ([1, 0], 0)])
def test_lengths_and_tails(lens, T):
    """empty sequences, sequences shorter than the tail, no tail, ragged tails."""
    rng = np.random.default_rng(24)
    B, H, g, d = 2, 2, 2, 64
    torch, gc, oc = _cache_pair(B, H, d, 768, T, "q4_0", "q8_0")
    n = max(max(lens), 1)
    k, v = _kv(rng, B, n, H, d)
    append_both(gc, oc, k, v, n_new_per_seq=lens, torch=torch)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    got = gpu_decode(gc, q, "f32", torch)
    ref = ko.decode_attention(oc, q)
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got[b] == 0)
    assert_close(got, ref, what=f"lens={lens},T={T}")


@pytest.mark.parametrize("flags", ["k_off", "v_off", "both_off"])
def test_rotation_switches(flags):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    f = kvq.KVQ_ROT_AUTO | {"k_off": kvq.KVQ_ROT_K_OFF, "v_off": kvq.KVQ_ROT_V_OFF,
                            "both_off": kvq.KVQ_ROT_K_OFF | kvq.KVQ_ROT_V_OFF}[flags]
    rng = np.random.default_rng(25)
    B, H, g, d, T = 2, 2, 2, 128, 24
    torch, gc, oc = _cache_pair(B, H, d, 320, T, "q8_0", "q5_0", flags=f)
    k, v = _kv(rng, B, 300, H, d)
    append_both(gc, oc, k, v, torch=torch)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=flags)


@pytest.mark.parametrize("q_dtype,out_dtype", [("bf16", "f32"), ("f16", "bf16"), ("f32", "f16")])
def test_dtypes_and_scale(q_dtype, out_dtype):
    rng = np.random.default_rng(26)
    B, H, g, d, T = 2, 2, 4, 128, 64
    torch, gc, oc = _cache_pair(B, H, d, 512, T, "q4_0", "q4_0")
    k, v = _kv(rng, B, 500, H, d)
    append_both(gc, oc, k, v, torch=torch)
    from kvq_testlib import to_dev
    q = to_dev(rng.standard_normal((B, H * g, d)).astype(np.float32), q_dtype, torch).float().cpu().numpy()
    for scale in (0.0, 0.2):
        got = gpu_decode(gc, q, q_dtype, torch, out_dtype=out_dtype, scale=scale)
        ref = ko.decode_attention(oc, q, scale=scale)
        if out_dtype == "f32":
            assert_close(got, ref, what=f"{q_dtype}->{out_dtype} scale={scale}")
        else:
            # the stored output adds one rounding of its own type (half a unit, relative)
            unit = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}[out_dtype]
            assert np.all(np.abs(got - ref) <= 2e-3 + np.abs(ref) * unit), (q_dtype, out_dtype, scale)


def test_decode_steps_with_appends():
    """Append one token per sequence, decode, repeat: the tail ring wraps many times."""
    rng = np.random.default_rng(27)
    B, H, g, d, T = 3, 2, 3, 128, 16
    torch, gc, oc = _cache_pair(B, H, d, 256, T, "q8_0", "q4_0")
    k, v = _kv(rng, B, 100, H, d)
    append_both(gc, oc, k, v, n_new_per_seq=[100, 37, 0], torch=torch)
    for step in range(40):
        k, v = _kv(rng, B, 1, H, d)
        append_both(gc, oc, k, v, torch=torch)
        q = rng.standard_normal((B, H * g, d)).astype(np.float32)
        if step % 8 == 0 or step == 39:
            assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=f"step {step}")


@pytest.mark.parametrize("name,pairs", [("decode_b4_ctx64k", [(0, 0), (3, 2)]),
                                        ("decode_b32_ragged8k", [(0, 0), (17, 5), (31, 7)])])
def test_full_size_sampled_heads(name, pairs):
    """The full-size workloads in the bench's launch configuration; the oracle
    computes the sampled (sequence, KV head) pairs."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, 0)
    rot = ko.rotation_enabled(w.head_dim)
    max_ctx = w.max_ctx()
    gc = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, max_ctx, w.tail_len, w.k_type, w.v_type)
    # pre-rotate with the oracle's FWHT (the matrix product at this size is slow); it is pinned equal
    grp = ko.rotation_group(w.head_dim)
    nps = torch.tensor(inp.lengths.astype(np.int32)).cuda()
    for b in range(w.batch):
        yk = ko.fwht(inp.k_hist[b:b + 1], grp).astype(np.float32) if rot else inp.k_hist[b:b + 1]
        yv = ko.fwht(inp.v_hist[b:b + 1], grp).astype(np.float32) if rot else inp.v_hist[b:b + 1]
        # append sequence b only
        sel = torch.zeros(w.batch, dtype=torch.int32, device="cuda")
        sel[b] = int(inp.lengths[b])
        full_k = torch.zeros((w.batch,) + yk.shape[1:], dtype=torch.float32, device="cuda")
        full_v = torch.zeros_like(full_k)
        full_k[b] = torch.from_numpy(yk[0]).cuda()
        full_v[b] = torch.from_numpy(yv[0]).cuda()
        kvq.kvq_rotate_quantize_append(gc.desc, full_k, full_v, n_new_per_seq=sel, prerotated=True)
        del full_k, full_v
        torch.cuda.synchronize()
    assert np.array_equal(gc.seq_len.cpu().numpy(), inp.lengths)
    got = gpu_decode(gc, inp.q, w.dtype, torch)
    for b, h in pairs:
        oc = ko.OracleCache(1, 1, w.head_dim, max_ctx, w.tail_len, w.k_type, w.v_type, rot, rot)
        n = int(inp.lengths[b])
        yk = ko.fwht(inp.k_hist[b, :n, h], grp).astype(np.float32)
        yv = ko.fwht(inp.v_hist[b, :n, h], grp).astype(np.float32)
        oc.append(yk[None, :, None], yv[None, :, None], prerotated=True)
        heads = slice(h * w.group, (h + 1) * w.group)
        ref = ko.decode_attention(oc, inp.q[b:b + 1, heads])
        assert_close(got[b:b + 1, heads], ref, what=f"{name} b={b} h={h}")
