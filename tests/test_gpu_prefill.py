"""GPU prefill attention (tcgen05) vs the float64 oracle on the same cache.

Bar: max-abs 2e-3 and rel-L2 1e-3.  Covers the prompt workload (reduced, and
sampled heads at full size), causal and non-causal, explicit query positions,
GQA groups that do and do not divide 128, head_dim 64, tails longer than the
prompt and no tail, every format pair, q / out dtypes."""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from rotated_bit_kv_kvq_gb300 import workloads as wl
from kvq_testlib import append_both, assert_close, require_gpu, to_dev

pytestmark = pytest.mark.gpu


def gpu_prefill(gc, q_np, q_dtype, torch, causal=True, q_pos0=None, out_dtype="f32", scale=0.0):
    from rotated_bit_kv_kvq_gb300 import kvq
    q = to_dev(q_np, q_dtype, torch)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    out = torch.full(q.shape, float("nan"), dtype=tdt, device="cuda")
    wsb = kvq.kvq_prefill_workspace_bytes(gc.desc, q.shape[2], q.shape[1])
    assert wsb > 0
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN fp16 pattern: stale bytes must not leak
    pos = None if q_pos0 is None else torch.tensor(np.asarray(q_pos0, np.int32)).cuda()
    kvq.kvq_prefill_attention(gc.desc, q, out, ws, q_pos0=pos, causal=causal, chunk=512, scale=scale)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == 0, (st, bits)
    return out.float().cpu().numpy().astype(np.float64)


def _pair(B, H, d, max_ctx, T, kt, vt):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    gc = kvq.KVCache(B, H, d, max_ctx, T, kt, vt)
    rot = ko.rotation_enabled(d)
    return torch, gc, ko.OracleCache(B, H, d, max_ctx, T, kt, vt, rot, rot)


def _kv(rng, B, n, H, d):
    k = rng.standard_normal((B, n, H, d)).astype(np.float32)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    k[..., 5] *= 20
    v[..., 17 % d] *= 20
    return k, v


def test_prompt_workload_reduced():
    w = wl.WORKLOADS["prefill_b2_4k"].scaled(ctx=640, tail_len=64)
    torch, gc, oc = _pair(w.batch, w.n_kv_heads, w.head_dim, w.max_ctx(), w.tail_len, w.k_type, w.v_type)
    inp = wl.make_inputs(w, 0)
    append_both(gc, oc, inp.k_hist, inp.v_hist, torch=torch)
    got = gpu_prefill(gc, inp.q, w.dtype, torch)
    ref = ko.prefill_attention(oc, inp.q)
    assert_close(got, ref, what="prompt workload reduced")


@pytest.mark.parametrize("kt", ["q4_0", "q5_0", "q8_0", "q4_1", "q5_1"])
@pytest.mark.parametrize("vt", ["q4_0", "q8_0", "q4_1", "q5_1"])
def test_format_pairs_causal(kt, vt):
    rng = np.random.default_rng(31)
    B, H, g, d, T, n = 2, 2, 4, 128, 40, 300
    torch, gc, oc = _pair(B, H, d, 320, T, kt, vt)
    k, v = _kv(rng, B, n, H, d)
    append_both(gc, oc, k, v, torch=torch)
    q = rng.standard_normal((B, n, H * g, d)).astype(np.float32)
    assert_close(gpu_prefill(gc, q, "f32", torch), ko.prefill_attention(oc, q), what=f"{kt}/{vt}")


@pytest.mark.parametrize("g", [1, 2, 3, 8, 12])
def test_gqa_groups_and_head_dim_64(g):
    rng = np.random.default_rng(32)
    B, H, d, T, n = 1, 2, 64, 16, 200
    torch, gc, oc = _pair(B, H, d, 256, T, "q8_0", "q4_0")
    k, v = _kv(rng, B, n, H, d)
    append_both(gc, oc, k, v, torch=torch)
    q = rng.standard_normal((B, n, H * g, d)).astype(np.float32)
    assert_close(gpu_prefill(gc, q, "f32", torch), ko.prefill_attention(oc, q), what=f"g={g}")


def test_non_causal_and_query_positions():
    """A chunk of queries in the middle of the sequence (q_pos0 given), causal
    and not; different lengths per sequence."""
    rng = np.random.default_rng(33)
    B, H, g, d, T = 2, 2, 2, 128, 32
    torch, gc, oc = _pair(B, H, d, 448, T, "q5_0", "q5_0")
    k, v = _kv(rng, B, 400, H, d)
    append_both(gc, oc, k, v, n_new_per_seq=[400, 260], torch=torch)
    q = rng.standard_normal((B, 96, H * g, d)).astype(np.float32)
    pos0 = [150, 70]
    for causal in (True, False):
        got = gpu_prefill(gc, q, "f32", torch, causal=causal, q_pos0=pos0)
        ref = ko.prefill_attention(oc, q, q_pos0=pos0, causal=causal)
        assert_close(got, ref, what=f"causal={causal}")


@pytest.mark.parametrize("T", [0, 512])
def test_tail_off_and_tail_longer_than_prompt(T):
    rng = np.random.default_rng(34)
    B, H, g, d, n = 1, 2, 4, 128, 230
    torch, gc, oc = _pair(B, H, d, 256, T, "q4_0", "q4_0")
    k, v = _kv(rng, B, n, H, d)
    append_both(gc, oc, k, v, torch=torch)
    q = rng.standard_normal((B, n, H * g, d)).astype(np.float32)
    assert_close(gpu_prefill(gc, q, "f32", torch), ko.prefill_attention(oc, q), what=f"T={T}")


@pytest.mark.parametrize("q_dtype,out_dtype", [("bf16", "f32"), ("f16", "bf16")])
def test_dtypes_and_scale(q_dtype, out_dtype):
    rng = np.random.default_rng(35)
    B, H, g, d, T, n = 2, 1, 4, 128, 32, 150
    torch, gc, oc = _pair(B, H, d, 192, T, "q8_0", "q8_0")
    k, v = _kv(rng, B, n, H, d)
    append_both(gc, oc, k, v, torch=torch)
    q = to_dev(rng.standard_normal((B, n, H * g, d)).astype(np.float32), q_dtype, torch).float().cpu().numpy()
    for scale in (0.0, 0.15):
        got = gpu_prefill(gc, q, q_dtype, torch, out_dtype=out_dtype, scale=scale)
        ref = ko.prefill_attention(oc, q, scale=scale)
        if out_dtype == "f32":
            assert_close(got, ref, what=f"{q_dtype} scale={scale}")
        else:
            unit = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}[out_dtype]
            assert np.all(np.abs(got - ref) <= 2e-3 + np.abs(ref) * unit)


def test_negative_query_position_is_reported():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(36)
    gc = kvq.KVCache(1, 1, 64, 64, 0, "q4_0", "q4_0")
    k = to_dev(rng.standard_normal((1, 10, 1, 64)).astype(np.float32), "f32", torch)
    kvq.kvq_rotate_quantize_append(gc.desc, k, k)
    q = to_dev(rng.standard_normal((1, 20, 1, 64)).astype(np.float32), "f32", torch)  # 20 > 10 keys
    out = torch.full(q.shape, 7.0, device="cuda")
    ws = torch.empty(kvq.kvq_prefill_workspace_bytes(gc.desc, 1, 20), dtype=torch.uint8, device="cuda")
    kvq.kvq_prefill_attention(gc.desc, q, out, ws)   # q_pos0 = 10 - 20 < 0
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == kvq.KVQ_ERR_DEVICE_RANGE and bits == kvq.KVQ_DEV_ERR_PREFILL_RANGE
    assert bool((out == 0).all())


def test_prompt_workload_full_size_sampled_heads():
    """2 prompts x 4096 tokens, 32/8 heads, d=128, q4_0, tail 256: the launch
    the bench times; the oracle computes two query heads of two KV heads."""
    w = wl.WORKLOADS["prefill_b2_4k"]
    torch, gc, _ = _pair(w.batch, w.n_kv_heads, w.head_dim, w.max_ctx(), w.tail_len, w.k_type, w.v_type)
    from rotated_bit_kv_kvq_gb300 import kvq
    inp = wl.make_inputs(w, 0)
    grp = ko.rotation_group(w.head_dim)
    yk = ko.fwht(inp.k_hist, grp).astype(np.float32)
    yv = ko.fwht(inp.v_hist, grp).astype(np.float32)
    kvq.kvq_rotate_quantize_append(gc.desc, to_dev(yk, "f32", torch), to_dev(yv, "f32", torch), prerotated=True)
    got = gpu_prefill(gc, inp.q, w.dtype, torch)
    for b, kvh in ((0, 0), (1, 5)):
        oc = ko.OracleCache(1, 1, w.head_dim, w.max_ctx(), w.tail_len, w.k_type, w.v_type, True, True)
        oc.append(yk[b:b + 1, :, kvh:kvh + 1], yv[b:b + 1, :, kvh:kvh + 1], prerotated=True)
        # the oracle cache holds one KV head: give it the group's query heads
        qg = inp.q[b:b + 1, :, kvh * w.group:(kvh + 1) * w.group]
        ref = ko.prefill_attention(oc, qg, heads=[0, w.group - 1])
        assert_close(got[b:b + 1, :, kvh * w.group + np.array([0, w.group - 1])], ref[:, :, [0, w.group - 1]],
                     what=f"b={b} kvh={kvh}")
