"""The failure path on the GPU without a fault: a bounded wait that nothing
completes gives up, the status word says so, kvq_sync_status reports
KVQ_ERR_TIMEOUT and clears it, and the context keeps working."""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from kvq_testlib import append_both, assert_close, gpu_decode, require_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(91)
    B, H, g, d, T = 1, 2, 2, 64, 8
    gc = kvq.KVCache(B, H, d, 128, T, "q8_0", "q4_0")
    oc = ko.OracleCache(B, H, d, 128, T, "q8_0", "q4_0", True, True)
    kvq.kvq_selftest_wait_timeout(gc.desc, 1 << 20)      # about half a millisecond
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == kvq.KVQ_ERR_TIMEOUT and bits == kvq.KVQ_DEV_ERR_TIMEOUT
    st, bits = kvq.kvq_sync_status(gc.desc)                # cleared by the first read
    assert st == 0 and bits == 0
    k = rng.standard_normal((B, 50, H, d)).astype(np.float32)
    v = rng.standard_normal((B, 50, H, d)).astype(np.float32)
    append_both(gc, oc, k, v, torch=torch)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what="decode after a timeout")
