"""Host logic of the bench (no GPU): algorithmic byte counts against the per-unit
figures, the recorded-traffic hash check, the clock-sample parsing and the
device-side wait ahead of a timed region.

Per body token-head: (d/32) blocks of K and V (34 + 18 bytes for q8_0 / q4_0);
per tail token-head: bf16 K and V (4 d bytes); per query head: bf16 q in and
out (4 d bytes).  Per appended token-head: bf16 K and V in (4 d), packed blocks
out, and bf16 tail rows out (4 d) for the last tail_len tokens of a call."""

import bench
from rotated_bit_kv_kvq_gb300 import workloads as wl


def test_headline_decode_bytes():
    w = wl.WORKLOADS[wl.HEADLINE]
    assert (w.batch, w.n_kv_heads, w.n_q_heads, w.head_dim, w.tail_len) == (4, 4, 24, 256, 1024)
    assert (w.k_type, w.v_type) == ("q8_0", "q4_0")
    per_body = (256 // 32) * (34 + 18)            # 416 B per token-head
    per_tail = 4 * 256
    n = 65536
    exp = 4 * 4 * ((n - 1024) * per_body + 1024 * per_tail) + 4 * 24 * 4 * 256
    assert exp == 446_267_392
    assert bench.decode_bytes(w, [n] * 4) == exp


def test_decode_bytes_short_and_ragged():
    w = wl.WORKLOADS[wl.HEADLINE]
    # shorter than the tail: every token from the tail; empty sequences still read q / write out
    assert bench.decode_bytes(w, [10, 0]) == 4 * 10 * 4 * 256 + 2 * 24 * 4 * 256
    assert bench.decode_bytes(w, [1025]) == 4 * (416 + 1024 * 1024) + 24 * 4 * 256


def test_append_bytes():
    w = wl.WORKLOADS[wl.HEADLINE]
    heads = 4 * 4
    assert bench.append_bytes(w, 1) == heads * (4 * 256 + 416 + 4 * 256)
    # a long append writes only its last tail_len tokens to the ring
    assert bench.append_bytes(w, 5000) == heads * (5000 * (4 * 256 + 416) + 1024 * 4 * 256)


def test_recorded_traffic_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    """The ncu DRAM bytes in profiles/ count only while the kernel source hashes the same."""
    import hashlib
    import json
    import os
    src_dir = tmp_path / "rotated_bit_kv_kvq_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "k.cuh"
    src.write_bytes(b"kernel v1")
    rec = {"bytes_per_launch": 123, "source_sha256": hashlib.sha256(b"kernel v1").hexdigest()}
    (tmp_path / "profiles" / "decode_b4_ctx64k_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k.cuh") == 123
    src.write_bytes(b"kernel v2")
    assert bench.recorded_traffic("k.cuh") is None
    os.remove(tmp_path / "profiles" / "decode_b4_ctx64k_traffic.json")
    assert bench.recorded_traffic("k.cuh") is None


def test_clock_sampler_parses_clocks_and_throttle_reasons(tmp_path):
    """nvidia-smi CSV rows -> median SM clock, max clock and the active throttle reasons."""
    class _Proc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    rows = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active, 0",
        "0, 1980, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active, 100",
        "0, 2070, 2070, 1000.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active, 97",
        "0, 1950, 2070, 1380.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active, 100",
        "garbage line",
    ]
    with open(cs.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    cs.f = open(cs.path, "a")
    cs.proc = _Proc()
    r = cs.stop()
    # the median SM clock is that of the samples taken under load (utilization >= 50%)
    assert r["sm_mhz"] == 1980.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 4
    assert r["samples_under_load"] == 3
    assert r["reasons"] == ["sw_power_cap"]
    # without nvidia-smi the line says so instead of inventing clocks
    none = bench.ClockSampler(0)
    assert none.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_hold_device_uses_the_device_wait_when_present():
    """The device-side wait ahead of a timed region's start event: called on the
    current stream through torch's wait kernel when the torch build has one, a
    no-op otherwise (never an error that would stop the bench)."""
    import types
    calls = []
    fake = types.SimpleNamespace(cuda=types.SimpleNamespace(_sleep=lambda cycles: calls.append(cycles)))
    bench.hold_device(fake)
    assert calls == [200_000]
    bench.hold_device(fake, cycles=1000)
    assert calls == [200_000, 1000]
    bench.hold_device(types.SimpleNamespace(cuda=types.SimpleNamespace()))  # no wait kernel: nothing happens


def test_reference_step_bytes_are_a_pairs_share():
    """The reference arm's per-step bytes (one pair's append and decode) times the
    number of (sequence, KV head) pairs equal the repo arm's step bytes."""
    w = wl.WORKLOADS[wl.HEADLINE]
    pairs = w.batch * w.n_kv_heads
    for n in (65536, 65555, 500, 1024, 1025):
        assert pairs * bench.pair_step_bytes(w, n, 1) == bench.decode_bytes(w, [n] * w.batch) + bench.append_bytes(w, 1)
