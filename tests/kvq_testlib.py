"""Shared helpers of the parity tests: build the same cache on the GPU (through
the C ABI) and in the CPU oracle, from the same seeded inputs."""

from __future__ import annotations

import numpy as np
import pytest

from oracle import kvq_oracle as ko

ATOL = 2e-3   # max-abs bound on attention outputs
RTOL = 1e-3   # rel-L2 bound on attention outputs


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


def to_dev(x: np.ndarray, dtype: str, torch):
    """float32 numpy -> device tensor of the workload dtype ('f32', 'bf16', 'f16')."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    elif dtype == "f16":
        t = t.to(torch.float16)
    return t.cuda()


def prerotate(x: np.ndarray, rot: bool) -> np.ndarray:
    """The oracle's rotated float32 values (float64 product, rounded to float32)."""
    return ko.rotate(x).astype(np.float32) if rot else np.asarray(x, dtype=np.float32)


def append_both(gcache, ocache, k, v, n_new_per_seq=None, torch=None, chunk=4096):
    """Append the same float32 K/V ([B][n][H][d]) to the GPU cache (pre-rotated by
    the oracle, so both sides quantize identical values) and to the oracle cache."""
    from rotated_bit_kv_kvq_gb300 import kvq
    yk = prerotate(k, ocache.rot["k"])
    yv = prerotate(v, ocache.rot["v"])
    nps_dev = None
    if n_new_per_seq is not None:
        nps_dev = torch.tensor(np.asarray(n_new_per_seq, dtype=np.int32)).cuda()
    kvq.kvq_rotate_quantize_append(gcache.desc, to_dev(yk, "f32", torch), to_dev(yv, "f32", torch),
                                   n_new_per_seq=nps_dev, prerotated=True)
    ocache.append(yk, yv, n_new_per_seq=n_new_per_seq, prerotated=True)


def gpu_blocks(gcache, seq, head, which, t0, count, qtype, d, torch):
    """GGUF array-of-structs bytes of body blocks read back from the GPU."""
    from rotated_bit_kv_kvq_gb300 import kvq
    nbytes = count * (d // 32) * ko.GGML_BLOCK_BYTES[qtype]
    buf = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    kvq.kvq_dequant_debug(gcache.desc, seq, head, which, t0, count, blocks=buf)
    torch.cuda.synchronize()
    return buf[:nbytes].cpu().numpy().reshape(count, d // 32, ko.GGML_BLOCK_BYTES[qtype])


def gpu_values(gcache, seq, head, which, t0, count, d, torch, original_basis=False):
    from rotated_bit_kv_kvq_gb300 import kvq
    out = torch.zeros((max(count, 1), d), dtype=torch.float32, device="cuda")
    kvq.kvq_dequant_debug(gcache.desc, seq, head, which, t0, count, out=out, original_basis=original_basis)
    torch.cuda.synchronize()
    return out[:count].cpu().numpy().astype(np.float64)


def gpu_decode(gcache, q_np, q_dtype, torch, out_dtype="f32", scale=0.0):
    from rotated_bit_kv_kvq_gb300 import kvq
    q = to_dev(q_np, q_dtype, torch)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    out = torch.empty(q.shape, dtype=tdt, device="cuda")
    wsb = kvq.kvq_decode_workspace_bytes(gcache.desc, q.shape[1])
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    kvq.kvq_decode_attention(gcache.desc, q, out, ws, scale=scale)
    st, bits = kvq.kvq_sync_status(gcache.desc)
    assert st == 0, (st, bits)
    return out.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, atol=ATOL, rtol=RTOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    maxabs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / denom) if denom > 0 else float(np.linalg.norm(got - ref))
    assert maxabs <= atol, f"{what}: max-abs {maxabs:.3e} > {atol}"
    assert rel <= rtol, f"{what}: rel-L2 {rel:.3e} > {rtol}"
    return maxabs, rel
