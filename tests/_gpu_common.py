"""Helpers shared by the GPU parity tests: move GPU-quantized buffers to the
oracle's numpy form, and compare results."""
import numpy as np
import torch


def nv_to_np(t):
    return (t.payload.cpu().numpy(), t.sf.cpu().numpy(), np.float32(t.g.cpu().item()))


def mx_to_np(t):
    return (t.payload_t.cpu().numpy(), t.sf.cpu().numpy())


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def sample_rows(B, H, N, heads, rows_per_head, seed):
    """Flat row ids (b*H+h)*N+i: chosen heads, rows spread over [0, N) incl. both ends."""
    rng = np.random.default_rng(seed)
    out = []
    for bh in heads:
        r = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=min(N, rows_per_head), replace=False)]))
        out.extend(int(bh) * N + int(i) for i in r)
    return np.array(sorted(set(out)), dtype=np.int64)


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
