"""Shared test helpers: host<->device conversion and the layer tolerance check."""
import numpy as np

# Layer-output tolerance: |gpu - ref| <= ATOL + RTOL |ref| elementwise, and
# cosine(gpu, ref) > COS_MIN over the flattened output, so that an all-zero
# output cannot pass ("CuteDSL NVFP4 MoE adds SwiGLU-OAI and ReLU2",
# 关键源码片段: atol 3e-2 plus a cosine check; rtol tightened to 2e-2).
ATOL, RTOL, COS_MIN = 3e-2, 2e-2, 0.99
# Relative L2 error ||gpu - ref|| / ||ref|| over the whole compared output:
# a stricter diagnostic than the elementwise bound (bf16 rounding of the
# output alone gives ~1e-3).
REL_L2_MAX = 1e-2


def dev_bf16(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bits(t) -> np.ndarray:
    """bf16 torch tensor -> uint16 bits (numpy)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(
        np.float64)


def assert_layer_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "out") -> dict:
    got = bits_to_f64(got_bits)
    ref = bits_to_f64(ref_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    nref = np.linalg.norm(ref)
    cos = float(np.dot(got.ravel(), ref.ravel()) / (np.linalg.norm(got) * nref)) if nref > 0 \
        else float(np.linalg.norm(got) == 0)
    rel_l2 = float(np.linalg.norm(got - ref) / nref) if nref > 0 else 0.0
    stats = {"max_abs": float(err.max()) if err.size else 0.0, "cos": cos, "rel_l2": rel_l2,
             "n_bad": int(bad.sum())}
    assert not bad.any(), f"{what}: {stats}"
    assert cos > COS_MIN, f"{what}: {stats}"
    assert rel_l2 <= REL_L2_MAX, f"{what}: {stats}"
    return stats
