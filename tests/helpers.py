"""Shared test helpers: parity metrics and GPU runners for numpy inputs."""
import numpy as np

# Acceptance bounds for bf16 activations with fp32 accumulation.
MAX_ABS_OVER_RMS = 2e-2
REL_L1 = 5e-3


def parity(gpu: np.ndarray, ref: np.ndarray) -> dict:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), "non-finite GPU output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    diff = np.abs(gpu - ref)
    return {"rms": rms, "max_abs": float(diff.max()) if diff.size else 0.0,
            "max_over_rms": float(diff.max() / rms) if rms > 0 else 0.0,
            "rel_l1": float(diff.sum() / max(np.abs(ref).sum(), 1e-300))}


def assert_parity(gpu, ref, label=""):
    m = parity(gpu, ref)
    assert m["max_abs"] <= MAX_ABS_OVER_RMS * m["rms"], (label, m)
    assert m["rel_l1"] <= REL_L1, (label, m)
    return m


def to_device_tokens(t: dict, device="cuda"):
    import torch
    x = torch.from_numpy(np.ascontiguousarray(t["x"]).view(np.int16)).to(device)
    ids = torch.from_numpy(np.ascontiguousarray(t["topk_ids"], dtype=np.int32)).to(device)
    tw = torch.from_numpy(np.ascontiguousarray(t["topk_weights"], dtype=np.float32)).to(device)
    return x.view(torch.bfloat16), ids, tw


def gpu_forward(pw, t: dict, workspace=None) -> np.ndarray:
    import torch
    x, ids, tw = to_device_tokens(t)
    out = pw.forward(x, ids, tw, workspace=workspace)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()
