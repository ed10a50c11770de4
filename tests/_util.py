"""Helpers shared by the GPU tests: move synthetic inputs to the device and
compare against the oracle."""
import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_dev(a, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device="cuda", dtype=torch.float32 if dtype == "f32" else torch.bfloat16).contiguous()


def to_host(t):
    import torch
    return t.to(torch.float32).cpu().numpy().astype(np.float64)
