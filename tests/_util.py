"""Helpers shared by the GPU tests: move synthetic inputs to the device and
compare against the oracle."""
import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}


def forward_err(got, ref, dtype):
    """Error of a forward output under its dtype's measure: element-wise with a
    1%-of-row floor (oracle.elem_rel_err) for fp32 storage, row-normwise
    (oracle.row_rel_err) for bf16 storage, where rounding the features to
    bf16 alone moves an element-wise ratio far past 2e-2."""
    import oracle as O
    return O.elem_rel_err(got, ref) if dtype == "f32" else O.row_rel_err(got, ref)


def to_dev(a, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device="cuda", dtype=torch.float32 if dtype == "f32" else torch.bfloat16).contiguous()


def to_host(t):
    import torch
    return t.to(torch.float32).cpu().numpy().astype(np.float64)


def to_dev_unaligned(a, dtype):
    """Like to_dev, but the tensor starts one element past a 16-byte boundary
    (the calls must take their paths for unaligned pointers)."""
    import torch
    t = to_dev(a, dtype)
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device=t.device)
    u = buf[1:1 + t.numel()].view(t.shape)
    u.copy_(t)
    assert u.data_ptr() % 16 != 0
    return u
