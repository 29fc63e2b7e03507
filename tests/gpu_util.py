"""Helpers shared by the GPU parity tests: host <-> device transfer of the
generator's storage arrays and the tolerance rule."""
import numpy as np

import datagen

TOL = {"f32": 1e-5, "bf16": 2e-2}
LOSS_TOL_BF16 = 1e-3


def dev(a, device="cuda"):
    """numpy storage array (float32 / float64 / bf16 bits / ints) -> CUDA tensor."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t):
    """CUDA tensor -> float64 numpy (exact widening)."""
    import torch
    if t.dtype == torch.bfloat16:
        return datagen.to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    return t.double().cpu().numpy()


def bits(t):
    """Raw storage bits of a CUDA tensor (for bit-exact checks)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def storage(dtype):
    import torch
    return torch.float32 if dtype == "f32" else torch.bfloat16
