"""Shared test helpers: moving seeded numpy inputs to the GPU and back."""
import numpy as np
import torch


def dev(x, dtype=None):
    """numpy -> CUDA tensor; float32 arrays become ``dtype`` (bf16 values
    produced by synth.round_bf16 convert exactly)."""
    a = np.ascontiguousarray(x)
    if not a.flags.writeable:  # e.g. a broadcast view: torch wants its own copy
        a = a.copy()
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.detach().float().cpu().numpy() if t.is_floating_point() else t.detach().cpu().numpy()


def i32(x):
    return dev(np.asarray(x, np.int32))


def zeros_i32(*shape):
    return torch.zeros(shape, dtype=torch.int32, device="cuda")


def within(got, ref, atol, rtol):
    """Element-wise |got - ref| <= atol + rtol |ref|; returns (ok, max excess)."""
    err = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    return bool((err <= 0).all()), float(err.max())
