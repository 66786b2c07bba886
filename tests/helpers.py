"""Shared test helpers: host <-> device marshalling of the seeded inputs and the parity bar."""
import numpy as np

# Parity bar for bf16 attention outputs: an element passes if it is within 2e-2
# absolutely or within 1e-2 relatively of the fp64 oracle.
ATTN_ABS = 2e-2
ATTN_REL = 1e-2
# fp32 latent noise against the fp64 oracle.
NOISE_ABS = 1e-6


def bf16_dev(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).to(device).view(torch.bfloat16)


def bits_host(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


def i64_dev(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int64) if np.asarray(a).dtype == np.uint64
                            else np.ascontiguousarray(a, np.int64)).to(device)


def attn_close(got, ref):
    """(ok, max_abs, max_rel) under the either-or bar."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    ok = np.all((err <= ATTN_ABS) | (err <= ATTN_REL * np.abs(ref)))
    rel = err / np.maximum(np.abs(ref), 1e-30)
    return bool(ok), float(err.max(initial=0.0)), float(rel.max(initial=0.0))
