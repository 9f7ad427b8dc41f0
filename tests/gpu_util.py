"""Moving numpy storage arrays to and from CUDA tensors, and bitwise
comparison.  Conversions only: no reduction arithmetic lives here."""
from __future__ import annotations

import numpy as np

NP_BITS = {"int32": np.int32, "int64": np.int64, "float32": np.uint32, "bfloat16": np.uint16}


def torch_dtype(torch, dtype: str):
    return {"int32": torch.int32, "int64": torch.int64, "float32": torch.float32,
            "bfloat16": torch.bfloat16}[dtype]


def to_device(torch, xs, dtype: str, device, offset: int = 0):
    """Copy numpy storage arrays to the device.  offset > 0 places each buffer
    `offset` elements into a larger allocation (a deliberately misaligned
    base that still lies inside its allocation)."""
    out = []
    for x in xs:
        if dtype == "bfloat16":
            t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(x))
        if offset:
            big = torch.empty(x.size + offset, dtype=t.dtype, device=device)
            big[offset:].copy_(t)
            out.append(big[offset:])
        else:
            out.append(t.to(device))
    return out


def empty_like_rank(torch, n: int, numel: int, dtype: str, device, offset: int = 0,
                    fill=None):
    tdt = torch_dtype(torch, dtype)
    out = []
    for _ in range(n):
        big = torch.empty(numel + offset, dtype=tdt, device=device)
        if fill is not None:
            big.fill_(fill)
        out.append(big[offset:] if offset else big)
    return out


def to_host(t, dtype: str) -> np.ndarray:
    """A device tensor's bytes as the numpy storage type (bf16 as uint16)."""
    if dtype == "bfloat16":
        import torch
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bits(a: np.ndarray, dtype: str) -> np.ndarray:
    return np.ascontiguousarray(a).view(NP_BITS[dtype])


def assert_bits_equal(got, want, dtype: str, msg: str = ""):
    g, w = bits(got, dtype), bits(want, dtype)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{msg}: {bad.size} of {g.size} elements differ; first at "
                             f"{bad[:5].tolist()}: got {g[bad[:5]].tolist()} "
                             f"want {w[bad[:5]].tolist()}")
