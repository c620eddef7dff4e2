"""Helpers shared by the tests: bf16 bit arrays <-> torch tensors and error measures."""
import numpy as np

from matrix_orthogonalizing_optimizer_gb300 import inputs


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bits_to_torch(bits, device="cuda"):
    """bf16 tensor of the given bits; rows padded in storage to 16 bytes when needed."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)
    return padded_copy(t)


def padded_copy(t):
    """Copy of t whose rows start on 16-byte boundaries (storage padded, view unpadded)."""
    import torch
    cols = t.shape[-1]
    al = 16 // t.element_size()
    if cols % al == 0:
        return t
    ld = (cols + al - 1) // al * al
    buf = torch.zeros((*t.shape[:-1], ld), dtype=t.dtype, device=t.device)
    v = buf[..., :cols]
    v.copy_(t)
    return v


def empty_like_padded(t, fill=None):
    import torch
    cols = t.shape[-1]
    al = 16 // t.element_size()
    ld = (cols + al - 1) // al * al
    buf = torch.empty((*t.shape[:-1], ld), dtype=t.dtype, device=t.device)
    if fill is not None:
        buf.fill_(fill)
    return buf[..., :cols]


def torch_to_bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def torch_to_f64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def bf16_input(seed, shape, scale=1.0, stream=0, dist="gaussian"):
    """(bits uint16, float64 decoded) of a seeded bf16 input."""
    if dist == "gaussian":
        x = inputs.gaussian(seed, shape, scale, stream=stream)
    elif dist == "student_t":
        x = inputs.student_t(seed, shape, stream=stream) * scale
    else:
        raise ValueError(dist)
    bits = inputs.round_to_bf16_bits(x)
    return bits, inputs.bf16_bits_to_f32(bits).astype(np.float64)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (for normal values)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def f16_input(seed, shape, scale=1.0, stream=0):
    """(float16 array, float64 decoded) of a seeded input rounded once to fp16 (numpy's
    float16 conversion rounds to nearest even)."""
    x16 = (inputs.gaussian(seed, shape, scale, stream=stream)).astype(np.float16)
    return x16, x16.astype(np.float64)


def f16_to_torch(x16, device="cuda"):
    import torch
    return padded_copy(torch.from_numpy(np.ascontiguousarray(x16)).to(device))
