"""Test helpers: moving synthetic inputs to the GPU and comparing outputs."""
import numpy as np


def bits_to_f64(bits):
    b = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_dev(L, device="cuda"):
    """numpy layer dict (bf16 as uint16 bits) -> torch CUDA tensors."""
    import torch
    out = {}
    for key, v in L.items():
        if v is None:
            out[key] = None
        elif key == "x":
            out[key] = torch.from_numpy(v.view(np.int16)).to(device).view(torch.bfloat16)
        else:
            out[key] = torch.from_numpy(np.ascontiguousarray(v)).to(device)
    return out


def bf16_tensor_bits(t):
    """CUDA/CPU bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def row_rel_l2(got_bits, ref_bits):
    """max over rows of ||got - ref||_2 / ||ref||_2 (and the elementwise max
    |err| / ||ref_row||_2)."""
    g, r = bits_to_f64(got_bits), bits_to_f64(ref_bits)
    num = np.sqrt(((g - r) ** 2).sum(axis=-1))
    den = np.sqrt((r ** 2).sum(axis=-1))
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max()), float((np.abs(g - r).max(axis=-1) / den).max())


# The layer output bar: row-L2-normalised relative error with fp32 accumulation.
OUTPUT_RTOL = 1e-2


def concatenated_fc1(w1, s1, kmajor=False):
    """FC1 weights and block scales with interleaved gate/linear columns
    (2m, 2m + 1) rewritten in the concatenated order (m, I + m) of
    swiglu_fusion = 2: column c of the result is column 2c (c < I) or
    2(c - I) + 1 of the input.  w1 packed [E, H, I] (low nibble = even
    column), s1 [E, 2I, H/bs] ([E, H/bs, 2I] when kmajor)."""
    w1 = np.asarray(w1, np.uint8)
    E, H, half = w1.shape
    codes = np.empty((E, H, 2 * half), np.uint8)
    codes[..., 0::2] = w1 & 0xF
    codes[..., 1::2] = w1 >> 4
    perm = np.concatenate([np.arange(0, 2 * half, 2), np.arange(1, 2 * half, 2)])
    c2 = codes[..., perm]
    w1c = (c2[..., 0::2] | (c2[..., 1::2] << 4)).astype(np.uint8)
    s1 = np.asarray(s1, np.uint8)
    s1c = s1[:, :, perm] if kmajor else s1[:, perm, :]
    return np.ascontiguousarray(w1c), np.ascontiguousarray(s1c)
