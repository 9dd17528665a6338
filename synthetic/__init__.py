"""Seeded synthetic inputs for the QMoE W4A16 layer.

This module only draws random inputs with the shapes and value distributions
of the workloads the pages describe; it holds none of the layer's arithmetic
(no decoding, no routing, no matmul).  Both the oracle-side tests and the CUDA
side read the same arrays from here.

Workloads (decode shapes from the NVFP4 MTP decode / verify measurements and
the 20B-class MXFP4 decode shape on the pages; prefill from the dequant +
grouped-GEMM fallback):

============================  ====  ===  ==  ====  ====  ======
name                             T    E   k     H     I  format
============================  ====  ===  ==  ====  ====  ======
tiny_nvfp4_decode                1    8   2   256   128  NVFP4
nvfp4_mtp_decode                 4  256   8  2048   512  NVFP4
mxfp4_decode                     8   32   4  2880  2880  MXFP4
nvfp4_verify_edge (ties)         8  256   8  4096  2048  NVFP4
nvfp4_prefill                 2048  128   8  2048  1536  NVFP4
============================  ====  ===  ==  ====  ====  ======

Value recipes:
  * activations x ~ N(0, 1), rounded to bf16 (returned as uint16 bit patterns);
  * router logits fp32 ~ N(0, std^2) (std = sqrt(2) for nvfp4_mtp_decode);
  * E2M1 codes uniform over all 16 codes (uniform bytes, two codes per byte);
  * NVFP4 block scales: uniform over the 32 positive E4M3 codes with value in
    [0.25, 4) (exponent field 5..8, any mantissa); per-expert fp32 global
    scale 2^-u, u uniform in {0..4};
  * MXFP4 block scales: E8M0 byte uniform in [120, 134]; no global scale;
  * ties: for every token, 25 logits are copied onto other experts of the
    same row, and the k-th largest value is copied onto a lower-index expert
    outside the top k, so the k-th place is decided by the tie rule.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

NVFP4 = 0
MXFP4 = 1
BLOCK = {NVFP4: 16, MXFP4: 32}


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    E: int
    k: int
    H: int
    I: int
    fmt: int
    logit_std: float = 1.0
    ties: bool = False
    normalize: int = 1
    alpha: float = 1.0
    beta: float = 0.0
    limit: float = math.inf
    note: str = field(default="", compare=False)

    @property
    def bs(self) -> int:
        return BLOCK[self.fmt]

    @property
    def R(self) -> int:
        return self.T * self.k


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_nvfp4_decode", 1, 8, 2, 256, 128, NVFP4,
                 note="tiny NVFP4 decode"),
        Workload("nvfp4_mtp_decode", 4, 256, 8, 2048, 512, NVFP4, logit_std=math.sqrt(2.0),
                 note="NVFP4 MTP decode, 4 token rows"),
        Workload("mxfp4_decode", 8, 32, 4, 2880, 2880, MXFP4,
                 note="MXFP4 decode, 8 token rows"),
        Workload("nvfp4_verify_edge", 8, 256, 8, 4096, 2048, NVFP4, ties=True,
                 note="NVFP4 MTP verify at the 64-row GEMV window edge, with ties"),
        Workload("nvfp4_prefill", 2048, 128, 8, 2048, 1536, NVFP4,
                 note="NVFP4 prefill: dequant + tensor-core grouped GEMM"),
    ]
}


def rng_for(seed: int, stream: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def uniform_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).reshape(shape).copy()


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float -> bf16 bit patterns (uint16), rounded by torch's own cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations(rng, T, H) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


def logits(rng, T, E, std=1.0, ties=False, k=1) -> np.ndarray:
    lg = (rng.standard_normal((T, E)) * std).astype(np.float32)
    if ties:
        ndup = int(0.1 * E) if E >= 20 else 1
        for t in range(T):
            row = lg[t]
            src = rng.choice(E, size=ndup, replace=False)
            dst = rng.choice(E, size=ndup, replace=False)
            for s, d in zip(src, dst):
                if s != d:
                    row[d] = row[s]
            # boundary tie: the k-th value (value desc, index asc) also lands on
            # a lower-index expert that is outside the top k
            order = np.lexsort((np.arange(E), -row.astype(np.float64)))
            kth = order[k - 1]
            outside = np.setdiff1d(np.arange(kth), order[:k])
            if outside.size:
                row[rng.choice(outside)] = row[kth]
    return lg


def nvfp4_scales(rng, shape) -> np.ndarray:
    idx = rng.integers(0, 32, size=shape, dtype=np.int64)
    return (((idx // 8) + 5) << 3 | (idx % 8)).astype(np.uint8)


def mxfp4_scales(rng, shape) -> np.ndarray:
    return rng.integers(120, 135, size=shape, dtype=np.int64).astype(np.uint8)


def global_scales(rng, E) -> np.ndarray:
    u = rng.integers(0, 5, size=E)
    return np.ldexp(np.ones(E, np.float32), -u).astype(np.float32)


def block_scales(rng, fmt, shape) -> np.ndarray:
    return nvfp4_scales(rng, shape) if fmt == NVFP4 else mxfp4_scales(rng, shape)


def expert_weights(rng, fmt, E, K, N):
    """One FC's packed codes [E, K, N/2], block scales [E, N, K/bs] and global
    scales [E] (None for MXFP4)."""
    bs = BLOCK[fmt]
    packed = uniform_bytes(rng, (E, K, N // 2))
    scales = block_scales(rng, fmt, (E, N, K // bs))
    g = global_scales(rng, E) if fmt == NVFP4 else None
    return packed, scales, g


def layer(w: Workload, seed: int = 0) -> dict:
    """All inputs of one MoE layer for workload ``w``."""
    rng = rng_for(seed, 1)
    x = activations(rng, w.T, w.H)
    lg = logits(rng, w.T, w.E, w.logit_std, w.ties, w.k)
    w1, s1, g1 = expert_weights(rng, w.fmt, w.E, w.H, 2 * w.I)
    w2, s2, g2 = expert_weights(rng, w.fmt, w.E, w.I, w.H)
    return dict(x=x, logits=lg, w1=w1, s1=s1, g1=g1, w2=w2, s2=s2, g2=g2)


def small(name="small", T=3, E=6, k=2, H=64, I=32, fmt=NVFP4, **kw) -> Workload:
    """A small custom workload (for tests)."""
    return Workload(name, T, E, k, H, I, fmt, **kw)
