"""Seeded synthetic workloads for the NVFP4 grouped GEMM (shared by tests and bench).

This module only *makes inputs*: problem sizes, fp32 draws and their NVFP4
quantisation into the bytes both the GPU path and the CPU oracle consume. It
holds none of the GEMM's arithmetic (no decoding, no products, no sums).

The five workloads follow the shapes of the "nvfp4 group gemm" task
(submission 499344, custom_kernel docstring: per group A [m, k/2] fp4x2,
B [n, k/2] fp4x2, per-16 e4m3 scales, fp16 C [m, n], l = 1):

  ``tiny``     G=2: (128,128,256), (64,256,256)
  ``decode``   G=8, m_g ~ U[40,192], n=4096, k=7168          (weight streaming)
  ``prefill``  G=8, m_g=1024, n=4096, k=7168                 (tensor bound)
  ``ragged``   G=4, m_g=(1,17,333,1000), n=7168, k=2048; B ~ N(0, 0.02^2)
               with 1% of elements multiplied by 50 (e4m3 subnormal scales)
  ``zipf64``   G=64, 16384 tokens routed over 60 active experts with
               popularity proportional to rank^-1.2, 4 idle experts (m=0)
               scattered among them; n=2048, k=7168

Quantisation (per row, per 16-element K block):
  sf   = e4m3fn(round-to-nearest-even(min(amax/6, 448)))   (torch's fp8 cast)
  code = e2m1 round-to-nearest-even, saturating at 6, of x / sf
         (all codes +0 when sf decodes to 0)
  two codes per byte, the even k in the low nibble.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

WORKLOADS = ("tiny", "decode", "prefill", "ragged", "zipf64")

# e2m1 magnitudes are 0, .5, 1, 1.5, 2, 3, 4, 6 (codes 0..7). A magnitude v is
# encoded by counting the decision boundaries <= v; on an exact boundary the
# even code wins, so the boundaries between an even code and the next odd one
# (0.25, 1.25, 2.5, 5.0) round down.
_E2M1_BOUNDS = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=torch.float32)
_TIES_DOWN = torch.tensor([0.25, 1.25, 2.5, 5.0], dtype=torch.float32)


@dataclass
class GroupedProblem:
    """One grouped call's inputs, host side (numpy, C-contiguous)."""

    name: str
    seed: int
    problem_sizes: list            # [(m, n, k, l)]
    A: list = field(default_factory=list)      # uint8 [m, k/2]
    B: list = field(default_factory=list)      # uint8 [n, k/2]
    SFA: list = field(default_factory=list)    # uint8 [m, k/16] row-major e4m3fn codes
    SFB: list = field(default_factory=list)    # uint8 [n, k/16]

    @property
    def group_count(self) -> int:
        return len(self.problem_sizes)

    def flops(self) -> float:
        return float(sum(2 * m * n * k for m, n, k, _ in self.problem_sizes if m > 0 and n > 0 and k > 0))

    def algorithmic_bytes(self) -> float:
        """A + B + scales + C over groups with m, n, k > 0 (no padding, B once)."""
        tot = 0
        for m, n, k, _ in self.problem_sizes:
            if m > 0 and n > 0 and k > 0:
                tot += m * k // 2 + n * k // 2 + m * k // 16 + n * k // 16 + 2 * m * n
        return float(tot)


def _rng(seed: int, name: str, *stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), WORKLOADS.index(name), *[int(s) for s in stream]])


def problem_sizes(name: str, seed: int = 0) -> list:
    """(m, n, k, l) per group for a named workload."""
    if name == "tiny":
        return [(128, 128, 256, 1), (64, 256, 256, 1)]
    if name == "decode":
        ms = np.random.default_rng(seed).integers(40, 193, 8)
        return [(int(m), 4096, 7168, 1) for m in ms]
    if name == "prefill":
        return [(1024, 4096, 7168, 1)] * 8
    if name == "ragged":
        return [(m, 7168, 2048, 1) for m in (1, 17, 333, 1000)]
    if name == "zipf64":
        return [(m, 2048, 7168, 1) for m in zipf_routing(seed)]
    raise ValueError(f"unknown workload {name!r}; expected one of {WORKLOADS}")


def zipf_routing(seed: int = 0, tokens: int = 16384, experts: int = 64, idle: int = 4,
                 s: float = 1.2) -> list:
    """Token counts per expert: 60 active experts with popularity ~ rank^-s,
    a multinomial draw of all tokens over them, 4 idle experts, and a seeded
    permutation that scatters ranks and idle experts over the group indices."""
    rng = _rng(seed, "zipf64", 0xD15)
    active = experts - idle
    p = np.arange(1, active + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    counts = rng.multinomial(tokens, p)
    m = np.concatenate([counts, np.zeros(idle, dtype=counts.dtype)])
    m = m[rng.permutation(experts)]
    return [int(x) for x in m]


def quantize_nvfp4(x: torch.Tensor):
    """fp32 [rows, k] (k % 16 == 0) -> (codes uint8 [rows, k/2], sf uint8 [rows, k/16])."""
    assert x.dtype == torch.float32 and x.dim() == 2 and x.shape[1] % 16 == 0
    rows, k = x.shape
    blocks = x.reshape(rows, k // 16, 16)
    amax = blocks.abs().amax(dim=2)
    sf8 = torch.clamp(amax / 6.0, max=448.0).to(torch.float8_e4m3fn)
    sf_dec = sf8.to(torch.float32)
    safe = torch.where(sf_dec > 0, sf_dec, torch.ones_like(sf_dec))
    v = torch.where((sf_dec > 0)[..., None], blocks / safe[..., None], torch.zeros_like(blocks))
    mag = v.abs()
    code = torch.bucketize(mag, _E2M1_BOUNDS, right=True)
    code = code - torch.isin(mag, _TIES_DOWN).to(code.dtype)
    code = code | ((v < 0).to(code.dtype) << 3)
    code = code.to(torch.uint8).reshape(rows, k // 2, 2)
    packed = code[..., 0] | (code[..., 1] << 4)
    return packed.contiguous().numpy(), sf8.view(torch.uint8).contiguous().numpy()


def _draw(rng: np.random.Generator, rows: int, k: int, name: str, role: int) -> torch.Tensor:
    x = rng.standard_normal((rows, k), dtype=np.float32)
    if name == "ragged" and role == 1:
        x *= np.float32(0.02)
        mask = rng.random((rows, k), dtype=np.float32) < np.float32(0.01)
        x[mask] *= np.float32(50.0)
    return torch.from_numpy(x)


def _quantize_rows(rng, rows, k, name, role, chunk_rows=1024):
    codes = np.empty((rows, k // 2), dtype=np.uint8)
    sf = np.empty((rows, k // 16), dtype=np.uint8)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        c, s = quantize_nvfp4(_draw(rng, r1 - r0, k, name, role))
        codes[r0:r1] = c
        sf[r0:r1] = s
    return codes, sf


def make_problem(name: str, seed: int = 0, sizes=None) -> GroupedProblem:
    """Generate the full seeded inputs of a workload (or of explicit sizes,
    drawn like ``name``). Role streams: A = 0, B = 1 per group."""
    if sizes is None:
        sizes = problem_sizes(name, seed)
    sizes = [tuple(int(v) for v in s) for s in sizes]
    prob = GroupedProblem(name=name, seed=seed, problem_sizes=sizes)
    for g, (m, n, k, _l) in enumerate(sizes):
        a, sfa = _quantize_rows(_rng(seed, name, g, 0), max(m, 0), max(k, 0), name, 0)
        b, sfb = _quantize_rows(_rng(seed, name, g, 1), max(n, 0), max(k, 0), name, 1)
        prob.A.append(a)
        prob.SFA.append(sfa)
        prob.B.append(b)
        prob.SFB.append(sfb)
    return prob


def random_codes(rng: np.random.Generator, rows: int, k: int, *, sf_codes=None):
    """Uniformly random e2m1 bytes and e4m3 scale codes (sign clear, no NaN)
    for edge-case tests; ``sf_codes`` restricts the scale codes drawn."""
    a = rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    if sf_codes is None:
        sf_codes = np.arange(0, 0x7F, dtype=np.uint8)
    sf = rng.choice(np.asarray(sf_codes, dtype=np.uint8), size=(rows, k // 16))
    return a, sf.astype(np.uint8)
