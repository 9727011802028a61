"""Device-resident operands of one grouped call (torch used for memory only).

``DeviceProblem.upload`` copies a host :class:`~.workloads.GroupedProblem` to
the GPU and reorders its row-major scales into the atom layout with the
library's packer kernel; ``run`` issues one ``nvfp4_grouped_gemm``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import grouped_gemm, pack_scales_tensor

SENTINEL_F16 = 0x7E00  # fp16 quiet NaN, marks C entries the kernel must not touch


@dataclass
class DeviceProblem:
    problem_sizes: list
    A: list = field(default_factory=list)
    B: list = field(default_factory=list)
    SFA: list = field(default_factory=list)     # atom layout
    SFB: list = field(default_factory=list)
    C: list = field(default_factory=list)

    @classmethod
    def upload(cls, prob, device="cuda", stream=None, fill_c=SENTINEL_F16):
        dp = cls(problem_sizes=list(prob.problem_sizes))
        for g, (m, n, k, _l) in enumerate(prob.problem_sizes):
            a = torch.from_numpy(np.ascontiguousarray(prob.A[g])).to(device)
            b = torch.from_numpy(np.ascontiguousarray(prob.B[g])).to(device)
            sfa = torch.from_numpy(np.ascontiguousarray(prob.SFA[g])).to(device)
            sfb = torch.from_numpy(np.ascontiguousarray(prob.SFB[g])).to(device)
            dp.A.append(a)
            dp.B.append(b)
            dp.SFA.append(pack_scales_tensor(sfa, k, stream) if m > 0 and k > 0 else sfa)
            dp.SFB.append(pack_scales_tensor(sfb, k, stream) if n > 0 and k > 0 else sfb)
            c = torch.full((max(m, 0), max(n, 0)), fill_c, dtype=torch.int16, device=device)
            dp.C.append(c.view(torch.float16))
        return dp

    def run(self, stream=None) -> None:
        ptr = lambda t: 0 if t is None or t.numel() == 0 else int(t.data_ptr())
        grouped_gemm(self.problem_sizes, [ptr(t) for t in self.A], [ptr(t) for t in self.B],
                     [ptr(t) for t in self.SFA], [ptr(t) for t in self.SFB], [ptr(t) for t in self.C], stream)

    def c_host(self):
        return [c.cpu().numpy() for c in self.C]
