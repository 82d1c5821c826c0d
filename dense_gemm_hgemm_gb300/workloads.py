"""The workloads the library is measured and checked on (shapes, dtypes, input scales).

Each entry names what it is with its sizes.  The input recipe is
``inputs.make_operands`` with the listed scales.
"""
from __future__ import annotations

from dataclasses import dataclass

SWEEP_SIZES = (64, 128, 256, 512, 1024, 2048, 4096)


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str          # operand type: "f16", "bf16" or "i8"
    a_scale: float = 1.0
    b_scale: float = 1.0

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def in_elt(self) -> int:
        return 1 if self.dtype == "i8" else 2

    @property
    def out_elt(self) -> int:
        return 4 if self.dtype == "i8" else 2

    @property
    def compulsory_bytes(self) -> int:
        """A, B and C each moved once."""
        return (self.M * self.K + self.N * self.K) * self.in_elt + self.M * self.N * self.out_elt


SKINNY = Workload("hgemm_tn_64x4096x64_f16", 64, 4096, 64, "f16")
HEADLINE_SWEEP = Workload("hgemm_tn_128x2048x128_f16", 128, 2048, 128, "f16")
SQUARE_8192 = Workload("hgemm_tn_8192x8192x8192_f16", 8192, 8192, 8192, "f16", 0.1, 0.1)
FFN_BF16 = Workload("ffn_bf16_tn_4096x14336x4096", 4096, 14336, 4096, "bf16", 1.0, 0.02)
INT8_4096 = Workload("igemm_tn_4096x4096x4096_i8_i32", 4096, 4096, 4096, "i8")

NAMED = (SKINNY, HEADLINE_SWEEP, SQUARE_8192, FFN_BF16, INT8_4096)


def sweep_shapes():
    """The 343-shape fp16 sweep: every (M, N, K) with M, N, K in SWEEP_SIZES."""
    return [Workload("sweep_%dx%dx%d_f16" % (m, n, k), m, n, k, "f16")
            for m in SWEEP_SIZES for n in SWEEP_SIZES for k in SWEEP_SIZES]
