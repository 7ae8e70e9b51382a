"""Shared helpers of the GPU parity tests: padded device copies, canaries,
and the tolerance checks against the oracle.

Tolerances (the bounds the GEMM is held to):
  * fp32 SIMT path: |out - ref| <= 1e-5 * (|A||B|)_ij + 1e-6
  * fp16/bf16 inputs, fp32 output: |out - ref| <= 2e-3 * (|A||B|)_ij and the
    relative Frobenius error ||out - ref|| / ||ref|| <= 1e-4
  * bf16 output: |out - ref| <= 2e-3 * (|A||B|)_ij + ulp_bf16(ref) / 2 (the
    accumulation bound plus the final rounding to bf16, which the |A||B|
    bound does not contain and which dominates at small K) and
    |out - ref| <= ulp_bf16(ref) + 1e-5 * (|A||B|)_ij (rounding of the fp32
    result to bf16 plus fp32 accumulation error); the Frobenius criterion is
    applied to an fp32-output launch of the same kernel, because rounding to
    bf16 alone already gives about 1e-3 relative Frobenius error.
  * when beta != 0 every bound gains 2^-23 * |beta * C0| (fp32 rounding of the
    beta term; 2^-7 for a bf16 C0), which the |A||B| bound does not cover.
ref and |A||B| always come from the oracle in fp64.
"""
import numpy as np
import torch

from stage_software_pipelining_gb300.workloads import (GEMM_BF16_BF16, GEMM_F32, IN_DTYPE,
                                                       OUT_DTYPE)

CANARY = 12345.0


def round_up(x, m):
    return (x + m - 1) // m * m


def to_device_padded(t: torch.Tensor, col_major: bool = False, pad_rows: int = 0):
    """Copy a host matrix to the GPU in a buffer whose leading dimension is
    rounded up to 16 bytes (plus extra padding), filled with NaN outside it.

    Returns the device view with the logical shape of t."""
    elem = t.element_size()
    mult = 16 // elem
    if col_major:           # t is a K x N view of an N x K row-major tensor
        base = t.t()
        rows, cols = base.shape
        ld = round_up(max(cols, 1), mult) + mult
        buf = torch.full((rows + pad_rows, ld), float("nan"), dtype=t.dtype, device="cuda")
        buf[:rows, :cols].copy_(base)
        return buf[:rows, :cols].t()
    rows, cols = t.shape
    ld = round_up(max(cols, 1), mult) + mult
    buf = torch.full((rows + pad_rows, ld), float("nan"), dtype=t.dtype, device="cuda")
    buf[:rows, :cols].copy_(t)
    return buf[:rows, :cols]


class GuardedC:
    """C inside a larger buffer: one canary row above, one below, canary
    columns to the right.  check() asserts the canaries survived."""

    def __init__(self, M, N, dtype, init=None):
        elem = torch.tensor([], dtype=dtype).element_size()
        mult = 16 // elem
        self.ld = round_up(max(N, 1), mult) + 2 * mult
        self.buf = torch.full((M + 2, self.ld), CANARY, dtype=dtype, device="cuda")
        self.M, self.N = M, N
        self.view = self.buf[1:M + 1, :N]
        if init is not None:
            self.view.copy_(init)

    def check(self):
        b = self.buf.float().cpu()
        inside = torch.zeros_like(b, dtype=torch.bool)
        inside[1:self.M + 1, :self.N] = True
        outside = b[~inside]
        expect = torch.tensor(CANARY, dtype=self.buf.dtype).float()   # canary as stored
        assert torch.all(outside == expect), "a write landed outside C"


def _beta_term(beta, C0):
    if beta == 0.0 or C0 is None:
        return 0.0
    c = C0.double().numpy()
    rel = 2.0 ** -7 if C0.dtype == torch.bfloat16 else 2.0 ** -23
    return rel * np.abs(beta * c)


def ulp_bf16(x):
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_against_oracle(out, ref, absb, dtype, beta=0.0, C0=None, what="", frob=True):
    """Elementwise bound (and Frobenius for fp32-output tensor-core runs)."""
    out = np.asarray(out, dtype=np.float64)
    err = np.abs(out - ref)
    bt = _beta_term(beta, C0)
    if dtype == GEMM_F32:
        bound = 1e-5 * absb + 1e-6 + bt
    elif dtype == GEMM_BF16_BF16:
        bound = 2e-3 * absb + 0.5 * ulp_bf16(ref) + bt
    else:
        bound = 2e-3 * absb + bt
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} entries out of bound; first at {tuple(idx)}: "
            f"out={out[tuple(idx)]!r} ref={ref[tuple(idx)]!r} bound={np.broadcast_to(bound, err.shape)[tuple(idx)]!r}")
    if dtype == GEMM_BF16_BF16:
        b2 = ulp_bf16(ref) + 1e-5 * absb + bt
        bad = ~(err <= b2)
        assert not bad.any(), f"{what}: bf16 output more than one ulp away at " \
                              f"{tuple(np.argwhere(bad)[0])}"
    elif dtype != GEMM_F32 and frob:
        den = np.linalg.norm(ref)
        if den > 0:
            rel = np.linalg.norm(out - ref) / den
            assert rel <= 1e-4, f"{what}: relative Frobenius error {rel:.3e} > 1e-4"
    return float(err.max()) if err.size else 0.0


def in_out_dtypes(code):
    return IN_DTYPE[code], OUT_DTYPE[code]
