"""The comparison an E4M3 forward result must pass against the fp64 oracle
(shared by the GPU tests and by the CPU test that shows it can fail).

The kernel rounds the softmax weights to E4M3 before the second product and
O to bf16, so element by element the error may reach the oracle's rigorous
rounding bound (``oracle.fp8_error_model``) plus the bf16 rounding of O.  A
bound that loose alone cannot see a slip that moves O by a fraction of it (a
wrong V tile, a dropped key tile), so the root-mean-square error over the
tensor is also held to RMS_MULT times the model's expected rounding error:
rounding errors average out across keys, slips do not.  The LSE comes from
fp32 sums of unrounded weights and is held to LSE_ATOL."""
import numpy as np
import torch

from _gpu_helpers import max_err

LSE_ATOL = 1e-3
RMS_MULT = 2.0        # RMS error <= RMS_MULT * sqrt(mean expected squared error)
BF16_REL = 2.0 ** -8  # per-element allowance for rounding O to bf16 (half ulp is <= 2^-8 |O|)
ABS_SLACK = 1e-4      # fp32 sums and the hardware exp2


def _np64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, np.float64)


def check(o, lse, o_ref, l_ref, bound, msq, what):
    o, lse = _np64(o), _np64(lse)
    err = o - o_ref
    tol = bound + BF16_REL * np.abs(o_ref) + ABS_SLACK
    worst = float((np.abs(err) - tol).max())
    assert worst <= 0, f"{what}: O error exceeds the per-element bound by {worst:.3e}"
    # bf16 output rounding: uniform error over a grid step of at most 2^-7 |O|
    expect = np.sqrt(float((msq + (2.0 ** -7 * o_ref) ** 2 / 12.0).mean()))
    rms = float(np.sqrt((err ** 2).mean()))
    assert rms <= RMS_MULT * expect, f"{what}: RMS O error {rms:.3e} > {RMS_MULT} x expected {expect:.3e}"
    el = max_err(lse, l_ref)
    assert el <= LSE_ATOL, f"{what}: LSE max-abs error {el:.3e} > {LSE_ATOL}"
