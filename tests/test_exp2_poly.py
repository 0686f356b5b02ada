"""The polynomial exponential that the softmax kernels use for part of their
exponentials (Cody-Waite range reduction in base 2 and a minimax polynomial
found by the Remez exchange algorithm, exact_attention_44_gb300/exp2_poly.py).

CPU: the constants compiled into the kernels are the generator's output, the
generator's polynomial is minimax (equioscillating error), and the kernel's
steps in fp32 stay within the stated relative error of numpy's float64 exp2
over the whole range the softmax feeds it.  GPU: the device routine against
CUDA's own exp2f, through a test hook of the library."""
import os
import re

import numpy as np
import pytest

from exact_attention_44_gb300 import exp2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BOUND = 2.0 ** -18  # 3.8e-6: the degree-4 minimax error (2.6e-6) plus fp32 rounding of the steps


def _kernel_constants():
    text = open(os.path.join(ROOT, "exact_attention_44_gb300", "csrc", "fa_ptx.cuh")).read()
    found = dict(re.findall(r"EXP2_C(\d) = (0x[0-9a-fA-Fp.+-]+)f", text))
    return [float.fromhex(found[str(i)]) for i in range(5)]


def test_kernel_constants_are_the_generators():
    assert _kernel_constants() == exp2_poly.coefficients_f32()


def test_polynomial_is_minimax_on_the_reduced_range():
    c, err = exp2_poly.remez()
    t = np.linspace(-0.5, 0.5, 400001)
    e = np.polyval(c[::-1], t) / np.exp2(t) - 1
    # the error levels out: its largest magnitude is the levelled one, reached
    # with alternating signs at degree + 2 points
    assert abs(np.max(np.abs(e)) - err) < 1e-3 * err
    peaks = np.flatnonzero(np.abs(np.abs(e) - err) < 1e-3 * err)
    signs = np.sign(e[peaks])
    assert np.count_nonzero(np.diff(signs)) + 1 >= exp2_poly.DEGREE + 2
    assert 2e-6 < err < 3e-6
    # lower degrees are worse (degree 3: ~7.5e-5), so degree 4 is the smallest that
    # stays far below the fp16 rounding of P (2^-11)
    assert exp2_poly.remez(3)[1] > 2.0 ** -14


def test_fp32_steps_match_exp2_over_the_softmax_range():
    x = np.linspace(-126.0, 8.0, 4_000_001).astype(np.float32)
    x = np.concatenate([x, np.arange(-126, 9, dtype=np.float32), np.float32([-0.5, 0.5, -1.5, 1.5, 7.999])])
    y = exp2_poly.evaluate_f32(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    assert np.max(rel) < BOUND
    # exact powers of two stay within the bound too, and the result never leaves (0, 2^8]
    assert np.all(y > 0) and np.all(y <= 256.0 * (1 + BOUND))


def test_arguments_below_the_normal_range_give_a_tiny_positive_value():
    y = exp2_poly.evaluate_f32(np.float32([-126.5, -127, -200, -1e30, -np.inf]))
    assert np.all(np.isfinite(y)) and np.all(y > 0) and np.all(y < 2.0 ** -125)


@pytest.mark.gpu
def test_device_routine_against_cuda_exp2f():
    import torch

    import exact_attention_44_gb300 as fa
    fa.build()
    fa.load()
    x = torch.linspace(-126.0, 8.0, 2_000_001, dtype=torch.float64).float().cuda()
    x = torch.cat([x, torch.arange(-126, 9, dtype=torch.float32, device="cuda")])
    y = fa.fa_debug_exp2(x)
    ref = torch.exp2(x)  # CUDA's exp2f
    torch.cuda.synchronize()
    rel = (y.double() / ref.double() - 1).abs().max().item()
    assert rel < BOUND + 2.0 ** -22, rel  # exp2f's own error is at most a couple of ulp
    # odd length: the last element has no partner in its pair
    z = fa.fa_debug_exp2(torch.tensor([0.0, 1.0, -3.0], device="cuda"))
    assert torch.allclose(z, torch.tensor([1.0, 2.0, 0.125], device="cuda"), rtol=BOUND)
