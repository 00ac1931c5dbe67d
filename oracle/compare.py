"""Comparisons of GPU results with the oracle, at stated tolerances (test only).

Tolerances (the stated bar: bit-exact for masks, indices and layouts; 1 bf16
ulp after float32 accumulation for bf16 outputs; max-abs 1e-5 for float32
outputs), with the two places where float32 arithmetic itself cannot meet
the literal figure made explicit:

* bf16 outputs computed from a float32 expression: the GPU value must be
  within 1 ulp of the exact (float64) value rounded to bf16, OR within an
  absolute floor of 2**-16 times the magnitude of the expression's terms.
  The floor matters only where the result cancels to far below its terms
  (a float32 evaluation carries an absolute error of a few 2**-24 of the
  terms, which there exceeds a bf16 ulp of the result); 2**-16 is 256 float32
  units, well above that error and below a bf16 ulp of any non-cancelled
  value.
* float32 per-token outputs (mean, rstd): |gpu - ref| <= 1e-5 * max(1, |ref|).
* float32 sums over tokens (dgamma, dbeta, dbias): |gpu - ref| <=
  1e-5 * max(1, rss) where rss is the root-sum-square of the summed terms,
  the natural scale of a sum of mixed-sign terms; float32 rounding of the
  terms and of the sum stays orders of magnitude below it, while a wrong,
  missing or extra term moves the sum by about rss.
"""
import numpy as np

from .bf16 import bf16_round, order_key

FLOOR_REL = 2.0 ** -16


def bf16_bits(x):
    """uint16 bit patterns of a torch bf16 tensor / float32 array of bf16 values."""
    if hasattr(x, "view") and hasattr(x, "dtype") and "bfloat16" in str(x.dtype):
        import torch
        return x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _bf16_tests(gpu_bits, ref_exact, magnitude, max_ulp):
    """(within max_ulp of the rounded exact value, within the magnitude floor)."""
    ref_bits = bf16_bits(bf16_round(ref_exact))
    ulps = np.abs(order_key(gpu_bits) - order_key(ref_bits))
    gpu = (np.asarray(gpu_bits).astype(np.uint32) << np.uint32(16)).view(np.float32)
    abs_err = np.abs(gpu.astype(np.float64) - np.asarray(ref_exact, dtype=np.float64))
    return ulps <= max_ulp, abs_err <= FLOOR_REL * np.asarray(magnitude, dtype=np.float64)


def bf16_mismatch(gpu_bits, ref_exact, magnitude, max_ulp=1):
    """Boolean mask of elements failing the bf16 tolerance."""
    near, floor = _bf16_tests(gpu_bits, ref_exact, magnitude, max_ulp)
    return ~(near | floor)


def bf16_floor_only(gpu_bits, ref_exact, magnitude, max_ulp=1):
    """Boolean mask of elements that pass the bf16 tolerance only through the
    magnitude floor (more than max_ulp from the rounded exact value, but
    within 2**-16 of the expression's terms): the cancelled results the floor
    exists for.  Tests bound how many there are, so that the floor cannot
    quietly stand in for the 1-ulp bar."""
    near, floor = _bf16_tests(gpu_bits, ref_exact, magnitude, max_ulp)
    return ~near & floor


def floor_only_bound(n):
    """Most elements out of n that may pass only through the magnitude floor.

    A float32 evaluation misses the 1-ulp bar only where its result cancels
    to below about 2**-15 of the expression's terms; with the workloads'
    distributions that is a few elements in ten million (a float32 emulation
    of the LayerNorm output on the s = h = 4096 inputs: 2 of 8,388,608).  The
    bound allows eight times that rate plus a constant for small tensors."""
    return 8 + int(2e-6 * n)


def f32_rel_mismatch(gpu, ref, tol=1e-5):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(gpu - ref) > tol * np.maximum(1.0, np.abs(ref))


def colsum_mismatch(gpu, ref, rss, tol=1e-5):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(gpu - ref) > tol * np.maximum(1.0, np.asarray(rss, dtype=np.float64))
