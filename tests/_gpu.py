"""Helpers shared by the GPU parity tests.

Acceptance bars. Exchanges are bit-exact. Attention outputs and gradients must
be within max-abs 2e-2 and mean-abs 2e-3 of the fp64 oracle for bf16 inputs,
and within 1e-4 for fp32.

The absolute bound is widened by one ulp of the element type relative to the
reference: |x - ref| <= atol + rtol * |ref|. A bf16 value at or above 8 is
spaced 1/16 from its neighbours, so rounding alone can put it more than 2e-2
from the exact result. The early keys' dV (a sum over every later query of the
GQA group) reaches such magnitudes. rtol = 2^-7 is one bf16 ulp: half an ulp
for the final rounding and half for the fp32 arithmetic before it. The
mean-abs bound stays absolute. The tests also report the plain max-abs.
"""
import math

import torch

F64 = torch.float64

TOL = {
    torch.bfloat16: {"atol": 2e-2, "rtol": 2.0 ** -7, "mean": 2e-3},
    torch.float32: {"atol": 1e-4, "rtol": 1e-6, "mean": 1e-4},
}


def errors(gpu: torch.Tensor, ref: torch.Tensor):
    d = (gpu.detach().cpu().to(F64) - ref.cpu().to(F64)).abs()
    if d.numel() == 0:
        return 0.0, 0.0
    return float(d.max()), float(d.mean())


def assert_close(name, gpu, ref, dtype, check_mean=True):
    """Element-wise bound; the mean-abs bound too unless the sample is biased.

    A sample chosen for its large values (keys at document starts, say) is not
    a fair sample for a whole-tensor mean: for those, only the element-wise
    bound applies.
    """
    t = TOL[dtype]
    g = gpu.detach().cpu().to(F64)
    r = ref.cpu().to(F64)
    d = (g - r).abs()
    if d.numel() == 0:
        return 0.0, 0.0
    mx, mean = float(d.max()), float(d.mean())
    assert math.isfinite(mx), f"{name}: non-finite output"
    bound = t["atol"] + t["rtol"] * r.abs()
    worst = float((d / bound).max())
    assert worst <= 1.0, (f"{name}: |x-ref| exceeds atol {t['atol']} + rtol {t['rtol']:.3g}*|ref| "
                          f"(worst ratio {worst:.3g}, max-abs {mx:.3g})")
    if check_mean:
        assert mean <= t["mean"], f"{name}: mean-abs {mean:.3g} > {t['mean']}"
    return mx, mean


def to_cuda(shards):
    return [s.cuda() for s in shards]


def cat_cpu(shards):
    return torch.cat([s.cpu() for s in shards], 0)
