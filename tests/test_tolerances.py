"""CPU measurements behind the parity tolerances that are not plain
precision statements (tests/_harness.py).

The short convolution's fp16 / bf16 outputs are allowed CONV_Y_ABS absolute
beside the one-step bar: the kernel forms y's pre-activation as an fp32 sum
of the bias and KW products, whose error, for outputs near zero, is many
16-bit steps.  Here that sum is evaluated as the kernel does (fp32, one
rounding per fused multiply-add, in the same order) on the layer-shape
workloads, and its error against the exact value must stay well inside the
floor."""
import numpy as np
import torch

from kda_linear_attention_gated_gb300 import workloads
from _harness import CONV_Y_ABS


def _fma32(a, b, c):
    # a * b + c rounded once to fp32 (the fp64 product of two fp32 values is exact)
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def test_conv_fp32_sum_error_is_inside_the_absolute_floor():
    worst, worst_rel = 0.0, 0.0
    for dt, seed in [(torch.bfloat16, 80 + j) for j in range(6)] + [(torch.float16, 60), (torch.bfloat16, 60)]:
        s = workloads.make_conv(n=16, t=5, dtype=dt, seed=seed, reset_p=0.25, pad_p=0.1)
        W, x = s.window.double().numpy(), s.x.double().numpy()
        w, b = s.weight.double().numpy(), s.bias.double().numpy()
        kw, T = w.shape[1], s.max_t
        for r in range(s.conv_slot.shape[0]):
            slot = int(s.conv_slot[r])
            if slot < 0:
                continue
            acc = int(s.accepted[r]) - 1
            zero_hist = s.reset is not None and int(s.reset[r]) != 0
            hist = np.zeros((kw - 1, x.shape[1])) if zero_hist else W[slot, acc:acc + kw - 1]
            z = np.concatenate([hist, x[r * T:(r + 1) * T]], 0)
            for t in range(T):
                exact = b + sum(w[:, i] * z[t + i] for i in range(kw))
                s32 = b.astype(np.float32)
                for i in range(kw):
                    s32 = _fma32(w[:, i].astype(np.float32), z[t + i].astype(np.float32), s32)
                err = np.abs(s32.astype(np.float64) - exact)
                mag = np.abs(b) + sum(np.abs(w[:, i] * z[t + i]) for i in range(kw))
                worst = max(worst, float(err.max()))
                worst_rel = max(worst_rel, float((err / mag).max()))
    # the fp32 error bound of a (KW + 1)-term sum, against the sum of |terms|
    assert worst_rel <= (4 + 1) * 2.0 ** -24
    # SiLU's slope is below 1.1, so y inherits at most 1.1x this: the floor
    # leaves more than a factor 2 beyond it
    assert 1.1 * worst <= CONV_Y_ABS / 2, worst
