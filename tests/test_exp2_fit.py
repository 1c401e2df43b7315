"""The forward kernels' optional FMA-pipe 2^x (exp2_fma2 in attn_fwd_common.cuh): its cubic
for 2^f on [0, 1) and the Cody-Waite composition 2^x = 2^floor(x) * 2^f stay within the
stated relative error of 7.5e-5 (far below the bf16 rounding of P, 2^-9), evaluated here in
float32 from the coefficients as they stand in the source (no GPU needed)."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "content_adaptive_sparse_gb300",
                   "csrc", "attn_fwd_common.cuh")


def _coefficients():
    text = open(SRC).read()
    body = text[text.index("uint64_t exp2_fma2("):]
    body = body[:body.index("\n}\n")]
    vals = [float(v) for v in re.findall(r"f2_pack\(([-0-9.e]+)f, \1f\)", body)]
    # in order of use: -127 clamp is not a pair; magic 1.5 * 2^23; then c3, c2, c1, c0
    vals = [v for v in vals if v not in (12582912.0,)]
    assert len(vals) == 4, vals
    return [np.float32(v) for v in vals]


def _cubic(f):
    c3, c2, c1, c0 = _coefficients()
    f = f.astype(np.float32)
    q = (c3 * f + c2).astype(np.float32)
    q = (q * f + c1).astype(np.float32)
    return (q * f + c0).astype(np.float32)


def test_cubic_fit_on_unit_interval():
    f = np.linspace(0.0, 1.0, 1_000_001, endpoint=False, dtype=np.float64)
    rel = np.abs(_cubic(f).astype(np.float64) - np.exp2(f)) / np.exp2(f)
    assert rel.max() <= 7.5e-5, rel.max()


def test_composed_exp2_over_the_kernel_range():
    x = np.concatenate([np.linspace(-126.0, 8.0, 400_001), np.array([-126.0, -1e-7, 0.0, 7.999, 8.0])])
    n = np.floor(x)
    f = (x - n).astype(np.float32)
    got = _cubic(f).astype(np.float64) * np.exp2(n)
    rel = np.abs(got - np.exp2(x)) / np.exp2(x)
    assert rel.max() <= 7.5e-5, rel.max()
