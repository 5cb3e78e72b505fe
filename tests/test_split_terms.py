"""The float32 accuracy claim behind the tensor-core products of the basis fit and the predictor fit, checked in
plain float arithmetic on the CPU.

Those products split every float32 operand into three bf16 terms, x = h + m + l with h = bf16(x), m = bf16(x - h),
l = bf16(x - h - m), and keep six of the nine term products (hh, hm, mh, hl, lh, mm). This file checks two things:
- the split is exact for float32 values across the exponent range;
- the three dropped products stay under 2^-23 |x| |y| per product, so a six-product dot product is within
  2^-23 sum_k |a_k| |b_k| of the exact one. That is the size of float32 rounding.
"""
import numpy as np
import torch


def bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).to(torch.float32)      # round to nearest even, back to float32 exactly


def split3(x: torch.Tensor):
    h = bf16(x)
    r1 = x - h                  # float32 arithmetic, exact
    m = bf16(r1)
    l = bf16(r1 - m)
    return h, m, l


def test_three_bf16_terms_are_exact():
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 8)).to(torch.float32)
    x = torch.cat([x, torch.tensor([1.0, -1.0, 3.0e38, -1.2e-30, 0.1, 1 / 3, 2 ** -100 * 1.2345678], dtype=torch.float32)])
    h, m, l = split3(x)
    total = h.double() + m.double() + l.double()
    assert torch.equal(total, x.double())
    # each term is a bf16 value
    for t in (h, m, l):
        assert torch.equal(t, bf16(t))


def test_six_products_keep_float32_accuracy():
    g = torch.Generator().manual_seed(1)
    A = torch.randn(64, 300, generator=g) * torch.exp(torch.randn(64, 1, generator=g))
    B = torch.randn(48, 300, generator=g) * torch.exp(torch.randn(48, 1, generator=g))
    ta, tb = split3(A), split3(B)
    pairs = [(0, 0), (0, 1), (1, 0), (0, 2), (2, 0), (1, 1)]
    C = sum(ta[i].double() @ tb[j].double().T for i, j in pairs)
    exact = A.double() @ B.double().T
    bound = 2.0 ** -23 * (A.double().abs() @ B.double().abs().T)
    assert torch.all((C - exact).abs() <= bound)
    # and three products (dropping hl, lh, mm) would not: their size is 2^-16, far above float32 rounding
    C3 = sum(ta[i].double() @ tb[j].double().T for i, j in pairs[:3])
    assert float(((C3 - exact).abs() / bound).max()) > 8.0


def test_one_bf16_term_is_far_from_float32():
    # why the split: a plain bf16 product (one term each) is off by about 2^-8 relative
    g = torch.Generator().manual_seed(2)
    A = torch.randn(32, 256, generator=g)
    B = torch.randn(32, 256, generator=g)
    one = bf16(A).double() @ bf16(B).double().T
    exact = A.double() @ B.double().T
    rel = float(((one - exact).abs() / (A.double().abs() @ B.double().abs().T)).max())
    assert rel > 2.0 ** -12
    assert np.isfinite(rel)
