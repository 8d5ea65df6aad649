"""Test-side model of the library's tensor-core arithmetic (3xTF32 and TF32).

A diagnostic description of how the kernels accumulate, checked against the
library's GEMM in tests/test_gpu_tc_arith.py and used to reason about the
accuracy of fp32-class products.  No parity gate reads it: every gate is against
the float64 oracle (relaxed at most to twice a plain float32 run's error).

The rule, as measured on crafted TF32-exact inputs through the library's own
GEMM (one MMA instruction = eight products of one K = 8 slice):
  * the eight exact products and the running fp32 accumulator are aligned to the
    largest exponent E among them; each addend is truncated toward zero at
    resolution 2^(E - 25), i.e. two bits below the fp32 ulp at E;
  * the truncated addends are summed exactly and the sum is rounded to fp32
    toward zero.
So 1 + 0.75 ulp gives 1, 1 - 1.25 * 2^-24 gives 1 - 2^-24 (the small addend is
truncated first), 1 + 4 * 2^-25 is exact, and 2^10 - 2^10 + 3 * 2^-20 gives 0.
The GEMM kernels issue, per K = 8 slice, lo*hi, hi*lo and hi*hi (3xTF32) or one
hi*hi (TF32).  For B a multiple of 256 the 3xTF32 kernel starts a fresh partial
accumulator every PARTIAL_SUB slices and adds the partials in fp32 with
round-to-nearest, in order; other sizes accumulate over the whole K.

Everything runs in float64 torch on whatever device the inputs live on.
"""

import torch

GUARD = 25          # addend resolution: 2^(E - GUARD)
PARTIAL_SUB = 2     # K = 8 slices per partial in the B % 256 == 0 3xTF32 kernel


def rna_tf32(t):
    """fp32 -> TF32 (10 explicit mantissa bits), ties away from zero."""
    bits = t.float().contiguous().view(torch.int32)
    return ((bits + 0x1000) & ~0x1FFF).view(torch.float32)


def split_tf32(t):
    hi = rna_tf32(t)
    return hi, rna_tf32(t.float() - hi)


def rz32(x):
    """float64 -> float32, rounded toward zero."""
    f = x.float()
    over = f.double().abs() > x.abs()
    return torch.where(over, torch.nextafter(f, torch.zeros_like(f)), f)


def mma_accumulate(acc, prods):
    """One MMA instruction: acc (..., n, m) fp32, prods (..., 8, n, m) exact float64."""
    a = acc.double()
    mx = torch.maximum(prods.abs().amax(dim=-3), a.abs())
    e = torch.floor(torch.log2(torch.where(mx > 0, mx, torch.ones_like(mx))))
    res = torch.exp2(e - GUARD)
    s = (torch.trunc(prods / res.unsqueeze(-3)) * res.unsqueeze(-3)).sum(dim=-3)
    s = s + torch.trunc(a / res) * res
    return rz32(s)


def gemm(a, b, prec, partial_sub=None):
    """C = a @ b (2-D fp32 operands) as the kernels form it.

    prec "3xtf32" splits both operands into TF32 hi + lo and issues lo*hi, hi*lo,
    hi*hi per slice; "tf32" rounds them to TF32 and issues one product.
    partial_sub=None accumulates over all of K; an integer starts a fresh partial
    every partial_sub slices, the partials summed in order with round-to-nearest."""
    if prec == "3xtf32":
        ah, al = split_tf32(a)
        bh, bl = split_tf32(b)
        passes = [(al, bh), (ah, bl), (ah, bh)]
    elif prec == "tf32":
        passes = [(rna_tf32(a), rna_tf32(b))]
    else:
        raise ValueError(prec)
    n, K = a.shape
    m = b.shape[1]
    if K % 8:
        raise ValueError("K must be a multiple of 8")
    steps = K // 8
    sub = steps if partial_sub is None else partial_sub
    if steps % sub:
        raise ValueError("partial length must divide K / 8")
    ng = steps // sub
    acc = torch.zeros((ng, n, m), dtype=torch.float32, device=a.device)
    lane = torch.arange(8, device=a.device)
    for s in range(sub):
        idx = (torch.arange(ng, device=a.device) * sub * 8 + s * 8)[:, None] + lane[None]
        for x, y in passes:
            xs = x.double()[:, idx].permute(1, 2, 0)          # (ng, 8, n)
            ys = y.double()[idx]                              # (ng, 8, m)
            acc = mma_accumulate(acc, xs.unsqueeze(-1) * ys.unsqueeze(-2))
    out = acc[0]
    for g in range(1, ng):
        out = out + acc[g]
    return out


def partial_sub_for(b, prec):
    return PARTIAL_SUB if (prec == "3xtf32" and b % 256 == 0) else None
