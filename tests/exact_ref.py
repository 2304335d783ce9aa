"""Exact rational brute force used to pin the oracle (tests only).

Everything here works on Python ``fractions.Fraction`` values decoded from raw bf16
bits with ``struct``: no floating-point rounding happens until the final, explicitly
written round-to-nearest-even. It shares no code with the oracle or the CUDA path.
"""
from __future__ import annotations

import struct
from fractions import Fraction


def bf16_bits_to_fraction(h: int) -> Fraction:
    """Exact value of a finite bf16 pattern."""
    (f,) = struct.unpack("<f", struct.pack("<I", (int(h) & 0xFFFF) << 16))
    return Fraction(f)  # a float converts to Fraction exactly


def _floor_log2(q: Fraction) -> int:
    """floor(log2(q)) for q > 0, exactly."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    # now 2^(e-1) < q < 2^(e+1); fix up
    if q >= Fraction(2) ** e:
        while q >= Fraction(2) ** (e + 1):
            e += 1
    else:
        while q < Fraction(2) ** e:
            e -= 1
    return e


def fraction_to_bf16_bits(q: Fraction) -> int:
    """Round an exact rational to bf16, nearest with ties to even, overflow to inf."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = -q if q < 0 else q
    E = _floor_log2(a)
    qexp = max(E, -126) - 7
    n = a / (Fraction(2) ** qexp)
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = Fraction(fl) * (Fraction(2) ** qexp)
    if r >= Fraction(2) ** 128:
        return sign | 0x7F80
    (u,) = struct.unpack("<I", struct.pack("<f", float(r)))
    return sign | ((u >> 16) & 0x7FFF)


def dot_exact(xbits, wbits) -> Fraction:
    return sum((bf16_bits_to_fraction(a) * bf16_bits_to_fraction(b)
                for a, b in zip(xbits, wbits)), Fraction(0))


def linear_exact(X, W, R=None):
    """Exact y[b][n] = sum_k X[b,k] W[n,k] (+ R[b,n]) as Fractions (nested lists)."""
    B, N = len(X), len(W)
    out = []
    for b in range(B):
        row = []
        for n in range(N):
            s = dot_exact(X[b], W[n])
            if R is not None:
                s += bf16_bits_to_fraction(R[b][n])
            row.append(s)
        out.append(row)
    return out
