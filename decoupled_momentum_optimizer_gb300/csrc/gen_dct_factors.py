"""Emit dct32_factors.cuh: straight-line DCT-IV blocks for the 32-point DCT.

The CUDA kernels factor the orthonormal 32-point DCT-II by the even/odd split
C_N(x)_{2j} = C_{N/2}(x_n + x_{N-1-n})_j,  C_N(x)_{2j+1} = S_{N/2}(x_n - x_{N-1-n})_j,
where S_M is the DCT-IV of size M, S_M[j][n] = cos(pi (2n+1)(2j+1) / (4M)).
Every S block here is pre-scaled by 1/4 (the orthonormal factor sqrt(2/32) of all
coefficients but X_0), and the last 2-point stage uses cos(pi/4)/4 = sqrt(1/32).

Blocks of size 8 and 16 are computed through a complex DFT of half the size.
With a_p = d[2p], b_p = d[M-1-2p], c_p = a_p - i b_p and t = pi/(4M):
    S_q = e^{i(4q+1)t} * sum_p (c_p e^{i 4p t}) e^{2 pi i p q/(M/2)},
    out[2q] = Re S_q,   out[M-1-2q] = Im S_q,
(split the sum over even n = 2p and odd n = M-1-2p; the cross terms of the
DCT-IV kernel collapse to the pre-twiddle e^{i4pt}, a size-M/2 DFT, and the
post-twiddle e^{i(4q+1)t}).  The DFT is a recursive radix-2 decimation in time.
Blocks of size 2 and 4 are plain products.  Costs: 16 -> 116 flops, 8 -> 44.

The program is recorded as a list of operations on named values; it is printed
as CUDA (float32 constants as hexadecimal literals, folded by the compiler into
FFMA immediates) and can be executed in numpy float32 by ``evaluate`` so that a
CPU test can check the emitted arithmetic against the float64 DCT-IV matrix.
The constants are computed in float64 with the host libm and rounded once.

Run from this folder: ``python gen_dct_factors.py > dct32_factors.cuh``.
"""

import math
import struct
import sys


def f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def f32_hex(v):
    f = f32(v)
    if f == 0.0:
        return "0.0f"
    mant, exp = f.hex().split("p")
    mant = mant.rstrip("0").rstrip(".") if "." in mant else mant
    return f"{mant}p{exp}f"


class Program:
    """Straight-line float32 program: ops are (kind, dst, args)."""

    def __init__(self, n_in):
        self.ops = []
        self.count = 0
        self.inputs = [f"d[{i}]" for i in range(n_in)]

    def _t(self):
        self.count += 1
        return f"t{self.count}"

    def add(self, a, b):
        t = self._t()
        self.ops.append(("add", t, (a, b)))
        return t

    def sub(self, a, b):
        t = self._t()
        self.ops.append(("sub", t, (a, b)))
        return t

    def mul(self, a, c):
        t = self._t()
        self.ops.append(("mul", t, (a, c)))
        return t

    def fma(self, a, c, b):  # a * c + b, c a constant
        t = self._t()
        self.ops.append(("fma", t, (a, c, b)))
        return t

    def neg(self, a):
        t = self._t()
        self.ops.append(("neg", t, (a,)))
        return t

    def out(self, j, a):
        self.ops.append(("out", f"o[{j}]", (a,)))

    def flops(self):
        return sum(1 for k, _, _ in self.ops if k in ("add", "sub", "mul", "fma"))

    def to_cuda(self, name):
        lines = [f"__device__ __forceinline__ void {name}(const float* d, float* o) {{"]
        for kind, dst, args in self.ops:
            if kind == "add":
                lines.append(f"  const float {dst} = {args[0]} + {args[1]};")
            elif kind == "sub":
                lines.append(f"  const float {dst} = {args[0]} - {args[1]};")
            elif kind == "mul":
                lines.append(f"  const float {dst} = {args[0]} * {f32_hex(args[1])};")
            elif kind == "fma":
                lines.append(f"  const float {dst} = fmaf({args[0]}, {f32_hex(args[1])}, {args[2]});")
            elif kind == "neg":
                lines.append(f"  const float {dst} = -{args[0]};")
            elif kind == "out":
                lines.append(f"  {dst} = {args[0]};")
        lines.append("}")
        return "\n".join(lines) + "\n"

    def evaluate(self, d):
        """Run the program in numpy float32 on input rows d[..., n_in]; returns outputs."""
        import numpy as np

        env = {f"d[{i}]": np.asarray(d[..., i], dtype=np.float32) for i in range(d.shape[-1])}
        outs = {}
        for kind, dst, args in self.ops:
            if kind == "add":
                env[dst] = (env[args[0]] + env[args[1]]).astype(np.float32)
            elif kind == "sub":
                env[dst] = (env[args[0]] - env[args[1]]).astype(np.float32)
            elif kind == "mul":
                env[dst] = (env[args[0]] * np.float32(f32(args[1]))).astype(np.float32)
            elif kind == "fma":
                a = env[args[0]].astype(np.float64)
                env[dst] = (a * f32(args[1]) + env[args[2]].astype(np.float64)).astype(np.float32)
            elif kind == "neg":
                env[dst] = (-env[args[0]]).astype(np.float32)
            elif kind == "out":
                outs[int(dst[2:-1])] = env[args[0]]
        return np.stack([outs[j] for j in range(len(outs))], axis=-1)


def dct4_direct(M, scale=0.25):
    P = Program(M)
    for j in range(M):
        acc = None
        for n in range(M):
            c = scale * math.cos(math.pi * (2 * n + 1) * (2 * j + 1) / (4 * M))
            acc = P.mul(P.inputs[n], c) if acc is None else P.fma(P.inputs[n], c, acc)
        P.out(j, acc)
    return P


def _cmul_const(P, z, ang):
    """z * e^{i ang} for a constant angle; z = (re, im) names; trivial angles are free."""
    re, im = z
    c, s = math.cos(ang), math.sin(ang)
    k = round(ang / (math.pi / 2))
    if abs(ang - k * math.pi / 2) < 1e-15:
        k %= 4
        if k == 0:
            return (re, im)
        if k == 1:
            return (P.neg(im), re)
        if k == 2:
            return (P.neg(re), P.neg(im))
        return (im, P.neg(re))
    r = P.fma(re, c, P.mul(im, -s))  # re c - im s
    i = P.fma(re, s, P.mul(im, c))   # re s + im c
    return (r, i)


def _dft_pos(P, w):
    """sum_p w_p e^{+2 pi i p q / L} for q < L (radix-2, decimation in time)."""
    L = len(w)
    if L == 1:
        return list(w)
    E = _dft_pos(P, w[0::2])
    O = _dft_pos(P, w[1::2])
    out = [None] * L
    for q in range(L // 2):
        t = _cmul_const(P, O[q], 2 * math.pi * q / L)
        out[q] = (P.add(E[q][0], t[0]), P.add(E[q][1], t[1]))
        out[q + L // 2] = (P.sub(E[q][0], t[0]), P.sub(E[q][1], t[1]))
    return out


def dct4_fft(M, scale=0.25):
    P = Program(M)
    t = math.pi / (4 * M)
    H = M // 2
    w = []
    for p in range(H):
        a, b = P.inputs[2 * p], P.inputs[M - 1 - 2 * p]
        # c_p = a - i b, times e^{i 4 p t}
        w.append(_cmul_const(P, (a, P.neg(b)), 4 * p * t))
    W = _dft_pos(P, w)
    for q in range(H):
        ang = (4 * q + 1) * t
        c, s = scale * math.cos(ang), scale * math.sin(ang)
        re, im = W[q]
        P.out(2 * q, P.fma(re, c, P.mul(im, -s)))
        P.out(M - 1 - 2 * q, P.fma(re, s, P.mul(im, c)))
    return P


def blocks():
    return {16: dct4_fft(16), 8: dct4_fft(8), 4: dct4_direct(4), 2: dct4_direct(2)}


def emit(out):
    w = out.write
    w("// Generated by gen_dct_factors.py -- do not edit.\n")
    w("// demo_dct4_M(d, o): o[j] = sum_n cos(pi (2n+1)(2j+1) / (4M)) / 4 * d[n].\n")
    w("// The DCT-IV is symmetric, so the same block serves the forward and inverse transform.\n")
    w("// M = 16 and 8 go through a complex DFT of size M/2 (see the generator).\n")
    w("#pragma once\n\n")
    for M, P in blocks().items():
        w(f"// {P.flops()} flops\n")
        w(P.to_cuda(f"demo_dct4_{M}"))
        w("\n")
    w("// sqrt(1/32) = cos(pi/4) / 4: the DC factor and the 2-point stage factor.\n")
    w(f"#define DEMO_DCT_C0 ({f32_hex(0.25 * math.cos(math.pi / 4))})\n")


if __name__ == "__main__":
    emit(sys.stdout)
