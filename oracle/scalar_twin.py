"""Pure-Python scalar twin of the C oracle, for tiny shapes only.

Test infrastructure: it restates the same definitions (pack into bitmask +
fixed-step values, unpack, fp64 product) with Python integers and floats so
that the C oracle can be cross-checked against an independent implementation.
binary16 decoding here uses ``struct``'s ``'e'`` format, not the C decoder.

Source: "SparseDecoding: Decoding-Aware Pruning for Accurate and Efficient LLM
Inference", Abstract -- N:M sparse matrix-vector kernel with bitmask indexing
and fixed-step traversal.
"""
from __future__ import annotations

import struct


def h2f(bits: int) -> float:
    return struct.unpack("<e", struct.pack("<H", bits & 0xFFFF))[0]


def pack(W, mask, N, M):
    """W, mask: lists of rows (ints = fp16 bit patterns, 0/1).  Returns
    (values rows, mask-word rows, bad-group count)."""
    values, words, bad = [], [], 0
    for wrow, mrow in zip(W, mask):
        K = len(wrow)
        vrow = []
        mw = [0] * ((K + 31) // 32)
        for g in range(K // M):
            kept = [k for k in range(g * M, g * M + M) if mrow[k]]
            for k in kept:
                mw[k // 32] |= 1 << (k % 32)
            if len(kept) != N:
                bad += 1
            take = [wrow[k] for k in kept[:N]]
            vrow.extend(take + [0] * (N - len(take)))
        values.append(vrow)
        words.append(mw)
    return values, words, bad


def unpack(values, words, K, N, M):
    out = []
    for vrow, mw in zip(values, words):
        row = [0] * K
        for g in range(K // M):
            j = 0
            for k in range(g * M, g * M + M):
                if (mw[k // 32] >> (k % 32)) & 1 and j < N:
                    row[k] = vrow[g * N + j]
                    j += 1
        out.append(row)
    return out


def spmv(values, words, K, N, M, xs):
    """xs: list of vectors (fp16 bit patterns).  Returns (y, s) as
    [batch][rows] lists of floats."""
    ys, ss = [], []
    for x in xs:
        yb, sb = [], []
        for vrow, mw in zip(values, words):
            acc = 0.0
            sab = 0.0
            v = 0
            for g in range(K // M):
                j = 0
                for k in range(g * M, g * M + M):
                    if (mw[k // 32] >> (k % 32)) & 1 and j < N:
                        p = h2f(vrow[v + j]) * h2f(x[k])
                        acc += p
                        sab += abs(p)
                        j += 1
                v += N
            yb.append(acc)
            sb.append(sab)
        ys.append(yb)
        ss.append(sb)
    return ys, ss
