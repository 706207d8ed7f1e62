"""IEEE special-value inputs for the reduce-scatter and placement tests.

Each case is a column of N bf16 values, one per rank, chosen so that a
plausible deviation from the reading taken for the reduce-scatter (fp32 sum
in ascending rank order from +0.0f, every add and the final multiply rounded
to nearest even, subnormals kept, NaN and infinity per IEEE 754) changes the
result: flushing subnormals to zero, starting the sum from -0.0f, summing in
another order (pairwise, reversed), or fusing the scale into the last add.

This module holds inputs and the closed-form results the oracle is pinned
against; it contains none of the oracle's or the kernels' arithmetic.
"""
from __future__ import annotations

import math

import numpy as np

PZERO, NZERO = 0x0000, 0x8000
ONE, NONE = 0x3F80, 0xBF80
SUB_MIN, NSUB_MIN = 0x0001, 0x8001     # +-2^-133, the smallest bf16 subnormal
SUB_MAX = 0x007F                        # 127 * 2^-133, the largest bf16 subnormal
MIN_NORMAL = 0x0080                     # 2^-126
MAX, NMAX = 0x7F7F, 0xFF7F              # +-(2 - 2^-7) * 2^127, the largest finite bf16
PINF, NINF = 0x7F80, 0xFF80
QNAN, QNAN_PAYLOAD, NQNAN_PAYLOAD = 0x7FC0, 0x7FC5, 0xFFD3
SNAN, NSNAN = 0x7F81, 0xFFA1            # quiet bit clear
BIG, NBIG = 0x7180, 0xF180              # +-2^100: BIG + 1 rounds back to BIG


def _col(n, head, fill=PZERO):
    """The first len(head) ranks hold `head`, the rest `fill` (N = 1 keeps head[0])."""
    return [head[k] if k < len(head) else fill for k in range(n)]


def cases(n: int):
    """(name, values[N]) for N ranks."""
    mid, last = n // 2, n - 1
    nan_at = lambda k, bits: [bits if j == k else ONE for j in range(n)]  # noqa: E731
    return [
        ("all_neg_zero", [NZERO] * n),
        ("neg_zero_then_pos_zero", _col(n, [NZERO], PZERO)),
        ("subnormal_min_sum", [SUB_MIN] * n),
        ("subnormal_cancel", _col(n, [SUB_MIN, NSUB_MIN])),
        ("subnormal_to_normal", [SUB_MAX] * n),
        ("min_normal", _col(n, [MIN_NORMAL])),
        ("pos_inf_last", [ONE] * last + [PINF]),
        ("neg_inf_first", _col(n, [NINF], NMAX)),
        ("inf_minus_inf", _col(n, [PINF, NINF])),
        ("qnan_payload_mid", nan_at(mid, QNAN_PAYLOAD)),
        ("neg_qnan_payload_first", nan_at(0, NQNAN_PAYLOAD)),
        ("snan_last", nan_at(last, SNAN)),
        ("nan_then_inf", _col(n, [NSNAN, PINF])),
        ("overflow", [MAX] * n),
        ("neg_overflow", [NMAX] * n),
        ("overflow_then_back", _col(n, [MAX, MAX, NMAX, NMAX])),
        ("max_alternating", _col(n, [MAX, NMAX, MAX, NMAX])),
        ("cancel_big_one_first", _col(n, [BIG, ONE, NBIG])),
        ("cancel_big_pair_first", _col(n, [BIG, NBIG, ONE])),
        ("ones", [ONE] * n),
    ]


def expected(name: str, n: int, scale: float):
    """Closed-form result of a case for a power-of-two `scale` (so the final
    multiply is exact unless it underflows), as float64; math.nan for NaN.
    Derived by hand from the sequential fp32 sum, not by running it."""
    assert scale > 0 and math.frexp(scale)[0] == 0.5, "power-of-two scale only"
    fmax = (2 - 2 ** -23) * 2.0 ** 127
    bmax = (2 - 2 ** -7) * 2.0 ** 127
    s = {
        "all_neg_zero": 0.0,             # +0 + (-0) = +0 under round to nearest
        "neg_zero_then_pos_zero": 0.0,
        "subnormal_min_sum": n * 2.0 ** -133,
        "subnormal_cancel": 2.0 ** -133 if n == 1 else 0.0,
        "subnormal_to_normal": n * 127 * 2.0 ** -133,
        "min_normal": 2.0 ** -126,
        "pos_inf_last": math.inf,
        "neg_inf_first": -math.inf,
        "inf_minus_inf": math.inf if n == 1 else math.nan,
        "qnan_payload_mid": math.nan,
        "neg_qnan_payload_first": math.nan,
        "snan_last": math.nan,
        "nan_then_inf": math.nan,
        # MAX + MAX is 2^128 - 2^121, past the rounding boundary (2 - 2^-24) * 2^127
        "overflow": bmax if n == 1 else math.inf,
        "neg_overflow": -bmax if n == 1 else -math.inf,
        # Inf stays Inf: a pairwise sum would give Inf + -Inf = NaN
        "overflow_then_back": {1: bmax}.get(n, math.inf),
        # MAX - MAX = 0 exactly at every even step
        "max_alternating": bmax if n in (1, 3) else 0.0,
        # 2^100 + 1 rounds to 2^100, so the one is lost; in the other order it survives
        "cancel_big_one_first": {1: 2.0 ** 100, 2: 2.0 ** 100}.get(n, 0.0),
        "cancel_big_pair_first": {1: 2.0 ** 100}.get(n, 0.0 if n == 2 else 1.0),
        "ones": float(n),
    }[name]
    if math.isnan(s) or math.isinf(s):
        return s
    assert abs(s) <= fmax
    v = s * scale
    # the product is exact unless it falls below 2^-126 (then it rounds to a
    # multiple of 2^-149; every case here lands on one exactly or on zero)
    if v != 0 and abs(v) < 2.0 ** -126:
        q = v / 2.0 ** -149
        assert q == int(q), (name, n, scale)
    return v


def shapes(n: int):
    """Parameters that put the cases into every kernel path: 16-byte vector
    runs, < 8-element tails, 1-D tensors, a tensor with fewer rows than ranks
    (empty ranks, padding tiles) and rows that do not divide by N."""
    return [(3 * n + 1, 24), (2 * n + 3, 8), (5 * n + 2,), (max(1, n - 1), 16), (4 * n, 40), ()]


def grads(n: int, shps, seed: int = 0):
    """grads[k][p]: rank k's bf16 bits of parameter p.  Element e of p holds
    case (e + 3p) mod C; one case in eight is replaced by random finite
    values so the special values sit among ordinary ones."""
    rng = np.random.default_rng(seed + n)
    cs = [np.asarray(v, dtype=np.uint16) for _, v in cases(n)]
    out = [[None] * len(shps) for _ in range(n)]
    for p, s in enumerate(shps):
        m = int(np.prod(s)) if len(s) else 1
        idx = (np.arange(m) + 3 * p) % len(cs)
        vals = np.stack([cs[i] for i in idx], axis=1) if m else np.zeros((n, 0), np.uint16)
        noise = rng.integers(0, 8, size=m) == 0
        rnd = (rng.standard_normal((n, m)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        vals = np.where(noise[None, :], rnd, vals)
        for k in range(n):
            out[k][p] = np.ascontiguousarray(vals[k])
    return out


def random_bits(rng, m: int, avoid: int):
    """m uniformly random 16-bit patterns (every NaN payload, subnormal and
    infinity included) with `avoid` (a sentinel) replaced."""
    b = rng.integers(0, 1 << 16, size=m, dtype=np.uint32).astype(np.uint16)
    b[b == avoid] = avoid ^ 0x0002
    return b
