"""Pure-Python brute force of decode attention over a logical token history.

Written independently of the C oracle (no shared code), with Python floats
(IEEE double) and math.exp. It works on the *logical* history -- a list of
(k, v) rows per sequence -- so it uses no cache layout at all. Only for tiny
inputs: it is slow on purpose.
"""
import math
import struct


def bf16_bits_to_float(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def attend(q_bits, hist_k_bits, hist_v_bits, L, sink, window, scale, G):
    """Output rows for one sequence.

    q_bits: [Hq][D] ints; hist_*_bits: [T][Hkv][D] ints (T >= L, token L-1 is
    the new one); sink: list of Hq floats or None; window: 0 = full.
    Returns [Hq][D] floats.
    """
    Hq = len(q_bits)
    D = len(q_bits[0])
    out = [[0.0] * D for _ in range(Hq)]
    if L <= 0:
        return out
    lo = max(0, L - window) if window > 0 else 0
    for h in range(Hq):
        g = h // G
        q = [bf16_bits_to_float(x) for x in q_bits[h]]
        scores = []
        for j in range(lo, L):
            k = [bf16_bits_to_float(x) for x in hist_k_bits[j][g]]
            scores.append(scale * sum(a * b for a, b in zip(q, k)))
        sigma = -math.inf if sink is None else float(sink[h])
        m = max([sigma] + scores)
        den = 0.0 if sigma == -math.inf else math.exp(sigma - m)
        num = [0.0] * D
        for idx, j in enumerate(range(lo, L)):
            w = math.exp(scores[idx] - m)
            den += w
            v = [bf16_bits_to_float(x) for x in hist_v_bits[j][g]]
            for d in range(D):
                num[d] += w * v[d]
        out[h] = [x / den for x in num]
    return out
