"""An independent, brute-force formulation of the candidate-selection path,
used only to pin the oracle on tiny inputs.

It shares nothing with the oracle's arithmetic: the order is built from the
float's class, value and sign (not from a bit-flipped integer key), block and
column selection are decided by counting how many items are strictly better
(not by sorting), and the mask applies the pages' per-column keep rule
(prhub report on vLLM PR #56628, key source excerpts) column by column,
restricted to columns below the clamped end (vLLM PR #57459, Summary: columns
at or past end are left untouched).
"""
import math
import struct


def rank(bits: int):
    """A sortable tuple reproducing IEEE-754 totalOrder for one fp32 pattern."""
    neg = bits >> 31
    exp = (bits >> 23) & 0xFF
    frac = bits & 0x7FFFFF
    if exp == 0xFF and frac != 0:  # NaN: -NaN below everything, +NaN above
        return (0, -frac, 0) if neg else (2, frac, 0)
    f = struct.unpack("<f", struct.pack("<I", bits))[0]
    return (1, f, 0 if neg else 1)  # -0.0 just below +0.0


def better(ra, ia, rb, ib):
    """Item a strictly precedes item b: higher rank, or equal rank and lower index."""
    return ra > rb or (ra == rb and ia < ib)


NEG_INF_BITS = 0xFF800000


def path(row_bits, W, s, e, B, Kb, K):
    """Whole path on one row given as a list of W fp32 bit patterns.
    Returns (masked bit list, cand list of Kb+1, topk list of K)."""
    s = max(s, 0)
    ec = min(e, W)
    NB = -(-W // B)
    live = list(range(s, ec)) if ec > s else []
    # block scores: max by rank over each block's live columns, -inf elsewhere
    score = []
    for j in range(NB):
        cols = [c for c in live if (c - s) // B == j]
        if cols:
            best = max(cols, key=lambda c: rank(row_bits[c]))
            score.append(rank(row_bits[best]))
        else:
            score.append(rank(NEG_INF_BITS))
    # block top-k: j is chosen when fewer than Kb blocks are strictly better
    chosen = [j for j in range(NB)
              if sum(better(score[i], i, score[j], j) for i in range(NB)) < Kb]
    cand = chosen + [-1] * (Kb - len(chosen))
    pin = (e - 1 - s) // B if e > s else -1
    cand = cand + [pin]
    # flags with set semantics; packed column past the buffer -> edge
    flags, edge = set(), False
    for b in cand:
        if b < 0:
            continue
        if s + b * B < W:
            flags.add(b)
        else:
            edge = True
    masked = list(row_bits)
    for c in range(W):
        valid = s <= c < e and c < W
        keep = valid and (((c - s) // B) in flags or (c == W - 1 and edge))
        if c < ec and not keep:
            masked[c] = NEG_INF_BITS
    # row top-k: c is chosen when fewer than K live columns are strictly better
    picked = [c for c in live
              if sum(better(rank(masked[d]), d, rank(masked[c]), c) for d in live) < K]
    topk = picked + [-1] * (K - len(picked))
    return masked, cand, topk


def to_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


VALUE_POOL = [float("-inf"), -1.0, 0.0, 1.0, 2.0]
EXOTIC_POOL = [-0.0, 0.5, float("inf")]
NAN_BITS = [0x7FC00000, 0xFFC00000, 0x7F800001, 0xFFFFFFFF]


def isnan_bits(b):
    return ((b >> 23) & 0xFF) == 0xFF and (b & 0x7FFFFF) != 0


__all__ = ["rank", "better", "path", "to_bits", "VALUE_POOL", "EXOTIC_POOL", "NAN_BITS",
           "NEG_INF_BITS", "isnan_bits", "math"]
