"""Writes tests/golden/tie_blocks.json: NVFP4 key blocks whose {4,6} search
ties exactly in binary32.

Method: BitDecoding-FP4 evaluation config (config.py), RECIPE
outlier_aware_key_quantization, adaptive block-scale search: a block keeps
the amax->4 scale only when its squared reconstruction error is strictly
lower than with amax->6, so a tie keeps amax->6.

The blocks are plain bf16 keys (no centering, no rotation) under one
per-tensor scale g.  A block is kept when

  * the oracle's two squared-error sums are equal (a tie, so it keeps 6), and
  * forming x - v*S with one rounding instead of two (a fused multiply-add)
    would make the amax->4 sum strictly lower, so the block flips.

Such blocks catch a kernel that contracts the reconstruction product into
the subtraction.  The search draws seeded normal keys and evaluates both
candidates with numpy binary32 arithmetic (one rounding per operation, the
oracle's order), then confirms every kept block with the oracle itself.

Run from the repository root:  python tests/golden/make_tie_blocks.py
"""
from __future__ import annotations

import json
import os
import sys
from fractions import Fraction

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "..", ".."))
import oracle  # noqa: E402

F32 = np.float32
G = float(F32(1.0) / F32(448.0))
SEED = 20261203
WANT = 48


def _tables():
    e2m1 = oracle.e2m1_value(np.arange(16)).astype(F32)
    e4m3 = oracle.e4m3_value(np.arange(256)).astype(F32)
    return e2m1, e4m3


def _sse_tree(w):
    """w[..., i] += w[..., i + h] for h = 8, 4, 2, 1 in binary32."""
    w = w.copy()
    h = 8
    while h >= 1:
        w[..., :h] = (w[..., :h] + w[..., h:2 * h]).astype(F32)
        h //= 2
    return w[..., 0]


def _candidate(x, m, g, e2m1, e4m3):
    """Squared-error sum of every block of x [N][16] under amax -> m."""
    amax = np.abs(x).max(axis=1).astype(F32)
    t = F32(m) * F32(g)
    s = (amax / t).astype(F32)
    b = oracle.e4m3_encode(s)
    S = (e4m3[b] * F32(g)).astype(F32)
    with np.errstate(divide="ignore"):
        inv = (F32(1.0) / S).astype(F32)
    zero = (S == 0) | np.isinf(inv)
    q = (x * inv[:, None]).astype(F32)
    codes = oracle.e2m1_encode(q).reshape(x.shape)
    xh = (e2m1[codes] * S[:, None]).astype(F32)
    xh[zero] = 0
    e = (x - xh).astype(F32)
    return _sse_tree((e * e).astype(F32)), e2m1[codes], S


def _rn32(fr: Fraction) -> float:
    """Round an exact rational to the nearest binary32, ties to even."""
    f = F32(float(fr))
    lo, hi = np.nextafter(f, F32(-np.inf)), np.nextafter(f, F32(np.inf))
    best = min((lo, f, hi), key=lambda c: (abs(Fraction(float(c)) - fr),
                                           int(np.array(c, F32).view(np.uint32)) & 1))
    return float(best)


def fused_sse(x, val, S) -> float:
    """The sum when each error x - v*S is rounded once (a fused multiply-add)."""
    e = np.array([_rn32(Fraction(float(xi)) - Fraction(float(vi)) * Fraction(float(S)))
                  for xi, vi in zip(x, val)], F32)
    return float(_sse_tree((e * e).astype(F32)[None, :])[0])


def main():
    e2m1, e4m3 = _tables()
    rng = np.random.default_rng(SEED)
    kept = []
    tried = 0
    while len(kept) < WANT and tried < 400:
        tried += 1
        raw = rng.standard_normal((1 << 19, 16)).astype(F32)
        bf = (raw.view(np.uint32) + 0x7FFF + ((raw.view(np.uint32) >> 16) & 1)) >> 16
        x = (bf.astype(np.uint32) << 16).view(F32)
        e6, v6, S6 = _candidate(x, 6, G, e2m1, e4m3)
        e4, v4, S4 = _candidate(x, 4, G, e2m1, e4m3)
        for i in np.nonzero(e4 == e6)[0]:
            f6 = fused_sse(x[i], v6[i], S6[i])
            f4 = fused_sse(x[i], v4[i], S4[i])
            if not f4 < f6:
                continue
            m, _, _, _, oe4, oe6 = oracle.four_six_block(x[i], G)
            if m == 6 and oe4 == oe6:
                kept.append(bf[i].astype(np.uint16).tolist())
    out = {
        "source": "BitDecoding-FP4 evaluation config (config.py), RECIPE outlier_aware_key_quantization, "
                  "adaptive block-scale search: amax->4 only when strictly better, so ties keep amax->6",
        "g": G,
        "seed": SEED,
        "blocks_bf16": kept,
    }
    path = os.path.join(os.path.dirname(__file__), "tie_blocks.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(f"{len(kept)} tie blocks from {tried} batches of {1 << 19} -> {path}")


if __name__ == "__main__":
    main()
