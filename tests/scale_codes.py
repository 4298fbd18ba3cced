"""Seeded UE5M3 scale-code inputs for the rebias tests: codes built bit by
bit from a binade and a mantissa (the UE5M3 layout: 5 exponent bits with bias
15, 3 mantissa bits, exponent field 0 subnormal), with a chosen binade span
per row."""
import numpy as np


def codes_with_span(rng, rows, nb, span):
    """UE5M3 codes whose non-zero values span exactly `span` binades per row
    (some zero codes and subnormal codes included)."""
    out = np.zeros((rows, nb), np.uint8)
    for r in range(rows):
        top = int(rng.integers(span - 16, 17))          # binade of the largest scale
        binades = rng.integers(top - span, top + 1, nb)
        binades[0], binades[1] = top, top - span
        for i, b in enumerate(binades):
            m = int(rng.integers(0, 7 if b == 16 else 8))      # 0xFF is not a value
            if b >= -14:
                out[r, i] = ((b + 15) << 3) | m
            else:                                        # subnormal: m/8 * 2^-14 with binade b
                sh = -14 - b                              # 1..3
                out[r, i] = (1 << (3 - sh)) | (m >> sh) if sh <= 3 else 0
        zero = rng.random(nb) < 0.1
        zero[:2] = False
        out[r, zero] = 0
    return out
