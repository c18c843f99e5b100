"""Corner-case 16-element blocks for the NVFP4 quantiser (test input
generator; it draws inputs and reads the E4M3 value grid from the oracle,
and computes none of the quantisation itself).

The recipe (scale byte E4M3_RNE_satfinite(amax / (6 g)), element codes
e2m1_RNE_satfinite(x / (s g)), ties to the even code, zero codes keeping the
sign of x) has exactly one correct byte stream, so the corners of its
rounding decisions are what a bit-exact test must reach:

  * element ties x = midpoint * s * g at each of the seven e2m1 midpoints,
    both signs (exact in bf16 when g is a power of two; the nearest bf16 and
    its neighbours otherwise);
  * amax on, and one bf16 ulp either side of, 6 g times every E4M3 midpoint
    (scale ties and near-ties, subnormal scales included);
  * saturation: amax / (6 g) at and above 448, elements beyond 6 s g;
  * the underflow edge of the scale (amax / (6 g) around 2^-10);
  * all-zero, all-negative-zero and mixed-sign-zero blocks.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

GLOBAL_SCALES = {
    "2^-60": 2.0 ** -60,
    "1/2688": float(np.float32(1.0 / 2688.0)),
    "1": 1.0,
    "2^60": 2.0 ** 60,
}
E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def bf16(x) -> np.ndarray:
    """Round to bf16 (RNE) and return the float64 values."""
    return torch.tensor(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def bf16_step(x: float, n: int) -> float:
    """The bf16 value n bit patterns away from the bf16 value x (for x > 0:
    n ulps up or down)."""
    bits = np.array([x], np.float64).astype(np.float32).view(np.uint32)[0] >> 16
    bits = np.array([(int(bits) + n) & 0xFFFF], np.uint32) << 16
    return float(bits.view(np.float32)[0])


def fill_below(rng, amax: float, n: int) -> np.ndarray:
    """n random bf16 values with |x| <= amax, random signs."""
    x = bf16(rng.uniform(-1.0, 1.0, n) * amax)
    return np.clip(x, -amax, amax)


def e4m3_grid():
    return [O.e4m3_value(c) for c in range(0x7F)]   # 0 .. 448


def adversarial_blocks(g: float, seed: int) -> np.ndarray:
    """[n, 16] float64 blocks; every value is exactly a bf16 value."""
    rng = np.random.default_rng(seed)
    e4 = e4m3_grid()
    e4_mids = [(e4[i] + e4[i + 1]) / 2 for i in range(0x7E)]
    blocks = []

    # -- element ties at every e2m1 midpoint, both signs ------------------
    for sc in list(range(1, 0x7F, 5)) + [0x7E]:
        s = e4[sc]
        amax = float(bf16(6.0 * s * g))
        vals = [amax]
        for m in E2M1_MIDS:
            t = float(bf16(m * s * g))
            vals += [t, -t]
        vals.append(-amax)
        blk = np.array(vals[:16])
        rng.shuffle(blk)
        blocks.append(blk)
        # the bf16 neighbours of every midpoint (near-ties on both sides)
        for d in (-1, 1):
            vals = [amax]
            for m in E2M1_MIDS:
                t = min(bf16_step(float(bf16(m * s * g)), d), amax)
                vals += [t, -t]
            vals.append(float(bf16(s * g)))
            blk = np.array(vals[:16])
            rng.shuffle(blk)
            blocks.append(blk)

    # -- scale ties: amax = 6 g m at every E4M3 midpoint, +-1 bf16 ulp ------
    for m in e4_mids:
        a0 = float(bf16(6.0 * g * m))
        for d in (-1, 0, 1):
            amax = bf16_step(a0, d) if d else a0
            if amax <= 0:
                continue
            rest = fill_below(rng, amax, 15)
            blk = np.concatenate([[amax if rng.random() < 0.5 else -amax], rest])
            rng.shuffle(blk)
            blocks.append(blk)

    # -- saturation: amax / (6 g) at and above 448 -------------------------
    for t in (448.0, 450.0, 463.0, 464.0, 465.0, 480.0, 1000.0, 1.0e5):
        amax = float(bf16(6.0 * g * t))
        over = [float(bf16(6.0 * 448.0 * g * f)) for f in (1.0, 1.02, 1.04, 1.1, 1.5)]
        over = [v for v in over if v <= amax]
        blk = np.concatenate([[amax, -amax], over, [-v for v in over],
                              fill_below(rng, amax, 14 - 2 * len(over))])
        rng.shuffle(blk)
        blocks.append(blk)

    # -- the scale's underflow edge (2^-9 is the smallest E4M3 subnormal) ----
    for t in (2.0 ** -12, 2.0 ** -11, 0.99 * 2.0 ** -10, 2.0 ** -10, 1.01 * 2.0 ** -10,
              1.5 * 2.0 ** -10, 2.0 ** -9, 3.0 * 2.0 ** -10, 2.0 ** -8, 2.0 ** -7):
        amax = float(bf16(6.0 * g * t))
        blk = np.concatenate([[-amax], fill_below(rng, amax, 15)])
        rng.shuffle(blk)
        blocks.append(blk)

    # -- zeros ----------------------------------------------------------------
    blocks.append(np.zeros(16))
    blocks.append(-np.zeros(16))
    mixed = np.zeros(16)
    mixed[::2] = -0.0
    blocks.append(mixed)
    tiny = -np.zeros(16)
    tiny[5] = float(bf16(6.0 * g * 2.0 ** -8))
    blocks.append(tiny)

    # -- ordinary blocks over many magnitudes --------------------------------
    for _ in range(64):
        scale = 10.0 ** rng.uniform(-3, 3) * g
        blocks.append(bf16(rng.standard_normal(16) * scale))

    out = np.stack(blocks)
    assert np.all(np.isfinite(out))
    assert np.array_equal(out, bf16(out)), "every block value must be a bf16 value"
    return out
