"""CPU checks of the corner-case block generator used by the adversarial GPU
quantiser test: the blocks really sit on the rounding decisions, and the
oracle's answer on every one of them equals the exact rational recipe."""
import numpy as np
import pytest

import oracle as O
from quant_corners import E2M1_MIDS, GLOBAL_SCALES, adversarial_blocks, e4m3_grid
from test_oracle_pins import exact_block


def test_blocks_hit_the_decisions():
    """With g = 1 some element quotients sit exactly on an e2m1 midpoint, some
    amax / 6 exactly on an E4M3 midpoint, and scales saturate and underflow."""
    blocks = adversarial_blocks(1.0, seed=0)
    e4 = e4m3_grid()
    e4_mids = {(e4[i] + e4[i + 1]) / 2 for i in range(0x7E)}
    scale_ties = sum(1 for b in blocks if np.abs(b).max() / 6.0 in e4_mids)
    elem_ties, sat, zero_scale = 0, 0, 0
    for b in blocks:
        _, sf = O.quantize_block16(b, 1.0)
        s = O.e4m3_value(sf)
        sat += sf == 0x7E and np.abs(b).max() / 6.0 > 448
        zero_scale += sf == 0
        if s > 0:
            elem_ties += sum(1 for x in b if abs(x) / s in E2M1_MIDS)
    assert scale_ties >= 100 and elem_ties >= 200, (scale_ties, elem_ties)
    assert sat >= 4 and zero_scale >= 6, (sat, zero_scale)


@pytest.mark.parametrize("gname", list(GLOBAL_SCALES))
def test_oracle_on_corner_blocks_is_exact(gname):
    """The oracle's bytes on every corner block equal the exact rational
    evaluation of the recipe (Fractions): the GPU test compares against
    these bytes."""
    g = GLOBAL_SCALES[gname]
    for b in adversarial_blocks(g, seed=7):
        packed, sf = O.quantize_block16(b, g)
        want_p, want_sf = exact_block(b.tolist(), g)
        assert sf == want_sf
        assert packed.tolist() == want_p
