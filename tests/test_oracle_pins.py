"""The oracle checked against what the pages and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


# Each planted mistake (see the ORC_MUTANT branches of the oracle source) must
# fail at least one pin; otherwise the pins would not guard that part.
MUTANTS = {
    1: "ql byte index masked to 5 bits",
    2: "qh byte index taken as r/4",
    3: "low and high ql nibbles swapped",
    4: "-32 centering dropped",
    5: "neighbouring sub-block's scale",
    6: "sub-block number used as the activation block",
    7: "super-block scale d dropped",
    8: "sign flip on odd sub-blocks",
    9: "da read with the [K/32][N] layout",
    10: "quantiser divides amax by 128",
    11: "quantiser truncates",
    12: "f16 subnormals flushed",
    13: "f16 exponent bias off by one",
    14: "sequential byte map (ql[e/2], qh[e/4])",
    15: "q4_K: min of sub-blocks 0-3 read from the scale bytes",
    16: "q4_K: top bits of scales 4-7 taken from the min bytes",
    17: "q4_K: low and high nibbles swapped",
    18: "q4_K: min term added instead of subtracted",
    19: "q4_K: neighbouring sub-block's activation scale",
}


@pytest.mark.parametrize("k", sorted(MUTANTS), ids=lambda k: f"m{k}")
def test_planted_mistake_is_caught(k):
    bad = oracle_pins.failing_pins(oracle.Oracle(mutant=k))
    assert bad, f"no pin catches planted mistake {k}: {MUTANTS[k]}"


def test_row_parallel_driver_matches(orc):
    """mmq_all (the large-shape driver over disjoint row ranges) gives exactly
    the single-threaded result, with ragged row splits."""
    from q6_int8_mmq_gb300 import synth
    M, K, N = 77, 768, 19
    raw = synth.q6k_raw_weights(0x51360B01, M, K)
    xq, da = orc.quantize(synth.activations(0x51360B02, N, K, outlier_frac=0.05))
    Y = orc.mmq(raw, M, K, xq, da)
    for t in (1, 3, 8, 77):
        assert np.array_equal(orc.mmq_all(raw, M, K, xq, da, threads=t), Y)
