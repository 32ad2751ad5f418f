"""Self-test of the oracle pins: every planted mistake must fail at least one pin.

Each mutant is the oracle compiled with one MUT_* switch (a dropped Q4_K min term, flipped IQ1_M sign
polarity, swapped Q4_0 nibbles, a missing -8 offset, round-half-away quantization, swapped Q4_K
sc/m fields, per-32 instead of per-16 IQ1_M sub-scales, an off-by-one scale index, a wrong f16
exponent bias, a permuted operand in the integer dot, swapped W8A8 scales, the q6_K high bit pair read
from the wrong field, MoE output rows stored slot-major, the block scale d taken from a rounded reciprocal
of 127, the Q4_K min term added instead of subtracted, the block sum s accumulated as a float sum of d*q,
bf16 ties rounded up instead of to even).  The pin suite runs in a
subprocess against the mutant and must fail.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MUTANTS = ["MUT_ROUND_AWAY", "MUT_DROP_MIN", "MUT_SIGN_POLARITY", "MUT_NIBBLE_SWAP", "MUT_Q4_0_NO_OFFSET",
           "MUT_Q4K_FIELD_SWAP", "MUT_IQ1_SCALE_GROUP32", "MUT_SCALE_INDEX", "MUT_F16_BIAS",
           "MUT_PARTIAL_TRANSPOSE", "MUT_W8A8_SCALE_SWAP", "MUT_Q6K_HIGH_PAIR", "MUT_MOE_SLOT_MAJOR",
           "MUT_SCALE_RECIP", "MUT_MIN_SIGN", "MUT_SUM_ORDER", "MUT_BF16_HALF_UP"]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_planted_mistake(mutant, tmp_path):
    lib = oracle.build(out=str(tmp_path / f"lib_{mutant}.so"), defines=[mutant])
    env = dict(os.environ, MMQ_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"{mutant} passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
