"""Planted mistakes: build deliberately wrong copies of the oracle and check
that the pins above catch every one of them (CPU only)."""
import os

import pytest

import oracle
from oracle import build as obuild

import test_oracle_formats as F
import test_oracle_gemv as G

PINS = [F.test_q4_0_golden_blocks, F.test_q4_k_golden_superblocks,
        F.test_q4_k_scale_packing_roundtrip_all_pairs,
        G.test_q4_0_roundtrip_representable_blocks, G.test_q4_0_integer_closed_form_exact,
        G.test_q4_k_roundtrip_representable_superblocks, G.test_q4_k_integer_closed_form_exact,
        lambda: G.test_q4_0_gemv_vs_numpy_matmul(2, 3, 64), F.test_af4_g64_golden_words]


@pytest.mark.parametrize("plant", ["ORACLE_PLANT_NIBBLE_SWAP", "ORACLE_PLANT_DROP_OFFSET",
                                   "ORACLE_PLANT_Q4K_HIGH_BITS", "ORACLE_PLANT_X_INDEX",
                                   "ORACLE_PLANT_AF4_HALVES", "ORACLE_PLANT_AF4_ROW_MAJOR"])
def test_planted_mistake_is_caught(plant, tmp_path):
    path = obuild.build(force=True, out=os.path.join(tmp_path, f"lib_{plant}.so"), defines=[plant])
    oracle.use_library(path)
    try:
        failed = []
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(getattr(pin, "__name__", "pin"))
        assert failed, f"no pin caught {plant}"
    finally:
        oracle.use_library(None)
