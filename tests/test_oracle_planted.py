"""Each pin must bite: rebuild the oracle with one planted mistake (ORACLE_PLANT_* switch, on the
CPU) and check that at least one pin fails for it."""
import numpy as np
import pytest

import oracle as O
from qwen3_decoder_transformer_gb300 import TINY, synth
from tests import test_oracle_generation as TG
from tests import test_oracle_model as TM
from tests import test_oracle_pins as TP

PLANTS = ["ORACLE_PLANT_GAMMA_BEFORE_CAST", "ORACLE_PLANT_LINEAR_DROP_LAST_K", "ORACLE_PLANT_SILU_SIGN",
          "ORACLE_PLANT_ROPE_ADJACENT", "ORACLE_PLANT_ROPE_SIGN", "ORACLE_PLANT_SCALE_BY_DIM",
          "ORACLE_PLANT_GQA_MODULO", "ORACLE_PLANT_NO_QNORM", "ORACLE_PLANT_DROP_ATTN_RESIDUAL",
          "ORACLE_PLANT_MASK_CAUSAL_ONLY"]


def _run_all_checks():
    failed = []
    for chk in TP.ALL_CHECKS:
        try:
            chk()
        except AssertionError:
            failed.append(chk.__name__)
    w = synth.make_weights(TINY, 0)
    m = O.Model(TINY, synth.weights_to_numpy(w))
    try:
        TM.check_matches_f64_statement(w, m)
    except AssertionError:
        failed.append("check_matches_f64_statement")
    for chk in TG.ALL_CHECKS:
        try:
            chk(m)
        except AssertionError:
            failed.append(chk.__name__)
    return failed


@pytest.mark.parametrize("plant", PLANTS)
def test_planted_mistake_is_caught(plant, tmp_path):
    path = O.build(defines=[plant], out=str(tmp_path / f"{plant}.so"))
    O.use_library(path)
    try:
        failed = _run_all_checks()
    finally:
        O.use_library(None)
    assert failed, f"no pin caught {plant}"


def test_clean_build_passes_all():
    assert _run_all_checks() == []
