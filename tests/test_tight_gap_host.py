"""CPU checks of the tight-gap input construction (tests/qsa_check.tune_boundary):
on seeded units of every regime the GPU tight-gap tests use, the oracle's
boundary gap lands in the window, the selected set is the one before tuning,
and only unselected blocks' keys change."""
import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from sparse_attention_decode_qsa_gb300 import synth
from tests import qsa_check as QC


@pytest.mark.parametrize("plant,skew", [(False, False), (True, False), (False, True), (True, True)])
def test_tune_boundary_places_the_gap_in_the_window(plant, skew):
    n, budget = 8190, 2048
    codes, scales = synth.index_keys(n, seed=11)
    if plant:
        synth.plant(scales, synth.planted_uniform(n // 4, 512, seed=12), n)
    q, w = synth.index_query_skewed(seed=13) if skew else synth.index_query(seed=13)
    sb = scales.contiguous().view(torch.int16).numpy().view(np.uint16)
    cand, _ = synth.index_keys(4096, seed=14)
    qd, wd = q.double().numpy(), w.double().numpy()
    blk0 = O.c4_block_scores(O.token_scores(codes.numpy(), sb, qd, wd))
    sel0 = O.select_blocks(blk0, budget)
    c2, s2, b, t = QC.tune_boundary(codes.numpy(), sb, qd, wd, budget, cand.numpy())
    blk = O.c4_block_scores(O.token_scores(c2, s2, qd, wd))
    assert QC.TIGHT_GAP[0] <= O.boundary_gap(blk, budget) <= QC.TIGHT_GAP[1]
    assert np.array_equal(O.select_blocks(blk, budget), sel0)
    assert b not in set(sel0.tolist()) and t == 4 * b
    changed = np.nonzero((c2 != codes.numpy()).any(axis=1) | (s2 != sb))[0]
    assert not np.isin(changed // 4, sel0).any()          # selected blocks untouched
