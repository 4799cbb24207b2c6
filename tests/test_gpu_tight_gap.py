"""Bit-exact selection at the boundary gap the parity bar names.

The selected-block sets must equal the oracle's on inputs whose fp64 score
gap at the top-k boundary is at least 1e-3.  Planted inputs have gaps far
larger than that, so these tests build inputs whose gap lies just above it:
after the seeded generator has drawn a unit, tests/qsa_check.tune_boundary
(oracle arithmetic only) rewrites the key of one unselected block so that the
oracle's gap falls in [1.1e-3, 1.9e-3].  Index score and top-k then run
through the C ABI, and every unit's selection is compared bit for bit.

Four input regimes, each over 2 requests x 4 layers (one context ragged):
  natural   no planted blocks; scores at their natural magnitude (~10-60)
  planted   512 planted blocks (scales x64), so both boundary blocks score
            in the hundreds and fp32 rounding is largest
  skewed    index-query elements log-uniform over [2^-12, 1] of the largest,
            so small elements reach the subnormal range of the query's e4m3
            pieces; no planting
  skewed_planted  both
The block-score error of every block is reported relative to
sum_h w_h |sc| sum_d |q k| (the scale of the fp32 rounding error).
"""
import numpy as np
import pytest
import torch

import sparse_attention_decode_qsa_gb300 as Q
from sparse_attention_decode_qsa_gb300 import synth, workloads
from tests import qsa_check as QC

pytestmark = pytest.mark.gpu

CTXS = [32768, 32766]
LAYERS = 4
REGIMES = {
    "natural": dict(plant=False, skew=False),
    "planted": dict(plant=True, skew=False),
    "skewed": dict(plant=False, skew=True),
    "skewed_planted": dict(plant=True, skew=True),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    Q.lib()


def _build(regime: str, seed: int):
    spec = REGIMES[regime]
    plant = (lambda l, r, n: synth.planted_uniform(n // 4, 512, synth.mix_seed(seed, 90, l, r))) \
        if spec["plant"] else (lambda l, r, n: [])
    wl = workloads.build(LAYERS, CTXS, [Q.KV_HBM] * len(CTXS), plant, staging_rows=0, seed=seed)
    c = wl.cache
    for l in range(LAYERS):
        for r, h in enumerate(wl.handles):
            u = wl.unit(l, r)
            if spec["skew"]:
                qs, ws = synth.index_query_skewed(synth.mix_seed(seed, 70, l, r))
                wl.q_idx[u], wl.w[u] = qs.cuda(), ws.cuda()
            n = wl.ctxs[r]
            codes = c.index_keys[h.index, l, :n].cpu().numpy()
            sbits = QC.bits16(c.index_scales[h.index, l, :n])
            cand, _ = synth.index_keys(4096, synth.mix_seed(seed, 71, l, r))
            codes2, sbits2, _, _ = QC.tune_boundary(
                codes, sbits, wl.q_idx[u].cpu().double().numpy(), wl.w[u].cpu().double().numpy(),
                wl.budget, cand.numpy())
            c.index_keys[h.index, l, :n] = torch.from_numpy(codes2).cuda()
            c.index_scales[h.index, l, :n] = torch.from_numpy(sbits2.view(np.float16)).cuda()
    torch.cuda.synchronize()
    return wl


@pytest.mark.parametrize("regime", list(REGIMES))
def test_selection_bit_exact_at_tight_boundary_gap(regime):
    wl = _build(regime, seed={"natural": 41, "planted": 42, "skewed": 43, "skewed_planted": 44}[regime])
    try:
        wl.step()
        torch.cuda.synchronize()
        st, det = wl.cache.poll_error()
        assert st == 0, f"device error word {st} detail {det}"
        worst, a_max, margin = 0.0, 0.0, float("inf")
        for l in range(LAYERS):
            for r in range(wl.n_req):
                ref = QC.oracle_unit(wl, l, r)
                lo, hi = QC.TIGHT_GAP
                assert lo <= ref["gap"] <= hi, (l, r, ref["gap"])
                QC.check_unit(wl, l, r, ref=ref)               # selection bit-exact, attention
                nb = ref["blk"].shape[0]
                g = wl.blk[wl.unit(l, r), :nb].cpu().double().numpy()
                rel = np.abs(g - ref["blk"]) / np.maximum(ref["mag_blk"], 1e-30)
                worst = max(worst, float(rel.max()))
                # the two blocks at the boundary and their error scale
                order = np.lexsort((np.arange(nb), -ref["blk"]))
                K = len(ref["sel"])
                a_b = float(ref["mag_blk"][order[K - 1]] + ref["mag_blk"][order[K]])
                a_max = max(a_max, a_b)
                margin = min(margin, ref["gap"] / a_b)
        # margin: the gap over the two boundary blocks' summed error scales;
        # the selection is safe while it exceeds the error ratio seen anywhere
        print(f"{regime}: worst block-score error / sum|w sc q k| = {worst:.3e}; "
              f"boundary sum|w sc q k| up to {a_max:.3e}; min gap / that = {margin:.3e}")
    finally:
        wl.close()
