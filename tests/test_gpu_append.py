"""Parity of the producer side (qsa_request_advance + qsa_append_token, through
the C ABI) with the fp64 oracle.

Bars: stored index-key codes and fp16 scales bit-exact with
oracle.quantize_index_key of the same fp32 keys; slot tables equal to the
oracle's layouts after the appends; KV rows byte-exact where the placement
puts them; and a decode step over the grown context meets the usual bars
(selection bit-exact on a >= 1e-3 boundary gap, attention within 2e-3).
The oracle is fed only generator bytes and the test's own keys and rows,
never what the kernels wrote.
"""
import numpy as np
import pytest
import torch

import sparse_attention_decode_qsa_gb300 as Q
from oracle import qsa_oracle as O
from sparse_attention_decode_qsa_gb300 import synth, workloads
from tests import qsa_check as QC

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    Q.lib()


def _clean(wl):
    st, det = wl.cache.poll_error()
    assert st == 0, f"device error word {st} detail {det}"


def _edge_keys(seed, m):
    """m index keys (fp32 [m][64]) of every magnitude plus the quantiser's
    edge cases: zero key, signed zeros, exact E4M3 midpoints, saturating
    scales, values far below the scale."""
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(m, 64, generator=g)
    k *= torch.exp2(torch.randint(-40, 40, (m, 1), generator=g).float())
    k[0] = 0.0
    k[1] = -0.0
    k[1, 7] = 1e-3
    k[2] = torch.tensor([448.0, 1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, -2.0 ** -10,
                         2.0 ** -9] + [0.0] * 56)
    k[3] = 3.0e7 * torch.randn(64, generator=g)
    k[4] = 1e-30 * torch.randn(64, generator=g)
    k[5, :] = 1.0
    k[5, 0] = 1e-12
    return k


def test_append_quantizes_index_keys_like_the_oracle():
    R, n0, G = 16, 40, 24
    wl = workloads.build(1, [n0] * R, [Q.KV_HBM] * R, lambda l, r, n: [], staging_rows=8,
                         seed=3, grow=G)
    try:
        c, hs, dev = wl.cache, wl.handles, wl.cache.pool.device
        keys = [_edge_keys(100 + s, R) for s in range(G)]
        rows = [synth.kv_rows(R, 200 + s) for s in range(G)]
        for s in range(G):
            for h in hs:
                c.advance(h)
            c.append_token(hs, 0, 1, keys[s].to(dev), rows[s].to(dev))
        torch.cuda.synchronize()
        _clean(wl)
        for r, h in enumerate(hs):
            info = c.request_info(h)
            assert info.ctx_len == n0 + G and info.max_ctx == n0 + G
            codes = c.index_keys[h.index, 0, n0:n0 + G].cpu().numpy()
            scales = QC.bits16(c.index_scales[h.index, 0, n0:n0 + G])
            for s in range(G):
                ref_codes, ref_bits = O.quantize_index_key(keys[s][r].numpy())
                assert int(scales[s]) == ref_bits, (r, s)
                assert np.array_equal(codes[s], ref_codes), (r, s)
            slots = c.slot_table[h.index, 0, :n0 + G].cpu().numpy()
            assert np.array_equal(slots, O.resident_slot_row(n0 + G, 0, info.hbm_row_base,
                                                             info.layer_rows))
            got = c.pool[info.hbm_row_base + n0:info.hbm_row_base + n0 + G].cpu()
            assert torch.equal(got, torch.stack([rows[s][r] for s in range(G)]))
    finally:
        wl.close()


def test_append_host_only_request():
    n0, G = 1000, 9
    wl = workloads.build(2, [n0], [Q.KV_HOST], lambda l, r, n: [], staging_rows=8, seed=4, grow=G)
    try:
        c, h, dev = wl.cache, wl.handles[0], wl.cache.pool.device
        keys = [torch.randn(2, 64, generator=torch.Generator().manual_seed(s)) for s in range(G)]
        rows = [synth.kv_rows(2, 300 + s) for s in range(G)]
        stats0 = c.stats()
        for s in range(G):
            c.advance(h)
            for l in range(2):
                c.append_token([h], l, 1, keys[s][l:l + 1].to(dev), rows[s][l:l + 1].to(dev))
        torch.cuda.synchronize()
        _clean(wl)
        assert c.stats() == stats0                      # no HBM rows leased by appending
        for l in range(2):
            assert np.all(c.slot_table[h.index, l, :n0 + G].cpu().numpy() == -1)
            for s in range(G):
                assert torch.equal(wl.host[0][l, n0 + s], rows[s][l])
                codes, bits = O.quantize_index_key(keys[s][l].numpy())
                assert np.array_equal(c.index_keys[h.index, l, n0 + s].cpu().numpy(), codes)
                assert int(QC.bits16(c.index_scales[h.index, l, n0 + s:n0 + s + 1])[0]) == bits
    finally:
        wl.close()


@pytest.mark.parametrize("hot_rows", [0, 2048])
def test_append_ring_request_then_decode_step_matches_the_oracle(hot_rows):
    """Two offloaded requests with a 512-token HBM tail ring grow by 260
    tokens at both layers (every append hands a ring row over and makes the
    token it held cold); the slot tables, ring rows and host history follow
    the oracle's layouts, and a decode step over the grown context matches
    the oracle run on the generator's bytes plus the test's own keys and rows
    (also with a hot cache, whose fetch moves the selected cold rows into
    HBM before attention)."""
    L, R, n0, G, ring = 2, 2, 3000, 260, 512
    seed = 21
    wl = workloads.build(L, [n0] * R, [Q.KV_HOST_RING] * R,
                         lambda l, r, n: synth.planted_hot_cold(n // 4, 512, ring // 4,
                                                                synth.mix_seed(seed, 90, l, r)),
                         ring=ring, staging_rows=64, seed=seed, grow=G, hot_rows=hot_rows)
    try:
        c, hs, dev = wl.cache, wl.handles, wl.cache.pool.device
        n = n0 + G
        gen_codes = [[c.index_keys[h.index, l, :n0].cpu().numpy() for h in hs] for l in range(L)]
        gen_scales = [[QC.bits16(c.index_scales[h.index, l, :n0]) for h in hs] for l in range(L)]
        all_rows = [[wl.host[r][l, :n0].clone() for r in range(R)] for l in range(L)]
        new_keys = [[[] for _ in range(R)] for _ in range(L)]
        g = torch.Generator().manual_seed(seed)
        for s in range(G):
            for h in hs:
                c.advance(h)
            for l in range(L):
                k = torch.randn(R, 64, generator=g)
                rows = synth.kv_rows(R, synth.mix_seed(seed, 7, s, l))
                c.append_token(hs, l, 1, k.to(dev), rows.to(dev))
                for r in range(R):
                    new_keys[l][r].append(k[r].numpy())
                    all_rows[l][r] = torch.cat([all_rows[l][r], rows[r:r + 1]])
        torch.cuda.synchronize()
        _clean(wl)
        codes_all, scales_all = {}, {}
        for l in range(L):
            for r, h in enumerate(hs):
                info = c.request_info(h)
                q = [O.quantize_index_key(k) for k in new_keys[l][r]]
                codes_all[l, r] = np.concatenate([gen_codes[l][r], np.stack([x[0] for x in q])])
                scales_all[l, r] = np.concatenate([gen_scales[l][r],
                                                   np.array([x[1] for x in q], dtype=np.uint16)])
                assert np.array_equal(c.index_keys[h.index, l, :n].cpu().numpy(), codes_all[l, r])
                assert np.array_equal(QC.bits16(c.index_scales[h.index, l, :n]), scales_all[l, r])
                want_slots = O.ring_slot_row(n, l, info.hbm_row_base, ring)
                assert np.array_equal(c.slot_table[h.index, l, :n].cpu().numpy(), want_slots)
                assert torch.equal(wl.host[r][l, n0:n], all_rows[l][r][n0:n])
                hot = np.arange(n - ring, n)
                got = c.pool[torch.as_tensor(want_slots[hot], dtype=torch.int64, device=dev)].cpu()
                assert torch.equal(got, all_rows[l][r][hot])
        # decode step over the grown context
        for r in range(R):
            wl.ctxs[r] = n
        wl.step()
        torch.cuda.synchronize()
        _clean(wl)
        for l in range(L):
            for r, h in enumerate(hs):
                info = c.request_info(h)
                u = wl.unit(l, r)
                q_idx, w = wl.q_idx[u].double().cpu().numpy(), wl.w[u].double().cpu().numpy()
                S = O.token_scores(codes_all[l, r], scales_all[l, r], q_idx, w)
                blk = O.c4_block_scores(S)
                assert O.boundary_gap(blk, wl.budget) >= QC.MIN_GAP
                sel = O.select_blocks(blk, wl.budget)
                toks = O.selected_tokens(sel, n)
                slot = O.ring_slot_row(n, l, info.hbm_row_base, ring)
                rows_np = all_rows[l][r].numpy()
                holder = {int(slot[t]): t for t in range(n) if slot[t] >= 0}
                pool = {s_: rows_np[t] for s_, t in holder.items()}
                got_rows = O.gather_rows(toks, slot, pool, rows_np)
                out, lse = O.decode_attention(QC.bits16(wl.q[u]), got_rows, wl.softmax_scale)
                k = int(wl.nsel[u].item())
                assert np.array_equal(wl.sel[u, :k].cpu().numpy(), sel), (l, r)
                absk = np.abs(O.decode_e4m3(codes_all[l, r])) * \
                    np.abs(O.decode_fp16(scales_all[l, r]))[:, None]
                mag_blk = O.c4_block_scores((absk @ np.abs(q_idx).T) @ np.abs(w))
                err = np.abs(wl.blk[u, :(n + 3) // 4].double().cpu().numpy() - blk)
                assert np.all(err <= QC.SCORE_REL_TOL * mag_blk + 1e-30)
                assert np.abs(wl.out[u].double().cpu().numpy() - out).max() <= QC.ATTN_TOL
                assert np.abs(wl.lse[u].double().cpu().numpy() - lse).max() <= QC.ATTN_TOL
    finally:
        wl.close()


def test_append_rejects_stale_handles_and_bad_buffers():
    wl = workloads.build(1, [64], [Q.KV_HBM], lambda l, r, n: [], staging_rows=8, seed=5, grow=4)
    try:
        c, h, dev = wl.cache, wl.handles[0], wl.cache.pool.device
        k = torch.zeros(1, 64, device=dev)
        rows = torch.zeros(1, 2048, dtype=torch.uint8, device=dev)
        c.advance(h)
        with pytest.raises(Q.QsaError) as e:
            c.append_token([h], 0, 1, k[:, 1:], rows)      # 4-byte offset: not 16-byte aligned
        assert e.value.status == Q.ERR_INVALID_ARG
        c.request_end(h)
        with pytest.raises(Q.QsaError) as e:
            c.append_token([h], 0, 1, k, rows)
        assert e.value.status == Q.ERR_STALE_HANDLE
        wl.handles = []
    finally:
        wl.close()
