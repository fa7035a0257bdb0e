"""Edge cases and failure handling of the CUDA path, each against the oracle.

* Top-k with massive ties: tens of thousands of entries with one and the same score, alone and
  below a few larger scores; the selection must take the lowest indices among the tied entries.
* A block table that maps a sequence's page to nothing (host-side corruption): the device
  status word reports LCS_ERR_DEVICE_GUARD, and every other sequence's top-k and attention
  output still equal the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import DEV, assert_status_ok, dev_status, entry_rows_of, u8, workspace
from test_gpu_stages import _attend_case, _index_case

lcsa = pytest.importorskip("long_context_sparse_24_b300")

pytestmark = pytest.mark.gpu


def _topk(batch, cache, q_fp4, q_sc, hw, heads, m, k, st=None, flags=0):
    T = batch.total_new
    out_idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    out_cnt = torch.full((T,), -7, dtype=torch.int32, device=DEV)
    wsb = lcsa.lcs_index_topk_workspace(batch, heads, cache.keys, cache.paging, m, k)
    lcsa.csa_index_topk(batch, q_fp4, q_sc, hw, heads, cache.keys, cache.paging, m, k, flags, out_idx, out_cnt,
                        workspace(wsb), wsb, st)
    torch.cuda.synchronize()
    return out_idx.cpu().numpy(), out_cnt.cpu().numpy()


@pytest.mark.parametrize("k", [512, 1024])
@pytest.mark.parametrize("new", [[1, 1], [2, 3]])
def test_topk_all_scores_tied_takes_lowest_indices(k, new):
    # every key of a sequence is the same row: every score of a query is the same value
    m = 4
    lengths = [160004, 200000]                      # 40001 and 50000 entries
    cache, batch, *_, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, 4, 128, False, True, ties=True)
    st = dev_status()
    oi, oc = _topk(batch, cache, q_fp4, q_sc, hw, 4, m, k, st)
    assert_status_ok(st)
    assert np.array_equal(oc, np.full(batch.total_new, k))
    assert np.array_equal(oi, np.tile(np.arange(k), (batch.total_new, 1)))


def test_topk_ties_below_a_few_larger_scores():
    """300 entries spread over the sequence score above a sea of ~40000 tied entries: the top-k is
    those 300 plus the lowest-index tied entries, exactly as the oracle's sort gives."""
    m, k, heads, rank = 4, 512, 4, 128
    lengths, new = [165000, 120000], [1, 2]
    cache, batch, kcs, kss, qcs, qss, hws, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, heads, rank, False,
                                                                       True, ties=True)
    rng = np.random.default_rng(3)
    for b, L in enumerate(lengths):
        ne = L // m
        pick = np.sort(rng.choice(ne, size=300, replace=False))
        kc = kcs[b]
        kc[pick] = synth.e2m1_codes(99, b, 0, 300 * rank).reshape(300, rank)   # other rows: other scores
        rows = entry_rows_of(cache, b, pick)
        cache.keys.fp4[torch.as_tensor(rows, device=DEV)] = u8(synth.pack_e2m1(kc[pick]))
    st = dev_status()
    oi, oc = _topk(batch, cache, q_fp4, q_sc, hw, heads, m, k, st)
    assert_status_ok(st)
    qi = 0
    for b, L in enumerate(lengths):
        ref = oracle.index_scores(qcs[b], qss[b], hws[b], kcs[b], kss[b])
        for i in range(new[b]):
            t = L - new[b] + i
            n = oracle.visible_entries(t, m)
            sel = oracle.topk_select(ref[i, :n], k)
            assert oc[qi] == len(sel)
            assert np.array_equal(oi[qi, :len(sel)], sel), f"seq {b} query {i}"
            qi += 1


def test_unmapped_page_reports_guard_indexer():
    """Sequence 1's first page unmapped in the block table: the status reports the guard and the
    other sequences' top-k lists are still exact."""
    m, k, heads, rank = 4, 64, 4, 128
    lengths, new = [3000, 5000, 2600], [1, 1, 1]
    cache, batch, kcs, kss, qcs, qss, hws, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, heads, rank, False,
                                                                       True)
    cache.paging.block_table[1, 0] = -1
    st = dev_status()
    oi, oc = _topk(batch, cache, q_fp4, q_sc, hw, heads, m, k, st)
    assert int(st.item()) == 6, f"device status {int(st.item())}, expected LCS_ERR_DEVICE_GUARD"
    for qi, b in ((0, 0), (2, 2)):
        t = lengths[b] - 1
        n = oracle.visible_entries(t, m)
        ref = oracle.index_scores(qcs[b], qss[b], hws[b], kcs[b], kss[b])
        sel = oracle.topk_select(ref[0, :n], k)
        assert oc[qi] == len(sel) and np.array_equal(oi[qi, :len(sel)], sel), f"seq {b}"


@pytest.mark.parametrize("kind,lengths,new,m,k", [
    ("csa", [2000, 4100, 300], [1, 1, 1], 4, 512),
    ("csa", [900, 2200, 1500], [40, 9, 3], 4, 64),
    ("hca", [20000, 1500, 9000], [1, 1, 1], 128, 0),
])
def test_unmapped_page_reports_guard_attention(kind, lengths, new, m, k):
    _attend_case(kind, lengths, new, 64, 512, "fp8_split", m, k, corrupt_seq=1)


def _nope_tiny_rows(b, rows):
    """Every 9th entry row of sequence 0: RoPE dims +-2 and FP8 dims with amax = 2/400, so that
    |rope| / s_r = 448 * 400 exceeds the f16 range of the kernels' widened rows."""
    if b == 0:
        rows = rows.copy()
        sel = rows[::9]
        sel[:, :64] = np.where(sel[:, :64] < 0, -2.0, 2.0)
        sel[:, 64:] *= (2.0 / 400.0) / np.abs(sel[:, 64:]).max(axis=1, keepdims=True)
        rows[::9] = sel
    return rows


def test_rope_beyond_f16_range_reports_guard():
    """Rows whose RoPE dims exceed 65504 times the row's FP8 scale cannot be widened to f16: the
    call reports LCS_ERR_DEVICE_GUARD; the sequences without such rows still match the oracle."""
    _attend_case("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512,
                 rows_hook=_nope_tiny_rows, skip_seq=0, expect_status=6)


def test_bounded_waits_report_timeout_then_recover():
    """With the wait bound at 0 every pipeline wait of the tensor-core kernels gives up at once: the
    calls complete, the device status reads LCS_ERR_TIMEOUT and the context stays usable -- the
    same calls under the default bound then give the oracle's results."""
    m, k, heads, rank = 4, 64, 4, 128
    lengths, new = [3000, 5000], [1, 1]
    cache, batch, kcs, kss, qcs, qss, hws, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, heads, rank, False,
                                                                       True)
    prev = lcsa.lcs_set_wait_polls(0)
    try:
        st = dev_status()
        _topk(batch, cache, q_fp4, q_sc, hw, heads, m, k, st)
        assert int(st.item()) == 7, f"indexer: device status {int(st.item())}, expected LCS_ERR_TIMEOUT"
        for kind, lens, mm, kk in (("csa", [2000, 4100, 300], 4, 512), ("hca", [20000, 1500], 128, 0)):
            _attend_case(kind, lens, [1] * len(lens), 64, 512, "fp8_split", mm, kk, expect_status=7)
    finally:
        assert lcsa.lcs_set_wait_polls(prev) == 0
    st = dev_status()
    oi, oc = _topk(batch, cache, q_fp4, q_sc, hw, heads, m, k, st)
    assert_status_ok(st)
    for b, L in enumerate(lengths):
        ref = oracle.index_scores(qcs[b], qss[b], hws[b], kcs[b], kss[b])
        sel = oracle.topk_select(ref[0, :oracle.visible_entries(L - 1, m)], k)
        assert oc[b] == len(sel) and np.array_equal(oi[b, :len(sel)], sel), f"seq {b}"
    _attend_case("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512)


@pytest.mark.parametrize("spare", [32, 100, 140])
def test_topk_with_spare_sms_matches_oracle(spare):
    """The scorer sized for fewer SMs (longer runs, fewer run lists; at least 16 SMs remain) gives
    the oracle's top-k, as with every SM."""
    m, k, heads, rank = 4, 512, 4, 128
    lengths, new = [40000, 130000, 9000], [1, 1, 1]
    cache, batch, kcs, kss, qcs, qss, hws, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, heads, rank, False,
                                                                       True)
    st = dev_status()
    oi, oc = _topk(batch, cache, q_fp4, q_sc, hw, heads, m, k, st, flags=lcsa.LCS_INDEX_SPARE_SMS(spare))
    assert_status_ok(st)
    for b, L in enumerate(lengths):
        ref = oracle.index_scores(qcs[b], qss[b], hws[b], kcs[b], kss[b])
        sel = oracle.topk_select(ref[0, :oracle.visible_entries(L - 1, m)], k)
        assert oc[b] == len(sel) and np.array_equal(oi[b, :len(sel)], sel), f"seq {b}"


def test_topk_few_long_sequences_merge_kernel():
    """Two sequences of about a million tokens at k = 1024: more runs than the scorer's ring can
    stage, so the runs are capped to what the merge kernel stages and the merge kernel selects;
    the top-k equals the oracle's."""
    m, k, heads, rank = 4, 1024, 4, 128
    lengths, new = [1000000, 700001], [1, 1]
    cache, batch, kcs, kss, qcs, qss, hws, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, heads, rank, False,
                                                                       True)
    st = dev_status()
    oi, oc = _topk(batch, cache, q_fp4, q_sc, hw, heads, m, k, st)
    assert_status_ok(st)
    for b, L in enumerate(lengths):
        ref = oracle.index_scores(qcs[b], qss[b], hws[b], kcs[b], kss[b])
        sel = oracle.topk_select(ref[0, :oracle.visible_entries(L - 1, m)], k)
        assert oc[b] == len(sel) and np.array_equal(oi[b, :len(sel)], sel), f"seq {b}"
