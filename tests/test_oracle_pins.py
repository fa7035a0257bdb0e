"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: the pages' printed
values (tests/golden/pages_constants.json), closed forms, invariants, and special cases that
reduce to a library routine (numpy, scipy, torch CPU).  Each test names the plausible mistake
it would catch.
"""
import heapq
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))
RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ number formats

def test_e2m1_table_matches_page():
    # catches a wrong exponent bias or mantissa weight in the FP4 decoder
    pos = oracle.e2m1_value(np.arange(8))
    assert list(pos) == GOLDEN["e2m1_positive_values"]["value"]
    assert list(oracle.e2m1_value(np.arange(8, 16))) == [-v for v in pos]


def test_e2m1_15_distinct_values_drawn():
    codes = synth.e2m1_codes(0, 1, 0, 30000)
    vals = oracle.e2m1_value(codes)
    assert len(np.unique(vals)) == 15
    assert not np.any(codes == 8)          # negative zero never drawn


def test_fp4_to_fp8_lossless():
    # x-techcon section 4: FP4 -> FP8 conversion is lossless (FP8 has two more exponent bits)
    v = oracle.e2m1_value(np.arange(16))
    for e in (-1, 0, 1):
        x = v * 2.0 ** e
        assert np.array_equal(oracle.e4m3_round_satfinite(x), x)


def test_bf16_round_matches_torch():
    # torch's float32 -> bfloat16 cast is round-to-nearest-even; inputs are fp32 values
    x = (RNG.standard_normal(200000) * np.exp(RNG.uniform(-30, 30, 200000))).astype(np.float32)
    x = np.concatenate([x, np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0])])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_round(x.astype(np.float64)), ref)


def test_e4m3_round_matches_torch_in_range():
    x = RNG.uniform(-448, 448, 200000) * np.exp(RNG.uniform(-12, 0, 200000))
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_round_satfinite(x.astype(np.float64)), ref)
    # saturation (the format has no infinity; torch gives NaN past 464, the oracle saturates)
    assert oracle.e4m3_round_satfinite(np.array([500.0, -1e6]))[0] == 448.0
    assert oracle.e4m3_round_satfinite(np.array([-1e6]))[0] == -448.0


def test_e4m3_codes_match_torch():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_decode(codes), ref)
    back = oracle.e4m3_encode(ref)
    # +0/-0 both decode to 0; compare values for the zero codes and bytes elsewhere
    nz = ref != 0
    assert np.array_equal(back[nz], codes[nz])


def test_ue8m0_closed_form():
    assert list(oracle.ue8m0_value(np.array([126, 127, 128, 130]))) == [0.5, 1.0, 2.0, 8.0]


def test_row_format_sizes_and_two_percent():
    # x-techcon section 2: RoPE dims BF16, the rest FP8, about half of BF16.
    b = oracle.kv_bytes_per_token(512)
    assert b["row"] == 64 * 2 + 448 + 4 == 580
    assert 0.5 < b["row"] / (512 * 2) < 0.6
    # digipub: about 2% of a BF16 GQA8 cache at 1M.  The GQA8 baseline (8 KV heads x K and V x
    # head dim 128 x 2 bytes) is an assumption outside the pages; the CSA/HCA pair average
    # (layers alternate) of our stored bytes lands at about 2%.
    pair = (b["csa"] + b["hca"]) / 2
    gqa8 = 8 * 2 * 128 * 2
    assert abs(pair / gqa8 - GOLDEN["kv_vs_bf16_gqa8_at_1m"]["value_approx"]) < 0.003


def test_quantize_rows_fp8_split():
    x = RNG.standard_normal((64, 512))
    f = oracle.quantize_rows(x, "fp8_split")
    deq = f["deq"]
    # RoPE slice within half a bf16 ulp; FP8 slice within half an e4m3 ulp of x/s times s
    assert np.all(np.abs(deq[:, :64] - x[:, :64]) <= np.abs(x[:, :64]) * 2 ** -8 + 1e-300)
    s = f["scale"].astype(np.float64)[:, None]
    assert np.all(np.abs(deq[:, 64:] - x[:, 64:]) <= np.maximum(np.abs(x[:, 64:]) * 2 ** -4, s * 2 ** -10) + 1e-6 * s)
    # the largest magnitude of every row maps to the largest code (448 * s)
    assert np.allclose(np.max(np.abs(deq[:, 64:]), axis=1), f["scale"].astype(np.float64) * 448.0, rtol=0, atol=0)
    assert np.array_equal(oracle.dequantize_rows(f), deq)
    # zero row: scale 1, all codes zero
    z = oracle.quantize_rows(np.zeros((1, 512)), "fp8_split")
    assert z["scale"][0] == 1.0 and not np.any(z["deq"])


# ------------------------------------------------------------------ compression

def test_counts_closed_form():
    n = GOLDEN["compressed_len_1m"]["tokens"]
    m = GOLDEN["csa_ratio"]["value"]
    assert oracle.num_entries(n, m) == 262144
    assert abs(oracle.num_entries(n, m) - GOLDEN["compressed_len_1m"]["value_approx"]) / 250000 < 0.05
    assert oracle.num_entries(n, GOLDEN["hca_ratio"]["value"]) == 8192
    for n in range(0, 50):
        for m in (1, 2, 4, 8):
            nf = oracle.num_entries(n, m)
            assert math.ceil(n / m) == nf + (1 if n % m else 0)
    # one cache block of LCM(4,128) raw tokens holds 32 CSA entries and 1 HCA entry
    blk = GOLDEN["cache_block_raw_tokens"]["value"]
    assert math.lcm(4, 128) == blk and blk // 4 == 32 and blk // 128 == 1


def _rand_seq(n, d=16):
    return RNG.standard_normal((n, d))


@pytest.mark.parametrize("m,overlap", [(4, True), (4, False), (2, True), (8, False)])
def test_weights_sum_to_one(m, overlap):
    raw = _rand_seq(10 * m)
    w = RNG.standard_normal(16)
    bias = RNG.standard_normal(2 * m if overlap else m)
    _, ws = oracle.compress(raw, w, bias, m, overlap, return_weights=True)
    for a in ws:
        assert abs(a.sum() - 1.0) <= 1e-15 and np.all(a > 0)


@pytest.mark.parametrize("m,overlap", [(4, True), (128, False)])
def test_constant_window_gives_that_row(m, overlap):
    row = RNG.standard_normal(16)
    raw = np.tile(row, (3 * m, 1))
    bias = RNG.standard_normal(2 * m if overlap else m) * 3
    c = oracle.compress(raw, RNG.standard_normal(16), bias, m, overlap)
    assert np.allclose(c, row[None, :], rtol=0, atol=1e-14)


def test_ratio_one_is_identity():
    raw = _rand_seq(37)
    c = oracle.compress(raw, RNG.standard_normal(16), RNG.standard_normal(1), 1, False)
    assert np.array_equal(c, raw)


@pytest.mark.parametrize("m,overlap", [(4, True), (4, False), (128, False)])
def test_uniform_weights_give_mean(m, overlap):
    # w = 0 and b = 0: softmax weights are uniform, the entry is the mean of the rows that exist
    raw = _rand_seq(5 * m + 3)
    nb = 2 * m if overlap else m
    c = oracle.compress(raw, np.zeros(16), np.zeros(nb), m, overlap)
    for j in range(c.shape[0]):
        lo = max((j - 1) * m if overlap else j * m, 0)
        assert np.allclose(c[j], np.mean(raw[lo:(j + 1) * m], axis=0), rtol=0, atol=1e-14)


@pytest.mark.parametrize("m,overlap", [(4, True), (4, False)])
def test_one_hot_bias_picks_offset(m, overlap):
    # catches an off-by-one in the window offsets or in which block comes first
    raw = _rand_seq(6 * m)
    nb = 2 * m if overlap else m
    for o in range(nb):
        bias = np.zeros(nb)
        bias[o] = 2000.0
        c = oracle.compress(raw, np.zeros(16), bias, m, overlap)
        for j in range(c.shape[0]):
            lo = (j - 1) * m if overlap else j * m
            if lo + o >= 0:
                assert np.allclose(c[j], raw[lo + o], rtol=0, atol=1e-12)
            else:       # the favoured row does not exist: uniform over the rows that do
                assert np.allclose(c[j], np.mean(raw[max(lo, 0):(j + 1) * m], axis=0), atol=1e-12)


def test_weights_equal_scipy_softmax_of_bias():
    m = 4
    raw = _rand_seq(8 * m)
    bias = RNG.standard_normal(2 * m) * 2
    _, ws = oracle.compress(raw, np.zeros(16), bias, m, True, return_weights=True)
    assert np.allclose(ws[0], scipy.special.softmax(bias[m:]), rtol=1e-15, atol=0)
    for a in ws[1:]:
        assert np.allclose(a, scipy.special.softmax(bias), rtol=1e-14, atol=0)


def test_linear_score_term_acts_on_keys():
    # a score vector w along one coordinate: the heavier row in the softmax is the one with the
    # larger value on that coordinate (sign error in z would flip this)
    m = 4
    raw = _rand_seq(2 * m)
    w = np.zeros(16); w[3] = 1e5
    c = oracle.compress(raw, w, np.zeros(2 * m), m, True)
    assert np.allclose(c[1], raw[np.argmax(raw[:, 3])], atol=1e-10)


def test_entries_in_convex_hull():
    m = 4
    raw = _rand_seq(40 * m)
    c = oracle.compress(raw, RNG.standard_normal(16), RNG.standard_normal(2 * m), m, True)
    for j in range(c.shape[0]):
        rows = raw[max((j - 1) * m, 0):(j + 1) * m]
        assert np.all(c[j] <= rows.max(0) + 1e-12) and np.all(c[j] >= rows.min(0) - 1e-12)


@pytest.mark.parametrize("m,overlap", [(4, True), (128, False), (1, False), (2, True)])
def test_blocked_equals_per_entry(m, overlap):
    raw = _rand_seq(7 * m + 1)
    w = RNG.standard_normal(16)
    bias = RNG.standard_normal(2 * m if overlap else m)
    a = oracle.compress(raw, w, bias, m, overlap)
    b = oracle.compress_blocked(raw, w, bias, m, overlap)
    assert np.allclose(a, b, rtol=0, atol=1e-13)
    for first in range(0, a.shape[0]):
        part = oracle.compress_blocked(raw, w, bias, m, overlap, first, a.shape[0] - first)
        assert np.allclose(part, a[first:], rtol=0, atol=1e-13)


def test_compression_is_causal_and_local():
    # entry j changes only if a token inside its span changes
    m = 4
    raw = _rand_seq(12 * m)
    w = RNG.standard_normal(16); bias = RNG.standard_normal(2 * m)
    c0 = oracle.compress(raw, w, bias, m, True)
    raw2 = raw.copy(); raw2[5 * m + 1] += 1.0
    c1 = oracle.compress(raw2, w, bias, m, True)
    changed = np.where(np.any(c0 != c1, axis=1))[0]
    assert list(changed) == [5, 6]


# ------------------------------------------------------------------ indexer and top-k

def _idx_inputs(t, hi, r, n, seed=3, scaled=True):
    qc = synth.e2m1_codes(seed, 1, 0, t * hi * r).reshape(t, hi, r)
    kc = synth.e2m1_codes(seed, 2, 0, n * r).reshape(n, r)
    if scaled:
        qs = synth.ue8m0_scales(seed, 3, 0, t * hi * r // 32).reshape(t, hi, r // 32)
        ks = synth.ue8m0_scales(seed, 4, 0, n * r // 32).reshape(n, r // 32)
    else:
        qs = np.full((t, hi, r // 32), 127, np.uint8)
        ks = np.full((n, r // 32), 127, np.uint8)
    hw = synth.head_weights(seed, 5, 0, t * hi).reshape(t, hi)
    return qc, qs, hw, kc, ks


def test_index_score_is_integer_dot_product_unscaled():
    # one head, unit scales, unit weight: the score is the plain dot product of the e2m1 values
    qc, qs, _, kc, ks = _idx_inputs(3, 1, 64, 50, scaled=False)
    s = oracle.index_scores(qc, qs, None, kc, ks)
    qi = (2 * oracle.e2m1_value(qc)).astype(np.int64)     # 2 * e2m1 is an integer
    ki = (2 * oracle.e2m1_value(kc)).astype(np.int64)
    ref = np.dot(qi[:, 0, :], ki.T) / 4.0
    assert np.array_equal(s, ref)


def test_index_score_block_scale_homogeneity():
    qc, qs, hw, kc, ks = _idx_inputs(2, 4, 128, 40)
    s = oracle.index_scores(qc, qs, hw, kc, ks)
    assert np.array_equal(oracle.index_scores(qc, qs, hw, kc, ks + 1), 2 * s)
    # doubling one block's key scale adds that block's contribution once more
    ks2 = ks.copy(); ks2[:, 1] += 1
    qv = oracle.blockscaled_values(qc, qs)[:, :, 32:64]
    kv = oracle.blockscaled_values(kc, ks)[:, 32:64]
    extra = np.einsum("th,thn->tn", hw, np.einsum("thr,nr->thn", qv, kv))
    assert np.array_equal(oracle.index_scores(qc, qs, hw, kc, ks2), s + extra)


def test_index_score_head_combination():
    qc, qs, hw, kc, ks = _idx_inputs(2, 4, 128, 30)
    s = oracle.index_scores(qc, qs, hw, kc, ks)
    per = [oracle.index_scores(qc[:, h:h + 1], qs[:, h:h + 1], None, kc, ks) for h in range(4)]
    assert np.array_equal(s, sum(hw[:, h:h + 1] * per[h] for h in range(4)))
    r = oracle.index_scores(qc, qs, hw, kc, ks, relu=True)
    assert np.array_equal(r, sum(hw[:, h:h + 1] * np.maximum(per[h], 0) for h in range(4)))
    assert np.all(r >= s)


def test_index_scores_exact_in_fp32():
    # every score of the generator's ranges is exactly representable in fp32
    qc, qs, hw, kc, ks = _idx_inputs(4, 4, 128, 2000)
    s = oracle.index_scores(qc, qs, hw, kc, ks)
    assert np.array_equal(s.astype(np.float32).astype(np.float64), s)
    assert np.all(np.abs(s) < 2 ** 24 * 2 ** -5)
    assert np.array_equal(np.round(s * 32), s * 32)


def test_topk_matches_heapq():
    for n, k in [(1, 1), (10, 3), (64, 64), (64, 65), (300, 17), (1000, 64)]:
        s = RNG.integers(-5, 5, n).astype(np.float64)        # many ties
        got = oracle.topk_select(s, k)
        ref = sorted(-negj for (_, negj) in heapq.nlargest(min(k, n), ((s[j], -j) for j in range(n))))
        assert list(got) == ref


def test_topk_ties_lowest_index_and_small_n():
    assert list(oracle.topk_select(np.zeros(100), 7)) == list(range(7))
    assert list(oracle.topk_select(np.arange(5.0), 10)) == [0, 1, 2, 3, 4]
    s = RNG.standard_normal(500)
    assert np.array_equal(oracle.topk_select(s, 40), oracle.topk_select(np.exp(s) * 3 + 1, 40))


# ------------------------------------------------------------------ attention

def test_attend_matches_torch_sdpa():
    h, r, d = 8, 37, 64
    q = RNG.standard_normal((h, d)); k = RNG.standard_normal((r, d)); v = RNG.standard_normal((r, d))
    scale = 0.3
    o, lse = oracle.attend(q, k, scale, v)
    tq = torch.from_numpy(q)[None, :, None, :]                 # [1, H, 1, D]
    tk = torch.from_numpy(k)[None, None].expand(1, h, r, d)
    tv = torch.from_numpy(v)[None, None].expand(1, h, r, d)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, :, 0].numpy()
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, scipy.special.logsumexp(scale * q @ k.T, axis=1), rtol=1e-14, atol=1e-12)


def test_attend_special_cases():
    q = RNG.standard_normal((4, 32)); rows = RNG.standard_normal((9, 32))
    o, lse = oracle.attend(q, rows[:1], 0.5)
    assert np.array_equal(o, np.repeat(rows[:1], 4, 0))
    assert np.allclose(lse, 0.5 * q @ rows[0])
    o, lse = oracle.attend(np.zeros((4, 32)), rows, 0.5)
    assert np.allclose(o, rows.mean(0)[None], atol=1e-14) and np.allclose(lse, math.log(9))


def test_window_positions():
    assert list(oracle.window_positions(0)) == [0]
    assert list(oracle.window_positions(5)) == list(range(6))
    assert list(oracle.window_positions(1000)) == list(range(873, 1001))
    assert len(oracle.window_positions(1000)) == GOLDEN["window"]["value"]
    assert oracle.visible_entries(3, 4) == 1 and oracle.visible_entries(2, 4) == 0
    assert oracle.visible_entries(127, 128) == 1 and oracle.visible_entries(126, 128) == 0


def test_ratio_one_full_topk_no_window_is_causal_mqa():
    # m=1, no overlap, k >= every N(t), window 0: CSA is standard causal multi-query attention
    n, h, d = 40, 4, 32
    raw = oracle.bf16_round(RNG.standard_normal((n, d)))
    q = RNG.standard_normal((n, h, d))
    ent = oracle.compress(raw, RNG.standard_normal(d), RNG.standard_normal(1), 1, False)
    outs = []
    for t in range(n):
        sel = oracle.topk_select(RNG.standard_normal(oracle.visible_entries(t, 1)), 10 ** 6)
        rows = oracle.csa_query_rows(t, sel, ent, raw, window=0)
        outs.append(oracle.attend(q[t], rows, 0.2)[0])
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]                 # [1, H, n, D]
    tk = torch.from_numpy(raw)[None, None].expand(1, h, n, d)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tk, is_causal=True, scale=0.2)
    assert np.allclose(np.stack(outs), ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_hca_is_csa_with_all_entries():
    # I3: HCA equals CSA with k covering every visible entry, on the same cache
    n, m, d = 700, 4, 32
    raw = RNG.standard_normal((n, d)); ent = RNG.standard_normal((n // m, d))
    q = RNG.standard_normal((3, d))
    for t in (3, 130, 699):
        sel = oracle.topk_select(RNG.standard_normal(oracle.visible_entries(t, m)), 10 ** 6)
        a = oracle.attend(q, oracle.csa_query_rows(t, sel, ent, raw), 0.1)[0]
        b = oracle.attend(q, oracle.hca_query_rows(t, m, ent, raw), 0.1)[0]
        assert np.allclose(a, b, rtol=1e-13, atol=1e-13)


def _small_layer(seed, n, h=4, d=128, m=4, r=64, hi=2, k=8, fmt="fp8_split"):
    s = seed
    raw = synth.bf16_bits_to_f32(synth.normal_bf16(s, 1, 0, n * d)).reshape(n, d).astype(np.float64)
    w = synth.bf16_bits_to_f32(synth.normal_bf16(s, 2, 0, d)).astype(np.float64) / 8
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(s, 3, 0, 2 * m)).astype(np.float64) / 2
    q_pos = np.arange(n - 6, n)
    q = synth.bf16_bits_to_f32(synth.normal_bf16(s, 4, 0, 6 * h * d)).reshape(6, h, d).astype(np.float64)
    qc = synth.e2m1_codes(s, 5, 0, 6 * hi * r).reshape(6, hi, r)
    qs = synth.ue8m0_scales(s, 6, 0, 6 * hi * r // 32).reshape(6, hi, r // 32)
    hw = synth.head_weights(s, 7, 0, 6 * hi).reshape(6, hi)
    kc = synth.e2m1_codes(s, 8, 0, (n // m) * r).reshape(n // m, r)
    ks = synth.ue8m0_scales(s, 9, 0, (n // m) * r // 32).reshape(n // m, r // 32)
    return raw, dict(w=w, bias=bias, m=m, overlap=True, row_format=fmt, q=q, q_pos=q_pos,
                     idx_q_codes=qc, idx_q_scales=qs, head_w=hw, idx_k_codes=kc, idx_k_scales=ks,
                     top_k=k, softmax_scale=1 / math.sqrt(d))


def test_layer_is_causal():
    # I6: changing tokens after a query's position leaves that query's output unchanged
    raw, kw = _small_layer(11, 200)
    kw2 = dict(kw)
    kw2["q"] = kw["q"][:3]; kw2["q_pos"] = kw["q_pos"][:3]
    for key in ("idx_q_codes", "idx_q_scales", "head_w"):
        kw2[key] = kw[key][:3]
    a = oracle.csa_layer(raw[:kw2["q_pos"][-1] + 1], **kw2)
    raw2 = raw.copy(); raw2[kw2["q_pos"][-1] + 1:] += 3.0
    b = oracle.csa_layer(raw2, **kw2)
    assert np.array_equal(a["o"], b["o"])
    assert all(np.array_equal(x, y) for x, y in zip(a["topk"], b["topk"]))


def test_layer_full_topk_equals_dense_over_visible():
    # I2: with k >= N(t), CSA equals one softmax over every visible entry and the window
    raw, kw = _small_layer(12, 160, k=10 ** 6)
    out = oracle.csa_layer(raw, **kw)
    ent = out["entries"]["deq"]; win = out["window"]["deq"]
    for i, t in enumerate(kw["q_pos"]):
        rows = np.concatenate([ent[:oracle.visible_entries(int(t), 4)], win[oracle.window_positions(int(t))]])
        ref = oracle.attend(kw["q"][i], rows, kw["softmax_scale"])[0]
        assert np.allclose(out["o"][i], ref, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------------------------------------
# Per-channel compression weights (the variant reading: chenxutan section 4.2 sketch)
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("m,overlap", [(4, True), (4, False), (2, True), (1, False)])
def test_per_channel_weights_are_a_softmax_per_channel(m, overlap):
    n, d = 37, 24
    raw = RNG.standard_normal((n, d)); sc = RNG.standard_normal((n, d)) * 2
    bias = RNG.standard_normal(((2 * m if overlap else m), d))
    out, ws = oracle.compress_per_channel(raw, sc, bias, m, overlap, return_weights=True)
    for j, a in enumerate(ws):
        lo, hi = oracle.entry_span(j, m, overlap)
        t = np.arange(max(lo, 0), hi)
        assert np.allclose(a.sum(axis=0), 1.0, atol=1e-15)
        assert np.allclose(a, scipy.special.softmax(sc[t] + bias[t - lo], axis=0), rtol=1e-13, atol=1e-15)
        assert np.allclose(out[j], np.einsum("td,td->d", a, raw[t]), rtol=1e-13, atol=1e-13)


def test_per_channel_with_equal_channels_is_the_scalar_reading():
    # every channel scored by the scalar w . k_t and one bias per offset: the per-channel softmax is
    # the same in every channel, and the entries are those of the scalar compressor
    n, d, m = 41, 16, 4
    raw = RNG.standard_normal((n, d)); w = RNG.standard_normal(d); b = RNG.standard_normal(2 * m)
    sc = np.repeat((raw @ w)[:, None], d, axis=1)
    per = oracle.compress_per_channel(raw, sc, np.repeat(b[:, None], d, axis=1), m, True)
    assert np.allclose(per, oracle.compress(raw, w, b, m, True), rtol=1e-13, atol=1e-13)


def test_per_channel_channels_are_independent_and_local():
    n, d, m = 40, 12, 4
    raw = RNG.standard_normal((n, d)); sc = RNG.standard_normal((n, d))
    bias = RNG.standard_normal((2 * m, d))
    a = oracle.compress_per_channel(raw, sc, bias, m, True)
    raw2, sc2 = raw.copy(), sc.copy()
    raw2[:, 5] += 3.0; sc2[:, 5] -= 2.0                   # channel 5 only
    b = oracle.compress_per_channel(raw2, sc2, bias, m, True)
    keep = [c for c in range(d) if c != 5]
    assert np.array_equal(a[:, keep], b[:, keep]) and not np.allclose(a[:, 5], b[:, 5])
    raw3 = raw.copy(); raw3[20] += 5.0                    # token 20 (block 5) reaches entries 5 and 6 only
    c = oracle.compress_per_channel(raw3, sc, bias, m, True)
    changed = [j for j in range(n // m) if not np.array_equal(a[j], c[j])]
    assert changed == [5, 6]


def test_per_channel_constant_window_and_ratio_one():
    n, d = 24, 8
    row = RNG.standard_normal(d)
    raw = np.tile(row, (n, 1)); sc = RNG.standard_normal((n, d))
    out = oracle.compress_per_channel(raw, sc, RNG.standard_normal((8, d)), 4, True)
    assert np.allclose(out, np.tile(row, (n // 4, 1)), rtol=1e-14, atol=1e-14)
    raw = RNG.standard_normal((n, d))
    assert np.array_equal(oracle.compress_per_channel(raw, sc, np.zeros((1, d)), 1, False), raw)


def _brute_rows(t, selected, entries, window_rows, window=128):
    """The rows a CSA query attends, gathered one by one: the listed entries in list order, then
    the window tokens from max(0, t - window + 1) up to t itself."""
    rows = []
    for j in selected:
        rows.append(entries[int(j)])
    p = max(0, t - window + 1)
    while p <= t:
        rows.append(window_rows[p])
        p += 1
    return np.array(rows)


def _softmax_attend_loops(q, rows, scale):
    """One head at a time, one row at a time: max, exponentials, weighted sum (plain loops)."""
    h_n, d = q.shape
    out = np.zeros((h_n, rows.shape[1]))
    for h in range(h_n):
        logits = [scale * float(np.dot(q[h], r)) for r in rows]
        mx = max(logits)
        w = [math.exp(z - mx) for z in logits]
        tot = sum(w)
        for wi, r in zip(w, rows):
            out[h] += (wi / tot) * r
    return out


def test_csa_query_rows_gathers_the_selected_entries():
    # k < N(t): only the listed entries join the window rows, in list order, whatever their positions
    ent = RNG.standard_normal((300, 16))
    win = RNG.standard_normal((1300, 16))
    for t, sel in [(1199, np.array([0, 7, 8, 150, 299])), (1199, np.array([299, 3])), (40, np.array([5])),
                   (1000, np.sort(RNG.choice(250, size=37, replace=False))), (7, np.zeros(0, np.int64))]:
        got = oracle.csa_query_rows(t, sel, ent, win)
        ref = _brute_rows(t, sel, ent, win)
        assert got.shape == ref.shape and np.array_equal(got, ref), (t, sel[:4])


def test_csa_layer_top_k_smaller_than_visible_entries_by_loops():
    # the whole layer with k < N(t): the top-k of explicitly computed scores (a full sort per query),
    # the rows gathered one by one and a loop softmax give the oracle's outputs
    raw, kw = _small_layer(13, 240, k=5)
    out = oracle.csa_layer(raw, **kw)
    ent = out["entries"]["deq"]; win = out["window"]["deq"]
    qv = oracle.blockscaled_values(kw["idx_q_codes"], kw["idx_q_scales"])
    kv = oracle.blockscaled_values(kw["idx_k_codes"], kw["idx_k_scales"])
    for i, t in enumerate(kw["q_pos"]):
        n = oracle.visible_entries(int(t), 4)
        assert n > kw["top_k"]
        sc = [sum(kw["head_w"][i, h] * float(np.dot(qv[i, h], kv[j])) for h in range(qv.shape[1]))
              for j in range(n)]
        order = sorted(range(n), key=lambda j: (-sc[j], j))
        sel = sorted(order[:kw["top_k"]])
        assert list(out["topk"][i]) == sel
        ref = _softmax_attend_loops(kw["q"][i], _brute_rows(int(t), sel, ent, win), kw["softmax_scale"])
        assert np.allclose(out["o"][i], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------------
# Block-scaled FP4 quantisation (the indexer's key / query production, x-techcon section 4)
# ------------------------------------------------------------------------------------------------

def _e2m1_table():
    codes = np.arange(16, dtype=np.uint8)
    return codes, oracle.e2m1_value(codes)


def test_e2m1_block_quantize_round_trips_representable_blocks():
    """Blocks of E2M1 values times 2^e whose largest magnitude is 4 or 6 come back as the same
    codes and scale exponent e (zero stored as +0)."""
    rng = np.random.default_rng(11)
    nb = 200
    mags = rng.integers(0, 8, size=(nb, 32))
    mags[np.arange(nb), rng.integers(0, 32, size=nb)] = rng.choice([6, 7], size=nb)   # 4.0 or 6.0
    signs = rng.integers(0, 2, size=(nb, 32))
    codes = (mags | (signs << 3)).astype(np.uint8)
    codes[mags == 0] = 0
    e = rng.integers(-40, 40, size=nb)
    x = oracle.e2m1_value(codes) * np.ldexp(1.0, e)[:, None]
    got_c, got_s = oracle.e2m1_block_quantize(x.reshape(1, -1))
    assert np.array_equal(got_c.reshape(nb, 32), codes)
    assert np.array_equal(got_s.reshape(nb).astype(np.int64) - 127, e)


def test_e2m1_block_quantize_nearest_value_ties_to_even_brute_force():
    """Every element's stored value is a nearest one among all 15 E2M1 values times the block
    scale (checked by exhaustive search); on a tie the code's mantissa bit is 0; the scale is the
    smallest power of two with amax <= 6 * scale."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((64, 128)) * np.ldexp(1.0, rng.integers(-10, 10, size=(64, 1)))
    # exact ties: block 0 of row 0 holds the midpoints between neighbouring E2M1 values (scale 1)
    x[0, :8] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]
    x[0, 8:32] = -np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 3 + [0.0] * 3)
    codes, scales = oracle.e2m1_block_quantize(x)
    tc, tv = _e2m1_table()
    for i in range(x.shape[0]):
        for blk in range(4):
            sc = oracle.ue8m0_value(scales[i, blk])
            xb = x[i, blk * 32:(blk + 1) * 32]
            amax = np.abs(xb).max()
            assert 6.0 * sc >= amax and (amax == 0 or 6.0 * sc / 2 < amax)
            for j in range(32):
                c = codes[i, blk * 32 + j]
                err = np.abs(xb[j] - tv * sc)
                best = err.min()
                assert abs(xb[j] - oracle.e2m1_value(c) * sc) == best
                if np.count_nonzero(np.isclose(err, best, rtol=0, atol=0)) > 1 and best > 0:
                    assert (c & 1) == 0
    assert list(codes[0, :8]) == [0, 2, 2, 4, 4, 6, 6, 7]


def test_e2m1_block_quantize_zero_and_extremes():
    codes, scales = oracle.e2m1_block_quantize(np.zeros((2, 64)))
    assert not codes.any() and np.all(scales == 0)                 # 2^-127, all +0
    big = np.full((1, 32), 3.0e38)
    c, s = oracle.e2m1_block_quantize(big)
    assert s[0, 0] == 127 + 126 and np.all(c == 6)                # 3e38 = 4 * 2^126 (rounded)
    tiny = np.full((1, 32), 1e-40)
    c, s = oracle.e2m1_block_quantize(tiny)
    assert s[0, 0] == 0                                            # clamped at 2^-127


# ------------------------------------------------------------------------------------------------
# Attention sink (NEXT-2 reading)
# ------------------------------------------------------------------------------------------------

def test_attend_with_sink_is_softmax_with_a_zero_value_row():
    """A sink logit s is one more row whose logit is s (whatever q) and whose value is zero:
    checked against torch's scaled_dot_product_attention over the rows plus such a row, and
    against the limits s -> -inf (plain attention) and s -> +inf (output 0)."""
    rng = np.random.default_rng(31)
    H, D, R = 8, 64, 50
    q = rng.standard_normal((H, D))
    rows = rng.standard_normal((R, D))
    sink = rng.standard_normal(H) * 3
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attend_with_sink(q, rows, scale, sink)
    # per head, the sink row: key chosen so that scale * q_h . key = sink_h, value 0
    for h in range(H):
        key = q[h] * (sink[h] / (scale * (q[h] @ q[h])))
        k_all = torch.from_numpy(np.vstack([rows, key]))[None]
        v_all = torch.from_numpy(np.vstack([rows, np.zeros(D)]))[None]
        ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q[h:h + 1])[None], k_all, v_all,
                                                               scale=scale)[0, 0].numpy()
        assert np.allclose(o[h], ref, rtol=1e-12, atol=1e-12)
        logits = np.append(scale * rows @ q[h], sink[h])
        assert np.isclose(lse[h], scipy.special.logsumexp(logits), rtol=1e-13)
    o0, lse0 = oracle.attend(q, rows, scale)
    o1, _ = oracle.attend_with_sink(q, rows, scale, np.full(H, -1e300))
    assert np.allclose(o1, o0, rtol=0, atol=1e-15)
    o2, _ = oracle.attend_with_sink(q, rows, scale, np.full(H, 1e4))
    assert np.all(np.abs(o2) < 1e-300)
