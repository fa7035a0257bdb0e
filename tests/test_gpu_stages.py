"""Stage-level parity of the CUDA path with the oracle (compression, indexer + top-k, attention).

Each stage is fed seeded inputs; attention is fed the oracle's own quantised rows so that its
comparison isolates the attention arithmetic.  Top-k index sets and counts are compared
bit-exactly, indexer scores bit-exactly, stored rows to within one storage ulp, attention
outputs within max-abs 3e-2 / rel-L2 1e-2.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import *  # noqa: F401,F403
from harness import DEV

lcsa = pytest.importorskip("long_context_sparse_24_b300")
from long_context_sparse_24_b300 import buffers  # noqa: E402

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------------------- generator

def test_gpu_generator_matches_numpy():
    import synth.gpu as sg
    sg.build()
    out = torch.empty(70001, dtype=torch.bfloat16, device=DEV)
    sg.normal_bf16(out, 5, 77, 12345)
    ref = synth.normal_bf16(5, 77, 12345, 70001)
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref)
    pk = torch.empty(4099, dtype=torch.uint8, device=DEV)
    sg.e2m1_packed(pk, 6, 78, 1000)
    assert np.array_equal(pk.cpu().numpy(), synth.pack_e2m1(synth.e2m1_codes(6, 78, 1000, 8198)))
    sc = torch.empty(5000, dtype=torch.uint8, device=DEV)
    sg.ue8m0(sc, 7, 79, 3)
    assert np.array_equal(sc.cpu().numpy(), synth.ue8m0_scales(7, 79, 3, 5000))


# ---------------------------------------------------------------------------------------- compression

def _score_rows_np(seed, seq, n, dim):
    """Per-channel score rows of a sequence's raw tokens (bf16 bit patterns [n, dim], N(0,1))."""
    return synth.normal_bf16(seed, synth.tensor_id(synth.COMP_SCORES, 0, seq), 0, n * dim, None).reshape(n, dim)


def _per_channel_bias(seed, dim, m, overlap):
    nb = 2 * m if overlap else m
    return bits_to_f64(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B, 1), 0, nb * dim)).reshape(nb, dim) * 0.5


def _compress_run(lengths, chunk_plan, m, overlap, dim, fmt, seed=21, block_order_seed=None, per_channel=False):
    """Compress len(lengths) sequences fed in calls: chunk_plan[c][b] new tokens of seq b in call c.
    per_channel: score rows per token (a per-channel compressor) instead of the scalar weights."""
    S = len(lengths)
    fmtc = buffers.row_format_code(fmt)
    cap = max(lengths) + 256
    bps = math.ceil(cap / 128)
    order = None
    if block_order_seed is not None:
        order = np.random.default_rng(block_order_seed).permutation(S * bps).tolist()
    new_cap = max(sum(c) for c in chunk_plan)
    cache = buffers.alloc_layer(S, cap, dim, fmtc, m, overlap, new_cap, DEV, block_order=order,
                                per_channel=per_channel)
    w, bias = compressor_params(seed, 0, dim, m, overlap)
    if per_channel:
        bias = _per_channel_bias(seed, dim, m, overlap)
    comp = lcsa.Compressor(to_dev_f32(w), to_dev_f32(bias), m, overlap)
    raws = [raw_rows_gpu(seed, 0, b, lengths[b], dim) for b in range(S)]
    scs = [to_dev_bf16_bits(_score_rows_np(seed, b, lengths[b], dim)) for b in range(S)] if per_channel else None
    st = dev_status()
    pos = [0] * S
    for call in chunk_plan:
        after = [pos[b] + call[b] for b in range(S)]
        batch = buffers.make_batch(after, call, DEV, max_seq_len=cap)
        parts = [raws[b][pos[b]:after[b]] for b in range(S)]
        raw = torch.cat(parts).contiguous() if batch.total_new else torch.empty((1, dim), dtype=torch.bfloat16, device=DEV)
        if per_channel:
            sc = (torch.cat([scs[b][pos[b]:after[b]] for b in range(S)]).contiguous() if batch.total_new
                  else torch.empty((1, dim), dtype=torch.bfloat16, device=DEV))
            lcsa.csa_compress(batch, raw, comp, cache.state, cache.entries, cache.paging, st, scores=sc)
        else:
            fn = lcsa.csa_compress if overlap or m < 128 else lcsa.hca_compress
            fn(batch, raw, comp, cache.state, cache.entries, cache.paging, st)
        lcsa.lcs_window_commit(batch, cache.state, st)
        pos = after
    torch.cuda.synchronize()
    assert_status_ok(st)
    assert pos == list(lengths)
    return cache, w, bias


@pytest.mark.parametrize("m,overlap,dim,fmt", [(4, True, 512, "fp8_split"), (4, True, 128, "bf16"),
                                               (128, False, 512, "fp8_split"), (1, False, 128, "fp8_split"),
                                               (8, True, 128, "fp8_split"), (2, False, 512, "fp8_split")])
def test_compress_matches_oracle(m, overlap, dim, fmt):
    lengths = [1, 3, 300, 517] if m < 128 else [100, 300, 1100]
    cache, w, bias = _compress_run(lengths, [lengths], m, overlap, dim, fmt, block_order_seed=3)
    for b, L in enumerate(lengths):
        raw = bits_to_f64(raw_rows_np(21, 0, b, L, dim))
        nf = L // m
        if nf:
            orc = oracle.quantize_rows(oracle.compress_blocked(raw, w, bias, m, overlap), fmt)
            gpu = read_rows(cache.entries, entry_rows_of(cache, b, range(nf)))
            compare_quantized(gpu, orc, f"entries seq {b}")
        # window ring: the last min(L,128) raw rows, quantised bit-exactly like the oracle
        ps = np.arange(max(0, L - 128), L)
        gw = read_rows(cache.state.window, b * 128 + ps % 128)
        ow = oracle.quantize_rows(raw[ps], fmt)
        for key in ("bf16", "nope", "rope", "scale"):
            if key in ow:
                assert np.array_equal(gw[key], ow[key]), f"window {key} seq {b}"
        # pending ring holds the rows a future entry still needs
        slots = cache.state.pending_slots
        full = L // m
        keep_lo = max(0, (full - 1) * m if overlap else full * m)
        pend = cache.state.pending[b].view(torch.int16).cpu().numpy().view(np.uint16)
        rb = raw_rows_np(21, 0, b, L, dim)
        for p in range(keep_lo, L):
            assert np.array_equal(pend[p % slots], rb[p])


@pytest.mark.parametrize("m,overlap", [(4, True), (128, False)])
def test_compress_incremental_equals_one_shot(m, overlap):
    # decode-time appends (one token per call, ragged chunks) give the same bits as one prefill call
    lengths = [263, 517, 130] if m == 4 else [300, 520, 129]
    rng = np.random.default_rng(5)
    plan, left = [], list(lengths)
    while any(left):
        call = []
        for b in range(3):
            c = min(left[b], int(rng.choice([0, 1, 1, 1, 3, 17, 64])))
            call.append(c)
            left[b] -= c
        plan.append(call)
    dim = 512
    one, _, _ = _compress_run(lengths, [lengths], m, overlap, dim, "fp8_split")
    inc, _, _ = _compress_run(lengths, plan, m, overlap, dim, "fp8_split")
    for b, L in enumerate(lengths):
        rows = entry_rows_of(one, b, range(L // m))
        a, c = read_rows(one.entries, rows), read_rows(inc.entries, rows)
        for key in ("nope", "rope", "scale"):
            assert np.array_equal(a[key], c[key]), (b, key)
    for key in ("nope", "rope", "scale"):
        assert torch.equal(getattr(one.state.window, key), getattr(inc.state.window, key))


@pytest.mark.parametrize("m,overlap,dim,fmt", [(4, True, 512, "fp8_split"), (4, True, 128, "bf16"),
                                               (2, False, 512, "fp8_split"), (1, False, 128, "fp8_split")])
def test_compress_per_channel_matches_oracle(m, overlap, dim, fmt):
    """The per-channel reading (a score row per token, softmax per channel) against the oracle."""
    lengths = [1, 3, 300, 517]
    cache, _, _ = _compress_run(lengths, [lengths], m, overlap, dim, fmt, block_order_seed=4, per_channel=True)
    bias = _per_channel_bias(21, dim, m, overlap)
    for b, L in enumerate(lengths):
        nf = L // m
        if not nf:
            continue
        raw = bits_to_f64(raw_rows_np(21, 0, b, L, dim))
        sc = bits_to_f64(_score_rows_np(21, b, L, dim))
        orc = oracle.quantize_rows(oracle.compress_per_channel(raw, sc, bias, m, overlap), fmt)
        gpu = read_rows(cache.entries, entry_rows_of(cache, b, range(nf)))
        compare_quantized(gpu, orc, f"per-channel entries seq {b}")


def test_compress_per_channel_incremental_equals_one_shot():
    # the pending score rows carry the overlapping block across calls: same bits as one call
    lengths = [263, 517, 130]
    rng = np.random.default_rng(6)
    plan, left = [], list(lengths)
    while any(left):
        call = []
        for b in range(3):
            c = min(left[b], int(rng.choice([0, 1, 1, 1, 3, 17, 64])))
            call.append(c)
            left[b] -= c
        plan.append(call)
    one, _, _ = _compress_run(lengths, [lengths], 4, True, 512, "fp8_split", per_channel=True)
    inc, _, _ = _compress_run(lengths, plan, 4, True, 512, "fp8_split", per_channel=True)
    for b, L in enumerate(lengths):
        rows = entry_rows_of(one, b, range(L // 4))
        a, c = read_rows(one.entries, rows), read_rows(inc.entries, rows)
        for key in ("nope", "rope", "scale"):
            assert np.array_equal(a[key], c[key]), (b, key)


# ---------------------------------------------------------------------------------------- indexer

def _index_case(lengths, new, m, k, heads, rank, relu, scaled, seed=31, ties=False):
    S = len(lengths)
    cap = max(lengths) + 128
    order = np.random.default_rng(seed).permutation(S * math.ceil(cap / 128)).tolist()
    cache = buffers.alloc_layer(S, cap, 512, lcsa.LCS_ROW_FP8_SPLIT, m, True, 0, DEV, index_rank=rank,
                                block_order=order)
    batch = buffers.make_batch(lengths, new, DEV, max_seq_len=cap)
    kcs, kss, qcs, qss, hws = [], [], [], [], []
    for b in range(S):
        ne = lengths[b] // m
        kc, ks = index_inputs(seed, 0, b, ne, rank, scaled)
        if ties:
            kc[:] = kc[:1]
            ks[:] = ks[:1]
        rows = entry_rows_of(cache, b, range(ne))
        if ne:
            cache.keys.fp4[torch.as_tensor(rows, device=DEV)] = u8(synth.pack_e2m1(kc))
            cache.keys.scale[torch.as_tensor(rows, device=DEV)] = u8(ks)
        qc, qs, hw = query_index_inputs(seed, 0, b, lengths[b] - new[b], new[b], heads, rank, scaled)
        kcs.append(kc); kss.append(ks); qcs.append(qc); qss.append(qs); hws.append(hw)
    qc_all = np.concatenate(qcs)
    q_fp4 = u8(synth.pack_e2m1(qc_all))
    q_sc = u8(np.concatenate(qss))
    hw_all = to_dev_f32(np.concatenate(hws))
    return cache, batch, kcs, kss, qcs, qss, hws, q_fp4, q_sc, hw_all


@pytest.mark.parametrize("heads,rank,relu,scaled,new,lengths", [
    # up to 4 queries per sequence at rank 128: tensor-core (tcgen05) scorer
    (4, 128, False, True, [1, 1, 1], [37, 600, 2100]),
    (4, 128, True, True, [1, 1, 1], [37, 600, 2100]),
    (4, 128, False, True, [1, 1, 1], [5, 9000, 4100]),
    (4, 128, False, True, [2, 1, 4], [37, 600, 2100]),
    (1, 128, False, True, [4, 1, 3], [37, 600, 2100]),
    (2, 128, True, True, [3, 4, 1], [37, 600, 2100]),
    (8, 128, False, True, [1, 1, 1], [37, 600, 2100]),
    (8, 128, False, True, [2, 1, 2], [300, 4600, 2100]),
    # longer runs of queries at rank 128: up to 16 per sequence, the fused scorer in groups of up
    # to 4 queries; beyond, the tensor-core prefill scorer (groups of 16 queries, 8 at Hi = 8;
    # ragged last groups; causal limits inside a tile; runs of 256 tiles) and the select kernel
    (4, 128, False, True, [1, 5, 40], [37, 600, 2100]),
    (2, 128, True, True, [2, 1, 9], [37, 600, 2100]),
    (4, 128, False, True, [17, 40, 33], [600, 2100, 5000]),
    (4, 128, True, True, [16, 5, 48], [300, 2100, 4100]),
    (1, 128, False, True, [33, 6, 70], [300, 2100, 4100]),
    (8, 128, False, True, [9, 20, 5], [37, 600, 2100]),
    (8, 128, True, True, [3, 24, 7], [37, 600, 2100]),
    (4, 128, False, True, [5, 21], [600, 140000]),
    (4, 128, False, True, [5, 12], [600, 140000]),
    # long sequences: 14 to 27 tiles per CTA, so that the stage, block-scale and accumulator rings
    # all wrap several times under random scores
    (4, 128, False, True, [1, 3], [600000, 1000000]),
    (2, 128, True, True, [1, 1], [1000000, 300000]),
    # rank 64: warp-MMA scorer
    (1, 64, False, False, [1, 7, 33], [37, 600, 2100]),
    (8, 64, False, True, [1, 3, 17], [37, 600, 2100]),
])
def test_index_scores_exact_and_topk_sets(heads, rank, relu, scaled, new, lengths):
    m, k = 4, 24
    cache, batch, kcs, kss, qcs, qss, hws, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, heads, rank, relu, scaled)
    flags = lcsa.LCS_INDEX_RELU if relu else 0
    T = batch.total_new
    ld = (max(lengths) + 128) // m
    scores = torch.full((T, ld), float("nan"), device=DEV)
    st = dev_status()
    lcsa.csa_index_scores(batch, q_fp4, q_sc, hw, heads, cache.keys, cache.paging, m, flags, scores, ld, st)
    out_idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    out_cnt = torch.full((T,), -7, dtype=torch.int32, device=DEV)
    wsb = lcsa.lcs_index_topk_workspace(batch, heads, cache.keys, cache.paging, m, k)
    ws = workspace(wsb)
    lcsa.csa_index_topk(batch, q_fp4, q_sc, hw, heads, cache.keys, cache.paging, m, k, flags, out_idx, out_cnt,
                        ws, wsb, st)
    torch.cuda.synchronize()
    assert_status_ok(st)
    sc = scores.cpu().numpy(); oi = out_idx.cpu().numpy(); oc = out_cnt.cpu().numpy()
    qi = 0
    for b in range(len(lengths)):
        ref = oracle.index_scores(qcs[b], qss[b], hws[b], kcs[b], kss[b], relu)
        for i in range(new[b]):
            t = lengths[b] - new[b] + i
            n = oracle.visible_entries(t, m)
            assert np.array_equal(sc[qi, :n].astype(np.float64), ref[i, :n]), f"scores seq {b} query {i}"
            sel = oracle.topk_select(ref[i, :n], k)
            assert oc[qi] == len(sel)
            assert np.array_equal(oi[qi, :len(sel)], sel), f"top-k seq {b} query {i}"
            assert np.all(oi[qi, len(sel):] == -1)
            qi += 1
    # the scoring and selection phases as two calls give the same bits
    idx2 = torch.full((T, k), -9, dtype=torch.int32, device=DEV)
    cnt2 = torch.full((T,), -9, dtype=torch.int32, device=DEV)
    ws2 = workspace(wsb)
    lcsa.csa_index_topk(batch, q_fp4, q_sc, hw, heads, cache.keys, cache.paging, m, k,
                        flags | lcsa.LCS_INDEX_SCORE_ONLY, None, None, ws2, wsb, st)
    lcsa.csa_index_topk(batch, q_fp4, q_sc, hw, heads, cache.keys, cache.paging, m, k,
                        flags | lcsa.LCS_INDEX_SELECT_ONLY, idx2, cnt2, ws2, wsb, st)
    torch.cuda.synchronize()
    assert_status_ok(st)
    assert np.array_equal(idx2.cpu().numpy(), oi) and np.array_equal(cnt2.cpu().numpy(), oc)


def test_topk_ties_take_lowest_index():
    m, k = 4, 24
    lengths, new = [400, 1000], [1, 2]
    cache, batch, *_, q_fp4, q_sc, hw = _index_case(lengths, new, m, k, 4, 128, False, True, ties=True)
    out_idx = torch.empty((batch.total_new, k), dtype=torch.int32, device=DEV)
    out_cnt = torch.empty((batch.total_new,), dtype=torch.int32, device=DEV)
    wsb = lcsa.lcs_index_topk_workspace(batch, 4, cache.keys, cache.paging, m, k)
    lcsa.csa_index_topk(batch, q_fp4, q_sc, hw, 4, cache.keys, cache.paging, m, k, 0, out_idx, out_cnt,
                        workspace(wsb), wsb)
    torch.cuda.synchronize()
    assert np.array_equal(out_idx.cpu().numpy(), np.tile(np.arange(k), (batch.total_new, 1)))


# ---------------------------------------------------------------------------------------- attention

def _attend_case(kind, lengths, new, heads, dim, fmt, m, k, seed=41, scale=None, split=False, sink=None,
                 corrupt_seq=None, rows_hook=None, skip_seq=None, expect_status=None, separate_v=False,
                 sink_fused=False):
    """Fill an entry cache / window ring / new rows with oracle-quantised rows and run one call.
    corrupt_seq: unmap that sequence's first cache block before the call (host-side corruption of
    the block table); the call must then report LCS_ERR_DEVICE_GUARD and every other sequence must
    still match the oracle.  rows_hook(b, entry_rows): may change a sequence's entry rows (fp64)
    before they are quantised.  separate_v: value rows of their own (entries, window ring and new
    rows numbered like the key rows, drawn from other streams) passed as `values`.  sink: per-head
    sink logits, applied by lcs_attention_sink after the call, or with sink_fused by the attention
    call itself.  expect_status: the device status the call must report (outputs
    are not checked when it is LCS_ERR_TIMEOUT); skip_seq: a sequence whose outputs are not
    checked."""
    S = len(lengths)
    fmtc = buffers.row_format_code(fmt)
    cap = max(lengths) + 128
    order = np.random.default_rng(seed).permutation(S * math.ceil(cap / 128)).tolist()
    T = sum(new)
    cache = buffers.alloc_layer(S, cap, dim, fmtc, m, kind == "csa", T, DEV, block_order=order)
    batch = buffers.make_batch(lengths, new, DEV, max_seq_len=cap)
    rng = np.random.default_rng(seed)
    ent_deq, win_deq, sels, qs = [], [], [], []
    vals, vent_deq, vwin_deq = None, [], []
    if separate_v:
        vals = lcsa.Values(buffers.alloc_rows(fmtc, dim, cache.entries.num_rows, DEV),
                           buffers.alloc_rows(fmtc, dim, cache.state.window.num_rows, DEV),
                           buffers.alloc_rows(fmtc, dim, cache.state.new_rows.num_rows, DEV)
                           if cache.state.new_rows is not None else None)
        vrng = np.random.default_rng(seed + 1)
    for b in range(S):
        L, q_n = lengths[b], new[b]
        n0 = L - q_n
        ne = L // m
        ent_f = rng.standard_normal((max(ne, 1), dim))
        if rows_hook is not None:
            ent_f = rows_hook(b, ent_f)
        ent = oracle.quantize_rows(ent_f, fmt)
        if ne:
            sub = {kk: v[:ne] for kk, v in ent.items() if kk != "format"}
            sub["format"] = ent["format"]
            write_rows(cache.entries, entry_rows_of(cache, b, range(ne)), sub)
        ent_deq.append(ent["deq"][:ne])
        # raw rows of the last 128 + new positions
        p_lo = max(0, n0 - 128)
        raw = bits_to_f64(raw_rows_np(seed, 0, b, L - p_lo, dim, start=p_lo))
        wq = oracle.quantize_rows(raw, fmt)
        wd = np.zeros((L, dim)); wd[p_lo:L] = wq["deq"]
        win_deq.append(wd)
        ring_pos = np.arange(p_lo, n0)
        if ring_pos.size:
            sub = {kk: v[:n0 - p_lo] for kk, v in wq.items() if kk not in ("format", "deq")}
            sub["format"] = wq["format"]
            write_rows(cache.state.window, b * 128 + ring_pos % 128, sub)
        sub = {kk: v[n0 - p_lo:] for kk, v in wq.items() if kk not in ("format", "deq")}
        sub["format"] = wq["format"]
        q0 = sum(new[:b])
        if q_n:
            write_rows(cache.state.new_rows, np.arange(q0, q0 + q_n), sub)
        if separate_v:
            # value rows with the key rows' numbers: entries, ring and new rows
            vent = oracle.quantize_rows(vrng.standard_normal((max(ne, 1), dim)) * 3.0, fmt)
            if ne:
                sub = {kk: v[:ne] for kk, v in vent.items() if kk != "format"}
                sub["format"] = vent["format"]
                write_rows(vals.entries, entry_rows_of(cache, b, range(ne)), sub)
            vent_deq.append(vent["deq"][:ne])
            vq = oracle.quantize_rows(bits_to_f64(raw_rows_np(seed, 1, b, L - p_lo, dim, start=p_lo)), fmt)
            vd = np.zeros((L, dim)); vd[p_lo:L] = vq["deq"]
            vwin_deq.append(vd)
            if ring_pos.size:
                sub = {kk: v[:n0 - p_lo] for kk, v in vq.items() if kk not in ("format", "deq")}
                sub["format"] = vq["format"]
                write_rows(vals.window, b * 128 + ring_pos % 128, sub)
            if q_n:
                sub = {kk: v[n0 - p_lo:] for kk, v in vq.items() if kk not in ("format", "deq")}
                sub["format"] = vq["format"]
                write_rows(vals.new_rows, np.arange(q0, q0 + q_n), sub)
        for i in range(q_n):
            t = n0 + i
            n = oracle.visible_entries(t, m)
            if kind == "csa":
                s = np.sort(rng.choice(n, size=min(k, n), replace=False)) if n else np.zeros(0, np.int64)
                sels.append(s)
        qs.append(queries_np(seed, 0, b, n0, q_n, heads, dim))
    q_bits = np.concatenate(qs)
    q = to_dev_bf16_bits(q_bits)
    if corrupt_seq is not None:
        cache.paging.block_table[corrupt_seq, 0] = -1
    out = torch.empty((T, heads, dim), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, heads), dtype=torch.float32, device=DEV)
    scale = scale if scale is not None else 1 / math.sqrt(dim)
    st = dev_status()
    sink_dev = torch.from_numpy(sink.astype(np.float32)).to(DEV) if sink is not None else None
    fsink = sink_dev if sink_fused else None
    if kind == "csa":
        idx = np.full((T, k), -1, np.int32)
        for i, s in enumerate(sels):
            idx[i, :len(s)] = s
        idx_t = torch.from_numpy(idx).to(DEV)
        cnt_t = torch.tensor([len(s) for s in sels], dtype=torch.int32, device=DEV)
        wsb = lcsa.lcs_attend_workspace(batch, heads, dim, k + 128)
        if split:
            # window part on a second stream, then the top-k part with the merge
            ws = workspace(wsb)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            lcsa.csa_attend_window(batch, q, heads, k, m, cache.entries, cache.paging, cache.state, scale, ws, wsb,
                                   st, stream=side, values=vals)
            torch.cuda.current_stream().wait_stream(side)
            lcsa.csa_attend_topk(batch, q, heads, idx_t, cnt_t, k, m, cache.entries, cache.paging, cache.state,
                                 scale, out, lse, ws, wsb, st, values=vals, sink=fsink)
            # the one call plans the window rows into the entries' list (other splits, so other
            # rounding): it is checked against the oracle as well
            one_out = torch.empty_like(out)
            one_lse = torch.empty_like(lse)
            lcsa.csa_attend(batch, q, heads, idx_t, cnt_t, k, m, cache.entries, cache.paging, cache.state, scale,
                            one_out, one_lse, workspace(wsb), wsb, st, values=vals, sink=fsink)
        else:
            lcsa.csa_attend(batch, q, heads, idx_t, cnt_t, k, m, cache.entries, cache.paging, cache.state, scale, out,
                            lse, workspace(wsb), wsb, st, values=vals, sink=fsink)
    else:
        wsb = lcsa.lcs_attend_workspace(batch, heads, dim, cap // m + 128)
        lcsa.hca_attend(batch, q, heads, m, cache.entries, cache.paging, cache.state, scale, out, lse,
                        workspace(wsb), wsb, st, values=vals, sink=fsink)
    if sink is not None and not sink_fused:
        lcsa.lcs_attention_sink(out, lse, sink_dev)
        if kind == "csa" and split:
            lcsa.lcs_attention_sink(one_out, one_lse, sink_dev)
    torch.cuda.synchronize()
    want = expect_status if expect_status is not None else (6 if corrupt_seq is not None else 0)
    got = int(st.item())
    assert got == want, f"device status {got} ({lcsa.STATUS_NAMES.get(got)}), expected {lcsa.STATUS_NAMES[want]}"
    if want == 7:
        return
    if corrupt_seq is not None:
        skip_seq = corrupt_seq
    results = [(out, lse, "")] + ([(one_out, one_lse, " (one call)")] if kind == "csa" and split else [])
    qf = bits_to_f64(q_bits)
    for res_out, res_lse, tag in results:
        o = bf16_tensor_to_f64(res_out); l = res_lse.cpu().numpy()
        qi = 0
        for b in range(S):
            n0 = lengths[b] - new[b]
            if b == skip_seq:
                qi += new[b]
                continue
            for i in range(new[b]):
                t = n0 + i
                vrows = None
                if kind == "csa":
                    rows = oracle.csa_query_rows(t, sels[qi], ent_deq[b], win_deq[b])
                    if separate_v:
                        vrows = oracle.csa_query_rows(t, sels[qi], vent_deq[b], vwin_deq[b])
                else:
                    rows = oracle.hca_query_rows(t, m, ent_deq[b], win_deq[b])
                    if separate_v:
                        vrows = oracle.hca_query_rows(t, m, vent_deq[b], vwin_deq[b])
                if sink is None:
                    ro, rl = oracle.attend(qf[qi], rows, scale, values=vrows)
                else:
                    ro, rl = oracle.attend_with_sink(qf[qi], rows, scale, sink.astype(np.float32).astype(np.float64),
                                                     values=vrows)
                check_outputs(o[qi], ro, f"{kind} seq {b} query {i}{tag}")
                assert np.allclose(l[qi], rl, atol=2e-3, rtol=1e-4), f"lse seq {b} query {i}{tag}"
                qi += 1


@pytest.mark.parametrize("kind,lengths,new,heads,dim,fmt,m,k", [
    ("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512),       # decode, split-KV
    ("csa", [900, 2200], [40, 9], 64, 512, "fp8_split", 4, 64),                # prefill chunk
    ("csa", [3000], [3], 128, 512, "fp8_split", 4, 256),                       # 128 heads = 2 groups
    ("csa", [2000], [3], 96, 512, "fp8_split", 4, 256),                        # a partial head group
    ("csa", [5000, 2600], [300, 200], 128, 512, "fp8_split", 4, 512),          # prefill: one list per CTA
    ("hca", [3000], [200], 128, 512, "fp8_split", 128, 0),
    ("csa", [50, 700], [50, 20], 8, 128, "bf16", 4, 64),                       # small-model rows
    ("csa", [600], [5], 8, 128, "fp8_split", 4, 64),
    ("csa", [130, 7], [1, 7], 16, 512, "fp8_split", 4, 32),                    # N(t) < k, short seqs
    ("hca", [20000, 1500, 128], [1, 1, 1], 64, 512, "fp8_split", 128, 0),      # HCA decode
    ("hca", [3000], [17], 64, 512, "fp8_split", 128, 0),
    # many queries: several 128-row tiles per CTA (online softmax across tiles, O rescaled)
    ("hca", [40000 - 700 * i for i in range(40)], [1] * 40, 64, 512, "fp8_split", 128, 0),
    ("csa", [3000 + 37 * i for i in range(120)], [1] * 120, 64, 512, "fp8_split", 4, 1024),
])
def test_attend_matches_oracle(kind, lengths, new, heads, dim, fmt, m, k):
    _attend_case(kind, lengths, new, heads, dim, fmt, m, k)


@pytest.mark.parametrize("kind,lengths,new,heads,dim,fmt,m,k,split", [
    ("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512, False),   # decode
    ("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512, True),    # two calls
    ("csa", [900, 2200], [40, 9], 64, 512, "fp8_split", 4, 64, False),            # prefill chunk
    ("csa", [3000], [3], 96, 512, "fp8_split", 4, 256, False),                    # partial head group
    ("csa", [130, 7], [1, 7], 16, 512, "fp8_split", 4, 32, False),                # N(t) < k
    ("hca", [20000, 1500, 128], [1, 1, 1], 64, 512, "fp8_split", 128, 0, False),
    ("hca", [3000], [17], 128, 512, "fp8_split", 128, 0, False),
    ("csa", [50, 700], [50, 20], 8, 128, "bf16", 4, 64, False),
    ("csa", [600], [5], 8, 128, "fp8_split", 4, 64, False),
])
def test_attend_separate_values_matches_oracle(kind, lengths, new, heads, dim, fmt, m, k, split):
    """Separate value rows (a value set numbered like each key set) against the oracle's attention
    with values apart from keys."""
    _attend_case(kind, lengths, new, heads, dim, fmt, m, k, split=split, separate_v=True)


@pytest.mark.parametrize("kind,lengths,new,heads,dim,fmt,m,k,split", [
    ("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512, False),
    ("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512, True),   # window part apart
    ("csa", [900, 2200], [40, 9], 64, 512, "fp8_split", 4, 64, False),
    ("hca", [3000], [17], 64, 512, "fp8_split", 128, 0, False),
    ("csa", [50, 700], [50, 20], 8, 128, "bf16", 4, 64, False),
    # several tiles per CTA: lse from the online softmax across tiles
    ("hca", [40000 - 700 * i for i in range(40)], [1] * 40, 64, 512, "fp8_split", 128, 0, False),
    ("csa", [3000 + 37 * i for i in range(120)], [1] * 120, 64, 512, "fp8_split", 4, 1024, False),
])
@pytest.mark.parametrize("fused", [False, True])
def test_attention_sink_matches_oracle(kind, lengths, new, heads, dim, fmt, m, k, split, fused):
    """Per-head sink logits around the logits' range, applied by lcs_attention_sink after the
    attention or folded into the attention's own normalisation (single-split epilogues and the
    combine), against the oracle's softmax with the sink term (outputs and lse)."""
    sink = np.random.default_rng(7).standard_normal(heads) * 2.0
    _attend_case(kind, lengths, new, heads, dim, fmt, m, k, sink=sink, split=split, sink_fused=fused)


@pytest.mark.parametrize("kind,lengths,new,heads,dim,fmt,m,k", [
    ("csa", [2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 4, 512),
    ("hca", [3000], [17], 64, 512, "fp8_split", 128, 0),
    ("csa", [50, 700], [50, 20], 8, 128, "bf16", 4, 64),
])
def test_attention_sink_with_separate_values(kind, lengths, new, heads, dim, fmt, m, k):
    """The folded sink together with separate value rows (warp-MMA kernel), against the oracle."""
    sink = np.random.default_rng(8).standard_normal(heads) * 3.0
    _attend_case(kind, lengths, new, heads, dim, fmt, m, k, sink=sink, sink_fused=True, separate_v=True)


@pytest.mark.parametrize("lengths,new,heads,dim,fmt,k", [
    ([2000, 4100, 300], [1, 1, 1], 64, 512, "fp8_split", 512),     # decode: window part computed apart
    ([900, 2200], [40, 9], 64, 512, "fp8_split", 64),              # multi-token chunk, window from new rows
    ([130, 7], [1, 7], 16, 512, "fp8_split", 32),                  # short sequences, N(t) < k
    ([50, 700], [50, 20], 8, 128, "bf16", 64),                     # no separate window part: all in the top-k call
])
def test_attend_window_then_topk_and_one_call(lengths, new, heads, dim, fmt, k):
    _attend_case("csa", lengths, new, heads, dim, fmt, 4, k, split=True)


# ---------------------------------------------------------------------------------------- staging

def test_stage_copy_pinned_and_device():
    """lcs_stage_copy: pinned host -> device, device -> pinned host and device -> device in one
    launch, aligned and unaligned buffers, odd sizes; bytes equal."""
    g = torch.Generator().manual_seed(5)
    sizes = [2 * 1024 * 1024, 1000003, 17, 4096]
    host = [torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory() for n in sizes]
    dev = [torch.zeros(n + 1, dtype=torch.uint8, device=DEV) for n in sizes]
    pairs = [(dev[0][:sizes[0]], host[0]), (dev[1][1:], host[1]), (dev[2][:17], host[2]), (dev[3][:4096], host[3])]
    lcsa.lcs_stage_copy(pairs)
    torch.cuda.synchronize()
    for (d, h) in pairs:
        assert torch.equal(d.cpu(), h)
    back = [torch.zeros(n, dtype=torch.uint8).pin_memory() for n in sizes[:2]]
    other = torch.zeros(sizes[2], dtype=torch.uint8, device=DEV)
    lcsa.lcs_stage_copy([(back[0], dev[0][:sizes[0]]), (back[1], dev[1][1:]), (other, dev[2][:17])])
    torch.cuda.synchronize()
    assert torch.equal(back[0], host[0]) and torch.equal(back[1], host[1])
    assert torch.equal(other.cpu(), host[2])
    with pytest.raises(lcsa.LcsError):
        lcsa.lcs_stage_copy([(dev[2][:17], torch.zeros(17, dtype=torch.uint8))])   # pageable host memory


# ---------------------------------------------------------------------------------------- FP4 keys

@pytest.mark.parametrize("r", [128, 64, 160])
def test_quantize_e2m1_matches_oracle(r):
    """lcs_quantize_e2m1 against the oracle's block-scaled FP4: codes and scale bytes bit-exact,
    including exact ties, all-zero blocks, subnormal and near-maximum BF16 inputs."""
    rng = np.random.default_rng(21 + r)
    rows = 1500
    x = rng.standard_normal((rows, r)) * np.ldexp(1.0, rng.integers(-30, 30, size=(rows, 1)))
    x[0, :32] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2 + [-0.25, -0.75, -1.25, -1.75,
                                                                      -2.5, -3.5, -5.0, -6.0] * 2
    x[1, :32] = 0.0
    x[2, :32] = rng.standard_normal(32) * 1e-39          # BF16 subnormals
    x[3, :32] = np.clip(rng.standard_normal(32), -3.0, 3.0) * 1e38   # near the BF16 maximum
    x[4, :] = rng.integers(-7, 8, size=r) * 0.5          # values already on the E2M1 grid
    bits = synth.f32_to_bf16_bits(x.astype(np.float32))
    xv = synth.bf16_bits_to_f32(bits).astype(np.float64)
    codes, scales = oracle.e2m1_block_quantize(xv)
    xd = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    cd = torch.full((rows, r // 2), 0xAB, dtype=torch.uint8, device=DEV)
    sd = torch.full((rows, r // 32), 0xAB, dtype=torch.uint8, device=DEV)
    lcsa.lcs_quantize_e2m1(xd, cd, sd)
    torch.cuda.synchronize()
    assert np.array_equal(sd.cpu().numpy(), scales)
    assert np.array_equal(cd.cpu().numpy(), synth.pack_e2m1(codes))
