"""End-to-end parity on the five synthetic workloads, through the layer driver (compress ->
indexer top-k -> attention -> window commit) against the fp64 oracle.

Small workload: every query is checked.  Large workloads run at their full sizes on the GPU
and are checked on sampled sequences / queries that the oracle computes one by one (the
entries they need are compressed by the oracle from the raw rows of their own spans).
Top-k index sets and counts: bit-exact.  Outputs: max-abs 3e-2 / rel-L2 1e-2.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.gpu as sg
from harness import DEV, OUT_MAX_ABS, OUT_REL_L2, bits_to_f64, check_outputs, to_dev_bf16_bits

lcsa = pytest.importorskip("long_context_sparse_24_b300")
from long_context_sparse_24_b300.layer import Layer  # noqa: E402

pytestmark = pytest.mark.gpu


def _comp_params(seed, layer, dim, m, overlap):
    wscale = np.float32(1 / 16 if dim >= 512 else 1 / 8)
    w = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_W, layer), 0, dim)) * wscale
    nb = 2 * m if overlap else m
    b = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B, layer), 0, nb)) * np.float32(0.5)
    return w.astype(np.float32), b.astype(np.float32)


def _raw_f64(seed, layer, seq, t0, n, dim):
    return bits_to_f64(synth.normal_bf16(seed, synth.tensor_id(synth.RAW, layer, seq), t0 * dim, n * dim)).reshape(n, dim)


def _fill_keys(layer_obj, seed, lay, seq, n_ent, rank, scaled=True):
    """Indexer keys of entries 0..n_ent-1 of one sequence (identity paging) on the device."""
    if n_ent <= 0:
        return
    bps = layer_obj.cache.paging.max_blocks_per_seq
    epb = layer_obj.cache.paging.entries_per_block
    table = layer_obj.cache.paging.block_table[seq].cpu().numpy()
    assert np.array_equal(table, np.arange(seq * bps, (seq + 1) * bps))
    r0 = seq * bps * epb
    sg.e2m1_packed(layer_obj.cache.keys.fp4[r0:r0 + n_ent], seed, synth.tensor_id(synth.IDX_K, lay, seq), 0)
    if scaled:
        sg.ue8m0(layer_obj.cache.keys.scale[r0:r0 + n_ent], seed, synth.tensor_id(synth.IDX_KS, lay, seq), 0)


def _keys_np(seed, lay, seq, n_ent, rank, scaled=True):
    kc = synth.e2m1_codes(seed, synth.tensor_id(synth.IDX_K, lay, seq), 0, n_ent * rank).reshape(n_ent, rank)
    if scaled:
        ks = synth.ue8m0_scales(seed, synth.tensor_id(synth.IDX_KS, lay, seq), 0, n_ent * rank // 32)
        ks = ks.reshape(n_ent, rank // 32)
    else:
        ks = np.full((n_ent, rank // 32), 127, np.uint8)
    return kc, ks


def _query_inputs(seed, lay, seq, t0, n, heads, dim, hi, rank, scaled=True, q_scale_bits=None):
    q = synth.normal_bf16(seed, synth.tensor_id(synth.QUERY, lay, seq), t0 * heads * dim, n * heads * dim, q_scale_bits)
    q = q.reshape(n, heads, dim)
    qc = synth.e2m1_codes(seed, synth.tensor_id(synth.IDX_Q, lay, seq), t0 * hi * rank, n * hi * rank)
    qc = qc.reshape(n, hi, rank)
    if scaled:
        qs = synth.ue8m0_scales(seed, synth.tensor_id(synth.IDX_QS, lay, seq), t0 * hi * rank // 32,
                                n * hi * rank // 32).reshape(n, hi, rank // 32)
        hw = synth.head_weights(seed, synth.tensor_id(synth.HEAD_W, lay, seq), t0 * hi, n * hi).reshape(n, hi)
    else:
        qs = np.full((n, hi, rank // 32), 127, np.uint8)
        hw = np.ones((n, hi), np.float32)
    return q, qc, qs, hw


def _dev_u8(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8)).to(DEV)


# ------------------------------------------------------------------------------------------ small

@pytest.mark.parametrize("fmt", ["bf16", "fp8_split"])
def test_csa_tiny_prefill_then_decode(fmt):
    """4096-token sequence, 8 heads, D=128, indexer rank 64 (1 head, unscaled), k=64: prefill of
    all 4096 tokens (every query checked), then 64 decode steps (every step checked)."""
    wl = synth.CONFIGS["csa_tiny"]
    seed, D, H, m, k, r, hi = wl.seed, wl.dim, wl.heads, wl.m, wl.top_k, wl.index_rank, wl.index_heads
    n, steps = wl.new_tokens, 64
    fmtc = lcsa.LCS_ROW_BF16 if fmt == "bf16" else lcsa.LCS_ROW_FP8_SPLIT
    lay = Layer("csa", 1, n + steps + 128, H, D, fmtc, m, top_k=k, index_heads=hi, index_rank=r, max_new=n,
                softmax_scale=1.0, device=DEV)
    w, b = _comp_params(seed, 0, D, m, True)
    lay.set_compressor(torch.from_numpy(w).to(DEV), torch.from_numpy(b).to(DEV))
    total = n + steps
    raw = _raw_f64(seed, 0, 0, 0, total, D)
    raw_dev = to_dev_bf16_bits(synth.normal_bf16(seed, synth.tensor_id(synth.RAW, 0, 0), 0, total * D).reshape(total, D))
    _fill_keys(lay, seed, 0, 0, total // m, r, scaled=False)
    kc, ks = _keys_np(seed, 0, 0, total // m, r, scaled=False)
    q, qc, qs, hw = _query_inputs(seed, 0, 0, 0, total, H, D, hi, r, scaled=False,
                                  q_scale_bits=synth.INV_SQRT128_BITS)
    ref = oracle.csa_layer(raw, w.astype(np.float64), b.astype(np.float64), m, True, fmt,
                           bits_to_f64(q), np.arange(total), qc, qs, hw, kc, ks, k, 1.0)
    # prefill: all n tokens in one call
    out = torch.empty((n, H, D), dtype=torch.bfloat16, device=DEV)
    batch = lay.batch([n], [n])
    lay.step(batch, raw_dev[:n], to_dev_bf16_bits(q[:n]), out, idx_q_fp4=_dev_u8(synth.pack_e2m1(qc[:n])),
             idx_q_scale=_dev_u8(qs[:n]), head_w=torch.from_numpy(hw[:n]).to(DEV))
    torch.cuda.synchronize()
    assert int(lay.status.item()) == 0
    got_idx = lay.topk_idx[:n].cpu().numpy()
    got_cnt = lay.topk_cnt[:n].cpu().numpy()
    o = out.float().cpu().numpy().astype(np.float64)
    for t in range(n):
        sel = ref["topk"][t]
        assert got_cnt[t] == len(sel), t
        assert np.array_equal(got_idx[t, :len(sel)], sel), t
    check_outputs(o, ref["o"][:n], "prefill")
    # decode: one token per call
    out1 = torch.empty((1, H, D), dtype=torch.bfloat16, device=DEV)
    for s in range(steps):
        t = n + s
        batch = lay.batch([t + 1], [1])
        lay.step(batch, raw_dev[t:t + 1], to_dev_bf16_bits(q[t:t + 1]), out1,
                 idx_q_fp4=_dev_u8(synth.pack_e2m1(qc[t:t + 1])), idx_q_scale=_dev_u8(qs[t:t + 1]),
                 head_w=torch.from_numpy(hw[t:t + 1]).to(DEV))
        torch.cuda.synchronize()
        sel = ref["topk"][t]
        assert np.array_equal(lay.topk_idx[0, :len(sel)].cpu().numpy(), sel), t
        check_outputs(out1.float().cpu().numpy()[0].astype(np.float64), ref["o"][t], f"decode step {s}")
    assert int(lay.status.item()) == 0


def test_hybrid_stack_ragged_decode_matches_oracle():
    """A CSA layer and an HCA layer on one shared, permuted block table (blocks of 128 raw
    tokens), ragged sequences, two decode steps through HybridStack; every sequence's output of
    every layer against the oracle, top-k sets bit-exact."""
    from long_context_sparse_24_b300 import buffers
    from long_context_sparse_24_b300.model import HybridStack
    seed, D, H, k, hi, r = 23, 512, 64, 64, 4, 128
    lengths = [900, 2600, 259]
    S, steps = len(lengths), 2
    cap = max(lengths) + steps + 128
    order = np.random.default_rng(seed).permutation(S * math.ceil(cap / 128)).tolist()
    stack = HybridStack(2, S, cap, H, D, lcsa.LCS_ROW_FP8_SPLIT, top_k=k, index_heads=hi, index_rank=r,
                        block_order=order, device=DEV)
    assert stack.kinds == ["csa", "hca"]
    params = []
    for li, lay in enumerate(stack.layers):
        w, b = _comp_params(seed, li, D, lay.m, lay.overlap)
        lay.set_compressor(torch.from_numpy(w).to(DEV), torch.from_numpy(b).to(DEV))
        params.append((w.astype(np.float64), b.astype(np.float64)))
        raws = []
        for s_, L in enumerate(lengths):
            t = torch.empty((L, D), dtype=torch.bfloat16, device=DEV)
            sg.normal_bf16(t, seed, synth.tensor_id(synth.RAW, li, s_), 0)
            raws.append(t)
        lay.fill(lay.batch(lengths, lengths), torch.cat(raws).contiguous())
    # indexer keys of the CSA layer through the shared block table
    csa = stack.layers[0]
    table = csa.cache.paging.block_table.cpu().numpy()
    keys = []
    for s_, L in enumerate(lengths):
        ne = (L + steps) // 4
        kc, ks = _keys_np(seed, 0, s_, ne, r)
        rows = table[s_, np.arange(ne) // 32].astype(np.int64) * 32 + np.arange(ne) % 32
        ridx = torch.as_tensor(rows, device=DEV)
        csa.cache.keys.fp4[ridx] = _dev_u8(synth.pack_e2m1(kc))
        csa.cache.keys.scale[ridx] = _dev_u8(ks)
        keys.append((kc, ks))
    for st in range(steps):
        pos = [L + st for L in lengths]
        raw_new, q_in, outs, iq, iqs, ihw, qref = [], [], [], [], [], [], []
        for li, lay in enumerate(stack.layers):
            rn = torch.empty((S, D), dtype=torch.bfloat16, device=DEV)
            for s_ in range(S):
                sg.normal_bf16(rn[s_], seed, synth.tensor_id(synth.RAW, li, s_), pos[s_] * D)
            raw_new.append(rn)
            qs_, qcs, qss, hws = [], [], [], []
            for s_ in range(S):
                q, qc, qsc, hw = _query_inputs(seed, li, s_, pos[s_], 1, H, D, hi, r)
                qs_.append(q); qcs.append(qc); qss.append(qsc); hws.append(hw)
            qb = np.concatenate(qs_)
            qref.append((qb, qcs, qss, hws))
            q_in.append(to_dev_bf16_bits(qb))
            outs.append(torch.empty((S, H, D), dtype=torch.bfloat16, device=DEV))
            if lay.kind == "csa":
                iq.append(_dev_u8(synth.pack_e2m1(np.concatenate(qcs))))
                iqs.append(_dev_u8(np.concatenate(qss)))
                ihw.append(torch.from_numpy(np.concatenate(hws)).to(DEV))
            else:
                iq.append(None); iqs.append(None); ihw.append(None)
        batch = stack.batch([p + 1 for p in pos], [1] * S)
        stack.step(batch, raw_new, q_in, outs, iq, iqs, ihw)
        torch.cuda.synchronize()
        assert stack.status == [0, 0]
        for li, lay in enumerate(stack.layers):
            o = outs[li].float().cpu().numpy().astype(np.float64)
            w, b = params[li]
            qb, qcs, qss, hws = qref[li]
            for s_ in range(S):
                raw = _raw_f64(seed, li, s_, 0, pos[s_] + 1, D)
                qf = bits_to_f64(qb[s_:s_ + 1])
                if lay.kind == "csa":
                    kc, ks = keys[s_]
                    ref = oracle.csa_layer(raw, w, b, 4, True, "fp8_split", qf, [pos[s_]], qcs[s_], qss[s_], hws[s_],
                                           kc, ks, k, 1 / math.sqrt(D))
                    n_sel = len(ref["topk"][0])
                    assert np.array_equal(lay.topk_idx[s_, :n_sel].cpu().numpy(), ref["topk"][0]), (st, s_)
                else:
                    ref = oracle.hca_layer(raw, w, b, 128, "fp8_split", qf, [pos[s_]], 1 / math.sqrt(D))
                check_outputs(o[s_], ref["o"][0], f"step {st} layer {li} seq {s_}")


# ------------------------------------------------------------------------------------------ large
#
# Full-size workloads, one step each in the layer driver's launch configuration.  The device
# inputs come from the seeded generator's CUDA build (spot-checked against its numpy build);
# the oracle recomputes the sampled queries from the numpy generator: their top-k over every
# visible entry, the selected entries compressed from their own raw spans, the window rows.

def _entries_from_spans(seed, lay, seq, js, m, overlap, w, b, dim):
    """Oracle entries js (fp64, before quantisation), each compressed from its own raw span."""
    out = np.empty((len(js), dim))
    for i, j in enumerate(js):
        j = int(j)
        if overlap and j > 0:
            raw = _raw_f64(seed, lay, seq, (j - 1) * m, 2 * m, dim)
            out[i] = oracle.compress(raw, w, b, m, True, 1, 1)[0]
        else:
            raw = _raw_f64(seed, lay, seq, j * m, m, dim)
            out[i] = oracle.compress(raw, w, b, m, overlap, 0, 1)[0]
    return out


def _fill_context(lay, seed, li, lengths, dim, chunk=16384):
    raw_chunk = torch.empty((len(lengths) * chunk, dim), dtype=torch.bfloat16, device=DEV)
    for c0 in range(0, max(lengths), chunk):
        ns = [max(0, min(chunk, L - c0)) for L in lengths]
        off = 0
        for s_, n in enumerate(ns):
            if n:
                sg.normal_bf16(raw_chunk[off:off + n], seed, synth.tensor_id(synth.RAW, li, s_), c0 * dim)
                off += n
        lay.fill(lay.batch([min(L, c0 + n) if n else L for L, n in zip(lengths, ns)], ns), raw_chunk[:off])
    del raw_chunk


def _check_csa_query(lay, seed, s_, t, row, q_np, qc, qs, hw, w, b, out_row, label, li=0):
    m, k, D = lay.m, lay.top_k, lay.dim
    n = oracle.visible_entries(t, m)
    kc, ks = _keys_np(seed, li, s_, n, lay.index_rank)
    sel = oracle.topk_select(oracle.index_scores(qc, qs, hw, kc, ks)[0, :n], k)
    assert int(lay.topk_cnt[row].item()) == len(sel), label
    assert np.array_equal(lay.topk_idx[row, :len(sel)].cpu().numpy(), sel), label
    ent = oracle.quantize_rows(_entries_from_spans(seed, li, s_, sel, m, True, w, b, D), "fp8_split")["deq"]
    lo = max(0, t - 127)
    win = oracle.quantize_rows(_raw_f64(seed, li, s_, lo, t + 1 - lo, D), "fp8_split")["deq"]
    o, _ = oracle.attend(bits_to_f64(q_np), np.concatenate([ent, win]), lay.scale)
    check_outputs(out_row, o, label)


def test_csa_decode_32x128k_full_size_sampled():
    """32 sequences x 131,072 cached tokens, 64 heads, D=512, k=512: one decode step; sequences
    0, 13 and 31 checked against the oracle (top-k bit-exact, outputs)."""
    _csa_decode_full_size_sampled("csa_decode", (0, 13, 31))


def test_csa_decode_32x1m_full_size_sampled():
    """32 sequences x 1,048,576 cached tokens, 64 heads, D=512, k=1024 (the 1M-context decode
    workload): one decode step in the layer driver's launch configuration, where each of the fused
    scorer's runs cuts its candidate buffer during the scan and the query's last CTA merges nine
    run lists; sequences 0, 17 and 31 checked against the oracle (top-k over 262,144 entries
    bit-exact, outputs)."""
    _csa_decode_full_size_sampled("csa_decode_1m", (0, 17, 31))


def _csa_decode_full_size_sampled(name, sampled):
    wl = synth.CONFIGS[name]
    seed, S, L, H, D, m, k, hi, r = wl.seed, wl.num_seqs, wl.ctx_len, wl.heads, wl.dim, wl.m, wl.top_k, \
        wl.index_heads, wl.index_rank
    lay = Layer("csa", S, L + 256, H, D, lcsa.LCS_ROW_FP8_SPLIT, m, top_k=k, index_heads=hi, index_rank=r,
                max_new=1, device=DEV)
    w, b = _comp_params(seed, 0, D, m, True)
    lay.set_compressor(torch.from_numpy(w).to(DEV), torch.from_numpy(b).to(DEV))
    _fill_context(lay, seed, 0, [L] * S, D)
    for s_ in range(S):
        _fill_keys(lay, seed, 0, s_, (L + 1) // m, r)
    ins = [_query_inputs(seed, 0, s_, L, 1, H, D, hi, r) for s_ in range(S)]
    raw_new = torch.empty((S, D), dtype=torch.bfloat16, device=DEV)
    for s_ in range(S):
        sg.normal_bf16(raw_new[s_], seed, synth.tensor_id(synth.RAW, 0, s_), L * D)
    q_dev = to_dev_bf16_bits(np.concatenate([x[0] for x in ins]))
    out = torch.empty((S, H, D), dtype=torch.bfloat16, device=DEV)
    lay.step(lay.batch([L + 1] * S, [1] * S), raw_new, q_dev, out,
             idx_q_fp4=_dev_u8(synth.pack_e2m1(np.concatenate([x[1] for x in ins]))),
             idx_q_scale=_dev_u8(np.concatenate([x[2] for x in ins])),
             head_w=torch.from_numpy(np.concatenate([x[3] for x in ins])).to(DEV))
    torch.cuda.synchronize()
    assert int(lay.status.item()) == 0
    o = out.float().cpu().numpy().astype(np.float64)
    w64, b64 = w.astype(np.float64), b.astype(np.float64)
    for s_ in sampled:
        q, qc, qs, hw = ins[s_]
        _check_csa_query(lay, seed, s_, L, s_, q[0], qc, qs, hw, w64, b64, o[s_], f"{name} seq {s_}")
    del lay, out
    torch.cuda.empty_cache()


def test_csa_prefill_1m_plus_16k_full_size_sampled():
    """One sequence, 1,048,576 cached tokens + a 16,384-token chunk, 128 heads, D=512, k=1024:
    one prefill step; queries 0, 1, 4099, 9000 and 16383 of the chunk checked against the
    oracle (top-k over all visible entries bit-exact, outputs)."""
    wl = synth.CONFIGS["csa_prefill"]
    seed, L, T, H, D, m, k, hi, r = wl.seed, wl.ctx_len, wl.new_tokens, wl.heads, wl.dim, wl.m, wl.top_k, \
        wl.index_heads, wl.index_rank
    lay = Layer("csa", 1, L + T + 256, H, D, lcsa.LCS_ROW_FP8_SPLIT, m, top_k=k, index_heads=hi, index_rank=r,
                max_new=T, device=DEV)
    w, b = _comp_params(seed, 0, D, m, True)
    lay.set_compressor(torch.from_numpy(w).to(DEV), torch.from_numpy(b).to(DEV))
    _fill_context(lay, seed, 0, [L], D, chunk=65536)
    _fill_keys(lay, seed, 0, 0, (L + T) // m, r)
    raw_new = torch.empty((T, D), dtype=torch.bfloat16, device=DEV)
    sg.normal_bf16(raw_new, seed, synth.tensor_id(synth.RAW, 0, 0), L * D)
    q_dev = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    sg.normal_bf16(q_dev, seed, synth.tensor_id(synth.QUERY, 0, 0), L * H * D)
    iq = torch.empty((T, hi, r // 2), dtype=torch.uint8, device=DEV)
    sg.e2m1_packed(iq, seed, synth.tensor_id(synth.IDX_Q, 0, 0), L * hi * r)
    iqs = torch.empty((T, hi, r // 32), dtype=torch.uint8, device=DEV)
    sg.ue8m0(iqs, seed, synth.tensor_id(synth.IDX_QS, 0, 0), L * hi * r // 32)
    hw = synth.head_weights(seed, synth.tensor_id(synth.HEAD_W, 0, 0), L * hi, T * hi).reshape(T, hi)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    lay.step(lay.batch([L + T], [T]), raw_new, q_dev, out, idx_q_fp4=iq, idx_q_scale=iqs,
             head_w=torch.from_numpy(np.ascontiguousarray(hw)).to(DEV))
    torch.cuda.synchronize()
    assert int(lay.status.item()) == 0
    # the device-side generator agrees with the numpy one on the sampled queries' inputs
    w64, b64 = w.astype(np.float64), b.astype(np.float64)
    for i in (0, 1, 4099, 9000, T - 1):
        q, qc, qs, hw_i = _query_inputs(seed, 0, 0, L + i, 1, H, D, hi, r)
        assert np.array_equal(q_dev[i].view(torch.int16).cpu().numpy().view(np.uint16), q[0]), i
        assert np.array_equal(iq[i].cpu().numpy(), synth.pack_e2m1(qc[0])), i
        assert np.array_equal(hw[i], hw_i[0]), i
        _check_csa_query(lay, seed, 0, L + i, i, q[0], qc, qs, hw_i, w64, b64,
                         out[i].float().cpu().numpy().astype(np.float64), f"query {i}")
    del lay, out, q_dev
    torch.cuda.empty_cache()


def test_hca_decode_64x1m_full_size_sampled():
    """64 sequences x 1,048,576 cached tokens, 64 heads, D=512: one decode step; sequences 0
    and 63 checked against dense oracle attention over all 8,192 entries + the window."""
    wl = synth.CONFIGS["hca_decode"]
    seed, S, L, H, D, m = wl.seed, wl.num_seqs, wl.ctx_len, wl.heads, wl.dim, wl.m
    lay = Layer("hca", S, L + 256, H, D, lcsa.LCS_ROW_FP8_SPLIT, m, max_new=1, device=DEV)
    w, b = _comp_params(seed, 0, D, m, False)
    lay.set_compressor(torch.from_numpy(w).to(DEV), torch.from_numpy(b).to(DEV))
    _fill_context(lay, seed, 0, [L] * S, D, chunk=8192)
    raw_new = torch.empty((S, D), dtype=torch.bfloat16, device=DEV)
    for s_ in range(S):
        sg.normal_bf16(raw_new[s_], seed, synth.tensor_id(synth.RAW, 0, s_), L * D)
    qs_np = [synth.normal_bf16(seed, synth.tensor_id(synth.QUERY, 0, s_), L * H * D, H * D).reshape(H, D)
             for s_ in range(S)]
    out = torch.empty((S, H, D), dtype=torch.bfloat16, device=DEV)
    lay.step(lay.batch([L + 1] * S, [1] * S), raw_new, to_dev_bf16_bits(np.stack(qs_np)), out)
    torch.cuda.synchronize()
    assert int(lay.status.item()) == 0
    o = out.float().cpu().numpy().astype(np.float64)
    w64, b64 = w.astype(np.float64), b.astype(np.float64)
    for s_ in (0, S - 1):
        ref = _hca_dense_ref(seed, 0, s_, L, m, D, w64, b64, bits_to_f64(qs_np[s_]), lay.scale)
        check_outputs(o[s_], ref, f"seq {s_}")
    del lay, out
    torch.cuda.empty_cache()


def _hca_dense_ref(seed, li, s_, t, m, D, w64, b64, q64, scale, chunk=65536):
    """Oracle HCA output of the query at position t: every entry compressed from the sequence's
    raw rows (drawn by the device-side generator in chunks, spot-checked against numpy), then
    the window rows."""
    n = oracle.visible_entries(t, m)
    ent = np.empty((n, D))
    raw_dev = torch.empty((chunk, D), dtype=torch.bfloat16, device=DEV)
    for c0 in range(0, n * m, chunk):
        sg.normal_bf16(raw_dev, seed, synth.tensor_id(synth.RAW, li, s_), c0 * D)
        bits = raw_dev.view(torch.int16).cpu().numpy().view(np.uint16)
        if c0 in (0, 7 * chunk):
            ref_bits = synth.normal_bf16(seed, synth.tensor_id(synth.RAW, li, s_), c0 * D, 8 * D).reshape(8, D)
            assert np.array_equal(bits[:8], ref_bits)
        rows = min(chunk, n * m - c0)
        ent[c0 // m:(c0 + rows) // m] = oracle.compress_blocked(bits_to_f64(bits[:rows]), w64, b64, m, False)
    ent_q = oracle.quantize_rows(ent, "fp8_split")["deq"]
    lo = max(0, t - 127)
    win = oracle.quantize_rows(_raw_f64(seed, li, s_, lo, t + 1 - lo, D), "fp8_split")["deq"]
    ref, _ = oracle.attend(q64, np.concatenate([ent_q, win]), scale)
    return ref


def test_mixed_decode_16x8_layers_full_size_sampled():
    """16 sequences of log-uniform lengths in [4096, 1M), 8 layers alternating CSA (k = 1024) and
    HCA on one shared block table, one decode step through HybridStack; the longest and the
    shortest sequence checked on every layer (CSA: top-k bit-exact, output; HCA: output against a
    dense oracle over every entry)."""
    from long_context_sparse_24_b300.model import HybridStack
    wl = synth.CONFIGS["mixed_decode"]
    seed, S, H, D, k, hi, r = wl.seed, wl.num_seqs, wl.heads, wl.dim, wl.top_k, wl.index_heads, wl.index_rank
    lengths = [int(x) for x in synth.mixed_lengths(seed, S)]
    cap = max(lengths) + 256
    stack = HybridStack(wl.layers, S, cap, H, D, lcsa.LCS_ROW_FP8_SPLIT, top_k=k, index_heads=hi, index_rank=r,
                        device=DEV)
    params = []
    for li, lay in enumerate(stack.layers):
        w, b = _comp_params(seed, li, D, lay.m, lay.overlap)
        lay.set_compressor(torch.from_numpy(w).to(DEV), torch.from_numpy(b).to(DEV))
        params.append((w.astype(np.float64), b.astype(np.float64)))
        _fill_context(lay, seed, li, lengths, D, chunk=8192)
        if lay.kind == "csa":
            for s_ in range(S):
                _fill_keys(lay, seed, li, s_, (lengths[s_] + 1) // 4, r)
    raw_new, q_in, outs, iq, iqs, ihw, ins = [], [], [], [], [], [], []
    for li, lay in enumerate(stack.layers):
        rn = torch.empty((S, D), dtype=torch.bfloat16, device=DEV)
        for s_ in range(S):
            sg.normal_bf16(rn[s_], seed, synth.tensor_id(synth.RAW, li, s_), lengths[s_] * D)
        raw_new.append(rn)
        x = [_query_inputs(seed, li, s_, lengths[s_], 1, H, D, hi, r) for s_ in range(S)]
        ins.append(x)
        q_in.append(to_dev_bf16_bits(np.concatenate([v[0] for v in x])))
        outs.append(torch.empty((S, H, D), dtype=torch.bfloat16, device=DEV))
        if lay.kind == "csa":
            iq.append(_dev_u8(synth.pack_e2m1(np.concatenate([v[1] for v in x]))))
            iqs.append(_dev_u8(np.concatenate([v[2] for v in x])))
            ihw.append(torch.from_numpy(np.concatenate([v[3] for v in x])).to(DEV))
        else:
            iq.append(None); iqs.append(None); ihw.append(None)
    stack.step(stack.batch([L + 1 for L in lengths], [1] * S), raw_new, q_in, outs, iq, iqs, ihw)
    torch.cuda.synchronize()
    assert stack.status == [0] * wl.layers
    picks = (int(np.argmax(lengths)), int(np.argmin(lengths)))
    for li in range(wl.layers):
        lay = stack.layers[li]
        o = outs[li].float().cpu().numpy().astype(np.float64)
        w64, b64 = params[li]
        for s_ in picks:
            q, qc, qs, hw = ins[li][s_]
            if lay.kind == "csa":
                _check_csa_query(lay, seed, s_, lengths[s_], s_, q[0], qc, qs, hw, w64, b64, o[s_],
                                 f"layer {li} seq {s_}", li=li)
            else:
                ref = _hca_dense_ref(seed, li, s_, lengths[s_], lay.m, D, w64, b64, bits_to_f64(q[0]), lay.scale)
                check_outputs(o[s_], ref, f"layer {li} seq {s_}")
    del stack, outs
    torch.cuda.empty_cache()
