"""Oracle: a plain, slow fp64 CPU statement of the CSA / HCA hybrid compressed attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module.  The CUDA library never calls it, and it shares no
code with the CUDA library (the seeded inputs come from ``synth``, which holds no step of the
method).

Sources (the pages this restates; section names as printed on each page):

* x-techcon  -- m.x-techcon.com/article/133366, section "2. 核心技术创新：混合压缩注意力":
  CSA step 1 (every m=4 raw tokens -> one entry: learned per-token weight plus a positional
  bias, softmax-normalised, weighted sum, adjacent blocks overlap), step 2 (lightning indexer,
  low-rank relevance, per-query top-k, k=1024 Pro / 512 Flash), step 3 (sliding window of the
  most recent 128 uncompressed tokens attended together with the selected entries), the HCA
  paragraph (m'=128, no sparse selection, dense attention, shared-KV multi-query attention),
  the efficiency paragraph (RoPE dims BF16, the rest FP8, indexer QK path FP4), and section
  "4. 底层基础设施优化" (FP4 -> FP8 is lossless; state cache for the window and the tail;
  compressed cache in blocks of LCM(4,128) raw tokens).
* csdn       -- deepseek.csdn.net/69ef40b30a2f6a37c5a66073, "CSA" (4 tokens -> 1 block,
  1M tokens -> about 250K blocks), "HCA" (looks at all compressed blocks), "KV cache".
* digipub    -- digipub.cc "DeepSeek V4來了", section "把賬算在注意力機制上" (4 -> 1 entry,
  128 -> 1 entry, top-k sparse attention continuing V3.2's DSA).
* chenxutan  -- chenxutan.com/d/4230 "万字深度解析 DeepSeek V4", section 4.2 (C4A compressor
  sketch: overlapping 2*ratio state, softmax then weighted sum), 4.5 (RoPE dims = 64 in BF16,
  the rest FP8 E4M3) and 6.2 (FP4 E2M1 value set 0, 0.5, 1, 1.5, 2, 3, 4, 6).

Readings where the pages are silent or ambiguous (each one also listed in the design notes):

* compression score is a scalar per raw token: z_t = w . k_t + b[offset of t in the window];
* CSA entry j covers raw tokens [(j-1)m, (j+1)m) (two blocks, offsets 0..2m-1); HCA entry j
  covers [jm, (j+1)m); rows before token 0 do not exist and are left out of the softmax;
* an entry exists once its last token has arrived: a query at position t sees entries
  j < N(t) = floor((t+1)/m) and window tokens max(0, t-127) .. t (its own token included);
* the indexer score is sum_h w_h * phi(q_h . k) over per-32 block-scaled e2m1 values, phi the
  identity by default or ReLU by flag; top-k keeps the largest scores, ties to the lowest j,
  and takes all N(t) entries when N(t) <= k;
* shared KV: one row serves as key and value (an optional separate value row is supported);
* FP8 rows: scale s = fp32(amax)/448 over the non-RoPE dims (1 when amax = 0), code =
  E4M3 round-to-nearest-even, saturating to +-448, of fp32(x)/s; the 64 RoPE dims are BF16.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
invariants, special cases that reduce to library routines, the pages' printed values).  What
DeepSeek-V4 itself computes beyond these readings is not fixed by the pages.
"""
from __future__ import annotations

import numpy as np

WINDOW = 128          # x-techcon section 2, CSA step 3: the most recent 128 tokens
ROPE_DIMS = 64        # chenxutan section 4.5: rope_dim = 64
FP8_MAX = 448.0       # largest finite E4M3 magnitude (OCP 8-bit floating point, E4M3FN)


# ---------------------------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------------------------

def e2m1_value(codes: np.ndarray) -> np.ndarray:
    """Value of FP4 E2M1 codes: 1 sign, 2 exponent (bias 1), 1 mantissa bit.

    chenxutan section 6.2 prints the positive values 0, 0.5, 1, 1.5, 2, 3, 4, 6.
    """
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    mant = (c & 1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * mant, np.ldexp(1.0 + 0.5 * mant, (e - 1).astype(np.int64)))
    return sign * mag


def ue8m0_value(b: np.ndarray) -> np.ndarray:
    """UE8M0 block scale: 2**(b - 127)."""
    return np.ldexp(1.0, np.asarray(b).astype(np.int64) - 127)


def _round_to_grid(x: np.ndarray, mant_bits: int, min_exp: int) -> np.ndarray:
    """Round to a binary float grid with ``mant_bits`` fraction bits, ties to even.

    Spacing at |x| in [2**e, 2**(e+1)) is 2**(e - mant_bits); below 2**min_exp the spacing is
    fixed at 2**(min_exp - mant_bits) (subnormals).  x / spacing is exact (power of two) and
    numpy's round is round-half-to-even.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = f * 2**e, 0.5 <= |f| < 1
    e = np.maximum(e - 1, min_exp)
    spacing = np.ldexp(1.0, (e - mant_bits).astype(np.int64))
    return np.round(x / spacing) * spacing


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (8-bit significand, fp32 exponent range), ties to even."""
    return _round_to_grid(x, 7, -126)


def e4m3_round_satfinite(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (bias 7, 3 mantissa bits, subnormals below 2**-6),
    ties to even, saturating to +-448 (the format has no infinity)."""
    r = _round_to_grid(x, 3, -6)
    return np.clip(r, -FP8_MAX, FP8_MAX)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Byte code of values already on the E4M3 grid (|v| <= 448)."""
    v = np.asarray(v, dtype=np.float64)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    a = np.abs(v)
    code = np.zeros(v.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    code[sub] = np.round(a[sub] / 2.0 ** -9).astype(np.int64)
    _, e = np.frexp(a[~sub])
    e = e - 1
    mant = np.round((a[~sub] / np.ldexp(1.0, e) - 1.0) * 8).astype(np.int64)
    code[~sub] = ((e + 7) << 3) | mant
    return (code | (sign.astype(np.int64) << 7)).astype(np.uint8)


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    c = np.asarray(b).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    mant = (c & 7).astype(np.float64)
    mag = np.where(e == 0, mant * 2.0 ** -9, np.ldexp(1.0 + mant / 8.0, (e - 7).astype(np.int64)))
    return sign * mag


E2M1_MAX = 6.0       # largest E2M1 magnitude (chenxutan section 6.2)


def e2m1_block_quantize(x: np.ndarray, block: int = 32) -> tuple[np.ndarray, np.ndarray]:
    """Block-scaled FP4 of x [..., r] (r a multiple of ``block``): E2M1 codes [..., r] and UE8M0
    scale bytes [..., r/block].

    The pages fix the format (E2M1 values with a power-of-two scale per 32 elements, x-techcon
    section 4; latetalk: "blockwise scale") but not how the scale is chosen.  Reading taken:
    the smallest power of two 2**e with amax <= 6 * 2**e, so that no element saturates, with e
    clamped to the UE8M0 range [-127, 127] (all-zero blocks get e = -127); each element is
    x / 2**e rounded to the nearest E2M1 value, ties to the even code (the one whose mantissa
    bit is 0); a zero result is stored as +0 (code 0).
    """
    x = np.asarray(x, dtype=np.float64)
    shp = x.shape
    blocks = x.reshape(shp[:-1] + (shp[-1] // block, block))
    amax = np.abs(blocks).max(axis=-1)
    # smallest e with 6 * 2**e >= amax: start from frexp and correct by one step either way
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / E2M1_MAX)), -127.0)
    e = e.astype(np.int64)
    e = np.where(np.ldexp(E2M1_MAX, e - 1) >= amax, e - 1, e)
    e = np.where(np.ldexp(E2M1_MAX, e) < amax, e + 1, e)
    e = np.clip(e, -127, 127)
    v = blocks / np.ldexp(1.0, e)[..., None]
    r = np.clip(_round_to_grid(v, 1, 0), -E2M1_MAX, E2M1_MAX)
    mag = np.abs(r)
    table = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    codes = np.zeros(mag.shape, dtype=np.int64)
    for val, code in table.items():
        codes[mag == val] = code
    codes = np.where((r < 0) & (codes != 0), codes | 8, codes)
    return codes.reshape(shp).astype(np.uint8), (e + 127).astype(np.uint8)


def bf16_bits(v: np.ndarray) -> np.ndarray:
    """Bit pattern of values already on the bf16 grid."""
    return (np.asarray(v, dtype=np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------------------------
# Row storage format (x-techcon section 2 efficiency paragraph; chenxutan section 4.5)
# ---------------------------------------------------------------------------------------------

def quantize_rows(x: np.ndarray, row_format: str) -> dict:
    """Quantise rows [R, D] to the stored row format.

    ``bf16``: every dim rounded to bf16.  ``fp8_split``: dims [0, 64) (the RoPE slice) rounded to
    bf16; dims [64, D) stored as E4M3 codes with one fp32 scale per row.
    Returns the stored fields and ``deq``, the exact value of the stored row.
    """
    x = np.asarray(x, dtype=np.float64)
    if row_format == "bf16":
        deq = bf16_round(x)
        return {"format": "bf16", "bf16": bf16_bits(deq), "deq": deq}
    assert row_format == "fp8_split"
    rope = bf16_round(x[:, :ROPE_DIMS])
    nope32 = x[:, ROPE_DIMS:].astype(np.float32)
    amax = np.max(np.abs(nope32), axis=1)
    scale = np.where(amax > 0, amax / np.float32(FP8_MAX), np.float32(1.0)).astype(np.float32)
    y = (nope32 / scale[:, None]).astype(np.float32)
    q = e4m3_round_satfinite(y.astype(np.float64))
    deq = np.concatenate([rope, q * scale.astype(np.float64)[:, None]], axis=1)
    return {"format": "fp8_split", "rope": bf16_bits(rope), "nope": e4m3_encode(q),
            "scale": scale, "deq": deq}


def dequantize_rows(fields: dict) -> np.ndarray:
    if fields["format"] == "bf16":
        return (fields["bf16"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rope = (fields["rope"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nope = e4m3_decode(fields["nope"]) * fields["scale"].astype(np.float64)[:, None]
    return np.concatenate([rope, nope], axis=1)


# ---------------------------------------------------------------------------------------------
# Compression (x-techcon section 2 CSA step 1 and the HCA paragraph; chenxutan section 4.2)
# ---------------------------------------------------------------------------------------------

def num_entries(n: int, m: int) -> int:
    """Complete entries of a sequence of n raw tokens: floor(n/m).  The n mod m tail stays in
    the state cache (x-techcon section 4, KV cache management)."""
    return n // m


def visible_entries(t: int, m: int) -> int:
    """Entries a query at absolute position t may use: N(t) = floor((t+1)/m)."""
    return (t + 1) // m


def entry_span(j: int, m: int, overlap: bool) -> tuple[int, int]:
    """Raw-token range [lo, hi) entry j is made from; lo may be negative (missing rows)."""
    return ((j - 1) * m if overlap else j * m), (j + 1) * m


def compression_weights(z: np.ndarray) -> np.ndarray:
    """Softmax over the window's rows."""
    a = np.exp(z - np.max(z))
    return a / np.sum(a)


def compress(raw: np.ndarray, w: np.ndarray, bias: np.ndarray, m: int, overlap: bool,
             first: int = 0, count: int | None = None, return_weights: bool = False):
    """Compressed entries ``first .. first+count-1`` of a raw sequence [n, D] (fp64).

    For entry j with window rows t in [lo, hi) clipped at 0: z_t = w . k_t + b[t - lo],
    alpha = softmax(z) over the existing rows, c_j = sum_t alpha_t k_t.
    ``bias`` has 2m entries (overlapping CSA windows) or m entries (HCA).
    """
    raw = np.asarray(raw, dtype=np.float64)
    n = raw.shape[0]
    total = num_entries(n, m)
    if count is None:
        count = total - first
    assert 0 <= first and first + count <= total
    assert bias.shape[0] == (2 * m if overlap else m)
    out = np.empty((count, raw.shape[1]), dtype=np.float64)
    weights = []
    for i, j in enumerate(range(first, first + count)):
        lo, hi = entry_span(j, m, overlap)
        t = np.arange(max(lo, 0), hi)
        z = raw[t] @ w + bias[t - lo]
        a = compression_weights(z)
        out[i] = a @ raw[t]
        if return_weights:
            weights.append(a)
    return (out, weights) if return_weights else out


def compress_per_channel(raw: np.ndarray, scores: np.ndarray, bias: np.ndarray, m: int, overlap: bool,
                         first: int = 0, count: int | None = None, return_weights: bool = False):
    """Entries ``first .. first+count-1`` with per-channel weights (the variant reading).

    chenxutan section 4.2 sketches the compressor with a score vector per raw token (one score per
    channel, from its own projection), a softmax over the window's tokens taken channel by
    channel, and a channel-by-channel weighted sum; x-techcon section 2 adds a positional bias,
    here one per window offset and channel.  For entry j with window rows t in [lo, hi) clipped at
    0: z[t, d] = scores[t, d] + bias[t - lo, d]; alpha[:, d] = softmax over the existing rows of
    z[:, d]; c[d] = sum_t alpha[t, d] raw[t, d].  ``scores`` [n, D] are the already projected score
    rows; ``bias`` is [2m, D] (overlapping windows) or [m, D].
    """
    raw = np.asarray(raw, dtype=np.float64)
    scores = np.asarray(scores, dtype=np.float64)
    n = raw.shape[0]
    total = num_entries(n, m)
    if count is None:
        count = total - first
    assert 0 <= first and first + count <= total and scores.shape == raw.shape
    assert bias.shape == ((2 * m if overlap else m), raw.shape[1])
    out = np.empty((count, raw.shape[1]), dtype=np.float64)
    weights = []
    for i, j in enumerate(range(first, first + count)):
        lo, hi = entry_span(j, m, overlap)
        t = np.arange(max(lo, 0), hi)
        z = scores[t] + bias[t - lo]                       # [rows, D]
        a = np.exp(z - z.max(axis=0, keepdims=True))
        a = a / a.sum(axis=0, keepdims=True)               # softmax over the rows, per channel
        out[i] = (a * raw[t]).sum(axis=0)
        if return_weights:
            weights.append(a)
    return (out, weights) if return_weights else out


def compress_blocked(raw: np.ndarray, w: np.ndarray, bias: np.ndarray, m: int, overlap: bool,
                     first: int = 0, count: int | None = None) -> np.ndarray:
    """The same entries as ``compress``, evaluated a block of m rows at a time (for long
    sequences).  Entry 0 of an overlapping compressor has only its second block."""
    raw = np.asarray(raw, dtype=np.float64)
    n, d = raw.shape
    total = num_entries(n, m)
    if count is None:
        count = total - first
    out = np.empty((count, d), dtype=np.float64)
    if count == 0:
        return out
    j0 = first
    if overlap and first == 0:
        out[0] = compress(raw[:m], w, bias, m, overlap, 0, 1)[0]
        j0 = 1
    js = np.arange(j0, first + count)
    if js.size:
        lo = (js[0] - 1) * m if overlap else js[0] * m
        hi = (js[-1] + 1) * m
        blocks = raw[lo:hi].reshape(-1, m, d)                    # blocks lo/m .. hi/m-1
        zb = blocks @ w                                         # [nb, m]
        if overlap:
            z = np.concatenate([zb[:-1], zb[1:]], axis=1) + bias  # [count', 2m]
            rows = np.concatenate([blocks[:-1], blocks[1:]], axis=1)
        else:
            z = zb + bias
            rows = blocks
        a = np.exp(z - z.max(axis=1, keepdims=True))
        a /= a.sum(axis=1, keepdims=True)
        out[j0 - first:] = np.einsum("jr,jrd->jd", a, rows)
    return out


# ---------------------------------------------------------------------------------------------
# Lightning indexer and top-k (x-techcon section 2 CSA step 2 and section 4 FP4 QAT;
# digipub "把賬算在注意力機制上")
# ---------------------------------------------------------------------------------------------

def blockscaled_values(codes: np.ndarray, scales: np.ndarray, block: int = 32) -> np.ndarray:
    """e2m1 codes [..., r] times their per-32 UE8M0 scales [..., r/32] (exact in fp64)."""
    v = e2m1_value(codes)
    s = np.repeat(ue8m0_value(scales), block, axis=-1)
    return v * s


def index_scores(q_codes: np.ndarray, q_scales: np.ndarray, head_w: np.ndarray | None,
                 k_codes: np.ndarray, k_scales: np.ndarray, relu: bool = False) -> np.ndarray:
    """score[t, j] = sum_h w[t,h] * phi(qhat[t,h,:] . khat[j,:]).

    q_codes [T, Hi, r], q_scales [T, Hi, r/32], head_w [T, Hi] (None: all ones),
    k_codes [N, r], k_scales [N, r/32].  Every product is a multiple of 2**-4 for the
    generator's ranges and every sum stays far below 2**53, so fp64 is exact here.
    """
    qv = blockscaled_values(q_codes, q_scales)
    kv = blockscaled_values(k_codes, k_scales)
    per_head = np.einsum("thr,nr->thn", qv, kv)
    if relu:
        per_head = np.maximum(per_head, 0.0)
    if head_w is None:
        head_w = np.ones(per_head.shape[:2])
    return np.einsum("th,thn->tn", np.asarray(head_w, dtype=np.float64), per_head)


def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores (ties: lower index first), returned in ascending order.
    All indices when len(scores) <= k."""
    n = scores.shape[0]
    if n <= k:
        return np.arange(n, dtype=np.int64)
    order = np.lexsort((np.arange(n), -scores))    # primary: score desc, secondary: index asc
    return np.sort(order[:k])


# ---------------------------------------------------------------------------------------------
# Attention (x-techcon section 2: CSA step 3 and the HCA paragraph)
# ---------------------------------------------------------------------------------------------

def window_positions(t: int, window: int = WINDOW) -> np.ndarray:
    return np.arange(max(0, t - window + 1), t + 1)


def attend(q: np.ndarray, keys: np.ndarray, softmax_scale: float, values: np.ndarray | None = None):
    """Multi-query attention of all heads q [H, D] over one shared set of rows [R, D]:
    one softmax per head over all rows.  Returns (o [H, Dv] fp64, lse [H] fp64)."""
    values = keys if values is None else values
    logits = softmax_scale * (np.asarray(q, np.float64) @ np.asarray(keys, np.float64).T)
    mx = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - mx)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ np.asarray(values, np.float64)) / l
    return o, (mx + np.log(l))[:, 0]


def attend_with_sink(q: np.ndarray, keys: np.ndarray, softmax_scale: float, sink: np.ndarray,
                     values: np.ndarray | None = None):
    """``attend`` with a per-head sink logit sink[H]: one more softmax term per head that takes
    probability mass but carries no value (o = sum_r p_r v_r / (sum_r p_r + exp(sink))).

    The csdn attention-details table names an attention sink without defining it; this is the
    common definition of a learned per-head sink logit (a reading from outside the pages)."""
    values = keys if values is None else values
    logits = softmax_scale * (np.asarray(q, np.float64) @ np.asarray(keys, np.float64).T)
    sink = np.asarray(sink, np.float64)[:, None]
    mx = np.maximum(logits.max(axis=1, keepdims=True), sink)
    p = np.exp(logits - mx)
    l = p.sum(axis=1, keepdims=True) + np.exp(sink - mx)
    o = (p @ np.asarray(values, np.float64)) / l
    return o, (mx + np.log(l))[:, 0]


def csa_query_rows(t: int, selected: np.ndarray, entries: np.ndarray, window_rows: np.ndarray,
                   window: int = WINDOW):
    """Rows one CSA query attends to: the selected entries, then its window rows.
    ``window_rows`` is indexed by absolute token position."""
    return np.concatenate([entries[selected], window_rows[window_positions(t, window)]], axis=0)


def hca_query_rows(t: int, m: int, entries: np.ndarray, window_rows: np.ndarray, window: int = WINDOW):
    """Rows one HCA query attends to: every visible entry, then its window rows."""
    return np.concatenate([entries[:visible_entries(t, m)], window_rows[window_positions(t, window)]],
                          axis=0)


# ---------------------------------------------------------------------------------------------
# One sequence through a whole layer
# ---------------------------------------------------------------------------------------------

def csa_layer(raw, w, bias, m, overlap, row_format, q, q_pos, idx_q_codes, idx_q_scales, head_w,
              idx_k_codes, idx_k_scales, top_k, softmax_scale, relu=False):
    """CSA for the queries at positions q_pos of one sequence of raw rows [n, D].

    Returns a dict with the quantised entries, the top-k index lists, outputs (fp64 and bf16)
    and lse.  idx_k_* cover at least floor(n/m) entries.
    """
    n = raw.shape[0]
    entries = compress_blocked(raw, w, bias, m, overlap)
    ent_q = quantize_rows(entries, row_format)
    win_q = quantize_rows(raw, row_format)
    n_ent = entries.shape[0]
    scores = index_scores(idx_q_codes, idx_q_scales, head_w,
                          idx_k_codes[:n_ent], idx_k_scales[:n_ent], relu)
    sel, outs, lses = [], [], []
    for i, t in enumerate(q_pos):
        nt = visible_entries(int(t), m)
        s = topk_select(scores[i, :nt], top_k)
        rows = csa_query_rows(int(t), s, ent_q["deq"], win_q["deq"])
        o, lse = attend(q[i], rows, softmax_scale)
        sel.append(s); outs.append(o); lses.append(lse)
    o = np.stack(outs)
    return {"entries": ent_q, "window": win_q, "topk": sel, "scores": scores,
            "o": o, "o_bf16": bf16_round(o), "lse": np.stack(lses)}


def hca_layer(raw, w, bias, m, row_format, q, q_pos, softmax_scale):
    entries = compress_blocked(raw, w, bias, m, False)
    ent_q = quantize_rows(entries, row_format)
    win_q = quantize_rows(raw, row_format)
    outs, lses = [], []
    for i, t in enumerate(q_pos):
        rows = hca_query_rows(int(t), m, ent_q["deq"], win_q["deq"])
        o, lse = attend(q[i], rows, softmax_scale)
        outs.append(o); lses.append(lse)
    o = np.stack(outs)
    return {"entries": ent_q, "window": win_q, "o": o, "o_bf16": bf16_round(o), "lse": np.stack(lses)}


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def kv_bytes_per_token(dim: int = 512, rope: int = ROPE_DIMS, index_rank: int = 128) -> dict:
    """Stored bytes per raw token and layer for the row format (x-techcon section 2 efficiency
    paragraph) with scalar fp32 FP8 scales, FP4 indexer keys with UE8M0 per-32 scales."""
    row = rope * 2 + (dim - rope) + 4
    idx = index_rank // 2 + index_rank // 32
    return {"row": row, "csa": row / 4 + idx / 4, "hca": row / 128, "index_key": idx}

