"""Test-side helpers: build seeded inputs, run the library through its binding, read results back,
and compare with the oracle.  Imports the oracle (allowed in tests only)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth
import long_context_sparse_24_b300 as lcsa
from long_context_sparse_24_b300 import buffers

DEV = "cuda"
OUT_MAX_ABS = 3e-2      # bf16 attention outputs vs the fp64 oracle
OUT_REL_L2 = 1e-2


def raw_rows_np(seed: int, layer: int, seq: int, n: int, dim: int, start: int = 0) -> np.ndarray:
    """bf16 bit patterns [n, dim] of raw tokens start .. start+n-1."""
    tid = synth.tensor_id(synth.RAW, layer, seq)
    return synth.normal_bf16(seed, tid, start * dim, n * dim).reshape(n, dim)


def raw_rows_gpu(seed: int, layer: int, seq: int, n: int, dim: int, start: int = 0) -> torch.Tensor:
    import synth.gpu as sg
    out = torch.empty((n, dim), dtype=torch.bfloat16, device=DEV)
    sg.normal_bf16(out, seed, synth.tensor_id(synth.RAW, layer, seq), start * dim)
    return out


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def compressor_params(seed: int, layer: int, dim: int, m: int, overlap: bool):
    """w ~ N(0,1)/16 for D=512 (1/8 for D=128), bias ~ N(0,1)/2, as fp32 (exact values)."""
    wscale = 1 / 16 if dim >= 512 else 1 / 8
    w = bits_to_f64(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_W, layer), 0, dim)) * wscale
    nb = 2 * m if overlap else m
    b = bits_to_f64(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B, layer), 0, nb)) * 0.5
    return w, b


def to_dev_f32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)


def to_dev_bf16_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def read_rows(rows: lcsa.RowSet, idx) -> dict:
    """Fetch rows (by physical row index) back to the host in the oracle's field layout."""
    idx_t = torch.as_tensor(np.asarray(idx, dtype=np.int64), device=DEV)
    if rows.format == lcsa.LCS_ROW_BF16:
        b = rows.nope.index_select(0, idx_t).view(torch.int16).cpu().numpy().view(np.uint16)
        return {"format": "bf16", "bf16": b}
    nope = rows.nope.index_select(0, idx_t).cpu().numpy()
    rope = rows.rope.index_select(0, idx_t).view(torch.int16).cpu().numpy().view(np.uint16)
    scale = rows.scale.index_select(0, idx_t).cpu().numpy()
    return {"format": "fp8_split", "nope": nope, "rope": rope, "scale": scale}


def write_rows(rows: lcsa.RowSet, idx, fields: dict) -> None:
    idx_t = torch.as_tensor(np.asarray(idx, dtype=np.int64), device=DEV)
    if rows.format == lcsa.LCS_ROW_BF16:
        rows.nope.index_copy_(0, idx_t, to_dev_bf16_bits(fields["bf16"]))
        return
    rows.nope.index_copy_(0, idx_t, torch.from_numpy(np.ascontiguousarray(fields["nope"])).to(DEV))
    rows.rope.index_copy_(0, idx_t, to_dev_bf16_bits(fields["rope"]))
    rows.scale.index_copy_(0, idx_t, torch.from_numpy(np.ascontiguousarray(fields["scale"], dtype=np.float32)).to(DEV))


def entry_rows_of(cache: buffers.LayerCache, seq: int, js) -> np.ndarray:
    table = cache.paging.block_table.cpu().numpy()
    epb = cache.paging.entries_per_block
    js = np.asarray(js, dtype=np.int64)
    return table[seq, js // epb].astype(np.int64) * epb + js % epb


def compare_quantized(gpu: dict, orc: dict, what: str, max_mismatch_frac: float = 1e-3) -> None:
    """GPU-quantised rows vs oracle-quantised rows of the same fp64 values: the GPU computes in
    fp32, so a code may land one step away where the value sits on a rounding boundary."""
    g = oracle.dequantize_rows(gpu)
    o = orc["deq"]
    if gpu["format"] == "bf16":
        diff = gpu["bf16"] != orc["bf16"]
        tol = np.abs(o) * 2.0 ** -7 + 1e-30
    else:
        s = orc["scale"].astype(np.float64)
        assert np.allclose(gpu["scale"], orc["scale"], rtol=1e-5, atol=0), f"{what}: row scales"
        diff = np.concatenate([gpu["rope"] != orc["rope"], gpu["nope"] != orc["nope"]], axis=1)
        tol = np.concatenate([np.abs(o[:, :64]) * 2.0 ** -7,
                              np.maximum(np.abs(o[:, 64:]) * 2.0 ** -3, s[:, None] * 2.0 ** -9)], axis=1) * 1.001
    frac = diff.mean() if diff.size else 0.0
    assert frac <= max_mismatch_frac, f"{what}: {frac:.2e} of stored values differ"
    bad = np.abs(g - o) > tol
    assert not bad.any(), f"{what}: {bad.sum()} values beyond one storage ulp"


def index_inputs(seed: int, layer: int, seq: int, n_entries: int, rank: int, block_scaled: bool = True):
    kc = synth.e2m1_codes(seed, synth.tensor_id(synth.IDX_K, layer, seq), 0, n_entries * rank).reshape(n_entries, rank)
    if block_scaled:
        ks = synth.ue8m0_scales(seed, synth.tensor_id(synth.IDX_KS, layer, seq), 0, n_entries * rank // 32)
        ks = ks.reshape(n_entries, rank // 32)
    else:
        ks = np.full((n_entries, rank // 32), 127, np.uint8)
    return kc, ks


def query_index_inputs(seed: int, layer: int, seq: int, t0: int, n: int, heads: int, rank: int,
                       block_scaled: bool = True, weighted: bool = True):
    """Indexer query codes/scales/weights for the tokens at positions t0 .. t0+n-1."""
    qc = synth.e2m1_codes(seed, synth.tensor_id(synth.IDX_Q, layer, seq), t0 * heads * rank, n * heads * rank)
    qc = qc.reshape(n, heads, rank)
    if block_scaled:
        qs = synth.ue8m0_scales(seed, synth.tensor_id(synth.IDX_QS, layer, seq), t0 * heads * rank // 32,
                                n * heads * rank // 32).reshape(n, heads, rank // 32)
    else:
        qs = np.full((n, heads, rank // 32), 127, np.uint8)
    hw = (synth.head_weights(seed, synth.tensor_id(synth.HEAD_W, layer, seq), t0 * heads, n * heads).reshape(n, heads)
          if weighted else np.ones((n, heads), np.float32))
    return qc, qs, hw


def queries_np(seed: int, layer: int, seq: int, t0: int, n: int, heads: int, dim: int, scale_bits=None):
    tid = synth.tensor_id(synth.QUERY, layer, seq)
    return synth.normal_bf16(seed, tid, t0 * heads * dim, n * heads * dim, scale_bits).reshape(n, heads, dim)


def u8(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8)).to(DEV)


def check_outputs(gpu_o: np.ndarray, orc_o: np.ndarray, what: str) -> None:
    err = np.abs(gpu_o - orc_o)
    assert np.isfinite(gpu_o).all(), f"{what}: non-finite outputs"
    assert err.max() <= OUT_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    rl2 = oracle.rel_l2(gpu_o, orc_o)
    assert rl2 <= OUT_REL_L2, f"{what}: rel L2 {rl2:.3e}"


def bf16_tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def workspace(nbytes: int) -> torch.Tensor:
    # zeros: the index workspace's leading counters must start at zero
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=DEV)


def dev_status() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def assert_status_ok(st: torch.Tensor) -> None:
    v = int(st.item())
    assert v == 0, f"device status {v} ({lcsa.STATUS_NAMES.get(v)})"


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [n for n in dir() if not n.startswith("_")] + ["math"]
