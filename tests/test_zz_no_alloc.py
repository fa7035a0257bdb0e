"""The allocation-free indexer entry point (csa_index_topk_noalloc).

Some callers cannot allocate device memory (graph capture owned by another framework, runtimes
with a fixed memory pool), so this entry point takes no workspace and uses a fixed scratch
array of the library instead.  Its results must equal those of csa_index_topk with a
caller-provided workspace, on consecutive calls that reuse the same scratch.  The file sorts
last so that a run stopping at the first failure has run every other test first.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth
from harness import (DEV, assert_status_ok, dev_status, entry_rows_of, index_inputs, query_index_inputs,
                     to_dev_f32, u8, workspace)

lcsa = pytest.importorskip("long_context_sparse_24_b300")
from long_context_sparse_24_b300 import buffers  # noqa: E402

pytestmark = pytest.mark.gpu


def _case(seed, lengths, new, m=4, heads=4, rank=128):
    S = len(lengths)
    cap = max(lengths) + 128
    cache = buffers.alloc_layer(S, cap, 512, lcsa.LCS_ROW_FP8_SPLIT, m, True, 0, DEV, index_rank=rank)
    batch = buffers.make_batch(lengths, new, DEV, max_seq_len=cap)
    qc, qs, hw = [], [], []
    for b in range(S):
        ne = lengths[b] // m
        kc, ks = index_inputs(seed, 0, b, ne, rank)
        rows = torch.as_tensor(entry_rows_of(cache, b, range(ne)), device=DEV)
        cache.keys.fp4[rows] = u8(synth.pack_e2m1(kc))
        cache.keys.scale[rows] = u8(ks)
        c, s, w = query_index_inputs(seed, 0, b, lengths[b] - new[b], new[b], heads, rank)
        qc.append(c); qs.append(s); hw.append(w)
    return (cache, batch, u8(synth.pack_e2m1(np.concatenate(qc))), u8(np.concatenate(qs)),
            to_dev_f32(np.concatenate(hw)))


def _call_c_abi_noalloc(batch, q_fp4, q_sc, hw, heads, cache, m, k, out_idx, out_cnt, st, flags=0):
    """Call the exported C symbol directly (the C ABI, no Python wrapper logic)."""
    lib = ctypes.CDLL(lcsa.LIB_PATH)
    fn = lib.csa_index_topk_noalloc
    fn.restype = ctypes.c_int32
    P, vp, i32 = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [P(lcsa.lcs_batch), vp, vp, vp, i32, P(lcsa.lcs_index_keys), P(lcsa.lcs_paging), i32, i32, i32,
                   vp, vp, vp, vp]
    b, kk, pg = batch.c(), cache.keys.c(), cache.paging.c()
    return fn(ctypes.byref(b), q_fp4.data_ptr(), q_sc.data_ptr(), hw.data_ptr(), heads, ctypes.byref(kk),
              ctypes.byref(pg), m, k, flags, out_idx.data_ptr() if out_idx is not None else None,
              out_cnt.data_ptr() if out_cnt is not None else None, st.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("first,second", [
    ((61, [5000, 131, 20000], [1, 1, 1], 512), (62, [9000, 700], [3, 2], 64)),
])
def test_noalloc_topk_equals_workspace_entry_point_twice(first, second):
    for seed, lengths, new, k in (first, second):       # two calls in a row share the scratch
        m, heads = 4, 4
        cache, batch, q_fp4, q_sc, hw = _case(seed, lengths, new)
        T = batch.total_new
        ref_idx = torch.full((T, k), -5, dtype=torch.int32, device=DEV)
        ref_cnt = torch.full((T,), -5, dtype=torch.int32, device=DEV)
        wsb = lcsa.lcs_index_topk_workspace(batch, heads, cache.keys, cache.paging, m, k)
        lcsa.csa_index_topk(batch, q_fp4, q_sc, hw, heads, cache.keys, cache.paging, m, k, 0, ref_idx, ref_cnt,
                            workspace(wsb), wsb)
        got_idx = torch.full((T, k), -9, dtype=torch.int32, device=DEV)
        got_cnt = torch.full((T,), -9, dtype=torch.int32, device=DEV)
        st = dev_status()
        rc = _call_c_abi_noalloc(batch, q_fp4, q_sc, hw, heads, cache, m, k, got_idx, got_cnt, st)
        assert rc == 0, lcsa.lcs_status_string(rc)
        torch.cuda.synchronize()
        assert_status_ok(st)
        assert torch.equal(got_idx, ref_idx)
        assert torch.equal(got_cnt, ref_cnt)


def test_noalloc_score_then_select_phases_share_the_scratch():
    """A scoring-only call leaves its results in the shared scratch; the selection-only call that
    follows on the same stream reads them.  Together they equal one call with a caller-provided
    workspace (same batch, m and k)."""
    seed, lengths, new, k, m, heads = 63, [7000, 300, 12000], [1, 2, 1], 256, 4, 4
    cache, batch, q_fp4, q_sc, hw = _case(seed, lengths, new)
    T = batch.total_new
    ref_idx = torch.full((T, k), -5, dtype=torch.int32, device=DEV)
    ref_cnt = torch.full((T,), -5, dtype=torch.int32, device=DEV)
    wsb = lcsa.lcs_index_topk_workspace(batch, heads, cache.keys, cache.paging, m, k)
    lcsa.csa_index_topk(batch, q_fp4, q_sc, hw, heads, cache.keys, cache.paging, m, k, 0, ref_idx, ref_cnt,
                        workspace(wsb), wsb)
    got_idx = torch.full((T, k), -9, dtype=torch.int32, device=DEV)
    got_cnt = torch.full((T,), -9, dtype=torch.int32, device=DEV)
    st = dev_status()
    rc = _call_c_abi_noalloc(batch, q_fp4, q_sc, hw, heads, cache, m, k, None, None, st,
                             flags=lcsa.LCS_INDEX_SCORE_ONLY)
    assert rc == 0, lcsa.lcs_status_string(rc)
    rc = _call_c_abi_noalloc(batch, q_fp4, q_sc, hw, heads, cache, m, k, got_idx, got_cnt, st,
                             flags=lcsa.LCS_INDEX_SELECT_ONLY)
    assert rc == 0, lcsa.lcs_status_string(rc)
    torch.cuda.synchronize()
    assert_status_ok(st)
    assert torch.equal(got_idx, ref_idx)
    assert torch.equal(got_cnt, ref_cnt)


def test_noalloc_rejects_requests_beyond_its_scratch():
    # a chunk of 300 queries over a 131072-entry sequence at rank 64 keeps every score key: 157 MB of
    # scratch, refused, nothing launched
    cap = 4 * 131072 + 128
    batch = buffers.make_batch([cap - 128], [300], DEV, max_seq_len=cap)
    z = torch.zeros(16, dtype=torch.int32, device=DEV)
    keys = lcsa.IndexKeys(z, z, 64, 1)
    pg = lcsa.Paging(z, 32, 1)
    assert lcsa.lcs_index_topk_workspace(batch, 4, keys, pg, 4, 512) > lcsa.NOALLOC_SCRATCH_BYTES
    with pytest.raises(lcsa.LcsError) as e:
        lcsa.csa_index_topk_noalloc(batch, z, z, None, 4, keys, pg, 4, 512, 0, z, z)
    assert e.value.status == 8
