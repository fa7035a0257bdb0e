"""The C ABI library: loads, exports every entry point the header declares, validates arguments
on the host (no GPU needed for any call here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "lcsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:lcs_status|size_t|int32_t|uint32_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_operations():
    names = header_functions()
    for n in ("csa_compress", "hca_compress", "csa_index_topk", "csa_attend", "hca_attend"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import long_context_sparse_24_b300 as lcsa
    lib = ctypes.CDLL(lcsa.LIB_PATH)
    for n in header_functions():
        assert hasattr(lib, n), n
    assert set(header_functions()) == set(lcsa.EXPORTED)


def test_abi_version_and_status_strings():
    import long_context_sparse_24_b300 as lcsa
    assert lcsa.lcs_abi_version() == 3
    assert lcsa.lcs_status_string(0) == "ok"
    assert "workspace" in lcsa.lcs_status_string(8)


def _batch(lcsa, **kw):
    b = lcsa.lcs_batch(1, 0x1000, 0x2000, 1, 1, 10)
    for k, v in kw.items():
        setattr(b, k, v)
    return b


def test_host_validation_without_gpu():
    import long_context_sparse_24_b300 as lcsa
    L = lcsa._lib
    rows = lcsa.lcs_rows(lcsa.LCS_ROW_FP8_SPLIT, 512, 10, 0x1000, 0x2000, 0x3000)
    pag = lcsa.lcs_paging(32, 4, 0x4000)
    st = lcsa.lcs_state(rows, 0x5000, 8, rows)
    comp = lcsa.lcs_compressor(0x6000, 0x7000, 4, 1)
    by = ctypes.byref
    # null batch
    assert L.csa_compress(None, 0x1000, by(comp), by(st), by(rows), by(pag), None, None) == 1
    # ratio not a power of two
    bad = lcsa.lcs_compressor(0x6000, 0x7000, 3, 1)
    assert L.csa_compress(by(_batch(lcsa)), 0x1000, by(bad), by(st), by(rows), by(pag), None, None) == 4
    # HCA rejects overlapping windows
    assert L.hca_compress(by(_batch(lcsa)), 0x1000, by(comp), by(st), by(rows), by(pag), None, None) == 4
    # pending slots must be 2m for an overlapping compressor
    st_bad = lcsa.lcs_state(rows, 0x5000, 4, rows)
    assert L.csa_compress(by(_batch(lcsa)), 0x1000, by(comp), by(st_bad), by(rows), by(pag), None, None) == 2
    # misaligned raw rows
    assert L.csa_compress(by(_batch(lcsa)), 0x1001, by(comp), by(st), by(rows), by(pag), None, None) == 3
    # unsupported head dim
    rows_bad = lcsa.lcs_rows(lcsa.LCS_ROW_FP8_SPLIT, 256, 10, 0x1000, 0x2000, 0x3000)
    assert L.csa_compress(by(_batch(lcsa)), 0x1000, by(comp), by(st), by(rows_bad), by(pag), None, None) == 4
    keys = lcsa.lcs_index_keys(0x1000, 0x2000, 128, 10)
    # indexer: 3 heads unsupported, k = 0 unsupported, missing workspace
    args = lambda heads, k, ws, wsb: (by(_batch(lcsa)), 0x1000, 0x2000, None, heads, by(keys), by(pag), 4, k, 0,
                                      0x3000, 0x4000, ws, wsb, None, None)
    assert L.csa_index_topk(*args(3, 16, 0x8000, 1 << 20)) == 4
    assert L.csa_index_topk(*args(4, 0, 0x8000, 1 << 20)) == 4
    assert L.csa_index_topk(*args(4, 16, None, 0)) == 8
    assert L.csa_index_topk(*args(4, 16, 0x8000, 1)) == 8
    # flags beyond ReLU, the two phases and the spare-SM count
    assert L.csa_index_topk(by(_batch(lcsa)), 0x1000, 0x2000, None, 4, by(keys), by(pag), 4, 16, 1 << 16, 0x3000,
                            0x4000, 0x8000, 1 << 20, None, None) == 1
    assert lcsa.LCS_INDEX_SPARE_SMS(32) == 32 << 8 and lcsa.LCS_INDEX_SPARE_SMS(300) == (300 & 0xFF) << 8
    # attention: heads 24 unsupported; topk list missing
    assert L.csa_attend(by(_batch(lcsa)), 0x1000, 24, 0x2000, None, 16, 4, by(rows), by(pag), by(st), None, None, 1.0,
                        0x3000, None, None, 0, None, None) == 4
    assert L.csa_attend(by(_batch(lcsa)), 0x1000, 64, None, None, 16, 4, by(rows), by(pag), by(st), None, None, 1.0,
                        0x3000, None, None, 0, None, None) == 1


def test_separate_values_host_validation():
    """Value sets must match their key counterparts' format, dim and row count, and come with new
    rows exactly when the state has them; a matching set passes to the workspace check."""
    import long_context_sparse_24_b300 as lcsa
    L = lcsa._lib
    by = ctypes.byref
    fp8 = lambda n: lcsa.lcs_rows(lcsa.LCS_ROW_FP8_SPLIT, 512, n, 0x1000, 0x2000, 0x3000)
    entries, ring, new = fp8(64), fp8(128), fp8(4)
    pag = lcsa.lcs_paging(32, 2, 0x4000)
    st = lcsa.lcs_state(ring, 0x5000, 8, new)
    b = _batch(lcsa)
    call = lambda v, heads=64: L.csa_attend(by(b), 0x1000, heads, 0x2000, None, 16, 4, by(entries), by(pag), by(st),
                                            by(v) if v is not None else None, None, 1.0, 0x3000, None, None, 0, None,
                                            None)
    hcall = lambda v, sink=None: L.hca_attend(by(b), 0x1000, 64, 128, by(entries), by(pag), by(st), by(v), sink, 1.0,
                                              0x3000, None, None, 0, None, None)
    good = lcsa.lcs_values(fp8(64), fp8(128), fp8(4))
    # one value set with fewer rows, another format, new rows missing
    assert call(lcsa.lcs_values(fp8(63), fp8(128), fp8(4))) == 2
    assert call(lcsa.lcs_values(fp8(64), fp8(129), fp8(4))) == 2
    assert call(lcsa.lcs_values(fp8(64), fp8(128), fp8(5))) == 2
    bf = lcsa.lcs_rows(lcsa.LCS_ROW_BF16, 512, 64, 0x1000, None, None)
    assert call(lcsa.lcs_values(bf, fp8(128), fp8(4))) == 2
    assert call(lcsa.lcs_values(fp8(64), fp8(128), lcsa.lcs_rows(lcsa.LCS_ROW_FP8_SPLIT, 512, 0, None, None, None))) == 2
    # a value set without its scales, or misaligned
    assert call(lcsa.lcs_values(lcsa.lcs_rows(lcsa.LCS_ROW_FP8_SPLIT, 512, 64, 0x1000, 0x2000, None), fp8(128),
                                fp8(4))) == 1
    assert call(lcsa.lcs_values(lcsa.lcs_rows(lcsa.LCS_ROW_FP8_SPLIT, 512, 64, 0x1008, 0x2000, 0x3000), fp8(128),
                                fp8(4))) == 3
    # matching sets get as far as the workspace check (none given), as do calls without values
    assert call(good) == 8 and call(None) == 8
    assert hcall(good) == 8
    assert hcall(lcsa.lcs_values(fp8(64), fp8(100), fp8(4))) == 2
    # a sink pointer not 4-byte aligned
    assert hcall(good, 0x5002) == 3 and hcall(good, 0x5004) == 8


def test_stage_copy_host_validation():
    import long_context_sparse_24_b300 as lcsa
    L = lcsa._lib
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    nine = (vp * 9)(*([0x1000] * 9))
    assert L.lcs_stage_copy(9, nine, nine, (sz * 9)(*([16] * 9)), None) == 4      # more than 8 copies
    assert L.lcs_stage_copy(0, None, None, None, None) == 0                      # nothing to copy
    assert L.lcs_stage_copy(1, None, None, None, None) == 1                      # missing lists
    assert L.lcs_stage_copy(1, (vp * 1)(None), (vp * 1)(0x1000), (sz * 1)(16), None) == 1   # NULL destination
    lcsa.lcs_stage_copy([], stream=0)                                             # binding: empty list


def test_quantize_e2m1_host_validation():
    import long_context_sparse_24_b300 as lcsa
    L = lcsa._lib
    assert L.lcs_quantize_e2m1(0x1000, 4, 48, 0x2000, 0x3000, None) == 4        # r not a multiple of 32
    assert L.lcs_quantize_e2m1(0x1000, 4, 8192, 0x2000, 0x3000, None) == 4      # r too large
    assert L.lcs_quantize_e2m1(0x1000, 0, 128, 0x2000, 0x3000, None) == 0       # no rows: nothing to do
    assert L.lcs_quantize_e2m1(None, 4, 128, 0x2000, 0x3000, None) == 1         # missing input
    assert L.lcs_quantize_e2m1(0x1008, 4, 128, 0x2000, 0x3000, None) == 3       # input not 16-byte aligned
    assert L.lcs_quantize_e2m1(0x1000, 4, 128, 0x2004, 0x3000, None) == 3       # codes not 8-byte aligned


def test_attention_sink_host_validation():
    import long_context_sparse_24_b300 as lcsa
    L = lcsa._lib
    assert L.lcs_attention_sink(0x1000, 0x2000, 0x3000, 4, 64, 100, None) == 4   # dim not a multiple of 8
    assert L.lcs_attention_sink(0x1000, 0x2000, 0x3000, 0, 64, 512, None) == 0   # nothing to do
    assert L.lcs_attention_sink(None, 0x2000, 0x3000, 4, 64, 512, None) == 1     # missing output
    assert L.lcs_attention_sink(0x1008, 0x2000, 0x3000, 4, 64, 512, None) == 3   # output not 16-byte aligned


def test_workspace_sizes():
    import long_context_sparse_24_b300 as lcsa
    keys = lcsa.lcs_index_keys(0x10000, 0x20000, 128, 32 * 32768)
    pg = lcsa.lcs_paging(32, 1024, 0x3000)
    # decode (one query per sequence, rank 128): the top-k runs inside the scorer and the workspace
    # holds per-run lists of k keys, far less than a key per (query, entry)
    b = lcsa.lcs_batch(32, 0x1000, 0x2000, 32, 1, 131072)
    n = lcsa._lib.lcs_index_topk_workspace(ctypes.byref(b), 4, ctypes.byref(keys), ctypes.byref(pg), 4, 512)
    assert 32 * 512 * 8 <= n < 32 * (131072 // 4) * 4
    # zero between calls: a ticket (int32) and a shared threshold (u64) per sequence and query
    assert lcsa._lib.lcs_index_topk_workspace_zeroed(ctypes.byref(b)) == 256 + 256
    # up to 16 queries per sequence at rank 128: query groups, still lists of k keys per query and run
    b = lcsa.lcs_batch(64, 0x1000, 0x2000, 1024, 16, 131072)
    n = lcsa._lib.lcs_index_topk_workspace(ctypes.byref(b), 4, ctypes.byref(keys), ctypes.byref(pg), 4, 512)
    assert 1024 * 512 * 8 <= n < 1024 * (131072 // 4) * 4
    assert lcsa._lib.lcs_index_topk_workspace_zeroed(ctypes.byref(b)) == 1024 * 4 + 1024 * 8
    # a prefill chunk: the prefill scorer writes every score key (4 bytes per query and visible entry)
    b = lcsa.lcs_batch(1, 0x1000, 0x2000, 2048, 2048, 131072)
    n = lcsa._lib.lcs_index_topk_workspace(ctypes.byref(b), 4, ctypes.byref(keys), ctypes.byref(pg), 4, 512)
    assert n >= 2048 * (131072 // 4) * 4
    assert lcsa._lib.lcs_index_topk_workspace_zeroed(ctypes.byref(b)) == 2048 * 4 + 2048 * 8
    # rank 64: every score key of every (query, visible entry) pair
    keys64 = lcsa.lcs_index_keys(0x10000, 0x20000, 64, 32 * 32768)
    n = lcsa._lib.lcs_index_topk_workspace(ctypes.byref(b), 4, ctypes.byref(keys64), ctypes.byref(pg), 4, 512)
    assert n >= 2048 * (131072 // 4) * 4
