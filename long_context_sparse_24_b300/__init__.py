"""Python binding of the CSA / HCA hybrid compressed attention library (``liblcsa.so``).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.  The
functions carry the names of the C entry points declared in ``include/lcsa.h``; torch tensors
are passed by ``data_ptr()`` and the kernels are enqueued on the current CUDA stream.  There is
no CPU fallback: importing the module fails when the built library is missing.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblcsa.so")

LCS_ROW_BF16 = 0
LCS_ROW_FP8_SPLIT = 1
LCS_INDEX_RELU = 1
LCS_INDEX_SCORE_ONLY = 2
LCS_INDEX_SELECT_ONLY = 4


def LCS_INDEX_SPARE_SMS(n: int) -> int:
    """csa_index_topk flag: leave n SMs (0..255) free for work run next to the call."""
    return (int(n) & 0xFF) << 8
WINDOW = 128
ROPE_DIMS = 64
BLOCK_TOKENS = 128

STATUS_NAMES = {0: "LCS_OK", 1: "LCS_ERR_INVALID_ARG", 2: "LCS_ERR_SHAPE", 3: "LCS_ERR_ALIGNMENT",
                4: "LCS_ERR_UNSUPPORTED", 5: "LCS_ERR_CUDA", 6: "LCS_ERR_DEVICE_GUARD", 7: "LCS_ERR_TIMEOUT",
                8: "LCS_ERR_WORKSPACE"}


class LcsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python long_context_sparse_24_b300/build.py` "
                      "(nvcc, sm_103a); there is no fallback implementation")
_lib = ctypes.CDLL(LIB_PATH)

c_i32, c_i64, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t


class lcs_batch(ctypes.Structure):
    _fields_ = [("num_seqs", c_i32), ("cu_new", c_vp), ("seq_len", c_vp), ("total_new", c_i32),
                ("max_new", c_i32), ("max_seq_len", c_i32)]


class lcs_rows(ctypes.Structure):
    _fields_ = [("format", c_i32), ("dim", c_i32), ("num_rows", c_i64), ("nope", c_vp), ("rope", c_vp),
                ("scale", c_vp)]


class lcs_paging(ctypes.Structure):
    _fields_ = [("entries_per_block", c_i32), ("max_blocks_per_seq", c_i32), ("block_table", c_vp)]


class lcs_state(ctypes.Structure):
    _fields_ = [("window", lcs_rows), ("pending", c_vp), ("pending_slots", c_i32), ("new_rows", lcs_rows),
                ("pending_scores", c_vp)]


class lcs_values(ctypes.Structure):
    _fields_ = [("entries", lcs_rows), ("window", lcs_rows), ("new_rows", lcs_rows)]


class lcs_compressor(ctypes.Structure):
    _fields_ = [("w", c_vp), ("bias", c_vp), ("m", c_i32), ("overlap", c_i32), ("scores", c_vp)]


class lcs_index_keys(ctypes.Structure):
    _fields_ = [("fp4", c_vp), ("scale", c_vp), ("rank", c_i32), ("num_rows", c_i64)]


P = ctypes.POINTER
_SIGS = {
    "lcs_abi_version": (c_i32, []),
    "lcs_stage_copy": (c_i32, [c_i32, c_vp, c_vp, c_vp, c_vp]),
    "lcs_quantize_e2m1": (c_i32, [c_vp, c_i64, c_i32, c_vp, c_vp, c_vp]),
    "lcs_attention_sink": (c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_vp]),
    "lcs_status_string": (ctypes.c_char_p, [c_i32]),
    "lcs_device_check": (c_i32, []),
    "csa_compress": (c_i32, [P(lcs_batch), c_vp, P(lcs_compressor), P(lcs_state), P(lcs_rows), P(lcs_paging),
                             c_vp, c_vp]),
    "hca_compress": (c_i32, [P(lcs_batch), c_vp, P(lcs_compressor), P(lcs_state), P(lcs_rows), P(lcs_paging),
                             c_vp, c_vp]),
    "lcs_window_commit": (c_i32, [P(lcs_batch), P(lcs_state), c_vp, c_vp]),
    "lcs_index_topk_workspace": (c_sz, [P(lcs_batch), c_i32, P(lcs_index_keys), P(lcs_paging), c_i32, c_i32]),
    "lcs_index_topk_workspace_zeroed": (c_sz, [P(lcs_batch)]),
    "lcs_set_wait_polls": (ctypes.c_uint32, [ctypes.c_uint32]),
    "lcs_mma_probe": (c_i32, [c_i32, c_i32, c_i32, c_vp, c_vp]),
    "csa_index_topk": (c_i32, [P(lcs_batch), c_vp, c_vp, c_vp, c_i32, P(lcs_index_keys), P(lcs_paging), c_i32,
                               c_i32, c_i32, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "csa_index_scores": (c_i32, [P(lcs_batch), c_vp, c_vp, c_vp, c_i32, P(lcs_index_keys), P(lcs_paging), c_i32,
                                 c_i32, c_vp, c_i64, c_vp, c_vp]),
    "csa_index_topk_noalloc": (c_i32, [P(lcs_batch), c_vp, c_vp, c_vp, c_i32, P(lcs_index_keys), P(lcs_paging),
                                       c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp]),
    "lcs_attend_workspace": (c_sz, [P(lcs_batch), c_i32, c_i32, c_i32]),
    "csa_attend": (c_i32, [P(lcs_batch), c_vp, c_i32, c_vp, c_vp, c_i32, c_i32, P(lcs_rows), P(lcs_paging),
                           P(lcs_state), P(lcs_values), c_vp, ctypes.c_float, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "csa_attend_window": (c_i32, [P(lcs_batch), c_vp, c_i32, c_i32, c_i32, P(lcs_rows), P(lcs_paging), P(lcs_state),
                                  P(lcs_values), ctypes.c_float, c_vp, c_sz, c_vp, c_vp]),
    "csa_attend_topk": (c_i32, [P(lcs_batch), c_vp, c_i32, c_vp, c_vp, c_i32, c_i32, P(lcs_rows), P(lcs_paging),
                                P(lcs_state), P(lcs_values), c_vp, ctypes.c_float, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "hca_attend": (c_i32, [P(lcs_batch), c_vp, c_i32, c_i32, P(lcs_rows), P(lcs_paging), P(lcs_state),
                           P(lcs_values), c_vp, ctypes.c_float, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, what: str) -> None:
    if status != 0:
        raise LcsError(status, what)


# ---------------------------------------------------------------------------------------------
# Host-side descriptions of the caller-owned buffers
# ---------------------------------------------------------------------------------------------

@dataclasses.dataclass
class Batch:
    cu_new: object            # device int32 [num_seqs+1]
    seq_len: object           # device int32 [num_seqs]
    num_seqs: int
    total_new: int
    max_new: int
    max_seq_len: int

    def c(self) -> lcs_batch:
        return lcs_batch(self.num_seqs, _ptr(self.cu_new), _ptr(self.seq_len), self.total_new, self.max_new,
                         self.max_seq_len)


@dataclasses.dataclass
class RowSet:
    format: int
    dim: int
    num_rows: int
    nope: object = None
    rope: object = None
    scale: object = None

    def c(self) -> lcs_rows:
        return lcs_rows(self.format, self.dim, self.num_rows, _ptr(self.nope), _ptr(self.rope), _ptr(self.scale))


@dataclasses.dataclass
class Paging:
    block_table: object       # device int32 [num_seqs, max_blocks_per_seq]
    entries_per_block: int
    max_blocks_per_seq: int

    def c(self) -> lcs_paging:
        return lcs_paging(self.entries_per_block, self.max_blocks_per_seq, _ptr(self.block_table))


@dataclasses.dataclass
class State:
    window: RowSet
    pending: object
    pending_slots: int
    new_rows: Optional[RowSet] = None
    pending_scores: object = None   # per-channel compressors: bf16 [num_seqs, pending_slots, D]

    def c(self) -> lcs_state:
        nr = self.new_rows.c() if self.new_rows is not None else lcs_rows(self.window.format, self.window.dim, 0,
                                                                            None, None, None)
        return lcs_state(self.window.c(), _ptr(self.pending), self.pending_slots, nr, _ptr(self.pending_scores))


@dataclasses.dataclass
class Values:
    """Separate value rows: each set numbered like its key counterpart (entry cache, window ring,
    new rows of the call)."""
    entries: RowSet
    window: RowSet
    new_rows: Optional[RowSet] = None

    def c(self) -> lcs_values:
        nr = self.new_rows.c() if self.new_rows is not None else lcs_rows(self.window.format, self.window.dim, 0,
                                                                            None, None, None)
        return lcs_values(self.entries.c(), self.window.c(), nr)


def _values_ref(values: Optional[Values]):
    """(ctypes argument, keep-alive) for an optional Values."""
    if values is None:
        return None, None
    v = values.c()
    return ctypes.byref(v), v


@dataclasses.dataclass
class Compressor:
    w: object                 # device f32 [D] (scalar weights)
    bias: object              # device f32 [2m] or [m]; per-channel: [2m, D] or [m, D]
    m: int
    overlap: bool

    def c(self, scores=None) -> lcs_compressor:
        return lcs_compressor(_ptr(self.w), _ptr(self.bias), self.m, 1 if self.overlap else 0, _ptr(scores))


@dataclasses.dataclass
class IndexKeys:
    fp4: object               # device uint8 [rows, r/2]
    scale: object             # device uint8 [rows, r/32]
    rank: int
    num_rows: int

    def c(self) -> lcs_index_keys:
        return lcs_index_keys(_ptr(self.fp4), _ptr(self.scale), self.rank, self.num_rows)


# ---------------------------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------------------------

def lcs_abi_version() -> int:
    return _lib.lcs_abi_version()


def lcs_status_string(status: int) -> str:
    return _lib.lcs_status_string(status).decode()


def lcs_device_check() -> int:
    return _lib.lcs_device_check()


def csa_compress(batch: Batch, raw, comp: Compressor, state: State, entries: RowSet, paging: Paging,
                 dev_status=None, stream=None, scores=None) -> None:
    """scores: per-channel score rows of the new tokens (bf16 [total_new, D]) for a per-channel
    compressor, else None."""
    b, c, s, e, p = batch.c(), comp.c(scores), state.c(), entries.c(), paging.c()
    _check(_lib.csa_compress(ctypes.byref(b), _ptr(raw), ctypes.byref(c), ctypes.byref(s), ctypes.byref(e),
                             ctypes.byref(p), _ptr(dev_status), _stream(stream)), "csa_compress")


def hca_compress(batch: Batch, raw, comp: Compressor, state: State, entries: RowSet, paging: Paging,
                 dev_status=None, stream=None) -> None:
    b, c, s, e, p = batch.c(), comp.c(), state.c(), entries.c(), paging.c()
    _check(_lib.hca_compress(ctypes.byref(b), _ptr(raw), ctypes.byref(c), ctypes.byref(s), ctypes.byref(e),
                             ctypes.byref(p), _ptr(dev_status), _stream(stream)), "hca_compress")


def lcs_quantize_e2m1(x, codes, scales, stream=None) -> None:
    """Block-scaled FP4 of BF16 rows x [rows, r]: codes [rows, r/2] uint8, scales [rows, r/32] uint8."""
    rows, r = int(x.shape[0]), int(x.shape[-1])
    _check(_lib.lcs_quantize_e2m1(_ptr(x), rows, r, _ptr(codes), _ptr(scales), _stream(stream)), "lcs_quantize_e2m1")


def lcs_attention_sink(out, out_lse, sink, stream=None) -> None:
    """Per-head sink logits sink [heads] applied to attention outputs out [T, heads, D] and lse [T, heads]."""
    T, H, D = int(out.shape[0]), int(out.shape[1]), int(out.shape[2])
    _check(_lib.lcs_attention_sink(_ptr(out), _ptr(out_lse), _ptr(sink), T, H, D, _stream(stream)),
           "lcs_attention_sink")


def lcs_stage_copy(pairs, stream=None) -> None:
    """Copy each (dst, src) tensor pair (device or pinned host, same byte size) with one kernel."""
    n = len(pairs)
    dst = (c_vp * max(n, 1))(*[_ptr(d) for d, _ in pairs])
    src = (c_vp * max(n, 1))(*[_ptr(s_) for _, s_ in pairs])
    nbytes = []
    for d, s_ in pairs:
        nb = s_.numel() * s_.element_size()
        if d.numel() * d.element_size() != nb:
            raise ValueError("lcs_stage_copy: destination and source sizes differ")
        nbytes.append(nb)
    sizes = (c_sz * max(n, 1))(*nbytes)
    _check(_lib.lcs_stage_copy(n, dst, src, sizes, _stream(stream)), "lcs_stage_copy")


def lcs_window_commit(batch: Batch, state: State, dev_status=None, stream=None) -> None:
    b, s = batch.c(), state.c()
    _check(_lib.lcs_window_commit(ctypes.byref(b), ctypes.byref(s), _ptr(dev_status), _stream(stream)),
           "lcs_window_commit")


def lcs_index_topk_workspace(batch: Batch, heads: int, keys: IndexKeys, paging: Paging, m: int, k: int) -> int:
    b, kk, p = batch.c(), keys.c(), paging.c()
    return _lib.lcs_index_topk_workspace(ctypes.byref(b), heads, ctypes.byref(kk), ctypes.byref(p), m, k)


def lcs_index_topk_workspace_zeroed(batch: Batch) -> int:
    b = batch.c()
    return _lib.lcs_index_topk_workspace_zeroed(ctypes.byref(b))


def lcs_set_wait_polls(polls: int) -> int:
    return int(_lib.lcs_set_wait_polls(polls))


def lcs_mma_probe(kind: int, mmas_per_cta: int, ctas: int, dev_status=None, stream=None) -> None:
    _check(_lib.lcs_mma_probe(kind, mmas_per_cta, ctas, _ptr(dev_status), _stream(stream)), "lcs_mma_probe")


def csa_index_topk(batch: Batch, q_fp4, q_scale, head_w, heads: int, keys: IndexKeys, paging: Paging, m: int,
                   k: int, flags: int, out_idx, out_cnt, workspace, workspace_bytes: int, dev_status=None,
                   stream=None) -> None:
    b, kk, p = batch.c(), keys.c(), paging.c()
    _check(_lib.csa_index_topk(ctypes.byref(b), _ptr(q_fp4), _ptr(q_scale), _ptr(head_w), heads, ctypes.byref(kk),
                               ctypes.byref(p), m, k, flags, _ptr(out_idx), _ptr(out_cnt), _ptr(workspace),
                               workspace_bytes, _ptr(dev_status), _stream(stream)), "csa_index_topk")


def csa_index_scores(batch: Batch, q_fp4, q_scale, head_w, heads: int, keys: IndexKeys, paging: Paging, m: int,
                     flags: int, out_scores, ld: int, dev_status=None, stream=None) -> None:
    b, kk, p = batch.c(), keys.c(), paging.c()
    _check(_lib.csa_index_scores(ctypes.byref(b), _ptr(q_fp4), _ptr(q_scale), _ptr(head_w), heads,
                                 ctypes.byref(kk), ctypes.byref(p), m, flags, _ptr(out_scores), ld,
                                 _ptr(dev_status), _stream(stream)), "csa_index_scores")


NOALLOC_SCRATCH_BYTES = 8 << 20


def csa_index_topk_noalloc(batch: Batch, q_fp4, q_scale, head_w, heads: int, keys: IndexKeys, paging: Paging,
                           m: int, k: int, flags: int, out_idx, out_cnt, dev_status=None, stream=None) -> None:
    """csa_index_topk without a workspace argument, for callers that cannot allocate: the scratch
    is the library's fixed device array (NOALLOC_SCRATCH_BYTES).  Calls must not overlap on the GPU."""
    b, kk, p = batch.c(), keys.c(), paging.c()
    _check(_lib.csa_index_topk_noalloc(ctypes.byref(b), _ptr(q_fp4), _ptr(q_scale), _ptr(head_w), heads,
                                       ctypes.byref(kk), ctypes.byref(p), m, k, flags, _ptr(out_idx), _ptr(out_cnt),
                                       _ptr(dev_status), _stream(stream)), "csa_index_topk_noalloc")


def lcs_attend_workspace(batch: Batch, heads: int, dim: int, max_rows: int) -> int:
    b = batch.c()
    return _lib.lcs_attend_workspace(ctypes.byref(b), heads, dim, max_rows)


def csa_attend(batch: Batch, q, heads: int, topk_idx, topk_cnt, k: int, m: int, entries: RowSet, paging: Paging,
               state: State, softmax_scale: float, out, out_lse, workspace, workspace_bytes: int, dev_status=None,
               stream=None, values: Optional[Values] = None, sink=None) -> None:
    b, e, p, s = batch.c(), entries.c(), paging.c(), state.c()
    vr, _keep = _values_ref(values)
    _check(_lib.csa_attend(ctypes.byref(b), _ptr(q), heads, _ptr(topk_idx), _ptr(topk_cnt), k, m, ctypes.byref(e),
                           ctypes.byref(p), ctypes.byref(s), vr, _ptr(sink), softmax_scale, _ptr(out), _ptr(out_lse),
                           _ptr(workspace), workspace_bytes, _ptr(dev_status), _stream(stream)), "csa_attend")


def csa_attend_window(batch: Batch, q, heads: int, k: int, m: int, entries: RowSet, paging: Paging, state: State,
                      softmax_scale: float, workspace, workspace_bytes: int, dev_status=None, stream=None,
                      values: Optional[Values] = None) -> None:
    b, e, p, s = batch.c(), entries.c(), paging.c(), state.c()
    vr, _keep = _values_ref(values)
    _check(_lib.csa_attend_window(ctypes.byref(b), _ptr(q), heads, k, m, ctypes.byref(e), ctypes.byref(p),
                                  ctypes.byref(s), vr, softmax_scale, _ptr(workspace), workspace_bytes, _ptr(dev_status),
                                  _stream(stream)), "csa_attend_window")


def csa_attend_topk(batch: Batch, q, heads: int, topk_idx, topk_cnt, k: int, m: int, entries: RowSet, paging: Paging,
                    state: State, softmax_scale: float, out, out_lse, workspace, workspace_bytes: int,
                    dev_status=None, stream=None, values: Optional[Values] = None, sink=None) -> None:
    b, e, p, s = batch.c(), entries.c(), paging.c(), state.c()
    vr, _keep = _values_ref(values)
    _check(_lib.csa_attend_topk(ctypes.byref(b), _ptr(q), heads, _ptr(topk_idx), _ptr(topk_cnt), k, m,
                                ctypes.byref(e), ctypes.byref(p), ctypes.byref(s), vr, _ptr(sink), softmax_scale, _ptr(out),
                                _ptr(out_lse), _ptr(workspace), workspace_bytes, _ptr(dev_status), _stream(stream)),
           "csa_attend_topk")


def hca_attend(batch: Batch, q, heads: int, m: int, entries: RowSet, paging: Paging, state: State,
               softmax_scale: float, out, out_lse, workspace, workspace_bytes: int, dev_status=None,
               stream=None, values: Optional[Values] = None, sink=None) -> None:
    b, e, p, s = batch.c(), entries.c(), paging.c(), state.c()
    vr, _keep = _values_ref(values)
    _check(_lib.hca_attend(ctypes.byref(b), _ptr(q), heads, m, ctypes.byref(e), ctypes.byref(p), ctypes.byref(s),
                           vr, _ptr(sink), softmax_scale, _ptr(out), _ptr(out_lse), _ptr(workspace), workspace_bytes,
                           _ptr(dev_status), _stream(stream)), "hca_attend")
