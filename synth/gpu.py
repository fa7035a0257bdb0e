"""ctypes loader of ``synth/libsynth_gpu.so``: the seeded generator filling device buffers."""
from __future__ import annotations

import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth_gpu.so")
SRC = os.path.join(HERE, "gen.cu")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-shared",
                    "-Xcompiler", "-fPIC", "-o", LIB + ".tmp", SRC], check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} missing: run synth.gpu.build()")
        _lib = ctypes.CDLL(LIB)
        u32, u64, vp = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p
        _lib.synth_normal_bf16.argtypes = [u32, u32, u64, u64, vp, vp]
        _lib.synth_e2m1_packed.argtypes = [u32, u32, u64, u64, vp, vp]
        _lib.synth_ue8m0.argtypes = [u32, u32, u64, u64, ctypes.c_int, ctypes.c_int, vp, vp]
        for f in (_lib.synth_normal_bf16, _lib.synth_e2m1_packed, _lib.synth_ue8m0):
            f.restype = ctypes.c_int
    return _lib


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def normal_bf16(out, seed: int, tid: int, start: int) -> None:
    """Fill the bf16 tensor ``out`` (contiguous) with draws start .. start+numel-1."""
    assert out.is_contiguous()
    rc = lib().synth_normal_bf16(seed, tid, start, out.numel(), out.data_ptr(), _stream())
    if rc:
        raise RuntimeError("synth_normal_bf16 launch failed")


def e2m1_packed(out, seed: int, tid: int, start_code: int) -> None:
    """Fill the uint8 tensor ``out`` with packed codes start_code .. start_code+2*numel-1."""
    assert out.is_contiguous()
    rc = lib().synth_e2m1_packed(seed, tid, start_code, out.numel(), out.data_ptr(), _stream())
    if rc:
        raise RuntimeError("synth_e2m1_packed launch failed")


def ue8m0(out, seed: int, tid: int, start: int, lo: int = -1, hi: int = 1) -> None:
    assert out.is_contiguous()
    rc = lib().synth_ue8m0(seed, tid, start, out.numel(), lo, hi, out.data_ptr(), _stream())
    if rc:
        raise RuntimeError("synth_ue8m0 launch failed")
