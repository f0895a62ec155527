"""ctypes front end of the C oracle (``pmg_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring). Builds the C file with
gcc on first use into ``oracle/_build/`` (git-ignored) and calls it on numpy
arrays held in host memory.

Source: "MLA cache gather scheduled per logical page" (prhub.com.cn, vllm PR
#51739), section "关键源码片段", test_cp_gather_cache_mla_large_uneven_sequences
(the per-token expected output) and the map_gather_page_task listing (output
placement from cu_seq_lens and seq_starts).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pmg_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpmg_oracle.so")

# dtype codes of the oracle's C interface
DTYPE_CODES = {"bf16": 0, "fp16": 1, "fp32": 2, "fp8_e4m3": 3, "u8": 4}
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp32": 4, "fp8_e4m3": 1, "u8": 1}

BAD_LOGICAL = 1
BAD_PHYS = 2
BAD_START = 4
BAD_CU = 8
BAD_TOKEN = 32

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load(path: str) -> ctypes.CDLL:
    """Load an oracle library build and declare its C signatures."""
    L = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    L.pmg_oracle_gather.restype = ctypes.c_int
    L.pmg_oracle_gather.argtypes = [
        vp, i64, i64, i64, vp, i64, vp, vp, i32, i64, i32, i32,
        ctypes.c_int, ctypes.c_int, ctypes.c_float, vp, i64]
    L.pmg_oracle_e4m3_to_f32.restype = ctypes.c_float
    L.pmg_oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.pmg_oracle_bf16_to_f32.restype = ctypes.c_float
    L.pmg_oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.pmg_oracle_f16_to_f32.restype = ctypes.c_float
    L.pmg_oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.pmg_oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.pmg_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.pmg_oracle_f32_to_f16.restype = ctypes.c_uint16
    L.pmg_oracle_f32_to_f16.argtypes = [ctypes.c_float]
    L.pmg_oracle_pair_supported.restype = ctypes.c_int
    L.pmg_oracle_pair_supported.argtypes = [ctypes.c_int, ctypes.c_int]
    L.pmg_oracle_gather_tokens.restype = ctypes.c_int
    L.pmg_oracle_gather_tokens.argtypes = [
        vp, i64, i64, i64, vp, i64, vp, vp, i32, i64, i32, i32,
        ctypes.c_int, ctypes.c_int, ctypes.c_float, vp, i64]
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    return a.ctypes.data


def gather(cache: np.ndarray, block_table: np.ndarray, cu_seq_lens: np.ndarray,
           seq_starts: np.ndarray | None, num_reqs: int, total_tokens: int, block_size: int,
           entry_size: int, src_dtype: str, dst_dtype: str, scale: float, dst: np.ndarray) -> int:
    """Run the oracle gather into ``dst`` (modified in place). Returns the flag bits.

    cache: array of shape [num_blocks, block_size, row_stride] (any numpy dtype
    with the source element size; uint8/uint16/float32 views are typical), last
    dimension contiguous. block_table: int32 [num_reqs, block_table_stride].
    cu_seq_lens: int32 [num_reqs + 1]. seq_starts: int32 [num_reqs] or None.
    dst: array [rows, dst_row_stride] of the destination element size, last
    dimension contiguous.
    """
    es, ed = ELEM_BYTES[src_dtype], ELEM_BYTES[dst_dtype]
    assert cache.ndim == 3 and cache.itemsize == es and (cache.strides[2] == es or cache.size == 0)
    assert dst.ndim == 2 and dst.itemsize == ed and (dst.strides[1] == ed or dst.size == 0)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    assert bt.ndim == 2
    cu = np.ascontiguousarray(cu_seq_lens, dtype=np.int32)
    assert cu.shape[0] >= num_reqs + 1
    ss = None if seq_starts is None else np.ascontiguousarray(seq_starts, dtype=np.int32)
    rc = lib().pmg_oracle_gather(
        _ptr(cache), cache.shape[1] * cache.shape[2] if cache.size == 0 else cache.strides[0] // es,
        cache.shape[2] if cache.size == 0 else cache.strides[1] // es, cache.shape[0],
        _ptr(bt), bt.shape[1], _ptr(cu), _ptr(ss), int(num_reqs), int(total_tokens),
        int(block_size), int(entry_size), DTYPE_CODES[src_dtype], DTYPE_CODES[dst_dtype],
        float(scale), _ptr(dst), dst.shape[1] if dst.size == 0 else dst.strides[0] // ed)
    if rc < 0:
        raise ValueError("oracle: call outside the defined domain (dtype pair or sizes)")
    return rc


def gather_tokens(cache: np.ndarray, block_table: np.ndarray, token_to_seq: np.ndarray, cu_seq_lens: np.ndarray,
                  num_reqs: int, num_tokens: int, block_size: int, entry_size: int, src_dtype: str, dst_dtype: str,
                  scale: float, dst: np.ndarray) -> int:
    """The per-token indexed gather (output row t from request token_to_seq[t])
    into ``dst`` (modified in place). Array conventions as in gather()."""
    es, ed = ELEM_BYTES[src_dtype], ELEM_BYTES[dst_dtype]
    assert cache.ndim == 3 and cache.itemsize == es and (cache.strides[2] == es or cache.size == 0)
    assert dst.ndim == 2 and dst.itemsize == ed and (dst.strides[1] == ed or dst.size == 0)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    t2s = np.ascontiguousarray(token_to_seq, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seq_lens, dtype=np.int32)
    assert t2s.shape[0] >= num_tokens and cu.shape[0] >= num_reqs + 1
    rc = lib().pmg_oracle_gather_tokens(
        _ptr(cache), cache.shape[1] * cache.shape[2] if cache.size == 0 else cache.strides[0] // es,
        cache.shape[2] if cache.size == 0 else cache.strides[1] // es, cache.shape[0],
        _ptr(bt), bt.shape[1], _ptr(t2s), _ptr(cu), int(num_reqs), int(num_tokens), int(block_size),
        int(entry_size), DTYPE_CODES[src_dtype], DTYPE_CODES[dst_dtype], float(scale), _ptr(dst),
        dst.shape[1] if dst.size == 0 else dst.strides[0] // ed)
    if rc < 0:
        raise ValueError("oracle: call outside the defined domain (dtype pair or sizes)")
    return rc


def pair_supported(src_dtype: str, dst_dtype: str) -> bool:
    return bool(lib().pmg_oracle_pair_supported(DTYPE_CODES[src_dtype], DTYPE_CODES[dst_dtype]))


def e4m3_to_f32(code: int) -> float:
    return lib().pmg_oracle_e4m3_to_f32(code)


def bf16_to_f32(bits: int) -> float:
    return lib().pmg_oracle_bf16_to_f32(bits)


def f16_to_f32(bits: int) -> float:
    return lib().pmg_oracle_f16_to_f32(bits)


def f32_to_bf16(x: float) -> int:
    return lib().pmg_oracle_f32_to_bf16(x)


def f32_to_f16(x: float) -> int:
    return lib().pmg_oracle_f32_to_f16(x)


def convert_array(src_bits: np.ndarray, src_dtype: str, dst_dtype: str, scale: float = 1.0) -> np.ndarray:
    """Convert a 1-D array of source element bit patterns through the oracle's
    gather (one request, one block, identity table). Returns dst bit patterns."""
    es, ed = ELEM_BYTES[src_dtype], ELEM_BYTES[dst_dtype]
    sdt = {1: np.uint8, 2: np.uint16, 4: np.uint32}[es]
    ddt = {1: np.uint8, 2: np.uint16, 4: np.uint32}[ed]
    n = int(src_bits.shape[0])
    cache = np.ascontiguousarray(src_bits.astype(sdt)).reshape(1, 1, n)
    dst = np.zeros((1, n), dtype=ddt)
    flag = gather(cache, np.zeros((1, 1), np.int32), np.array([0, 1], np.int32), None, 1, 1, 1, n,
                  src_dtype, dst_dtype, scale, dst)
    assert flag == 0
    return dst[0]
