"""Thin ctypes binding of ``libpmg.so`` (declared in ``include/pmg.h``).

Argument marshalling only: shapes, strides, dtypes and raw pointers are taken
from torch tensors and passed to the C ABI; every step of the gather runs in
the CUDA kernels of ``csrc/pmg_gather.cu``. There is no fallback: if the
library is missing or a call fails, a PmgError is raised.

The call mirrors ops.cp_gather_cache(src_cache, dst, block_table, cu_seq_lens,
batch_size, seq_starts) of "MLA cache gather scheduled per logical page"
(prhub.com.cn, vllm PR #51739, section "关键源码片段"), with the dtype pair,
the FP8 scale, an error flag and the stream made explicit.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from .build import LIB_PATH

PMG_OK = 0
STATUS_NAMES = {0: "PMG_OK", 1: "PMG_ERR_NULL", 2: "PMG_ERR_ARG", 3: "PMG_ERR_DTYPE", 4: "PMG_ERR_ALIGN",
                5: "PMG_ERR_UNSUPPORTED", 6: "PMG_ERR_CUDA"}

DTYPE_CODES = {"bf16": 0, "fp16": 1, "fp32": 2, "fp8_e4m3": 3, "u8": 4}
TORCH_DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2, torch.float8_e4m3fn: 3, torch.uint8: 4}

FLAG_LOGICAL_BLOCK = 1
FLAG_PHYS_BLOCK = 2
FLAG_SEQ_START = 4
FLAG_CU_ORDER = 8
FLAG_TIMEOUT = 16
FLAG_TOKEN = 32

OPT_FORCE_SIMT = 1
OPT_FORCE_SCALAR = 2
OPT_IMPLIED_END = 4
OPT_EARLY_METADATA = 8

PATH_NAMES = {0: "none", 1: "bulk", 2: "vector", 3: "scalar", 4: "realign"}
WORKSPACE_INTS = 4
MAX_REQS_PLAN = 4096       # requests one launch plans; more need a workspace
MAX_REQS = 1 << 20         # requests one call accepts


class PmgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status})")


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libpmg.so once. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise PmgError(6, f"CUDA library {LIB_PATH} is missing; build it with "
                              "paged_mla_kv_cache_gb300.build.build_library()")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, u32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p
        gather_args = [vp, i64, i64, i64, vp, i64, vp, vp, i32, i64, i32, i32, i32, i32, vp, vp, i64, vp, vp]
        L.pmg_gather.restype = ctypes.c_int
        L.pmg_gather.argtypes = gather_args
        L.pmg_gather_ex.restype = ctypes.c_int
        L.pmg_gather_ex.argtypes = gather_args[:18] + [vp, vp, u32]
        L.pmg_gather_noalloc.restype = ctypes.c_int
        L.pmg_gather_noalloc.argtypes = gather_args
        L.pmg_debug_noalloc_scratch.restype = ctypes.c_int
        L.pmg_debug_noalloc_scratch.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(i64)]
        L.pmg_gather_tokens.restype = ctypes.c_int
        L.pmg_gather_tokens.argtypes = [vp, i64, i64, i64, vp, i64, vp, vp, i32, i64, i32, i32, i32, i32, vp, vp, i64,
                                        vp, vp, vp, u32]
        L.pmg_select_path.restype = ctypes.c_int
        L.pmg_select_path.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, i64, i32, i32, i32, i32, vp, i64, u32,
                                      ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.pmg_debug_plan.restype = ctypes.c_int
        L.pmg_debug_plan.argtypes = [vp, vp, i32, i64, i32, vp, i64, vp, vp, vp, u32]
        L.pmg_status_string.restype = ctypes.c_char_p
        L.pmg_status_string.argtypes = [ctypes.c_int]
        L.pmg_version.restype = ctypes.c_int
        L.pmg_version.argtypes = []
        _lib = L
        return _lib


def status_string(status: int) -> str:
    return load_library().pmg_status_string(status).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _table_width(block_table: torch.Tensor) -> int:
    if block_table.dim() != 2 or block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32 [num_reqs, block_table_stride]")
    if block_table.shape[0] > 1 and block_table.stride(0) != block_table.shape[1] or (
            block_table.shape[1] > 1 and block_table.stride(1) != 1):
        raise ValueError("block_table must be contiguous")
    return block_table.shape[1]


def _layout(cache: torch.Tensor, dst: torch.Tensor):
    if cache.dim() != 3:
        raise ValueError("cache must be [num_blocks, block_size, entry_size] (a padded row is a strided view)")
    if dst.dim() != 2:
        raise ValueError("dst must be [total_tokens, entry_size]")
    if cache.shape[2] > 1 and cache.stride(2) != 1 or dst.shape[1] > 1 and dst.stride(1) != 1:
        raise ValueError("the entry dimension must be contiguous")
    if cache.dtype not in TORCH_DTYPE_CODES or dst.dtype not in TORCH_DTYPE_CODES:
        raise ValueError(f"unsupported dtype {cache.dtype} -> {dst.dtype}")
    return TORCH_DTYPE_CODES[cache.dtype], TORCH_DTYPE_CODES[dst.dtype]


def gather(cache: torch.Tensor, dst: torch.Tensor, block_table: torch.Tensor, cu_seq_lens: torch.Tensor,
           seq_starts: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None,
           error_flag: Optional[torch.Tensor] = None, num_reqs: Optional[int] = None, stream=None,
           options: int = 0, workspace: Optional[torch.Tensor] = None) -> None:
    """Gather the cached entries of every request into dst (asynchronous).

    cache        [num_blocks, block_size, entry_size] device tensor; a padded
                 row stride is expressed as a view (stride(1) > entry_size).
    dst          [total_tokens, entry_size] device tensor (may be a row-strided view).
    block_table  int32 [num_reqs, block_table_stride]; row stride = stride(0).
    cu_seq_lens  int32 [num_reqs + 1] (or [num_reqs] with OPT_IMPLIED_END).
    seq_starts   int32 [num_reqs] or None.
    scale        fp32 device scalar tensor or None (1.0); used for fp8 sources.
    error_flag   int32 device tensor of one element or None.
    num_reqs     defaults to the request count implied by cu_seq_lens.
    workspace    int32 device tensor of WORKSPACE_INTS zeros (see new_workspace), or
                 None: dynamic work distribution on the TMA paths.
    """
    src_code, dst_code = _layout(cache, dst)
    if num_reqs is None:
        num_reqs = cu_seq_lens.shape[0] - (0 if options & OPT_IMPLIED_END else 1)
    bt_stride = _table_width(block_table)
    st = load_library().pmg_gather_ex(
        _ptr(cache), cache.stride(0), cache.stride(1), cache.shape[0],
        _ptr(block_table), bt_stride, _ptr(cu_seq_lens), _ptr(seq_starts), int(num_reqs),
        dst.shape[0], cache.shape[1], cache.shape[2], src_code, dst_code, _ptr(scale),
        _ptr(dst), dst.stride(0), _ptr(error_flag), _ptr(workspace),
        _stream_handle(stream), int(options))
    if st != PMG_OK:
        raise PmgError(st, "pmg_gather")


def gather_noalloc(cache: torch.Tensor, dst: torch.Tensor, block_table: torch.Tensor, cu_seq_lens: torch.Tensor,
                   seq_starts: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None,
                   error_flag: Optional[torch.Tensor] = None, num_reqs: Optional[int] = None, stream=None) -> None:
    """gather() for callers that cannot allocate device memory: the dynamic
    work split runs on the library's own static scratch instead of a caller
    workspace (pmg_gather_noalloc). Calls that overlap on the GPU must not use
    it concurrently; make the first call on a device outside stream capture."""
    src_code, dst_code = _layout(cache, dst)
    if num_reqs is None:
        num_reqs = cu_seq_lens.shape[0] - 1
    st = load_library().pmg_gather_noalloc(
        _ptr(cache), cache.stride(0), cache.stride(1), cache.shape[0],
        _ptr(block_table), _table_width(block_table), _ptr(cu_seq_lens), _ptr(seq_starts), int(num_reqs),
        dst.shape[0], cache.shape[1], cache.shape[2], src_code, dst_code, _ptr(scale),
        _ptr(dst), dst.stride(0), _ptr(error_flag), _stream_handle(stream))
    if st != PMG_OK:
        raise PmgError(st, "pmg_gather_noalloc")


def debug_noalloc_scratch() -> Tuple[int, int]:
    """(device address, int32 elements) of the static scratch that
    gather_noalloc uses on the current device (pmg_debug_noalloc_scratch); a
    test hook."""
    ptr = ctypes.c_void_p()
    n = ctypes.c_int64()
    st = load_library().pmg_debug_noalloc_scratch(ctypes.byref(ptr), ctypes.byref(n))
    if st != PMG_OK:
        raise PmgError(st, "pmg_debug_noalloc_scratch")
    return int(ptr.value), int(n.value)


def gather_tokens(cache: torch.Tensor, dst: torch.Tensor, block_table: torch.Tensor, token_to_seq: torch.Tensor,
                  cu_seq_lens: torch.Tensor, scale: Optional[torch.Tensor] = None,
                  error_flag: Optional[torch.Tensor] = None, num_reqs: Optional[int] = None, stream=None,
                  options: int = 0, workspace: Optional[torch.Tensor] = None) -> None:
    """Per-token indexed gather (pmg_gather_tokens): dst row t comes from
    request token_to_seq[t] at position t - cu_seq_lens[token_to_seq[t]].
    dst has num_tokens = len(token_to_seq) rows used. workspace as in gather()."""
    src_code, dst_code = _layout(cache, dst)
    if num_reqs is None:
        num_reqs = cu_seq_lens.shape[0] - 1
    st = load_library().pmg_gather_tokens(
        _ptr(cache), cache.stride(0), cache.stride(1), cache.shape[0],
        _ptr(block_table), _table_width(block_table), _ptr(token_to_seq), _ptr(cu_seq_lens), int(num_reqs),
        token_to_seq.shape[0], cache.shape[1], cache.shape[2], src_code, dst_code, _ptr(scale),
        _ptr(dst), dst.stride(0), _ptr(error_flag), _ptr(workspace), _stream_handle(stream), int(options))
    if st != PMG_OK:
        raise PmgError(st, "pmg_gather_tokens")


def new_workspace(device) -> torch.Tensor:
    """A zeroed scheduling workspace for gather(..., workspace=...). One per
    stream: concurrent calls must not share one."""
    return torch.zeros(WORKSPACE_INTS, dtype=torch.int32, device=device)


def select_path(cache: torch.Tensor, dst: torch.Tensor, block_table: torch.Tensor, cu_seq_lens: torch.Tensor,
                num_reqs: Optional[int] = None, options: int = 0) -> Tuple[str, int]:
    """The path and access width (elements) pmg_gather_ex would use. Host only:
    tensors may live anywhere, only their pointers' alignment is looked at."""
    src_code, dst_code = _layout(cache, dst)
    if num_reqs is None:
        num_reqs = cu_seq_lens.shape[0] - (0 if options & OPT_IMPLIED_END else 1)
    path = ctypes.c_int32(-1)
    unit = ctypes.c_int32(-1)
    bt_stride = _table_width(block_table)
    st = load_library().pmg_select_path(
        _ptr(cache), cache.stride(0), cache.stride(1), cache.shape[0], _ptr(block_table), bt_stride,
        _ptr(cu_seq_lens), int(num_reqs), dst.shape[0], cache.shape[1], cache.shape[2], src_code, dst_code,
        _ptr(dst), dst.stride(0), int(options),
        ctypes.byref(path), ctypes.byref(unit))
    if st != PMG_OK:
        raise PmgError(st, "pmg_select_path")
    return PATH_NAMES[path.value], unit.value


def debug_plan(cu_seq_lens: torch.Tensor, seq_starts: Optional[torch.Tensor], total_tokens: int, block_size: int,
               max_tasks: int, error_flag: Optional[torch.Tensor] = None, num_reqs: Optional[int] = None,
               stream=None, options: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Run the device page-task mapper alone. Returns (tasks int32 [max_tasks, 5],
    num_tasks int64 [1]) as device tensors; rows past num_tasks are untouched (-1)."""
    dev = cu_seq_lens.device
    if num_reqs is None:
        num_reqs = cu_seq_lens.shape[0] - (0 if options & OPT_IMPLIED_END else 1)
    tasks = torch.full((max(max_tasks, 0), 5), -1, dtype=torch.int32, device=dev)
    num = torch.full((1,), -1, dtype=torch.int64, device=dev)
    st = load_library().pmg_debug_plan(
        _ptr(cu_seq_lens), _ptr(seq_starts), int(num_reqs), int(total_tokens), int(block_size),
        _ptr(tasks) if max_tasks > 0 else None, int(max_tasks), _ptr(num), _ptr(error_flag),
        _stream_handle(stream), int(options))
    if st != PMG_OK:
        raise PmgError(st, "pmg_debug_plan")
    return tasks, num
