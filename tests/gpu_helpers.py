"""Shared helpers of the GPU parity tests: run one workload through the CUDA
library (via the binding) and through the CPU oracle on the same inputs, with
sentinel-filled destinations and guard regions around the device output."""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np
import torch

from oracle import gather as og
from paged_mla_kv_cache_gb300 import binding
from paged_mla_kv_cache_gb300.workloads import ELEM_BYTES, NP_BITS, TORCH_DTYPES, Workload, tensor_bits

GUARD_BYTES = 4096
FILL = 0xA5


def oracle_run(wl: Workload, dst_row_stride: Optional[int] = None, cu: Optional[np.ndarray] = None,
               seq_starts: Optional[np.ndarray] = "wl", block_table: Optional[np.ndarray] = None,
               total_tokens: Optional[int] = None) -> Tuple[np.ndarray, int]:
    """Oracle output as raw bits [T, row_stride] (sentinel-filled) and its flag."""
    ed = ELEM_BYTES[wl.dst_dtype]
    rs = wl.entry_size if dst_row_stride is None else dst_row_stride
    T = wl.total_tokens if total_tokens is None else total_tokens
    dst = np.full((T, rs * ed), FILL, dtype=np.uint8).view(NP_BITS[ed])
    cache = tensor_bits(wl.cache)
    cache = cache[:, :, :]  # [nb, B, row_stride] view with the padded stride
    cache_view = np.lib.stride_tricks.as_strided(
        cache, shape=(cache.shape[0], cache.shape[1], wl.entry_size), strides=cache.strides)
    ss = (None if wl.seq_starts is None else wl.seq_starts.numpy()) if isinstance(seq_starts, str) else seq_starts
    flag = og.gather(cache_view, wl.block_table.numpy() if block_table is None else block_table,
                     wl.cu_seq_lens.numpy() if cu is None else cu, ss, wl.num_reqs, T, wl.block_size,
                     wl.entry_size, wl.src_dtype, wl.dst_dtype, wl.scale, dst)
    return dst, flag


class DeviceCase:
    """A workload moved to the GPU with a guarded, sentinel-filled destination."""

    def __init__(self, wl: Workload, dst_row_stride: Optional[int] = None, device: str = "cuda:0",
                 cu: Optional[np.ndarray] = None, seq_starts="wl", block_table: Optional[np.ndarray] = None,
                 total_tokens: Optional[int] = None, with_scale: bool = True, workspace: bool = False):
        self.wl = wl
        self.device = device
        ed = ELEM_BYTES[wl.dst_dtype]
        self.rs = wl.entry_size if dst_row_stride is None else dst_row_stride
        self.T = wl.total_tokens if total_tokens is None else total_tokens
        # cache: full padded tensor, then a [nb, B, E] view
        full = wl.cache.to(device)
        self.cache_full = full
        self.cache = full[:, :, :wl.entry_size]
        self.block_table = (wl.block_table if block_table is None else torch.from_numpy(block_table)).to(device)
        self.cu = (wl.cu_seq_lens if cu is None else torch.from_numpy(cu)).to(device)
        if isinstance(seq_starts, str):
            self.seq_starts = None if wl.seq_starts is None else wl.seq_starts.to(device)
        else:
            self.seq_starts = None if seq_starts is None else torch.from_numpy(seq_starts).to(device)
        self.scale = torch.tensor([wl.scale], dtype=torch.float32, device=device) if with_scale else None
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws = binding.new_workspace(device) if workspace else None
        nbytes = self.T * self.rs * ed
        self.raw = torch.full((GUARD_BYTES * 2 + nbytes,), FILL, dtype=torch.uint8, device=device)
        body = self.raw[GUARD_BYTES:GUARD_BYTES + nbytes]
        self.dst_full = body.view(TORCH_DTYPES[wl.dst_dtype] if wl.dst_dtype != "u8" else torch.uint8).view(
            self.T, self.rs)
        self.dst = self.dst_full[:, :wl.entry_size]

    def run(self, options: int = 0, stream=None) -> None:
        binding.gather(self.cache, self.dst, self.block_table, self.cu, self.seq_starts, self.scale, self.err,
                       num_reqs=self.wl.num_reqs, stream=stream, options=options, workspace=self.ws)

    def result(self) -> Tuple[np.ndarray, int, bool]:
        """(dst bits [T, row_stride], flag, guards intact)."""
        torch.cuda.synchronize(self.device)
        raw = self.raw.cpu().numpy()
        guards_ok = bool(np.all(raw[:GUARD_BYTES] == FILL) and np.all(raw[-GUARD_BYTES:] == FILL))
        if self.ws is not None:
            assert int(self.ws.abs().sum().item()) == 0, f"workspace not reset: {self.ws.tolist()}"
        ed = ELEM_BYTES[self.wl.dst_dtype]
        body = raw[GUARD_BYTES:len(raw) - GUARD_BYTES].view(NP_BITS[ed]).reshape(self.T, self.rs)
        return body, int(self.err.item()), guards_ok


def nan_mask(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)
    if dtype == "fp16":
        return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)
    if dtype == "fp32":
        return ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x007FFFFF) != 0)
    return np.zeros(bits.shape, dtype=bool)


def assert_same(got: np.ndarray, want: np.ndarray, dtype: str, converting: bool) -> None:
    """Bit-exact equality; for a converting gather, NaN matches NaN whatever the payload."""
    assert got.shape == want.shape
    if converting:
        gn, wn = nan_mask(got, dtype), nan_mask(want, dtype)
        assert np.array_equal(gn, wn), "NaN positions differ"
        diff = (got != want) & ~gn
    else:
        diff = got != want
    n = int(np.count_nonzero(diff))
    if n:
        idx = np.argwhere(diff)[:5]
        raise AssertionError(f"{n} elements differ; first at {idx.tolist()}: got "
                             f"{[hex(int(got[tuple(i)])) for i in idx]} want {[hex(int(want[tuple(i)])) for i in idx]}")
