"""Seeded synthetic inputs for the paged MLA KV-cache gather.

This module only draws inputs: caches, block tables, cu_seq_lens and
seq_starts. It holds none of the gather's arithmetic, and both the CUDA path
and the CPU oracle read the same arrays it returns.

The shapes follow "MLA cache gather scheduled per logical page" (prhub.com.cn,
vllm PR #51739): block_size 64 and 576-element MLA entries, uneven request
lengths such as {17, 32768, 71} with starts {3, 17, 5}, and shuffled physical
blocks (section "关键源码片段", the test
test_cp_gather_cache_mla_large_uneven_sequences), plus the single-60K,
single-300K and skewed scenarios of the benchmark named in section "实现拆解"
item 4. All data are synthetic: there is no dataset.

Conventions:
- A request's block-table row covers its whole context from token 0, so row r
  holds ceil((start_r + len_r) / block_size) valid block ids; unused entries
  are -1.
- Multi-request tables take consecutive slices of one seeded permutation of
  the physical blocks, so no cache row is read twice.
- Values: bf16 caches are N(0, 1); fp8 caches hold clamp(N(0, 1) / scale,
  -448, 448) cast to float8_e4m3fn (no NaN codes).
- Seeds: base 20261202 plus a per-workload index.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

SEED_BASE = 20261202

TORCH_DTYPES = {
    "bf16": torch.bfloat16,
    "fp16": torch.float16,
    "fp32": torch.float32,
    "fp8_e4m3": torch.float8_e4m3fn,
    "u8": torch.uint8,
}
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp32": 4, "fp8_e4m3": 1, "u8": 1}
# numpy dtype of the same width, for handing raw bits to host code
NP_BITS = {1: np.uint8, 2: np.uint16, 4: np.uint32}


@dataclasses.dataclass
class Workload:
    name: str
    cache: torch.Tensor            # [num_blocks, block_size, row_stride], src dtype, CPU
    block_table: torch.Tensor      # int32 [num_reqs, block_table_stride], CPU
    cu_seq_lens: torch.Tensor      # int32 [num_reqs + 1], CPU
    seq_starts: Optional[torch.Tensor]  # int32 [num_reqs] or None, CPU
    lens: List[int]
    num_reqs: int
    total_tokens: int
    block_size: int
    entry_size: int
    src_dtype: str
    dst_dtype: str
    scale: float = 1.0

    @property
    def num_blocks(self) -> int:
        return int(self.cache.shape[0])

    @property
    def rows(self) -> int:
        """Output rows the call defines: sum of request lengths."""
        return int(sum(self.lens))

    def algorithmic_bytes(self) -> int:
        """Bytes read plus bytes written per call, counting only the entries
        (no padding, no block table)."""
        return self.rows * self.entry_size * (ELEM_BYTES[self.src_dtype] + ELEM_BYTES[self.dst_dtype])

    def cache_bits(self) -> np.ndarray:
        """The cache as an unsigned-integer numpy array of the element width (a view)."""
        return tensor_bits(self.cache)

    def new_dst(self, fill_byte: int = 0xA5, row_stride: Optional[int] = None) -> np.ndarray:
        """A host destination [total_tokens, row_stride] filled with a sentinel byte."""
        ed = ELEM_BYTES[self.dst_dtype]
        rs = self.entry_size if row_stride is None else row_stride
        buf = np.full((self.total_tokens, rs * ed), fill_byte, dtype=np.uint8)
        return buf.view(NP_BITS[ed])


def tensor_bits(t: torch.Tensor) -> np.ndarray:
    """Reinterpret a CPU tensor as a numpy array of unsigned integers of the same width."""
    es = t.element_size()
    as_int = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[es]
    return t.view(as_int).numpy().view(NP_BITS[es])


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _fill_cache(shape, src_dtype: str, scale: float, seed: int) -> torch.Tensor:
    g = _gen(seed)
    if src_dtype == "u8":
        return torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    vals = torch.randn(shape, generator=g, dtype=torch.float32)
    if src_dtype == "fp8_e4m3":
        vals = (vals / scale).clamp_(-448.0, 448.0)
    return vals.to(TORCH_DTYPES[src_dtype])


def pages_to_hold(start: int, length: int, block_size: int) -> int:
    """Blocks a request's table row needs to hold tokens [0, start + length)."""
    return -(-(start + length) // block_size)


def _table_from_permutation(perm: np.ndarray, need: List[int]) -> np.ndarray:
    stride = max(max(need), 1)
    bt = np.full((len(need), stride), -1, dtype=np.int32)
    pos = 0
    for r, n in enumerate(need):
        bt[r, :n] = perm[pos:pos + n]
        pos += n
    assert pos <= perm.shape[0], "not enough physical blocks for the requested lengths"
    return bt


def make_workload(name: str, lens: List[int], starts: Optional[List[int]], block_size: int, entry_size: int,
                  num_blocks: Optional[int], src_dtype: str, dst_dtype: str, scale: float, seed: int,
                  row_stride: Optional[int] = None, independent_rows: bool = False,
                  cu_offset: int = 0, total_tokens: Optional[int] = None) -> Workload:
    """Build one workload. num_blocks None picks the smallest multiple of 1024
    (or of 64 below 1024 blocks) that holds every request."""
    rng = np.random.default_rng(seed)
    R = len(lens)
    st = [0] * R if starts is None else list(starts)
    need = [pages_to_hold(st[r], lens[r], block_size) for r in range(R)]
    if num_blocks is None:
        total_need = max(max(need) if independent_rows else sum(need), 1)
        unit = 1024 if total_need > 1024 else 64
        num_blocks = -(-total_need // unit) * unit
    if independent_rows:
        bt = np.stack([rng.permutation(num_blocks).astype(np.int32) for _ in range(R)]) if R else np.zeros((0, 1), np.int32)
    else:
        bt = _table_from_permutation(rng.permutation(num_blocks).astype(np.int32), need) if R else np.zeros((0, 1), np.int32)
    cu = np.zeros(R + 1, dtype=np.int64)
    cu[0] = cu_offset
    cu[1:] = cu_offset + np.cumsum(lens)
    T = int(cu[-1]) if total_tokens is None else int(total_tokens)
    rs = entry_size if row_stride is None else row_stride
    cache = _fill_cache((num_blocks, block_size, rs), src_dtype, scale, seed + 7919)
    return Workload(
        name=name, cache=cache, block_table=torch.from_numpy(bt),
        cu_seq_lens=torch.from_numpy(cu.astype(np.int32)),
        seq_starts=None if starts is None else torch.tensor(st, dtype=torch.int32),
        lens=list(lens), num_reqs=R, total_tokens=T, block_size=block_size, entry_size=entry_size,
        src_dtype=src_dtype, dst_dtype=dst_dtype, scale=scale)


# --- the five named workloads -------------------------------------------------

def tiny(seed: int = SEED_BASE + 0) -> Workload:
    """4 requests {17, 71, 130, 0}, no starts, B=64, 576 bf16, 64 blocks; T=218."""
    return make_workload("tiny raw gather", [17, 71, 130, 0], None, 64, 576, 64, "bf16", "bf16", 1.0, seed)


def single_60k(seed: int = SEED_BASE + 1) -> Workload:
    """1 request of 60,000 tokens, B=64, 576 bf16, 1024 shuffled blocks."""
    return make_workload("single-60K raw gather", [60000], None, 64, 576, 1024, "bf16", "bf16", 1.0, seed)


def single_300k(seed: int = SEED_BASE + 2) -> Workload:
    """1 request of 300,000 tokens, B=64, 576 bf16, 5000 shuffled blocks."""
    return make_workload("single-300K raw gather", [300000], None, 64, 576, 5000, "bf16", "bf16", 1.0, seed)


SKEW8_LENS = [32768, 17, 71, 4096, 1, 513, 0, 8191]


def skew8(seed: int = SEED_BASE + 3) -> Workload:
    """8 requests, starts uniform in [0, 200], fp8 e4m3 (scale 0.05) -> bf16, 1024 blocks."""
    rng = np.random.default_rng(seed + 1)
    starts = rng.integers(0, 201, len(SKEW8_LENS)).tolist()
    return make_workload("skew-8 fp8 upconvert", SKEW8_LENS, starts, 64, 576, 1024, "fp8_e4m3", "bf16", 0.05, seed)


def skew64_lens(seed: int) -> List[int]:
    """64 log-uniform lengths in [1, 32768] with 4 forced to zero."""
    rng = np.random.default_rng(seed + 2)
    u = rng.uniform(0.0, math.log(32768.0), 64)
    lens = np.clip(np.round(np.exp(u)), 1, 32768).astype(np.int64)
    zero = rng.choice(64, 4, replace=False)
    lens[zero] = 0
    return [int(x) for x in lens]


def skew64(mode: str = "raw", seed: int = SEED_BASE + 4) -> Workload:
    """64 requests, starts in [0, 200], entries in a padded 640-element row
    stride; mode 'raw' (bf16 copy) or 'dequant' (fp8 e4m3, scale 0.02 -> bf16)."""
    lens = skew64_lens(seed)
    rng = np.random.default_rng(seed + 1)
    starts = rng.integers(0, 201, 64).tolist()
    if mode == "raw":
        return make_workload("skew-64 mixed raw", lens, starts, 64, 576, None, "bf16", "bf16", 1.0, seed,
                             row_stride=640)
    if mode == "dequant":
        return make_workload("skew-64 mixed dequant", lens, starts, 64, 576, None, "fp8_e4m3", "bf16", 0.02,
                             seed, row_stride=640)
    raise ValueError(mode)


def fp32_1m(seed: int = SEED_BASE + 6) -> Workload:
    """1 request of 1,000,000 tokens of 576 fp32 elements (2304 bytes per
    entry), raw copy, B=64, 16384 shuffled blocks: the output passes 2^31 bytes
    after about 932K rows, where the review section ("评论区精华") of the page
    reports int32 overflow of output_token_begin * entry_bytes."""
    return make_workload("fp32-1M raw gather", [1_000_000], None, 64, 576, 16384, "fp32", "fp32", 1.0, seed)


def p1test(cache_dtype: str = "bf16", use_seq_starts: bool = True, seed: int = SEED_BASE + 5) -> Workload:
    """The page's uneven test: lens {17, 32768, 71}, starts {3, 17, 5}, 1024
    blocks, every table row an independent permutation of all blocks.
    cache_dtype 'bf16' copies bf16; 'fp8_e4m3' copies the fp8 bytes."""
    starts = [3, 17, 5] if use_seq_starts else None
    return make_workload("P1 uneven test", [17, 32768, 71], starts, 64, 576, 1024, cache_dtype, cache_dtype,
                         1.0, seed, independent_rows=True)


CONFIGS: Dict[str, object] = {
    "tiny": tiny,
    "60k": single_60k,
    "300k": single_300k,
    "skew8": skew8,
    "skew64_raw": lambda: skew64("raw"),
    "skew64_dequant": lambda: skew64("dequant"),
    "fp32_1m": fp32_1m,
}
