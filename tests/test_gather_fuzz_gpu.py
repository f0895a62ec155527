"""Randomized GPU parity: many small random gathers across every path and
option, each compared with the oracle element by element (tolerance 0, NaN
matches NaN for converting gathers). Seeds are fixed, so a failure reproduces.

Each case draws: a dtype pair, block size, entry size, padded or dense rows on
either side, request lengths (zeros included), seq_starts or none, an offset
cu[0], total_tokens above or below the sum of lengths, a path option (default,
SIMT, scalar, early metadata) and whether a scheduling workspace is passed.
"""
import numpy as np
import pytest
import torch

from paged_mla_kv_cache_gb300 import binding
from paged_mla_kv_cache_gb300 import workloads as W

from gpu_helpers import DeviceCase, assert_same, oracle_run

pytestmark = pytest.mark.gpu

PAIRS = [("bf16", "bf16"), ("fp16", "fp16"), ("fp32", "fp32"), ("fp8_e4m3", "fp8_e4m3"), ("u8", "u8"),
         ("fp8_e4m3", "bf16"), ("fp8_e4m3", "fp16"), ("fp8_e4m3", "fp32"), ("bf16", "fp32"), ("fp16", "fp32")]
OPTIONS = [0, binding.OPT_FORCE_SIMT, binding.OPT_FORCE_SCALAR, binding.OPT_EARLY_METADATA]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    return cuda_lib


def _case(seed):
    rng = np.random.default_rng(90_000 + seed)
    src, dst = PAIRS[int(rng.integers(0, len(PAIRS)))]
    B = int(rng.choice([1, 2, 5, 16, 64, 128]))
    E = int(rng.choice([1, 3, 8, 16, 64, 576]))
    row_stride = E + int(rng.choice([0, 0, 1, 8, 64]))
    dst_stride = E + int(rng.choice([0, 0, 3, 16]))
    R = int(rng.integers(1, 40))
    lens = [int(x) if rng.random() > 0.15 else 0 for x in rng.integers(0, 6 * B + 40, R)]
    starts = [int(x) for x in rng.integers(0, 3 * B + 1, R)] if rng.random() < 0.6 else None
    off = int(rng.integers(0, 5))
    total = off + sum(lens) + int(rng.integers(-min(sum(lens), 30), 6))
    wl = W.make_workload("fuzz", lens, starts, B, E, None, src, dst, float(rng.choice([1.0, 0.05, 3.0])),
                         90_000 + seed, row_stride=row_stride, cu_offset=off, total_tokens=max(total, 0))
    options = int(rng.choice(OPTIONS))
    workspace = bool(rng.random() < 0.5)
    return wl, dst_stride, options, workspace


@pytest.mark.parametrize("seed", range(300))
def test_random_gather(seed):
    wl, dst_stride, options, workspace = _case(seed)
    case = DeviceCase(wl, dst_row_stride=dst_stride, workspace=workspace)
    case.run(options=options)
    got, flag, guards = case.result()
    want, oflag = oracle_run(wl, dst_row_stride=dst_stride)
    assert guards, "guard regions written"
    assert flag == oflag
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


def _case_many(seed):
    """100 to 300 requests: several passes of the plan and its check, and both
    sides of the 256-request limit of the one-warp plan."""
    rng = np.random.default_rng(95_000 + seed)
    src, dst = PAIRS[int(rng.integers(0, len(PAIRS)))]
    B = int(rng.choice([1, 16, 64]))
    E = int(rng.choice([8, 64, 576]))
    R = int(rng.integers(100, 301))
    lens = [int(x) if rng.random() > 0.15 else 0 for x in rng.integers(0, 2 * B + 9, R)]
    starts = [int(x) for x in rng.integers(0, B + 1, R)] if rng.random() < 0.6 else None
    total = sum(lens) - int(rng.integers(0, 10))
    wl = W.make_workload("fuzz-many", lens, starts, B, E, None, src, dst, 0.05, 95_000 + seed,
                         total_tokens=max(total, 0))
    return wl, int(rng.choice(OPTIONS)), bool(rng.random() < 0.5)


@pytest.mark.parametrize("seed", range(30))
def test_random_gather_many_requests(seed):
    wl, options, workspace = _case_many(seed)
    case = DeviceCase(wl, workspace=workspace)
    case.run(options=options)
    got, flag, guards = case.result()
    want, oflag = oracle_run(wl)
    assert guards, "guard regions written"
    assert flag == oflag
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


@pytest.mark.parametrize("seed", range(40))
def test_random_gather_cu_not_non_decreasing(seed):
    """cu_seq_lens with random decreases (and now and then a negative first
    entry): requests after a decrease lose their rows or, when their rows would
    start below an earlier boundary, are skipped with flag 8; everything else
    is copied. Half the cases have more than 256 requests (the plan built by
    the whole CTA), the rest fewer (the one-warp plan)."""
    rng = np.random.default_rng(97_000 + seed)
    if seed % 2:
        wl, options, workspace = _case_many(seed + 100)
    else:
        wl, _, options, workspace = _case(seed + 500)
    cu = wl.cu_seq_lens.numpy().astype(np.int64)
    R = wl.num_reqs
    for _ in range(int(rng.integers(1, 4))):
        i = int(rng.integers(0, R + 1))
        cu[i] = cu[i] - int(rng.integers(1, 40)) if rng.random() < 0.8 else cu[i] + int(rng.integers(1, 10))
    if rng.random() < 0.2:
        cu[0] = -int(rng.integers(1, 5))
    cu = cu.astype(np.int32)
    case = DeviceCase(wl, cu=cu, workspace=workspace)
    case.run(options=options)
    got, flag, guards = case.result()
    want, oflag = oracle_run(wl, cu=cu)
    assert guards, "guard regions written"
    assert flag == oflag
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)
