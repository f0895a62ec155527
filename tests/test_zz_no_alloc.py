"""The allocation-free entry point, pmg_gather_noalloc, on the GPU.

pmg_gather_noalloc exists for callers that may not call cudaMalloc: a serving
engine that reserves nearly all of HBM for its own KV-cache pool at start-up,
a plugin inside a framework that owns every allocation, a latency-bound path
that cannot take cudaMalloc's implicit device synchronisation. It runs the
dynamic work split on a static scratch array inside the library instead of a
caller workspace. Its output must equal the CPU oracle's and pmg_gather_ex's
(with a workspace) bit for bit, a NaN matching any NaN for converting gathers,
on two calls in a row, since the second call starts from whatever the first
left in the shared scratch; and a call must start from a cleared claim counter
even when the scratch holds stale values.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it; it passes alone in a fresh process
as well as after the rest.
"""
import os

import numpy as np
import pytest
import torch

from paged_mla_kv_cache_gb300 import binding
from paged_mla_kv_cache_gb300 import workloads as W

from gpu_helpers import DeviceCase, assert_same, oracle_run

pytestmark = pytest.mark.gpu

# the dynamic split engages when a CTA owns at least this many rows (the
# library's default; PMG_SCHED_MIN_ROWS would change it)
MIN_ROWS_DYNAMIC = 32
# an upper bound on resident CTAs per SM of the TMA kernels (shared memory
# keeps them at 2 for byte copies and at 4 or 5 for converting gathers)
MAX_CTAS_PER_SM = 8


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    return cuda_lib


def _dynamic_split_runs(wl) -> bool:
    """Whether every CTA of the launch owns enough rows for the dynamic split
    (the part of the work split that uses the scratch)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return wl.rows // (MAX_CTAS_PER_SM * sms) >= MIN_ROWS_DYNAMIC


def _noalloc(case, wl):
    binding.gather_noalloc(case.cache, case.dst, case.block_table, case.cu, case.seq_starts, case.scale,
                           case.err, num_reqs=wl.num_reqs)


@pytest.mark.parametrize("name,dynamic", [("60k", True), ("skew64_raw", True), ("skew64_dequant", True),
                                          ("skew8", True), ("tiny", False)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(name, dynamic):
    assert "PMG_SCHED_MIN_ROWS" not in os.environ
    wl = W.CONFIGS[name]()
    converting = wl.src_dtype != wl.dst_dtype
    case = DeviceCase(wl)
    path, _ = binding.select_path(case.cache, case.dst, case.block_table, case.cu, num_reqs=wl.num_reqs)
    assert path == "bulk"
    assert _dynamic_split_runs(wl) == dynamic

    want, oflag = oracle_run(wl)
    assert oflag == 0
    ref = DeviceCase(wl, workspace=True)
    ref.run()
    ref_out, ref_flag, ref_guards = ref.result()
    assert ref_guards and ref_flag == 0

    for call in range(2):
        case.dst_full.view(torch.uint8).fill_(0xA5)
        _noalloc(case, wl)
        got, flag, guards = case.result()
        assert guards, f"call {call}: guard regions written"
        assert flag == 0, f"call {call}: flag {flag}"
        assert_same(got, want, wl.dst_dtype, converting)
        assert_same(got, ref_out, wl.dst_dtype, converting)


class _DeviceInts:
    """A raw device int32 array seen as a torch tensor (no copy)."""

    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False), "version": 3}


@pytest.mark.parametrize("name", ["60k", "skew8"])
def test_noalloc_starts_from_a_cleared_counter_over_stale_scratch(name):
    """Stale values in the shared scratch (a counter far past the last item)
    would make every claim fail; the call clears the counter on its stream
    before the launch, so the output is still complete."""
    wl = W.CONFIGS[name]()
    assert _dynamic_split_runs(wl)
    want, _ = oracle_run(wl)
    case = DeviceCase(wl)
    ptr, n = binding.debug_noalloc_scratch()
    assert n >= binding.WORKSPACE_INTS
    scratch = torch.as_tensor(_DeviceInts(ptr, n), device="cuda:0")
    for call in range(2):
        torch.cuda.synchronize()
        scratch.fill_(0x7FFFFFFF)
        case.dst_full.view(torch.uint8).fill_(0xA5)
        _noalloc(case, wl)
        got, flag, guards = case.result()
        assert guards and flag == 0, (call, flag)
        assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


def test_noalloc_large_batch_matches_oracle_and_workspace_entry_point():
    """More requests than one launch plans: the scratch also carries what the
    launches over groups of requests pass on."""
    rng = np.random.default_rng(65)
    R = binding.MAX_REQS_PLAN + 900
    lens = [int(x) for x in rng.integers(0, 20, R)]
    wl = W.make_workload("large", lens, [int(x) for x in rng.integers(0, 30, R)], 16, 64, None, "bf16", "bf16",
                         1.0, 65)
    want, oflag = oracle_run(wl)
    assert oflag == 0
    ref = DeviceCase(wl, workspace=True)
    ref.run()
    ref_out, ref_flag, _ = ref.result()
    case = DeviceCase(wl)
    for _ in range(2):
        case.dst_full.view(torch.uint8).fill_(0xA5)
        _noalloc(case, wl)
        got, flag, guards = case.result()
        assert guards and flag == ref_flag == 0
        assert_same(got, want, "bf16", False)
        assert_same(got, ref_out, "bf16", False)


def test_noalloc_rejects_what_pmg_gather_rejects():
    wl = W.tiny()
    case = DeviceCase(wl)
    with pytest.raises(binding.PmgError) as e:
        binding.gather_noalloc(case.cache, case.dst, case.block_table, case.cu, num_reqs=binding.MAX_REQS + 1)
    assert e.value.status == 5  # PMG_ERR_UNSUPPORTED
