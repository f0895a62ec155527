"""The allocation-free entry point, pmg_gather_noalloc, against the regular one.

pmg_gather_noalloc exists for callers that cannot call cudaMalloc (an engine
that owns nearly all of HBM through its own pool, code inside a CUDA stream
capture, latency-bound paths): it runs the dynamic work split on a static
scratch array inside the library instead of a caller workspace. Its output must
equal pmg_gather_ex's with a workspace, bit for bit (a NaN matching any NaN for
converting gathers), on two calls in a row, since the second call starts from
whatever the first left in the shared scratch.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it; it passes alone in a fresh process
as well as after the rest.
"""
import numpy as np
import pytest
import torch

from paged_mla_kv_cache_gb300 import binding
from paged_mla_kv_cache_gb300 import workloads as W

from gpu_helpers import DeviceCase, assert_same

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    return cuda_lib


# single-60K and both skew-64 modes put at least 128 rows on every CTA, so
# the dynamic split (the part that uses the scratch) really runs
@pytest.mark.parametrize("name", ["60k", "skew64_raw", "skew64_dequant", "skew8", "tiny"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    wl = W.CONFIGS[name]()
    ref = DeviceCase(wl, workspace=True)
    ref.run()
    want, want_flag, want_guards = ref.result()
    assert want_guards and want_flag == 0

    case = DeviceCase(wl)
    for call in range(2):
        case.dst_full.view(torch.uint8).fill_(0xA5)
        binding.gather_noalloc(case.cache, case.dst, case.block_table, case.cu, case.seq_starts, case.scale,
                               case.err, num_reqs=wl.num_reqs)
        got, flag, guards = case.result()
        assert guards, f"call {call}: guard regions written"
        assert flag == 0, f"call {call}: flag {flag}"
        assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


def test_noalloc_large_batch_matches_workspace_entry_point():
    """More requests than one launch plans: the scratch also carries the verdict
    of the whole-array cu_seq_lens check."""
    rng = np.random.default_rng(65)
    R = binding.MAX_REQS_PLAN + 900
    lens = [int(x) for x in rng.integers(0, 20, R)]
    wl = W.make_workload("large", lens, [int(x) for x in rng.integers(0, 30, R)], 16, 64, None, "bf16", "bf16",
                         1.0, 65)
    ref = DeviceCase(wl, workspace=True)
    ref.run()
    want, want_flag, _ = ref.result()
    case = DeviceCase(wl)
    for _ in range(2):
        case.dst_full.view(torch.uint8).fill_(0xA5)
        binding.gather_noalloc(case.cache, case.dst, case.block_table, case.cu, case.seq_starts, case.scale,
                               case.err, num_reqs=wl.num_reqs)
        got, flag, guards = case.result()
        assert guards and flag == want_flag == 0
        assert_same(got, want, "bf16", False)


def test_noalloc_rejects_what_pmg_gather_rejects():
    wl = W.tiny()
    case = DeviceCase(wl)
    with pytest.raises(binding.PmgError) as e:
        binding.gather_noalloc(case.cache, case.dst, case.block_table, case.cu, num_reqs=binding.MAX_REQS + 1)
    assert e.value.status == 5  # PMG_ERR_UNSUPPORTED
