"""GPU parity of the per-token indexed gather (pmg_gather_tokens) against the
oracle's per-token definition, element by element, tolerance 0 (NaN matches
NaN for converting gathers).

Source: "indexer kernels take shape arguments at run time" (prhub.com.cn, vllm
PR #56153), section "关键源码片段" (_cp_gather_indexer_quant_cache_kernel):
output token t reads request token_to_seq[t] at position t - cu_seqlen[b],
every index masked before use.
"""
import numpy as np
import pytest
import torch

from oracle import gather as og
from paged_mla_kv_cache_gb300 import binding
from paged_mla_kv_cache_gb300 import workloads as W

from gpu_helpers import GUARD_BYTES, FILL, assert_same

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    return cuda_lib


def token_to_seq_from_cu(cu: np.ndarray, T: int) -> np.ndarray:
    t2s = np.full(T, -1, np.int32)
    for r in range(len(cu) - 1):
        t2s[cu[r]:cu[r + 1]] = r
    return t2s


def _run(wl: W.Workload, t2s: np.ndarray, cu: np.ndarray, options=0, dst_row_stride=None, expect_flag=0,
         workspace=False):
    T = int(t2s.shape[0])
    ed = W.ELEM_BYTES[wl.dst_dtype]
    rs = wl.entry_size if dst_row_stride is None else dst_row_stride
    # oracle
    want = np.full((T, rs * ed), FILL, np.uint8).view(W.NP_BITS[ed])
    cache_bits = W.tensor_bits(wl.cache)
    cache_view = np.lib.stride_tricks.as_strided(cache_bits, shape=(cache_bits.shape[0], cache_bits.shape[1],
                                                                    wl.entry_size), strides=cache_bits.strides)
    oflag = og.gather_tokens(cache_view, wl.block_table.numpy(), t2s, cu, len(cu) - 1, T, wl.block_size,
                             wl.entry_size, wl.src_dtype, wl.dst_dtype, wl.scale, want)
    # device, with guard regions around dst
    dev = "cuda:0"
    full = wl.cache.to(dev)
    nbytes = T * rs * ed
    raw = torch.full((2 * GUARD_BYTES + nbytes,), FILL, dtype=torch.uint8, device=dev)
    body = raw[GUARD_BYTES:GUARD_BYTES + nbytes]
    dst_full = body.view(W.TORCH_DTYPES[wl.dst_dtype]).view(T, rs)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = binding.new_workspace(dev) if workspace else None
    binding.gather_tokens(full[:, :, :wl.entry_size], dst_full[:, :wl.entry_size], wl.block_table.to(dev),
                          torch.from_numpy(t2s).to(dev), torch.from_numpy(cu).to(dev),
                          torch.tensor([wl.scale], dtype=torch.float32, device=dev), err, num_reqs=len(cu) - 1,
                          options=options, workspace=ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert int(ws.abs().sum().item()) == 0, f"workspace not reset: {ws.tolist()}"
    r = raw.cpu().numpy()
    assert np.all(r[:GUARD_BYTES] == FILL) and np.all(r[-GUARD_BYTES:] == FILL), "guard regions written"
    got = r[GUARD_BYTES:len(r) - GUARD_BYTES].view(W.NP_BITS[ed]).reshape(T, rs)
    assert oflag == expect_flag
    assert int(err.item()) == oflag
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


def _consistent(wl):
    cu = wl.cu_seq_lens.numpy().copy()
    return token_to_seq_from_cu(cu, int(cu[-1])), cu


@pytest.mark.parametrize("name", ["tiny", "60k", "skew8", "skew64_raw", "skew64_dequant"])
@pytest.mark.parametrize("options", [0, binding.OPT_FORCE_SIMT, binding.OPT_FORCE_SCALAR,
                                     binding.OPT_EARLY_METADATA])
def test_named_workloads(name, options):
    wl = W.CONFIGS[name]()
    if wl.seq_starts is not None:  # the per-token gather has no seq_starts: positions start at 0
        wl = W.make_workload(wl.name, wl.lens, None, wl.block_size, wl.entry_size, wl.num_blocks, wl.src_dtype,
                             wl.dst_dtype, wl.scale, 77, row_stride=wl.cache.shape[2])
    t2s, cu = _consistent(wl)
    _run(wl, t2s, cu, options=options, workspace=options == binding.OPT_EARLY_METADATA)


PAIRS = [("bf16", "bf16"), ("fp32", "fp32"), ("u8", "u8"), ("fp8_e4m3", "bf16"), ("fp8_e4m3", "fp16"),
         ("fp8_e4m3", "fp32"), ("bf16", "fp32"), ("fp16", "fp32")]


@pytest.mark.parametrize("src,dst", PAIRS)
@pytest.mark.parametrize("B,E,rs", [(16, 576, None), (64, 576, 640), (3, 7, None), (1, 8, 9), (4, 16, None)])
@pytest.mark.parametrize("options", [0, binding.OPT_FORCE_SIMT])
def test_dtype_shapes(src, dst, B, E, rs, options):
    rng = np.random.default_rng(B * 100 + E)
    lens = [int(x) for x in rng.integers(0, 5 * B + 9, 7)]
    wl = W.make_workload("tok", lens, None, B, E, None, src, dst, 0.05, 31, row_stride=rs)
    t2s, cu = _consistent(wl)
    _run(wl, t2s, cu, options=options)


@pytest.mark.parametrize("dtypes", [("bf16", "bf16"), ("fp8_e4m3", "bf16")])
@pytest.mark.parametrize("B", [1, 16, 64])
def test_identity_table_runs_cross_pages(dtypes, B):
    """Physically consecutive blocks: adjacent source rows run across page
    boundaries and across requests, so one bulk copy spans several pages."""
    lens = [0, 3 * B + 5, 1, 0, 7 * B, 2 * B - 1, 40]
    need = [-(-L // B) for L in lens]
    nb = sum(need) + 2
    wl = W.make_workload("tok", lens, None, B, 576, nb, dtypes[0], dtypes[1], 0.05, 39)
    bt = np.full((len(lens), max(need)), -1, np.int32)
    pos = 1
    for r, n in enumerate(need):
        bt[r, :n] = np.arange(pos, pos + n, dtype=np.int32)
        pos += n
    wl.block_table = torch.from_numpy(bt)
    t2s, cu = _consistent(wl)
    _run(wl, t2s, cu)


@pytest.mark.parametrize("seed", range(6))
def test_invalid_tokens_break_runs(seed):
    """Invalid tokens scattered through contiguous runs: the runs split around
    them and only the valid rows are written."""
    rng = np.random.default_rng(400 + seed)
    wl = W.make_workload("tok", [int(x) for x in rng.integers(1, 300, 9)], None, 64, 576, None, "bf16", "bf16",
                         1.0, 41 + seed)
    t2s, cu = _consistent(wl)
    t2s = t2s.copy()
    idx = rng.choice(len(t2s), max(1, len(t2s) // 17), replace=False)
    t2s[idx] = rng.choice([-1, 9, 100], idx.shape[0]).astype(np.int32)
    _run(wl, t2s, cu, expect_flag=og.BAD_TOKEN, workspace=bool(seed % 2))


def test_invalid_tokens_are_skipped_and_flagged():
    wl = W.make_workload("tok", [40, 30, 25, 50], None, 16, 64, None, "bf16", "bf16", 1.0, 33)
    t2s, cu = _consistent(wl)
    rng = np.random.default_rng(34)
    idx = rng.choice(len(t2s), 20, replace=False)
    t2s = t2s.copy()
    t2s[idx[:5]] = -3                         # request id below range
    t2s[idx[5:10]] = 4                        # request id past num_reqs
    t2s[idx[10:20]] = (t2s[idx[10:20]] + 1) % 4  # a real request whose rows do not contain t
    _run(wl, t2s, cu, expect_flag=og.BAD_TOKEN)


def test_block_bounds_flags():
    wl = W.make_workload("tok", [40, 30, 25], None, 16, 64, None, "bf16", "bf16", 1.0, 35)
    t2s, cu = _consistent(wl)
    bt = wl.block_table.numpy().copy()
    bt[1, 1] = -1
    wl.block_table = torch.from_numpy(bt)
    _run(wl, t2s, cu, expect_flag=og.BAD_PHYS)
    wl2 = W.make_workload("tok", [40, 30, 25], None, 16, 64, None, "bf16", "bf16", 1.0, 36)
    cu2 = wl2.cu_seq_lens.numpy().copy()
    cu2[2:] += 30  # request 1 now owns 60 rows, past its 2-wide table row
    t2s2 = token_to_seq_from_cu(cu2, int(cu2[-1]))
    _run(wl2, t2s2, cu2, expect_flag=og.BAD_LOGICAL | og.BAD_PHYS)


def test_no_requests_every_token_flagged():
    wl = W.make_workload("tok", [10], None, 16, 64, None, "bf16", "bf16", 1.0, 37)
    _run(wl, np.zeros(10, np.int32), np.array([0], np.int32), expect_flag=og.BAD_TOKEN)


@pytest.mark.parametrize("workspace", [False, True])
def test_single_300k_tokens(workspace):
    """300K tokens of one request through the per-token path (with a
    workspace: the dynamic row split)."""
    wl = W.single_300k()
    t2s, cu = _consistent(wl)
    _run(wl, t2s, cu, workspace=workspace)


@pytest.mark.parametrize("T", [500_000, 1_000_000])
def test_many_small_rows_use_the_larger_tiles(T):
    """Enough tokens for 16- and 32-token warp tiles (small calls use 8)."""
    rng = np.random.default_rng(T % 97)
    lens = [int(x) for x in rng.integers(1, 2 * T // 50, 50)]
    lens[-1] += T - sum(lens) if T > sum(lens) else 0
    wl = W.make_workload("tok", lens, None, 64, 8, None, "fp8_e4m3", "bf16", 0.05, 38)
    t2s, cu = _consistent(wl)
    _run(wl, t2s, cu)
