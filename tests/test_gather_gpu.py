"""GPU parity: the CUDA gather against the CPU oracle, element by element.

Source of the operation: "MLA cache gather scheduled per logical page"
(prhub.com.cn, vllm PR #51739): section "关键源码片段" (the uneven-length
test and the page mapper), section "实现拆解" items 1 and 3 (raw copy, FP8
upconvert and maybe-dequant; long uneven requests, seq_starts on and off,
shuffled blocks, partial pages, unaligned strides, zero-length requests) and
the review section "评论区精华" (block-table bounds and int32 overflow).

Tolerance: 0. Byte copies must match bit for bit; converting gathers must too,
except that a NaN matches any NaN (no workload below draws NaN codes except
the all-codes test).
"""
import numpy as np
import pytest
import torch

from oracle import gather as og
from oracle import plan as op
from paged_mla_kv_cache_gb300 import binding
from paged_mla_kv_cache_gb300 import workloads as W

from gpu_helpers import GUARD_BYTES, DeviceCase, assert_same, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    return cuda_lib


def _check(wl, options=0, dst_row_stride=None, expect_flag=0, workspace=False, **kw):
    case = DeviceCase(wl, dst_row_stride=dst_row_stride, workspace=workspace, **kw)
    case.run(options=options)
    got, flag, guards = case.result()
    want, oflag = oracle_run(wl, dst_row_stride=dst_row_stride, **{k: v for k, v in kw.items()
                                                                    if k in ("cu", "seq_starts", "block_table",
                                                                             "total_tokens")})
    assert guards, "guard regions around dst were written"
    assert oflag == expect_flag
    assert flag == oflag, f"device flag {flag} != oracle flag {oflag}"
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)
    return case


# --- the five named workloads at full size, in the launch configuration the
# benchmark times ------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "60k", "300k", "skew8", "skew64_raw", "skew64_dequant"])
@pytest.mark.parametrize("workspace", [False, True])
def test_named_workloads_full_size(name, workspace):
    wl = W.CONFIGS[name]()
    _check(wl, workspace=workspace)


@pytest.mark.parametrize("name", ["60k", "skew8", "skew64_dequant"])
def test_workspace_reuse_across_calls_and_graph_replays(name):
    """A workspace serves back-to-back calls (each leaves it zeroed), also when
    the calls are replayed from a CUDA graph."""
    wl = W.CONFIGS[name]()
    case = DeviceCase(wl, workspace=True)
    for _ in range(5):
        case.run()
    want, _ = oracle_run(wl)
    got, flag, guards = case.result()
    assert guards and flag == 0
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)
    case.dst_full.view(torch.uint8).fill_(0xA5)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream()
        for _ in range(3):
            case.run(stream=s)
    for _ in range(4):
        g.replay()
    got, flag, guards = case.result()
    assert guards and flag == 0
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


@pytest.mark.parametrize("name", ["tiny", "60k", "300k", "skew8", "skew64_raw", "skew64_dequant"])
@pytest.mark.parametrize("workspace", [False, True])
def test_named_workloads_early_metadata(name, workspace):
    """PMG_OPT_EARLY_METADATA: the plan runs before the previous grid is done;
    the result is the same."""
    _check(W.CONFIGS[name](), options=binding.OPT_EARLY_METADATA, workspace=workspace)


@pytest.mark.parametrize("name", ["60k", "skew8", "skew64_dequant"])
def test_early_metadata_back_to_back_graph(name):
    """Back-to-back calls replayed from a CUDA graph with early metadata: each
    call overlaps the previous one's tail; outputs and the workspace stay right."""
    wl = W.CONFIGS[name]()
    want, _ = oracle_run(wl)
    case = DeviceCase(wl, workspace=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream()
        for _ in range(4):
            case.run(options=binding.OPT_EARLY_METADATA, stream=s)
    for _ in range(3):
        g.replay()
    got, flag, guards = case.result()
    assert guards and flag == 0
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


@pytest.mark.parametrize("name", ["tiny", "60k", "skew8", "skew64_raw"])
@pytest.mark.parametrize("options", [binding.OPT_FORCE_SIMT, binding.OPT_FORCE_SCALAR])
def test_named_workloads_other_paths(name, options):
    _check(W.CONFIGS[name](), options=options)


# --- the page's own uneven test ----------------------------------------------

@pytest.mark.parametrize("cache_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("use_seq_starts", [False, True])
def test_p1_uneven_lengths(cache_dtype, use_seq_starts):
    wl = W.p1test(cache_dtype, use_seq_starts)
    _check(wl)


# --- dtype matrix, block sizes, entry sizes, strides --------------------------

PAIRS = [("bf16", "bf16"), ("fp16", "fp16"), ("fp32", "fp32"), ("fp8_e4m3", "fp8_e4m3"), ("u8", "u8"),
         ("fp8_e4m3", "bf16"), ("fp8_e4m3", "fp16"), ("fp8_e4m3", "fp32"), ("bf16", "fp32"), ("fp16", "fp32")]


def _small(seed, src, dst, B, E, row_stride=None, starts=True, R=6, maxlen=None, scale=0.05):
    rng = np.random.default_rng(seed)
    maxlen = maxlen or 3 * B + 5
    lens = [int(x) for x in rng.integers(0, maxlen, R)]
    lens[int(rng.integers(0, R))] = 0
    st = [int(x) for x in rng.integers(0, 2 * B + 1, R)] if starts else None
    return W.make_workload("small", lens, st, B, E, None, src, dst, scale, seed, row_stride=row_stride)


@pytest.mark.parametrize("src,dst", PAIRS)
@pytest.mark.parametrize("B,E", [(1, 576), (16, 7), (64, 576), (128, 8), (16, 512), (64, 656), (3, 1)])
def test_dtype_block_entry_matrix(src, dst, B, E):
    seed = sum(map(ord, src + dst)) * 1000 + B * 10 + E
    wl = _small(seed, src, dst, B, E)
    _check(wl)
    _check(wl, workspace=True)


@pytest.mark.parametrize("src,dst", PAIRS)
@pytest.mark.parametrize("options", [0, binding.OPT_FORCE_SIMT, binding.OPT_FORCE_SCALAR])
def test_padded_rows_both_sides(src, dst, options):
    """Cache rows padded to 640 elements, dst rows padded to 600."""
    wl = _small(7, src, dst, 64, 576, row_stride=640, R=5, maxlen=300)
    _check(wl, options=options, dst_row_stride=600)
    _check(wl, options=options, dst_row_stride=600, workspace=True)


@pytest.mark.parametrize("row_stride,dst_stride", [(577, None), (576, 579), (581, 583)])
def test_odd_strides_force_narrow_units(row_stride, dst_stride):
    wl = _small(11, "bf16", "bf16", 16, 576, row_stride=row_stride, R=4, maxlen=70)
    _check(wl, dst_row_stride=dst_stride)
    wl8 = _small(12, "fp8_e4m3", "bf16", 16, 576, row_stride=row_stride, R=4, maxlen=70)
    _check(wl8, dst_row_stride=dst_stride)


@pytest.mark.parametrize("scale", [1.0, 0.05, 0.02, 2.0 ** -12, 1e30, 3.0e-39])
@pytest.mark.parametrize("dst", ["bf16", "fp16", "fp32"])
def test_all_fp8_codes(scale, dst):
    """Every e4m3 code (NaN included) through the dequant path."""
    codes = np.tile(np.arange(256, dtype=np.uint8), 4)  # 1024 elements: 4 rows of 256
    cache = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).reshape(4, 1, 256)
    wl = W.Workload("codes", cache, torch.tensor([[2, 0, 3, 1]], dtype=torch.int32),
                    torch.tensor([0, 4], dtype=torch.int32), None, [4], 1, 4, 1, 256, "fp8_e4m3", dst, scale)
    for opt in (0, binding.OPT_FORCE_SCALAR):
        _check(wl, options=opt)


# --- edge cases ---------------------------------------------------------------

def test_many_requests_at_the_limit():
    rng = np.random.default_rng(3)
    R = binding.MAX_REQS_PLAN
    lens = [int(x) for x in rng.integers(0, 40, R)]
    starts = [int(x) for x in rng.integers(0, 100, R)]
    wl = W.make_workload("many", lens, starts, 16, 64, None, "bf16", "bf16", 1.0, 5)
    _check(wl)


def test_single_token_requests_and_zero_lengths():
    lens = [1, 0, 1, 0, 0, 1, 1, 0]
    wl = W.make_workload("ones", lens, [63, 5, 0, 0, 1, 64, 127, 3], 64, 576, None, "bf16", "bf16", 1.0, 9)
    _check(wl)


def test_cu_offset_and_clamp_at_total_tokens():
    wl = W.make_workload("clamp", [100, 50, 70], [5, 0, 9], 16, 576, None, "bf16", "bf16", 1.0, 13, cu_offset=10,
                         total_tokens=150)
    _check(wl)


def test_empty_calls_write_nothing():
    wl = W.make_workload("empty", [0, 0, 0], [1, 2, 3], 16, 32, None, "bf16", "bf16", 1.0, 14, total_tokens=8)
    _check(wl)
    wl0 = W.make_workload("noreq", [], None, 16, 32, 4, "bf16", "bf16", 1.0, 15, total_tokens=4)
    _check(wl0)
    wlT = W.make_workload("zeroT", [5], None, 16, 32, None, "bf16", "bf16", 1.0, 16, total_tokens=0)
    _check(wlT)


def test_non_default_stream():
    wl = W.skew8()
    case = DeviceCase(wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        case.run(stream=s)
    s.synchronize()
    got, flag, guards = case.result()
    want, oflag = oracle_run(wl)
    assert guards and flag == oflag == 0
    assert_same(got, want, "bf16", True)


def test_repeated_calls_are_deterministic():
    wl = W.skew64("dequant")
    case = DeviceCase(wl)
    case.run()
    first, _, _ = case.result()
    case.dst_full.view(torch.uint8).fill_(0x3C)
    case.run()
    second, flag, guards = case.result()
    assert guards and flag == 0
    assert np.array_equal(first, second)


# --- invalid data: skipped rows, flags, untouched output (review section) -------

def _flag_case(**kw):
    base = dict(lens=[40, 30, 25], starts=[3, 0, 7], B=16, E=64)
    base.update(kw)
    return W.make_workload("flags", base["lens"], base["starts"], base["B"], base["E"], None, "bf16", "bf16", 1.0,
                           21)


def test_logical_block_past_table_row():
    wl = _flag_case()
    bt = wl.block_table.numpy().copy()
    # request 1 (len 30) now starts at 40: its row holds 2 ids in a 3-wide
    # table, so logical block 2 is the -1 padding and blocks 3, 4 are past the row
    ss = np.array([3, 40, 7], np.int32)
    _check(wl, seq_starts=ss, expect_flag=og.BAD_LOGICAL | og.BAD_PHYS)


@pytest.mark.parametrize("bad", [-1, 10 ** 6, -(2 ** 31)])
def test_physical_block_out_of_range(bad):
    wl = _flag_case()
    bt = wl.block_table.numpy().copy()
    bt[1, 1] = bad
    bt[2, 0] = bad
    _check(wl, block_table=bt, expect_flag=og.BAD_PHYS)


def test_negative_seq_start():
    wl = _flag_case()
    _check(wl, seq_starts=np.array([3, -5, 7], np.int32), expect_flag=og.BAD_START)


# cu_seq_lens that is not non-decreasing: the page's clamp gives a request
# after a decrease no rows; a request whose rows would start below row 0 or
# below an earlier boundary (overlapping or out-of-order rows) is skipped with
# flag 8, and every other request is copied (T = 95, lengths 40/30/25)
@pytest.mark.parametrize("cu,flag", [
    ([0, 40, 30, 30], 0),             # a decrease, no rows after it
    ([0, 40, 70, 60], 0),             # the last request has no rows
    ([0, 40, 30, 95], og.BAD_CU),     # request 2 would overlap request 0
    ([-1, 40, 70, 95], og.BAD_CU),    # request 0 would start at row -1
    ([50, 60, 0, 20], og.BAD_CU),     # request 2 comes out of order (no overlap)
    ([0, 40, 20, 60], og.BAD_CU),     # rows 40-59 of the skipped request stay untouched
])
def test_cu_seq_lens_not_non_decreasing(cu, flag):
    wl = _flag_case()
    _check(wl, cu=np.array(cu, np.int32), expect_flag=flag)


def test_huge_seq_start_no_overflow():
    wl = _flag_case()
    _check(wl, seq_starts=np.array([3, 2 ** 31 - 10, 7], np.int32), expect_flag=og.BAD_LOGICAL)


# --- batches beyond one launch's plan: run in groups of requests -------------

def _large(R, seed, src="bf16", dst="bf16", E=64, B=16):
    rng = np.random.default_rng(seed)
    lens = [int(x) if rng.random() > 0.1 else 0 for x in rng.integers(0, 24, R)]
    starts = [int(x) for x in rng.integers(0, 40, R)]
    return W.make_workload("large", lens, starts, B, E, None, src, dst, 0.05, seed)


@pytest.mark.parametrize("src,dst,options", [("bf16", "bf16", 0), ("fp8_e4m3", "bf16", 0),
                                             ("bf16", "bf16", binding.OPT_FORCE_SIMT)])
def test_large_batch_in_groups(src, dst, options):
    wl = _large(2 * binding.MAX_REQS_PLAN + 1808, 61, src, dst)
    _check(wl, options=options, workspace=True)


def test_large_batch_needs_a_workspace():
    wl = _large(binding.MAX_REQS_PLAN + 1, 62)
    case = DeviceCase(wl)
    with pytest.raises(binding.PmgError) as e:
        case.run()
    assert e.value.status == 5


@pytest.mark.parametrize("where", ["inside_last_group", "across_group_boundary"])
def test_large_batch_cu_decrease(where):
    """A decrease of cu_seq_lens in a batch run as several launches: the request
    after it starts below an earlier boundary and is skipped (flag 8). Across a
    group boundary, the earlier boundary belongs to the group before, so the
    group launches must pass it on through the workspace."""
    wl = _large(2 * binding.MAX_REQS_PLAN + 100, 63)
    cu = wl.cu_seq_lens.numpy().copy()
    i = len(cu) - 20 if where == "inside_last_group" else 2 * binding.MAX_REQS_PLAN
    cu[i] = cu[i - 1] - 1
    assert cu[i + 1] > cu[i]  # the request starting at boundary i has rows
    _check(wl, cu=cu, expect_flag=og.BAD_CU, workspace=True)
    # the workspace is left zeroed for the next call
    case = DeviceCase(wl, workspace=True)
    case.run()
    case.run()
    got, flag, guards = case.result()
    want, _ = oracle_run(wl)
    assert guards and flag == 0
    assert_same(got, want, "bf16", False)


def test_large_batch_implied_end():
    wl = _large(binding.MAX_REQS_PLAN + 700, 64)
    T = wl.total_tokens - 5
    cu_short = wl.cu_seq_lens.numpy()[:-1].copy()
    cu_full = np.concatenate([cu_short, [max(T, int(cu_short[-1]))]]).astype(np.int32)
    want, oflag = oracle_run(wl, cu=cu_full, total_tokens=T)
    case = DeviceCase(wl, cu=cu_short, total_tokens=T, workspace=True)
    case.run(options=binding.OPT_IMPLIED_END)
    got, flag, guards = case.result()
    assert guards and oflag == 0 and flag == 0
    assert_same(got, want, "bf16", False)


# --- implied terminal entry (has_terminal_start = false) -----------------------

@pytest.mark.parametrize("T_cut", [0, 7, 27, 40])
def test_implied_end_convention(T_cut):
    """cu_seq_lens without its terminal entry: the last request ends at total_tokens."""
    wl = W.make_workload("implied", [40, 30, 32], [3, 0, 7], 16, 64, None, "bf16", "bf16", 1.0, 31)
    T = 102 - T_cut
    cu_short = wl.cu_seq_lens.numpy()[:-1].copy()
    # the oracle takes the explicit form: the last request ends at total_tokens
    cu_full = np.concatenate([cu_short, [max(T, int(cu_short[-1]))]]).astype(np.int32)
    want, oflag = oracle_run(wl, cu=cu_full, total_tokens=T)
    case = DeviceCase(wl, cu=cu_short, total_tokens=T)
    case.run(options=binding.OPT_IMPLIED_END)
    got, flag, guards = case.result()
    assert guards and oflag == 0 and flag == oflag
    assert_same(got, want, "bf16", False)


# --- the device mapper alone ---------------------------------------------------

def _plan_case(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 60))
    B = int(rng.choice([1, 2, 16, 64]))
    lens = [int(x) if rng.random() > 0.2 else 0 for x in rng.integers(0, 6 * B + 3, R)]
    starts = [int(x) for x in rng.integers(0, 3 * B, R)] if rng.random() < 0.6 else None
    off = int(rng.integers(0, 4))
    cu = np.concatenate([[off], off + np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1]) - int(rng.integers(0, 3))
    return cu, starts, R, max(T, 0), B


@pytest.mark.parametrize("seed", range(30))
def test_debug_plan_matches_oracle_plan(seed):
    cu, starts, R, T, B = _plan_case(seed)
    want = op.page_tasks(cu.tolist(), starts, R, T, B)
    dev = "cuda:0"
    ss = None if starts is None else torch.tensor(starts, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    tasks, num = binding.debug_plan(torch.from_numpy(cu).to(dev), ss, T, B, len(want) + 3, error_flag=err)
    assert int(num.item()) == len(want)
    got = [tuple(int(x) for x in row) for row in tasks.cpu().numpy()[:len(want)]]
    assert got == want
    assert np.all(tasks.cpu().numpy()[len(want):] == -1)
    assert int(err.item()) == 0


def test_debug_plan_golden_cases():
    import json, os
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))["cases"]
    for c in cases:
        cu = torch.tensor(c["cu_seq_lens"], dtype=torch.int32, device="cuda:0")
        ss = None if c["seq_starts"] is None else torch.tensor(c["seq_starts"], dtype=torch.int32, device="cuda:0")
        tasks, num = binding.debug_plan(cu, ss, c["total_tokens"], c["block_size"], 16)
        n = int(num.item())
        assert n == len(c["tasks"]), c["name"]
        assert [list(map(int, r)) for r in tasks.cpu().numpy()[:n]] == c["tasks"], c["name"]


# --- 64-bit addressing: output offsets past 2^31 bytes --------------------------

@pytest.mark.slow
def test_int64_output_offsets_fp32_1m_tokens():
    """fp32 raw copy of 576-element entries (2304 B) over 1,000,000 tokens: the
    output byte offset passes 2^31 near token 932,068."""
    B, E, T = 64, 576, 1_000_000
    nb = T // B + 2
    # id-coded values: element (b, s, e) holds b << 16 | s << 10 | e (as fp32 bits)
    b = np.arange(nb, dtype=np.uint32)[:, None, None]
    s = np.arange(B, dtype=np.uint32)[None, :, None]
    e = np.arange(E, dtype=np.uint32)[None, None, :]
    bits = ((b << 16) | (s << 10) | e).astype(np.uint32)
    perm = np.random.default_rng(41).permutation(nb).astype(np.int32)
    cache = torch.from_numpy(bits.view(np.float32))
    wl = W.Workload("int64", cache, torch.from_numpy(perm[None, :].copy()),
                    torch.tensor([0, T], dtype=torch.int32), torch.tensor([17], dtype=torch.int32), [T], 1, T, B, E,
                    "fp32", "fp32", 1.0)
    _check(wl)


# --- the context-parallel calling pattern: a slice of a larger workspace ------

@pytest.mark.parametrize("name", ["skew8", "skew64_raw"])
def test_cp_workspace_slice_eager_and_graph(name):
    """The page's context-parallel prefill gathers into workspace[:toks] and
    leaves the workspace tail to an all-gather (section "实现拆解" item 2). Here
    the gather writes rows [off, off + T) of a larger workspace, from an eager
    call and from a captured CUDA graph; every other row keeps its contents."""
    wl = W.CONFIGS[name]()
    want, oflag = oracle_run(wl)
    assert oflag == 0
    dev = "cuda:0"
    ed = W.ELEM_BYTES[wl.dst_dtype]
    off, tail = 300, 1000
    rows = off + wl.total_tokens + tail
    ws = torch.full((rows, wl.entry_size * ed), 0x3C, dtype=torch.uint8, device=dev)
    dst = ws.view(W.TORCH_DTYPES[wl.dst_dtype])[off:off + wl.total_tokens]
    cache = wl.cache.to(dev)[:, :, :wl.entry_size]
    bt, cu = wl.block_table.to(dev), wl.cu_seq_lens.to(dev)
    ss = None if wl.seq_starts is None else wl.seq_starts.to(dev)
    scale = torch.tensor([wl.scale], dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sched = binding.new_workspace(dev)

    def call(stream=None):
        binding.gather(cache, dst, bt, cu, ss, scale, err, stream=stream, workspace=sched)

    def check():
        torch.cuda.synchronize()
        host = ws.cpu().numpy()
        assert np.all(host[:off] == 0x3C) and np.all(host[off + wl.total_tokens:] == 0x3C)
        got = host[off:off + wl.total_tokens].view(W.NP_BITS[ed])
        assert int(err.item()) == 0
        assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)

    call()
    check()
    ws.fill_(0x3C)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(torch.cuda.current_stream())
    g.replay()
    g.replay()
    check()


# --- the exported pmg_gather symbol itself (no workspace, no options) ---------

@pytest.mark.parametrize("name", ["tiny", "skew8", "skew64_dequant"])
def test_pmg_gather_symbol_through_ctypes(name):
    """pmg_gather, the call of ops.cp_gather_cache(src_cache, dst, block_table,
    cu_seq_lens, batch_size, seq_starts) in section "关键源码片段" with strides,
    dtypes, scale and stream made explicit, called directly through ctypes
    with raw pointers, against the oracle."""
    wl = W.CONFIGS[name]()
    want, oflag = oracle_run(wl)
    case = DeviceCase(wl)
    L = binding.load_library()
    codes = binding.DTYPE_CODES
    st = L.pmg_gather(
        case.cache.data_ptr(), case.cache.stride(0), case.cache.stride(1), case.cache.shape[0],
        case.block_table.data_ptr(), case.block_table.shape[1], case.cu.data_ptr(),
        None if case.seq_starts is None else case.seq_starts.data_ptr(), wl.num_reqs, case.T, wl.block_size,
        wl.entry_size, codes[wl.src_dtype], codes[wl.dst_dtype], case.scale.data_ptr(), case.dst.data_ptr(),
        case.dst.stride(0), case.err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.status_string(st)
    got, flag, guards = case.result()
    assert guards and flag == oflag == 0
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


def test_fp32_1m_named_workload_with_workspace():
    """The 1M-token fp32 raw copy the benchmark times (2304-byte entries, output
    offsets past 2^31 bytes), in the benchmark's launch configuration."""
    _check(W.CONFIGS["fp32_1m"](), workspace=True)


# --- the converting kernel's ring, chosen at launch from the rows each CTA
# will hold (T / (4 x SMs)): two stages up to 128 rows per CTA, else three over
# back-to-back or padded rows; cases on both sides of the boundary -----------

def _rows_per_cta(T):
    return T // (4 * torch.cuda.get_device_properties(0).multi_processor_count)


@pytest.mark.parametrize("rows_per_cta,src,dst,row_stride", [
    (120, "fp8_e4m3", "bf16", None),   # two stages
    (128, "fp8_e4m3", "fp16", None),   # the boundary: two stages
    (129, "fp8_e4m3", "bf16", None),   # three stages, back-to-back rows
    (200, "fp8_e4m3", "fp32", None),
    (140, "bf16", "fp32", None),
    (129, "fp8_e4m3", "bf16", 640),    # three stages, padded rows
    (100, "fp16", "fp32", 640),
])
@pytest.mark.parametrize("workspace", [False, True])
def test_converter_ring_across_launch_sizes(rows_per_cta, src, dst, row_stride, workspace):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = rows_per_cta * 4 * sms + 3
    assert _rows_per_cta(T) == rows_per_cta
    # three requests with unaligned starts: partial first and last pages
    lens = [T // 2, 1, T - T // 2 - 1]
    wl = W.make_workload(f"ring at {rows_per_cta} rows per CTA", lens, [37, 0, 63], 64, 576, None, src, dst, 0.05,
                         9100 + rows_per_cta, row_stride=row_stride)
    case = _check(wl, workspace=workspace)
    assert binding.select_path(case.cache, case.dst, case.block_table, case.cu)[0] == "bulk"


# --- the realigning byte copy: raw copies whose rows are not 16-byte aligned
# (odd strides on either side, or a base that is not 16-byte aligned) ---------

def _realign_case(seed, dtype, E, src_stride, dst_stride, src_off=0, dst_off=0, B=16, R=5, out_dtype=None,
                  scale=1.0):
    out_dtype = out_dtype or dtype
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(0, 3 * B + 5, R)]
    lens[int(rng.integers(0, R))] = 0
    starts = [int(x) for x in rng.integers(0, 2 * B + 1, R)]
    assert src_off + E <= src_stride
    wl = W.make_workload("realign", lens, starts, B, E, None, dtype, out_dtype, scale, seed, row_stride=src_stride)
    T, ed = wl.total_tokens, W.ELEM_BYTES[out_dtype]
    # oracle on the same element window of each cache row
    cache_bits = W.tensor_bits(wl.cache)
    view = np.lib.stride_tricks.as_strided(cache_bits[:, :, src_off:], shape=(cache_bits.shape[0], B, E),
                                           strides=cache_bits.strides)
    want = np.full((T, dst_stride * ed), 0xA5, np.uint8).view(W.NP_BITS[ed])
    oflag = og.gather(view, wl.block_table.numpy(), wl.cu_seq_lens.numpy(), wl.seq_starts.numpy(), R, T, B, E,
                      dtype, out_dtype, scale, want)
    # device: cache window at element src_off; dst rows of dst_stride elements
    # starting dst_off elements into a guarded buffer
    dev = "cuda:0"
    full = wl.cache.to(dev)
    cache = full[:, :, src_off:src_off + E]
    body_elems = dst_off + T * dst_stride
    raw = torch.full((2 * GUARD_BYTES + body_elems * ed,), 0xA5, dtype=torch.uint8, device=dev)
    flat = raw[GUARD_BYTES:GUARD_BYTES + body_elems * ed].view(W.TORCH_DTYPES[out_dtype])
    dst = flat[dst_off:].view(T, dst_stride)[:, :E]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    path, _ = binding.select_path(cache, dst, wl.block_table.to(dev), wl.cu_seq_lens.to(dev))
    binding.gather(cache, dst, wl.block_table.to(dev), wl.cu_seq_lens.to(dev), wl.seq_starts.to(dev),
                   torch.tensor([scale], device=dev), err, num_reqs=R)
    torch.cuda.synchronize()
    r = raw.cpu().numpy()
    assert np.all(r[:GUARD_BYTES] == 0xA5) and np.all(r[-GUARD_BYTES:] == 0xA5), "guard regions written"
    body = r[GUARD_BYTES:len(r) - GUARD_BYTES]
    assert np.all(body[:dst_off * ed] == 0xA5), "bytes before the first row written"
    got = body[dst_off * ed:].view(W.NP_BITS[ed]).reshape(T, dst_stride)
    assert oflag == 0 and int(err.item()) == 0
    assert_same(got, want, out_dtype, out_dtype != dtype)
    return path


@pytest.mark.parametrize("dtype,E,src_stride,dst_stride,src_off,dst_off", [
    ("bf16", 576, 577, 576, 0, 0),     # source rows step 2 bytes off alignment per row
    ("bf16", 576, 576, 577, 0, 0),     # destination rows do
    ("bf16", 576, 581, 583, 0, 0),
    ("bf16", 576, 580, 580, 0, 0),     # 8-byte aligned rows
    ("bf16", 576, 584, 576, 1, 0),     # aligned row stride, window 2 bytes into each row
    ("bf16", 576, 576, 576, 0, 3),     # output starts 6 bytes into the buffer
    ("bf16", 576, 592, 584, 7, 5),
    ("bf16", 8, 9, 11, 0, 0),          # 16-byte rows, always split over two words
    ("u8", 17, 17, 17, 0, 0),
    ("u8", 31, 36, 31, 3, 1),
    ("u8", 100, 101, 103, 0, 0),
    ("u8", 1000, 1024, 1001, 15, 13),
    ("fp8_e4m3", 576, 577, 577, 0, 0),  # fp8 raw copy: byte rows
    ("fp32", 5, 5, 5, 0, 0),           # 20-byte rows
    ("fp32", 7, 9, 7, 1, 2),
    ("fp32", 290, 290, 291, 0, 1),
])
def test_realigning_copy(dtype, E, src_stride, dst_stride, src_off, dst_off):
    path = _realign_case(500 + E + src_stride + 7 * src_off + 13 * dst_off, dtype, E, src_stride, dst_stride,
                         src_off, dst_off)
    assert path == "realign"


@pytest.mark.parametrize("B,R", [(64, 3), (1, 40), (128, 2)])
def test_realigning_copy_pages_and_requests(B, R):
    """Full pages, one-token pages and long pages, many requests."""
    assert _realign_case(77 + B + R, "bf16", 576, 579, 577, 1, 1, B=B, R=R) == "realign"


def test_realigning_copy_matches_forced_scalar():
    """The realigning copy and the one-element-per-access kernel write the same
    bytes (and the same untouched padding) on a named-size workload with odd
    strides on both sides."""
    wl = _small(31, "bf16", "bf16", 64, 576, row_stride=579, R=6)
    a = DeviceCase(wl, dst_row_stride=581)
    assert binding.select_path(a.cache, a.dst, a.block_table, a.cu)[0] == "realign"
    a.run()
    b = DeviceCase(wl, dst_row_stride=581)
    b.run(options=binding.OPT_FORCE_SCALAR)
    ga, fa, _ = a.result()
    gb, fb, _ = b.result()
    assert fa == fb == 0
    assert np.array_equal(ga, gb)


@pytest.mark.parametrize("src,dst,E,src_stride,dst_stride,src_off,dst_off", [
    ("fp8_e4m3", "bf16", 576, 577, 576, 0, 0),   # odd source rows, aligned output rows
    ("fp8_e4m3", "bf16", 576, 576, 577, 0, 0),   # output rows 2 bytes off per row
    ("fp8_e4m3", "bf16", 576, 592, 576, 5, 3),   # windows off alignment on both sides
    ("fp8_e4m3", "bf16", 572, 572, 572, 0, 0),   # aligned rows, not a whole number of converter units
    ("fp8_e4m3", "bf16", 9, 9, 9, 0, 0),         # 18-byte output rows: two partial words
    ("fp8_e4m3", "fp16", 576, 579, 581, 0, 0),
    ("fp8_e4m3", "fp32", 576, 577, 577, 0, 0),
    ("fp8_e4m3", "fp32", 5, 5, 5, 0, 1),         # 20-byte output rows
    ("bf16", "fp32", 576, 577, 578, 0, 0),
    ("bf16", "fp32", 8, 9, 8, 1, 0),
    ("fp16", "fp32", 100, 101, 103, 0, 1),
    ("fp16", "fp32", 100, 112, 100, 7, 0),
])
def test_realigning_converting_gather(src, dst, E, src_stride, dst_stride, src_off, dst_off):
    scale = 0.05 if src == "fp8_e4m3" else 1.0
    path = _realign_case(900 + E + src_stride + 7 * src_off + 13 * dst_off, src, E, src_stride, dst_stride,
                         src_off, dst_off, out_dtype=dst, scale=scale)
    assert path == "realign"
