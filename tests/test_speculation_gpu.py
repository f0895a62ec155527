"""The speculative start of the TMA paths, under real overlap.

Without the caller's early-metadata promise, a small batch still plans and
resolves its first batch before the previous grid in the stream is known to be
done, and checks both against the inputs as they are after the wait. Here the
previous grid is itself a gather whose output IS the next gather's
cu_seq_lens and block table: it starts (programmatic dependent launch) while
the first one still writes them, so its speculative reads can see the old
tables. Old and new tables are both valid, so every speculative read stays in
bounds; the result must equal the oracle on the NEW tables, bit for bit, on
every repetition, whichever way each race went.

Source for the expected output: "MLA cache gather scheduled per logical page"
(prhub.com.cn, vllm PR #51739), section "关键源码片段", the per-token
expected output of test_cp_gather_cache_mla_large_uneven_sequences.
"""
import numpy as np
import pytest
import torch

from oracle import gather as og
from paged_mla_kv_cache_gb300 import binding
from paged_mla_kv_cache_gb300 import workloads as W

from gpu_helpers import assert_same

pytestmark = pytest.mark.gpu

R, STRIDE, B, NB = 3, 16, 16, 64
T2S = 64         # token_to_seq at [T2S, T2S + 256)
META_INTS = 320  # cu at [0, R], block table at [16, 16 + R * STRIDE)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    return cuda_lib


def _meta(rng, lens):
    """Valid cu, block table and token_to_seq packed into META_INTS int32
    (token_to_seq is -1 past the last request)."""
    m = np.zeros(META_INTS, np.int32)
    m[:R + 1] = np.concatenate([[0], np.cumsum(lens)])
    perm = rng.permutation(NB).astype(np.int32)
    m[16:16 + R * STRIDE] = perm[:R * STRIDE]
    m[T2S:] = -1
    for r in range(R):
        m[T2S + m[r]:T2S + m[r + 1]] = r
    return m


def _oracle(cache_bits, meta, E, src, dst_dtype, scale, T):
    cu = meta[:R + 1].copy()
    bt = meta[16:16 + R * STRIDE].reshape(R, STRIDE).copy()
    ed = W.ELEM_BYTES[dst_dtype]
    want = np.full((T, E * ed), 0xA5, np.uint8).view(W.NP_BITS[ed])
    flag = og.gather(cache_bits, bt, cu, None, R, T, B, E, src, dst_dtype, scale, want)
    return want, flag


@pytest.mark.parametrize("src,dst", [("bf16", "bf16"), ("fp8_e4m3", "bf16")])
@pytest.mark.parametrize("same", [False, True])
def test_metadata_written_by_the_previous_grid(src, dst, same):
    dev = "cuda:0"
    E = 64
    rng = np.random.default_rng(71 if same else 72)
    # the gathered cache: NB blocks of B slots
    wl = W.make_workload("spec", [B * NB], None, B, E, NB, src, dst, 0.05, 73)
    cache = wl.cache.to(dev)
    cache_bits = W.tensor_bits(wl.cache)
    scale = torch.tensor([wl.scale], dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # the first gather copies one fp32 row of META_INTS elements: the tables
    one_bt = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    one_cu = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    meta = torch.empty(META_INTS, dtype=torch.int32, device=dev)
    cu_dev = meta[:R + 1]
    bt_dev = meta[16:16 + R * STRIDE].view(R, STRIDE)
    for it in range(24):
        lens_new = [int(x) for x in rng.integers(1, 5 * B, R)]
        lens_old = [int(x) for x in rng.integers(1, 5 * B, R)]
        new = _meta(rng, lens_new)
        old = new.copy() if same else _meta(rng, lens_old)
        T = int(max(new[R], old[R]))
        src_row = torch.from_numpy(new.view(np.float32).copy()).to(dev).view(1, 1, META_INTS)
        meta.copy_(torch.from_numpy(old))
        out = torch.full((T, E), 0, dtype=W.TORCH_DTYPES[dst], device=dev)
        out.view(torch.uint8).fill_(0xA5)
        err.zero_()
        torch.cuda.synchronize()
        # queue both behind a busy kernel so that they start back to back
        torch.cuda._sleep(200_000)
        binding.gather(src_row, meta.view(torch.float32).view(1, META_INTS), one_bt, one_cu, error_flag=err)
        binding.gather(cache, out, bt_dev, cu_dev, None, scale, err, num_reqs=R)
        torch.cuda.synchronize()
        assert np.array_equal(meta.cpu().numpy(), new)
        want, flag = _oracle(cache_bits, new, E, src, dst, wl.scale, T)
        got = out.cpu().view(torch.uint8).numpy().view(W.NP_BITS[W.ELEM_BYTES[dst]]).reshape(T, E)
        assert int(err.item()) == flag == 0
        assert_same(got, want, dst, src != dst)


@pytest.mark.parametrize("src,dst", [("bf16", "bf16"), ("fp8_e4m3", "bf16")])
def test_token_metadata_written_by_the_previous_grid(src, dst):
    """The same race for the per-token entry point: token_to_seq, cu_seq_lens
    and the block table come from the previous grid."""
    dev = "cuda:0"
    E = 64
    rng = np.random.default_rng(74)
    wl = W.make_workload("spec", [B * NB], None, B, E, NB, src, dst, 0.05, 75)
    cache = wl.cache.to(dev)
    cache_bits = W.tensor_bits(wl.cache)
    scale = torch.tensor([wl.scale], dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    one_bt = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    one_cu = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    meta = torch.empty(META_INTS, dtype=torch.int32, device=dev)
    for it in range(24):
        new = _meta(rng, [int(x) for x in rng.integers(1, 5 * B, R)])
        old = _meta(rng, [int(x) for x in rng.integers(1, 5 * B, R)])
        T = int(new[R])
        src_row = torch.from_numpy(new.view(np.float32).copy()).to(dev).view(1, 1, META_INTS)
        meta.copy_(torch.from_numpy(old))
        out = torch.full((T, E), 0, dtype=W.TORCH_DTYPES[dst], device=dev)
        out.view(torch.uint8).fill_(0xA5)
        err.zero_()
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000)
        binding.gather(src_row, meta.view(torch.float32).view(1, META_INTS), one_bt, one_cu, error_flag=err)
        binding.gather_tokens(cache, out, meta[16:16 + R * STRIDE].view(R, STRIDE), meta[T2S:T2S + T],
                              meta[:R + 1], scale, err, num_reqs=R)
        torch.cuda.synchronize()
        assert np.array_equal(meta.cpu().numpy(), new)
        ed = W.ELEM_BYTES[dst]
        want = np.full((T, E * ed), 0xA5, np.uint8).view(W.NP_BITS[ed])
        flag = og.gather_tokens(cache_bits, new[16:16 + R * STRIDE].reshape(R, STRIDE).copy(),
                                new[T2S:T2S + T].copy(), new[:R + 1].copy(), R, T, B, E, src, dst, wl.scale, want)
        got = out.cpu().view(torch.uint8).numpy().view(W.NP_BITS[ed]).reshape(T, E)
        assert int(err.item()) == flag == 0
        assert_same(got, want, dst, src != dst)


def _align4(n):
    return (n + 3) // 4 * 4


@pytest.mark.parametrize("R,with_ss,implied", [(200, True, False), (130, False, True), (40, True, True),
                                               (256, True, False)])
def test_many_requests_metadata_race(R, with_ss, implied):
    """The same race with a larger batch: the check after the wait reads
    cu_seq_lens and seq_starts in several passes of 128 entries; seq_starts
    and the implied-end convention change under the race too."""
    dev = "cuda:0"
    B, E, NB2, STRIDE2 = 16, 64, 1024, 4
    rng = np.random.default_rng(700 + R + 7 * with_ss + 3 * implied)
    wl = W.make_workload("spec", [B * NB2], None, B, E, NB2, "bf16", "bf16", 1.0, 76)
    cache = wl.cache.to(dev)
    cache_bits = W.tensor_bits(wl.cache)
    SS = _align4(R + 1)
    BT = SS + _align4(R)
    META = _align4(BT + R * STRIDE2)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    one_bt = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    one_cu = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    meta = torch.empty(META, dtype=torch.int32, device=dev)
    opts = binding.OPT_IMPLIED_END if implied else 0

    def make():
        lens = rng.integers(0, 2 * B + 1, R)
        starts = rng.integers(0, B, R) if with_ss else np.zeros(R, np.int64)
        m = np.zeros(META, np.int32)
        m[:R + 1] = np.concatenate([[0], np.cumsum(lens)])
        m[SS:SS + R] = starts
        m[BT:BT + R * STRIDE2] = rng.permutation(NB2)[:R * STRIDE2]
        return m

    for it in range(12):
        new, old = make(), make()
        T = int(new[R])
        src_row = torch.from_numpy(new.view(np.float32).copy()).to(dev).view(1, 1, META)
        meta.copy_(torch.from_numpy(old))
        out = torch.empty((T, E), dtype=torch.bfloat16, device=dev)
        out.view(torch.uint8).fill_(0xA5)
        err.zero_()
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000)
        binding.gather(src_row, meta.view(torch.float32).view(1, META), one_bt, one_cu, error_flag=err)
        binding.gather(cache, out, meta[BT:BT + R * STRIDE2].view(R, STRIDE2), meta[:R + (0 if implied else 1)],
                       meta[SS:SS + R] if with_ss else None, None, err, num_reqs=R, options=opts)
        torch.cuda.synchronize()
        assert np.array_equal(meta.cpu().numpy(), new)
        cu = new[:R + 1].copy()
        if implied:
            cu[R] = max(T, int(cu[R - 1]))
        want = np.full((T, E), 0xA5A5, np.uint16)
        flag = og.gather(cache_bits, new[BT:BT + R * STRIDE2].reshape(R, STRIDE2).copy(), cu,
                         new[SS:SS + R].copy() if with_ss else None, R, T, B, E, "bf16", "bf16", 1.0, want)
        got = out.cpu().view(torch.int16).numpy().view(np.uint16)
        assert int(err.item()) == flag == 0
        assert_same(got, want, "bf16", False)


@pytest.mark.parametrize("src,dst", [("bf16", "bf16"), ("fp8_e4m3", "bf16")])
@pytest.mark.parametrize("form", ["zero_to_T", "offset_start", "short_end", "implied_zero", "implied_offset"])
def test_single_request_plan_guess_under_race(src, dst, form):
    """One request without seq_starts: the TMA paths plan from cu_seq_lens =
    [0, T] (or [0] with the implied end) before reading it, and keep that plan
    only if the values read after the previous grid completes agree. Here the
    previous grid writes the next call's cu_seq_lens and block table; forms
    that differ from the guess (a start above 0, an end below T) must give the
    oracle's result on the new tables, bit for bit."""
    dev = "cuda:0"
    E, STRIDE1 = 64, 24
    rng = np.random.default_rng({"zero_to_T": 81, "offset_start": 82, "short_end": 83, "implied_zero": 84,
                                 "implied_offset": 85}[form] + (100 if src != dst else 0))
    wl = W.make_workload("spec1", [B * NB], None, B, E, NB, src, dst, 0.05, 86)
    cache = wl.cache.to(dev)
    cache_bits = W.tensor_bits(wl.cache)
    scale = torch.tensor([wl.scale], dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    one_bt = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    one_cu = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    implied = form.startswith("implied")
    opts = binding.OPT_IMPLIED_END if implied else 0
    meta = torch.empty(64, dtype=torch.int32, device=dev)
    for it in range(16):
        T = int(rng.integers(B, STRIDE1 * B))
        c0 = int(rng.integers(1, B)) if form in ("offset_start", "implied_offset") else 0
        c1 = int(rng.integers(c0 + 1, T)) if form == "short_end" else T
        new = np.zeros(64, np.int32)
        new[0], new[1] = c0, (0 if implied else c1)
        new[16:16 + STRIDE1] = rng.permutation(NB)[:STRIDE1]
        old = np.zeros(64, np.int32)
        old[0], old[1] = 0, (0 if implied else T)  # the form the guess assumes
        old[16:16 + STRIDE1] = rng.permutation(NB)[:STRIDE1]
        src_row = torch.from_numpy(new.view(np.float32).copy()).to(dev).view(1, 1, 64)
        meta.copy_(torch.from_numpy(old))
        out = torch.empty((T, E), dtype=W.TORCH_DTYPES[dst], device=dev)
        out.view(torch.uint8).fill_(0xA5)
        err.zero_()
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000)
        binding.gather(src_row, meta.view(torch.float32).view(1, 64), one_bt, one_cu, error_flag=err)
        binding.gather(cache, out, meta[16:16 + STRIDE1].view(1, STRIDE1), meta[:1 if implied else 2], None, scale,
                       err, num_reqs=1, options=opts)
        torch.cuda.synchronize()
        assert np.array_equal(meta.cpu().numpy(), new)
        cu = np.array([c0, T if implied else c1], np.int32)
        ed = W.ELEM_BYTES[dst]
        want = np.full((T, E * ed), 0xA5, np.uint8).view(W.NP_BITS[ed])
        flag = og.gather(cache_bits, new[16:16 + STRIDE1].reshape(1, STRIDE1).copy(), cu, None, 1, T, B, E, src,
                         dst, wl.scale, want)
        got = out.cpu().view(torch.uint8).numpy().view(W.NP_BITS[ed]).reshape(T, E)
        assert int(err.item()) == flag == 0
        assert_same(got, want, dst, src != dst)
