"""Pins for the oracle gather and the oracle page plan.

Source: "MLA cache gather scheduled per logical page" (prhub.com.cn, vllm PR
#51739), section "关键源码片段": the per-token expected output of
test_cp_gather_cache_mla_large_uneven_sequences and the
GatherPageTask / map_gather_page_task listing.

What ties the oracle to something other than itself:
- hand-worked cases (tests/golden/hand_cases.json), worked from the page's
  definition without running any code;
- a second route to the same output through library routines only: gather
  whole logical pages of a request with numpy fancy indexing, reshape to a
  token-contiguous context, slice [start, start + len);
- closed forms: identity block table gives a plain slice of the flattened
  cache; invariants: relabelling physical blocks, seq_starts of zeros vs
  none, row count = sum of lengths;
- for the plan, two formulations (walk each request's pages; linear scan
  over requests from a flat id) against each other and against the hand
  cases, and a brute-force check that the tasks tile the rows exactly once.
"""
import json
import os

import numpy as np
import pytest

from oracle import gather as og
from oracle import plan as op

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _id_cache(num_blocks: int, block_size: int, entry_size: int, row_stride: int | None = None) -> np.ndarray:
    """fp32-width cache whose element (b, s, e) holds the bits b<<20 | s<<10 | e."""
    rs = entry_size if row_stride is None else row_stride
    b = np.arange(num_blocks, dtype=np.uint32)[:, None, None]
    s = np.arange(block_size, dtype=np.uint32)[None, :, None]
    e = np.arange(rs, dtype=np.uint32)[None, None, :]
    return (b << 20) | (s << 10) | e


def _decode_row(row: np.ndarray):
    return int(row[0] >> 20), int((row[0] >> 10) & 0x3FF)


SENTINEL32 = 0xA5A5A5A5


def _run(case, entry_size=3, dtype="fp32"):
    B = case["block_size"]
    nb = case["num_blocks"]
    cache = _id_cache(nb, B, entry_size)
    bt = np.array(case["block_table"], dtype=np.int32)
    cu = np.array(case["cu_seq_lens"], dtype=np.int32)
    ss = None if case["seq_starts"] is None else np.array(case["seq_starts"], dtype=np.int32)
    T = case["total_tokens"]
    dst = np.full((T, entry_size), SENTINEL32, dtype=np.uint32)
    flag = og.gather(cache, bt, cu, ss, len(cu) - 1, T, B, entry_size, dtype, dtype, 1.0, dst)
    return flag, dst


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_cases_plan(case):
    cu, ss = case["cu_seq_lens"], case["seq_starts"]
    R, T, B = len(cu) - 1, case["total_tokens"], case["block_size"]
    expected = [tuple(t) for t in case["tasks"]]
    assert op.page_tasks(cu, ss, R, T, B) == expected
    assert [op.task_by_scan(t, cu, ss, R, T, B) for t in range(len(expected))] == expected
    assert op.task_by_scan(len(expected), cu, ss, R, T, B) is None
    assert op.num_tasks(cu, ss, R, T, B) == len(expected)


@pytest.mark.parametrize("case", [c for c in _cases() if "rows" in c], ids=lambda c: c["name"])
def test_hand_cases_gather(case):
    flag, dst = _run(case)
    assert flag == case["flag"]
    for i, want in enumerate(case["rows"]):
        if want is None:
            assert np.all(dst[i] == SENTINEL32), f"row {i} written"
        else:
            b, s = want
            assert _decode_row(dst[i]) == (b, s), f"row {i}"
            assert np.array_equal(dst[i], _id_cache(b + 1, s + 1, dst.shape[1])[b, s]), f"row {i} elements"


def test_tiny_config_row_count():
    case = _cases()[0]
    tasks = op.page_tasks(case["cu_seq_lens"], None, 4, 218, 64)
    assert sum(e - b for (_, _, b, e, _) in tasks) == 218 == 17 + 71 + 130 + 0


def _random_case(rng, R_max=12, B_choices=(1, 2, 3, 4, 16, 64), with_starts=None, e=5):
    R = int(rng.integers(0, R_max + 1))
    B = int(rng.choice(B_choices))
    lens = [int(x) if rng.random() > 0.2 else 0 for x in rng.integers(0, 5 * B + 3, R)]
    use = rng.random() < 0.5 if with_starts is None else with_starts
    starts = [int(x) for x in rng.integers(0, 3 * B + 2, R)] if use else None
    st = starts or [0] * R
    need = [-(-(st[r] + lens[r]) // B) for r in range(R)]
    stride = max(need + [1]) + int(rng.integers(0, 3))
    nb = max(sum(need), 1) + int(rng.integers(0, 4))
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((max(R, 1), stride), -1, dtype=np.int32)
    pos = 0
    for r in range(R):
        bt[r, :need[r]] = perm[pos:pos + need[r]]
        pos += need[r]
    off = int(rng.integers(0, 3))
    cu = np.concatenate([[off], off + np.cumsum(lens, dtype=np.int64)]).astype(np.int32)
    T = int(cu[-1]) + int(rng.integers(0, 3))
    return dict(R=R, B=B, lens=lens, starts=starts, bt=bt, nb=nb, cu=cu, T=T, E=e)


def _library_route(c, cache):
    """Expected rows through numpy only: per request, take all of its logical
    pages (fancy indexing on the block axis), reshape to [pages*B, E] and slice."""
    out = {}
    st = c["starts"] or [0] * c["R"]
    for r in range(c["R"]):
        L, s = c["lens"][r], st[r]
        if L == 0:
            continue
        npages = -(-(s + L) // c["B"])
        ctx = cache[c["bt"][r, :npages].astype(np.int64)].reshape(npages * c["B"], -1)
        seg = ctx[s:s + L]
        for i in range(L):
            out[int(c["cu"][r]) + i] = seg[i]
    return out


@pytest.mark.parametrize("seed", range(40))
def test_random_against_library_route(seed):
    rng = np.random.default_rng(seed)
    c = _random_case(rng)
    cache = _id_cache(c["nb"], c["B"], c["E"])
    dst = np.full((c["T"], c["E"]), SENTINEL32, dtype=np.uint32)
    flag = og.gather(cache, c["bt"], c["cu"], None if c["starts"] is None else np.array(c["starts"], np.int32),
                     c["R"], c["T"], c["B"], c["E"], "fp32", "fp32", 1.0, dst)
    assert flag == 0
    want = _library_route(c, cache)
    assert len(want) == sum(c["lens"])  # row count = sum of lengths
    for i in range(c["T"]):
        if i in want:
            assert np.array_equal(dst[i], want[i]), f"row {i}"
        else:
            assert np.all(dst[i] == SENTINEL32), f"row {i} written"


@pytest.mark.parametrize("seed", range(40))
def test_plan_two_formulations_and_tiling(seed):
    rng = np.random.default_rng(1000 + seed)
    c = _random_case(rng)
    cu, ss, R, T, B = c["cu"].tolist(), c["starts"], c["R"], c["T"], c["B"]
    tasks = op.page_tasks(cu, ss, R, T, B)
    assert [op.task_by_scan(t, cu, ss, R, T, B) for t in range(len(tasks))] == tasks
    assert op.task_by_scan(len(tasks), cu, ss, R, T, B) is None
    # brute force: the tasks tile each request's rows exactly once, in order,
    # and every task stays inside one page
    covered = []
    st = ss or [0] * R
    for (r, lb, b, e, out) in tasks:
        assert 0 <= b < e <= B
        for k in range(e - b):
            p = lb * B + b + k
            covered.append((out + k, r, p))
    expect = []
    for r in range(R):
        for i in range(c["lens"][r]):
            expect.append((int(cu[r]) + i, r, st[r] + i))
    assert covered == expect


def test_closed_form_identity_table():
    """One request over an identity table: the output is a slice of the flattened cache."""
    B, E, nb = 16, 7, 9
    rng = np.random.default_rng(5)
    cache = rng.integers(0, 2 ** 16, (nb, B, E), dtype=np.uint16)
    for s, L in [(0, 1), (0, nb * B), (5, 100), (17, 31), (15, 1), (0, 0)]:
        bt = np.arange(nb, dtype=np.int32)[None, :]
        dst = np.zeros((L, E), dtype=np.uint16)
        flag = og.gather(cache, bt, np.array([0, L], np.int32), np.array([s], np.int32), 1, L, B, E,
                         "bf16", "bf16", 1.0, dst)
        assert flag == 0
        assert np.array_equal(dst, cache.reshape(-1, E)[s:s + L])


def test_closed_form_permuted_table_whole_pages():
    """Page-aligned request over a permuted table: the output is cache[perm] flattened."""
    B, E, nb = 8, 4, 12
    rng = np.random.default_rng(6)
    cache = rng.integers(0, 2 ** 16, (nb, B, E), dtype=np.uint16)
    perm = rng.permutation(nb).astype(np.int32)
    dst = np.zeros((nb * B, E), dtype=np.uint16)
    flag = og.gather(cache, perm[None, :], np.array([0, nb * B], np.int32), None, 1, nb * B, B, E,
                     "fp16", "fp16", 1.0, dst)
    assert flag == 0
    assert np.array_equal(dst, cache[perm].reshape(-1, E))


@pytest.mark.parametrize("seed", range(10))
def test_invariants(seed):
    rng = np.random.default_rng(2000 + seed)
    c = _random_case(rng, with_starts=False)
    cache = rng.integers(0, 256, (c["nb"], c["B"], c["E"]), dtype=np.uint8)

    def run(cache_, bt_, ss_):
        d = np.full((c["T"], c["E"]), 0x5A, dtype=np.uint8)
        f = og.gather(cache_, bt_, c["cu"], ss_, c["R"], c["T"], c["B"], c["E"], "u8", "u8", 1.0, d)
        assert f == 0
        return d

    base = run(cache, c["bt"], None)
    # seq_starts of zeros is the same as no seq_starts
    assert np.array_equal(run(cache, c["bt"], np.zeros(max(c["R"], 1), np.int32)), base)
    # relabel physical blocks: cache'[pi[b]] = cache[b], table' = pi[table]
    pi = rng.permutation(c["nb"]).astype(np.int32)
    cache2 = np.empty_like(cache)
    cache2[pi] = cache
    bt2 = np.where(c["bt"] >= 0, pi[np.maximum(c["bt"], 0)], -1).astype(np.int32)
    assert np.array_equal(run(cache2, bt2, None), base)


def test_padded_row_stride_reads_only_entries():
    """A padded row stride: columns past entry_size are never read or written."""
    B, E, RS, nb = 4, 3, 5, 3
    cache = _id_cache(nb, B, E, row_stride=RS)
    bt = np.array([[2, 0, 1]], np.int32)
    dst = np.full((10, 6), SENTINEL32, dtype=np.uint32)  # dst row stride 6 > E
    flag = og.gather(cache, bt, np.array([0, 10], np.int32), np.array([1], np.int32), 1, 10, B, E,
                     "fp32", "fp32", 1.0, dst)
    assert flag == 0
    for i in range(10):
        p = 1 + i
        b, s = [2, 0, 1][p // B], p % B
        assert np.array_equal(dst[i, :E], cache[b, s, :E])
        assert np.all(dst[i, E:] == SENTINEL32)


def test_out_of_domain_calls():
    cache = np.zeros((1, 1, 1), np.uint16)
    dst = np.zeros((1, 1), np.uint16)
    with pytest.raises(ValueError):
        og.gather(cache, np.zeros((1, 1), np.int32), np.array([0, 1], np.int32), None, 1, 1, 0, 1,
                  "bf16", "bf16", 1.0, dst)
    with pytest.raises(ValueError):
        og.gather(cache, np.zeros((1, 1), np.int32), np.array([0, 1], np.int32), None, 1, 1, 1, 1,
                  "bf16", "fp16", 1.0, dst)
