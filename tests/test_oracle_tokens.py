"""Pins for the oracle's per-token indexed gather.

Source: "indexer kernels take shape arguments at run time" (prhub.com.cn, vllm
PR #56153), section "关键源码片段" (_cp_gather_indexer_quant_cache_kernel):
output token t reads request token_to_seq[t] at position t - cu_seqlen[b],
with every index masked before use.

Pins: hand-worked golden cases (tests/golden/token_cases.json), and equality
with the page gather's oracle (itself pinned) whenever token_to_seq names each
token's own request, which is the only case where the two definitions say the
same thing.
"""
import json
import os

import numpy as np
import pytest

from oracle import gather as og

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "token_cases.json")
FILL = 0xA5A5A5A5


def _id_cache(nb, B, E):
    b = np.arange(nb, dtype=np.uint32)[:, None, None]
    s = np.arange(B, dtype=np.uint32)[None, :, None]
    e = np.arange(E, dtype=np.uint32)[None, None, :]
    return (b << 20) | (s << 10) | e


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_cases(case):
    E = 3
    cache = _id_cache(case["num_blocks"], case["block_size"], E)
    t2s = np.array(case["token_to_seq"], np.int32)
    cu = np.array(case["cu_seq_lens"], np.int32)
    dst = np.full((len(t2s), E), FILL, np.uint32)
    flag = og.gather_tokens(cache, np.array(case["block_table"], np.int32), t2s, cu, len(cu) - 1, len(t2s),
                            case["block_size"], E, "fp32", "fp32", 1.0, dst)
    assert flag == case["flag"]
    for i, want in enumerate(case["rows"]):
        if want is None:
            assert np.all(dst[i] == FILL), f"row {i} written"
        else:
            assert (int(dst[i, 0] >> 20), int((dst[i, 0] >> 10) & 0x3FF)) == tuple(want), f"row {i}"
            assert np.array_equal(dst[i], cache[want[0], want[1]])


def token_to_seq_from_cu(cu: np.ndarray, T: int) -> np.ndarray:
    t2s = np.full(T, -1, np.int32)
    for r in range(len(cu) - 1):
        t2s[cu[r]:cu[r + 1]] = r
    return t2s


@pytest.mark.parametrize("seed", range(25))
def test_matches_page_gather_when_token_to_seq_is_consistent(seed):
    rng = np.random.default_rng(500 + seed)
    R = int(rng.integers(1, 10))
    B = int(rng.choice([1, 3, 16, 64]))
    lens = [int(x) if rng.random() > 0.2 else 0 for x in rng.integers(0, 4 * B + 5, R)]
    need = [-(-lens[r] // B) for r in range(R)]
    nb = max(sum(need), 1)
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((R, max(need + [1])), -1, np.int32)
    pos = 0
    for r in range(R):
        bt[r, :need[r]] = perm[pos:pos + need[r]]
        pos += need[r]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    E = 5
    cache = rng.integers(0, 2 ** 16, (nb, B, E), dtype=np.uint16)
    a = np.full((T, E), 0x5A5A, np.uint16)
    b = a.copy()
    fa = og.gather(cache, bt, cu, None, R, T, B, E, "bf16", "bf16", 1.0, a)
    fb = og.gather_tokens(cache, bt, token_to_seq_from_cu(cu, T), cu, R, T, B, E, "bf16", "bf16", 1.0, b)
    assert fa == fb == 0
    assert np.array_equal(a, b)
    # dequant too: fp8 codes without NaN through both definitions
    c8 = rng.integers(0, 0x7E, (nb, B, E), dtype=np.uint8)
    a8 = np.zeros((T, E), np.uint16)
    b8 = a8.copy()
    og.gather(c8, bt, cu, None, R, T, B, E, "fp8_e4m3", "bf16", 0.05, a8)
    og.gather_tokens(c8, bt, token_to_seq_from_cu(cu, T), cu, R, T, B, E, "fp8_e4m3", "bf16", 0.05, b8)
    assert np.array_equal(a8, b8)
