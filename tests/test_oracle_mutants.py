"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of oracle/pmg_oracle.c (an
index off by one, a dropped seq_starts, a missing clamp at total_tokens, the
wrong row stride, truncation or round-half-up instead of round-half-even, a
wrong FP8 exponent bias or subnormal scale, a dropped dequant scale, an
accepted request whose rows start below an earlier cu_seq_lens boundary, an
accepted negative start), builds it with gcc, and
runs a battery of the pins against it: hand-worked golden cases, the numpy-only
second route, closed forms, and the conversion checks against torch and
numpy. Every mutant must fail at least one pin. The committed oracle is never
modified and the CUDA path is not involved.
"""
import contextlib
import json
import os
import subprocess

import numpy as np
import pytest
import torch

from oracle import gather as og

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pmg_oracle.c")
GOLDEN = os.path.join(ROOT, "tests", "golden", "hand_cases.json")

MUTANTS = {
    "slot off by one": ("const int64_t slot = p % B;", "const int64_t slot = (p + 1) % B;"),
    "logical block off by one": ("const int64_t logical = p / B;", "const int64_t logical = (p + 1) / B;"),
    "seq_starts ignored": ("const int64_t p = start + i;", "const int64_t p = i;"),
    "no clamp at total_tokens": ("const int64_t oe = cu_seq_lens[r + 1] < T ? cu_seq_lens[r + 1] : T;",
                                 "const int64_t oe = cu_seq_lens[r + 1];"),
    "dst row stride ignored": ("uint8_t* d = dst + (ob + i) * dst_token_stride * ed;",
                               "uint8_t* d = dst + (ob + i) * entry_size * ed;"),
    "bf16 truncation": ("u += 0x7FFFu + lsb;", "u += 0u * lsb;"),
    "bf16 round half up": ("u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;"),
    "e4m3 exponent bias": ("mag = ldexpf((float)(8 + m), e - 10);", "mag = ldexpf((float)(8 + m), e - 11);"),
    "e4m3 subnormal scale": ("mag = ldexpf((float)m, -9);", "mag = ldexpf((float)m, -10);"),
    "fp16 ties away from zero": ("if (rem > half || (rem == half && (q & 1u))) q += 1u;", "if (rem >= half) q += 1u;"),
    "dequant scale dropped": ("v = pmg_oracle_e4m3_to_f32(s[0]) * scale;", "v = pmg_oracle_e4m3_to_f32(s[0]) * 1.0f;"),
    # (rows below row 0 stay refused: a mutant must not write outside its dst)
    "rows below an earlier boundary accepted": ("if (len > 0 && ob < below) {", "if (len > 0 && ob < 0) {"),
    "earlier boundaries forgotten": ("if (ob > floor_row) floor_row = ob;", ";"),
    "negative start accepted": ("if (len > 0 && start < 0) {", "if (len > 0 && start < -1000000) {"),
    "token position off by one": ("const int64_t pos = t - first_row;", "const int64_t pos = t - first_row + 1;"),
    "token row range unchecked": ("if (t < first_row || t >= end_row) {", "if (t >= end_row + 1000000) {"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: expression not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib),
                           str(path), "-lm"])
    return og.load(str(lib))


@contextlib.contextmanager
def _using(lib):
    saved = og._lib
    og._lib = lib
    try:
        yield
    finally:
        og._lib = saved


def _id_cache(nb, B, E, rs=None):
    rs = E if rs is None else rs
    b = np.arange(nb, dtype=np.uint32)[:, None, None]
    s = np.arange(B, dtype=np.uint32)[None, :, None]
    e = np.arange(rs, dtype=np.uint32)[None, None, :]
    return (b << 20) | (s << 10) | e


GUARD_ROWS = 64


def _guarded(rows, cols, fill=0xA5A5A5A5):
    """(buffer, view): a destination of `rows` rows inside GUARD_ROWS sentinel
    rows on each side, so that a mutant that writes a row before 0 or past the
    end writes into memory the test owns (and fails the guard check) instead of
    corrupting the heap."""
    buf = np.full((rows + 2 * GUARD_ROWS, cols), 0x5A5A5A5A, np.uint32)
    view = buf[GUARD_ROWS:GUARD_ROWS + rows]
    view[:] = fill
    return buf, view


def _guards_intact(buf):
    return bool(np.all(buf[:GUARD_ROWS] == 0x5A5A5A5A)) and bool(np.all(buf[-GUARD_ROWS:] == 0x5A5A5A5A))


def _pin_hand_cases():
    for c in json.load(open(GOLDEN))["cases"]:
        if "rows" not in c:
            continue
        E = 3
        cache = _id_cache(c["num_blocks"], c["block_size"], E)
        cu = np.array(c["cu_seq_lens"], np.int32)
        T = c["total_tokens"]
        buf, dst = _guarded(T, E)
        ss = None if c["seq_starts"] is None else np.array(c["seq_starts"], np.int32)
        flag = og.gather(cache, np.array(c["block_table"], np.int32), cu, ss, len(cu) - 1, T, c["block_size"], E,
                         "fp32", "fp32", 1.0, dst)
        if flag != c["flag"] or not _guards_intact(buf):
            return False
        for i, want in enumerate(c["rows"]):
            if want is None:
                if not np.all(dst[i] == 0xA5A5A5A5):
                    return False
            elif (int(dst[i, 0] >> 20), int((dst[i, 0] >> 10) & 0x3FF)) != tuple(want):
                return False
    return True


def _pin_library_route():
    rng = np.random.default_rng(7)
    for _ in range(20):
        R, B, E = int(rng.integers(1, 8)), int(rng.choice([1, 3, 16])), 4
        lens = [int(x) for x in rng.integers(0, 4 * B + 3, R)]
        starts = [int(x) for x in rng.integers(0, 2 * B + 1, R)]
        need = [-(-(starts[r] + lens[r]) // B) for r in range(R)]
        nb = max(sum(need), 1)
        perm = rng.permutation(nb).astype(np.int32)
        bt = np.full((R, max(need + [1])), -1, np.int32)
        pos = 0
        for r in range(R):
            bt[r, :need[r]] = perm[pos:pos + need[r]]
            pos += need[r]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        cache = _id_cache(nb, B, E)
        buf, dst = _guarded(T, E)
        if og.gather(cache, bt, cu, np.array(starts, np.int32), R, T, B, E, "fp32", "fp32", 1.0, dst) != 0:
            return False
        if not _guards_intact(buf):
            return False
        for r in range(R):
            if lens[r] == 0:
                continue
            ctx = cache[bt[r, :need[r]].astype(np.int64)].reshape(need[r] * B, -1)
            if not np.array_equal(dst[cu[r]:cu[r + 1]], ctx[starts[r]:starts[r] + lens[r]]):
                return False
    return True


def _pin_padded_and_clamp():
    cache = _id_cache(3, 4, 3, rs=5)
    gbuf, dst = _guarded(10, 6)
    og.gather(cache, np.array([[2, 0, 1]], np.int32), np.array([0, 10], np.int32), np.array([1], np.int32), 1, 10,
              4, 3, "fp32", "fp32", 1.0, dst)
    if not _guards_intact(gbuf):
        return False
    for i in range(10):
        p = 1 + i
        if not np.array_equal(dst[i, :3], cache[[2, 0, 1][p // 4], p % 4, :3]) or not np.all(dst[i, 3:] == 0xA5A5A5A5):
            return False
    # rows past total_tokens are never written (the buffer is larger than any
    # row a mistaken oracle could reach, so a mutant cannot write out of bounds)
    cache = _id_cache(4, 4, 2)
    buf = np.full((20, 2), 0x5A5A5A5A, np.uint32)
    buf[:6] = 0xA5A5A5A5
    og.gather(cache, np.array([[0, 1, 2, 3]], np.int32), np.array([2, 14], np.int32), None, 1, 6, 4, 2, "fp32",
              "fp32", 1.0, buf)
    return bool(np.all(buf[6:] == 0x5A5A5A5A)) and bool(np.all(buf[:2] == 0xA5A5A5A5))


def _same(a, b, nan):
    an, bn = nan(a), nan(b)
    return np.array_equal(an, bn) and np.array_equal(a[~an], b[~bn])


def _pin_conversions():
    codes = np.arange(256, dtype=np.uint8)
    f32nan = lambda x: ((x & 0x7F800000) == 0x7F800000) & ((x & 0x7FFFFF) != 0)
    ours = np.array([og.e4m3_to_f32(int(c)) for c in codes], np.float32).view(np.uint32)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy().view(np.uint32)
    if not _same(ours, ref, f32nan):
        return False
    bfnan = lambda x: ((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)
    hnan = lambda x: ((x & 0x7C00) == 0x7C00) & ((x & 0x3FF) != 0)
    for scale in (0.05, 1.0):
        got = og.convert_array(codes, "fp8_e4m3", "bf16", scale)
        want = (torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float() * scale).to(torch.bfloat16)
        if not _same(got, want.view(torch.int16).numpy().view(np.uint16), bfnan):
            return False
    rng = np.random.default_rng(3)
    bits = np.concatenate([rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32),
                           np.array([0x3F808000, 0x3F818000, 0x00018000], np.uint32)])
    ours = np.fromiter((og.f32_to_bf16(float(x)) for x in bits.view(np.float32)), np.uint16, count=len(bits))
    ref = torch.from_numpy(bits.view(np.float32).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if not _same(ours, ref, bfnan):
        return False
    near = ((rng.integers(0, 2, 20000, dtype=np.uint32) << 31) | (rng.integers(97, 144, 20000, dtype=np.uint32) << 23)
            | rng.integers(0, 2 ** 23, 20000, dtype=np.uint32))
    ties = np.array([0x3F801000, 0x3F803000, 0x33000000, 0x33800000], np.uint32)  # fp16 ties, subnormal ties
    near = np.concatenate([near, ties])
    ours = np.fromiter((og.f32_to_f16(float(x)) for x in near.view(np.float32)), np.uint16, count=len(near))
    with np.errstate(over="ignore"):
        ref = near.view(np.float32).astype(np.float16).view(np.uint16)
    return _same(ours, ref, hnan)


def _pin_token_cases():
    for c in json.load(open(os.path.join(ROOT, "tests", "golden", "token_cases.json")))["cases"]:
        E = 3
        cache = _id_cache(c["num_blocks"], c["block_size"], E)
        t2s = np.array(c["token_to_seq"], np.int32)
        cu = np.array(c["cu_seq_lens"], np.int32)
        buf, dst = _guarded(len(t2s), E)
        flag = og.gather_tokens(cache, np.array(c["block_table"], np.int32), t2s, cu, len(cu) - 1, len(t2s),
                                c["block_size"], E, "fp32", "fp32", 1.0, dst)
        if flag != c["flag"] or not _guards_intact(buf):
            return False
        for i, want in enumerate(c["rows"]):
            if want is None:
                if not np.all(dst[i] == 0xA5A5A5A5):
                    return False
            elif not np.array_equal(dst[i], cache[want[0], want[1]]):
                return False
    return True


PINS = [_pin_hand_cases, _pin_library_route, _pin_padded_and_clamp, _pin_conversions, _pin_token_cases]


def _run(pin) -> bool:
    """A pin that raises (e.g. an unexpected flag from a helper) has failed."""
    try:
        return bool(pin())
    except Exception:
        return False


def test_pins_pass_on_the_real_oracle():
    assert all(pin() for pin in PINS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_fails_a_pin(tmp_path, name):
    old, new = MUTANTS[name]
    mutant = _build_mutant(tmp_path, name, old, new)
    with _using(mutant):
        results = {pin.__name__: _run(pin) for pin in PINS}
    assert not all(results.values()), f"mutant '{name}' passed every pin: {results}"
