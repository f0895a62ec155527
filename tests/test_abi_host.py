"""CPU-only checks of the C ABI: the library builds and loads, exports every
entry point include/pmg.h declares, and rejects bad calls on the host before
any CUDA call (the host half of every entry point makes none)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from paged_mla_kv_cache_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pmg.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(pmg_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    assert declared_functions() == ["pmg_debug_noalloc_scratch", "pmg_debug_plan", "pmg_gather", "pmg_gather_ex",
                                    "pmg_gather_noalloc", "pmg_gather_tokens", "pmg_select_path",
                                    "pmg_status_string", "pmg_version"]


def test_library_exports_every_declared_symbol(cuda_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (pmg_\w+)$", out.stdout, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(cuda_lib, name)
    assert cuda_lib.pmg_version() == 1


def test_status_strings(cuda_lib):
    for st in range(7):
        assert binding.status_string(st).startswith(binding.STATUS_NAMES[st])
    assert binding.status_string(99) == "unknown pmg status"


def _args(**over):
    # host stand-ins: the host half only looks at pointer values
    a = dict(cache=16 * 1024, cbs=64 * 576, cts=576, nb=8, bt=4096, bts=4, cu=8192, ss=0, R=2, T=100, B=64,
             E=576, sdt=0, ddt=0, scale=0, dst=32 * 1024, dts=576, err=0, ws=0, opt=0)
    a.update(over)
    return a


def _gather(L, a):
    return L.pmg_gather_ex(a["cache"] or None, a["cbs"], a["cts"], a["nb"], a["bt"] or None, a["bts"],
                           a["cu"] or None, a["ss"] or None, a["R"], a["T"], a["B"], a["E"], a["sdt"], a["ddt"],
                           a["scale"] or None, a["dst"] or None, a["dts"], a["err"] or None, a["ws"] or None, None,
                           a["opt"])


def _path(L, a):
    p, u = ctypes.c_int32(-1), ctypes.c_int32(-1)
    st = L.pmg_select_path(a["cache"] or None, a["cbs"], a["cts"], a["nb"], a["bt"] or None, a["bts"],
                           a["cu"] or None, a["R"], a["T"], a["B"], a["E"], a["sdt"], a["ddt"], a["dst"] or None,
                           a["dts"], a["opt"], ctypes.byref(p), ctypes.byref(u))
    return st, binding.PATH_NAMES.get(p.value), u.value


@pytest.mark.parametrize("over,status", [
    (dict(cache=0), 1), (dict(bt=0), 1), (dict(cu=0), 1), (dict(dst=0), 1),
    (dict(sdt=9), 3), (dict(sdt=0, ddt=1), 3), (dict(sdt=3, ddt=4), 3), (dict(sdt=2, ddt=0), 3),
    (dict(R=-1), 2), (dict(T=-1), 2), (dict(B=0), 2), (dict(E=0), 2), (dict(dts=575), 2), (dict(cts=-1), 2),
    (dict(nb=-1), 2), (dict(opt=64), 2),
    (dict(R=binding.MAX_REQS + 1), 5),
    (dict(R=binding.MAX_REQS_PLAN + 1), 5),  # more than one launch plans needs a workspace
    (dict(cache=16 * 1024 + 1), 4), (dict(dst=32 * 1024 + 1), 4), (dict(bt=4098), 4), (dict(ss=8194), 4),
    (dict(ws=64 * 1024 + 8), 4),
])
def test_host_validation_rejects(cuda_lib, over, status):
    assert _gather(cuda_lib, _args(**over)) == status
    st, _, _ = _path(cuda_lib, _args(**over))
    if "ss" not in over and "ws" not in over and over.get("R") != binding.MAX_REQS_PLAN + 1:
        # select_path takes no seq_starts or workspace (and accepts large batches)
        assert st == status


@pytest.mark.parametrize("over", [dict(R=0), dict(T=0), dict(R=0, cache=0, bt=0, cu=0, dst=0)])
def test_nothing_to_do_launches_nothing(cuda_lib, over):
    # returns OK without touching CUDA (there is no GPU here)
    assert _gather(cuda_lib, _args(**over)) == 0
    st, path, unit = _path(cuda_lib, _args(**over))
    assert st == 0 and path == "none" and unit == 0


@pytest.mark.parametrize("over,path,unit", [
    (dict(), "bulk", 0),                                                  # bf16 576, 16-B aligned rows
    (dict(opt=binding.OPT_FORCE_SIMT), "vector", 8),                      # 16 B = 8 bf16
    (dict(opt=binding.OPT_FORCE_SCALAR), "scalar", 1),
    (dict(cts=640, cbs=64 * 640), "bulk", 0),                             # padded rows, still 16-B aligned
    (dict(cts=577, cbs=64 * 577), "realign", 0),                          # 1154-B row starts: realigned 16-B words
    (dict(cts=577, cbs=64 * 577, opt=binding.OPT_FORCE_SIMT), "scalar", 1),  # forced SIMT: one bf16 per access
    (dict(cts=580, cbs=64 * 580), "realign", 0),                          # 8-B aligned rows: realigned too
    (dict(cts=580, cbs=64 * 580, opt=binding.OPT_FORCE_SIMT), "vector", 4),
    (dict(dts=577), "realign", 0),                                        # only the output rows unaligned
    (dict(E=7, cts=7, cbs=64 * 7, dts=7), "scalar", 1),
    (dict(sdt=3, ddt=0), "bulk", 0),                                      # fp8 -> bf16: TMA in, converter warps out
    (dict(sdt=3, ddt=0, opt=binding.OPT_FORCE_SIMT), "vector", 16),       # fp8 -> bf16 SIMT, 16 codes per load
    (dict(sdt=3, ddt=0, cts=577, cbs=64 * 577), "realign", 0),           # odd fp8 rows: realigned words
    (dict(sdt=3, ddt=0, cts=577, cbs=64 * 577, opt=binding.OPT_FORCE_SIMT), "scalar", 1),
    (dict(sdt=3, ddt=0, cts=640, cbs=64 * 640, dts=600), "bulk", 0),      # padded rows on both sides
    (dict(sdt=3, ddt=0, E=572, cts=572, cbs=64 * 572, dts=572), "realign", 0),  # 572 % 8 != 0: no TMA units
    (dict(sdt=3, ddt=0, E=572, cts=572, cbs=64 * 572, dts=572, opt=binding.OPT_FORCE_SIMT), "vector", 4),
    (dict(sdt=3, ddt=2, dst=32 * 1024 + 16), "bulk", 0),                  # fp32 out, 16-B aligned
    (dict(sdt=3, ddt=2, dst=32 * 1024 + 4), "realign", 0),                # fp32 out, only 4-B aligned rows
    (dict(sdt=3, ddt=2, dst=32 * 1024 + 4, opt=binding.OPT_FORCE_SIMT), "scalar", 1),
    (dict(sdt=0, ddt=2), "bulk", 0),                                      # bf16 -> fp32
    (dict(sdt=0, ddt=2, dts=578), "realign", 0),                          # bf16 -> fp32, 8-B aligned out rows
    (dict(sdt=0, ddt=2, dts=578, opt=binding.OPT_FORCE_SIMT), "vector", 2),
    (dict(sdt=3, ddt=0, E=7, cts=7, cbs=64 * 7, dts=7), "scalar", 1),    # 14-B output rows: below one word
    (dict(sdt=2, ddt=2), "bulk", 0),                                      # fp32 copy
    (dict(sdt=4, ddt=4, E=5, cts=5, cbs=320, dts=5), "scalar", 1),       # u8 odd rows
    (dict(sdt=4, ddt=4, E=12, cts=12, cbs=768, dts=12), "vector", 4),     # u8 rows of 12 B: 4-byte units
    (dict(sdt=4, ddt=4, E=17, cts=17, cbs=64 * 17, dts=17), "realign", 0),  # u8 rows of 17 B
    (dict(sdt=2, ddt=2, E=5, cts=5, cbs=320, dts=5), "realign", 0),       # fp32 rows of 20 B
])
def test_path_selection(cuda_lib, over, path, unit):
    st, p, u = _path(cuda_lib, _args(**over))
    assert st == 0
    assert (p, u) == (path, unit)


def test_binding_requires_contiguous_table():
    bt = torch.zeros(3, 8, dtype=torch.int32)[:, :4]
    cache = torch.zeros(2, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.select_path(cache, torch.zeros(4, 8, dtype=torch.bfloat16), bt, torch.zeros(4, dtype=torch.int32))


def test_binding_select_path_on_cpu_tensors(cuda_lib):
    cache = torch.zeros(4, 64, 640, dtype=torch.bfloat16)[:, :, :576]
    dst = torch.zeros(10, 576, dtype=torch.bfloat16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    cu = torch.tensor([0, 4, 10], dtype=torch.int32)
    path, unit = binding.select_path(cache, dst, bt, cu)
    assert path in ("bulk", "vector")  # depends on the allocator's alignment of these host tensors
    path, unit = binding.select_path(cache, dst, bt, cu, options=binding.OPT_FORCE_SCALAR)
    assert (path, unit) == ("scalar", 1)


def _tokens(L, **over):
    a = dict(cache=16 * 1024, cbs=64 * 576, cts=576, nb=8, bt=4096, bts=4, t2s=8192, cu=12288, R=2, T=100, B=64,
             E=576, sdt=0, ddt=0, scale=0, dst=32 * 1024, dts=576, err=0, ws=0, opt=0)
    a.update(over)
    return L.pmg_gather_tokens(a["cache"] or None, a["cbs"], a["cts"], a["nb"], a["bt"] or None, a["bts"],
                               a["t2s"] or None, a["cu"] or None, a["R"], a["T"], a["B"], a["E"], a["sdt"], a["ddt"],
                               a["scale"] or None, a["dst"] or None, a["dts"], a["err"] or None, a["ws"] or None,
                               None, a["opt"])


@pytest.mark.parametrize("over,status", [
    (dict(t2s=0), 1), (dict(dst=0), 1), (dict(cache=0), 1), (dict(cu=0), 1),
    (dict(sdt=0, ddt=1), 3), (dict(T=-1), 2), (dict(B=0), 2), (dict(dts=100), 2), (dict(opt=4), 2),
    (dict(opt=16), 2), (dict(T=2 ** 31), 5), (dict(t2s=8194), 4), (dict(cache=16 * 1024 + 1), 4),
    (dict(ws=40 * 1024 + 8), 4),
    (dict(T=0), 0), (dict(T=0, t2s=0, dst=0), 0),
])
def test_token_gather_host_validation(cuda_lib, over, status):
    assert _tokens(cuda_lib, **over) == status
