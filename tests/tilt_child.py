"""Child process of test_tilt_gpu.py: GPU parity against the oracle on the
workloads whose static split the tilt reaches, under the scheduling variables
the parent put in the environment (the library reads them once per process).
Prints one line "tilt-child ok <cases>" when every case matched."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path[:0] = [os.path.dirname(HERE), HERE]

import torch  # noqa: E402

from paged_mla_kv_cache_gb300 import workloads as W  # noqa: E402
from gpu_helpers import DeviceCase, assert_same, oracle_run  # noqa: E402
from test_gather_tokens_gpu import _run as run_tokens, token_to_seq_from_cu  # noqa: E402


def page_case(wl, workspace):
    case = DeviceCase(wl, workspace=workspace)
    case.run()
    got, flag, guards = case.result()
    want, oflag = oracle_run(wl)
    assert guards, f"{wl.name}: guard regions written"
    assert oflag == 0 and flag == 0, f"{wl.name}: flags {flag} / {oflag}"
    assert_same(got, want, wl.dst_dtype, wl.src_dtype != wl.dst_dtype)


def main():
    assert torch.cuda.is_available()
    sk = W.skew8()
    starts = sk.seq_starts.tolist()
    page = [
        W.skew8(),
        W.make_workload("skew-8 lengths, bf16", W.SKEW8_LENS, starts, 64, 576, 1024, "bf16", "bf16", 1.0, 11),
        W.make_workload("one fp8 request, 30000", [30000], None, 64, 576, 1024, "fp8_e4m3", "bf16", 0.05, 12),
        # 32 rows per CTA of the converter's grid on a 152-SM part: the smallest split the tilt takes
        W.make_workload("8 x 2432 fp8", [2432] * 8, None, 64, 576, 512, "fp8_e4m3", "bf16", 0.05, 13),
        W.make_workload("3 fp8 requests, 7 rows short of a stage", [9001, 77, 11000], [5, 0, 63], 64, 576, 512,
                        "fp8_e4m3", "fp32", 0.05, 14),
    ]
    n = 0
    for wl in page:
        for ws in (False, True):
            page_case(wl, ws)
            n += 1
    tok = W.make_workload("skew-8 lengths, per token", W.SKEW8_LENS, None, 64, 576, 1024, "fp8_e4m3", "bf16", 0.05,
                          15)
    cu = tok.cu_seq_lens.numpy().copy()
    t2s = token_to_seq_from_cu(cu, int(cu[-1]))
    for ws in (False, True):
        run_tokens(tok, t2s, cu, workspace=ws)
        n += 1
    torch.cuda.synchronize()
    print(f"tilt-child ok {n}", flush=True)


if __name__ == "__main__":
    main()
