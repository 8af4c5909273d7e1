"""The device-side timeout path: a bounded wait gives up, the kernel records
W4_ERR_TIMEOUT in the workspace status word and returns, w4_check_status
reports it and re-zeroes the split-K counters, and the next call on that
workspace is correct again.

The wait is made to run out from the host, with no fault: the workspace's
split-K tile counters are pre-set so that their high half (the count of
contributors that have written their partial sums, which the last arriving
warp of a split tile waits for) starts at -32768 and can never reach its
target.  The last arriver waits its 2 s limit, gives up, sets the status
word and returns; every other warp of its CTA sees the CTA's abort flag and
returns too.  Nothing traps, faults or hangs.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import w4synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
HEADER = 256              # status word + spare, then the split-K counters
COUNTER_BYTES = 64 * 1024


def test_split_k_wait_times_out_and_recovers(gpu_lib):
    w4 = gpu_lib
    M, N, K = 40, 384, 2048
    e = w4synth.gen_w4a8(M, N, K, group_size=-1, seed=41)
    a = e["a"].to(DEV)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], K, N)
    sched = w4.schedule_names().index("tc64_sk")  # 3 tiles of 8 stages over 12 CTAs: split tiles
    nbytes = w4.workspace_size(M, N, K, torch.int8, -1)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    ws[HEADER:HEADER + COUNTER_BYTES].view(torch.int32).fill_(-(2 ** 31))  # 0x80000000
    torch.cuda.synchronize()

    t0 = time.time()
    w4.gemm(a, b, e["wtype"], N, group_size=-1, out_dtype=torch.int32, ws=ws, schedule=sched)
    st = w4.check_status(ws)
    waited = time.time() - t0
    assert st == w4.ERR_TIMEOUT, w4.status_string(st)
    assert waited >= 1.5, f"returned after {waited:.2f} s: the wait did not run to its limit"
    # the status word and the counters are zero again
    assert int(ws[:HEADER + COUNTER_BYTES].view(torch.int32).abs().sum()) == 0

    # the same workspace serves the next call correctly
    acc = w4.gemm(a, b, e["wtype"], N, group_size=-1, out_dtype=torch.int32, ws=ws,
                  schedule=sched)
    assert w4.check_status(ws) == w4.OK
    ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], None, -1, K, N)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref)
