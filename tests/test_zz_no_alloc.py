"""w4_gemm_noalloc: the GEMM entry point that takes no workspace.

It serves callers that cannot allocate device memory where they run the GEMM
(a plug-in in a framework that owns all device memory and gives extensions
no allocator, or a latency-critical loop that must not call cudaMalloc,
which can synchronize the device); its scratch is a fixed array inside
libw4.  These tests call it through the C ABI twice in a row and check each
result against the CPU oracle (float outputs within the parity bound, int32
accumulators bit-exact, W4A8 fp16 within one ulp), and against w4_gemm's
result with a caller workspace.  The file is named to be collected last.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import w4synth
from parity import assert_fp16_within_ulp, assert_within

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _scratch_bytes():
    """W4_NOALLOC_SCRATCH_BYTES as include/w4.h defines it."""
    text = open(os.path.join(ROOT, "include", "w4.h")).read()
    m = re.search(r"#define\s+W4_NOALLOC_SCRATCH_BYTES\s+\(([^)]*)\)", text)
    expr = m.group(1).replace("u", "")
    assert re.fullmatch(r"[0-9 *]+", expr), expr
    return eval(expr)


def _noalloc(lib):
    f = lib.w4_gemm_noalloc
    i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    f.argtypes = [p, i32, i64, i64, p, i32, i64, p, i32, p, i64, p, p, p, i32, p]
    f.restype = i32
    return f


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call(w4, a, a_code, b, wtype, N, s, s_code, z, gs, tok, ch, out, out_code):
    f = _noalloc(w4.load())
    M, K = a.shape
    st = f(_ptr(a), a_code, M, K, _ptr(b), wtype, N, _ptr(s), s_code, _ptr(z), gs, _ptr(tok),
           _ptr(ch), _ptr(out), out_code, torch.cuda.current_stream().cuda_stream)
    return st


def test_noalloc_w4a16_matches_oracle(gpu_lib):
    w4 = gpu_lib
    M, N, K = 16, 4096, 14336
    d = w4synth.gen_w4a16(M, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4,
                          layout=w4.NK_EXLLAMA, group_size=128, zeros=True, seed=11)
    a, s, z = d["a"].to(DEV), d["s"].to(DEV), d["z"].to(DEV)
    b = w4.prepack_B(d["w"].to(DEV), d["wtype"], d["layout"], K, N)
    # this shape runs the streamed stream-K schedule, so the scratch holds
    # the staged activations and partial sums
    assert w4.schedule_names()[w4.default_schedule(M, N, K, torch.bfloat16, 128)] == "ds16_sk"
    ref, absref = oracle.w4a16(d["a"], d["w"], d["layout"], d["wtype"], d["s"], d["z"], 128, K, N)
    with_ws = w4.gemm(a, b, d["wtype"], N, scales=s, zeros=z, group_size=128)
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        st = _call(w4, a, w4.BF16, b, d["wtype"], N, s, w4.BF16, z, 128, None, None, out, w4.BF16)
        assert st == w4.OK, w4.load().w4_last_error().decode()
        torch.cuda.synchronize()
        assert_within(out.double().cpu().numpy(), ref, absref, "bf16", f"noalloc call {call}")
        # the same schedule adds its partial sums in the same order
        assert torch.equal(out, with_ws), f"noalloc call {call} differs from w4_gemm"


@pytest.mark.parametrize("gs", [-1, 128])
def test_noalloc_w4a8_matches_oracle(gpu_lib, gs):
    w4 = gpu_lib
    M, N, K = 8, 8192, 21760
    e = w4synth.gen_w4a8(M, N, K, group_size=gs, seed=12)
    a = e["a"].to(DEV)
    sg = None if e["sg"] is None else e["sg"].to(DEV)
    tok, ch = e["s_tok"].to(DEV), e["s_ch"].to(DEV)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], K, N)
    ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], e["sg"], gs, K, N)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref16 = oracle.w4a8_scale(ref.reshape(-1), rows.reshape(-1), cols.reshape(-1), e["s_tok"],
                              e["s_ch"])
    with_ws = w4.gemm(a, b, e["wtype"], N, scales=sg, group_size=gs, out_dtype=torch.int32)
    for call in range(2):
        acc = torch.zeros((M, N), dtype=torch.int32, device=DEV)
        st = _call(w4, a, w4.S8, b, e["wtype"], N, sg, w4.S8, None, gs, None, None, acc, w4.S32)
        assert st == w4.OK, w4.load().w4_last_error().decode()
        out = torch.zeros((M, N), dtype=torch.float16, device=DEV)
        st = _call(w4, a, w4.S8, b, e["wtype"], N, sg, w4.S8, None, gs, tok, ch, out, w4.F16)
        assert st == w4.OK, w4.load().w4_last_error().decode()
        torch.cuda.synchronize()
        assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref), f"call {call}"
        assert torch.equal(acc, with_ws), f"call {call} differs from w4_gemm"
        assert_fp16_within_ulp(out.double().cpu().numpy().reshape(-1), ref16, f"call {call}")


def test_noalloc_rejects_problems_above_its_scratch(gpu_lib):
    w4 = gpu_lib
    M, N, K = 1024, 8192, 21760  # the bf16 copy of a alone is 44.6 MB
    assert w4.workspace_size(M, N, K, torch.int8, -1) > _scratch_bytes()
    a = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    b = torch.zeros(w4.prepacked_size(K, N), dtype=torch.uint8, device=DEV)
    out = torch.full((M, N), 3, dtype=torch.int32, device=DEV)
    st = _call(w4, a, w4.S8, b, w4.INT4, N, None, w4.S8, None, -1, None, None, out, w4.S32)
    assert st == w4.ERR_WORKSPACE
    assert "workspace too small" in w4.load().w4_last_error().decode()
    torch.cuda.synchronize()
    assert int((out != 3).sum()) == 0  # nothing ran
