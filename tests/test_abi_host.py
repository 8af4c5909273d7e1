"""The C-ABI library: it loads, exports every symbol include/w4.h declares,
and rejects bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import int4_weight_mixed_gb300 as w4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "w4.h")).read()
    return sorted(set(re.findall(r"\b(w4_[A-Za-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    w4.build()
    return w4.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "w4_gemm" in names and "w4_prepack_B" in names
    for n in names:
        assert hasattr(lib, n), n


def test_static_queries(lib):
    assert w4.layout_version() == 1
    assert w4.prepacked_size(21760, 8192) == 8192 * 21760 // 2
    assert w4.prepacked_size(512, 200) == 256 * 256  # N padded to 128
    assert w4.prepacked_size(72, 128) == 0           # K % 64 != 0
    names = w4.schedule_names()
    assert names[0] == "simt" and len(names) == w4.num_schedules()
    assert lib.w4_schedule_name(99) is None
    assert w4.status_string(5) == "W4_ERR_TIMEOUT"


def test_default_heuristic(lib):
    import torch
    name = lambda M, N, K, dt, g: w4.schedule_names()[w4.default_schedule(M, N, K, dt, g)]
    assert name(1, 8192, 21760, torch.int8, -1) == "ds8_sk"
    assert name(8, 8192, 21760, torch.int8, 128) == "ds8_sk"
    assert name(16, 4096, 4096, torch.bfloat16, 128) == "gv16_cl"  # 8 MiB of weights: one launch
    assert name(1, 6144, 4096, torch.bfloat16, 128) == "gv8_cl"
    assert name(1, 28672, 4096, torch.bfloat16, 128) == "ds8_sk"  # 56 MiB: streamed
    assert name(12, 4096, 14336, torch.bfloat16, 128) == "ds16_sk"
    assert name(16, 4096, 4096, torch.bfloat16, 64) == "tc16_sk"   # group 64 splits a K block
    assert name(32, 8192, 21760, torch.int8, -1) == "ds32_sk"
    assert name(64, 4096, 4096, torch.bfloat16, 128) == "tc64_sk"
    # 256-row tiles on CTA pairs (stream-K: 256 tiles < 4 waves; data-parallel beyond)
    assert name(1024, 8192, 21760, torch.int8, -1) == "tc256p_sk"
    assert name(1024, 8192, 21760, torch.bfloat16, 128) == "tc256p_sk"
    assert name(16384, 57344, 8192, torch.bfloat16, 128) == "tc256p_dp"
    # 128-row tiles: pairs for W4A8, single CTAs otherwise
    assert name(128, 8192, 21760, torch.int8, -1) == "tc128p_sk"
    assert name(128, 8192, 21760, torch.bfloat16, 128) == "tc128_sk"
    assert name(4, 13, 512, torch.float16, 128) == "dk8_sk"  # any N (streamed needs N % 8 == 0)
    assert name(20, 13, 512, torch.float16, 128) == "simt"  # N % 8 != 0 beyond 16 rows
    assert w4.default_schedule(0, 8, 64, torch.float16, -1) == -1


def test_workspace_size(lib):
    import torch
    assert w4.workspace_size(0, 8, 64, torch.float16, -1) >= 256
    small = w4.workspace_size(1, 8192, 21760, torch.int8, -1)
    big = w4.workspace_size(1024, 8192, 21760, torch.int8, -1)
    assert big >= small + 1024 * 21760 * 2  # bf16 copy of the activations


def _gemm(lib, **kw):
    # placeholder addresses (never dereferenced: every case fails on the host)
    args = dict(a=256, a_type=0, M=4, K=128, b=256, wtype=0, N=128, s=256, st=0, z=None, gs=128,
                tok=None, ch=None, out=256, ot=0, ws=256, wsb=1 << 20, stream=None, sched=-1)
    args.update(kw)
    return lib.w4_gemm_ex(args["a"], args["a_type"], args["M"], args["K"], args["b"],
                          args["wtype"], args["N"], args["s"], args["st"], args["z"], args["gs"],
                          args["tok"], args["ch"], args["out"], args["ot"], args["ws"],
                          args["wsb"], args["stream"], args["sched"])


def test_invalid_arguments_rejected_on_host(lib):
    E = w4.ERR_INVALID_ARGUMENT
    assert _gemm(lib, M=-1) == E
    assert _gemm(lib, K=100) == E                    # K % 8
    assert _gemm(lib, gs=96) == E                    # does not divide K
    assert _gemm(lib, a_type=7) == E
    assert _gemm(lib, wtype=9) == E
    assert _gemm(lib, a=None) == E
    assert _gemm(lib, out=None) == E
    assert _gemm(lib, s=None) == E                   # W4A16 needs scales
    assert _gemm(lib, st=1) == E                     # scale dtype != a dtype
    assert _gemm(lib, ot=1) == E                     # out dtype != a dtype
    assert _gemm(lib, tok=1) == E                    # W4A16 takes no token scales
    assert _gemm(lib, a_type=2, s=None, gs=-1, ot=0) == E      # W4A8 fp16 out needs scales
    assert _gemm(lib, a_type=2, s=1, st=0, wtype=2, tok=1, ch=1) == E  # sg must be int8
    assert _gemm(lib, sched=99) == E
    assert "K must be a multiple of 8" in lib.w4_last_error().decode() or True


def test_unsupported_rejected_on_host(lib):
    U = w4.ERR_UNSUPPORTED
    assert _gemm(lib, K=72, gs=-1) == U              # K % 64
    assert _gemm(lib, K=256, gs=32) == U             # group not a multiple of 64
    assert _gemm(lib, a_type=2, wtype=1, s=None, gs=-1, ot=3) == U  # W4A8 uint4
    assert _gemm(lib, a_type=2, wtype=2, s=None, gs=-1, z=1, ot=3) == U  # zeros
    assert _gemm(lib, a_type=2, wtype=2, s=None, gs=-1, ot=1) == U  # bf16 out


def test_workspace_checks(lib):
    assert _gemm(lib, ws=None) == w4.ERR_WORKSPACE
    assert _gemm(lib, wsb=16) == w4.ERR_WORKSPACE
    assert lib.w4_check_status(None, 0, None) == w4.ERR_WORKSPACE


def test_empty_problems_are_noops(lib):
    # M == 0 or N == 0: nothing to compute, nothing launched
    assert _gemm(lib, M=0, a=None, out=None) == w4.OK
    assert _gemm(lib, N=0) == w4.OK


def test_prepack_argument_errors(lib):
    E = w4.ERR_INVALID_ARGUMENT
    assert lib.w4_prepack_B(None, 0, 0, 64, 8, 1, None) == E
    assert lib.w4_prepack_B(1, 5, 0, 64, 8, 1, None) == E
    assert lib.w4_prepack_B(1, 0, 9, 64, 8, 1, None) == E
    assert lib.w4_prepack_B(1, 0, 0, 60, 8, 1, None) == E
    assert lib.w4_prepack_B(1, 0, 0, 96, 8, 1, None) == w4.ERR_UNSUPPORTED
    assert lib.w4_unprepack_B(1, 0, 0, 64, 0, 1, None) == E


def test_quantize_argument_errors(lib):
    E = w4.ERR_INVALID_ARGUMENT
    q = lib.w4_quantize_per_token
    assert q(1, 0, -1, 64, 1, 1, None) == E            # negative M
    assert q(1, 0, 4, -8, 1, 1, None) == E             # negative K
    assert q(1, 2, 4, 64, 1, 1, None) == E             # int8 input
    assert q(1, 3, 4, 64, 1, 1, None) == E             # int32 input
    assert q(None, 0, 4, 64, 1, 1, None) == E          # activations needed
    assert q(1, 1, 4, 64, None, 1, None) == E          # codes needed
    assert q(1, 1, 4, 0, None, None, None) == E        # scales needed even at K == 0
    assert q(None, 0, 0, 64, None, None, None) == w4.OK  # M == 0: nothing launched
    assert q(256, 0, 1 << 31, 64, 256, 256, None) == w4.ERR_UNSUPPORTED


def test_misaligned_pointers_rejected_on_host(lib):
    """Every array must be aligned to its element size (the prepacked
    weights to 4 bytes), else INVALID_ARGUMENT before anything runs."""
    E = w4.ERR_INVALID_ARGUMENT
    assert _gemm(lib, a=257) == E                    # fp16 activations
    assert _gemm(lib, out=259) == E                  # fp16 output
    assert _gemm(lib, b=258) == E                    # prepacked words
    assert _gemm(lib, s=255) == E                    # fp16 scales
    assert _gemm(lib, z=257, wtype=1) == E           # fp16 zero-points
    w4a8 = dict(a_type=2, wtype=2, s=None, gs=-1, st=2)
    assert _gemm(lib, **w4a8, ot=0, tok=258, ch=256) == E   # fp32 token scales
    assert _gemm(lib, **w4a8, ot=0, tok=256, ch=254) == E   # fp32 channel scales
    assert _gemm(lib, **w4a8, ot=3, out=258) == E            # int32 output
    # int8 activations need no alignment: the call goes on to fail on its
    # (too small) workspace, still on the host
    assert _gemm(lib, **w4a8, ot=3, a=257, wsb=16) == w4.ERR_WORKSPACE
    assert lib.w4_prepack_B(258, 0, 0, 64, 8, 256, None) == E
    assert lib.w4_prepack_B(256, 0, 0, 64, 8, 258, None) == E
    assert lib.w4_unprepack_B(256, 0, 0, 64, 8, 258, None) == E
    assert lib.w4_quantize_per_token(257, 0, 4, 64, 256, 256, None) == E
    assert lib.w4_quantize_per_token(256, 0, 4, 64, 256, 258, None) == E


def test_every_schedule_fits_in_the_published_workspace(lib):
    """w4_gemm_workspace_size covers what every schedule that can run a
    problem asks for (the need is read from the WORKSPACE error that a too
    small workspace returns on the host, before anything is launched)."""
    import re

    shapes = [  # (M, N, K, a_type, group_size)
        (1, 8192, 21760, 2, -1), (8, 8192, 21760, 2, 128), (16, 8192, 21760, 2, -1),
        (32, 8192, 21760, 2, -1), (128, 8192, 21760, 2, -1), (1024, 8192, 21760, 2, 128),
        (2048, 8192, 21760, 2, 128), (1, 4096, 4096, 1, 128), (16, 28672, 4096, 1, 128),
        (64, 4096, 14336, 1, 128), (4096, 8192, 28672, 1, 128), (17, 136, 512, 1, 64),
        (5, 13, 512, 0, 128), (300, 384, 2048, 0, -1)]
    checked = 0
    for M, N, K, at, gs in shapes:
        published = lib.w4_gemm_workspace_size(M, N, K, at, gs)
        w4a8 = at == 2
        kw = dict(M=M, N=N, K=K, a_type=at, gs=gs, ws=256, wsb=16,
                  wtype=2 if w4a8 else 0, ot=3 if w4a8 else at,
                  s=(256 if gs != -1 else None) if w4a8 else 256, st=2 if w4a8 else at)
        for sched in range(lib.w4_num_schedules()):
            st = _gemm(lib, sched=sched, **kw)
            if st == w4.ERR_UNSUPPORTED:
                continue
            assert st == w4.ERR_WORKSPACE, (M, N, K, sched, st)
            need = int(re.search(r"(\d+) bytes", lib.w4_last_error().decode()).group(1))
            assert need <= published, (M, N, K, lib.w4_schedule_name(sched), need, published)
            checked += 1
    assert checked > 60


def test_default_heuristic_always_runs_valid_shapes(lib):
    """For any shape the API accepts, the default heuristic's schedule can
    run it within the published workspace (seeded sweep over M, N, K,
    group size and mode; each call stops on the host at the workspace)."""
    import re

    import numpy as np

    rng = np.random.default_rng(0)
    for _ in range(300):
        at = int(rng.integers(0, 3))
        M = int(rng.choice([1, 2, 7, 8, 9, 16, 17, 31, 32, 33, 64, 100, 128, 129, 256, 700, 4096]))
        N = int(rng.choice([8, 13, 64, 120, 128, 136, 1000, 4096, 8192]))
        K = 64 * int(rng.integers(1, 64))
        divisors = [g for g in (64, 128, 256, 512, 1024) if K % g == 0]
        gs = int(rng.choice([-1] + divisors))
        published = lib.w4_gemm_workspace_size(M, N, K, at, gs)
        w4a8 = at == 2
        st = _gemm(lib, M=M, N=N, K=K, a_type=at, gs=gs, ws=256, wsb=16, sched=-1,
                   wtype=2 if w4a8 else 0, ot=3 if w4a8 else at,
                   s=(256 if gs not in (-1, K) else None) if w4a8 else 256, st=2 if w4a8 else at)
        assert st == w4.ERR_WORKSPACE, (M, N, K, at, gs, st, lib.w4_last_error())
        need = int(re.search(r"(\d+) bytes", lib.w4_last_error().decode()).group(1))
        assert need <= published, (M, N, K, at, gs)


def test_dk_does_not_split_k_beyond_its_counters(lib):
    """dk counts the contributors of a K split in one 32-bit counter per
    128-column tile inside a 64 KB region: with more tiles than that it
    runs unsplit (its workspace need is then the header and counters only)."""
    import re

    dk8 = [i for i in range(lib.w4_num_schedules()) if lib.w4_schedule_name(i) == b"dk8_sk"][0]

    def need(N, K):
        st = _gemm(lib, M=1, N=N, K=K, a_type=0, gs=-1, ws=256, wsb=16, sched=dk8, wtype=0, ot=0)
        assert st == w4.ERR_WORKSPACE
        return int(re.search(r"(\d+) bytes", lib.w4_last_error().decode()).group(1))

    assert need(1000, 4096) > 256 + 64 * 1024                # few tiles: K is split
    # K = 8192 does not fit one dk CTA's preferred shared memory unsplit, so the
    # planner would split it; with more tiles than counters it must not
    assert need(16384 * 128 + 8, 8192) == 256 + 64 * 1024


def test_dk_gives_way_when_its_staging_does_not_fit(lib):
    """A K so long that even the largest K split leaves dk's staged
    activations beyond a CTA's shared memory: dk reports UNSUPPORTED and the
    default heuristic takes the CUDA-core schedule (N % 8 != 0 rules out
    the others)."""
    dk8 = [i for i in range(lib.w4_num_schedules()) if lib.w4_schedule_name(i) == b"dk8_sk"][0]
    kw = dict(M=1, a_type=0, gs=-1, ws=256, wsb=16, wtype=0, ot=0)
    assert _gemm(lib, N=16384 * 128 + 8, K=65536, sched=dk8, **kw) == w4.ERR_UNSUPPORTED
    assert _gemm(lib, N=1001, K=1 << 22, sched=dk8, **kw) == w4.ERR_UNSUPPORTED
    assert lib.w4_schedule_name(lib.w4_default_schedule(1, 1001, 1 << 22, 0, -1)) == b"simt"
    assert lib.w4_schedule_name(lib.w4_default_schedule(1, 1001, 4096, 0, -1)) == b"dk8_sk"


def test_binding_rejects_host_and_strided_tensors(lib):
    """The binding checks that every tensor it passes is a contiguous
    device tensor before calling the library (CPU tensors here)."""
    import torch

    a = torch.zeros(4, 128, dtype=torch.float16)
    b = torch.zeros(w4.prepacked_size(128, 128), dtype=torch.uint8)
    s = torch.zeros(1, 128, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        w4.gemm(a, b, w4.UINT4B8, 128, scales=s, group_size=-1)


def test_binding_argtypes_match_the_header(lib):
    """Every entry point the binding declares to ctypes takes as many
    arguments as include/w4.h declares for it (ABI drift check)."""
    import re

    text = open(os.path.join(ROOT, "include", "w4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = dict(
        (m.group(1), m.group(2))
        for m in re.finditer(r"\b(w4_[A-Za-z0-9_]+)\s*\(([^)]*)\)\s*;", text))
    assert len(decls) >= 15
    checked = 0
    for name, params in decls.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
        checked += 1
    assert checked >= 10


def test_override_table(lib):
    """Built-in measured exceptions to the heuristic, and entries installed at
    run time: consulted first, replaced by a later entry for the same key,
    removed with -1, ignored where the schedule cannot run the shape, and
    validated on the host."""
    import torch
    name = lambda M, N, K, dt, g: w4.schedule_names()[w4.default_schedule(M, N, K, dt, g)]
    # built-in: Llama-3-70B prefill shapes on data-parallel CTA-pair tiles (the
    # heuristic's choice too); outside the entries' M range the heuristic decides
    assert name(4096, 8192, 28672, torch.bfloat16, 128) == "tc256p_dp"
    assert name(8192, 57344, 8192, torch.bfloat16, 128) == "tc256p_dp"
    assert name(16384, 57344, 8192, torch.bfloat16, 128) == "tc256p_dp"
    assert name(2048, 8192, 28672, torch.bfloat16, 128) == "tc256p_sk"  # 512 tiles < 4 waves
    # installed at run time
    assert name(64, 4096, 4096, torch.bfloat16, 128) == "tc64_sk"
    w4.override_schedule(torch.bfloat16, 33, 64, 4096, 4096, 128, "tc128_sk")
    assert name(64, 4096, 4096, torch.bfloat16, 128) == "tc128_sk"
    assert name(64, 4096, 4096, torch.float16, 128) == "tc64_sk"     # other dtype: untouched
    assert name(64, 4096, 4096, torch.bfloat16, -1) == "tc64_sk"     # other group size
    w4.override_schedule(torch.bfloat16, 33, 64, 4096, 4096, 128, "tc64_sk")
    assert name(48, 4096, 4096, torch.bfloat16, 128) == "tc64_sk"
    w4.override_schedule(torch.bfloat16, 33, 64, 4096, 4096, 128, "ds8_sk")  # cannot run M=64
    assert name(64, 4096, 4096, torch.bfloat16, 128) == "tc64_sk"
    w4.override_schedule(torch.bfloat16, 33, 64, 4096, 4096, 128, None)       # removed
    assert name(64, 4096, 4096, torch.bfloat16, 128) == "tc64_sk"
    E = w4.ERR_INVALID_ARGUMENT
    assert lib.w4_override_schedule(7, 1, 2, 8, 64, -1, 1) == E      # a_type
    assert lib.w4_override_schedule(1, 5, 2, 8, 64, -1, 1) == E      # empty range
    assert lib.w4_override_schedule(1, 1, 2, 8, 72, -1, 1) == E      # K % 64
    assert lib.w4_override_schedule(1, 1, 2, 8, 256, 96, 1) == E     # group size
    assert lib.w4_override_schedule(1, 1, 2, 8, 64, -1, 99) == E     # schedule index



def test_dynamic_and_fp8_argument_checks(lib):
    """The dynamic-quantization call and fp8 activations reject bad arguments
    on the host; the dynamic workspace covers the GEMM's plus the codes."""
    E, U = w4.ERR_INVALID_ARGUMENT, w4.ERR_UNSUPPORTED
    f = lib.w4_gemm_dynamic
    base = dict(a=256, at=0, M=4, K=256, b=256, wt=2, N=128, s=None, st=2, gs=-1, ch=256, act=2,
                bias=None, out=256, tok=None, ws=256, wsb=1 << 24, stream=None)

    def call(**kw):
        d = dict(base, **kw)
        return f(d["a"], d["at"], d["M"], d["K"], d["b"], d["wt"], d["N"], d["s"], d["st"],
                 d["gs"], d["ch"], d["act"], d["bias"], d["out"], d["tok"], d["ws"], d["wsb"],
                 d["stream"])
    assert call(at=2) == E                      # int8 input
    assert call(act=1) == E                     # act_type must be int8 or E4M3
    assert call(a=None) == E
    assert call(K=100) == E                     # K % 8
    assert call(K=320, act=4) == U              # fp8 wants K % 128
    assert call(ws=None) == w4.ERR_WORKSPACE
    assert call(wsb=16) == w4.ERR_WORKSPACE
    assert call(M=0, a=None) == w4.OK
    # the codes never overlap the header + split-K counters, even when the
    # GEMM part itself (the clustered schedule) needs only the header
    for M in (1, 7, 16):
        nd = lib.w4_gemm_dynamic_workspace_size(M, 1024, 4096, 2, -1)
        assert nd >= 256 + 64 * 1024 + M * 4096 + M * 4
    nd = lib.w4_gemm_dynamic_workspace_size(300, 1024, 4096, 2, -1)
    assert nd >= lib.w4_gemm_workspace_size(300, 1024, 4096, 2, -1) + 300 * 4096 + 300 * 4
    # fp8 activations through the plain GEMM call: per-channel, fp16 out, K % 128
    assert _gemm(lib, a_type=4, wtype=2, s=None, gs=-1, ot=0, tok=256, ch=256, K=192) == U
    assert _gemm(lib, a_type=4, wtype=2, s=256, st=2, gs=128, ot=0, tok=256, ch=256) == U
    assert _gemm(lib, a_type=4, wtype=2, s=None, gs=-1, ot=3) == U
    assert _gemm(lib, a_type=4, wtype=1, s=None, gs=-1, ot=0, tok=256, ch=256) == U
    names = w4.schedule_names()
    pick = lambda M, N, K: names[lib.w4_default_schedule(M, N, K, 4, -1)]
    assert pick(1, 8192, 21760) == "gv8_cl" and pick(16, 8192, 21760) == "gv16_cl"
    assert pick(1024, 8192, 21760).startswith("tc")
    q = lib.w4_quantize_per_token_fp8
    assert q(1, 2, 4, 64, 1, 1, None) == E      # int8 input
    assert q(1, 0, -1, 64, 1, 1, None) == E
    assert q(None, 0, 0, 64, None, None, None) == w4.OK
