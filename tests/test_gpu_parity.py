"""GPU parity: libw4 (through the C ABI) against the CPU oracle.

Float outputs: every element within 4e-3 * sum_k|a_k w_k| + 1 ulp of the
output type.  W4A8 int32 accumulators: bit-exact.  W4A8 fp16 outputs:
within 1 fp16 ulp of the fp64 reference.  Small cases compare every
element; full-size cases compare sampled elements that the oracle computes
one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import w4synth
from parity import assert_fp16_near, assert_fp16_within_ulp, assert_within

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ALL = ["simt", "tc16_sk", "tc32_sk", "tc64_sk", "tc128_sk", "tc128_dp", "tc256_sk", "tc256_dp",
       "tc128x2_sk", "tc128x2_dp", "tc128x2_kp", "tc256p_sk", "tc256p_dp", "tc128p_sk"]
DK = ["dk8_sk", "dk16_sk"]
DS = ["ds8_sk", "ds16_sk", "ds32_sk"]
GV = ["gv8_cl", "gv16_cl", "gv32_cl"]
ROWS = {"dk8_sk": 8, "dk16_sk": 16, "ds8_sk": 8, "ds16_sk": 16, "ds32_sk": 32, "gv8_cl": 8,
        "gv16_cl": 16, "gv32_cl": 32}


def sched(w4, name):
    return w4.schedule_names().index(name)


def fmt(dt):
    return "f16" if dt == torch.float16 else "bf16"


def run_w4a16(w4, d, schedule=-1):
    b = w4.prepack_B(d["w"].to(DEV), d["wtype"], d["layout"], d["K"], d["N"])
    z = None if d["z"] is None else d["z"].to(DEV)
    out = w4.gemm(d["a"].to(DEV), b, d["wtype"], d["N"], scales=d["s"].to(DEV), zeros=z,
                  group_size=d["group_size"], schedule=schedule)
    torch.cuda.synchronize()
    return out.cpu()


def oracle_w4a16(d):
    return oracle.w4a16(d["a"], d["w"], d["layout"], d["wtype"], d["s"], d["z"], d["group_size"],
                        d["K"], d["N"])


def samples(M, N, count=384, seed=0):
    """Random output elements plus the corners, and 16 elements of the last
    row tile x last column tile (ragged or not)."""
    rng = np.random.default_rng(seed)
    tail_r = M - 1 - rng.integers(0, min(M, 256), 16)
    tail_c = N - 1 - rng.integers(0, min(N, 128), 16)
    rows = np.concatenate([[0, M - 1, M // 2], tail_r, rng.integers(0, M, count)])
    cols = np.concatenate([[0, N - 1, min(127, N - 1)], tail_c, rng.integers(0, N, count)])
    return rows.astype(np.int64), cols.astype(np.int64)


# --------------------------------------------------------------- CTA pairs ---
@pytest.mark.parametrize("name", ["tc256p_sk", "tc256p_dp", "tc128p_sk"])
@pytest.mark.parametrize("M,N", [(256, 256), (100, 384), (300, 640)])
def test_pair_w4a8_int32_exact(gpu_lib, name, M, N):
    """Two CTAs of a cluster share each MMA: int32 accumulators bit-exact,
    with a pair tile whose second CTA has no weight columns (N = 384, 640:
    odd 128-column tile counts) or no activation rows (M = 100)."""
    w4 = gpu_lib
    e = w4synth.gen_w4a8(M, N, 1024, group_size=-1, seed=M + N)
    acc = run_w4a8(w4, e, torch.int32, sched(w4, name))
    ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], None, -1, e["K"], e["N"])
    assert np.array_equal(acc.numpy().astype(np.int64), ref)


# ----------------------------------------------------------------- prepack ---

@pytest.mark.parametrize("layout", [0, 1, 2])
def test_prepack_round_trip(gpu_lib, layout):
    w4 = gpu_lib
    K, N = 512, 200
    w = w4synth.random_words(w4synth.packed_shape(layout, K, N), torch.Generator().manual_seed(1))
    wd = w.to(DEV)
    packs = {}
    for wtype in (w4.UINT4B8, w4.UINT4, w4.INT4):
        b = w4.prepack_B(wd, wtype, layout, K, N)
        assert b.numel() == w4.prepacked_size(K, N)
        back = w4.unprepack_B(b, wtype, layout, K, N)
        assert torch.equal(back.cpu(), w)
        packs[wtype] = b.cpu()
    # uint4 and uint4b8 prepack identically; int4 flips the top bit of each nibble
    assert torch.equal(packs[w4.UINT4], packs[w4.UINT4B8])
    flipped = (packs[w4.UINT4B8].view(torch.int32) ^ int(np.int32(np.uint32(0x88888888))))
    n_pad_words = packs[w4.INT4].view(torch.int32)
    valid = torch.zeros(256 // 128, K // 32, 128, 4, dtype=torch.bool)
    valid[:, :, :, :] = True
    valid[1, :, 200 - 128:, :] = False  # padding rows stay zero
    assert torch.equal(n_pad_words.view(2, K // 32, 128, 4)[valid],
                       flipped.view(2, K // 32, 128, 4)[valid])
    assert int(n_pad_words.view(2, K // 32, 128, 4)[~valid].abs().sum()) == 0


def test_prepack_layouts_agree(gpu_lib):
    w4 = gpu_lib
    K, N = 256, 384
    rng = np.random.default_rng(2)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    bufs = [w4.prepack_B(torch.from_numpy(oracle.pack(q, L)).to(DEV), w4.UINT4, L, K, N).cpu()
            for L in (0, 1, 2)]
    assert torch.equal(bufs[0], bufs[1]) and torch.equal(bufs[0], bufs[2])


# ------------------------------------------------------------------- W4A16 ---

@pytest.mark.parametrize("name", ALL + ["dk16_sk"])
def test_tiny_w4a16_every_schedule(gpu_lib, name):
    w4 = gpu_lib
    d = w4synth.tiny_w4a16(seed=0)
    got = run_w4a16(w4, d, sched(w4, name))
    ref, absref = oracle_w4a16(d)
    assert_within(got.double().numpy(), ref, absref, "f16", f"tiny {name}")


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("zeros", [False, True])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_w4a16_several_tiles(gpu_lib, name, zeros, dt):
    """Every schedule, both activation types, with and without pre-scaled
    zero-points (fp16 with zero-points on every tensor-core schedule)."""
    w4 = gpu_lib
    d = w4synth.gen_w4a16(40, 384, 1024, act_dtype=dt,
                          wtype=w4.UINT4 if zeros else w4.UINT4B8, layout=w4.KN_SEQ,
                          group_size=128, zeros=zeros, seed=3)
    got = run_w4a16(w4, d, sched(w4, name))
    ref, absref = oracle_w4a16(d)
    assert_within(got.double().numpy(), ref, absref, fmt(dt), f"{fmt(dt)} {name} zeros={zeros}")


@pytest.mark.parametrize("M", [256, 1000])
@pytest.mark.parametrize("name", ["tc128_sk", "tc256_sk", "tc256_dp", "tc128x2_kp", "tc256p_sk",
                                  "tc256p_dp", "tc128p_sk"])
def test_w4a16_f16_zero_points_large_m(gpu_lib, name, M):
    """fp16 activations with uint4 + pre-scaled zero-points on the wide
    tensor-core tiles (the large-M path), ragged N, several K groups."""
    w4 = gpu_lib
    d = w4synth.gen_w4a16(M, 1160, 2048, act_dtype=torch.float16, wtype=w4.UINT4,
                          layout=w4.NK_EXLLAMA, group_size=128, zeros=True, seed=M + 7)
    got = run_w4a16(w4, d, sched(w4, name))
    rows, cols = samples(M, d["N"], count=384, seed=M)
    sub = got[torch.from_numpy(rows), torch.from_numpy(cols)].double().numpy()
    ref, absref = oracle.w4a16_elems(d["a"], d["w"], d["layout"], d["wtype"], d["s"], d["z"], 128,
                                     d["K"], d["N"], rows, cols)
    assert_within(sub, ref, absref, "f16", f"f16 zero-points {name} M={M}")


@pytest.mark.parametrize("M,N,K,gs,dt", [
    (1, 8, 576, -1, torch.float16),       # smallest tc tile row, K not a multiple of 128
    (3, 200, 640, 128, torch.bfloat16),   # ragged N inside a 128 tile
    (17, 136, 512, 64, torch.bfloat16),   # group 64, ragged M and N
    (100, 13, 256, 128, torch.float16),   # N % 8 != 0 -> CUDA-core schedule
    (5, 13, 256, 128, torch.bfloat16),    # N % 8 != 0, skinny M -> mma.sync schedule
    (12, 200, 576, -1, torch.float16),    # skinny M, ragged N, K not a multiple of 128
    (300, 256, 192, -1, torch.bfloat16),  # M spanning two 256-row tiles
])
def test_w4a16_ragged(gpu_lib, M, N, K, gs, dt):
    w4 = gpu_lib
    d = w4synth.gen_w4a16(M, N, K, act_dtype=dt, wtype=w4.UINT4, layout=w4.NK_EXLLAMA,
                          group_size=gs, zeros=True, seed=M + N)
    got = run_w4a16(w4, d)
    ref, absref = oracle_w4a16(d)
    assert_within(got.double().numpy(), ref, absref, fmt(dt), f"ragged {M}x{N}x{K}")


@pytest.mark.parametrize("name", DK + DS + GV)
@pytest.mark.parametrize("M", [1, 3, 8, 13, 16, 27, 32])
@pytest.mark.parametrize("dt,zeros,gs", [(torch.bfloat16, True, 128), (torch.float16, False, 128),
                                          (torch.bfloat16, False, -1), (torch.float16, True, 256)])
def test_dk_w4a16(gpu_lib, name, M, dt, zeros, gs):
    w4 = gpu_lib
    if M > ROWS[name]:
        pytest.skip("more rows than the schedule's tile")
    d = w4synth.gen_w4a16(M, 392, 1280, act_dtype=dt, wtype=w4.UINT4 if zeros else w4.UINT4B8,
                          layout=w4.NK_EXLLAMA, group_size=gs, zeros=zeros, seed=M)
    got = run_w4a16(w4, d, sched(w4, name))
    ref, absref = oracle_w4a16(d)
    assert_within(got.double().numpy(), ref, absref, fmt(dt), f"{name} M={M}")


@pytest.mark.parametrize("name", DS + GV)
@pytest.mark.parametrize("M,N,K,gs,dt", [
    (5, 200, 576, -1, torch.bfloat16),    # K not a multiple of 128: half-full last block
    (8, 136, 640, 128, torch.float16),    # ragged N, odd number of K blocks
    (1, 8, 64, -1, torch.bfloat16),       # one 64-wide K block, one 8-column tile
    (3, 4096, 4096, 128, torch.float16),  # several tiles per CTA's stream-K range
])
def test_ds_ragged(gpu_lib, name, M, N, K, gs, dt):
    w4 = gpu_lib
    d = w4synth.gen_w4a16(M, N, K, act_dtype=dt, wtype=w4.UINT4, layout=w4.NK_EXLLAMA,
                          group_size=gs, zeros=True, seed=M + K)
    got = run_w4a16(w4, d, sched(w4, name))
    ref, absref = oracle_w4a16(d)
    assert_within(got.double().numpy(), ref, absref, fmt(dt), f"{name} {M}x{N}x{K}")


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("name", ["default", "ds8_sk", "ds16_sk", "ds32_sk", "dk16_sk", "tc16_sk",
                                  "tc64_sk", "simt", "gv8_cl", "gv16_cl", "gv32_cl", "tc256p_sk"])
def test_w4a16_power_of_two_scales_exact(gpu_lib, dt, name):
    # exact products and sums: the GPU output must equal the exact result
    # rounded once (to nearest even) to the output type.  The activations are
    # small integers, so the fp16 staging of the streamed schedule (odd pairs
    # divided by 16) is exact too.
    w4 = gpu_lib
    M, N, K = 8, 256, 512
    d = w4synth.gen_w4a16(M, N, K, act_dtype=dt, wtype=w4.UINT4B8, group_size=128, seed=5)
    d["s"] = torch.full_like(d["s"], 0.0625)
    d["a"] = torch.randint(-4, 5, (M, K), generator=torch.Generator().manual_seed(5)).to(dt)
    got = run_w4a16(w4, d, -1 if name == "default" else sched(w4, name))
    ref, _ = oracle_w4a16(d)
    assert torch.equal(got, torch.from_numpy(ref).to(dt))


def test_w4a16_zero_point_eight_equals_symmetric(gpu_lib):
    w4 = gpu_lib
    d = w4synth.gen_w4a16(16, 256, 512, act_dtype=torch.bfloat16, wtype=w4.UINT4B8,
                          group_size=128, seed=6)
    sym = run_w4a16(w4, d)
    d2 = dict(d, wtype=w4.UINT4, z=(d["s"].float() * 8).to(torch.bfloat16))
    asym = run_w4a16(w4, d2)
    assert torch.equal(sym, asym)


@pytest.mark.parametrize("N,K", w4synth.DECODE_SHAPES)
@pytest.mark.parametrize("M", w4synth.DECODE_M)
def test_decode_sweep_llama3_8b(gpu_lib, N, K, M):
    w4 = gpu_lib
    d = w4synth.gen_w4a16(M, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4,
                          layout=w4.NK_EXLLAMA, group_size=128, zeros=True, seed=0)
    got = run_w4a16(w4, d).double().numpy()
    rows, cols = samples(M, N, seed=M)
    ref, absref = oracle.w4a16_elems(d["a"], d["w"], d["layout"], d["wtype"], d["s"], d["z"], 128,
                                     K, N, rows, cols)
    assert_within(got[rows, cols], ref, absref, "bf16", f"decode {M}x{N}x{K}")


@pytest.mark.parametrize("N,K", w4synth.PREFILL_SHAPES)
@pytest.mark.parametrize("M", w4synth.PREFILL_M)
def test_prefill_llama3_70b(gpu_lib, N, K, M):
    """Every (N, K) x M point of the Llama-3-70B MLP prefill workload, on
    sampled elements that include the last row and column tiles."""
    w4 = gpu_lib
    d = w4synth.gen_w4a16(M, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4B8,
                          layout=w4.NK_EXLLAMA, group_size=128, zeros=False, seed=0)
    got = run_w4a16(w4, d)
    rows, cols = samples(M, N, count=192, seed=N)
    sub = got[torch.from_numpy(rows), torch.from_numpy(cols)].double().numpy()
    ref, absref = oracle.w4a16_elems(d["a"], d["w"], d["layout"], d["wtype"], d["s"], None, 128,
                                     K, N, rows, cols)
    assert_within(sub, ref, absref, "bf16", f"prefill {M}x{N}x{K}")


@pytest.mark.parametrize("name", ["tc128x2_sk", "tc128x2_dp", "tc128x2_kp"])
def test_prefill_two_weight_tiles(gpu_lib, name):
    """CTAs covering two 128-column weight tiles at a full prefill shape
    (ragged last weight tile: N = 8192 + 128 is an odd number of tiles)."""
    w4 = gpu_lib
    M, N, K = 1000, 8320, 8192
    d = w4synth.gen_w4a16(M, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4,
                          layout=w4.NK_EXLLAMA, group_size=128, zeros=True, seed=5)
    got = run_w4a16(w4, d, sched(w4, name))
    rows, cols = samples(M, N, count=192, seed=N)
    cols[:64] = N - 1 - np.arange(64)  # the lone last tile
    sub = got[torch.from_numpy(rows), torch.from_numpy(cols)].double().numpy()
    ref, absref = oracle.w4a16_elems(d["a"], d["w"], d["layout"], d["wtype"], d["s"], d["z"], 128,
                                     K, N, rows, cols)
    assert_within(sub, ref, absref, "bf16", f"two tiles {name}")


# -------------------------------------------------------------------- W4A8 ---

def run_w4a8(w4, e, out_dtype, schedule=-1):
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], e["K"], e["N"])
    sg = None if e["sg"] is None else e["sg"].to(DEV)
    kw = {}
    if out_dtype == torch.float16:
        kw = dict(token_scales=e["s_tok"].to(DEV), channel_scales=e["s_ch"].to(DEV))
    out = w4.gemm(e["a"].to(DEV), b, e["wtype"], e["N"], scales=sg, group_size=e["group_size"],
                  out_dtype=out_dtype, schedule=schedule, **kw)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("name", ["simt", "tc16_sk", "tc32_sk", "tc64_sk", "tc128_sk", "tc128_dp",
                                  "tc128x2_kp", "tc256_kp", "tc256_sk", "tc256_dp", "dk8_sk",
                                  "dk16_sk", "ds8_sk", "ds16_sk", "ds32_sk", "gv8_cl", "gv16_cl",
                                  "gv32_cl", "tc256p_sk", "tc256p_dp", "tc128p_sk"])
@pytest.mark.parametrize("gs", [-1, 128])
def test_w4a8_int32_bit_exact(gpu_lib, name, gs):
    w4 = gpu_lib
    M = {"dk8_sk": 8, "dk16_sk": 13, "ds8_sk": 7, "ds16_sk": 16, "ds32_sk": 29, "gv8_cl": 5,
         "gv16_cl": 11, "gv32_cl": 32}.get(name, 40)
    e = w4synth.gen_w4a8(M, 384, 2048, group_size=gs, seed=7)
    acc = run_w4a8(w4, e, torch.int32, sched(w4, name))
    ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], e["sg"], gs, e["K"], e["N"])
    assert np.array_equal(acc.numpy().astype(np.int64), ref)


@pytest.mark.parametrize("gs", [-1, 128])
def test_w4a8_extreme_magnitudes_exact(gpu_lib, gs):
    """Largest |partial sums| the QQQ shapes allow: int8 -128/127 against
    int4 -8 (x group scale 16), K = 21760."""
    w4 = gpu_lib
    M, N, K = 4, 256, 21760
    q = np.full((K, N), 8, dtype=np.uint8)           # int4 -8 everywhere
    q[:, 1::2] = 7                                   # and +7 in odd columns
    w = torch.from_numpy(oracle.pack(q, oracle.NK_EXLLAMA))
    a = torch.full((M, K), -128, dtype=torch.int8)
    a[1] = 127
    a[2, ::2] = 127
    a[3] = torch.randint(-128, 128, (K,), generator=torch.Generator().manual_seed(0)).to(torch.int8)
    sg = torch.full((K // 128, N), 16, dtype=torch.int8) if gs == 128 else None
    e = dict(a=a, w=w, sg=sg, layout=oracle.NK_EXLLAMA, wtype=w4.INT4, K=K, N=N, group_size=gs)
    names = ("tc16_sk", "tc128_dp", "simt", "dk8_sk", "ds8_sk", "tc256_sk", "tc256_dp", "gv8_cl",
             "gv32_cl") + (
        ("tc128x2_kp", "tc256_kp") if gs == -1 else ())
    for name in names:
        acc = run_w4a8(w4, e, torch.int32, sched(w4, name))
        ref = oracle.w4a8(a, w, oracle.NK_EXLLAMA, w4.INT4, sg, gs, K, N)
        assert np.array_equal(acc.numpy().astype(np.int64), ref), name


@pytest.mark.parametrize("name", ["tc256p_sk", "tc256p_dp", "tc128p_sk"])
@pytest.mark.parametrize("gs", [-1, 128])
def test_w4a8_extreme_magnitudes_pairs(gpu_lib, name, gs):
    """The same largest partial sums on CTA pairs, over enough weight tiles
    that a unit spans several exact chunks (the int32 running sum of the
    256-row tiles in global scratch, of the 128-row tiles in tensor memory)
    and stream-K tiles are shared by several pairs."""
    w4 = gpu_lib
    M, N, K = 5, 2048, 21760
    q = np.full((K, N), 8, dtype=np.uint8)
    q[:, 1::2] = 7
    w = torch.from_numpy(oracle.pack(q, oracle.NK_EXLLAMA))
    a = torch.full((M, K), -128, dtype=torch.int8)
    a[1] = 127
    a[2, ::2] = 127
    a[3] = torch.randint(-128, 128, (K,), generator=torch.Generator().manual_seed(1)).to(torch.int8)
    a[4, 1::2] = 127
    sg = torch.full((K // 128, N), 16, dtype=torch.int8) if gs == 128 else None
    e = dict(a=a, w=w, sg=sg, layout=oracle.NK_EXLLAMA, wtype=w4.INT4, K=K, N=N, group_size=gs)
    acc = run_w4a8(w4, e, torch.int32, sched(w4, name))
    ref = oracle.w4a8(a, w, oracle.NK_EXLLAMA, w4.INT4, sg, gs, K, N)
    assert np.array_equal(acc.numpy().astype(np.int64), ref)


@pytest.mark.parametrize("M", w4synth.QQQ_CH_M)
def test_w4a8_qqq_per_channel(gpu_lib, M):
    w4 = gpu_lib
    e = w4synth.gen_w4a8(M, w4synth.QQQ_N, w4synth.QQQ_K, group_size=-1, seed=0)
    out = run_w4a8(w4, e, torch.float16).double().numpy()
    acc = run_w4a8(w4, e, torch.int32).numpy().astype(np.int64)
    rows, cols = samples(M, e["N"], count=256, seed=M)
    ref_acc = oracle.w4a8_elems(e["a"], e["w"], e["layout"], e["wtype"], None, -1, e["K"],
                                e["N"], rows, cols)
    assert np.array_equal(acc[rows, cols], ref_acc)
    ref = oracle.w4a8_scale(ref_acc, rows, cols, e["s_tok"], e["s_ch"])
    assert_fp16_within_ulp(out[rows, cols], ref, f"qqq per-channel M={M}")


@pytest.mark.parametrize("name", ["tc128x2_kp", "tc256_kp", "tc256p_sk", "tc128p_sk"])
@pytest.mark.parametrize("M", [128, 1024])
def test_w4a8_qqq_per_channel_split_k(gpu_lib, M, name):
    """Two weight tiles per CTA, K split so that no unit passes one exact
    fp32 chunk: bit-exact int32 at the full QQQ shape."""
    w4 = gpu_lib
    e = w4synth.gen_w4a8(M, w4synth.QQQ_N, w4synth.QQQ_K, group_size=-1, seed=1)
    acc = run_w4a8(w4, e, torch.int32, sched(w4, name)).numpy().astype(np.int64)
    rows, cols = samples(M, e["N"], count=256, seed=M + 1)
    ref_acc = oracle.w4a8_elems(e["a"], e["w"], e["layout"], e["wtype"], None, -1, e["K"],
                                e["N"], rows, cols)
    assert np.array_equal(acc[rows, cols], ref_acc)


@pytest.mark.parametrize("M", w4synth.QQQ_G128_M)
def test_w4a8_qqq_g128(gpu_lib, M):
    w4 = gpu_lib
    e = w4synth.gen_w4a8(M, w4synth.QQQ_N, w4synth.QQQ_K, group_size=128, seed=0)
    out = run_w4a8(w4, e, torch.float16).double().numpy()
    acc = run_w4a8(w4, e, torch.int32).numpy().astype(np.int64)
    rows, cols = samples(M, e["N"], count=256, seed=M)
    ref_acc = oracle.w4a8_elems(e["a"], e["w"], e["layout"], e["wtype"], e["sg"], 128, e["K"],
                                e["N"], rows, cols)
    assert np.array_equal(acc[rows, cols], ref_acc)
    ref = oracle.w4a8_scale(ref_acc, rows, cols, e["s_tok"], e["s_ch"])
    assert_fp16_within_ulp(out[rows, cols], ref, f"qqq g128 M={M}")


# ------------------------------------------------------------ edge cases ---

def test_empty_and_k_zero(gpu_lib):
    w4 = gpu_lib
    b = torch.zeros(1, dtype=torch.uint8, device=DEV)
    s = torch.ones(1, 8, dtype=torch.float16, device=DEV)
    out = w4.gemm(torch.empty(0, 64, dtype=torch.float16, device=DEV), b, w4.UINT4B8, 8,
                  scales=s, group_size=-1)
    assert out.shape == (0, 8)
    out = torch.full((3, 8), 7.0, dtype=torch.float16, device=DEV)
    w4.gemm(torch.empty(3, 0, dtype=torch.float16, device=DEV), b, w4.UINT4B8, 8, scales=s,
            group_size=-1, out=out)
    torch.cuda.synchronize()
    assert int(out.abs().sum()) == 0


def test_deterministic_stream_k(gpu_lib):
    w4 = gpu_lib
    d = w4synth.gen_w4a16(16, 4096, 4096, act_dtype=torch.bfloat16, wtype=w4.UINT4,
                          group_size=128, zeros=True, seed=9)
    a = run_w4a16(w4, d)
    b = run_w4a16(w4, d)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["tc16_sk", "tc32_sk", "tc256p_sk", "tc128p_sk"])
def test_stream_k_many_contributors(gpu_lib, name):
    """One weight tile over a long K: stream-K spreads its stages over more
    than 32 CTAs, so the tile's last arriving warp adds over 32 other partial
    sums (the slot of each computed in turn rather than held by a lane)."""
    w4 = gpu_lib
    N, K = 128, 32768
    e = w4synth.gen_w4a8(8, N, K, group_size=-1, seed=31)
    got = run_w4a8(w4, e, torch.int32, schedule=sched(w4, name))
    ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], e["sg"], e["group_size"], K, N)
    assert np.array_equal(got.numpy().astype(np.int64), ref)
    d = w4synth.gen_w4a16(8, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4, group_size=128,
                          zeros=True, seed=32)
    o1 = run_w4a16(w4, d, schedule=sched(w4, name))
    o2 = run_w4a16(w4, d, schedule=sched(w4, name))
    assert torch.equal(o1, o2)  # partial sums are added in K order
    ref, absref = oracle_w4a16(d)
    assert_within(o1.double().numpy(), ref, absref, "bf16", f"{name} many contributors")


@pytest.mark.parametrize("name", GV)
@pytest.mark.parametrize("N,K", [(128, 32768), (200, 21760), (1032, 4160), (8, 64)])
def test_gv_cluster_reduction(gpu_lib, name, N, K):
    """The clustered schedule splits each 128-column tile's K blocks over up
    to 16 CTAs and adds their partial sums through distributed shared memory
    in K order: int32 bit-exact (W4A8 per-channel and g128), bf16 within the
    bound and bitwise repeatable; ragged N, K not a multiple of 128, a single
    64-wide K block."""
    w4 = gpu_lib
    M = ROWS[name] - 3
    for gs in ([-1, 128] if K % 128 == 0 and N % 16 == 0 else [-1]):
        e = w4synth.gen_w4a8(M, N, K, group_size=gs, seed=N + K)
        got = run_w4a8(w4, e, torch.int32, schedule=sched(w4, name))
        ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], e["sg"], gs, K, N)
        assert np.array_equal(got.numpy().astype(np.int64), ref), f"{name} gs={gs}"
    d = w4synth.gen_w4a16(M, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4,
                          group_size=128 if K % 128 == 0 else -1, zeros=True, seed=N + K + 1)
    o1 = run_w4a16(w4, d, schedule=sched(w4, name))
    o2 = run_w4a16(w4, d, schedule=sched(w4, name))
    assert torch.equal(o1, o2)
    ref, absref = oracle_w4a16(d)
    assert_within(o1.double().numpy(), ref, absref, "bf16", f"{name} {N}x{K}")


def test_misaligned_workspace_rejected(gpu_lib):
    w4 = gpu_lib
    d = w4synth.tiny_w4a16(seed=2)
    b = w4.prepack_B(d["w"].to(DEV), d["wtype"], d["layout"], d["K"], d["N"])
    nbytes = w4.workspace_size(d["M"], d["N"], d["K"], d["a"].dtype, d["group_size"])
    ws = torch.zeros(nbytes + 16, dtype=torch.uint8, device=DEV)[8:]
    with pytest.raises(w4.W4Error) as ei:
        w4.gemm(d["a"].to(DEV), b, d["wtype"], d["N"], scales=d["s"].to(DEV),
                group_size=d["group_size"], ws=ws)
    assert ei.value.status == w4.ERR_WORKSPACE


def test_check_status_clean(gpu_lib):
    w4 = gpu_lib
    d = w4synth.tiny_w4a16(seed=1)
    run_w4a16(w4, d)
    ws = w4.workspace(DEV, 256)
    assert w4.check_status(ws) == w4.OK


def test_invalid_on_device_pointers(gpu_lib):
    w4 = gpu_lib
    d = w4synth.tiny_w4a16(seed=0)
    b = w4.prepack_B(d["w"].to(DEV), d["wtype"], d["layout"], d["K"], d["N"])
    with pytest.raises(w4.W4Error) as ei:
        w4.gemm(d["a"].to(DEV), b, d["wtype"], d["N"], scales=d["s"].to(DEV).bfloat16(),
                group_size=128)
    assert ei.value.status == w4.ERR_INVALID_ARGUMENT


def test_back_to_back_calls(gpu_lib):
    """Calls of several schedules enqueued back to back on one stream, sharing
    the cached workspace, with no synchronization between them: the launches
    that overlap a previous call's tail (activation staging, programmatic
    dependents) must leave every result equal to its oracle."""
    w4 = gpu_lib
    N, K = 1024, 2048
    e1 = w4synth.gen_w4a8(1, N, K, group_size=-1, seed=21)
    e2 = w4synth.gen_w4a8(8, N, K, group_size=-1, seed=22)
    e3 = w4synth.gen_w4a8(300, N, K, group_size=-1, seed=23)
    e4 = w4synth.gen_w4a8(24, N, K, group_size=128, seed=24)
    d5 = w4synth.gen_w4a16(5, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4, group_size=128,
                           zeros=True, seed=25)
    jobs = []
    for e in (e1, e2, e3, e4, e1, e3):
        b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], e["K"], e["N"])
        sg = None if e["sg"] is None else e["sg"].to(DEV)
        jobs.append((e, b, e["a"].to(DEV), sg))
    b5 = w4.prepack_B(d5["w"].to(DEV), d5["wtype"], d5["layout"], K, N)
    a5, s5, z5 = d5["a"].to(DEV), d5["s"].to(DEV), d5["z"].to(DEV)
    torch.cuda.synchronize()
    outs = []
    for i, (e, b, a, sg) in enumerate(jobs):
        outs.append(w4.gemm(a, b, e["wtype"], N, scales=sg, group_size=e["group_size"],
                            out_dtype=torch.int32))
        if i == 2:
            out5 = w4.gemm(a5, b5, d5["wtype"], N, scales=s5, zeros=z5, group_size=128)
    torch.cuda.synchronize()
    for (e, _, _, _), got in zip(jobs, outs):
        ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], e["sg"], e["group_size"], K, N)
        assert np.array_equal(got.cpu().numpy().astype(np.int64), ref)
    ref, absref = oracle_w4a16(d5)
    assert_within(out5.cpu().double().numpy(), ref, absref, "bf16", "back to back W4A16")


# ------------------------------------------- per-token int8 quantization ---
# Codes and scales are decided in fp32 on both sides: bit-exact.

def _quant_gpu(w4, a_dev):
    q, s = w4.quantize_per_token(a_dev)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _assert_quant_equal(q, s, rq, rs, what):
    assert np.array_equal(s.view(np.int32), rs.view(np.int32)), f"{what}: scales differ"
    bad = np.argwhere(q != rq)
    assert bad.size == 0, f"{what}: {len(bad)} codes differ, first {bad[:3].tolist()}"


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,K", [(1, 21760), (16, 21760), (37, 4096), (5, 72), (3, 13), (2, 8),
                                 (0, 64), (4, 0), (1024, 21760), (3, 65536), (2, 65600),
                                 (7, 2048), (2000, 4096), (400, 8)])
def test_quantize_per_token_bit_exact(gpu_lib, M, K, dt):
    w4 = gpu_lib
    a = w4synth.gen_act16(M, K, dt, seed=M + K)
    q, s = _quant_gpu(w4, a.to(DEV))
    rq, rs = oracle.quant_per_token(a)
    _assert_quant_equal(q, s, rq, rs, f"M={M} K={K} {fmt(dt)}")


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("aligned", [True, False])
def test_quantize_special_rows(gpu_lib, dt, aligned):
    """Zero rows, one outlier, equal values, exact ties and near-ties,
    the largest and the smallest magnitudes of the type, on the vectorised
    path and (a view one element off 16-byte alignment) the element-wise
    one."""
    w4 = gpu_lib
    K = 264
    a = w4synth.gen_act16(12, K, dt, seed=21).float()
    a[0] = 0.0
    a[1] = 0.0
    a[1, 100] = -3.0
    a[2] = 1.5
    a[3, :3] = torch.tensor([0.80615234375, 0.041259765625, 0.092041015625])
    a[4, :2] = torch.tensor([3110.0, 1555.0])
    a[5, :2] = torch.tensor([12.0078125, 6.00390625])
    a[6, :8] = torch.tensor([-254.0, 127.0, 63.5, 0.5, 0.0, 65.0, -65.0, 5.0])
    big = 65504.0 if dt == torch.float16 else 3.0e38
    a[7] *= big / a[7].abs().max()
    small = 6.0e-5 if dt == torch.float16 else 1.0e-38
    a[8] *= small / a[8].abs().max()
    a[9, ::2] = -a[9, ::2].abs()
    a[10] = torch.arange(K, dtype=torch.float32) - K / 2
    a = a.to(dt)
    if aligned:
        a_dev = a.to(DEV)
    else:
        buf = torch.zeros(a.numel() + 1, dtype=dt, device=DEV)
        buf[1:] = a.reshape(-1).to(DEV)
        a_dev = buf[1:].view(a.shape)
        assert a_dev.data_ptr() % 16 != 0
    q, s = _quant_gpu(w4, a_dev)
    rq, rs = oracle.quant_per_token(a)
    _assert_quant_equal(q, s, rq, rs, f"special rows {fmt(dt)} aligned={aligned}")
    assert s[0] == 0 and not q[0].any()


@pytest.mark.parametrize("M", [5, 300])
def test_quantize_feeds_w4a8(gpu_lib, M):
    """fp16 activations -> GPU per-token codes -> GPU W4A8 GEMM, against the
    oracle's codes through the oracle's W4A8: int32 bit-exact, fp16 within
    one ulp."""
    w4 = gpu_lib
    N, K = 384, 2048
    e = w4synth.gen_w4a8(M, N, K, group_size=-1, seed=11)
    a16 = w4synth.gen_act16(M, K, torch.float16, seed=12)
    q, s = w4.quantize_per_token(a16.to(DEV))
    rq, rs = oracle.quant_per_token(a16)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], K, N)
    acc = w4.gemm(q, b, e["wtype"], N, group_size=-1, out_dtype=torch.int32)
    out = w4.gemm(q, b, e["wtype"], N, group_size=-1, token_scales=s,
                  channel_scales=e["s_ch"].to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), rq)
    ref = oracle.w4a8(rq, e["w"], e["layout"], e["wtype"], None, -1, K, N)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    refo = oracle.w4a8_scale(ref.reshape(-1), rows.reshape(-1), cols.reshape(-1),
                             rs.astype(np.float64), e["s_ch"])
    assert_fp16_within_ulp(out.cpu().double().numpy().reshape(-1), refo, f"quantized W4A8 M={M}")



# ------------------------------------------------------------------- bias ---
# out = round(sum + bias[n]) (W4A16) / fp16_rn(acc * s_tok * s_ch + bias[n]) (W4A8)

BIAS_SCHEDULES = ["simt", "tc16_sk", "tc64_sk", "tc128_sk", "tc256_sk", "tc256_dp", "tc128x2_kp",
                  "dk8_sk", "dk16_sk", "ds8_sk", "ds16_sk", "ds32_sk", "gv8_cl", "gv16_cl",
                  "gv32_cl", "tc256p_sk", "tc256p_dp", "tc128p_sk"]


@pytest.mark.parametrize("name", BIAS_SCHEDULES)
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_w4a16_bias_every_engine(gpu_lib, name, dt):
    w4 = gpu_lib
    M = min(ROWS.get(name, 40), 40) - 1
    N, K = 392 if not name.startswith("tc") else 384, 1280
    d = w4synth.gen_w4a16(M, N, K, act_dtype=dt, wtype=w4.UINT4, layout=w4.NK_EXLLAMA,
                          group_size=128, zeros=True, seed=M + 77)
    bias = (torch.randn(N, generator=torch.Generator().manual_seed(5)) * 0.5).to(dt)
    b = w4.prepack_B(d["w"].to(DEV), d["wtype"], d["layout"], K, N)
    got = w4.gemm(d["a"].to(DEV), b, d["wtype"], N, scales=d["s"].to(DEV), zeros=d["z"].to(DEV),
                  group_size=128, schedule=sched(w4, name), bias=bias.to(DEV))
    torch.cuda.synchronize()
    ref, absref = oracle_w4a16(d)
    assert_within(got.cpu().double().numpy(), oracle.add_bias(ref, None, bias), absref, fmt(dt),
                  f"bias {name}")


@pytest.mark.parametrize("name", BIAS_SCHEDULES)
@pytest.mark.parametrize("gs", [128, -1])
def test_w4a8_bias_every_engine(gpu_lib, name, gs):
    """Bias on the W4A8 fp16 epilogue, with group scales and per-channel (on
    CTA pairs these are different kernel instances)."""
    w4 = gpu_lib
    M = min(ROWS.get(name, 40), 40) - 2
    N, K = 384, 2048
    e = w4synth.gen_w4a8(M, N, K, group_size=gs, seed=M + 88)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], K, N)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    rows, cols = rows.reshape(-1), cols.reshape(-1)
    acc = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], e["sg"], gs, K, N).reshape(-1)
    prod = oracle.w4a8_scale(acc, rows, cols, e["s_tok"], e["s_ch"])
    # a bias near minus the product in some columns (cancellation), random elsewhere
    bias = torch.from_numpy(-prod.reshape(M, N)[0]).to(torch.float16)
    bias[1::2] = (torch.randn(N // 2, generator=torch.Generator().manual_seed(6))).half()
    sg = e["sg"].to(DEV) if gs > 0 else None
    got = w4.gemm(e["a"].to(DEV), b, e["wtype"], N, scales=sg, group_size=gs,
                  token_scales=e["s_tok"].to(DEV), channel_scales=e["s_ch"].to(DEV),
                  schedule=sched(w4, name), bias=bias.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.add_bias(prod, cols, bias)
    assert_fp16_near(got.cpu().double().numpy().reshape(-1), ref,
                     np.abs(prod) + np.abs(bias.double().numpy()[cols]), f"bias {name}")


def test_bias_k_zero_and_rejections(gpu_lib):
    w4 = gpu_lib
    N = 136
    bias = torch.randn(N, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).to(DEV)
    b = torch.zeros(1, dtype=torch.uint8, device=DEV)
    s = torch.ones(1, N, dtype=torch.bfloat16, device=DEV)
    out = w4.gemm(torch.empty(3, 0, dtype=torch.bfloat16, device=DEV), b, w4.UINT4B8, N,
                  scales=s, group_size=-1, bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(out, bias.expand(3, N))  # a product over no K is zero
    e = w4synth.gen_w4a8(4, N, 256, group_size=-1, seed=8)
    bp = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], 256, N)
    with pytest.raises(w4.W4Error) as ei:  # the raw int32 output takes no bias
        w4.gemm(e["a"].to(DEV), bp, e["wtype"], N, group_size=-1, out_dtype=torch.int32,
                bias=torch.zeros(N, dtype=torch.int32, device=DEV))
    assert ei.value.status == w4.ERR_INVALID_ARGUMENT


def test_autotune_installs_the_fastest_schedule(gpu_lib):
    """autotune() times every schedule that can run the problem on the GPU,
    installs the fastest as the default for that shape, and the default
    call then runs it, with results still equal to the oracle."""
    w4 = gpu_lib
    M, N, K = 24, 1024, 2048
    e = w4synth.gen_w4a8(M, N, K, group_size=-1, seed=61)
    a = e["a"].to(DEV)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], K, N)
    times = w4.autotune(a, b, e["wtype"], N, group_size=-1, out_dtype=torch.int32, reps=5)
    names = w4.schedule_names()
    assert len(times) >= 5 and all(t > 0 for t in times.values())
    best = min(times, key=times.get)
    try:
        assert names[w4.default_schedule(M, N, K, torch.int8, -1)] == best
        acc = w4.gemm(a, b, e["wtype"], N, group_size=-1, out_dtype=torch.int32)
        torch.cuda.synchronize()
        ref = oracle.w4a8(e["a"], e["w"], e["layout"], e["wtype"], None, -1, K, N)
        assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref)
    finally:
        w4.override_schedule(torch.int8, M, M, N, K, -1, None)



# ------------------------------------------------- W4A8, fp8 activations ---
# out = fp16(acc * s_tok * s_ch), acc the fp32 sum of exact E4M3 x int4
# products: within 4e-3 * sum|terms| * s_tok * s_ch + 1 fp16 ulp.

F8_SCHEDULES = ["simt", "tc16_sk", "tc32_sk", "tc64_sk", "tc128_sk", "tc128_dp", "tc256_sk",
                "tc256_dp", "tc128x2_sk", "tc128x2_kp", "tc256_kp", "gv8_cl", "gv16_cl",
                "gv32_cl", "tc256p_sk", "tc256p_dp", "tc128p_sk"]


def run_fp8(w4, e, schedule=-1, bias=None):
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], e["K"], e["N"])
    a = e["a"].to(DEV).view(torch.float8_e4m3fn)
    out = w4.gemm(a, b, e["wtype"], e["N"], group_size=-1, token_scales=e["s_tok"].to(DEV),
                  channel_scales=e["s_ch"].to(DEV), schedule=schedule, bias=bias)
    torch.cuda.synchronize()
    return out.cpu().double().numpy()


def fp8_ref(e, rows=None, cols=None):
    ref, absref = oracle.w4a8_fp8(e["a"].numpy(), e["w"], e["layout"], e["wtype"], e["K"], e["N"])
    sc = np.outer(e["s_tok"].double().numpy(), e["s_ch"].double().numpy())
    ref, absref = ref * sc, absref * sc
    if rows is not None:
        return ref[rows, cols], absref[rows, cols]
    return ref, absref


@pytest.mark.parametrize("name", F8_SCHEDULES)
def test_w4a8_fp8_every_schedule(gpu_lib, name):
    w4 = gpu_lib
    M = min(ROWS.get(name, 40), 40) - 3
    e = w4synth.gen_w4a8_fp8(M, 384, 2048, seed=M + 5)
    got = run_fp8(w4, e, sched(w4, name))
    ref, absref = fp8_ref(e)
    assert_within(got, ref, absref, "f16", f"fp8 {name}")


@pytest.mark.parametrize("name", ["tc64_sk", "tc256_sk", "gv16_cl", "tc256p_sk", "tc256p_dp",
                                  "tc128p_sk"])
def test_w4a8_fp8_bias(gpu_lib, name):
    """fp8 activations with a bias: added in fp32 to the scaled sum before the
    one rounding to fp16 (the bias is exact in fp32, so the bound is the
    product's plus the final rounding)."""
    w4 = gpu_lib
    M = min(ROWS.get(name, 40), 40) - 5
    e = w4synth.gen_w4a8_fp8(M, 384, 2048, seed=M + 15)
    bias = (torch.randn(384, generator=torch.Generator().manual_seed(16)) * 4).half()
    got = run_fp8(w4, e, sched(w4, name), bias=bias.to(DEV))
    ref, absref = fp8_ref(e)
    assert_within(got, ref + bias.double().numpy()[None, :], absref, "f16", f"fp8 bias {name}")


@pytest.mark.parametrize("M", [1, 8, 32, 128, 1024])
def test_w4a8_fp8_qqq_shape(gpu_lib, M):
    """The QQQ sweep shape (N=8192, K=21760) with fp8 activations, default
    schedule, on sampled elements computed one by one."""
    w4 = gpu_lib
    N, K = w4synth.QQQ_N, w4synth.QQQ_K
    e = w4synth.gen_w4a8_fp8(M, N, K, seed=M)
    got = run_fp8(w4, e)
    rows, cols = samples(M, N, count=48, seed=M)
    a = e["a"][torch.from_numpy(np.unique(rows))]
    # the oracle on the sampled rows only (full N), then the sampled columns
    ur = np.unique(rows)
    sub = dict(e, a=a, M=len(ur), s_tok=e["s_tok"][torch.from_numpy(ur)])
    ref, absref = fp8_ref(sub)
    idx = np.searchsorted(ur, rows)
    assert_within(got[rows, cols], ref[idx, cols], absref[idx, cols], "f16", f"fp8 QQQ M={M}")


# ----------------------------------------- stage slots reused many times ---
# N=8192 and a long K give every CTA of a forced tensor-core schedule dozens
# of pipeline stages, so each shared-memory stage slot is refilled many
# times and each converter group waits on slots whose previous stage another
# group converted (a wait that passed on the previous stage's phase would
# convert stale bytes).

SLOT_SCHEDULES = ["tc16_sk", "tc32_sk", "tc64_sk", "tc128_sk", "tc128x2_sk", "tc256_sk",
                  "tc256p_sk", "tc128p_sk"]
SLOT_BM = {"tc16_sk": 16, "tc32_sk": 32, "tc64_sk": 64, "tc128_sk": 128, "tc128x2_sk": 128,
           "tc256_sk": 256, "tc256p_sk": 256, "tc128p_sk": 128}


@pytest.mark.parametrize("name", SLOT_SCHEDULES)
def test_w4a8_int32_stage_slots_cycle(gpu_lib, name):
    w4 = gpu_lib
    M, N, K = SLOT_BM[name] - 3, 8192, 16384
    e = w4synth.gen_w4a8(M, N, K, group_size=-1, seed=61)
    acc = run_w4a8(w4, e, torch.int32, sched(w4, name)).numpy().astype(np.int64)
    rows, cols = samples(M, N, count=256, seed=62)
    ref = oracle.w4a8_elems(e["a"], e["w"], e["layout"], e["wtype"], None, -1, K, N, rows, cols)
    assert np.array_equal(acc[rows, cols], ref), name


@pytest.mark.parametrize("name", SLOT_SCHEDULES)
def test_w4a8_fp8_stage_slots_cycle(gpu_lib, name):
    w4 = gpu_lib
    M, N, K = SLOT_BM[name] - 3, 8192, 16384
    e = w4synth.gen_w4a8_fp8(M, N, K, seed=63)
    got = run_fp8(w4, e, sched(w4, name))
    ur = np.unique(np.array([0, M // 2, M - 1]))
    sub = dict(e, a=e["a"][torch.from_numpy(ur)], M=len(ur),
               s_tok=e["s_tok"][torch.from_numpy(ur)])
    ref, absref = fp8_ref(sub)
    assert_within(got[ur], ref, absref, "f16", f"fp8 slots {name}")


@pytest.mark.parametrize("name", SLOT_SCHEDULES)
def test_w4a16_stage_slots_cycle(gpu_lib, name):
    w4 = gpu_lib
    M, N, K = SLOT_BM[name] - 3, 8192, 16384
    d = w4synth.gen_w4a16(M, N, K, act_dtype=torch.bfloat16, wtype=w4.UINT4,
                          layout=w4.NK_EXLLAMA, group_size=128, zeros=True, seed=64)
    got = run_w4a16(w4, d, sched(w4, name)).double().numpy()
    rows, cols = samples(M, N, count=256, seed=65)
    ref, absref = oracle.w4a16_elems(d["a"], d["w"], d["layout"], d["wtype"], d["s"], d["z"], 128,
                                     K, N, rows, cols)
    assert_within(got[rows, cols], ref, absref, "bf16", f"w4a16 slots {name}")


def test_w4a8_fp8_rejections(gpu_lib):
    w4 = gpu_lib
    e = w4synth.gen_w4a8_fp8(4, 256, 512, seed=1)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], 512, 256)
    a = e["a"].to(DEV).view(torch.float8_e4m3fn)
    with pytest.raises(w4.W4Error) as ei:  # raw int32 output: the sum is not an integer
        w4.gemm(a, b, e["wtype"], 256, group_size=-1, out_dtype=torch.int32)
    assert ei.value.status == w4.ERR_UNSUPPORTED
    with pytest.raises(w4.W4Error) as ei:  # per-group scales
        w4.gemm(a, b, e["wtype"], 256, scales=torch.ones(4, 256, dtype=torch.int8, device=DEV),
                group_size=128, token_scales=e["s_tok"].to(DEV), channel_scales=e["s_ch"].to(DEV))
    assert ei.value.status == w4.ERR_UNSUPPORTED
    with pytest.raises(w4.W4Error) as ei:  # ds cannot run fp8
        w4.gemm(a, b, e["wtype"], 256, group_size=-1, token_scales=e["s_tok"].to(DEV),
                channel_scales=e["s_ch"].to(DEV), schedule=sched(w4, "ds8_sk"))
    assert ei.value.status == w4.ERR_UNSUPPORTED



# ------------------------------------------- per-token fp8 quantization ---

@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,K", [(1, 21760), (16, 21760), (37, 4096), (5, 72), (3, 13),
                                 (1024, 21760), (2, 40000), (3, 65536), (2, 65600),
                                 (2000, 4096)])
def test_quantize_per_token_fp8_bit_exact(gpu_lib, M, K, dt):
    w4 = gpu_lib
    a = w4synth.gen_act16(M, K, dt, seed=M + 3 * K)
    q, s = w4.quantize_per_token_fp8(a.to(DEV))
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token_fp8(a)
    assert np.array_equal(s.cpu().numpy().view(np.int32), rs.view(np.int32)), "scales"
    bad = np.argwhere(q.cpu().view(torch.uint8).numpy() != rq)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:3].tolist()}"


@pytest.mark.parametrize("aligned", [True, False])
def test_quantize_fp8_special_rows(gpu_lib, aligned):
    """Zero rows, an outlier, ties between E4M3 values, the subnormal range,
    the largest and the smallest bf16 magnitudes."""
    w4 = gpu_lib
    K = 264
    dt = torch.bfloat16
    a = w4synth.gen_act16(8, K, dt, seed=31).float()
    a[0] = 0.0
    a[1] = 0.0
    a[1, 7] = -448.0
    a[2, :6] = torch.tensor([448.0, 9.0, 11.0, 13.0, -15.0, 0.0068359375])  # ties / subnormal step
    a[3] *= 3.0e38 / a[3].abs().max()
    a[4] *= 1.0e-38 / a[4].abs().max()
    a[5, ::3] = 1000.0
    a = a.to(dt)
    if aligned:
        a_dev = a.to(DEV)
    else:
        buf = torch.zeros(a.numel() + 1, dtype=dt, device=DEV)
        buf[1:] = a.reshape(-1).to(DEV)
        a_dev = buf[1:].view(a.shape)
    q, s = w4.quantize_per_token_fp8(a_dev)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token_fp8(a)
    assert np.array_equal(s.cpu().numpy().view(np.int32), rs.view(np.int32))
    assert np.array_equal(q.cpu().view(torch.uint8).numpy(), rq)
    assert s[0].item() == 0 and int(q[0].view(torch.uint8).sum()) == 0


# --------------------------- W4A8 with dynamic per-token quantization ---

@pytest.mark.parametrize("M", [1, 7, 24, 40, 300, 1024])
@pytest.mark.parametrize("gs", [-1, 128])
def test_gemm_dynamic_int8_equals_two_steps(gpu_lib, M, gs):
    """The fused call gives exactly what quantize_per_token followed by the
    W4A8 gemm gives (same codes, same schedule), and its codes / scales are
    the oracle's (through token_scales_out and the product)."""
    w4 = gpu_lib
    N, K = 1024, 4096
    e = w4synth.gen_w4a8(M, N, K, group_size=gs, seed=M + 2)
    a16 = w4synth.gen_act16(M, K, torch.float16, seed=M + 9).to(DEV)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], K, N)
    sg = None if e["sg"] is None else e["sg"].to(DEV)
    sch = e["s_ch"].to(DEV)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3)).half().to(DEV)
    stok = torch.empty(M, dtype=torch.float32, device=DEV)
    out = w4.gemm_dynamic(a16, b, e["wtype"], N, torch.int8, scales=sg, group_size=gs,
                          channel_scales=sch, bias=bias, token_scales_out=stok)
    q, s = w4.quantize_per_token(a16)
    ref2 = w4.gemm(q, b, e["wtype"], N, scales=sg, group_size=gs, token_scales=s,
                   channel_scales=sch, bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(stok, s)
    assert torch.equal(out, ref2)
    rq, rs = oracle.quant_per_token(a16.cpu())
    assert np.array_equal(s.cpu().numpy().view(np.int32), rs.view(np.int32))
    rows, cols = samples(M, N, count=64, seed=M)
    acc = oracle.w4a8_elems(rq, e["w"], e["layout"], e["wtype"], e["sg"], gs, K, N, rows, cols)
    prod = oracle.w4a8_scale(acc, rows, cols, rs.astype(np.float64), e["s_ch"])
    assert_fp16_near(out.cpu().double().numpy()[rows, cols], oracle.add_bias(prod, cols, bias.cpu()),
                     np.abs(prod) + np.abs(bias.cpu().double().numpy()[cols]), f"dynamic M={M}")


@pytest.mark.parametrize("M", [1, 24, 300])
def test_gemm_dynamic_fp8(gpu_lib, M):
    """fp8 activations quantized inside the call: the oracle's E4M3 codes and
    scales through the oracle's W4A8-fp8 product, within the float bound."""
    w4 = gpu_lib
    N, K = 512, 2048
    e = w4synth.gen_w4a8(M, N, K, group_size=-1, seed=M + 4)
    a16 = w4synth.gen_act16(M, K, torch.bfloat16, seed=M + 5)
    b = w4.prepack_B(e["w"].to(DEV), e["wtype"], e["layout"], K, N)
    out = w4.gemm_dynamic(a16.to(DEV), b, e["wtype"], N, torch.float8_e4m3fn, group_size=-1,
                          channel_scales=e["s_ch"].to(DEV))
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token_fp8(a16)
    ref, absref = oracle.w4a8_fp8(rq, e["w"], e["layout"], e["wtype"], K, N)
    sc = np.outer(rs.astype(np.float64), e["s_ch"].double().numpy())
    assert_within(out.cpu().double().numpy(), ref * sc, absref * sc, "f16", f"dynamic fp8 M={M}")
