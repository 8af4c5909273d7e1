"""Pins for the CPU oracle: values the pages print, hand-worked examples,
closed forms, invariants and library routines (CPU only, no GPU).

Each test would fail under a plausible slip in the oracle: a wrong shift
table or word index, a dropped zero-point or scale, a wrong sign or group
index, a transposed operand.
"""
import numpy as np
import pytest
import torch

import oracle
import w4synth
from conftest import golden_kv, golden_lines

LAYOUTS = [oracle.KN_SEQ, oracle.NK_SEQ, oracle.NK_EXLLAMA]


def _word_array(words_hex, layout):
    w = np.array([np.uint32(int(h, 16)).view(np.int32) for h in words_hex], dtype=np.int32)
    # K=8, N=len(words): KN_SEQ is [1, N], NK layouts are [N, 1]
    return w.reshape(1, -1) if layout == oracle.KN_SEQ else w.reshape(-1, 1)


# ---------------------------------------------------------------- packing ---

def test_exllama_words_match_page_formula():
    rows = golden_lines("exllama_pack.txt")
    q = np.array([[int(x) for x in r[:8]] for r in rows], dtype=np.uint8).T  # [8, N]
    w = oracle.pack(q, oracle.NK_EXLLAMA)
    expect = _word_array([r[8] for r in rows], oracle.NK_EXLLAMA)
    assert np.array_equal(w, expect)
    assert np.array_equal(oracle.unpack(expect, oracle.NK_EXLLAMA, 8, q.shape[1]), q)


def test_exllama_shift_table():
    shifts = [int(x) for x in golden_lines("exllama_shifts.txt")[0]]
    for j, sh in enumerate(shifts):
        for v in range(16):
            word = np.array([[np.uint32(v << sh).view(np.int32)]], dtype=np.int32)
            q = oracle.unpack(word, oracle.NK_EXLLAMA, 8, 1)[:, 0]
            expect = np.zeros(8, np.uint8)
            expect[j] = v
            assert np.array_equal(q, expect), (j, v)


def test_sequential_words():
    rows = golden_lines("sequential_pack.txt")
    q = np.array([[int(x) for x in r[:8]] for r in rows], dtype=np.uint8).T
    for layout in (oracle.KN_SEQ, oracle.NK_SEQ):
        expect = _word_array([r[8] for r in rows], layout)
        assert np.array_equal(oracle.pack(q, layout), expect)
        assert np.array_equal(oracle.unpack(expect, layout, 8, q.shape[1]), q)


def test_kn_and_nk_are_transposes():
    rng = np.random.default_rng(1)
    q = rng.integers(0, 16, size=(64, 24), dtype=np.uint8)
    assert np.array_equal(oracle.pack(q, oracle.KN_SEQ), oracle.pack(q, oracle.NK_SEQ).T)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_pack_unpack_round_trip(layout):
    rng = np.random.default_rng(layout)
    K, N = 96, 40
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    w = oracle.pack(q, layout)
    assert np.array_equal(oracle.unpack(w, layout, K, N), q)
    words = w4synth.random_words(w4synth.packed_shape(layout, K, N), torch.Generator().manual_seed(3))
    assert np.array_equal(oracle.pack(oracle.unpack(words, layout, K, N), layout), words.numpy())


@pytest.mark.parametrize("layout", LAYOUTS)
def test_every_nibble_in_every_position(layout):
    # brute force over one word: each of the 8 positions x 16 values
    for j in range(8):
        for v in range(16):
            q = np.zeros((8, 1), np.uint8)
            q[j, 0] = v
            w = oracle.pack(q, layout)
            assert oracle.nibble(w, layout, 8, 1, j, 0) == v
            assert sum(oracle.nibble(w, layout, 8, 1, k, 0) for k in range(8)) == v


def test_value_table():
    for r in golden_lines("values.txt"):
        q, b8, u4, i4 = (int(x) for x in r)
        assert oracle.value(q, oracle.UINT4B8) == b8
        assert oracle.value(q, oracle.UINT4) == u4
        assert oracle.value(q, oracle.INT4) == i4


# ----------------------------------------------------------------- W4A16 ---

def _one_col(q_list, layout=oracle.NK_EXLLAMA):
    q = np.array(q_list, dtype=np.uint8).reshape(8, 1)
    return oracle.pack(q, layout)


def test_w4a16_worked_example():
    g = golden_kv("worked_examples.txt")
    a = np.array([[float(x) for x in g["w4a16_a"]]])
    for layout in LAYOUTS:
        w = _one_col([int(x) for x in g["w4a16_q"]], layout)
        s = np.array([[float(g["w4a16_s"][0])]])
        ref, absref = oracle.w4a16(a, w, layout, oracle.UINT4B8, s, None, -1, 8, 1)
        assert ref[0, 0] == float(g["w4a16_ref"][0])
        assert absref[0, 0] == float(g["w4a16_absref"][0])
        z = np.array([[float(g["w4a16_z_uint4"][0])]])
        ref2, _ = oracle.w4a16(a, w, layout, oracle.UINT4, s, z, -1, 8, 1)
        assert ref2[0, 0] == float(g["w4a16_ref"][0])


def _pow2_problem(M, N, K, gs, seed, zeros):
    """Inputs whose every product and sum is exact in fp64: fp16 activations,
    power-of-two scales, power-of-two-multiple zero-points."""
    rng = np.random.default_rng(seed)
    G = K // gs
    a = torch.randn(M, K, generator=torch.Generator().manual_seed(seed)).to(torch.float16)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s = (2.0 ** rng.integers(-8, -3, size=(G, N))).astype(np.float64)
    z = (rng.integers(0, 16, size=(G, N)) * s).astype(np.float64) if zeros else None
    return a, q, s, z


@pytest.mark.parametrize("wtype", [oracle.UINT4B8, oracle.UINT4])
@pytest.mark.parametrize("zeros", [False, True])
def test_w4a16_equals_blockwise_library_matmul(wtype, zeros):
    M, N, K, gs = 5, 24, 256, 64
    a, q, s, z = _pow2_problem(M, N, K, gs, 7 + wtype, zeros)
    w = oracle.pack(q, oracle.KN_SEQ)
    ref, _ = oracle.w4a16(a, w, oracle.KN_SEQ, wtype, s, z, gs, K, N)
    v = q.astype(np.float64) - (8.0 if wtype == oracle.UINT4B8 else 0.0)
    a64 = a.to(torch.float64).numpy()
    expect = np.zeros((M, N))
    for gi in range(K // gs):
        blk = slice(gi * gs, (gi + 1) * gs)
        what = v[blk] * s[gi][None, :] - (z[gi][None, :] if zeros else 0.0)
        expect += a64[:, blk] @ what
    assert np.array_equal(ref, expect)


def test_w4a16_unit_scale_is_plain_matmul():
    M, N, K = 3, 17, 64
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    a = torch.randn(M, K, generator=torch.Generator().manual_seed(5)).to(torch.float16)
    w = oracle.pack(q, oracle.NK_SEQ)
    ref, _ = oracle.w4a16(a, w, oracle.NK_SEQ, oracle.UINT4, np.ones((1, N)), None, -1, K, N)
    assert np.array_equal(ref, a.to(torch.float64).numpy() @ q.astype(np.float64))


def test_w4a16_one_hot_rows_give_dequantized_weights():
    M, N, K, gs = 8, 16, 128, 32
    a, q, s, z = _pow2_problem(M, N, K, gs, 11, True)
    a = torch.zeros(K, K, dtype=torch.float16)
    a[torch.arange(K), torch.arange(K)] = 1.0
    w = oracle.pack(q, oracle.NK_EXLLAMA)
    ref, _ = oracle.w4a16(a, w, oracle.NK_EXLLAMA, oracle.UINT4, s, z, gs, K, N)
    # row k of the product is w_hat[k, :]; check against the scale/zero of k's group
    for k in (0, 31, 32, 100, 127):
        gi = k // gs
        assert np.array_equal(ref[k], q[k].astype(np.float64) * s[gi] - z[gi])


def test_w4a16_invariants():
    M, N, K = 4, 32, 256
    d = w4synth.gen_w4a16(M, N, K, act_dtype=torch.bfloat16, wtype=oracle.UINT4,
                          layout=oracle.NK_EXLLAMA, group_size=128, zeros=True, seed=2)
    args = (d["w"], d["layout"])
    # zero-points that are all zero equal no zero-points
    r0, _ = oracle.w4a16(d["a"], *args, oracle.UINT4, d["s"], torch.zeros_like(d["z"]), 128, K, N)
    r1, _ = oracle.w4a16(d["a"], *args, oracle.UINT4, d["s"], None, 128, K, N)
    assert np.array_equal(r0, r1)
    # uint4 with w_z = 8*s equals uint4b8 (exact: 8*s is a power-of-two multiple)
    r2, _ = oracle.w4a16(d["a"], *args, oracle.UINT4, d["s"], d["s"].double() * 8, 128, K, N)
    r3, _ = oracle.w4a16(d["a"], *args, oracle.UINT4B8, d["s"], None, 128, K, N)
    assert np.allclose(r2, r3, rtol=0, atol=1e-12)
    # group_size = K equals per-channel with the one scale row broadcast
    s1 = d["s"][:1]
    r4, _ = oracle.w4a16(d["a"], *args, oracle.UINT4B8, s1.repeat(2, 1), None, 128, K, N)
    r5, _ = oracle.w4a16(d["a"], *args, oracle.UINT4B8, s1, None, -1, K, N)
    assert np.array_equal(r4, r5)
    # rows are independent: M=1 (a GEMV) equals the matching row of the batch
    full, absfull = oracle.w4a16(d["a"], *args, oracle.UINT4, d["s"], d["z"], 128, K, N)
    for m in range(M):
        row, _ = oracle.w4a16(d["a"][m:m + 1], *args, oracle.UINT4, d["s"], d["z"], 128, K, N)
        assert np.array_equal(row[0], full[m])
    # |ref| <= sum|terms|, and linear in a
    assert np.all(np.abs(full) <= absfull + 1e-12)
    a2 = (d["a"].double() * 2).to(torch.bfloat16)  # exact doubling
    r6, _ = oracle.w4a16(a2, *args, oracle.UINT4, d["s"], d["z"], 128, K, N)
    assert np.array_equal(r6, 2 * full)
    # sampled elements equal the full product at those positions
    rows = np.array([0, 3, 1, 2]); cols = np.array([0, 31, 7, 16])
    e, ea = oracle.w4a16_elems(d["a"], *args, oracle.UINT4, d["s"], d["z"], 128, K, N, rows, cols)
    assert np.array_equal(e, full[rows, cols]) and np.array_equal(ea, absfull[rows, cols])


def test_w4a16_layouts_agree():
    M, N, K = 3, 24, 128
    rng = np.random.default_rng(9)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    a = torch.randn(M, K, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    s = torch.rand(1, N, generator=torch.Generator().manual_seed(10)).to(torch.bfloat16)
    outs = [oracle.w4a16(a, oracle.pack(q, L), L, oracle.UINT4B8, s, None, -1, K, N)[0]
            for L in LAYOUTS]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


# ------------------------------------------------------------------ W4A8 ---

def test_w4a8_worked_example():
    g = golden_kv("worked_examples.txt")
    a = np.array([[int(x) for x in g["w4a8_a"]]], dtype=np.int8)
    for layout in LAYOUTS:
        w = _one_col([int(x) for x in g["w4a8_q"]], layout)
        acc = oracle.w4a8(a, w, layout, oracle.INT4, None, -1, 8, 1)
        assert acc[0, 0] == int(g["w4a8_acc_channel"][0])
        sg = np.array([[int(x)] for x in g["w4a8_sg"]], dtype=np.int8)  # [G=2, N=1]
        acc2 = oracle.w4a8(a, w, layout, oracle.INT4, sg, 4, 8, 1)
        assert acc2[0, 0] == int(g["w4a8_acc_g4"][0])


def test_w4a8_equals_integer_matmul():
    M, N, K = 6, 40, 512
    d = w4synth.gen_w4a8(M, N, K, group_size=128, seed=4)
    q = oracle.unpack(d["w"], d["layout"], K, N).astype(np.int64)
    v = np.where(q >= 8, q - 16, q)
    a = d["a"].numpy().astype(np.int64)
    acc = oracle.w4a8(d["a"], d["w"], d["layout"], oracle.INT4, None, -1, K, N)
    assert np.array_equal(acc, a @ v)
    sg = d["sg"].numpy().astype(np.int64)
    accg = oracle.w4a8(d["a"], d["w"], d["layout"], oracle.INT4, d["sg"], 128, K, N)
    assert np.array_equal(accg, a @ (v * np.repeat(sg, 128, axis=0)))
    # unit group scales equal per-channel; constant group scale c multiplies by c
    ones = torch.ones_like(d["sg"])
    assert np.array_equal(oracle.w4a8(d["a"], d["w"], d["layout"], oracle.INT4, ones, 128, K, N), acc)
    assert np.array_equal(oracle.w4a8(d["a"], d["w"], d["layout"], oracle.INT4, ones * 5, 128, K, N), 5 * acc)
    # uint4b8 and int4 hold the same values once the top bit of each nibble is flipped
    flipped = (d["w"].numpy().view(np.uint32) ^ np.uint32(0x88888888)).view(np.int32)
    assert np.array_equal(oracle.w4a8(d["a"], flipped, d["layout"], oracle.UINT4B8, None, -1, K, N), acc)
    rows = np.array([0, 5, 2]); cols = np.array([39, 0, 17])
    assert np.array_equal(oracle.w4a8_elems(d["a"], d["w"], d["layout"], oracle.INT4, d["sg"], 128,
                                            K, N, rows, cols), accg[rows, cols])


def test_w4a8_extreme_accumulator_fits_int32():
    # the largest |acc| the QQQ shape allows: K=21760, a=-127, v=-8, sg=16
    K, N = 21760, 1
    q = np.full((K, N), 8, dtype=np.uint8)  # int4 nibble 8 -> -8
    w = oracle.pack(q, oracle.NK_EXLLAMA)
    a = np.full((1, K), -127, dtype=np.int8)
    sg = np.full((K // 128, N), 16, dtype=np.int8)
    acc = oracle.w4a8(a, w, oracle.NK_EXLLAMA, oracle.INT4, sg, 128, K, N)
    assert acc[0, 0] == 21760 * 127 * 8 * 16 and acc[0, 0] < 2**31


def test_w4a8_scale_closed_form():
    acc = np.array([3, -7, 1 << 20]); rows = np.array([0, 1, 1]); cols = np.array([1, 0, 1])
    s_tok = np.array([0.5, 0.25]); s_ch = np.array([2.0, 0.125])
    ref = oracle.w4a8_scale(acc, rows, cols, s_tok, s_ch)
    assert list(ref) == [3 * 0.5 * 0.125, -7 * 0.25 * 2.0, (1 << 20) * 0.25 * 0.125]


# --------------------------------------------- per-token int8 quantization ---
# Reading of vLLM PR #6547 "Enable Dynamic Per Token fp8" (one scale per
# token, from that token's values) with the symmetric int8 activations of
# pytorch/ao PR #1113: s = amax / 127, q = round-half-even(a / s), in fp32.

def test_quant_worked_example():
    # amax 254 -> s = 2 exactly; 127/2 = 63.5 and 65/2 = 32.5 are ties (to
    # even: 64 and 32), 63.5/2 = 31.75 -> 32, 0.5/2 = 0.25 -> 0
    a = torch.tensor([[-254.0, 127.0, 63.5, 0.5, 0.0, 65.0, -65.0, 5.0],
                      [0.0] * 8,
                      [3.0, -3.0, 1.5, 0.0, 0.0, 0.0, 0.0, 0.0]], dtype=torch.float16)
    q, s = oracle.quant_per_token(a)
    assert s.dtype == np.float32 and list(s[:2]) == [2.0, 0.0]
    assert q[0].tolist() == [-127, 64, 32, 0, 0, 32, -32, 2]
    assert q[1].tolist() == [0] * 8
    # amax 3: s = fl32(3/127); 3/s and -3/s round to +-127, 1.5/s = 63.5(1+d) -> 63 or 64
    assert q[2, 0] == 127 and q[2, 1] == -127 and q[2, 2] in (63, 64)


def test_quant_error_bound_and_extremes():
    g = torch.Generator().manual_seed(3)
    for dt in (torch.float16, torch.bfloat16):
        a = torch.randn(24, 1000, generator=g).to(dt)
        a[5, 17] = 40.0  # an outlier channel
        q, s = oracle.quant_per_token(a)
        x = a.double().numpy()
        amax = np.abs(x).max(axis=1)
        s64 = s.astype(np.float64)
        # 127 steps of s reach amax (to the rounding of one fp32 division)
        assert np.all(np.abs(s64 * 127 - amax) <= amax * 2.0**-23)
        # every code within half a step of the value, |q| <= 127
        err = np.abs(q.astype(np.float64) * s64[:, None] - x)
        assert np.all(err <= s64[:, None] * (0.5 + 1e-5))
        assert np.abs(q.astype(np.int32)).max() <= 127
        # the largest |a| of a row maps to +-127 with its sign
        am = np.abs(x).argmax(axis=1)
        r = np.arange(x.shape[0])
        assert np.array_equal(q[r, am].astype(np.int32), 127 * np.sign(x[r, am]).astype(np.int32))


def test_quant_symmetry_scaling_rows_independent():
    g = torch.Generator().manual_seed(4)
    a = torch.randn(9, 300, generator=g).to(torch.bfloat16)
    q, s = oracle.quant_per_token(a)
    qn, sn = oracle.quant_per_token(-a)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    for e in (-3, 5):  # powers of two scale s and leave the codes
        qe, se = oracle.quant_per_token(a.float() * 2.0**e)
        assert np.array_equal(qe, q) and np.array_equal(se, s * np.float32(2.0**e))
    for m in (0, 4, 8):  # each row on its own (M = 1) gives the same result
        q1, s1 = oracle.quant_per_token(a[m:m + 1])
        assert np.array_equal(q1[0], q[m]) and s1[0] == s[m]
    qz, sz = oracle.quant_per_token(np.zeros((3, 0), np.float32))
    assert qz.shape == (3, 0) and list(sz) == [0.0, 0.0, 0.0]


def test_quant_brute_force_exact_rationals():
    """Codes against exact rational arithmetic: the nearest integer to a/s
    (ties to even) for the returned fp32 s, except where a/s lies so close
    to a half-integer that rounding the quotient to fp32 may decide it."""
    from fractions import Fraction

    g = torch.Generator().manual_seed(5)
    a = (torch.rand(6, 64, generator=g) * 20 - 10).to(torch.float16)
    a[2, :8] = torch.tensor([2.5, -2.5, 10.0, 0.125, -7.75, 3.0, 1.0, 0.0])
    q, s = oracle.quant_per_token(a)
    x = a.float().numpy()
    checked = 0
    for m in range(x.shape[0]):
        sm = Fraction(float(s[m]))
        for k in range(x.shape[1]):
            t = Fraction(float(x[m, k])) / sm
            fl = t.numerator // t.denominator
            frac = t - fl
            exact = fl + (1 if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and fl % 2) else 0)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 1 << 16) * (abs(t) + 1):
                assert q[m, k] in (fl, fl + 1)
                continue
            assert q[m, k] == exact, (m, k, t)
            checked += 1
    assert checked > 370


def test_quant_feeds_w4a8_within_quantization_error():
    """Dynamic quantization then W4A8 approximates the fp64 product a x v
    to within the codes' error: |acc*s_tok - a.v| <= sum_k (s/2)|v_k|."""
    M, N, K = 5, 48, 256
    g = torch.Generator().manual_seed(6)
    a = torch.randn(M, K, generator=g).to(torch.float16)
    w = w4synth.random_words(w4synth.packed_shape(oracle.NK_EXLLAMA, K, N), g)
    q, s = oracle.quant_per_token(a)
    acc = oracle.w4a8(q, w, oracle.NK_EXLLAMA, oracle.INT4, None, -1, K, N)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    approx = oracle.w4a8_scale(acc.reshape(-1), rows.reshape(-1), cols.reshape(-1),
                               s.astype(np.float64), np.ones(N)).reshape(M, N)
    v = np.vectorize(lambda t: oracle.value(int(t), oracle.INT4))(
        oracle.unpack(w, oracle.NK_EXLLAMA, K, N)).astype(np.float64)
    exact = a.double().numpy() @ v
    bound = (s.astype(np.float64)[:, None] / 2) * np.abs(v).sum(axis=0)[None, :] * (1 + 1e-4)
    assert np.all(np.abs(approx - exact) <= bound)
    assert np.abs(approx - exact).max() > 0  # the codes are not exact here


def test_quant_quotient_rounded_once_in_fp32():
    """Codes decided by one correctly rounded fp32 division a / s (worked
    with exact rationals):
      amax 0.80615234375: s = amax/127 = 0.00634765625 exactly, and
        0.041259765625 / s = 6.5, 0.092041015625 / s = 14.5 exactly
        (ties, to even: 6 and 14);
      amax 3110: s = fl32(3110/127) = 24.488189697265625; 1555 / s is
        63.5 - 1.87e-6, which rounds to the fp32 value 63.5 (a tie: 64);
      amax 12.0078125: 6.00390625 / s is 63.5 - 2.25e-6, whose fp32 value
        63.499996... gives 63.
    Multiplying by a rounded reciprocal 1/s instead gives 7, 15, 63, 64."""
    a = torch.tensor([[0.80615234375, 0.041259765625, 0.092041015625],
                      [3110.0, 1555.0, 0.0],
                      [12.0078125, 6.00390625, 0.0]], dtype=torch.float16)
    q, s = oracle.quant_per_token(a)
    assert s[0] == np.float32(0.00634765625) and s[1] == np.float32(24.488189697265625)
    assert q.tolist() == [[127, 6, 14], [127, 64, 0], [127, 63, 0]]


# ------------------------------------------------- fp8 (E4M3) activations ---
# vLLM PR #9855: QQQ-style W4A8 "including fp8 activations"; the format is
# read as OCP E4M3 (bias 7, subnormals m/8 * 2^-6, S.1111.111 NaN, max 448).

def test_e4m3_decode_worked_codes():
    # values worked by hand from the format definition
    table = {0x00: 0.0, 0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x08: 2.0**-6, 0x30: 0.5, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x4C: 6.0, 0x50: 8.0, 0x77: 240.0,
             0x78: 256.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xC0: -2.0, 0xFE: -448.0}
    got = oracle.e4m3_decode(np.array(list(table), dtype=np.uint8))
    assert list(got) == list(table.values())
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    assert np.signbit(oracle.e4m3_decode(np.array([0x80], np.uint8)))[0]


def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], lib[ok])


def test_e4m3_encode_ties_saturation_round_trip():
    x = np.float32([1.0625, 1.1875, 3.125, 3.25, 0.5 * 2**-9, 1.5 * 2**-9, 7.5 * 2**-9, 448, 464,
                    470, 500, -1e30, -0.0, 0.0])
    # ties go to the even mantissa: 1.0625 -> 1.0 (m=0), 1.1875 -> 1.25 (m=2),
    # 3.125 (between 3.0 = 1.5*2 and 3.25 = 1.625*2) -> 3.0 (m=4); 3.25 is exact
    # (0x45); subnormal ties 0.5 and 1.5 steps of 2^-9 -> 0 and 2 steps;
    # 7.5 * 2^-9 -> 2^-6 (0x08); 448 and above saturate to 448 (470 would round
    # to the NaN pattern 0x7F without the saturation)
    got = oracle.e4m3_encode(x).tolist()
    assert got == [0x38, 0x3A, 0x44, 0x45, 0x00, 0x02, 0x08, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00]
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(finite).astype(np.float32)), finite)


def test_e4m3_encode_matches_torch_in_range_and_is_nearest():
    g = torch.Generator().manual_seed(8)
    x = torch.cat([torch.randn(20000, generator=g) * 40, torch.randn(20000, generator=g) * 0.01,
                   (torch.rand(5000, generator=g) - 0.5) * 895])
    x = x[x.abs() < 448]
    ours = oracle.e4m3_encode(x)
    lib = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
    # nearest: no finite code is closer than the chosen one
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = vals[~np.isnan(vals)]
    xs = x.double().numpy()[:500]
    best = np.abs(finite[None, :] - xs[:, None]).min(axis=1)
    assert np.array_equal(np.abs(oracle.e4m3_decode(ours[:500]) - xs), best)


def test_quant_fp8_scale_bound_and_invariants():
    g = torch.Generator().manual_seed(9)
    a = torch.randn(16, 700, generator=g).to(torch.bfloat16)
    a[3] = 0.0
    q, s = oracle.quant_per_token_fp8(a)
    x = a.double().numpy()
    v = oracle.e4m3_decode(q)
    amax = np.abs(x).max(axis=1)
    s64 = s.astype(np.float64)
    assert s[3] == 0 and not q[3].any()
    live = amax > 0
    assert np.all(np.abs(s64[live] * 448 - amax[live]) <= amax[live] * 2.0**-23)
    # each code within half a step of E4M3 at its magnitude (relative 2^-4, or
    # 2^-10 absolute in the subnormal range), on the scale of the row
    t = x[live] / s64[live, None]
    step = np.where(np.abs(t) >= 2.0**-6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(t), 2.0**-6))) - 3),
                    2.0**-9)
    assert np.all(np.abs(v[live] - t) <= step / 2 * (1 + 1e-5) + 1e-12)
    # the largest |a| of a row maps to +-448
    r = np.flatnonzero(live)
    am = np.abs(x[r]).argmax(axis=1)
    assert np.array_equal(np.abs(v[r, am]), np.full(r.size, 448.0))
    qn, sn = oracle.quant_per_token_fp8(-a)
    assert np.array_equal(oracle.e4m3_decode(qn)[live], -v[live]) and np.array_equal(sn, s)
    q2, s2 = oracle.quant_per_token_fp8(a.float() * 8.0)
    assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(8.0))


def test_w4a8_fp8_exact_matmul_and_bound():
    M, N, K = 6, 40, 384
    g = torch.Generator().manual_seed(10)
    a = torch.randn(M, K, generator=g).to(torch.float16)
    w = w4synth.random_words(w4synth.packed_shape(oracle.NK_EXLLAMA, K, N), g)
    q, s = oracle.quant_per_token_fp8(a)
    ref, absref = oracle.w4a8_fp8(q, w, oracle.NK_EXLLAMA, oracle.INT4, K, N)
    v = np.vectorize(lambda t: oracle.value(int(t), oracle.INT4))(
        oracle.unpack(w, oracle.NK_EXLLAMA, K, N)).astype(np.float64)
    dec = oracle.e4m3_decode(q)
    assert np.array_equal(ref, dec @ v)          # exact: multiples of 2^-9 below 2^44
    assert np.array_equal(absref, np.abs(dec) @ np.abs(v))
    # uint4b8 weights hold the same values as int4 once each nibble's top bit flips
    flipped = (w.numpy().view(np.uint32) ^ np.uint32(0x88888888)).view(np.int32)
    assert np.array_equal(oracle.w4a8_fp8(q, flipped, oracle.NK_EXLLAMA, oracle.UINT4B8, K, N)[0], ref)
    # dequantized, the product stays within the codes' error of the fp64 a x v
    exact = a.double().numpy() @ v
    err = np.abs(ref * s.astype(np.float64)[:, None] - exact)
    bound = (np.abs(a.double().numpy()) * 2.0**-4 + s.astype(np.float64)[:, None] * 2.0**-10) @ np.abs(v)
    assert np.all(err <= bound)


def test_bias_worked_examples():
    """The bias step: the hand-worked W4A16 and W4A8 examples of
    tests/golden/worked_examples.txt plus a bias on their column."""
    g = golden_kv("worked_examples.txt")
    a = np.array([float(x) for x in g["w4a16_a"]]).reshape(1, 8)
    q = np.array([int(x) for x in g["w4a16_q"]], dtype=np.uint8).reshape(8, 1)
    w = oracle.pack(q, oracle.NK_EXLLAMA)
    s = np.full((1, 1), float(g["w4a16_s"][0]))
    ref, _ = oracle.w4a16(a, w, oracle.NK_EXLLAMA, oracle.UINT4B8, s, None, -1, 8, 1)
    got = oracle.add_bias(ref, None, np.array([float(g["w4a16_bias"][0])]))
    assert got[0, 0] == float(g["w4a16_ref_bias"][0])
    a8 = np.array([int(x) for x in g["w4a8_a"]], dtype=np.int8).reshape(1, 8)
    q8 = np.array([int(x) for x in g["w4a8_q"]], dtype=np.uint8).reshape(8, 1)
    w8 = oracle.pack(q8, oracle.NK_EXLLAMA)
    acc = oracle.w4a8(a8, w8, oracle.NK_EXLLAMA, oracle.INT4, None, -1, 8, 1)
    st, sc, bias = (float(x) for x in g["w4a8_scales_bias"])
    r = oracle.w4a8_scale(acc.reshape(-1), np.array([0]), np.array([0]), np.array([st]),
                          np.array([sc]))
    assert oracle.add_bias(r, np.array([0]), np.array([bias]))[0] == float(g["w4a8_ref_bias"][0])


def test_bias_is_a_per_column_shift():
    """A zero bias changes nothing; the bias shifts every row of a column by
    the same amount, independently of the product; flat and full forms
    agree."""
    rng = np.random.default_rng(3)
    ref = rng.integers(-1000, 1000, (5, 7)).astype(np.float64)  # sums stay exact
    assert np.array_equal(oracle.add_bias(ref, None, np.zeros(7)), ref)
    b = (rng.integers(-64, 64, 7) / 8).astype(np.float16)
    full = oracle.add_bias(ref, None, b)
    assert np.array_equal(full - ref, np.broadcast_to(b.astype(np.float64), (5, 7)))
    rows, cols = np.meshgrid(np.arange(5), np.arange(7), indexing="ij")
    flat = oracle.add_bias(ref.reshape(-1), cols.reshape(-1), b)
    assert np.array_equal(flat, full.reshape(-1))
