"""Seeded synthetic inputs for the 4-bit-weight GEMM (shared by tests and bench).

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no unpacking, no dequantization, no products).  Packed
weights are drawn as uniformly random int32 words, which is the same thing
as independent uniform nibbles 0..15 in every one of the input layouts.

Workload shapes and value distributions follow the pages' workloads:

* W4A16 tiny: A fp16 [16, 512] ~ N(0, 1); uint4b8 weights; fp16 group-128
  scales U[0.005, 0.02].
* W4A16 decode on Llama-3-8B linear shapes (N, K) in {(4096, 4096),
  (6144, 4096), (28672, 4096), (4096, 14336)}, M in {1, 4, 16, 64}: A bf16
  ~ N(0, 1); uint4 weights with integer zero-points z in 0..15 stored
  pre-scaled as bf16(z * s); bf16 scales U[0.005, 0.02]; group 128.
* W4A8 (QQQ style) at N=8192, K=21760: A int8 U{-127..127}; fp32 per-token
  scales U[0.01, 0.05]; int4 weights U{-8..7}; fp32 per-channel scales
  U[0.001, 0.01]; per-group variant with int8 group scales U{1..16}.
* W4A16 prefill on Llama-3-70B MLP shapes (N, K) in {(57344, 8192),
  (8192, 28672)}, M in {4096, 8192, 16384}: uint4b8, bf16 scales, group 128.
"""
from __future__ import annotations

import torch

KN_SEQ, NK_SEQ, NK_EXLLAMA = 0, 1, 2
UINT4B8, UINT4, INT4 = 0, 1, 2

DECODE_SHAPES = [(4096, 4096), (6144, 4096), (28672, 4096), (4096, 14336)]
DECODE_M = [1, 4, 16, 64]
QQQ_N, QQQ_K = 8192, 21760
QQQ_CH_M = [1, 8, 32, 128, 512, 1024]
QQQ_G128_M = [1, 16, 256, 2048]
PREFILL_SHAPES = [(57344, 8192), (8192, 28672)]
PREFILL_M = [4096, 8192, 16384]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def random_words(shape, g: torch.Generator) -> torch.Tensor:
    """Uniform int32 words (= uniform independent nibbles in any layout)."""
    w = torch.randint(-(2**31), 2**31, tuple(shape), generator=g, dtype=torch.int64)
    return w.to(torch.int32)


def packed_shape(layout: int, K: int, N: int):
    return (K // 8, N) if layout == KN_SEQ else (N, K // 8)


def uniform(shape, lo: float, hi: float, g: torch.Generator, dtype) -> torch.Tensor:
    x = torch.rand(tuple(shape), generator=g, dtype=torch.float32) * (hi - lo) + lo
    return x.to(dtype)


def gen_w4a16(M: int, N: int, K: int, act_dtype=torch.bfloat16, wtype: int = UINT4B8,
              layout: int = NK_EXLLAMA, group_size: int = 128, zeros: bool = False,
              seed: int = 0) -> dict:
    """CPU tensors for one W4A16 problem.

    Returns a [M,K] act_dtype ~N(0,1); w packed int32 in `layout`;
    s [G,N] act_dtype U[0.005,0.02]; z [G,N] act_dtype = round(z_int * s)
    with z_int U{0..15} (pre-scaled zero-point), or None.
    """
    g = _gen(seed)
    gs = K if group_size == -1 else group_size
    G = K // gs if K else 0
    a = torch.randn((M, K), generator=g, dtype=torch.float32).to(act_dtype)
    w = random_words(packed_shape(layout, K, N), g)
    s = uniform((G, N), 0.005, 0.02, g, act_dtype)
    z = None
    if zeros:
        z_int = torch.randint(0, 16, (G, N), generator=g, dtype=torch.int32)
        # z_int * s is exact in fp32 (4-bit times 8/11-bit); one rounding to act_dtype.
        z = (z_int.to(torch.float32) * s.to(torch.float32)).to(act_dtype)
    return dict(a=a, w=w, s=s, z=z, M=M, N=N, K=K, layout=layout, wtype=wtype,
                group_size=group_size)


def gen_w4a8(M: int, N: int, K: int, group_size: int = -1, layout: int = NK_EXLLAMA,
             seed: int = 0) -> dict:
    """CPU tensors for one W4A8 (QQQ-style) problem.

    a [M,K] int8 U{-127..127}; s_tok [M] fp32 U[0.01,0.05]; w int4 words
    (two's complement nibbles, U{-8..7}); s_ch [N] fp32 U[0.001,0.01];
    sg [G,N] int8 U{1..16} when group_size == 128, else None.
    """
    g = _gen(seed)
    a = torch.randint(-127, 128, (M, K), generator=g, dtype=torch.int32).to(torch.int8)
    s_tok = uniform((M,), 0.01, 0.05, g, torch.float32)
    w = random_words(packed_shape(layout, K, N), g)
    s_ch = uniform((N,), 0.001, 0.01, g, torch.float32)
    sg = None
    if group_size not in (-1, K):
        sg = torch.randint(1, 17, (K // group_size, N), generator=g,
                           dtype=torch.int32).to(torch.int8)
    return dict(a=a, s_tok=s_tok, w=w, s_ch=s_ch, sg=sg, M=M, N=N, K=K, layout=layout,
                wtype=INT4, group_size=group_size)


def gen_w4a8_fp8(M: int, N: int, K: int, layout: int = NK_EXLLAMA, seed: int = 0) -> dict:
    """CPU tensors for one W4A8 problem with fp8 activations: a [M,K] E4M3
    codes (uint8) drawn uniformly from the 254 finite codes (0x7F and 0xFF,
    the NaNs, are replaced by their neighbours 0x7E, 0xFE); s_tok [M] fp32
    U[0.01,0.05]; int4 weight words; s_ch [N] fp32 U[0.001,0.01].  Per-channel
    only."""
    g = _gen(seed)
    codes = torch.randint(0, 256, (M, K), generator=g, dtype=torch.int32)
    codes = torch.where((codes & 0x7F) == 0x7F, codes - 1, codes).to(torch.uint8)
    s_tok = uniform((M,), 0.01, 0.05, g, torch.float32)
    w = random_words(packed_shape(layout, K, N), g)
    s_ch = uniform((N,), 0.001, 0.01, g, torch.float32)
    return dict(a=codes, s_tok=s_tok, w=w, s_ch=s_ch, M=M, N=N, K=K, layout=layout, wtype=INT4,
                group_size=-1)


def gen_act16(M: int, K: int, dtype=torch.float16, seed: int = 0) -> torch.Tensor:
    """Activations [M, K] ~ N(0, 1) in fp16 / bf16 (the W4A16 activation
    distribution): the input of the per-token int8 quantization."""
    return torch.randn(M, K, generator=_gen(seed)).to(dtype)


def tiny_w4a16(seed: int = 0) -> dict:
    """The tiny W4A16 case: fp16 [16,512] x uint4b8 [512,256], g128."""
    return gen_w4a16(16, 256, 512, act_dtype=torch.float16, wtype=UINT4B8,
                     layout=NK_EXLLAMA, group_size=128, zeros=False, seed=seed)
