"""CPU oracle for the 4-bit-weight mixed-precision GEMM (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product library never imports,
links or runs anything here, and the two share no code.

The arithmetic lives in plain C (``w4_oracle.c``: fp64 sums with k
ascending, int64 integer sums, OpenMP across output elements); this module
only marshals numpy / torch CPU arrays into it.  Conversions of fp16 / bf16
inputs to fp64 are exact.

What each function computes, and the page it follows:

* ``unpack`` / ``pack`` / ``nibble`` — the three input layouts.  ExLlama
  shuffle: vLLM API page "rdna_hybrid_w4a16", ``pack_int4_exllama_shuffle``.
  Sequential layouts (K-value j at bits 4j) are a reading.
* ``value`` — uint4b8 is q-8 (ZP_BIAS 8 on the same page), uint4 is q,
  int4 is the two's complement nibble.
* ``w4a16`` / ``w4a16_elems`` — Machete Readme, "Overview":
  w_hat = w_q * w_s - w_z (pre-scaled zero-point), out = a x w_hat.
* ``w4a8`` / ``w4a8_elems`` / ``w4a8_scale`` — pytorch/ao PR #1113
  "support W4A8 Marlin kernel": int8 x int4 (per-channel) or int8 x
  (int4 * group scale) (per-group), exact integer accumulator, then
  acc * s_tok[m] * s_ch[n].
* ``e4m3_decode`` / ``e4m3_encode`` / ``quant_per_token_fp8`` / ``w4a8_fp8``
  — the fp8 activations of vLLM PR #9855 ("including fp8 activations"),
  read as OCP E4M3 (bias 7, largest value 448, no infinity): decoding,
  round-to-nearest-even encoding saturated at 448, per-token scales
  amax/448, and the exact fp64 product of decoded activations with int4
  weights.
* ``add_bias`` — the vLLM API page "rdna_hybrid_w4a16",
  ``_rdna_hybrid_w4a16_apply_impl``: the layer bias added to the product.
* ``quant_per_token`` — vLLM PR #6547 "Enable Dynamic Per Token fp8" (one
  activation scale per token, computed from that token at run time) with
  the symmetric int8 activations of pytorch/ao PR #1113: s = amax/127 and
  q = round-half-even(a/s) in fp32 (the formula is a reading; the pages
  print none).

Every function is pinned by ``tests/test_oracle_pins.py``; none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

KN_SEQ, NK_SEQ, NK_EXLLAMA = 0, 1, 2
UINT4B8, UINT4, INT4 = 0, 1, 2

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile w4_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.or_nibble.argtypes = [p, i32, i64, i64, i64, i64]
            lib.or_nibble.restype = i32
            lib.or_unpack.argtypes = [p, i32, i64, i64, p]
            lib.or_pack.argtypes = [p, i32, i64, i64, p]
            lib.or_value.argtypes = [i32, i32]
            lib.or_value.restype = i32
            lib.or_w4a16.argtypes = [i64, i64, i64, p, p, i32, i32, p, p, i64, p, p]
            lib.or_w4a16_elems.argtypes = [i64, i64, i64, p, p, i32, i32, p, p, i64, i64, p, p, p, p]
            lib.or_w4a8.argtypes = [i64, i64, i64, p, p, i32, i32, p, i64, p]
            lib.or_w4a8_elems.argtypes = [i64, i64, i64, p, p, i32, i32, p, i64, i64, p, p, p]
            lib.or_w4a8_scale.argtypes = [i64, p, p, p, p, p, p]
            lib.or_quant_per_token.argtypes = [i64, i64, p, p, p]
            lib.or_e4m3_decode_n.argtypes = [i64, p, p]
            lib.or_e4m3_encode_n.argtypes = [i64, p, p]
            lib.or_quant_per_token_fp8.argtypes = [i64, i64, p, p, p]
            lib.or_w4a8_fp8.argtypes = [i64, i64, i64, p, p, i32, i32, p, p]
            lib.or_num_threads.restype = i32
            _lib = lib
    return _lib


def _np(x, dtype):
    """CPU numpy copy in `dtype` (exact for fp16/bf16 -> float64)."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if dtype == np.float64:
                x = x.to(torch.float64)
            return np.ascontiguousarray(x.numpy().astype(dtype, copy=False))
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x).astype(dtype, copy=False))


def _ptr(arr):
    return None if arr is None else arr.ctypes.data


def num_threads() -> int:
    return int(_load().or_num_threads())


def value(q: int, wtype: int) -> int:
    return int(_load().or_value(int(q), int(wtype)))


def nibble(w, layout: int, K: int, N: int, k: int, n: int) -> int:
    w = _np(w, np.int32)
    return int(_load().or_nibble(_ptr(w), layout, K, N, k, n))


def unpack(w, layout: int, K: int, N: int) -> np.ndarray:
    """Logical nibbles q[K, N] (uint8, 0..15) from packed words."""
    w = _np(w, np.int32)
    q = np.empty((K, N), dtype=np.uint8)
    _load().or_unpack(_ptr(w), layout, K, N, _ptr(q))
    return q


def pack(q, layout: int) -> np.ndarray:
    """Pack logical nibbles q[K, N] into int32 words of `layout`."""
    q = _np(q, np.uint8)
    K, N = q.shape
    shape = (K // 8, N) if layout == KN_SEQ else (N, K // 8)
    w = np.empty(shape, dtype=np.int32)
    _load().or_pack(_ptr(q), layout, K, N, _ptr(w))
    return w


def w4a16(a, w, layout, wtype, s, z, group_size, K, N):
    """fp64 reference and sum of |terms|, each [M, N]."""
    a = _np(a, np.float64)
    M = a.shape[0]
    w = _np(w, np.int32)
    s = _np(s, np.float64)
    z = None if z is None else _np(z, np.float64)
    gs = K if group_size in (-1, None) else group_size
    ref = np.empty((M, N), np.float64)
    absref = np.empty((M, N), np.float64)
    _load().or_w4a16(M, N, K, _ptr(a), _ptr(w), layout, wtype, _ptr(s), _ptr(z), gs,
                     _ptr(ref), _ptr(absref))
    return ref, absref


def w4a16_elems(a, w, layout, wtype, s, z, group_size, K, N, rows, cols):
    a = _np(a, np.float64)
    M = a.shape[0]
    w = _np(w, np.int32)
    s = _np(s, np.float64)
    z = None if z is None else _np(z, np.float64)
    rows = _np(rows, np.int64)
    cols = _np(cols, np.int64)
    gs = K if group_size in (-1, None) else group_size
    ref = np.empty(rows.shape[0], np.float64)
    absref = np.empty(rows.shape[0], np.float64)
    _load().or_w4a16_elems(M, N, K, _ptr(a), _ptr(w), layout, wtype, _ptr(s), _ptr(z), gs,
                           rows.shape[0], _ptr(rows), _ptr(cols), _ptr(ref), _ptr(absref))
    return ref, absref


def w4a8(a, w, layout, wtype, sg, group_size, K, N):
    """Exact int64 accumulator [M, N]."""
    a = _np(a, np.int8)
    M = a.shape[0]
    w = _np(w, np.int32)
    sg = None if sg is None else _np(sg, np.int8)
    gs = K if group_size in (-1, None) else group_size
    acc = np.empty((M, N), np.int64)
    _load().or_w4a8(M, N, K, _ptr(a), _ptr(w), layout, wtype, _ptr(sg), gs, _ptr(acc))
    return acc


def w4a8_elems(a, w, layout, wtype, sg, group_size, K, N, rows, cols):
    a = _np(a, np.int8)
    M = a.shape[0]
    w = _np(w, np.int32)
    sg = None if sg is None else _np(sg, np.int8)
    rows = _np(rows, np.int64)
    cols = _np(cols, np.int64)
    gs = K if group_size in (-1, None) else group_size
    acc = np.empty(rows.shape[0], np.int64)
    _load().or_w4a8_elems(M, N, K, _ptr(a), _ptr(w), layout, wtype, _ptr(sg), gs,
                          rows.shape[0], _ptr(rows), _ptr(cols), _ptr(acc))
    return acc


def w4a8_scale(acc, rows, cols, s_tok, s_ch):
    """fp64 acc * s_tok[rows] * s_ch[cols] for flat (acc, rows, cols) lists."""
    acc = _np(acc, np.int64).reshape(-1)
    rows = _np(rows, np.int64).reshape(-1)
    cols = _np(cols, np.int64).reshape(-1)
    s_tok = _np(s_tok, np.float64)
    s_ch = _np(s_ch, np.float64)
    ref = np.empty(acc.shape[0], np.float64)
    _load().or_w4a8_scale(acc.shape[0], _ptr(acc), _ptr(rows), _ptr(cols), _ptr(s_tok),
                          _ptr(s_ch), _ptr(ref))
    return ref


def add_bias(ref, cols, bias):
    """The bias step after the product: ref[i] + bias[cols[i]] in fp64 (the
    bias, fp16 / bf16, converted exactly).  vLLM API page "rdna_hybrid_w4a16",
    _rdna_hybrid_w4a16_apply_impl: the layer bias is added to the GEMM
    result.  Works on flat (ref, cols) lists or on a full [M, N] ref (cols
    None)."""
    ref = np.asarray(ref, dtype=np.float64)
    b = _np(bias, np.float64).reshape(-1)
    if cols is None:
        return ref + b[np.newaxis, :]
    return ref + b[_np(cols, np.int64).reshape(-1)]


def quant_per_token(a):
    """Per-token int8 codes [M, K] and fp32 scales [M] of fp16/bf16/fp32
    activations a [M, K] (converted to fp32 exactly)."""
    try:
        import torch

        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().to(torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    M, K = a.shape
    q = np.empty((M, K), np.int8)
    s = np.empty(M, np.float32)
    _load().or_quant_per_token(M, K, _ptr(a), _ptr(q), _ptr(s))
    return q, s


def _f32(a):
    try:
        import torch

        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().to(torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of E4M3 codes (uint8 array of any shape; NaN for 0x7F/0xFF)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, np.float64)
    _load().or_e4m3_decode_n(c.size, _ptr(c), _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of finite fp32 values, nearest-even, saturated at 448."""
    x = _f32(x)
    out = np.empty(x.shape, np.uint8)
    _load().or_e4m3_encode_n(x.size, _ptr(x), _ptr(out))
    return out


def quant_per_token_fp8(a):
    """Per-token E4M3 codes [M, K] (uint8) and fp32 scales [M]."""
    a = _f32(a)
    M, K = a.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty(M, np.float32)
    _load().or_quant_per_token_fp8(M, K, _ptr(a), _ptr(q), _ptr(s))
    return q, s


def w4a8_fp8(a_codes, w, layout, wtype, K, N):
    """Exact fp64 sum_k decode(a) * v(q) [M, N] and the sum of |terms|."""
    a = np.ascontiguousarray(np.asarray(a_codes, dtype=np.uint8))
    M = a.shape[0]
    w = _np(w, np.int32)
    ref = np.empty((M, N), np.float64)
    absref = np.empty((M, N), np.float64)
    _load().or_w4a8_fp8(M, N, K, _ptr(a), _ptr(w), layout, wtype, _ptr(ref), _ptr(absref))
    return ref, absref
