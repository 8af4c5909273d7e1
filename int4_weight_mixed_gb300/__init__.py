"""int4_weight_mixed_gb300 — Python binding of libw4 (GB300 4-bit-weight GEMM).

Argument marshalling only: every step of the product runs in libw4's CUDA
kernels.  PyTorch supplies device memory (outputs, workspaces) and the
current stream.  There is no CPU fallback: if libw4.so is missing or cannot
be loaded, every call raises.

    b = prepack_B(w_q, wtype, layout, K, N)          # once per weight
    out = gemm(a, b, wtype, N, scales=s, zeros=z, group_size=128)

Names follow the C ABI in include/w4.h (w4_prepack_B, w4_gemm, ...), which
follows the Machete Readme "API" section (prepack, then gemm with b_type,
b_scales, b_group_size, and an optional schedule).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build_lib

UINT4B8, UINT4, INT4 = 0, 1, 2
KN_SEQ, NK_SEQ, NK_EXLLAMA = 0, 1, 2
F16, BF16, S8, S32, E4M3 = 0, 1, 2, 3, 4
OK, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)

_DTYPE_CODE = {torch.float16: F16, torch.bfloat16: BF16, torch.int8: S8, torch.int32: S32,
               torch.float8_e4m3fn: E4M3}
_CODE_DTYPE = {v: k for k, v in _DTYPE_CODE.items()}

_lib = None
_lock = threading.Lock()
_ws_cache: dict = {}


class W4Error(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}: {message}")


def library_path() -> str:
    return _build_lib.LIB


def build(force: bool = False) -> str:
    """Compile libw4.so for sm_103a in-tree (see _build_lib.py)."""
    return _build_lib.build(force=force)


def load():
    """Load libw4.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libw4.so not found at {path}: the CUDA extension is missing; "
                "run __graft_entry__.build() or python -m int4_weight_mixed_gb300._build_lib")
        lib = ctypes.CDLL(path)
        i64, i32, p, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        lib.w4_layout_version.restype = i32
        lib.w4_prepacked_size.argtypes = [i64, i64]
        lib.w4_prepacked_size.restype = sz
        lib.w4_prepack_B.argtypes = [p, i32, i32, i64, i64, p, p]
        lib.w4_prepack_B.restype = i32
        lib.w4_unprepack_B.argtypes = [p, i32, i32, i64, i64, p, p]
        lib.w4_unprepack_B.restype = i32
        lib.w4_gemm_workspace_size.argtypes = [i64, i64, i64, i32, i64]
        lib.w4_gemm_workspace_size.restype = sz
        gemm_args = [p, i32, i64, i64, p, i32, i64, p, i32, p, i64, p, p, p, i32, p, sz, p]
        lib.w4_gemm.argtypes = gemm_args
        lib.w4_gemm.restype = i32
        lib.w4_gemm_ex.argtypes = gemm_args + [i32]
        lib.w4_gemm_ex.restype = i32
        lib.w4_gemm_bias.argtypes = gemm_args[:13] + [p] + gemm_args[13:] + [i32]
        lib.w4_gemm_bias.restype = i32
        lib.w4_num_schedules.restype = i32
        lib.w4_schedule_name.argtypes = [i32]
        lib.w4_schedule_name.restype = ctypes.c_char_p
        lib.w4_default_schedule.argtypes = [i64, i64, i64, i32, i64]
        lib.w4_default_schedule.restype = i32
        lib.w4_override_schedule.argtypes = [i32, i64, i64, i64, i64, i64, i32]
        lib.w4_override_schedule.restype = i32
        lib.w4_quantize_per_token.argtypes = [p, i32, i64, i64, p, p, p]
        lib.w4_quantize_per_token.restype = i32
        lib.w4_gemm_dynamic_workspace_size.argtypes = [i64, i64, i64, i32, i64]
        lib.w4_gemm_dynamic_workspace_size.restype = sz
        lib.w4_gemm_dynamic.argtypes = [p, i32, i64, i64, p, i32, i64, p, i32, i64, p, i32, p,
                                        p, p, p, sz, p]
        lib.w4_gemm_dynamic.restype = i32
        lib.w4_quantize_per_token_fp8.argtypes = [p, i32, i64, i64, p, p, p]
        lib.w4_quantize_per_token_fp8.restype = i32
        lib.w4_check_status.argtypes = [p, sz, p]
        lib.w4_check_status.restype = i32
        lib.w4_status_string.argtypes = [i32]
        lib.w4_status_string.restype = ctypes.c_char_p
        lib.w4_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().w4_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise W4Error(status, where, load().w4_last_error().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dense_on(device, **tensors):
    """The kernels read every array densely from its first element: each
    given tensor must be a contiguous CUDA tensor on `device`."""
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda or t.device != device:
            raise ValueError(f"{name} must be a CUDA tensor on {device} (got {t.device})")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def layout_version() -> int:
    return load().w4_layout_version()


def prepacked_size(K: int, N: int) -> int:
    return int(load().w4_prepacked_size(K, N))


def prepack_B(w_q: torch.Tensor, wtype: int, layout: int, K: int, N: int,
              out: torch.Tensor | None = None) -> torch.Tensor:
    """w4_prepack_B: packed int32 words (device) -> prepacked uint8 buffer."""
    lib = load()
    assert w_q.dtype == torch.int32 and w_q.is_cuda and w_q.is_contiguous()
    _dense_on(w_q.device, out=out)
    nbytes = prepacked_size(K, N)
    if out is None:
        out = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=w_q.device)
    _check(lib.w4_prepack_B(_ptr(w_q), wtype, layout, K, N, _ptr(out), _stream(w_q.device)),
           "w4_prepack_B")
    return out


def unprepack_B(b_packed: torch.Tensor, wtype: int, layout: int, K: int, N: int) -> torch.Tensor:
    lib = load()
    _dense_on(b_packed.device, b_packed=b_packed)
    shape = (K // 8, N) if layout == KN_SEQ else (N, K // 8)
    w_q = torch.empty(shape, dtype=torch.int32, device=b_packed.device)
    _check(lib.w4_unprepack_B(_ptr(b_packed), wtype, layout, K, N, _ptr(w_q),
                              _stream(b_packed.device)), "w4_unprepack_B")
    return w_q


def workspace_size(M: int, N: int, K: int, a_dtype: torch.dtype, group_size: int) -> int:
    return int(load().w4_gemm_workspace_size(M, N, K, _DTYPE_CODE[a_dtype], group_size))


def workspace(device, nbytes: int) -> torch.Tensor:
    """A zero-filled workspace of at least nbytes, cached per (device, stream).

    Calls on the same stream are ordered, so sharing is safe; the library
    leaves its counters at zero after every call.  Not available while the
    stream is capturing a CUDA graph: an allocation there would come from the
    graph's private pool and its zero-fill would be recorded into the graph,
    so callers that capture pass a workspace allocated beforehand."""
    dev = torch.device(device)
    if torch.cuda.is_current_stream_capturing():
        raise RuntimeError("w4: pass ws= (allocated before capture) to calls captured in a "
                           "CUDA graph")
    key = (dev.index, _stream(dev))
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        _ws_cache[key] = ws
    return ws


def num_schedules() -> int:
    return load().w4_num_schedules()


def schedule_names() -> list:
    lib = load()
    return [lib.w4_schedule_name(i).decode() for i in range(lib.w4_num_schedules())]


def default_schedule(M: int, N: int, K: int, a_dtype: torch.dtype, group_size: int) -> int:
    return load().w4_default_schedule(M, N, K, _DTYPE_CODE[a_dtype], group_size)


def override_schedule(a_dtype: torch.dtype, m_lo: int, m_hi: int, N: int, K: int,
                      group_size: int, schedule) -> None:
    """w4_override_schedule: problems of this shape with M in [m_lo, m_hi]
    run `schedule` (index or name) by default; None / -1 removes the entry."""
    if schedule is None:
        schedule = -1
    elif isinstance(schedule, str):
        schedule = schedule_names().index(schedule)
    _check(load().w4_override_schedule(_DTYPE_CODE[a_dtype], m_lo, m_hi, N, K, group_size,
                                       schedule), "w4_override_schedule")


def autotune(a: torch.Tensor, b_packed: torch.Tensor, wtype: int, N: int, install: bool = True,
             reps: int = 20, **kw) -> dict:
    """Time every schedule that can run this problem (the arguments of
    gemm()) with CUDA events on the current stream, and, with install=True,
    make the fastest the default for exactly this shape (w4_override_schedule
    for this M).  Returns {schedule name: microseconds per call}.  The calls
    write `out` (or a scratch output) and use `ws` (or the cached workspace)."""
    M, K = a.shape
    names = schedule_names()
    kw = dict(kw)
    kw.pop("schedule", None)
    group_size = kw.get("group_size", -1)
    if kw.get("ws") is None:
        kw["ws"] = workspace(a.device, workspace_size(M, N, K, a.dtype, group_size))
    times = {}
    stream = torch.cuda.current_stream(a.device)
    for si, name in enumerate(names):
        if name == "simt" and M * N * K > (1 << 31):
            continue  # the CUDA-core schedule is a correctness path
        try:
            gemm(a, b_packed, wtype, N, schedule=si, **kw)  # warm-up; UNSUPPORTED -> skip
        except W4Error as e:
            if e.status == ERR_UNSUPPORTED:
                continue
            raise
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            gemm(a, b_packed, wtype, N, schedule=si, **kw)
        e1.record(stream)
        e1.synchronize()
        times[name] = e0.elapsed_time(e1) * 1e3 / reps
    if install and times:
        best = min(times, key=times.get)
        override_schedule(a.dtype, M, M, N, K, group_size, best)
    return times


def gemm(a: torch.Tensor, b_packed: torch.Tensor, wtype: int, N: int,
         scales: torch.Tensor | None = None, zeros: torch.Tensor | None = None,
         group_size: int = -1, token_scales: torch.Tensor | None = None,
         channel_scales: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
         out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
         schedule: int = -1, bias: torch.Tensor | None = None) -> torch.Tensor:
    """w4_gemm_ex / w4_gemm_bias: out[M,N] = a[M,K] x dequant(W) (+ bias).

    W4A16: a fp16/bf16, scales [G,N] of a's dtype, zeros [G,N] pre-scaled or
    None.  W4A8: a int8, scales = int8 group scales [G,N] or None
    (per-channel), token_scales [M] and channel_scales [N] fp32 for fp16
    output, or out_dtype=torch.int32 for the raw accumulator.  bias: [N] of
    the output dtype, added before the output rounding, or None.
    """
    lib = load()
    _dense_on(a.device, a=a, b_packed=b_packed, scales=scales, zeros=zeros,
              token_scales=token_scales, channel_scales=channel_scales, out=out, ws=ws,
              bias=bias)
    M, K = a.shape
    a_code = _DTYPE_CODE[a.dtype]
    if out_dtype is None:
        out_dtype = torch.float16 if a.dtype in (torch.int8, torch.float8_e4m3fn) else a.dtype
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    if ws is None:  # (a given workspace is checked against the plan by the library)
        ws = workspace(a.device, workspace_size(M, N, K, a.dtype, group_size))
    scale_code = _DTYPE_CODE[scales.dtype] if scales is not None else a_code
    if bias is None:
        st = lib.w4_gemm_ex(_ptr(a), a_code, M, K, _ptr(b_packed), wtype, N, _ptr(scales),
                            scale_code, _ptr(zeros), group_size, _ptr(token_scales),
                            _ptr(channel_scales), _ptr(out), _DTYPE_CODE[out_dtype], _ptr(ws),
                            ws.numel(), _stream(a.device), schedule)
        _check(st, "w4_gemm")
    else:
        if bias.dtype != out_dtype or bias.numel() != N:
            raise ValueError(f"bias must be [{N}] of {out_dtype}")
        st = lib.w4_gemm_bias(_ptr(a), a_code, M, K, _ptr(b_packed), wtype, N, _ptr(scales),
                              scale_code, _ptr(zeros), group_size, _ptr(token_scales),
                              _ptr(channel_scales), _ptr(bias), _ptr(out),
                              _DTYPE_CODE[out_dtype], _ptr(ws), ws.numel(), _stream(a.device),
                              schedule)
        _check(st, "w4_gemm_bias")
    return out


def gemm_dynamic(a: torch.Tensor, b_packed: torch.Tensor, wtype: int, N: int,
                 act_dtype: torch.dtype = torch.int8, scales: torch.Tensor | None = None,
                 group_size: int = -1, channel_scales: torch.Tensor | None = None,
                 bias: torch.Tensor | None = None, out: torch.Tensor | None = None,
                 token_scales_out: torch.Tensor | None = None,
                 ws: torch.Tensor | None = None) -> torch.Tensor:
    """w4_gemm_dynamic: fp16/bf16 activations quantized per token to int8
    (act_dtype torch.int8) or E4M3 (torch.float8_e4m3fn) inside the call,
    then the W4A8 product; fp16 out [M, N]."""
    lib = load()
    _dense_on(a.device, a=a, b_packed=b_packed, scales=scales, channel_scales=channel_scales,
              bias=bias, out=out, token_scales_out=token_scales_out, ws=ws)
    M, K = a.shape
    act = _DTYPE_CODE[act_dtype]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=a.device)
    if ws is None:  # (a given workspace is checked against the plan by the library)
        ws = workspace(a.device, int(lib.w4_gemm_dynamic_workspace_size(M, N, K, act, group_size)))
    scale_code = _DTYPE_CODE[scales.dtype] if scales is not None else S8
    _check(lib.w4_gemm_dynamic(_ptr(a), _DTYPE_CODE[a.dtype], M, K, _ptr(b_packed), wtype, N,
                               _ptr(scales), scale_code, group_size, _ptr(channel_scales), act,
                               _ptr(bias), _ptr(out), _ptr(token_scales_out), _ptr(ws),
                               ws.numel(), _stream(a.device)), "w4_gemm_dynamic")
    return out


def quantize_per_token(a: torch.Tensor, out: torch.Tensor | None = None,
                       scales: torch.Tensor | None = None):
    """w4_quantize_per_token: fp16/bf16 activations [M, K] -> (int8 codes
    [M, K], fp32 per-token scales [M]), the `a` and `token_scales` of a
    W4A8 gemm."""
    lib = load()
    assert a.dim() == 2 and a.is_cuda and a.is_contiguous()
    M, K = a.shape
    if out is None:
        out = torch.empty(M, K, dtype=torch.int8, device=a.device)
    if scales is None:
        scales = torch.empty(M, dtype=torch.float32, device=a.device)
    assert out.dtype == torch.int8 and out.is_contiguous() and out.shape == (M, K)
    assert scales.dtype == torch.float32 and scales.is_contiguous() and scales.numel() == M
    _check(lib.w4_quantize_per_token(_ptr(a), _DTYPE_CODE[a.dtype], M, K, _ptr(out), _ptr(scales),
                                     _stream(a.device)), "w4_quantize_per_token")
    return out, scales


def quantize_per_token_fp8(a: torch.Tensor, out: torch.Tensor | None = None,
                           scales: torch.Tensor | None = None):
    """w4_quantize_per_token_fp8: fp16/bf16 activations [M, K] -> (E4M3
    codes [M, K] as torch.float8_e4m3fn, fp32 per-token scales [M]), the `a`
    and `token_scales` of a W4A8 gemm with fp8 activations."""
    lib = load()
    assert a.dim() == 2 and a.is_cuda and a.is_contiguous()
    M, K = a.shape
    if out is None:
        out = torch.empty(M, K, dtype=torch.float8_e4m3fn, device=a.device)
    if scales is None:
        scales = torch.empty(M, dtype=torch.float32, device=a.device)
    assert out.dtype in (torch.float8_e4m3fn, torch.uint8) and out.is_contiguous()
    assert out.shape == (M, K)
    assert scales.dtype == torch.float32 and scales.is_contiguous() and scales.numel() == M
    _check(lib.w4_quantize_per_token_fp8(_ptr(a), _DTYPE_CODE[a.dtype], M, K, _ptr(out),
                                         _ptr(scales), _stream(a.device)),
           "w4_quantize_per_token_fp8")
    return out, scales


def check_status(ws: torch.Tensor) -> int:
    """w4_check_status: sync and report a device-side timeout recorded in ws."""
    return load().w4_check_status(_ptr(ws), ws.numel(), _stream(ws.device))
