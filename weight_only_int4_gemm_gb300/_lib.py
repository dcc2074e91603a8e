"""ctypes binding of ``libw4a16.so``: argument marshalling only.

Every function here has the name of the C entry point it wraps, takes torch
tensors (device memory and streams come from PyTorch), checks dtypes and
shapes enough to build the call, and raises ``W4A16Error`` on a non-OK
status.  All arithmetic happens in the library's CUDA kernels; there is no
fallback of any kind -- if the library is missing, loading fails loudly.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")
GROUP = 128

PATH_AUTO, PATH_SKINNY, PATH_TCGEN05 = -1, 0, 1
EPI_NONE, EPI_BIAS, EPI_SILU_MUL = 0, 1, 2
PATH_NAMES = {PATH_SKINNY: "skinny", PATH_TCGEN05: "tcgen05"}

_STATUS = {0: "W4A16_OK", 1: "W4A16_ERR_NULL", 2: "W4A16_ERR_SHAPE", 3: "W4A16_ERR_ALIGN",
           4: "W4A16_ERR_UNSUPPORTED", 5: "W4A16_ERR_WORKSPACE", 6: "W4A16_ERR_CUDA",
           7: "W4A16_ERR_TIMEOUT", 8: "W4A16_ERR_BOUNDS"}

# (name, restype, argtypes) of every exported symbol, in header order.
_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "w4a16_packed_bytes": (_S, [_I, _I, _I, _I]),
    "w4a16_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "w4a16_pack": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "w4a16_gemm": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _S, _P]),
    "w4a16_gemm_fused": (_I, [_P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _S, _P]),
    "w4a16_gemm_path": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _S, _I, _P]),
    "w4a16_dequant_ref": (_I, [_P, _P, _I, _P, _I, _I, _I, _P]),
    "w4a16_gemm_static_scratch": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P]),
    "w4a16_select_path": (_I, [_I, _I, _I]),
    "w4a16_kernel_name": (ctypes.c_char_p, [_I, _I, _I]),
    "w4a16_debug_forced_timeout": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _S, _I, _P]),
    "w4a16_device_status": (_I, [_I]),
    "w4a16_packed_check": (_I, [_P, _I, _I, _I, _I, _P]),
    "w4a16_quantize_rtn": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "w4a16_grouped_workspace_bytes": (_S, [_I, _I, _I, _I, _I, _I]),
    "w4a16_gemm_grouped": (_I, [_P, _P, _I, _I, _P, _P, _I, _P, _I, _I, _I, _I, _P, _S, _P]),
    "w4a16_status_string": (ctypes.c_char_p, [_I]),
    "w4a16_debug_build": (_I, []),
    "w4a16_gemm_f16": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _S, _P]),
    "w4a16_gemm_f16_path": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _S, _I, _P]),
    "w4a16_dequant_ref_f16": (_I, [_P, _P, _I, _P, _I, _I, _I, _P]),
    "w4a16_debug_shrink_code_bound": (_I, [_S]),
    "w4a16_describe_plan": (_I, [_I, _I, _I, _I, _I, _P]),
    # include/w8a8_fp8.h
    "w8a8_fp8_quantize_act": (_I, [_P, _I, _I, _P, _P, _P]),
    "w8a8_fp8_quantize_weight": (_I, [_P, _I, _I, _P, _P, _P]),
    "w8a8_fp8_packed_bytes": (_S, [_I, _I]),
    "w8a8_fp8_pack_weight": (_I, [_P, _I, _I, _P, _P]),
    "w8a8_fp8_workspace_bytes": (_S, [_I, _I, _I]),
    "w8a8_fp8_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _S, _P]),
}


class W4A16Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)} ({msg})")
        self.status = status


_lock = threading.Lock()
_lib = None
_debug_lib = None
DEBUG_LIB_PATH = os.path.join(_HERE, "libw4a16_debug.so")


_active = threading.local()


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built); inside
    `debug_library()` the debug build instead."""
    lib = getattr(_active, "lib", None)
    if lib is not None:
        return lib
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {LIB_PATH} is missing "
                "(run __graft_entry__.build() or python -m weight_only_int4_gemm_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def load_debug() -> ctypes.CDLL:
    """The debug build of the library (W4A16_DEBUG: device-side bounds checks
    that report W4A16_ERR_BOUNDS through w4a16_device_status), with the same
    C ABI; raises if it has not been built (build.build_library(debug=True))."""
    global _debug_lib
    with _lock:
        if _debug_lib is not None:
            return _debug_lib
        if not os.path.exists(DEBUG_LIB_PATH):
            raise RuntimeError(f"debug library not built: {DEBUG_LIB_PATH} is missing")
        lib = ctypes.CDLL(DEBUG_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _debug_lib = lib
        return lib


@contextlib.contextmanager
def debug_library():
    """Route this thread's calls of the binding to the debug build."""
    prev = getattr(_active, "lib", None)
    _active.lib = load_debug()
    try:
        yield _active.lib
    finally:
        _active.lib = prev


def _check(fn: str, status: int):
    if status != 0:
        msg = load().w4a16_status_string(status).decode()
        raise W4A16Error(fn, status, msg)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")


def w4a16_packed_bytes(K: int, N: int, has_zeros: bool) -> int:
    return int(load().w4a16_packed_bytes(K, N, GROUP, 1 if has_zeros else 0))


def w4a16_workspace_bytes(B: int, K: int, N: int) -> int:
    v = int(load().w4a16_workspace_bytes(B, K, N, GROUP))
    if v == ctypes.c_size_t(-1).value:
        raise ValueError(f"invalid shape B={B} K={K} N={N}")
    return v


def w4a16_select_path(B: int, K: int, N: int) -> int:
    return int(load().w4a16_select_path(B, K, N))


class PlanInfo(ctypes.Structure):
    """w4a16_plan_info (include/w4a16.h)."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "kernel", "batch_rows", "batch_tiles", "col_tiles", "k_splits", "groups_per_split",
        "grid", "ctas_per_sm", "issuers", "acc_buffers", "tile_slots", "x_slots", "code_slots",
        "block_rows", "tmem_cols")] + [("smem_bytes", ctypes.c_size_t),
                                       ("workspace_bytes", ctypes.c_size_t)]


KERNEL_NAMES = {0: "skinny_kernel", 1: "tc_kernel", 2: "wide_kernel"}


def w4a16_describe_plan(B: int, K: int, N: int, num_sms: int = 0) -> dict:
    """The launch plan of w4a16_gemm for (B, K, N): for the current device
    (num_sms = 0) or, without a device, for one with num_sms SMs."""
    info = PlanInfo()
    _check("w4a16_describe_plan",
           load().w4a16_describe_plan(B, K, N, GROUP, num_sms, ctypes.addressof(info)))
    d = {name: getattr(info, name) for name, _ in PlanInfo._fields_}
    d["kernel_name"] = KERNEL_NAMES[d["kernel"]]
    return d


def w4a16_kernel_name(B: int, K: int, N: int) -> str:
    return load().w4a16_kernel_name(B, K, N).decode()


def w4a16_pack(qweight: torch.Tensor, qzeros: torch.Tensor | None = None, *,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Repack canonical codes (int32 [K/8][N]) and zeros (int32 [K/128][N/8])."""
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    _need(qweight, torch.int32, (K // 8, N), "qweight")
    if qzeros is not None:
        _need(qzeros, torch.int32, (K // GROUP, N // 8), "qzeros")
    nbytes = w4a16_packed_bytes(K, N, qzeros is not None)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=qweight.device)
    _check("w4a16_pack", load().w4a16_pack(
        qweight.data_ptr(), None if qzeros is None else qzeros.data_ptr(), K, N, GROUP,
        out.data_ptr(), _stream(stream)))
    return out


class Workspace:
    """A zero-filled device workspace per device, grown on demand."""

    def __init__(self):
        self._bufs: dict[int, torch.Tensor] = {}

    def get(self, nbytes: int, device: torch.device) -> torch.Tensor | None:
        if nbytes == 0:
            return None
        idx = device.index if device.index is not None else torch.cuda.current_device()
        buf = self._bufs.get(idx)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
            self._bufs[idx] = buf
        return buf


_default_ws = Workspace()


def w4a16_gemm(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, has_zeros: bool,
               N: int | None = None, *, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, path: int = PATH_AUTO,
               stream=None) -> torch.Tensor:
    """y[B][N] = x[B][K] . dequant(packed, scales)."""
    B, K = x.shape
    N = scales.shape[1] if N is None else N
    _need(x, torch.bfloat16, (B, K), "x")
    _need(scales, torch.bfloat16, (K // GROUP, N), "scales")
    if packed.numel() * packed.element_size() < w4a16_packed_bytes(K, N, has_zeros):
        raise ValueError("packed: too small for this shape")
    if out is None:
        out = torch.empty((B, N), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (B, N), "out")
    need = w4a16_workspace_bytes(B, K, N)
    if workspace is None:
        workspace = _default_ws.get(need, x.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load()
    if path == PATH_AUTO:
        st = lib.w4a16_gemm(x.data_ptr(), packed.data_ptr(), scales.data_ptr(),
                            1 if has_zeros else 0, out.data_ptr(), B, K, N, GROUP,
                            ws_ptr, ws_bytes, _stream(stream))
        _check("w4a16_gemm", st)
    else:
        st = lib.w4a16_gemm_path(x.data_ptr(), packed.data_ptr(), scales.data_ptr(),
                                 1 if has_zeros else 0, out.data_ptr(), B, K, N, GROUP,
                                 ws_ptr, ws_bytes, int(path), _stream(stream))
        _check("w4a16_gemm_path", st)
    return out


def w4a16_gemm_f16(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, has_zeros: bool,
                   N: int | None = None, *, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, path: int = PATH_AUTO,
                   stream=None) -> torch.Tensor:
    """fp16-activation variant: y[B][N] (fp16) = x[B][K] (fp16) . dequant(packed,
    scales (fp16))."""
    B, K = x.shape
    N = scales.shape[1] if N is None else N
    _need(x, torch.float16, (B, K), "x")
    _need(scales, torch.float16, (K // GROUP, N), "scales")
    if packed.numel() * packed.element_size() < w4a16_packed_bytes(K, N, has_zeros):
        raise ValueError("packed: too small for this shape")
    if out is None:
        out = torch.empty((B, N), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, (B, N), "out")
    need = w4a16_workspace_bytes(B, K, N)
    if workspace is None:
        workspace = _default_ws.get(need, x.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w4a16_gemm_f16_path", load().w4a16_gemm_f16_path(
        x.data_ptr(), packed.data_ptr(), scales.data_ptr(), 1 if has_zeros else 0,
        out.data_ptr(), B, K, N, GROUP, ws_ptr, ws_bytes, int(path), _stream(stream)))
    return out


def w4a16_dequant_ref_f16(packed: torch.Tensor, scales: torch.Tensor, has_zeros: bool, K: int, *,
                          out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Dequantised W[K][N] (fp16) from fp16 scales, through the fp16 decode."""
    N = scales.shape[1]
    _need(scales, torch.float16, (K // GROUP, N), "scales")
    if out is None:
        out = torch.empty((K, N), dtype=torch.float16, device=scales.device)
    _need(out, torch.float16, (K, N), "out")
    _check("w4a16_dequant_ref_f16", load().w4a16_dequant_ref_f16(
        packed.data_ptr(), scales.data_ptr(), 1 if has_zeros else 0, out.data_ptr(), K, N,
        GROUP, _stream(stream)))
    return out


def w4a16_gemm_fused(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                     has_zeros: bool, epilogue: int, bias: torch.Tensor | None = None, *,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """w4a16_gemm with a fused epilogue (EPI_BIAS and/or EPI_SILU_MUL): bias
    bf16 [N]; with EPI_SILU_MUL the N columns are interleaved gate/up pairs and
    the output is [B][N/2]."""
    B, K = x.shape
    N = scales.shape[1]
    _need(x, torch.bfloat16, (B, K), "x")
    _need(scales, torch.bfloat16, (K // GROUP, N), "scales")
    if packed.numel() * packed.element_size() < w4a16_packed_bytes(K, N, has_zeros):
        raise ValueError("packed: too small for this shape")
    if bias is not None:
        _need(bias, torch.bfloat16, (N,), "bias")
    n_out = N // 2 if epilogue & EPI_SILU_MUL else N
    if out is None:
        out = torch.empty((B, n_out), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (B, n_out), "out")
    need = w4a16_workspace_bytes(B, K, N)
    if workspace is None:
        workspace = _default_ws.get(need, x.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w4a16_gemm_fused", load().w4a16_gemm_fused(
        x.data_ptr(), packed.data_ptr(), scales.data_ptr(), 1 if has_zeros else 0,
        None if bias is None else bias.data_ptr(), int(epilogue), out.data_ptr(), B, K, N, GROUP,
        ws_ptr, ws_bytes, _stream(stream)))
    return out


def w4a16_dequant_ref(packed: torch.Tensor, scales: torch.Tensor, has_zeros: bool, K: int, *,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Dequantised W[K][N] (bf16) through the kernels' own decode routine."""
    N = scales.shape[1]
    _need(scales, torch.bfloat16, (K // GROUP, N), "scales")
    if out is None:
        out = torch.empty((K, N), dtype=torch.bfloat16, device=scales.device)
    _need(out, torch.bfloat16, (K, N), "out")
    _check("w4a16_dequant_ref", load().w4a16_dequant_ref(
        packed.data_ptr(), scales.data_ptr(), 1 if has_zeros else 0, out.data_ptr(), K, N,
        GROUP, _stream(stream)))
    return out


def w4a16_grouped_workspace_bytes(T: int, E: int, max_rows: int, K: int, N: int) -> int:
    v = int(load().w4a16_grouped_workspace_bytes(T, E, max_rows, K, N, GROUP))
    if v == ctypes.c_size_t(-1).value:
        raise ValueError(f"invalid grouped shape T={T} E={E} max_rows={max_rows} K={K} N={N}")
    return v


def w4a16_gemm_grouped(x: torch.Tensor, offsets: torch.Tensor, packed: torch.Tensor,
                       scales: torch.Tensor, has_zeros: bool, max_rows: int, *,
                       out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Mixture-of-experts GEMM: rows offsets[e] .. offsets[e+1]-1 of x use expert
    e's weights.  packed: uint8 [E][packed_bytes]; scales: bf16 [E][K/128][N];
    offsets: int32 [E+1] on the device."""
    T, K = x.shape
    E, G, N = scales.shape
    _need(x, torch.bfloat16, (T, K), "x")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(scales, torch.bfloat16, (E, K // GROUP, N), "scales")
    _need(packed, torch.uint8, (E, w4a16_packed_bytes(K, N, has_zeros)), "packed")
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (T, N), "out")
    need = w4a16_grouped_workspace_bytes(T, E, max_rows, K, N)
    if workspace is None:
        workspace = _default_ws.get(need, x.device)
    _check("w4a16_gemm_grouped", load().w4a16_gemm_grouped(
        x.data_ptr(), offsets.data_ptr(), E, T, packed.data_ptr(), scales.data_ptr(),
        1 if has_zeros else 0, out.data_ptr(), max_rows, K, N, GROUP, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def w4a16_quantize_rtn(w: torch.Tensor, *, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Offline quantizer (round to nearest, MSE-optimal clipping): bf16 W [K][N]
    -> (canonical qweight int32 [K/8][N], scales bf16 [K/128][N])."""
    K, N = w.shape
    _need(w, torch.bfloat16, (K, N), "w")
    qweight = torch.empty((K // 8, N), dtype=torch.int32, device=w.device)
    scales = torch.empty((K // GROUP, N), dtype=torch.bfloat16, device=w.device)
    _check("w4a16_quantize_rtn", load().w4a16_quantize_rtn(
        w.data_ptr(), K, N, GROUP, qweight.data_ptr(), scales.data_ptr(), _stream(stream)))
    return qweight, scales


def w4a16_debug_forced_timeout(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                               has_zeros: bool, out: torch.Tensor, wait_ms: int,
                               workspace: torch.Tensor | None = None, stream=None) -> int:
    """Run the tensor-core kernel with one wait that must expire (test hook);
    returns the launch status (the device status word then reads TIMEOUT)."""
    B, K = x.shape
    N = scales.shape[1]
    need = w4a16_workspace_bytes(B, K, N)
    if workspace is None:
        workspace = _default_ws.get(need, x.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return int(load().w4a16_debug_forced_timeout(
        x.data_ptr(), packed.data_ptr(), scales.data_ptr(), 1 if has_zeros else 0,
        out.data_ptr(), B, K, N, GROUP, ws_ptr, ws_bytes, int(wait_ms), _stream(stream)))


def w4a16_device_status(clear: bool = True) -> int:
    return int(load().w4a16_device_status(1 if clear else 0))


def w4a16_packed_check(packed: torch.Tensor, K: int, N: int, has_zeros: bool,
                       stream=None) -> int:
    """Status of a packed blob's tag against (K, N, has_zeros) and the
    library's layout version (0 = OK); synchronises the stream."""
    return int(load().w4a16_packed_check(packed.data_ptr(), K, N, GROUP, 1 if has_zeros else 0,
                                         _stream(stream)))


# ---- W8A8-FP8 comparison path (include/w8a8_fp8.h)

def w8a8_fp8_quantize_act(x: torch.Tensor, *, out: tuple | None = None,
                          stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Dynamic per-token quantisation: bf16 x [B][K] -> (E4M3 codes uint8 [B][K],
    fp32 scales [B])."""
    B, K = x.shape
    _need(x, torch.bfloat16, (B, K), "x")
    if out is None:
        out = (torch.empty((B, K), dtype=torch.uint8, device=x.device),
               torch.empty(B, dtype=torch.float32, device=x.device))
    xq, sx = out
    _need(xq, torch.uint8, (B, K), "xq")
    _need(sx, torch.float32, (B,), "sx")
    _check("w8a8_fp8_quantize_act", load().w8a8_fp8_quantize_act(
        x.data_ptr(), B, K, xq.data_ptr(), sx.data_ptr(), _stream(stream)))
    return xq, sx


def w8a8_fp8_quantize_weight(w: torch.Tensor, *, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Per-output-channel quantisation: bf16 W [K][N] -> (E4M3 codes uint8 [N][K],
    fp32 scales [N])."""
    K, N = w.shape
    _need(w, torch.bfloat16, (K, N), "w")
    wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    sw = torch.empty(N, dtype=torch.float32, device=w.device)
    _check("w8a8_fp8_quantize_weight", load().w8a8_fp8_quantize_weight(
        w.data_ptr(), K, N, wq.data_ptr(), sw.data_ptr(), _stream(stream)))
    return wq, sw


def w8a8_fp8_packed_bytes(K: int, N: int) -> int:
    return int(load().w8a8_fp8_packed_bytes(K, N))


def w8a8_fp8_pack_weight(wq: torch.Tensor, *, stream=None) -> torch.Tensor:
    """[N][K] E4M3 codes -> the GEMM's tiled, pre-swizzled weight layout (uint8)."""
    N, K = wq.shape
    _need(wq, torch.uint8, (N, K), "wq")
    packed = torch.empty(w8a8_fp8_packed_bytes(K, N), dtype=torch.uint8, device=wq.device)
    _check("w8a8_fp8_pack_weight", load().w8a8_fp8_pack_weight(
        wq.data_ptr(), K, N, packed.data_ptr(), _stream(stream)))
    return packed


def w8a8_fp8_workspace_bytes(B: int, K: int, N: int) -> int:
    v = int(load().w8a8_fp8_workspace_bytes(B, K, N))
    if v == ctypes.c_size_t(-1).value:
        raise ValueError(f"invalid shape B={B} K={K} N={N}")
    return v


def w8a8_fp8_gemm(xq: torch.Tensor, sx: torch.Tensor, packed: torch.Tensor, sw: torch.Tensor, *,
                  out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """y[B][N] = (sx * dec(xq)) . (sw * dec(wq))^T, bf16; `packed` from
    w8a8_fp8_pack_weight(wq)."""
    B, K = xq.shape
    N = sw.shape[0]
    _need(xq, torch.uint8, (B, K), "xq")
    _need(packed, torch.uint8, (w8a8_fp8_packed_bytes(K, N),), "packed")
    _need(sx, torch.float32, (B,), "sx")
    _need(sw, torch.float32, (N,), "sw")
    if out is None:
        out = torch.empty((B, N), dtype=torch.bfloat16, device=xq.device)
    _need(out, torch.bfloat16, (B, N), "out")
    need = w8a8_fp8_workspace_bytes(B, K, N)
    if workspace is None:
        workspace = _default_ws.get(need, xq.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w8a8_fp8_gemm", load().w8a8_fp8_gemm(
        xq.data_ptr(), sx.data_ptr(), packed.data_ptr(), sw.data_ptr(), out.data_ptr(), B, K, N,
        ws_ptr, ws_bytes, _stream(stream)))
    return out
