"""CPU oracle for the W4A16 group-128 linear layer -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, compiled with gcc, OpenMP
over output columns).  This module only compiles it and marshals numpy arrays
through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the library under
``weight_only_int4_gemm_gb300`` never does, and the two share no code.

Sources, by page title and section:
  * "Give Me BF16 or Give Me Death" (summary), "W4A16-INT Quantization":
    group-128 scales along K; dequantise-then-multiply inference.
  * "When quantization pays -- and when it does not", "Counting c from the
    kernel, not from intuition": uint4 codes with bias 8, exact (q - 8) first,
    then one bf16 multiply by the group scale.
  * "When quantization pays -- and when it does not", "The three regimes"
    (mixture-of-experts paragraphs): each routed expert's GEMM sees only
    its own rows (``gemm_grouped``).
  * "Give Me BF16 or Give Me Death", "W4A16-INT Quantization": round to
    nearest with MSE-optimal clipping (``quantize_rtn_mse``).
  * "Give Me BF16 or Give Me Death", "W4A16-INT Quantization", paragraph
    "Inference with W4A16": the same layer with fp16 activations, scales,
    weights and output (``f16_*``, ``dequant_f16``, ``gemm_f16``; C source
    ``w4a16_f16_oracle.c``).
  * "Give Me BF16 or Give Me Death", "W8A8-FP Quantization": per-channel FP8
    weights, dynamic per-token FP8 activations, their product
    (``fp8_quantize_rows``, ``fp8_quantize_cols``, ``fp8_gemm``; C source
    ``w8a8_fp8_oracle.c``).

Parity status: every function here is pinned -- ``tests/test_oracle_pins.py``
(exhaustive nearest-bf16 check, integer special cases, exact-rational brute
force, invariants, hand-built unpack cases, the 4.125-bit accounting),
``tests/test_quantizer_pins.py`` (quantizer), ``tests/test_grouped_pins.py``
(closed-form expert routing), ``tests/test_epilogue_pins.py`` (closed-form
bias and SiLU-gate cases, an independent tanh route to silu) and
``tests/test_fp8_pins.py`` (E4M3 codec
against the format's published constants and brute-force nearest search,
scale invariants, exact integer GEMM) and ``tests/test_f16_pins.py`` (binary16
codec against numpy's float16 and an exhaustive tie enumeration, every code
times every finite fp16 scale against numpy, exact-rational brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "w8a8_fp8_oracle.c"), os.path.join(_HERE, "w4a16_f16_oracle.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 128


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and \
            os.path.getmtime(_LIB) >= max(os.path.getmtime(p) for p in _SRCS):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int)
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_code.argtypes = [u32p, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_code.restype = ctypes.c_int
        lib.oracle_zero.argtypes = [u32p, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_zero.restype = ctypes.c_int
        lib.oracle_dequant_one.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint16]
        lib.oracle_dequant_one.restype = ctypes.c_uint16
        lib.oracle_dequant.argtypes = [u32p, u16p, u32p, ctypes.c_int, ctypes.c_int, u16p]
        lib.oracle_dequant.restype = None
        lib.oracle_gemm_cols.argtypes = [u16p, u32p, u16p, u32p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, i32p, ctypes.c_int, u16p, f64p, f64p]
        lib.oracle_gemm_cols.restype = None
        lib.oracle_bf16_from_double_array.argtypes = [f64p, ctypes.c_longlong, u16p]
        lib.oracle_bf16_from_double_array.restype = None
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_threads.restype = None
        lib.oracle_quantize_rtn_mse.argtypes = [u16p, ctypes.c_int, ctypes.c_int, u32p, u16p]
        lib.oracle_quantize_rtn_mse.restype = None
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_from_double.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
        lib.oracle_fp8_quantize_rows.argtypes = [u16p, ctypes.c_int, ctypes.c_int, u8p, f32p]
        lib.oracle_fp8_quantize_rows.restype = None
        lib.oracle_fp8_quantize_cols.argtypes = [u16p, ctypes.c_int, ctypes.c_int, u8p, f32p]
        lib.oracle_fp8_quantize_cols.restype = None
        lib.oracle_fp8_gemm_cols.argtypes = [u8p, f32p, u8p, f32p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, i32p, ctypes.c_int, u16p, f64p, f64p]
        lib.oracle_fp8_gemm_cols.restype = None
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_f16_from_double.restype = ctypes.c_uint16
        lib.oracle_f16_from_double_array.argtypes = [f64p, ctypes.c_longlong, u16p]
        lib.oracle_f16_from_double_array.restype = None
        lib.oracle_dequant_one_f16.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint16]
        lib.oracle_dequant_one_f16.restype = ctypes.c_uint16
        lib.oracle_dequant_f16.argtypes = [u32p, u16p, u32p, ctypes.c_int, ctypes.c_int, u16p]
        lib.oracle_dequant_f16.restype = None
        lib.oracle_gemm_cols_f16.argtypes = [u16p, u32p, u16p, u32p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, i32p, ctypes.c_int, u16p, f64p, f64p]
        lib.oracle_gemm_cols_f16.restype = None
        lib.oracle_format_bits_per_weight.argtypes = [ctypes.c_longlong, ctypes.c_longlong,
                                                      ctypes.c_int]
        lib.oracle_format_bits_per_weight.restype = ctypes.c_double
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype in (np.uint16, np.int16), a.dtype
    return a.view(np.uint16)


def _as_u32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype in (np.uint32, np.int32), a.dtype
    return a.view(np.uint32)


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits) & 0xFFFF)


def bf16_from_double(v: float) -> int:
    return int(_load().oracle_bf16_from_double(float(v)))


def code(qweight: np.ndarray, k: int, n: int) -> int:
    q = _as_u32(qweight)
    return _load().oracle_code(_ptr(q, ctypes.c_uint32), q.shape[1], k, n)


def zero(qzeros: np.ndarray | None, N: int, g: int, n: int) -> int:
    z = None if qzeros is None else _as_u32(qzeros)
    return _load().oracle_zero(_ptr(z, ctypes.c_uint32), N, g, n)


def dequant_one(q: int, z: int, scale_bits: int) -> int:
    return int(_load().oracle_dequant_one(int(q), int(z), int(scale_bits) & 0xFFFF))


def dequant(qweight, scales, qzeros=None) -> np.ndarray:
    """W[K][N] as bf16 bit patterns (uint16)."""
    q = _as_u32(qweight)
    s = _as_u16(scales)
    z = None if qzeros is None else _as_u32(qzeros)
    K = q.shape[0] * 8
    N = q.shape[1]
    assert s.shape == (K // GROUP, N)
    if z is not None:
        assert z.shape == (K // GROUP, N // 8)
    out = np.empty((K, N), dtype=np.uint16)
    _load().oracle_dequant(_ptr(q, ctypes.c_uint32), _ptr(s, ctypes.c_uint16),
                           _ptr(z, ctypes.c_uint32), K, N, _ptr(out, ctypes.c_uint16))
    return out


def gemm(x, qweight, scales, qzeros=None, cols=None):
    """Reference GEMM on the listed output columns (all when ``cols`` is None).

    Returns ``(y_bits uint16 [B][ncols], acc float64 [B][ncols],
    bound float64 [B][ncols])``.
    """
    xb = _as_u16(x)
    q = _as_u32(qweight)
    s = _as_u16(scales)
    z = None if qzeros is None else _as_u32(qzeros)
    B, K = xb.shape
    N = q.shape[1]
    assert q.shape[0] * 8 == K
    assert s.shape == (K // GROUP, N)
    if z is not None:
        assert z.shape == (K // GROUP, N // 8)
    c = np.arange(N, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, dtype=np.int32)
    nc = int(c.shape[0])
    y = np.empty((B, nc), dtype=np.uint16)
    acc = np.empty((B, nc), dtype=np.float64)
    bound = np.empty((B, nc), dtype=np.float64)
    _load().oracle_gemm_cols(_ptr(xb, ctypes.c_uint16), _ptr(q, ctypes.c_uint32),
                             _ptr(s, ctypes.c_uint16), _ptr(z, ctypes.c_uint32),
                             B, K, N, _ptr(c, ctypes.c_int), nc,
                             _ptr(y, ctypes.c_uint16), _ptr(acc, ctypes.c_double),
                             _ptr(bound, ctypes.c_double))
    return y, acc, bound


def bf16_round(v) -> np.ndarray:
    """RNE_bf16 of every element of a float64 array (bit patterns)."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_from_double_array(_ptr(a, ctypes.c_double), a.size,
                                          _ptr(out, ctypes.c_uint16))
    return out


# ---- fp16-activation variant (w4a16_f16_oracle.c)

def f16_to_double(bits: int) -> float:
    return _load().oracle_f16_to_double(int(bits) & 0xFFFF)


def f16_from_double(v: float) -> int:
    return int(_load().oracle_f16_from_double(float(v)))


def f16_round(v) -> np.ndarray:
    """RNE_f16 of every element of a float64 array (bit patterns)."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_f16_from_double_array(_ptr(a, ctypes.c_double), a.size,
                                         _ptr(out, ctypes.c_uint16))
    return out


def dequant_one_f16(q: int, z: int, scale_bits: int) -> int:
    return int(_load().oracle_dequant_one_f16(int(q), int(z), int(scale_bits) & 0xFFFF))


def dequant_f16(qweight, scales, qzeros=None) -> np.ndarray:
    """W[K][N] as fp16 bit patterns (uint16), scales fp16 bits [K/128][N]."""
    q = _as_u32(qweight)
    s = _as_u16(scales)
    z = None if qzeros is None else _as_u32(qzeros)
    K = q.shape[0] * 8
    N = q.shape[1]
    assert s.shape == (K // GROUP, N)
    if z is not None:
        assert z.shape == (K // GROUP, N // 8)
    out = np.empty((K, N), dtype=np.uint16)
    _load().oracle_dequant_f16(_ptr(q, ctypes.c_uint32), _ptr(s, ctypes.c_uint16),
                               _ptr(z, ctypes.c_uint32), K, N, _ptr(out, ctypes.c_uint16))
    return out


def gemm_f16(x, qweight, scales, qzeros=None, cols=None):
    """fp16 reference GEMM (x, scales, y fp16 bits) on the listed columns.

    Returns ``(y_bits uint16 [B][ncols], acc float64, bound float64)`` with
    bound = 2e-3 * sum|x*w| + 2^-24 * (1 + sum|x|)."""
    xb = _as_u16(x)
    q = _as_u32(qweight)
    s = _as_u16(scales)
    z = None if qzeros is None else _as_u32(qzeros)
    B, K = xb.shape
    N = q.shape[1]
    assert q.shape[0] * 8 == K
    assert s.shape == (K // GROUP, N)
    if z is not None:
        assert z.shape == (K // GROUP, N // 8)
    c = np.arange(N, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, dtype=np.int32)
    nc = int(c.shape[0])
    y = np.empty((B, nc), dtype=np.uint16)
    acc = np.empty((B, nc), dtype=np.float64)
    bound = np.empty((B, nc), dtype=np.float64)
    _load().oracle_gemm_cols_f16(_ptr(xb, ctypes.c_uint16), _ptr(q, ctypes.c_uint32),
                                 _ptr(s, ctypes.c_uint16), _ptr(z, ctypes.c_uint32),
                                 B, K, N, _ptr(c, ctypes.c_int), nc,
                                 _ptr(y, ctypes.c_uint16), _ptr(acc, ctypes.c_double),
                                 _ptr(bound, ctypes.c_double))
    return y, acc, bound


EPI_BIAS, EPI_SILU_MUL = 1, 2
SILU_SLOPE_MAX = 1.1  # sup |d/dg silu(g)| = 1.0998...


def silu(g):
    """silu(g) = g / (1 + e^-g), float64."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def gemm_epilogue(x, qweight, scales, qzeros=None, bias=None, mode=0, cols=None):
    """GEMM with a fused output epilogue, on the exact sums of ``gemm``.

    mode: EPI_BIAS adds bias[n] (bf16 bits [N]); EPI_SILU_MUL treats columns
    (2j, 2j+1) as (gate, up) and returns h[b][j] = RNE_bf16(silu(g) * u).
    With EPI_SILU_MUL, ``cols`` (if given) lists gate columns 2j; their up
    partners are added.  Returns (y bits, value before rounding, bound): the
    bound is the GEMM bound carried through the epilogue -- for the SiLU form
    1.1 * b_g * (|u| + b_u) + |silu(g)| * b_u (slope of silu at most 1.1) plus
    one bf16 step of the result, 2^-7 |h|.
    """
    silu_mode = bool(mode & EPI_SILU_MUL)
    if silu_mode and cols is not None:
        gates = np.asarray(cols, dtype=np.int64)
        assert np.all(gates % 2 == 0)
        cols = np.stack([gates, gates + 1], axis=1).reshape(-1)
    _, acc, bound = gemm(x, qweight, scales, qzeros, cols=cols)
    N = _as_u32(qweight).shape[1]
    c = np.arange(N) if cols is None else np.asarray(cols)
    v = acc.copy()
    if mode & EPI_BIAS:
        bb = _as_u16(bias).astype(np.uint32)
        bvals = (bb << 16).view(np.float32).astype(np.float64)[c]
        v = v + bvals[None, :]
        bound = bound + 2.0 ** -7 * np.abs(bvals)[None, :]
    if not silu_mode:
        return bf16_round(v), v, bound
    g, u = v[:, 0::2], v[:, 1::2]
    bg, bu = bound[:, 0::2], bound[:, 1::2]
    h = silu(g) * u
    hb = SILU_SLOPE_MAX * bg * (np.abs(u) + bu) + np.abs(silu(g)) * bu + 2.0 ** -7 * np.abs(h) + 1e-6
    return bf16_round(h), h, hb


def gemm_grouped(x, offsets, qweights, scales, qzeros=None, cols=None):
    """Mixture-of-experts GEMM ("When quantization pays -- and when it does
    not", section "The three regimes", the mixture-of-experts paragraphs: a
    routed expert's weights multiply only the rows sent to it).

    Rows offsets[e] .. offsets[e+1]-1 of x [T][K] use expert e's weights
    (qweights[e], scales[e], qzeros[e]); each expert is one ``gemm`` on its
    rows.  Returns ``(y, acc, bound)`` over all T rows, like ``gemm``.
    """
    xb = _as_u16(x)
    T = xb.shape[0]
    off = np.asarray(offsets, dtype=np.int64)
    E = off.shape[0] - 1
    assert off[0] == 0 and off[E] == T and np.all(np.diff(off) >= 0)
    N = _as_u32(qweights[0]).shape[1]
    nc = N if cols is None else len(cols)
    y = np.zeros((T, nc), dtype=np.uint16)
    acc = np.zeros((T, nc), dtype=np.float64)
    bound = np.zeros((T, nc), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        ye, ae, be = gemm(xb[r0:r1], qweights[e], scales[e],
                          None if qzeros is None else qzeros[e], cols=cols)
        y[r0:r1], acc[r0:r1], bound[r0:r1] = ye, ae, be
    return y, acc, bound


def quantize_rtn_mse(w) -> tuple[np.ndarray, np.ndarray]:
    """MSE-optimal clipping quantizer (round to nearest): bf16 bits w [K][N] ->
    (canonical qweight uint32 [K/8][N], scales bf16 bits uint16 [K/128][N])."""
    w = _as_u16(w)
    K, N = w.shape
    qw = np.zeros((K // 8, N), dtype=np.uint32)
    sc = np.zeros((K // 128, N), dtype=np.uint16)
    _load().oracle_quantize_rtn_mse(_ptr(w, ctypes.c_uint16), K, N, _ptr(qw, ctypes.c_uint32),
                                    _ptr(sc, ctypes.c_uint16))
    return qw, sc


# ---- W8A8-FP8 comparison path ("Give Me BF16 or Give Me Death", section
# "W8A8-FP Quantization: 8-Bit Floating-Point Weights and Activations")

def e4m3_to_double(code: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(code)))


def e4m3_from_double(v: float) -> int:
    return int(_load().oracle_e4m3_from_double(float(v)))


def fp8_quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Dynamic per-token quantisation: bf16 bits x [B][K] -> (E4M3 codes uint8
    [B][K], binary32 scales [B])."""
    x = _as_u16(x)
    B, K = x.shape
    codes = np.zeros((B, K), dtype=np.uint8)
    sc = np.zeros(B, dtype=np.float32)
    _load().oracle_fp8_quantize_rows(_ptr(x, ctypes.c_uint16), B, K,
                                     _ptr(codes, ctypes.c_uint8), _ptr(sc, ctypes.c_float))
    return codes, sc


def fp8_quantize_cols(w) -> tuple[np.ndarray, np.ndarray]:
    """Per-output-channel weight quantisation: bf16 bits W [K][N] -> (E4M3
    codes uint8 [N][K], binary32 scales [N])."""
    w = _as_u16(w)
    K, N = w.shape
    codes = np.zeros((N, K), dtype=np.uint8)
    sc = np.zeros(N, dtype=np.float32)
    _load().oracle_fp8_quantize_cols(_ptr(w, ctypes.c_uint16), K, N,
                                     _ptr(codes, ctypes.c_uint8), _ptr(sc, ctypes.c_float))
    return codes, sc


def fp8_gemm(xq, sx, wq, sw, cols=None):
    """y = (s_x q_x) . (s_w q_w) on the listed columns: returns (y bf16 bits
    [B][ncols], acc = exact code sum float64, bound float64)."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    B, K = xq.shape
    N = wq.shape[0]
    assert wq.shape == (N, K) and sx.shape == (B,) and sw.shape == (N,)
    assert K <= 1 << 15, "the exact-sum argument holds for K <= 2^15"
    c = np.arange(N, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, dtype=np.int32)
    nc = int(c.shape[0])
    y = np.empty((B, nc), dtype=np.uint16)
    acc = np.empty((B, nc), dtype=np.float64)
    bound = np.empty((B, nc), dtype=np.float64)
    _load().oracle_fp8_gemm_cols(_ptr(xq, ctypes.c_uint8), _ptr(sx, ctypes.c_float),
                                 _ptr(wq, ctypes.c_uint8), _ptr(sw, ctypes.c_float), B, K, N,
                                 _ptr(c, ctypes.c_int), nc, _ptr(y, ctypes.c_uint16),
                                 _ptr(acc, ctypes.c_double), _ptr(bound, ctypes.c_double))
    return y, acc, bound


def format_bits_per_weight(K: int, N: int, has_zeros: bool) -> float:
    return float(_load().oracle_format_bits_per_weight(K, N, 1 if has_zeros else 0))


def set_threads(n: int) -> None:
    """Threads for the oracle's OpenMP loops from now on."""
    _load().oracle_set_threads(int(n))


def omp_threads() -> int:
    """Threads the oracle's OpenMP loops use (OMP_NUM_THREADS, else all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    return os.cpu_count() or 1
