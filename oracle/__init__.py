"""CPU oracle for the blockwise-FP8 MoE grouped matmul — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C, fp64 sums, fp32 where the
method fixes fp32); this module only builds it with gcc and marshals numpy
arrays through ctypes.  bf16 values travel as ``numpy.uint16`` bit patterns and
e4m3 codes as ``numpy.uint8``.

Layouts are the method's natural ones (not the CUDA library's):
  xq [M, K] uint8, xs [M, K/128] float32                 (1x128 LHS blocks)
  wq [G, K, N] uint8, ws [G, K/128, N/128] float32        (128x128 RHS blocks;
      e4m3 codes, or e2m1 codes one per byte for the 4-bit weights)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK = 0
ERR_NEGATIVE_GROUP = 1
ERR_GROUPS_EXCEED_M = 2
ERR_SHAPE = 3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (OpenMP when available).

    Built without fast-math and with FMA contraction off, so fp32 scale
    arithmetic is plain IEEE binary32 on every host.
    """
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode_array.argtypes = [P, I64, P]
        lib.oracle_e4m3_decode_array.argtypes = [P, I64, P]
        lib.oracle_e2m1_decode.restype = ctypes.c_double
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode_array.argtypes = [P, I64, P]
        lib.oracle_e2m1_decode_array.argtypes = [P, I64, P]
        lib.oracle_quantize_rhs_e2m1.argtypes = [P, I64, I64, I64, P, P]
        lib.oracle_gmm_fp8_w4.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, P]
        lib.oracle_round_to_bf16.restype = ctypes.c_uint16
        lib.oracle_round_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_to_bf16_array.argtypes = [P, I64, P]
        lib.oracle_bf16_to_double_array.argtypes = [P, I64, P]
        lib.oracle_quantize_lhs.argtypes = [P, I64, I64, P, P]
        lib.oracle_quantize_rhs.argtypes = [P, I64, I64, I64, P, P]
        lib.oracle_group_offsets.argtypes = [P, I64, I64, P]
        lib.oracle_group_tiles.argtypes = [P, I64, I64, I64, P, P, P]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_gmm_fp8.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, P]
        lib.oracle_gmm_bf16.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_int, P]
        lib.oracle_tgmm_bf16.argtypes = [P, P, P, I64, I64, I64, I64, P]
        lib.oracle_dgrad_bf16.argtypes = [P, P, P, I64, I64, I64, I64, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__({1: "negative group size", 2: "sum(group_sizes) > M",
                          3: "bad shape"}.get(status, f"status {status}"))
        self.status = status


def _check(st: int):
    if st != OK:
        raise OracleError(st)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ----------------------------------------------------------------------------
# codecs
# ----------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_decode(codes) -> np.ndarray:
    """FP4 E2M1 value of each code (the low 4 bits of each byte)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e2m1_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e2m1_encode(values) -> np.ndarray:
    """FP4 E2M1 code (0..15) of each fp32 value: nearest, ties to even, saturating at 6."""
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def round_to_bf16(values) -> np.ndarray:
    """fp64 -> fp32 (nearest) -> bf16 (nearest, ties to even), as uint16 bits."""
    v = _c(values, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_round_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_bf16_to_double_array(_ptr(b), b.size, _ptr(out))
    return out


def silu(v: float) -> float:
    return float(_load().oracle_silu(float(v)))


# ----------------------------------------------------------------------------
# quantization
# ----------------------------------------------------------------------------

def quantize_lhs(x_bf16) -> tuple[np.ndarray, np.ndarray]:
    """1x128 dynamic quantization of X [M, K] -> (xq [M,K] u8, xs [M,K/128] f32)."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    xq = np.empty((M, K), np.uint8)
    xs = np.empty((M, K // 128), np.float32)
    _check(_load().oracle_quantize_lhs(_ptr(x), M, K, _ptr(xq), _ptr(xs)))
    return xq, xs


def quantize_rhs(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """128x128 quantization of W [G, K, N] -> (wq [G,K,N] u8, ws [G,K/128,N/128] f32)."""
    w = _c(w_bf16, np.uint16)
    G, K, N = w.shape
    wq = np.empty((G, K, N), np.uint8)
    ws = np.empty((G, K // 128, N // 128), np.float32)
    _check(_load().oracle_quantize_rhs(_ptr(w), G, K, N, _ptr(wq), _ptr(ws)))
    return wq, ws


def quantize_rhs_e2m1(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """4-bit weights: 128x128 blocks, scale = absmax / 6, e2m1 codes ->
    (wq [G,K,N] u8, one code per byte; ws [G,K/128,N/128] f32)."""
    w = _c(w_bf16, np.uint16)
    G, K, N = w.shape
    wq = np.empty((G, K, N), np.uint8)
    ws = np.empty((G, K // 128, N // 128), np.float32)
    _check(_load().oracle_quantize_rhs_e2m1(_ptr(w), G, K, N, _ptr(wq), _ptr(ws)))
    return wq, ws


# ----------------------------------------------------------------------------
# group metadata
# ----------------------------------------------------------------------------

def group_offsets(group_sizes, M: int) -> np.ndarray:
    s = _c(group_sizes, np.int32)
    off = np.empty(s.size + 1, np.int64)
    _check(_load().oracle_group_offsets(_ptr(s), s.size, M, _ptr(off)))
    return off


def group_tiles(group_sizes, M: int, bm: int) -> tuple[np.ndarray, np.ndarray]:
    """Returns (offsets [G+1], tiles [T, 3] = (g, row0, row1))."""
    s = _c(group_sizes, np.int32)
    G = s.size
    off = np.empty(G + 1, np.int64)
    cap = (M + bm - 1) // bm + G
    tiles = np.empty((max(cap, 1), 3), np.int64)
    nt = ctypes.c_int64(0)
    _check(_load().oracle_group_tiles(_ptr(s), G, M, bm, _ptr(off), _ptr(tiles),
                                      ctypes.byref(nt)))
    return off, tiles[: nt.value].copy()


# ----------------------------------------------------------------------------
# GEMMs (fp64 results; round with round_to_bf16 for the bf16 output)
# ----------------------------------------------------------------------------

def gmm_fp8(xq, xs, wq, ws, group_sizes, fuse: bool = False) -> np.ndarray:
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.float32)
    s = _c(group_sizes, np.int32)
    M, K = xq.shape
    G, K2, Nw = wq.shape
    assert K2 == K and s.size == G
    N = Nw // 2 if fuse else Nw
    out = np.empty((M, N), np.float64)
    _check(_load().oracle_gmm_fp8(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), _ptr(s), G, M, K, N,
                                  int(bool(fuse)), _ptr(out)))
    return out


def gmm_fp8_w4(xq, xs, wq4, ws, group_sizes, fuse: bool = False) -> np.ndarray:
    """gmm_fp8 with e2m1 weight codes (one per byte, [G, K, Nw]) and their
    128x128 scales; the activations stay e4m3 in 1x128 blocks."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    wq4 = _c(wq4, np.uint8)
    ws = _c(ws, np.float32)
    s = _c(group_sizes, np.int32)
    M, K = xq.shape
    G, K2, Nw = wq4.shape
    assert K2 == K and s.size == G
    N = Nw // 2 if fuse else Nw
    out = np.empty((M, N), np.float64)
    _check(_load().oracle_gmm_fp8_w4(_ptr(xq), _ptr(xs), _ptr(wq4), _ptr(ws), _ptr(s), G, M, K, N,
                                     int(bool(fuse)), _ptr(out)))
    return out


def gmm_bf16(x, w, group_sizes, fuse: bool = False) -> np.ndarray:
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    s = _c(group_sizes, np.int32)
    M, K = x.shape
    G, K2, Nw = w.shape
    assert K2 == K and s.size == G
    N = Nw // 2 if fuse else Nw
    out = np.empty((M, N), np.float64)
    _check(_load().oracle_gmm_bf16(_ptr(x), _ptr(w), _ptr(s), G, M, K, N, int(bool(fuse)),
                                   _ptr(out)))
    return out


def tgmm_bf16(x, dy, group_sizes) -> np.ndarray:
    x = _c(x, np.uint16)
    dy = _c(dy, np.uint16)
    s = _c(group_sizes, np.int32)
    M, K = x.shape
    M2, N = dy.shape
    assert M2 == M
    G = s.size
    out = np.empty((G, K, N), np.float64)
    _check(_load().oracle_tgmm_bf16(_ptr(x), _ptr(dy), _ptr(s), G, M, K, N, _ptr(out)))
    return out


def dgrad_bf16(dy, w, group_sizes) -> np.ndarray:
    """dx[m, k] = sum_n dy[m, n] * w[g][k, n] (fp64); dy [M, N], w [G, K, N]."""
    dy = _c(dy, np.uint16)
    w = _c(w, np.uint16)
    s = _c(group_sizes, np.int32)
    M, N = dy.shape
    G, K, N2 = w.shape
    assert N2 == N and s.size == G
    out = np.empty((M, K), np.float64)
    _check(_load().oracle_dgrad_bf16(_ptr(dy), _ptr(w), _ptr(s), G, M, K, N, _ptr(out)))
    return out


# ----------------------------------------------------------------------------
# accuracy metrics of the method's own methodology ("GEMM Kernel 性能优化十问",
# Q9.2): element-wise allclose, SQNR in dB, and the error in units in the last
# place of the expected value.
# ----------------------------------------------------------------------------

def sqnr_db(ref, test) -> float:
    ref = np.asarray(ref, np.float64)
    test = np.asarray(test, np.float64)
    noise = float(np.sum((ref - test) ** 2))
    signal = float(np.sum(ref ** 2))
    if noise == 0.0:
        return float("inf")
    return 10.0 * np.log10(signal / noise)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits, normal range)."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(v > 0, v, 2.0 ** -126)))
    e = np.maximum(e, -126)
    return 2.0 ** (e - 7)
