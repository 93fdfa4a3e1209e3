"""Python binding of the C ABI in include/gmm.h (argument marshalling only).

Every function named like a C entry point passes its tensors' device
pointers, the sizes and the stream straight to the library; every step of the
computation runs in the library's CUDA kernels.  The convenience wrappers
below (``quantize_lhs``, ``fp8_fwd``, ...) additionally allocate the outputs
with torch, which here is only the device-memory allocator.

The library must have been built (``fp8_blockwise_quantized_gb300.build``);
without it every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgmm_gb300.so")

GMM_OK = 0
GMM_ERR_GROUP_SIZES = 6
GMM_ERR_TIMEOUT = 7
STATUS_NAMES = {0: "GMM_OK", 1: "GMM_ERR_NULL", 2: "GMM_ERR_SHAPE", 3: "GMM_ERR_ALIGN",
                4: "GMM_ERR_UNSUPPORTED", 5: "GMM_ERR_CUDA", 6: "GMM_ERR_GROUP_SIZES",
                7: "GMM_ERR_TIMEOUT", 8: "GMM_ERR_WORKSPACE"}

EXPORTED = ["gmm_status_string", "gmm_last_cuda_error", "gmm_workspace_bytes", "gmm_tiles_offset",
            "gmm_group_metadata", "gmm_quantize_lhs", "gmm_quantize_rhs", "gmm_fp8_fwd",
            "gmm_bf16_fwd", "tgmm_bf16", "gmm_get_device_status", "gmm_fp8_fwd_noalloc",
            "gmm_bf16_dgrad", "gmm_fp8_fwd_swiglu_quant", "gmm_selftest_wait_timeout", "gmm_fp8_fwd_tiled",
            "gmm_fp8_fwd_swiglu_quant_tiled", "gmm_quantize_rhs_w4", "gmm_fp8_w4_fwd",
            "gmm_fp8_w4_fwd_swiglu_quant", "tgmm_bf16_tiled"]


class TileConfig(ctypes.Structure):
    """gmm_fp8_tile_config: bn (128 | 256), ctas (1 .. SMs), unit_order
    (1 row-tile major, 2 column-block major), cta_group (1 one CTA per
    128-row tile, 2 CTA pairs on 256-row tiles), stages (operand ring
    slots), tmem_bufs (TMEM partial buffers); 0 keeps a field's default.
    A shorter tuple leaves the remaining fields 0."""
    _fields_ = [("bn", ctypes.c_int), ("ctas", ctypes.c_int), ("unit_order", ctypes.c_int),
                ("cta_group", ctypes.c_int), ("stages", ctypes.c_int), ("tmem_bufs", ctypes.c_int)]

    def astuple(self):
        return (self.bn, self.ctas, self.unit_order, self.cta_group, self.stages, self.tmem_bufs)


class TgmmConfig(ctypes.Structure):
    """gmm_tgmm_tile_config: stages (4..6), claim_ahead (1..12), max_batch
    (1..4); 0 keeps a field's default.  A shorter tuple leaves the rest 0."""
    _fields_ = [("stages", ctypes.c_int), ("claim_ahead", ctypes.c_int), ("max_batch", ctypes.c_int)]

    def astuple(self):
        return (self.stages, self.claim_ahead, self.max_batch)


class GmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.gmm_status_string(status).decode()
        if status == 5:
            msg += f" ({lib.gmm_last_cuda_error().decode()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


_lib = None


def load():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run fp8_blockwise_quantized_gb300.build.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.gmm_status_string.restype = ctypes.c_char_p
    lib.gmm_status_string.argtypes = [I]
    lib.gmm_last_cuda_error.restype = ctypes.c_char_p
    lib.gmm_last_cuda_error.argtypes = []
    lib.gmm_workspace_bytes.restype = SZ
    lib.gmm_workspace_bytes.argtypes = [I, I64]
    lib.gmm_tiles_offset.restype = SZ
    lib.gmm_tiles_offset.argtypes = [I]
    lib.gmm_group_metadata.restype = I
    lib.gmm_group_metadata.argtypes = [P, I, I64, P, SZ, P]
    lib.gmm_quantize_lhs.restype = I
    lib.gmm_quantize_lhs.argtypes = [P, I64, I64, P, P, P]
    lib.gmm_quantize_rhs.restype = I
    lib.gmm_quantize_rhs.argtypes = [P, I, I64, I64, P, P, P]
    lib.gmm_fp8_fwd.restype = I
    lib.gmm_fp8_fwd.argtypes = [P, P, P, P, P, I, I64, I64, I64, I, P, P, SZ, P]
    lib.gmm_fp8_fwd_tiled.restype = I
    lib.gmm_fp8_fwd_tiled.argtypes = [P, P, P, P, P, I, I64, I64, I64, I, P, P, SZ, P,
                                      ctypes.POINTER(TileConfig)]
    lib.gmm_bf16_fwd.restype = I
    lib.gmm_bf16_fwd.argtypes = [P, P, P, I, I64, I64, I64, I, P, P, SZ, P]
    lib.tgmm_bf16.restype = I
    lib.tgmm_bf16.argtypes = [P, P, P, I, I64, I64, I64, P, P, SZ, P]
    lib.tgmm_bf16_tiled.restype = I
    lib.tgmm_bf16_tiled.argtypes = [P, P, P, I, I64, I64, I64, P, P, SZ, P, ctypes.POINTER(TgmmConfig)]
    lib.gmm_fp8_fwd_swiglu_quant.restype = I
    lib.gmm_fp8_fwd_swiglu_quant.argtypes = [P, P, P, P, P, I, I64, I64, I64, P, P, P, P, SZ, P]
    lib.gmm_fp8_fwd_swiglu_quant_tiled.restype = I
    lib.gmm_fp8_fwd_swiglu_quant_tiled.argtypes = [P, P, P, P, P, I, I64, I64, I64, P, P, P, P, SZ, P,
                                                   ctypes.POINTER(TileConfig)]
    lib.gmm_bf16_dgrad.restype = I
    lib.gmm_bf16_dgrad.argtypes = [P, P, P, I, I64, I64, I64, P, P, SZ, P]
    lib.gmm_get_device_status.restype = I
    lib.gmm_get_device_status.argtypes = [P, P]
    lib.gmm_selftest_wait_timeout.restype = I
    lib.gmm_selftest_wait_timeout.argtypes = [P, SZ, I, P]
    lib.gmm_fp8_fwd_noalloc.restype = I
    lib.gmm_fp8_fwd_noalloc.argtypes = [P, P, P, P, P, I, I64, I64, I64, I, P, P]
    lib.gmm_quantize_rhs_w4.restype = I
    lib.gmm_quantize_rhs_w4.argtypes = [P, I, I64, I64, P, P, P]
    lib.gmm_fp8_w4_fwd.restype = I
    lib.gmm_fp8_w4_fwd.argtypes = [P, P, P, P, P, I, I64, I64, I64, I, P, P, SZ, P, ctypes.POINTER(TileConfig)]
    lib.gmm_fp8_w4_fwd_swiglu_quant.restype = I
    lib.gmm_fp8_w4_fwd_swiglu_quant.argtypes = [P, P, P, P, P, I, I64, I64, I64, P, P, P, P, SZ, P,
                                                ctypes.POINTER(TileConfig)]
    _lib = lib
    return lib


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr() if t.numel() > 0 else None
    return int(t)


def _s(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str):
    if status != GMM_OK:
        raise GmmError(status, where)


# ---------------------------------------------------------------------------
# C entry points, same names and argument order
# ---------------------------------------------------------------------------

def gmm_workspace_bytes(G: int, M: int) -> int:
    return int(load().gmm_workspace_bytes(G, M))


def gmm_tiles_offset(G: int) -> int:
    return int(load().gmm_tiles_offset(G))


def gmm_group_metadata(group_sizes, G, M, workspace, workspace_bytes, stream=None) -> int:
    return load().gmm_group_metadata(_p(group_sizes), G, M, _p(workspace), workspace_bytes, _s(stream))


def gmm_quantize_lhs(x, M, K, xq, xs, stream=None) -> int:
    return load().gmm_quantize_lhs(_p(x), M, K, _p(xq), _p(xs), _s(stream))


def gmm_quantize_rhs(w, G, K, N, wq, ws, stream=None) -> int:
    return load().gmm_quantize_rhs(_p(w), G, K, N, _p(wq), _p(ws), _s(stream))


def gmm_fp8_fwd(xq, xs, wq, ws, group_sizes, G, M, K, N, fuse_silu_mul, out, workspace,
                workspace_bytes, stream=None) -> int:
    return load().gmm_fp8_fwd(_p(xq), _p(xs), _p(wq), _p(ws), _p(group_sizes), G, M, K, N,
                              int(fuse_silu_mul), _p(out), _p(workspace), workspace_bytes, _s(stream))


def gmm_fp8_fwd_tiled(xq, xs, wq, ws, group_sizes, G, M, K, N, fuse_silu_mul, out, workspace,
                      workspace_bytes, stream=None, config=None) -> int:
    """config: a TileConfig, a (bn, ctas, unit_order[, cta_group[, stages[, tmem_bufs]]]) tuple, or None."""
    if config is not None and not isinstance(config, TileConfig):
        config = TileConfig(*config)
    return load().gmm_fp8_fwd_tiled(_p(xq), _p(xs), _p(wq), _p(ws), _p(group_sizes), G, M, K, N,
                                    int(fuse_silu_mul), _p(out), _p(workspace), workspace_bytes, _s(stream),
                                    ctypes.byref(config) if config is not None else None)


def gmm_fp8_fwd_swiglu_quant(xq, xs, wq, ws, group_sizes, G, M, K, N, h, hq, hs, workspace,
                             workspace_bytes, stream=None) -> int:
    return load().gmm_fp8_fwd_swiglu_quant(_p(xq), _p(xs), _p(wq), _p(ws), _p(group_sizes), G, M, K, N, _p(h),
                                           _p(hq), _p(hs), _p(workspace), workspace_bytes, _s(stream))


def gmm_fp8_fwd_swiglu_quant_tiled(xq, xs, wq, ws, group_sizes, G, M, K, N, h, hq, hs, workspace,
                                   workspace_bytes, stream=None, config=None) -> int:
    """config: a TileConfig, a (bn, ctas, unit_order[, cta_group[, stages[, tmem_bufs]]]) tuple, or None."""
    if config is not None and not isinstance(config, TileConfig):
        config = TileConfig(*config)
    return load().gmm_fp8_fwd_swiglu_quant_tiled(_p(xq), _p(xs), _p(wq), _p(ws), _p(group_sizes), G, M, K, N,
                                                 _p(h), _p(hq), _p(hs), _p(workspace), workspace_bytes, _s(stream),
                                                 ctypes.byref(config) if config is not None else None)


def _cfg(config):
    if config is None:
        return None
    if not isinstance(config, TileConfig):
        config = TileConfig(*config)
    return ctypes.byref(config)


def gmm_quantize_rhs_w4(w, G, K, N, wq4, ws, stream=None) -> int:
    return load().gmm_quantize_rhs_w4(_p(w), G, K, N, _p(wq4), _p(ws), _s(stream))


def gmm_fp8_w4_fwd(xq, xs, wq4, ws, group_sizes, G, M, K, N, fuse_silu_mul, out, workspace, workspace_bytes,
                   stream=None, config=None) -> int:
    return load().gmm_fp8_w4_fwd(_p(xq), _p(xs), _p(wq4), _p(ws), _p(group_sizes), G, M, K, N, int(fuse_silu_mul),
                                 _p(out), _p(workspace), workspace_bytes, _s(stream), _cfg(config))


def gmm_fp8_w4_fwd_swiglu_quant(xq, xs, wq4, ws, group_sizes, G, M, K, N, h, hq, hs, workspace, workspace_bytes,
                                stream=None, config=None) -> int:
    return load().gmm_fp8_w4_fwd_swiglu_quant(_p(xq), _p(xs), _p(wq4), _p(ws), _p(group_sizes), G, M, K, N, _p(h),
                                              _p(hq), _p(hs), _p(workspace), workspace_bytes, _s(stream),
                                              _cfg(config))


def gmm_bf16_fwd(x, w, group_sizes, G, M, K, N, fuse_silu_mul, out, workspace, workspace_bytes,
                 stream=None) -> int:
    return load().gmm_bf16_fwd(_p(x), _p(w), _p(group_sizes), G, M, K, N, int(fuse_silu_mul),
                               _p(out), _p(workspace), workspace_bytes, _s(stream))


def gmm_bf16_dgrad(dy, w, group_sizes, G, M, K, N, dx, workspace, workspace_bytes, stream=None) -> int:
    return load().gmm_bf16_dgrad(_p(dy), _p(w), _p(group_sizes), G, M, K, N, _p(dx), _p(workspace),
                                 workspace_bytes, _s(stream))


def tgmm_bf16(x, dy, group_sizes, G, M, K, N, dw, workspace, workspace_bytes, stream=None) -> int:
    return load().tgmm_bf16(_p(x), _p(dy), _p(group_sizes), G, M, K, N, _p(dw), _p(workspace),
                            workspace_bytes, _s(stream))


def tgmm_bf16_tiled(x, dy, group_sizes, G, M, K, N, dw, workspace, workspace_bytes, stream=None,
                    config=None) -> int:
    """config: a TgmmConfig, a (stages, claim_ahead, max_batch) tuple, or None (defaults)."""
    if config is not None and not isinstance(config, TgmmConfig):
        config = TgmmConfig(*config)
    return load().tgmm_bf16_tiled(_p(x), _p(dy), _p(group_sizes), G, M, K, N, _p(dw), _p(workspace),
                                  workspace_bytes, _s(stream), ctypes.byref(config) if config is not None else None)


def gmm_get_device_status(workspace, stream=None) -> int:
    return load().gmm_get_device_status(_p(workspace), _s(stream))


def gmm_selftest_wait_timeout(workspace, workspace_bytes, limit_ms, stream=None) -> int:
    return load().gmm_selftest_wait_timeout(_p(workspace), workspace_bytes, int(limit_ms), _s(stream))


def gmm_fp8_fwd_noalloc(xq, xs, wq, ws, group_sizes, G, M, K, N, fuse_silu_mul, out,
                        stream=None) -> int:
    """gmm_fp8_fwd for callers that cannot allocate: no workspace argument;
    the metadata lives in the library's static device array (see gmm.h)."""
    return load().gmm_fp8_fwd_noalloc(_p(xq), _p(xs), _p(wq), _p(ws), _p(group_sizes), G, M, K, N,
                                      int(fuse_silu_mul), _p(out), _s(stream))


# ---------------------------------------------------------------------------
# convenience wrappers: allocate outputs with torch, call the C entry points
# ---------------------------------------------------------------------------

class Workspace:
    """A zero-initialised device workspace sized for (G, M)."""

    def __init__(self, G: int, M: int, device="cuda"):
        self.G, self.M = G, M
        self.nbytes = gmm_workspace_bytes(G, M)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    def fits(self, G: int, M: int) -> bool:
        return gmm_workspace_bytes(G, M) <= self.nbytes

    def status(self, stream=None) -> int:
        return gmm_get_device_status(self.buf, stream)

    def header(self) -> list[int]:
        return self.buf[:16].view(torch.int32).tolist()

    def offsets(self) -> list[int]:
        return self.buf[32:32 + 4 * (self.G + 1)].view(torch.int32).tolist()

    def tiles(self) -> torch.Tensor:
        n = self.header()[3]
        off = gmm_tiles_offset(self.G)
        return self.buf[off:off + 16 * n].view(torch.int32).view(n, 4)[:, :3]

    def _order_offset(self) -> int:
        return gmm_tiles_offset(self.G) + 16 * ((self.M + 127) // 128 + self.G)

    def order(self) -> list[int]:
        """The group ids sorted by size, largest first (ties by id)."""
        off = self._order_offset()
        return self.buf[off:off + 4 * self.G].view(torch.int32).tolist()

    def pair_tiles(self) -> torch.Tensor:
        """The 256-row tiles {g, row0, row1} (the CTA-pair FP8 kernel's)."""
        n = self.buf[24:28].view(torch.int32).item()
        off = self._order_offset() + 16 * ((self.G + 3) // 4)
        return self.buf[off:off + 16 * n].view(torch.int32).view(n, 4)[:, :3]


def _ws(ws, G, M, device):
    if ws is None or not ws.fits(G, M):
        ws = Workspace(G, M, device)
    return ws


def _ws_for(group_sizes, ws, G, M, device):
    """Workspace of a grouped call.  group_sizes=None reuses the metadata that
    an earlier call (or group_metadata) left in `ws`, so `ws` must be given."""
    if group_sizes is None:
        if ws is None or not ws.fits(G, M):
            raise ValueError("group_sizes=None reuses the metadata in `workspace`: pass that workspace")
        return ws
    return _ws(ws, G, M, device)


def quantize_lhs(x: torch.Tensor, stream=None):
    """x bf16 [M, K] -> (xq uint8 [M, K] e4m3 codes, xs float32 [K/128, M])."""
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    xs = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    _check(gmm_quantize_lhs(x, M, K, xq, xs, stream), "gmm_quantize_lhs")
    return xq, xs


def quantize_rhs(w: torch.Tensor, stream=None):
    """w bf16 [G, K, N] -> (wq uint8 [G, N, K] e4m3 codes, ws float32 [G, K/128, N/128])."""
    G, K, N = w.shape
    wq = torch.empty((G, N, K), dtype=torch.uint8, device=w.device)
    ws = torch.empty((G, K // 128, N // 128), dtype=torch.float32, device=w.device)
    _check(gmm_quantize_rhs(w, G, K, N, wq, ws, stream), "gmm_quantize_rhs")
    return wq, ws


def quantize_rhs_w4(w: torch.Tensor, stream=None):
    """w bf16 [G, K, N] -> (wq4 uint8 [G, N, K/2] packed E2M1 codes, ws float32 [G, K/128, N/128])."""
    G, K, N = w.shape
    wq4 = torch.empty((G, N, K // 2), dtype=torch.uint8, device=w.device)
    ws = torch.empty((G, K // 128, N // 128), dtype=torch.float32, device=w.device)
    _check(gmm_quantize_rhs_w4(w, G, K, N, wq4, ws, stream), "gmm_quantize_rhs_w4")
    return wq4, ws


def fp8_w4_fwd(xq, xs, wq4, ws, group_sizes, fuse=False, out=None, workspace=None, stream=None, config=None):
    """The FP8 forward with 4-bit weights (wq4 [G, Nw, K/2] from quantize_rhs_w4)."""
    M, K = xq.shape
    G, Nw, K2 = wq4.shape
    assert 2 * K2 == K
    N = Nw // 2 if fuse else Nw
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    ws_ = _ws_for(group_sizes, workspace, G, M, xq.device)
    _check(gmm_fp8_w4_fwd(xq, xs, wq4, ws, group_sizes, G, M, K, N, fuse, out, ws_.buf, ws_.nbytes, stream, config),
           "gmm_fp8_w4_fwd")
    return out


def fp8_w4_fwd_swiglu_quant(xq, xs, wq4, ws, group_sizes, with_h=True, workspace=None, stream=None, config=None,
                            out=None):
    """Fused wi with 4-bit weights: returns (h or None, hq, hs) as fp8_fwd_swiglu_quant."""
    M, K = xq.shape
    G, Nw, K2 = wq4.shape
    assert 2 * K2 == K
    N = Nw // 2
    if out is not None:
        h, hq, hs = out
    else:
        h = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device) if with_h else None
        hq = torch.empty((M, N), dtype=torch.uint8, device=xq.device)
        hs = torch.empty((N // 128, M), dtype=torch.float32, device=xq.device)
    ws_ = _ws_for(group_sizes, workspace, G, M, xq.device)
    _check(gmm_fp8_w4_fwd_swiglu_quant(xq, xs, wq4, ws, group_sizes, G, M, K, N, h, hq, hs, ws_.buf, ws_.nbytes,
                                       stream, config), "gmm_fp8_w4_fwd_swiglu_quant")
    return h, hq, hs


def fp8_fwd(xq, xs, wq, ws, group_sizes, fuse=False, out=None, workspace=None, stream=None, config=None):
    """config: a tile configuration (see TileConfig), or None for the defaults."""
    M, K = xq.shape
    G, Nw, K2 = wq.shape
    assert K2 == K
    N = Nw // 2 if fuse else Nw
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    ws_ = _ws_for(group_sizes, workspace, G, M, xq.device)
    if config is None:
        _check(gmm_fp8_fwd(xq, xs, wq, ws, group_sizes, G, M, K, N, fuse, out, ws_.buf, ws_.nbytes,
                           stream), "gmm_fp8_fwd")
    else:
        _check(gmm_fp8_fwd_tiled(xq, xs, wq, ws, group_sizes, G, M, K, N, fuse, out, ws_.buf, ws_.nbytes,
                                 stream, config), "gmm_fp8_fwd_tiled")
    return out


def fp8_fwd_swiglu_quant(xq, xs, wq, ws, group_sizes, with_h=True, workspace=None, stream=None, config=None,
                         out=None):
    """Fused wi: returns (h or None, hq [M, N] e4m3 codes, hs [N/128, M]).
    config: a tile configuration (see TileConfig), or None for the defaults;
    out: an (h, hq, hs) triple to write into instead of new tensors."""
    M, K = xq.shape
    G, Nw, K2 = wq.shape
    assert K2 == K
    N = Nw // 2
    if out is not None:
        h, hq, hs = out
    else:
        h = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device) if with_h else None
        hq = torch.empty((M, N), dtype=torch.uint8, device=xq.device)
        hs = torch.empty((N // 128, M), dtype=torch.float32, device=xq.device)
    ws_ = _ws_for(group_sizes, workspace, G, M, xq.device)
    if config is None:
        _check(gmm_fp8_fwd_swiglu_quant(xq, xs, wq, ws, group_sizes, G, M, K, N, h, hq, hs, ws_.buf, ws_.nbytes,
                                        stream), "gmm_fp8_fwd_swiglu_quant")
    else:
        _check(gmm_fp8_fwd_swiglu_quant_tiled(xq, xs, wq, ws, group_sizes, G, M, K, N, h, hq, hs, ws_.buf,
                                              ws_.nbytes, stream, config), "gmm_fp8_fwd_swiglu_quant_tiled")
    return h, hq, hs


def bf16_fwd(x, w, group_sizes, fuse=False, out=None, workspace=None, stream=None):
    M, K = x.shape
    G, K2, Nw = w.shape
    assert K2 == K
    N = Nw // 2 if fuse else Nw
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_ = _ws_for(group_sizes, workspace, G, M, x.device)
    _check(gmm_bf16_fwd(x, w, group_sizes, G, M, K, N, fuse, out, ws_.buf, ws_.nbytes, stream),
           "gmm_bf16_fwd")
    return out


def dgrad(dy, w, group_sizes, dx=None, workspace=None, stream=None):
    """dx [M, K] = dy [M, N] . w[g]^T per group, w [G, K, N]."""
    M, N = dy.shape
    G, K, N2 = w.shape
    assert N2 == N
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    ws_ = _ws_for(group_sizes, workspace, G, M, dy.device)
    _check(gmm_bf16_dgrad(dy, w, group_sizes, G, M, K, N, dx, ws_.buf, ws_.nbytes, stream), "gmm_bf16_dgrad")
    return dx


def tgmm(x, dy, group_sizes, dw=None, workspace=None, stream=None, config=None):
    M, K = x.shape
    M2, N = dy.shape
    assert M2 == M
    if group_sizes is not None:
        G = group_sizes.numel()
    elif dw is not None:
        G = dw.shape[0]
    elif workspace is not None:
        G = workspace.G
    else:
        raise ValueError("group_sizes=None reuses the metadata in `workspace`: pass that workspace")
    if dw is None:
        dw = torch.empty((G, K, N), dtype=torch.bfloat16, device=x.device)
    ws_ = _ws_for(group_sizes, workspace, G, M, x.device)
    if config is None:
        _check(tgmm_bf16(x, dy, group_sizes, G, M, K, N, dw, ws_.buf, ws_.nbytes, stream), "tgmm_bf16")
    else:
        _check(tgmm_bf16_tiled(x, dy, group_sizes, G, M, K, N, dw, ws_.buf, ws_.nbytes, stream, config),
               "tgmm_bf16_tiled")
    return dw


def group_metadata(group_sizes, M, workspace=None, stream=None) -> Workspace:
    G = group_sizes.numel()
    ws_ = _ws(workspace, G, M, group_sizes.device)
    _check(gmm_group_metadata(group_sizes, G, M, ws_.buf, ws_.nbytes, stream), "gmm_group_metadata")
    return ws_
