"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/gmm.h declares, and rejects bad arguments on
the host before any CUDA call is made."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gmm.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_blockwise_quantized_gb300 import build as b
    b.build()
    import fp8_blockwise_quantized_gb300 as g
    return g.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared()
    for need in ["gmm_quantize_lhs", "gmm_fp8_fwd", "gmm_bf16_fwd", "tgmm_bf16", "gmm_quantize_rhs",
                 "gmm_group_metadata", "gmm_workspace_bytes", "gmm_get_device_status"]:
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    from fp8_blockwise_quantized_gb300 import LIB_PATH, EXPORTED
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared():
        assert name in exported, f"{name} declared in gmm.h but not exported"
        assert hasattr(lib, name)
    assert sorted(EXPORTED) == sorted(_declared())


def test_status_strings(lib):
    for code in range(9):
        s = lib.gmm_status_string(code).decode()
        assert s.startswith("GMM_")
    assert "unknown" in lib.gmm_status_string(99).decode()


def test_workspace_size(lib):
    for G, M in [(1, 0), (4, 512), (32, 8192), (256, 65536), (4096, 1)]:
        n = lib.gmm_workspace_bytes(G, M)
        tiles = (M + 127) // 128 + G
        assert n >= 32 + 4 * (G + 1) + 16 * tiles
        off = lib.gmm_tiles_offset(G)
        assert off % 16 == 0 and off >= 32 + 4 * (G + 1)
        pair_tiles = (M + 255) // 256 + G
        # + the size-ordered group ids, + the 256-row tiles
        assert n == off + 16 * tiles + (4 * G + 15) // 16 * 16 + 16 * pair_tiles
    assert lib.gmm_workspace_bytes(0, 10) == 0


FAKE = 1 << 20  # an aligned non-null pointer value; never dereferenced on the host


def _fp8(lib, **kw):
    a = dict(xq=FAKE, xs=FAKE, wq=FAKE, ws=FAKE, gs=FAKE, G=4, M=512, K=256, N=256, fuse=0, out=FAKE,
             work=FAKE, wbytes=1 << 20)
    a.update(kw)
    return lib.gmm_fp8_fwd(a["xq"], a["xs"], a["wq"], a["ws"], a["gs"], a["G"], a["M"], a["K"], a["N"],
                           a["fuse"], a["out"], a["work"], a["wbytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(K=100), 2), (dict(N=0), 2), (dict(G=0), 2), (dict(G=5000), 2), (dict(M=-1), 2),
    (dict(M=1 << 31), 2), (dict(wq=None), 1), (dict(out=None), 1), (dict(gs=FAKE + 4), 3),
    (dict(xq=FAKE + 8), 3), (dict(out=FAKE + 2), 3), (dict(work=None), 8), (dict(wbytes=16), 8),
    (dict(work=FAKE + 4), 3),
])
def test_fp8_host_validation(lib, kw, code):
    assert _fp8(lib, **kw) == code


def _tiled(lib, cfg, **kw):
    import ctypes
    from fp8_blockwise_quantized_gb300 import TileConfig
    a = dict(xq=FAKE, xs=FAKE, wq=FAKE, ws=FAKE, gs=FAKE, G=4, M=512, K=256, N=256, fuse=0, out=FAKE,
             work=FAKE, wbytes=1 << 20)
    a.update(kw)
    return lib.gmm_fp8_fwd_tiled(a["xq"], a["xs"], a["wq"], a["ws"], a["gs"], a["G"], a["M"], a["K"], a["N"],
                                 a["fuse"], a["out"], a["work"], a["wbytes"], None, ctypes.byref(TileConfig(*cfg)))


@pytest.mark.parametrize("cfg,kw,code", [
    ((64, 0, 0), {}, 4), ((256, 0, 0), dict(N=384), 4), ((128, 0, 0), dict(fuse=1), 4),
    ((0, -1, 0), {}, 4), ((0, 0, 3), {}, 4), ((0, 0, -1), {}, 4),
    ((256, 0, 2), dict(K=100), 2), ((128, 0, 1), dict(wq=None), 1),
    # CTA pairs: 256-column units (not with bn 128 or N % 256 != 0), even CTA counts
    ((0, 0, 0, 2), dict(N=384), 4), ((128, 0, 0, 2), {}, 4), ((0, 7, 0, 2), {}, 4), ((0, 0, 0, 3), {}, 4),
    ((0, 0, 0, -1), {}, 4),
    # compiled ring depths and TMEM buffer counts only
    ((256, 0, 0, 1, 4, 0), {}, 4), ((128, 0, 0, 1, 2, 0), {}, 4), ((0, 0, 0, 0, 0, 3), {}, 4),
    ((256, 0, 0, 1, 0, 4), {}, 4), ((0, 0, 0, 2, 5, 0), {}, 4), ((0, 0, 0, 2, 0, 2), {}, 4),
    ((0, 0, 0, 0, -1, 0), {}, 4),
])
def test_tile_config_host_validation(lib, cfg, kw, code):
    # rejected on the host, before any device call
    assert _tiled(lib, cfg, **kw) == code


@pytest.mark.parametrize("cfg", [(3, 0, 0), (7, 0, 0), (0, 13, 0), (0, -1, 0), (0, 0, 5), (0, 0, -2)])
def test_tgmm_config_host_validation(lib, cfg):
    import ctypes
    from fp8_blockwise_quantized_gb300 import TgmmConfig
    # rejected on the host, before any device call
    assert lib.tgmm_bf16_tiled(FAKE, FAKE, FAKE, 4, 512, 256, 256, FAKE, FAKE, 1 << 20, None,
                               ctypes.byref(TgmmConfig(*cfg))) == 4


def test_null_group_sizes_is_not_a_host_error(lib):
    # group_sizes = NULL reuses the workspace's metadata: shape errors are still
    # reported first, and a missing weight is still a null-pointer error
    assert _fp8(lib, gs=None, K=100) == 2
    assert _fp8(lib, gs=None, wq=None) == 1
    assert lib.tgmm_bf16(FAKE, FAKE, None, 4, 512, 256, 256, None, FAKE, 1 << 20, None) == 1


def test_host_validation_other_calls(lib):
    # quantize: shape / null / alignment
    assert lib.gmm_quantize_lhs(FAKE, 10, 100, FAKE, FAKE, None) == 2
    assert lib.gmm_quantize_lhs(None, 10, 128, FAKE, FAKE, None) == 1
    assert lib.gmm_quantize_lhs(FAKE + 1, 10, 128, FAKE, FAKE, None) == 3
    assert lib.gmm_quantize_lhs(None, 0, 128, None, None, None) == 0  # empty: nothing to do
    assert lib.gmm_quantize_rhs(FAKE, 2, 128, 130, FAKE, FAKE, None) == 2
    assert lib.gmm_quantize_rhs(FAKE, 2, 128, 128, None, FAKE, None) == 1
    # bf16 fwd and tgmm
    assert lib.gmm_bf16_fwd(FAKE, FAKE, FAKE, 4, 512, 256, 200, 0, FAKE, FAKE, 1 << 20, None) == 2
    assert lib.gmm_bf16_fwd(FAKE, None, FAKE, 4, 512, 256, 256, 0, FAKE, FAKE, 1 << 20, None) == 1
    assert lib.tgmm_bf16(FAKE, FAKE, FAKE, 4, 512, 256, 256, None, FAKE, 1 << 20, None) == 1
    assert lib.tgmm_bf16(FAKE, FAKE, FAKE, 4, 512, 256, 256, FAKE, FAKE, 8, None) == 8
    assert lib.gmm_group_metadata(None, 4, 512, FAKE, 1 << 20, None) == 1
    assert lib.gmm_get_device_status(None, None) == 8


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import fp8_blockwise_quantized_gb300.binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        b.load()
