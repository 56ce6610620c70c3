"""CPU-only checks of the C ABI: the library builds, loads and exports every
symbol include/dsa.h declares, workspace sizes are consistent, and invalid
arguments are rejected on the host before anything touches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    from dsa_sparse_attention_lightning_gb300 import _build, _lib
    _build.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(dsa_\w+)\s*\(", text, re.M)))


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ("dsa_indexer_score", "dsa_topk", "dsa_sparse_mla_decode", "dsa_decode_step",
              "dsa_sparse_mla_decode_nvfp4", "dsa_topk_workspace_size",
              "dsa_check_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from dsa_sparse_attention_lightning_gb300 import _lib
    bound = {n for n, _, _ in _lib.SIGNATURES}
    for name in declared_symbols():
        assert hasattr(lib, name), f"libdsa.so does not export {name}"
        assert name in bound, f"python binding does not bind {name}"


def test_version_and_status_strings(lib):
    assert lib.dsa_version() >= 10000
    for s in range(6):
        assert lib.dsa_status_string(s)
    assert lib.dsa_status_string(0) == b"ok"


def test_workspace_sizes(lib):
    # per row: a threshold, a count, one (offset, count) pair per 2048-score
    # chunk and room for 8192 (key, position) candidates (longer candidate
    # lists fall back to a pass over the scores)
    assert lib.dsa_topk_workspace_size(4, 1000, 64) >= 4 * 8192 * 8
    grow = lib.dsa_topk_workspace_size(8, 1 << 20, 2048) - lib.dsa_topk_workspace_size(8, 1 << 10, 2048)
    assert 0 < grow <= 8 * 512 * 8 + 256
    assert lib.dsa_sparse_mla_workspace_size(64, 64, 2048) >= 64 * 64 * 512 * 4
    assert lib.dsa_decode_step_workspace_size(16, 64, 512, 64, 2048) >= \
        lib.dsa_topk_workspace_size(64, 512 * 64, 2048)
    assert lib.dsa_indexer_score_workspace_size(-1) == 0
    assert lib.dsa_topk_workspace_size(4, 100, 0) == 0


FAKE = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: validation fails first


def test_topk_rejects_bad_arguments(lib):
    ws_need = lib.dsa_topk_workspace_size(2, 128, 16)
    # k out of range
    assert lib.dsa_topk(FAKE, 128, FAKE, 2, 128, 0, FAKE, FAKE, ws_need, None) == 1
    assert lib.dsa_topk(FAKE, 128, FAKE, 2, 128, 4096, FAKE, FAKE, ws_need, None) == 2
    # ld smaller than max_len, or not a multiple of 4
    assert lib.dsa_topk(FAKE, 64, FAKE, 2, 128, 16, FAKE, FAKE, ws_need, None) == 1
    assert lib.dsa_topk(FAKE, 130, FAKE, 2, 128, 16, FAKE, FAKE, ws_need, None) == 1
    # missing pointers, missing or small workspace
    assert lib.dsa_topk(None, 128, FAKE, 2, 128, 16, FAKE, FAKE, ws_need, None) == 1
    assert lib.dsa_topk(FAKE, 128, FAKE, 2, 128, 16, FAKE, None, ws_need, None) == 3
    assert lib.dsa_topk(FAKE, 128, FAKE, 2, 128, 16, FAKE, FAKE, ws_need - 1, None) == 3
    assert lib.dsa_topk(FAKE, 128, FAKE, 2, 128, 16, FAKE, ctypes.c_void_p((1 << 20) + 8),
                        ws_need, None) == 3


def test_mla_and_step_reject_bad_shapes(lib):
    ws = lib.dsa_sparse_mla_workspace_size(1, 64, 64)
    args = lambda H, k: (FAKE, H, 0.1, FAKE, 4, 1.0, FAKE, 1, 4, FAKE, FAKE, FAKE, k, 1, FAKE,
                         None, FAKE, ws, None)
    assert lib.dsa_sparse_mla_decode(*args(48, 64)) == 2       # H not built
    assert lib.dsa_sparse_mla_decode(*args(64, 4096)) == 2     # k > 2048
    assert lib.dsa_sparse_mla_decode(*args(64, 0)) == 1
    for f in (lib.dsa_sparse_mla_decode, lib.dsa_sparse_mla_decode_nvfp4):
        assert f(*args(48, 64)) == 2
        assert f(*args(64, 4096)) == 2
        assert f(*args(64, 0)) == 1
        assert f(*args(64, 64)[:-3], FAKE, ws - 1, None) == 3          # workspace too small
    wss = lib.dsa_decode_step_workspace_size(1, 1, 4, 64, 64)
    step = lambda qt, H: (FAKE, qt, None, FAKE, FAKE, FAKE, 4, 1.0, FAKE, 1, 4, FAKE, FAKE, 1,
                          FAKE, H, 0.1, 64, FAKE, None, None, FAKE, wss, None)
    assert lib.dsa_decode_step(*step(7, 64)) == 2              # unknown q dtype
    assert lib.dsa_decode_step(*step(1, 64)) == 1              # E4M3 without q_scale
    assert lib.dsa_decode_step(*step(0, 24)) == 2
    step4 = lambda qs, H: (FAKE, qs, FAKE, FAKE, FAKE, 4, 1.0, FAKE, 1, 4, FAKE, FAKE, 1, FAKE,
                           H, 0.1, 64, FAKE, None, None, FAKE, wss, None)
    assert lib.dsa_decode_step_fp4(*step4(FAKE, 24)) == 2      # H not built
    assert lib.dsa_decode_step_fp4(*step4(None, 64)) == 1      # no MXFP4 query scales
    assert lib.dsa_indexer_score(FAKE, 0, None, FAKE, FAKE, 4, FAKE, 1, 4, FAKE, FAKE, 1, FAKE,
                                 100, FAKE, 1 << 20, None) == 1   # ld < max_pages * 64


def test_topk_dcp_rejects_bad_arguments(lib):
    ws = lib.dsa_topk_dcp_workspace_size(2, 128, 16, 8)
    assert ws > lib.dsa_topk_workspace_size(2, 128, 16)
    assert lib.dsa_topk_dcp_workspace_size(2, 128, 16, 0) == 0
    call = lambda k, W, ws_bytes=ws, R=2, work=FAKE: lib.dsa_topk_dcp(
        FAKE, 128, FAKE, R, 128, k, W, FAKE, None, work, ws_bytes, None)
    assert call(16, 0) == 1                          # no shards
    assert call(16, 33) == 2                         # more shards than the resend mask holds
    assert call(4096, 8) == 2                        # k > 2048
    assert call(0, 8) == 1
    assert call(16, 8, R=9000) == 2                  # R * W > 65535
    assert call(16, 8, ws_bytes=ws - 1) == 3
    assert call(16, 8, work=None) == 3


def test_write_kv_rejects_bad_arguments(lib):
    odd = ctypes.c_void_p((1 << 20) + 4)             # 4-byte aligned only
    call = lambda T=2, ls=1.0, eps=1e-6, k=FAKE, lat=FAKE, kc=FAKE: lib.dsa_write_kv(
        k, FAKE, FAKE, eps, lat, ls, FAKE, 1, 4, FAKE, FAKE, T, kc, FAKE, 4, None, None)
    assert call(T=-1) == 1
    assert call(ls=0.0) == 1 and call(ls=-2.0) == 1 and call(ls=float("inf")) == 1
    assert call(eps=-1.0) == 1
    assert call(k=None) == 1
    assert call(k=odd) == 1                          # k_raw must be 8-byte aligned
    assert call(lat=ctypes.c_void_p((1 << 20) + 8)) == 1   # latent must be 16-byte aligned
    assert call(kc=odd) == 1
    assert call(T=0) == 0                            # nothing to write: no GPU work at all


def test_write_kv_mxfp4_rejects_bad_arguments(lib):
    odd = ctypes.c_void_p((1 << 20) + 4)
    call = lambda T=2, ls=1.0, eps=1e-6, k=FAKE, kc=FAKE: lib.dsa_write_kv_mxfp4(
        k, FAKE, FAKE, eps, FAKE, ls, FAKE, 1, 4, FAKE, FAKE, T, kc, FAKE, 4, None, None)
    assert call(T=-1) == 1
    assert call(ls=0.0) == 1 and call(eps=-1.0) == 1
    assert call(k=None) == 1 and call(k=odd) == 1 and call(kc=odd) == 1
    assert call(T=0) == 0


def test_indexer_score_mxfp4_rejects_bad_arguments(lib):
    ws = lib.dsa_indexer_score_workspace_size(3)
    call = lambda R=3, qc=FAKE, qs=FAKE, ld=256, work=FAKE, ws_bytes=ws, mp=4: (
        lib.dsa_indexer_score_mxfp4(qc, qs, FAKE, FAKE, 8, FAKE, 2, mp, FAKE, FAKE, R, FAKE, ld,
                                    work, ws_bytes, None))
    assert call(R=-1) == 1
    assert call(R=70000) == 2
    assert call(qc=None) == 1 and call(qs=None) == 1
    assert call(qc=ctypes.c_void_p((1 << 20) + 8)) == 1    # codes must be 16-byte aligned
    assert call(qs=ctypes.c_void_p((1 << 20) + 2)) == 1    # scales must be 4-byte aligned
    assert call(ld=255) == 1 and call(ld=128) == 1          # ld % 4, ld < max_pages * 64
    assert call(work=None) == 3 and call(ws_bytes=ws - 1) == 3


def test_indexer_score_noalloc_rejects_bad_arguments(lib):
    call = lambda R=2, qt=0, st=None, ld=256, q=FAKE: lib.dsa_indexer_score_noalloc(
        q, qt, None, FAKE, FAKE, 4, FAKE, 1, 4, FAKE, FAKE, R, FAKE, ld, st, None)
    assert call(R=65) == 2                               # more rows than the fixed scratch holds
    assert call(st=ctypes.c_void_p((1 << 20) + 2)) == 1  # status word not 4-byte aligned
    assert call(qt=1) == 1                               # E4M3 query without its scales
    assert call(qt=5) == 2
    assert call(ld=255) == 1 and call(ld=128) == 1
    assert call(q=None) == 1


def test_selftest_rejects_bad_arguments(lib):
    need = lib.dsa_selftest_workspace_size()
    assert need >= 768
    assert lib.dsa_selftest_bounded_wait(0, FAKE, need, None) == 1          # wait_us < 1
    assert lib.dsa_selftest_bounded_wait(2_000_000, FAKE, need, None) == 1  # > 1 s
    assert lib.dsa_selftest_bounded_wait(100, None, need, None) == 3
    assert lib.dsa_selftest_bounded_wait(100, FAKE, need - 1, None) == 3


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from dsa_sparse_attention_lightning_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.load()
