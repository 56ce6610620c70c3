"""Python access to the float64 CPU oracle (``dsa_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition of one DSA
decode step (indexer scores, top-k, sparse MLA) that the CUDA library is
checked against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It never imports the
CUDA package, and the CUDA package never imports it.

``build()`` compiles ``dsa_oracle.c`` with the host C compiler (float64,
OpenMP) into ``liboracle.so`` next to this file.  The functions below only
marshal numpy arrays into the C calls; all arithmetic is in the C file.
``decode_step`` chains the three C calls in the order the pages give (score,
select, attend), selecting on the float64 scores.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PAGE = 64
IDX_HEADS = 32
IDX_DIM = 128
KEY_PAGE_BYTES = PAGE * IDX_DIM + PAGE * 4
MX_BLOCK = 32
MX_KEY_BYTES = IDX_DIM // 2
MX_SCALES = IDX_DIM // MX_BLOCK
MX_KEY_PAGE_BYTES = PAGE * (MX_KEY_BYTES + MX_SCALES)
LAT_DIM = 576
V_DIM = 512
NV_BLOCK = 16
NV_ROW_BYTES = V_DIM // 2 + V_DIM // NV_BLOCK + (LAT_DIM - V_DIM)   # 352


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle.so`` (skipped when up to date)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = dbl
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_indexer_scores.argtypes = [P, P, P, P, P, i64, P, i32, i32, P, P, i32, P, i64]
        lib.oracle_indexer_scores.restype = ctypes.c_int
        lib.oracle_topk.argtypes = [P, i64, P, i32, i32, P]
        lib.oracle_topk.restype = ctypes.c_int
        lib.oracle_topk_dcp.argtypes = [P, i64, P, i32, i32, i32, P, P]
        lib.oracle_topk_dcp.restype = ctypes.c_int
        lib.oracle_e4m3_encode.argtypes = [dbl]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_write_kv.argtypes = [P, P, P, dbl, P, dbl, P, i32, i32, P, P, i32, P, P, i64,
                                        P, P, P]
        lib.oracle_write_kv.restype = ctypes.c_int
        lib.oracle_sparse_mla.argtypes = [P, i32, dbl, P, i64, dbl, P, i32, i32, P, P, P, i32, i32,
                                          P, P]
        lib.oracle_sparse_mla.restype = ctypes.c_int
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_decode.restype = dbl
        lib.oracle_e2m1_encode.argtypes = [dbl]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_decode.restype = dbl
        lib.oracle_mx_quantize.argtypes = [P, ctypes.c_int, P, P]
        lib.oracle_mx_quantize.restype = ctypes.c_int
        lib.oracle_write_key_mx.argtypes = [P, P, P, dbl, P, i32, i32, P, P, i32, P, i64, P]
        lib.oracle_write_key_mx.restype = ctypes.c_int
        lib.oracle_indexer_scores_mx.argtypes = [P, P, P, P, i64, P, i32, i32, P, P, i32, P, i64]
        lib.oracle_indexer_scores_mx.restype = ctypes.c_int
        lib.oracle_nvfp4_latent_decode.argtypes = [P, dbl, P]
        lib.oracle_nvfp4_latent_decode.restype = None
        lib.oracle_nvfp4_latent_encode.argtypes = [P, P]
        lib.oracle_nvfp4_latent_encode.restype = None
        lib.oracle_sparse_mla_nvfp4.argtypes = [P, i32, dbl, P, i64, dbl, P, i32, i32, P, P, P,
                                                i32, i32, P, P]
        lib.oracle_sparse_mla_nvfp4.restype = ctypes.c_int
        _lib = lib
        return lib


def _c(a, dtype):
    """Contiguous numpy array of the given dtype (no copy when already so)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def e4m3_decode(code: int) -> float:
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def indexer_scores(q_idx, w, key_cache, block_table, row_req, row_len, *, q_scale=None,
                   ld=None):
    """Float64 scores [R, ld]; entries past row_len are NaN.

    ``q_idx`` is uint16 bf16 bits [R,32,128], or uint8 E4M3 codes [R,32,128]
    together with ``q_scale`` fp32 [R,32].
    """
    lib = _load()
    q_idx = np.asarray(q_idx)
    R = int(np.asarray(row_len).shape[0])
    row_len = _c(row_len, np.int32)
    row_req = _c(row_req, np.int32)
    block_table = _c(block_table, np.int32)
    B, max_pages = block_table.shape
    ld = int(ld if ld is not None else max(1, int(row_len.max(initial=0))))
    scores = np.full((R, ld), np.nan, dtype=np.float64)
    key_cache = _c(key_cache, np.uint8)
    num_pages = key_cache.size // KEY_PAGE_BYTES
    w = _c(w, np.float32)
    if q_idx.dtype == np.uint16:
        qb, q8, qs = _c(q_idx, np.uint16), None, None
    else:
        qb, q8, qs = None, _c(q_idx, np.uint8), _c(q_scale, np.float32)
    st = lib.oracle_indexer_scores(_ptr(qb), _ptr(q8), _ptr(qs), _ptr(w), _ptr(key_cache),
                                   num_pages, _ptr(block_table), B, max_pages, _ptr(row_req),
                                   _ptr(row_len), R, _ptr(scores), ld)
    if st != 0:
        raise ValueError(f"oracle_indexer_scores failed with status {st}")
    return scores


def topk(scores, row_len, k):
    """int32 [R, k] positions in rank order (score desc, index asc), -1 padded."""
    lib = _load()
    scores = _c(scores, np.float64)
    R, ld = scores.shape
    row_len = _c(row_len, np.int32)
    idx = np.empty((R, k), dtype=np.int32)
    st = lib.oracle_topk(_ptr(scores), ld, _ptr(row_len), R, int(k), _ptr(idx))
    if st != 0:
        raise ValueError(f"oracle_topk failed with status {st}")
    return idx


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def write_kv(k_raw, gamma, beta, eps, latent, latent_scale, block_table, tok_req, tok_pos,
             key_cache, latent_cache):
    """The Write step on copies of the caches.

    ``k_raw`` uint16 bf16 bits [T,128], ``latent`` uint16 bf16 bits [T,576].
    Returns (key_cache, latent_cache, key_pre [T,128], lat_pre [T,576],
    key_scale [T]): the written caches and the float64 values before rounding."""
    lib = _load()
    k_raw = _c(k_raw, np.uint16)
    latent = _c(latent, np.uint16)
    T = k_raw.shape[0]
    block_table = _c(block_table, np.int32)
    B, max_pages = block_table.shape
    key_cache = np.array(key_cache, dtype=np.uint8, copy=True, order="C")
    latent_cache = np.array(latent_cache, dtype=np.uint8, copy=True, order="C")
    num_pages = key_cache.size // KEY_PAGE_BYTES
    key_pre = np.zeros((T, IDX_DIM))
    lat_pre = np.zeros((T, LAT_DIM))
    key_scale = np.zeros(T)
    st = lib.oracle_write_kv(_ptr(k_raw), _ptr(_c(gamma, np.float64)), _ptr(_c(beta, np.float64)),
                             float(eps), _ptr(latent), float(latent_scale), _ptr(block_table), B,
                             max_pages, _ptr(_c(tok_req, np.int32)), _ptr(_c(tok_pos, np.int32)), T,
                             _ptr(key_cache), _ptr(latent_cache), num_pages, _ptr(key_pre),
                             _ptr(lat_pre), _ptr(key_scale))
    if st != 0:
        raise ValueError(f"oracle_write_kv failed with status {st}")
    return key_cache, latent_cache, key_pre, lat_pre, key_scale


def e2m1_decode(nibble: int) -> float:
    return float(_load().oracle_e2m1_decode(int(nibble) & 0xF))


def e2m1_encode(x: float) -> int:
    return int(_load().oracle_e2m1_encode(float(x)))


def e8m0_decode(code: int) -> float:
    return float(_load().oracle_e8m0_decode(int(code) & 0xFF))


def mx_quantize(v):
    """MXFP4 of float64 values [..., n] (n a multiple of 32).

    Returns (codes uint8 [..., n/2], two per byte, low nibble first; scales
    uint8 E8M0 [..., n/32])."""
    lib = _load()
    v = _c(v, np.float64)
    n = v.shape[-1]
    flat = v.reshape(-1, n)
    codes = np.zeros((flat.shape[0], n // 2), dtype=np.uint8)
    scales = np.zeros((flat.shape[0], n // MX_BLOCK), dtype=np.uint8)
    for i in range(flat.shape[0]):
        st = lib.oracle_mx_quantize(_ptr(flat[i]), n, _ptr(codes[i]), _ptr(scales[i]))
        if st != 0:
            raise ValueError(f"oracle_mx_quantize failed with status {st}")
    return codes.reshape(v.shape[:-1] + (n // 2,)), scales.reshape(v.shape[:-1] + (n // MX_BLOCK,))


def write_key_mx(k_raw, gamma, beta, eps, block_table, tok_req, tok_pos, key_cache):
    """The Write step of MXFP4 index keys on a copy of the key cache.

    Returns (key_cache, key_pre [T,128]): the written cache and the float64
    normalized keys."""
    lib = _load()
    k_raw = _c(k_raw, np.uint16)
    T = k_raw.shape[0]
    block_table = _c(block_table, np.int32)
    B, max_pages = block_table.shape
    key_cache = np.array(key_cache, dtype=np.uint8, copy=True, order="C")
    num_pages = key_cache.size // MX_KEY_PAGE_BYTES
    key_pre = np.zeros((T, IDX_DIM))
    st = lib.oracle_write_key_mx(_ptr(k_raw), _ptr(_c(gamma, np.float64)),
                                 _ptr(_c(beta, np.float64)), float(eps), _ptr(block_table), B,
                                 max_pages, _ptr(_c(tok_req, np.int32)),
                                 _ptr(_c(tok_pos, np.int32)), T, _ptr(key_cache), num_pages,
                                 _ptr(key_pre))
    if st != 0:
        raise ValueError(f"oracle_write_key_mx failed with status {st}")
    return key_cache, key_pre


def indexer_scores_mx(q_codes, q_scales, w, key_cache, block_table, row_req, row_len, *,
                      ld=None):
    """Float64 scores [R, ld] over MXFP4 keys; entries past row_len are NaN.

    ``q_codes`` uint8 [R,32,64] packed E2M1, ``q_scales`` uint8 E8M0 [R,32,4],
    ``key_cache`` pages of MX_KEY_PAGE_BYTES."""
    lib = _load()
    R = int(np.asarray(row_len).shape[0])
    row_len = _c(row_len, np.int32)
    row_req = _c(row_req, np.int32)
    block_table = _c(block_table, np.int32)
    B, max_pages = block_table.shape
    ld = int(ld if ld is not None else max(1, int(row_len.max(initial=0))))
    scores = np.full((R, ld), np.nan, dtype=np.float64)
    key_cache = _c(key_cache, np.uint8)
    num_pages = key_cache.size // MX_KEY_PAGE_BYTES
    st = lib.oracle_indexer_scores_mx(_ptr(_c(q_codes, np.uint8)), _ptr(_c(q_scales, np.uint8)),
                                      _ptr(_c(w, np.float32)), _ptr(key_cache), num_pages,
                                      _ptr(block_table), B, max_pages, _ptr(row_req),
                                      _ptr(row_len), R, _ptr(scores), ld)
    if st != 0:
        raise ValueError(f"oracle_indexer_scores_mx failed with status {st}")
    return scores


def nvfp4_latent_encode(v):
    """NVFP4 latent rows (uint8 [..., 352]) of float64 values [..., 576]
    already divided by the per-tensor scale."""
    lib = _load()
    v = _c(v, np.float64)
    flat = v.reshape(-1, LAT_DIM)
    rows = np.zeros((flat.shape[0], NV_ROW_BYTES), dtype=np.uint8)
    for i in range(flat.shape[0]):
        lib.oracle_nvfp4_latent_encode(_ptr(flat[i]), _ptr(rows[i]))
    return rows.reshape(v.shape[:-1] + (NV_ROW_BYTES,))


def nvfp4_latent_decode(rows, latent_scale):
    """float64 [..., 576] values of NVFP4 latent rows uint8 [..., 352]."""
    lib = _load()
    rows = _c(rows, np.uint8)
    flat = rows.reshape(-1, NV_ROW_BYTES)
    out = np.zeros((flat.shape[0], LAT_DIM))
    for i in range(flat.shape[0]):
        lib.oracle_nvfp4_latent_decode(_ptr(flat[i]), float(latent_scale), _ptr(out[i]))
    return out.reshape(rows.shape[:-1] + (LAT_DIM,))


def sparse_mla_nvfp4(q, softmax_scale, latent_cache, latent_scale, block_table, row_req,
                     row_len, idx):
    """(out float64 [R,H,512], lse float64 [R,H]) over NVFP4 latent pages
    (uint8 [pages][64][352])."""
    lib = _load()
    q = _c(q, np.uint16)
    R, H, _ = q.shape
    idx = _c(idx, np.int32)
    k = idx.shape[1]
    latent_cache = _c(latent_cache, np.uint8)
    num_pages = latent_cache.size // (PAGE * NV_ROW_BYTES)
    block_table = _c(block_table, np.int32)
    B, max_pages = block_table.shape
    out = np.zeros((R, H, V_DIM))
    lse = np.zeros((R, H))
    st = lib.oracle_sparse_mla_nvfp4(_ptr(q), H, float(softmax_scale), _ptr(latent_cache),
                                     num_pages, float(latent_scale), _ptr(block_table), B,
                                     max_pages, _ptr(_c(row_req, np.int32)),
                                     _ptr(_c(row_len, np.int32)), _ptr(idx), k, R, _ptr(out),
                                     _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle_sparse_mla_nvfp4 failed with status {st}")
    return out, lse


def topk_dcp(scores, row_len, k, W):
    """Top-k by the decode-context-parallel exchange over W token shards.

    Returns (idx int32 [R, k] in rank order, -1 padded; resend uint32 [R],
    bit s set when shard s's full local top-k was gathered)."""
    lib = _load()
    scores = _c(scores, np.float64)
    R, ld = scores.shape
    row_len = _c(row_len, np.int32)
    idx = np.empty((R, k), dtype=np.int32)
    resend = np.empty(R, dtype=np.uint32)
    st = lib.oracle_topk_dcp(_ptr(scores), ld, _ptr(row_len), R, int(k), int(W), _ptr(idx),
                             _ptr(resend))
    if st != 0:
        raise ValueError(f"oracle_topk_dcp failed with status {st}")
    return idx, resend


def sparse_mla(q, softmax_scale, latent_cache, latent_scale, block_table, row_req, row_len, idx):
    """Float64 (out [R,H,512], lse [R,H]) of exact attention over the selected rows.

    ``q`` is uint16 bf16 bits [R,H,576]; ``idx`` int32 [R,k] (-1 = unused slot).
    """
    lib = _load()
    q = _c(q, np.uint16)
    R, H, _ = q.shape
    idx = _c(idx, np.int32)
    k = idx.shape[1]
    block_table = _c(block_table, np.int32)
    B, max_pages = block_table.shape
    latent_cache = _c(latent_cache, np.uint8)
    num_pages = latent_cache.size // (PAGE * LAT_DIM)
    out = np.zeros((R, H, V_DIM), dtype=np.float64)
    lse = np.zeros((R, H), dtype=np.float64)
    st = lib.oracle_sparse_mla(_ptr(q), H, float(softmax_scale), _ptr(latent_cache), num_pages,
                               float(latent_scale), _ptr(block_table), B, max_pages,
                               _ptr(_c(row_req, np.int32)), _ptr(_c(row_len, np.int32)), _ptr(idx),
                               k, R, _ptr(out), _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle_sparse_mla failed with status {st}")
    return out, lse


def decode_step(inp, k=2048):
    """Score -> select -> attend for one decode step, all in the oracle.

    ``inp`` is a mapping of numpy arrays with the keys produced by the input
    generator (``q_idx``, ``w``, ``key_cache``, ``block_table``, ``row_req``,
    ``row_len``, ``q``, ``latent_cache``, ``latent_scale``, ``softmax_scale``
    and optionally ``q_idx_scale``).  Returns (scores, idx, out, lse), all
    float64 except idx.
    """
    scores = indexer_scores(inp["q_idx"], inp["w"], inp["key_cache"], inp["block_table"],
                            inp["row_req"], inp["row_len"], q_scale=inp.get("q_idx_scale"))
    idx = topk(np.nan_to_num(scores, nan=0.0), inp["row_len"], k)
    out, lse = sparse_mla(inp["q"], inp["softmax_scale"], inp["latent_cache"],
                          inp["latent_scale"], inp["block_table"], inp["row_req"],
                          inp["row_len"], idx)
    return scores, idx, out, lse
