"""ctypes binding of libdsa (include/dsa.h).

Argument marshalling only: every function here takes torch tensors, checks
their dtype, shape and device, and passes raw pointers and the current CUDA
stream to the C entry point of the same name.  All work runs in libdsa's
kernels.  There is no fallback: if libdsa.so is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DSA_OK = 0
DSA_ERR_DEVICE_CHECK = 5
DSA_BF16 = 0
DSA_E4M3 = 1
PAGE = 64
IDX_HEADS = 32
IDX_DIM = 128
KEY_PAGE_BYTES = 8448
MXFP4_KEY_PAGE_BYTES = 4352   # 64 x 64 E2M1 code bytes, then 64 x 4 E8M0 scale bytes
LAT_DIM = 576
V_DIM = 512
NVFP4_ROW_BYTES = 352

# (name, restype, argtypes) of every exported symbol, in header order.
P, I32, I64, SZ, F32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = [
    ("dsa_version", I32, []),
    ("dsa_status_string", ctypes.c_char_p, [I32]),
    ("dsa_last_cuda_error", I32, []),
    ("dsa_last_cuda_error_string", ctypes.c_char_p, []),
    ("dsa_device_info", I32, [P, P, P]),
    ("dsa_indexer_score_workspace_size", SZ, [I32]),
    ("dsa_indexer_score", I32, [P, I32, P, P, P, I64, P, I32, I32, P, P, I32, P, I64, P, SZ, P]),
    ("dsa_indexer_score_mxfp4", I32, [P, P, P, P, I64, P, I32, I32, P, P, I32, P, I64, P, SZ, P]),
    ("dsa_indexer_score_noalloc", I32, [P, I32, P, P, P, I64, P, I32, I32, P, P, I32, P, I64, P,
                                        P]),
    ("dsa_topk_workspace_size", SZ, [I32, I64, I32]),
    ("dsa_topk", I32, [P, I64, P, I32, I64, I32, P, P, SZ, P]),
    ("dsa_write_kv", I32, [P, P, P, F32, P, F32, P, I32, I32, P, P, I32, P, P, I64, P, P]),
    ("dsa_write_kv_mxfp4", I32, [P, P, P, F32, P, F32, P, I32, I32, P, P, I32, P, P, I64, P, P]),
    ("dsa_topk_dcp_workspace_size", SZ, [I32, I64, I32, I32]),
    ("dsa_topk_dcp", I32, [P, I64, P, I32, I64, I32, I32, P, P, P, SZ, P]),
    ("dsa_sparse_mla_workspace_size", SZ, [I32, I32, I32]),
    ("dsa_sparse_mla_decode", I32, [P, I32, F32, P, I64, F32, P, I32, I32, P, P, P, I32, I32, P,
                                    P, P, SZ, P]),
    ("dsa_sparse_mla_decode_nvfp4", I32, [P, I32, F32, P, I64, F32, P, I32, I32, P, P, P, I32,
                                          I32, P, P, P, SZ, P]),
    ("dsa_decode_step_workspace_size", SZ, [I32, I32, I32, I32, I32]),
    ("dsa_decode_step", I32, [P, I32, P, P, P, P, I64, F32, P, I32, I32, P, P, I32, P, I32, F32,
                              I32, P, P, P, P, SZ, P]),
    ("dsa_decode_step_fp4", I32, [P, P, P, P, P, I64, F32, P, I32, I32, P, P, I32, P, I32, F32,
                                  I32, P, P, P, P, SZ, P]),
    ("dsa_check_device_status", I32, [P, P, P]),
    ("dsa_selftest_workspace_size", SZ, []),
    ("dsa_selftest_bounded_wait", I32, [I32, P, SZ, P]),
]

_lock = threading.Lock()
_lib = None


class DSAError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: status {status} ({text})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libdsa.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                                  "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().dsa_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != DSA_OK:
        text = status_string(status)
        if status == 4:
            text += ": " + load().dsa_last_cuda_error_string().decode()
        raise DSAError(fn, status, text)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def version() -> int:
    return int(load().dsa_version())


def device_info():
    n, a, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("dsa_device_info", load().dsa_device_info(ctypes.byref(n), ctypes.byref(a),
                                                     ctypes.byref(b)))
    return n.value, a.value, b.value


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is None:
        return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    _need(workspace, "workspace", torch.uint8, device)
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace has {workspace.numel()} bytes, needs {nbytes}")
    return workspace


def _q_idx_type(q_idx: torch.Tensor) -> int:
    if q_idx.dtype == torch.bfloat16:
        return DSA_BF16
    if q_idx.dtype == torch.uint8:
        return DSA_E4M3
    raise TypeError("q_idx must be bfloat16 or uint8 (E4M3 codes)")


def indexer_score_workspace_size(R: int) -> int:
    return int(load().dsa_indexer_score_workspace_size(int(R)))


def dsa_indexer_score(q_idx, w, key_cache, block_table, row_req, row_len, *, q_scale=None,
                      scores=None, workspace=None):
    """fp32 scores [R, max_pages*64]; entries at or past row_len are left unwritten."""
    dev = key_cache.device
    R = row_len.shape[0]
    B, max_pages = block_table.shape
    qt = _q_idx_type(q_idx)
    _need(w, "w", torch.float32, dev)
    _need(key_cache, "key_cache", torch.uint8, dev)
    for n, t in (("block_table", block_table), ("row_req", row_req), ("row_len", row_len)):
        _need(t, n, torch.int32, dev)
    if q_scale is not None:
        _need(q_scale, "q_scale", torch.float32, dev)
    ld = max_pages * PAGE
    if scores is None:
        scores = torch.empty((R, ld), dtype=torch.float32, device=dev)
    _need(scores, "scores", torch.float32, dev)
    ws = _workspace(indexer_score_workspace_size(R), dev, workspace)
    _check("dsa_indexer_score", load().dsa_indexer_score(
        _ptr(q_idx), qt, _ptr(q_scale), _ptr(w), _ptr(key_cache), key_cache.numel() // KEY_PAGE_BYTES,
        _ptr(block_table), B, max_pages, _ptr(row_req), _ptr(row_len), R, _ptr(scores),
        scores.shape[1], _ptr(ws), ws.numel(), _stream(dev)))
    return scores


def dsa_indexer_score_mxfp4(q_codes, q_scales, w, key_cache, block_table, row_req, row_len, *,
                            scores=None, workspace=None):
    """fp32 scores [R, max_pages*64] over MXFP4 keys and an MXFP4 query.

    ``q_codes`` uint8 [R,32,64] (E2M1, dim 2j in the low nibble of byte j),
    ``q_scales`` uint8 [R,32,4] (E8M0), ``key_cache`` uint8 pages of
    MXFP4_KEY_PAGE_BYTES.  Entries at or past row_len are left unwritten."""
    dev = key_cache.device
    R = row_len.shape[0]
    B, max_pages = block_table.shape
    _need(q_codes, "q_codes", torch.uint8, dev)
    _need(q_scales, "q_scales", torch.uint8, dev)
    _need(w, "w", torch.float32, dev)
    _need(key_cache, "key_cache", torch.uint8, dev)
    for n, t in (("block_table", block_table), ("row_req", row_req), ("row_len", row_len)):
        _need(t, n, torch.int32, dev)
    ld = max_pages * PAGE
    if scores is None:
        scores = torch.empty((R, ld), dtype=torch.float32, device=dev)
    _need(scores, "scores", torch.float32, dev)
    ws = _workspace(indexer_score_workspace_size(R), dev, workspace)
    _check("dsa_indexer_score_mxfp4", load().dsa_indexer_score_mxfp4(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), _ptr(key_cache),
        key_cache.numel() // MXFP4_KEY_PAGE_BYTES, _ptr(block_table), B, max_pages,
        _ptr(row_req), _ptr(row_len), R, _ptr(scores), scores.shape[1], _ptr(ws), ws.numel(),
        _stream(dev)))
    return scores


def topk_workspace_size(R: int, max_len: int, k: int) -> int:
    return int(load().dsa_topk_workspace_size(int(R), int(max_len), int(k)))


def dsa_topk(scores, row_len, k, *, max_len=None, idx=None, workspace=None):
    """int32 [R, k]: selected positions in ascending order, -1 padded."""
    dev = scores.device
    _need(scores, "scores", torch.float32, dev)
    _need(row_len, "row_len", torch.int32, dev)
    R, ld = scores.shape
    max_len = ld if max_len is None else int(max_len)
    if idx is None:
        idx = torch.empty((R, k), dtype=torch.int32, device=dev)
    _need(idx, "idx", torch.int32, dev)
    ws = _workspace(topk_workspace_size(R, max_len, k), dev, workspace)
    _check("dsa_topk", load().dsa_topk(_ptr(scores), ld, _ptr(row_len), R, max_len, int(k),
                                       _ptr(idx), _ptr(ws), ws.numel(), _stream(dev)))
    return idx


def dsa_write_kv(k_raw, gamma, beta, eps, latent, latent_scale, block_table, tok_req, tok_pos,
                 key_cache, latent_cache, *, dev_status=None, mxfp4_keys=False):
    """The Write step: new tokens' index keys and latent rows into the caches (in place).

    With ``mxfp4_keys`` the index keys go to pages of MXFP4_KEY_PAGE_BYTES
    (dsa_write_kv_mxfp4)."""
    dev = key_cache.device
    _need(k_raw, "k_raw", torch.bfloat16, dev)
    _need(latent, "latent", torch.bfloat16, dev)
    _need(gamma, "gamma", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(key_cache, "key_cache", torch.uint8, dev)
    _need(latent_cache, "latent_cache", torch.uint8, dev)
    for n, t in (("block_table", block_table), ("tok_req", tok_req), ("tok_pos", tok_pos)):
        _need(t, n, torch.int32, dev)
    T = k_raw.shape[0]
    B, max_pages = block_table.shape
    num_pages = key_cache.numel() // (MXFP4_KEY_PAGE_BYTES if mxfp4_keys else KEY_PAGE_BYTES)
    name = "dsa_write_kv_mxfp4" if mxfp4_keys else "dsa_write_kv"
    _check(name, getattr(load(), name)(
        _ptr(k_raw), _ptr(gamma), _ptr(beta), float(eps), _ptr(latent), float(latent_scale),
        _ptr(block_table), B, max_pages, _ptr(tok_req), _ptr(tok_pos), T, _ptr(key_cache),
        _ptr(latent_cache), num_pages, _ptr(dev_status) if dev_status is not None else None,
        _stream(dev)))
    return key_cache, latent_cache


def topk_dcp_workspace_size(R: int, max_len: int, k: int, W: int) -> int:
    return int(load().dsa_topk_dcp_workspace_size(int(R), int(max_len), int(k), int(W)))


def dsa_topk_dcp(scores, row_len, k, W, *, max_len=None, idx=None, resend=None, workspace=None):
    """(idx int32 [R, k], resend uint32 [R]): dsa_topk by the context-parallel exchange."""
    dev = scores.device
    _need(scores, "scores", torch.float32, dev)
    _need(row_len, "row_len", torch.int32, dev)
    R, ld = scores.shape
    max_len = ld if max_len is None else int(max_len)
    if idx is None:
        idx = torch.empty((R, k), dtype=torch.int32, device=dev)
    if resend is None:
        resend = torch.empty((R,), dtype=torch.int32, device=dev)
    _need(idx, "idx", torch.int32, dev)
    _need(resend, "resend", torch.int32, dev)
    ws = _workspace(topk_dcp_workspace_size(R, max_len, k, W), dev, workspace)
    _check("dsa_topk_dcp", load().dsa_topk_dcp(_ptr(scores), ld, _ptr(row_len), R, max_len, int(k),
                                               int(W), _ptr(idx), _ptr(resend), _ptr(ws),
                                               ws.numel(), _stream(dev)))
    return idx, resend


def sparse_mla_workspace_size(R: int, H: int, k: int) -> int:
    return int(load().dsa_sparse_mla_workspace_size(int(R), int(H), int(k)))


def dsa_sparse_mla_decode(q, latent_cache, latent_scale, block_table, row_req, row_len, idx, *,
                          softmax_scale, out=None, lse=None, workspace=None):
    """bf16 out [R,H,512] and fp32 lse [R,H] of attention over the selected rows."""
    return _sparse_mla("dsa_sparse_mla_decode", LAT_DIM, q, latent_cache, latent_scale,
                       block_table, row_req, row_len, idx, softmax_scale, out, lse, workspace)


def dsa_sparse_mla_decode_nvfp4(q, latent_cache, latent_scale, block_table, row_req, row_len,
                                idx, *, softmax_scale, out=None, lse=None, workspace=None):
    """As dsa_sparse_mla_decode over an NVFP4 latent cache uint8 [pages, 64, 352]."""
    return _sparse_mla("dsa_sparse_mla_decode_nvfp4", NVFP4_ROW_BYTES, q, latent_cache,
                       latent_scale, block_table, row_req, row_len, idx, softmax_scale, out, lse,
                       workspace)


def _sparse_mla(fn, row_bytes, q, latent_cache, latent_scale, block_table, row_req, row_len, idx,
                softmax_scale, out, lse, workspace):
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(latent_cache, "latent_cache", torch.uint8, dev)
    _need(idx, "idx", torch.int32, dev)
    for n, t in (("block_table", block_table), ("row_req", row_req), ("row_len", row_len)):
        _need(t, n, torch.int32, dev)
    R, H, _ = q.shape
    k = idx.shape[1]
    B, max_pages = block_table.shape
    if out is None:
        out = torch.empty((R, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    ws = _workspace(sparse_mla_workspace_size(R, H, k), dev, workspace)
    _check(fn, getattr(load(), fn)(
        _ptr(q), H, float(softmax_scale), _ptr(latent_cache),
        latent_cache.numel() // (PAGE * row_bytes), float(latent_scale), _ptr(block_table), B,
        max_pages, _ptr(row_req), _ptr(row_len), _ptr(idx), k, R, _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel(), _stream(dev)))
    return out, lse


def decode_step_workspace_size(B: int, R: int, max_pages: int, H: int, k: int) -> int:
    return int(load().dsa_decode_step_workspace_size(int(B), int(R), int(max_pages), int(H),
                                                     int(k)))


def dsa_decode_step(q_idx, w, key_cache, latent_cache, latent_scale, block_table, row_req,
                    row_len, q, *, softmax_scale, k=2048, q_scale=None, out=None, lse=None,
                    idx_out=None, workspace=None):
    """The whole step (Score -> Select -> Attend); returns (out, lse)."""
    dev = q.device
    qt = _q_idx_type(q_idx)
    _need(q, "q", torch.bfloat16, dev)
    _need(w, "w", torch.float32, dev)
    _need(key_cache, "key_cache", torch.uint8, dev)
    _need(latent_cache, "latent_cache", torch.uint8, dev)
    for n, t in (("block_table", block_table), ("row_req", row_req), ("row_len", row_len)):
        _need(t, n, torch.int32, dev)
    if q_scale is not None:
        _need(q_scale, "q_scale", torch.float32, dev)
    R, H, _ = q.shape
    B, max_pages = block_table.shape
    num_pages = key_cache.numel() // KEY_PAGE_BYTES
    if latent_cache.numel() != num_pages * PAGE * LAT_DIM:
        raise ValueError("key_cache and latent_cache must hold the same number of pages")
    if out is None:
        out = torch.empty((R, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=dev)
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32, dev)
    ws = _workspace(decode_step_workspace_size(B, R, max_pages, H, k), dev, workspace)
    _check("dsa_decode_step", load().dsa_decode_step(
        _ptr(q_idx), qt, _ptr(q_scale), _ptr(w), _ptr(key_cache), _ptr(latent_cache), num_pages,
        float(latent_scale), _ptr(block_table), B, max_pages, _ptr(row_req), _ptr(row_len), R,
        _ptr(q), H, float(softmax_scale), int(k), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws),
        ws.numel(), _stream(dev)))
    return out, lse


def dsa_decode_step_fp4(q_codes, q_scales, w, key_cache, latent_cache, latent_scale, block_table,
                        row_req, row_len, q, *, softmax_scale, k=2048, out=None, lse=None,
                        idx_out=None, workspace=None):
    """The whole step over MXFP4 index keys (pages of MXFP4_KEY_PAGE_BYTES) and
    NVFP4 latent rows (uint8 [pages, 64, 352]) with an MXFP4 indexer query
    (``q_codes`` uint8 [R,32,64], ``q_scales`` uint8 [R,32,4]); returns (out, lse)."""
    dev = q.device
    _need(q_codes, "q_codes", torch.uint8, dev)
    _need(q_scales, "q_scales", torch.uint8, dev)
    _need(q, "q", torch.bfloat16, dev)
    _need(w, "w", torch.float32, dev)
    _need(key_cache, "key_cache", torch.uint8, dev)
    _need(latent_cache, "latent_cache", torch.uint8, dev)
    for n, t in (("block_table", block_table), ("row_req", row_req), ("row_len", row_len)):
        _need(t, n, torch.int32, dev)
    R, H, _ = q.shape
    B, max_pages = block_table.shape
    num_pages = key_cache.numel() // MXFP4_KEY_PAGE_BYTES
    if latent_cache.numel() != num_pages * PAGE * NVFP4_ROW_BYTES:
        raise ValueError("key_cache and latent_cache must hold the same number of pages")
    if out is None:
        out = torch.empty((R, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=dev)
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32, dev)
    ws = _workspace(decode_step_workspace_size(B, R, max_pages, H, k), dev, workspace)
    _check("dsa_decode_step_fp4", load().dsa_decode_step_fp4(
        _ptr(q_codes), _ptr(q_scales), _ptr(w), _ptr(key_cache), _ptr(latent_cache), num_pages,
        float(latent_scale), _ptr(block_table), B, max_pages, _ptr(row_req), _ptr(row_len), R,
        _ptr(q), H, float(softmax_scale), int(k), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws),
        ws.numel(), _stream(dev)))
    return out, lse


def check_device_status(workspace: torch.Tensor) -> int:
    """Synchronise and return the device status bits of the last call using ``workspace``."""
    bits = ctypes.c_uint32(0)
    st = load().dsa_check_device_status(_ptr(workspace), _stream(workspace.device),
                                        ctypes.byref(bits))
    if st not in (DSA_OK, DSA_ERR_DEVICE_CHECK):
        _check("dsa_check_device_status", st)
    return int(bits.value)


def selftest_workspace_size() -> int:
    return int(load().dsa_selftest_workspace_size())


def selftest_bounded_wait(wait_us: int, workspace: torch.Tensor) -> None:
    """Enqueue the library's bounded-wait self-test on the current stream.

    One CTA waits ``wait_us`` microseconds on a barrier nothing arrives on,
    raises the timeout bit in ``workspace``'s status word, drains its bulk copy
    of ``workspace[256:512]`` into ``workspace[512:768]`` and frees its tensor
    memory.  Read the result with :func:`check_device_status`.
    """
    _need(workspace, "workspace", torch.uint8)
    if workspace.device.type != "cuda":
        raise ValueError("workspace must be CUDA device memory")
    _check("dsa_selftest_bounded_wait", load().dsa_selftest_bounded_wait(
        int(wait_us), _ptr(workspace), workspace.numel(), _stream(workspace.device)))
