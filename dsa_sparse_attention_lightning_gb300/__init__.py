"""One decode step of a DSA (DeepSeek-style sparse attention) layer on GB300.

The compute runs in libdsa.so (hand-written CUDA for sm_103a behind the C ABI
in include/dsa.h); this package holds its ctypes binding, the build script,
the seeded input generator and the byte model.
"""
from ._lib import (DSAError, check_device_status, decode_step_workspace_size, device_info,
                   dsa_decode_step, dsa_decode_step_fp4, dsa_indexer_score, dsa_indexer_score_mxfp4,
                   dsa_sparse_mla_decode, dsa_sparse_mla_decode_nvfp4, dsa_topk,
                   dsa_topk_dcp, dsa_write_kv, topk_dcp_workspace_size,
                   indexer_score_workspace_size, load, selftest_bounded_wait,
                   selftest_workspace_size, sparse_mla_workspace_size, topk_workspace_size,
                   version)

__all__ = [
    "DSAError", "check_device_status", "decode_step_workspace_size", "device_info",
    "dsa_decode_step", "dsa_decode_step_fp4", "dsa_indexer_score", "dsa_indexer_score_mxfp4", "dsa_sparse_mla_decode",
    "dsa_sparse_mla_decode_nvfp4", "dsa_topk",
    "dsa_topk_dcp", "dsa_write_kv", "topk_dcp_workspace_size",
    "indexer_score_workspace_size", "load", "selftest_bounded_wait", "selftest_workspace_size",
    "sparse_mla_workspace_size", "topk_workspace_size", "version",
]
