"""dsa_indexer_score_noalloc: the indexer scan for callers that cannot pass a
workspace (stream capture, allocator-free decode loops, hosts that own all
allocation).  Its scratch is a fixed array inside the library, shared by all
calls on a GPU; this test calls it twice in a row through the C ABI, with
different shapes so that the second call starts from the first call's
leftovers, and checks both against dsa_indexer_score with a workspace.

This file is collected last on purpose: a run that stops at its first failure
has run every other test before this one."""
import ctypes

import numpy as np
import pytest
import torch

import helpers
from dsa_sparse_attention_lightning_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_attention_lightning_gb300 import _build, _lib
    _build.build()
    return _lib.load()


def _noalloc(lib, inp, scores, dev_status=None):
    q_idx = inp["q_idx"]
    bt = inp["block_table"]
    B, max_pages = bt.shape
    R = inp["row_len"].shape[0]
    qt = 0 if q_idx.dtype == torch.bfloat16 else 1
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.dsa_indexer_score_noalloc(
        p(q_idx), qt, p(inp["q_idx_scale"]), p(inp["w"]), p(inp["key_cache"]),
        inp["key_cache"].numel() // 8448, p(bt), B, max_pages, p(inp["row_req"]),
        p(inp["row_len"]), R, p(scores), scores.shape[1], p(dev_status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice(lib):
    import dsa_sparse_attention_lightning_gb300 as dsa
    cases = [
        inputs.Workload("na1", [5000, 700, 3000], [4, 1, 3], H=16, seed=21, shift_frac=0.05),
        inputs.Workload("na2", [1500, 9000], [2, 1], H=16, seed=22, q_idx_fp8=True),
    ]
    for wl in cases:                           # two calls in a row, on the shared array
        inp = inputs.make_inputs(wl, device="cuda")
        ref = dsa.dsa_indexer_score(inp["q_idx"], inp["w"], inp["key_cache"],
                                    inp["block_table"], inp["row_req"], inp["row_len"],
                                    q_scale=inp["q_idx_scale"])
        got = torch.full_like(ref, float("nan"))
        status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, inp, got, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        lens = inp["row_len"].cpu().numpy()
        helpers.assert_scores_close(got.cpu().numpy(), ref.cpu().numpy(), lens)


def test_noalloc_rejects_too_many_rows(lib):
    R = 65                                      # DSA_NOALLOC_MAX_ROWS + 1
    fake = ctypes.c_void_p(1 << 20)
    assert lib.dsa_indexer_score_noalloc(fake, 0, None, fake, fake, 4, fake, 1, 4, fake, fake, R,
                                         fake, 256, None, None) == 2
