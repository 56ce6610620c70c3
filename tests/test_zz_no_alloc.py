"""dsa_indexer_score_noalloc: the indexer scan for callers that cannot pass a
workspace -- code that captures a stream into a CUDA graph (no allocation is
allowed during capture), decode loops that must not enter the allocator (it
may synchronise the device), and hosts that own every allocation.  Its
scratch is a fixed array inside the library, shared by all calls on a GPU.

This test calls it twice in a row through the C ABI, with different shapes so
that the second call starts from the first call's leftovers, the first with
a status word of the caller's and the second with none (the status then lives
in the array).  Both calls run the same kernels on the same inputs as
dsa_indexer_score with a workspace, so their scores must be bit-identical to
it; the first case is also checked against the float64 oracle.

This file is collected last on purpose: a run that stops at its first failure
has run every other test before this one."""
import ctypes

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


def test_noalloc_matches_workspace_entry_point_twice(lib, oracle_mod):
    import dsa_sparse_attention_lightning_gb300 as dsa
    cases = [
        (inputs.Workload("na1", [5000, 700, 3000], [4, 1, 3], H=16, seed=21, shift_frac=0.05),
         True),
        (inputs.Workload("na2", [1500, 9000], [2, 1], H=16, seed=22, q_idx_fp8=True), False),
    ]
    for wl, own_status in cases:                # two calls in a row, on the shared array
        inp = inputs.make_inputs(wl, device="cuda")
        ref = dsa.dsa_indexer_score(inp["q_idx"], inp["w"], inp["key_cache"],
                                    inp["block_table"], inp["row_req"], inp["row_len"],
                                    q_scale=inp["q_idx_scale"])
        got = torch.full_like(ref, float("nan"))
        status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda") if own_status else None
        assert _noalloc(lib, inp, got, status) == 0
        torch.cuda.synchronize()
        if own_status:
            assert int(status.item()) == 0
        lens = inp["row_len"].cpu().tolist()
        for r, L in enumerate(lens):              # same kernels, same inputs: same bits
            assert torch.equal(got[r, :L], ref[r, :L]), f"{wl.name} row {r}: scores differ"
        if own_status:
            host = inputs.to_numpy(inp)
            ora = oracle_mod.indexer_scores(host["q_idx"], host["w"], host["key_cache"],
                                            host["block_table"], host["row_req"],
                                            host["row_len"], q_scale=host["q_idx_scale"])
            helpers.assert_scores_close(got.cpu().numpy(), ora, host["row_len"])


def test_noalloc_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(1 << 20)             # never dereferenced: validation fails first
    call = lambda R, st=None: lib.dsa_indexer_score_noalloc(
        fake, 0, None, fake, fake, 4, fake, 1, 4, fake, fake, R, fake, 256, st, None)
    assert call(65) == 2                        # DSA_NOALLOC_MAX_ROWS + 1
    assert call(2, ctypes.c_void_p((1 << 20) + 2)) == 1   # status word not 4-byte aligned
