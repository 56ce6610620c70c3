"""GPU parity of dsa_decode_step_fp4: the fused step over MXFP4 index keys and
NVFP4 latent rows (the pages' 10,080-byte-per-token configuration).

The fused step runs the same kernels as the separate calls
(dsa_indexer_score_mxfp4, dsa_topk, dsa_sparse_mla_decode_nvfp4), so its
selection and its output must equal theirs bit for bit; the selection is also
checked against the float64 oracle's (outside near-ties) and the attention
output against the oracle's on the step's own selection."""
import numpy as np
import pytest
import torch

import helpers
from dsa_sparse_attention_lightning_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
MX_PAGE = 4352


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dsa_sparse_attention_lightning_gb300 as m
    from dsa_sparse_attention_lightning_gb300 import _build
    _build.build()
    m.load()
    return m


def _mx_bytes(g, shape_codes, shape_scales):
    """Random MXFP4 bytes: uniform E2M1 code bytes, E8M0 scales 2^-3 .. 2^3."""
    codes = torch.randint(0, 256, shape_codes, generator=g, device=DEV, dtype=torch.int32)
    scales = torch.randint(124, 131, shape_scales, generator=g, device=DEV, dtype=torch.int32)
    return codes.to(torch.uint8), scales.to(torch.uint8)


def _fp4_inputs(wl):
    inp = inputs.make_inputs(wl, device=DEV)
    nv, nls = inputs.nvfp4_latent_cache(inp, wl)
    num_pages = inp["key_cache"].shape[0]
    g = torch.Generator(device=DEV).manual_seed(7919 * wl.seed + 5)
    kc, ks = _mx_bytes(g, (num_pages, 64 * 64), (num_pages, 64 * 4))
    key_cache = torch.cat([kc, ks], dim=1).contiguous()
    qc, qs = _mx_bytes(g, (wl.R, 32, 64), (wl.R, 32, 4))
    return inp, nv, nls, key_cache, qc.contiguous(), qs.contiguous()


def _run(dsa, wl, inp, nv, nls, key_cache, qc, qs):
    idx = torch.full((wl.R, wl.k), -7, dtype=torch.int32, device=DEV)
    out, lse = dsa.dsa_decode_step_fp4(qc, qs, inp["w"], key_cache, nv, nls, inp["block_table"],
                                       inp["row_req"], inp["row_len"], inp["q"],
                                       softmax_scale=inp["softmax_scale"], k=wl.k, idx_out=idx)
    scores = dsa.dsa_indexer_score_mxfp4(qc, qs, inp["w"], key_cache, inp["block_table"],
                                         inp["row_req"], inp["row_len"])
    ref_idx = dsa.dsa_topk(scores, inp["row_len"], wl.k)
    ref_out, ref_lse = dsa.dsa_sparse_mla_decode_nvfp4(
        inp["q"], nv, nls, inp["block_table"], inp["row_req"], inp["row_len"], ref_idx,
        softmax_scale=inp["softmax_scale"])
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_idx)
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    return idx, out, lse, scores


def _check_oracle(oracle_mod, wl, inp, nv, nls, key_cache, qc, qs, idx, out, lse, scores, rows):
    host = inputs.to_numpy({k: inp[k] for k in ("w", "block_table", "row_req", "row_len", "q")})
    sub = {k: np.ascontiguousarray(host[k][rows]) for k in ("w", "row_req", "row_len", "q")}
    ld = scores.shape[1]
    ora_s = oracle_mod.indexer_scores_mx(qc[rows].cpu().numpy(), qs[rows].cpu().numpy(), sub["w"],
                                         key_cache.cpu().numpy(), host["block_table"],
                                         sub["row_req"], sub["row_len"], ld=ld)
    helpers.assert_scores_close(scores[rows].cpu().numpy(), ora_s, sub["row_len"])
    ora_idx = oracle_mod.topk(ora_s, sub["row_len"], wl.k)
    gi = idx[rows].cpu().numpy()
    helpers.assert_topk_equal_outside_near_ties(gi, ora_idx, ora_s, sub["row_len"], wl.k)
    oo, ol = oracle_mod.sparse_mla_nvfp4(sub["q"], inp["softmax_scale"], nv.cpu().numpy(), nls,
                                         host["block_table"], sub["row_req"], sub["row_len"],
                                         np.ascontiguousarray(gi))
    helpers.assert_out_close(out[rows].float().cpu().numpy(), oo)
    lg = lse[rows].cpu().numpy()
    fin = np.isfinite(ol)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.allclose(lg[fin], ol[fin], rtol=1e-4, atol=1e-4)


CASES = [
    inputs.Workload("fp4_ragged", [3000, 700, 5000, 64], [2, 1, 4, 1], H=64, k=512, seed=61),
    inputs.Workload("fp4_short_h16", [1, 63, 65, 2047, 2049], [1, 1, 2, 1, 3], H=16, seed=62),
    inputs.Workload("fp4_wide_h32", [6000, 3000], [11, 5], H=32, k=1024, seed=63),
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_fp4_step_matches_separate_calls_and_oracle(dsa, oracle_mod, wl):
    args = _fp4_inputs(wl)
    idx, out, lse, scores = _run(dsa, wl, *args)
    _check_oracle(oracle_mod, wl, *args, idx, out, lse, scores, list(range(wl.R)))


def test_fp4_step_full_size_sampled_rows(dsa, oracle_mod):
    """16 requests x 4 rows at 256K context, H = 64: every row against the
    separate calls, two sampled rows against the oracle."""
    wl = inputs.config(2)
    args = _fp4_inputs(wl)
    del args[0]["latent_cache"]
    idx, out, lse, scores = _run(dsa, wl, *args)
    _check_oracle(oracle_mod, wl, *args, idx, out, lse, scores, [0, wl.R - 1])
