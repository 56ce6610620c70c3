"""GPU parity of dsa_sparse_mla_decode_nvfp4 (sparse MLA over 352-byte NVFP4
latent rows) against the float64 oracle: element by element on small
workloads (several tiles, ragged tails, scattered padding, one and two head
groups), with block scales inside and below the range the kernel splits
exactly, plus the device checks, and sampled rows at the benchmark's full
sizes."""
import numpy as np
import pytest
import torch

import helpers
from dsa_sparse_attention_lightning_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dsa_sparse_attention_lightning_gb300 as m
    from dsa_sparse_attention_lightning_gb300 import _build
    _build.build()
    m.load()
    return m


CASES = [
    inputs.Workload("nv_one_row", [4096], [1], H=16, seed=40, paged=False),
    inputs.Workload("nv_ragged", [3000, 700, 5000, 64], [2, 1, 4, 1], H=64, k=512, seed=41),
    inputs.Workload("nv_short", [1, 63, 65, 2047, 2049], [1, 1, 2, 1, 3], H=32, seed=42),
    inputs.Workload("nv_h128", [9000], [3], H=128, k=1024, seed=43),
    inputs.Workload("nv_many_rows_h16", [300, 1000, 257] * 20, [7] * 60, H=16, k=256, seed=44),
]


def _random_idx(host, k, seed):
    """Valid ids of each row scattered among -1 slots (all of a short row)."""
    rng = np.random.default_rng(seed)
    R = host["row_len"].shape[0]
    idx = np.full((R, k), -1, np.int32)
    for r, L in enumerate(host["row_len"]):
        n = min(k, int(L))
        sel = rng.choice(int(L), n, replace=False).astype(np.int32) if L else np.zeros(0, np.int32)
        idx[r, rng.choice(k, n, replace=False)] = sel
    return idx


def _check(dsa, oracle_mod, wl, inp, cache, lat_scale, idx, rows=None):
    out, lse = dsa.dsa_sparse_mla_decode_nvfp4(
        inp["q"], cache, lat_scale, inp["block_table"], inp["row_req"], inp["row_len"],
        torch.from_numpy(idx).to(DEV), softmax_scale=inp["softmax_scale"])
    torch.cuda.synchronize()
    rows = list(range(wl.R)) if rows is None else rows
    q = inp["q"][rows].cpu().view(torch.int16).numpy().view(np.uint16)
    oo, ol = oracle_mod.sparse_mla_nvfp4(
        q, inp["softmax_scale"], cache.cpu().numpy(), lat_scale,
        inp["block_table"].cpu().numpy(), inp["row_req"][rows].cpu().numpy(),
        inp["row_len"][rows].cpu().numpy(), np.ascontiguousarray(idx[rows]))
    err = helpers.assert_out_close(out[rows].float().cpu().numpy(), oo)
    lg = lse[rows].cpu().numpy()
    fin = np.isfinite(ol)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.allclose(lg[fin], ol[fin], rtol=1e-4, atol=1e-4)
    return err


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_sparse_mla_nvfp4_matches_oracle(dsa, oracle_mod, wl):
    inp = inputs.make_inputs(wl, device=DEV)
    cache, ls = inputs.nvfp4_latent_cache(inp, wl)
    idx = _random_idx(inputs.to_numpy({"row_len": inp["row_len"]}), wl.k, wl.seed)
    _check(dsa, oracle_mod, wl, inp, cache, ls, idx)


def test_sparse_mla_nvfp4_small_block_scales(dsa, oracle_mod):
    """Block scales from 2^-3 to 15: below 0.5 the two E4M3 terms round (at most
    2^-8 of latent_scale per element), above it they are exact."""
    wl = inputs.Workload("nv_scales", [5000, 1200], [3, 2], H=64, k=2048, seed=45)
    inp = inputs.make_inputs(wl, device=DEV)
    cache, ls = inputs.nvfp4_latent_cache(inp, wl, scale_bytes=(0x20, 0x58), latent_scale=1 / 32)
    idx = _random_idx(inputs.to_numpy({"row_len": inp["row_len"]}), wl.k, wl.seed)
    _check(dsa, oracle_mod, wl, inp, cache, ls, idx)


def test_sparse_mla_nvfp4_device_checks(dsa):
    wl = inputs.Workload("nv_bad", [300], [1], H=16, k=64, seed=46)
    inp = inputs.make_inputs(wl, device=DEV)
    cache, ls = inputs.nvfp4_latent_cache(inp, wl)
    ws = torch.empty(dsa.sparse_mla_workspace_size(1, 16, 5), dtype=torch.uint8, device=DEV)
    call = lambda bt, idx: dsa.dsa_sparse_mla_decode_nvfp4(
        inp["q"], cache, ls, bt, inp["row_req"], inp["row_len"], idx,
        softmax_scale=inp["softmax_scale"], workspace=ws)
    idx = torch.tensor([[0, 5, 299, 300, -1]], dtype=torch.int32, device=DEV)   # 300 >= len
    out, _ = call(inp["block_table"], idx)
    assert dsa.check_device_status(ws) & 0x4
    assert torch.isfinite(out.float()).all()
    bt = inp["block_table"].clone()
    bt[0, 2] = 10_000_000                        # page id out of range
    ok = torch.tensor([[0, 5, 130, 299, -1]], dtype=torch.int32, device=DEV)
    call(bt, ok)
    assert dsa.check_device_status(ws) & 0x2
    call(inp["block_table"], ok)                 # a clean call clears the word
    assert dsa.check_device_status(ws) == 0


def test_sparse_mla_nvfp4_deterministic(dsa):
    wl = CASES[1]
    inp = inputs.make_inputs(wl, device=DEV)
    cache, ls = inputs.nvfp4_latent_cache(inp, wl)
    idx = torch.from_numpy(_random_idx(inputs.to_numpy({"row_len": inp["row_len"]}), wl.k,
                                       wl.seed)).to(DEV)
    a = dsa.dsa_sparse_mla_decode_nvfp4(inp["q"], cache, ls, inp["block_table"], inp["row_req"],
                                        inp["row_len"], idx, softmax_scale=inp["softmax_scale"])
    b = dsa.dsa_sparse_mla_decode_nvfp4(inp["q"], cache, ls, inp["block_table"], inp["row_req"],
                                        inp["row_len"], idx, softmax_scale=inp["softmax_scale"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ----------------------------------------------- full benchmark sizes, sampled
@pytest.mark.parametrize("ci", [2, 3], ids=[inputs.config(i).name for i in (2, 3)])
def test_sparse_mla_nvfp4_full_size_sampled_rows(dsa, oracle_mod, ci):
    wl = inputs.config(ci)
    inp = inputs.make_inputs(wl, device=DEV)
    cache, ls = inputs.nvfp4_latent_cache(inp, wl)
    del inp["latent_cache"]
    idx = _random_idx(inputs.to_numpy({"row_len": inp["row_len"]}), wl.k, wl.seed)
    rows = sorted({0, wl.R - 1, wl.R // 2, 1 % wl.R})
    _check(dsa, oracle_mod, wl, inp, cache, ls, idx, rows=rows)
