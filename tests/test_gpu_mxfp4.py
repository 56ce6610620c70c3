"""GPU parity of the MXFP4 index-key path (68-byte keys: 64 bytes of E2M1 codes
and four E8M0 block scales) against the float64 oracle: the scorer on the
block-scaled FP4 tensor cores and the Write step's MX quantization."""
import numpy as np
import pytest
import torch

import helpers
from dsa_sparse_attention_lightning_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
MX_PAGE = 4352
E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dsa_sparse_attention_lightning_gb300 as m
    from dsa_sparse_attention_lightning_gb300 import _build
    _build.build()
    m.load()
    return m


def _mx_values(rng, shape):
    """Normal values with a per-vector magnitude, a few blocks 2^-8 smaller and a
    few all zero (so that block exponents spread within a vector)."""
    v = rng.standard_normal(shape) * rng.uniform(0.2, 5.0, shape[:-1] + (1,))
    blocks = v.reshape(shape[:-1] + (shape[-1] // 32, 32))
    blocks[rng.random(blocks.shape[:-1]) < 0.05] *= 2.0 ** -8
    blocks[rng.random(blocks.shape[:-1]) < 0.02] = 0.0
    return blocks.reshape(shape)


def _mx_cache(oracle_mod, rng, num_pages):
    codes, scales = oracle_mod.mx_quantize(_mx_values(rng, (num_pages, 64, 128)))
    return np.concatenate([codes.reshape(num_pages, 64 * 64),
                           scales.reshape(num_pages, 64 * 4)], axis=1)


MX_CASES = [
    inputs.Workload("mx_ragged", [3000, 700, 5000, 64], [2, 1, 4, 1], H=16, seed=21),
    inputs.Workload("mx_short_rows", [1, 63, 65, 2047, 2049], [1, 1, 2, 1, 3], H=16, seed=22),
    # more than four rows per request: groups 4 + 4 + 3 and 4 + 1
    inputs.Workload("mx_wide", [6000, 3000], [11, 5], H=16, seed=23),
]


@pytest.mark.parametrize("wl", MX_CASES, ids=[w.name for w in MX_CASES])
def test_indexer_mxfp4_matches_oracle(dsa, oracle_mod, wl):
    host = inputs.to_numpy(inputs.make_inputs(wl, device="cpu"))
    rng = np.random.default_rng(wl.seed + 100)
    num_pages = host["key_cache"].shape[0]
    cache = _mx_cache(oracle_mod, rng, num_pages)
    R = host["row_len"].shape[0]
    qc, qs = oracle_mod.mx_quantize(_mx_values(rng, (R, 32, 128)))
    w = host["w"]
    g = dsa.dsa_indexer_score_mxfp4(
        torch.from_numpy(qc).to(DEV), torch.from_numpy(qs).to(DEV), torch.from_numpy(w).to(DEV),
        torch.from_numpy(cache).to(DEV), torch.from_numpy(host["block_table"]).to(DEV),
        torch.from_numpy(host["row_req"]).to(DEV), torch.from_numpy(host["row_len"]).to(DEV))
    torch.cuda.synchronize()
    ora = oracle_mod.indexer_scores_mx(qc, qs, w, cache, host["block_table"], host["row_req"],
                                       host["row_len"], ld=g.shape[1])
    helpers.assert_scores_close(g.cpu().numpy(), ora, host["row_len"])


def _near_pow2(a, rel=1e-5):
    """Block maxima whose float64 value is within rel of a power of two: the fp32
    kernel may take the neighbouring exponent there."""
    with np.errstate(divide="ignore"):
        l2 = np.log2(np.where(a > 0, a, 1.0))
    return (a > 0) & (np.abs(l2 - np.round(l2)) < rel)


def test_write_kv_mxfp4_matches_oracle(dsa, oracle_mod):
    rng = np.random.default_rng(12)
    T, B, max_pages = 200, 4, 16
    num_pages = B * max_pages
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, max_pages)
    req = np.repeat(np.arange(B), T // B).astype(np.int32)
    pos = np.concatenate([rng.choice(max_pages * 64, T // B, replace=False)
                          for _ in range(B)]).astype(np.int32)
    x = (rng.standard_normal((T, 128)) * 3.0 + 0.5).astype(np.float32)
    x[5] = 1.5                                        # constant key: a zero normalized key
    lat = rng.standard_normal((T, 576)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    gamma[32:64] *= 2.0 ** -6                          # one block far smaller than the others
    eps, ls = 1e-6, 0.0125
    kc0 = np.full((num_pages, MX_PAGE), 0x77, np.uint8)
    lc0 = np.full((num_pages, 64, 576), 0x7F, np.uint8)
    for b_vec in ((rng.standard_normal(128) * 0.1).astype(np.float32), np.zeros(128, np.float32)):
        kb = torch.from_numpy(x).to(torch.bfloat16)
        lb = torch.from_numpy(lat).to(torch.bfloat16)
        kc = torch.from_numpy(kc0).to(DEV)
        lc = torch.from_numpy(lc0).to(DEV)
        st = torch.full((1,), 7, dtype=torch.int32, device=DEV)
        dsa.dsa_write_kv(kb.to(DEV), torch.from_numpy(gamma).to(DEV),
                         torch.from_numpy(b_vec).to(DEV), eps, lb.to(DEV), ls,
                         torch.from_numpy(bt).to(DEV), torch.from_numpy(req).to(DEV),
                         torch.from_numpy(pos).to(DEV), kc, lc, dev_status=st, mxfp4_keys=True)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        kcg, lcg = kc.cpu().numpy(), lc.cpu().numpy()
        k16 = kb.view(torch.int16).numpy().view(np.uint16)
        okc, kpre = oracle_mod.write_key_mx(k16, gamma.astype(np.float64),
                                            b_vec.astype(np.float64), eps, bt, req, pos, kc0)
        _, olc, _, lpre, _ = oracle_mod.write_kv(
            k16, gamma.astype(np.float64), b_vec.astype(np.float64), eps,
            lb.view(torch.int16).numpy().view(np.uint16), ls, bt, req, pos,
            np.zeros((num_pages, 8448), np.uint8), lc0)
        mids = helpers.e4m3_midpoints(oracle_mod)
        written_k = np.zeros(kc0.shape, bool)
        written_l = np.zeros(lc0.shape[:2], bool)
        for t in range(T):
            page, slot = bt[req[t], pos[t] // 64], pos[t] % 64
            sc_off = 64 * 64 + 4 * slot
            g_sc, o_sc = kcg[page, sc_off:sc_off + 4], okc[page, sc_off:sc_off + 4]
            g_codes = kcg[page, 64 * slot:64 * slot + 64]
            o_codes = okc[page, 64 * slot:64 * slot + 64]
            g_nib = np.stack([g_codes & 0xF, g_codes >> 4], 1).reshape(128)
            o_nib = np.stack([o_codes & 0xF, o_codes >> 4], 1).reshape(128)
            for b in range(4):
                blk = slice(32 * b, 32 * b + 32)
                amax = np.abs(kpre[t, blk]).max()
                if g_sc[b] != o_sc[b]:
                    assert _near_pow2(amax), (t, b, g_sc[b], o_sc[b], amax)
                    continue
                scaled = np.abs(kpre[t, blk]) / 2.0 ** (int(o_sc[b]) - 127)
                near = np.abs(scaled[:, None] - E2M1_MIDPOINTS[None]).min(1) < 1e-5 * np.maximum(
                    scaled, 1.0)
                ok = near | (g_nib[blk] == o_nib[blk])
                assert ok.all(), (t, b, np.flatnonzero(~ok))
            ok = helpers.near_midpoint(lpre[t], mids) | (lcg[page, slot] == olc[page, slot])
            assert ok.all(), (t, np.flatnonzero(~ok))
            written_k[page, 64 * slot:64 * slot + 64] = True
            written_k[page, sc_off:sc_off + 4] = True
            written_l[page, slot] = True
        assert np.array_equal(kcg[~written_k], kc0[~written_k])
        assert np.array_equal(lcg[~written_l], lc0[~written_l])
        # the zero key: every block scale 2^-127 (code 0), every code 0
        page, slot = bt[req[5], pos[5] // 64], pos[5] % 64
        if not b_vec.any():
            assert (kcg[page, 64 * 64 + 4 * slot:64 * 64 + 4 * slot + 4] == 0).all()
            assert (kcg[page, 64 * slot:64 * slot + 64] == 0).all()


def test_write_kv_mxfp4_then_score(dsa, oracle_mod):
    """Keys written by the MX Write step and scored by the MX scorer agree with
    the oracle scoring the same cache bytes."""
    rng = np.random.default_rng(13)
    B, max_pages, ctx = 2, 8, [500, 300]
    num_pages = B * max_pages
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, max_pages)
    req = np.concatenate([np.full(c, b) for b, c in enumerate(ctx)]).astype(np.int32)
    pos = np.concatenate([np.arange(c) for c in ctx]).astype(np.int32)
    T = req.shape[0]
    kb = torch.from_numpy(rng.standard_normal((T, 128)).astype(np.float32)).to(torch.bfloat16)
    lb = torch.zeros((T, 576), dtype=torch.bfloat16)
    kc = torch.zeros((num_pages, MX_PAGE), dtype=torch.uint8, device=DEV)
    lc = torch.zeros((num_pages, 64, 576), dtype=torch.uint8, device=DEV)
    dsa.dsa_write_kv(kb.to(DEV), torch.ones(128, device=DEV), torch.zeros(128, device=DEV), 1e-6,
                     lb.to(DEV), 1.0, torch.from_numpy(bt).to(DEV), torch.from_numpy(req).to(DEV),
                     torch.from_numpy(pos).to(DEV), kc, lc, mxfp4_keys=True)
    rows_req = np.array([0, 0, 1], np.int32)
    rows_len = np.array([499, 500, 300], np.int32)
    qc, qs = oracle_mod.mx_quantize(_mx_values(rng, (3, 32, 128)))
    w = rng.uniform(-0.1, 0.3, (3, 32)).astype(np.float32)
    g = dsa.dsa_indexer_score_mxfp4(
        torch.from_numpy(qc).to(DEV), torch.from_numpy(qs).to(DEV), torch.from_numpy(w).to(DEV),
        kc, torch.from_numpy(bt).to(DEV), torch.from_numpy(rows_req).to(DEV),
        torch.from_numpy(rows_len).to(DEV))
    torch.cuda.synchronize()
    ora = oracle_mod.indexer_scores_mx(qc, qs, w, kc.cpu().numpy(), bt, rows_req, rows_len,
                                       ld=g.shape[1])
    helpers.assert_scores_close(g.cpu().numpy(), ora, rows_len)


def test_write_kv_mxfp4_flags_bad_tokens(dsa):
    kc = torch.full((4, MX_PAGE), 0x77, dtype=torch.uint8, device=DEV)
    lc = torch.full((4, 64, 576), 0x7F, dtype=torch.uint8, device=DEV)
    bt = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device=DEV)
    kb = torch.randn(3, 128, device=DEV).to(torch.bfloat16)
    lb = torch.randn(3, 576, device=DEV).to(torch.bfloat16)
    one, zero = torch.ones(128, device=DEV), torch.zeros(128, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    req = torch.tensor([0, 5, 1], dtype=torch.int32, device=DEV)     # request 5 does not exist
    pos = torch.tensor([3, 0, 200], dtype=torch.int32, device=DEV)   # 200 >= 2 pages x 64
    dsa.dsa_write_kv(kb, one, zero, 1e-6, lb, 0.05, bt, req, pos, kc, lc, dev_status=st,
                     mxfp4_keys=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0x1                       # DSA_DEV_BAD_ROW
    assert (kc[0, 3 * 64:4 * 64] != 0x77).any()        # the valid token was written
    assert (kc[1:] == 0x77).all() and (lc[1:] == 0x7F).all()
