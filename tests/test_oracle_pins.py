"""Pins for the float64 oracle: closed forms, library routines, brute force.

Each test ties one part of the oracle to something other than the oracle
itself, chosen so that a plausible slip (a dropped head or dimension, a wrong
page or slot, the scale read from the wrong token, ReLU in the wrong place, a
wrong softmax shift or log-sum-exp) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from dsa_sparse_attention_lightning_gb300 import inputs, traffic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PAGE, D, NH, LAT, V = 64, 128, 32, 576, 512


def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            rows[parts[0]] = parts[1:]
    return rows


def _bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def _e4m3(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_vals(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def _key_cache(codes, scales):
    """Pack [ntok,128] codes and [ntok] scales into identity-mapped 64-token pages."""
    n = codes.shape[0]
    npg = (n + PAGE - 1) // PAGE
    cache = np.full((npg, PAGE * D + PAGE * 4), 0x7F, dtype=np.uint8)
    sc = np.full((npg, PAGE), np.nan, dtype=np.float32)
    for t in range(n):
        cache[t // PAGE, (t % PAGE) * D:(t % PAGE + 1) * D] = codes[t]
        sc[t // PAGE, t % PAGE] = scales[t]
    cache[:, PAGE * D:] = sc.view(np.uint8).reshape(npg, PAGE * 4)
    bt = np.arange(npg, dtype=np.int32)[None, :]
    return cache, bt


def _latent_cache(codes):
    n = codes.shape[0]
    npg = (n + PAGE - 1) // PAGE
    cache = np.full((npg, PAGE, LAT), 0x7F, dtype=np.uint8)
    for t in range(n):
        cache[t // PAGE, t % PAGE] = codes[t]
    return cache, np.arange(npg, dtype=np.int32)[None, :]


# ---------------------------------------------------------------- E4M3 decode
def test_e4m3_all_codes_match_torch(oracle_mod):
    lib = _e4m3_vals(np.arange(256, dtype=np.uint8))
    ours = np.array([oracle_mod.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2  # 0x7f and 0xff only
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))


def test_e4m3_golden_table(oracle_mod):
    for code, (val,) in _read_golden("e4m3_codes.txt").items():
        got = oracle_mod.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


# ------------------------------------------------------------ indexer scores
def _rand_case(rng, n, scale_spread=True):
    k = rng.standard_normal((n, D)).astype(np.float32)
    codes = _e4m3(np.clip(k * 40, -448, 448))
    scales = (rng.uniform(0.5, 2.0, n) if scale_spread else np.ones(n)).astype(np.float32)
    return codes, scales


def test_indexer_single_head_is_relu_dot(oracle_mod):
    """w one-hot on head h, scale 1: score = max(0, q_h . k) (numpy float64 dot)."""
    rng = np.random.default_rng(1)
    n = 150
    codes, _ = _rand_case(rng, n)
    cache, bt = _key_cache(codes, np.ones(n, np.float32))
    q = _bf16_bits(rng.standard_normal((1, NH, D)))
    kd = _e4m3_vals(codes)
    for h in (0, 17, 31):
        w = np.zeros((1, NH), np.float32)
        w[0, h] = 1.0
        s = oracle_mod.indexer_scores(q, w, cache, bt, [0], [n])
        ref = np.maximum(0.0, kd @ _bf16_vals(q[0, h]))
        assert np.array_equal(s[0], ref) or np.allclose(s[0], ref, rtol=1e-13, atol=1e-12)
        assert (ref == 0).sum() > 10 and (ref > 0).sum() > 10   # both ReLU branches hit


def test_indexer_last_dim_and_scale_slot(oracle_mod):
    """Key nonzero only in dim 127, per-token scale 2^t: score = w*relu(q[127]*code)*2^t."""
    n = 70  # crosses a page boundary
    codes = np.zeros((n, D), np.uint8)
    codes[:, D - 1] = 0x38  # 1.0
    scales = np.array([2.0 ** (t % 7) for t in range(n)], np.float32)
    cache, bt = _key_cache(codes, scales)
    qv = np.zeros((1, NH, D), np.float32)
    qv[0, :, D - 1] = np.linspace(-1, 2, NH)
    q = _bf16_bits(qv)
    w = np.full((1, NH), 1.0 / NH, np.float32)
    s = oracle_mod.indexer_scores(q, w, cache, bt, [0], [n])
    qd = _bf16_vals(q[0, :, D - 1])
    per_tok = np.sum(np.float64(w[0]) * np.maximum(0.0, qd)) * scales.astype(np.float64)
    assert np.allclose(s[0], per_tok, rtol=1e-14)


def test_indexer_relu_is_per_head_before_weighting(oracle_mod):
    """Negative head weight: a head with positive logit contributes w*logit < 0."""
    n = 3
    codes = np.zeros((n, D), np.uint8)
    codes[:, 0] = 0x38
    cache, bt = _key_cache(codes, np.ones(n, np.float32))
    qv = np.zeros((1, NH, D), np.float32)
    qv[0, 0, 0] = 1.0     # head 0: logit +1
    qv[0, 1, 0] = -3.0    # head 1: logit -3 -> ReLU 0
    w = np.zeros((1, NH), np.float32)
    w[0, 0], w[0, 1] = -0.5, 1.0
    s = oracle_mod.indexer_scores(_bf16_bits(qv), w, cache, bt, [0], [n])
    assert np.array_equal(s[0], np.full(n, -0.5))   # ReLU of the sum would give 0


def test_indexer_zero_query_and_linearity(oracle_mod):
    rng = np.random.default_rng(2)
    n = 200
    codes, scales = _rand_case(rng, n)
    cache, bt = _key_cache(codes, scales)
    q = _bf16_bits(rng.standard_normal((1, NH, D)))
    w = rng.uniform(0.01, 0.1, (1, NH)).astype(np.float32)
    s1 = oracle_mod.indexer_scores(q, w, cache, bt, [0], [n])
    s4 = oracle_mod.indexer_scores(q, w * 4, cache, bt, [0], [n])
    assert np.array_equal(s4, 4 * s1)
    z = oracle_mod.indexer_scores(np.zeros_like(q), w, cache, bt, [0], [n])
    assert np.array_equal(z, np.zeros_like(z))


def test_indexer_paging_invariance_and_row_lengths(oracle_mod):
    """Scattering pages through a shuffled block table changes nothing; rows see
    exactly row_len tokens; entries beyond row_len stay untouched."""
    wl = inputs.Workload("pin", [300, 130], [3, 1], H=16, k=64, seed=7, paged=True,
                         shift_frac=0.05)
    a = inputs.to_numpy(inputs.make_inputs(wl))
    wl2 = inputs.Workload("pin", [300, 130], [3, 1], H=16, k=64, seed=7, paged=False,
                          shift_frac=0.05)
    b = inputs.to_numpy(inputs.make_inputs(wl2))
    sa = oracle_mod.indexer_scores(a["q_idx"], a["w"], a["key_cache"], a["block_table"],
                                   a["row_req"], a["row_len"])
    # rebuild identity-paged caches from the shuffled ones
    ka, bta = a["key_cache"], a["block_table"]
    kb = np.concatenate([ka[bta[bi, :(c + 63) // 64]] for bi, c in enumerate(wl.ctx)])
    starts = np.cumsum([0] + [(c + 63) // 64 for c in wl.ctx])
    btb = np.full_like(bta, -1)
    for bi, c in enumerate(wl.ctx):
        n = (c + 63) // 64
        btb[bi, :n] = np.arange(starts[bi], starts[bi] + n)
    sb = oracle_mod.indexer_scores(a["q_idx"], a["w"], kb, btb, a["row_req"], a["row_len"])
    assert np.array_equal(np.isnan(sa), np.isnan(sb))
    assert np.array_equal(np.nan_to_num(sa), np.nan_to_num(sb))
    for r, L in enumerate(a["row_len"]):
        assert not np.isnan(sa[r, :L]).any()
        assert np.isnan(sa[r, L:]).all()
    assert b["block_table"][0, 0] == 0


def test_indexer_einsum_crosscheck(oracle_mod):
    """Full random case against torch float64 einsum with torch's FP8 decode."""
    wl = inputs.Workload("pin", [257], [2], H=16, k=64, seed=3, shift_frac=0.05)
    a = inputs.to_numpy(inputs.make_inputs(wl))
    s = oracle_mod.indexer_scores(a["q_idx"], a["w"], a["key_cache"], a["block_table"],
                                  a["row_req"], a["row_len"])
    kc = a["key_cache"]
    bt = a["block_table"][0]
    ntok = 257
    pages = bt[np.arange(ntok) // 64]
    slots = np.arange(ntok) % 64
    codes = kc[:, :PAGE * D].reshape(-1, PAGE, D)[pages, slots]
    scales = kc[:, PAGE * D:].copy().view(np.float32)[pages, slots].astype(np.float64)
    kd = torch.from_numpy(_e4m3_vals(codes))
    q = torch.from_numpy(_bf16_vals(a["q_idx"]))
    logits = torch.einsum("rhd,sd->rhs", q, kd) * torch.from_numpy(scales)
    ref = (torch.from_numpy(a["w"].astype(np.float64))[:, :, None] * logits.clamp_min(0)).sum(1)
    for r, L in enumerate(a["row_len"]):
        assert np.allclose(s[r, :L], ref[r, :L].numpy(), rtol=1e-12, atol=1e-12)


def test_indexer_fp8_query_scale(oracle_mod):
    """E4M3 query with a (row, head) scale equals the bf16 path on the decoded values
    when those values are exact in bf16 (E4M3 values times a power of two are)."""
    rng = np.random.default_rng(4)
    n = 90
    codes, scales = _rand_case(rng, n)
    cache, bt = _key_cache(codes, scales)
    q8 = _e4m3(np.clip(rng.standard_normal((1, NH, D)) * 100, -448, 448))
    qs = (2.0 ** rng.integers(-8, 3, (1, NH))).astype(np.float32)
    w = rng.uniform(0.01, 0.1, (1, NH)).astype(np.float32)
    s8 = oracle_mod.indexer_scores(q8, w, cache, bt, [0], [n], q_scale=qs)
    qb = _bf16_bits(_e4m3_vals(q8) * qs[..., None])
    sb = oracle_mod.indexer_scores(qb, w, cache, bt, [0], [n])
    assert np.array_equal(s8, sb)


def test_indexer_rejects_bad_page(oracle_mod):
    codes = np.zeros((10, D), np.uint8)
    cache, bt = _key_cache(codes, np.ones(10, np.float32))
    with pytest.raises(ValueError):
        oracle_mod.indexer_scores(_bf16_bits(np.zeros((1, NH, D))), np.ones((1, NH), np.float32),
                                  cache, bt + 5, [0], [10])


# ----------------------------------------------------------------------- top-k
def _brute_topk(scores, L, k):
    order = np.lexsort((np.arange(L), -scores[:L]))
    out = np.full(k, -1, np.int32)
    out[:min(k, L)] = order[:k]
    return out


@pytest.mark.parametrize("L,k", [(1, 4), (5, 8), (100, 8), (1000, 64), (4096, 2048)])
def test_topk_brute_force_with_ties(oracle_mod, L, k):
    rng = np.random.default_rng(L + k)
    s = rng.integers(0, 20, (2, max(L, 1))).astype(np.float64)   # many exact ties
    s[1] = rng.standard_normal(max(L, 1))
    got = oracle_mod.topk(s, [L, L], k)
    for r in range(2):
        assert np.array_equal(got[r], _brute_topk(s[r], L, k))


def test_topk_all_equal_and_signed_zero(oracle_mod):
    s = np.zeros((2, 10))
    s[1, ::2] = -0.0
    got = oracle_mod.topk(s, [10, 10], 4)
    assert np.array_equal(got[0], [0, 1, 2, 3])
    assert np.array_equal(got[1], [0, 1, 2, 3])


def test_topk_len_below_k_and_zero(oracle_mod):
    s = np.array([[3.0, 1.0, 2.0, 9.0]])
    assert np.array_equal(oracle_mod.topk(s, [3], 5)[0], [0, 2, 1, -1, -1])
    assert np.array_equal(oracle_mod.topk(s, [0], 2)[0], [-1, -1])


# ------------------------------------------- top-k by the context-parallel exchange
# The pages state the invariant: the merged selection matches a single-GPU
# top-k exactly (SGLang post, "Decode: DSA with decode context parallelism";
# vLLM post, "An exact top-k merge with about 10x less traffic").
def _dcp_rows(rng, L, W):
    base = rng.standard_normal(L)
    conc = base.copy()
    conc[(W - 1)::W] += 10.0                    # shard W-1 holds every winner
    first = base.copy()
    first[:: 2 * W] += 10.0                     # half of shard 0's tokens win
    ties = rng.integers(0, 20, L).astype(np.float64)
    return np.stack([base, conc, first, ties, np.zeros(L)])


@pytest.mark.parametrize("W", [1, 2, 3, 8])
def test_topk_dcp_equals_single_shard_topk(oracle_mod, W):
    rng = np.random.default_rng(20 + W)
    L = 6000
    s = _dcp_rows(rng, L, W)
    for k in (7, 300, 2048):
        for lens in ([L] * 5, [L, 5000, 4097, 2 * W + 1, W - 1 if W > 1 else 0]):
            got, _ = oracle_mod.topk_dcp(s, lens, k, W)
            assert np.array_equal(got, oracle_mod.topk(s, lens, k))
            for r in range(s.shape[0]):
                assert np.array_equal(got[r], _brute_topk(s[r], lens[r], k))


def test_topk_dcp_resend_pattern(oracle_mod):
    W, k, L = 8, 2048, 32768
    rng = np.random.default_rng(3)
    base = rng.standard_normal(L)
    conc = base.copy()
    conc[3::W] += 10.0                          # shard 3: 4096 tokens above all others
    s = np.stack([conc, base, np.zeros(L)])
    idx, mask = oracle_mod.topk_dcp(s, [L, L, L], k, W)
    # only the shard holding every winner can hide any; spread winners (about
    # 256 per shard, below the 384 sent) and all-equal scores (the lowest
    # 2048 positions, 256 per shard) need no resend
    assert list(mask) == [1 << 3, 0, 0]
    assert np.all(idx[0] % W == 3)
    assert np.array_equal(idx[0], _brute_topk(conc, L, k))
    # one shard holds everything: 1.5 k candidates always cover the top-k
    _, m1 = oracle_mod.topk_dcp(s, [L, L, L], k, 1)
    assert list(m1) == [0, 0, 0]
    # short rows: no shard keeps a token back
    _, m2 = oracle_mod.topk_dcp(s, [300, 3000, 0], k, W)
    assert list(m2) == [0, 0, 0]


# --------------------------------------------------------------- the Write step
def _e4m3_midpoints(oracle_mod):
    vals = sorted({oracle_mod.e4m3_decode(c) for c in range(0x7F)})
    return np.array([(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])])


def _near_midpoint(v, mids, rel=1e-5):
    """True where |v| lies within rel * |v| of a rounding midpoint of E4M3."""
    a = np.abs(np.asarray(v, np.float64))
    j = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[j - 1]), np.abs(a - mids[j]))
    return d <= rel * np.maximum(a, 1e-30)


def test_e4m3_encode_round_trip_and_torch_cast(oracle_mod):
    for c in range(256):
        if c & 0x7F != 0x7F:
            assert oracle_mod.e4m3_encode(oracle_mod.e4m3_decode(c)) == c, hex(c)
    # golden ties (round to nearest even): 1.0625 between 1.0 (0x38) and 1.125
    # (0x39); 1.1875 between 1.125 and 1.25 (0x3A); saturation at 448 (0x7E)
    assert [oracle_mod.e4m3_encode(v) for v in (1.0625, 1.1875, 600.0, -1000.0)] == \
        [0x38, 0x3A, 0x7E, 0xFE]
    mids = _e4m3_midpoints(oracle_mod)
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(-448, 448, 3000), rng.standard_normal(3000) * 0.02,
                         mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, ref)


def _write_case(rng, T=40, B=3, max_pages=4):
    num_pages = B * max_pages
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, max_pages)
    req = np.repeat(np.arange(B), T // B + 1)[:T].astype(np.int32)
    pos = np.zeros(T, np.int32)
    for b in range(B):
        sel = req == b
        pos[sel] = rng.choice(max_pages * PAGE, int(sel.sum()), replace=False)
    x = rng.standard_normal((T, D)) * 3.0 + 0.5
    lat = rng.standard_normal((T, LAT))
    key_cache = np.full((num_pages, PAGE * D + PAGE * 4), 0x7F, np.uint8)
    latent_cache = np.full((num_pages, PAGE, LAT), 0x7F, np.uint8)
    return bt, req, pos, x, lat, key_cache, latent_cache


def test_write_kv_layernorm_scale_codes_and_placement(oracle_mod):
    rng = np.random.default_rng(5)
    bt, req, pos, x, lat, kc0, lc0 = _write_case(rng)
    gamma = rng.uniform(0.5, 1.5, D)
    beta = rng.standard_normal(D) * 0.1
    eps, ls = 1e-6, 0.0125
    kb, lb = _bf16_bits(x), _bf16_bits(lat)
    kc, lc, kpre, lpre, ks = oracle_mod.write_kv(kb, gamma, beta, eps, lb, ls, bt, req, pos,
                                                 kc0, lc0)
    # LayerNorm: torch's float64 layer_norm of the same bf16 inputs
    ln = torch.nn.functional.layer_norm(torch.from_numpy(_bf16_vals(kb)), (D,),
                                        torch.from_numpy(gamma), torch.from_numpy(beta), eps)
    assert np.allclose(kpre * ks[:, None], ln.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(ks, np.abs(ln.numpy()).max(1) / 448.0, rtol=1e-15)
    mids = _e4m3_midpoints(oracle_mod)
    written = np.zeros(kc0.shape, bool)
    for t in range(len(req)):
        page, slot = bt[req[t], pos[t] // PAGE], pos[t] % PAGE
        codes = kc[page, slot * D:(slot + 1) * D]
        vals = _e4m3_vals(codes)
        assert np.abs(vals).max() == 448.0            # the absmax element is exactly 448
        ref = torch.from_numpy(kpre[t].astype(np.float32)).to(torch.float8_e4m3fn)
        ok = ~_near_midpoint(kpre[t], mids)
        assert np.array_equal(codes[ok], ref.view(torch.uint8).numpy()[ok])
        assert kc[page, PAGE * D + slot * 4:PAGE * D + slot * 4 + 4].view(np.float32)[0] == \
            np.float32(ks[t])
        # the latent row: the generator's quantizer (torch cast of the fp32 quotient)
        lref = torch.from_numpy(_bf16_vals(lb[t]).astype(np.float32) / np.float32(ls))
        lref = lref.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        lok = ~_near_midpoint(lpre[t], mids)
        assert np.array_equal(lc[page, slot][lok], lref[lok])
        written[page, slot * D:(slot + 1) * D] = True
        written[page, PAGE * D + slot * 4:PAGE * D + slot * 4 + 4] = True
    assert np.all(kc[~written] == 0x7F)                # nothing else is touched


def test_write_kv_zero_key(oracle_mod):
    rng = np.random.default_rng(6)
    bt, req, pos, x, lat, kc0, lc0 = _write_case(rng, T=3)
    x[:] = 1.5                                         # constant key: LayerNorm gives beta = 0
    kc, _, _, _, ks = oracle_mod.write_kv(_bf16_bits(x), np.ones(D), np.zeros(D), 1e-6,
                                          _bf16_bits(lat), 1.0, bt, req, pos, kc0, lc0)
    assert np.all(ks == 1.0)
    for t in range(3):
        page, slot = bt[req[t], pos[t] // PAGE], pos[t] % PAGE
        assert np.all(kc[page, slot * D:(slot + 1) * D] == 0)


# ------------------------------------------------------------------ sparse MLA
def _mla_case(rng, n, H):
    codes = _e4m3(np.clip(rng.standard_normal((n, LAT)) * 100, -448, 448))
    cache, bt = _latent_cache(codes)
    q = _bf16_bits(rng.standard_normal((1, H, LAT)))
    return codes, cache, bt, q


def test_mla_dense_matches_sdpa(oracle_mod):
    """All tokens selected: equals float64 scaled_dot_product_attention."""
    rng = np.random.default_rng(5)
    n, H, s_l, sm = 150, 4, 0.0123, 1 / math.sqrt(192)
    codes, cache, bt, q = _mla_case(rng, n, H)
    idx = np.arange(n, dtype=np.int32)[None]
    out, lse = oracle_mod.sparse_mla(q, sm, cache, s_l, bt, [0], [n], idx)
    L = torch.from_numpy(_e4m3_vals(codes)) * s_l
    qd = torch.from_numpy(_bf16_vals(q[0]))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qd[None, :, None, :].expand(1, H, 1, LAT), L[None, None].expand(1, H, n, LAT),
        L[None, None, :, :V].expand(1, H, n, V), scale=sm)[0, :, 0]
    assert np.allclose(out[0], ref.numpy(), rtol=1e-10, atol=1e-12)
    ref_lse = torch.logsumexp(sm * (qd @ L.T), dim=-1)
    assert np.allclose(lse[0], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_mla_single_token_and_zero_query(oracle_mod):
    rng = np.random.default_rng(6)
    n, H, s_l = 80, 3, 0.5
    codes, cache, bt, q = _mla_case(rng, n, H)
    vals = _e4m3_vals(codes) * s_l
    idx = np.full((1, 8), -1, np.int32)
    idx[0, 5] = 71
    out, _ = oracle_mod.sparse_mla(q, 0.1, cache, s_l, bt, [0], [n], idx)
    assert np.array_equal(out[0], np.broadcast_to(vals[71, :V], (H, V)))
    sel = np.array([3, 9, 64, 70], np.int32)
    out0, lse0 = oracle_mod.sparse_mla(np.zeros_like(q), 0.1, cache, s_l, bt, [0], [n], sel[None])
    assert np.allclose(out0[0], np.broadcast_to(vals[sel, :V].mean(0), (H, V)), rtol=1e-13)
    assert np.allclose(lse0[0], math.log(4.0), rtol=1e-14)


def test_mla_split_merge_by_lse(oracle_mod):
    """Attention over A u B equals the LSE-weighted merge of A and B (exact softmax)."""
    rng = np.random.default_rng(8)
    n, H, s_l, sm = 200, 5, 0.02, 1 / math.sqrt(192)
    codes, cache, bt, q = _mla_case(rng, n, H)
    sel = rng.permutation(n)[:96].astype(np.int32)
    full, lf = oracle_mod.sparse_mla(q, sm, cache, s_l, bt, [0], [n], sel[None])
    a = np.where(np.arange(96) < 40, sel, -1).astype(np.int32)
    b = np.where(np.arange(96) >= 40, sel, -1).astype(np.int32)
    oa, la = oracle_mod.sparse_mla(q, sm, cache, s_l, bt, [0], [n], a[None])
    ob, lb = oracle_mod.sparse_mla(q, sm, cache, s_l, bt, [0], [n], b[None])
    lm = np.logaddexp(la, lb)
    merged = np.exp(la - lm)[..., None] * oa + np.exp(lb - lm)[..., None] * ob
    assert np.allclose(merged, full, rtol=1e-12, atol=1e-13)
    assert np.allclose(lm, lf, rtol=1e-13)
    # order of the selected slots does not matter
    perm, lp = oracle_mod.sparse_mla(q, sm, cache, s_l, bt, [0], [n], sel[::-1].copy()[None])
    assert np.allclose(perm, full, rtol=1e-12, atol=1e-13) and np.allclose(lp, lf, rtol=1e-13)


def test_mla_empty_row(oracle_mod):
    rng = np.random.default_rng(9)
    codes, cache, bt, q = _mla_case(rng, 10, 2)
    out, lse = oracle_mod.sparse_mla(q, 0.1, cache, 1.0, bt, [0], [0],
                                     np.full((1, 4), -1, np.int32))
    assert np.array_equal(out, np.zeros_like(out)) and np.all(np.isneginf(lse))


def test_topk_equal_context_is_dense(oracle_mod):
    """top-k with k >= context selects every token: sparse MLA == dense MLA."""
    wl = inputs.Workload("pin", [180], [2], H=4, k=256, seed=11)
    a = inputs.to_numpy(inputs.make_inputs(wl))
    _, idx, out, lse = oracle_mod.decode_step(a, k=256)
    dense = np.stack([np.where(np.arange(256) < L, np.arange(256), -1) for L in a["row_len"]])
    od, ld = oracle_mod.sparse_mla(a["q"], a["softmax_scale"], a["latent_cache"],
                                   a["latent_scale"], a["block_table"], a["row_req"],
                                   a["row_len"], dense.astype(np.int32))
    assert np.allclose(out, od, rtol=1e-12, atol=1e-13) and np.allclose(lse, ld, rtol=1e-13)


# ------------------------------------------------------------------ byte model
def test_byte_model_matches_pages():
    g = {k: float(v[0]) for k, v in _read_golden("byte_model.txt").items()}
    assert traffic.KEY_BYTES == g["index_key_bytes_per_token"]
    assert traffic.LATENT_BYTES == g["latent_bytes_per_token"]
    assert inputs.IDX_DIM * 2 == g["bf16_index_key_bytes_per_token"]
    ctx = 131072
    dense = ctx * traffic.dense_mla_bytes_per_token()
    dsa = traffic.dsa_bytes(ctx, int(g["selected_tokens"]))
    assert round(dense / 1e6, 1) == g["dense_bytes_128k"]
    assert round(dsa / 1e6, 1) == g["dsa_bytes_128k"]
    assert round(2 * ctx * 4 / 1e6) == g["index_scores_128k"]        # fp32, written + read
    assert round(dense / dsa) == g["single_row_reduction_128k"]
    four = ctx * traffic.KEY_BYTES + 4 * 2048 * traffic.LATENT_BYTES
    assert round(dense / four) == g["four_row_saving_128k"]
    assert round(traffic.dsa_bytes(1 << 20) / ((1 << 20) * 576), 2) == g[
        "dsa_share_of_dense_long_context"]
    assert 24 * traffic.LATENT_BYTES == g["kv_per_token_24_layers_k3_fp8"]
    assert 24 * (traffic.LATENT_BYTES + traffic.KEY_BYTES) == g["kv_per_token_24_layers_k31_fp8"]


def test_workload_bytes():
    assert traffic.algorithmic_bytes(inputs.config(0)) == 1_763_456
    assert traffic.algorithmic_bytes(inputs.config(1)) == 154_148_864
    assert traffic.algorithmic_bytes(inputs.config(2)) == 638_590_976
    assert traffic.algorithmic_bytes(inputs.config(3)) == 139_739_264
    assert round(traffic.scan_bytes(inputs.config(2)) / 16 / 1e6, 1) == 34.6
    assert inputs.config(4).row_lengths()[0] == 126_977    # row i sees tokens <= 126,976 + i


# ------------------------------------------------------- MXFP4 index keys
# Packed layout of one key: 64 bytes of E2M1 codes (dim 2j in the low nibble of
# byte j, dim 2j+1 in the high nibble), then per 64-token page 64 x 4 E8M0
# block scales (block b = dims 32b .. 32b+31).
MX_PAGE_BYTES = PAGE * (D // 2 + D // 32)


def _e2m1_grid():
    return np.array([float(v[0]) for c, v in _read_golden("e2m1_codes.txt").items()
                     if int(c, 16) < 8])


def _mx_key_cache(codes, scales):
    """Pack [ntok,64] code bytes and [ntok,4] scale bytes into identity-mapped pages."""
    n = codes.shape[0]
    npg = (n + PAGE - 1) // PAGE
    cache = np.full((npg, MX_PAGE_BYTES), 0xFF, dtype=np.uint8)   # 0xFF: NaN scale if read
    for t in range(n):
        p, s = divmod(t, PAGE)
        cache[p, s * 64:(s + 1) * 64] = codes[t]
        cache[p, PAGE * 64 + s * 4:PAGE * 64 + (s + 1) * 4] = scales[t]
    return cache, np.arange(npg, dtype=np.int32)[None, :]


def _grid_values(rng, shape, lo=-3, hi=2):
    """Values exactly on the MX grid: E2M1 magnitudes x sign x 2^p, p drawn per
    32-value block; about a tenth of the blocks all zero."""
    grid = _e2m1_grid()
    v = grid[rng.integers(0, 8, shape)] * rng.choice([-1.0, 1.0], shape)
    blocks = v.reshape(shape[:-1] + (shape[-1] // 32, 32))
    p = rng.integers(lo, hi + 1, blocks.shape[:-1] + (1,))
    blocks *= np.ldexp(1.0, p)
    blocks[rng.random(blocks.shape[:-1]) < 0.1] = 0.0
    return blocks.reshape(shape)


def test_e2m1_golden_table(oracle_mod):
    for code, (val,) in _read_golden("e2m1_codes.txt").items():
        got = oracle_mod.e2m1_decode(int(code, 16))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e2m1_encode_round_trip_and_golden_rounding(oracle_mod):
    for c in range(16):
        assert oracle_mod.e2m1_encode(oracle_mod.e2m1_decode(c)) == c
    for val, (code,) in _read_golden("e2m1_rounding.txt").items():
        assert oracle_mod.e2m1_encode(float(val)) == int(code, 16), val


def test_e2m1_encode_is_nearest(oracle_mod):
    """No grid point is strictly closer than the chosen one (brute force)."""
    grid = _e2m1_grid()
    rng = np.random.default_rng(40)
    for x in rng.uniform(-6.0, 6.0, 2000):
        got = oracle_mod.e2m1_decode(oracle_mod.e2m1_encode(x))
        assert math.copysign(1, got) == math.copysign(1, x)
        assert abs(x - got) <= np.min(np.abs(abs(x) - grid)) + 0.0


def test_e8m0_all_codes(oracle_mod):
    ours = np.array([oracle_mod.e8m0_decode(c) for c in range(256)])
    assert np.isnan(ours[255]) and not np.isnan(ours[:255]).any()
    assert all(ours[c] == math.ldexp(1.0, c - 127) for c in range(255))
    if hasattr(torch, "float8_e8m0fnu"):
        lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
        assert np.array_equal(np.isnan(lib), np.isnan(ours))
        assert np.array_equal(lib[:255], ours[:255])


def test_mx_quantize_scale_exponent_and_packing(oracle_mod):
    """The block exponent is floor(log2 amax) - 2 (via frexp); every code is the
    E2M1 encoding of v / scale; dim 2j sits in the low nibble of byte j."""
    rng = np.random.default_rng(41)
    v = rng.standard_normal((50, 128)) * np.ldexp(1.0, rng.integers(-20, 20, (50, 1)))
    v[3, 32:64] = 0.0
    codes, scales = oracle_mod.mx_quantize(v)
    assert codes.shape == (50, 64) and scales.shape == (50, 4)
    for i in range(50):
        for b in range(4):
            blk = v[i, 32 * b:32 * (b + 1)]
            amax = np.max(np.abs(blk))
            if amax == 0.0:
                assert scales[i, b] == 0
                assert not codes[i, 16 * b:16 * (b + 1)].any()
                continue
            assert int(scales[i, b]) - 127 == math.frexp(amax)[1] - 3
            sc = math.ldexp(1.0, int(scales[i, b]) - 127)
            assert 4.0 <= amax / sc < 8.0
            for j in (0, 1, 30, 31):
                d = 32 * b + j
                nib = codes[i, d // 2] & 0xF if d % 2 == 0 else codes[i, d // 2] >> 4
                assert nib == oracle_mod.e2m1_encode(v[i, d] / sc)


def test_mx_quantize_exact_on_grid_and_error_bound(oracle_mod):
    rng = np.random.default_rng(42)
    grid = _e2m1_grid()

    def decode(codes, scales):
        lo, hi = codes & 0xF, codes >> 4
        nib = np.stack([lo, hi], -1).reshape(codes.shape[:-1] + (-1,))
        mag = grid[nib & 7] * np.where(nib & 8, -1.0, 1.0)
        return mag * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=-1)

    v = _grid_values(rng, (40, 128), lo=-12, hi=12)
    assert np.array_equal(decode(*oracle_mod.mx_quantize(v)), v)
    v = rng.standard_normal((40, 128)) * rng.uniform(0.01, 100.0, (40, 1))
    codes, scales = oracle_mod.mx_quantize(v)
    sc = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=-1)
    err = np.abs(decode(codes, scales) - v) / sc
    # grid spacing 0.5 below 2, 1 below 4, 2 below 6; beyond 6 the clamp loses < 2
    a = np.abs(v) / sc
    bound = np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, np.where(a <= 6, 1.0, 2.0)))
    assert (err <= bound).all()


def test_indexer_mx_equals_fp8_scorer_on_shared_grid(oracle_mod):
    """Keys and queries on the MX grid are also E4M3 codes times a power-of-two
    per-token (per-head) scale, exactly.  The FP8 scorer, pinned above, must then
    give the same scores: this catches a wrong E2M1 value, nibble order, block
    scale index or bias in the MX path."""
    rng = np.random.default_rng(43)
    n, R = 150, 2
    kv = _grid_values(rng, (n, D))
    kc, ks = oracle_mod.mx_quantize(kv)
    cache_mx, bt = _mx_key_cache(kc, ks)
    # FP8 form: codes of kv / 2^base with ks = 2^base, base the smallest block exponent
    base = np.floor(np.log2(np.where(kv == 0, np.inf, np.abs(kv)).min(axis=1)))
    base = np.where(np.isfinite(base), base, 0.0)
    k8 = _e4m3(kv / np.ldexp(1.0, base.astype(np.int64))[:, None])
    assert np.array_equal(_e4m3_vals(k8) * np.ldexp(1.0, base.astype(np.int64))[:, None], kv)
    cache8, _ = _key_cache(k8, np.ldexp(1.0, base.astype(np.int64)).astype(np.float32))
    qv = _grid_values(rng, (R, NH, D))
    qc, qs = oracle_mod.mx_quantize(qv)
    qbase = np.floor(np.log2(np.where(qv == 0, np.inf, np.abs(qv)).min(axis=2)))
    qbase = np.where(np.isfinite(qbase), qbase, 0.0).astype(np.int64)
    q8 = _e4m3(qv / np.ldexp(1.0, qbase)[..., None])
    assert np.array_equal(_e4m3_vals(q8) * np.ldexp(1.0, qbase)[..., None], qv)
    w = rng.uniform(-0.05, 0.1, (R, NH)).astype(np.float32)
    row_len = [n, 97]
    s_mx = oracle_mod.indexer_scores_mx(qc, qs, w, cache_mx, bt, [0, 0], row_len)
    s_8 = oracle_mod.indexer_scores(q8, w, cache8, bt, [0, 0], row_len,
                                    q_scale=np.ldexp(1.0, qbase).astype(np.float32))
    assert np.array_equal(np.isnan(s_mx), np.isnan(s_8))
    assert np.allclose(np.nan_to_num(s_mx), np.nan_to_num(s_8), rtol=1e-14, atol=1e-300)
    assert (np.nan_to_num(s_mx) != 0).sum() > 100


def test_indexer_mx_last_dim_and_scale_slot(oracle_mod):
    """Key nonzero only in dim 127 (high nibble of byte 63, scale block 3), with a
    per-token exponent: score = sum_h w_h relu(q_h[127] * 2^e_t)."""
    n = 70  # crosses a page boundary
    kc = np.zeros((n, 64), np.uint8)
    kc[:, 63] = 0x20                        # dim 126 = 0, dim 127 = 1.0
    ks = np.full((n, 4), 127, np.uint8)
    e = np.array([t % 7 - 3 for t in range(n)])
    ks[:, 3] = 127 + e
    ks[:, :3] = 200                         # blocks 0-2 hold zeros; their scale must not leak
    cache, bt = _mx_key_cache(kc, ks)
    qc = np.zeros((1, NH, 64), np.uint8)
    grid_codes = np.array([0x2, 0xA, 0x7, 0xF, 0x1, 0x0] * 6)[:NH]   # +-1, +-6, 0.5, 0
    qc[0, :, 63] = (grid_codes << 4).astype(np.uint8)
    qs = np.full((1, NH, 4), 127, np.uint8)
    qs[0, :, 3] = 128                       # query block 3 scaled by 2
    w = np.linspace(0.5, 1.5, NH).astype(np.float32)[None]
    s = oracle_mod.indexer_scores_mx(qc, qs, w, cache, bt, [0], [n])
    qv = np.array([1.0, -1.0, 6.0, -6.0, 0.5, 0.0] * 6)[:NH] * 2.0
    per_head = np.maximum(0.0, qv)
    ref = np.array([np.sum(w[0].astype(np.float64) * per_head * 2.0 ** et) for et in e])
    assert np.allclose(s[0], ref, rtol=1e-14)


def test_indexer_mx_zero_query_and_linearity(oracle_mod):
    rng = np.random.default_rng(44)
    n = 130
    kc, ks = oracle_mod.mx_quantize(rng.standard_normal((n, D)))
    cache, bt = _mx_key_cache(kc, ks)
    qc, qs = oracle_mod.mx_quantize(rng.standard_normal((1, NH, D)))
    w = rng.uniform(0.01, 0.1, (1, NH)).astype(np.float32)
    s1 = oracle_mod.indexer_scores_mx(qc, qs, w, cache, bt, [0], [n])
    s4 = oracle_mod.indexer_scores_mx(qc, qs, w * 4, cache, bt, [0], [n])
    assert np.array_equal(s4, 4 * s1)
    z = oracle_mod.indexer_scores_mx(np.zeros_like(qc), qs, w, cache, bt, [0], [n])
    assert np.array_equal(z, np.zeros_like(z))


def test_write_key_mx_codes_and_placement(oracle_mod):
    """The MX Write step stores mx_quantize of torch's float64 layer_norm at the
    slot the shuffled block table names, and touches nothing else."""
    rng = np.random.default_rng(45)
    T, max_pages, num_pages = 40, 4, 9
    x = rng.standard_normal((T, D)) * 3 + 0.5
    k_raw = _bf16_bits(x)
    gamma = rng.uniform(0.5, 1.5, D)
    beta = rng.uniform(-0.2, 0.2, D)
    eps = 1e-6
    bt = rng.permutation(num_pages)[:2 * max_pages].astype(np.int32).reshape(2, max_pages)
    tok_req = rng.integers(0, 2, T).astype(np.int32)
    tok_pos = rng.choice(max_pages * PAGE, T, replace=False).astype(np.int32)
    cache0 = rng.integers(0, 256, (num_pages, MX_PAGE_BYTES)).astype(np.uint8)
    cache, key_pre = oracle_mod.write_key_mx(k_raw, gamma, beta, eps, bt, tok_req, tok_pos,
                                             cache0)
    ln = torch.nn.functional.layer_norm(torch.from_numpy(_bf16_vals(k_raw)), (D,),
                                        torch.from_numpy(gamma), torch.from_numpy(beta),
                                        eps).numpy()
    assert np.allclose(key_pre, ln, rtol=1e-12, atol=1e-12)
    codes, scales = oracle_mod.mx_quantize(key_pre)
    touched = np.zeros_like(cache0, dtype=bool)
    for t in range(T):
        pg = bt[tok_req[t], tok_pos[t] // PAGE]
        s = tok_pos[t] % PAGE
        assert np.array_equal(cache[pg, s * 64:(s + 1) * 64], codes[t])
        assert np.array_equal(cache[pg, PAGE * 64 + s * 4:PAGE * 64 + (s + 1) * 4], scales[t])
        touched[pg, s * 64:(s + 1) * 64] = True
        touched[pg, PAGE * 64 + s * 4:PAGE * 64 + (s + 1) * 4] = True
    assert np.array_equal(cache[~touched], cache0[~touched])


def test_mx_byte_model_matches_pages(oracle_mod):
    g = {k: float(v[0]) for k, v in _read_golden("byte_model.txt").items()}
    assert MX_PAGE_BYTES // PAGE == g["mxfp4_index_key_bytes_per_token"]
    assert oracle_mod.MX_KEY_PAGE_BYTES == MX_PAGE_BYTES
    assert round(100 * (1 - MX_PAGE_BYTES / PAGE / traffic.KEY_BYTES), 1) == g[
        "mxfp4_index_cache_saving"]
    assert 24 * (g["nvfp4_latent_bytes_per_token"] + MX_PAGE_BYTES // PAGE) == g[
        "kv_per_token_24_layers_k31_nvfp4_mxfp4"]
    assert traffic.MXFP4_KEY_BYTES == g["mxfp4_index_key_bytes_per_token"]
    wl = inputs.config(1)
    assert traffic.scan_bytes_mxfp4(wl) == sum(wl.ctx) * 68 + wl.R * NH * (68 + 4)


# ------------------------------------------------------------ NVFP4 latent
# Row of 352 bytes: 256 bytes of E2M1 codes of dims 0..511 (dim 2j in the low
# nibble of byte j), 32 unsigned-E4M3 block scales (byte b: dims 16b..16b+15),
# 64 E4M3 RoPE bytes (dims 512..575); every value times the per-tensor scale.
NV_ROW = 352


def test_nvfp4_latent_layout_last_dims(oracle_mod):
    row = np.zeros(NV_ROW, np.uint8)
    row[255] = 0x70                 # dim 510 = 0, dim 511 = E2M1 code 7 (6.0)
    row[256 + 31] = 0x30            # block 31 scale: E4M3 0.5
    row[256 + 32 + 63] = 0x40       # dim 575: E4M3 2.0
    L = oracle_mod.nvfp4_latent_decode(row, 0.25)
    want = np.zeros(LAT)
    want[511] = 6.0 * 0.5 * 0.25
    want[575] = 2.0 * 0.25
    assert np.array_equal(L, want)
    row[256 + 31] = 0xB0            # the scale is unsigned: its top bit is ignored
    assert np.array_equal(oracle_mod.nvfp4_latent_decode(row, 0.25), want)
    row[0] = 0x09                   # dim 0 = -0.5 (code 9), dim 1 = 0, block 0 scale still 0
    assert np.array_equal(oracle_mod.nvfp4_latent_decode(row, 0.25), want)
    row[256] = 0x38                 # block 0 scale 1.0
    want[0] = -0.5 * 0.25
    assert np.array_equal(oracle_mod.nvfp4_latent_decode(row, 0.25), want)


def _nv_grid_rows(rng, n, lo=-3, hi=3):
    """Latent rows every dim of which both NVFP4 and E4M3 hold exactly: per
    16-dim block E2M1 magnitudes x sign x 2^p with one element +-6 x 2^p (so the
    block scale is exactly 2^p), and E4M3 RoPE dims."""
    grid = _e2m1_grid()
    v = grid[rng.integers(0, 8, (n, 512))] * rng.choice([-1.0, 1.0], (n, 512))
    blocks = v.reshape(n, 32, 16)
    blocks[:, :, 0] = 6.0 * rng.choice([-1.0, 1.0], (n, 32))
    blocks *= np.ldexp(1.0, rng.integers(lo, hi + 1, (n, 32, 1)))
    rope = _e4m3_vals(_e4m3(rng.standard_normal((n, 64)) * 4))
    return np.concatenate([blocks.reshape(n, 512), rope], axis=1)


def test_nvfp4_encode_exact_on_shared_grid_and_error_bound(oracle_mod):
    rng = np.random.default_rng(50)
    v = _nv_grid_rows(rng, 20, lo=-6, hi=4)
    assert np.array_equal(oracle_mod.nvfp4_latent_decode(oracle_mod.nvfp4_latent_encode(v), 1.0), v)
    v = rng.standard_normal((20, LAT)) * rng.uniform(0.05, 20.0, (20, 1))
    rows = oracle_mod.nvfp4_latent_encode(v)
    d = oracle_mod.nvfp4_latent_decode(rows, 1.0)
    s = _e4m3_vals(rows[:, 256:288] & 0x7F)                # block scales
    amax = np.abs(v[:, :512]).reshape(20, 32, 16).max(-1)
    # E2M1 half-spacing is at most 1 below 6; beyond 6 * s the clamp loses amax - 6 s
    bound = s + np.maximum(0.0, amax - 6 * s)
    err = np.abs(d[:, :512] - v[:, :512]).reshape(20, 32, 16).max(-1)
    assert (err <= bound * (1 + 1e-12)).all()
    assert np.array_equal(d[:, 512:], _e4m3_vals(_e4m3(v[:, 512:])))


def test_mla_nvfp4_equals_fp8_on_shared_grid(oracle_mod):
    """Latent rows on the shared grid: NVFP4 and FP8 caches hold the same
    values, so the NVFP4 attention must equal the pinned FP8 attention."""
    rng = np.random.default_rng(51)
    n, H, k, ls = 150, 8, 96, 0.125
    vals = _nv_grid_rows(rng, n)
    fp8, bt = _latent_cache(_e4m3(vals))
    assert np.array_equal(_e4m3_vals(_e4m3(vals)), vals)
    nv = np.zeros((fp8.shape[0], PAGE, NV_ROW), np.uint8)
    rows = oracle_mod.nvfp4_latent_encode(vals)
    for t in range(n):
        nv[t // PAGE, t % PAGE] = rows[t]
    q = _bf16_bits(rng.standard_normal((2, H, LAT)) * 0.05)
    idx = np.full((2, k), -1, np.int32)
    idx[0, :90] = rng.choice(n, 90, replace=False)
    idx[1, :k] = rng.choice(120, k, replace=False)
    args = (ls, bt, [0, 0], [n, 120], idx)
    o8, l8 = oracle_mod.sparse_mla(q, 1 / math.sqrt(192), fp8, *args)
    o4, l4 = oracle_mod.sparse_mla_nvfp4(q, 1 / math.sqrt(192), nv, *args)
    assert np.allclose(o4, o8, rtol=1e-13, atol=1e-15) and np.allclose(l4, l8, rtol=1e-14)


def test_nvfp4_byte_model(oracle_mod):
    g = {k: float(v[0]) for k, v in _read_golden("byte_model.txt").items()}
    assert oracle_mod.NV_ROW_BYTES == NV_ROW == g["nvfp4_latent_bytes_per_token"]
