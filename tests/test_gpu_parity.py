"""GPU parity: every entry point of the C ABI against the float64 oracle on the
same seeded inputs, element by element at sizes the oracle finishes in
seconds (several tiles, ragged tails), and on sampled rows at the
benchmark's full sizes."""
import numpy as np
import pytest
import torch

import helpers
from dsa_sparse_attention_lightning_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dsa_sparse_attention_lightning_gb300 as m
    from dsa_sparse_attention_lightning_gb300 import _build
    _build.build()
    m.load()
    return m


DEV = "cuda"

SMALL = [
    inputs.Workload("one_row_4k", [4096], [1], H=16, seed=0, paged=False),
    inputs.Workload("ragged_multi", [3000, 700, 5000, 64], [2, 1, 4, 1], H=64, k=512, seed=1,
                    shift_frac=0.05),
    inputs.Workload("short_rows", [1, 63, 65, 2047, 2049], [1, 1, 2, 1, 3], H=32, seed=2),
    inputs.Workload("h128", [9000], [3], H=128, k=1024, seed=3, shift_frac=0.05),
    inputs.Workload("fp8_query", [6000, 2500], [4, 2], H=64, k=2048, seed=4, q_idx_fp8=True),
    # more than four rows per request with an E4M3 query: groups 4 + 4 + 3 and 4 + 1
    inputs.Workload("fp8_query_wide", [6000, 3000], [11, 5], H=32, k=1024, seed=7,
                    q_idx_fp8=True),
]


# Many short units: CTA ranges hold whole units (written straight out) as well
# as cut ones (merged by the combine), for one and for two head groups.
MLA_WIDE = [
    inputs.Workload("many_rows_h16", [300, 1000, 257] * 20, [7] * 60, H=16, k=256, seed=5),
    inputs.Workload("many_units_h128", [700, 260] * 10, [5] * 20, H=128, k=256, seed=6),
]


def _sub(host, rows):
    """Host inputs restricted to the given rows (caches and block table unchanged)."""
    h = dict(host)
    for key in ("q_idx", "q_idx_scale", "w", "row_req", "row_len", "q"):
        if h.get(key) is not None:
            h[key] = np.ascontiguousarray(h[key][rows])
    return h


def _run_step(dsa, inp, k, **kw):
    R = inp["row_len"].shape[0]
    idx = torch.full((R, k), -7, dtype=torch.int32, device=DEV)
    out, lse = dsa.dsa_decode_step(inp["q_idx"], inp["w"], inp["key_cache"], inp["latent_cache"],
                                   inp["latent_scale"], inp["block_table"], inp["row_req"],
                                   inp["row_len"], inp["q"], softmax_scale=inp["softmax_scale"],
                                   k=k, q_scale=inp["q_idx_scale"], idx_out=idx, **kw)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


# ------------------------------------------------------------------ scores
@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_indexer_scores_match_oracle(dsa, oracle_mod, wl):
    inp = inputs.make_inputs(wl, device=DEV)
    scores = dsa.dsa_indexer_score(inp["q_idx"], inp["w"], inp["key_cache"], inp["block_table"],
                                   inp["row_req"], inp["row_len"], q_scale=inp["q_idx_scale"])
    torch.cuda.synchronize()
    host = inputs.to_numpy(inp)
    ora = oracle_mod.indexer_scores(host["q_idx"], host["w"], host["key_cache"],
                                    host["block_table"], host["row_req"], host["row_len"],
                                    q_scale=host["q_idx_scale"])
    helpers.assert_scores_close(scores.cpu().numpy(), ora, host["row_len"])


# ------------------------------------------------------------------- top-k
# Rows of at most 49152 scores are selected by one CTA per row in shared
# memory, wider score buffers by the sample / collect / finalize kernels; a
# buffer padded to WIDE columns (poison past the data) takes the second path.
WIDE = 65536
TOPK_PATHS = {"row_in_smem": None, "sample_collect": WIDE}


def _topk_bitexact(dsa, oracle_mod, scores32, row_len, k, pad_to=None):
    R, ld = scores32.shape
    ld4 = (ld + 3) // 4 * 4
    if pad_to is not None:
        ld4 = max(ld4, pad_to)
    buf = np.full((R, ld4), 1e30, np.float32)
    buf[:, :ld] = scores32
    g = dsa.dsa_topk(torch.from_numpy(buf).to(DEV), torch.tensor(row_len, dtype=torch.int32,
                                                                 device=DEV), k)
    torch.cuda.synchronize()
    g = g.cpu().numpy()
    o = oracle_mod.topk(buf.astype(np.float64), row_len, k)
    for r in range(R):
        gs = g[r]
        n = min(k, row_len[r])
        assert np.all(gs[n:] == -1), f"row {r}: padding"
        assert np.all(np.diff(gs[:n]) > 0), f"row {r}: not ascending"
        assert np.array_equal(gs[:n], np.sort(o[r, :n])), f"row {r}: selection differs"


@pytest.mark.parametrize("path", list(TOPK_PATHS))
@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_topk_bitexact_on_oracle_scores(dsa, oracle_mod, wl, path):
    host = inputs.to_numpy(inputs.make_inputs(wl, device="cpu"))
    ora = oracle_mod.indexer_scores(host["q_idx"], host["w"], host["key_cache"],
                                    host["block_table"], host["row_req"], host["row_len"],
                                    q_scale=host["q_idx_scale"])
    s32 = np.nan_to_num(ora, nan=0.0).astype(np.float32)
    _topk_bitexact(dsa, oracle_mod, s32, list(host["row_len"]), wl.k, TOPK_PATHS[path])


@pytest.mark.parametrize("path", list(TOPK_PATHS))
def test_topk_ties_signs_and_edges(dsa, oracle_mod, path):
    rng = np.random.default_rng(0)
    L = 20000
    rows = [
        rng.integers(0, 50, L).astype(np.float32),          # heavy exact ties at the cut
        np.zeros(L, np.float32),                            # all equal
        np.where(rng.random(L) < 0.5, -0.0, 0.0).astype(np.float32),
        -np.abs(rng.standard_normal(L)).astype(np.float32),  # all negative
        rng.standard_normal(L).astype(np.float32),
        np.full(L, 3.0, np.float32),
        rng.standard_normal(L).astype(np.float32) * 1e-30,  # subnormal-adjacent scale
        rng.integers(0, 3, L).astype(np.float32) * 1e6,
    ]
    s = np.stack(rows)
    lens = [L, L, L, L, 2048, 2049, 4097, 1]
    pad = TOPK_PATHS[path]
    for k in (2048, 1, 7, 1000):
        _topk_bitexact(dsa, oracle_mod, s, lens, k, pad)
    _topk_bitexact(dsa, oracle_mod, s[:2], [0, 5], 16, pad)
    # the largest row the one-CTA path holds, and one past it (other path)
    for L2 in (49152, 49153):
        big = rng.integers(0, 200, (1, L2)).astype(np.float32)
        _topk_bitexact(dsa, oracle_mod, big, [L2], 2048, pad)


@pytest.mark.parametrize("path", list(TOPK_PATHS))
def test_topk_rows_built_against_the_sample(dsa, oracle_mod, path):
    """The selection is exact whatever a fixed sample of the row suggests: rows
    whose best scores sit only outside, or only inside, the sampled blocks
    (every 16th block of 32 scores), so the candidate threshold is far too low
    (candidates overflow) or too high (fewer than k candidates)."""
    rng = np.random.default_rng(2)
    L = 40000
    pos = np.arange(L)
    in_sample = (pos // 32) % 16 == 0
    hidden = rng.standard_normal(L).astype(np.float32)
    hidden[~in_sample] += 10.0                           # best scores never sampled
    only = rng.standard_normal(L).astype(np.float32)
    only[in_sample] += 10.0                              # 2528 sampled highs, then noise
    short = rng.standard_normal(L).astype(np.float32)
    short[in_sample & (pos < 16384)] += 10.0             # 1024 sampled highs < k
    s = np.stack([hidden, only, short])
    _topk_bitexact(dsa, oracle_mod, s, [L, L, 16384], 2048, TOPK_PATHS[path])


def test_topk_long_row_split_over_chunks(dsa, oracle_mod):
    rng = np.random.default_rng(1)
    L = 1 << 20
    s = rng.standard_normal((1, L)).astype(np.float32)
    s[0, rng.choice(L, 3000, replace=False)] = 5.5      # 3000 exact ties straddling the cut
    _topk_bitexact(dsa, oracle_mod, s, [L], 2048)


def test_topk_many_long_rows_full_size(dsa, oracle_mod):
    """64 rows of up to 262144 scores (16 requests x 4 rows at 256K context),
    the sample / collect / finalize path: random rows, exact ties straddling the cut,
    winners only at the end of the row, all scores equal, rising in steps,
    thresholds from the sample far too low (more candidates than the list
    holds) and too high (fewer than k), both taking the whole-row select, and
    ragged lengths."""
    rng = np.random.default_rng(5)
    R, L = 64, 262144
    pos = np.arange(L)
    s = rng.standard_normal((R, L)).astype(np.float32)
    s[1, rng.choice(L, 3000, replace=False)] = 5.5
    s[2] = (pos * 1e-3).astype(np.float32)                 # rising: the last 2048 win
    s[3] = 1.0                                             # all equal: the first 2048
    s[4] = (pos // 4096).astype(np.float32)                # rising in steps of exact ties
    s[5, :] = 1.0
    s[5, (pos // 32) % 64 == 0] = 2.0                      # half the sampled blocks: 4096 ties
    sampled = (pos // 32) % 32 == 0                        # the blocks the sample reads at 256K
    s[6, ~sampled] += 10.0                                 # threshold far too low: the list
    s[10, sampled & (pos < 16384)] += 10.0                 # overflows; too high: < k candidates
    lens = [L] * R
    lens[7], lens[8], lens[9] = 49153, 100001, 2048
    _topk_bitexact(dsa, oracle_mod, s, lens, 2048)


# ------------------------------------------------------------------ the Write step
def test_write_kv_matches_oracle(dsa, oracle_mod):
    rng = np.random.default_rng(11)
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
    beta = (rng.standard_normal(128) * 0.1).astype(np.float32)
    beta_zero = np.zeros(128, np.float32)
    eps, ls = 1e-6, 0.0125
    kc0 = np.full((num_pages, 8448), 0x7F, np.uint8)
    lc0 = np.full((num_pages, 64, 576), 0x7F, np.uint8)
    for b_vec in (beta, beta_zero):
        kb = torch.from_numpy(x).to(torch.bfloat16)
        lb = torch.from_numpy(lat).to(torch.bfloat16)
        kc = torch.from_numpy(kc0).to(DEV)
        lc = torch.from_numpy(lc0).to(DEV)
        st = torch.full((1,), 7, dtype=torch.int32, device=DEV)
        dsa.dsa_write_kv(kb.to(DEV), torch.from_numpy(gamma).to(DEV), torch.from_numpy(b_vec).to(DEV),
                         eps, lb.to(DEV), ls, torch.from_numpy(bt).to(DEV),
                         torch.from_numpy(req).to(DEV), torch.from_numpy(pos).to(DEV), kc, lc,
                         dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        kcg, lcg = kc.cpu().numpy(), lc.cpu().numpy()
        okc, olc, kpre, lpre, ks = oracle_mod.write_kv(
            kb.view(torch.int16).numpy().view(np.uint16), gamma.astype(np.float64),
            b_vec.astype(np.float64), eps, lb.view(torch.int16).numpy().view(np.uint16), ls, bt,
            req, pos, kc0, lc0)
        mids = helpers.e4m3_midpoints(oracle_mod)
        written_k = np.zeros(kc0.shape, bool)
        written_l = np.zeros(lc0.shape[:2], bool)
        for t in range(T):
            page, slot = bt[req[t], pos[t] // 64], pos[t] % 64
            # the scale within 1e-6 relative; the codes equal except at rounding midpoints
            g_ks = kcg[page, 8192 + 4 * slot:8196 + 4 * slot].view(np.float32)[0]
            assert abs(g_ks - ks[t]) <= 1e-6 * ks[t], t
            keys = slice(128 * slot, 128 * slot + 128)
            ok = helpers.near_midpoint(kpre[t], mids) | (kcg[page, keys] == okc[page, keys])
            assert ok.all(), (t, np.flatnonzero(~ok))
            ok = helpers.near_midpoint(lpre[t], mids) | (lcg[page, slot] == olc[page, slot])
            assert ok.all(), (t, np.flatnonzero(~ok))
            written_k[page, keys] = True
            written_k[page, 8192 + 4 * slot:8196 + 4 * slot] = True
            written_l[page, slot] = True
        # bytes of slots the call does not own are untouched
        assert np.array_equal(kcg[~written_k], kc0[~written_k])
        assert np.array_equal(lcg[~written_l], lc0[~written_l])


def test_write_kv_flags_bad_tokens(dsa):
    kc = torch.full((4, 8448), 0x7F, dtype=torch.uint8, device=DEV)
    lc = torch.full((4, 64, 576), 0x7F, dtype=torch.uint8, device=DEV)
    bt = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device=DEV)
    kb = torch.randn(3, 128, device=DEV).to(torch.bfloat16)
    lb = torch.randn(3, 576, device=DEV).to(torch.bfloat16)
    one, zero = torch.ones(128, device=DEV), torch.zeros(128, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    req = torch.tensor([0, 5, 1], dtype=torch.int32, device=DEV)     # request 5 does not exist
    pos = torch.tensor([3, 0, 200], dtype=torch.int32, device=DEV)   # 200 >= 2 pages x 64
    dsa.dsa_write_kv(kb, one, zero, 1e-6, lb, 0.05, bt, req, pos, kc, lc, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0x1                       # DSA_DEV_BAD_ROW
    assert (kc[0, 3 * 128:4 * 128] != 0x7F).any()      # the valid token was written
    assert (kc[1:] == 0x7F).all() and (lc[1:] == 0x7F).all()


# ------------------------------------------- top-k by the context-parallel exchange
def _dcp_rows(rng, L, W):
    base = rng.standard_normal(L).astype(np.float32)
    conc = base.copy()
    conc[(W - 1)::W] += 10.0                    # shard W-1 holds every winner
    first = base.copy()
    first[:: 2 * W] += 10.0                     # half of shard 0's tokens win
    ties = rng.integers(0, 20, L).astype(np.float32)
    return np.stack([base, conc, first, ties, np.zeros(L, np.float32)])


def _dcp_check(dsa, oracle_mod, s32, lens, k, W):
    sc = torch.from_numpy(s32).to(DEV)
    rl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    g_idx, g_res = dsa.dsa_topk_dcp(sc, rl, k, W)
    t_idx = dsa.dsa_topk(sc, rl, k)
    torch.cuda.synchronize()
    g_idx, t_idx = g_idx.cpu().numpy(), t_idx.cpu().numpy()
    assert np.array_equal(g_idx, t_idx), "exchange differs from the single-shard top-k"
    o_idx, o_res = oracle_mod.topk_dcp(s32.astype(np.float64), lens, k, W)
    assert np.array_equal(g_res.cpu().numpy().view(np.uint32), o_res), "resend pattern"
    for r in range(s32.shape[0]):
        n = min(k, lens[r])
        assert np.array_equal(g_idx[r, :n], np.sort(o_idx[r, :n]))
        assert np.all(g_idx[r, n:] == -1)
    return o_res


@pytest.mark.parametrize("W", [1, 2, 3, 8])
def test_topk_dcp_matches_topk_and_oracle(dsa, oracle_mod, W):
    rng = np.random.default_rng(40 + W)
    L = 20000
    s32 = _dcp_rows(rng, L, W)
    for k in (7, 300, 2048):
        for lens in ([L] * 5, [L, 5000, 4097, 2 * W + 1, max(W - 1, 0)]):
            _dcp_check(dsa, oracle_mod, s32, lens, k, W)


def test_topk_dcp_full_size_rows(dsa, oracle_mod):
    """256K rows (shards of 32K: one-CTA top-k; the member rows: the
    sample / collect path) and one 1M row, eight shards."""
    rng = np.random.default_rng(7)
    W, k = 8, 2048
    s32 = _dcp_rows(rng, 262144, W)[:3]
    res = _dcp_check(dsa, oracle_mod, s32, [262144, 262144, 200000], k, W)
    assert res[1] == 1 << (W - 1)
    big = rng.standard_normal((1, 1 << 20)).astype(np.float32)
    big[0, 5::W] += 5.0
    res = _dcp_check(dsa, oracle_mod, big, [1 << 20], k, W)
    assert res[0] == 1 << 5


# --------------------------------------------------------------- sparse MLA
@pytest.mark.parametrize("wl", SMALL + MLA_WIDE, ids=[w.name for w in SMALL + MLA_WIDE])
def test_sparse_mla_matches_oracle(dsa, oracle_mod, wl):
    inp = inputs.make_inputs(wl, device=DEV)
    host = inputs.to_numpy(inp)
    rng = np.random.default_rng(wl.seed)
    idx = np.full((wl.R, wl.k), -1, np.int32)
    for r, L in enumerate(host["row_len"]):
        n = min(wl.k, L)
        sel = rng.choice(L, n, replace=False).astype(np.int32) if L else np.zeros(0, np.int32)
        pos = rng.choice(wl.k, n, replace=False)       # valid ids scattered among -1 slots
        idx[r, pos] = sel
    out, lse = dsa.dsa_sparse_mla_decode(inp["q"], inp["latent_cache"], inp["latent_scale"],
                                         inp["block_table"], inp["row_req"], inp["row_len"],
                                         torch.from_numpy(idx).to(DEV),
                                         softmax_scale=inp["softmax_scale"])
    torch.cuda.synchronize()
    oo, ol = oracle_mod.sparse_mla(host["q"], host["softmax_scale"], host["latent_cache"],
                                   host["latent_scale"], host["block_table"], host["row_req"],
                                   host["row_len"], idx)
    helpers.assert_out_close(out.float().cpu().numpy(), oo)
    lg = lse.cpu().numpy()
    fin = np.isfinite(ol)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.allclose(lg[fin], ol[fin], rtol=1e-4, atol=1e-4)


def test_sparse_mla_dense_equivalence(dsa, oracle_mod):
    """k >= context: the step's sparse attention equals dense MLA over every token."""
    wl = inputs.Workload("dense", [1500, 900], [2, 1], H=64, k=2048, seed=9)
    inp = inputs.make_inputs(wl, device=DEV)
    idx, out, lse = _run_step(dsa, inp, wl.k)
    host = inputs.to_numpy(inp)
    dense = np.full((wl.R, wl.k), -1, np.int32)
    for r, L in enumerate(host["row_len"]):
        dense[r, :L] = np.arange(L)
        assert np.array_equal(idx[r], dense[r])
    od, ld = oracle_mod.sparse_mla(host["q"], host["softmax_scale"], host["latent_cache"],
                                   host["latent_scale"], host["block_table"], host["row_req"],
                                   host["row_len"], dense)
    helpers.assert_out_close(out, od)
    assert np.allclose(lse, ld, rtol=1e-4, atol=1e-4)


# ------------------------------------------------------------ fused step
@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_decode_step_matches_oracle(dsa, oracle_mod, wl):
    inp = inputs.make_inputs(wl, device=DEV)
    idx, out, lse = _run_step(dsa, inp, wl.k)
    host = inputs.to_numpy(inp)
    scores, oidx, oout, olse = oracle_mod.decode_step(host, k=wl.k)
    helpers.assert_topk_equal_outside_near_ties(idx, oidx, scores, host["row_len"], wl.k)
    # attention is compared on the GPU's own selection (the oracle attends over it)
    oo, ol = oracle_mod.sparse_mla(host["q"], host["softmax_scale"], host["latent_cache"],
                                   host["latent_scale"], host["block_table"], host["row_req"],
                                   host["row_len"], idx)
    helpers.assert_out_close(out, oo)
    for r in range(wl.R):
        if helpers.selected(idx[r]) == helpers.selected(oidx[r]):
            helpers.assert_out_close(out[r], oout[r])


def test_decode_step_deterministic_and_batch_invariant(dsa):
    wl = inputs.Workload("inv", [5000, 3000, 7000], [4, 1, 2], H=64, seed=12, shift_frac=0.05)
    inp = inputs.make_inputs(wl, device=DEV)
    a = _run_step(dsa, inp, wl.k)
    b = _run_step(dsa, inp, wl.k)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # rows 4 (request 1) alone: same selection, same output
    sub = dict(inp)
    for key in ("q_idx", "w", "row_req", "row_len", "q"):
        sub[key] = inp[key][4:5].contiguous()
    c = _run_step(dsa, sub, wl.k)
    assert np.array_equal(c[0][0], a[0][4])
    assert np.abs(c[1][0] - a[1][4]).max() <= 1e-2


def test_step_attention_equals_standalone_call_on_reused_memory(dsa):
    """The fused step launches its attention kernel while the selection kernel
    is still finishing (programmatic dependent launch).  Two steps in a row,
    each with freshly allocated selection, output and workspace buffers (so
    they land on memory the previous calls used), must give exactly what the
    standalone attention call gives on the step's own selection: a read of
    the selection that ran ahead of its producer shows up here as stale data."""
    wl = inputs.config(1)                        # 16 x 4 rows, 32K: units cut over CTAs
    inp = inputs.make_inputs(wl, device=DEV)
    for _ in range(3):
        idx = torch.full((wl.R, wl.k), -7, dtype=torch.int32, device=DEV)
        out, lse = dsa.dsa_decode_step(inp["q_idx"], inp["w"], inp["key_cache"],
                                       inp["latent_cache"], inp["latent_scale"],
                                       inp["block_table"], inp["row_req"], inp["row_len"],
                                       inp["q"], softmax_scale=inp["softmax_scale"], k=wl.k,
                                       idx_out=idx)
        out2, lse2 = dsa.dsa_sparse_mla_decode(inp["q"], inp["latent_cache"], inp["latent_scale"],
                                               inp["block_table"], inp["row_req"],
                                               inp["row_len"], idx,
                                               softmax_scale=inp["softmax_scale"])
        torch.cuda.synchronize()
        assert torch.equal(out, out2) and torch.equal(lse, lse2)


# ------------------------------------------------- selection on built rows
# The step's selection must equal dsa_topk over the full scores of
# dsa_indexer_score bit for bit (the same kernels run on the same inputs),
# also on rows built against the top-k's sampled threshold.
def _step_vs_full_scores(dsa, inp, k):
    R = inp["row_len"].shape[0]
    idx = torch.full((R, k), -7, dtype=torch.int32, device=DEV)
    dsa.dsa_decode_step(inp["q_idx"], inp["w"], inp["key_cache"], inp["latent_cache"],
                        inp["latent_scale"], inp["block_table"], inp["row_req"], inp["row_len"],
                        inp["q"], softmax_scale=inp["softmax_scale"], k=k,
                        q_scale=inp["q_idx_scale"], idx_out=idx)
    scores = dsa.dsa_indexer_score(inp["q_idx"], inp["w"], inp["key_cache"], inp["block_table"],
                                   inp["row_req"], inp["row_len"], q_scale=inp["q_idx_scale"])
    ref = dsa.dsa_topk(scores, inp["row_len"], k)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref)
    return idx.cpu().numpy(), scores


def _set_keys(inp, scale_of_pos):
    """Every token's index key = one fixed E4M3 code vector, its scale
    scale_of_pos(position) (so the scores follow the scale)."""
    kc = inp["key_cache"]
    P = kc.shape[0]
    codes = kc[:, :64 * 128].view(P, 64, 128)
    scales = kc[:, 64 * 128:].view(torch.float32).view(P, 64)
    g = torch.Generator(device=DEV).manual_seed(99)
    vec = torch.randn(128, generator=g, device=DEV)
    code = (vec / vec.abs().max() * 448).to(torch.float8_e4m3fn).view(torch.uint8)
    bt = inp["block_table"].long()
    for b, L in enumerate(inp["ctx"]):
        pos = torch.arange(L, device=DEV)
        pg, sl = bt[b, pos // 64], pos % 64
        codes[pg, sl] = code
        scales[pg, sl] = scale_of_pos(pos).float()


@pytest.mark.parametrize("rows", [[2, 1, 1, 3], [8, 8, 8, 8]], ids=["7_rows", "32_rows"])
@pytest.mark.parametrize("pattern", ["equal", "rising", "rising_steps", "ties_at_cut"])
def test_step_selection_adversarial_rows(dsa, oracle_mod, pattern, rows):
    """Rows built against the selection: all scores equal (ties broken by
    position), scores rising along the context (the winners come last),
    rising in steps (long runs of exact ties), and many exact ties at the
    cut; rows long enough for the sample / collect / finalize path (7 or 32
    rows) and short ones for the one-CTA path."""
    ctx = [300000, 70000, 5000, 2100]
    wl = inputs.Workload("sel_adv", ctx, rows, H=16, k=2048, seed=31)
    inp = inputs.make_inputs(wl, device=DEV)
    inp["ctx"] = ctx
    f = {"equal": lambda p: torch.ones_like(p, dtype=torch.float64),
         "rising": lambda p: 1.0 + p.double() * 1e-4,
         "rising_steps": lambda p: 1.0 + (p // 4096).double(),
         "ties_at_cut": lambda p: torch.where(p % 7 == 0, 2.0, 1.0).double()}[pattern]
    _set_keys(inp, f)
    idx, scores = _step_vs_full_scores(dsa, inp, wl.k)
    lens = inp["row_len"].cpu().numpy()
    s32 = scores.cpu().numpy()
    s32 = np.where(np.arange(s32.shape[1])[None, :] < lens[:, None], s32, 0)   # past len: unset
    o = oracle_mod.topk(s32.astype(np.float64), lens, wl.k)
    for r, L in enumerate(lens):
        n = min(wl.k, L)
        assert np.all(np.diff(idx[r, :n]) > 0) and np.all(idx[r, n:] == -1)
        assert np.array_equal(idx[r, :n], np.sort(o[r, :n])), f"row {r}"
        if pattern == "equal":
            assert np.array_equal(idx[r, :n], np.arange(n))


def test_device_checks_flag_bad_values(dsa):
    wl = inputs.Workload("bad", [300], [1], H=16, k=64, seed=13)
    inp = inputs.make_inputs(wl, device=DEV)
    ws = torch.empty(dsa.decode_step_workspace_size(1, 1, wl.max_pages, 16, 64), dtype=torch.uint8,
                     device=DEV)
    bt = inp["block_table"].clone()
    bt[0, 2] = 10_000_000                        # page id out of range
    dsa.dsa_decode_step(inp["q_idx"], inp["w"], inp["key_cache"], inp["latent_cache"],
                        inp["latent_scale"], bt, inp["row_req"], inp["row_len"], inp["q"],
                        softmax_scale=inp["softmax_scale"], k=64, workspace=ws)
    assert dsa.check_device_status(ws) & 0x2
    idx = torch.tensor([[0, 5, 299, 300, -1]], dtype=torch.int32, device=DEV)   # 300 >= len
    wsm = torch.empty(dsa.sparse_mla_workspace_size(1, 16, 5), dtype=torch.uint8, device=DEV)
    dsa.dsa_sparse_mla_decode(inp["q"], inp["latent_cache"], inp["latent_scale"],
                              inp["block_table"], inp["row_req"], inp["row_len"], idx,
                              softmax_scale=inp["softmax_scale"], workspace=wsm)
    assert dsa.check_device_status(wsm) & 0x4
    # a clean call clears the word
    dsa.dsa_decode_step(inp["q_idx"], inp["w"], inp["key_cache"], inp["latent_cache"],
                        inp["latent_scale"], inp["block_table"], inp["row_req"], inp["row_len"],
                        inp["q"], softmax_scale=inp["softmax_scale"], k=64, workspace=ws)
    assert dsa.check_device_status(ws) == 0


def test_bounded_wait_runs_out_and_context_stays_usable(dsa):
    """A wait that nothing satisfies ends in the timeout bit, not a hang: the
    self-test CTA gives up after its 2 ms limit, drains the bulk copy it had in
    flight, frees its tensor memory and returns; later launches on the same
    context run normally."""
    import time
    ws = torch.zeros(dsa.selftest_workspace_size(), dtype=torch.uint8, device=DEV)
    pattern = ((torch.arange(256, device=DEV) * 7 + 3) % 251).to(torch.uint8)
    ws[256:512] = pattern
    for _ in range(2):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dsa.selftest_bounded_wait(2000, ws)
        bits = dsa.check_device_status(ws)
        dt = time.perf_counter() - t0
        assert bits == 0x8
        assert torch.equal(ws[512:768], pattern)
        assert 1.5e-3 <= dt < 1.0
        ws[512:768] = 0
    wl = inputs.Workload("after_timeout", [900], [2], H=16, k=64, seed=14)
    inp = inputs.make_inputs(wl, device=DEV)
    wss = torch.empty(dsa.decode_step_workspace_size(1, 2, wl.max_pages, 16, 64),
                      dtype=torch.uint8, device=DEV)
    out, lse = dsa.dsa_decode_step(inp["q_idx"], inp["w"], inp["key_cache"], inp["latent_cache"],
                                   inp["latent_scale"], inp["block_table"], inp["row_req"],
                                   inp["row_len"], inp["q"], softmax_scale=inp["softmax_scale"],
                                   k=64, workspace=wss)
    assert dsa.check_device_status(wss) == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


# ----------------------------------------------- full benchmark sizes, sampled
FULL = [1, 2, 3, 4]


@pytest.mark.parametrize("ci", FULL, ids=[inputs.config(i).name for i in FULL])
def test_full_size_sampled_rows(dsa, oracle_mod, ci):
    wl = inputs.config(ci)
    inp = inputs.make_inputs(wl, device=DEV)
    idx, out, lse = _run_step(dsa, inp, wl.k)
    host = inputs.to_numpy(inp)
    rows = sorted({0, wl.R - 1, wl.R // 2, 1 % wl.R})
    sub = _sub(host, rows)
    scores, oidx, _, _ = oracle_mod.decode_step(sub, k=wl.k)
    helpers.assert_topk_equal_outside_near_ties(idx[rows], oidx, scores, sub["row_len"], wl.k)
    oo, ol = oracle_mod.sparse_mla(sub["q"], sub["softmax_scale"], sub["latent_cache"],
                                   sub["latent_scale"], sub["block_table"], sub["row_req"],
                                   sub["row_len"], idx[rows])
    helpers.assert_out_close(out[rows], oo)
    assert np.allclose(lse[rows], ol, rtol=1e-4, atol=1e-4)
    # every row: selection size, ascending ids, finite output
    for r in range(wl.R):
        n = min(wl.k, int(host["row_len"][r]))
        assert np.all(np.diff(idx[r, :n]) > 0) and np.all(idx[r, n:] == -1)
    assert np.isfinite(out).all()
    if wl.planted:
        planted = set(host["planted"][0].tolist())
        assert helpers.selected(idx[0]) == planted
