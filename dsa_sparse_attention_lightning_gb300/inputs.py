"""Seeded synthetic inputs for one DSA decode step.

This module only draws random numbers and lays them out in the cache formats
the library reads; it holds none of the step's arithmetic (no score, no
selection, no attention).  The same tensors feed the CUDA library and, copied
to the host, the float64 oracle.

Shapes follow the pages' decode microbenchmark (TokenSpeed post on Kimi K3.1
Pro, "Reducing indexer overhead on AMD MI350X": 16 requests x 4 verification
rows at 16K-1M tokens) and the model's attention shapes (vLLM Day-0 post,
"What Kimi K3.1 Pro changes": indexer 32 heads x 128 dims, FP8 keys; the AMD
Instinct post's overview table: 576-wide latent = 512 KV + 64 RoPE).

Cache layouts (all caller-owned device memory):
  key_cache    uint8 [num_pages, 8448]: per 64-token page, 64 x 128 E4M3 key
               bytes, then 64 little-endian fp32 key scales.
  latent_cache uint8 [num_pages, 64, 576]: E4M3 latent rows, one fp32 scale
               for the whole tensor.
  block_table  int32 [B, max_pages]: page of each 64-token block of each
               request (both caches share it); unused entries are -1.
Slots past a request's context in its last page, and spare pages, hold the
E4M3 NaN code 0x7F so that any read of them shows up as NaN.

Key quantization (the generator's, not part of the step): per token,
scale = absmax / 448 and code = RNE(key / scale) as E4M3 (torch's float8
cast); an all-zero key gets scale 1.  The latent uses one absmax/448 scale for
the whole cache.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

PAGE = 64
IDX_HEADS = 32
IDX_DIM = 128
KEY_PAGE_BYTES = PAGE * IDX_DIM + PAGE * 4
LAT_DIM = 576
V_DIM = 512
E4M3_MAX = 448.0
E4M3_NAN = 0x7F


@dataclasses.dataclass
class Workload:
    """One decode step's shape and data recipe."""
    name: str
    ctx: List[int]                 # context length of each request
    rows: List[int]                # query rows of each request
    H: int = 64                    # MLA query heads
    k: int = 2048                  # tokens selected per row
    seed: int = 0
    paged: bool = True             # shuffled block table (else identity)
    shift_frac: float = 0.0        # fraction of tokens given a +3 sigma direction
    planted: int = 0               # tokens planted along the weighted query
    q_idx_fp8: bool = False        # E4M3 indexer query + fp32 (row, head) scale
    spare_pages: int = 2           # poisoned pages not referenced by any request
    softmax_scale: float = 1.0 / math.sqrt(192.0)

    @property
    def B(self) -> int:
        return len(self.ctx)

    @property
    def R(self) -> int:
        return int(sum(self.rows))

    def row_lengths(self) -> List[int]:
        """Row j of a request with c tokens and n rows sees c - n + 1 + j tokens."""
        out = []
        for c, n in zip(self.ctx, self.rows):
            out += [c - n + 1 + j for j in range(n)]
        return out

    @property
    def max_pages(self) -> int:
        return max(1, max((c + PAGE - 1) // PAGE for c in self.ctx))


def config(i: int) -> Workload:
    """The five workloads of the benchmark contract (0-based)."""
    if i == 0:   # tiny decode step
        return Workload("tiny_1x1_ctx4096_h16", [4096], [1], H=16, seed=0, paged=False)
    if i == 1:   # batched verification decode, 32K
        return Workload("decode_16x4_ctx32768_h64", [32768] * 16, [4] * 16, H=64, seed=1,
                        shift_frac=0.05)
    if i == 2:   # batched verification decode, 256K
        return Workload("decode_16x4_ctx262144_h64", [262144] * 16, [4] * 16, H=64, seed=2,
                        shift_frac=0.05)
    if i == 3:   # one long stream, 1M, planted winners
        return Workload("decode_1x1_ctx1048576_h64", [1048576], [1], H=64, seed=3,
                        planted=2048)
    if i == 4:   # prefill chunk of 4096 rows at 128K, FP8 indexer query
        return Workload("prefill_4096rows_ctx131072_h64", [131072], [4096], H=64, seed=4,
                        q_idx_fp8=True)
    raise ValueError(i)


def _e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """E4M3 codes (uint8) of values already scaled into [-448, 448]."""
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def _absmax_scale(x: torch.Tensor, dim: int) -> torch.Tensor:
    amax = x.abs().amax(dim=dim, keepdim=True)
    return torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))


def make_inputs(wl: Workload, device="cpu", chunk_tokens: int = 1 << 20) -> Dict[str, object]:
    """Draw the step's inputs on ``device`` (seeded by ``wl.seed``).

    Returns torch tensors: q_idx (bf16 [R,32,128], or uint8 E4M3 codes with
    q_idx_scale fp32 [R,32]), w fp32 [R,32], key_cache, latent_cache,
    latent_scale (float), block_table, row_req, row_len (int32), q bf16
    [R,H,576], softmax_scale (float), k (int) and the planted positions (per
    request, int64, possibly empty).
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(wl.seed))
    B, R = wl.B, wl.R

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)

    # ---- rows -----------------------------------------------------------
    row_req = torch.tensor([b for b, n in enumerate(wl.rows) for _ in range(n)],
                           dtype=torch.int32, device=dev)
    row_len = torch.tensor(wl.row_lengths(), dtype=torch.int32, device=dev)

    # ---- indexer query and head weights ---------------------------------
    qi = randn(R, IDX_HEADS, IDX_DIM)
    w = torch.softmax(randn(R, IDX_HEADS), dim=-1).contiguous()
    if wl.q_idx_fp8:
        q_idx_scale = _absmax_scale(qi, dim=2)                       # [R,32,1]
        q_idx = _e4m3_codes(qi / q_idx_scale).contiguous()
        q_idx_scale = q_idx_scale.squeeze(-1).contiguous()
    else:
        q_idx = qi.to(torch.bfloat16).contiguous()
        q_idx_scale = None

    # ---- pages and block table -------------------------------------------
    pages_per_req = [(c + PAGE - 1) // PAGE for c in wl.ctx]
    used = int(sum(pages_per_req))
    num_pages = used + int(wl.spare_pages)
    if wl.paged:
        perm = torch.randperm(num_pages, generator=g, device=dev)[:used]
    else:
        perm = torch.arange(used, device=dev)
    block_table = torch.full((B, wl.max_pages), -1, dtype=torch.int32, device=dev)
    off = 0
    for b, n in enumerate(pages_per_req):
        block_table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n

    key_cache = torch.full((num_pages, KEY_PAGE_BYTES), E4M3_NAN, dtype=torch.uint8, device=dev)
    key_vals = key_cache[:, :PAGE * IDX_DIM].view(num_pages, PAGE, IDX_DIM)
    key_scales = key_cache[:, PAGE * IDX_DIM:].view(torch.float32)       # [num_pages, 64]
    key_scales.fill_(float("nan"))

    # ---- index keys, request by request ---------------------------------
    planted_pos = []
    for b, c in enumerate(wl.ctx):
        bt = block_table[b, :pages_per_req[b]].to(torch.int64)
        shift_u = None
        shifted = None
        if wl.shift_frac > 0:
            u = randn(IDX_DIM)
            shift_u = 3.0 * u / u.norm()
            n_shift = int(round(wl.shift_frac * c))
            shifted = torch.randperm(c, generator=g, device=dev)[:n_shift]
        planted = None
        plant_dir = None
        if wl.planted > 0:
            planted = torch.randperm(c, generator=g, device=dev)[:wl.planted]
            r0 = int(sum(wl.rows[:b]))
            v = (w[r0].unsqueeze(-1) * qi[r0]).sum(0)
            plant_dir = 1.5 * math.sqrt(IDX_DIM) * v / v.norm()
        planted_pos.append(planted.cpu() if planted is not None
                           else torch.empty(0, dtype=torch.int64))
        for t0 in range(0, c, chunk_tokens):
            t1 = min(c, t0 + chunk_tokens)
            kv = randn(t1 - t0, IDX_DIM)
            if shifted is not None:
                sel = shifted[(shifted >= t0) & (shifted < t1)] - t0
                kv[sel] += shift_u
            if planted is not None:
                sel = planted[(planted >= t0) & (planted < t1)] - t0
                kv[sel] = plant_dir + 0.1 * randn(int(sel.numel()), IDX_DIM)
            sc = _absmax_scale(kv, dim=1)                                   # [n,1]
            codes = _e4m3_codes(kv / sc)
            tok = torch.arange(t0, t1, device=dev)
            pg = bt[tok // PAGE]
            slot = tok % PAGE
            key_vals[pg, slot] = codes
            key_scales[pg, slot] = sc.squeeze(1)

    # ---- latent rows (one per token, one scale for the tensor) -----------
    # Drawn twice from a generator of their own: the first pass finds the
    # absmax for the tensor-wide scale, the second quantizes the same values.
    latent_cache = torch.full((num_pages, PAGE, LAT_DIM), E4M3_NAN, dtype=torch.uint8, device=dev)
    lat_seed = int(torch.randint(0, 2**62, (1,), generator=g, device=dev).item())
    amax = 0.0
    for quantize in (False, True):
        gl = torch.Generator(device=dev)
        gl.manual_seed(lat_seed)
        if quantize:
            latent_scale = amax / E4M3_MAX if amax > 0 else 1.0
        for b, c in enumerate(wl.ctx):
            bt = block_table[b, :pages_per_req[b]].to(torch.int64)
            for t0 in range(0, c, chunk_tokens):
                t1 = min(c, t0 + chunk_tokens)
                x = torch.randn(t1 - t0, LAT_DIM, generator=gl, device=dev, dtype=torch.float32)
                if not quantize:
                    amax = max(amax, float(x.abs().amax()))
                    continue
                tok = torch.arange(t0, t1, device=dev)
                latent_cache[bt[tok // PAGE], tok % PAGE] = _e4m3_codes(x / latent_scale)

    # ---- MLA query --------------------------------------------------------
    q = randn(R, wl.H, LAT_DIM).to(torch.bfloat16).contiguous()

    return {
        "q_idx": q_idx, "q_idx_scale": q_idx_scale, "w": w,
        "key_cache": key_cache, "latent_cache": latent_cache, "latent_scale": latent_scale,
        "block_table": block_table, "row_req": row_req, "row_len": row_len,
        "q": q, "softmax_scale": float(wl.softmax_scale), "k": int(wl.k),
        "planted": planted_pos,
    }


NVFP4_ROW_BYTES = 352        # 256 code bytes + 32 block scales + 64 RoPE bytes
NVFP4_SCALE_BYTES = (0x38, 0x48)   # block scales drawn from E4M3 codes 1.0 .. 3.75
NVFP4_LATENT_SCALE = 0.15


def nvfp4_latent_cache(inp: Dict[str, object], wl: Workload,
                       scale_bytes=NVFP4_SCALE_BYTES, latent_scale: float = NVFP4_LATENT_SCALE):
    """An NVFP4 latent cache for ``inp``'s block table: uint8 [num_pages, 64, 352].

    Random bytes in the row layout of dsa_sparse_mla_decode_nvfp4: uniform
    E2M1 code bytes (every nibble equally likely), block-scale bytes uniform
    in [scale_bytes[0], scale_bytes[1]), and RoPE bytes that are the E4M3
    codes of N(0, 1) / latent_scale.  The default scale range spreads each
    block's magnitude over two binades, as the absmax / 6 scales of Gaussian
    blocks do; with the default latent_scale the values have a mean square
    of about 1, as the FP8 latent's have.  Slots outside every request's
    context hold 0x7F, whose scale byte decodes to NaN, so a stray read shows
    up.  Seeded by ``wl.seed``.  Returns (cache, latent_scale).
    """
    bt = inp["block_table"]
    dev = bt.device
    num_pages = inp["latent_cache"].shape[0]
    g = torch.Generator(device=dev)
    g.manual_seed(1_000_003 * int(wl.seed) + 12_345)
    cache = torch.empty((num_pages, PAGE, NVFP4_ROW_BYTES), dtype=torch.uint8, device=dev)
    cache[:, :, :256] = torch.randint(0, 256, (num_pages, PAGE, 256), generator=g, device=dev,
                                      dtype=torch.int32).to(torch.uint8)
    cache[:, :, 256:288] = torch.randint(int(scale_bytes[0]), int(scale_bytes[1]),
                                         (num_pages, PAGE, 32), generator=g, device=dev,
                                         dtype=torch.int32).to(torch.uint8)
    rope = torch.randn(num_pages, PAGE, 64, generator=g, device=dev, dtype=torch.float32)
    cache[:, :, 288:] = _e4m3_codes(rope / latent_scale)
    valid = torch.zeros((num_pages, PAGE), dtype=torch.bool, device=dev)
    for b, c in enumerate(wl.ctx):
        n = (c + PAGE - 1) // PAGE
        if n == 0:
            continue
        pages = bt[b, :n].to(torch.int64)
        valid[pages[:-1]] = True
        valid[pages[-1], :c - (n - 1) * PAGE] = True
    cache[~valid] = E4M3_NAN
    return cache, float(latent_scale)


def to_numpy(inp: Dict[str, object]) -> Dict[str, object]:
    """Host copies for the oracle: bf16 as uint16 bits, E4M3 as uint8 codes."""
    out = {}
    for key, v in inp.items():
        if isinstance(v, torch.Tensor):
            t = v.detach().cpu()
            if t.dtype == torch.bfloat16:
                out[key] = t.view(torch.int16).numpy().view(np.uint16)
            else:
                out[key] = t.numpy()
        elif isinstance(v, list):
            out[key] = [x.numpy() if isinstance(x, torch.Tensor) else x for x in v]
        else:
            out[key] = v
    return out
