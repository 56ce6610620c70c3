"""Algorithmic bytes and FLOPs of one DSA decode step (the roofline numerators).

The byte model is the pages' own argument for DSA (vLLM Day-0 post, "Sparse
attention cuts long-context decode bandwidth"; TokenSpeed post, "Sparse
attention in Kimi K3.1 Pro"): the indexer scan reads one 132-byte FP8 key per
context token (128 E4M3 values + one fp32 scale), then attention reads the
576-byte FP8 latent row of only the k selected tokens, against 576 bytes per
context token for dense MLA.
"""
from __future__ import annotations

from .inputs import IDX_DIM, IDX_HEADS, LAT_DIM, V_DIM, Workload

KEY_BYTES = IDX_DIM + 4          # 132 B per token per layer
MXFP4_KEY_BYTES = IDX_DIM // 2 + IDX_DIM // 32   # 68 B: E2M1 codes + one E8M0 scale per 32 dims
LATENT_BYTES = LAT_DIM           # 576 B per token per layer (FP8)
NVFP4_LATENT_BYTES = 352         # the same row in NVFP4 + E4M3 RoPE


def dense_mla_bytes_per_token() -> int:
    """Latent bytes dense MLA reads per context token per layer."""
    return LATENT_BYTES


def dsa_bytes(ctx: int, k: int = 2048) -> int:
    """Index-key scan over ``ctx`` tokens plus ``min(k, ctx)`` latent rows (one row)."""
    return ctx * KEY_BYTES + min(k, ctx) * LATENT_BYTES


def scan_bytes(wl: Workload) -> int:
    """Index keys of every request's context (read once for all its rows)."""
    return int(sum(wl.ctx) * KEY_BYTES)


def scan_bytes_mxfp4(wl: Workload) -> int:
    """MXFP4 index keys of every request's context, the MXFP4 query (codes and
    scales) and the head weights."""
    return int(sum(wl.ctx) * MXFP4_KEY_BYTES + wl.R * IDX_HEADS * (MXFP4_KEY_BYTES + 4))


def gather_bytes(wl: Workload) -> int:
    """Latent rows gathered for every row (no credit for rows shared by rows)."""
    return int(sum(min(wl.k, n) for n in wl.row_lengths()) * LATENT_BYTES)


def gather_bytes_nvfp4(wl: Workload) -> int:
    """352 B NVFP4 latent row per selected token (256 B codes, 32 B scales, 64 B RoPE)."""
    return int(sum(min(wl.k, n) for n in wl.row_lengths()) * NVFP4_LATENT_BYTES)


def query_output_bytes(wl: Workload) -> int:
    qi = wl.R * IDX_HEADS * (IDX_DIM * (1 if wl.q_idx_fp8 else 2) + (4 if wl.q_idx_fp8 else 0))
    w = wl.R * IDX_HEADS * 4
    q = wl.R * wl.H * LAT_DIM * 2
    out = wl.R * wl.H * V_DIM * 2
    return int(qi + w + q + out)


def algorithmic_bytes(wl: Workload) -> int:
    """Minimum bytes one step moves: keys + gathered latents + queries + output.

    Score buffers, candidate lists, block tables and split partials are
    overhead and earn no credit.
    """
    return scan_bytes(wl) + gather_bytes(wl) + query_output_bytes(wl)


def algorithmic_bytes_fp4(wl: Workload) -> int:
    """The same for the step over MXFP4 index keys and NVFP4 latent rows."""
    return scan_bytes_mxfp4(wl) + gather_bytes_nvfp4(wl) + wl.R * wl.H * (LAT_DIM + V_DIM) * 2


def scan_flops(wl: Workload) -> int:
    """2 * 32 heads * 128 dims per (row, visible token)."""
    return int(2 * IDX_HEADS * IDX_DIM * sum(wl.row_lengths()))


def mla_flops(wl: Workload) -> int:
    """2 * H * (576 + 512) per (row, selected token)."""
    return int(2 * wl.H * (LAT_DIM + V_DIM) * sum(min(wl.k, n) for n in wl.row_lengths()))
