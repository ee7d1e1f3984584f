"""Helpers shared by the tests: tensor <-> numpy bit views, small specs."""

import numpy as np
import torch

from block_sparse_attention_qsa_gb300 import synth


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw storage of a tensor as numpy: BF16 -> uint16 bits, uint8 as is."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_numpy_inputs(inp: dict) -> dict:
    return {k: bits(v) for k, v in inp.items()}


def unpage(cache: np.ndarray, page_table_row: np.ndarray, n_tokens: int) -> np.ndarray:
    """Contiguous per-token view [T][H_kv][D] of one request's paged cache,
    assembled page by page (independent of any per-position lookup)."""
    P = cache.shape[2]
    parts = []
    for page in page_table_row:
        if page < 0:
            break
        parts.append(np.transpose(cache[int(page)], (1, 0, 2)))  # [P][H_kv][D]
    full = np.concatenate(parts, axis=0)
    return full[:n_tokens]


def small_spec(first_pos, n_q=4, n_idx_heads=1, kv_dtype="bf16", paged=True, seed=777, batch=None):
    fp = list(first_pos)
    return synth.Spec(f"small-{fp[0]}", len(fp) if batch is None else batch, n_q, fp, n_idx_heads,
                      kv_dtype, paged, seed)
