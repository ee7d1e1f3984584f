"""Seeded synthetic inputs for the QSA decode / MTP-verify step.

This module only draws random numbers and stores them in the formats the step
consumes (BF16, FP8-E4M3 with a per-head FP32 scale, int32 positions and page
tables). It holds none of the method's arithmetic: no compressed keys, scores,
selection or attention. Both the CPU oracle's tests and the CUDA path's tests
and benchmark draw their inputs from here, so the two sides see identical
bytes.

Random numbers come from a counter-based SplitMix64 (Steele, Lea, Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014): output ``i`` of
stream ``seed`` is ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)``. Normals use
the Box-Muller transform on pairs of 24-bit uniforms, in float32, then
round-to-nearest-even to BF16. Generation is chunked and indexed by element,
so results do not depend on the chunk size or on the number of threads.

Workloads follow the pages' decode / MTP-verify setting (arex-research.com,
"SWE-Smith 与 AgentX" and "四类优化"): a first turn of 50,000 tokens that grows
by 800 tokens per turn over 10-15 turns, 4 verify queries per request, 16 query
heads over 2 KV heads of dim 128, and a paged KV cache of 64-token pages.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

_MASK64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB

SEED_BASE = 20261202

# tensor ids that offset the seed of each drawn tensor
T_QIDX, T_IDXKEYS, T_Q, T_K, T_V, T_PAGES, T_CTX = 1, 2, 3, 4, 5, 6, 7

HEAD_DIM = 128
N_Q_HEADS = 16
N_KV_HEADS = 2
PAGE_SIZE = 64
BLOCK = 4
E4M3_MAX = 448.0


def _s64(c: int) -> int:
    c &= _MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def _srl(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 lanes holding uint64 bit patterns."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def splitmix64(counter: torch.Tensor, seed: int) -> torch.Tensor:
    """Output number ``counter`` of the SplitMix64 stream started at ``seed``.

    ``counter`` is int64; the result is int64 holding the uint64 bit pattern.
    """
    z = counter * _s64(_GAMMA) + _s64(seed + _GAMMA)
    z = (z ^ _srl(z, 30)) * _s64(_MIX1)
    z = (z ^ _srl(z, 27)) * _s64(_MIX2)
    return z ^ _srl(z, 31)


def splitmix64_py(i: int, seed: int) -> int:
    """Scalar pure-Python SplitMix64, used to pin the tensor version."""
    z = (seed + (i + 1) * _GAMMA) & _MASK64
    z = ((z ^ (z >> 30)) * _MIX1) & _MASK64
    z = ((z ^ (z >> 27)) * _MIX2) & _MASK64
    return z ^ (z >> 31)


def _uniform24(counter: torch.Tensor, seed: int) -> torch.Tensor:
    """Uniform float32 in (0, 1) from the top 24 bits of SplitMix64."""
    bits = _srl(splitmix64(counter, seed), 40)
    return (bits.to(torch.float32) + 0.5) * (1.0 / 16777216.0)


_CHUNK = 1 << 24


def normal_f32(n: int, seed: int, device="cpu") -> torch.Tensor:
    """``n`` standard normals (float32) by Box-Muller on counter pairs."""
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = _normal_range(s, e, seed, device)
    return out


def normal_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    n = 1
    for d in shape:
        n *= d
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        # draw the chunk with its global counters so chunking never changes values
        out[s:e] = _normal_range(s, e, seed, device).to(torch.bfloat16)
    return out.view(*shape)


def _normal_range(s: int, e: int, seed: int, device) -> torch.Tensor:
    idx = torch.arange(s, e, dtype=torch.int64, device=device)
    pair = idx >> 1
    u1 = _uniform24(2 * pair, seed)
    u2 = _uniform24(2 * pair + 1, seed)
    r = torch.sqrt(-2.0 * torch.log(u1))
    ang = (2.0 * math.pi) * u2
    return torch.where((idx & 1) == 0, r * torch.cos(ang), r * torch.sin(ang))


def uint_below(n: int, bound: int, seed: int) -> List[int]:
    """``n`` integers drawn uniformly from 0..bound-1 (host, exact)."""
    return [splitmix64_py(i, seed) % bound for i in range(n)]


def permutation(n: int, seed: int) -> torch.Tensor:
    """A seeded random permutation of 0..n-1 (argsort of SplitMix64 keys)."""
    keys = splitmix64(torch.arange(n, dtype=torch.int64), seed)
    return torch.argsort(keys, stable=True).to(torch.int32)


def quantize_e4m3(x: torch.Tensor, per_head_dim: int):
    """Per-KV-head FP8-E4M3 storage of ``x`` with one FP32 scale per head.

    ``x`` has the KV-head index on dimension ``per_head_dim``. The scale is
    amax/448 over that head; codes are round-to-nearest-even of x/scale,
    clamped to +-448 (no NaN can be produced). Returns (codes uint8, scales
    float32 [H_kv]).
    """
    xf = x.to(torch.float32)
    dims = [d for d in range(xf.dim()) if d != per_head_dim]
    amax = xf.abs().amax(dim=dims)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    shape = [1] * xf.dim()
    shape[per_head_dim] = -1
    y = (xf / scale.view(shape)).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.to(torch.float32)


@dataclasses.dataclass
class Spec:
    """Shape of one synthetic QSA step.

    ``first_pos[r]`` is the position of request r's first query token; its
    ``n_q`` verify queries sit at ``first_pos[r] .. first_pos[r] + n_q - 1``
    and their own K/V are already in the cache, so the request holds
    ``first_pos[r] + n_q`` tokens.
    """

    name: str
    batch: int
    n_q: int
    first_pos: List[int]
    n_idx_heads: int = 1
    kv_dtype: str = "bf16"  # "bf16" or "fp8"
    paged: bool = True  # False: identity page table (contiguous KV)
    seed: int = SEED_BASE
    n_q_heads: int = N_Q_HEADS
    n_kv_heads: int = N_KV_HEADS
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE

    def q_pos(self) -> List[List[int]]:
        return [[p + j for j in range(self.n_q)] for p in self.first_pos]

    def tokens(self) -> List[int]:
        return [p + self.n_q for p in self.first_pos]

    def max_blocks(self) -> int:
        # blocks whose 4 tokens all exist in the cache
        return max(1, max(t // BLOCK for t in self.tokens()))

    def pages_per_request(self) -> List[int]:
        return [(t + self.page_size - 1) // self.page_size for t in self.tokens()]

    def max_pages(self) -> int:
        return max(self.pages_per_request())

    def num_pages(self) -> int:
        return sum(self.pages_per_request())


def turn_growth_positions(batch: int, seed: int, first: int = 50000, per_turn: int = 800,
                          turns: int = 15) -> List[int]:
    """Context lengths first + per_turn * t, t uniform in 0..turns-1."""
    return [first + per_turn * t for t in uint_below(batch, turns, seed)]


def spec_for(config: int, batch: Optional[int] = None, ctx: Optional[int] = None, replica: int = 0) -> Spec:
    """The five workloads of the decode / verify step, by number.

    0: batch 1, one query at position 4,098 (1,024 full blocks + a 3-token
       partial block), 1 index head, contiguous BF16 KV.
    1: batch 1, 4 verify queries at 50,000..50,003, paged BF16 KV.
    2: batch 32, 4 verify queries, contexts 50,000 + 800*t (t uniform 0..14),
       paged BF16 KV.
    3: as 2 with FP8-E4M3 KV, one FP32 scale per KV head.
    4: batch ``batch`` x context ``ctx`` in {131,072, 262,144}, 4 verify
       queries, 4 index heads, FP8-E4M3 paged KV.
    """
    # replica r of a multi-GPU run draws its own requests (its shard of the
    # global batch) from the same distribution
    seed = SEED_BASE + 1000 * config + 100_000 * replica
    if config == 0:
        return Spec("tiny-decode-b1-ctx4099", 1, 1, [4098], 1, "bf16", False, seed)
    if config == 1:
        return Spec("verify-b1-ctx50k", 1, 4, [50000], 1, "bf16", True, seed)
    if config in (2, 3):
        b = 32 if batch is None else batch
        pos = turn_growth_positions(b, seed + T_CTX)
        kv = "bf16" if config == 2 else "fp8"
        return Spec(f"verify-b{b}-ctx50k-turns-{kv}", b, 4, pos, 1, kv, True, seed)
    if config == 4:
        b = 1 if batch is None else batch
        L = 131072 if ctx is None else ctx
        return Spec(f"longctx-b{b}-ctx{L}-idx4-fp8", b, 4, [L] * b, 4, "fp8", True, seed + b * 7 + L)
    raise ValueError(f"unknown config {config}")


def make_inputs(spec: Spec, device="cpu", with_index_keys: bool = True) -> Dict[str, torch.Tensor]:
    """Draw every input tensor of ``spec`` on ``device``.

    Returns a dict with
      q_idx     bf16  [B][n_q][H_idx][128]   index queries
      idx_keys  bf16  [B][4*max_blocks][H_idx][128]  per-token index keys
                (only tokens of full blocks matter; the compressed key of a
                block is derived from these by the method, not here)
      q         bf16  [B][n_q][H_q][128]     attention queries
      k_cache, v_cache  bf16 or uint8 (E4M3 codes) [num_pages][H_kv][P][128]
      k_scale, v_scale  float32 [H_kv] (ones for BF16)
      page_table int32 [B][max_pages] (-1 beyond a request's pages)
      q_pos      int32 [B][n_q]
    """
    s = spec.seed
    B, nq, H, D = spec.batch, spec.n_q, spec.n_idx_heads, spec.head_dim
    out: Dict[str, torch.Tensor] = {}
    out["q_idx"] = normal_bf16((B, nq, H, D), s + T_QIDX, device)
    if with_index_keys:
        out["idx_keys"] = normal_bf16((B, BLOCK * spec.max_blocks(), H, D), s + T_IDXKEYS, device)
    out["q"] = normal_bf16((B, nq, spec.n_q_heads, D), s + T_Q, device)
    shape = (spec.num_pages(), spec.n_kv_heads, spec.page_size, D)
    k = normal_bf16(shape, s + T_K, device)
    v = normal_bf16(shape, s + T_V, device)
    if spec.kv_dtype == "fp8":
        out["k_cache"], out["k_scale"] = quantize_e4m3(k, 1)
        del k
        out["v_cache"], out["v_scale"] = quantize_e4m3(v, 1)
        del v
    elif spec.kv_dtype == "bf16":
        out["k_cache"], out["v_cache"] = k, v
        out["k_scale"] = torch.ones(spec.n_kv_heads, dtype=torch.float32, device=device)
        out["v_scale"] = torch.ones(spec.n_kv_heads, dtype=torch.float32, device=device)
    else:
        raise ValueError(spec.kv_dtype)
    n_pages = spec.num_pages()
    perm = permutation(n_pages, s + T_PAGES) if spec.paged else torch.arange(n_pages, dtype=torch.int32)
    pt = torch.full((B, spec.max_pages()), -1, dtype=torch.int32)
    off = 0
    for r, npg in enumerate(spec.pages_per_request()):
        pt[r, :npg] = perm[off:off + npg]
        off += npg
    out["page_table"] = pt.to(device)
    out["q_pos"] = torch.tensor(spec.q_pos(), dtype=torch.int32, device=device)
    return out
