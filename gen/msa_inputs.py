"""Seeded synthetic inputs for MSA block-sparse GQA attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no scores, no pooling, no selection, no softmax).  The same
bf16 bits it returns are handed both to the CUDA library and to the CPU oracle.

Workloads (sizes and head layout from the method's deployment setting: GQA with
4 KV groups of 128 dims, one index query head per group and one shared index key,
64-token blocks, k = 16 blocks per query):

  tiny     N=1024,  H_q=8,  H_kv=2, d_h=64,  d_idx=32, k=4
  p32k     N=32768, H_q=32, H_kv=4, d_h=128, d_idx=64, k=16, per-block K offsets
  p128k    N=131072, same heads, per-block K offsets + 8 hot blocks
  decode   32 sequences, cache lengths ~ U[65536, 262144], same heads
  p1m      N=1048576, as p32k

Random draws use torch generators (CPU or CUDA, seeded); float32 normals are
rounded to bf16 with torch's round-to-nearest-even conversion.  Tensors come back
as torch.bfloat16 on the requested device; ``to_bits`` gives the uint16 view the
oracle takes.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

__all__ = [
    "PrefillConfig", "DecodeConfig", "CONFIGS", "prefill_inputs", "decode_inputs", "to_pages",
    "to_bits", "from_bits", "bf16_bits_to_f64", "nblocks", "ceil_div", "BLOCK",
]

BLOCK = 64


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    N: int
    H_q: int
    H_kv: int
    d_h: int
    d_idx: int
    k: int
    block_size: int = BLOCK
    block_offset_std: float = 0.0   # std of the per-(group, block) K offset vector
    hot_blocks: int = 0             # number of hot blocks drawn from the first 64 blocks


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    S: int
    len_lo: int
    len_hi: int          # inclusive
    H_q: int
    H_kv: int
    d_h: int
    d_idx: int
    k: int
    block_size: int = BLOCK


CONFIGS = {
    "tiny": PrefillConfig("tiny", 1024, 8, 2, 64, 32, 4),
    "p32k": PrefillConfig("p32k", 32768, 32, 4, 128, 64, 16, block_offset_std=0.5),
    "p128k": PrefillConfig("p128k", 131072, 32, 4, 128, 64, 16, block_offset_std=0.5,
                           hot_blocks=8),
    "decode": DecodeConfig("decode", 32, 65536, 262144, 32, 4, 128, 64, 16),
    "p1m": PrefillConfig("p1m", 1 << 20, 32, 4, 128, 64, 16, block_offset_std=0.5),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, device):
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def _ints(g, shape, device, lo=-3, hi=3):
    return torch.randint(lo, hi + 1, shape, generator=g, device=device).to(torch.float32)


def prefill_inputs(cfg: PrefillConfig, seed: int = 0, device="cpu", variant="gauss",
                   N: int | None = None):
    """Draw Q [N,H_q,d_h], K,V [N,H_kv,d_h], Q_idx [N,H_kv,d_idx], K_idx [N,d_idx] (bf16).

    variant "gauss": i.i.d. N(0,1) plus the config's structure (block offsets on K,
    hot blocks).  variant "int": i.i.d. integers uniform in [-3, 3] (every product
    and sum then stays exact in fp32).  variant "zero_q": as gauss but Q = 0.
    variant "const_kidx": as gauss but every K_idx row is the same vector.
    ``N`` overrides the config's length (same head layout).
    """
    n = cfg.N if N is None else int(N)
    g = _gen(device, seed)
    draw = _ints if variant == "int" else _normal
    q = draw(g, (n, cfg.H_q, cfg.d_h), device)
    k = draw(g, (n, cfg.H_kv, cfg.d_h), device)
    v = draw(g, (n, cfg.H_kv, cfg.d_h), device)
    q_idx = draw(g, (n, cfg.H_kv, cfg.d_idx), device)
    k_idx = draw(g, (n, cfg.d_idx), device)
    meta = {"N": n, "seed": seed, "variant": variant}
    if variant != "int":
        nblk = (n + cfg.block_size - 1) // cfg.block_size
        if cfg.block_offset_std > 0:
            # one offset vector per (KV group, block), shared by the block's tokens
            off = _normal(g, (cfg.H_kv, nblk, cfg.d_h), device) * cfg.block_offset_std
            tok_blk = torch.arange(n, device=device) // cfg.block_size
            k += off[:, tok_blk, :].permute(1, 0, 2)
        if cfg.hot_blocks > 0:
            pool = min(64, nblk)
            perm = torch.randperm(pool, generator=g, device=device)
            hot = torch.sort(perm[: min(cfg.hot_blocks, pool)]).values
            u = _normal(g, (cfg.d_idx,), device)
            u = u / u.norm()
            u2 = _normal(g, (cfg.d_h,), device)
            u2 = u2 / u2.norm()
            hot_tok = (hot[:, None] * cfg.block_size
                       + torch.arange(cfg.block_size, device=device)[None, :]).reshape(-1)
            hot_tok = hot_tok[hot_tok < n]
            q_idx += 2.0 * u
            k_idx[hot_tok] += 12.0 * u
            q += 2.0 * u2
            k[hot_tok] += 12.0 * u2
            meta["hot_blocks"] = hot.tolist()
        if variant == "zero_q":
            q.zero_()
        if variant == "const_kidx":
            k_idx[:] = k_idx[0:1].clone()
    bf = torch.bfloat16
    return dict(q=q.to(bf), k=k.to(bf), v=v.to(bf), q_idx=q_idx.to(bf), k_idx=k_idx.to(bf),
                meta=meta)


def decode_inputs(cfg: DecodeConfig, seed: int = 0, device="cpu", S: int | None = None,
                  len_lo: int | None = None, len_hi: int | None = None, variant="gauss"):
    """Draw a packed varlen cache and one new query per sequence.

    Returns q [S,H_q,d_h], q_idx [S,H_kv,d_idx], k_cache/v_cache [sum L,H_kv,d_h],
    k_idx_cache [sum L,d_idx] (bf16) and cu_seqlens [S+1] (int64, on ``device``).
    The newest token of sequence s is cache row cu_seqlens[s+1]-1.
    """
    s = cfg.S if S is None else int(S)
    lo = cfg.len_lo if len_lo is None else int(len_lo)
    hi = cfg.len_hi if len_hi is None else int(len_hi)
    g = _gen("cpu", seed)
    lens = torch.randint(lo, hi + 1, (s,), generator=g)
    cu = torch.zeros(s + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    total = int(cu[-1])
    gd = _gen(device, seed + 7919)
    draw = _ints if variant == "int" else _normal
    q = draw(gd, (s, cfg.H_q, cfg.d_h), device)
    q_idx = draw(gd, (s, cfg.H_kv, cfg.d_idx), device)
    k = draw(gd, (total, cfg.H_kv, cfg.d_h), device)
    v = draw(gd, (total, cfg.H_kv, cfg.d_h), device)
    k_idx = draw(gd, (total, cfg.d_idx), device)
    bf = torch.bfloat16
    return dict(q=q.to(bf), q_idx=q_idx.to(bf), k_cache=k.to(bf), v_cache=v.to(bf),
                k_idx_cache=k_idx.to(bf), cu_seqlens=cu.to(device),
                meta={"S": s, "lens": lens.tolist(), "seed": seed, "variant": variant})


def to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> contiguous numpy uint16 array of its bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> torch.bfloat16 tensor (CPU)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def nblocks(n: int, block: int = BLOCK) -> int:
    return (n + block - 1) // block


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def to_pages(d, seed, extra=3):
    """Scatter a packed decode cache (rows cu_seqlens[s] .. cu_seqlens[s+1]-1 per sequence) into
    64-token pages in a random order: `extra` unused pages, noise in the rows of a last page
    past the sequence's end, and page-table entries past a sequence's last block set to an id
    far out of range (they must never be read).  Layout only, no arithmetic of the method.
    Returns (k_pages, v_pages, k_idx_pages, page_table [S, max_pages] int32, seq_lens int64)."""
    cu = d["cu_seqlens"].cpu().numpy()
    lens = cu[1:] - cu[:-1]
    nb = (lens + 63) // 64
    npages = int(nb.sum()) + extra
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    perm = torch.randperm(npages, generator=g, device="cuda").cpu().numpy()
    kc, vc, kic = d["k_cache"], d["v_cache"], d["k_idx_cache"]
    kp = torch.randn((npages * 64,) + tuple(kc.shape[1:]), generator=g, device="cuda").to(kc.dtype)
    vp = torch.randn((npages * 64,) + tuple(vc.shape[1:]), generator=g, device="cuda").to(vc.dtype)
    kip = torch.randn((npages * 64,) + tuple(kic.shape[1:]), generator=g, device="cuda").to(kic.dtype)
    S, max_pages = len(lens), int(nb.max())
    pt = np.full((S, max_pages), 1 << 30, np.int32)
    dst, src, nxt = [], [], 0
    for s in range(S):
        for b in range(int(nb[s])):
            pg = int(perm[nxt])
            nxt += 1
            pt[s, b] = pg
            n = min(64, int(lens[s]) - 64 * b)
            dst.append(pg * 64 + np.arange(n))
            src.append(int(cu[s]) + 64 * b + np.arange(n))
    dst = torch.from_numpy(np.concatenate(dst)).cuda()
    src = torch.from_numpy(np.concatenate(src)).cuda()
    kp[dst], vp[dst], kip[dst] = kc[src], vc[src], kic[src]
    shape = lambda t: t.view((npages, 64) + tuple(t.shape[1:]))
    return (shape(kp), shape(vp), shape(kip), torch.from_numpy(pt).cuda(),
            torch.from_numpy(lens.astype(np.int64)).cuda())
