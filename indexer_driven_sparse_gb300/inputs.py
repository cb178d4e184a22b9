"""Seeded synthetic inputs for the five workloads (shared by tests, bench and smoke).

This module draws random tensors and nothing else: it holds none of the
method's arithmetic (no pooling, scoring, selection or attention), so both the
CUDA path and the CPU oracle can consume what it makes.

Distributions (no page measures this path on a dataset; all inputs are synthetic):

* "gaussian": every bf16 tensor is N(0,1)/sqrt(dim), dim = head_dim (256) for
  Q/K/V and idx_dim (128) for the indexer query and raw indexer keys.
* "planted": Q/K/V as above, but the indexer tensors carry a rank-8 component
  so that block scores are spread rather than near-tied: U is an orthonormal
  128x8 basis; block b draws z_b ~ N(0, I8) and its tokens' raw keys are
  U z_b + eps/sqrt(128); a query draws a ~ N(0, I8) and q_idx = U a + eta/sqrt(128).
* "sharp": Q/K/V ~ N(0,1) (logit std about 1) instead of N(0,1)/sqrt(256).
* "planted_sharp": the planted indexer tensors with sharp Q/K/V (the prefill chunk's
  selection structure with outputs large enough to grade by relative error).
* Prefill queries can be temporally correlated: a_i = rho a_(i-1) + sqrt(1-rho^2) xi_i,
  which makes consecutive queries' selections overlap (rho is chosen so that
  the mean overlap of consecutive top-512 selections is about 0.72, the value
  measured on real text in "125B MoE を 3090 3 枚で運用する vLLM 最適化編", section 5).

Creation order for one layer with one generator: raw indexer keys, indexer
queries, queries, K, V (for "planted": U first, then the latents, then noise).
Small cases draw on the CPU generator (bit-stable across machines); large ones
draw on the device generator of the same seed so that tens of GiB are made in
milliseconds.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 256
IDX_DIM = 128
RATIO = 4
PLANTED_RANK = 8
# Consecutive-query correlation of the prefill indexer queries; tuned offline on
# the oracle so that consecutive top-512 selections share ~72% of their blocks.
PREFILL_RHO = 0.985


@dataclass
class Layer:
    raw_idx_k: torch.Tensor      # [T_total, IDX_DIM] bf16
    q_idx: torch.Tensor          # [Nq, IDX_DIM] bf16
    q: torch.Tensor              # [Nq, Hq, HEAD_DIM] bf16
    k_cache: torch.Tensor        # [T_total, Hkv, HEAD_DIM] bf16
    v_cache: torch.Tensor        # [T_total, Hkv, HEAD_DIM] bf16


@dataclass
class Workload:
    name: str
    n_q_heads: int
    n_kv_heads: int
    ctx_len: list                # decode: p per sequence; prefill: [p0]
    n_chunk: int = 0             # prefill: chunk queries (0 for decode)
    layers: list = field(default_factory=list)

    @property
    def batch(self) -> int:
        return len(self.ctx_len)

    @property
    def tok_off(self) -> list:
        """Flat ragged token layout: sequence s owns tokens [tok_off[s], tok_off[s+1])."""
        if self.n_chunk:
            return [0, self.ctx_len[0] + self.n_chunk]
        off = [0]
        for p in self.ctx_len:
            off.append(off[-1] + p + 1)      # history p tokens + the current token
        return off

    @property
    def n_tokens(self) -> int:
        return self.tok_off[-1]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, scale=1.0):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    return t


def _planted_basis(g, device):
    a = _randn((IDX_DIM, PLANTED_RANK), g, device).double()
    u, _ = torch.linalg.qr(a.cpu())
    return u.to(device=device, dtype=torch.float32)


def _layer(n_tok: int, n_q: int, hq: int, hkv: int, kind: str, g, device,
           block_of_token=None, rho: float = 0.0) -> Layer:
    s_idx = 1.0 / math.sqrt(IDX_DIM)
    s_head = 1.0 if kind in ("sharp", "planted_sharp") else 1.0 / math.sqrt(HEAD_DIM)
    if kind in ("planted", "planted_sharp"):
        u = _planted_basis(g, device)
        if block_of_token is None:
            block_of_token = torch.arange(n_tok, device=device) // RATIO
        n_blk = int(block_of_token.max().item()) + 1 if n_tok else 0
        z = _randn((n_blk, PLANTED_RANK), g, device)
        raw = z[block_of_token] @ u.T
        raw.add_(_randn((n_tok, IDX_DIM), g, device, s_idx))
        a = _randn((n_q, PLANTED_RANK), g, device)
        if rho > 0.0:
            c = math.sqrt(1.0 - rho * rho)
            for i in range(1, n_q):            # AR(1) chain of query latents
                a[i] = rho * a[i - 1] + c * a[i]
        q_idx = a @ u.T
        q_idx.add_(_randn((n_q, IDX_DIM), g, device, s_idx))
    else:
        raw = _randn((n_tok, IDX_DIM), g, device, s_idx)
        q_idx = _randn((n_q, IDX_DIM), g, device, s_idx)
    q = _randn((n_q, hq, HEAD_DIM), g, device, s_head)
    k = _randn((n_tok, hkv, HEAD_DIM), g, device, s_head)
    v = _randn((n_tok, hkv, HEAD_DIM), g, device, s_head)
    bf = torch.bfloat16
    return Layer(raw.to(bf), q_idx.to(bf), q.to(bf), k.to(bf), v.to(bf))


def decode_workload(name: str, ctx_len, n_layers: int, n_q_heads: int, n_kv_heads: int = 2,
                    kind: str = "gaussian", seed: int = 0, device="cpu") -> Workload:
    """Decode batch: one query per sequence at position p = ctx_len[s]; the
    sequence's cache holds p + 1 tokens (the current token's K/V is at index p)."""
    w = Workload(name, n_q_heads, n_kv_heads, [int(p) for p in ctx_len])
    g = _gen(seed, device)
    blocks = None
    if kind in ("planted", "planted_sharp"):
        # block index of every flat token, so that blocks never straddle sequences
        parts, base = [], 0
        for p in w.ctx_len:
            parts.append(torch.arange(p + 1, device=device) // RATIO + base)
            base += (p + 1 + RATIO - 1) // RATIO
        blocks = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.long, device=device)
    for _ in range(n_layers):
        w.layers.append(_layer(w.n_tokens, w.batch, n_q_heads, n_kv_heads, kind, g, device, blocks))
    return w


def prefill_workload(name: str, p0: int, n_chunk: int, n_q_heads: int = 16, n_kv_heads: int = 2,
                     kind: str = "planted", rho: float = PREFILL_RHO, seed: int = 0,
                     device="cpu") -> Workload:
    """Prefill chunk: n_chunk new queries at positions p0 .. p0+n_chunk-1 over a
    cache of p0 + n_chunk tokens (the chunk's own K/V already appended)."""
    w = Workload(name, n_q_heads, n_kv_heads, [int(p0)], n_chunk=int(n_chunk))
    g = _gen(seed, device)
    w.layers.append(_layer(w.n_tokens, n_chunk, n_q_heads, n_kv_heads, kind, g, device, rho=rho))
    return w


def batched_ctx_lens(batch: int = 32, lo: int = 4096, hi: int = 65536, seed: int = 0,
                     short_draw: bool = False) -> list:
    """Per-sequence contexts uniform on [lo, hi]. The short draw replaces 8 of
    them with lengths around the dense/sparse threshold and the degenerate ends."""
    g = _gen(seed, "cpu")
    lens = torch.randint(lo, hi + 1, (batch,), generator=g).tolist()
    if short_draw:
        for i, p in enumerate([0, 1, 3, 4, 2050, 2051, 2052, 2055]):
            lens[(i * 4 + 1) % batch] = p
    return lens


# ----------------------------------------------------------------------------- named workloads

def tiny_decode(seed=0, device="cpu", kind="gaussian"):
    """Batch 1 at context 4096 (1024 blocks -> 512), 1 layer, 8 query / 2 KV heads."""
    return decode_workload("tiny_decode_ctx4096", [4096], 1, 8, 2, kind, seed, device)


def long_decode(seed=0, device="cuda", n_layers=12, kind="planted"):
    """Batch 1 at context 131072, 12 layers, 16 query / 2 KV heads, planted indexer."""
    return decode_workload("long_decode_ctx131072", [131072], n_layers, 16, 2, kind, seed, device)


def batched_decode(seed=0, device="cuda", n_layers=12, short_draw=False, kind="gaussian"):
    """Batch 32, contexts uniform in [4096, 65536], 12 layers, 8 query / 2 KV heads."""
    lens = batched_ctx_lens(short_draw=short_draw, seed=seed)
    name = "batched_decode_b32" + ("_short" if short_draw else "")
    return decode_workload(name, lens, n_layers, 8, 2, kind, seed, device)


def million_decode(seed=0, device="cuda", n_layers=12, kind="planted"):
    """Batch 1 at context 1,048,320 (262,080 blocks), 12 layers, 16 query / 2 KV heads."""
    return decode_workload("million_decode_ctx1048320", [1048320], n_layers, 16, 2, kind, seed, device)


def prefill_chunk(seed=0, device="cuda", kind="planted", rho=PREFILL_RHO, p0=262144, n_chunk=4096):
    """4096 chunk queries over a 262,144-token history, 16 query / 2 KV heads."""
    return prefill_workload(f"prefill_chunk_p{p0}_n{n_chunk}", p0, n_chunk, 16, 2, kind, rho, seed, device)


# ----------------------------------------------------------------------------- sparse MLA (FP8 rows)

MLA_ROW_BYTES = 656        # 512 E4M3 latent codes, 4 fp32 group scales, 64 bf16 rotary dims
MLA_QK_DIM = 576


@dataclass
class MlaWorkload:
    kv: torch.Tensor           # [n_tokens, 656] uint8 rows
    q: torch.Tensor            # [B, H, 576] bf16
    rows: torch.Tensor         # [B, max_rows] int32 selected token ids (ascending, -1 padded)
    n_rows: torch.Tensor       # [B] int32


def mla_workload(n_tokens: int, n_rows, n_heads: int = 64, seed: int = 0, device="cpu") -> MlaWorkload:
    """A synthetic FP8 sparse-MLA cache and a batch of decode queries, each with its own
    selected rows. Row bytes: random E4M3 codes (sign and a magnitude byte drawn from
    0x08..0x77, normal values 2^-6 .. 240), four fp32 scales 2^-9 * U(0.5, 1) and 64 bf16
    rotary values N(0,1)/8. Queries are bf16 16 N(0,1) (logits of std about 1 under the
    1/sqrt(576) scale, so the softmax is far from uniform). Each query's rows are a uniform random
    subset of the tokens, ascending. Creation order: codes, scales, rope, queries, subsets."""
    g = _gen(seed, device)
    n_rows = [int(n) for n in n_rows]
    B, mr = len(n_rows), max(max(n_rows, default=1), 1)
    sign = torch.randint(0, 2, (n_tokens, 512), generator=g, device=device, dtype=torch.int32)
    mag = torch.randint(0x08, 0x78, (n_tokens, 512), generator=g, device=device, dtype=torch.int32)
    codes = (sign * 128 + mag).to(torch.uint8)
    scales = torch.rand((n_tokens, 4), generator=g, device=device, dtype=torch.float32).mul_(0.5).add_(0.5)
    scales.mul_(2.0 ** -9)
    rope = _randn((n_tokens, 64), g, device, 1.0 / 8.0).to(torch.bfloat16)
    kv = torch.cat([codes, scales.view(torch.uint8), rope.view(torch.uint8)], dim=1).contiguous()
    q = _randn((B, n_heads, MLA_QK_DIM), g, device, 16.0).to(torch.bfloat16)
    rows = torch.full((B, mr), -1, dtype=torch.int32, device=device)
    for b, n in enumerate(n_rows):
        if n:
            sel = torch.randperm(n_tokens, generator=g, device=device)[:n].sort().values
            rows[b, :n] = sel.to(torch.int32)
    return MlaWorkload(kv, q, rows, torch.tensor(n_rows, dtype=torch.int32, device=device))
