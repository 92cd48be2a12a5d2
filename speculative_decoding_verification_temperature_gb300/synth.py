"""Seeded synthetic inputs for the verify step (tests, smoke check, bench).

This module only makes inputs: Gaussian logits shaped like the workloads of
the pages (vocabularies of LLaMA-2 32000, LLaMA-3 128256 and Qwen 151936 /
152064 tokens), draft tokens drawn from the draft distribution, token trees,
and the uniform numbers the verify step consumes.  It holds none of the
verify arithmetic (no acceptance ratio, residual or inverse CDF); draft
tokens are drawn with the Gumbel-max trick, which is not what the verify
step computes.

Uniforms come from splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the 64-bit finaliser constants
as published with the public-domain reference implementation): the e-th
output of the stream seeded with ``seed`` is mixed from
``seed + (e+1) * 0x9E3779B97F4A7C15``, and uniform ``e`` is
``((s_e >> 41) + 0.5) * 2**-23``, a number in (0, 1) that is exact in fp32,
so every consumer sees bit-identical uniforms.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+n-1 of the splitmix64 stream for ``seed``."""
    with np.errstate(over="ignore"):
        e = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + e * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniforms(seed: int, shape, offset: int = 0) -> np.ndarray:
    """float32 uniforms in (0, 1), row-major over ``shape``."""
    n = int(np.prod(shape))
    s = splitmix64(seed, n, offset)
    u = ((s >> np.uint64(41)).astype(np.float64) + 0.5) * 2.0 ** -23
    return u.astype(np.float32).reshape(shape)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) of a bf16 tensor, on the host."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(
        np.uint16)


def host_logits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a logits tensor in the form the oracle takes: float32
    values, or raw uint16 bits for bf16."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    assert t.dtype == torch.float32
    return t.detach().cpu().contiguous().numpy()


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, sigma=1.0):
    return torch.randn(shape, generator=g, device=device,
                       dtype=torch.float32) * float(sigma)


def gumbel_argmax(logits: torch.Tensor, T: float, g: torch.Generator,
                  draws: int = 1, chunk: int = 1 << 26) -> torch.Tensor:
    """Draw ``draws`` tokens per row of ``logits`` [..., V] from
    softmax(logits / T) by the Gumbel-max trick (argmax of logits/T plus
    Gumbel noise, in float64); T == 0 gives the row argmax (lowest index on
    ties).  Returns int32 [..., draws]."""
    lead = logits.shape[:-1]
    V = logits.shape[-1]
    flat = logits.reshape(-1, V)
    rows = flat.shape[0]
    out = torch.empty((rows, draws), dtype=torch.int32, device=logits.device)
    if T == 0:
        # torch.argmax returns the first maximal index
        out[:] = torch.argmax(flat.float(), dim=1, keepdim=True).to(
            torch.int32)
        return out.reshape(*lead, draws)
    step = max(1, chunk // max(1, V * draws))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        z = flat[r0:r1].to(torch.float64).unsqueeze(1) / float(T)
        u = torch.rand((r1 - r0, draws, V), generator=g,
                       device=logits.device, dtype=torch.float64)
        u.clamp_(min=1e-300)
        gmb = -torch.log(-torch.log(u))
        out[r0:r1] = torch.argmax(z + gmb, dim=2).to(torch.int32)
    return out.reshape(*lead, draws)


def _cast(t: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    return t.to(dtype).contiguous()


# --------------------------------------------------------------------------
# linear verify inputs
# --------------------------------------------------------------------------
@dataclass
class LinearCase:
    target: torch.Tensor          # [B, gamma+1, V]
    draft: torch.Tensor           # [B, gamma (or K+1 for fan-out), V]
    tokens: torch.Tensor          # [B, gamma] int32
    uniforms: torch.Tensor        # [B, gamma+1] float32
    T: float
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, G1, V = self.target.shape
        return B, G1 - 1, V


def linear_case(B, gamma, V, dtype=torch.float32, T=1.0, seed=0,
                sigma_t=3.0, sigma_d=1.0, spike=0.0, draft_rows=None,
                device="cpu") -> LinearCase:
    """Target ~ N(0, sigma_t^2) (+ ``spike`` at one uniformly chosen token
    per target row), draft = target + N(0, sigma_d^2) at the same
    positions; ``draft_rows`` (default gamma) lets the draft carry extra
    lookahead rows for fan-out.  Draft tokens are drawn from
    softmax(draft / T) of the rounded logits (argmax at T == 0)."""
    g = _gen(seed, device)
    dr = gamma if draft_rows is None else draft_rows
    rows = max(gamma + 1, dr)
    base = _randn((B, rows, V), g, device, sigma_t)
    if spike:
        idx = torch.randint(0, V, (B, rows, 1), generator=g, device=device)
        base.scatter_add_(2, idx, torch.full((B, rows, 1), float(spike),
                                             device=device))
    target = _cast(base[:, :gamma + 1], dtype)
    draft = _cast(base[:, :dr] + _randn((B, dr, V), g, device, sigma_d),
                  dtype)
    tok = gumbel_argmax(draft[:, :gamma].float(), T, g)[..., 0]
    u = torch.from_numpy(uniforms(seed * 7919 + 17, (B, gamma + 1))).to(
        device)
    return LinearCase(target, draft, tok.contiguous(), u, float(T),
                      dict(seed=seed))


# --------------------------------------------------------------------------
# K-candidate (diffusion self-selection) inputs
# --------------------------------------------------------------------------
@dataclass
class KcandCase:
    target: torch.Tensor          # [B, K, gamma+1, V]
    draft: torch.Tensor           # [B, gamma, V] shared marginals
    tokens: torch.Tensor          # [B, K, gamma]
    uniforms: torch.Tensor        # [B, K, gamma+1]
    T: float


def kcand_case(B, K, gamma, V, dtype=torch.bfloat16, T=1.0, seed=0,
               sigma_t=3.0, sigma_d=1.0, sigma_k=0.5,
               device="cpu") -> KcandCase:
    """Base rows ~ N(0, sigma_t^2) per (b, j); the shared draft marginal of
    position j is base + N(0, sigma_d^2); candidate k's target row at
    position 0 is the base row (same prefix for all k), at j >= 1 it is
    base + N(0, sigma_k^2) of its own.  The K drafts are iid joint samples
    from the marginals."""
    g = _gen(seed, device)
    base = _randn((B, gamma + 1, V), g, device, sigma_t)
    draft32 = base[:, :gamma] + _randn((B, gamma, V), g, device, sigma_d)
    draft = _cast(draft32, dtype)
    target = torch.empty((B, K, gamma + 1, V), dtype=dtype, device=device)
    for k in range(K):
        tk = base.clone()
        tk[:, 1:] += _randn((B, gamma, V), g, device, sigma_k)
        target[:, k] = tk.to(dtype)
    tok = gumbel_argmax(draft.float(), T, g, draws=K)  # [B, gamma, K]
    tok = tok.permute(0, 2, 1).contiguous()
    u = torch.from_numpy(uniforms(seed * 7919 + 29, (B, K, gamma + 1))).to(
        device)
    return KcandCase(target, draft, tok, u, float(T))


# --------------------------------------------------------------------------
# token-tree inputs
# --------------------------------------------------------------------------
@dataclass
class TreeCase:
    target: torch.Tensor          # [B, N, V]
    draft: torch.Tensor           # [B, N, V]
    parent: torch.Tensor          # [B, N] int32, parent[0] = -1
    node_tokens: torch.Tensor     # [B, N] int32 (slot 0 unused: -1)
    uniforms: torch.Tensor        # [B, N] float32
    T: float


def tree_case(B, N, V, dtype=torch.bfloat16, T=0.8, seed=0, sigma_t=3.0,
              sigma_d=1.0, max_depth=8, branch=4,
              device="cpu") -> TreeCase:
    """Node rows: target ~ N(0, sigma_t^2), draft = target + N(0,
    sigma_d^2).  Shape: best-first expansion by cumulative draft log-prob
    at temperature T (lowest node id on ties); a node at depth d gets the
    top max(1, branch - d) tokens of its draft row as children (in rank
    order, by logit then lower id); nodes at ``max_depth`` are leaves; stop
    at N nodes."""
    g = _gen(seed, device)
    target32 = _randn((B, N, V), g, device, sigma_t)
    draft32 = target32 + _randn((B, N, V), g, device, sigma_d)
    target = _cast(target32, dtype)
    draft = _cast(draft32, dtype)
    Tl = T if T > 0 else 1.0
    parent = np.full((B, N), -1, np.int32)
    toks = np.full((B, N), -1, np.int32)
    kmax = max(1, branch)
    # log-probs and ranked tokens of every row, computed once per sequence
    for b in range(B):
        d32 = draft[b].float()
        logq = (d32 / Tl - torch.logsumexp(d32 / Tl, dim=1,
                                           keepdim=True)).double().cpu()
        # rank by (logit desc, id asc): stable sort of the negated logits
        order = torch.sort(-d32, dim=1, stable=True).indices[:, :kmax].cpu()
        depth = [0] * N
        cum = [0.0] * N
        heap = [(0.0, 0)]
        count = 1
        while count < N and heap:
            _, u = heapq.heappop(heap)
            k = max(1, branch - depth[u])
            for r in range(k):
                if count >= N:
                    break
                t = int(order[u, r])
                v = count
                count += 1
                parent[b, v] = u
                toks[b, v] = t
                depth[v] = depth[u] + 1
                cum[v] = cum[u] + float(logq[u, t])
                if depth[v] < max_depth:
                    heapq.heappush(heap, (-cum[v], v))
        if count < N:
            raise ValueError("tree shape cannot reach %d nodes" % N)
    u = torch.from_numpy(uniforms(seed * 7919 + 43, (B, N))).to(device)
    return TreeCase(target, draft,
                    torch.from_numpy(parent).to(device),
                    torch.from_numpy(toks).to(device), u, float(T))


# --------------------------------------------------------------------------
# The five workloads (sizes of the pages' setting; seed = 1000 + index)
# --------------------------------------------------------------------------
WORKLOADS = {
    "tiny": "tiny linear verify: B=1, gamma=4, V=1000, fp32, T=1.0",
    "linear": "linear verify: B=32, gamma=8, V=32000, bf16, spike +8, "
              "T in {0, 0.7, 1.0}",
    "kcand": "diffusion K-candidate self-selection: B=64, K=8, gamma=16, "
             "V=152064, bf16, T=1.0",
    "tree": "tree verify: B=16, N=64 nodes (depth <= 8, top-k children "
            "k = 4..1), V=151936, bf16, T=0.8",
    "large": "large-batch verify + fan-out: B=256, gamma=8, V=128256, "
             "fp32, T=1.0, geometric fan-out a=0.8 r=1 K=8 budget 64",
}


def tiny(round_index=0, device="cpu") -> LinearCase:
    return linear_case(1, 4, 1000, torch.float32, 1.0,
                       seed=1000 + round_index, sigma_t=2.0, sigma_d=1.0,
                       device=device)


def linear(T=1.0, round_index=0, device="cpu") -> LinearCase:
    return linear_case(32, 8, 32000, torch.bfloat16, T,
                       seed=1001 + 97 * round_index, sigma_t=3.0,
                       sigma_d=1.5, spike=8.0, device=device)


def kcand(round_index=0, device="cpu") -> KcandCase:
    return kcand_case(64, 8, 16, 152064, torch.bfloat16, 1.0,
                      seed=1002 + 97 * round_index, device=device)


def tree(round_index=0, device="cpu") -> TreeCase:
    return tree_case(16, 64, 151936, torch.bfloat16, 0.8,
                     seed=1003 + 97 * round_index, device=device)


def large(round_index=0, device="cpu", B=256) -> LinearCase:
    """The large workload: B=256 sequences (fewer only for profiling runs),
    gamma=8, V=128256 fp32, T=1, 9 draft rows."""
    return linear_case(B, 8, 128256, torch.float32, 1.0,
                       seed=1004 + 97 * round_index, sigma_t=3.0,
                       sigma_d=1.0, draft_rows=9, device=device)
