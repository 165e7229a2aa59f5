"""Seeded synthetic inputs shaped like the TriForce decode-step workloads.

Shared by the tests, the smoke check and the benchmark.  Holds no arithmetic
of the method itself: only random draws, the planted-chunk recipe and the
harness-side sampling of draft tokens (the drafter's job, outside the path).

Recipe (every draw seeded):
* K, V, q (decode query) and Q (verify queries) ~ N(0, 1), rounded to bf16.
* Planted relevant chunks: per (sequence, KV head) round(frac * C_b) chunks,
  drawn uniformly without replacement; every valid row of a planted chunk is
  3 * q_hat + N(0, 0.5^2) with q_hat the unit vector of the group's summed
  decode query.  This gives the top-k a clear margin.
* Spec accept: target logits N(0, 2^2); draft logits = target + N(0, 1); for
  the two-level step the tiny drafter's logits add another N(0, 1).  Draft
  tokens are sampled from the draft distribution, uniforms are U[0, 1).
"""

from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    L: int  # context (max of the per-sequence lengths for ragged batches)
    layers: int
    chunk: int
    budget: int  # tokens; kc = budget // chunk chunks
    n_sink: int
    window: int
    T: int  # verify query tokens (gamma + 1)
    gamma: int  # accept step draft length
    vocab: int
    planted_frac: float
    seed: int
    ragged: bool = False  # per-sequence lengths uniform in [L_min, L]
    L_min: int = 0

    @property
    def kc(self) -> int:
        return self.budget // self.chunk

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


# The five workloads: a tiny single-layer step, one Llama2-7B-128K-shaped layer
# at 32K, the full 32-layer Llama2-7B cache at 128K, a Llama-3-8B-style GQA
# batch at 128K, and a ragged mixed batch.
TINY = Workload("tiny-1layer-mha8-4k", 1, 8, 8, 128, 4096, 1, 8, 512, 4, 252, 5, 4, 32000, 0.02, 0)
LLAMA2_7B_32K_1LAYER = Workload("llama2-7b-32k-1layer", 1, 32, 32, 128, 32768, 1, 8, 4096, 4, 252, 6, 5, 32000, 0.01, 1)
LLAMA2_7B_128K = Workload("llama2-7b-128k-32layer", 1, 32, 32, 128, 131072, 32, 8, 4096, 4, 252, 6, 5, 32000, 0.01, 2)
LLAMA3_8B_GQA_128K = Workload("llama3-8b-gqa-128k-b4", 4, 32, 8, 128, 131072, 32, 8, 4096, 4, 252, 6, 5, 32000, 0.01, 3)
MIXED_BATCH = Workload("mixed-b8-gqa-16k-128k", 8, 32, 8, 128, 131072, 16, 8, 4096, 4, 252, 6, 5, 32000, 0.01, 4,
                       ragged=True, L_min=16384)

WORKLOADS = {w.name: w for w in (TINY, LLAMA2_7B_32K_1LAYER, LLAMA2_7B_128K, LLAMA3_8B_GQA_128K, MIXED_BATCH)}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_normal(gen, shape, std=1.0, device="cpu") -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def seq_lens_for(w: Workload, device="cpu") -> torch.Tensor:
    """Per-sequence context lengths (int32).  Ragged batches draw U[L_min, L]."""
    if not w.ragged:
        return torch.full((w.B,), w.L, dtype=torch.int32, device=device)
    g = generator(w.seed * 7919 + 17, "cpu")
    lens = torch.randint(w.L_min, w.L + 1, (w.B,), generator=g, dtype=torch.int64)
    return lens.to(torch.int32).to(device)


def decode_queries(w: Workload, layer: int, device="cpu"):
    """q [B, Hq, D] bf16 (decode query) and Q [B, Hq, T, D] bf16 (verify queries)."""
    g = generator(w.seed * 1_000_003 + 101 * layer + 1, device)
    q = bf16_normal(g, (w.B, w.Hq, w.D), device=device)
    Q = bf16_normal(g, (w.B, w.Hq, w.T, w.D), device=device)
    return q, Q


def planted_chunks(w: Workload, layer: int, seq_lens_cpu: torch.Tensor):
    """Planted chunk ids per (b, g): a list of lists of int64 tensors (CPU)."""
    g = generator(w.seed * 1_000_003 + 101 * layer + 2, "cpu")
    out = []
    for b in range(w.B):
        L = int(seq_lens_cpu[b])
        C = -(-L // w.chunk)
        n = int(round(w.planted_frac * C))
        row = []
        for _ in range(w.Hkv):
            perm = torch.randperm(C, generator=g)[:n]
            row.append(torch.sort(perm).values)
        out.append(row)
    return out


def kv_cache(w: Workload, layer: int, q: torch.Tensor, seq_lens_cpu: torch.Tensor, device="cpu",
             K_out: torch.Tensor | None = None, V_out: torch.Tensor | None = None,
             fill_invalid: float | None = None):
    """K, V [B, Hkv, Lmax, D] bf16 with planted chunks aligned to the decode query.

    K_out / V_out may be preallocated views (e.g. one layer of a multi-layer
    cache).  fill_invalid, when given, overwrites positions >= L_b with that
    value (e.g. NaN) so tests can show they are never read into a result.
    """
    gen = generator(w.seed * 1_000_003 + 101 * layer + 3, device)
    shape = (w.B, w.Hkv, w.L, w.D)
    if K_out is None:
        K_out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if V_out is None:
        V_out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    # Draw in slabs to bound the fp32 temporary.
    for b in range(w.B):
        for h in range(w.Hkv):
            K_out[b, h].copy_(bf16_normal(gen, (w.L, w.D), device=device))
            V_out[b, h].copy_(bf16_normal(gen, (w.L, w.D), device=device))
    planted = planted_chunks(w, layer, seq_lens_cpu)
    gp = generator(w.seed * 1_000_003 + 101 * layer + 4, device)
    qg = q.float().reshape(w.B, w.Hkv, w.G, w.D).sum(dim=2)  # [B, Hkv, D]
    qhat = qg / qg.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    for b in range(w.B):
        L = int(seq_lens_cpu[b])
        for h in range(w.Hkv):
            ids = planted[b][h]
            if ids.numel() == 0:
                continue
            rows = (ids[:, None] * w.chunk + torch.arange(w.chunk)[None, :]).reshape(-1)
            rows = rows[rows < L].to(device)
            noise = torch.randn((rows.numel(), w.D), generator=gp, device=device) * 0.5
            K_out[b, h, rows] = (3.0 * qhat[b, h][None, :] + noise).to(torch.bfloat16)
    if fill_invalid is not None:
        for b in range(w.B):
            L = int(seq_lens_cpu[b])
            K_out[b, :, L:] = fill_invalid
            V_out[b, :, L:] = fill_invalid
    return K_out, V_out, planted


def accept_inputs(B, gamma, vocab, seed, device="cpu", tgt_std=2.0, drf_noise=1.0):
    """One verification level: target logits [B, gamma+1, V], draft logits
    [B, gamma, V], draft tokens sampled from softmax(draft), uniforms."""
    g = generator(seed * 1_000_003 + 11, device)
    tgt = torch.randn((B, gamma + 1, vocab), generator=g, device=device) * tgt_std
    drf = tgt[:, :gamma] + torch.randn((B, gamma, vocab), generator=g, device=device) * drf_noise
    x = sample_tokens(drf, g)
    u_acc = torch.rand((B, gamma), generator=g, device=device)
    u_res = torch.rand((B,), generator=g, device=device)
    return tgt.contiguous(), drf.contiguous(), x, u_acc, u_res


def sample_tokens(logits: torch.Tensor, gen: torch.Generator) -> torch.Tensor:
    """Draw one token per row from softmax(logits) (the drafter's own sampling)."""
    B, R, Vn = logits.shape
    probs = torch.softmax(logits.double(), dim=-1).reshape(B * R, Vn)
    x = torch.multinomial(probs, 1, replacement=True, generator=gen).reshape(B, R)
    return x.to(torch.int32)


def two_level_inputs(B, gamma1, vocab, seed, device="cpu"):
    """Hierarchical step inputs: p (target, gamma1+2 rows), q (retrieval drafter,
    gamma1+1 rows), r (tiny drafter, gamma1 rows), tiny-drafter tokens x ~ r and
    the uniforms of both levels."""
    g = generator(seed * 1_000_003 + 13, device)
    gamma2 = gamma1 + 1
    p = torch.randn((B, gamma2 + 1, vocab), generator=g, device=device) * 2.0
    q = p[:, :gamma2] + torch.randn((B, gamma2, vocab), generator=g, device=device)
    r = q[:, :gamma1] + torch.randn((B, gamma1, vocab), generator=g, device=device)
    x = sample_tokens(r, g)
    u1 = torch.rand((B, gamma1), generator=g, device=device)
    ur1 = torch.rand((B,), generator=g, device=device)
    u2 = torch.rand((B, gamma2), generator=g, device=device)
    ur2 = torch.rand((B,), generator=g, device=device)
    return dict(p=p.contiguous(), q=q.contiguous(), r=r.contiguous(), x=x, u1=u1, ur1=ur1, u2=u2, ur2=ur2)



def tree_accept_inputs(B, T, vocab, seed, device="cpu", tgt_std=2.0, drf_noise=1.0, branching=None):
    """A candidate tree per sequence: parent [B, T] (candidate j extends a
    uniformly drawn earlier candidate or the prefix, -1), verifier logits
    [B, T+1, V] (row 0 the prefix, row 1+j after candidate j), the drafter's
    logits at every node (the prefix and each candidate) = the verifier's at
    that node + noise, drf [B, T, V] = the row of candidate j's parent, tokens
    drawn independently from those rows (siblings are independent draws) and
    uniforms.  branching=k gives every node up to k children in order instead
    (a complete k-ary tree laid out breadth first)."""
    g = generator(seed * 1_000_003 + 17, device)
    if branching:
        parent = torch.tensor([(j // branching) - 1 for j in range(T)], dtype=torch.int32, device=device)
        parent = parent[None].repeat(B, 1)
    else:
        span = torch.arange(T, device=device, dtype=torch.float32)[None] + 1.0  # choices -1 .. j-1
        parent = (torch.rand((B, T), generator=g, device=device) * span).floor().to(torch.int32) - 1
    tgt = torch.randn((B, T + 1, vocab), generator=g, device=device) * tgt_std
    node_drf = tgt + torch.randn((B, T + 1, vocab), generator=g, device=device) * drf_noise
    rows = (parent.long() + 1).clamp(0, T)  # node index of the parent: 0 = prefix, 1 + i = candidate i
    drf = torch.gather(node_drf, 1, rows[:, :, None].expand(B, T, vocab)) if T > 0 else node_drf[:, :0]
    x = sample_tokens(drf, g) if T > 0 else torch.zeros((B, 0), dtype=torch.int32, device=device)
    u_acc = torch.rand((B, T), generator=g, device=device)
    u_res = torch.rand((B,), generator=g, device=device)
    return dict(tgt=tgt.contiguous(), drf=drf.contiguous(), x=x.contiguous(), parent=parent.contiguous(),
                u_acc=u_acc, u_res=u_res)
