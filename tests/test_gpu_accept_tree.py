"""GPU parity of tf_spec_accept_tree (accept / resample over a candidate tree)
against the float64 oracle, and against tf_spec_accept on chains.

Tolerance as for the chain call: n_acc, next token, kept tokens and kept
candidate indices bit-exact, except sequences where the oracle took a decision
with a uniform within 1e-6 of its boundary (counted; at V = 32000 that is a
few per cent of the draws, since a token's CDF step is ~1/V wide).
"""

import numpy as np
import pytest
import torch
from scipy import stats

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O

pytestmark = pytest.mark.gpu

EDGE = 1e-6


def run_tree(cuda_lib, d, temperature=1.0):
    dev = "cuda"
    r = cuda_lib.tf_spec_accept_tree(d["tgt"].to(dev), d["drf"].to(dev), d["x"].to(dev), d["parent"].to(dev),
                                     d["u_acc"].to(dev), d["u_res"].to(dev), temperature=temperature)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in r]


def check_against_oracle(d, got, temperature=1.0, max_edge_frac=0.25):
    o = O.spec_accept_tree(d["tgt"].double().numpy(), d["drf"].double().numpy(), d["x"].numpy(),
                           d["parent"].numpy(), d["u_acc"].double().numpy(), d["u_res"].double().numpy(),
                           temperature)
    n_acc, nxt, out, nodes = got
    T = d["x"].shape[1]
    same = ((n_acc == o["n_acc"]) & (nxt == o["next"]) & np.all(out == o["out_tokens"], axis=1) &
            np.all(nodes[:, :T] == o["acc_nodes"], axis=1))
    edge = o["margin"] < EDGE
    bad = ~same & ~edge
    assert not bad.any(), f"{bad.sum()} sequences differ away from a decision boundary: {np.nonzero(bad)[0][:10]}"
    # At V = 32000 a draw's CDF step is ~1/V wide, so ~2e-6 * V of the uniforms
    # land within 1e-6 of one of its ends: the count is a property of the
    # oracle's draws; it must leave most sequences compared exactly.
    assert edge.mean() <= max_edge_frac
    return o


@pytest.mark.parametrize("B,T,V,branching", [
    (64, 8, 7, None),        # tiny vocabulary, random trees
    (64, 8, 1000, None),
    (96, 12, 32000, None),   # the workloads' vocabulary
    (16, 14, 32000, 2),      # a complete binary tree (every node has two children)
    (16, 12, 32000, 3),      # three-way branching
], ids=["v7", "v1000", "v32000", "binary-v32000", "ternary-v32000"])
def test_tree_accept_matches_oracle(cuda_lib, B, T, V, branching):
    d = synth.tree_accept_inputs(B, T, V, seed=T * 7 + V % 97, branching=branching)
    got = run_tree(cuda_lib, d)
    o = check_against_oracle(d, got)
    assert o["n_acc"].max() >= 1  # the walk goes below the prefix for some sequences


def test_tree_accept_edge_inputs(cuda_lib):
    # Invalid tokens (the subtree is removed), parent links outside [-1, j)
    # (read as the prefix), temperature != 1.
    d = synth.tree_accept_inputs(48, 10, 2000, seed=5)
    x, par = d["x"].clone(), d["parent"].clone()
    x[::5, 0] = -1
    x[1::7, 3] = 2000
    par[::3, 6] = 6       # points at itself
    par[1::4, 9] = 40     # past the end
    par[2::5, 4] = -7     # below -1
    d["x"], d["parent"] = x, par
    check_against_oracle(d, run_tree(cuda_lib, d, temperature=0.7), temperature=0.7)


def test_tree_accept_without_candidates(cuda_lib):
    d = synth.tree_accept_inputs(9, 0, 500, seed=3)
    n_acc, nxt, out, _ = run_tree(cuda_lib, d)
    o = O.spec_accept_tree(d["tgt"].double().numpy(), d["drf"].double().numpy(), d["x"].numpy(),
                           d["parent"].numpy(), d["u_acc"].double().numpy(), d["u_res"].double().numpy())
    assert np.all(n_acc == 0)
    ok = (nxt == o["next"]) | (o["margin"] < EDGE)
    assert ok.all() and np.array_equal(out[:, 0][ok], nxt[ok])


@pytest.mark.parametrize("V", [5000, 32000])
def test_chain_tree_equals_chain_call(cuda_lib, V):
    """parent[j] = j - 1 with the chain call's own inputs: the same values
    (ratio tests, residual weights, scan), so the outputs agree bit for bit."""
    B, gamma = 32, 6
    tgt, drf, x, ua, ur = synth.accept_inputs(B, gamma, V, seed=V % 13)
    x[::4, 4] = -1  # some drafts end early
    dev = "cuda"
    chain = (torch.arange(gamma, dtype=torch.int32) - 1)[None].repeat(B, 1)
    a = cuda_lib.tf_spec_accept(tgt.to(dev), drf.to(dev), x.to(dev), ua.to(dev), ur.to(dev))
    b = cuda_lib.tf_spec_accept_tree(tgt.to(dev), drf.to(dev), x.to(dev), chain.to(dev), ua.to(dev), ur.to(dev))
    torch.cuda.synchronize()
    for u, v in zip(a, b[:3]):
        assert torch.equal(u, v)
    d = dict(tgt=tgt, drf=drf, x=x, parent=chain, u_acc=ua, u_res=ur)
    check_against_oracle(d, [t.cpu().numpy() for t in b])


def test_branching_root_chi_square_on_gpu(cuda_lib):
    """Three siblings drawn from the root's drafter distribution: the first
    emitted token follows the verifier's prefix row (V = 16, 2*10^5 trials)."""
    N, V, k = 200_000, 16, 3
    rng = np.random.default_rng(12)
    tgt = rng.standard_normal((k + 1, V)) * 2.0
    qr = tgt[0] + rng.standard_normal(V)
    q = np.exp(qr - qr.max())
    q /= q.sum()
    dev = "cuda"
    tg = torch.tensor(tgt, dtype=torch.float32)[None].repeat(N, 1, 1).to(dev)
    dr = torch.tensor(np.tile(qr, (k, 1)), dtype=torch.float32)[None].repeat(N, 1, 1).to(dev)
    x = torch.from_numpy(rng.choice(V, size=(N, k), p=q).astype(np.int32)).to(dev)
    par = torch.full((N, k), -1, dtype=torch.int32, device=dev)
    ua = torch.from_numpy(rng.random((N, k)).astype(np.float32)).to(dev)
    ur = torch.from_numpy(rng.random(N).astype(np.float32)).to(dev)
    n_acc, nxt, out, nodes = cuda_lib.tf_spec_accept_tree(tg, dr, x, par, ua, ur)
    first = out[:, 0].cpu().numpy()
    p0 = np.exp(tgt[0] - tgt[0].max())
    p0 /= p0.sum()
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, p0 * N).pvalue > 1e-3
