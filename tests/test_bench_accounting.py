"""The benchmark's work accounting (no kernels run).

The headline metric is effective TFLOP/s: the algorithmic FLOPs of one step
divided by its time.  The attention's FLOPs are counted from the selected
blocks with their actual (unpadded) token counts: 4 d per (query token,
selected key token) pair, 2 d for q·k and 2 d for p·v; the linear read
2 d² + 2 d per query token; the absorb 2 d² + d per evicted token and head;
the block scores 2 d per (query block, key block) pair (Hybrid Forcing,
English technical summary, sections 2.A.1 and 2.A.2).  These tests count the
same work token by token on small workloads with ragged blocks and compare it
with `bench.step_flops`, which counts it with array arithmetic."""

import itertools

import numpy as np
import pytest

import bench
from hybrid_sparse_linear_scores_b300.workloads import Workload


def _workload(nf, beta, C, W, heads, K):
    return Workload("acct", 1, heads, 64, nf, C, W, beta, seed=0, recipe="normal", topk=K, absorbed_frames=4)


def _brute_attention_flops(w, idx):
    d, nf, beta, bpf = w.head_dim, w.tokens_per_frame, w.block_size, w.blocks_per_frame
    total = 0
    for bh in range(w.heads_total):
        for c in range(w.chunk_frames):
            for i in range(nf):                      # every query token of the chunk
                qb = c * bpf + i // beta
                for kb in idx[bh, qb]:
                    j = kb % bpf                     # the key block's block within its frame
                    rows = sum(1 for t in range(nf) if t // beta == j)
                    total += 4 * d * rows
    return total


@pytest.mark.parametrize("nf,beta,C,W,heads,K", [(100, 32, 2, 3, 2, 3), (64, 64, 1, 2, 1, 1), (130, 64, 3, 4, 2, 5),
                                                  (97, 32, 1, 1, 3, 4)])
def test_attention_flops_count_actual_tokens(nf, beta, C, W, heads, K):
    w = _workload(nf, beta, C, W, heads, K)
    rng = np.random.default_rng(nf + beta + K)
    nkb, nqb = w.n_kb(0), w.n_qb()
    k = w.k_for(0)
    idx = np.stack([np.stack([np.sort(rng.choice(nkb, size=k, replace=False)) for _ in range(nqb)])
                    for _ in range(w.heads_total)]).astype(np.int32)
    fl = bench.step_flops(w, idx, n_ev_tokens=0)
    assert fl["attn"] == _brute_attention_flops(w, idx)


def test_linear_absorb_and_score_flops():
    w = _workload(100, 32, 2, 3, 2, 3)
    idx = np.zeros((w.heads_total, w.n_qb(), w.k_for(0)), np.int32)
    n_ev = 7 * w.tokens_per_frame
    fl = bench.step_flops(w, idx, n_ev_tokens=n_ev)
    d, BH = w.head_dim, w.heads_total
    q_tokens = w.chunk_frames * w.tokens_per_frame
    lin = sum(2 * d * d + 2 * d for _ in range(q_tokens)) * BH
    absorb = sum(2 * d * d + d for _ in range(n_ev)) * BH
    score = sum(2 * d for _ in itertools.product(range(w.n_qb()), range(w.n_kb(0)))) * BH
    assert (fl["lin"], fl["absorb"], fl["score"]) == (lin, absorb, score)
    assert fl["total"] == fl["attn"] + lin + absorb + score


def test_realistic_step_work():
    """The realistic workload's fixed terms, in the figures the documentation
    quotes (1.85 GFLOP of linear read for 12 heads x 4680 query tokens)."""
    from hybrid_sparse_linear_scores_b300.workloads import CONFIGS
    w = CONFIGS["realistic"]
    idx = np.zeros((w.heads_total, w.n_qb(), w.k_for(0)), np.int32)
    fl = bench.step_flops(w, idx, n_ev_tokens=0)
    assert fl["lin"] == (2 * 128 * 128 + 2 * 128) * 4680 * 12
    assert abs(fl["lin"] / 1e9 - 1.85) < 0.01
