"""Pins for the oracle's preselection (SnapKV-style, "KTransformers 长上下文稀疏注意力实战…"
§4.4 "预选择 Preselect" and the §4.6 `preselect_block()` pseudocode).

The oracle is checked against an independent restatement built from library
routines: torch's softmax over each local query's causal logits, summed over the
unit's query heads, and torch's `avg_pool1d` (stride 1, zero padding kernel//2,
padding counted in the divisor) over the Context tokens only, as the pseudocode
slices the vote vector between the Initial and Local parts before pooling.  A
block's score is the largest pooled vote of its tokens; the oracle's
preselection for every `count` from 1 to C must be the top `count` blocks of
that ranking (ties to the lower block).  Comparing every count compares the
whole ranking.

The inputs plant strong-vote tokens where a plausible slip would change the
ranking, and `test_inputs_expose_plausible_mistakes` shows, for each slip, that
the restatement with the slip ranks differently on these very inputs, so an
oracle carrying it would fail the comparison:
  * SHARED votes summed over one KV head instead of all of them;
  * pooling each block on its own instead of along the Context tokens;
  * pooling the whole sequence instead of only the Context tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

BS = 128


def _decode(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _logical(pool, kv, b, h):
    n = int(kv.seq_lens[b])
    rows = [pool[kv.block_table[b, t // BS], h, t % BS] for t in range(n)]
    return _decode(np.array(rows).reshape(n, kv.d))


def _votes(kv, w, b, heads):
    """Sum over the local queries (position n-T+i sees tokens <= its position)
    and the query heads of `heads`' groups of softmax(q k^T * scale): [n]."""
    p = w.params
    G = p.num_q_heads // kv.H_kv
    n = int(kv.seq_lens[b])
    T = w.q_local.shape[1]
    vote = torch.zeros(n, dtype=torch.float64)
    for h in heads:
        K = torch.from_numpy(_logical(kv.k_pool, kv, b, h))
        for i in range(T):
            pos = n - T + i
            for g in range(G):
                q = torch.from_numpy(_decode(w.q_local[b, i, h * G + g]))
                logits = (K[:pos + 1] @ q) * p.softmax_scale
                vote[:pos + 1] += torch.softmax(logits, dim=0)
    return vote


def _block_scores(vote, c0, c1, kernel, *, per_block=False, whole_sequence=False):
    """Largest pooled vote of each Context block c0..c1-1."""
    pool = lambda x: torch.nn.functional.avg_pool1d(
        x[None, None], kernel, stride=1, padding=kernel // 2, count_include_pad=True)[0, 0]
    if whole_sequence:
        pooled = pool(vote)[c0 * BS:c1 * BS]
    elif per_block:
        pooled = torch.cat([pool(vote[j * BS:(j + 1) * BS]) for j in range(c0, c1)])
    else:
        pooled = pool(vote[c0 * BS:c1 * BS])
    return pooled.reshape(c1 - c0, BS).max(dim=1).values.numpy()


def _ranking(scores, c0):
    return [c0 + j for j in sorted(range(len(scores)), key=lambda j: (-scores[j], j))]


def _unit_heads(p, H_kv, u):
    return list(range(H_kv)) if p.head_mode == synth.HEAD_SHARED else [u]


def _plant(w, kv, b, h, token, beta):
    """Make the key of `token` (KV head h) point along the sum of the group's
    local queries, scaled by beta, so that its softmax vote dominates."""
    G = w.params.num_q_heads // kv.H_kv
    u = _decode(w.q_local[b, :, h * G:(h + 1) * G]).reshape(-1, kv.d).sum(axis=0)
    u /= np.linalg.norm(u)
    row = (beta * u).astype(np.float16).view(np.uint16)
    kv.k_pool[kv.block_table[b, token // BS], h, token % BS] = row


def _planted_workload(seed, head_mode, H_kv, n_blocks_ctx=8):
    """One sequence: Initial 1 block, Context n_blocks_ctx blocks, Local 2
    blocks of which the last is partial; strong-vote tokens next to the
    Initial/Local edges, on a Context block boundary, and in one block for the
    last KV head only."""
    n = BS * (1 + n_blocks_ctx + 1) + 37
    w = synth.custom(seed, [n], num_q_heads=2 * H_kv, num_kv_heads=H_kv, rep=synth.REP_QUEST,
                     head_mode=head_mode, local_queries=8, initial_blocks=1, local_blocks=2)
    kv = oracle.KV.of(w)
    c0, c1 = 1, 1 + n_blocks_ctx
    # the last tokens of the Initial block and the first of the Local window:
    # only pooling across the Context edge lets them raise blocks c0 and c1-1
    for t in (BS - 3, BS - 2, BS - 1, c1 * BS, c1 * BS + 1, c1 * BS + 2):
        _plant(w, kv, 0, 0, t, 26.0)
    # the last token of block 4: pooling along the Context tokens spills it
    # into block 5, pooling each block on its own does not
    _plant(w, kv, 0, 0, 5 * BS - 1, 30.0)
    # a token in the middle of block 6 that only the last KV head sees
    _plant(w, kv, 0, H_kv - 1, 6 * BS + 60, 34.0)
    # two moderate tokens elsewhere, so that the rest of the ranking is not noise
    _plant(w, kv, 0, 0, 2 * BS + 90, 18.0)
    _plant(w, kv, 0, min(1, H_kv - 1), 7 * BS + 10, 20.0)
    return w, kv, c0, c1


def _check_against_restatement(w, kv, c0, c1, kernel):
    p = w.params
    SEL = 1 if p.head_mode == synth.HEAD_SHARED else kv.H_kv
    C = c1 - c0
    expected = []
    for u in range(SEL):
        s = _block_scores(_votes(kv, w, 0, _unit_heads(p, kv.H_kv, u)), c0, c1, kernel)
        expected.append((s, _ranking(s, c0)))
    for count in range(1, C + 1):
        presel, pcnt = oracle.preselect(kv, p, w.q_local, kernel=kernel, count=count)
        for u in range(SEL):
            s, rank = expected[u]
            assert pcnt[0, u] == count
            kth, nxt = s[rank[count - 1] - c0], (s[rank[count] - c0] if count < C else -np.inf)
            if abs(kth - nxt) <= 1e-12 * abs(kth):
                continue   # an exact-arithmetic tie at the cut: either block is right
            assert list(presel[0, u, :count]) == sorted(rank[:count]), (u, count)


@pytest.mark.parametrize("kernel", [5, 13])
@pytest.mark.parametrize("H_kv", [2, 3])
def test_shared_preselection_matches_library_restatement(kernel, H_kv):
    w, kv, c0, c1 = _planted_workload(70 + H_kv, synth.HEAD_SHARED, H_kv)
    _check_against_restatement(w, kv, c0, c1, kernel)


@pytest.mark.parametrize("kernel", [1, 5, 13])
def test_separate_preselection_matches_library_restatement(kernel):
    w, kv, c0, c1 = _planted_workload(75, synth.HEAD_SEPARATE, 2)
    _check_against_restatement(w, kv, c0, c1, kernel)


def test_random_votes_ragged_two_sequences_match_library_restatement():
    # no plants: two ragged sequences, three KV heads, SEPARATE, kernel 7
    w = synth.custom(77, [BS * 9 + 100, BS * 7 + 1], num_q_heads=6, num_kv_heads=3,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE, local_queries=5,
                     initial_blocks=1, local_blocks=2)
    kv = oracle.KV.of(w)
    for b, n in enumerate(w.seq_lens):
        nb = (int(n) + BS - 1) // BS
        c0, c1 = 1, nb - 2
        count = (c1 - c0) // 2
        presel, pcnt = oracle.preselect(kv, w.params, w.q_local, kernel=7, count=count)
        for u in range(3):
            s = _block_scores(_votes(kv, w, b, [u]), c0, c1, 7)
            assert pcnt[b, u] == count
            assert list(presel[b, u, :count]) == sorted(_ranking(s, c0)[:count]), (b, u)


def test_inputs_expose_plausible_mistakes():
    # each slip, restated, ranks the planted inputs differently from the correct
    # restatement (which the tests above tie to the oracle)
    kernel = 13
    w, kv, c0, c1 = _planted_workload(72, synth.HEAD_SHARED, 2)
    all_heads = _votes(kv, w, 0, [0, 1])
    right = _ranking(_block_scores(all_heads, c0, c1, kernel), c0)
    one_head = _ranking(_block_scores(_votes(kv, w, 0, [0]), c0, c1, kernel), c0)
    per_block = _ranking(_block_scores(all_heads, c0, c1, kernel, per_block=True), c0)
    whole = _ranking(_block_scores(all_heads, c0, c1, kernel, whole_sequence=True), c0)
    for name, wrong in (("one KV head", one_head), ("per-block pooling", per_block),
                        ("whole-sequence pooling", whole)):
        # a difference in the top half, so a mid-size count already shows it
        assert any(sorted(wrong[:m]) != sorted(right[:m]) for m in range(1, 5)), name
    # and the oracle agrees with the correct ranking at those counts
    for m in range(1, 5):
        presel, _ = oracle.preselect(kv, w.params, w.q_local, kernel=kernel, count=m)
        assert list(presel[0, 0, :m]) == sorted(right[:m])
