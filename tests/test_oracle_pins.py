"""Pins for the CPU oracle: each test checks the oracle against something other
than itself — a library routine, a closed form, an invariant stated by the
article, brute force on tiny inputs, or a number the article prints.

Article: "KTransformers 长上下文稀疏注意力实战：单张 24GB GPU 跑通 1M Token KVCache 的
完整方案" (sections cited as §N.M).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def decode(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def small_kv(seed, lens, H_kv=2, d=128, bs=128, permute=True):
    """A paged KV with random pages, built here (not with the oracle)."""
    lens = np.asarray(lens, dtype=np.int32)
    nbs = [(int(n) + bs - 1) // bs for n in lens]
    P = max(1, sum(nbs))
    rng = np.random.default_rng(seed)
    order = rng.permutation(P) if permute else np.arange(P)
    table = np.zeros((len(lens), max(1, max(nbs))), dtype=np.int32)
    off = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = order[off:off + nb]
        off += nb
    k = f16(rng.standard_normal((P, H_kv, bs, d)))
    v = f16(rng.standard_normal((P, H_kv, bs, d)))
    return oracle.KV(k, v, table, lens, block_size=bs)


def logical_keys(kv, b, h):
    """[n][d] decoded keys of sequence b, KV head h, gathered through the table."""
    n = int(kv.seq_lens[b])
    rows = [kv.k_pool[kv.block_table[b, t // kv.bs], h, t % kv.bs] for t in range(n)]
    return decode(np.array(rows).reshape(n, kv.d))


def logical_values(kv, b, h):
    n = int(kv.seq_lens[b])
    rows = [kv.v_pool[kv.block_table[b, t // kv.bs], h, t % kv.bs] for t in range(n)]
    return decode(np.array(rows).reshape(n, kv.d))


# --------------------------------------------------------------------------- binary16

def test_f16_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, ours[0x8000]) == -1.0 and math.copysign(1.0, ours[0]) == 1.0


def test_generator_encoder_matches_numpy_rounding():
    x = RNG.standard_normal(200000) * np.exp(RNG.uniform(-22, 11, 200000))
    x = np.concatenate([x, [0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0**-24, 2.0**-25,
                            3 * 2.0**-26, -(2.0**-14) * 1.5]])
    with np.errstate(over="ignore"):  # values past the binary16 range become inf on purpose
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(synth.f16_bits(x), ref)


def test_generator_is_counter_based_and_seeded():
    a = synth.normal_f16((1000,), 7, 3)
    b = synth.normal_f16((400,), 7, 3, first=600)
    assert np.array_equal(a[600:], b)
    assert not np.array_equal(a, synth.normal_f16((1000,), 8, 3))
    z = decode(synth.normal_f16((1 << 20,), 1, 1))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


# --------------------------------------------------------------------------- partition

@pytest.mark.parametrize("n,I,L,expect", [
    (4096, 1, 4, (32, 1, 28)),          # tiny workload: 27 context blocks
    (131072, 1, 32, (1024, 1, 992)),    # 128K, Local 4096: 991 context blocks
    (1048576, 1, 32, (8192, 1, 8160)),  # 1M: 8159 context blocks
    (1000, 1, 2, (8, 1, 6)),            # ragged tail: last block has 104 tokens
    (384, 1, 2, (3, 1, 1)),             # nb == I + L: no context
    (200, 1, 4, (2, 1, 1)),             # nb < I + L: all dense
    (0, 1, 4, (0, 0, 0)),
])
def test_partition_hand_cases(n, I, L, expect):
    assert oracle.partition(n, I, L) == expect


def test_attended_tokens_match_article():
    rows = [list(map(int, l.split())) for l in open(os.path.join(GOLDEN, "attended_tokens.txt"))
            if l.strip() and not l.startswith("#")]
    for bs, local_tokens, k, init_tokens, attended in rows:
        for n in (131072, 262144, 1048576):
            nb, c0, c1 = oracle.partition(n, init_tokens // bs, local_tokens // bs, bs)
            sel = oracle.select(np.arange(c1 - c0, dtype=np.float64), c0, k)
            tokens = (c0 + sel.size + (nb - c1)) * bs
            assert tokens == attended


def test_kv_layout_matches_article_memory_table():
    # 32 layers x our per-layer K+V pool bytes per token, against §6.2's table.
    w = synth.custom(0, [1024], num_q_heads=32, num_kv_heads=8)
    per_token_layer = (w.k_pool.nbytes + w.v_pool.nbytes) / (w.num_pages * 128)
    rows = [l.split() for l in open(os.path.join(GOLDEN, "memory_table.txt"))
            if l.strip() and not l.startswith("#")]
    for ctx, gb, checked in rows:
        if checked != "1":
            continue
        total_gb = 32 * per_token_layer * int(ctx) / 1e9
        decimals = len(gb.split(".")[1])
        assert math.floor(total_gb * 10**decimals) / 10**decimals == float(gb)


# --------------------------------------------------------------------------- reps

@pytest.mark.parametrize("rep", [synth.REP_MAX, synth.REP_QUEST])
def test_max_min_reps_are_numpy_extrema(rep):
    kv = small_kv(1, [128 * 5 + 17], H_kv=2)
    p = synth.Params(num_q_heads=2, initial_blocks=1, local_blocks=1, top_k=2, rep=rep,
                     head_mode=synth.HEAD_SEPARATE)
    for h in range(2):
        K = logical_keys(kv, 0, h)
        for j in range(5):
            r = decode(oracle.block_reps(kv, p, 0, j, h))
            blk = K[j * 128:(j + 1) * 128]
            if rep == synth.REP_MAX:
                assert np.array_equal(r[0], blk.max(axis=0))
            else:
                assert np.array_equal(r[0], blk.min(axis=0))
                assert np.array_equal(r[1], blk.max(axis=0))


def test_signed_zero_total_order():
    # a channel holding only +0 and -0: max picks +0, min picks -0 (binary16 totalOrder)
    k = np.zeros((1, 1, 128, 128), dtype=np.uint16)
    k[0, 0, ::2, 0] = 0x8000
    k[0, 0, :, 1] = 0x8000
    kv = oracle.KV(k, k, np.zeros((1, 1), np.int32), [128])
    p = synth.Params(num_q_heads=1, initial_blocks=0, local_blocks=1, top_k=1,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE)
    r = oracle.block_reps(kv, p, 0, 0, 0)
    assert r[1, 0] == 0x0000 and r[0, 0] == 0x8000
    assert r[1, 1] == 0x8000 and r[0, 1] == 0x8000
    assert r[1, 2] == 0x0000 and r[0, 2] == 0x0000


def test_mean_rep_is_exact_mean_rounded_once():
    kv = small_kv(2, [128 * 3], H_kv=1)
    # add some large and tiny magnitudes so that naive float32 sums would round
    kv.k_pool[0, 0, :, :8] = f16(RNG.standard_normal((128, 8)) * 3000)
    kv.k_pool[0, 0, :, 8:16] = f16(RNG.standard_normal((128, 8)) * 1e-6)
    p = synth.Params(num_q_heads=1, initial_blocks=0, local_blocks=1, top_k=1,
                     rep=synth.REP_MEAN, head_mode=synth.HEAD_SEPARATE)
    K = logical_keys(kv, 0, 0)
    for j in range(3):
        got = oracle.block_reps(kv, p, 0, j, 0)
        for c in range(128):
            exact = sum(Fraction(float(x)) for x in K[j * 128:(j + 1) * 128, c]) / 128
            want = np.float32(float(exact))  # float(Fraction) is exact here (< 53 bits)
            assert got[c].view(np.uint32) == want.view(np.uint32)


def test_fix_reps_are_strided_rows():
    kv = small_kv(3, [128 * 2], H_kv=2)
    p = synth.Params(num_q_heads=2, initial_blocks=0, local_blocks=1, top_k=1,
                     rep=synth.REP_FIX, head_mode=synth.HEAD_SEPARATE, fix_stride=32)
    for h in range(2):
        for j in range(2):
            r = oracle.block_reps(kv, p, 0, j, h)
            page = kv.block_table[0, j]
            assert np.array_equal(r, kv.k_pool[page, h, [0, 32, 64, 96]])


# --------------------------------------------------------------------------- scores

def test_quest_score_is_an_upper_bound_of_every_key_in_the_block():
    # §3.1: the Quest score bounds q.k from above for every token of the block.
    kv = small_kv(4, [128 * 12], H_kv=1)
    p = synth.Params(num_q_heads=1, initial_blocks=0, local_blocks=1, top_k=1,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE)
    K = logical_keys(kv, 0, 0)
    for trial in range(20):
        q = decode(f16(RNG.standard_normal(128) * (1 + trial)))
        for j in range(12):
            reps = decode(oracle.block_reps(kv, p, 0, j, 0))
            s = oracle.head_block_score(q, reps, synth.REP_QUEST)
            true_max = (K[j * 128:(j + 1) * 128] @ q).max()
            slack = 1e-12 * np.abs(q).sum() * np.abs(K).max()
            assert s >= true_max - slack


def test_quest_score_sign_special_cases():
    # q >= 0 elementwise: the bound is q.kmax; q <= 0: the bound is q.kmin.
    kv = small_kv(5, [128 * 4], H_kv=1)
    p = synth.Params(num_q_heads=1, initial_blocks=0, local_blocks=1, top_k=1,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE)
    K = logical_keys(kv, 0, 0)
    q = decode(f16(np.abs(RNG.standard_normal(128))))
    for j in range(4):
        reps = decode(oracle.block_reps(kv, p, 0, j, 0))
        blk = K[j * 128:(j + 1) * 128]
        assert oracle.head_block_score(q, reps, synth.REP_QUEST) == pytest.approx(
            float(np.dot(q, blk.max(axis=0))), rel=1e-12)
        assert oracle.head_block_score(-q, reps, synth.REP_QUEST) == pytest.approx(
            float(np.dot(-q, blk.min(axis=0))), rel=1e-12)


def test_quest_is_tight_for_a_constant_block():
    k = np.tile(f16(RNG.standard_normal(128)), (1, 1, 128, 1)).reshape(1, 1, 128, 128)
    kv = oracle.KV(k, k, np.zeros((1, 1), np.int32), [128])
    p = synth.Params(num_q_heads=1, initial_blocks=0, local_blocks=1, top_k=1,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE)
    reps = decode(oracle.block_reps(kv, p, 0, 0, 0))
    q = decode(f16(RNG.standard_normal(128)))
    assert oracle.head_block_score(q, reps, synth.REP_QUEST) == pytest.approx(
        float(np.dot(q, decode(k[0, 0, 0]))), rel=1e-12)


def test_multi_rep_score_is_best_rep_dot():
    reps = RNG.standard_normal((4, 128))
    q = RNG.standard_normal(128)
    best = max(float(np.dot(q, r)) for r in reps)
    assert oracle.head_block_score(q, reps, synth.REP_FIX) == pytest.approx(best, rel=1e-12)
    assert oracle.head_block_score(q, reps[:1], synth.REP_MAX) == pytest.approx(
        float(np.dot(q, reps[0])), rel=1e-12)


def _single_head_view(w, hq):
    """Workload of one query head over its own KV head (MHA, 1 head)."""
    G = w.params.num_q_heads // w.num_kv_heads
    h = hq // G
    kv = oracle.KV(w.k_pool[:, h:h + 1].copy(), w.v_pool[:, h:h + 1].copy(), w.block_table,
                   w.seq_lens)
    p = synth.Params(**{**w.params.__dict__, "num_q_heads": 1})
    return kv, np.ascontiguousarray(w.q[:, hq:hq + 1]), p


@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
@pytest.mark.parametrize("rep", [synth.REP_MAX, synth.REP_QUEST, synth.REP_FIX])
def test_unit_score_is_sum_of_single_head_scores(mode, rep):
    # SHARED joins all query heads, SEPARATE the heads of one KV head (§4.5); each
    # single-head score is computed by a 1-head oracle run over that head's own keys.
    w = synth.custom(11, [128 * 9 + 50, 128 * 6], num_q_heads=8, num_kv_heads=2, rep=rep,
                     head_mode=mode, top_k=3)
    multi = oracle.sparse_step(oracle.KV.of(w), w.q, w.params)["unit_scores"]
    G = 4
    singles = []
    for hq in range(8):
        kv1, q1, p1 = _single_head_view(w, hq)
        p1.head_mode = synth.HEAD_SEPARATE
        singles.append(oracle.sparse_step(kv1, q1, p1)["unit_scores"][:, 0])
    singles = np.array(singles)  # [hq][B][MB]
    if mode == synth.HEAD_SHARED:
        want = np.nansum(singles, axis=0)[:, None]
    else:
        want = np.stack([np.nansum(singles[u * G:(u + 1) * G], axis=0) for u in range(2)], 1)
    ctx = ~np.isnan(multi)
    assert np.allclose(multi[ctx], want[ctx], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- selection

def test_select_matches_brute_force_with_ties():
    for trial in range(200):
        C = int(RNG.integers(0, 60))
        k = int(RNG.integers(0, 70))
        s = RNG.integers(0, 6, C).astype(np.float64)  # many exact ties
        c0 = int(RNG.integers(0, 5))
        got = oracle.select(s, c0, k)
        order = sorted(range(C), key=lambda i: (-s[i], i))[:min(k, C)]
        assert list(got) == sorted(c0 + i for i in order)


# --------------------------------------------------------------------------- attention

def test_attend_matches_torch_sdpa_fp64():
    torch = pytest.importorskip("torch")
    kv = small_kv(6, [128 * 3 + 77], H_kv=2)
    q = f16(RNG.standard_normal((4, 128)))
    scale = 1 / math.sqrt(128)
    out = oracle.dense(kv, q[None], 4, scale)[0]
    for hq in range(4):
        h = hq // 2
        K = torch.tensor(logical_keys(kv, 0, h))[None, None]
        V = torch.tensor(logical_values(kv, 0, h))[None, None]
        Q = torch.tensor(decode(q[hq]))[None, None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)
        assert np.allclose(out[hq], ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-14)


def test_attend_hand_worked_d4_n6():
    # d = 4, 6 tokens in blocks of 2, scale 1/2.  q = (2,0,0,0) and key t has
    # first component a_t = (0,0,1,1,2,2), so the logits are a_t and the weights
    # are 1, 1, e, e, e^2, e^2.  V rows are small integers.
    a = [0, 0, 1, 1, 2, 2]
    k = np.zeros((3, 1, 2, 4))
    v = np.zeros((3, 1, 2, 4))
    V = np.array([[1, 2, 3, 4], [5, 6, 7, 8], [-1, 0, 1, 2], [2, 2, 2, 2],
                  [0, 1, 0, 1], [4, -4, 4, -4]], dtype=np.float64)
    for t in range(6):
        k[t // 2, 0, t % 2] = [a[t], 1.0, -1.0, 0.5]
        v[t // 2, 0, t % 2] = V[t]
    kv = oracle.KV(f16(k), f16(v), np.array([[0, 1, 2]], np.int32), [6], block_size=2)
    q = f16([[2.0, 0.0, 0.0, 0.0]])
    out = oracle.attend(kv, 0, 0, 1, q[0], [0, 1, 2], 0.5)
    e = math.e
    want = (V[0] + V[1] + e * (V[2] + V[3]) + e * e * (V[4] + V[5])) / (2 + 2 * e + 2 * e * e)
    assert np.allclose(out, want, rtol=1e-14)
    # a selection of blocks {0, 2} drops the middle pair
    out2 = oracle.attend(kv, 0, 0, 1, q[0], [0, 2], 0.5)
    want2 = (V[0] + V[1] + e * e * (V[4] + V[5])) / (2 + 2 * e * e)
    assert np.allclose(out2, want2, rtol=1e-14)


def test_uniform_logits_give_mean_of_values():
    kv = small_kv(7, [128 * 2 + 5], H_kv=1)
    q = np.zeros((1, 1, 128), dtype=np.uint16)
    out = oracle.dense(kv, q, 1, 1 / math.sqrt(128))[0, 0]
    assert np.allclose(out, logical_values(kv, 0, 0).mean(axis=0), rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- the step

@pytest.mark.parametrize("rep", [synth.REP_MAX, synth.REP_MEAN, synth.REP_QUEST, synth.REP_FIX])
@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_selecting_every_block_is_dense_attention(rep, mode):
    w = synth.custom(8, [128 * 7 + 3, 128 * 5], num_q_heads=4, num_kv_heads=2, rep=rep,
                     head_mode=mode, top_k=100)
    kv = oracle.KV.of(w)
    r = oracle.sparse_step(kv, w.q, w.params)
    dense = oracle.dense(kv, w.q, 4, w.params.softmax_scale)
    assert np.allclose(r["out"], dense, rtol=1e-12, atol=1e-14)


def test_initial_and_local_always_attended():
    w = synth.custom(9, [128 * 20 + 9, 128 * 11, 128 * 3], num_q_heads=4, num_kv_heads=2,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE, top_k=3,
                     initial_blocks=2, local_blocks=3)
    kv = oracle.KV.of(w)
    r = oracle.sparse_step(kv, w.q, w.params)
    for b, n in enumerate(w.seq_lens):
        nb, c0, c1 = oracle.partition(int(n), 2, 3)
        for u in range(2):
            cnt = r["cnt"][b, u]
            sel = r["sel"][b, u, :cnt]
            assert cnt == min(3, c1 - c0)
            assert np.all((sel >= c0) & (sel < c1)) and np.all(np.diff(sel) > 0)
            blocks = list(range(c0)) + list(sel) + list(range(c1, nb))
            for g in range(2):
                hq = u * 2 + g
                want = oracle.attend(kv, b, hq, 4, w.q[b, hq], blocks, w.params.softmax_scale)
                assert np.allclose(r["out"][b, hq], want, rtol=1e-13, atol=1e-15)


def test_block_size_one_with_max_reps_is_exact_topk_logits():
    # §4.5: block_size 1 turns block selection into token selection; with a Max rep
    # of one token the block score is q.k, so selection is the top-k logits.
    n, d = 300, 16
    k = f16(RNG.standard_normal((n, 1, 1, d)))
    kv = oracle.KV(k, k, np.arange(n, dtype=np.int32)[None], [n], block_size=1)
    p = synth.Params(num_q_heads=1, initial_blocks=0, local_blocks=1, top_k=25,
                     rep=synth.REP_MAX, head_mode=synth.HEAD_SEPARATE)
    q = f16(RNG.standard_normal((1, 1, d)))
    r = oracle.sparse_step(kv, q, p)
    logits = decode(k[:, 0, 0]) @ decode(q[0, 0])
    ctx = np.arange(n - 1)
    top = sorted(ctx, key=lambda t: (-logits[t], t))[:25]
    assert list(r["sel"][0, 0, :r["cnt"][0, 0]]) == sorted(top)


def test_planted_blocks_are_selected_by_every_head():
    w = synth.tiny()
    r = oracle.sparse_step(oracle.KV.of(w), w.q, w.params)
    planted = {j for _, j in w.needles}
    assert len(planted) == 3
    for u in range(8):
        assert planted <= set(r["sel"][0, u, :r["cnt"][0, u]].tolist())


# --------------------------------------------------------------------------- dynamic

def test_dynamic_scores_with_one_query_rank_tokens_by_logit():
    # T = 1 and G = 1: the accumulated score is one softmax row, so the 4 reps of
    # each block are its 4 largest logits (ties: lower index), in token order.
    w = synth.custom(10, [128 * 4], num_q_heads=1, num_kv_heads=1, rep=synth.REP_DYNAMIC,
                     num_reps=4, local_queries=1, local_blocks=1, initial_blocks=0)
    kv = oracle.KV.of(w)
    acc = oracle.dynamic_token_scores(kv, w.params, 0, 0, w.q_local[0])
    K = logical_keys(kv, 0, 0)
    logits = K @ decode(w.q_local[0, 0, 0])
    assert abs(acc.sum() - 1.0) < 1e-12
    for j in range(4):
        reps = oracle.block_reps(kv, w.params, 0, j, 0, dyn_scores=acc)
        blk = list(range(j * 128, (j + 1) * 128))
        top = sorted(sorted(blk, key=lambda t: (-logits[t], t))[:4])
        page = kv.block_table[0, j]
        assert np.array_equal(reps, kv.k_pool[page, 0, [t - j * 128 for t in top]])


def test_dynamic_scores_zero_queries_closed_form():
    # q = 0: each query position pos spreads weight 1/(pos+1) over tokens 0..pos,
    # so acc[t] = G * sum over the T positions pos >= t of 1/(pos + 1).
    n, T, G = 300, 5, 2
    w = synth.custom(12, [n], num_q_heads=2, num_kv_heads=1, rep=synth.REP_DYNAMIC,
                     local_queries=T)
    kv = oracle.KV.of(w)
    ql = np.zeros_like(w.q_local[0])
    acc = oracle.dynamic_token_scores(kv, w.params, 0, 0, ql)
    pos = np.arange(n - T, n)
    want = np.array([G * sum(1.0 / (p + 1) for p in pos if p >= t) for t in range(n)])
    assert np.allclose(acc, want, rtol=1e-12)
    assert acc.sum() == pytest.approx(T * G, rel=1e-12)


# --------------------------------------------------------------------------- preselection

@pytest.mark.parametrize("k", [1, 3, 5])
def test_avg_pool_closed_forms(k):
    # a unit impulse spreads 1/k over the k positions around it; a constant c
    # stays c where the window fits and loses the padded part at the ends
    n, c = 23, 2.5
    x = np.zeros(n)
    x[10] = 1.0
    got = oracle.avg_pool1d(x, k)
    want = np.zeros(n)
    want[10 - k // 2:10 + k // 2 + 1] = 1.0 / k
    assert np.allclose(got, want, rtol=0, atol=1e-15)
    got = oracle.avg_pool1d(np.full(n, c), k)
    inside = [min(k, t + k // 2 + 1, n - t + k // 2) for t in range(n)]
    assert np.allclose(got, c * np.array(inside) / k, rtol=1e-15)


def test_preselect_one_query_no_pooling_is_top_blocks_by_max_logit():
    # T = 1, G = 1, kernel 1: the vote is one softmax row over the tokens the
    # last query sees, monotone in the logit, so the preselected blocks are the
    # context blocks with the largest maximum logit (ties: lower block)
    n = 128 * 12 + 40
    w = synth.custom(41, [n], num_q_heads=1, num_kv_heads=1, rep=synth.REP_QUEST,
                     local_queries=1, initial_blocks=1, local_blocks=2)
    kv = oracle.KV.of(w)
    presel, pcnt = oracle.preselect(kv, w.params, w.q_local, kernel=1, count=4)
    K = logical_keys(kv, 0, 0)
    logits = K @ decode(w.q_local[0, 0, 0])
    nb = (n + 127) // 128
    c0, c1 = 1, nb - 2
    best = {j: logits[j * 128:(j + 1) * 128].max() for j in range(c0, c1)}
    want = sorted(sorted(best, key=lambda j: (-best[j], j))[:4])
    assert pcnt[0, 0] == 4 and list(presel[0, 0]) == want


def test_preselect_count_covers_all_context_blocks():
    w = synth.custom(42, [128 * 9 + 5, 128 * 6], num_q_heads=4, num_kv_heads=2,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE, local_queries=8,
                     initial_blocks=1, local_blocks=2)
    kv = oracle.KV.of(w)
    presel, pcnt = oracle.preselect(kv, w.params, w.q_local, kernel=5, count=64)
    for b, n in enumerate(w.seq_lens):
        nb = (int(n) + 127) // 128
        ctx = list(range(1, nb - 2))
        for u in range(2):
            assert pcnt[b, u] == len(ctx)
            assert list(presel[b, u, :len(ctx)]) == ctx


def test_step_restricted_to_everything_equals_unrestricted_step():
    w = synth.custom(43, [128 * 20 + 7, 128 * 11], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SHARED, top_k=3,
                     local_queries=4)
    kv = oracle.KV.of(w)
    ref = oracle.sparse_step(kv, w.q, w.params, w.q_local)
    presel, pcnt = oracle.preselect(kv, w.params, w.q_local, kernel=3, count=1000)
    got = oracle.sparse_step_presel(kv, w.q, w.params, presel, pcnt, w.q_local)
    assert np.array_equal(got["sel"], ref["sel"]) and np.array_equal(got["cnt"], ref["cnt"])
    assert np.array_equal(got["out"], ref["out"])


def test_step_restricted_selection_is_top_k_of_the_preselection():
    w = synth.custom(44, [128 * 30 + 3], num_q_heads=8, num_kv_heads=2, rep=synth.REP_MAX,
                     head_mode=synth.HEAD_SEPARATE, top_k=3, local_queries=4)
    kv = oracle.KV.of(w)
    presel, pcnt = oracle.preselect(kv, w.params, w.q_local, kernel=5, count=6)
    got = oracle.sparse_step_presel(kv, w.q, w.params, presel, pcnt, w.q_local)
    for u in range(2):
        cand = presel[0, u, :pcnt[0, u]]
        sc = got["unit_scores"][0, u]
        want = sorted(sorted(cand, key=lambda j: (-sc[j], j))[:3])
        assert got["cnt"][0, u] == 3 and list(got["sel"][0, u, :3]) == want


def test_score_select_attend_over_own_reps_is_the_step():
    # the entry that takes representative values reproduces the step when
    # given the oracle's own reps (Quest, SEPARATE, ragged batch)
    w = synth.custom(45, [128 * 14 + 9, 128 * 8], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE, top_k=3)
    kv = oracle.KV.of(w)
    ref = oracle.sparse_step(kv, w.q, w.params)
    R = w.params.reps_per_block()
    rv = np.zeros((w.batch, w.max_blocks, 2, R, 128))
    for b in range(w.batch):
        for j in range(int(w.seq_lens[b]) // 128):
            rv[b, j] = decode(ref["reps"][b, j])
    got = oracle.score_select_attend(kv, w.q, w.params, rv)
    assert np.array_equal(got["sel"], ref["sel"]) and np.array_equal(got["cnt"], ref["cnt"])
    assert np.array_equal(got["out"], ref["out"])
