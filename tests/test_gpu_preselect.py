"""GPU parity of the preselection [LC §4.4, §4.6 preselect_block()] and of the
selection restricted to it, against the oracle.

The preselected set must equal the oracle's except for blocks whose score
(largest pooled vote) lies within 1e-5 of the count-th score; the restricted
step is checked on the oracle's own preselection, so its parity does not
depend on those near-ties.
"""
import numpy as np
import pytest

import oracle
import synth
from kt_testlib import TOL, ZONE, DevWorkload, row_rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300  # noqa: F401


def _block_scores(w, kernel):
    """Oracle block scores per unit: largest pooled vote of each Context block."""
    kv = oracle.KV.of(w)
    p = w.params
    SEL = 1 if p.head_mode == synth.HEAD_SHARED else w.num_kv_heads
    out = {}
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        nb = (n + 127) // 128
        c0 = min(p.initial_blocks, nb)
        c1 = max(c0, nb - p.local_blocks)
        per_head = [oracle.dynamic_token_scores(kv, p, b, h, w.q_local[b])
                    for h in range(w.num_kv_heads)]
        for u in range(SEL):
            heads = range(w.num_kv_heads) if SEL == 1 else [u]
            vote = sum(per_head[h][c0 * 128:c1 * 128] for h in heads)
            pooled = oracle.avg_pool1d(vote, kernel)
            out[b, u] = (c0, pooled.reshape(-1, 128).max(axis=1) if c1 > c0 else np.zeros(0))
    return out


def _mask_to_sets(mask, SEL, B):
    mask = mask.cpu().numpy().astype(np.uint32)
    sets = {}
    for b in range(B):
        for u in range(SEL):
            bits = np.unpackbits(mask[b, u].view(np.uint8), bitorder="little")
            sets[b, u] = set(np.nonzero(bits)[0].tolist())
    return sets


def _gpu_preselect(dw, kernel, count):
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = dw.w
    T = w.q_local.shape[1]
    mw = kt.kt_preselect_mask_words(dw.kv)
    mask = torch.full((w.batch, dw.SEL, mw), -1, dtype=torch.int32, device="cuda")  # all bits
    cnt = torch.full((w.batch, dw.SEL), -1, dtype=torch.int32, device="cuda")
    ws = kt.workspace(kt.KT_OP_PRESELECT, dw.kv, dw.params, T)
    kt.kt_preselect_blocks(dw.kv, dw.params, dw.q_local, T, kernel, count, mask, cnt, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    return mask, cnt


@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
@pytest.mark.parametrize("kernel,count", [(1, 4), (5, 6), (13, 40)])
def test_preselection_matches_oracle(mode, kernel, count):
    w = synth.custom(61, [128 * 40 + 17, 128 * 23, 128 * 3], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_QUEST, head_mode=mode, top_k=3, local_queries=8,
                     initial_blocks=1, local_blocks=2)
    dw = DevWorkload(w)
    mask, cnt = _gpu_preselect(dw, kernel, count)
    presel, pcnt = oracle.preselect(oracle.KV.of(w), w.params, w.q_local, kernel, count)
    assert np.array_equal(cnt.cpu().numpy(), pcnt)
    got = _mask_to_sets(mask, dw.SEL, w.batch)
    scores = _block_scores(w, kernel)
    for (b, u), g in got.items():
        want = set(presel[b, u, :pcnt[b, u]].tolist())
        if g == want:
            continue
        c0, sc = scores[b, u]
        sk = np.sort(sc)[::-1][pcnt[b, u] - 1]
        for j in g.symmetric_difference(want):
            assert abs(sc[j - c0] - sk) <= ZONE * abs(sk), (b, u, j)


def _mask_from_lists(presel, pcnt, mw):
    B, SEL, _ = presel.shape
    mask = np.zeros((B, SEL, mw), dtype=np.uint32)
    for b in range(B):
        for u in range(SEL):
            for j in presel[b, u, :pcnt[b, u]]:
                mask[b, u, j // 32] |= np.uint32(1) << np.uint32(j % 32)
    return mask


def _restricted_agrees(sel, cnt, ref, presel, pcnt, b, u):
    c = int(ref["cnt"][b, u])
    if int(cnt[b, u]) != c:
        return False, False
    got = sel[b, u, :c].tolist()
    if got != sorted(got) or len(set(got)) != c:
        return False, False
    want = ref["sel"][b, u, :c].tolist()
    if got == want:
        return True, True
    sc = ref["unit_scores"][b, u]
    cand = presel[b, u, :pcnt[b, u]]
    sk = np.sort(sc[cand])[::-1][c - 1]
    for j in set(got).symmetric_difference(want):
        if j not in cand or abs(sc[j] - sk) > ZONE * abs(sk):
            return False, False
    return True, False


@pytest.mark.parametrize("rep", [synth.REP_QUEST, synth.REP_MAX, synth.REP_FIX])
@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
@pytest.mark.parametrize("count", [2, 9])
@pytest.mark.parametrize("cap", [0, 8])
def test_step_restricted_to_preselection(rep, mode, count, cap):
    # count 2 < top_k: every preselected block is chosen; count 9: top 4 of 9.
    # cap 8: eight CTAs, so a scoring slice holds more blocks than its slots
    # and publishes through the threshold search over its unmasked keys
    import block_sparse_long_quest_gb300 as kt
    kt.kt_set_max_ctas(cap)
    try:
        _restricted_step_case(rep, mode, count)
    finally:
        kt.kt_set_max_ctas(0)


def _restricted_step_case(rep, mode, count):
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(62, [128 * 37 + 29, 128 * 20 + 100, 300], num_q_heads=8, num_kv_heads=2,
                     rep=rep, head_mode=mode, top_k=4, local_queries=4, fix_stride=32)
    kv = oracle.KV.of(w)
    presel, pcnt = oracle.preselect(kv, w.params, w.q_local, 5, count)
    ref = oracle.sparse_step_presel(kv, w.q, w.params, presel, pcnt, w.q_local)
    dw = DevWorkload(w)
    dw.build_reps()
    mw = kt.kt_preselect_mask_words(dw.kv)
    mask = to_dev(_mask_from_lists(presel, pcnt, mw).view(np.int32))
    pc = to_dev(pcnt)
    B, SEL, k = w.batch, dw.SEL, w.params.top_k
    for path in ("step", "select"):
        sel = torch.full((B, SEL, k), -1, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, SEL), -1, dtype=torch.int32, device="cuda")
        ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
        if path == "step":
            out = torch.full((B, w.params.num_q_heads, 128), float("nan"), device="cuda")
            kt.kt_sparse_decode_step_presel(dw.q, dw.kv, dw.reps, dw.params, mask, pc, sel, cnt,
                                            out, ws)
        else:
            kt.kt_score_select_blocks_presel(dw.q, dw.kv, dw.reps, dw.params, mask, sel, cnt,
                                             None, ws)
            out, _ = dw.attend(sel, cnt, ws)
        assert kt.kt_read_device_status(ws) == kt.KT_OK
        s_, c_, o_ = sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
        G = w.params.num_q_heads // w.num_kv_heads
        for b in range(B):
            for u in range(SEL):
                ok, exact = _restricted_agrees(s_, c_, ref, presel, pcnt, b, u)
                assert ok, (path, b, u, s_[b, u], ref["sel"][b, u])
                if exact:
                    hs = list(range(w.params.num_q_heads)) if SEL == 1 else list(range(u * G, (u + 1) * G))
                    assert row_rel_err(o_[b, hs], ref["out"][b, hs]).max() <= TOL


def test_preselect_then_restricted_step_end_to_end():
    # the library's own preselection feeds the restricted one-launch step
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(63, [128 * 60 + 5], num_q_heads=16, num_kv_heads=4, rep=synth.REP_QUEST,
                     head_mode=synth.HEAD_SEPARATE, top_k=4, local_queries=8)
    dw = DevWorkload(w)
    dw.build_reps()
    mask, pcnt = _gpu_preselect(dw, 5, 12)
    sel = torch.full((1, 4, 4), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((1, 4), -1, dtype=torch.int32, device="cuda")
    out = torch.zeros((1, 16, 128), device="cuda")
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
    kt.kt_sparse_decode_step_presel(dw.q, dw.kv, dw.reps, dw.params, mask, pcnt, sel, cnt, out, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    sets = _mask_to_sets(mask, 4, 1)
    s_, c_ = sel.cpu().numpy(), cnt.cpu().numpy()
    for u in range(4):
        assert c_[0, u] == 4
        assert set(s_[0, u].tolist()) <= sets[0, u]
