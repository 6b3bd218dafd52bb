"""Parity at the workloads' full sizes, through kt_sparse_decode_step (the call
bench.py times), against the oracle on sampled outputs: all reps, and the
selection and attention output of the sampled selection units.

Sizes: 128K tokens (32/8 heads, SHARED), 1M tokens (SEPARATE; KV heads 0-1
checked), 16 paged sequences of 8K-64K tokens (every rep method and head mode),
and the Dynamic 128K layer (KV head 0's token scores and reps).
"""
import numpy as np
import pytest

import oracle
import synth
from kt_testlib import (TOL, DevWorkload, build_dynamic, check_dynamic_reps, check_reps,
                        row_rel_err, selection_agrees)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300  # noqa: F401


def _check_step(w, dw, units):
    """Selection + output of the given units against the oracle."""
    import block_sparse_long_quest_gb300 as kt
    sel, cnt, out, ws = dw.step()
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    ref = oracle.sparse_step(oracle.KV.of(w), w.q, w.params, w.q_local, units=units)
    if w.params.rep != synth.REP_DYNAMIC:
        # reps of the sampled units' KV heads, bit for bit
        got = dw.reps_view()
        R = w.params.reps_per_block()
        heads = range(w.num_kv_heads) if w.params.head_mode == synth.HEAD_SHARED \
            else range(units[0], units[1])
        for b in range(w.batch):
            for j in range(int(w.seq_lens[b]) // 128):
                for h in heads:
                    a = got[w.block_table[b, j], h]
                    r = ref["reps"][b, j, h]
                    if w.params.rep == synth.REP_MEAN:
                        assert np.array_equal(a.reshape(-1).view(np.uint32),
                                              r.reshape(-1).view(np.uint32))
                    else:
                        assert np.array_equal(a, r.reshape(R, 128)), (b, j, h)
    sel, cnt, out = sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
    G = w.params.num_q_heads // w.num_kv_heads
    compared = 0
    for b in range(w.batch):
        for u in range(units[0], units[1]):
            ok, exact = selection_agrees(sel, cnt, ref, b, u)
            assert ok, (b, u, sel[b, u], ref["sel"][b, u])
            if exact:
                heads = range(w.params.num_q_heads) if w.params.head_mode == synth.HEAD_SHARED \
                    else range(u * G, (u + 1) * G)
                err = row_rel_err(out[b, list(heads)], ref["out"][b, list(heads)])
                assert err.max() <= TOL, err.max()
                compared += 1
    assert compared > 0
    return ref


def test_128k_shared_quest_full_size():
    import block_sparse_long_quest_gb300 as kt
    w = synth.long128k()
    dw = DevWorkload(w)
    dw.build_reps()
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
    _check_step(w, dw, (0, 1))


@pytest.mark.parametrize("rep", [synth.REP_QUEST, synth.REP_MAX, synth.REP_FIX])
def test_1m_separate_full_size_sampled_heads(rep):
    w = synth.long1m(rep=rep)
    dw = DevWorkload(w)
    dw.build_reps()
    _check_step(w, dw, (0, 2))


@pytest.mark.parametrize("rep", [synth.REP_MAX, synth.REP_MEAN, synth.REP_QUEST, synth.REP_FIX])
@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_batched_paged_full_size(rep, mode):
    w = synth.batched(rep=rep, head_mode=mode)
    dw = DevWorkload(w)
    dw.build_reps()
    units = (0, 1) if mode == synth.HEAD_SHARED else (0, 8)
    _check_step(w, dw, units)


def test_dynamic_128k_full_size_head0():
    w = synth.dynamic128k()
    dw = DevWorkload(w)
    got = build_dynamic(dw)
    kv = oracle.KV.of(w)
    ref0 = oracle.dynamic_token_scores(kv, w.params, 0, 0, w.q_local[0])
    assert np.abs(got[0, 0, :ref0.size] - ref0).max() <= 1e-4 * ref0.max()
    # reps of KV head 0 for every full block, against the oracle's choice
    scores = np.zeros((1, w.num_kv_heads, w.max_blocks * 128))
    scores[0, 0, :ref0.size] = ref0
    checked, differ, bad = check_dynamic_reps(dw, scores, heads=[0])
    assert checked == 1024 and not bad, bad[:3]
