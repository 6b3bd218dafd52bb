"""GPU parity of the Dynamic representative build (accumulated softmax scores of
the last T queries; the best tokens of each block) against the oracle, and of
the decode step over Dynamic reps."""
import numpy as np
import pytest

import oracle
import synth
from kt_testlib import (DevWorkload, build_dynamic, check_dynamic_reps, check_units,
                        rep_values_of_gpu_tokens)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300  # noqa: F401


@pytest.mark.parametrize("G,T,R", [(1, 1, 4), (4, 16, 4), (2, 7, 3), (4, 64, 4), (8, 32, 1)])
def test_dynamic_token_scores_and_reps(G, T, R):
    lens = [128 * 9 + 50, 128 * 6, 40, 128 * 3 + 1]
    w = synth.custom(51, lens, num_q_heads=2 * G, num_kv_heads=2, rep=synth.REP_DYNAMIC,
                     num_reps=R, local_queries=T, top_k=3)
    dw = DevWorkload(w)
    got = build_dynamic(dw)
    ref = oracle.sparse_step(oracle.KV.of(w), w.q, w.params, w.q_local, want_dyn_scores=True)
    for b, n in enumerate(w.seq_lens):
        for h in range(2):
            r = ref["dyn_scores"][b, h, :n]
            g = got[b, h, :n]
            assert np.abs(g - r).max() <= 1e-4 * max(r.max(), 1e-30)
    checked, differ, bad = check_dynamic_reps(dw, ref["dyn_scores"])
    assert checked > 0 and not bad, bad[:3]


@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_dynamic_full_step_selection_and_output(mode):
    """Every block's reps are checked against the oracle's token scores (a
    token inside the 1e-5 zone of the block's cut may stand in for another);
    the oracle then scores the blocks with the reps the GPU chose, and every
    unit's selection and output is compared (check_units).  When no rep
    differs, that is exactly the oracle's own step."""
    w = synth.custom(52, [128 * 40 + 17, 128 * 25], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_DYNAMIC, num_reps=4, local_queries=16, top_k=5,
                     head_mode=mode, num_needles=2)
    dw = DevWorkload(w)
    build_dynamic(dw)
    kv = oracle.KV.of(w)
    own = oracle.sparse_step(kv, w.q, w.params, w.q_local, want_dyn_scores=True)
    checked, differ, bad = check_dynamic_reps(dw, own["dyn_scores"])
    assert checked > 0 and not bad, bad[:3]
    ref = oracle.score_select_attend(kv, w.q, w.params, rep_values_of_gpu_tokens(w, dw))
    if differ == 0:
        assert np.array_equal(ref["sel"], own["sel"]) and np.array_equal(ref["cnt"], own["cnt"])
    sel, cnt, out, ws = dw.step()
    exact, zone = check_units(w, kv, sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy(),
                              ref, (0, dw.SEL))
    assert exact + zone == w.batch * dw.SEL
