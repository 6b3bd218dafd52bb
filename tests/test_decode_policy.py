"""Selection reuse while decoding ([LC §4.5] token_step / layer_step /
dense_layer_num, [LC §4.6] decode loop): the oracle's action function pinned
to the decode loop's reuse rule, and the library's host-side policy checked
against it (no GPU work)."""
import itertools

import pytest

import oracle

DENSE, SELECT, REUSE = oracle.LAYER_DENSE, oracle.LAYER_SELECT, oracle.LAYER_REUSE


def decode_loop_rule(num_tokens, num_layers, lstride, tstride):
    """The reuse rule of the decode loop of [LC §4.6] (no dense layers),
    restated: every layer group g = layer // lstride keeps one stored
    selection; a (token, layer) pair makes a new one, and stores it for its
    group, exactly when the token is a multiple of tstride and the layer a
    multiple of lstride; every other pair reuses its group's.  Returns the
    (action, slot) sequence in decode order and checks that no group is read
    before it was stored."""
    stored = set()
    seq = []
    for tok in range(num_tokens):
        for lay in range(num_layers):
            group = lay // lstride
            fresh = tok % tstride == 0 and lay % lstride == 0
            if fresh:
                stored.add(group)
            else:
                assert group in stored
            seq.append((SELECT if fresh else REUSE, group))
    return seq


@pytest.mark.parametrize("layers,lstep,tstep", [(1, 1, 1), (4, 1, 1), (4, 2, 1), (5, 2, 3),
                                               (32, 1, 100), (7, 7, 2), (6, 4, 1)])
def test_action_matches_the_decode_loop_rule(layers, lstep, tstep):
    tokens = 2 * tstep + 1
    want = decode_loop_rule(tokens, layers, lstep, tstep)
    got = [oracle.decode_layer_action(layers, 0, lstep, tstep, t, l)
           for t in range(tokens) for l in range(layers)]
    assert got == want


def test_worked_cases():
    # the YAML of [HOWTO] Step 3: layer_step 1, token_step 100
    assert oracle.decode_layer_action(32, 0, 1, 100, 0, 5) == (SELECT, 5)
    assert oracle.decode_layer_action(32, 0, 1, 100, 99, 5) == (REUSE, 5)
    assert oracle.decode_layer_action(32, 0, 1, 100, 100, 5) == (SELECT, 5)
    # two dense layers (the 2 of [LC §5.2] / the YAML's dense_layer_num)
    assert oracle.decode_layer_action(32, 2, 1, 100, 0, 0) == (DENSE, -1)
    assert oracle.decode_layer_action(32, 2, 1, 100, 7, 1) == (DENSE, -1)
    assert oracle.decode_layer_action(32, 2, 1, 100, 0, 2) == (SELECT, 0)
    # layer_step 2 after 1 dense layer: layers 1-2 share slot 0, 3-4 slot 1
    acts = [oracle.decode_layer_action(5, 1, 2, 1, 0, l) for l in range(5)]
    assert acts == [(DENSE, -1), (SELECT, 0), (REUSE, 0), (SELECT, 1), (REUSE, 1)]


def test_every_slot_is_written_before_it_is_read():
    for layers, dense, lstep, tstep in itertools.product([1, 3, 8], [0, 1, 3], [1, 2, 3],
                                                         [1, 2, 5]):
        if dense > layers:
            continue
        written = set()
        for t in range(2 * tstep + 1):
            for l in range(layers):
                a, s = oracle.decode_layer_action(layers, dense, lstep, tstep, t, l)
                if a == SELECT:
                    written.add(s)
                elif a == REUSE:
                    assert s in written
                else:
                    assert l < dense and s == -1


def test_selection_count_over_a_window():
    # selections per token window = number of slots (one per layer group),
    # and a window of token_step tokens selects once per slot
    layers, dense, lstep, tstep = 10, 2, 3, 4
    slots = -(-(layers - dense) // lstep)
    n_sel = sum(oracle.decode_layer_action(layers, dense, lstep, tstep, t, l)[0] == SELECT
                for t in range(tstep) for l in range(layers))
    assert n_sel == slots


def test_invalid_policies_rejected():
    for args in [(0, 0, 1, 1, 0, 0), (4, 5, 1, 1, 0, 0), (4, 0, 0, 1, 0, 0), (4, 0, 1, 0, 0, 0),
                 (4, 0, 1, 1, -1, 0), (4, 0, 1, 1, 0, 4)]:
        with pytest.raises(ValueError):
            oracle.decode_layer_action(*args)


# ---- the library's host-side policy (libkt.so loads without a GPU) ----------

def test_library_policy_matches_the_oracle():
    kt = pytest.importorskip("block_sparse_long_quest_gb300")
    for layers, dense, lstep, tstep in itertools.product([1, 2, 5, 9], [0, 1, 2], [1, 2, 4],
                                                         [1, 3]):
        if dense > layers:
            continue
        pol = kt.reuse_policy(layers, dense, lstep, tstep)
        assert kt.kt_decode_history_slots(pol) == -(-(layers - dense) // lstep)
        for t in range(2 * tstep + 1):
            for l in range(layers):
                assert kt.kt_decode_layer_action(pol, t, l) == \
                    oracle.decode_layer_action(layers, dense, lstep, tstep, t, l)


def test_library_rejects_invalid_policies():
    kt = pytest.importorskip("block_sparse_long_quest_gb300")
    for bad in [(0, 0, 1, 1), (4, 5, 1, 1), (4, 0, 0, 1), (4, 0, 1, 0)]:
        pol = kt.reuse_policy(*bad)
        with pytest.raises(kt.KtError):
            kt.kt_decode_history_slots(pol)
        with pytest.raises(kt.KtError):
            kt.kt_decode_layer_action(pol, 0, 0)
    pol = kt.reuse_policy(4, 0, 1, 1)
    for t, l in [(-1, 0), (0, -1), (0, 4)]:
        with pytest.raises(kt.KtError):
            kt.kt_decode_layer_action(pol, t, l)


# ---- the oracle's attention over a stored selection --------------------------

@pytest.mark.parametrize("head_mode", [oracle.HEAD_SEPARATE, oracle.HEAD_SHARED])
def test_attention_over_a_stored_selection_is_the_step_on_its_own_selection(head_mode):
    import numpy as np

    import synth
    w = synth.custom(71, [128 * 9 + 40, 128 * 6], num_q_heads=4, num_kv_heads=2, top_k=3,
                     head_mode=head_mode)
    kv = oracle.KV.of(w)
    ref = oracle.sparse_step(kv, w.q, w.params)
    got = oracle.attend_selection(kv, w.q, w.params, ref["sel"], ref["cnt"])
    assert np.allclose(got, ref["out"], rtol=1e-12, atol=1e-15)
    # a different selection gives a different result (the ids are used)
    sel2 = ref["sel"].copy()
    sel2[0, 0, 0] = next(j for j in range(1, 9) if j not in set(ref["sel"][0, 0].tolist()))
    sel2[0, 0].sort()
    other = oracle.attend_selection(kv, w.q, w.params, sel2, ref["cnt"])
    assert not np.allclose(other[0], got[0])
