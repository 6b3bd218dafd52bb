"""GPU parity of decoding over several layers and tokens with selection reuse
([LC §4.5] token_step / layer_step / dense_layer_num, [LC §4.6] decode loop)
and of the token append, against the oracle.

Every (token, layer) takes the oracle's action.  A fresh selection must agree
with the oracle's (near-ties as in the other parity tests); an attention over a
stored selection is compared with the oracle's attention over the same stored
block ids at the current lengths.  The pools start with room for the appended
tokens, so the appends complete blocks and move the Local window forward
(Context grows under a reused selection).
"""
import numpy as np
import pytest

import oracle
import synth
from kt_testlib import TOL, DevWorkload, check_reps, row_rel_err, selection_agrees, to_dev

pytestmark = pytest.mark.gpu

CAP = [128 * 7 + 2, 128 * 10 + 3]    # pages allocated for these lengths
START = [128 * 7 - 2, 128 * 10 - 1]  # lengths when decoding starts
TOKENS = 5                           # decode steps; an append after each but the last


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300  # noqa: F401


def _layer(l, rep, head_mode):
    p = synth.Params(num_q_heads=8, initial_blocks=1, local_blocks=2, top_k=3, rep=rep,
                     head_mode=head_mode, num_reps=4 if rep == synth.REP_FIX else 1,
                     fix_stride=32)
    w = synth.make_workload(f"decode-l{l}", seed=61, seq_lens=CAP, num_q_heads=8,
                            num_kv_heads=2, params=p, layer=l, permute_pages=True)
    w.seq_lens = np.asarray(START, dtype=np.int32)
    return w


@pytest.mark.parametrize("rep,head_mode", [(synth.REP_QUEST, synth.HEAD_SEPARATE),
                                           (synth.REP_MAX, synth.HEAD_SHARED),
                                           (synth.REP_MEAN, synth.HEAD_SEPARATE),
                                           (synth.REP_FIX, synth.HEAD_SHARED)])
def test_decode_loop_with_reuse_and_append(rep, head_mode):
    import torch
    import block_sparse_long_quest_gb300 as kt
    L, dense, lstep, tstep = 3, 1, 2, 2
    pol = kt.reuse_policy(L, dense, lstep, tstep)
    slots = kt.kt_decode_history_slots(pol)
    layers = [_layer(l, rep, head_mode) for l in range(L)]
    devs = [DevWorkload(w) for w in layers]
    for dw in devs:
        dw.build_reps()
    B, H_q, H_kv, k = len(START), 8, 2, 3
    SEL = devs[0].SEL
    hist_sel = torch.full((slots, B, SEL, k), -1, dtype=torch.int32, device="cuda")
    hist_cnt = torch.zeros((slots, B, SEL), dtype=torch.int32, device="cuda")
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, devs[0].kv, devs[0].params)
    seen = set()
    for t in range(TOKENS):
        for l, (w, dw) in enumerate(zip(layers, devs)):
            q = synth.normal_f16((B, H_q, 128), 62 + t, 900 + l)
            q_dev = to_dev(q)
            out = torch.full((B, H_q, 128), float("nan"), dtype=torch.float32, device="cuda")
            before = (hist_sel.clone(), hist_cnt.clone())
            kt.kt_decode_layer(pol, t, l, q_dev, dw.kv, dw.reps, dw.params, hist_sel, hist_cnt,
                               out, ws)
            action, slot = oracle.decode_layer_action(L, dense, lstep, tstep, t, l)
            assert kt.kt_decode_layer_action(pol, t, l) == (action, slot)
            seen.add(action)
            kv = oracle.KV.of(w)
            got = out.cpu().numpy()
            if action == oracle.LAYER_DENSE:
                want = oracle.dense(kv, q, H_q, w.params.softmax_scale)
            else:
                sel = hist_sel[slot].cpu().numpy()
                cnt = hist_cnt[slot].cpu().numpy()
                if action == oracle.LAYER_SELECT:
                    ref = oracle.sparse_step(kv, q, w.params)
                    for b in range(B):
                        for u in range(SEL):
                            assert selection_agrees(sel, cnt, ref, b, u)[0]
                else:
                    # the stored selection is read, not rewritten
                    assert torch.equal(before[0], hist_sel) and torch.equal(before[1], hist_cnt)
                want = oracle.attend_selection(kv, q, w.params, sel, cnt)
            assert row_rel_err(got, want).max() <= TOL, (t, l, action)
        if t + 1 < TOKENS:
            for l, (w, dw) in enumerate(zip(layers, devs)):
                kn = synth.normal_f16((B, H_kv, 128), 63 + t, 900 + l)
                vn = synth.normal_f16((B, H_kv, 128), 64 + t, 900 + l)
                kt.kt_append_kv(dw.kv, dw.params, to_dev(kn), to_dev(vn), dw.reps, ws)
                for b in range(B):
                    n = int(w.seq_lens[b])
                    page = w.block_table[b, n // 128]
                    w.k_pool[page, :, n % 128, :] = kn[b]
                    w.v_pool[page, :, n % 128, :] = vn[b]
                    w.seq_lens[b] = n + 1
    assert seen == {oracle.LAYER_DENSE, oracle.LAYER_SELECT, oracle.LAYER_REUSE}
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    # the appended rows, the lengths and the reps of the completed blocks
    for w, dw in zip(layers, devs):
        assert np.array_equal(dw.lens.cpu().numpy(), w.seq_lens)
        assert np.array_equal(dw.k.cpu().numpy().view(np.uint16), w.k_pool)
        assert np.array_equal(dw.v.cpu().numpy().view(np.uint16), w.v_pool)
        ref = oracle.sparse_step(oracle.KV.of(w), w.q, w.params)
        assert check_reps(dw, ref["reps"]) == 0


def test_append_without_room_is_flagged():
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(65, [128 * 3], num_q_heads=4, num_kv_heads=2, top_k=1)  # table full
    dw = DevWorkload(w)
    dw.build_reps()
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    kn = to_dev(synth.normal_f16((1, 2, 128), 66, 1))
    k_before = dw.k.clone()
    kt.kt_append_kv(dw.kv, dw.params, kn, kn, dw.reps, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_ERR_DEVICE_CHECK
    assert int(dw.lens.cpu()[0]) == 128 * 3
    assert torch.equal(k_before, dw.k)
