"""GPU-internal consistency of the decode path (no oracle needed for the
comparison itself, though each output is also checked against the oracle):

* split-count invariance: the split-K partition of a segment across CTAs
  (kt_set_max_ctas forces 1, 2, 7 or the default one-per-SM CTAs per segment)
  changes only the grouping of the fp32 sums, so outputs agree within 64
  binary32 units in the last place (2^-18, normwise per row), and
  in the one-launch step the scoring slices change without changing the
  selection outside the near-tie zone;
* paged vs identity block table: the same logical KV stored in randomly
  permuted pages or in pages 0, 1, 2, ... gives bit-identical reps and
  selections and outputs within the same bound.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from kt_testlib import TOL, DevWorkload, check_units, row_rel_err

pytestmark = pytest.mark.gpu
# regrouping fp32 sums of up to ~10^4 weighted terms (online-softmax partials
# merged in a different tree) moves a row by a few tens of ulp
INVARIANCE = 2.0 ** -18


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300  # noqa: F401


@pytest.fixture
def cap():
    import block_sparse_long_quest_gb300 as kt
    yield kt.kt_set_max_ctas
    kt.kt_set_max_ctas(0)


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_attention_output_independent_of_split_count(mode, cap):
    # one sequence, two KV heads: a cap of 2, 4, 14 CTAs gives each segment
    # 1, 2, 7 CTAs; 0 gives the default (one per SM, ~76 per segment)
    import torch
    w = synth.custom(81, [128 * 60 + 77], num_q_heads=8, num_kv_heads=2, rep=synth.REP_QUEST,
                     head_mode=mode, top_k=12, initial_blocks=2, local_blocks=5)
    dw = DevWorkload(w)
    kv = oracle.KV.of(w)
    ref = oracle.sparse_step(kv, w.q, w.params)
    sel = torch.from_numpy(ref["sel"]).cuda()
    cnt = torch.from_numpy(ref["cnt"]).cuda()
    outs = {}
    for ctas in (2, 4, 14, 0):
        cap(ctas)
        out, ws = dw.attend(sel, cnt)
        outs[ctas] = out.cpu().numpy()
        assert row_rel_err(outs[ctas][0], ref["out"][0]).max() <= TOL, ctas
    for ctas in (2, 4, 14):
        assert row_rel_err(outs[ctas][0], outs[0][0]).max() <= INVARIANCE, ctas


def test_dense_output_independent_of_split_count(cap):
    w = synth.custom(82, [128 * 33 + 5, 128 * 9], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_QUEST)
    dw = DevWorkload(w)
    want = oracle.dense(oracle.KV.of(w), w.q, 8, w.params.softmax_scale)
    outs = {}
    for ctas in (4, 8, 28, 0):
        cap(ctas)
        out, _ = dw.dense()
        outs[ctas] = out.cpu().numpy()
        assert row_rel_err(outs[ctas], want).max() <= TOL, ctas
    for ctas in (4, 8, 28):
        assert row_rel_err(outs[ctas], outs[0]).max() <= INVARIANCE, ctas


@pytest.mark.parametrize("rep,mode", [(synth.REP_QUEST, synth.HEAD_SHARED),
                                      (synth.REP_MAX, synth.HEAD_SEPARATE),
                                      (synth.REP_FIX, synth.HEAD_SHARED)])
def test_step_independent_of_split_count(rep, mode, cap):
    # the one-launch step at several CTA counts: the scoring slices and the
    # split-K partition both change
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(83, [128 * 200 + 31], num_q_heads=16, num_kv_heads=4, rep=rep,
                     head_mode=mode, top_k=16, initial_blocks=1, local_blocks=8)
    dw = DevWorkload(w)
    dw.build_reps()
    kv = oracle.KV.of(w)
    ref = oracle.sparse_step(kv, w.q, w.params)
    sms = _sms()
    results = {}
    for ctas in (4, 8, 28, min(100, sms), 0):
        cap(ctas)
        if ctas == 0:
            assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
        sel, cnt, out, ws = dw.step()
        assert kt.kt_read_device_status(ws) == kt.KT_OK
        sel, cnt, out = sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
        check_units(w, kv, sel, cnt, out, ref, (0, dw.SEL))
        results[ctas] = (sel, cnt, out)
    sel0, cnt0, out0 = results[0]
    for ctas, (sel, cnt, out) in results.items():
        for u in range(dw.SEL):
            if np.array_equal(sel[0, u], sel0[0, u]):
                heads = list(range(16)) if mode == synth.HEAD_SHARED else \
                    list(range(4 * u, 4 * u + 4))
                assert row_rel_err(out[0, heads], out0[0, heads]).max() <= INVARIANCE, ctas


def _identity_copy(w):
    """The same logical KV with page = running block index (identity table)."""
    P = w.num_pages
    order = []
    table = np.zeros_like(w.block_table)
    for b, n in enumerate(w.seq_lens):
        nb = (int(n) + 127) // 128
        for j in range(nb):
            table[b, j] = len(order)
            order.append(int(w.block_table[b, j]))
    rest = [pg for pg in range(P) if pg not in set(order)]
    perm = np.array(order + rest, dtype=np.int64)
    return dataclasses.replace(w, k_pool=np.ascontiguousarray(w.k_pool[perm]),
                               v_pool=np.ascontiguousarray(w.v_pool[perm]), block_table=table)


@pytest.mark.parametrize("rep,mode", [(synth.REP_QUEST, synth.HEAD_SHARED),
                                      (synth.REP_MEAN, synth.HEAD_SEPARATE),
                                      (synth.REP_FIX, synth.HEAD_SEPARATE)])
def test_paged_and_identity_tables_agree(rep, mode):
    w = synth.custom(84, [128 * 37 + 3, 128 * 52, 128 * 20 + 100], num_q_heads=8,
                     num_kv_heads=2, rep=rep, head_mode=mode, top_k=6, permute_pages=True)
    wi = _identity_copy(w)
    assert not np.array_equal(w.block_table, wi.block_table)
    res = []
    for x in (w, wi):
        dw = DevWorkload(x)
        dw.build_reps()
        reps = dw.reps_view()
        by_block = {(b, j): reps[x.block_table[b, j]].copy()
                    for b in range(x.batch) for j in range(int(x.seq_lens[b]) // 128)}
        sel, cnt, out, _ = dw.step()
        res.append((by_block, sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()))
    (r0, s0, c0, o0), (r1, s1, c1, o1) = res
    for key in r0:
        assert np.array_equal(r0[key].view(np.uint8), r1[key].view(np.uint8)), key
    assert np.array_equal(s0, s1) and np.array_equal(c0, c1)
    assert row_rel_err(o0, o1).max() <= INVARIANCE
    ref = oracle.sparse_step(oracle.KV.of(w), w.q, w.params)
    assert row_rel_err(o0, ref["out"]).max() <= TOL


def test_one_launch_step_across_tag_wrap_with_changing_layouts():
    # one workspace shared by one-launch steps of two layouts (SHARED: one
    # unit of many slices; SEPARATE: two units), alternated for more than one
    # cycle of the 12-bit slot tags: every launch writes every slot of the
    # region, so no slot left by the other layout can pass for a live one,
    # and the last outputs equal those of fresh workspaces bit for bit
    import torch
    import block_sparse_long_quest_gb300 as kt
    ws_, dws, refs = [], [], []
    # SHARED over 40 blocks: one-block slices, 152 slots; SEPARATE over 400
    # blocks: six-block slices keeping five, 760 slots
    for mode, nblk in ((synth.HEAD_SHARED, 40), (synth.HEAD_SEPARATE, 400)):
        w = synth.custom(85, [128 * nblk + 9], num_q_heads=8, num_kv_heads=2,
                         rep=synth.REP_QUEST, head_mode=mode, top_k=5)
        dw = DevWorkload(w)
        dw.build_reps()
        assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
        _, _, ref, _ = dw.step()  # a fresh workspace
        dws.append(dw)
        refs.append(ref)
        ws_.append(kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params))
    ws = ws_[0] if ws_[0].numel() >= ws_[1].numel() else ws_[1]
    bufs = []
    for dw in dws:
        B, k = dw.w.batch, dw.w.params.top_k
        bufs.append((torch.empty((B, dw.SEL, k), dtype=torch.int32, device="cuda"),
                     torch.empty((B, dw.SEL), dtype=torch.int32, device="cuda"),
                     torch.full((B, dw.w.params.num_q_heads, 128), float("nan"),
                                device="cuda")))
    n = 4200  # > 4095 launches: the slot tags wrap
    for i in range(n):
        dw = dws[i % 2]
        sel, cnt, out = bufs[i % 2]
        kt.kt_sparse_decode_step(dw.q, dw.kv, dw.reps, dw.params, sel, cnt, out, ws)
    torch.cuda.synchronize()
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    for j in range(2):
        assert torch.equal(bufs[j][2], refs[j]), j
