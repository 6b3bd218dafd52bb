"""GPU parity: every libkt call against the CPU oracle on the same seeded inputs.

Bit-exact for representatives and block indices (outside the 1e-5 boundary
zone of the k-th score); 2e-3 max normwise relative error per output row for
attention (fp16 KV, fp32 accumulation).
"""
import numpy as np
import pytest

import oracle
import synth
from kt_testlib import TOL, DevWorkload, check_reps, row_rel_err, selection_agrees

pytestmark = pytest.mark.gpu

REPS = [synth.REP_MAX, synth.REP_MEAN, synth.REP_QUEST, synth.REP_FIX]
MODES = [synth.HEAD_SHARED, synth.HEAD_SEPARATE]

# ragged lengths: several 64-token units, partial tail blocks (<=64 and >64),
# a sequence with no Context part and one shorter than a block
RAGGED = [128 * 37 + 29, 128 * 20 + 100, 128 * 9, 300, 100, 128 * 61 + 64]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300  # noqa: F401  (fails loudly without libkt.so)


def _oracle(w, **kw):
    return oracle.sparse_step(oracle.KV.of(w), w.q, w.params, w.q_local, **kw)


@pytest.mark.parametrize("rep", REPS)
def test_reps_bit_exact_ragged_paged(rep):
    w = synth.custom(21, RAGGED, num_q_heads=8, num_kv_heads=4, rep=rep, fix_stride=32)
    dw = DevWorkload(w)
    dw.build_reps()
    ref = _oracle(w)["reps"]
    assert check_reps(dw, ref) == 0


def test_reps_signed_zero_and_extremes():
    w = synth.custom(22, [128 * 4], num_q_heads=2, num_kv_heads=2, rep=synth.REP_QUEST)
    k = w.k_pool
    k[:, :, :, 0] = 0x8000          # only -0
    k[:, :, ::2, 1] = 0x0000        # +0 and -0 mixed
    k[:, :, 1::2, 1] = 0x8000
    k[:, :, :, 2] = 0x7BFF          # max finite
    k[:, :, 5, 3] = 0xFBFF          # min finite in one row
    k[:, :, :, 4] = 0x0001          # smallest subnormal
    k[:, :, 7, 4] = 0x8001
    for rep in (synth.REP_QUEST, synth.REP_MAX, synth.REP_MEAN):
        w.params.rep = rep
        dw = DevWorkload(w)
        dw.build_reps()
        assert check_reps(dw, _oracle(w)["reps"]) == 0


@pytest.mark.parametrize("rep", REPS)
@pytest.mark.parametrize("mode", MODES)
def test_selection_matches_oracle(rep, mode):
    w = synth.custom(23, RAGGED, num_q_heads=16, num_kv_heads=4, rep=rep, head_mode=mode,
                     top_k=5, fix_stride=32, num_needles=2)
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, sc, ws = dw.select()
    ref = _oracle(w)
    sel, cnt, sc = sel.cpu().numpy(), cnt.cpu().numpy(), sc.cpu().numpy()
    import block_sparse_long_quest_gb300 as kt
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    for b in range(w.batch):
        for u in range(dw.SEL):
            ok, exact = selection_agrees(sel, cnt, ref, b, u)
            assert ok, (b, u, sel[b, u], ref["sel"][b, u])
            c = int(cnt[b, u])
            if exact and c:
                want = ref["unit_scores"][b, u][sel[b, u, :c]]
                assert np.allclose(sc[b, u, :c], want, rtol=1e-4, atol=1e-4 * np.abs(want).max())


def test_selection_large_topk_and_many_chunks():
    # many context blocks per unit: several selection CTAs, radix merge, k > 32
    w = synth.custom(24, [128 * 700 + 7, 128 * 300], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SEPARATE, top_k=100)
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, _, _ = dw.select()
    ref = _oracle(w)
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    for b in range(2):
        for u in range(2):
            assert selection_agrees(sel, cnt, ref, b, u)[0]


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_dense_attention_matches_oracle(G):
    w = synth.custom(25, RAGGED, num_q_heads=2 * G, num_kv_heads=2)
    dw = DevWorkload(w)
    out, ws = dw.dense()
    kv = oracle.KV.of(w)
    ref = oracle.dense(kv, w.q, 2 * G, w.params.softmax_scale)
    err = row_rel_err(out.cpu().numpy(), ref)
    assert err.max() <= TOL, err.max()
    import block_sparse_long_quest_gb300 as kt
    assert kt.kt_read_device_status(ws) == kt.KT_OK


@pytest.mark.parametrize("mode", MODES)
def test_sparse_attention_given_oracle_selection(mode):
    w = synth.custom(26, RAGGED, num_q_heads=16, num_kv_heads=4, rep=synth.REP_QUEST,
                     head_mode=mode, top_k=6, initial_blocks=2, local_blocks=3)
    ref = _oracle(w)
    dw = DevWorkload(w)
    from kt_testlib import to_dev
    out, ws = dw.attend(to_dev(ref["sel"]), to_dev(ref["cnt"]))
    err = row_rel_err(out.cpu().numpy(), ref["out"])
    assert err.max() <= TOL, err.max()
    import block_sparse_long_quest_gb300 as kt
    assert kt.kt_read_device_status(ws) == kt.KT_OK


@pytest.mark.parametrize("rep", REPS)
@pytest.mark.parametrize("mode", MODES)
def test_full_step_matches_oracle(rep, mode):
    w = synth.custom(27, RAGGED, num_q_heads=16, num_kv_heads=4, rep=rep, head_mode=mode,
                     top_k=4, num_needles=3)
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, out, ws = dw.step()
    ref = _oracle(w)
    sel, cnt, out = sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
    G = 4
    compared = 0
    for b in range(w.batch):
        for u in range(dw.SEL):
            ok, exact = selection_agrees(sel, cnt, ref, b, u)
            assert ok
            if exact:
                heads = range(16) if dw.SEL == 1 else range(u * G, (u + 1) * G)
                err = row_rel_err(out[b, list(heads)], ref["out"][b, list(heads)])
                assert err.max() <= TOL, err.max()
                compared += 1
    assert compared > 0
    import block_sparse_long_quest_gb300 as kt
    assert kt.kt_read_device_status(ws) == kt.KT_OK


def test_selecting_every_block_equals_dense():
    w = synth.custom(28, RAGGED, num_q_heads=8, num_kv_heads=2, rep=synth.REP_MAX,
                     head_mode=synth.HEAD_SEPARATE, top_k=1024)
    dw = DevWorkload(w)
    dw.build_reps()
    _, _, out, _ = dw.step()
    dense, _ = dw.dense()
    err = row_rel_err(out.cpu().numpy(), dense.cpu().numpy())
    assert err.max() <= TOL


def test_tiny_workload_selects_planted_blocks():
    w = synth.tiny()
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, out, _ = dw.step()
    ref = _oracle(w)
    assert check_reps(dw, ref["reps"]) == 0
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    planted = {j for _, j in w.needles}
    for u in range(8):
        assert planted <= set(sel[0, u, :cnt[0, u]].tolist())
        assert selection_agrees(sel, cnt, ref, 0, u)[0]
    assert row_rel_err(out.cpu().numpy(), ref["out"]).max() <= TOL


def test_bad_block_table_entry_is_reported_not_faulted():
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(29, [128 * 12], num_q_heads=4, num_kv_heads=2, top_k=3)
    dw = DevWorkload(w)
    dw.build_reps()
    dw.table[0, 11] = w.num_pages + 7   # a Local block pointing outside the pool
    _, _, out, ws = dw.step()
    assert kt.kt_read_device_status(ws) == kt.KT_ERR_DEVICE_CHECK
    assert kt.kt_read_device_status(ws) == kt.KT_OK  # reading clears it


def test_bounded_wait_times_out_with_status():
    import torch
    import block_sparse_long_quest_gb300 as kt
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    kt.kt_selftest_bounded_wait(ws, 1000)
    assert kt.kt_read_device_status(ws) == kt.KT_ERR_TIMEOUT


@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_one_launch_step_timeout_records_status_and_recovers(mode):
    # one CTA publishes no candidate slots: its unit's slot polls run out (2 ms
    # limit), the launch records KT_ERR_TIMEOUT and finishes, and the same
    # workspace then serves a normal step with the normal result
    import ctypes

    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(36, [128 * 60 + 5], num_q_heads=8, num_kv_heads=2, top_k=4,
                     head_mode=mode)
    dw = DevWorkload(w)
    dw.build_reps()
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    s0, c0, o0, _ = dw.step(ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    sel, cnt, out = torch.zeros_like(s0), torch.zeros_like(c0), torch.zeros_like(o0)
    st = kt.lib.kt_selftest_step_timeout(
        dw.q.data_ptr(), ctypes.byref(dw.kv), dw.reps.data_ptr(), ctypes.byref(dw.params),
        sel.data_ptr(), cnt.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(), 0, 2000,
        torch.cuda.current_stream().cuda_stream)
    assert st == kt.KT_OK, kt.status_string(st)
    assert kt.kt_read_device_status(ws) == kt.KT_ERR_TIMEOUT
    s2, c2, o2, _ = dw.step(ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    assert (s2 == s0).all() and (c2 == c0).all() and (o2 == o0).all()
    ref = _oracle(w)
    for u in range(dw.SEL):
        assert selection_agrees(s2.cpu().numpy(), c2.cpu().numpy(), ref, 0, u)[0]


def test_workspace_reuse_is_stable():
    # counters are reset by each call: repeated calls give identical results
    w = synth.custom(30, RAGGED, num_q_heads=8, num_kv_heads=2, top_k=4)
    dw = DevWorkload(w)
    dw.build_reps()
    s1, c1, o1, ws = dw.step()
    s2, c2, o2, _ = dw.step(ws)
    assert (s1 == s2).all() and (c1 == c2).all()
    assert (o1 == o2).all()  # deterministic merge order


def test_one_workspace_serves_every_call():
    # select, attend and step share one workspace (sized for the step) in any order
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(31, RAGGED, num_q_heads=8, num_kv_heads=2, top_k=4,
                     head_mode=synth.HEAD_SEPARATE)
    dw = DevWorkload(w)
    dw.build_reps()
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    s0, c0, o0, _ = dw.step(ws)
    out_a, _ = dw.attend(s0, c0, ws)
    s1, c1, _, _ = dw.select(ws)
    dense, _ = dw.dense(ws)
    s2, c2, o2, _ = dw.step(ws)
    # the step and the selection call may sum the block scores in different
    # orders (tensor cores vs CUDA cores): each must agree with the oracle
    ref = _oracle(w)
    for sel, cnt in ((s0, c0), (s1, c1)):
        sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
        for b in range(w.batch):
            for u in range(dw.SEL):
                assert selection_agrees(sel, cnt, ref, b, u)[0]
    assert (s0 == s2).all() and (c0 == c2).all()
    # repeated steps agree bit for bit; the one-launch step and the
    # attention-only call group the split-K merge differently (rounding only)
    assert (o0 == o2).all()
    assert row_rel_err(o0.cpu().numpy(), out_a.cpu().numpy()).max() <= 2.0 ** -18
    assert kt.kt_read_device_status(ws) == kt.KT_OK


def test_more_segments_than_sms_and_empty_sequence():
    # 45 sequences x 4 KV heads = 180 segments (more than the SM count), one empty
    import block_sparse_long_quest_gb300 as kt
    lens = [0] + [128 * (3 + (i * 7) % 11) + (i * 37) % 128 for i in range(44)]
    w = synth.custom(32, lens, num_q_heads=8, num_kv_heads=4, top_k=3,
                     head_mode=synth.HEAD_SEPARATE)
    dw = DevWorkload(w)
    dw.build_reps()
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 2  # two-kernel path
    sel, cnt, out, ws = dw.step()
    dense, _ = dw.dense()
    ref = _oracle(w)
    out, sel, cnt = out.cpu().numpy(), sel.cpu().numpy(), cnt.cpu().numpy()
    assert np.all(out[0] == 0.0) and np.all(dense.cpu().numpy()[0] == 0.0)
    d_ref = oracle.dense(oracle.KV.of(w), w.q, 8, w.params.softmax_scale)
    assert row_rel_err(dense.cpu().numpy()[1:], d_ref[1:]).max() <= TOL
    for b in range(1, w.batch):
        for u in range(4):
            ok, exact = selection_agrees(sel, cnt, ref, b, u)
            assert ok
            if exact:
                assert row_rel_err(out[b, 2 * u:2 * u + 2], ref["out"][b, 2 * u:2 * u + 2]).max() <= TOL
    import block_sparse_long_quest_gb300 as kt
    assert kt.kt_read_device_status(ws) == kt.KT_OK


def test_step_after_query_change_uses_the_new_selection():
    # The one-launch step tags each unit's published selection with a launch
    # counter; a step with new queries must never attend the previous one.
    import block_sparse_long_quest_gb300 as kt
    from kt_testlib import to_dev
    w = synth.custom(33, RAGGED, num_q_heads=16, num_kv_heads=4, rep=synth.REP_QUEST,
                     head_mode=synth.HEAD_SEPARATE, top_k=4, num_needles=3)
    dw = DevWorkload(w)
    dw.build_reps()
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1  # one-launch path
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    q_first = w.q.copy()
    for it in range(6):
        q = q_first.copy() if it % 2 else synth.normal_f16(w.q.shape, 33, 900 + it, sigma=2.0)
        dw.q.copy_(to_dev(q))
        w.q = q
        sel, cnt, out, _ = dw.step(ws)
        ref = _oracle(w)
        sel, cnt, out = sel.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
        for b in range(w.batch):
            for u in range(dw.SEL):
                ok, exact = selection_agrees(sel, cnt, ref, b, u)
                assert ok, (it, b, u)
                if exact:
                    hs = list(range(4 * u, 4 * u + 4))
                    assert row_rel_err(out[b, hs], ref["out"][b, hs]).max() <= TOL
        assert kt.kt_read_device_status(ws) == kt.KT_OK



def test_host_buffer_step_replays_and_follows_host_inputs():
    # kt_sparse_decode_step_host (upload, step, download, sync) on a stream and
    # on the legacy default stream: outputs follow the host query as it
    # changes between calls and match the oracle
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(35, [128 * 20 + 9], num_q_heads=8, num_kv_heads=2, top_k=4,
                     head_mode=synth.HEAD_SHARED)
    dw = DevWorkload(w)
    dw.build_reps()
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    sel = torch.zeros((1, 1, 4), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    q_dev = torch.empty_like(dw.q)
    out_dev = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
    q_host = torch.empty_like(dw.q, device="cpu").pin_memory()
    out_host = torch.empty_like(out_dev, device="cpu").pin_memory()
    stream = torch.cuda.Stream()
    rng = np.random.default_rng(7)
    for i in range(4):
        qb = rng.standard_normal(w.q.shape).astype(np.float16)
        q_host.copy_(torch.from_numpy(qb))
        st = stream if i < 3 else 0  # the last call on the legacy default stream
        kt.kt_sparse_decode_step_host(q_host, q_dev, dw.kv, dw.reps, dw.params, sel, cnt, out_dev,
                                      out_host, ws, st)
        w2 = synth.custom(35, [128 * 20 + 9], num_q_heads=8, num_kv_heads=2, top_k=4,
                          head_mode=synth.HEAD_SHARED)
        w2.q = qb.view(np.uint16)
        ref = oracle.sparse_step(oracle.KV.of(w2), w2.q, w2.params)
        assert row_rel_err(out_host.numpy(), ref["out"]).max() <= TOL, i
    assert kt.kt_read_device_status(ws) == kt.KT_OK


def test_host_buffer_step_mapped_reads_and_writes_host_memory():
    # q_dev and out_dev NULL: the step kernel reads the page-locked query and
    # writes the output over the host link; the output equals the device
    # step's bit for bit, follows the host query between calls and matches the
    # oracle; pageable host memory is refused before any launch
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(36, [128 * 24 + 17], num_q_heads=16, num_kv_heads=4, top_k=5,
                     head_mode=synth.HEAD_SHARED)
    dw = DevWorkload(w)
    dw.build_reps()
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    sel = torch.zeros((1, 1, 5), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    q_host = torch.empty_like(dw.q, device="cpu").pin_memory()
    out_host = torch.empty((1, 16, 128), dtype=torch.float32, device="cpu").pin_memory()
    out_dev = torch.empty((1, 16, 128), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    rng = np.random.default_rng(11)
    for i in range(3):
        qb = rng.standard_normal(w.q.shape).astype(np.float16)
        q_host.copy_(torch.from_numpy(qb))
        out_host.fill_(float("nan"))
        kt.kt_sparse_decode_step_host(q_host, None, dw.kv, dw.reps, dw.params, sel, cnt, None,
                                      out_host, ws, stream)
        got = out_host.clone()
        q_dev = q_host.cuda()
        kt.kt_sparse_decode_step(q_dev, dw.kv, dw.reps, dw.params, sel, cnt, out_dev, ws, stream)
        stream.synchronize()
        assert torch.equal(got, out_dev.cpu()), i
        w2 = synth.custom(36, [128 * 24 + 17], num_q_heads=16, num_kv_heads=4, top_k=5,
                          head_mode=synth.HEAD_SHARED)
        w2.q = qb.view(np.uint16)
        ref = oracle.sparse_step(oracle.KV.of(w2), w2.q, w2.params)
        assert row_rel_err(got.numpy(), ref["out"]).max() <= TOL, i
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    pageable = torch.empty_like(dw.q, device="cpu")
    with pytest.raises(kt.KtError) as e:
        kt.kt_sparse_decode_step_host(pageable, None, dw.kv, dw.reps, dw.params, sel, cnt, None,
                                      out_host, ws, stream)
    assert e.value.status == kt.KT_ERR_INVALID_ARG


@pytest.mark.parametrize("rep", REPS)
@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_host_buffer_step_mapped_every_scoring_path(rep, mode):
    # the copy-free host step reads the query in every scoring path of the
    # one-launch step (CUDA-core columns and lines, tensor cores, fp32 Mean,
    # multi-rep Fix): bit for bit the device step's output
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(37, [128 * 60 + 5, 128 * 21], num_q_heads=8, num_kv_heads=2, rep=rep,
                     head_mode=mode, top_k=6, fix_stride=32)
    dw = DevWorkload(w)
    dw.build_reps()
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
    sel_d, cnt_d, out_d, ws = dw.step()
    q_host = dw.q.cpu().pin_memory()
    out_host = torch.full(tuple(out_d.shape), float("nan"), dtype=torch.float32).pin_memory()
    sel = torch.full_like(sel_d, -1)
    cnt = torch.full_like(cnt_d, -1)
    kt.kt_sparse_decode_step_host(q_host, None, dw.kv, dw.reps, dw.params, sel, cnt, None,
                                  out_host, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    assert torch.equal(cnt, cnt_d) and torch.equal(sel, sel_d)
    assert torch.equal(out_host, out_d.cpu())
