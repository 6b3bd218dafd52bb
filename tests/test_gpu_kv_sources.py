"""GPU parity of the two other KV sources of the attention:

* Q8_0 pools ("How to Implement Long Context Inference (Up to 139K Tokens) with
  KTransformers", Step 1 kv_type): the quantisation is bit-exact against the
  oracle's, the attention over the codes matches the oracle's attention over
  the dequantised values, and on KV that Q8_0 stores exactly it equals the fp16
  attention bit for bit;
* K/V pools in page-locked host memory read over NVLink-C2C ("KTransformers
  长上下文稀疏注意力实战…" §4.1: the KV cache stays in CPU memory): the same
  arithmetic as the device pools, so the output is identical bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
from kt_testlib import TOL, DevWorkload, row_rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300  # noqa: F401


def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


class Q8Pools:
    """Q8_0 pools of a DevWorkload, quantised on the GPU."""

    def __init__(self, dw):
        import torch
        import block_sparse_long_quest_gb300 as kt
        P, H, bs, d = dw.w.k_pool.shape
        self.k_code = torch.empty((P, H, bs, d), dtype=torch.int8, device="cuda")
        self.v_code = torch.empty_like(self.k_code)
        self.k_scale = torch.empty((P, H, bs, d // 32), dtype=torch.float16, device="cuda")
        self.v_scale = torch.empty_like(self.k_scale)
        kt.kt_quantize_kv_q8_0(dw.kv, self.k_code, self.k_scale, self.v_code, self.v_scale)
        self.kvq = kt.paged_kv_q8(self.k_code, self.k_scale, self.v_code, self.v_scale,
                                  dw.table, dw.lens)

    def attend(self, dw, sel, cnt):
        import torch
        import block_sparse_long_quest_gb300 as kt
        out = torch.full((dw.w.batch, dw.w.params.num_q_heads, 128), float("nan"),
                         dtype=torch.float32, device="cuda")
        ws = kt.workspace(kt.KT_OP_SPARSE_ATTN, dw.kv, dw.params)
        kt.kt_sparse_decode_attn_q8_0(dw.q, self.kvq, dw.params, sel, cnt, out, ws)
        assert kt.kt_read_device_status(ws) == kt.KT_OK
        return out


def test_quantise_bit_exact_against_oracle():
    w = synth.custom(91, [128 * 7 + 33, 128 * 4], num_q_heads=4, num_kv_heads=2,
                     rep=synth.REP_QUEST, permute_pages=True)
    k = w.k_pool.view(np.float16).astype(np.float64) * 3.0
    k[0, 0, 5, 32:64] = 0.0                     # an all-zero group
    k[1, 1, 9, :32] = np.linspace(-60000, 60000, 32)  # a group near the binary16 range
    k[2, 0, 3, 64:96] = 1e-6                    # a subnormal scale
    w.k_pool = _f16(k)
    dw = DevWorkload(w)
    qp = Q8Pools(dw)
    want_kc, want_ks = oracle.quantize_q8_0(w.k_pool)
    want_vc, want_vs = oracle.quantize_q8_0(w.v_pool)
    assert np.array_equal(qp.k_code.cpu().numpy(), want_kc)
    assert np.array_equal(qp.v_code.cpu().numpy(), want_vc)
    assert np.array_equal(qp.k_scale.cpu().numpy().view(np.uint16), want_ks)
    assert np.array_equal(qp.v_scale.cpu().numpy().view(np.uint16), want_vs)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_q8_attention_matches_oracle(G, mode):
    import torch
    lens = [128 * 30 + 77, 128 * 9, 128 * 5 + 1]
    w = synth.custom(92, lens, num_q_heads=2 * G, num_kv_heads=2, rep=synth.REP_QUEST,
                     head_mode=mode, top_k=5, permute_pages=True)
    dw = DevWorkload(w)
    kv = oracle.KV.of(w)
    ref = oracle.sparse_step(kv, w.q, w.params)          # selection from the fp16 reps
    sel = torch.from_numpy(ref["sel"]).cuda()
    cnt = torch.from_numpy(ref["cnt"]).cuda()
    got = Q8Pools(dw).attend(dw, sel, cnt).cpu().numpy()
    want = oracle.attend_selection_q8(oracle.KVQ(kv), w.q, w.params, ref["sel"], ref["cnt"])
    assert row_rel_err(got, want).max() <= TOL


def test_q8_of_exactly_stored_kv_equals_fp16_attention():
    # every 32-channel group on its own grid m * 2^-e (|m| <= 127, one at 127):
    # Q8_0 stores it exactly, so the dequantised blocks are the fp16 blocks
    import torch
    rng = np.random.default_rng(93)
    w = synth.custom(93, [128 * 12 + 40, 128 * 6], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_QUEST, top_k=3, permute_pages=True)
    P = w.num_pages
    for name in ("k_pool", "v_pool"):
        e = rng.integers(0, 9, size=(P, 2, 128, 4, 1))
        m = rng.integers(-127, 128, size=(P, 2, 128, 4, 32))
        m[..., 0] = 127
        setattr(w, name, _f16((m * 2.0 ** -e).reshape(P, 2, 128, 128)))
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, _, _ = dw.select()
    fp16_out, _ = dw.attend(sel, cnt)
    q8_out = Q8Pools(dw).attend(dw, sel, cnt)
    assert torch.equal(q8_out, fp16_out)


def _q8_step(dw, qp):
    import torch
    import block_sparse_long_quest_gb300 as kt
    B, k = dw.w.batch, dw.w.params.top_k
    sel = torch.full((B, dw.SEL, k), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, dw.SEL), -1, dtype=torch.int32, device="cuda")
    out = torch.full((B, dw.w.params.num_q_heads, 128), float("nan"), dtype=torch.float32,
                     device="cuda")
    ws = kt.workspace(kt.KT_OP_SPARSE_STEP, dw.kv, dw.params)
    kt.kt_sparse_decode_step_q8_0(dw.q, qp.kvq, dw.reps, dw.params, sel, cnt, out, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    return sel, cnt, out


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_q8_step_matches_fp16_selection_and_oracle(G, mode):
    # the one-launch step over Q8_0 pools: the selection (from the fp16 reps)
    # equals the fp16 step's, and the output matches the oracle's attention
    # over the dequantised blocks of that selection
    import torch
    import block_sparse_long_quest_gb300 as kt
    lens = [128 * 30 + 77, 128 * 9, 128 * 5 + 1]
    w = synth.custom(96, lens, num_q_heads=2 * G, num_kv_heads=2, rep=synth.REP_QUEST,
                     head_mode=mode, top_k=5, permute_pages=True)
    dw = DevWorkload(w)
    dw.build_reps()
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
    sel16, cnt16, _, _ = dw.step()
    sel, cnt, out = _q8_step(dw, Q8Pools(dw))
    assert torch.equal(cnt, cnt16)
    for b in range(w.batch):
        for u in range(dw.SEL):
            c = int(cnt[b, u])
            assert torch.equal(sel[b, u, :c], sel16[b, u, :c]), (b, u)
    want = oracle.attend_selection_q8(oracle.KVQ(oracle.KV.of(w)), w.q, w.params,
                                      sel.cpu().numpy(), cnt.cpu().numpy())
    assert row_rel_err(out.cpu().numpy(), want).max() <= TOL


def test_q8_step_of_exactly_stored_kv_equals_fp16_step():
    # KV on per-group grids is stored exactly by Q8_0: the Q8_0 step's
    # output equals the fp16 step's bit for bit
    import torch
    rng = np.random.default_rng(97)
    w = synth.custom(97, [128 * 12 + 40, 128 * 6], num_q_heads=8, num_kv_heads=2,
                     rep=synth.REP_QUEST, top_k=3, permute_pages=True)
    P = w.num_pages
    for name in ("k_pool", "v_pool"):
        e = rng.integers(0, 9, size=(P, 2, 128, 4, 1))
        m = rng.integers(-127, 128, size=(P, 2, 128, 4, 32))
        m[..., 0] = 127
        setattr(w, name, _f16((m * 2.0 ** -e).reshape(P, 2, 128, 128)))
    dw = DevWorkload(w)
    dw.build_reps()
    sel16, cnt16, out16, _ = dw.step()
    sel, cnt, out = _q8_step(dw, Q8Pools(dw))
    assert torch.equal(cnt, cnt16) and torch.equal(out, out16)


def _pinned_copy(t):
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, device="cpu", pin_memory=True)
    h.copy_(t.cpu())
    return h


@pytest.mark.parametrize("G", [1, 4, 8])
def test_host_kv_equals_device_kv(G):
    import torch
    import block_sparse_long_quest_gb300 as kt
    lens = [128 * 25 + 3, 128 * 11, 200]
    w = synth.custom(94, lens, num_q_heads=2 * G, num_kv_heads=2, rep=synth.REP_QUEST,
                     head_mode=synth.HEAD_SEPARATE, top_k=4, permute_pages=True)
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, _, _ = dw.select()
    dev_out, _ = dw.attend(sel, cnt)
    hk, hv = _pinned_copy(dw.k), _pinned_copy(dw.v)
    kvh = kt.paged_kv(hk, hv, dw.table, dw.lens)
    out = torch.full_like(dev_out, float("nan"))
    ws = kt.workspace(kt.KT_OP_SPARSE_ATTN, dw.kv, dw.params)
    kt.kt_sparse_decode_attn_hostkv(dw.q, kvh, dw.params, sel, cnt, out, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    assert torch.equal(out, dev_out)
    ref = oracle.attend_selection(oracle.KV.of(w), w.q, w.params, sel.cpu().numpy(),
                                  cnt.cpu().numpy())
    assert row_rel_err(out.cpu().numpy(), ref).max() <= TOL


def test_host_kv_rejects_device_pools():
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(95, [128 * 6], num_q_heads=4, num_kv_heads=2, rep=synth.REP_QUEST)
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, _, _ = dw.select()
    out, ws = dw.attend(sel, cnt)
    with pytest.raises(kt.KtError) as e:
        kt.kt_sparse_decode_attn_hostkv(dw.q, dw.kv, dw.params, sel, cnt, out, ws)
    assert e.value.status == kt.KT_ERR_INVALID_ARG


def test_128k_q8_and_host_kv_full_size():
    # the 128K layer: selection from the fp16 reps, then the attention from
    # Q8_0 pools (against the oracle on KV heads 0 and 5) and from host memory
    # (bit-identical to the device pools)
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.long128k()
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, _, _ = dw.select()
    dev_out, _ = dw.attend(sel, cnt)
    q8 = Q8Pools(dw).attend(dw, sel, cnt).cpu().numpy()
    kv = oracle.KV.of(w)
    kvq = oracle.KVQ(kv)
    s, c = sel.cpu().numpy(), cnt.cpu().numpy()
    nb, c0, c1 = oracle.partition(int(w.seq_lens[0]), 1, 32)
    blocks = list(range(c0)) + [int(j) for j in s[0, 0, :int(c[0, 0])]] + list(range(c1, nb))
    for hq in (0, 1, 21, 23):
        want = oracle.attend_q8(kvq, 0, hq, 32, w.q[0, hq], blocks, w.params.softmax_scale)
        assert row_rel_err(q8[0, hq], want) <= TOL, hq
    # the one-launch step over the Q8_0 pools: the fp16 step's selection,
    # the oracle's Q8_0 attention on KV heads 0 and 5
    sel16, cnt16, _, _ = dw.step()
    qsel, qcnt, qout = _q8_step(dw, Q8Pools(dw))
    assert torch.equal(qcnt, cnt16) and torch.equal(qsel[0, 0, :32], sel16[0, 0, :32])
    qout = qout.cpu().numpy()
    qs = qsel.cpu().numpy()
    blocks = list(range(c0)) + [int(j) for j in qs[0, 0, :int(qcnt[0, 0])]] + list(range(c1, nb))
    for hq in (0, 3, 20, 22):
        want = oracle.attend_q8(kvq, 0, hq, 32, w.q[0, hq], blocks, w.params.softmax_scale)
        assert row_rel_err(qout[0, hq], want) <= TOL, hq
    hk, hv = _pinned_copy(dw.k), _pinned_copy(dw.v)
    out = torch.full_like(dev_out, float("nan"))
    ws = kt.workspace(kt.KT_OP_SPARSE_ATTN, dw.kv, dw.params)
    kt.kt_sparse_decode_attn_hostkv(dw.q, kt.paged_kv(hk, hv, dw.table, dw.lens), dw.params, sel,
                                    cnt, out, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    assert torch.equal(out, dev_out)


@pytest.mark.parametrize("rep", [synth.REP_MAX, synth.REP_MEAN, synth.REP_QUEST, synth.REP_FIX])
@pytest.mark.parametrize("mode", [synth.HEAD_SHARED, synth.HEAD_SEPARATE])
def test_q8_step_every_scoring_path(rep, mode):
    # the Q8_0 one-launch step in every scoring path of the step (the reps
    # stay fp16): the fp16 step's selection, the oracle's Q8_0 attention
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(98, [128 * 60 + 5, 128 * 21], num_q_heads=8, num_kv_heads=2, rep=rep,
                     head_mode=mode, top_k=6, fix_stride=32, permute_pages=True)
    dw = DevWorkload(w)
    dw.build_reps()
    assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
    sel16, cnt16, _, _ = dw.step()
    sel, cnt, out = _q8_step(dw, Q8Pools(dw))
    assert torch.equal(cnt, cnt16) and torch.equal(sel, sel16)
    want = oracle.attend_selection_q8(oracle.KVQ(oracle.KV.of(w)), w.q, w.params,
                                      sel.cpu().numpy(), cnt.cpu().numpy())
    assert row_rel_err(out.cpu().numpy(), want).max() <= TOL


def test_q8_step_tensor_core_scoring_slices():
    # slices of many blocks per CTA (SEPARATE, ~2000 blocks per sequence, the
    # CTAs capped at 32 so that a slice holds ~125 blocks): the tensor-core
    # scoring path and the per-slice threshold search, over Q8_0 pools
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = synth.custom(99, [128 * 2000 + 77], num_q_heads=8, num_kv_heads=2, rep=synth.REP_QUEST,
                     head_mode=synth.HEAD_SEPARATE, top_k=16, local_blocks=8)
    dw = DevWorkload(w)
    dw.build_reps()
    kt.kt_set_max_ctas(32)
    try:
        assert kt.kt_sparse_decode_step_kernels(dw.kv, dw.params) == 1
        sel16, cnt16, _, _ = dw.step()
        sel, cnt, out = _q8_step(dw, Q8Pools(dw))
    finally:
        kt.kt_set_max_ctas(0)
    assert torch.equal(cnt, cnt16) and torch.equal(sel, sel16)
    want = oracle.attend_selection_q8(oracle.KVQ(oracle.KV.of(w)), w.q, w.params,
                                      sel.cpu().numpy(), cnt.cpu().numpy())
    assert row_rel_err(out.cpu().numpy(), want).max() <= TOL
