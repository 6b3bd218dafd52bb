"""The allocation-free attention entry point.

Some callers cannot allocate device memory: a kernel plugged into an engine or
framework that only hands it its input and output buffers (the host owns every
other byte of device memory), or a latency-critical path where a cudaMalloc,
which can synchronise the device, is not allowed.  kt_sparse_decode_attn_noalloc
serves them with scratch memory that lives in a fixed array of the library.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes alone in a fresh process and after the
rest of the suite.
"""
import ctypes

import numpy as np
import pytest

import synth
from kt_testlib import TOL, DevWorkload, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kt():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_long_quest_gb300 as kt
    return kt


def test_noalloc_attention_matches_workspace_call_twice(kt):
    import torch
    w = synth.custom(41, [128 * 37 + 29, 128 * 20 + 100, 300, 128 * 61 + 64], num_q_heads=16,
                     num_kv_heads=4, top_k=5, head_mode=synth.HEAD_SEPARATE, num_needles=2)
    dw = DevWorkload(w)
    dw.build_reps()
    sel, cnt, _, _ = dw.select()
    want, ws = dw.attend(sel, cnt)  # the existing entry point, with a workspace
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    want = want.cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        out = torch.full_like(dw.q, float("nan"), dtype=torch.float32)
        st = kt.lib.kt_sparse_decode_attn_noalloc(dw.q.data_ptr(), ctypes.byref(dw.kv),
                                                  ctypes.byref(dw.params), sel.data_ptr(),
                                                  cnt.data_ptr(), out.data_ptr(), stream)
        assert st == kt.KT_OK, kt.status_string(st)
        dev_status = ctypes.c_int32(-1)
        assert kt.lib.kt_noalloc_read_status(stream, ctypes.byref(dev_status)) == kt.KT_OK
        assert dev_status.value == kt.KT_OK, kt.status_string(dev_status.value)
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert row_rel_err(got, want).max() <= TOL


def test_noalloc_rejects_shapes_beyond_its_scratch(kt):
    import torch
    # 700 sequences x 1 KV head x G = 8: more partial slots than the 1 MiB array holds
    lens = torch.full((700,), 128, dtype=torch.int32, device="cuda")
    table = torch.zeros((700, 1), dtype=torch.int32, device="cuda")
    pool = torch.zeros((1, 1, 128, 128), dtype=torch.float16, device="cuda")
    kv = kt.paged_kv(pool, pool, table, lens)
    p = kt.sparse_params(8, 1, 1, 4, kt.KT_REP_QUEST, kt.KT_HEAD_SHARED)
    q = torch.zeros((700, 8, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((700, 8, 128), dtype=torch.float32, device="cuda")
    sel = torch.zeros((700, 1, 4), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((700, 1), dtype=torch.int32, device="cuda")
    st = kt.lib.kt_sparse_decode_attn_noalloc(q.data_ptr(), ctypes.byref(kv), ctypes.byref(p),
                                              sel.data_ptr(), cnt.data_ptr(), out.data_ptr(),
                                              None)
    assert st == kt.KT_ERR_WORKSPACE_TOO_SMALL
