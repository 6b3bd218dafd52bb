"""Host-only checks of the C ABI: the library loads without a GPU, exports every
symbol include/kt.h declares, sizes workspaces, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import block_sparse_long_quest_gb300 as kt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # aligned, never dereferenced: validation fails before any launch


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kt.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kt_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 14
    lib = ctypes.CDLL(kt._LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(kt.EXPORTS) == names


def kv(batch=1, H_kv=8, head_dim=128, block_size=128, max_blocks=1024, pages=1024, ptr=FAKE):
    return kt.PagedKV(ptr, ptr, ptr, ptr, batch, H_kv, head_dim, block_size, max_blocks, pages)


def params(**kw):
    base = dict(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=32,
                rep=kt.KT_REP_QUEST, head_mode=kt.KT_HEAD_SHARED)
    base.update(kw)
    extra = {k: base.pop(k) for k in ("num_reps", "fix_stride", "softmax_scale") if k in base}
    return kt.sparse_params(**base, **extra)


def ws_bytes(op, k, p, T=0):
    n = ctypes.c_size_t(0)
    st = kt.lib.kt_workspace_bytes(op, ctypes.byref(k), ctypes.byref(p), T, ctypes.byref(n))
    return st, n.value


def test_status_strings():
    for s in range(7):
        assert kt.status_string(s)
    assert kt.status_string(99) == "unknown status"


def test_reps_per_block_and_pool_bytes():
    assert kt.kt_reps_per_block(params(rep=kt.KT_REP_MAX)) == 1
    assert kt.kt_reps_per_block(params(rep=kt.KT_REP_QUEST)) == 2
    assert kt.kt_reps_per_block(params(rep=kt.KT_REP_FIX, fix_stride=32)) == 4
    assert kt.kt_reps_per_block(params(rep=kt.KT_REP_DYNAMIC, num_reps=4)) == 4
    # 128K Quest: 1024 pages x 8 heads x 2 rows x 256 B = 4 MiB
    assert kt.kt_reps_pool_bytes(kv(), params()) == 1024 * 8 * 2 * 256
    assert kt.kt_reps_pool_bytes(kv(), params(rep=kt.KT_REP_MEAN)) == 1024 * 8 * 512


@pytest.mark.parametrize("op", [kt.KT_OP_SCORE_SELECT, kt.KT_OP_SPARSE_ATTN,
                                kt.KT_OP_DENSE_ATTN, kt.KT_OP_SPARSE_STEP])
def test_workspace_sizes_are_modest(op):
    st, n = ws_bytes(op, kv(), params())
    assert st == kt.KT_OK and 256 <= n < 32 << 20
    st, n2 = ws_bytes(op, kv(batch=16, max_blocks=512, pages=16 * 512), params(top_k=16))
    assert st == kt.KT_OK and n2 >= 256


@pytest.mark.parametrize("k,p,status", [
    (kv(head_dim=64), params(), kt.KT_ERR_UNSUPPORTED),
    (kv(block_size=64), params(), kt.KT_ERR_UNSUPPORTED),
    (kv(batch=0), params(), kt.KT_ERR_INVALID_ARG),
    (kv(batch=300), params(), kt.KT_ERR_UNSUPPORTED),           # 2400 segments
    (kv(ptr=FAKE + 4), params(), kt.KT_ERR_INVALID_ARG),         # misaligned
    (kv(ptr=0), params(), kt.KT_ERR_INVALID_ARG),
    (kv(), params(num_q_heads=30), kt.KT_ERR_INVALID_ARG),       # not a multiple of H_kv
    (kv(), params(num_q_heads=128), kt.KT_ERR_UNSUPPORTED),      # G = 16
    (kv(), params(local_blocks=0), kt.KT_ERR_UNSUPPORTED),
    (kv(), params(top_k=0), kt.KT_ERR_INVALID_ARG),
    (kv(), params(top_k=5000), kt.KT_ERR_UNSUPPORTED),
    (kv(), params(rep=9), kt.KT_ERR_INVALID_ARG),
    (kv(), params(head_mode=3), kt.KT_ERR_INVALID_ARG),
    (kv(), params(rep=kt.KT_REP_FIX, fix_stride=3), kt.KT_ERR_INVALID_ARG),
    (kv(), params(rep=kt.KT_REP_DYNAMIC, num_reps=64), kt.KT_ERR_UNSUPPORTED),
    (kv(), params(softmax_scale=-1.0), kt.KT_ERR_INVALID_ARG),
])
def test_invalid_arguments(k, p, status):
    st, _ = ws_bytes(kt.KT_OP_SPARSE_STEP, k, p)
    assert st == status
    st = kt.lib.kt_sparse_decode_step(FAKE, ctypes.byref(k), FAKE, ctypes.byref(p), FAKE, FAKE,
                                      FAKE, FAKE, 1 << 30, None)
    assert st == status
    assert kt.lib.kt_sparse_decode_step_kernels(ctypes.byref(k), ctypes.byref(p)) == -status


def test_step_kernel_count_is_one_or_two():
    # 1 needs a device with enough SMs; without one the two-kernel plan stands
    n = kt.kt_sparse_decode_step_kernels(kv(), params())
    assert n in (1, 2)
    with pytest.raises(kt.KtError):
        kt.kt_sparse_decode_step_kernels(kv(batch=0), params())


def test_calls_reject_null_and_small_workspace_without_a_device():
    k, p = kv(), params()
    st = kt.lib.kt_score_select_blocks(None, ctypes.byref(k), FAKE, ctypes.byref(p), FAKE, FAKE,
                                       None, FAKE, 1 << 30, None)
    assert st == kt.KT_ERR_INVALID_ARG
    st = kt.lib.kt_sparse_decode_attn(FAKE, ctypes.byref(k), ctypes.byref(p), FAKE, FAKE, FAKE,
                                      FAKE, 16, None)
    assert st == kt.KT_ERR_WORKSPACE_TOO_SMALL
    st = kt.lib.kt_dense_decode_attn(FAKE, ctypes.byref(k), 32, 0.088, FAKE, FAKE, 16, None)
    assert st == kt.KT_ERR_WORKSPACE_TOO_SMALL
    st = kt.lib.kt_build_block_reps(ctypes.byref(k), ctypes.byref(p), -1, 4, FAKE, None)
    assert st == kt.KT_ERR_INVALID_ARG
    st = kt.lib.kt_build_block_reps(ctypes.byref(k), ctypes.byref(params(rep=kt.KT_REP_DYNAMIC,
                                                                         num_reps=4)),
                                    0, 4, FAKE, None)
    assert st == kt.KT_ERR_INVALID_ARG
    assert kt.lib.kt_selftest_bounded_wait(None, 256, 10, None) == kt.KT_ERR_INVALID_ARG
    v = ctypes.c_int32(0)
    assert kt.lib.kt_read_device_status(None, 256, None, ctypes.byref(v)) == kt.KT_ERR_INVALID_ARG
    # the host-buffer step: a NULL host buffer, or only one of the two device
    # buffers left NULL, is refused before anything touches a device
    st = kt.lib.kt_sparse_decode_step_host(None, FAKE, ctypes.byref(k), FAKE, ctypes.byref(p),
                                           FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == kt.KT_ERR_INVALID_ARG
    st = kt.lib.kt_sparse_decode_step_host(FAKE, None, ctypes.byref(k), FAKE, ctypes.byref(p),
                                           FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == kt.KT_ERR_INVALID_ARG
    # the Q8_0 step: no pools struct, or scale rows missing
    st = kt.lib.kt_sparse_decode_step_q8_0(FAKE, None, FAKE, ctypes.byref(p), FAKE, FAKE, FAKE,
                                           FAKE, 1 << 30, None)
    assert st == kt.KT_ERR_INVALID_ARG
    kq = kt.PagedKVQ8(k_code=FAKE, k_scale=None, v_code=FAKE, v_scale=FAKE,
                      block_table=k.block_table, seq_lens=k.seq_lens, batch=k.batch,
                      num_kv_heads=k.num_kv_heads, head_dim=k.head_dim,
                      block_size=k.block_size, max_blocks_per_seq=k.max_blocks_per_seq,
                      num_pages=k.num_pages)
    st = kt.lib.kt_sparse_decode_step_q8_0(FAKE, ctypes.byref(kq), FAKE, ctypes.byref(p), FAKE,
                                           FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == kt.KT_ERR_INVALID_ARG
