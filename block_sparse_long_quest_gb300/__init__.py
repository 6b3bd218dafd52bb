"""Python binding of libkt (block-sparse long-context decode attention, GB300).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of libkt.so, behind the C ABI declared in include/kt.h.  Tensors are
passed as raw device pointers together with torch's current CUDA stream.  If
libkt.so is missing this module raises at import; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as _LIB_PATH, build  # noqa: F401

KT_OK = 0
KT_ERR_INVALID_ARG = 1
KT_ERR_UNSUPPORTED = 2
KT_ERR_WORKSPACE_TOO_SMALL = 3
KT_ERR_CUDA = 4
KT_ERR_DEVICE_CHECK = 5
KT_ERR_TIMEOUT = 6

KT_REP_MAX, KT_REP_MEAN, KT_REP_QUEST, KT_REP_FIX, KT_REP_DYNAMIC = 0, 1, 2, 3, 4
KT_HEAD_SHARED, KT_HEAD_SEPARATE = 0, 1
(KT_OP_SCORE_SELECT, KT_OP_SPARSE_ATTN, KT_OP_DENSE_ATTN, KT_OP_SPARSE_STEP,
 KT_OP_DYNAMIC_REPS, KT_OP_PRESELECT) = 0, 1, 2, 3, 4, 5
KT_LAYER_DENSE, KT_LAYER_SELECT, KT_LAYER_REUSE = 0, 1, 2

# Every symbol declared in include/kt.h.
EXPORTS = (
    "kt_status_string", "kt_reps_per_block", "kt_reps_pool_bytes", "kt_workspace_bytes",
    "kt_workspace_init", "kt_build_block_reps", "kt_build_dynamic_reps",
    "kt_score_select_blocks", "kt_sparse_decode_attn", "kt_sparse_decode_step",
    "kt_sparse_decode_step_host", "kt_dense_decode_attn", "kt_read_device_status",
    "kt_selftest_bounded_wait", "kt_sparse_decode_attn_noalloc", "kt_sparse_decode_step_kernels",
    "kt_preselect_mask_words", "kt_preselect_blocks", "kt_score_select_blocks_presel",
    "kt_sparse_decode_step_presel", "kt_decode_history_slots", "kt_decode_layer_action",
    "kt_decode_layer", "kt_append_kv", "kt_set_max_ctas", "kt_set_phase_stamps",
    "kt_sparse_decode_attn_hostkv", "kt_quantize_kv_q8_0", "kt_sparse_decode_attn_q8_0",
    "kt_noalloc_read_status", "kt_selftest_step_timeout", "kt_sparse_decode_step_q8_0",
)


class KtError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {status_string(status)} (status {status})")


class PagedKV(ctypes.Structure):
    """kt_paged_kv: device pointers + shapes of the paged K/V pools."""
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


class SparseParams(ctypes.Structure):
    """kt_sparse_params."""
    _fields_ = [("num_q_heads", ctypes.c_int32), ("initial_blocks", ctypes.c_int32),
                ("local_blocks", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("num_reps", ctypes.c_int32), ("fix_stride", ctypes.c_int32),
                ("rep", ctypes.c_int32), ("head_mode", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]


class PagedKVQ8(ctypes.Structure):
    """kt_paged_kv_q8: Q8_0 code and scale pools + block table and lengths."""
    _fields_ = [("k_code", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_code", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


class ReusePolicy(ctypes.Structure):
    """kt_reuse_policy: dense layers and the selection reuse strides."""
    _fields_ = [("num_layers", ctypes.c_int32), ("dense_layer_num", ctypes.c_int32),
                ("layer_step", ctypes.c_int32), ("token_step", ctypes.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libkt.so not built ({_LIB_PATH}); run "
                          "block_sparse_long_quest_gb300.build() or __graft_entry__.build()")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, sz, P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.POINTER
    sig = {
        "kt_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "kt_reps_per_block": (i32, [P(SparseParams)]),
        "kt_reps_pool_bytes": (sz, [P(PagedKV), P(SparseParams)]),
        "kt_workspace_bytes": (ctypes.c_int, [ctypes.c_int, P(PagedKV), P(SparseParams), i32,
                                              P(sz)]),
        "kt_workspace_init": (ctypes.c_int, [vp, sz, vp]),
        "kt_build_block_reps": (ctypes.c_int, [P(PagedKV), P(SparseParams), i32, i32, vp, vp]),
        "kt_build_dynamic_reps": (ctypes.c_int, [P(PagedKV), P(SparseParams), vp, i32, i32, i32,
                                                 vp, vp, vp, sz, vp]),
        "kt_score_select_blocks": (ctypes.c_int, [vp, P(PagedKV), vp, P(SparseParams), vp, vp,
                                                  vp, vp, sz, vp]),
        "kt_sparse_decode_attn": (ctypes.c_int, [vp, P(PagedKV), P(SparseParams), vp, vp, vp,
                                                 vp, sz, vp]),
        "kt_sparse_decode_step": (ctypes.c_int, [vp, P(PagedKV), vp, P(SparseParams), vp, vp,
                                                 vp, vp, sz, vp]),
        "kt_sparse_decode_step_kernels": (i32, [P(PagedKV), P(SparseParams)]),
        "kt_preselect_mask_words": (i32, [P(PagedKV)]),
        "kt_preselect_blocks": (ctypes.c_int, [P(PagedKV), P(SparseParams), vp, i32, i32, i32,
                                               vp, vp, vp, sz, vp]),
        "kt_score_select_blocks_presel": (ctypes.c_int, [vp, P(PagedKV), vp, P(SparseParams),
                                                         vp, vp, vp, vp, vp, sz, vp]),
        "kt_sparse_decode_step_presel": (ctypes.c_int, [vp, P(PagedKV), vp, P(SparseParams),
                                                        vp, vp, vp, vp, vp, vp, sz, vp]),
        "kt_sparse_decode_step_host": (ctypes.c_int, [vp, vp, P(PagedKV), vp, P(SparseParams),
                                                      vp, vp, vp, vp, vp, sz, vp]),
        "kt_dense_decode_attn": (ctypes.c_int, [vp, P(PagedKV), i32, ctypes.c_float, vp, vp, sz,
                                                vp]),
        "kt_read_device_status": (ctypes.c_int, [vp, sz, vp, P(i32)]),
        "kt_selftest_bounded_wait": (ctypes.c_int, [vp, sz, i32, vp]),
        "kt_selftest_step_timeout": (ctypes.c_int, [vp, P(PagedKV), vp, P(SparseParams), vp, vp,
                                                    vp, vp, sz, i32, i32, vp]),
        "kt_noalloc_read_status": (ctypes.c_int, [vp, P(i32)]),
        "kt_sparse_decode_attn_noalloc": (ctypes.c_int, [vp, P(PagedKV), P(SparseParams), vp,
                                                         vp, vp, vp]),
        "kt_decode_history_slots": (i32, [P(ReusePolicy)]),
        "kt_decode_layer_action": (ctypes.c_int, [P(ReusePolicy), i32, i32, P(i32), P(i32)]),
        "kt_decode_layer": (ctypes.c_int, [P(ReusePolicy), i32, i32, vp, P(PagedKV), vp,
                                           P(SparseParams), vp, vp, vp, vp, sz, vp]),
        "kt_append_kv": (ctypes.c_int, [P(PagedKV), P(SparseParams), vp, vp, vp, vp, sz, vp]),
        "kt_set_max_ctas": (ctypes.c_int, [i32]),
        "kt_set_phase_stamps": (ctypes.c_int, [vp, i32]),
        "kt_sparse_decode_attn_hostkv": (ctypes.c_int, [vp, P(PagedKV), P(SparseParams), vp, vp,
                                                        vp, vp, sz, vp]),
        "kt_quantize_kv_q8_0": (ctypes.c_int, [P(PagedKV), vp, vp, vp, vp, i32, i32, vp]),
        "kt_sparse_decode_attn_q8_0": (ctypes.c_int, [vp, P(PagedKVQ8), P(SparseParams), vp, vp,
                                                      vp, vp, sz, vp]),
        "kt_sparse_decode_step_q8_0": (ctypes.c_int, [vp, P(PagedKVQ8), vp, P(SparseParams), vp,
                                                      vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


def status_string(status: int) -> str:
    return lib.kt_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status, call):
    if status != KT_OK:
        raise KtError(status, call)


def paged_kv(k_pool, v_pool, block_table, seq_lens) -> PagedKV:
    """k_pool/v_pool: fp16 [P][H_kv][128][128]; block_table: int32 [B][MB]; seq_lens: int32 [B]."""
    P, H_kv, bs, d = k_pool.shape
    return PagedKV(_ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(seq_lens),
                   int(seq_lens.shape[0]), H_kv, d, bs, int(block_table.shape[1]), P)


def sparse_params(num_q_heads, initial_blocks, local_blocks, top_k, rep, head_mode, *,
                  num_reps=1, fix_stride=32, softmax_scale=None) -> SparseParams:
    if softmax_scale is None:
        softmax_scale = 128 ** -0.5
    return SparseParams(num_q_heads, initial_blocks, local_blocks, top_k, num_reps, fix_stride,
                        rep, head_mode, softmax_scale)


def kt_reps_per_block(params: SparseParams) -> int:
    return int(lib.kt_reps_per_block(ctypes.byref(params)))


def kt_reps_pool_bytes(kv: PagedKV, params: SparseParams) -> int:
    return int(lib.kt_reps_pool_bytes(ctypes.byref(kv), ctypes.byref(params)))


def kt_workspace_bytes(op: int, kv: PagedKV, params: SparseParams, T: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.kt_workspace_bytes(op, ctypes.byref(kv), ctypes.byref(params), T, ctypes.byref(n)),
           "kt_workspace_bytes")
    return int(n.value)


def kt_workspace_init(ws, stream=None):
    _check(lib.kt_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "kt_workspace_init")


def workspace(op: int, kv: PagedKV, params: SparseParams, T: int = 0, device="cuda"):
    """A zero-filled workspace tensor (uint8) for `op`, allocated by torch."""
    import torch
    ws = torch.empty(kt_workspace_bytes(op, kv, params, T), dtype=torch.uint8, device=device)
    kt_workspace_init(ws)
    return ws


def kt_build_block_reps(kv, params, first_block, num_blocks, reps_pool, stream=None):
    _check(lib.kt_build_block_reps(ctypes.byref(kv), ctypes.byref(params), first_block,
                                   num_blocks, _ptr(reps_pool), _stream(stream)),
           "kt_build_block_reps")


def kt_build_dynamic_reps(kv, params, q_local, T, first_block, num_blocks, reps_pool,
                          token_scores, ws, stream=None):
    _check(lib.kt_build_dynamic_reps(ctypes.byref(kv), ctypes.byref(params), _ptr(q_local), T,
                                     first_block, num_blocks, _ptr(reps_pool),
                                     _ptr(token_scores), _ptr(ws), ws.numel(), _stream(stream)),
           "kt_build_dynamic_reps")


def reuse_policy(num_layers, dense_layer_num=0, layer_step=1, token_step=1) -> ReusePolicy:
    return ReusePolicy(num_layers, dense_layer_num, layer_step, token_step)


def kt_decode_history_slots(pol) -> int:
    n = lib.kt_decode_history_slots(ctypes.byref(pol))
    if n < 0:
        raise KtError(-n, "kt_decode_history_slots")
    return n


def kt_decode_layer_action(pol, token_idx, layer_idx):
    """(action, slot) of decode step token_idx at layer layer_idx."""
    a, sl = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.kt_decode_layer_action(ctypes.byref(pol), token_idx, layer_idx, ctypes.byref(a),
                                      ctypes.byref(sl)), "kt_decode_layer_action")
    return a.value, sl.value


def kt_decode_layer(pol, token_idx, layer_idx, q, kv, reps_pool, params, hist_sel, hist_cnt, out,
                    ws, stream=None):
    _check(lib.kt_decode_layer(ctypes.byref(pol), token_idx, layer_idx, _ptr(q), ctypes.byref(kv),
                               _ptr(reps_pool), ctypes.byref(params), _ptr(hist_sel),
                               _ptr(hist_cnt), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "kt_decode_layer")


def kt_append_kv(kv, params, k_new, v_new, reps_pool, ws, stream=None):
    _check(lib.kt_append_kv(ctypes.byref(kv), ctypes.byref(params), _ptr(k_new), _ptr(v_new),
                            _ptr(reps_pool), _ptr(ws), ws.numel(), _stream(stream)),
           "kt_append_kv")


def kt_preselect_mask_words(kv):
    n = lib.kt_preselect_mask_words(ctypes.byref(kv))
    if n < 0:
        raise KtError(-n, "kt_preselect_mask_words")
    return n


def kt_preselect_blocks(kv, params, q_local, T, kernel_size, count, presel_mask, presel_cnt, ws,
                        stream=None):
    _check(lib.kt_preselect_blocks(ctypes.byref(kv), ctypes.byref(params), _ptr(q_local), T,
                                   kernel_size, count, _ptr(presel_mask), _ptr(presel_cnt),
                                   _ptr(ws), ws.numel(), _stream(stream)),
           "kt_preselect_blocks")


def kt_score_select_blocks_presel(q, kv, reps_pool, params, presel_mask, sel, cnt, sel_scores,
                                  ws, stream=None):
    _check(lib.kt_score_select_blocks_presel(_ptr(q), ctypes.byref(kv), _ptr(reps_pool),
                                             ctypes.byref(params), _ptr(presel_mask), _ptr(sel),
                                             _ptr(cnt), _ptr(sel_scores), _ptr(ws), ws.numel(),
                                             _stream(stream)),
           "kt_score_select_blocks_presel")


def kt_sparse_decode_step_presel(q, kv, reps_pool, params, presel_mask, presel_cnt, sel, cnt,
                                 out, ws, stream=None):
    _check(lib.kt_sparse_decode_step_presel(_ptr(q), ctypes.byref(kv), _ptr(reps_pool),
                                            ctypes.byref(params), _ptr(presel_mask),
                                            _ptr(presel_cnt), _ptr(sel), _ptr(cnt), _ptr(out),
                                            _ptr(ws), ws.numel(), _stream(stream)),
           "kt_sparse_decode_step_presel")


def kt_score_select_blocks(q, kv, reps_pool, params, sel, cnt, sel_scores, ws, stream=None):
    _check(lib.kt_score_select_blocks(_ptr(q), ctypes.byref(kv), _ptr(reps_pool),
                                      ctypes.byref(params), _ptr(sel), _ptr(cnt),
                                      _ptr(sel_scores), _ptr(ws), ws.numel(), _stream(stream)),
           "kt_score_select_blocks")


def kt_sparse_decode_attn(q, kv, params, sel, cnt, out, ws, stream=None):
    _check(lib.kt_sparse_decode_attn(_ptr(q), ctypes.byref(kv), ctypes.byref(params), _ptr(sel),
                                     _ptr(cnt), _ptr(out), _ptr(ws), ws.numel(),
                                     _stream(stream)),
           "kt_sparse_decode_attn")


def kt_sparse_decode_step(q, kv, reps_pool, params, sel, cnt, out, ws, stream=None):
    _check(lib.kt_sparse_decode_step(_ptr(q), ctypes.byref(kv), _ptr(reps_pool),
                                     ctypes.byref(params), _ptr(sel), _ptr(cnt), _ptr(out),
                                     _ptr(ws), ws.numel(), _stream(stream)),
           "kt_sparse_decode_step")


def kt_sparse_decode_step_kernels(kv, params):
    """Launches per kt_sparse_decode_step for this shape: 1 (one cooperative
    launch) or 2 (selection + attention)."""
    n = lib.kt_sparse_decode_step_kernels(ctypes.byref(kv), ctypes.byref(params))
    if n < 0:
        raise KtError(-n, "kt_sparse_decode_step_kernels")
    return n


def kt_sparse_decode_attn_hostkv(q, kv, params, sel, cnt, out, ws, stream=None):
    """kt_sparse_decode_attn with kv's K/V pools in page-locked host memory."""
    _check(lib.kt_sparse_decode_attn_hostkv(_ptr(q), ctypes.byref(kv), ctypes.byref(params),
                                            _ptr(sel), _ptr(cnt), _ptr(out), _ptr(ws), ws.numel(),
                                            _stream(stream)),
           "kt_sparse_decode_attn_hostkv")


def paged_kv_q8(k_code, k_scale, v_code, v_scale, block_table, seq_lens) -> PagedKVQ8:
    P, H_kv, bs, d = k_code.shape
    return PagedKVQ8(_ptr(k_code), _ptr(k_scale), _ptr(v_code), _ptr(v_scale), _ptr(block_table),
                     _ptr(seq_lens), seq_lens.numel(), H_kv, d, bs, block_table.shape[1], P)


def kt_quantize_kv_q8_0(kv, k_code, k_scale, v_code, v_scale, first_page=0, num_pages=None,
                        stream=None):
    n = kv.num_pages - first_page if num_pages is None else num_pages
    _check(lib.kt_quantize_kv_q8_0(ctypes.byref(kv), _ptr(k_code), _ptr(k_scale), _ptr(v_code),
                                   _ptr(v_scale), first_page, n, _stream(stream)),
           "kt_quantize_kv_q8_0")


def kt_sparse_decode_step_q8_0(q, kvq, reps_pool, params, sel, cnt, out, ws, stream=None):
    _check(lib.kt_sparse_decode_step_q8_0(_ptr(q), ctypes.byref(kvq), _ptr(reps_pool),
                                          ctypes.byref(params), _ptr(sel), _ptr(cnt), _ptr(out),
                                          _ptr(ws), ws.numel(), _stream(stream)),
           "kt_sparse_decode_step_q8_0")


def kt_sparse_decode_attn_q8_0(q, kvq, params, sel, cnt, out, ws, stream=None):
    _check(lib.kt_sparse_decode_attn_q8_0(_ptr(q), ctypes.byref(kvq), ctypes.byref(params),
                                          _ptr(sel), _ptr(cnt), _ptr(out), _ptr(ws), ws.numel(),
                                          _stream(stream)),
           "kt_sparse_decode_attn_q8_0")


def kt_set_phase_stamps(stamps, max_ctas: int = 0):
    """Record per-CTA phase stamps of this thread's attention launches into a
    uint64 device tensor of >= max_ctas * 16 entries (None: off)."""
    if stamps is None:
        _check(lib.kt_set_phase_stamps(None, 0), "kt_set_phase_stamps")
    else:
        _check(lib.kt_set_phase_stamps(_ptr(stamps), int(max_ctas or stamps.numel() // 16)),
               "kt_set_phase_stamps")


def kt_set_max_ctas(max_ctas: int):
    """Cap the CTAs of this thread's attention launches (0: one per SM)."""
    _check(lib.kt_set_max_ctas(int(max_ctas)), "kt_set_max_ctas")


def kt_sparse_decode_step_host(q_host, q_dev, kv, reps_pool, params, sel, cnt, out_dev,
                               out_host, ws, stream=None):
    _check(lib.kt_sparse_decode_step_host(_ptr(q_host), _ptr(q_dev), ctypes.byref(kv),
                                          _ptr(reps_pool), ctypes.byref(params), _ptr(sel),
                                          _ptr(cnt), _ptr(out_dev), _ptr(out_host), _ptr(ws),
                                          ws.numel(), _stream(stream)),
           "kt_sparse_decode_step_host")


def kt_dense_decode_attn(q, kv, num_q_heads, softmax_scale, out, ws, stream=None):
    _check(lib.kt_dense_decode_attn(_ptr(q), ctypes.byref(kv), num_q_heads, softmax_scale,
                                    _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "kt_dense_decode_attn")


def kt_read_device_status(ws, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib.kt_read_device_status(_ptr(ws), ws.numel(), _stream(stream), ctypes.byref(v)),
           "kt_read_device_status")
    return int(v.value)


def kt_selftest_bounded_wait(ws, spin_limit, stream=None):
    _check(lib.kt_selftest_bounded_wait(_ptr(ws), ws.numel(), spin_limit, _stream(stream)),
           "kt_selftest_bounded_wait")


def kt_sparse_decode_attn_noalloc(q, kv, params, sel, cnt, out, stream=None):
    """kt_sparse_decode_attn without a workspace (scratch in a fixed 1 MiB
    device array of the library); for callers that cannot allocate."""
    _check(lib.kt_sparse_decode_attn_noalloc(_ptr(q), ctypes.byref(kv), ctypes.byref(params),
                                             _ptr(sel), _ptr(cnt), _ptr(out), _stream(stream)),
           "kt_sparse_decode_attn_noalloc")
