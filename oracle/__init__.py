"""CPU oracle for block-sparse long-context decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The product path
(``block_sparse_long_quest_gb300``) never imports this package, and this
package never imports the product.

The arithmetic lives in ``kt_oracle.c`` (plain single-threaded C, double
precision); this module only compiles it and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kt_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

REP_MAX, REP_MEAN, REP_QUEST, REP_FIX, REP_DYNAMIC = 0, 1, 2, 3, 4
HEAD_SHARED, HEAD_SEPARATE = 0, 1


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _KV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("H_kv", ctypes.c_int64), ("d", ctypes.c_int64),
                ("bs", ctypes.c_int64), ("max_blocks", ctypes.c_int64), ("P", ctypes.c_int64)]


class _Params(ctypes.Structure):
    _fields_ = [("H_q", ctypes.c_int64), ("initial_blocks", ctypes.c_int64),
                ("local_blocks", ctypes.c_int64), ("top_k", ctypes.c_int64),
                ("rep", ctypes.c_int64), ("head_mode", ctypes.c_int64),
                ("num_reps", ctypes.c_int64), ("fix_stride", ctypes.c_int64),
                ("softmax_scale", ctypes.c_double)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        L.orc_f16_to_double.restype = ctypes.c_double
        L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_f16_array.restype = None
        L.orc_f16_array.argtypes = [vp, vp, i64]
        L.orc_partition.restype = None
        L.orc_partition.argtypes = [i64, i64, i64, i64, vp, vp, vp]
        L.orc_reps_per_block.restype = i64
        L.orc_reps_per_block.argtypes = [vp, i64]
        L.orc_block_reps.restype = None
        L.orc_block_reps.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        L.orc_dynamic_token_scores.restype = None
        L.orc_dynamic_token_scores.argtypes = [vp, i64, i64, vp, vp, i64, vp]
        L.orc_head_block_score.restype = ctypes.c_double
        L.orc_head_block_score.argtypes = [vp, vp, i64, i64, i64]
        L.orc_select.restype = i64
        L.orc_select.argtypes = [vp, i64, i64, i64, vp]
        L.orc_attend.restype = None
        L.orc_attend.argtypes = [vp, i64, i64, i64, vp, vp, i64, ctypes.c_double, vp]
        L.orc_dense.restype = None
        L.orc_dense.argtypes = [vp, vp, i64, ctypes.c_double, vp]
        L.orc_build_all_reps.restype = ctypes.c_int
        L.orc_build_all_reps.argtypes = [vp, vp, vp, i64, vp, vp, vp, vp, i64, i64]
        L.orc_score_select_attend.restype = ctypes.c_int
        L.orc_score_select_attend.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64]
        L.orc_sparse_step.restype = ctypes.c_int
        L.orc_sparse_step.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, i64, i64]
        L.orc_sparse_step_presel.restype = ctypes.c_int
        L.orc_sparse_step_presel.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, i64, i64, vp,
                                             vp, i64]
        L.orc_avg_pool1d.restype = None
        L.orc_avg_pool1d.argtypes = [vp, i64, i64, vp]
        L.orc_preselect.restype = ctypes.c_int
        L.orc_preselect.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp]
        L.orc_f32_to_f16.restype = ctypes.c_uint16
        L.orc_f32_to_f16.argtypes = [ctypes.c_float]
        L.orc_quantize_q8_0.restype = None
        L.orc_quantize_q8_0.argtypes = [vp, i64, vp, vp]
        L.orc_attend_q8.restype = None
        L.orc_attend_q8.argtypes = [vp, i64, i64, i64, vp, vp, i64, ctypes.c_double, vp]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class KV:
    """Paged KV view handed to the C oracle (keeps the arrays alive)."""

    def __init__(self, k_pool, v_pool, block_table, seq_lens, block_size=128):
        self.k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
        self.v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
        self.block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        self.seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        P, H_kv, bs, d = self.k_pool.shape
        assert bs == block_size
        self.H_kv, self.d, self.bs, self.P = H_kv, d, bs, P
        self.B = self.seq_lens.size
        self.max_blocks = self.block_table.shape[1]
        self.s = _KV(self.k_pool.ctypes.data, self.v_pool.ctypes.data,
                     self.block_table.ctypes.data, self.seq_lens.ctypes.data,
                     self.B, H_kv, d, bs, self.max_blocks, P)

    @classmethod
    def of(cls, w):
        return cls(w.k_pool, w.v_pool, w.block_table, w.seq_lens)


class _KVQ(ctypes.Structure):
    _fields_ = [("k_code", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_code", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("H_kv", ctypes.c_int64), ("d", ctypes.c_int64),
                ("bs", ctypes.c_int64), ("max_blocks", ctypes.c_int64), ("P", ctypes.c_int64)]


def f32_to_f16(x: float) -> int:
    """binary32 -> binary16 bits, round to nearest even."""
    return int(lib().orc_f32_to_f16(ctypes.c_float(x)))


def quantize_q8_0(bits):
    """[..., 128] binary16 bits -> (codes int8 [..., 128], scales binary16 bits [..., 4])
    (the oracle's Q8_0 reading: 4 groups of 32 channels per row)."""
    x = np.ascontiguousarray(bits, dtype=np.uint16)
    rows = x.size // 128
    code = np.zeros(x.shape, dtype=np.int8)
    scale = np.zeros(x.shape[:-1] + (4,), dtype=np.uint16)
    lib().orc_quantize_q8_0(x.ctypes.data, rows, code.ctypes.data, scale.ctypes.data)
    return code, scale


class KVQ:
    """Q8_0 K/V pools (codes + binary16 scales) with the block table of a KV."""

    def __init__(self, kv: "KV"):
        self.kv = kv
        self.k_code, self.k_scale = quantize_q8_0(kv.k_pool)
        self.v_code, self.v_scale = quantize_q8_0(kv.v_pool)
        self.s = _KVQ(self.k_code.ctypes.data, self.k_scale.ctypes.data,
                      self.v_code.ctypes.data, self.v_scale.ctypes.data,
                      kv.block_table.ctypes.data, kv.seq_lens.ctypes.data,
                      kv.B, kv.H_kv, kv.d, kv.bs, kv.max_blocks, kv.P)


def attend_q8(kvq: KVQ, b: int, hq: int, num_q_heads: int, q_bits, blocks, scale: float):
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bl = np.ascontiguousarray(blocks, dtype=np.int32)
    out = np.zeros(kvq.kv.d, dtype=np.float64)
    lib().orc_attend_q8(ctypes.byref(kvq.s), b, hq, num_q_heads, q.ctypes.data, bl.ctypes.data,
                        bl.size, scale, out.ctypes.data)
    return out


def attend_selection_q8(kvq: KVQ, q, p, sel, cnt) -> np.ndarray:
    """attend_selection over the dequantised Q8_0 K and V: [B][H_q][d]."""
    kv = kvq.kv
    q = np.ascontiguousarray(q, dtype=np.uint16)
    H_q = p.num_q_heads
    G = H_q // kv.H_kv
    out = np.zeros((kv.B, H_q, kv.d), dtype=np.float64)
    for b in range(kv.B):
        nb, c0, c1 = partition(int(kv.seq_lens[b]), p.initial_blocks, p.local_blocks, kv.bs)
        for hq in range(H_q):
            u = 0 if p.head_mode == HEAD_SHARED else hq // G
            blocks = list(range(c0)) + [int(j) for j in sel[b, u, :int(cnt[b, u])]] + \
                list(range(c1, nb))
            out[b, hq] = attend_q8(kvq, b, hq, H_q, q[b, hq], blocks, p.softmax_scale)
    return out


def params(p) -> _Params:
    return _Params(p.num_q_heads, p.initial_blocks, p.local_blocks, p.top_k, p.rep,
                   p.head_mode, p.num_reps, p.fix_stride, float(p.softmax_scale))


def f16_to_double(bits) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().orc_f16_array(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def partition(n: int, initial_blocks: int, local_blocks: int, block_size: int = 128):
    a = (ctypes.c_int64 * 3)()
    lib().orc_partition(n, block_size, initial_blocks, local_blocks, ctypes.byref(a, 0),
                        ctypes.byref(a, 8), ctypes.byref(a, 16))
    return int(a[0]), int(a[1]), int(a[2])


def reps_per_block(p, block_size: int = 128) -> int:
    pp = params(p)
    return int(lib().orc_reps_per_block(ctypes.byref(pp), block_size))


def block_reps(kv: KV, p, b: int, j: int, h: int, dyn_scores=None):
    pp = params(p)
    R = reps_per_block(p, kv.bs)
    h16 = np.zeros((R, kv.d), dtype=np.uint16)
    f32 = np.zeros(kv.d, dtype=np.float32)
    ds = None if dyn_scores is None else np.ascontiguousarray(dyn_scores, dtype=np.float64)
    lib().orc_block_reps(ctypes.byref(kv.s), b, j, h, ctypes.byref(pp), _ptr(ds),
                         h16.ctypes.data, f32.ctypes.data)
    return f32 if p.rep == REP_MEAN else h16


def dynamic_token_scores(kv: KV, p, b: int, h: int, q_local_b):
    pp = params(p)
    ql = np.ascontiguousarray(q_local_b, dtype=np.uint16)
    n = int(kv.seq_lens[b])
    acc = np.zeros(max(n, 1), dtype=np.float64)
    lib().orc_dynamic_token_scores(ctypes.byref(kv.s), b, h, ctypes.byref(pp), ql.ctypes.data,
                                   ql.shape[0], acc.ctypes.data)
    return acc[:n]


def head_block_score(q, reps, rep: int) -> float:
    q = np.ascontiguousarray(q, dtype=np.float64)
    reps = np.ascontiguousarray(reps, dtype=np.float64)
    R, d = reps.shape
    return float(lib().orc_head_block_score(q.ctypes.data, reps.ctypes.data, R, d, rep))


def select(scores, c0: int, k: int) -> np.ndarray:
    s = np.ascontiguousarray(scores, dtype=np.float64)
    sel = np.zeros(max(k, 1), dtype=np.int32)
    cnt = lib().orc_select(s.ctypes.data, c0, s.size, k, sel.ctypes.data)
    return sel[:cnt]


def attend(kv: KV, b: int, hq: int, num_q_heads: int, q_bits, blocks, scale: float):
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bl = np.ascontiguousarray(blocks, dtype=np.int32)
    out = np.zeros(kv.d, dtype=np.float64)
    lib().orc_attend(ctypes.byref(kv.s), b, hq, num_q_heads, q.ctypes.data, bl.ctypes.data,
                     bl.size, scale, out.ctypes.data)
    return out


def dense(kv: KV, q, num_q_heads: int, scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint16)
    out = np.zeros((kv.B, num_q_heads, kv.d), dtype=np.float64)
    lib().orc_dense(ctypes.byref(kv.s), q.ctypes.data, num_q_heads, scale, out.ctypes.data)
    return out


def sparse_step(kv: KV, q, p, q_local=None, *, units=None, want_reps=True,
                want_dyn_scores=False):
    """One decode step of the method; returns a dict of numpy outputs.

    reps are indexed by LOGICAL block: [B][max_blocks][H_kv][R][d] (binary16
    bits) or [B][max_blocks][H_kv][d] (Mean, binary32).  unit_scores is
    [B][SEL][max_blocks] with NaN outside the context range.
    """
    pp = params(p)
    B, H_kv, d, MB = kv.B, kv.H_kv, kv.d, kv.max_blocks
    R = reps_per_block(p, kv.bs)
    SEL = 1 if p.head_mode == HEAD_SHARED else H_kv
    lo, hi = (0, SEL) if units is None else units
    q = np.ascontiguousarray(q, dtype=np.uint16)
    ql = None if q_local is None else np.ascontiguousarray(q_local, dtype=np.uint16)
    T = 0 if ql is None else ql.shape[1]
    reps_h16 = reps_f32 = None
    if want_reps:
        if p.rep == REP_MEAN:
            reps_f32 = np.zeros((B, MB, H_kv, d), dtype=np.float32)
        else:
            reps_h16 = np.zeros((B, MB, H_kv, R, d), dtype=np.uint16)
    dyn = np.zeros((B, H_kv, MB * kv.bs), dtype=np.float64) if want_dyn_scores else None
    us = np.full((B, SEL, MB), np.nan, dtype=np.float64)
    sel = np.full((B, SEL, max(p.top_k, 1)), -1, dtype=np.int32)
    cnt = np.zeros((B, SEL), dtype=np.int32)
    out = np.zeros((B, p.num_q_heads, d), dtype=np.float64)
    rc = lib().orc_sparse_step(ctypes.byref(kv.s), q.ctypes.data, ctypes.byref(pp), _ptr(ql), T,
                               _ptr(reps_h16), _ptr(reps_f32), _ptr(dyn), us.ctypes.data,
                               sel.ctypes.data, cnt.ctypes.data, out.ctypes.data, lo, hi)
    if rc != 0:
        raise ValueError("oracle rejected the parameters")
    return dict(reps=reps_f32 if p.rep == REP_MEAN else reps_h16, unit_scores=us, sel=sel,
                cnt=cnt, out=out, dyn_scores=dyn)


def score_select_attend(kv: KV, q, p, rv, *, units=None):
    """Score, select and attend ([LC §3.1, §4.3, §4.5, §4.6]) over given
    representative values rv [B][max_blocks][H_kv][R][d] (double, by logical
    block); returns unit_scores, sel, cnt, out as sparse_step does."""
    pp = params(p)
    B, H_kv, d, MB = kv.B, kv.H_kv, kv.d, kv.max_blocks
    R = reps_per_block(p, kv.bs)
    rv = np.ascontiguousarray(rv, dtype=np.float64)
    if rv.shape != (B, MB, H_kv, R, d):
        raise ValueError(f"rv must be [B][max_blocks][H_kv][R][d] = {(B, MB, H_kv, R, d)}")
    SEL = 1 if p.head_mode == HEAD_SHARED else H_kv
    lo, hi = (0, SEL) if units is None else units
    q = np.ascontiguousarray(q, dtype=np.uint16)
    us = np.full((B, SEL, MB), np.nan, dtype=np.float64)
    sel = np.full((B, SEL, max(p.top_k, 1)), -1, dtype=np.int32)
    cnt = np.zeros((B, SEL), dtype=np.int32)
    out = np.zeros((B, p.num_q_heads, d), dtype=np.float64)
    rc = lib().orc_score_select_attend(ctypes.byref(kv.s), q.ctypes.data, ctypes.byref(pp),
                                       rv.ctypes.data, us.ctypes.data, sel.ctypes.data,
                                       cnt.ctypes.data, out.ctypes.data, lo, hi)
    if rc != 0:
        raise ValueError("oracle rejected the parameters")
    return dict(unit_scores=us, sel=sel, cnt=cnt, out=out)


def avg_pool1d(x, kernel: int) -> np.ndarray:
    """Zero-padded average pooling, window kernel (odd), stride 1 [LC §4.6]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().orc_avg_pool1d(x.ctypes.data, x.size, kernel, out.ctypes.data)
    return out


def preselect(kv: KV, p, q_local, kernel: int, count: int):
    """Preselected context blocks per unit [LC §4.4, §4.6 preselect_block()]:
    (presel [B][SEL][count] ascending, -1 padded; presel_cnt [B][SEL])."""
    pp = params(p)
    SEL = 1 if p.head_mode == HEAD_SHARED else kv.H_kv
    ql = np.ascontiguousarray(q_local, dtype=np.uint16)
    presel = np.full((kv.B, SEL, count), -1, dtype=np.int32)
    pcnt = np.zeros((kv.B, SEL), dtype=np.int32)
    rc = lib().orc_preselect(ctypes.byref(kv.s), ctypes.byref(pp), ql.ctypes.data, ql.shape[1],
                             kernel, count, presel.ctypes.data, pcnt.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the preselection parameters")
    return presel, pcnt


def sparse_step_presel(kv: KV, q, p, presel, presel_cnt, q_local=None, *, units=None):
    """sparse_step with each unit's selection restricted to its preselected
    blocks; returns sel, cnt, out, unit_scores."""
    pp = params(p)
    B, d, MB = kv.B, kv.d, kv.max_blocks
    SEL = 1 if p.head_mode == HEAD_SHARED else kv.H_kv
    lo, hi = (0, SEL) if units is None else units
    q = np.ascontiguousarray(q, dtype=np.uint16)
    ql = None if q_local is None else np.ascontiguousarray(q_local, dtype=np.uint16)
    T = 0 if ql is None else ql.shape[1]
    presel = np.ascontiguousarray(presel, dtype=np.int32)
    pcnt = np.ascontiguousarray(presel_cnt, dtype=np.int32)
    us = np.full((B, SEL, MB), np.nan, dtype=np.float64)
    sel = np.full((B, SEL, max(p.top_k, 1)), -1, dtype=np.int32)
    cnt = np.zeros((B, SEL), dtype=np.int32)
    out = np.zeros((B, p.num_q_heads, d), dtype=np.float64)
    rc = lib().orc_sparse_step_presel(ctypes.byref(kv.s), q.ctypes.data, ctypes.byref(pp),
                                      _ptr(ql), T, us.ctypes.data, sel.ctypes.data,
                                      cnt.ctypes.data, out.ctypes.data, lo, hi,
                                      presel.ctypes.data, pcnt.ctypes.data, presel.shape[-1])
    if rc != 0:
        raise ValueError("oracle rejected the parameters")
    return dict(unit_scores=us, sel=sel, cnt=cnt, out=out)


# ---- decoding with selection reuse [LC §4.5 token_step / layer_step /
# dense_layer_num; §4.6 decode loop] -------------------------------------------
LAYER_DENSE, LAYER_SELECT, LAYER_REUSE = 0, 1, 2


def decode_layer_action(num_layers: int, dense_layer_num: int, layer_step: int,
                        token_step: int, token_idx: int, layer_idx: int):
    """(action, slot) of decode step token_idx at layer layer_idx.

    The first dense_layer_num layers attend every block ([LC §4.5]).  The
    decode loop of [LC §4.6] reselects at (token, layer) when token % token_step
    == 0 and layer % layer_step == 0 and otherwise reuses the selection kept
    for layer // layer_step; here the layer index is counted among the sparse
    layers (layer - dense_layer_num), so every slot is written before it is
    read."""
    if not (num_layers >= 1 and 0 <= dense_layer_num <= num_layers and layer_step >= 1
            and token_step >= 1 and token_idx >= 0 and 0 <= layer_idx < num_layers):
        raise ValueError("invalid policy or index")
    if layer_idx < dense_layer_num:
        return LAYER_DENSE, -1
    l = layer_idx - dense_layer_num
    if token_idx % token_step == 0 and l % layer_step == 0:
        return LAYER_SELECT, l // layer_step
    return LAYER_REUSE, l // layer_step


def attend_selection(kv: KV, q, p, sel, cnt) -> np.ndarray:
    """Attention of every query head over Initial + the given selection of
    its unit + Local at the current lengths ([LC §4.6] attn over
    kvcache_after_retrieval), as [B][H_q][d]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    H_q = p.num_q_heads
    G = H_q // kv.H_kv
    out = np.zeros((kv.B, H_q, kv.d), dtype=np.float64)
    for b in range(kv.B):
        nb, c0, c1 = partition(int(kv.seq_lens[b]), p.initial_blocks, p.local_blocks, kv.bs)
        for hq in range(H_q):
            u = 0 if p.head_mode == HEAD_SHARED else hq // G
            blocks = list(range(c0)) + [int(j) for j in sel[b, u, :int(cnt[b, u])]] + \
                list(range(c1, nb))
            out[b, hq] = attend(kv, b, hq, H_q, q[b, hq], blocks, p.softmax_scale)
    return out


class StepTimer:
    """The per-step part of the oracle (score, select, attend) over reps built
    once up front; used to time the CPU baseline on the same work as one GPU
    decode step."""

    def __init__(self, kv: KV, p, q_local=None):
        self.kv, self.p = kv, p
        self.pp = params(p)
        R = reps_per_block(p, kv.bs)
        self.rv = np.zeros((kv.B, kv.max_blocks, kv.H_kv, R, kv.d), dtype=np.float64)
        ql = None if q_local is None else np.ascontiguousarray(q_local, dtype=np.uint16)
        T = 0 if ql is None else ql.shape[1]
        SEL = 1 if p.head_mode == HEAD_SHARED else kv.H_kv
        rc = lib().orc_build_all_reps(ctypes.byref(kv.s), ctypes.byref(self.pp), _ptr(ql), T,
                                      self.rv.ctypes.data, None, None, None, 0, SEL)
        if rc != 0:
            raise ValueError("oracle rejected the parameters")
        self.SEL = SEL
        self.sel = np.zeros((kv.B, SEL, max(p.top_k, 1)), dtype=np.int32)
        self.cnt = np.zeros((kv.B, SEL), dtype=np.int32)
        self.out = np.zeros((kv.B, p.num_q_heads, kv.d), dtype=np.float64)

    def step(self, q):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        rc = lib().orc_score_select_attend(ctypes.byref(self.kv.s), q.ctypes.data,
                                           ctypes.byref(self.pp), self.rv.ctypes.data, None,
                                           self.sel.ctypes.data, self.cnt.ctypes.data,
                                           self.out.ctypes.data, 0, self.SEL)
        if rc != 0:
            raise ValueError("oracle rejected the parameters")
        return self.out
