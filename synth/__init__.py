"""Seeded synthetic inputs for block-sparse long-context decode attention.

This package is the only code that the CUDA path's tests/benchmark and the CPU
oracle share.  It draws random numbers and lays them out; it holds none of the
method's arithmetic (no representatives, scores, selection or attention).

Shapes follow the workloads of the KTransformers long-context sparse attention
article ("KTransformers 长上下文稀疏注意力实战：单张 24GB GPU 跑通 1M Token
KVCache 的完整方案"): InternLM2.5-7B-Chat-1M-style layers with 32 query heads,
8 KV heads, head_dim 128, fp16 KV cut into 128-token blocks (§1, §4.3, §5.1,
§6.2 memory table: 4 KiB of K+V per token per layer).

Random numbers: SplitMix64 as a counter-based generator and the Box-Muller
transform, rounded once to binary16 (see synth.c).  Each tensor draws from its
own stream; stream ids are the STREAM_* constants below (+ 16 * layer).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

BLOCK = 128
HEAD_DIM = 128

# Stream ids (one per tensor kind; + 16 * layer for multi-layer workloads).
STREAM_K = 1
STREAM_V = 2
STREAM_Q = 3
STREAM_QLOCAL = 4
STREAM_NEEDLE = 5
STREAM_LENS = 6
STREAM_PERM = 7
STREAM_OUTLIER = 8

# Rep method and head-mode codes (same numbering as the C interface).
REP_MAX, REP_MEAN, REP_QUEST, REP_FIX, REP_DYNAMIC = 0, 1, 2, 3, 4
HEAD_SHARED, HEAD_SEPARATE = 0, 1
REP_NAMES = {REP_MAX: "max", REP_MEAN: "mean", REP_QUEST: "quest", REP_FIX: "fix",
             REP_DYNAMIC: "dynamic"}


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, portable C)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, i64, vp, dp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.synth_u64.restype = u64
        L.synth_u64.argtypes = [u64, u64, u64]
        L.synth_fill_u64.restype = None
        L.synth_fill_u64.argtypes = [vp, u64, u64, u64, u64]
        L.synth_f16_from_double.restype = ctypes.c_uint16
        L.synth_f16_from_double.argtypes = [dp]
        L.synth_fill_normal_f16.restype = ctypes.c_int
        L.synth_fill_normal_f16.argtypes = [vp, u64, u64, u64, u64, dp, dp, vp, i64, ctypes.c_int]
        L.synth_fill_normal_f64.restype = None
        L.synth_fill_normal_f64.argtypes = [vp, u64, u64, u64, u64]
        L.synth_f16_from_double_array.restype = None
        L.synth_f16_from_double_array.argtypes = [vp, vp, u64]
        _lib = L
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def u64(seed: int, stream: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_fill_u64(out.ctypes.data, n, seed, stream, first)
    return out


def normal_f16(shape, seed: int, stream: int, *, mean: float = 0.0, sigma: float = 1.0,
               chan_scale: Optional[np.ndarray] = None, out: Optional[np.ndarray] = None,
               first: int = 0) -> np.ndarray:
    """binary16 bit patterns (uint16) of mean + sigma*scale[c]*N(0,1)."""
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    cs = None
    d = 0
    if chan_scale is not None:
        cs = np.ascontiguousarray(chan_scale, dtype=np.float64)
        d = cs.size
    rc = lib().synth_fill_normal_f16(out.ctypes.data, n, seed, stream, first, mean, sigma,
                                     cs.ctypes.data if cs is not None else None, d, _threads())
    assert rc == 0
    return out


def fill_normal_f16_ptr(addr: int, n: int, seed: int, stream: int, *, first: int = 0,
                        sigma: float = 1.0, chan_scale: Optional[np.ndarray] = None) -> None:
    """Same as normal_f16 but into raw host memory (e.g. a pinned torch tensor)."""
    cs = None
    d = 0
    if chan_scale is not None:
        cs = np.ascontiguousarray(chan_scale, dtype=np.float64)
        d = cs.size
    rc = lib().synth_fill_normal_f16(addr, n, seed, stream, first, 0.0, sigma,
                                     cs.ctypes.data if cs is not None else None, d, _threads())
    assert rc == 0


def normal_f64(n: int, seed: int, stream: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_fill_normal_f64(out.ctypes.data, n, seed, stream, first)
    return out


def f16_bits(x: np.ndarray) -> np.ndarray:
    """Round doubles to binary16 (nearest-even) with the generator's encoder."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().synth_f16_from_double_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def uniform_ints(n: int, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive), by Lemire-free modulo of the top
    bits; the bias is below 2^-40 for the ranges used here."""
    w = u64(seed, stream, n)
    span = hi - lo + 1
    return (lo + ((w >> np.uint64(11)) % np.uint64(span)).astype(np.int64)).astype(np.int64)


def permutation(n: int, seed: int, stream: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by the stream (Knuth, TAOCP 3.4.2)."""
    w = u64(seed, stream, max(n, 1))
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(w[i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Params:
    """Selection parameters (names follow the article's §4.5 parameter list)."""
    num_q_heads: int
    initial_blocks: int          # Initial part, in 128-token blocks (§4.2)
    local_blocks: int            # Local window, in blocks (local_windows_len / 128)
    top_k: int                   # second_select_num / second_block_count
    rep: int                     # representative_type / anchor_type
    head_mode: int               # head_select_mode: SHARED or SEPARATE
    num_reps: int = 1            # representative_num / anchor_num
    fix_stride: int = 32         # stride of the Fix method (4 reps per block at 32)
    softmax_scale: float = 1.0 / np.sqrt(HEAD_DIM)

    def reps_per_block(self) -> int:
        if self.rep in (REP_MAX, REP_MEAN):
            return 1
        if self.rep == REP_QUEST:
            return 2
        if self.rep == REP_FIX:
            return BLOCK // self.fix_stride
        return self.num_reps


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    k_pool: np.ndarray            # uint16 [P][H_kv][128][128]  (binary16 bits)
    v_pool: np.ndarray            # uint16 [P][H_kv][128][128]
    block_table: np.ndarray       # int32 [B][max_blocks]
    seq_lens: np.ndarray          # int32 [B]
    q: np.ndarray                 # uint16 [B][H_q][128]
    params: Params
    q_local: Optional[np.ndarray] = None   # uint16 [B][T][H_q][128]
    needles: Optional[list] = None         # [(b, block)]

    @property
    def batch(self):
        return int(self.seq_lens.shape[0])

    @property
    def num_kv_heads(self):
        return int(self.k_pool.shape[1])

    @property
    def num_pages(self):
        return int(self.k_pool.shape[0])

    @property
    def max_blocks(self):
        return int(self.block_table.shape[1])


def needle_blocks(initial_blocks: int, num_ctx: int, count: int) -> list:
    """Context blocks spread evenly: I_b + floor((j + 1/2) * C / count)."""
    return [initial_blocks + int((j + 0.5) * num_ctx // count) for j in range(count)]


def plant_needles(k_pool, block_table, q, b, blocks, seed, stream, *, gain=2.0, sigma=0.5):
    """Keys of a planted block: gain * (mean of the group's query heads) + N(0, sigma^2).

    For multi-head attention the group is the single query head of that KV head.
    """
    H_kv = k_pool.shape[1]
    H_q = q.shape[1]
    G = H_q // H_kv
    qd = q[b].view(np.float16).astype(np.float64)           # [H_q][d]
    target = gain * qd.reshape(H_kv, G, HEAD_DIM).mean(axis=1)  # [H_kv][d]
    per_block = H_kv * BLOCK * HEAD_DIM
    for i, j in enumerate(blocks):
        z = normal_f64(per_block, seed, stream, first=(b * 4096 + i) * per_block)
        vals = target[:, None, :] + sigma * z.reshape(H_kv, BLOCK, HEAD_DIM)
        k_pool[block_table[b, j]] = f16_bits(vals)


def make_workload(name: str, *, seed: int, seq_lens, num_q_heads: int, num_kv_heads: int,
                  params: Params, layer: int = 0, permute_pages: bool = False,
                  outlier_channels: int = 0, outlier_gain: float = 8.0,
                  num_needles: int = 0, local_queries: int = 0) -> Workload:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.size
    nbs = [(int(n) + BLOCK - 1) // BLOCK for n in seq_lens]
    max_blocks = max(1, max(nbs))
    P = max(1, sum(nbs))
    so = 16 * layer
    table = np.zeros((B, max_blocks), dtype=np.int32)
    order = permutation(P, seed, STREAM_PERM + so) if permute_pages else np.arange(P)
    off = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = order[off:off + nb]
        off += nb
    scale = None
    if outlier_channels:
        chans = permutation(HEAD_DIM, seed, STREAM_OUTLIER + so)[:outlier_channels]
        scale = np.ones(HEAD_DIM)
        scale[chans] = outlier_gain
    k_pool = normal_f16((P, num_kv_heads, BLOCK, HEAD_DIM), seed, STREAM_K + so, chan_scale=scale)
    v_pool = normal_f16((P, num_kv_heads, BLOCK, HEAD_DIM), seed, STREAM_V + so)
    q = normal_f16((B, num_q_heads, HEAD_DIM), seed, STREAM_Q + so)
    q_local = None
    if local_queries:
        q_local = normal_f16((B, local_queries, num_q_heads, HEAD_DIM), seed, STREAM_QLOCAL + so)
    needles = []
    if num_needles:
        for b in range(B):
            C = nbs[b] - params.initial_blocks - params.local_blocks
            if C <= 0:
                continue
            blocks = needle_blocks(params.initial_blocks, C, min(num_needles, C))
            plant_needles(k_pool, table, q, b, blocks, seed, STREAM_NEEDLE + so)
            needles += [(b, j) for j in blocks]
    return Workload(name=name, seed=seed, k_pool=k_pool, v_pool=v_pool, block_table=table,
                    seq_lens=seq_lens, q=q, params=params, q_local=q_local, needles=needles)


# The five workloads.  Initial 128 tokens = 1 block; Local 4096 tokens = 32 blocks.

def tiny(seed: int = 0) -> Workload:
    """8 q heads = 8 KV heads, 4096 tokens, Initial 1 / Local 4 blocks, Quest,
    per-head top-4, 3 planted blocks with keys 2*q + N(0, 0.5^2)."""
    p = Params(num_q_heads=8, initial_blocks=1, local_blocks=4, top_k=4, rep=REP_QUEST,
               head_mode=HEAD_SEPARATE)
    return make_workload("tiny-4k-mha-quest", seed=seed, seq_lens=[4096], num_q_heads=8,
                         num_kv_heads=8, params=p, num_needles=3)


def long128k(seed: int = 1, *, layer: int = 0, seq_len: int = 131072) -> Workload:
    """InternLM2.5-7B-1M-shaped layer at 128K: GQA 32/8, Quest, SHARED top-32, K with
    4 outlier channels x8, 16 planted needle blocks."""
    p = Params(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=32, rep=REP_QUEST,
               head_mode=HEAD_SHARED)
    return make_workload("128k-gqa4-quest-shared-k32", seed=seed, seq_lens=[seq_len],
                         num_q_heads=32, num_kv_heads=8, params=p, layer=layer,
                         outlier_channels=4, num_needles=16)


def long1m(seed: int = 2, *, layer: int = 0, rep: int = REP_QUEST,
           seq_len: int = 1048576) -> Workload:
    """1M tokens per layer, GQA 32/8, SEPARATE top-32 per KV head, Max or Quest reps,
    64 planted needle blocks; layers 0..3 use streams offset by 16*layer."""
    p = Params(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=32, rep=rep,
               head_mode=HEAD_SEPARATE)
    return make_workload(f"1m-gqa4-{REP_NAMES[rep]}-separate-k32", seed=seed,
                         seq_lens=[seq_len], num_q_heads=32, num_kv_heads=8, params=p,
                         layer=layer, num_needles=64)


def batched_lengths(seed: int = 3, batch: int = 16, lo: int = 8192, hi: int = 65536):
    return uniform_ints(batch, lo, hi, seed, STREAM_LENS)


def batched(seed: int = 3, *, rep: int = REP_QUEST, head_mode: int = HEAD_SHARED,
            batch: int = 16, lo: int = 8192, hi: int = 65536) -> Workload:
    """16 sequences, lengths uniform on [8192, 65536], pages randomly permuted in one
    pool, GQA 32/8, Local 2048 (16 blocks), top-16."""
    p = Params(num_q_heads=32, initial_blocks=1, local_blocks=16, top_k=16, rep=rep,
               head_mode=head_mode, fix_stride=32)
    lens = batched_lengths(seed, batch, lo, hi)
    return make_workload(f"batched{batch}-paged-{REP_NAMES[rep]}-"
                         f"{'shared' if head_mode == HEAD_SHARED else 'separate'}-k16",
                         seed=seed, seq_lens=lens, num_q_heads=32, num_kv_heads=8, params=p,
                         permute_pages=True)


def dynamic128k(seed: int = 4, *, seq_len: int = 131072, head_mode: int = HEAD_SHARED,
                local_queries: int = 64, layer: int = 0) -> Workload:
    """128K, GQA 32/8, Dynamic reps (4 per block) from the last 64 local-window
    queries, top-32, Local 4096."""
    p = Params(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=32, rep=REP_DYNAMIC,
               head_mode=head_mode, num_reps=4)
    return make_workload("128k-gqa4-dynamic4-k32", seed=seed, seq_lens=[seq_len],
                         num_q_heads=32, num_kv_heads=8, params=p, layer=layer,
                         local_queries=local_queries)


def custom(seed: int, seq_lens, *, num_q_heads=8, num_kv_heads=2, initial_blocks=1,
           local_blocks=2, top_k=4, rep=REP_QUEST, head_mode=HEAD_SEPARATE, num_reps=1,
           fix_stride=32, permute_pages=True, local_queries=0, num_needles=0,
           outlier_channels=0) -> Workload:
    """Small parity cases: any lengths (ragged tails included), any GQA ratio."""
    p = Params(num_q_heads=num_q_heads, initial_blocks=initial_blocks,
               local_blocks=local_blocks, top_k=top_k, rep=rep, head_mode=head_mode,
               num_reps=num_reps, fix_stride=fix_stride)
    return make_workload(f"custom-s{seed}", seed=seed, seq_lens=seq_lens,
                         num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, params=p,
                         permute_pages=permute_pages, local_queries=local_queries,
                         num_needles=num_needles, outlier_channels=outlier_channels)
