"""Helpers shared by the GPU tests: move a synthetic workload to the device,
run the libkt calls through the binding, and compare against the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synth

TOL = 2e-3  # max normwise relative error per (sequence, query head) row
ZONE = 1e-5  # selection boundary zone, relative to the k-th score


def to_dev(a, dtype=None):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


class DevWorkload:
    """A synth.Workload on the GPU plus the binding's structs."""

    def __init__(self, w: synth.Workload):
        import block_sparse_long_quest_gb300 as kt
        self.w = w
        self.k = to_dev(w.k_pool)
        self.v = to_dev(w.v_pool)
        self.table = to_dev(w.block_table)
        self.lens = to_dev(w.seq_lens)
        self.q = to_dev(w.q)
        self.q_local = to_dev(w.q_local) if w.q_local is not None else None
        self.kv = kt.paged_kv(self.k, self.v, self.table, self.lens)
        p = w.params
        self.params = kt.sparse_params(p.num_q_heads, p.initial_blocks, p.local_blocks, p.top_k,
                                       p.rep, p.head_mode, num_reps=p.num_reps,
                                       fix_stride=p.fix_stride, softmax_scale=p.softmax_scale)

    @property
    def SEL(self):
        return 1 if self.w.params.head_mode == synth.HEAD_SHARED else self.w.num_kv_heads

    def build_reps(self):
        import torch
        import block_sparse_long_quest_gb300 as kt
        n = kt.kt_reps_pool_bytes(self.kv, self.params)
        self.reps = torch.zeros(n, dtype=torch.uint8, device="cuda")
        kt.kt_build_block_reps(self.kv, self.params, 0, self.w.max_blocks, self.reps)
        return self.reps

    def reps_view(self):
        """[P][H_kv][R][d] numpy view of the device reps (uint16 bits or float32)."""
        R = synth.Params.reps_per_block(self.w.params)
        a = self.reps.cpu().numpy()
        if self.w.params.rep == synth.REP_MEAN:
            return a.view(np.float32).reshape(self.w.num_pages, self.w.num_kv_heads, R, 128)
        return a.view(np.uint16).reshape(self.w.num_pages, self.w.num_kv_heads, R, 128)

    def select(self, ws=None):
        import torch
        import block_sparse_long_quest_gb300 as kt
        B, k = self.w.batch, self.w.params.top_k
        sel = torch.full((B, self.SEL, k), -1, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, self.SEL), -1, dtype=torch.int32, device="cuda")
        sc = torch.zeros((B, self.SEL, k), dtype=torch.float32, device="cuda")
        if ws is None:
            ws = kt.workspace(kt.KT_OP_SCORE_SELECT, self.kv, self.params)
        kt.kt_score_select_blocks(self.q, self.kv, self.reps, self.params, sel, cnt, sc, ws)
        return sel, cnt, sc, ws

    def attend(self, sel, cnt, ws=None):
        import torch
        import block_sparse_long_quest_gb300 as kt
        out = torch.full((self.w.batch, self.w.params.num_q_heads, 128), float("nan"),
                         dtype=torch.float32, device="cuda")
        if ws is None:
            ws = kt.workspace(kt.KT_OP_SPARSE_ATTN, self.kv, self.params)
        kt.kt_sparse_decode_attn(self.q, self.kv, self.params, sel, cnt, out, ws)
        return out, ws

    def step(self, ws=None):
        import torch
        import block_sparse_long_quest_gb300 as kt
        B, k = self.w.batch, self.w.params.top_k
        sel = torch.full((B, self.SEL, k), -1, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, self.SEL), -1, dtype=torch.int32, device="cuda")
        out = torch.full((B, self.w.params.num_q_heads, 128), float("nan"), dtype=torch.float32,
                         device="cuda")
        if ws is None:
            ws = kt.workspace(kt.KT_OP_SPARSE_STEP, self.kv, self.params)
        kt.kt_sparse_decode_step(self.q, self.kv, self.reps, self.params, sel, cnt, out, ws)
        return sel, cnt, out, ws

    def dense(self, ws=None):
        import torch
        import block_sparse_long_quest_gb300 as kt
        out = torch.full((self.w.batch, self.w.params.num_q_heads, 128), float("nan"),
                         dtype=torch.float32, device="cuda")
        if ws is None:
            ws = kt.workspace(kt.KT_OP_DENSE_ATTN, self.kv, self.params)
        kt.kt_dense_decode_attn(self.q, self.kv, self.w.params.num_q_heads,
                                self.w.params.softmax_scale, out, ws)
        return out, ws


def row_rel_err(got, want):
    """max_i |a_i - r_i| / max_i |r_i| per row (last axis)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    num = np.abs(got - want).max(axis=-1)
    den = np.maximum(np.abs(want).max(axis=-1), 1e-30)
    return num / den


def check_reps(dw: DevWorkload, ref):
    """GPU reps (per page) must equal the oracle's (per logical block) bit for bit."""
    w = dw.w
    got = dw.reps_view()
    mism = 0
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        for j in range(n // 128):
            page = w.block_table[b, j]
            a = got[page]
            r = ref[b, j]
            if w.params.rep == synth.REP_MEAN:
                ok = np.array_equal(a.reshape(r.shape).view(np.uint32), r.view(np.uint32))
            else:
                ok = np.array_equal(a, r)
            mism += 0 if ok else 1
    return mism


def selection_agrees(gpu_sel, gpu_cnt, oracle_res, b, u):
    """Set equality outside the boundary zone.  Returns (ok, exact_equal)."""
    cnt = int(oracle_res["cnt"][b, u])
    if int(gpu_cnt[b, u]) != cnt:
        return False, False
    want = set(oracle_res["sel"][b, u, :cnt].tolist())
    got_list = gpu_sel[b, u, :cnt].tolist()
    got = set(got_list)
    if got_list != sorted(got_list) or len(got) != cnt:
        return False, False
    if got == want:
        return True, True
    scores = oracle_res["unit_scores"][b, u]
    ctx = ~np.isnan(scores)
    vals = np.sort(scores[ctx])[::-1]
    sk = vals[cnt - 1]
    zone = np.abs(scores - sk) <= ZONE * max(abs(sk), 1e-30)
    for j in got.symmetric_difference(want):
        if not zone[j]:
            return False, False
    return True, False


def build_dynamic(dw):
    """Dynamic reps on the GPU; returns the accumulated token scores (numpy)."""
    import torch
    import block_sparse_long_quest_gb300 as kt
    w = dw.w
    T = w.q_local.shape[1]
    n = kt.kt_reps_pool_bytes(dw.kv, dw.params)
    dw.reps = torch.zeros(n, dtype=torch.uint8, device="cuda")
    scores = torch.full((w.batch, w.num_kv_heads, w.max_blocks * 128), -1.0,
                        dtype=torch.float32, device="cuda")
    ws = kt.workspace(kt.KT_OP_DYNAMIC_REPS, dw.kv, dw.params, T)
    kt.kt_build_dynamic_reps(dw.kv, dw.params, dw.q_local, T, 0, w.max_blocks, dw.reps, scores, ws)
    assert kt.kt_read_device_status(ws) == kt.KT_OK
    return scores.cpu().numpy()


def dynamic_rep_tokens(w, reps_view, b, j, h):
    """Token offsets (within block j) whose key rows form the GPU reps."""
    page = w.block_table[b, j]
    rows = w.k_pool[page, h]            # [128][128]
    out = []
    for r in reps_view[page, h]:
        hit = np.nonzero((rows == r).all(axis=1))[0]
        out.append(int(hit[0]) if hit.size else -1)
    return out


def check_dynamic_reps(dw, ref_scores, zone=ZONE, heads=None):
    """GPU reps equal the oracle's choice of tokens, except where the tokens'
    oracle scores sit within `zone` (relative) of the R-th best score.
    Returns (#blocks checked, #blocks that differ inside the zone, bad list)."""
    w = dw.w
    R = w.params.num_reps
    got = dw.reps_view()
    checked = differ = 0
    bad = []
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        for h in (range(w.num_kv_heads) if heads is None else heads):
            sc = ref_scores[b, h]
            for j in range(n // 128):
                blk = sc[j * 128:(j + 1) * 128]
                order = sorted(range(128), key=lambda t: (-blk[t], t))
                want = sorted(order[:R])
                toks = dynamic_rep_tokens(w, got, b, j, h)
                checked += 1
                if toks == want:
                    continue
                rth = blk[order[R - 1]]
                tol = zone * max(abs(rth), 1e-30)
                if -1 in toks or any(abs(blk[t] - rth) > tol
                                     for t in set(toks).symmetric_difference(want)):
                    bad.append((b, h, j, toks, want))
                else:
                    differ += 1
    return checked, differ, bad


def unit_heads(w, u):
    """Query heads whose selection unit is u."""
    G = w.params.num_q_heads // w.num_kv_heads
    if w.params.head_mode == synth.HEAD_SHARED:
        return list(range(w.params.num_q_heads))
    return list(range(u * G, (u + 1) * G))


def check_units(w, kv, sel, cnt, out, ref, units, batches=None):
    """Selection and output of units [units[0], units[1]) of every sequence.

    The selected set must equal the oracle's outside the near-tie zone
    (selection_agrees).  The output of the unit's query heads is compared with
    the oracle's output when the sets are equal; when they differ only inside
    the zone the GPU made another valid selection, and its output is compared
    with the oracle's attention over that (just validated) set, so no unit's
    output goes unchecked.  Returns (#units with equal sets, #units with a
    valid zone difference)."""
    p = w.params
    n_exact = n_zone = 0
    for b in (range(w.batch) if batches is None else batches):
        nb, c0, c1 = oracle.partition(int(w.seq_lens[b]), p.initial_blocks, p.local_blocks)
        for u in range(units[0], units[1]):
            ok, exact = selection_agrees(sel, cnt, ref, b, u)
            assert ok, (b, u, sel[b, u], ref["sel"][b, u])
            heads = unit_heads(w, u)
            if exact:
                want = ref["out"][b, heads]
                n_exact += 1
            else:
                blocks = list(range(c0)) + [int(j) for j in sel[b, u, :int(cnt[b, u])]] + \
                    list(range(c1, nb))
                want = np.stack([oracle.attend(kv, b, hq, p.num_q_heads, w.q[b, hq], blocks,
                                               p.softmax_scale) for hq in heads])
                n_zone += 1
            err = row_rel_err(out[b, heads], want)
            assert err.max() <= TOL, (b, u, err.max())
    return n_exact, n_zone


def parallel(fn, jobs, threads=16):
    """fn over jobs in host threads (the oracle's C calls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(threads, max(1, len(jobs)))) as ex:
        return list(ex.map(fn, jobs))


def dynamic_oracle_scores(w, kv, heads=None):
    """Oracle token scores [B][H_kv][max_blocks*128] of the given KV heads (all
    by default), one host thread per (sequence, KV head)."""
    B, H_kv = w.batch, w.num_kv_heads
    heads = range(H_kv) if heads is None else heads
    out = np.zeros((B, H_kv, w.max_blocks * 128))
    jobs = [(b, h) for b in range(B) for h in heads]
    res = parallel(lambda bh: oracle.dynamic_token_scores(kv, w.params, bh[0], bh[1],
                                                          w.q_local[bh[0]]), jobs)
    for (b, h), r in zip(jobs, res):
        out[b, h, :r.size] = r
    return out


def rep_values_of_gpu_tokens(w, dw):
    """[B][max_blocks][H_kv][R][128] (double): the key rows, taken from the
    input K, of the tokens whose rows the GPU chose as Dynamic reps.  Call it
    after check_dynamic_reps has shown every choice to be valid."""
    R = w.params.num_reps
    got = dw.reps_view()
    rv = np.zeros((w.batch, w.max_blocks, w.num_kv_heads, R, 128))
    for b in range(w.batch):
        for j in range(int(w.seq_lens[b]) // 128):
            page = w.block_table[b, j]
            for h in range(w.num_kv_heads):
                toks = dynamic_rep_tokens(w, got, b, j, h)
                assert -1 not in toks, (b, j, h)
                rows = w.k_pool[page, h, toks]
                rv[b, j, h] = rows.view(np.float16).astype(np.float64)
    return rv


def oracle_step_by_unit(w, kv, units, **kw):
    """oracle.sparse_step of each unit in `units` (SEPARATE) in parallel host
    threads, merged into one result (reps, unit_scores, sel, cnt, out)."""
    res = parallel(lambda u: oracle.sparse_step(kv, w.q, w.params, w.q_local, units=(u, u + 1),
                                                **kw), list(units))
    ref = res[0]
    G = w.params.num_q_heads // w.num_kv_heads
    for u, r in zip(units, res):
        for key in ("unit_scores", "sel", "cnt"):
            ref[key][:, u] = r[key][:, u]
        ref["out"][:, u * G:(u + 1) * G] = r["out"][:, u * G:(u + 1) * G]
        if ref.get("reps") is not None:
            ref["reps"][:, :, u] = r["reps"][:, :, u]
    return ref
