// attn.cu — split-K decode attention over a block list (sparse or dense).
//
// Computes, for every query head h of every sequence b,
//   out[b][h] = softmax(q_h . K_S^T * scale) V_S
// over the token set S = Initial blocks + selected Context blocks + Local blocks
// (sparse; article "KTransformers 长上下文稀疏注意力实战…", §4.2 and §4.6
// attn(query, kvcache_after_retrieval)) or over every block (dense, the full
// scan of §1).
//
// Work decomposition (one launch, grid = max(#SMs, segments)):
//   - A segment is one (sequence, KV head) pair; its work is a list of 128-token
//     blocks in two phases: phase A = the Initial and Local blocks (known from
//     seq_lens alone), phase B = the selected Context blocks (known once the
//     selection has finished).  Every segment gets at least one CTA; the
//     remaining CTAs go to segments in proportion to their work (cumulative
//     rounding, identical on every CTA).  CTA i of a segment with n CTAs takes
//     the i-th n-th of its phase-A blocks and of its phase-B blocks, so a CTA
//     only ever holds one online-softmax state.
//   - A producer warp turns blocks into block-table lookups and 2-D TMA loads
//     (four 16 KB boxes: K and V, two 64-channel halves each, 128-byte swizzle)
//     into a 3-stage shared-memory ring.  Phase-B work waits on
//     griddepcontrol.wait, so when this kernel is a programmatic dependent of
//     the selection kernel, the Initial/Local blocks stream while selection
//     runs.
//   - Eight consumer warps each take 16 tokens of a block: S = q K^T and
//     O += P V on mma.sync m16n8k16 (fp16 in, fp32 accumulate).  Query heads
//     are rows 0..G-1 of the A operand; in P V the fp16 split P = P_hi + P_lo
//     puts P_hi in rows 0..7 and P_lo in rows 8..15 of the same fragment, so P
//     keeps ~22 bits.  Online softmax in base 2 per warp.
//   - At the end the eight warp states are merged through shared memory.  A
//     segment served by one CTA is written to out directly; otherwise each CTA
//     writes an (m, l, acc) partial, takes a ticket, and the CTA completing the
//     count merges the segment's partials in CTA order (deterministic).
//
// The one-launch decode step (attn_kernel<SK>, SK != SK_NONE; a cooperative
// launch of one CTA per SM) also makes the selection (§3.1, §4.3, §4.5): while
// the producer waits, the consumer warps stage and score one slice of a
// selection unit's Context blocks (fused_score), publish the slice's best keys
// with a ticket, then wait for the unit's tickets and pick the unit's top-k
// (fused_merge) and hand this CTA's share of the chosen pages to the producer.
// Each segment's first CTA merges the partials (every CTA is resident).  SK
// selects the scoring path at compile time, so a launch carries only the code
// it runs.
#include "select_common.cuh"

namespace kt {
namespace {

constexpr int STAGES = 3;
constexpr int CONSUMERS = 8;
constexpr int NCT = CONSUMERS * 32;
constexpr int THREADS = NCT + 32;
constexpr int UNIT = 128;                      // tokens per work unit (one block)
constexpr int BOX_BYTES = UNIT * 64 * 2;       // 128 tokens x 64 channels fp16
constexpr int KV_STAGE_BYTES = 4 * BOX_BYTES;  // K lo, K hi, V lo, V hi
constexpr int Q_BYTES = MAX_G * D * 2;
constexpr int HALF_WARPS = CONSUMERS / 2;
constexpr int SCRATCH_FLOATS = HALF_WARPS * MAX_G * (D + 2);
static_assert(SCRATCH_FLOATS * 4 == ATTN_SCRATCH_BYTES, "scratch size shared with the host");
static_assert(NCT == ATTN_CONSUMER_THREADS, "consumer threads shared with the host");
static_assert(STAGES * KV_STAGE_BYTES == ATTN_RING_BYTES, "ring size shared with the host");

struct StageInfo {
  int ntok, end, pad0, pad1;
};

struct SmemLayout {
  static constexpr int kv = 0;
  static constexpr int q = kv + STAGES * KV_STAGE_BYTES;
  static constexpr int scratch = q + Q_BYTES;
  static constexpr int cum = scratch + SCRATCH_FLOATS * 4;  // [MAX_SEGS+1] work prefix
  static constexpr int info = cum + (MAX_SEGS + 1) * 4;
  static constexpr int bars = (info + STAGES * (int)sizeof(StageInfo) + 15) & ~15;
  static constexpr int bcast = bars + (2 * STAGES + 5) * 8;
  static constexpr int total = bcast + 64 * 4;
};
constexpr int SMEM_BYTES = SmemLayout::total + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "attention shared memory exceeds the per-CTA limit");
static_assert(SmemLayout::cum == SmemLayout::scratch + ATTN_SCRATCH_BYTES &&
                  ATTN_MERGE_BYTES == ATTN_SCRATCH_BYTES + (MAX_SEGS + 1) * 4,
              "the fused merge area is scratch + block prefix, contiguous");

struct Params {
  CUtensorMap kmap, vmap;
  const __half* q;
  const int32_t* table;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* cnt;
  const int32_t* sel_pages;
  float* out;
  int* status;
  int* counters;
  float* parts;
  int B, H_kv, G, max_blocks, P, I_b, L_b, top_k, SEL, dense, slot_floats;
  float scale_log2;
  // fused step only: in-kernel selection (fused_score, fused_merge)
  const void* reps;
  int rep, R, ncpu, f_chunk, kk_f;
  unsigned long long* f_cand;
  int* f_cand_pages;
  int* f_counters;
  int* f_polled;
  int32_t* sel_out;
  int32_t* cnt_out;
  const uint32_t* presel_mask;
  const int32_t* presel_cnt;
  int mask_words;
};

struct Part {
  int n, nb, c0, c1;
};

__device__ __forceinline__ Part partition(int n, int I, int L) {
  Part p;
  p.n = n;
  p.nb = (n + BS - 1) / BS;
  p.c0 = min(I, p.nb);
  p.c1 = max(p.c0, p.nb - L);
  return p;
}

__device__ __forceinline__ int seq_len(const Params& p, int b) {
  int n = __ldg(p.seq_lens + b);
  if (n < 0 || n > p.max_blocks * BS) {
    set_status(p.status, KT_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : p.max_blocks * BS;
  }
  return n;
}

// Phase-A blocks of a sequence and the most phase-B blocks it can have.
__device__ __forceinline__ int blocks_a(const Part& pt, int dense) {
  return dense ? pt.nb : pt.c0 + (pt.nb - pt.c1);
}
__device__ __forceinline__ int blocks_b_max(const Part& pt, int dense, int top_k) {
  return dense ? 0 : min(top_k, pt.c1 - pt.c0);
}

// Inclusive prefix over S counts computed by one warp: pref[0] = 0,
// pref[s+1] = pref[s] + count(s).
template <class F>
__device__ void warp_prefix(int* pref, int S, F count, int lane) {
  const int per = (S + 31) / 32;
  const int lo = min(S, lane * per), hi = min(S, lo + per);
  int sum = 0;
  for (int s = lo; s < hi; ++s) {
    sum += count(s);
    pref[s + 1] = sum;
  }
  int incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - sum;
  for (int s = lo; s < hi; ++s) pref[s + 1] += excl;
  if (lane == 0) pref[0] = 0;
  __syncwarp();
}

// Number of ids in a[0, n) smaller than id; a is 16-byte aligned, n a multiple of 4.
__device__ __forceinline__ int count_less_u32(const uint32_t* a, int n, uint32_t id) {
  int r0 = 0, r1 = 0;
  int m = 0;
#pragma unroll 1
  for (; m + 16 <= n; m += 16) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(a + m);
    const uint4 v1 = *reinterpret_cast<const uint4*>(a + m + 4);
    const uint4 v2 = *reinterpret_cast<const uint4*>(a + m + 8);
    const uint4 v3 = *reinterpret_cast<const uint4*>(a + m + 12);
    r0 += (v0.x < id ? 1 : 0) + (v0.y < id ? 1 : 0) + (v0.z < id ? 1 : 0) + (v0.w < id ? 1 : 0) +
          (v1.x < id ? 1 : 0) + (v1.y < id ? 1 : 0) + (v1.z < id ? 1 : 0) + (v1.w < id ? 1 : 0);
    r1 += (v2.x < id ? 1 : 0) + (v2.y < id ? 1 : 0) + (v2.z < id ? 1 : 0) + (v2.w < id ? 1 : 0) +
          (v3.x < id ? 1 : 0) + (v3.y < id ? 1 : 0) + (v3.z < id ? 1 : 0) + (v3.w < id ? 1 : 0);
  }
#pragma unroll 1
  for (; m < n; m += 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(a + m);
    r0 += (v.x < id ? 1 : 0) + (v.y < id ? 1 : 0) + (v.z < id ? 1 : 0) + (v.w < id ? 1 : 0);
  }
  return r0 + r1;
}

// Fused step: where the scoring CTA stages its slice's representative rows in
// the KV ring.  When a whole nominal slice fits, it sits at the top of the
// ring and the stages below it stay free for the Initial/Local blocks;
// otherwise rounds use the two halves from offset 0.  Also returns the row
// stride (fp16 rows are padded by 16 bytes for conflict-free ldmatrix).
__device__ __forceinline__ uint32_t fused_stage_off(const Params& p, uint32_t* stride = nullptr,
                                                    bool* single = nullptr) {
  constexpr uint32_t RING = STAGES * KV_STAGE_BYTES;
  const int nkv = p.SEL == 1 ? p.H_kv : 1;
  const bool f32 = p.rep == KT_REP_MEAN;
  const uint32_t bbytes = (uint32_t)(nkv * p.R * D * (f32 ? 4 : 2));
  const uint32_t sb = f32 ? bbytes : bbytes + 16;
  const uint64_t need = (uint64_t)p.f_chunk * sb;
  if (stride) *stride = sb;
  if (single) *single = need <= RING;
  return need <= RING ? (uint32_t)(RING - need) : 0u;
}

// Mean reps (fp32) scored on the CUDA cores; kept out of line, away from the
// common fp16 path.
__device__ __noinline__ void fused_score_f32(const uint4* sbuf, int sstride, int nblk, int j0,
                                             int P, const int* pg, const float* wts, int V,
                                             unsigned long long* keys, int warp, int lane,
                                             int* status) {
  if (V <= 32) selc::score_linear_smem<1, true, CONSUMERS>(sbuf, sstride, nblk, j0, P, pg, wts, V, keys, warp, lane, status);
  else if (V <= 64) selc::score_linear_smem<2, true, CONSUMERS>(sbuf, sstride, nblk, j0, P, pg, wts, V, keys, warp, lane, status);
  else if (V <= 128) selc::score_linear_smem<4, true, CONSUMERS>(sbuf, sstride, nblk, j0, P, pg, wts, V, keys, warp, lane, status);
  else selc::score_linear_smem<8, true, CONSUMERS>(sbuf, sstride, nblk, j0, P, pg, wts, V, keys, warp, lane, status);
}

// Fused step: the linear weight rows of KV heads g0 .. g0+nkv-1 of sequence bu
// (query heads summed in ascending order per channel; Quest: the negative and
// positive parts, paired with the kmin and kmax rows).  Same values as the
// selection kernel.
__device__ __forceinline__ void fused_weights(const Params& p, float* wts, int bu, int g0, int nkv,
                                           int ctid) {
  const int H_q = p.H_kv * p.G;
  const __half* qu = p.q + ((size_t)bu * H_q + (size_t)g0 * p.G) * D;
#pragma unroll 1
  for (int it = ctid; it < nkv * (D / 8); it += NCT) {
    const int gi = it / (D / 8), c8 = it % (D / 8);
    uint4 v[MAX_G];
#pragma unroll
    for (int hh = 0; hh < MAX_G; ++hh)
      v[hh] = hh < p.G ? __ldg(reinterpret_cast<const uint4*>(qu + (size_t)(gi * p.G + hh) * D) + c8)
                       : make_uint4(0u, 0u, 0u, 0u);
    float sum[8], neg[8], pos[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sum[e] = neg[e] = pos[e] = 0.0f;
#pragma unroll
    for (int hh = 0; hh < MAX_G; ++hh) {
      if (hh < p.G) {
        const __half2* h2 = reinterpret_cast<const __half2*>(&v[hh]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h2[e]);
          sum[2 * e] += f.x;
          neg[2 * e] += fminf(f.x, 0.0f);
          pos[2 * e] += fmaxf(f.x, 0.0f);
          sum[2 * e + 1] += f.y;
          neg[2 * e + 1] += fminf(f.y, 0.0f);
          pos[2 * e + 1] += fmaxf(f.y, 0.0f);
        }
      }
    }
    if (p.rep == KT_REP_QUEST) {
      float4* wn = reinterpret_cast<float4*>(wts + (gi * 2 + 0) * D + c8 * 8);  // kmin row
      float4* wp = reinterpret_cast<float4*>(wts + (gi * 2 + 1) * D + c8 * 8);  // kmax row
      wn[0] = make_float4(neg[0], neg[1], neg[2], neg[3]);
      wn[1] = make_float4(neg[4], neg[5], neg[6], neg[7]);
      wp[0] = make_float4(pos[0], pos[1], pos[2], pos[3]);
      wp[1] = make_float4(pos[4], pos[5], pos[6], pos[7]);
    } else {
      float4* w = reinterpret_cast<float4*>(wts + gi * D + c8 * 8);
      w[0] = make_float4(sum[0], sum[1], sum[2], sum[3]);
      w[1] = make_float4(sum[4], sum[5], sum[6], sum[7]);
    }
  }
}

// Fused step, consumer warps of CTA c < U*ncpu: score slice c % ncpu (nominal
// Context blocks I_b + s*f_chunk ...) of selection unit c / ncpu with the same
// weights, dot products and keys as the selection kernel, keep the slice's best
// kk_f (key 0 = empty slot) in the unit's candidate table and take a ticket.
// Arrives on bar_scored once its representative loads are done (every CTA).
// The block-table entries of the nominal slice do not depend on the sequence
// length, so they load together with the length and the query rows.
template <int SK, class Bar>
__device__ void fused_score(const Params& p, uint8_t* scr, unsigned int* hist,
                            unsigned long long* sh_u64, int* sh_int, int ctid, int warp, int lane,
                            Bar bar_c, uint32_t bar_scored, const uint8_t* ring,
                            uint32_t ring_u32, uint32_t bar_reps) {
  const int U = p.B * p.SEL;
  const int u = blockIdx.x / p.ncpu;
  if (u >= U) {
    if (ctid == 0) mbar_arrive(bar_scored);
    return;
  }
  const int cs = blockIdx.x % p.ncpu;
  const int bu = u / p.SEL, g0 = p.SEL == 1 ? 0 : u % p.SEL;
  const int nkv = p.SEL == 1 ? p.H_kv : 1;
  const int Rw = p.rep == KT_REP_QUEST ? 2 : 1;
  const bool f32 = p.rep == KT_REP_MEAN;
  const bool multi = p.rep == KT_REP_FIX || p.rep == KT_REP_DYNAMIC;  // max over reps per head
  const FusedScoreLayout Ls = fused_score_layout(multi ? 0 : nkv * Rw * D, p.f_chunk, p.kk_f);
  float* wts = reinterpret_cast<float*>(scr);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(scr + Ls.keys);
  int* pgs = reinterpret_cast<int*>(scr + Ls.pgs);

  const int js = p.I_b + cs * p.f_chunk;
#pragma unroll 1
  for (int i = ctid; i < p.f_chunk; i += NCT) {
    const int j = js + i;
    pgs[i] = j < p.max_blocks ? __ldg(p.table + (size_t)bu * p.max_blocks + j) : -1;
  }
  // the slice's candidate slots start empty (key 0, page -1): keys of equal
  // value share a rank and empty keys are never written, so some may stay so
  unsigned long long* cand = p.f_cand + ((size_t)u * p.ncpu + cs) * p.kk_f;
  int* cpage = p.f_cand_pages + ((size_t)u * p.ncpu + cs) * p.kk_f;
#pragma unroll 1
  for (int i = ctid; i < p.kk_f; i += NCT) {
    cand[i] = 0ull;
    cpage[i] = -1;
  }
  const Part pu = partition(seq_len(p, bu), p.I_b, p.L_b);
  const int je = min(js + p.f_chunk, pu.c1);
  const int nloc = max(0, je - js);  // js >= c0 whenever the slice is not empty
  if (ctid == 0 && (nloc & 1)) keys[nloc] = 0ull;  // the ranking's zero padding
  bar_c();
  if (nloc > 0) {
    // the slice's representative rows, staged into the (still idle) KV ring by
    // bulk copies in rounds of up to ring-size bytes, then scored from there
    // fp16 reps (Max, Quest) are scored on the tensor cores from rows padded
    // by 16 bytes (conflict-free ldmatrix); fp32 reps (Mean) on the CUDA cores
    const int V = nkv * p.R * D / (f32 ? 4 : 8);
    const uint32_t bbytes = (uint32_t)V * 16;  // one block's rows for the unit's heads
    const uint32_t sb = f32 ? bbytes : bbytes + 16;
    const size_t head_bytes = (size_t)p.R * D * (f32 ? 4 : 2);
    // one round when the slice fits the ring, else rounds alternating between
    // its two halves so that the next round's copies fly while one is scored;
    // each warp issues its share of a round (its expect-tx, then its copies)
    constexpr uint32_t RING = STAGES * KV_STAGE_BYTES, HALF = RING / 2;
    bool single = false;
    const uint32_t off = fused_stage_off(p, nullptr, &single);
    const int rcap = single ? nloc : (int)(HALF / sb);
    const int nrounds = (nloc + rcap - 1) / rcap;
    auto buf_off = [&](int r) { return single ? off : (uint32_t)(r & 1) * HALF; };
    auto issue = [&](int r) {
      const int r0 = r * rcap, nr = min(rcap, nloc - r0);
      const uint32_t base = ring_u32 + buf_off(r);
      const uint32_t bar = (r & 1) ? bar_reps + 8 : bar_reps;
      const int i0 = warp * nr / CONSUMERS, i1 = (warp + 1) * nr / CONSUMERS;
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(i1 - i0) * bbytes);
      __syncwarp();
#pragma unroll 1
      for (int i = i0 + lane; i < i1; i += 32) {
        const int page = pgs[r0 + i];
        const bool ok = page >= 0 && page < p.P;  // out of range: scored -inf, flagged
        bulk_load(base + (uint32_t)i * sb,
                  static_cast<const uint8_t*>(p.reps) +
                      ((size_t)(ok ? page : 0) * p.H_kv + g0) * head_bytes,
                  bbytes, bar);
      }
    };
    issue(0);
    if (nrounds > 1) issue(1);
    // the query-dependent weights are folded while the copies fly
    if (!multi) {
      fused_weights(p, wts, bu, g0, nkv, ctid);
      bar_c();
    }
    // fp16 reps: a few blocks per CTA on the CUDA cores, many on the tensor
    // cores, whose B fragments replace the weights in place (the launch's
    // path SK follows from the largest slice, fused_score_kind)
    if constexpr (SK == SK_MMA) selc::weights_to_frags<NCT>(wts, V * 8, ctid, bar_c);
#pragma unroll 1
    for (int r = 0; r < nrounds; ++r) {
      const int r0 = r * rcap, nr = min(rcap, nloc - r0);
      mbar_wait((r & 1) ? bar_reps + 8 : bar_reps, (uint32_t)(r >> 1) & 1u, p.status);
      const uint32_t base = ring_u32 + buf_off(r);
      const uint4* sbuf = reinterpret_cast<const uint4*>(ring + buf_off(r));
#define KT_SCORE(NV, F) selc::score_linear_smem<NV, F, CONSUMERS>(sbuf, (int)(sb / 16), nr, js + r0, p.P, pgs + r0, wts, V, keys + r0, warp, lane, p.status)
#define KT_COLS(VC) selc::score_linear_cols<VC, CONSUMERS>(sbuf, (int)(sb / 16), nr, js + r0, p.P, pgs + r0, wts, keys + r0, red, warp, lane, p.status, bar_c)
      if constexpr (SK == SK_MULTI) {
        selc::score_multi_mma_smem<CONSUMERS>(
            base, (int)sb, nr, js + r0, p.P, pgs + r0,
            p.q + ((size_t)bu * p.H_kv * p.G + (size_t)g0 * p.G) * D, p.G, nkv, p.R, keys + r0,
            reinterpret_cast<float*>(hist), warp, lane, p.status, bar_c);
      } else if constexpr (SK == SK_F32) {
        fused_score_f32(sbuf, (int)(sb / 16), nr, js + r0, p.P, pgs + r0, wts, V, keys + r0, warp,
                        lane, p.status);
      } else if constexpr (SK == SK_MMA) {
        selc::score_mma_smem<CONSUMERS>(base, (int)sb, nr, js + r0, p.P, pgs + r0,
                                        reinterpret_cast<const uint2*>(wts), V * 8, keys + r0,
                                        reinterpret_cast<float*>(hist), warp, lane, p.status,
                                        bar_c);
      } else if constexpr (SK == SK_COLS) {
        // one pass: every thread owns one 16-byte column of the few blocks
        float* red = reinterpret_cast<float*>(hist);
        if (V == 256) KT_COLS(256);
        else if (V == 128) KT_COLS(128);
        else KT_COLS(64);
      } else {
        // one pass of the CUDA-core path: each warp reduces its few blocks
        if (V <= 32) KT_SCORE(1, false);
        else if (V <= 64) KT_SCORE(2, false);
        else if (V <= 128) KT_SCORE(4, false);
        else KT_SCORE(8, false);
      }
#undef KT_SCORE
#undef KT_COLS
      bar_c();  // this half is refilled by round r + 2, the ring by the producer
      if (r + 2 < nrounds) issue(r + 2);
    }
  }
  if (ctid == 0) mbar_arrive(bar_scored);  // the producer may start its own loads
  // the slice's best min(nloc, kk_f) keys, written in descending key order
  // (empty slots: key 0, page -1), then the ticket
  bool few = nloc <= p.kk_f;  // every key of the slice is a candidate
  if (p.presel_mask) {
    // preselection: blocks outside it get key 0, the empty slot; with at most
    // kk_f real keys left they are all candidates
    const uint32_t* mk = p.presel_mask + (size_t)u * p.mask_words;
    int real = 0;
#pragma unroll 1
    for (int i = ctid; i < nloc; i += NCT) {
      const int j = js + i;
      if (!((__ldg(mk + (j >> 5)) >> (j & 31)) & 1u)) keys[i] = 0ull;
      else ++real;
    }
    real = selc::warp_sum_int(real);
    if (ctid == 0) sh_int[3] = 0;
    bar_c();
    if (lane == 0) atomicAdd(&sh_int[3], real);
    bar_c();
    few = few || sh_int[3] <= p.kk_f;
  }
  // SK_COLS launches have slices of at most top_k blocks: always `few`
  if (SK != SK_COLS && !few) {
    auto emit = [&](int r, int i) {
      cand[r] = keys[i];
      cpage[r] = pgs[i];
    };
    unsigned long long* ck = reinterpret_cast<unsigned long long*>(scr + Ls.bkey);
    int* ci = reinterpret_cast<int*>(scr + Ls.bidx);
    int* ix = reinterpret_cast<int*>(scr + Ls.idx);
    // slices hold at most FUSED_MAX_CHUNK = 8 NCT blocks (the host's plan)
    if constexpr (SK != SK_COLS)
      selc::topk_sorted_reg<NCT>(keys, nloc, p.kk_f, ck, ci, ix, hist, sh_u64, sh_int, ctid,
                                 bar_c, emit);
  } else {
    // with nloc odd, keys[nloc] is the zero padding
    const int npad = (nloc + 1) & ~1;
#pragma unroll 1
    for (int i = ctid; i < nloc; i += NCT) {
      const unsigned long long key = keys[i];
      if (key != 0ull) {
        const int r = selc::count_greater(keys, npad, key);
        if (r < p.kk_f) {
          cand[r] = key;
          cpage[r] = pgs[i];
        }
      }
    }
  }
  bar_c();
  if (ctid == 0) red_release_gpu_add(p.f_counters + u, 1);
}

// Fused step, consumer warps of every CTA: wait (bounded) for every scoring
// slice of this segment's selection unit, pick the unit's top-k from the
// candidate table, order the chosen blocks by id and keep this CTA's share
// [i0, i1) of their page ids in the merge area's slice.  One CTA per unit
// writes sel / cnt.  Returns i1 - i0.
//
// The per-slice lists are sorted, so the keff-th largest of their first J
// keys (J lists' heads, ncpu * J >= keff) is a lower bound T0 for the unit's
// keff-th largest key: only keys >= T0 can be chosen, and they are few
// (at most keff / J lists reach T0 at their J-th key).  Those are ranked
// exactly by counting; the same keys as the selection kernel give the same
// blocks.
template <class Bar>
__device__ int fused_merge(const Params& p, uint8_t* scr, unsigned int* hist,
                           unsigned long long* sh_u64, int* sh_int, int b, int h, int ci,
                           int ncta, int ctid, Bar bar_c) {
  const int unit = b * p.SEL + (p.SEL == 1 ? 0 : h);
  const Part pt = partition(seq_len(p, b), p.I_b, p.L_b);
  int keff = min(p.top_k, pt.c1 - pt.c0);
  if (p.presel_mask) keff = min(keff, max(0, __ldg(p.presel_cnt + unit)));
  if (ctid == 0) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
      if (ld_acquire_gpu(p.f_counters + unit) >= p.ncpu) break;
      if ((i & 63u) == 63u && globaltimer() - t0 > WAIT_LIMIT_NS) {
        set_status(p.status, KT_ERR_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
  }
  bar_c();
  const int kk = p.kk_f, nslots = p.ncpu * kk;
  const FusedMergeLayout Lm = fused_merge_layout(p.ncpu, kk, min(p.top_k, nslots));
  unsigned long long* all = reinterpret_cast<unsigned long long*>(scr + Lm.all);
  int* allp = reinterpret_cast<int*>(scr + Lm.allp);
  unsigned long long* heads = reinterpret_cast<unsigned long long*>(scr + Lm.heads);
  unsigned long long* ckey = reinterpret_cast<unsigned long long*>(scr + Lm.ck);
  int* cslot = reinterpret_cast<int*>(scr + Lm.cs);
  int* idx = reinterpret_cast<int*>(scr + Lm.idx);
  uint32_t* cid = reinterpret_cast<uint32_t*>(scr + Lm.cid);
  int* slice = reinterpret_cast<int*>(scr + Lm.slice);
  const bool writer = ci == 0 && (p.SEL != 1 || h == 0);
  if (keff <= 0) {
    if (writer && ctid == 0) p.cnt_out[unit] = 0;
    return 0;
  }
  // gather: slots ctid + r*NCT of the unit's table into registers (one round
  // trip), their pages and keys into shared memory, and the head sample
  constexpr int GP = FUSED_GATHER_PER_THREAD;
  const unsigned long long* src = p.f_cand + (size_t)unit * nslots;
  const int* srcp = p.f_cand_pages + (size_t)unit * nslots;
  const int J = Lm.J, H = Lm.nheads, Hpad = (H + 1) & ~1;
  unsigned long long kx[GP];
  int px[GP];
#pragma unroll
  for (int r = 0; r < GP; ++r) {
    const int s = ctid + r * NCT;
    kx[r] = s < nslots ? __ldcg(src + s) : 0ull;
    px[r] = s < nslots ? __ldcg(srcp + s) : -1;
  }
  // head sample with its common leading bits (AND / OR) and nonzero count
  unsigned long long h_and = ~0ull, h_or = 0ull;
  int h_nz = 0;
#pragma unroll 1
  for (int hh = ctid; hh < Hpad; hh += NCT) {
    const unsigned long long key = hh < H ? __ldcg(src + (hh / J) * kk + (hh % J)) : 0ull;
    heads[hh] = key;
    if (key != 0ull) {
      h_and &= key;
      h_or |= key;
      ++h_nz;
    }
  }
#pragma unroll
  for (int r = 0; r < GP; ++r) {
    const int s = ctid + r * NCT;
    if (s < nslots) {
      all[s] = kx[r];
      allp[s] = px[r];
    }
  }
  const int kpad = (keff + 3) & ~3;
#pragma unroll 1
  for (int i = ctid; i < kpad; i += NCT) {
    idx[i] = -1;
    cid[i] = 0xFFFFFFFFu;
  }
#pragma unroll 1
  for (int i = ctid; i < Lm.mcap; i += NCT) ckey[i] = 0ull;
  hist[ctid] = 0u;  // NCT == 256 bins
  {
    const int lane = ctid & 31, w = ctid >> 5;
    const uint32_t a_lo = __reduce_and_sync(0xffffffffu, (uint32_t)h_and);
    const uint32_t a_hi = __reduce_and_sync(0xffffffffu, (uint32_t)(h_and >> 32));
    const uint32_t o_lo = __reduce_or_sync(0xffffffffu, (uint32_t)h_or);
    const uint32_t o_hi = __reduce_or_sync(0xffffffffu, (uint32_t)(h_or >> 32));
    const unsigned nz = __reduce_add_sync(0xffffffffu, (unsigned)h_nz);
    if (lane == 0) {
      sh_u64[2 + w] = ((unsigned long long)a_hi << 32) | a_lo;
      sh_u64[2 + CONSUMERS + w] = ((unsigned long long)o_hi << 32) | o_lo;
      hist[256 + w] = nz;
    }
  }
  if (ctid == 0) sh_int[0] = 0;
  bar_c();
  // T0: lower edge of the 8-bit digit bin (just below the heads' common
  // leading bits) that holds the keff-th largest head.  At least keff heads,
  // hence keys, are >= T0, so T0 bounds the keff-th largest key from below;
  // with fewer than keff nonzero heads every nonzero key stays (T0 = 1).
  // Every warp scans the histogram itself.
  unsigned long long T0 = 1ull;
  {
    unsigned long long a = ~0ull, o = 0ull;
    int nz = 0;
#pragma unroll
    for (int w = 0; w < CONSUMERS; ++w) {
      a &= sh_u64[2 + w];
      o |= sh_u64[2 + CONSUMERS + w];
      nz += (int)hist[256 + w];
    }
    if (nz >= keff) {
      const unsigned long long diff = a ^ o;
      const int hi = diff ? 64 - __clzll((long long)diff) : 0;
      const int shift = hi > 8 ? hi - 8 : 0;
      const unsigned long long pmask = hi >= 64 ? 0ull : ~((1ull << hi) - 1);
      const unsigned long long prefix = a & pmask;
#pragma unroll 1
      for (int hh = ctid; hh < H; hh += NCT) {
        const unsigned long long key = heads[hh];
        if (key != 0ull) atomicAdd(&hist[(unsigned)((key >> shift) & 255ull)], 1u);
      }
      bar_c();
      // lane l holds digits 255-8l .. 248-8l (descending)
      const int lane = ctid & 31;
      unsigned int c[8], local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
        local += c[i];
      }
      unsigned int incl = local;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const unsigned int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      const unsigned int excl = incl - local;
      const bool hit = excl < (unsigned)keff && (unsigned)keff <= incl;
      int digit = 0;  // 256 + digit once found
      unsigned int above = excl;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        above += c[i];
        if (hit && digit == 0 && above >= (unsigned)keff) digit = 256 + 255 - 8 * lane - i;
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
      digit = __shfl_sync(0xffffffffu, digit, src < 0 ? 0 : src) - 256;
      if (digit >= 0) T0 = prefix | (static_cast<unsigned long long>(digit) << shift);
      if (T0 == 0ull) T0 = 1ull;
    }
  }
  // keys >= T0 with their slots: one shared atomic per warp
  {
    const int lane = ctid & 31;
    const unsigned int lt = (1u << lane) - 1u;
    unsigned int bal[GP];
    int tot = 0;
#pragma unroll
    for (int r = 0; r < GP; ++r) {
      bal[r] = __ballot_sync(0xffffffffu, kx[r] >= T0);
      tot += __popc(bal[r]);
    }
    int o = 0;
    if (lane == 0 && tot) o = atomicAdd(&sh_int[0], tot);
    o = __shfl_sync(0xffffffffu, o, 0);
#pragma unroll
    for (int r = 0; r < GP; ++r) {
      const int pos = o + __popc(bal[r] & lt);
      if (kx[r] >= T0 && pos < Lm.mcap) {
        ckey[pos] = kx[r];
        cslot[pos] = ctid + r * NCT;
      }
      o += __popc(bal[r]);
    }
  }
  bar_c();
  const int M = sh_int[0];
  if (M <= Lm.mcap) {
    // exact rank among them; the chosen keep their block ids for the ordering
#pragma unroll 1
    for (int i = ctid; i < M; i += NCT) {
      const unsigned long long key = ckey[i];
      const int r = selc::count_greater(ckey, (M + 1) & ~1, key);
      if (r < keff) {
        idx[r] = cslot[i];
        cid[r] = 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
      }
    }
  } else {
    // many keys near the bound: radix selection over the whole table
    selc::select_top<NCT>(all, nslots, keff, idx, ckey, cslot, hist, sh_u64, sh_int, ctid, bar_c);
#pragma unroll 1
    for (int i = ctid; i < keff; i += NCT)
      cid[i] = 0xFFFFFFFFu - static_cast<uint32_t>(all[idx[i]] & 0xFFFFFFFFull);
  }
  bar_c();
  if (ctid == 0 && M < keff) set_status(p.status, KT_ERR_DEVICE_CHECK);
  // position of a chosen block = chosen blocks with a smaller id
  const int i0 = (int)((long long)ci * keff / ncta), i1 = (int)((long long)(ci + 1) * keff / ncta);
#pragma unroll 1
  for (int i = ctid; i < keff; i += NCT) {
    const uint32_t id = cid[i];
    const int r = min(count_less_u32(cid, kpad, id), keff - 1);
    const int x = idx[i];
    if (writer) p.sel_out[(size_t)unit * p.top_k + r] = x >= 0 ? static_cast<int32_t>(id) : -1;
    if (r >= i0 && r < i1) slice[r - i0] = x >= 0 ? allp[x] : -1;
  }
  if (writer && ctid == 0) p.cnt_out[unit] = keff;
  bar_c();
  return i1 - i0;
}

template <int SK>
__global__ void __launch_bounds__(THREADS, 1) attn_kernel(const __grid_constant__ Params p) {
  constexpr bool FUSED = SK != SK_NONE;
  extern __shared__ uint8_t smem_raw[];
  __shared__ unsigned int f_hist[FUSED ? 512 : 1];
  __shared__ unsigned long long f_sh_u64[FUSED ? 2 + 2 * CONSUMERS : 1];
  __shared__ int f_sh_int[FUSED ? 4 : 1];
  // 1024-byte aligned (128-byte swizzled TMA boxes); offsetting the array
  // itself keeps the accesses below in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grid = gridDim.x, cta = blockIdx.x;
  const int S = p.B * p.H_kv, H_q = p.H_kv * p.G;
  int* cum = reinterpret_cast<int*>(smem + SmemLayout::cum);
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + SmemLayout::info);
  int* bcast = reinterpret_cast<int*>(smem + SmemLayout::bcast);
  float* scratch = reinterpret_cast<float*>(smem + SmemLayout::scratch);
  const uint32_t bar_full = smem_u32(smem + SmemLayout::bars);
  const uint32_t bar_empty = bar_full + STAGES * 8;
  const uint32_t bar_q = bar_empty + STAGES * 8;
  const uint32_t bar_sel = bar_q + 8;      // fused: this CTA's selected pages are ready
  const uint32_t bar_scored = bar_sel + 8;  // fused: this CTA's scoring loads are done
  const uint32_t bar_reps = bar_scored + 8;  // fused: staged reps landed (two, one per ring half)
  const uint32_t kv_base = smem_u32(smem + SmemLayout::kv);
  auto bar_c = [] { named_bar_sync(1, NCT); };
  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, CONSUMERS);
    }
    mbar_init(bar_q, 1);
    mbar_init(bar_sel, 1);
    mbar_init(bar_scored, 1);
    mbar_init(bar_reps, CONSUMERS);
    mbar_init(bar_reps + 8, CONSUMERS);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- set-up: segment work prefix -> this CTA's segment and slice.  In the
  // fused step the consumer warps score their selection slice meanwhile.
  if (warp == CONSUMERS) {
    if (lane == 0) {
      prefetch_tensormap(&p.kmap);
      prefetch_tensormap(&p.vmap);
    }
    // weight of a segment: its phase-A blocks + the most phase-B blocks + 1
    warp_prefix(cum, S, [&](int s) {
      const Part pt = partition(seq_len(p, s / p.H_kv), p.I_b, p.L_b);
      return blocks_a(pt, p.dense) + blocks_b_max(pt, p.dense, p.top_k) + 1;
    }, lane);
    // in place: cum[s] -> first CTA of segment s = s + floor(extra * cum[s] / W)
    const long long extra = grid - S, W = cum[S];
    __syncwarp();
    for (int s = lane; s <= S; s += 32) cum[s] = s + (int)(extra * cum[s] / W);
    __syncwarp();
  } else if (FUSED) {
    fused_score<SK>(p, reinterpret_cast<uint8_t*>(scratch), f_hist, f_sh_u64, f_sh_int, tid, warp,
                lane, bar_c, bar_scored, smem + SmemLayout::kv, kv_base, bar_reps);
  }
  if (!FUSED) __syncthreads();
  else if (warp != CONSUMERS) named_bar_sync(2, THREADS);
  // CTAs of segment s: [cum[s], cum[s+1])
  int seg;
  {
    int lo = 0, hi = S - 1;  // largest s with first(s) <= cta
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= cta) lo = mid; else hi = mid - 1;
    }
    seg = lo;
  }
  const int f0 = cum[seg], ncta = cum[seg + 1] - f0, ci = cta - f0;
  // fused: CTAs that wait on this segment's selection unit (SHARED: every
  // segment of the sequence)
  const int npoll = (p.SEL == 1) ? cum[(seg / p.H_kv + 1) * p.H_kv] - cum[(seg / p.H_kv) * p.H_kv]
                                 : ncta;
  // fused: the consumers may overwrite `cum` once the producer has read it
  if (FUSED && warp == CONSUMERS) named_bar_arrive(2, THREADS);
  const int b = seg / p.H_kv, h = seg % p.H_kv;
  const Part pt = partition(seq_len(p, b), p.I_b, p.L_b);
  const int nA = blocks_a(pt, p.dense);
  const int a0 = (int)((long long)ci * nA / ncta), a1 = (int)((long long)(ci + 1) * nA / ncta);

  if (warp == CONSUMERS) {
    // =========================== producer warp ===============================
    const uint64_t policy = l2_evict_first_policy();
    if (lane == 0) {
      const uint32_t qbytes = (uint32_t)p.G * D * 2;
      mbar_arrive_expect_tx(bar_q, qbytes);
      bulk_load(smem_u32(smem + SmemLayout::q), p.q + ((size_t)b * H_q + h * p.G) * D, qbytes,
                bar_q);
    }
    // fused: this CTA's selected page ids, written by the consumer warps
    const int* fslice = nullptr;
    if (FUSED) {
      const FusedMergeLayout Lm =
          fused_merge_layout(p.ncpu, p.kk_f, min(p.top_k, p.ncpu * p.kk_f));
      fslice = reinterpret_cast<const int*>(smem + SmemLayout::scratch + Lm.slice);
    }
    uint32_t it = 0;
    bool ok = true;
    bool scored = !FUSED;
    // phase 0: list index i -> Initial/Local block; phase 1: i -> selected block
    auto produce = [&](int phase, int u0, int u1) {
      for (int base = u0; base < u1 && ok; base += 32) {
        const int i = base + lane;
        int ntok = 0, row = 0;
        if (i < u1) {
          int j, page = -1;
          if (phase == 0) {
            j = (p.dense || i < pt.c0) ? i : pt.c1 + (i - pt.c0);
            page = p.table[(size_t)b * p.max_blocks + j];
          } else if (FUSED) {
            j = pt.c0;  // a selected Context block: full
            page = fslice[i];
          } else if (p.sel_pages == nullptr) {
            const int unit = p.SEL == 1 ? 0 : h;
            j = p.sel[((size_t)b * p.SEL + unit) * p.top_k + i];
            if (j < pt.c0 || j >= pt.c1) {
              set_status(p.status, KT_ERR_DEVICE_CHECK);
              j = -1;
            } else {
              page = p.table[(size_t)b * p.max_blocks + j];
            }
          } else {
            j = pt.c0;  // a selected Context block: full; its page comes with the selection
            page = p.sel_pages[((size_t)b * p.SEL + (p.SEL == 1 ? 0 : h)) * p.top_k + i];
          }
          if (j >= 0) {
            if (page < 0 || page >= p.P) {
              set_status(p.status, KT_ERR_DEVICE_CHECK);
            } else {
              ntok = min(UNIT, pt.n - j * BS);
              row = (page * p.H_kv + h) * BS;
            }
          }
        }
        const int nbatch = min(32, u1 - base);
        for (int k = 0; k < nbatch; ++k) {
          const int ntok_k = __shfl_sync(0xffffffffu, ntok, k);
          const int row_k = __shfl_sync(0xffffffffu, row, k);
          const uint32_t st = it % STAGES;
          int okl = 1;
          if (lane == 0) {
            if (it >= STAGES &&
                !mbar_wait(bar_empty + 8 * st, ((it / STAGES) - 1) & 1, p.status))
              okl = 0;
            // fused: the Initial/Local loads start once this CTA's slice is
            // scored, so the representative rows (the selection's critical
            // path) do not queue behind them in HBM; by then the stages that
            // held those rows are free as well
            if (okl && !scored && ntok_k > 0) {
              mbar_wait_sleep(bar_scored, 0, p.status, 64);
              scored = true;
            }
            if (okl) {
              info[st].ntok = ntok_k;
              info[st].end = 0;
              const uint32_t bar = bar_full + 8 * st;
              if (ntok_k > 0) {
                mbar_arrive_expect_tx(bar, KV_STAGE_BYTES);
                const uint32_t dst = kv_base + st * KV_STAGE_BYTES;
                tma_load_2d(dst, &p.kmap, 0, row_k, bar, policy);
                tma_load_2d(dst + BOX_BYTES, &p.kmap, 64, row_k, bar, policy);
                tma_load_2d(dst + 2 * BOX_BYTES, &p.vmap, 0, row_k, bar, policy);
                tma_load_2d(dst + 3 * BOX_BYTES, &p.vmap, 64, row_k, bar, policy);
              } else {
                mbar_arrive(bar);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
          if (!ok) break;
          ++it;
        }
      }
    };
    produce(0, a0, a1);
    if (FUSED) {
      // phase B: this CTA's share of the selected blocks, handed over by the
      // consumer warps once the unit's selection is complete
      int n1 = 0;
      if (lane == 0 && mbar_wait_sleep(bar_sel, 0, p.status, 128)) n1 = bcast[61];
      n1 = __shfl_sync(0xffffffffu, n1, 0);
      if (ok) produce(1, 0, n1);
    } else {
      // Phase B needs the selection: wait for the grid this launch depends on.
      griddep_wait();
      int nB = 0;
      if (!p.dense) {
        const int cmax = blocks_b_max(pt, 0, p.top_k);
        nB = p.cnt ? p.cnt[b * p.SEL + (p.SEL == 1 ? 0 : h)] : cmax;
        if (nB < 0 || nB > cmax) {
          set_status(p.status, KT_ERR_DEVICE_CHECK);
          nB = nB < 0 ? 0 : cmax;
        }
      }
      if (ok)
        produce(1, (int)((long long)ci * nB / ncta), (int)((long long)(ci + 1) * nB / ncta));
    }
    if (ok && lane == 0) {
      const uint32_t st = it % STAGES;
      if (it < STAGES || mbar_wait(bar_empty + 8 * st, ((it / STAGES) - 1) & 1, p.status)) {
        info[st].end = 1;
        info[st].ntok = 0;
        mbar_arrive(bar_full + 8 * st);
      }
    }
    return;
  }

  // ============================ consumer warps ===============================
  const int g = lane >> 2, t = lane & 3;
  const int ctid = tid;

  if constexpr (FUSED) {
    const int n1 = fused_merge(p, reinterpret_cast<uint8_t*>(scratch), f_hist, f_sh_u64,
                               f_sh_int, b, h, ci, ncta, ctid, bar_c);
    if (ctid == 0) {
      bcast[61] = n1;
      mbar_arrive(bar_sel);
      // the last of the unit's npoll waiting CTAs zeroes its tickets for the
      // next launch (every other waiter has read them by then)
      const int unit = b * p.SEL + (p.SEL == 1 ? 0 : h);
      if (atomicAdd(p.f_polled + unit, 1) == npoll - 1) {
        p.f_counters[unit] = 0;
        p.f_polled[unit] = 0;
      }
    }
  }
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  float m_run = -INFINITY, l_part = 0.0f;
  uint32_t qa[8][2];
  bool q_loaded = false;

  for (uint32_t it = 0;; ++it) {
    const uint32_t st = it % STAGES;
    if (!mbar_wait(bar_full + 8 * st, (it / STAGES) & 1, p.status)) break;
    const StageInfo in = info[st];
    if (in.end) break;
    if (in.ntok > 0 && !q_loaded) {
      if (!mbar_wait(bar_q, 0, p.status)) break;
      // query rows -> A fragments (rows >= G are zero)
      const __half* qs = reinterpret_cast<const __half*>(smem + SmemLayout::q);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        if (g < p.G) {
          qa[kk][0] = *reinterpret_cast<const uint32_t*>(qs + g * D + kk * 16 + 2 * t);
          qa[kk][1] = *reinterpret_cast<const uint32_t*>(qs + g * D + kk * 16 + 8 + 2 * t);
        } else {
          qa[kk][0] = qa[kk][1] = 0u;
        }
      }
      q_loaded = true;
    }
    if (in.ntok > warp * 16) {
      const uint32_t kb = kv_base + st * KV_STAGE_BYTES;
      const uint32_t vb = kb + 2 * BOX_BYTES;
      const int mi = lane >> 3, r = lane & 7;
      // ---- S = q K^T for this warp's 16 tokens: two n-tiles, each with two
      // independent accumulation chains over the 8 k-steps
      float s[2][2][4];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int c = 0; c < 2; ++c) s[a][c][0] = s[a][c][1] = s[a][c][2] = s[a][c][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int tok = warp * 16 + (mi >> 1) * 8 + r;
        const int chunk = kk * 2 + (mi & 1);
        const uint32_t addr = kb + (chunk >> 3) * BOX_BYTES + tok * 128 +
                              (((chunk & 7) ^ (tok & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, addr);
        mma_16816(s[0][kk & 1], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
        mma_16816(s[1][kk & 1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
      }
      // ---- online softmax (base 2), rows = query heads
      const int tok0 = warp * 16 + 2 * t;
      float x[4];
      x[0] = (tok0 < in.ntok) ? (s[0][0][0] + s[0][1][0]) * p.scale_log2 : -INFINITY;
      x[1] = (tok0 + 1 < in.ntok) ? (s[0][0][1] + s[0][1][1]) * p.scale_log2 : -INFINITY;
      x[2] = (tok0 + 8 < in.ntok) ? (s[1][0][0] + s[1][1][0]) * p.scale_log2 : -INFINITY;
      x[3] = (tok0 + 9 < in.ntok) ? (s[1][0][1] + s[1][1][1]) * p.scale_log2 : -INFINITY;
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      float pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = exp2f(x[i] - m_use);
      if (__any_sync(0xffffffffu, m_new != m_run)) {
        const float alpha = exp2f(m_run - m_use);
        l_part *= alpha;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc[i][0] *= alpha;
          acc[i][1] *= alpha;
          acc[i][2] *= alpha;
          acc[i][3] *= alpha;
        }
      }
      m_run = m_new;
      l_part += (pr[0] + pr[1]) + (pr[2] + pr[3]);
      // ---- P = P_hi + P_lo (rows 0..7 hi, rows 8..15 lo)
      __half hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hi[i] = __float2half_rn(pr[i]);
        lo[i] = __float2half_rn(pr[i] - __half2float(hi[i]));
      }
      const uint32_t pa0 = pack_half2(hi[0], hi[1]);
      const uint32_t pa1 = pack_half2(lo[0], lo[1]);
      const uint32_t pa2 = pack_half2(hi[2], hi[3]);
      const uint32_t pa3 = pack_half2(lo[2], lo[3]);
      // ---- O += P V
#pragma unroll
      for (int cp = 0; cp < 8; ++cp) {
        const int tok = warp * 16 + (mi & 1) * 8 + r;
        const int chunk = cp * 2 + (mi >> 1);
        const uint32_t addr = vb + (chunk >> 3) * BOX_BYTES + tok * 128 +
                              (((chunk & 7) ^ (tok & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, addr);
        mma_16816(acc[2 * cp], pa0, pa1, pa2, pa3, b0, b1);
        mma_16816(acc[2 * cp + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * st);
  }

  // a CTA without units still owns the query copy it started: let it land
  if (!q_loaded && warp == 0) mbar_wait(bar_q, 0, p.status);

  // ---- merge the eight warp states: warps 4..7 into 0..3, then 0..3 --------
  float l_row = l_part;
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
  float o[32];  // this lane's 32 channels of head g: nt*8 + 2t (+1)
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    o[2 * nt] = acc[nt][0] + acc[nt][2];
    o[2 * nt + 1] = acc[nt][1] + acc[nt][3];
  }
  const int wl = warp & (HALF_WARPS - 1);
  float* sc = scratch + (wl * MAX_G + g) * (D + 2);
  if (warp >= HALF_WARPS && g < p.G) {
    if (t == 0) {
      sc[0] = m_run;
      sc[1] = l_row;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      sc[2 + nt * 8 + 2 * t] = o[2 * nt];
      sc[2 + nt * 8 + 2 * t + 1] = o[2 * nt + 1];
    }
  }
  named_bar_sync(1, NCT);
  if (warp < HALF_WARPS && g < p.G) {
    const float m2 = sc[0], l2 = sc[1];
    const float M = fmaxf(m_run, m2);
    const float wa = (M == -INFINITY) ? 0.0f : exp2f(m_run - M);
    const float wb = (M == -INFINITY) ? 0.0f : exp2f(m2 - M);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[2 * nt] = o[2 * nt] * wa + sc[2 + nt * 8 + 2 * t] * wb;
      o[2 * nt + 1] = o[2 * nt + 1] * wa + sc[2 + nt * 8 + 2 * t + 1] * wb;
    }
    l_row = l_row * wa + l2 * wb;
    m_run = M;
  }
  named_bar_sync(1, NCT);
  if (warp < HALF_WARPS && g < p.G) {
    if (t == 0) {
      sc[0] = m_run;
      sc[1] = l_row;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      sc[2 + nt * 8 + 2 * t] = o[2 * nt];
      sc[2 + nt * 8 + 2 * t + 1] = o[2 * nt + 1];
    }
  }
  named_bar_sync(1, NCT);
  // per head: M over the four states, weights, L
  float* fw = reinterpret_cast<float*>(bcast + 16);  // [G][4] weights
  float* fm = reinterpret_cast<float*>(bcast);       // [G] M, [G] L at +MAX_G
  if (ctid < p.G) {
    const int gg = ctid;
    float M = -INFINITY;
    for (int w = 0; w < HALF_WARPS; ++w) M = fmaxf(M, scratch[(w * MAX_G + gg) * (D + 2)]);
    float L = 0.0f;
    for (int w = 0; w < HALF_WARPS; ++w) {
      const float* s2 = scratch + (w * MAX_G + gg) * (D + 2);
      const float wt = (M == -INFINITY) ? 0.0f : exp2f(s2[0] - M);
      fw[gg * HALF_WARPS + w] = wt;
      L += s2[1] * wt;
    }
    fm[gg] = M;
    fm[MAX_G + gg] = L;
  }
  named_bar_sync(1, NCT);

  if (ncta == 1) {
    // the only CTA of its segment: normalise and write the output
    for (int idx = ctid; idx < p.G * D; idx += NCT) {
      const int gg = idx / D, c = idx % D;
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < HALF_WARPS; ++w)
        v = fmaf(scratch[(w * MAX_G + gg) * (D + 2) + 2 + c], fw[gg * HALF_WARPS + w], v);
      const float L = fm[MAX_G + gg];
      p.out[((size_t)b * H_q + h * p.G + gg) * D + c] = L > 0.0f ? v / L : 0.0f;
    }
    return;
  }

  // ---- partial (slot = this CTA): O[G][128], then m[G], then l[G] (base 2)
  const int slot_stride = p.slot_floats;
  float* dst = p.parts + (size_t)cta * slot_stride;
  for (int idx = ctid; idx < p.G * D; idx += NCT) {
    const int gg = idx / D, c = idx % D;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < HALF_WARPS; ++w)
      v = fmaf(scratch[(w * MAX_G + gg) * (D + 2) + 2 + c], fw[gg * HALF_WARPS + w], v);
    dst[gg * D + c] = v;
    if (c == 0) {
      dst[p.G * D + gg] = fm[gg];
      dst[p.G * D + p.G + gg] = fm[MAX_G + gg];
    }
  }
  named_bar_sync(1, NCT);
  if constexpr (FUSED) {
    // every CTA is resident: the segment's first CTA merges once the others'
    // partials are in; the others leave as soon as theirs is released
    if (ci != 0) {
      if (ctid == 0) red_release_gpu_add(p.counters + seg, 1);
      return;
    }
    if (ctid == 0) {
      const uint64_t t0 = globaltimer();
      for (uint32_t i = 0;; ++i) {
        if (ld_acquire_gpu(p.counters + seg) >= ncta - 1) break;
        if ((i & 63u) == 63u && globaltimer() - t0 > WAIT_LIMIT_NS) {
          set_status(p.status, KT_ERR_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
      p.counters[seg] = 0;  // all ncta - 1 tickets are in
    }
    named_bar_sync(1, NCT);
  } else {
    if (ctid == 0) {
      const int old = atom_acq_rel_gpu_add(p.counters + seg, 1);
      bcast[60] = (old + 1 == ncta) ? 1 : 0;
    }
    named_bar_sync(1, NCT);
    if (!bcast[60]) return;
  }

  // ---- last CTA of the segment: merge partials of CTAs f0 .. f0+ncta-1.
  // Each thread owns one float4 chunk of the G x 128 outputs and a share of
  // the partials, loaded 16 at a time with independent loads and merged
  // online; the shares are combined through shared memory in a fixed order.
  float* red = scratch;  // per thread: M, L, O.xyzw
  const int nchunk = p.G * D / 4;
  const int nsplit = NCT / nchunk;  // 1 (G=8), 2 (G=4), 4, 8
  const int chn = ctid % nchunk, sp = ctid / nchunk;
  const int f = 4 * chn, gg = f / D;
  const int i0 = sp * ncta / nsplit, i1 = (sp + 1) * ncta / nsplit;
  float M = -INFINITY, L = 0.0f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = i0; base < i1; base += 16) {
    const int nb = min(16, i1 - base);
    float m[16], l[16];
    float4 ov[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (k < nb) {
        const float* src = p.parts + (size_t)(f0 + base + k) * slot_stride;
        m[k] = __ldcg(src + p.G * D + gg);
        l[k] = __ldcg(src + p.G * D + p.G + gg);
        ov[k] = __ldcg(reinterpret_cast<const float4*>(src + f));
      } else {
        m[k] = -INFINITY;
        l[k] = 0.0f;
        ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mn = M;
#pragma unroll
    for (int k = 0; k < 16; ++k) Mn = fmaxf(Mn, m[k]);
    if (Mn == -INFINITY) continue;
    const float a = exp2f(M - Mn);  // 0 when M is -inf
    L *= a;
    O.x *= a;
    O.y *= a;
    O.z *= a;
    O.w *= a;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float w = exp2f(m[k] - Mn);  // 0 for empty partials
      L = fmaf(l[k], w, L);
      O.x = fmaf(ov[k].x, w, O.x);
      O.y = fmaf(ov[k].y, w, O.y);
      O.z = fmaf(ov[k].z, w, O.z);
      O.w = fmaf(ov[k].w, w, O.w);
    }
    M = Mn;
  }
  if (nsplit > 1) {
    named_bar_sync(1, NCT);  // scratch (red) was read above for the weights
    float* r6 = red + 6 * ctid;
    r6[0] = M;
    r6[1] = L;
    r6[2] = O.x;
    r6[3] = O.y;
    r6[4] = O.z;
    r6[5] = O.w;
    named_bar_sync(1, NCT);
    if (sp == 0) {
      for (int qd = 1; qd < nsplit; ++qd) {
        const float* o2 = red + 6 * (ctid + qd * nchunk);
        const float Mn = fmaxf(M, o2[0]);
        if (Mn == -INFINITY) continue;
        const float a = exp2f(M - Mn), w = exp2f(o2[0] - Mn);
        L = L * a + o2[1] * w;
        O.x = O.x * a + o2[2] * w;
        O.y = O.y * a + o2[3] * w;
        O.z = O.z * a + o2[4] * w;
        O.w = O.w * a + o2[5] * w;
        M = Mn;
      }
    }
  }
  if (sp == 0) {
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    *reinterpret_cast<float4*>(p.out + ((size_t)b * H_q + h * p.G + gg) * D + (f % D)) =
        make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
  }
  if (!FUSED && ctid == 0) p.counters[seg] = 0;
}

}  // namespace

// Per device: the shared-memory opt-in of both variants (0 = done, else the
// error), and the resident CTAs of the fused variant per SM.
int attn_smem_optin() {
  static std::atomic<int> slot[KT_MAX_DEVICES];
  return per_device_cached(slot, [] {
    cudaError_t e = cudaSuccess;
    for (const void* f : {(const void*)attn_kernel<SK_NONE>, (const void*)attn_kernel<SK_COLS>,
                          (const void*)attn_kernel<SK_LINEAR>, (const void*)attn_kernel<SK_MMA>,
                          (const void*)attn_kernel<SK_F32>, (const void*)attn_kernel<SK_MULTI>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    return (int)e;
  });
}

int attn_fused_max_ctas_per_sm() {
  static std::atomic<int> slot[KT_MAX_DEVICES];
  return per_device_cached(slot, [] {
    if (attn_smem_optin() != 0) return 0;
    int n = 0;
    // every instantiation needs the same resources; the largest register
    // count decides
    int m = 1 << 30;
    for (const void* f : {(const void*)attn_kernel<SK_COLS>, (const void*)attn_kernel<SK_LINEAR>,
                          (const void*)attn_kernel<SK_MMA>, (const void*)attn_kernel<SK_F32>,
                          (const void*)attn_kernel<SK_MULTI>}) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, THREADS, SMEM_BYTES) !=
          cudaSuccess)
        return 0;
      m = n < m ? n : m;
    }
    return m;
  });
}

cudaError_t launch_attention(const AttnLaunch& a, cudaStream_t stream) {
  const cudaError_t e = (cudaError_t)attn_smem_optin();
  if (e != cudaSuccess) return e;
  Params p;
  p.kmap = *a.kmap;
  p.vmap = *a.vmap;
  p.q = a.q;
  p.table = a.table;
  p.seq_lens = a.seq_lens;
  p.sel = a.sel;
  p.cnt = a.cnt;
  p.sel_pages = a.sel_pages;
  p.out = a.out;
  p.status = a.status;
  p.counters = a.counters;
  p.parts = a.parts;
  p.B = a.B;
  p.H_kv = a.H_kv;
  p.G = a.G;
  p.max_blocks = a.max_blocks;
  p.P = a.P;
  p.I_b = a.I_b;
  p.L_b = a.L_b;
  p.top_k = a.top_k;
  p.SEL = a.SEL;
  p.dense = a.dense;
  p.slot_floats = a.slot_floats;
  p.scale_log2 = a.scale_log2;
  p.reps = a.reps;
  p.rep = a.rep;
  p.R = a.R;
  p.ncpu = a.ncpu;
  p.f_chunk = a.f_chunk;
  p.kk_f = a.kk_f;
  p.f_cand = a.f_cand;
  p.f_cand_pages = a.f_cand_pages;
  p.f_counters = a.f_counters;
  p.f_polled = a.f_polled;
  p.sel_out = a.sel_out;
  p.cnt_out = a.cnt_out;
  p.presel_mask = a.presel_mask;
  p.presel_cnt = a.presel_cnt;
  p.mask_words = a.mask_words;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (a.fused) {
    // every CTA must be resident: the producers wait for selection flags set
    // by other CTAs of the same grid
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!a.fused) return cudaLaunchKernelEx(&cfg, attn_kernel<SK_NONE>, p);
  switch (a.sk) {
    case SK_COLS: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_COLS>, p);
    case SK_LINEAR: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_LINEAR>, p);
    case SK_MMA: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_MMA>, p);
    case SK_F32: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_F32>, p);
    case SK_MULTI: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_MULTI>, p);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kt
