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
//     into a 3-stage shared-memory ring.  Every launch is a programmatic
//     dependent of the kernel before it on the stream: it waits for that
//     kernel at entry, except behind the selection kernel, where phase B alone
//     waits (griddepcontrol.wait) and the Initial/Local blocks stream while
//     the selection runs.
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
// launch of one CTA per SM) also makes the selection (§3.1, §4.3, §4.5).
// While the producer finds the CTA's segment, the consumer warps stage and
// score one slice of a selection unit's Context blocks (fused_score) and
// write the slice's candidates to tagged slots; every CTA then reads its
// unit's slots until all carry this launch's tag, finds the top-k threshold
// (kth_largest_reg), orders the chosen blocks by id (fused_pick) and issues
// its first chosen blocks' loads itself.  Split-K
// partials are tagged words as well, and every CTA of a segment merges its
// share of the output channels from all of them.  No ticket, fence or atomic
// that anyone waits on is left: the tags come from a launch counter that each
// CTA advances by its share without waiting.  SK selects the scoring path at
// compile time, so a launch carries only the code it runs.
#include "select_common.cuh"

namespace kt {
namespace {

constexpr int STAGES = 3;
constexpr int CONSUMERS = 8;

// A compile-time int carried through generic lambdas.
template <int N>
struct IntC {
  static constexpr int value = N;
};
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

// Q8_0 source: per stage the int8 codes of K and V (16 KB each, 128-byte
// swizzled TMA boxes) and their binary16 scales (1 KB each); each consumer
// warp dequantises its 16 token rows into one fp16 block in the layout the
// fp16 stages have, at the start of the ring, and the int8 stages follow it.
constexpr int Q8_CODE_BYTES = UNIT * D;
constexpr int Q8_SCALE_BYTES = UNIT * (D / 32) * 2;
constexpr int Q8_STAGE_BYTES = 2 * Q8_CODE_BYTES + 2 * Q8_SCALE_BYTES;
constexpr int Q8_RING_OFF = KV_STAGE_BYTES;
static_assert(Q8_RING_OFF + STAGES * Q8_STAGE_BYTES <= STAGES * KV_STAGE_BYTES,
              "Q8_0 stages and the dequantised block fit the ring");
static_assert(Q8_STAGE_BYTES % 1024 == 0, "128-byte swizzled boxes need 1024-byte alignment");

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
  static constexpr int bcast = bars + (2 * STAGES + 6) * 8;
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
  // fused step only: in-kernel selection (fused_score, fused_pick)
  const void* reps;
  int rep, R, ncpu, f_chunk, kk_f;
  unsigned long long* f_cand;
  int f_cand_len;
  uint32_t* f_cpage;
  unsigned long long* f_sync;
  int32_t* sel_out;
  int32_t* cnt_out;
  const uint32_t* presel_mask;
  const int32_t* presel_cnt;
  int mask_words;
  unsigned long long* stamps;
  const __half* k_src;    // KVM_HOST: fp16 pools in device-accessible host memory
  const __half* v_src;
  const __half* k_scale;  // KVM_Q8: binary16 scales [P][H_kv][128][4]
  const __half* v_scale;
  int skip_publish;                  // fused, failure-path test only: CTA + 1, 0 = none
  int wait_at_entry;  // programmatic dependent: wait for the previous grid before any global access
  int q_mapped;       // q and out in page-locked host memory (plain loads, no bulk copy of q)
  unsigned long long poll_limit_ns;  // fused: bound of the slot and partial polls
};

// Phase stamp i of this CTA (global timer, ns) when stamps are requested.
#define KT_STAMP(p, i)                                                                  \
  do {                                                                                  \
    if ((p).stamps) (p).stamps[(size_t)blockIdx.x * KT_PHASE_STAMPS + (i)] = globaltimer(); \
  } while (0)

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
// weights, dot products and keys as the selection kernel and write the slice's
// best kk_f keys (key 0 = empty slot) to its tagged slots.
// Arrives on bar_scored once its staged representative rows are scored
// (every CTA; the ring is then free).
// The block-table entries of the nominal slice do not depend on the sequence
// length, so they load together with the length and the query rows.
template <int SK, class Bar>
__device__ void fused_score(const Params& p, uint8_t* scr, unsigned int* hist,
                            unsigned long long* sh_u64, int* sh_int, int ctid, int warp, int lane,
                            Bar bar_c, uint32_t bar_scored, const uint8_t* ring,
                            uint32_t ring_u32, uint32_t bar_reps) {
  const int U = p.B * p.SEL;
  const int u = blockIdx.x / p.ncpu;
  // this launch's epoch: its slot and partial tags, which every CTA needs for
  // the pick, are set once the slice's first loads are out; this CTA's share
  // of the advance to the next epoch is added once its slots are written
  // (every CTA passes there exactly once, whatever its waits gave)
  unsigned long long counter = 0;
  if (ctid == 0) {
    counter = ld_relaxed_gpu_u64(p.f_sync);
  }
  auto add_share = [&] {
    const unsigned long long c = blockIdx.x, g = gridDim.x;
    red_relaxed_gpu_add_u64(p.f_sync, (((c + 1) << FUSED_EPOCH_SHIFT) / g) -
                                          ((c << FUSED_EPOCH_SHIFT) / g));
  };
  auto set_tags = [&] {
    const unsigned long long epoch = counter >> FUSED_EPOCH_SHIFT;
    sh_int[12] = (int)(1u + (uint32_t)(epoch % FUSED_TAG_CYCLE));
    sh_int[15] = (int)(1u + (uint32_t)(epoch % 0xFFFFFFFEull));  // partial tag (never 0)
  };
  // the slots past this launch's layout get tag 0: each launch writes every slot
  auto fill_tail = [&] {
    const int used = U * p.ncpu * p.kk_f;
#pragma unroll 1
    for (int i = used + (int)blockIdx.x * NCT + ctid; i < p.f_cand_len; i += (int)gridDim.x * NCT) {
      st_relaxed_gpu_u64(p.f_cand + i, 0ull);
      st_relaxed_gpu_u32(p.f_cpage + i, 0u);
    }
  };
  if (u >= U) {
    fill_tail();
    if (ctid == 0) {
      set_tags();
      mbar_arrive(bar_scored);
      add_share();
    }
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
  const int n_bu = seq_len(p, bu);  // in flight with the block-table loads below
#pragma unroll 1
  for (int i = ctid; i < p.f_chunk; i += NCT) {
    const int j = js + i;
    pgs[i] = j < p.max_blocks ? __ldg(p.table + (size_t)bu * p.max_blocks + j) : -1;
  }
  fill_tail();
  // the slice's candidate and page slots, each written once below with this
  // launch's tag
  unsigned long long* cand = p.f_cand + ((size_t)u * p.ncpu + cs) * p.kk_f;
  uint32_t* cpage = p.f_cpage + ((size_t)u * p.ncpu + cs) * p.kk_f;
  const Part pu = partition(n_bu, p.I_b, p.L_b);
  const int je = min(js + p.f_chunk, pu.c1);
  const int nloc = max(0, je - js);  // js >= c0 whenever the slice is not empty
  if (ctid == 0) set_tags();
  bar_c();
  if (ctid == 0) KT_STAMP(p, 1);
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
      if (r == 0 && ctid == 0) KT_STAMP(p, 2);
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
  if (ctid == 0) {
    mbar_arrive(bar_scored);  // the staged rows are scored: the ring is free
    KT_STAMP(p, 3);
  }
  // the slice's best min(nloc, kk_f) keys as tagged slots, then its empty
  // slots; no fence: readers check each slot's tag (failure-path test: one
  // CTA publishes nothing, so its unit's polls time out)
  const uint32_t tag = (int)blockIdx.x + 1 == p.skip_publish ? 0u : (uint32_t)sh_int[12];
  if (p.presel_mask) {
    // preselection: blocks outside it get key 0, the empty slot
    const uint32_t* mk = p.presel_mask + (size_t)u * p.mask_words;
#pragma unroll 1
    for (int i = ctid; i < nloc; i += NCT) {
      const int j = js + i;
      if (!((__ldg(mk + (j >> 5)) >> (j & 31)) & 1u)) keys[i] = 0ull;
    }
    bar_c();
  }
  if (nloc <= p.kk_f) {
    // every key of the slice is a candidate: block i goes to slot i (a zero
    // key is an empty slot).  SK_COLS launches (slices of at most top_k
    // blocks) always take this path.
#pragma unroll 1
    for (int i = ctid; i < p.kk_f; i += NCT) {
      const bool in = i < nloc;
      st_relaxed_gpu_u64(cand + i, fused_slot(in ? keys[i] : 0ull, tag));
      st_relaxed_gpu_u32(cpage + i, in ? (((uint32_t)pgs[i] & 0xFFFFFu) << FUSED_TAG_BITS | tag) : tag);
    }
  } else if constexpr (SK != SK_COLS) {
    // the slice's best kk_f keys (slices hold at most FUSED_MAX_CHUNK = 8 NCT
    // blocks, the host's plan): the threshold on the keys held in registers
    // (key i of the slice in thread i % NCT, register i / NCT), with as few
    // registers a thread as the plan's slices need (the code runs once per
    // launch, so its length is part of its cost)
    auto top = [&](auto gps) {
      constexpr int GPS = decltype(gps)::value;
      unsigned long long kr[GPS];
      uint32_t pr[GPS];
#pragma unroll
      for (int r = 0; r < GPS; ++r) {
        const int i = ctid + r * NCT;
        kr[r] = i < nloc ? keys[i] : 0ull;
        pr[r] = i < nloc ? (uint32_t)pgs[i] : 0u;
      }
      // the threshold's scratch overlays the weights, keys and pages, all held
      // in registers or dead by now (its first barrier precedes its first store)
      unsigned int* hs = reinterpret_cast<unsigned int*>(scr);
      unsigned long long* bk = reinterpret_cast<unsigned long long*>(scr + FUSED_KTH_BINK);
      int* wc = reinterpret_cast<int*>(scr + FUSED_KTH_COUNTS);
      int N = 0;
      if (ctid == 0) *wc = 0;  // ordered before the atomics by the threshold's barriers
      const unsigned long long T =
          selc::kth_largest_reg<NCT, GPS>(kr, p.kk_f, hs, bk, sh_u64, sh_int, &N, ctid, bar_c);
      // the chosen keys into the first slots, one shared atomic per warp
      const unsigned int lt = (1u << lane) - 1u;
      unsigned int bal[GPS];
      int tot = 0;
#pragma unroll
      for (int r = 0; r < GPS; ++r) {
        bal[r] = __ballot_sync(0xffffffffu, kr[r] != 0ull && kr[r] >= T);
        tot += __popc(bal[r]);
      }
      int o = 0;
      if (lane == 0 && tot) o = atomicAdd(wc, tot);
      o = __shfl_sync(0xffffffffu, o, 0);
#pragma unroll
      for (int r = 0; r < GPS; ++r) {
        const int pos = o + __popc(bal[r] & lt);
        if (((bal[r] >> lane) & 1u) && pos < p.kk_f) {
          st_relaxed_gpu_u64(cand + pos, fused_slot(kr[r], tag));
          st_relaxed_gpu_u32(cpage + pos, (pr[r] & 0xFFFFFu) << FUSED_TAG_BITS | tag);
        }
        o += __popc(bal[r]);
      }
#pragma unroll 1
      for (int r = min(N, p.kk_f) + ctid; r < p.kk_f; r += NCT) {
        st_relaxed_gpu_u64(cand + r, tag);
        st_relaxed_gpu_u32(cpage + r, tag);
      }
    };
    if (p.f_chunk <= 2 * NCT) top(IntC<2>{});
    else if (p.f_chunk <= 4 * NCT) top(IntC<4>{});
    else top(IntC<FUSED_MAX_CHUNK / NCT>{});
  }
  // the slots carry their own validity: no fence
  if (ctid == 0) {
    KT_STAMP(p, 4);
    add_share();
  }
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

// Fused step, consumer warps of every CTA: read the candidate slots of this
// segment's selection unit until each carries this launch's tag (one round of
// loads once the unit's slices are published; no fence on either side), find
// the threshold of the unit's top keff keys (kth_largest_reg: keys held in
// registers, ties to the lower block as the keys order them), order the
// chosen blocks by id and return this CTA's share [i0, i0 + n) of them: n,
// with i0 in *i0_out.  The ascending ids stay in the pick layout's `sorted`
// array, where the producer reads them.  One CTA per unit writes sel / cnt.
template <int GP, class Bar>
__device__ int fused_pick(const Params& p, uint8_t* scr, unsigned long long* sh_u64, int* sh_int,
                          int b, int h, const Part& pt, int ci, int ncta, int ctid, Bar bar_c,
                          int* i0_out, uint32_t bar_seen) {
  const int unit = b * p.SEL + (p.SEL == 1 ? 0 : h);
  int keff = min(p.top_k, pt.c1 - pt.c0);
  if (p.presel_mask) keff = min(keff, max(0, __ldg(p.presel_cnt + unit)));
  const int nslots = p.ncpu * p.kk_f, kmax = min(p.top_k, nslots);
  const FusedPickLayout Lp = fused_pick_layout(nslots, kmax);
  int* sorted = reinterpret_cast<int*>(scr + Lp.sorted);
  int* sorted_pages = reinterpret_cast<int*>(scr + Lp.sorted_pages);
  const bool writer = ci == 0 && (p.SEL != 1 || h == 0);
  const uint32_t tag = (uint32_t)sh_int[12];
  uint32_t* ids = reinterpret_cast<uint32_t*>(scr + Lp.ids);
  int* pages = reinterpret_cast<int*>(scr + Lp.pages);
  const int kpad = (kmax + 3) & ~3;
  if (ctid == 0) sh_int[13] = 0;
#pragma unroll 1
  for (int i = ctid; i < kpad; i += NCT) ids[i] = 0xFFFFFFFFu;
  // every slot of the unit, read until all carry the tag (bounded)
  static_assert(GP <= FUSED_GATHER_PER_THREAD, "slots a thread holds");
  const unsigned long long* src = p.f_cand + (size_t)unit * nslots;
  const uint32_t* srcp = p.f_cpage + (size_t)unit * nslots;
  unsigned long long kx[GP];
  uint32_t px[GP];
  bool ok = false;
  const uint64_t t0 = globaltimer();
#pragma unroll 1
  for (;;) {
    ok = true;
#pragma unroll
    for (int r = 0; r < GP; ++r) {
      const int s = ctid + r * NCT;
      kx[r] = s < nslots ? ld_relaxed_gpu_u64(src + s) : static_cast<unsigned long long>(tag);
      px[r] = s < nslots ? ld_relaxed_gpu_u32(srcp + s) : tag;
      ok = ok && (static_cast<uint32_t>(kx[r]) & ((1u << FUSED_TAG_BITS) - 1u)) == tag &&
           (px[r] & ((1u << FUSED_TAG_BITS) - 1u)) == tag;
    }
    if (named_bar_and(1, NCT, ok || globaltimer() - t0 > p.poll_limit_ns)) break;
  }
  if (!ok) set_status(p.status, KT_ERR_TIMEOUT);
  if (ctid == 0) {
    mbar_arrive(bar_seen);  // the producer may start the Initial/Local loads
    KT_STAMP(p, 5);
  }
  *i0_out = 0;
  if (keff <= 0) {
    if (writer && ctid == 0) p.cnt_out[unit] = 0;
    return 0;
  }
#pragma unroll
  for (int r = 0; r < GP; ++r) kx[r] &= ~((1ull << FUSED_TAG_BITS) - 1ull);  // empty: 0
  int N = 0;
  const unsigned long long T = selc::kth_largest_reg<NCT, GP>(
      kx, keff, reinterpret_cast<unsigned int*>(scr + Lp.hist),
      reinterpret_cast<unsigned long long*>(scr + Lp.bink), sh_u64, sh_int, &N, ctid, bar_c);
  if (N < keff) {
    if (ctid == 0) set_status(p.status, KT_ERR_DEVICE_CHECK);
    keff = N;
    if (keff <= 0) {
      if (writer && ctid == 0) p.cnt_out[unit] = 0;
      return 0;
    }
  }
  // the chosen blocks' ids, one shared atomic per warp
  {
    const int lane = ctid & 31;
    const unsigned int lt = (1u << lane) - 1u;
    unsigned int bal[GP];
    int tot = 0;
#pragma unroll
    for (int r = 0; r < GP; ++r) {
      bal[r] = __ballot_sync(0xffffffffu, kx[r] != 0ull && kx[r] >= T);
      tot += __popc(bal[r]);
    }
    int o = 0;
    if (lane == 0 && tot) o = atomicAdd(&sh_int[13], tot);
    o = __shfl_sync(0xffffffffu, o, 0);
#pragma unroll
    for (int r = 0; r < GP; ++r) {
      const int pos = o + __popc(bal[r] & lt);
      if (((bal[r] >> lane) & 1u) && pos < kpad) {
        ids[pos] = static_cast<uint32_t>(fused_slot_block(kx[r]));
        pages[pos] = static_cast<int>(px[r] >> FUSED_TAG_BITS);
      }
      o += __popc(bal[r]);
    }
  }
  bar_c();
  // position of a chosen block = chosen blocks with a smaller id
#pragma unroll 1
  for (int i = ctid; i < keff; i += NCT) {
    const uint32_t id = ids[i];
    const int r = min(count_less_u32(ids, kpad, id), keff - 1);
    sorted[r] = static_cast<int>(id);
    sorted_pages[r] = pages[i];
    if (writer) p.sel_out[(size_t)unit * p.top_k + r] = static_cast<int32_t>(id);
  }
  if (writer && ctid == 0) p.cnt_out[unit] = keff;
  bar_c();
  const int i0 = ci * keff / ncta, i1 = (ci + 1) * keff / ncta;
  *i0_out = i0;
  return i1 - i0;
}

template <int SK, int KVM = KVM_F16>
__global__ void __launch_bounds__(THREADS, 1) attn_kernel(const __grid_constant__ Params p) {
  constexpr bool FUSED = SK != SK_NONE;
  static_assert(!FUSED || KVM != KVM_HOST, "the one-launch step reads device pools");
  extern __shared__ uint8_t smem_raw[];
  __shared__ unsigned int f_hist[FUSED ? 512 : 1];
  __shared__ unsigned long long f_sh_u64[FUSED ? 2 + 2 * CONSUMERS : 1];
  __shared__ int f_sh_int[FUSED ? 16 : 1];
  // 1024-byte aligned (128-byte swizzled TMA boxes); offsetting the array
  // itself keeps the accesses below in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // launched as a programmatic dependent of whatever precedes it on the
  // stream: only the launch itself overlaps that kernel's tail (a launch
  // behind the selection kernel waits later, before its selected blocks)
  if (p.wait_at_entry) griddep_wait();
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
  const uint32_t bar_seen = bar_reps + 16;   // fused: the unit's candidate slots are all seen
  const uint32_t kv_base = smem_u32(smem + SmemLayout::kv);
  auto bar_c = [] { named_bar_sync(1, NCT); };
  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      // host source: all 32 producer lanes arrive (each once its copies land)
      mbar_init(bar_full + 8 * i, KVM == KVM_HOST ? 32 : 1);
      mbar_init(bar_empty + 8 * i, CONSUMERS);
    }
    mbar_init(bar_q, 1);
    mbar_init(bar_sel, 1);
    mbar_init(bar_scored, 1);
    mbar_init(bar_reps, CONSUMERS);
    mbar_init(bar_reps + 8, CONSUMERS);
    mbar_init(bar_seen, 1);
    fence_mbar_init();
    KT_STAMP(p, 0);
  }
  __syncthreads();

  // ---- set-up: segment work prefix -> this CTA's segment and slice.  In the
  // fused step the consumer warps score their selection slice meanwhile.
  if (warp == CONSUMERS) {
    if (lane == 0 && KVM != KVM_HOST) {  // the host source uses no tensor maps
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
  // CTAs of segment s: [cum[s], cum[s+1]).  In the fused step the producer
  // finds this CTA's segment and its sequence's length while the consumers
  // score, and hands both over in shared memory (the consumers then use the
  // `cum` area for the pick).
  int seg, f0, ncta, n_b;
  if (FUSED && warp != CONSUMERS) {
    named_bar_sync(2, THREADS);
    seg = bcast[56];
    f0 = bcast[57];
    ncta = bcast[58];
    n_b = bcast[59];
  } else {
    if (!FUSED) __syncthreads();
    int lo = 0, hi = S - 1;  // largest s with first(s) <= cta
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= cta) lo = mid; else hi = mid - 1;
    }
    seg = lo;
    f0 = cum[seg];
    ncta = cum[seg + 1] - f0;
    n_b = seq_len(p, seg / p.H_kv);
    if (FUSED) {
      if (lane == 0) {
        bcast[56] = seg;
        bcast[57] = f0;
        bcast[58] = ncta;
        bcast[59] = n_b;
      }
      __syncwarp();
      named_bar_arrive(2, THREADS);
    }
  }
  const int ci = cta - f0;
  const int b = seg / p.H_kv, h = seg % p.H_kv;
  const Part pt = partition(n_b, p.I_b, p.L_b);
  const int nA = blocks_a(pt, p.dense);
  // 32-bit products: ci < 2^10 CTAs, nA < 2^20 blocks
  const int a0 = ci * nA / ncta, a1 = (ci + 1) * nA / ncta;

  if (warp == CONSUMERS) {
    // =========================== producer warp ===============================
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t qbytes = (uint32_t)p.G * D * 2;
    if (p.q_mapped) {
      // q in host memory: 16-byte loads over the link, then one arrival
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)b * H_q + h * p.G) * D);
      uint4* dst = reinterpret_cast<uint4*>(smem + SmemLayout::q);
      for (int i = lane; i < (int)(qbytes / 16); i += 32) dst[i] = src[i];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_q);
    } else if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, qbytes);
      bulk_load(smem_u32(smem + SmemLayout::q), p.q + ((size_t)b * H_q + h * p.G) * D, qbytes,
                bar_q);
    }
    // fused: the unit's chosen block ids in ascending order, written by the
    // consumer warps (this CTA's share starts at fi0); the page of each of this
    // CTA's first 32 Initial/Local blocks, looked up now
    const int* fsorted = nullptr;
    const int* fpages = nullptr;
    int fi0 = 0, pgA = -1;
    if (FUSED) {
      const int nsl = p.ncpu * p.kk_f;
      const FusedPickLayout Lp = fused_pick_layout(nsl, min(p.top_k, nsl));
      fsorted = reinterpret_cast<const int*>(smem + SmemLayout::scratch + Lp.sorted);
      fpages = reinterpret_cast<const int*>(smem + SmemLayout::scratch + Lp.sorted_pages);
      const int i = a0 + lane;
      if (i < a1) pgA = p.table[(size_t)b * p.max_blocks + (i < pt.c0 ? i : pt.c1 + (i - pt.c0))];
    }
    uint32_t it = 0;
    bool ok = true;
    // not fused: the unit's first 32 chosen ids, loaded together with the count
    int sel32 = -1;
    // phase 0: list index i -> Initial/Local block; phase 1: i -> selected block
    auto produce = [&](int phase, int u0, int u1) {
      for (int base = u0; base < u1 && ok; base += 32) {
        const int i = base + lane;
        int ntok = 0, row = 0;
        const int sel_i = (!FUSED && phase == 1) ? __shfl_sync(0xffffffffu, sel32, i & 31) : -1;
        if (i < u1) {
          int j, page = -1;
          if (phase == 0) {
            j = (p.dense || i < pt.c0) ? i : pt.c1 + (i - pt.c0);
            page = (FUSED && base == u0) ? pgA : p.table[(size_t)b * p.max_blocks + j];
          } else if (FUSED) {
            j = fsorted[fi0 + i];  // a selected Context block (full), with its page
            page = fpages[fi0 + i];
            if (j < pt.c0 || j >= pt.c1) {
              set_status(p.status, KT_ERR_DEVICE_CHECK);
              j = -1;
            }
          } else if (p.sel_pages == nullptr) {
            const int unit = p.SEL == 1 ? 0 : h;
            j = i < 32 ? sel_i : p.sel[((size_t)b * p.SEL + unit) * p.top_k + i];
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
            if (okl) {
              info[st].ntok = ntok_k;
              info[st].end = 0;
              const uint32_t bar = bar_full + 8 * st;
              if (ntok_k > 0) {
                if (it == 0) KT_STAMP(p, 7);
                if (phase == 1 && k == 0 && base == 0) KT_STAMP(p, 8);  // none issued by the consumers
                if constexpr (KVM == KVM_F16) {
                  mbar_arrive_expect_tx(bar, KV_STAGE_BYTES);
                  const uint32_t dst = kv_base + st * KV_STAGE_BYTES;
                  tma_load_2d(dst, &p.kmap, 0, row_k, bar, policy);
                  tma_load_2d(dst + BOX_BYTES, &p.kmap, 64, row_k, bar, policy);
                  tma_load_2d(dst + 2 * BOX_BYTES, &p.vmap, 0, row_k, bar, policy);
                  tma_load_2d(dst + 3 * BOX_BYTES, &p.vmap, 64, row_k, bar, policy);
                } else if constexpr (KVM == KVM_Q8) {
                  mbar_arrive_expect_tx(bar, Q8_STAGE_BYTES);
                  const uint32_t dst = kv_base + Q8_RING_OFF + st * Q8_STAGE_BYTES;
                  tma_load_2d(dst, &p.kmap, 0, row_k, bar, policy);
                  tma_load_2d(dst + Q8_CODE_BYTES, &p.vmap, 0, row_k, bar, policy);
                  bulk_load(dst + 2 * Q8_CODE_BYTES, p.k_scale + (size_t)row_k * (D / 32),
                            Q8_SCALE_BYTES, bar);
                  bulk_load(dst + 2 * Q8_CODE_BYTES + Q8_SCALE_BYTES,
                            p.v_scale + (size_t)row_k * (D / 32), Q8_SCALE_BYTES, bar);
                }
              } else if constexpr (KVM != KVM_HOST) {
                mbar_arrive(bar);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
          if (!ok) break;
          if constexpr (KVM == KVM_HOST) {
            // every lane: its 128 of the block's 4096 16-byte pieces (K and V,
            // each two 64-channel boxes in the 128-byte swizzled layout of the
            // TMA stages), then an arrival that completes once they have landed
            const uint32_t st = it % STAGES;
            if (ntok_k > 0) {
              const uint32_t dst = kv_base + st * KV_STAGE_BYTES;
#pragma unroll 4
              for (int idx = lane; idx < 4 * UNIT * 8; idx += 32) {
                const int bx = idx >> 10, r = (idx >> 3) & (UNIT - 1), c = idx & 7;
                const __half* src = (bx < 2 ? p.k_src : p.v_src) + ((size_t)row_k + r) * D +
                                    (bx & 1) * 64 + c * 8;
                cp_async_16(dst + bx * BOX_BYTES + r * 128 + ((c ^ (r & 7)) << 4), src);
              }
              cp_async_mbar_arrive_noinc(bar_full + 8 * st);
            } else {
              mbar_arrive(bar_full + 8 * st);
            }
          }
          ++it;
        }
      }
    };
    if (FUSED) {
      // The Initial/Local loads start once the unit's candidate slots have
      // all been read: data arriving at this SM would queue the selection's
      // own loads (the representative rows, the slot polls) behind it.  They
      // land while the top-k is picked.  This CTA's share of the chosen
      // blocks follows once the selection is made.
      // plain try_wait spins: a sleep between polls can outlast the wait itself
      if (lane == 0) mbar_wait(bar_seen, 0, p.status);
      __syncwarp();
    }
    // both phases run the one copy of `produce` (a second inlined copy would
    // be fetched cold on the way to the first selected load)
    int u0 = a0, u1 = a1;
#pragma unroll 1
    for (int phase = 0; phase < 2 && ok; ++phase) {
      if (phase == 1) {
        if (FUSED) {
          // the consumers issued the first npre chosen blocks into stages
          // it .. it + npre - 1 themselves; the rest follow from here
          int n1 = 0, i0 = 0, npre = 0;
          if (lane == 0 && mbar_wait(bar_sel, 0, p.status)) {
            n1 = bcast[61];
            i0 = bcast[62];
            npre = bcast[63];
          }
          u0 = __shfl_sync(0xffffffffu, npre, 0);
          u1 = __shfl_sync(0xffffffffu, n1, 0);
          fi0 = __shfl_sync(0xffffffffu, i0, 0);
          it += (uint32_t)u0;
        } else {
          // Phase B needs the selection: wait for the grid this launch depends on.
          griddep_wait();
          int nB = 0;
          if (!p.dense) {
            const int cmax = blocks_b_max(pt, 0, p.top_k);
            if (p.sel_pages == nullptr && lane < min(cmax, 32))
              sel32 = p.sel[((size_t)b * p.SEL + (p.SEL == 1 ? 0 : h)) * p.top_k + lane];
            nB = p.cnt ? p.cnt[b * p.SEL + (p.SEL == 1 ? 0 : h)] : cmax;
            if (nB < 0 || nB > cmax) {
              set_status(p.status, KT_ERR_DEVICE_CHECK);
              nB = nB < 0 ? 0 : cmax;
            }
          }
          u0 = (int)((long long)ci * nB / ncta);
          u1 = (int)((long long)(ci + 1) * nB / ncta);
        }
      }
      produce(phase, u0, u1);
    }
    if (ok) {
      const uint32_t st = it % STAGES;
      int okl = 0;
      if (lane == 0 &&
          (it < STAGES || mbar_wait(bar_empty + 8 * st, ((it / STAGES) - 1) & 1, p.status))) {
        info[st].end = 1;
        info[st].ntok = 0;
        okl = 1;
      }
      okl = __shfl_sync(0xffffffffu, okl, 0);
      // the end marker: one arrival, or one per lane for the host source
      if (okl && (KVM == KVM_HOST || lane == 0)) mbar_arrive(bar_full + 8 * st);
    }
    return;
  }

  // ============================ consumer warps ===============================
  const int g = lane >> 2, t = lane & 3;
  const int ctid = tid;

  if constexpr (FUSED) {
    int i0 = 0;
    // as few slot registers a thread as the unit's slots need
    const int nsl = p.ncpu * p.kk_f;
    uint8_t* scr = reinterpret_cast<uint8_t*>(scratch);
    const int n1 =
        nsl <= 3 * NCT
            ? fused_pick<3>(p, scr, f_sh_u64, f_sh_int, b, h, pt, ci, ncta, ctid, bar_c, &i0,
                            bar_seen)
        : nsl <= 5 * NCT
            ? fused_pick<5>(p, scr, f_sh_u64, f_sh_int, b, h, pt, ci, ncta, ctid, bar_c, &i0,
                            bar_seen)
            : fused_pick<FUSED_GATHER_PER_THREAD>(p, scr, f_sh_u64, f_sh_int, b, h, pt, ci, ncta,
                                                  ctid, bar_c, &i0, bar_seen);
    // The first of this CTA's chosen blocks go straight into the ring stages
    // that are still unused (the producer's Initial/Local loads took stages
    // 0 .. nil-1 and waited on none): issued here, one thread a block, not
    // handed to the producer warp, whose shared-memory reads would queue
    // behind the consumers' fragment loads once the attention starts.
    const int nil = a1 - a0;
    const int npre = nil < STAGES ? min(n1, STAGES - nil) : 0;
    if (ctid < npre) {
      const int nsl = p.ncpu * p.kk_f;
      const FusedPickLayout Lp = fused_pick_layout(nsl, min(p.top_k, nsl));
      const uint8_t* scr = reinterpret_cast<const uint8_t*>(scratch);
      const int j = reinterpret_cast<const int*>(scr + Lp.sorted)[i0 + ctid];
      const int page = reinterpret_cast<const int*>(scr + Lp.sorted_pages)[i0 + ctid];
      int ntok = 0;
      if (j < pt.c0 || j >= pt.c1 || page < 0 || page >= p.P) {
        set_status(p.status, KT_ERR_DEVICE_CHECK);
      } else {
        ntok = min(UNIT, pt.n - j * BS);
      }
      const uint32_t st = (uint32_t)(nil + ctid);
      info[st].ntok = ntok;
      info[st].end = 0;
      const uint32_t bar = bar_full + 8 * st;
      if (ntok > 0) {
        if (ctid == 0) KT_STAMP(p, 8);
        const int row = (page * p.H_kv + h) * BS;
        const uint64_t policy = l2_evict_first_policy();
        if constexpr (KVM == KVM_Q8) {
          mbar_arrive_expect_tx(bar, Q8_STAGE_BYTES);
          const uint32_t dst = kv_base + Q8_RING_OFF + st * Q8_STAGE_BYTES;
          tma_load_2d(dst, &p.kmap, 0, row, bar, policy);
          tma_load_2d(dst + Q8_CODE_BYTES, &p.vmap, 0, row, bar, policy);
          bulk_load(dst + 2 * Q8_CODE_BYTES, p.k_scale + (size_t)row * (D / 32), Q8_SCALE_BYTES,
                    bar);
          bulk_load(dst + 2 * Q8_CODE_BYTES + Q8_SCALE_BYTES, p.v_scale + (size_t)row * (D / 32),
                    Q8_SCALE_BYTES, bar);
        } else {
          mbar_arrive_expect_tx(bar, KV_STAGE_BYTES);
          const uint32_t dst = kv_base + st * KV_STAGE_BYTES;
          tma_load_2d(dst, &p.kmap, 0, row, bar, policy);
          tma_load_2d(dst + BOX_BYTES, &p.kmap, 64, row, bar, policy);
          tma_load_2d(dst + 2 * BOX_BYTES, &p.vmap, 0, row, bar, policy);
          tma_load_2d(dst + 3 * BOX_BYTES, &p.vmap, 64, row, bar, policy);
        }
      } else {
        mbar_arrive(bar);
      }
    }
    if (ctid == 0) {
      bcast[61] = n1;
      bcast[62] = i0;
      bcast[63] = npre;
      mbar_arrive(bar_sel);
      KT_STAMP(p, 6);
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
      if constexpr (KVM == KVM_Q8) {
        // this warp's 16 token rows of K and V: int8 code * binary16 scale,
        // rounded once to fp16, into the fp16 block at the start of the ring
        // in the layout of an fp16 stage (lane: one row, half its channels)
        const uint8_t* qst = smem + SmemLayout::kv + Q8_RING_OFF + st * Q8_STAGE_BYTES;
        const int rr = lane >> 1, hh = lane & 1, tok = warp * 16 + rr, sw = tok & 7;
#pragma unroll
        for (int kvs = 0; kvs < 2; ++kvs) {
          const uint8_t* codes = qst + kvs * Q8_CODE_BYTES + tok * 128;
          const __half* scl = reinterpret_cast<const __half*>(qst + 2 * Q8_CODE_BYTES +
                                                              kvs * Q8_SCALE_BYTES) + tok * (D / 32);
          uint8_t* row16 = smem + SmemLayout::kv + (2 * kvs + hh) * BOX_BYTES + tok * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c16 = 4 * hh + i;  // 16-channel piece of the int8 row
            const uint4 v = *reinterpret_cast<const uint4*>(codes + ((c16 ^ sw) << 4));
            const __half2 d2 = __half2half2(scl[c16 >> 1]);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint32_t h2[8];
            // code c as binary16: the byte c + 128 in the low mantissa of 1024
            // gives 1152 + c exactly; subtracting 1152 leaves c, and one
            // correctly rounded binary16 product gives round(c * scale)
            const __half2 bias = __float2half2_rn(1152.0f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t u = wv[j] ^ 0x80808080u;
              const uint32_t lo = __byte_perm(u, 0x64646464u, 0x5140);
              const uint32_t hi = __byte_perm(u, 0x64646464u, 0x7362);
              const __half2 lo2 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&lo), bias), d2);
              const __half2 hi2 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&hi), bias), d2);
              h2[2 * j] = *reinterpret_cast<const uint32_t*>(&lo2);
              h2[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi2);
            }
            *reinterpret_cast<uint4*>(row16 + (((2 * i) ^ sw) << 4)) =
                make_uint4(h2[0], h2[1], h2[2], h2[3]);
            *reinterpret_cast<uint4*>(row16 + (((2 * i + 1) ^ sw) << 4)) =
                make_uint4(h2[4], h2[5], h2[6], h2[7]);
          }
        }
        __syncwarp();
      }
      const uint32_t kb = KVM == KVM_Q8 ? kv_base : kv_base + st * KV_STAGE_BYTES;
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
  if (ctid == 0) KT_STAMP(p, 9);

  // ---- combine the eight warp states in one barrier round: each warp stores
  // (m, l, O[128]) per query head; then each thread combines two channels of a
  // head over the eight states.  The scratch and block-prefix areas hold them
  // for G <= 4; for larger G the (now idle) KV ring does, once every warp is
  // past its last block.
  constexpr int WST = D + 2;
  float* wst = scratch;
  if (p.G * CONSUMERS * WST * 4 > ATTN_MERGE_BYTES) {
    wst = reinterpret_cast<float*>(smem + SmemLayout::kv);
    named_bar_sync(1, NCT);
  }
  {
    float l_row = l_part;
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
    if (g < p.G) {
      float* sw = wst + (warp * p.G + g) * WST;
      if (t == 0) {
        sw[0] = m_run;
        sw[1] = l_row;
      }
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2*>(sw + 2 + nt * 8 + 2 * t) =
            make_float2(acc[nt][0] + acc[nt][2], acc[nt][1] + acc[nt][3]);
    }
  }
  named_bar_sync(1, NCT);
  const int slot_stride = p.slot_floats;
  float* dst = p.parts + (size_t)cta * slot_stride;  // partial: O[G][128], m[G], l[G] (base 2)
  // fused: tagged partial words (value bits | launch tag << 32), two per float
  // slot pair, so readers validate the data itself
  unsigned long long* dstw = reinterpret_cast<unsigned long long*>(p.parts) + (size_t)cta * slot_stride;
  const uint32_t ptag = FUSED ? (uint32_t)f_sh_int[15] : 0u;
#pragma unroll 1
  for (int idx = 2 * ctid; idx < p.G * D; idx += 2 * NCT) {
    const int gg = idx / D, c = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < CONSUMERS; ++w) M = fmaxf(M, wst[(w * p.G + gg) * WST]);
    float L = 0.0f, o0 = 0.0f, o1 = 0.0f;
#pragma unroll
    for (int w = 0; w < CONSUMERS; ++w) {
      const float* sw = wst + (w * p.G + gg) * WST;
      const float wt = (M == -INFINITY) ? 0.0f : exp2f(sw[0] - M);
      const float2 ov = *reinterpret_cast<const float2*>(sw + 2 + c);
      L = fmaf(sw[1], wt, L);
      o0 = fmaf(ov.x, wt, o0);
      o1 = fmaf(ov.y, wt, o1);
    }
    if (ncta == 1) {
      // the only CTA of its segment: normalise and write the output
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      *reinterpret_cast<float2*>(p.out + ((size_t)b * H_q + h * p.G + gg) * D + c) =
          make_float2(o0 * inv, o1 * inv);
    } else if (FUSED) {
      const unsigned long long hi = static_cast<unsigned long long>(ptag) << 32;
      st_relaxed_gpu_u64(dstw + gg * D + c, hi | __float_as_uint(o0));
      st_relaxed_gpu_u64(dstw + gg * D + c + 1, hi | __float_as_uint(o1));
      if (c == 0) {
        st_relaxed_gpu_u64(dstw + p.G * D + gg, hi | __float_as_uint(M));
        st_relaxed_gpu_u64(dstw + p.G * D + p.G + gg, hi | __float_as_uint(L));
      }
    } else {
      *reinterpret_cast<float2*>(dst + gg * D + c) = make_float2(o0, o1);
      if (c == 0) {
        dst[p.G * D + gg] = M;
        dst[p.G * D + p.G + gg] = L;
      }
    }
  }
  if (ncta == 1) {
    if (ctid == 0) KT_STAMP(p, 10);
    return;
  }
  if constexpr (FUSED) {
    // the tagged partial words are pushed out to L2 now (see the slots)
  }
  if constexpr (FUSED) {
    // every CTA is resident: each CTA of the segment merges its share of the
    // G x 128 output channels from every CTA's partial, reading the tagged
    // words until all carry this launch's tag (no fence, no ticket)
    if (ctid == 0) KT_STAMP(p, 10);
    if (ctid == 0) griddep_launch_dependents();  // the next launch may be scheduled
    // shares are whole groups of 4 channels (a group never straddles a head)
    const int GD = p.G * D, G4 = GD / 4;
    const int q0 = 4 * (ci * G4 / ncta), q1 = 4 * ((ci + 1) * G4 / ncta);
    const unsigned long long* base = reinterpret_cast<const unsigned long long*>(p.parts) +
                                     (size_t)f0 * slot_stride;
    const unsigned long long tagw = static_cast<unsigned long long>(ptag) << 32;
    const int lane = ctid & 31, wp = ctid >> 5;
    const uint64_t t0 = globaltimer();
    // rounds over the share: warp wp takes the 4 channels cb .. cb+3; its lane
    // k holds partial k0 + k (m, l and the 4 O words, one round of loads), and
    // butterflies over the lanes merge the partials in a fixed order
    const int rounds = (q1 - q0 + 4 * CONSUMERS - 1) / (4 * CONSUMERS);
#pragma unroll 1
    for (int rr = 0; rr < rounds; ++rr) {
      const int cb = q0 + 4 * (rr * CONSUMERS + wp);
      const bool has_ch = cb < q1;
      const int gg = has_ch ? cb / D : 0;
      float Mw = -INFINITY, Lw = 0.0f, Ow[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      bool ok = false;
#pragma unroll 1
      for (;;) {
        ok = true;
        Mw = -INFINITY;
        Lw = 0.0f;
        Ow[0] = Ow[1] = Ow[2] = Ow[3] = 0.0f;
#pragma unroll 1
        for (int k0 = 0; k0 < ncta; k0 += 32) {
          const bool has = has_ch && k0 + lane < ncta;
          const unsigned long long* src = base + (size_t)(k0 + lane) * slot_stride;
          const unsigned long long wm = has ? ld_relaxed_gpu_u64(src + GD + gg)
                                            : (tagw | __float_as_uint(-INFINITY));
          const unsigned long long wl = has ? ld_relaxed_gpu_u64(src + GD + p.G + gg) : tagw;
          unsigned long long wo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) wo[i] = has ? ld_relaxed_gpu_u64(src + cb + i) : tagw;
          const bool lane_ok = (wm >> 32) == ptag && (wl >> 32) == ptag &&
                               (wo[0] >> 32) == ptag && (wo[1] >> 32) == ptag &&
                               (wo[2] >> 32) == ptag && (wo[3] >> 32) == ptag;
          ok = ok && lane_ok;
          if (!__all_sync(0xffffffffu, lane_ok)) continue;  // not all in yet: poll again
          const float mk = __uint_as_float((uint32_t)wm);
          float M = mk;
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));
          const float Mn = fmaxf(Mw, M);
          if (Mn == -INFINITY) continue;  // warp-uniform
          const float w = exp2f(mk - Mn);  // 0 for lanes without a partial
          const float a0 = exp2f(Mw - Mn);  // 0 when Mw is -inf
          float v[5] = {__uint_as_float((uint32_t)wl) * w, __uint_as_float((uint32_t)wo[0]) * w,
                        __uint_as_float((uint32_t)wo[1]) * w, __uint_as_float((uint32_t)wo[2]) * w,
                        __uint_as_float((uint32_t)wo[3]) * w};
#pragma unroll
          for (int d = 16; d > 0; d >>= 1)
#pragma unroll
            for (int i = 0; i < 5; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], d);
          Lw = fmaf(Lw, a0, v[0]);
#pragma unroll
          for (int i = 0; i < 4; ++i) Ow[i] = fmaf(Ow[i], a0, v[1 + i]);
          Mw = Mn;
        }
        if (named_bar_and(1, NCT, ok || globaltimer() - t0 > p.poll_limit_ns)) break;
      }
      if (!ok) set_status(p.status, KT_ERR_TIMEOUT);
      if (ctid == 0) KT_STAMP(p, 11);
      const float inv = Lw > 0.0f ? 1.0f / Lw : 0.0f;
      if (has_ch && lane < 4) {
        const float ov = lane == 0 ? Ow[0] : lane == 1 ? Ow[1] : lane == 2 ? Ow[2] : Ow[3];
        p.out[((size_t)b * H_q + h * p.G) * D + cb + lane] = ov * inv;
      }
    }
    if (ctid == 0) KT_STAMP(p, 12);
    return;
  } else {
    named_bar_sync(1, NCT);
    if (ctid == 0) {
      griddep_launch_dependents();  // the next launch may be scheduled
      const int old = atom_acq_rel_gpu_add(p.counters + seg, 1);
      bcast[60] = (old + 1 == ncta) ? 1 : 0;
    }
    named_bar_sync(1, NCT);
    if (!bcast[60]) return;
  }

  // ---- the merging CTA: partials of CTAs f0 .. f0+ncta-1 in CTA order; each
  // thread owns two channels of one head and takes 16 partials per round of
  // independent loads, merged online
  if constexpr (!FUSED) {
#pragma unroll 1
  for (int idx = 2 * ctid; idx < p.G * D; idx += 2 * NCT) {
    const int gg = idx / D, c = idx % D;
    float M = -INFINITY, L = 0.0f, o0 = 0.0f, o1 = 0.0f;
#pragma unroll 1
    for (int base = 0; base < ncta; base += 16) {
      const int nb = min(16, ncta - base);
      float m[16], l[16];
      float2 ov[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k < nb) {
          const float* src = p.parts + (size_t)(f0 + base + k) * slot_stride;
          m[k] = __ldcg(src + p.G * D + gg);
          l[k] = __ldcg(src + p.G * D + p.G + gg);
          ov[k] = __ldcg(reinterpret_cast<const float2*>(src + gg * D + c));
        } else {
          m[k] = -INFINITY;
          l[k] = 0.0f;
          ov[k] = make_float2(0.f, 0.f);
        }
      }
      float Mn = M;
#pragma unroll
      for (int k = 0; k < 16; ++k) Mn = fmaxf(Mn, m[k]);
      if (Mn == -INFINITY) continue;
      const float a0 = exp2f(M - Mn);  // 0 when M is -inf
      L *= a0;
      o0 *= a0;
      o1 *= a0;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float w = exp2f(m[k] - Mn);  // 0 for empty partials
        L = fmaf(l[k], w, L);
        o0 = fmaf(ov[k].x, w, o0);
        o1 = fmaf(ov[k].y, w, o1);
      }
      M = Mn;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    *reinterpret_cast<float2*>(p.out + ((size_t)b * H_q + h * p.G + gg) * D + c) =
        make_float2(o0 * inv, o1 * inv);
  }
  if (ctid == 0) {
    p.counters[seg] = 0;
    KT_STAMP(p, 12);
  }
  }
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
                          (const void*)attn_kernel<SK_F32>, (const void*)attn_kernel<SK_MULTI>,
                          (const void*)attn_kernel<SK_NONE, KVM_HOST>,
                          (const void*)attn_kernel<SK_NONE, KVM_Q8>,
                          (const void*)attn_kernel<SK_COLS, KVM_Q8>,
                          (const void*)attn_kernel<SK_LINEAR, KVM_Q8>,
                          (const void*)attn_kernel<SK_MMA, KVM_Q8>,
                          (const void*)attn_kernel<SK_F32, KVM_Q8>,
                          (const void*)attn_kernel<SK_MULTI, KVM_Q8>})
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
                          (const void*)attn_kernel<SK_MULTI>,
                          (const void*)attn_kernel<SK_COLS, KVM_Q8>,
                          (const void*)attn_kernel<SK_LINEAR, KVM_Q8>,
                          (const void*)attn_kernel<SK_MMA, KVM_Q8>,
                          (const void*)attn_kernel<SK_F32, KVM_Q8>,
                          (const void*)attn_kernel<SK_MULTI, KVM_Q8>}) {
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
  p.f_cand_len = a.f_cand_len;
  p.f_cpage = a.f_cpage;
  p.f_sync = a.f_sync;
  p.sel_out = a.sel_out;
  p.cnt_out = a.cnt_out;
  p.presel_mask = a.presel_mask;
  p.presel_cnt = a.presel_cnt;
  p.mask_words = a.mask_words;
  p.stamps = a.stamps;
  p.k_src = static_cast<const __half*>(a.k_src);
  p.v_src = static_cast<const __half*>(a.v_src);
  p.k_scale = static_cast<const __half*>(a.k_scale);
  p.v_scale = static_cast<const __half*>(a.v_scale);
  p.skip_publish = a.skip_publish;
  p.poll_limit_ns = a.poll_limit_ns ? a.poll_limit_ns : WAIT_LIMIT_NS;
  p.wait_at_entry = (a.fused || !a.pdl) ? 1 : 0;
  p.q_mapped = a.q_mapped ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  // every launch may start while the previous kernel on the stream finishes
  // (the kernel waits for it, at entry or before its selected blocks)
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (a.fused) {
    // every CTA must be resident: CTAs wait for candidate slots and partials
    // written by other CTAs of the same grid
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  if (!a.fused) {
    if (a.kvm == KVM_HOST) return cudaLaunchKernelEx(&cfg, attn_kernel<SK_NONE, KVM_HOST>, p);
    if (a.kvm == KVM_Q8) return cudaLaunchKernelEx(&cfg, attn_kernel<SK_NONE, KVM_Q8>, p);
    return cudaLaunchKernelEx(&cfg, attn_kernel<SK_NONE>, p);
  }
  if (a.kvm == KVM_Q8) {
    switch (a.sk) {
      case SK_COLS: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_COLS, KVM_Q8>, p);
      case SK_LINEAR: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_LINEAR, KVM_Q8>, p);
      case SK_MMA: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_MMA, KVM_Q8>, p);
      case SK_F32: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_F32, KVM_Q8>, p);
      case SK_MULTI: return cudaLaunchKernelEx(&cfg, attn_kernel<SK_MULTI, KVM_Q8>, p);
    }
    return cudaErrorInvalidValue;
  }
  if (a.kvm != KVM_F16) return cudaErrorInvalidValue;
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
