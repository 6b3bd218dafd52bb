// attn.cu — split-K decode attention over a block list (sparse or dense).
//
// Computes, for every query head h of every sequence b,
//   out[b][h] = softmax(q_h . K_S^T * scale) V_S
// over the token set S = Initial blocks + selected Context blocks + Local blocks
// (sparse; article "KTransformers 长上下文稀疏注意力实战…", §4.2 and §4.6
// attn(query, kvcache_after_retrieval)) or over every block (dense, the full
// scan of §1).
//
// Work decomposition (one launch, persistent grid of `grid` CTAs):
//   - A work unit is 64 tokens (half a block) of one (sequence, KV head)
//     "segment": 16 KB of K + 16 KB of V.  Phase A holds the Initial and Local
//     units (known from seq_lens alone), phase B the selected Context units
//     (known once the selection has finished).  Each phase's units, ordered by
//     segment, are cut into `grid` equal contiguous ranges, one per CTA.
//   - A producer warp turns its units into block-table lookups and 2-D TMA
//     loads (four 8 KB boxes, 128-byte swizzle) into a 5-stage shared-memory
//     ring, plus a bulk copy of the segment's G query rows.  Phase-B work waits
//     on griddepcontrol.wait, so when this kernel is a programmatic dependent
//     of the selection kernel, Initial/Local streaming overlaps selection.
//   - Four consumer warps each take 16 tokens of a unit: S = q K^T and
//     O += P V on mma.sync m16n8k16 (fp16 in, fp32 accumulate).  Query heads
//     are rows 0..G-1 of the A operand; in P V the fp16 split P = P_hi + P_lo
//     puts P_hi in rows 0..7 and P_lo in rows 8..15 of the same fragment, so P
//     keeps ~22 bits.  Online softmax (base 2) per warp, merged at segment end.
//   - Each CTA writes one (m, l, acc) partial per segment it touched; the CTA
//     that takes a segment's last ticket merges the partials in CTA order
//     (deterministic) and writes out[b][h].
#include "kt_internal.cuh"

namespace kt {
namespace {

constexpr int STAGES = 5;
constexpr int CONSUMERS = 4;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int UNIT = 64;
constexpr int BOX_BYTES = UNIT * 64 * 2;       // 64 tokens x 64 channels fp16
constexpr int KV_STAGE_BYTES = 4 * BOX_BYTES;  // K lo, K hi, V lo, V hi
constexpr int Q_STAGE_BYTES = MAX_G * D * 2;
constexpr int SCRATCH_FLOATS = CONSUMERS * MAX_G * (D + 2);

struct StageInfo {
  int seg, ntok, phase, end;
};

struct SmemLayout {
  static constexpr int kv = 0;
  static constexpr int q = kv + STAGES * KV_STAGE_BYTES;
  static constexpr int scratch = q + STAGES * Q_STAGE_BYTES;
  static constexpr int prefA = scratch + SCRATCH_FLOATS * 4;
  static constexpr int prefB = prefA + (MAX_SEGS + 1) * 4;
  static constexpr int sl = prefB + (MAX_SEGS + 1) * 4;
  static constexpr int info = sl + MAX_SEGS * 4;
  static constexpr int bars = (info + STAGES * (int)sizeof(StageInfo) + 15) & ~15;
  static constexpr int bcast = bars + 2 * STAGES * 8;
  static constexpr int total = bcast + 64;
};
constexpr int SMEM_BYTES = SmemLayout::total + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "attention shared memory exceeds the per-CTA limit");

struct Params {
  CUtensorMap kmap, vmap;
  const __half* q;
  const int32_t* table;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* cnt;
  float* out;
  int* status;
  int* counters;
  float* parts;
  int B, H_kv, G, max_blocks, P, I_b, L_b, top_k, SEL, dense, slot_floats;
  float scale_log2;
};

struct Part {
  int nb, c0, c1;
};

__device__ __forceinline__ Part partition(int n, int I, int L) {
  Part p;
  p.nb = (n + BS - 1) / BS;
  p.c0 = min(I, p.nb);
  p.c1 = max(p.c0, p.nb - L);
  return p;
}

__device__ __forceinline__ int units_a(int n, int I, int L, int dense) {
  if (n <= 0) return 0;
  const Part p = partition(n, I, L);
  const int blocks = dense ? p.nb : p.c0 + (p.nb - p.c1);
  const int tail = n - (p.nb - 1) * BS;
  return 2 * blocks - (tail <= UNIT ? 1 : 0);
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

// Largest s in [0, S) with pref[s] <= u.
__device__ __forceinline__ int find_seg(const int* pref, int S, int u) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ long long range_start(int c, long long U, int NC) {
  return (long long)c * U / NC;
}

// CTA whose range holds unit u (0 <= u < U) when U units are split into NC
// ranges [floor(c U / NC), floor((c+1) U / NC)).
__device__ __forceinline__ int cta_of_unit(long long u, long long U, int NC) {
  return (int)(((u + 1) * NC + U - 1) / U - 1);
}

// Calls f(c) for every CTA c (ascending) whose non-empty range of a phase with
// U units overlaps units [x, y).  With U >= NC every range is non-empty, so the
// overlapping CTAs are the interval [cta(x), cta(y-1)]; with U < NC every
// non-empty range holds exactly one unit.
template <class F>
__device__ __forceinline__ void for_overlapping_ctas(long long x, long long y, long long U, int NC,
                                                     F f) {
  if (y <= x || U <= 0) return;
  if (U >= NC) {
    const int chi = cta_of_unit(y - 1, U, NC);
    for (int c = cta_of_unit(x, U, NC); c <= chi; ++c) f(c);
  } else {
    for (long long u = x; u < y; ++u) f(cta_of_unit(u, U, NC));
  }
}

__device__ __forceinline__ int count_overlapping_ctas(long long x, long long y, long long U,
                                                      int NC) {
  if (y <= x || U <= 0) return 0;
  if (U < NC) return (int)(y - x);
  return cta_of_unit(y - 1, U, NC) - cta_of_unit(x, U, NC) + 1;
}

__global__ void __launch_bounds__(THREADS, 1) attn_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = gridDim.x, cta = blockIdx.x;
  const int S = p.B * p.H_kv;
  int* prefA = reinterpret_cast<int*>(smem + SmemLayout::prefA);
  int* prefB = reinterpret_cast<int*>(smem + SmemLayout::prefB);
  int* sl = reinterpret_cast<int*>(smem + SmemLayout::sl);
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + SmemLayout::info);
  int* bcast = reinterpret_cast<int*>(smem + SmemLayout::bcast);
  float* scratch = reinterpret_cast<float*>(smem + SmemLayout::scratch);
  const uint32_t bar_full = smem_u32(smem + SmemLayout::bars);
  const uint32_t bar_empty = bar_full + STAGES * 8;
  const uint32_t kv_base = smem_u32(smem + SmemLayout::kv);
  const uint32_t q_base = smem_u32(smem + SmemLayout::q);

  // ---- set-up: sequence lengths, phase-A prefix, barriers -------------------
  for (int b = tid; b < p.B; b += THREADS) {
    int n = p.seq_lens[b];
    if (n < 0 || n > p.max_blocks * BS) {
      set_status(p.status, KT_ERR_DEVICE_CHECK);
      n = n < 0 ? 0 : p.max_blocks * BS;
    }
    sl[b] = n;
  }
  __syncthreads();
  if (warp == CONSUMERS)
    warp_prefix(prefA, S, [&](int s) { return units_a(sl[s / p.H_kv], p.I_b, p.L_b, p.dense); },
                lane);
  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, CONSUMERS);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int H_q = p.H_kv * p.G;
  // Segments of empty sequences produce no partial: write their zeros here.
  for (int s = cta; s < S; s += NC)
    if (sl[s / p.H_kv] == 0 && tid < CONSUMERS * 32)
      for (int g = 0; g < p.G; ++g)
        p.out[((size_t)(s / p.H_kv) * H_q + (s % p.H_kv) * p.G + g) * D + tid] = 0.0f;

  const long long UA = prefA[S];
  const long long a0 = range_start(cta, UA, NC), a1 = range_start(cta + 1, UA, NC);

  if (warp == CONSUMERS) {
    // =========================== producer warp ===============================
    const uint64_t policy = l2_evict_first_policy();
    uint32_t it = 0;
    bool ok = true;
    auto produce = [&](int phase, long long u0, long long u1, const int* pref) {
      for (long long base = u0; base < u1 && ok; base += 32) {
        const long long u = base + lane;
        int seg = 0, ntok = 0, row = 0;
        if (u < u1) {
          seg = find_seg(pref, S, (int)u);
          const int i = (int)(u - pref[seg]);
          const int b = seg / p.H_kv, h = seg % p.H_kv, n = sl[b];
          const Part pt = partition(n, p.I_b, p.L_b);
          int j, half;
          if (phase == 0) {
            if (p.dense || i < 2 * pt.c0) {
              j = i >> 1;
              half = i & 1;
            } else {
              const int i2 = i - 2 * pt.c0;
              j = pt.c1 + (i2 >> 1);
              half = i2 & 1;
            }
          } else {
            const int unit = p.SEL == 1 ? 0 : h;
            j = p.sel[((size_t)b * p.SEL + unit) * p.top_k + (i >> 1)];
            half = i & 1;
            if (j < pt.c0 || j >= pt.c1) {
              set_status(p.status, KT_ERR_DEVICE_CHECK);
              j = -1;
            }
          }
          if (j >= 0) {
            ntok = min(UNIT, n - j * BS - half * UNIT);
            const int page = p.table[(size_t)b * p.max_blocks + j];
            if (page < 0 || page >= p.P) {
              set_status(p.status, KT_ERR_DEVICE_CHECK);
              ntok = 0;
            } else {
              row = (page * p.H_kv + h) * BS + half * UNIT;
            }
          }
        }
        const int cnt_batch = (int)min(32LL, u1 - base);
        for (int k = 0; k < cnt_batch; ++k) {
          const int seg_k = __shfl_sync(0xffffffffu, seg, k);
          const int ntok_k = __shfl_sync(0xffffffffu, ntok, k);
          const int row_k = __shfl_sync(0xffffffffu, row, k);
          const uint32_t st = it % STAGES;
          int okl = 1;
          if (lane == 0) {
            if (it >= STAGES && !mbar_wait(bar_empty + 8 * st, ((it / STAGES) - 1) & 1, p.status))
              okl = 0;
            if (okl) {
              info[st].seg = seg_k;
              info[st].ntok = ntok_k;
              info[st].phase = phase;
              info[st].end = 0;
              const uint32_t bar = bar_full + 8 * st;
              if (ntok_k > 0) {
                const int b = seg_k / p.H_kv, h = seg_k % p.H_kv;
                const uint32_t qbytes = (uint32_t)p.G * D * 2;
                mbar_arrive_expect_tx(bar, KV_STAGE_BYTES + qbytes);
                const uint32_t dst = kv_base + st * KV_STAGE_BYTES;
                tma_load_2d(dst, &p.kmap, 0, row_k, bar, policy);
                tma_load_2d(dst + BOX_BYTES, &p.kmap, 64, row_k, bar, policy);
                tma_load_2d(dst + 2 * BOX_BYTES, &p.vmap, 0, row_k, bar, policy);
                tma_load_2d(dst + 3 * BOX_BYTES, &p.vmap, 64, row_k, bar, policy);
                bulk_load(q_base + st * Q_STAGE_BYTES, p.q + ((size_t)b * H_q + h * p.G) * D,
                          qbytes, bar);
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
    produce(0, a0, a1, prefA);
    // Phase B needs the selection: wait for the grid this launch depends on.
    griddep_wait();
    if (p.dense) {
      for (int s = lane; s <= S; s += 32) prefB[s] = 0;
      __syncwarp();
    } else {
      warp_prefix(prefB, S, [&](int s) {
        const int b = s / p.H_kv, h = s % p.H_kv;
        const Part pt = partition(sl[b], p.I_b, p.L_b);
        const int cmax = min(p.top_k, pt.c1 - pt.c0);
        int c = p.cnt[b * p.SEL + (p.SEL == 1 ? 0 : h)];
        if (c < 0 || c > cmax) {
          set_status(p.status, KT_ERR_DEVICE_CHECK);
          c = c < 0 ? 0 : cmax;
        }
        return 2 * c;
      }, lane);
    }
    const long long UB = prefB[S];
    if (ok) produce(1, range_start(cta, UB, NC), range_start(cta + 1, UB, NC), prefB);
    if (ok && lane == 0) {
      const uint32_t st = it % STAGES;
      if (it < STAGES || mbar_wait(bar_empty + 8 * st, ((it / STAGES) - 1) & 1, p.status)) {
        info[st].end = 1;
        info[st].seg = -1;
        info[st].phase = 1;
        info[st].ntok = 0;
        mbar_arrive(bar_full + 8 * st);
      }
    }
    return;
  }

  // ============================ consumer warps ===============================
  const int g = lane >> 2, t = lane & 3;
  const int ctid = tid;  // 0..127
  float acc[16][4];
  float m_run = -INFINITY, l_part = 0.0f;
  uint32_t qa[8][2];
  int cur_seg = -1, cur_phase = 0;
  bool a_tickets_done = false;
  bool q_loaded = false;
  const int slot_stride = p.slot_floats;
  const long long half_slots = (long long)NC + S;

  auto reset_state = [&]() {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    m_run = -INFINITY;
    l_part = 0.0f;
  };

  // Merge the four warps' states and write this CTA's partial for `seg`.
  auto flush = [&](int seg, int phase) {
    float l_row = l_part;
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
    if (g < p.G) {
      float* sc = scratch + (warp * MAX_G + g) * (D + 2);
      if (t == 0) {
        sc[0] = m_run;
        sc[1] = l_row;
      }
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        sc[2 + nt * 8 + 2 * t] = acc[nt][0] + acc[nt][2];
        sc[2 + nt * 8 + 2 * t + 1] = acc[nt][1] + acc[nt][3];
      }
    }
    named_bar_sync(1, CONSUMERS * 32);
    const long long slot = (phase == 0 ? 0 : half_slots) + cta + seg;
    float* dst = p.parts + slot * slot_stride;
    const int c = ctid;
    for (int gg = 0; gg < p.G; ++gg) {
      float M = -INFINITY;
      for (int w = 0; w < CONSUMERS; ++w) M = fmaxf(M, scratch[(w * MAX_G + gg) * (D + 2)]);
      float o = 0.0f, l = 0.0f;
      if (M != -INFINITY) {
        for (int w = 0; w < CONSUMERS; ++w) {
          const float* sc = scratch + (w * MAX_G + gg) * (D + 2);
          const float f = exp2f(sc[0] - M);
          o += sc[2 + c] * f;
          l += sc[1] * f;
        }
      }
      dst[gg * D + c] = o;  // slot: O[G][128], then m[G], then l[G]
      if (c == 0) {
        dst[p.G * D + gg] = M;
        dst[p.G * D + p.G + gg] = l;
      }
    }
    __threadfence();
    named_bar_sync(1, CONSUMERS * 32);
  };

  auto expected_parts = [&](int seg, long long UB) {
    return count_overlapping_ctas(prefA[seg], prefA[seg + 1], UA, NC) +
           count_overlapping_ctas(prefB[seg], prefB[seg + 1], UB, NC);
  };

  // Final merge of all partials of `seg` (CTA order, phase A then B).  Thread
  // 0 lists the partial slots (arithmetic only), then every consumer thread
  // owns float4 chunks of the G x 128 outputs and streams the partials with
  // independent loads (online max-rescaling, base 2).
  auto merge = [&](int seg, long long UB) {
    __threadfence();
    int* slots = reinterpret_cast<int*>(scratch);  // up to 2 * MAX_ATTN_CTAS entries
    if (ctid == 0) {
      int np = 0;
      for_overlapping_ctas(prefA[seg], prefA[seg + 1], UA, NC,
                           [&](int cc) { slots[np++] = cc + seg; });
      for_overlapping_ctas(prefB[seg], prefB[seg + 1], UB, NC,
                           [&](int cc) { slots[np++] = (int)half_slots + cc + seg; });
      bcast[1] = np;
    }
    named_bar_sync(1, CONSUMERS * 32);
    const int np = bcast[1];
    const int b = seg / p.H_kv, h = seg % p.H_kv;
    for (int f = 4 * ctid; f < p.G * D; f += 4 * CONSUMERS * 32) {
      const int gg = f / D, c = f % D;
      float M = -INFINITY, L = 0.0f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int i = 0; i < np; ++i) {
        const float* src = p.parts + (size_t)slots[i] * slot_stride;
        const float m = __ldcg(src + p.G * D + gg);
        const float l = __ldcg(src + p.G * D + p.G + gg);
        const float4 o = __ldcg(reinterpret_cast<const float4*>(src + f));
        if (m == -INFINITY) continue;
        const float Mn = fmaxf(M, m);
        const float a = exp2f(M - Mn), w = exp2f(m - Mn);
        L = L * a + l * w;
        O.x = O.x * a + o.x * w;
        O.y = O.y * a + o.y * w;
        O.z = O.z * a + o.z * w;
        O.w = O.w * a + o.w * w;
        M = Mn;
      }
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      float4* dst = reinterpret_cast<float4*>(p.out + ((size_t)b * H_q + h * p.G + gg) * D + c);
      *dst = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
    }
    if (ctid == 0) p.counters[seg] = 0;
    named_bar_sync(1, CONSUMERS * 32);
  };

  // Ticket for `seg`; the CTA that completes the count merges.
  auto ticket = [&](int seg, long long UB) {
    if (ctid == 0) {
      const int expect = expected_parts(seg, UB);
      const int old = atomicAdd(p.counters + seg, 1);
      bcast[0] = (old + 1 == expect) ? 1 : 0;
    }
    named_bar_sync(1, CONSUMERS * 32);
    const bool last = bcast[0] != 0;
    named_bar_sync(1, CONSUMERS * 32);
    if (last) merge(seg, UB);
  };

  reset_state();
  for (uint32_t it = 0;; ++it) {
    const uint32_t st = it % STAGES;
    if (!mbar_wait(bar_full + 8 * st, (it / STAGES) & 1, p.status)) break;
    const StageInfo in = info[st];
    if (in.end || in.seg != cur_seg || in.phase != cur_phase) {
      const long long UB = prefB[S];  // valid once phase B or the end marker is visible
      if (cur_seg >= 0) {
        flush(cur_seg, cur_phase);
        if (cur_phase == 1) ticket(cur_seg, UB);
      }
      if (!a_tickets_done && (in.end || in.phase == 1)) {
        a_tickets_done = true;
        if (a1 > a0) {
          const int s_first = find_seg(prefA, S, (int)a0);
          const int s_last = find_seg(prefA, S, (int)(a1 - 1));
          for (int s = s_first; s <= s_last; ++s) ticket(s, UB);
        }
      }
      if (in.end) break;
      cur_seg = in.seg;
      cur_phase = in.phase;
      reset_state();
      q_loaded = false;
    }
    if (in.ntok > 0 && !q_loaded) {
      // query rows of this segment -> A fragments (rows >= G are zero); the
      // stage's bulk copy of q completed with its K/V boxes.
      const __half* qs =
          reinterpret_cast<const __half*>(smem + SmemLayout::q + st * Q_STAGE_BYTES);
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
    if (in.ntok > 0) {
      const uint32_t kb = kv_base + st * KV_STAGE_BYTES;
      const uint32_t vb = kb + 2 * BOX_BYTES;
      const int mi = lane >> 3, r = lane & 7;
      // ---- S = q K^T for this warp's 16 tokens
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int tok = warp * 16 + (mi >> 1) * 8 + r;
        const int chunk = kk * 2 + (mi & 1);
        const uint32_t addr = kb + (chunk >> 3) * BOX_BYTES + tok * 128 +
                              (((chunk & 7) ^ (tok & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, addr);
        mma_16816(s[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
        mma_16816(s[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
      }
      // ---- online softmax (base 2), rows = query heads
      float x[4];
      const int tok0 = warp * 16 + 2 * t;
      x[0] = (tok0 < in.ntok) ? s[0][0] * p.scale_log2 : -INFINITY;
      x[1] = (tok0 + 1 < in.ntok) ? s[0][1] * p.scale_log2 : -INFINITY;
      x[2] = (tok0 + 8 < in.ntok) ? s[1][0] * p.scale_log2 : -INFINITY;
      x[3] = (tok0 + 9 < in.ntok) ? s[1][1] * p.scale_log2 : -INFINITY;
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
}

}  // namespace

cudaError_t launch_attention(const AttnLaunch& a, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  Params p;
  p.kmap = *a.kmap;
  p.vmap = *a.vmap;
  p.q = a.q;
  p.table = a.table;
  p.seq_lens = a.seq_lens;
  p.sel = a.sel;
  p.cnt = a.cnt;
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

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_kernel, p);
}

}  // namespace kt
