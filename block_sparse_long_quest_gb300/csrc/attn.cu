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
//   - Eight consumer warps each take 8 tokens of a unit (two warps per SM
//     sub-partition, so one hides the other's latency): S = q K^T on mma.sync
//     m16n8k16 and O += P V on m16n8k8 (fp16 in, fp32 accumulate).  Query
//     heads are rows 0..G-1 of the A operand; in P V the fp16 split
//     P = P_hi + P_lo puts P_hi in rows 0..7 and P_lo in rows 8..15 of the same
//     fragment, so P keeps ~22 bits.  Online softmax (base 2) per warp, merged
//     through shared memory when the CTA moves to another segment or phase.
//   - Each CTA writes one (m, l, acc) partial per segment and phase it touched
//     and, after its last unit, takes one ticket per partial; the CTA that
//     completes a segment's count merges its partials in CTA order
//     (deterministic) and writes out[b][h].
#include "kt_internal.cuh"

namespace kt {
namespace {

constexpr int STAGES = 4;
constexpr int CONSUMERS = 8;
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
  static constexpr int touched = sl + MAX_SEGS * 4;
  static constexpr int info = touched + 64 * 4;
  static constexpr int bars = (info + STAGES * (int)sizeof(StageInfo) + 15) & ~15;
  static constexpr int bcast = bars + 2 * STAGES * 8;
  static constexpr int total = bcast + 128 * 4;
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
    if (lane == 0) {
      prefetch_tensormap(&p.kmap);
      prefetch_tensormap(&p.vmap);
    }
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
  const int ctid = tid;  // 0 .. CONSUMERS*32-1
  constexpr int NCT = CONSUMERS * 32;
  float acc[16][4];
  float m_run = -INFINITY, l_part = 0.0f;
  uint32_t qa[8][2];
  int cur_seg = -1, cur_phase = 0;
  bool q_loaded = false;
  int* touched = reinterpret_cast<int*>(smem + SmemLayout::touched);  // (seg << 1 | phase)
  int ntouched = 0;  // maintained identically by every consumer thread
  const int slot_stride = p.slot_floats;
  const long long half_slots = (long long)NC + S;

  auto reset_state = [&]() {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    m_run = -INFINITY;
    l_part = 0.0f;
  };

  // Merge the eight warps' states and write this CTA's partial for (seg, phase).
  // Slot layout: O[G][128], then m[G], then l[G] (base-2 log domain).
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
    named_bar_sync(1, NCT);
    // per head: M = max over warps, weights exp2(m_w - M), L = sum l_w w
    float* fw = reinterpret_cast<float*>(bcast + 32);  // [G][CONSUMERS] weights
    float* fm = reinterpret_cast<float*>(bcast + 8);   // [G] M, then [G] L at +MAX_G
    if (ctid < p.G) {
      const int gg = ctid;
      float M = -INFINITY;
      for (int w = 0; w < CONSUMERS; ++w) M = fmaxf(M, scratch[(w * MAX_G + gg) * (D + 2)]);
      float L = 0.0f;
      for (int w = 0; w < CONSUMERS; ++w) {
        const float* sc = scratch + (w * MAX_G + gg) * (D + 2);
        const float wt = (M == -INFINITY) ? 0.0f : exp2f(sc[0] - M);
        fw[gg * CONSUMERS + w] = wt;
        L += sc[1] * wt;
      }
      fm[gg] = M;
      fm[MAX_G + gg] = L;
    }
    named_bar_sync(1, NCT);
    const long long slot = (phase == 0 ? 0 : half_slots) + cta + seg;
    float* dst = p.parts + slot * slot_stride;
    for (int idx = ctid; idx < p.G * D; idx += NCT) {
      const int gg = idx / D, c = idx % D;
      float o = 0.0f;
#pragma unroll
      for (int w = 0; w < CONSUMERS; ++w)
        o = fmaf(scratch[(w * MAX_G + gg) * (D + 2) + 2 + c], fw[gg * CONSUMERS + w], o);
      dst[gg * D + c] = o;
      if (c == 0) {
        dst[p.G * D + gg] = fm[gg];
        dst[p.G * D + p.G + gg] = fm[MAX_G + gg];
      }
    }
    if (ctid == 0) {
      if (ntouched < 64) touched[ntouched] = (seg << 1) | phase;
      else set_status(p.status, KT_ERR_DEVICE_CHECK);  // more partials than the list holds
    }
    ++ntouched;
    named_bar_sync(1, NCT);
  };

  auto expected_parts = [&](int seg, long long UB) {
    return count_overlapping_ctas(prefA[seg], prefA[seg + 1], UA, NC) +
           count_overlapping_ctas(prefB[seg], prefB[seg + 1], UB, NC);
  };

  // Final merge of all partials of `seg` (CTA order, phase A then B).  Thread
  // 0 lists the partial slots (arithmetic only).  Each thread then owns one
  // float4 chunk of the G x 128 outputs and a share of the partials, loads
  // them in batches of 16 with independent loads, and merges online (base 2);
  // the shares are combined through shared memory in a fixed order.
  auto merge = [&](int seg, long long UB) {
    int* slots = reinterpret_cast<int*>(scratch);
    float* red = scratch + 2 * MAX_ATTN_CTAS;  // per thread: M, L, O.xyzw
    if (ctid == 0) {
      int np = 0;
      for_overlapping_ctas(prefA[seg], prefA[seg + 1], UA, NC,
                           [&](int cc) { slots[np++] = cc + seg; });
      for_overlapping_ctas(prefB[seg], prefB[seg + 1], UB, NC,
                           [&](int cc) { slots[np++] = (int)half_slots + cc + seg; });
      bcast[1] = np;
    }
    named_bar_sync(1, NCT);
    const int np = bcast[1];
    const int b = seg / p.H_kv, h = seg % p.H_kv;
    const int nchunk = p.G * D / 4;             // float4 chunks of the output
    const int nsplit = NCT / nchunk;            // 1 (G=8), 2 (G=4), 4, 8
    const int ch = ctid % nchunk, sp = ctid / nchunk;
    const int f = 4 * ch, gg = f / D;
    const int i0 = sp * np / nsplit, i1 = (sp + 1) * np / nsplit;
    float M = -INFINITY, L = 0.0f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = i0; base < i1; base += 16) {
      const int nb = min(16, i1 - base);
      float m[16], l[16];
      float4 o[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k < nb) {
          const float* src = p.parts + (size_t)slots[base + k] * slot_stride;
          m[k] = __ldcg(src + p.G * D + gg);
          l[k] = __ldcg(src + p.G * D + p.G + gg);
          o[k] = __ldcg(reinterpret_cast<const float4*>(src + f));
        } else {
          m[k] = -INFINITY;
          l[k] = 0.0f;
          o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float Mn = M;
#pragma unroll
      for (int k = 0; k < 16; ++k) Mn = fmaxf(Mn, m[k]);
      if (Mn == -INFINITY) continue;
      const float a = exp2f(M - Mn);  // 0 when M is -inf
      L *= a;
      O.x *= a; O.y *= a; O.z *= a; O.w *= a;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float w = exp2f(m[k] - Mn);  // 0 for empty partials
        L = fmaf(l[k], w, L);
        O.x = fmaf(o[k].x, w, O.x);
        O.y = fmaf(o[k].y, w, O.y);
        O.z = fmaf(o[k].z, w, O.z);
        O.w = fmaf(o[k].w, w, O.w);
      }
      M = Mn;
    }
    if (nsplit > 1) {
      float* r = red + 6 * ctid;
      r[0] = M; r[1] = L; r[2] = O.x; r[3] = O.y; r[4] = O.z; r[5] = O.w;
      named_bar_sync(1, NCT);
      if (sp == 0) {
        for (int q = 1; q < nsplit; ++q) {
          const float* o2 = red + 6 * (ctid + q * nchunk);
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
    if (ctid == 0) p.counters[seg] = 0;
    named_bar_sync(1, NCT);
  };

  reset_state();
  for (uint32_t it = 0;; ++it) {
    const uint32_t st = it % STAGES;
    if (!mbar_wait(bar_full + 8 * st, (it / STAGES) & 1, p.status)) break;
    const StageInfo in = info[st];
    if (in.end || in.seg != cur_seg || in.phase != cur_phase) {
      if (cur_seg >= 0) flush(cur_seg, cur_phase);
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
    if (in.ntok > 0 && warp * 8 < in.ntok) {
      const uint32_t kb = kv_base + st * KV_STAGE_BYTES;
      const uint32_t vb = kb + 2 * BOX_BYTES;
      const int mi = lane >> 3, r = lane & 7;
      const int tok = warp * 8 + r;  // this warp's 8 tokens
      // ---- S = q K^T: one n-tile of 8 tokens, k = 128 channels as two
      // independent accumulation chains
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int chunk = 4 * j + mi;  // 8-channel chunks 4j .. 4j+3
        const uint32_t addr = kb + (chunk >> 3) * BOX_BYTES + tok * 128 +
                              (((chunk & 7) ^ (tok & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, addr);
        mma_16816(sa, qa[2 * j][0], 0u, qa[2 * j][1], 0u, b0, b1);
        mma_16816(sb, qa[2 * j + 1][0], 0u, qa[2 * j + 1][1], 0u, b2, b3);
      }
      // ---- online softmax (base 2), rows = query heads
      const int tk = warp * 8 + 2 * t;
      const float x0 = (tk < in.ntok) ? (sa[0] + sb[0]) * p.scale_log2 : -INFINITY;
      const float x1 = (tk + 1 < in.ntok) ? (sa[1] + sb[1]) * p.scale_log2 : -INFINITY;
      float mx = fmaxf(x0, x1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      const float p0 = exp2f(x0 - m_use), p1 = exp2f(x1 - m_use);
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
      l_part += p0 + p1;
      // ---- P = P_hi (row g) + P_lo (row g+8)
      const __half h0 = __float2half_rn(p0), h1 = __float2half_rn(p1);
      const __half l0 = __float2half_rn(p0 - __half2float(h0));
      const __half l1 = __float2half_rn(p1 - __half2float(h1));
      const uint32_t pa0 = pack_half2(h0, h1), pa1 = pack_half2(l0, l1);
      // ---- O += P V over this warp's 8 tokens (k = 8), 16 channel tiles
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int chunk = 4 * j + mi;
        const uint32_t addr = vb + (chunk >> 3) * BOX_BYTES + tok * 128 +
                              (((chunk & 7) ^ (tok & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, addr);
        mma_1688(acc[4 * j + 0], pa0, pa1, b0);
        mma_1688(acc[4 * j + 1], pa0, pa1, b1);
        mma_1688(acc[4 * j + 2], pa0, pa1, b2);
        mma_1688(acc[4 * j + 3], pa0, pa1, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * st);
  }

  // ---- tickets: one per partial this CTA wrote; the completing CTA merges
  const long long UB = prefB[S];  // the producer wrote it before the end marker
  __threadfence();
  named_bar_sync(1, NCT);
  int* lastflag = bcast + 96;  // 32 flags per round
  if (ntouched > 64) ntouched = 64;
  for (int base = 0; base < ntouched; base += 32) {
    const int n_here = min(32, ntouched - base);
    if (ctid < n_here) {
      const int code = touched[base + ctid];
      const int seg = code >> 1;
      const int old = atomicAdd(p.counters + seg, 1);
      lastflag[ctid] = (old + 1 == expected_parts(seg, UB)) ? (seg + 1) : 0;
    }
    named_bar_sync(1, NCT);
    for (int i = 0; i < n_here; ++i) {
      const int seg1 = lastflag[i];
      if (seg1) {
        __threadfence();
        merge(seg1 - 1, UB);
      }
    }
    named_bar_sync(1, NCT);
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
