// select.cu — block scoring and deterministic top-k selection.
//
// For each selection unit (a sequence and, in SEPARATE mode, one KV head) every
// Context block gets a unit score and the top-k blocks are chosen (article
// "KTransformers 长上下文稀疏注意力实战…": Quest bound §3.1, similarity to the
// representative tokens §4.3, top-k and head_select_mode §4.5).
//
//   head score   Quest      sum_c max(q_c kmax_c, q_c kmin_c)
//                Max/Mean   q . rep
//                Fix/Dyn    max_r q . rep_r
//   unit score   sum of head scores over the unit's query heads
//
// Linear methods (Max, Mean, Quest) fold the query heads of a KV head into one
// weight vector per representative row: for Quest max(q kmax, q kmin) equals
// relu(q) kmax + min(q, 0) kmin exactly (kmax >= kmin), so the unit score is a
// single dot product of the block's representative bytes with a precomputed
// fp32 weight vector.  Fix and Dynamic keep per-head dot products.
//
// Grid (chunks, units, batch): each CTA scores a chunk of Context blocks, keeps
// its chunk's top-k with a radix select over 64-bit keys
// (score-order bits << 32 | ~block), and the CTA that takes the unit's last
// ticket merges all chunk candidates, sorts the chosen blocks by id and writes
// sel / cnt / sel_scores.  Ties go to the lower block id; the result does not
// depend on CTA timing.
#include "kt_internal.cuh"

namespace kt {
namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;

struct Params {
  const __half* q;
  const void* reps;
  const int32_t* table;
  const int32_t* seq_lens;
  int32_t* sel;
  int32_t* cnt;
  float* sel_scores;
  int* status;
  int* counters;
  unsigned long long* cand;
  int* cand_pages;
  int32_t* sel_pages;
  int B, H_kv, G, max_blocks, P, I_b, L_b, top_k, rep, R, head_mode;
  int SEL, chunk, nchunks, kk;
  int trigger;
};

__device__ __forceinline__ float dot8(const float* w, uint4 v) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    s = fmaf(w[2 * i], f.x, s);
    s = fmaf(w[2 * i + 1], f.y, s);
  }
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long make_key(float score, int block) {
  return (static_cast<unsigned long long>(float_key(score)) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(block));
}

// k-th largest of N distinct keys in shared memory (1 <= k <= N), all threads
// of the CTA.  On return, a key is among the k largest iff
// (key & *mask_out) >= *prefix_out.  MSB-first radix select on 8-bit digits;
// the leading bits common to every key are skipped.  hist holds two 256-bin
// histograms used alternately, so each pass needs two barriers.
__device__ void radix_select(const unsigned long long* keys, int N, int k, unsigned int* hist,
                             unsigned long long* sh_u64, int* sh_int,
                             unsigned long long* prefix_out, unsigned long long* mask_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // common leading bits: AND and OR over all keys; clear both histograms
  unsigned long long a = ~0ull, o = 0ull;
  for (int i = tid; i < N; i += THREADS) {
    a &= keys[i];
    o |= keys[i];
  }
  for (int i = tid; i < 512; i += THREADS) hist[i] = 0u;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    a &= __shfl_xor_sync(0xffffffffu, a, d);
    o |= __shfl_xor_sync(0xffffffffu, o, d);
  }
  unsigned long long* red = sh_u64 + 2;  // [WARPS] ANDs, then [WARPS] ORs
  if (lane == 0) {
    red[warp] = a;
    red[WARPS + warp] = o;
  }
  __syncthreads();
  unsigned long long all_and = ~0ull, all_or = 0ull;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) {
    all_and &= red[w];
    all_or |= red[WARPS + w];
  }
  const unsigned long long diff = all_and ^ all_or;
  const int top = diff ? 63 - __clzll((long long)diff) : 0;  // highest differing bit
  // digit windows [lo, hi) of up to 8 bits, starting at the top differing bit
  int hi = top + 1;
  unsigned long long mask = (hi >= 64) ? 0ull : ~((1ull << hi) - 1);
  unsigned long long prefix = all_and & mask;
  int need = k;
  for (int pass = 0; hi > 0; ++pass) {
    const int shift = hi > 8 ? hi - 8 : 0;
    const unsigned long long dmask = (1ull << (hi - shift)) - 1;
    unsigned int* H = hist + 256 * (pass & 1);
    unsigned int* Hn = hist + 256 * ((pass + 1) & 1);
    for (int base = 0; base < N; base += THREADS) {
      // equal digits are counted once per warp: keys are often clustered
      const int i = base + tid;
      unsigned int bin = 256u;
      if (i < N) {
        const unsigned long long key = keys[i];
        if ((key & mask) == prefix) bin = (unsigned)((key >> shift) & dmask);
      }
      const unsigned int peers = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && lane == __ffs(peers) - 1) atomicAdd(&H[bin], (unsigned)__popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds digits 255-8l .. 248-8l (descending)
      unsigned int c[8];
      unsigned int local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = H[255 - 8 * lane - i];
        local += c[i];
      }
      unsigned int incl = local;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const unsigned int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      const unsigned int excl = incl - local;
      const bool hit = excl < (unsigned)need && (unsigned)need <= incl;
      const unsigned int ball = __ballot_sync(0xffffffffu, hit);
      const int src = __ffs(ball) - 1;
      if (lane == src) {
        unsigned int above = excl;
        int digit = 0;
        unsigned int bin = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above + c[i] >= (unsigned)need) {
            digit = 255 - 8 * lane - i;
            bin = c[i];
            break;
          }
          above += c[i];
        }
        const int need2 = need - (int)above;
        sh_u64[0] = prefix | (static_cast<unsigned long long>(digit) << shift);
        sh_u64[1] = mask | (dmask << shift);
        sh_int[0] = need2;
        sh_int[1] = (bin == (unsigned)need2) ? 1 : 0;
      }
    } else {
      for (int i = tid - 32; i < 256; i += THREADS - 32) Hn[i] = 0u;  // next pass's bins
    }
    __syncthreads();
    prefix = sh_u64[0];
    mask = sh_u64[1];
    need = sh_int[0];
    if (sh_int[1]) break;
    hi = shift;
  }
  __syncthreads();  // sh_* are rewritten by the caller
  *prefix_out = prefix;
  *mask_out = mask;
}

// Linear scoring (Max, Mean, Quest): each warp scores 8/NV blocks at a time;
// a lane holds NV 16-byte vectors of each block, and every load of the group is
// issued before any arithmetic.  V = 16-byte vectors per block and unit.
template <int NV, bool F32>
__device__ __forceinline__ void score_linear(const Params& p, int g0, int js, int je,
                                             const int* pg, const float* wts, int V,
                                             unsigned long long* keys, int warp, int lane) {
  constexpr int GB = 8 / NV;
  constexpr int VE = F32 ? 4 : 8;
  float w[NV][VE];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int vec = lane + 32 * v;
#pragma unroll
    for (int e = 0; e < VE; e += 4) {
      const float4 f = (vec < V) ? *reinterpret_cast<const float4*>(wts + vec * VE + e)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
      w[v][e] = f.x;
      w[v][e + 1] = f.y;
      w[v][e + 2] = f.z;
      w[v][e + 3] = f.w;
    }
  }
  const size_t head_bytes = (size_t)p.R * D * (F32 ? 4 : 2);
  for (int j0 = js + warp * GB; j0 < je; j0 += WARPS * GB) {
    uint4 x[GB][NV];
    int page[GB];
#pragma unroll
    for (int bi = 0; bi < GB; ++bi) {
      const int j = j0 + bi;
      page[bi] = (j < je) ? pg[j - js] : -1;
      const bool ok = page[bi] >= 0 && page[bi] < p.P;
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(p.reps) +
          ((size_t)(ok ? page[bi] : 0) * p.H_kv + g0) * head_bytes);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int vec = lane + 32 * v;
        x[bi][v] = (ok && vec < V) ? __ldg(src + vec) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int bi = 0; bi < GB; ++bi) {
      float acc = 0.0f;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        if (F32) {
          const float4 f = *reinterpret_cast<const float4*>(&x[bi][v]);
          acc = fmaf(w[v][0], f.x, acc);
          acc = fmaf(w[v][1], f.y, acc);
          acc = fmaf(w[v][2], f.z, acc);
          acc = fmaf(w[v][3], f.w, acc);
        } else {
          acc += dot8(w[v], x[bi][v]);
        }
      }
      acc = warp_sum(acc);
      const int j = j0 + bi;
      if (j < je) {
        const bool ok = page[bi] >= 0 && page[bi] < p.P;
        if (lane == 0) keys[j - js] = make_key(ok ? acc : -INFINITY, j);
        if (!ok && lane == 0) set_status(p.status, KT_ERR_DEVICE_CHECK);
      }
    }
  }
}

__global__ void __launch_bounds__(THREADS) select_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ unsigned int hist[512];
  __shared__ unsigned long long sh_u64[2 + 2 * WARPS];
  __shared__ int sh_int[4];

  if (p.trigger) griddep_launch_dependents();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = blockIdx.x, u = blockIdx.y, b = blockIdx.z;
  const int H_q = p.H_kv * p.G;
  const int nkv = p.head_mode == KT_HEAD_SHARED ? p.H_kv : 1;  // KV heads in the unit
  const int g0 = p.head_mode == KT_HEAD_SHARED ? 0 : u;
  const bool linear = p.rep == KT_REP_MAX || p.rep == KT_REP_MEAN || p.rep == KT_REP_QUEST;
  const int Rw = p.rep == KT_REP_QUEST ? 2 : 1;  // weight rows for linear methods
  // shared memory: weights (fp32), keys (u64), query rows (fp16), pages (int)
  float* wts = reinterpret_cast<float*>(smem);
  const int wfloats = linear ? nkv * Rw * D : (p.head_mode == KT_HEAD_SHARED ? H_q : p.G) * D;
  unsigned long long* keys =
      reinterpret_cast<unsigned long long*>(smem + ((wfloats * 4 + 15) & ~15));
  const int nq = nkv * p.G;  // query heads of the unit, contiguous from g0*G
  __half* qs = reinterpret_cast<__half*>(keys + ((p.chunk + 1) & ~1));  // 16-B aligned
  int* pg = reinterpret_cast<int*>(qs + nq * D);

  // ---- independent loads first: sequence length, the chunk's block-table
  // entries (when the sequence has Context blocks the chunk starts at block
  // I_b + chunk*CH) and the unit's query rows
  int n = p.seq_lens[b];
  const int js_nom = p.I_b + chunk * p.chunk;
  for (int t = tid; t < p.chunk; t += THREADS) {
    const int j = js_nom + t;
    pg[t] = (j < p.max_blocks) ? __ldg(p.table + (size_t)b * p.max_blocks + j) : -1;
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)b * H_q + g0 * p.G) * D);
    uint4* dst = reinterpret_cast<uint4*>(qs);
    for (int i = tid; i < nq * D / 8; i += THREADS) dst[i] = __ldg(src + i);
  }
  if (n < 0 || n > p.max_blocks * BS) {
    set_status(p.status, KT_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : p.max_blocks * BS;
  }
  const int nb = (n + BS - 1) / BS;
  const int c0 = min(p.I_b, nb), c1 = max(c0, nb - p.L_b);
  const int js = c0 + chunk * p.chunk, je = min(js + p.chunk, c1);  // js == js_nom if nloc > 0
  const int nloc = max(0, je - js);

  const size_t unit_base = (size_t)b * p.SEL + u;
  unsigned long long* my_cand = p.cand + (unit_base * p.nchunks + chunk) * p.kk;
  int* my_pages = p.cand_pages + (unit_base * p.nchunks + chunk) * p.kk;
  __syncthreads();

  if (nloc > 0) {
    // ---- weights (query heads summed in ascending order)
    if (linear) {
      for (int i = tid; i < nkv * D; i += THREADS) {
        const int gi = i / D, c = i % D;
        float sum = 0.0f, neg = 0.0f, pos = 0.0f;
        for (int hh = 0; hh < p.G; ++hh) {
          const float qv = __half2float(qs[(gi * p.G + hh) * D + c]);
          sum += qv;
          neg += fminf(qv, 0.0f);
          pos += fmaxf(qv, 0.0f);
        }
        if (p.rep == KT_REP_QUEST) {
          wts[(gi * 2 + 0) * D + c] = neg;  // pairs with the kmin row
          wts[(gi * 2 + 1) * D + c] = pos;  // pairs with the kmax row
        } else {
          wts[gi * D + c] = sum;
        }
      }
    } else {
      for (int i = tid; i < wfloats; i += THREADS) wts[i] = __half2float(qs[i]);
    }
    __syncthreads();

    // ---- scores
    if (linear) {
      const bool f32 = p.rep == KT_REP_MEAN;
      const int V = nkv * p.R * D / (f32 ? 4 : 8);  // 16-byte vectors per block
      if (f32) {
        if (V <= 32) score_linear<1, true>(p, g0, js, je, pg, wts, V, keys, warp, lane);
        else if (V <= 64) score_linear<2, true>(p, g0, js, je, pg, wts, V, keys, warp, lane);
        else if (V <= 128) score_linear<4, true>(p, g0, js, je, pg, wts, V, keys, warp, lane);
        else score_linear<8, true>(p, g0, js, je, pg, wts, V, keys, warp, lane);
      } else {
        if (V <= 32) score_linear<1, false>(p, g0, js, je, pg, wts, V, keys, warp, lane);
        else if (V <= 64) score_linear<2, false>(p, g0, js, je, pg, wts, V, keys, warp, lane);
        else if (V <= 128) score_linear<4, false>(p, g0, js, je, pg, wts, V, keys, warp, lane);
        else score_linear<8, false>(p, g0, js, je, pg, wts, V, keys, warp, lane);
      }
    } else {
      // Fix / Dynamic: per KV head, per query head, max over reps of q.rep;
      // lane owns channels 4*lane .. 4*lane+3.
      for (int j = js + warp; j < je; j += WARPS) {
        const int page = pg[j - js];
        float total = 0.0f;
        if (page < 0 || page >= p.P) {
          set_status(p.status, KT_ERR_DEVICE_CHECK);
          total = -INFINITY;
        } else {
          for (int gi = 0; gi < nkv; ++gi) {
            const int g = g0 + gi;
            const __half* rp =
                static_cast<const __half*>(p.reps) + ((size_t)page * p.H_kv + g) * p.R * D;
            for (int hh = 0; hh < p.G; ++hh) {
              const float* w =
                  wts + ((p.head_mode == KT_HEAD_SHARED ? g * p.G : 0) + hh) * D + 4 * lane;
              float best = -INFINITY;
              for (int r = 0; r < p.R; ++r) {
                const uint2 raw = __ldg(reinterpret_cast<const uint2*>(rp + r * D) + lane);
                const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
                const float2 f0 = __half22float2(h2[0]), f1 = __half22float2(h2[1]);
                float sc = w[0] * f0.x;
                sc = fmaf(w[1], f0.y, sc);
                sc = fmaf(w[2], f1.x, sc);
                sc = fmaf(w[3], f1.y, sc);
                sc = warp_sum(sc);
                best = fmaxf(best, sc);
              }
              total += best;
            }
          }
        }
        if (lane == 0) keys[j - js] = make_key(total, j);
      }
    }
    __syncthreads();

    // ---- this chunk's top-kk candidates; unused slots hold key 0, which is
    // below every real key
    if (nloc <= p.kk) {
      for (int i = tid; i < p.kk; i += THREADS) {
        my_cand[i] = i < nloc ? keys[i] : 0ull;
        my_pages[i] = i < nloc ? pg[i] : -1;
      }
    } else {
      unsigned long long prefix, mask;
      radix_select(keys, nloc, p.kk, hist, sh_u64, sh_int, &prefix, &mask);
      if (tid == 0) sh_int[2] = 0;
      __syncthreads();
      for (int i = tid; i < nloc; i += THREADS) {
        const unsigned long long key = keys[i];
        if ((key & mask) >= prefix) {
          const int pos = atomicAdd(&sh_int[2], 1);
          if (pos < p.kk) {
            my_cand[pos] = key;
            my_pages[pos] = pg[i];
          } else {
            set_status(p.status, KT_ERR_DEVICE_CHECK);
          }
        }
      }
    }
  }
  if (nloc <= 0)
    for (int i = tid; i < p.kk; i += THREADS) {
      my_cand[i] = 0ull;
      my_pages[i] = -1;
    }

  // ---- ticket: the last chunk CTA of this unit merges
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int old = atomicAdd(p.counters + unit_base, 1);
    sh_int[3] = (old == p.nchunks - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!sh_int[3]) return;
  __threadfence();

  // gather every candidate slot of the unit into shared memory (independent,
  // coalesced loads); empty slots are key 0
  unsigned long long* all = keys;
  const int nslots = p.nchunks * p.kk;
  const int max_keff = min(p.top_k, nslots);
  int* allp = reinterpret_cast<int*>(all + nslots + max_keff);  // pages of `all`
  int* chosenp = allp + nslots;                                  // pages of `chosen`
  const unsigned long long* src = p.cand + unit_base * (size_t)nslots;
  const int* srcp = p.cand_pages + unit_base * (size_t)nslots;
  int real = 0;
  for (int i = tid; i < nslots; i += THREADS) {
    const unsigned long long key = __ldcg(src + i);
    all[i] = key;
    allp[i] = __ldcg(srcp + i);
    real += key != 0ull ? 1 : 0;
  }
  real = warp_sum_int(real);
  if (tid == 0) sh_int[0] = 0;
  __syncthreads();
  if (lane == 0) atomicAdd(&sh_int[0], real);
  __syncthreads();
  const int total_real = sh_int[0];
  const int total = nslots;
  __syncthreads();

  const int keff = min(p.top_k, total_real);
  unsigned long long* chosen = all + total;  // keff entries
  if (keff > 0) {
    if (keff == total) {
      for (int i = tid; i < total; i += THREADS) {
        chosen[i] = all[i];
        chosenp[i] = allp[i];
      }
    } else {  // keff <= total_real: the zero slots are never chosen
      unsigned long long prefix, mask;
      radix_select(all, total, keff, hist, sh_u64, sh_int, &prefix, &mask);
      if (tid == 0) sh_int[2] = 0;
      __syncthreads();
      for (int i = tid; i < total; i += THREADS) {
        const unsigned long long key = all[i];
        if ((key & mask) >= prefix) {
          const int pos = atomicAdd(&sh_int[2], 1);
          if (pos < keff) {
            chosen[pos] = key;
            chosenp[pos] = allp[i];
          } else {
            set_status(p.status, KT_ERR_DEVICE_CHECK);
          }
        }
      }
    }
    __syncthreads();
    // ascending block order: rank by counting
    int32_t* sel_out = p.sel + unit_base * p.top_k;
    float* sc_out = p.sel_scores ? p.sel_scores + unit_base * p.top_k : nullptr;
    for (int i = tid; i < keff; i += THREADS) {
      const unsigned long long ki = chosen[i];
      const uint32_t id = 0xFFFFFFFFu - static_cast<uint32_t>(ki & 0xFFFFFFFFull);
      int rank = 0;
      for (int m = 0; m < keff; ++m) {
        const uint32_t idm = 0xFFFFFFFFu - static_cast<uint32_t>(chosen[m] & 0xFFFFFFFFull);
        rank += idm < id ? 1 : 0;
      }
      sel_out[rank] = static_cast<int32_t>(id);
      if (sc_out) sc_out[rank] = key_float(static_cast<uint32_t>(ki >> 32));
      if (p.sel_pages) p.sel_pages[unit_base * p.top_k + rank] = chosenp[i];
    }
  }
  if (tid == 0) {
    p.cnt[unit_base] = keff;
    p.counters[unit_base] = 0;
  }
}

}  // namespace

size_t select_smem_bytes(const SelectLaunch& a) {
  const bool linear = a.rep == KT_REP_MAX || a.rep == KT_REP_MEAN || a.rep == KT_REP_QUEST;
  const int nkv = a.head_mode == KT_HEAD_SHARED ? a.H_kv : 1;
  const int Rw = a.rep == KT_REP_QUEST ? 2 : 1;
  const int wfloats =
      linear ? nkv * Rw * D : (a.head_mode == KT_HEAD_SHARED ? a.H_kv * a.G : a.G) * D;
  const int chunk_keys = (a.plan.chunk + 1) & ~1;
  const int merged = a.plan.nchunks * a.plan.kk;
  // keys of all slots and of the chosen ones, plus their page ids (as ints)
  const int merge_keys = merged + (a.top_k < merged ? a.top_k : merged) +
                         (merged + (a.top_k < merged ? a.top_k : merged) + 1) / 2;
  const int nq = nkv * a.G;
  // keys + staged q rows + the chunk's page ids
  const int score_keys = chunk_keys + (nq * D * 2 + 7) / 8 + (a.plan.chunk * 4 + 7) / 8;
  const int nkeys = score_keys > merge_keys ? score_keys : merge_keys;
  return (size_t)((wfloats * 4 + 15) & ~15) + (size_t)nkeys * 8;
}

cudaError_t launch_select(const SelectLaunch& a, cudaStream_t stream) {
  Params p;
  p.q = a.q;
  p.reps = a.reps;
  p.table = a.table;
  p.seq_lens = a.seq_lens;
  p.sel = a.sel;
  p.cnt = a.cnt;
  p.sel_scores = a.sel_scores;
  p.status = a.status;
  p.counters = a.counters;
  p.cand = a.cand;
  p.cand_pages = a.cand_pages;
  p.sel_pages = a.sel_pages;
  p.B = a.B;
  p.H_kv = a.H_kv;
  p.G = a.G;
  p.max_blocks = a.max_blocks;
  p.P = a.P;
  p.I_b = a.I_b;
  p.L_b = a.L_b;
  p.top_k = a.top_k;
  p.rep = a.rep;
  p.R = a.R;
  p.head_mode = a.head_mode;
  p.SEL = a.plan.SEL;
  p.chunk = a.plan.chunk;
  p.nchunks = a.plan.nchunks;
  p.kk = a.plan.kk;
  p.trigger = a.trigger_dependents ? 1 : 0;
  const size_t smem = select_smem_bytes(a);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(smem > 48 * 1024 ? smem : 48 * 1024));
  if (e != cudaSuccess) return e;
  const dim3 grid(a.plan.nchunks, a.plan.SEL, a.B);
  select_kernel<<<grid, THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kt
