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
#include "select_common.cuh"

namespace kt {
namespace {

using selc::dot8;
using selc::make_key;
using selc::warp_sum;
using selc::warp_sum_int;


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
  const uint32_t* presel_mask;  // nullable [B][SEL][mask_words]
  int mask_words;
};

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
        if (V <= 32) selc::score_linear<1, true, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
        else if (V <= 64) selc::score_linear<2, true, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
        else if (V <= 128) selc::score_linear<4, true, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
        else selc::score_linear<8, true, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
      } else {
        if (V <= 32) selc::score_linear<1, false, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
        else if (V <= 64) selc::score_linear<2, false, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
        else if (V <= 128) selc::score_linear<4, false, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
        else selc::score_linear<8, false, WARPS>(p.reps, p.P, p.H_kv, p.R, g0, js, je, pg, wts, V, keys, warp, lane, p.status);
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
    // preselection: blocks outside it get key 0, the empty slot
    if (p.presel_mask) {
      const uint32_t* mk = p.presel_mask + unit_base * p.mask_words;
      for (int i = tid; i < nloc; i += THREADS) {
        const int j = js + i;
        if (!((__ldg(mk + (j >> 5)) >> (j & 31)) & 1u)) keys[i] = 0ull;
      }
      __syncthreads();
    }

    // ---- this chunk's top-kk candidates; unused slots hold key 0, which is
    // below every real key
    if (nloc <= p.kk) {
      for (int i = tid; i < p.kk; i += THREADS) {
        my_cand[i] = i < nloc ? keys[i] : 0ull;
        my_pages[i] = i < nloc ? pg[i] : -1;
      }
    } else {
      unsigned long long prefix, mask;
      selc::radix_select<THREADS>(keys, nloc, p.kk, hist, sh_u64, sh_int, &prefix, &mask, tid,
                                    [] { __syncthreads(); });
      if (tid == 0) sh_int[2] = 0;
      for (int i = tid; i < p.kk; i += THREADS) {  // slots left empty stay key 0
        my_cand[i] = 0ull;
        my_pages[i] = -1;
      }
      __syncthreads();
      for (int i = tid; i < nloc; i += THREADS) {
        const unsigned long long key = keys[i];
        if (key != 0ull && (key & mask) >= prefix) {
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
  __syncthreads();
  if (tid == 0) {
    const int old = atom_acq_rel_gpu_add(p.counters + unit_base, 1);
    sh_int[3] = (old == p.nchunks - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!sh_int[3]) return;

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
      selc::radix_select<THREADS>(all, total, keff, hist, sh_u64, sh_int, &prefix, &mask, tid,
                                    [] { __syncthreads(); });
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
  p.presel_mask = a.presel_mask;
  p.mask_words = a.mask_words;
  const size_t smem = select_smem_bytes(a);
  // the shared-memory opt-in only grows; it is raised when a call needs more
  static std::atomic<int> optin[KT_MAX_DEVICES];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int want = (int)(smem > 48 * 1024 ? smem : 48 * 1024);
  if (dev < 0 || dev >= KT_MAX_DEVICES || optin[dev].load(std::memory_order_relaxed) < want) {
    e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < KT_MAX_DEVICES) {
      int cur = optin[dev].load(std::memory_order_relaxed);
      while (cur < want && !optin[dev].compare_exchange_weak(cur, want)) {
      }
    }
  }
  const dim3 grid(a.plan.nchunks, a.plan.SEL, a.B);
  select_kernel<<<grid, THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kt
