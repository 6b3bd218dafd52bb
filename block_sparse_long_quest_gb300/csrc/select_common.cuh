// select_common.cuh — block scoring and radix top-k helpers shared by the
// selection kernel and the fused decode-step kernel.
#pragma once

#include "kt_internal.cuh"

namespace kt {
namespace selc {

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

// warp_sum of N independent values, the butterfly steps interleaved so that
// the N shuffle chains overlap; each value is summed in warp_sum's order.
template <int N>
__device__ __forceinline__ void warp_sum_n(float (&v)[N]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
  }
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


// This lane's share of a block's dot product with the weights: NV 16-byte
// vectors, fp16 (8 values each) or fp32 (4 values each), in a fixed order.
template <int NV, bool F32>
__device__ __forceinline__ float lane_dot(const float (&w)[NV][F32 ? 4 : 8], const uint4 (&x)[NV]) {
  float acc = 0.0f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if constexpr (F32) {
      const float4 f = *reinterpret_cast<const float4*>(&x[v]);
      acc = fmaf(w[v][0], f.x, acc);
      acc = fmaf(w[v][1], f.y, acc);
      acc = fmaf(w[v][2], f.z, acc);
      acc = fmaf(w[v][3], f.w, acc);
    } else {
      acc += dot8(w[v], x[v]);
    }
  }
  return acc;
}

// k-th largest of N distinct keys in shared memory (1 <= k <= N), all threads
// of the CTA.  On return, a key is among the k largest iff
// (key & *mask_out) >= *prefix_out.  MSB-first radix select on 8-bit digits;
// the leading bits common to every key are skipped.  hist holds two 256-bin
// histograms used alternately, so each pass needs two barriers.
//
// NT threads take part (thread index `tid` in [0, NT)); `bar` synchronises
// exactly those threads.  sh_u64 holds 2 + 2*NT/32 entries, sh_int 2.
template <int NT, class Bar>
__device__ void radix_select(const unsigned long long* keys, int N, int k, unsigned int* hist,
                             unsigned long long* sh_u64, int* sh_int,
                             unsigned long long* prefix_out, unsigned long long* mask_out,
                             int tid, Bar bar) {
  constexpr int WARPS = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  // common leading bits: AND and OR over all keys; clear both histograms
  unsigned long long a = ~0ull, o = 0ull;
#pragma unroll 1
  for (int i = tid; i < N; i += NT) {
    a &= keys[i];
    o |= keys[i];
  }
#pragma unroll 1
  for (int i = tid; i < 512; i += NT) hist[i] = 0u;
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
  bar();
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
#pragma unroll 1
  for (int pass = 0; hi > 0; ++pass) {
    const int shift = hi > 8 ? hi - 8 : 0;
    const unsigned long long dmask = (1ull << (hi - shift)) - 1;
    unsigned int* H = hist + 256 * (pass & 1);
    unsigned int* Hn = hist + 256 * ((pass + 1) & 1);
#pragma unroll 1
    for (int base = 0; base < N; base += NT) {
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
    bar();
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
#pragma unroll 1
      for (int i = tid - 32; i < 256; i += NT - 32) Hn[i] = 0u;  // next pass's bins
    }
    bar();
    prefix = sh_u64[0];
    mask = sh_u64[1];
    need = sh_int[0];
    if (sh_int[1]) break;
    hi = shift;
  }
  bar();  // sh_* are rewritten by the caller
  *prefix_out = prefix;
  *mask_out = mask;
}

// Threshold of the k largest nonzero keys held in registers (GP per thread;
// nonzero keys distinct): returns T > 0 such that exactly min(k, N) nonzero
// keys are >= T, and the count N of nonzero keys in *n_out.  MSB-first passes
// over 11-bit digits of the keys that share the running prefix, starting
// below the bits every key has in common: a 2048-bin histogram, scanned by
// all NT threads at once (PER bins each, warp shuffles, then the warp totals),
// locates the bin of the k-th key; once that bin holds at most NT keys they
// are ranked exactly by counting.  Every one of the NT threads calls it; bar
// synchronises them.  Scratch: hist 2048 u32 (16-byte aligned), bink NT u64,
// sh_u64 2 * NT / 32 + 1 entries, sh_int NT / 32 + 4 entries.
template <int NT, int GP, class Bar>
__device__ __forceinline__ unsigned long long kth_largest_reg(const unsigned long long (&kx)[GP], int k,
                                                           unsigned int* hist, unsigned long long* bink,
                                                           unsigned long long* sh_u64, int* sh_int,
                                                           int* n_out, int tid, Bar bar) {
  constexpr int WARPS = NT / 32, BINS = 2048, PER = BINS / NT;
  static_assert(PER == 8, "two 16-byte vectors of bins per thread");
  const int lane = tid & 31, warp = tid >> 5;
  int* wsum = sh_int + 4;  // [WARPS]
  // common leading bits and the count of the nonzero keys
  unsigned long long a = ~0ull, o = 0ull;
  int cnt = 0;
#pragma unroll
  for (int r = 0; r < GP; ++r)
    if (kx[r]) {
      a &= kx[r];
      o |= kx[r];
      ++cnt;
    }
  {
    // warp reductions as independent redux instructions (no shuffle chain)
    const uint32_t a_lo = __reduce_and_sync(0xffffffffu, static_cast<uint32_t>(a));
    const uint32_t a_hi = __reduce_and_sync(0xffffffffu, static_cast<uint32_t>(a >> 32));
    const uint32_t o_lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(o));
    const uint32_t o_hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(o >> 32));
    const int wc = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cnt)));
    if (lane == 0) {
      sh_u64[warp] = (static_cast<unsigned long long>(a_hi) << 32) | a_lo;
      sh_u64[WARPS + warp] = (static_cast<unsigned long long>(o_hi) << 32) | o_lo;
      wsum[warp] = wc;
    }
  }
  if (tid == 0) sh_int[3] = 0;
  bar();
  a = ~0ull;
  o = 0ull;
  int N = 0;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) {
    a &= sh_u64[w];
    o |= sh_u64[WARPS + w];
    N += wsum[w];
  }
  *n_out = N;
  if (N <= k) return 1ull;  // every nonzero key (uniform: N is the same in every thread)
  const unsigned long long diff = a ^ o;
  int hi = diff ? 64 - __clzll((long long)diff) : 0;  // bits below the common prefix
  unsigned long long mask = hi >= 64 ? 0ull : ~((1ull << hi) - 1);
  unsigned long long prefix = a & mask;
  int need = k, nb = N;
#pragma unroll 1
  while (nb > NT && hi > 0) {
    const int shift = hi > 11 ? hi - 11 : 0;
    const unsigned long long dmask = (1ull << (hi - shift)) - 1;
    bar();  // the previous pass's scan has read the histogram and wsum
    reinterpret_cast<uint4*>(hist)[2 * tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(hist)[2 * tid + 1] = make_uint4(0u, 0u, 0u, 0u);
    bar();
#pragma unroll
    for (int r = 0; r < GP; ++r)
      if (kx[r] && (kx[r] & mask) == prefix) atomicAdd(&hist[(unsigned)((kx[r] >> shift) & dmask)], 1u);
    bar();
    // thread t holds bins BINS-1-PER*t (first) .. BINS-PER-PER*t, descending
    const uint4 lo4 = reinterpret_cast<const uint4*>(hist)[2 * (NT - 1 - tid)];
    const uint4 hi4 = reinterpret_cast<const uint4*>(hist)[2 * (NT - 1 - tid) + 1];
    const unsigned c[PER] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};
    int local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) local += (int)c[i];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    bar();
    int excl = incl - local;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) excl += w < warp ? wsum[w] : 0;
    if (excl < need && need <= excl + local) {
      int above = excl;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        if (above + (int)c[i] >= need) {
          sh_int[0] = BINS - 1 - PER * tid - i;
          sh_int[1] = need - above;
          sh_int[2] = (int)c[i];
          break;
        }
        above += (int)c[i];
      }
    }
    bar();
    prefix |= static_cast<unsigned long long>(sh_int[0]) << shift;
    mask |= dmask << shift;
    need = sh_int[1];
    nb = sh_int[2];
    hi = shift;
  }
  // the keys sharing the final prefix (at most NT of them), ranked exactly
  {
    // one shared atomic per warp (ballots give each key its place)
    const unsigned int lt = (1u << lane) - 1u;
    unsigned int bal[GP];
    int tot = 0;
#pragma unroll
    for (int r = 0; r < GP; ++r) {
      bal[r] = __ballot_sync(0xffffffffu, kx[r] != 0ull && (kx[r] & mask) == prefix);
      tot += __popc(bal[r]);
    }
    int o0 = 0;
    if (lane == 0 && tot) o0 = atomicAdd(&sh_int[3], tot);
    o0 = __shfl_sync(0xffffffffu, o0, 0);
#pragma unroll
    for (int r = 0; r < GP; ++r) {
      const int pos = o0 + __popc(bal[r] & lt);
      // more than NT only if keys repeat (never for distinct keys)
      if (((bal[r] >> lane) & 1u) && pos < NT) bink[pos] = kx[r];
      o0 += __popc(bal[r]);
    }
  }
  if (nb > NT) nb = NT;
  bar();
  for (int i = tid; i < nb; i += NT) {
    const unsigned long long key = bink[i];
    int g = 0;
#pragma unroll 4
    for (int j = 0; j < nb; ++j) g += bink[j] > key ? 1 : 0;
    if (g == need - 1) sh_u64[2 * WARPS] = key;
  }
  bar();
  const unsigned long long t = sh_u64[2 * WARPS];
  bar();  // the caller may reuse the scratch
  return t;
}

// Indices of the k largest of N distinct keys in shared memory (1 <= k <= N),
// written unordered to idx_out[0, k).  MSB-first 8-bit digit histograms over
// the keys sharing the running prefix narrow the search until the bin holding
// the k-th key has at most NT keys (usually after one pass); keys in higher
// bins are taken outright and the bin's keys are ranked exactly among
// themselves.  Scratch: hist 512 bins, bkey/bidx NT entries, sh_u64
// 2 + 2*NT/32, sh_int 4.  All NT threads call it; `bar` synchronises them.
template <int NT, class Bar>
__device__ __noinline__ void select_top(const unsigned long long* keys, int N, int k, int* idx_out,
                           unsigned long long* bkey, int* bidx, unsigned int* hist,
                           unsigned long long* sh_u64, int* sh_int, int tid, Bar bar) {
  constexpr int WARPS = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  if (k >= N) {
    for (int i = tid; i < N; i += NT) idx_out[i] = i;
    bar();
    return;
  }
  unsigned long long a = ~0ull, o = 0ull;
#pragma unroll 1
  for (int i = tid; i < N; i += NT) {
    a &= keys[i];
    o |= keys[i];
  }
#pragma unroll 1
  for (int i = tid; i < 512; i += NT) hist[i] = 0u;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    a &= __shfl_xor_sync(0xffffffffu, a, d);
    o |= __shfl_xor_sync(0xffffffffu, o, d);
  }
  unsigned long long* red = sh_u64 + 2;
  if (lane == 0) {
    red[warp] = a;
    red[WARPS + warp] = o;
  }
  if (tid == 0) {
    sh_int[2] = 0;
    sh_int[3] = 0;
  }
  bar();
  unsigned long long all_and = ~0ull, all_or = 0ull;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) {
    all_and &= red[w];
    all_or |= red[WARPS + w];
  }
  const unsigned long long diff = all_and ^ all_or;
  int hi = diff ? 64 - __clzll((long long)diff) : 0;  // one past the top differing bit
  unsigned long long mask = (hi >= 64) ? 0ull : ~((1ull << hi) - 1);
  unsigned long long prefix = all_and & mask;
  int need = k;
#pragma unroll 1
  for (int pass = 0; hi > 0; ++pass) {
    const int shift = hi > 8 ? hi - 8 : 0;
    const unsigned long long dmask = (1ull << (hi - shift)) - 1;
    unsigned int* H = hist + 256 * (pass & 1);
    unsigned int* Hn = hist + 256 * ((pass + 1) & 1);
#pragma unroll 1
    for (int base = 0; base < N; base += NT) {
      const int i = base + tid;
      unsigned int bin = 256u;
      if (i < N) {
        const unsigned long long key = keys[i];
        if ((key & mask) == prefix) bin = (unsigned)((key >> shift) & dmask);
      }
      const unsigned int peers = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && lane == __ffs(peers) - 1) atomicAdd(&H[bin], (unsigned)__popc(peers));
    }
    bar();
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
      if (lane == __ffs(ball) - 1) {
        unsigned int above = excl;
        int digit = 0;
        unsigned int inbin = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above + c[i] >= (unsigned)need) {
            digit = 255 - 8 * lane - i;
            inbin = c[i];
            break;
          }
          above += c[i];
        }
        sh_u64[0] = prefix | (static_cast<unsigned long long>(digit) << shift);
        sh_u64[1] = mask | (dmask << shift);
        sh_int[0] = need - (int)above;
        sh_int[1] = (inbin <= (unsigned)NT || shift == 0) ? 1 : 0;
      }
    } else {
#pragma unroll 1
      for (int i = tid - 32; i < 256; i += NT - 32) Hn[i] = 0u;
    }
    bar();
    prefix = sh_u64[0];
    mask = sh_u64[1];
    need = sh_int[0];
    if (sh_int[1]) break;
    hi = shift;
  }
  // keys above the boundary bin are chosen; the bin's keys go to bkey/bidx
  const unsigned int lt = (1u << lane) - 1u;
#pragma unroll 1
  for (int base = 0; base < N; base += NT) {
    const int i = base + tid;
    unsigned long long key = 0ull, m = 0ull;
    if (i < N) {
      key = keys[i];
      m = key & mask;
    }
    const bool up = i < N && m > prefix, eq = i < N && m == prefix;
    const unsigned int bu = __ballot_sync(0xffffffffu, up);
    const unsigned int be = __ballot_sync(0xffffffffu, eq);
    int ou = 0, oe = 0;
    if (lane == 0) {
      if (bu) ou = atomicAdd(&sh_int[2], __popc(bu));
      if (be) oe = atomicAdd(&sh_int[3], __popc(be));
    }
    ou = __shfl_sync(0xffffffffu, ou, 0);
    oe = __shfl_sync(0xffffffffu, oe, 0);
    if (up) idx_out[ou + __popc(bu & lt)] = i;
    if (eq) {
      const int pos = oe + __popc(be & lt);
      if (pos < NT) {
        bkey[pos] = key;
        bidx[pos] = i;
      }
    }
  }
  bar();
  const int taken = sh_int[2], nb = min(sh_int[3], NT);
  if (tid < nb) {
    const unsigned long long key = bkey[tid];
    int r = 0;
#pragma unroll 4
    for (int s = 0; s < nb; ++s) r += bkey[s] > key ? 1 : 0;
    if (r < need && taken + r < k) idx_out[taken + r] = bidx[tid];
  }
  bar();
}


// Linear scoring (Max, Mean, Quest): each warp scores 8/NV blocks at a time;
// a lane holds NV 16-byte vectors of each block, and every load of the group is
// issued before any arithmetic.  V = 16-byte vectors per block and unit.
//
// reps: the representative pool; R rows of 128 per (page, KV head); P pages.
template <int NV, bool F32, int WARPS, bool PIPE = false>
__device__ __forceinline__ void score_linear(const void* reps, int P, int H_kv, int R, int g0,
                                             int js, int je, const int* pg, const float* wts,
                                             int V, unsigned long long* keys, int warp, int lane,
                                             int* status) {
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
  const size_t head_bytes = (size_t)R * D * (F32 ? 4 : 2);
  // PIPE: the next group's loads are in flight while the current group is
  // reduced (twice the registers)
  auto load = [&](int j0, uint4 (&x)[GB][NV], int (&page)[GB]) {
#pragma unroll
    for (int bi = 0; bi < GB; ++bi) {
      const int j = j0 + bi;
      page[bi] = (j < je) ? pg[j - js] : -1;
      const bool ok = page[bi] >= 0 && page[bi] < P;
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(reps) +
          ((size_t)(ok ? page[bi] : 0) * H_kv + g0) * head_bytes);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int vec = lane + 32 * v;
        x[bi][v] = (ok && vec < V) ? __ldg(src + vec) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  auto reduce = [&](int j0, const uint4 (&x)[GB][NV], const int (&page)[GB]) {
    float acc[GB];
#pragma unroll
    for (int bi = 0; bi < GB; ++bi) acc[bi] = lane_dot<NV, F32>(w, x[bi]);
    warp_sum_n(acc);
    if (lane == 0) {
#pragma unroll
      for (int bi = 0; bi < GB; ++bi) {
        const int j = j0 + bi;
        if (j < je) {
          const bool ok = page[bi] >= 0 && page[bi] < P;
          keys[j - js] = make_key(ok ? acc[bi] : -INFINITY, j);
          if (!ok) set_status(status, KT_ERR_DEVICE_CHECK);
        }
      }
    }
  };
  if constexpr (PIPE) {
    int j0 = js + warp * GB;
    if (j0 >= je) return;
    uint4 x[GB][NV];
    int page[GB];
    load(j0, x, page);
#pragma unroll 1
    for (; j0 < je; j0 += WARPS * GB) {
      uint4 xn[GB][NV];
      int pn[GB];
      const int jn = j0 + WARPS * GB;
      if (jn < je) load(jn, xn, pn);
      reduce(j0, x, page);
      if (jn < je) {
#pragma unroll
        for (int bi = 0; bi < GB; ++bi) {
          page[bi] = pn[bi];
#pragma unroll
          for (int v = 0; v < NV; ++v) x[bi][v] = xn[bi][v];
        }
      }
    }
  } else {
#pragma unroll 1
    for (int j0 = js + warp * GB; j0 < je; j0 += WARPS * GB) {
      uint4 x[GB][NV];
      int page[GB];
      load(j0, x, page);
      reduce(j0, x, page);
    }
  }
}

// score_linear over representatives already in shared memory: block i of
// the group (i < nblk) has its V 16-byte vectors at sbuf + i*sstride; its key goes to
// keys[i] with block id j0 + i, its page (for the range check) is pg[i].
// Same lane-to-vector mapping and summation order as score_linear, so the
// keys are identical.
template <int NV, bool F32, int WARPS>
__device__ __forceinline__ void score_linear_smem(const uint4* sbuf, int sstride, int nblk, int j0, int P,
                                                  const int* pg, const float* wts, int V,
                                                  unsigned long long* keys, int warp, int lane,
                                                  int* status) {
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
#pragma unroll 1
  for (int i0 = warp * GB; i0 < nblk; i0 += WARPS * GB) {
    uint4 x[GB][NV];
#pragma unroll
    for (int bi = 0; bi < GB; ++bi) {
      const int i = i0 + bi;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int vec = lane + 32 * v;
        x[bi][v] = (i < nblk && vec < V) ? sbuf[(size_t)i * sstride + vec] : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float acc[GB];
#pragma unroll
    for (int bi = 0; bi < GB; ++bi) acc[bi] = lane_dot<NV, F32>(w, x[bi]);
    warp_sum_n(acc);
    if (lane == 0) {
#pragma unroll
      for (int bi = 0; bi < GB; ++bi) {
        const int i = i0 + bi;
        if (i < nblk) {
          const bool ok = pg[i] >= 0 && pg[i] < P;
          keys[i] = make_key(ok ? acc[bi] : -INFINITY, j0 + i);
          if (!ok) set_status(status, KT_ERR_DEVICE_CHECK);
        }
      }
    }
  }
}

// Linear scoring of a few staged fp16 blocks on the CUDA cores, one 16-byte
// column of the blocks' rows per thread, so the weights are read once per CTA
// rather than once per warp.  V (64, 128 or 256) columns per block; phase
// s = tid / V of S = 32 WARPS / V takes blocks s, s + S, ... (nblk <= 8 S).
// Each thread forms its (up to) 8 block partials, a halving butterfly over
// lane bits 4, 3, 2 leaves block slot (lane >> 2) in every lane, then lanes 2
// and 1 are folded and the phase's warps added in warp order through
// red[WARPS * 8].  All WARPS warps call it (bar syncs them).  keys[i] receives
// block i's key with block id j0 + i.
template <int V, int WARPS, class Bar>
__device__ __forceinline__ void score_linear_cols(const uint4* sbuf, int sstride, int nblk, int j0,
                                                  int P, const int* pg, const float* wts,
                                                  unsigned long long* keys, float* red, int warp,
                                                  int lane, int* status, Bar bar) {
  static_assert(V == 64 || V == 128 || V == 256, "columns per block");
  constexpr int S = WARPS * 32 / V, WP = V / 32;
  const int tid = warp * 32 + lane;
  const int s = tid / V, c = tid % V;
  float w[8];
  {
    const float4 f0 = *reinterpret_cast<const float4*>(wts + c * 8);
    const float4 f1 = *reinterpret_cast<const float4*>(wts + c * 8 + 4);
    w[0] = f0.x; w[1] = f0.y; w[2] = f0.z; w[3] = f0.w;
    w[4] = f1.x; w[5] = f1.y; w[6] = f1.z; w[7] = f1.w;
  }
  uint4 x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = s + S * k;
    x[k] = i < nblk ? sbuf[(size_t)i * sstride + c] : make_uint4(0u, 0u, 0u, 0u);
  }
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const __half2* h = reinterpret_cast<const __half2*>(&x[k]);
    float e = 0.0f, o = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; q += 2) {
      const float2 f = __half22float2(h[q]), g = __half22float2(h[q + 1]);
      e = fmaf(w[2 * q], f.x, e);
      o = fmaf(w[2 * q + 1], f.y, o);
      e = fmaf(w[2 * q + 2], g.x, e);
      o = fmaf(w[2 * q + 3], g.y, o);
    }
    a[k] = e + o;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const bool up = lane & 16;
    const float send = up ? a[k] : a[k + 4], keep = up ? a[k + 4] : a[k];
    a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const bool up = lane & 8;
    const float send = up ? a[k] : a[k + 2], keep = up ? a[k + 2] : a[k];
    a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const bool up = lane & 4;
    const float send = up ? a[0] : a[1], keep = up ? a[1] : a[0];
    a[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  a[0] += __shfl_xor_sync(0xffffffffu, a[0], 2);
  a[0] += __shfl_xor_sync(0xffffffffu, a[0], 1);
  if ((lane & 3) == 0) red[warp * 8 + (lane >> 2)] = a[0];
  bar();
  if (tid < nblk) {
    const int ss = tid % S, k = tid / S;
    float v[WP];
#pragma unroll
    for (int q = 0; q < WP; ++q) v[q] = red[(ss * WP + q) * 8 + k];
    float sc = v[0];
#pragma unroll
    for (int q = 1; q < WP; ++q) sc += v[q];
    const int pgi = pg[tid];
    const bool ok = pgi >= 0 && pgi < P;
    keys[tid] = make_key(ok ? sc : -INFINITY, j0 + tid);
    if (!ok) set_status(status, KT_ERR_DEVICE_CHECK);
  }
}

// In place, the fp32 weights wts[K] (K a multiple of 16, at most 2048) become
// the B fragments of score_mma_smem: the weights split into fp16 hi + lo parts
// as B columns 0 (hi) and 1 (lo).  Fragment j of k-step ks, j = g * 4 + t
// (g = 0 hi, 1 lo), holds the fp16 pairs of k rows (2t, 2t + 1) and
// (2t + 8, 2t + 9) at ((uint2*)wts)[ks * 8 + j], i.e. in the same 64 bytes as
// the k-step's 16 weights: every thread reads before the barrier and writes
// after it.  All NT threads call it; on return the fragments are visible.
template <int NT, class Bar>
__device__ __forceinline__ void weights_to_frags(float* wts, int K, int tid, Bar bar) {
  constexpr int PER = 2048 / 2 / NT;  // fragments per thread at K = 2048
  uint2 v[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int e = tid + r * NT;
    const int ks = e >> 3, lo = (e >> 2) & 1, t = e & 3;
    v[r] = make_uint2(0u, 0u);
    if (e < K / 2) {
      const float2 wa = *reinterpret_cast<const float2*>(wts + ks * 16 + 2 * t);
      const float2 wb = *reinterpret_cast<const float2*>(wts + ks * 16 + 2 * t + 8);
      __half2 ha = __floats2half2_rn(wa.x, wa.y), hb = __floats2half2_rn(wb.x, wb.y);
      const __half2 la = __floats2half2_rn(wa.x - __low2float(ha), wa.y - __high2float(ha));
      const __half2 lb = __floats2half2_rn(wb.x - __low2float(hb), wb.y - __high2float(hb));
      if (lo) {
        ha = la;
        hb = lb;
      }
      v[r] = make_uint2(*reinterpret_cast<const uint32_t*>(&ha), *reinterpret_cast<const uint32_t*>(&hb));
    }
  }
  bar();
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int e = tid + r * NT;
    if (e < K / 2) reinterpret_cast<uint2*>(wts)[e] = v[r];
  }
  bar();
}

// Linear scoring of fp16 representatives on the tensor cores.  Blocks are
// staged in shared memory at a row stride of sb bytes (sbase, a shared-space
// address), K fp16 values each in the order of the weights.  The weights come
// as the B fragments of weights_to_frags (hi + lo fp16 parts as columns 0 and
// 1, the other columns zero), so one mma.sync m16n8k16 step reduces 16 blocks
// x 16 values into two fp32 partial sums per block; the score is their sum.
// Products of fp16 values are exact in fp32, and hi + lo carries the weight
// to about 2^-22.  Each 16-row group accumulates its k-steps in two chains
// (even, odd); every operand load is unconditional (k-steps clamped, masked
// after), so a warp keeps eight A and B fragments in flight.  With many groups
// each warp takes whole groups (w, w + WARPS, ...); with few, each group's K
// range is split over WARPS / groups warps and the partial sums are added
// through red[WARPS * 16] in warp order.  All WARPS warps call it (bar syncs
// them).  keys[i] receives block i's key with block id j0 + i.
template <int WARPS, class Bar>
__device__ __forceinline__ void score_mma_smem(uint32_t sbase, int sb, int nblk, int j0, int P,
                                               const int* pg, const uint2* wf, int K,
                                               unsigned long long* keys, float* red, int warp,
                                               int lane, int* status, Bar bar) {
  const int ngrp = (nblk + 15) >> 4;
  const int g = lane >> 2, t = lane & 3;
  const bool bcol = g < 2;  // lanes holding B columns 0 and 1
  const uint32_t koff = (uint32_t)((lane >> 4) * 16);  // bytes: k offset 0 or 8
  const int nks = K / 16;
  bool bad = false;
  auto emit = [&](int i, float score) {
    const int pgi = pg[i];
    const bool ok = pgi >= 0 && pgi < P;
    keys[i] = make_key(ok ? score : -INFINITY, j0 + i);
    bad |= !ok;
  };
  // acc (chains 0 and 1) += the 16 rows at ra x k-steps [k0, k1)
  auto run = [&](uint32_t ra, int k0, int k1, float (&acc)[2][4]) {
#pragma unroll 1
    for (int ks0 = k0; ks0 < k1; ks0 += 8) {
      uint32_t a[8][4];
      uint2 b[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int ks = min(ks0 + kk, k1 - 1);
        ldsm_x4(a[kk][0], a[kk][1], a[kk][2], a[kk][3], ra + (uint32_t)ks * 32u);
        const uint2 f = wf[ks * 8 + (lane & 7)];
        const bool on = bcol && ks0 + kk < k1;
        b[kk] = on ? f : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_16816_sched(acc[kk & 1], a[kk][0], a[kk][1], a[kk][2], a[kk][3], b[kk].x, b[kk].y);
    }
  };
  if (ngrp * 2 <= WARPS) {
    // split K: warp w -> group w / ns, k-steps part w % ns of ns
    const int ns = WARPS / ngrp;
    const int grp = warp / ns, part = warp % ns;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (grp < ngrp) {
      const int row = min(grp * 16 + (lane & 15), nblk - 1);
      run(sbase + (uint32_t)row * (uint32_t)sb + koff, part * nks / ns, (part + 1) * nks / ns, acc);
    }
    if (t == 0) {
      red[warp * 16 + g] = (acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1]);
      red[warp * 16 + g + 8] = (acc[0][2] + acc[0][3]) + (acc[1][2] + acc[1][3]);
    }
    bar();
    const int tid = warp * 32 + lane;
    if (tid < nblk) {
      const int gi = tid >> 4, r = tid & 15;
      float sc = 0.0f;
      for (int q = 0; q < ns; ++q) sc += red[(gi * ns + q) * 16 + r];
      emit(tid, sc);
    }
  } else {
#pragma unroll 1
    for (int gb = warp; gb < ngrp; gb += WARPS) {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int row = min(gb * 16 + (lane & 15), nblk - 1);  // past the end: ignored
      run(sbase + (uint32_t)row * (uint32_t)sb + koff, 0, nks, acc);
      if (t == 0) {
        const int i0 = gb * 16 + g, i1 = i0 + 8;
        const float s0 = (acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1]);
        const float s1 = (acc[0][2] + acc[0][3]) + (acc[1][2] + acc[1][3]);
        if (i0 < nblk) emit(i0, s0);
        if (i1 < nblk) emit(i1, s1);
      }
    }
  }
  if (bad) set_status(status, KT_ERR_DEVICE_CHECK);
}

// Multi-representative scoring (Fix, Dynamic) on the tensor cores: the head
// score of query head h is max_r q_h . rep_r of its KV head, the unit score
// the sum over the unit's heads.  Blocks are staged at a row stride of sb
// bytes as [KV head gi][rep r][128] fp16 (nkv KV heads from q_unit's heads,
// G query heads each).  One mma.sync tile holds 16 blocks x one (gi, r) x the
// G query heads (columns; the fp16 queries are exact), so the max over r is
// elementwise and the sum over a KV head's queries a 4-lane reduction.  With
// many tiles each warp takes whole tiles; with few, the KV heads of a tile are
// split over WARPS / tiles warps and the partial sums are added through
// red[WARPS * 16] in warp order.  All WARPS warps call it (bar syncs them).
template <int WARPS, class Bar>
__device__ __forceinline__ void score_multi_mma_smem(uint32_t sbase, int sb, int nblk, int j0,
                                                     int P, const int* pg, const __half* q_unit,
                                                     int G, int nkv, int R,
                                                     unsigned long long* keys, float* red,
                                                     int warp, int lane, int* status, Bar bar) {
  const int ntile = (nblk + 15) >> 4;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t koff = (uint32_t)((lane >> 4) * 16);
  // sum over KV heads gi = gi0, gi0 + gstep, ... of the head scores of the
  // tile's rows g and g + 8 (every lane of a quad returns the same sums)
  auto tile_sum = [&](int tile, int gi0, int gstep, float& s_lo, float& s_hi) {
    s_lo = s_hi = 0.0f;
    const int row = min(tile * 16 + (lane & 15), nblk - 1);
    const uint32_t ra = sbase + (uint32_t)row * (uint32_t)sb + koff;
#pragma unroll 1
    for (int gi = gi0; gi < nkv; gi += gstep) {
      uint32_t bf[8][2];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        bf[ks][0] = bf[ks][1] = 0u;
        if (g < G) {
          const __half* qr = q_unit + (size_t)(gi * G + g) * D + ks * 16 + 2 * t;
          bf[ks][0] = __ldg(reinterpret_cast<const unsigned int*>(qr));
          bf[ks][1] = __ldg(reinterpret_cast<const unsigned int*>(qr + 8));
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int r = 0; r < R; ++r) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t rr = ra + (uint32_t)((gi * R + r) * D * 2);
        uint32_t a[8][4];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) ldsm_x4(a[ks][0], a[ks][1], a[ks][2], a[ks][3], rr + ks * 32);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_16816(c, a[ks][0], a[ks][1], a[ks][2], a[ks][3], bf[ks][0], bf[ks][1]);
#pragma unroll
        for (int e = 0; e < 4; ++e) mx[e] = fmaxf(mx[e], c[e]);
      }
      // columns >= G are zero; sum the 8 columns of rows g and g + 8
      float lo = mx[0] + mx[1], hi = mx[2] + mx[3];
      lo += __shfl_xor_sync(0xffffffffu, lo, 1);
      hi += __shfl_xor_sync(0xffffffffu, hi, 1);
      lo += __shfl_xor_sync(0xffffffffu, lo, 2);
      hi += __shfl_xor_sync(0xffffffffu, hi, 2);
      s_lo += lo;
      s_hi += hi;
    }
  };
  auto emit = [&](int i, float score) {
    const bool ok = pg[i] >= 0 && pg[i] < P;
    keys[i] = make_key(ok ? score : -INFINITY, j0 + i);
    if (!ok) set_status(status, KT_ERR_DEVICE_CHECK);
  };
  if (ntile * 2 <= WARPS && nkv > 1) {
    const int ns = min(WARPS / ntile, nkv);
    const int tile = warp / ns, part = warp % ns;
    float lo = 0.f, hi = 0.f;
    if (tile < ntile) tile_sum(tile, part, ns, lo, hi);
    if (t == 0) {
      red[warp * 16 + g] = lo;
      red[warp * 16 + g + 8] = hi;
    }
    bar();
    const int tid = warp * 32 + lane;
    if (tid < nblk) {
      const int ti = tid >> 4, rw = tid & 15;
      float sc = 0.0f;
      for (int q = 0; q < ns; ++q) sc += red[(ti * ns + q) * 16 + rw];
      emit(tid, sc);
    }
    return;
  }
#pragma unroll 1
  for (int tile = warp; tile < ntile; tile += WARPS) {
    float lo, hi;
    tile_sum(tile, 0, 1, lo, hi);
    if (t == 0) {
      if (tile * 16 + g < nblk) emit(tile * 16 + g, lo);
      if (tile * 16 + g + 8 < nblk) emit(tile * 16 + g + 8, hi);
    }
  }
}

}  // namespace selc
}  // namespace kt
