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

// Number of keys in a[0, n) greater than key; a is 16-byte aligned and n even.
// Eight loads in flight per iteration.
__device__ __forceinline__ int count_greater(const unsigned long long* a, int n,
                                             unsigned long long key) {
  int r0 = 0, r1 = 0;
  int m = 0;
#pragma unroll 1
  for (; m + 8 <= n; m += 8) {
    const ulonglong2 v0 = *reinterpret_cast<const ulonglong2*>(a + m);
    const ulonglong2 v1 = *reinterpret_cast<const ulonglong2*>(a + m + 2);
    const ulonglong2 v2 = *reinterpret_cast<const ulonglong2*>(a + m + 4);
    const ulonglong2 v3 = *reinterpret_cast<const ulonglong2*>(a + m + 6);
    r0 += (v0.x > key ? 1 : 0) + (v0.y > key ? 1 : 0) + (v1.x > key ? 1 : 0) + (v1.y > key ? 1 : 0);
    r1 += (v2.x > key ? 1 : 0) + (v2.y > key ? 1 : 0) + (v3.x > key ? 1 : 0) + (v3.y > key ? 1 : 0);
  }
#pragma unroll 1
  for (; m < n; m += 2) {
    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(a + m);
    r0 += (v.x > key ? 1 : 0) + (v.y > key ? 1 : 0);
  }
  return r0 + r1;
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

// The k largest of N distinct keys in shared memory (1 <= k < N, k <= NT),
// emitted in descending order as emit(rank, index).  One 8-bit digit
// histogram (just below the keys' common leading bits) finds the bin of the
// k-th largest key; the keys from that bin up are ranked exactly by counting.
// When more than NT keys reach that bin, select_top narrows first (k <= NT).
// Scratch: hist 256 bins; ck (16-byte aligned) / ci NT entries; idx k
// entries; sh_u64 2 + 2*NT/32; sh_int 4.  All NT threads call it.
template <int NT, class Bar, class Emit>
__device__ void topk_sorted(const unsigned long long* keys, int N, int k,
                            unsigned long long* ck, int* ci, int* idx, unsigned int* hist,
                            unsigned long long* sh_u64, int* sh_int, int tid, Bar bar,
                            Emit emit) {
  constexpr int WARPS = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  unsigned long long a = ~0ull, o = 0ull;
#pragma unroll 1
  for (int i = tid; i < N; i += NT) {
    a &= keys[i];
    o |= keys[i];
  }
#pragma unroll 1
  for (int i = tid; i < 256; i += NT) hist[i] = 0u;
#pragma unroll 1
  for (int i = tid; i < NT; i += NT) ck[i] = 0ull;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    a &= __shfl_xor_sync(0xffffffffu, a, d);
    o |= __shfl_xor_sync(0xffffffffu, o, d);
  }
  if (lane == 0) {
    sh_u64[2 + warp] = a;
    sh_u64[2 + WARPS + warp] = o;
  }
  if (tid == 0) sh_int[0] = 0;
  bar();
  unsigned long long all_and = ~0ull, all_or = 0ull;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) {
    all_and &= sh_u64[2 + w];
    all_or |= sh_u64[2 + WARPS + w];
  }
  const unsigned long long diff = all_and ^ all_or;
  const int hi = diff ? 64 - __clzll((long long)diff) : 0;
  const int shift = hi > 8 ? hi - 8 : 0;
  const unsigned long long pmask = hi >= 64 ? 0ull : ~((1ull << hi) - 1);
  const unsigned long long prefix = all_and & pmask;
#pragma unroll 1
  for (int base = 0; base < N; base += NT) {
    const int i = base + tid;
    unsigned int bin = 256u;
    if (i < N) bin = (unsigned)((keys[i] >> shift) & 255ull);
    const unsigned int peers = __match_any_sync(0xffffffffu, bin);
    if (bin < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
  }
  bar();
  if (warp == 0) {
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
    if (excl < (unsigned)k && (unsigned)k <= incl) {
      unsigned int above = excl;
      int digit = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        above += c[i];
        if (above >= (unsigned)k) {
          digit = 255 - 8 * lane - i;
          break;
        }
      }
      sh_u64[0] = prefix | (static_cast<unsigned long long>(digit) << shift);
    }
  }
  bar();
  const unsigned long long T = sh_u64[0];
  {
    const unsigned int lt = (1u << lane) - 1u;
#pragma unroll 1
    for (int base = 0; base < N; base += NT) {
      const int i = base + tid;
      const bool take = i < N && keys[i] >= T;
      const unsigned int bal = __ballot_sync(0xffffffffu, take);
      int off = 0;
      if (lane == 0 && bal) off = atomicAdd(&sh_int[0], __popc(bal));
      off = __shfl_sync(0xffffffffu, off, 0) + __popc(bal & lt);
      if (take && off < NT) {
        ck[off] = keys[i];
        ci[off] = i;
      }
    }
  }
  bar();
  const int M = sh_int[0];
  if (M <= NT) {
#pragma unroll 1
    for (int i = tid; i < M; i += NT) {
      const int r = count_greater(ck, (M + 1) & ~1, ck[i]);
      if (r < k) emit(r, ci[i]);
    }
  } else {
    select_top<NT>(keys, N, k, idx, ck, ci, hist, sh_u64, sh_int, tid, bar);
#pragma unroll 1
    for (int i = tid; i < NT; i += NT) ck[i] = i < k ? keys[idx[i]] : 0ull;
    bar();
#pragma unroll 1
    for (int i = tid; i < k; i += NT) emit(count_greater(ck, (k + 1) & ~1, ck[i]), idx[i]);
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

// Linear scoring of fp16 representatives on the tensor cores.  Blocks are
// staged in shared memory at a row stride of sb bytes (sbase, a shared-space
// address), K fp16 values each in the order of the fp32 weights wts[K].  The
// weights are split into fp16 hi + lo parts, which form columns 0 and 1 of the
// B operand (the other columns are zero), so one mma.sync m16n8k16 step
// reduces 16 blocks x 16 values into two fp32 partial sums per block; the
// score is their sum.  Products of fp16 values are exact in fp32, and hi + lo
// carries the weight to about 2^-22.  With many 16-block groups each warp
// takes whole groups (w, w + WARPS, ...); with few, each group's K range is
// split over WARPS / groups warps and the partial sums are added through
// red[WARPS * 16] in warp order.  All WARPS warps call it (bar syncs them).
// keys[i] receives block i's key with block id j0 + i.
template <int WARPS, class Bar>
__device__ __forceinline__ void score_mma_smem(uint32_t sbase, int sb, int nblk, int j0, int P,
                                               const int* pg, const float* wts, int K,
                                               unsigned long long* keys, float* red, int warp,
                                               int lane, int* status, Bar bar) {
  constexpr int MAXG = 4;  // groups per warp per pass
  constexpr int KC = 16;   // k-steps whose weight fragments are held in registers
  const int ngrp = (nblk + 15) >> 4;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t koff = (uint32_t)((lane >> 4) * 16);  // bytes: k offset 0 or 8
  const int nks = K / 16;
  // weight fragments of k-steps ks0 .. ks0+kn-1 (kn <= KC): column 0 hi, 1 lo
  auto build = [&](int ks0, int kn, uint32_t (&bf)[KC][2]) {
#pragma unroll
    for (int kk = 0; kk < KC; ++kk) {
      bf[kk][0] = bf[kk][1] = 0u;
      if (kk < kn && g < 2) {
        const int ks = ks0 + kk;
        const float2 wa = *reinterpret_cast<const float2*>(wts + ks * 16 + 2 * t);
        const float2 wb = *reinterpret_cast<const float2*>(wts + ks * 16 + 2 * t + 8);
        __half2 ha = __floats2half2_rn(wa.x, wa.y), hb = __floats2half2_rn(wb.x, wb.y);
        if (g == 1) {
          ha = __floats2half2_rn(wa.x - __low2float(ha), wa.y - __high2float(ha));
          hb = __floats2half2_rn(wb.x - __low2float(hb), wb.y - __high2float(hb));
        }
        bf[kk][0] = *reinterpret_cast<uint32_t*>(&ha);
        bf[kk][1] = *reinterpret_cast<uint32_t*>(&hb);
      }
    }
  };
  // acc += rows of ra (16 blocks) x weights over k-steps ks0 .. ks0+kn-1,
  // eight A fragments in flight at a time
  auto run = [&](uint32_t ra, int ks0, int kn, const uint32_t (&bf)[KC][2], float (&acc)[4]) {
#pragma unroll
    for (int h = 0; h < KC; h += 8) {
      uint32_t a[8][4];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (h + kk < kn) ldsm_x4(a[kk][0], a[kk][1], a[kk][2], a[kk][3], ra + (uint32_t)(ks0 + h + kk) * 32u);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (h + kk < kn)
          mma_16816(acc, a[kk][0], a[kk][1], a[kk][2], a[kk][3], bf[h + kk][0], bf[h + kk][1]);
    }
  };
  auto emit = [&](int i, float score) {
    const bool ok = pg[i] >= 0 && pg[i] < P;
    keys[i] = make_key(ok ? score : -INFINITY, j0 + i);
    if (!ok) set_status(status, KT_ERR_DEVICE_CHECK);
  };
  if (ngrp * 2 <= WARPS) {
    // split K: warp w -> group w / ns, k-steps part w % ns of ns
    const int ns = WARPS / ngrp;
    const int grp = warp / ns, part = warp % ns;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (grp < ngrp) {
      const int row = min(grp * 16 + (lane & 15), nblk - 1);
      const uint32_t ra = sbase + (uint32_t)row * (uint32_t)sb + koff;
      const int k0 = part * nks / ns, k1 = (part + 1) * nks / ns;
#pragma unroll 1
      for (int ks0 = k0; ks0 < k1; ks0 += KC) {
        uint32_t bf[KC][2];
        const int kn = min(KC, k1 - ks0);
        build(ks0, kn, bf);
        run(ra, ks0, kn, bf, acc);
      }
    }
    if (t == 0) {
      red[warp * 16 + g] = acc[0] + acc[1];
      red[warp * 16 + g + 8] = acc[2] + acc[3];
    }
    bar();
    const int tid = warp * 32 + lane;
    if (tid < nblk) {
      const int gi = tid >> 4, r = tid & 15;
      float sc = 0.0f;
      for (int q = 0; q < ns; ++q) sc += red[(gi * ns + q) * 16 + r];
      emit(tid, sc);
    }
    return;
  }
#pragma unroll 1
  for (int gb = warp; gb < ngrp; gb += WARPS * MAXG) {
    float acc[MAXG][4];
    uint32_t rowaddr[MAXG];
#pragma unroll
    for (int m = 0; m < MAXG; ++m) {
      acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.0f;
      const int row = min((gb + m * WARPS) * 16 + (lane & 15), nblk - 1);  // past the end: ignored
      rowaddr[m] = sbase + (uint32_t)row * (uint32_t)sb + koff;
    }
#pragma unroll 1
    for (int ks0 = 0; ks0 < nks; ks0 += KC) {
      uint32_t bf[KC][2];
      const int kn = min(KC, nks - ks0);
      build(ks0, kn, bf);
#pragma unroll
      for (int m = 0; m < MAXG; ++m)
        if (gb + m * WARPS < ngrp) run(rowaddr[m], ks0, kn, bf, acc[m]);
    }
    if (t == 0) {
#pragma unroll
      for (int m = 0; m < MAXG; ++m) {
        const int grp = gb + m * WARPS;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = grp * 16 + g + 8 * h;
          if (grp < ngrp && i < nblk) emit(i, acc[m][2 * h] + acc[m][2 * h + 1]);
        }
      }
    }
  }
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
