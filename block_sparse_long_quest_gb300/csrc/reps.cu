// reps.cu — representative keys of full KV blocks (article "KTransformers
// 长上下文稀疏注意力实战…", §4.3 representative-token table; Quest §3.1).
//
//   Max    per-channel maximum                         1 fp16 row
//   Quest  per-channel minimum (row 0), maximum (row 1) 2 fp16 rows
//   Mean   per-channel mean, exact, rounded once        1 fp32 row
//   Fix    key rows at offsets 0, s, 2s, ...            128/s fp16 rows
//
// One CTA per (logical block, sequence); one warp per KV head slab of
// 128 x 128 fp16 (32 KB, contiguous).  A half-warp covers one 256-byte row, so
// every load is a coalesced 16-byte vector; 8 loads per lane are in flight.
//
// Max/min are exact: each binary16 pattern is mapped to a signed 16-bit key
// that orders like the binary16 total order (-0 < +0), and __vmaxs2/__vmins2
// compare two keys per 32-bit word.  Mean is exact: every binary16 value is an
// integer multiple of 2^-24 below 2^16, so the 128-token sum is accumulated as
// a 64-bit integer (< 2^47), converted once with round-to-nearest-even and
// scaled by 2^-31 (= 2^-24 / 128), which is exact.
#include "kt_internal.cuh"

namespace kt {
namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;

struct Params {
  const __half* k_pool;
  const int32_t* table;
  const int32_t* seq_lens;
  void* reps;
  int B, H_kv, max_blocks, P, rep, R, fix_stride, first_block;
};

// binary16 bits (two per word) -> keys ordered as signed 16-bit integers; the
// map flips the 15 magnitude bits of negative values and is its own inverse.
__device__ __forceinline__ uint32_t order_key2(uint32_t w) {
  return w ^ (((w >> 15) & 0x00010001u) * 0x7FFFu);
}

// binary16 bits -> value * 2^24 as an exact integer.
__device__ __forceinline__ long long f16_fixed(uint32_t h) {
  const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
  const long long mag = e ? ((long long)(m | 1024u) << (e - 1)) : (long long)m;
  return (h & 0x8000u) ? -mag : mag;
}

// first_block < 0: per sequence, the block that ends at its current length
// (the block the last appended token completed), if any.
__global__ void __launch_bounds__(THREADS) reps_kernel(const __grid_constant__ Params p) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.seq_lens[b];
  const int j = p.first_block >= 0 ? p.first_block + (int)blockIdx.x
                                   : (n > 0 && n % BS == 0 ? n / BS - 1 : -1);
  if (j < 0 || j >= p.max_blocks || (long long)(j + 1) * BS > n) return;  // full blocks only
  const int page = p.table[(size_t)b * p.max_blocks + j];
  if (page < 0 || page >= p.P) return;
  const int hw = lane >> 4, col = lane & 15;  // half-warp hw reads rows hw, hw+2, ...

  for (int h = warp; h < p.H_kv; h += WARPS) {
    const uint4* slab =
        reinterpret_cast<const uint4*>(p.k_pool + ((size_t)page * p.H_kv + h) * BS * D);
    const size_t rep_row0 = ((size_t)page * p.H_kv + h) * p.R;  // first rep row index
    if (p.rep == KT_REP_MAX || p.rep == KT_REP_QUEST) {
      uint32_t mx[4], mn[4];
      {
        const uint4 v = __ldg(slab + hw * 16 + col);
        mx[0] = mn[0] = order_key2(v.x);
        mx[1] = mn[1] = order_key2(v.y);
        mx[2] = mn[2] = order_key2(v.z);
        mx[3] = mn[3] = order_key2(v.w);
      }
#pragma unroll 8
      for (int t = hw + 2; t < BS; t += 2) {
        const uint4 v = __ldg(slab + t * 16 + col);
        const uint32_t k0 = order_key2(v.x), k1 = order_key2(v.y), k2 = order_key2(v.z),
                       k3 = order_key2(v.w);
        mx[0] = __vmaxs2(mx[0], k0);
        mx[1] = __vmaxs2(mx[1], k1);
        mx[2] = __vmaxs2(mx[2], k2);
        mx[3] = __vmaxs2(mx[3], k3);
        mn[0] = __vmins2(mn[0], k0);
        mn[1] = __vmins2(mn[1], k1);
        mn[2] = __vmins2(mn[2], k2);
        mn[3] = __vmins2(mn[3], k3);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mx[i] = __vmaxs2(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 16));
        mn[i] = __vmins2(mn[i], __shfl_xor_sync(0xffffffffu, mn[i], 16));
      }
      if (hw == 0) {
        uint4* out = reinterpret_cast<uint4*>(static_cast<__half*>(p.reps) + rep_row0 * D);
        const uint4 vmax = make_uint4(order_key2(mx[0]), order_key2(mx[1]), order_key2(mx[2]),
                                      order_key2(mx[3]));
        if (p.rep == KT_REP_MAX) {
          out[col] = vmax;
        } else {
          out[col] = make_uint4(order_key2(mn[0]), order_key2(mn[1]), order_key2(mn[2]),
                                order_key2(mn[3]));
          out[16 + col] = vmax;
        }
      }
    } else if (p.rep == KT_REP_MEAN) {
      long long acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0;
#pragma unroll 4
      for (int t = hw; t < BS; t += 2) {
        const uint4 v = __ldg(slab + t * 16 + col);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] += f16_fixed(w[i] & 0xFFFFu);
          acc[2 * i + 1] += f16_fixed(w[i] >> 16);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const long long o = __shfl_xor_sync(0xffffffffu, acc[i], 16);
        acc[i] += o;
      }
      if (hw == 0) {
        float4* out = reinterpret_cast<float4*>(static_cast<float*>(p.reps) + rep_row0 * D);
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __ll2float_rn(acc[i]) * 0x1.0p-31f;
        out[2 * col] = make_float4(f[0], f[1], f[2], f[3]);
        out[2 * col + 1] = make_float4(f[4], f[5], f[6], f[7]);
      }
    } else {  // KT_REP_FIX
      uint4* out = reinterpret_cast<uint4*>(static_cast<__half*>(p.reps) + rep_row0 * D);
      for (int r = hw; r < p.R; r += 2) out[r * 16 + col] = __ldg(slab + r * p.fix_stride * 16 + col);
    }
  }
}

struct AppendParams {
  const uint4* k_new;  // [B][H_kv][16] (128 fp16 per head)
  const uint4* v_new;
  uint4* k_pool;       // [P][H_kv][128][16]
  uint4* v_pool;
  const int32_t* table;
  int32_t* seq_lens;
  int* status;
  int H_kv, max_blocks, P;
};

// One decoded token per sequence (CTA b): the K and V rows of every KV head
// go to row n % 128 of the page of block n / 128, then n becomes n + 1.
__global__ void __launch_bounds__(THREADS) append_kernel(const __grid_constant__ AppendParams p) {
  const int b = blockIdx.x;
  const int n = p.seq_lens[b];
  const int j = n / BS;
  int page = -1;
  if (n >= 0 && j < p.max_blocks) page = p.table[(size_t)b * p.max_blocks + j];
  if (page < 0 || page >= p.P) {  // no room in the table, or a page outside the pool
    if (threadIdx.x == 0) set_status(p.status, KT_ERR_DEVICE_CHECK);
    return;
  }
  const int per = p.H_kv * (D / 8);  // 16-byte chunks of one token's rows
  for (int i = threadIdx.x; i < 2 * per; i += THREADS) {
    const int r = i % per, h = r / (D / 8), c = r % (D / 8);
    const uint4* src = (i < per ? p.k_new : p.v_new) + ((size_t)b * p.H_kv + h) * (D / 8) + c;
    uint4* dst = (i < per ? p.k_pool : p.v_pool) +
                 (((size_t)page * p.H_kv + h) * BS + n % BS) * (D / 8) + c;
    *dst = *src;
  }
  __syncthreads();  // every thread has read seq_lens[b]
  if (threadIdx.x == 0) p.seq_lens[b] = n + 1;
}

__global__ void selftest_wait_kernel(int* status, int spin_limit) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nobody arrives on this barrier: every poll fails until the limit.
    bool done = false;
    for (int i = 0; i < spin_limit && !done; ++i) done = mbar_try_wait(a, 0);
    if (!done) set_status(status, KT_ERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_reps(const RepsLaunch& a, cudaStream_t stream) {
  Params p;
  p.k_pool = a.k_pool;
  p.table = a.table;
  p.seq_lens = a.seq_lens;
  p.reps = a.reps;
  p.B = a.B;
  p.H_kv = a.H_kv;
  p.max_blocks = a.max_blocks;
  p.P = a.P;
  p.rep = a.rep;
  p.R = a.R;
  p.fix_stride = a.fix_stride;
  p.first_block = a.first_block;
  if (a.num_blocks <= 0) return cudaSuccess;
  const dim3 grid(a.num_blocks, a.B);
  reps_kernel<<<grid, THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream) {
  AppendParams p;
  p.k_new = static_cast<const uint4*>(a.k_new);
  p.v_new = static_cast<const uint4*>(a.v_new);
  p.k_pool = static_cast<uint4*>(a.k_pool);
  p.v_pool = static_cast<uint4*>(a.v_pool);
  p.table = a.table;
  p.seq_lens = a.seq_lens;
  p.status = a.status;
  p.H_kv = a.H_kv;
  p.max_blocks = a.max_blocks;
  p.P = a.P;
  if (a.B <= 0) return cudaSuccess;
  append_kernel<<<a.B, THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int* status, int spin_limit, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, spin_limit);
  return cudaGetLastError();
}

}  // namespace kt
