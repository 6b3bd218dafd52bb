// quant.cu — Q8_0 quantisation of the fp16 K/V pools.
//
// Each 128-channel row is stored as 4 groups of 32 channels: a binary16 scale
// and 32 signed 8-bit codes (the Q8_0 choice among the kv_type options of "How
// to Implement Long Context Inference (Up to 139K Tokens) with KTransformers",
// Step 1).  With amax the group's largest |x| in binary32, dd = amax / 127 and
// id = 1 / dd (0 when dd is 0), a code is round-half-away-from-zero(x * id),
// every operation rounded once in binary32, and the scale is dd rounded to
// binary16.  The codes are therefore exact: any binary32 implementation of
// the same steps gets the same bytes.
#include "kt_internal.cuh"

namespace kt {
namespace {

constexpr int QT = 256;  // threads; one CTA per (page, KV head) slab of K or V

__global__ void __launch_bounds__(QT) quant_kernel(QuantLaunch a) {
  const int slab = blockIdx.x;  // (page - first_page) * H_kv + head
  const bool is_v = blockIdx.y != 0;
  const size_t row0 = ((size_t)a.first_page * a.H_kv + slab) * BS;
  const __half* src = (is_v ? a.v_pool : a.k_pool) + row0 * D;
  int8_t* code = (is_v ? a.v_code : a.k_code) + row0 * D;
  __half* scale = (is_v ? a.v_scale : a.k_scale) + row0 * (D / 32);
  // 128 rows x 4 groups, two groups a thread
#pragma unroll 1
  for (int gi = threadIdx.x; gi < BS * (D / 32); gi += QT) {
    const int r = gi >> 2, g = gi & 3;
    const uint4* x4 = reinterpret_cast<const uint4*>(src + (size_t)r * D + g * 32);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(x4 + i);
    float x[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2* h2 = reinterpret_cast<const __half2*>(&v[i]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(h2[j]);
        x[i * 8 + 2 * j] = f.x;
        x[i * 8 + 2 * j + 1] = f.y;
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(x[j]));
    const float dd = __fdiv_rn(amax, 127.0f);
    const float id = dd != 0.0f ? __frcp_rn(dd) : 0.0f;
    uint32_t packed[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int c = (int)roundf(__fmul_rn(x[w * 4 + b], id));
        word |= (uint32_t)(uint8_t)(int8_t)c << (8 * b);
      }
      packed[w] = word;
    }
    uint4* dst = reinterpret_cast<uint4*>(code + (size_t)r * D + g * 32);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    scale[r * (D / 32) + g] = __float2half_rn(dd);
  }
}

}  // namespace

cudaError_t launch_quant(const QuantLaunch& a, cudaStream_t stream) {
  if (a.num_pages <= 0) return cudaSuccess;
  dim3 grid((unsigned)(a.num_pages * a.H_kv), 2);
  quant_kernel<<<grid, QT, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kt
