// preselect.cu — preselection of Context blocks from the local queries
// (article "KTransformers 长上下文稀疏注意力实战…", §4.4 "预选择 Preselect" and
// §4.6 preselect_block(): SnapKV-style votes, pooled, then the blocks of the
// best tokens).
//
// Inputs are the accumulated softmax probabilities of every token over the
// local query rows of each KV head (the Dynamic token scores, produced by the
// Dynamic passes into the workspace).  For a selection unit (a sequence and,
// in SEPARATE mode, one KV head) the vote of a Context token is the sum of
// those scores over the unit's KV heads; votes are average-pooled along the
// Context tokens (window kernel_size, zero padding of kernel_size/2, stride 1);
// a block's score is the largest pooled vote of its tokens, and the `count`
// best blocks (score descending, then block ascending) are preselected:
// taking tokens in descending pooled vote reaches each block at its largest
// one, so these are the blocks of the best tokens.  Output: one bit per
// block in a per-unit mask, and the number of preselected blocks.
#include "select_common.cuh"

namespace kt {
namespace {

constexpr int PS_THREADS = 256;
constexpr int PS_WARPS = PS_THREADS / 32;
constexpr int PS_MAX_HALF = 32;  // kernel_size <= 65

struct PreselParams {
  const float* votes;  // [B][H_kv][max_blocks * 128] token scores
  const int32_t* seq_lens;
  float* bscore;       // [B][SEL][max_blocks] score of Context block c0 + i at i
  uint32_t* mask;      // [B][SEL][mask_words]
  int32_t* cnt;        // [B][SEL]
  int* status;
  int B, H_kv, SEL, max_blocks, I_b, L_b, kernel, count, mask_words;
};

__device__ __forceinline__ void context_range(const PreselParams& p, int b, int& c0, int& c1) {
  int n = __ldg(p.seq_lens + b);
  if (n < 0 || n > p.max_blocks * BS) {
    set_status(p.status, KT_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : p.max_blocks * BS;
  }
  const int nb = (n + BS - 1) / BS;
  c0 = min(p.I_b, nb);
  c1 = max(c0, nb - p.L_b);
}

// Grid (block groups, SEL, B): warp w of CTA x scores Context blocks
// i = (x * PS_WARPS + w), + gridDim.x * PS_WARPS, ...  Lane l pools tokens
// 4l .. 4l+3 of the block from a shared copy of its votes and halo.
__global__ void __launch_bounds__(PS_THREADS) presel_score_kernel(const __grid_constant__ PreselParams p) {
  __shared__ float win[PS_WARPS][BS + 2 * PS_MAX_HALF];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.y, b = blockIdx.z;
  int c0, c1;
  context_range(p, b, c0, c1);
  const int C = c1 - c0, ntok = C * BS, half = p.kernel / 2;
  const int h0 = p.SEL == 1 ? 0 : u, h1 = p.SEL == 1 ? p.H_kv : u + 1;
  float* w = win[warp];
  for (int i = blockIdx.x * PS_WARPS + warp; i < C; i += gridDim.x * PS_WARPS) {
    // votes of Context tokens i*128 - half .. i*128 + 127 + half (0 outside)
    for (int e = lane; e < BS + 2 * half; e += 32) {
      const int v = i * BS - half + e;
      float s = 0.0f;
      if (v >= 0 && v < ntok)
        for (int h = h0; h < h1; ++h)
          s += __ldg(p.votes + ((size_t)b * p.H_kv + h) * p.max_blocks * BS + (size_t)c0 * BS + v);
      w[e] = s;
    }
    __syncwarp();
    float best = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t = lane * 4 + q;  // token t of the block: window w[t .. t + 2*half]
      float s = 0.0f;
      for (int e = 0; e <= 2 * half; ++e) s += w[t + e];
      best = fmaxf(best, s / (float)p.kernel);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (lane == 0) p.bscore[((size_t)b * p.SEL + u) * p.max_blocks + i] = best;
    __syncwarp();
  }
}

// One CTA per (unit, sequence): the `count` best blocks by score, as mask bits.
__global__ void __launch_bounds__(PS_THREADS) presel_select_kernel(const __grid_constant__ PreselParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ unsigned int hist[512];
  __shared__ unsigned long long sh_u64[2 + 2 * PS_WARPS];
  __shared__ int sh_int[4];
  __shared__ unsigned long long bkey[PS_THREADS];
  __shared__ int bidx[PS_THREADS];
  const int tid = threadIdx.x;
  const int u = blockIdx.x, b = blockIdx.y;
  int c0, c1;
  context_range(p, b, c0, c1);
  const int C = c1 - c0, k = min(p.count, C);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
  uint32_t* mk = reinterpret_cast<uint32_t*>(keys + p.max_blocks);
  int* idx = reinterpret_cast<int*>(mk + p.mask_words);
  const float* sc = p.bscore + ((size_t)b * p.SEL + u) * p.max_blocks;
  for (int i = tid; i < C; i += PS_THREADS) keys[i] = selc::make_key(sc[i], c0 + i);
  for (int i = tid; i < p.mask_words; i += PS_THREADS) mk[i] = 0u;
  __syncthreads();
  auto bar = [] { __syncthreads(); };
  if (k > 0) {
    selc::select_top<PS_THREADS>(keys, C, k, idx, bkey, bidx, hist, sh_u64, sh_int, tid, bar);
    for (int i = tid; i < k; i += PS_THREADS) {
      const int j = c0 + idx[i];
      atomicOr(&mk[j >> 5], 1u << (j & 31));
    }
  }
  __syncthreads();
  uint32_t* dst = p.mask + ((size_t)b * p.SEL + u) * p.mask_words;
  for (int i = tid; i < p.mask_words; i += PS_THREADS) dst[i] = mk[i];
  if (tid == 0) p.cnt[b * p.SEL + u] = k;
}

}  // namespace

size_t preselect_ws_bytes(int B, int H_kv, int SEL, int max_blocks) {
  return align256((size_t)B * H_kv * max_blocks * BS * 4) +
         align256((size_t)B * SEL * max_blocks * 4);
}

size_t preselect_smem_bytes(int max_blocks, int mask_words) {
  return (size_t)max_blocks * 8 + (size_t)mask_words * 4 + (size_t)max_blocks * 4;
}

cudaError_t launch_preselect(const PreselLaunch& a, cudaStream_t stream) {
  PreselParams p;
  p.votes = a.votes;
  p.seq_lens = a.seq_lens;
  p.bscore = a.bscore;
  p.mask = a.mask;
  p.cnt = a.cnt;
  p.status = a.status;
  p.B = a.B;
  p.H_kv = a.H_kv;
  p.SEL = a.SEL;
  p.max_blocks = a.max_blocks;
  p.I_b = a.I_b;
  p.L_b = a.L_b;
  p.kernel = a.kernel;
  p.count = a.count;
  p.mask_words = a.mask_words;
  const int groups = (a.max_blocks + PS_WARPS * 4 - 1) / (PS_WARPS * 4);  // 4 blocks a warp
  presel_score_kernel<<<dim3(groups, a.SEL, a.B), PS_THREADS, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = preselect_smem_bytes(a.max_blocks, a.mask_words);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(presel_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
  }
  presel_select_kernel<<<dim3(a.SEL, a.B), PS_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kt
