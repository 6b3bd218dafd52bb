// dynamic.cu — Dynamic representative tokens (article "KTransformers 长上下文稀疏
// 注意力实战…", §4.3 "Dynamic": each token gets an accumulated attention score,
// and the top-k tokens of each block become its representatives; the score is
// softmax(q k^T / sqrt(d)) as in §3.2).
//
// For KV head h of sequence b, the rows are the last T query positions
// pos_i = n - T + i (i < T) times the G query heads of h (row r = i*G + g);
// position pos sees tokens 0..pos.  The accumulated score of token t is
//   acc[t] = sum over rows r with t <= pos_r of exp(s_rt - m_r) / l_r,
// where s_rt = q_r . k_t * scale, m_r = max_t s_rt and l_r = sum_t exp(s_rt - m_r)
// over the tokens row r sees.  Three launches:
//   pass 1   one CTA per (block slice, KV head, sequence): S = Q K^T for every
//            block of its slice (mma.sync m16n8k16, Q fragments held in
//            registers, K blocks by 2-D TMA into a double buffer); per block and
//            row, the partial max and sum (base 2) go to the workspace.
//   combine  per (split, KV head, sequence): merge the partials of a range of
//            blocks per row.
//   pass 2   the same S for the requested blocks; p = exp2(s - M_r) / L_r summed
//            over rows per token; the num_reps best tokens of each full block
//            (ties: lower index) are copied, in token order, as its reps.
// The path is a dense contraction (M = T*G rows per KV head) plus one exp per
// logit per pass; K is read twice (once per pass).
#include "kt_internal.cuh"

namespace kt {
namespace {

constexpr int THREADS = 256;  // 8 warps; warp w owns rows 32w .. 32w+31
constexpr int MAX_ROWS = 256;
constexpr int BOX_BYTES = BS * 64 * 2;  // 128 tokens x 64 channels
constexpr int KBUF_BYTES = 2 * BOX_BYTES;
constexpr int NSPLIT = 8;

struct DynParams {
  CUtensorMap kmap;
  const __half* k_pool;
  const __half* q_local;  // [B][T][H_q][128]
  const int32_t* table;
  const int32_t* seq_lens;
  float2* stats;    // [B][H_kv][max_blocks][MAX_ROWS] (m, l) per block, base 2
  float2* split;    // [B][H_kv][NSPLIT][MAX_ROWS] combined over a block range
  __half* reps;     // [P][H_kv][R][128]
  float* token_scores;  // nullable [B][H_kv][max_blocks*128]
  int* status;
  int B, H_kv, G, T, max_blocks, P, R, first_block, num_blocks, pass, nslices;
  float scale_log2;
};

__device__ __forceinline__ int seq_len_checked(const DynParams& p, int b) {
  int n = __ldg(p.seq_lens + b);
  if (n < 0 || n > p.max_blocks * BS) {
    set_status(p.status, KT_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : p.max_blocks * BS;
  }
  return n;
}

// One CTA: KV head h of sequence b, blocks j = j_begin, j_begin + stride, ...
__global__ void __launch_bounds__(THREADS, 1) dyn_pass_kernel(const __grid_constant__ DynParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned (128-byte swizzled TMA boxes); offsetting the array
  // itself keeps the accesses below in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ float colsum[8][BS];
  __shared__ float tscore[BS];
  __shared__ float rowM[MAX_ROWS], rowInvL[MAX_ROWS];
  __shared__ int pick[BS];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n = seq_len_checked(p, b);
  const int nb = (n + BS - 1) / BS;
  const int rows = p.T * p.G;
  const int H_q = p.H_kv * p.G;
  // blocks handled: pass 1 all blocks, pass 2 the requested range
  const int jb = p.pass == 1 ? 0 : min(p.first_block, nb);
  const int je = p.pass == 1 ? nb : min(nb, p.first_block + p.num_blocks);
  const uint32_t bar0 = smem_u32(&bars[0]);
  const uint32_t kbase = smem_u32(smem);

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_mbar_init();
    prefetch_tensormap(&p.kmap);
  }
  // final row statistics for pass 2: combine the NSPLIT split partials
  if (p.pass == 2) {
    for (int r = tid; r < MAX_ROWS; r += THREADS) {
      float M = -INFINITY, L = 0.0f;
      if (r < rows) {
        const float2* sp = p.split + ((size_t)(b * p.H_kv + h) * NSPLIT) * MAX_ROWS + r;
        for (int q = 0; q < NSPLIT; ++q) {
          const float2 v = sp[(size_t)q * MAX_ROWS];
          if (v.x == -INFINITY) continue;
          const float Mn = fmaxf(M, v.x);
          L = L * exp2f(M - Mn) + v.y * exp2f(v.x - Mn);
          M = Mn;
        }
      }
      rowM[r] = M;
      rowInvL[r] = L > 0.0f ? 1.0f / L : 0.0f;
    }
  }
  // query fragments of this warp's two m-tiles (rows 32w .. 32w+31), all 8 k-steps
  uint32_t qa[2][8][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = warp * 32 + mt * 16 + g + 8 * hr;
      const __half* qrow = nullptr;
      if (r < rows) {
        const int i = r / p.G, gg = r % p.G;
        qrow = p.q_local + (((size_t)b * p.T + i) * H_q + h * p.G + gg) * D;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[mt][kk][hr] = qrow ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * t)) : 0u;
        qa[mt][kk][2 + hr] =
            qrow ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * t)) : 0u;
      }
    }
  }
  // positions of the four rows this thread holds: [mt][hr]
  int pos[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = warp * 32 + mt * 16 + g + 8 * hr;
      pos[mt][hr] = r < rows ? n - p.T + r / p.G : -1;  // -1: row absent, sees nothing
    }
  __syncthreads();

  auto issue = [&](int j, int buf) {
    const int page = p.table[(size_t)b * p.max_blocks + j];
    const uint32_t bar = bar0 + 8 * buf;
    if (page < 0 || page >= p.P) {
      set_status(p.status, KT_ERR_DEVICE_CHECK);
      mbar_arrive(bar);
      return false;
    }
    const int row = (page * p.H_kv + h) * BS;
    mbar_arrive_expect_tx(bar, KBUF_BYTES);
    const uint64_t pol = l2_evict_first_policy();
    tma_load_2d(kbase + buf * KBUF_BYTES, &p.kmap, 0, row, bar, pol);
    tma_load_2d(kbase + buf * KBUF_BYTES + BOX_BYTES, &p.kmap, 64, row, bar, pol);
    return true;
  };

  const int stride = p.nslices;
  int it = 0;
  if (tid == 0 && jb + slice < je) issue(jb + slice, 0);
  for (int j = jb + slice; j < je; j += stride, ++it) {
    const int buf = it & 1;
    if (tid == 0 && j + stride < je) issue(j + stride, buf ^ 1);
    if (!mbar_wait(bar0 + 8 * buf, (it >> 1) & 1, p.status)) break;
    const int page = p.table[(size_t)b * p.max_blocks + j];
    const bool page_ok = page >= 0 && page < p.P;
    const uint32_t kb = kbase + buf * KBUF_BYTES;
    const int mi = lane >> 3, r8 = lane & 7;

    // ---- S for this warp's 32 rows x 128 tokens, in two halves of 64 tokens
    float rm[2][2] = {{-INFINITY, -INFINITY}, {-INFINITY, -INFINITY}};
    float rl[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    float cs[16][2];
#pragma unroll
    for (int i = 0; i < 16; ++i) cs[i][0] = cs[i][1] = 0.0f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float s[2][8][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[mt][nt][0] = s[mt][nt][1] = s[mt][nt][2] = s[mt][nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {  // pairs of 8-token n-tiles
          const int tok = half * 64 + np * 16 + (mi >> 1) * 8 + r8;
          const int chunk = kk * 2 + (mi & 1);
          const uint32_t addr = kb + (chunk >> 3) * BOX_BYTES + tok * 128 +
                                (((chunk & 7) ^ (tok & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3, addr);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            mma_16816(s[mt][2 * np], qa[mt][kk][0], qa[mt][kk][1], qa[mt][kk][2], qa[mt][kk][3],
                      b0, b1);
            mma_16816(s[mt][2 * np + 1], qa[mt][kk][0], qa[mt][kk][1], qa[mt][kk][2],
                      qa[mt][kk][3], b2, b3);
          }
        }
      }
      // ---- mask, scale; pass 1: row max / sum; pass 2: normalised column sums.
      // A block that ends before the first query position is seen whole by
      // every present row: only absent rows are masked there.
      if (page_ok && (j + 1) * BS - 1 <= n - p.T) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              s[mt][nt][e] = pos[mt][e >> 1] >= 0 ? s[mt][nt][e] * p.scale_log2 : -INFINITY;
      } else {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int hr = e >> 1;
              const int tok = j * BS + half * 64 + nt * 8 + 2 * t + (e & 1);
              const bool vis = page_ok && tok < n && tok <= pos[mt][hr];
              s[mt][nt][e] = vis ? s[mt][nt][e] * p.scale_log2 : -INFINITY;
            }
      }
      if (p.pass == 1) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
              mx = fmaxf(mx, fmaxf(s[mt][nt][2 * hr], s[mt][nt][2 * hr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float Mn = fmaxf(rm[mt][hr], mx);
            if (Mn == -INFINITY) continue;
            float sum = 0.0f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
              sum += exp2f(s[mt][nt][2 * hr] - Mn) + exp2f(s[mt][nt][2 * hr + 1] - Mn);
            rl[mt][hr] = rl[mt][hr] * exp2f(rm[mt][hr] - Mn) + sum;
            rm[mt][hr] = Mn;
          }
      } else {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int r = warp * 32 + mt * 16 + g + 8 * hr;
            const float M = rowM[r], iL = rowInvL[r];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
              const float a0 = s[mt][nt][2 * hr], a1 = s[mt][nt][2 * hr + 1];
              cs[half * 8 + nt][0] += (a0 == -INFINITY) ? 0.0f : exp2f(a0 - M) * iL;
              cs[half * 8 + nt][1] += (a1 == -INFINITY) ? 0.0f : exp2f(a1 - M) * iL;
            }
          }
      }
    }
    __syncwarp();
    // the K buffer is free once every warp is past its ldmatrix reads
    __syncthreads();

    if (p.pass == 1) {
      // row sums over the four lanes of a row, then one write per row
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          float l = rl[mt][hr];
          l += __shfl_xor_sync(0xffffffffu, l, 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          const int r = warp * 32 + mt * 16 + g + 8 * hr;
          if (t == 0)
            p.stats[(((size_t)b * p.H_kv + h) * p.max_blocks + j) * MAX_ROWS + r] =
                make_float2(rm[mt][hr], l);
        }
      continue;
    }

    // ---- pass 2: token scores of block j = column sums over all rows
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = cs[i][e];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (g == 0) colsum[warp][i * 8 + 2 * t + e] = v;
      }
    __syncthreads();
    if (tid < BS) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += colsum[w][tid];
      tscore[tid] = v;
      if (p.token_scores) {
        const int tok = j * BS + tid;
        p.token_scores[((size_t)b * p.H_kv + h) * p.max_blocks * BS + tok] = tok < n ? v : 0.0f;
      }
    }
    __syncthreads();
    // reps exist for full blocks only: the num_reps best tokens (ties: lower
    // index), emitted in token order
    if ((j + 1) * BS <= n && page_ok) {
      // warp 0 takes the best token R times (score descending, then index
      // ascending): lane l holds tokens l, l+32, l+64, l+96
      if (warp == 0) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = tscore[lane + 32 * k];
        unsigned int taken = 0u;
#pragma unroll 1
        for (int rr = 0; rr < p.R; ++rr) {
          float bv = -INFINITY;
          int bi = 0x7fffffff;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int idx = lane + 32 * k;
            if (!((taken >> k) & 1u) && (v[k] > bv || (v[k] == bv && idx < bi))) {
              bv = v[k];
              bi = idx;
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
              bv = ov;
              bi = oi;
            }
          }
          if (bi < BS && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) pick[lane + 32 * k] = (taken >> k) & 1u;
      }
      __syncthreads();
      if (tid < BS && pick[tid]) {
        int order = 0;
        for (int u = 0; u < tid; ++u) order += pick[u];
        pick[tid] = 1 + order;  // 1-based output slot
      }
      __syncthreads();
      // copy the chosen rows: warp w copies tokens w, w+8, ... (16 lanes x 16 B)
      for (int tk = warp; tk < BS; tk += 8) {
        const int slot = pick[tk];
        if (slot && lane < 16) {
          const uint4* src =
              reinterpret_cast<const uint4*>(p.k_pool + (((size_t)page * p.H_kv + h) * BS + tk) * D);
          uint4* dst = reinterpret_cast<uint4*>(
              p.reps + (((size_t)page * p.H_kv + h) * p.R + (slot - 1)) * D);
          dst[lane] = __ldg(src + lane);
        }
      }
      __syncthreads();
    }
  }
}

// Combine per-block row statistics over a range of blocks.
__global__ void __launch_bounds__(MAX_ROWS) dyn_combine_kernel(const __grid_constant__ DynParams p) {
  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z, r = threadIdx.x;
  const int n = seq_len_checked(p, b);
  const int nb = (n + BS - 1) / BS;
  const int j0 = sp * nb / NSPLIT, j1 = (sp + 1) * nb / NSPLIT;
  float M = -INFINITY, L = 0.0f;
  const float2* src = p.stats + ((size_t)b * p.H_kv + h) * p.max_blocks * MAX_ROWS + r;
  for (int j = j0; j < j1; j += 8) {
    float2 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = (j + k < j1) ? __ldcg(src + (size_t)(j + k) * MAX_ROWS) : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (v[k].x == -INFINITY) continue;
      const float Mn = fmaxf(M, v[k].x);
      L = L * exp2f(M - Mn) + v[k].y * exp2f(v[k].x - Mn);
      M = Mn;
    }
  }
  p.split[(((size_t)b * p.H_kv + h) * NSPLIT + sp) * MAX_ROWS + r] = make_float2(M, L);
}

}  // namespace

size_t dynamic_ws_bytes(int B, int H_kv, int max_blocks) {
  return align256((size_t)B * H_kv * max_blocks * MAX_ROWS * sizeof(float2)) +
         align256((size_t)B * H_kv * NSPLIT * MAX_ROWS * sizeof(float2));
}

cudaError_t launch_dynamic(const DynLaunch& a, cudaStream_t stream) {
  DynParams p;
  p.kmap = *a.kmap;
  p.k_pool = a.k_pool;
  p.q_local = a.q_local;
  p.table = a.table;
  p.seq_lens = a.seq_lens;
  p.stats = reinterpret_cast<float2*>(a.ws);
  p.split = reinterpret_cast<float2*>(static_cast<uint8_t*>(a.ws) +
                                      align256((size_t)a.B * a.H_kv * a.max_blocks * MAX_ROWS *
                                               sizeof(float2)));
  p.reps = static_cast<__half*>(a.reps);
  p.token_scores = a.token_scores;
  p.status = a.status;
  p.B = a.B;
  p.H_kv = a.H_kv;
  p.G = a.G;
  p.T = a.T;
  p.max_blocks = a.max_blocks;
  p.P = a.P;
  p.R = a.R;
  p.first_block = a.first_block;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  const int smem = KBUF_BYTES * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(dyn_pass_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // slices per (KV head, sequence) so that the grid covers the SMs a few times
  int slices = (2 * a.num_sms + a.B * a.H_kv - 1) / (a.B * a.H_kv);
  if (slices < 1) slices = 1;
  if (slices > a.max_blocks) slices = a.max_blocks;
  p.nslices = slices;
  const dim3 grid(slices, a.H_kv, a.B);
  p.pass = 1;
  dyn_pass_kernel<<<grid, THREADS, smem, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dyn_combine_kernel<<<dim3(NSPLIT, a.H_kv, a.B), MAX_ROWS, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  p.pass = 2;
  dyn_pass_kernel<<<grid, THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kt
