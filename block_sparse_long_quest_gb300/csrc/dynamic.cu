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
// over the tokens row r sees.  Four launches:
//   pass 1   one CTA per (block slice, KV head, sequence): S = Q K^T for every
//            block of its slice on the 5th-generation tensor cores (tcgen05,
//            accumulators in tensor memory, K blocks by 2-D TMA into a double
//            buffer); per block and row, the partial max and sum (base 2) go to
//            the workspace.
//   combine  per (split, KV head, sequence): merge the partials of a range of
//            blocks per row.
//   pass 2   S^T for the requested blocks; p = exp2(s - M_r) / L_r summed over
//            rows per token, written per token.
//   pick     per (block, KV head, sequence): the num_reps best tokens of each
//            full block (ties: lower index) are copied, in token order, as its
//            reps.
// The path is a dense contraction (M = T*G rows per KV head) plus one exp per
// logit per pass; K is read twice (once per pass).
#include "kt_internal.cuh"

namespace kt {
namespace {

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
  float* token_scores;  // [B][H_kv][max_blocks*128] (the caller's or the workspace's)
  int* status;
  int B, H_kv, G, T, max_blocks, P, R, first_block, num_blocks, pass, nslices;
  float scale_log2;
};

// 2^x on the MUFU unit (PTX ex2.approx.ftz: relative error about 2^-22,
// results below 2^-126 flushed to zero; 2^-inf = 0)
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int seq_len_checked(const DynParams& p, int b) {
  int n = __ldg(p.seq_lens + b);
  if (n < 0 || n > p.max_blocks * BS) {
    set_status(p.status, KT_ERR_DEVICE_CHECK);
    n = n < 0 ? 0 : p.max_blocks * BS;
  }
  return n;
}

// ---- tcgen05 version of the two passes ---------------------------------------
// One CTA (16 epilogue warps + 1 control warp) per (block slice, KV head,
// sequence).  The T*G query rows live in shared memory as two K-major
// 128-byte-swizzled boxes (64 channels x 256 rows each); each K block arrives
// by TMA as two boxes (64 channels x 128 tokens) into a double buffer.  One
// thread issues the tcgen05.mma chains into one of two 256-column TMEM
// accumulators.  An epilogue warp reads the TMEM lanes of its quarter
// (warp % 4) and a quarter of the columns:
//   pass 1  S = Q K^T, two M = 128 tiles (rows 0-127, 128-255) x N = 128
//           tokens: a thread owns one row (its TMEM lane) and half of the
//           block's tokens; the two halves' (max, sum) meet in shared memory;
//   pass 2  S^T = K Q^T, M = 128 tokens x N = 256 rows: a thread owns one
//           token and sums exp2(s - M_r) / L_r over 64 of the rows; the four
//           row quarters meet in shared memory.
// Two or four warps meet on their own named barrier, so no warp waits for
// the whole CTA; the epilogue of block q overlaps the MMAs of block q + 1.
constexpr int TC_EPI_WARPS = 16;
constexpr int TC_THREADS = (TC_EPI_WARPS + 1) * 32;
constexpr int Q_BOX = MAX_ROWS * 128;  // 256 rows x 64 channels fp16
constexpr int TC_SMEM = 2 * Q_BOX + 2 * KBUF_BYTES + 1024;
constexpr uint32_t TMEM_COLS = 512;    // two 256-column accumulators
static_assert(TC_SMEM > 233472 / 2, "one CTA per SM: it holds all of TMEM");

__global__ void __launch_bounds__(TC_THREADS, 1) dyn_pass_tc_kernel(const __grid_constant__ DynParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bars[6];  // K full x2, MMA done x2, TMEM free x2
  __shared__ uint32_t tmem_base;
  __shared__ __align__(16) float rowC[MAX_ROWS];  // pass 2: M_r + log2 L_r
  __shared__ int rowPos[MAX_ROWS];
  __shared__ float2 pslot[2][MAX_ROWS];  // pass 1: second token half's (max, sum)
  __shared__ float part4[2][4][BS];      // pass 2: row quarters' sums

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n = seq_len_checked(p, b);
  const int nb = (n + BS - 1) / BS;
  const int rows = p.T * p.G;
  const int H_q = p.H_kv * p.G;
  const int jb = p.pass == 1 ? 0 : min(p.first_block, nb);
  const int je = p.pass == 1 ? nb : min(nb, p.first_block + p.num_blocks);
  const int stride = p.nslices;
  const int nmine = (jb + slice < je) ? (je - jb - slice + stride - 1) / stride : 0;
  const uint32_t sQ = smem_u32(smem), sK = sQ + 2 * Q_BOX;
  const uint32_t kfull = smem_u32(&bars[0]), mdone = kfull + 16, tfree = kfull + 32;

  if (tid == 0) {
    mbar_init(kfull, 1);
    mbar_init(kfull + 8, 1);
    mbar_init(mdone, 1);
    mbar_init(mdone + 8, 1);
    mbar_init(tfree, TC_EPI_WARPS);
    mbar_init(tfree + 8, TC_EPI_WARPS);
    fence_mbar_init();
    prefetch_tensormap(&p.kmap);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // rows: final statistics (pass 2) and query positions
  for (int r = tid; r < MAX_ROWS; r += TC_THREADS) {
    if (p.pass == 2) {
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
      rowC[r] = (L > 0.0f && M != -INFINITY) ? M + log2f(L) : INFINITY;
    }
    rowPos[r] = r < rows ? n - p.T + r / p.G : -1;  // -1: row absent, sees nothing
  }
  // query rows into the two swizzled boxes (16-byte chunk c of row r goes to
  // box c / 8, chunk slot (c % 8) ^ (r % 8))
  for (int idx = tid; idx < MAX_ROWS * 16; idx += TC_THREADS) {
    const int r = idx >> 4, c = idx & 15;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) {
      const __half* src = p.q_local + (((size_t)b * p.T + r / p.G) * H_q + h * p.G + r % p.G) * D;
      v = __ldg(reinterpret_cast<const uint4*>(src) + c);
    }
    *reinterpret_cast<uint4*>(smem + (c >> 3) * Q_BOX + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == TC_EPI_WARPS) {
    // ============================ control thread ============================
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      auto load = [&](int q) {
        const int j = jb + slice + q * stride, buf = q & 1;
        const int page = p.table[(size_t)b * p.max_blocks + j];
        if (page < 0 || page >= p.P) {  // the epilogue masks the whole block
          set_status(p.status, KT_ERR_DEVICE_CHECK);
          mbar_arrive(kfull + 8 * buf);
          return;
        }
        const int row = (page * p.H_kv + h) * BS;
        mbar_arrive_expect_tx(kfull + 8 * buf, KBUF_BYTES);
        tma_load_2d(sK + buf * KBUF_BYTES, &p.kmap, 0, row, kfull + 8 * buf, pol);
        tma_load_2d(sK + buf * KBUF_BYTES + BOX_BYTES, &p.kmap, 64, row, kfull + 8 * buf, pol);
      };
      if (nmine > 0) load(0);
      if (nmine > 1) load(1);
      for (int q = 0; q < nmine; ++q) {
        const int buf = q & 1;
        if (!mbar_wait(kfull + 8 * buf, (q >> 1) & 1, p.status)) break;
        if (q >= 2 && !mbar_wait(tfree + 8 * buf, ((q >> 1) - 1) & 1, p.status)) break;
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)buf * 256u;
        const uint32_t kb = sK + buf * KBUF_BYTES;
        if (p.pass == 1) {
          constexpr uint32_t id = umma_idesc_f16_f32(128, 128);
          for (int mt = 0; mt < 2; ++mt)
            for (int ks = 0; ks < 8; ++ks)
              umma_f16(dt + mt * 128,
                       umma_sdesc_sw128(sQ + (ks >> 2) * Q_BOX + mt * 128 * 128 + (ks & 3) * 32),
                       umma_sdesc_sw128(kb + (ks >> 2) * BOX_BYTES + (ks & 3) * 32), id, ks > 0);
        } else {
          constexpr uint32_t id = umma_idesc_f16_f32(128, 256);
          for (int ks = 0; ks < 8; ++ks)
            umma_f16(dt, umma_sdesc_sw128(kb + (ks >> 2) * BOX_BYTES + (ks & 3) * 32),
                     umma_sdesc_sw128(sQ + (ks >> 2) * Q_BOX + (ks & 3) * 32), id, ks > 0);
        }
        umma_commit(mdone + 8 * buf);
        if (q + 2 < nmine) {
          // the K buffer is free once these MMAs have read it
          if (!mbar_wait(mdone + 8 * buf, (q >> 1) & 1, p.status)) break;
          load(q + 2);
        }
      }
    }
    __syncwarp();
  } else {
    // ============================ epilogue warps ============================
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int* trow = p.table + (size_t)b * p.max_blocks;
    int page_next = nmine > 0 ? trow[jb + slice] : -1;  // loaded a block ahead
    for (int q = 0; q < nmine; ++q) {
      const int buf = q & 1, j = jb + slice + q * stride;
      const int page = page_next;
      if (q + 1 < nmine) page_next = trow[j + stride];
      const bool live = mbar_wait(mdone + 8 * buf, (q >> 1) & 1, p.status);
      tc_fence_after();
      const bool page_ok = live && page >= 0 && page < p.P;
      const bool whole = page_ok && (j + 1) * BS - 1 <= n - p.T;  // every present row sees it all
      if (p.pass == 1) {
        const int half = (warp >> 2) & 1, cpart = warp >> 3;  // M tile, token half
        const uint32_t dt = tmem + (uint32_t)buf * 256u + ((uint32_t)(quarter * 32) << 16) +
                            (uint32_t)(half * 128 + cpart * 64);
        const int r = half * 128 + quarter * 32 + lane;  // this thread's row
        const int pos = rowPos[r];
        const bool row_ok = page_ok && pos >= 0;
        const bool row_whole = whole && pos >= 0;  // no token of the block is masked
        float m = -INFINITY, l = 0.0f;
        // tcgen05.ld is warp-collective: every lane loads, masks apply after
        for (int c0 = 0; c0 < 64; c0 += 32) {
          float v[32];
          tmem_ld32(dt + c0, v);
          if (!row_whole) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int tok = j * BS + cpart * 64 + c0 + e;
              v[e] = (row_ok && tok < n && tok <= pos) ? v[e] : -INFINITY;
            }
          }
          float cm[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
          for (int e = 4; e < 32; ++e) cm[e & 3] = fmaxf(cm[e & 3], v[e]);
          const float cmax = fmaxf(fmaxf(cm[0], cm[1]), fmaxf(cm[2], cm[3])) * p.scale_log2;
          const float mn = fmaxf(m, cmax);
          if (mn != -INFINITY) {
            float sm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 32; ++e) sm4[e & 3] += ex2_fast(fmaf(v[e], p.scale_log2, -mn));
            l = l * ex2_fast(m - mn) + ((sm4[0] + sm4[1]) + (sm4[2] + sm4[3]));
            m = mn;
          }
        }
        // this warp is done with the TMEM buffer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tfree + 8 * buf);
        // the row's two token halves meet: warps w and w + 8 share barrier 1 + w % 8
        if (cpart == 1) pslot[buf][r] = make_float2(m, l);
        named_bar_sync(1 + (warp & 7), 64);
        if (cpart == 0) {
          const float2 o = pslot[buf][r];
          const float M = fmaxf(m, o.x);
          const float L = M == -INFINITY ? 0.0f : l * ex2_fast(m - M) + o.y * ex2_fast(o.x - M);
          p.stats[(((size_t)b * p.H_kv + h) * p.max_blocks + j) * MAX_ROWS + r] = make_float2(M, L);
        }
      } else {
        const int rq = warp >> 2;  // rows 64*rq .. +63
        const uint32_t dt = tmem + (uint32_t)buf * 256u + ((uint32_t)(quarter * 32) << 16) +
                            (uint32_t)(rq * 64);
        const int t = quarter * 32 + lane, tok = j * BS + t;  // this thread's token
        const bool tok_ok = page_ok && tok < n;
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        // tcgen05.ld is warp-collective: every lane loads, masks apply after.
        // exp2(s - M_r) / L_r = exp2(s - rowC[r]) with rowC = M + log2 L
        // (+inf for rows without tokens)
        for (int c0 = 0; c0 < 64; c0 += 32) {
          float v[32];
          tmem_ld32(dt + c0, v);
          const float4* rc = reinterpret_cast<const float4*>(rowC + rq * 64 + c0);
          if (whole) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 c = rc[e >> 2];
              acc4[0] += ex2_fast(fmaf(v[e], p.scale_log2, -c.x));
              acc4[1] += ex2_fast(fmaf(v[e + 1], p.scale_log2, -c.y));
              acc4[2] += ex2_fast(fmaf(v[e + 2], p.scale_log2, -c.z));
              acc4[3] += ex2_fast(fmaf(v[e + 3], p.scale_log2, -c.w));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int r = rq * 64 + c0 + e;
              const int pos = rowPos[r];
              if (tok_ok && pos >= 0 && tok <= pos)
                acc4[e & 3] += ex2_fast(fmaf(v[e], p.scale_log2, -rowC[r]));
            }
          }
        }
        // this warp is done with the TMEM buffer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tfree + 8 * buf);
        // the token's four row quarters meet: warps quarter + 4i share barrier 1 + quarter
        part4[buf][rq][t] = tok_ok ? (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]) : 0.0f;
        named_bar_sync(1 + quarter, 128);
        if (rq == 0) {
          const float v = (part4[buf][0][t] + part4[buf][1][t]) + (part4[buf][2][t] + part4[buf][3][t]);
          p.token_scores[((size_t)b * p.H_kv + h) * p.max_blocks * BS + (size_t)j * BS + t] = v;
        }
      }
    }
  }
  // all tcgen05 work of this CTA has completed once every epilogue warp has
  // seen its last commit; then the accumulators are released
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
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

// Reps of the requested full blocks: one warp per (block, KV head,
// sequence) takes the num_reps best tokens by accumulated score (descending,
// then index ascending) and copies their key rows, in token order.
constexpr int PICK_WARPS = 8;
__global__ void __launch_bounds__(PICK_WARPS * 32) dyn_pick_kernel(const __grid_constant__ DynParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int jj = blockIdx.x * PICK_WARPS + warp;
  const int n = seq_len_checked(p, b);
  const int j = p.first_block + jj;
  if (jj >= p.num_blocks || (j + 1) * BS > n) return;  // reps exist for full blocks only
  const int page = p.table[(size_t)b * p.max_blocks + j];
  if (page < 0 || page >= p.P) {
    if (lane == 0) set_status(p.status, KT_ERR_DEVICE_CHECK);
    return;
  }
  const float* sc = p.token_scores + ((size_t)b * p.H_kv + h) * p.max_blocks * BS + (size_t)j * BS;
  float v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = sc[lane + 32 * k];
  unsigned int taken = 0u;
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
  // output slot = chosen tokens before this one (token order); a half warp
  // copies each chosen 256-byte row
  const uint4* src = reinterpret_cast<const uint4*>(p.k_pool + ((size_t)page * p.H_kv + h) * BS * D);
  uint4* dst = reinterpret_cast<uint4*>(p.reps + ((size_t)page * p.H_kv + h) * p.R * D);
  int before = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    unsigned int bal = __ballot_sync(0xffffffffu, (taken >> k) & 1u);
    while (bal) {
      const int l0 = __ffs(bal) - 1;
      bal &= bal - 1u;
      const int l1 = bal ? __ffs(bal) - 1 : -1;  // a second row for the upper half warp
      if (l1 >= 0) bal &= bal - 1u;
      const int mine = lane < 16 ? l0 : l1;
      const int slot = lane < 16 ? before : before + 1;
      if (mine >= 0) dst[(size_t)slot * (D / 8) + (lane & 15)] = __ldg(src + (size_t)(mine + 32 * k) * (D / 8) + (lane & 15));
      before += l1 >= 0 ? 2 : 1;
    }
  }
}

}  // namespace

size_t dynamic_ws_bytes(int B, int H_kv, int max_blocks) {
  return align256((size_t)B * H_kv * max_blocks * MAX_ROWS * sizeof(float2)) +
         align256((size_t)B * H_kv * NSPLIT * MAX_ROWS * sizeof(float2)) +
         align256((size_t)B * H_kv * max_blocks * BS * sizeof(float));
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
  // token scores: the caller's array, else the workspace's
  p.token_scores = a.token_scores
                       ? a.token_scores
                       : reinterpret_cast<float*>(
                             static_cast<uint8_t*>(a.ws) +
                             align256((size_t)a.B * a.H_kv * a.max_blocks * MAX_ROWS * sizeof(float2)) +
                             align256((size_t)a.B * a.H_kv * NSPLIT * MAX_ROWS * sizeof(float2)));
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
  static std::atomic<int> optin[KT_MAX_DEVICES];
  cudaError_t e = (cudaError_t)per_device_cached(optin, [] {
    return (int)cudaFuncSetAttribute(dyn_pass_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     TC_SMEM);
  });
  if (e != cudaSuccess) return e;
  // slices per (KV head, sequence) so that the grid covers the SMs a few times
  int slices = (2 * a.num_sms + a.B * a.H_kv - 1) / (a.B * a.H_kv);
  if (slices < 1) slices = 1;
  if (slices > a.max_blocks) slices = a.max_blocks;
  p.nslices = slices;
  const dim3 grid(slices, a.H_kv, a.B);
  p.pass = 1;
  dyn_pass_tc_kernel<<<grid, TC_THREADS, TC_SMEM, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dyn_combine_kernel<<<dim3(NSPLIT, a.H_kv, a.B), MAX_ROWS, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  p.pass = 2;
  dyn_pass_tc_kernel<<<grid, TC_THREADS, TC_SMEM, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.R > 0 && p.reps && p.num_blocks > 0) {
    const dim3 pg((p.num_blocks + PICK_WARPS - 1) / PICK_WARPS, a.H_kv, a.B);
    dyn_pick_kernel<<<pg, PICK_WARPS * 32, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace kt
