// kt_api.cu — host side of the libkt C ABI: argument validation, workspace
// layout, TMA tensor maps and kernel launches.  No allocation, no hidden
// synchronisation (see kt.h for the contract of every call).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "kt_internal.cuh"

namespace kt {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kt_status check_kv(const kt_paged_kv* kv) {
  if (!kv || !kv->k_pool || !kv->v_pool || !kv->block_table || !kv->seq_lens)
    return KT_ERR_INVALID_ARG;
  if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(kv->block_table) ||
      !aligned16(kv->seq_lens))
    return KT_ERR_INVALID_ARG;
  if (kv->batch < 1 || kv->num_kv_heads < 1 || kv->max_blocks_per_seq < 1 || kv->num_pages < 1)
    return KT_ERR_INVALID_ARG;
  if (kv->head_dim != D || kv->block_size != BS) return KT_ERR_UNSUPPORTED;
  if ((long long)kv->batch * kv->num_kv_heads > MAX_SEGS || kv->batch > 65535)
    return KT_ERR_UNSUPPORTED;
  if ((long long)kv->num_pages * kv->num_kv_heads * BS > 0x7FFFFFFFLL) return KT_ERR_UNSUPPORTED;
  if ((long long)kv->max_blocks_per_seq * BS > 0x7FFFFFFFLL) return KT_ERR_UNSUPPORTED;
  return KT_OK;
}

kt_status check_heads(const kt_paged_kv* kv, int num_q_heads, float scale) {
  if (num_q_heads < 1 || num_q_heads % kv->num_kv_heads != 0) return KT_ERR_INVALID_ARG;
  if (num_q_heads / kv->num_kv_heads > MAX_G) return KT_ERR_UNSUPPORTED;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return KT_ERR_INVALID_ARG;
  return KT_OK;
}

kt_status check_params(const kt_paged_kv* kv, const kt_sparse_params* p) {
  if (!p) return KT_ERR_INVALID_ARG;
  kt_status s = check_heads(kv, p->num_q_heads, p->softmax_scale);
  if (s != KT_OK) return s;
  if (p->initial_blocks < 0 || p->local_blocks < 0 || p->top_k < 1) return KT_ERR_INVALID_ARG;
  if (p->local_blocks < 1 || p->top_k > MAX_TOPK) return KT_ERR_UNSUPPORTED;
  if (p->head_mode != KT_HEAD_SHARED && p->head_mode != KT_HEAD_SEPARATE)
    return KT_ERR_INVALID_ARG;
  switch (p->rep) {
    case KT_REP_MAX:
    case KT_REP_MEAN:
    case KT_REP_QUEST:
      break;
    case KT_REP_FIX:
      if (p->fix_stride < 1 || p->fix_stride > BS || BS % p->fix_stride != 0)
        return KT_ERR_INVALID_ARG;
      break;
    case KT_REP_DYNAMIC:
      if (p->num_reps < 1) return KT_ERR_INVALID_ARG;
      if (p->num_reps > MAX_DYN_REPS) return KT_ERR_UNSUPPORTED;
      break;
    default:
      return KT_ERR_INVALID_ARG;
  }
  return KT_OK;
}

int reps_rows(const kt_sparse_params* p) {
  switch (p->rep) {
    case KT_REP_MAX:
    case KT_REP_MEAN:
      return 1;
    case KT_REP_QUEST:
      return 2;
    case KT_REP_FIX:
      return p->fix_stride >= 1 ? BS / p->fix_stride : 0;
    case KT_REP_DYNAMIC:
      return p->num_reps;
    default:
      return 0;
  }
}

// One layout for every op: [status header][attention][selection][dynamic].
// Region offsets depend only on the shapes, so a workspace sized for a larger
// op serves every smaller one; kt_workspace_bytes(op) is the end of the last
// region that `op` uses.
WsLayout layout(kt_op op, const kt_paged_kv* kv, const kt_sparse_params* p, int T) {
  WsLayout L;
  std::memset(&L, 0, sizeof(L));
  const int B = kv->batch, H_kv = kv->num_kv_heads, S = B * H_kv;
  const int G = p->num_q_heads / H_kv;
  size_t off = 256;  // status header
  L.status = 0;
  L.slot_floats = ((2 * G + G * D) + 3) & ~3;
  L.attn_counters = off;
  off = align256(off + (size_t)S * 4);
  L.attn_parts = off;
  off = align256(off + (size_t)2 * (MAX_ATTN_CTAS + S) * L.slot_floats * 4);
  const size_t attn_end = off;
  L.sel = make_sel_plan(B, H_kv, kv->max_blocks_per_seq, p->initial_blocks, p->local_blocks,
                        p->top_k > 0 ? p->top_k : 1, p->head_mode);
  const size_t units = (size_t)B * L.sel.SEL;
  L.sel_counters = off;
  off = align256(off + units * 4);
  L.sel_cand = off;
  off = align256(off + units * L.sel.nchunks * L.sel.kk * 8);
  L.sel_cand_pages = off;
  off = align256(off + units * L.sel.nchunks * L.sel.kk * 4);
  L.sel_pages = off;
  off = align256(off + units * (size_t)(p->top_k > 0 ? p->top_k : 1) * 4);
  // fused step (selection inside the attention launch)
  const size_t fcap = (size_t)MAX_ATTN_CTAS *
                      (size_t)(p->top_k < FUSED_KK_CAP ? (p->top_k > 0 ? p->top_k : 1)
                                                       : FUSED_KK_CAP);
  L.f_sync = off;
  off = align256(off + 8);
  L.f_cand = off;
  L.f_cand_slots = fcap;
  off = align256(off + fcap * 8);
  L.f_cpage = off;
  off = align256(off + fcap * 4);
  const size_t sel_end = off;
  (void)T;
  L.dyn = off;
  L.dyn_bytes = (op == KT_OP_DYNAMIC_REPS || op == KT_OP_PRESELECT)
                    ? dynamic_ws_bytes(B, H_kv, kv->max_blocks_per_seq)
                    : 0;
  off = align256(off + L.dyn_bytes);
  const int SELp = p->head_mode == KT_HEAD_SHARED ? 1 : H_kv;
  L.presel_votes = off;
  L.presel_bscore = off + align256((size_t)B * H_kv * kv->max_blocks_per_seq * BS * 4);
  if (op == KT_OP_PRESELECT) off += preselect_ws_bytes(B, H_kv, SELp, kv->max_blocks_per_seq);
  L.total = op == KT_OP_DENSE_ATTN ? attn_end
            : (op == KT_OP_DYNAMIC_REPS || op == KT_OP_PRESELECT) ? off
                                                                   : sel_end;
  return L;
}

// ---- TMA tensor maps over the K / V pools ----------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [rows = pages*heads*128][128 channels] fp16, boxes of 64 channels x 128 rows
// (one block of one head, half its channels), 128-byte swizzle; the attention
// kernel's stage size and ldmatrix addressing assume exactly this box.
bool encode_pool_map(CUtensorMap* map, const void* pool, const kt_paged_kv* kv) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)kv->num_pages * kv->num_kv_heads * BS};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)BS};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(pool), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows][128] int8 Q8_0 codes, boxes of 128 bytes x 128 rows (one block of one
// KV head), 128-byte swizzle.
bool encode_code_map(CUtensorMap* map, const void* pool, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D};
  cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)BS};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The map depends only on the pool address, its extent and its element type:
// the last few are kept per thread, so a decode loop encodes each pool once.
bool make_pool_map(CUtensorMap* map, const void* pool, const kt_paged_kv* kv,
                   bool codes = false) {
  struct Entry {
    const void* pool;
    long long rows;
    int dev;
    bool codes;
    CUtensorMap map;
  };
  constexpr int N = 8;
  thread_local Entry cache[N];
  thread_local int used = 0, next = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const long long rows = (long long)kv->num_pages * kv->num_kv_heads * BS;
  for (int i = 0; i < used; ++i)
    if (cache[i].pool == pool && cache[i].rows == rows && cache[i].dev == dev &&
        cache[i].codes == codes) {
      *map = cache[i].map;
      return true;
    }
  if (!(codes ? encode_code_map(map, pool, rows) : encode_pool_map(map, pool, kv))) return false;
  Entry& e = cache[next];
  e.pool = pool;
  e.rows = rows;
  e.dev = dev;
  e.codes = codes;
  e.map = *map;
  next = (next + 1) % N;
  if (used < N) ++used;
  return true;
}

int num_sms() {
  static std::atomic<int> slot[KT_MAX_DEVICES];
  return per_device_cached(slot, [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
  });
}

// CTAs an attention launch may use from this host thread: one per SM, or
// fewer when the caller has set a cap (kt_set_max_ctas).
thread_local int max_ctas_cap = 0;
int cta_budget() {
  const int sms = num_sms();
  return (max_ctas_cap > 0 && max_ctas_cap < sms) ? max_ctas_cap : sms;
}

// Phase-stamp buffer of this host thread's attention launches (kt_set_phase_stamps).
thread_local unsigned long long* stamps_buf = nullptr;
thread_local int stamps_max_ctas = 0;
unsigned long long* stamps_for(int grid) { return grid <= stamps_max_ctas ? stamps_buf : nullptr; }

kt_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KT_OK : KT_ERR_CUDA; }

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

int mask_words_of(const kt_paged_kv* kv) { return (kv->max_blocks_per_seq + 31) / 32; }

kt_status select_impl(const void* q, const kt_paged_kv* kv, const void* reps,
                      const kt_sparse_params* p, int32_t* sel, int32_t* cnt, float* sel_scores,
                      void* ws, const WsLayout& L, bool trigger, cudaStream_t stream,
                      const uint32_t* presel_mask = nullptr) {
  SelectLaunch a;
  a.presel_mask = presel_mask;
  a.mask_words = mask_words_of(kv);
  a.q = static_cast<const __half*>(q);
  a.reps = reps;
  a.table = kv->block_table;
  a.seq_lens = kv->seq_lens;
  a.sel = sel;
  a.cnt = cnt;
  a.sel_scores = sel_scores;
  a.status = at<int>(ws, L.status);
  a.counters = at<int>(ws, L.sel_counters);
  a.cand = at<unsigned long long>(ws, L.sel_cand);
  a.cand_pages = at<int>(ws, L.sel_cand_pages);
  a.sel_pages = at<int32_t>(ws, L.sel_pages);
  a.B = kv->batch;
  a.H_kv = kv->num_kv_heads;
  a.G = p->num_q_heads / kv->num_kv_heads;
  a.max_blocks = kv->max_blocks_per_seq;
  a.P = kv->num_pages;
  a.I_b = p->initial_blocks;
  a.L_b = p->local_blocks;
  a.top_k = p->top_k;
  a.rep = p->rep;
  a.R = reps_rows(p);
  a.head_mode = p->head_mode;
  a.plan = L.sel;
  a.trigger_dependents = trigger;
  if (a.plan.chunk > SEL_MAX_CHUNK || select_smem_bytes(a) > 227 * 1024) return KT_ERR_UNSUPPORTED;
  return cuda_status(launch_select(a, stream));
}

// step_path: the selection ran in this call on this workspace, so its page ids
// (sel_pages) are used directly, and its counts are min(top_k, C) unless
// counts_vary (a preselection can leave fewer candidates; cnt is then read).
// KV source of an attention-only launch (KVM_*): for KVM_HOST the device
// addresses of the host pools; for KVM_Q8 the code and scale pools.
struct KvSource {
  int kvm = KVM_F16;
  const void* k_src = nullptr;
  const void* v_src = nullptr;
  const void* k_scale = nullptr;
  const void* v_scale = nullptr;
};

kt_status attn_impl(const void* q, const kt_paged_kv* kv, int num_q_heads, float scale,
                    const kt_sparse_params* p, const int32_t* sel, const int32_t* cnt, float* out,
                    void* ws, const WsLayout& L, bool dense, bool pdl, cudaStream_t stream,
                    bool step_path = false, bool counts_vary = false,
                    const KvSource& src = KvSource()) {
  CUtensorMap kmap, vmap;
  std::memset(&kmap, 0, sizeof(kmap));
  std::memset(&vmap, 0, sizeof(vmap));
  if (src.kvm == KVM_F16 &&
      (!make_pool_map(&kmap, kv->k_pool, kv) || !make_pool_map(&vmap, kv->v_pool, kv)))
    return KT_ERR_CUDA;
  if (src.kvm == KVM_Q8 && (!make_pool_map(&kmap, src.k_src, kv, true) ||
                            !make_pool_map(&vmap, src.v_src, kv, true)))
    return KT_ERR_CUDA;
  const int sms = cta_budget();
  if (sms <= 0) return KT_ERR_CUDA;
  AttnLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.kmap = &kmap;
  a.vmap = &vmap;
  a.q = static_cast<const __half*>(q);
  a.table = kv->block_table;
  a.seq_lens = kv->seq_lens;
  a.sel = sel;
  a.cnt = (step_path && !counts_vary) ? nullptr : cnt;
  a.sel_pages = step_path ? at<int32_t>(ws, L.sel_pages) : nullptr;
  a.out = out;
  a.status = at<int>(ws, L.status);
  a.counters = at<int>(ws, L.attn_counters);
  a.parts = at<float>(ws, L.attn_parts);
  a.B = kv->batch;
  a.H_kv = kv->num_kv_heads;
  a.G = num_q_heads / kv->num_kv_heads;
  a.max_blocks = kv->max_blocks_per_seq;
  a.P = kv->num_pages;
  a.I_b = dense ? 0 : p->initial_blocks;
  a.L_b = dense ? 1 : p->local_blocks;
  a.top_k = dense ? 1 : p->top_k;
  a.SEL = dense ? 1 : (p->head_mode == KT_HEAD_SHARED ? 1 : kv->num_kv_heads);
  a.dense = dense ? 1 : 0;
  a.slot_floats = L.slot_floats;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  // at least one CTA per (sequence, KV head) segment, at least one per SM
  const int nseg = kv->batch * kv->num_kv_heads;
  const int base = sms < MAX_ATTN_CTAS ? sms : MAX_ATTN_CTAS;
  a.grid = base > nseg ? base : nseg;
  a.pdl = pdl;
  a.stamps = stamps_for(a.grid);
  a.kvm = src.kvm;
  a.k_src = src.k_src;
  a.v_src = src.v_src;
  a.k_scale = src.k_scale;
  a.v_scale = src.v_scale;
  return cuda_status(launch_attention(a, stream));
}

}  // namespace
}  // namespace kt

using namespace kt;

extern "C" {

const char* kt_status_string(kt_status s) {
  switch (s) {
    case KT_OK: return "ok";
    case KT_ERR_INVALID_ARG: return "invalid argument";
    case KT_ERR_UNSUPPORTED: return "unsupported shape or method";
    case KT_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KT_ERR_CUDA: return "CUDA error";
    case KT_ERR_DEVICE_CHECK: return "device-side bounds check failed";
    case KT_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int32_t kt_reps_per_block(const kt_sparse_params* p) { return p ? reps_rows(p) : 0; }

size_t kt_reps_pool_bytes(const kt_paged_kv* kv, const kt_sparse_params* p) {
  if (!kv || !p || kv->num_pages < 1 || kv->num_kv_heads < 1 || kv->head_dim < 1) return 0;
  const int R = reps_rows(p);
  if (R <= 0) return 0;
  const size_t elem = p->rep == KT_REP_MEAN ? 4 : 2;
  return (size_t)kv->num_pages * kv->num_kv_heads * R * kv->head_dim * elem;
}

kt_status kt_workspace_bytes(kt_op op, const kt_paged_kv* kv, const kt_sparse_params* p,
                             int32_t T, size_t* bytes) {
  if (!bytes) return KT_ERR_INVALID_ARG;
  if (op < KT_OP_SCORE_SELECT || op > KT_OP_PRESELECT) return KT_ERR_INVALID_ARG;
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  if (op == KT_OP_DENSE_ATTN) {
    if (!p) return KT_ERR_INVALID_ARG;
    s = check_heads(kv, p->num_q_heads, p->softmax_scale);
  } else {
    s = check_params(kv, p);
  }
  if (s != KT_OK) return s;
  if (op == KT_OP_DYNAMIC_REPS && T < 1) return KT_ERR_INVALID_ARG;
  *bytes = layout(op, kv, p, T).total;
  return KT_OK;
}

kt_status kt_workspace_init(void* ws, size_t ws_bytes, kt_stream_t stream) {
  if (!ws || ws_bytes < 256) return KT_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

kt_status kt_build_block_reps(const kt_paged_kv* kv, const kt_sparse_params* p,
                              int32_t first_block, int32_t num_blocks, void* reps_pool,
                              kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!reps_pool || !aligned16(reps_pool) || first_block < 0 || num_blocks < 0)
    return KT_ERR_INVALID_ARG;
  if (p->rep == KT_REP_DYNAMIC) return KT_ERR_INVALID_ARG;  // kt_build_dynamic_reps
  if (num_blocks == 0) return KT_OK;
  RepsLaunch a;
  a.k_pool = static_cast<const __half*>(kv->k_pool);
  a.table = kv->block_table;
  a.seq_lens = kv->seq_lens;
  a.reps = reps_pool;
  a.B = kv->batch;
  a.H_kv = kv->num_kv_heads;
  a.max_blocks = kv->max_blocks_per_seq;
  a.P = kv->num_pages;
  a.rep = p->rep;
  a.R = reps_rows(p);
  a.fix_stride = p->fix_stride;
  a.first_block = first_block;
  const long long last = (long long)first_block + num_blocks;
  a.num_blocks = (int)((last > kv->max_blocks_per_seq ? kv->max_blocks_per_seq : last) -
                       first_block);
  if (a.num_blocks <= 0) return KT_OK;
  return cuda_status(launch_reps(a, (cudaStream_t)stream));
}

kt_status kt_build_dynamic_reps(const kt_paged_kv* kv, const kt_sparse_params* p,
                                const void* q_local, int32_t T, int32_t first_block,
                                int32_t num_blocks, void* reps_pool, float* token_scores,
                                void* ws, size_t ws_bytes, kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (p->rep != KT_REP_DYNAMIC) return KT_ERR_INVALID_ARG;
  if (!q_local || !reps_pool || !ws || !aligned16(q_local) || !aligned16(reps_pool) ||
      !aligned16(ws) || (token_scores && !aligned16(token_scores)))
    return KT_ERR_INVALID_ARG;
  if (T < 1 || first_block < 0 || num_blocks < 0) return KT_ERR_INVALID_ARG;
  const int G = p->num_q_heads / kv->num_kv_heads;
  if ((long long)T * G > MAX_DYN_ROWS) return KT_ERR_UNSUPPORTED;
  const WsLayout L = layout(KT_OP_DYNAMIC_REPS, kv, p, T);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap kmap;
  if (!make_pool_map(&kmap, kv->k_pool, kv)) return KT_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return KT_ERR_CUDA;
  DynLaunch a;
  a.kmap = &kmap;
  a.k_pool = static_cast<const __half*>(kv->k_pool);
  a.q_local = static_cast<const __half*>(q_local);
  a.table = kv->block_table;
  a.seq_lens = kv->seq_lens;
  a.ws = at<uint8_t>(ws, L.dyn);
  a.reps = reps_pool;
  a.token_scores = token_scores;
  a.status = at<int>(ws, L.status);
  a.B = kv->batch;
  a.H_kv = kv->num_kv_heads;
  a.G = G;
  a.T = T;
  a.max_blocks = kv->max_blocks_per_seq;
  a.P = kv->num_pages;
  a.R = p->num_reps;
  a.first_block = first_block;
  const long long last = (long long)first_block + num_blocks;
  a.num_blocks = (int)((last > kv->max_blocks_per_seq ? kv->max_blocks_per_seq : last) -
                       (first_block < kv->max_blocks_per_seq ? first_block
                                                             : kv->max_blocks_per_seq));
  if (a.num_blocks < 0) a.num_blocks = 0;
  a.num_sms = sms;
  a.scale_log2 = (float)((double)p->softmax_scale * 1.4426950408889634);
  return cuda_status(launch_dynamic(a, (cudaStream_t)stream));
}

kt_status kt_score_select_blocks(const void* q, const kt_paged_kv* kv, const void* reps_pool,
                                 const kt_sparse_params* p, int32_t* sel, int32_t* cnt,
                                 float* sel_scores, void* ws, size_t ws_bytes,
                                 kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q || !reps_pool || !sel || !cnt || !ws || !aligned16(q) || !aligned16(reps_pool) ||
      !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  const WsLayout L = layout(KT_OP_SCORE_SELECT, kv, p, 0);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  return select_impl(q, kv, reps_pool, p, sel, cnt, sel_scores, ws, L, false,
                     (cudaStream_t)stream);
}

kt_status kt_score_select_blocks_presel(const void* q, const kt_paged_kv* kv,
                                        const void* reps_pool, const kt_sparse_params* p,
                                        const uint32_t* presel_mask, int32_t* sel, int32_t* cnt,
                                        float* sel_scores, void* ws, size_t ws_bytes,
                                        kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q || !reps_pool || !sel || !cnt || !ws || !presel_mask || !aligned16(q) ||
      !aligned16(reps_pool) || !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  const WsLayout L = layout(KT_OP_SCORE_SELECT, kv, p, 0);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  return select_impl(q, kv, reps_pool, p, sel, cnt, sel_scores, ws, L, false,
                     (cudaStream_t)stream, presel_mask);
}

int32_t kt_preselect_mask_words(const kt_paged_kv* kv) {
  if (!kv || kv->max_blocks_per_seq < 1) return -(int32_t)KT_ERR_INVALID_ARG;
  return mask_words_of(kv);
}

kt_status kt_preselect_blocks(const kt_paged_kv* kv, const kt_sparse_params* p,
                              const void* q_local, int32_t T, int32_t kernel_size, int32_t count,
                              uint32_t* presel_mask, int32_t* presel_cnt, void* ws,
                              size_t ws_bytes, kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q_local || !presel_mask || !presel_cnt || !ws || !aligned16(q_local) || !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  if (T < 1 || count < 1 || kernel_size < 1 || (kernel_size % 2) == 0)
    return KT_ERR_INVALID_ARG;
  if (kernel_size > PRESEL_MAX_KERNEL) return KT_ERR_UNSUPPORTED;
  const int G = p->num_q_heads / kv->num_kv_heads;
  if ((long long)T * G > MAX_DYN_ROWS) return KT_ERR_UNSUPPORTED;
  const int mw = mask_words_of(kv);
  if (preselect_smem_bytes(kv->max_blocks_per_seq, mw) > 200 * 1024) return KT_ERR_UNSUPPORTED;
  const WsLayout L = layout(KT_OP_PRESELECT, kv, p, T);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap kmap;
  if (!make_pool_map(&kmap, kv->k_pool, kv)) return KT_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return KT_ERR_CUDA;
  // token votes: the Dynamic passes without representatives
  float* votes = at<float>(ws, L.presel_votes);
  DynLaunch d;
  d.kmap = &kmap;
  d.k_pool = static_cast<const __half*>(kv->k_pool);
  d.q_local = static_cast<const __half*>(q_local);
  d.table = kv->block_table;
  d.seq_lens = kv->seq_lens;
  d.ws = at<uint8_t>(ws, L.dyn);
  d.reps = nullptr;
  d.token_scores = votes;
  d.status = at<int>(ws, L.status);
  d.B = kv->batch;
  d.H_kv = kv->num_kv_heads;
  d.G = G;
  d.T = T;
  d.max_blocks = kv->max_blocks_per_seq;
  d.P = kv->num_pages;
  d.R = 0;
  d.first_block = 0;
  d.num_blocks = kv->max_blocks_per_seq;
  d.num_sms = sms;
  d.scale_log2 = (float)((double)p->softmax_scale * 1.4426950408889634);
  cudaError_t e = launch_dynamic(d, (cudaStream_t)stream);
  if (e != cudaSuccess) return KT_ERR_CUDA;
  PreselLaunch a;
  a.votes = votes;
  a.seq_lens = kv->seq_lens;
  a.bscore = at<float>(ws, L.presel_bscore);
  a.mask = presel_mask;
  a.cnt = presel_cnt;
  a.status = at<int>(ws, L.status);
  a.B = kv->batch;
  a.H_kv = kv->num_kv_heads;
  a.SEL = p->head_mode == KT_HEAD_SHARED ? 1 : kv->num_kv_heads;
  a.max_blocks = kv->max_blocks_per_seq;
  a.I_b = p->initial_blocks;
  a.L_b = p->local_blocks;
  a.kernel = kernel_size;
  a.count = count;
  a.mask_words = mw;
  return cuda_status(launch_preselect(a, (cudaStream_t)stream));
}

kt_status kt_sparse_decode_attn(const void* q, const kt_paged_kv* kv, const kt_sparse_params* p,
                                const int32_t* sel, const int32_t* cnt, float* out, void* ws,
                                size_t ws_bytes, kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q || !sel || !cnt || !out || !ws || !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  const WsLayout L = layout(KT_OP_SPARSE_ATTN, kv, p, 0);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  return attn_impl(q, kv, p->num_q_heads, p->softmax_scale, p, sel, cnt, out, ws, L, false, false,
                   (cudaStream_t)stream);
}

// Device address of a host pool the GPU can read (page-locked, mapped), or
// nullptr.  The last few answers are kept per host thread and device, so a
// decode loop (or a CUDA graph capture of one) queries each pool once.
static const void* host_pool_device_ptr(const void* p) {
  struct Entry {
    const void* host;
    const void* dev_ptr;
    int dev;
  };
  constexpr int N = 16;
  thread_local Entry cache[N];
  thread_local int used = 0, next = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  for (int i = 0; i < used; ++i)
    if (cache[i].host == p && cache[i].dev == dev) return cache[i].dev_ptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  cache[next] = Entry{p, at.devicePointer, dev};
  next = (next + 1) % N;
  if (used < N) ++used;
  return at.devicePointer;
}

kt_status kt_sparse_decode_attn_hostkv(const void* q, const kt_paged_kv* kv,
                                       const kt_sparse_params* p, const int32_t* sel,
                                       const int32_t* cnt, float* out, void* ws, size_t ws_bytes,
                                       kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q || !sel || !cnt || !out || !ws || !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  KvSource src;
  src.kvm = KVM_HOST;
  src.k_src = host_pool_device_ptr(kv->k_pool);
  src.v_src = host_pool_device_ptr(kv->v_pool);
  if (!src.k_src || !src.v_src || !aligned16(src.k_src) || !aligned16(src.v_src))
    return KT_ERR_INVALID_ARG;
  const WsLayout L = layout(KT_OP_SPARSE_ATTN, kv, p, 0);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  return attn_impl(q, kv, p->num_q_heads, p->softmax_scale, p, sel, cnt, out, ws, L, false, false,
                   (cudaStream_t)stream, false, false, src);
}

kt_status kt_quantize_kv_q8_0(const kt_paged_kv* kv, void* k_code, void* k_scale, void* v_code,
                              void* v_scale, int32_t first_page, int32_t num_pages,
                              kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  if (!k_code || !k_scale || !v_code || !v_scale || !aligned16(k_code) || !aligned16(k_scale) ||
      !aligned16(v_code) || !aligned16(v_scale))
    return KT_ERR_INVALID_ARG;
  if (first_page < 0 || num_pages < 0 || (long long)first_page + num_pages > kv->num_pages)
    return KT_ERR_INVALID_ARG;
  QuantLaunch a;
  a.k_pool = static_cast<const __half*>(kv->k_pool);
  a.v_pool = static_cast<const __half*>(kv->v_pool);
  a.k_code = static_cast<int8_t*>(k_code);
  a.k_scale = static_cast<__half*>(k_scale);
  a.v_code = static_cast<int8_t*>(v_code);
  a.v_scale = static_cast<__half*>(v_scale);
  a.first_page = first_page;
  a.num_pages = num_pages;
  a.H_kv = kv->num_kv_heads;
  return cuda_status(launch_quant(a, (cudaStream_t)stream));
}

// The shapes and table of Q8_0 pools as a kt_paged_kv (the code pools stand
// in for the fp16 pools in the checks; they are never read as fp16).
static kt_paged_kv kv_view_q8(const kt_paged_kv_q8* kvq) {
  kt_paged_kv kv;
  kv.k_pool = kvq->k_code;
  kv.v_pool = kvq->v_code;
  kv.block_table = kvq->block_table;
  kv.seq_lens = kvq->seq_lens;
  kv.batch = kvq->batch;
  kv.num_kv_heads = kvq->num_kv_heads;
  kv.head_dim = kvq->head_dim;
  kv.block_size = kvq->block_size;
  kv.max_blocks_per_seq = kvq->max_blocks_per_seq;
  kv.num_pages = kvq->num_pages;
  return kv;
}

kt_status kt_sparse_decode_attn_q8_0(const void* q, const kt_paged_kv_q8* kvq,
                                     const kt_sparse_params* p, const int32_t* sel,
                                     const int32_t* cnt, float* out, void* ws, size_t ws_bytes,
                                     kt_stream_t stream) {
  if (!kvq) return KT_ERR_INVALID_ARG;
  kt_paged_kv kv = kv_view_q8(kvq);
  kt_status s = check_kv(&kv);
  if (s != KT_OK) return s;
  s = check_params(&kv, p);
  if (s != KT_OK) return s;
  if (!kvq->k_scale || !kvq->v_scale || !aligned16(kvq->k_scale) || !aligned16(kvq->v_scale))
    return KT_ERR_INVALID_ARG;
  if (!q || !sel || !cnt || !out || !ws || !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  const WsLayout L = layout(KT_OP_SPARSE_ATTN, &kv, p, 0);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  KvSource src;
  src.kvm = KVM_Q8;
  src.k_src = kvq->k_code;
  src.v_src = kvq->v_code;
  src.k_scale = kvq->k_scale;
  src.v_scale = kvq->v_scale;
  return attn_impl(q, &kv, p->num_q_heads, p->softmax_scale, p, sel, cnt, out, ws, L, false,
                   false, (cudaStream_t)stream, false, false, src);
}

namespace kt {
namespace {

// Whether the one-launch step applies: linear reps, at most one attention CTA
// per SM per segment and per selection unit, and the in-kernel selection
// buffers fit the attention kernel's scratch.  Sets CTAs per unit and
// candidates per CTA.
bool fused_plan(const kt_paged_kv* kv, const kt_sparse_params* p, int sms, int* ncpu,
                int* chunk_out, int* kk) {
  const bool multi = p->rep == KT_REP_FIX || p->rep == KT_REP_DYNAMIC;
  if (sms < 1 || sms > MAX_ATTN_CTAS) return false;
  const long long S = (long long)kv->batch * kv->num_kv_heads;
  const int SEL = p->head_mode == KT_HEAD_SHARED ? 1 : kv->num_kv_heads;
  const long long U = (long long)kv->batch * SEL;
  if (S > sms || U > sms) return false;
  const int nc = (int)(sms / U);
  const int cmax = kv->max_blocks_per_seq - p->initial_blocks - p->local_blocks;
  const int chunk = cmax > 0 ? (cmax + nc - 1) / nc : 1;
  const int k = p->top_k < chunk ? p->top_k : chunk;
  if (k > FUSED_KK_CAP || chunk > FUSED_MAX_CHUNK) return false;
  const int nkv = SEL == 1 ? kv->num_kv_heads : 1;
  const int Rw = p->rep == KT_REP_QUEST ? 2 : 1;
  const bool f32 = p->rep == KT_REP_MEAN;
  const int V = nkv * reps_rows(p) * D / (f32 ? 4 : 8);
  if (!multi && V > 256) return false;  // linear CUDA-core scoring: 8 vectors a lane
  if ((long long)V * 16 + 16 > ATTN_RING_BYTES / 2) return false;  // a block per staging round
  const long long nslots = (long long)nc * k;
  if (nslots > FUSED_MAX_SLOTS) return false;
  const int kmax = (int)(p->top_k < nslots ? p->top_k : nslots);
  if (fused_score_layout(multi ? 0 : nkv * Rw * D, chunk, k).total > ATTN_SCRATCH_BYTES)
    return false;
  if (fused_pick_layout((int)nslots, kmax).total > ATTN_MERGE_BYTES) return false;
  // block ids and pages in tagged slots
  if (kv->max_blocks_per_seq > FUSED_MAX_BLOCKS || kv->num_pages > FUSED_MAX_PAGES) return false;
  if (attn_fused_max_ctas_per_sm() < 1) return false;
  *ncpu = nc;
  *chunk_out = chunk;
  *kk = k;
  return true;
}

}  // namespace
}  // namespace kt

int32_t kt_sparse_decode_step_kernels(const kt_paged_kv* kv, const kt_sparse_params* p) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return -(int32_t)s;
  s = check_params(kv, p);
  if (s != KT_OK) return -(int32_t)s;
  const int sms = cta_budget();
  int ncpu = 0, chunk = 0, kk = 0;
  return (sms > 0 && fused_plan(kv, p, sms, &ncpu, &chunk, &kk)) ? 1 : 2;
}

namespace kt {
namespace {

kt_status step_impl(const void* q, const kt_paged_kv* kv, const void* reps_pool,
                    const kt_sparse_params* p, const uint32_t* presel_mask,
                    const int32_t* presel_cnt, int32_t* sel, int32_t* cnt, float* out, void* ws,
                    size_t ws_bytes, kt_stream_t stream, int skip_publish = 0,
                    unsigned long long poll_limit_ns = 0, bool fused_only = false,
                    bool q_mapped = false, const KvSource& src = KvSource()) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q || !reps_pool || !sel || !cnt || !out || !ws || !aligned16(q) ||
      !aligned16(reps_pool) || !aligned16(out) || !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  const WsLayout L = layout(KT_OP_SPARSE_STEP, kv, p, 0);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  const int sms = cta_budget();
  int ncpu = 0, chunk = 0, kk = 0;
  if (sms > 0 && fused_plan(kv, p, sms, &ncpu, &chunk, &kk)) {
    // one launch: selection inside the attention kernel
    CUtensorMap kmap, vmap;
    const bool codes = src.kvm == KVM_Q8;
    if (!make_pool_map(&kmap, codes ? src.k_src : kv->k_pool, kv, codes) ||
        !make_pool_map(&vmap, codes ? src.v_src : kv->v_pool, kv, codes))
      return KT_ERR_CUDA;
    AttnLaunch a;
    std::memset(&a, 0, sizeof(a));
    a.kmap = &kmap;
    a.vmap = &vmap;
    a.kvm = src.kvm;
    a.k_src = src.k_src;
    a.v_src = src.v_src;
    a.k_scale = src.k_scale;
    a.v_scale = src.v_scale;
    a.q = static_cast<const __half*>(q);
    a.table = kv->block_table;
    a.seq_lens = kv->seq_lens;
    a.out = out;
    a.status = at<int>(ws, L.status);
    a.counters = at<int>(ws, L.attn_counters);
    a.parts = at<float>(ws, L.attn_parts);
    a.B = kv->batch;
    a.H_kv = kv->num_kv_heads;
    a.G = p->num_q_heads / kv->num_kv_heads;
    a.max_blocks = kv->max_blocks_per_seq;
    a.P = kv->num_pages;
    a.I_b = p->initial_blocks;
    a.L_b = p->local_blocks;
    a.top_k = p->top_k;
    a.SEL = p->head_mode == KT_HEAD_SHARED ? 1 : kv->num_kv_heads;
    a.dense = 0;
    a.slot_floats = L.slot_floats;
    a.scale_log2 = (float)((double)p->softmax_scale * 1.4426950408889634);
    a.grid = sms;
    a.fused = true;
    {
      const int nkv = a.SEL == 1 ? kv->num_kv_heads : 1;
      const int V = nkv * reps_rows(p) * D / (p->rep == KT_REP_MEAN ? 4 : 8);
      a.sk = fused_score_kind(p->rep, V, chunk, p->top_k);
    }
    a.reps = reps_pool;
    a.rep = p->rep;
    a.R = reps_rows(p);
    a.ncpu = ncpu;
    a.f_chunk = chunk;
    a.kk_f = kk;
    a.f_cand = at<unsigned long long>(ws, L.f_cand);
    a.f_cand_len = (int)L.f_cand_slots;
    a.f_cpage = at<uint32_t>(ws, L.f_cpage);
    a.f_sync = at<unsigned long long>(ws, L.f_sync);
    a.sel_out = sel;
    a.cnt_out = cnt;
    a.presel_mask = presel_mask;
    a.presel_cnt = presel_cnt;
    a.mask_words = mask_words_of(kv);
    a.stamps = stamps_for(a.grid);
    a.skip_publish = skip_publish;
    a.poll_limit_ns = poll_limit_ns;
    a.q_mapped = q_mapped;
    return cuda_status(launch_attention(a, (cudaStream_t)stream));
  }
  if (fused_only || q_mapped) return KT_ERR_UNSUPPORTED;
  s = select_impl(q, kv, reps_pool, p, sel, cnt, nullptr, ws, L, true, (cudaStream_t)stream,
                  presel_mask);
  if (s != KT_OK) return s;
  return attn_impl(q, kv, p->num_q_heads, p->softmax_scale, p, sel, cnt, out, ws, L, false, true,
                   (cudaStream_t)stream, true, presel_mask != nullptr, src);
}

}  // namespace
}  // namespace kt

kt_status kt_sparse_decode_step(const void* q, const kt_paged_kv* kv, const void* reps_pool,
                                const kt_sparse_params* p, int32_t* sel, int32_t* cnt,
                                float* out, void* ws, size_t ws_bytes, kt_stream_t stream) {
  return step_impl(q, kv, reps_pool, p, nullptr, nullptr, sel, cnt, out, ws, ws_bytes, stream);
}

kt_status kt_sparse_decode_step_q8_0(const void* q, const kt_paged_kv_q8* kvq,
                                     const void* reps_pool, const kt_sparse_params* p,
                                     int32_t* sel, int32_t* cnt, float* out, void* ws,
                                     size_t ws_bytes, kt_stream_t stream) {
  if (!kvq) return KT_ERR_INVALID_ARG;
  const kt_paged_kv kv = kv_view_q8(kvq);
  if (!kvq->k_scale || !kvq->v_scale || !aligned16(kvq->k_scale) || !aligned16(kvq->v_scale))
    return KT_ERR_INVALID_ARG;
  KvSource src;
  src.kvm = KVM_Q8;
  src.k_src = kvq->k_code;
  src.v_src = kvq->v_code;
  src.k_scale = kvq->k_scale;
  src.v_scale = kvq->v_scale;
  return step_impl(q, &kv, reps_pool, p, nullptr, nullptr, sel, cnt, out, ws, ws_bytes, stream, 0,
                   0, false, false, src);
}

kt_status kt_sparse_decode_step_presel(const void* q, const kt_paged_kv* kv,
                                       const void* reps_pool, const kt_sparse_params* p,
                                       const uint32_t* presel_mask, const int32_t* presel_cnt,
                                       int32_t* sel, int32_t* cnt, float* out, void* ws,
                                       size_t ws_bytes, kt_stream_t stream) {
  if (!presel_mask || !presel_cnt) return KT_ERR_INVALID_ARG;
  return step_impl(q, kv, reps_pool, p, presel_mask, presel_cnt, sel, cnt, out, ws, ws_bytes,
                   stream);
}

kt_status kt_sparse_decode_step_host(const void* q_host, void* q_dev, const kt_paged_kv* kv,
                                     const void* reps_pool, const kt_sparse_params* p,
                                     int32_t* sel, int32_t* cnt, float* out_dev,
                                     float* out_host, void* ws, size_t ws_bytes,
                                     kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q_host || !out_host) return KT_ERR_INVALID_ARG;
  const size_t qbytes = (size_t)kv->batch * p->num_q_heads * D * 2;
  const size_t obytes = (size_t)kv->batch * p->num_q_heads * D * 4;
  cudaStream_t st = (cudaStream_t)stream;
  if (!q_dev && !out_dev) {
    // page-locked host buffers mapped for the device: the step kernel reads
    // the query and writes the output over the link (no copies)
    const void* qd = host_pool_device_ptr(q_host);
    const void* od = host_pool_device_ptr(out_host);
    if (!qd || !od || !aligned16(qd) || !aligned16(od)) return KT_ERR_INVALID_ARG;
    s = step_impl(qd, kv, reps_pool, p, nullptr, nullptr, sel, cnt,
                  static_cast<float*>(const_cast<void*>(od)), ws, ws_bytes, stream, 0, 0, false,
                  true);
    if (s != KT_OK) return s;
    return cuda_status(cudaStreamSynchronize(st));
  }
  if (!q_dev || !out_dev) return KT_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(q_dev, q_host, qbytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return KT_ERR_CUDA;
  s = kt_sparse_decode_step(q_dev, kv, reps_pool, p, sel, cnt, out_dev, ws, ws_bytes, stream);
  if (s != KT_OK) return s;
  if (cudaMemcpyAsync(out_host, out_dev, obytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return KT_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(st));
}

kt_status kt_dense_decode_attn(const void* q, const kt_paged_kv* kv, int32_t num_q_heads,
                               float softmax_scale, float* out, void* ws, size_t ws_bytes,
                               kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_heads(kv, num_q_heads, softmax_scale);
  if (s != KT_OK) return s;
  if (!q || !out || !ws || !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return KT_ERR_INVALID_ARG;
  kt_sparse_params p;
  std::memset(&p, 0, sizeof(p));
  p.num_q_heads = num_q_heads;
  p.softmax_scale = softmax_scale;
  p.top_k = 1;
  p.local_blocks = 1;
  const WsLayout L = layout(KT_OP_DENSE_ATTN, kv, &p, 0);
  if (ws_bytes < L.total) return KT_ERR_WORKSPACE_TOO_SMALL;
  return attn_impl(q, kv, num_q_heads, softmax_scale, &p, nullptr, nullptr, out, ws, L, true,
                   false, (cudaStream_t)stream);
}

// ---- decoding with selection reuse [LC §4.5, §4.6 decode loop] --------------

namespace {
bool policy_ok(const kt_reuse_policy* pol) {
  return pol && pol->num_layers >= 1 && pol->dense_layer_num >= 0 &&
         pol->dense_layer_num <= pol->num_layers && pol->layer_step >= 1 && pol->token_step >= 1;
}
}  // namespace

int32_t kt_decode_history_slots(const kt_reuse_policy* pol) {
  if (!policy_ok(pol)) return -(int32_t)KT_ERR_INVALID_ARG;
  const int sparse = pol->num_layers - pol->dense_layer_num;
  return (sparse + pol->layer_step - 1) / pol->layer_step;
}

kt_status kt_decode_layer_action(const kt_reuse_policy* pol, int32_t token_idx,
                                 int32_t layer_idx, int32_t* action, int32_t* slot) {
  if (!policy_ok(pol) || !action || !slot || token_idx < 0 || layer_idx < 0 ||
      layer_idx >= pol->num_layers)
    return KT_ERR_INVALID_ARG;
  if (layer_idx < pol->dense_layer_num) {
    *action = KT_LAYER_DENSE;
    *slot = -1;
    return KT_OK;
  }
  const int l = layer_idx - pol->dense_layer_num;  // index among the sparse layers
  *slot = l / pol->layer_step;
  *action = (token_idx % pol->token_step == 0 && l % pol->layer_step == 0) ? KT_LAYER_SELECT
                                                                            : KT_LAYER_REUSE;
  return KT_OK;
}

kt_status kt_decode_layer(const kt_reuse_policy* pol, int32_t token_idx, int32_t layer_idx,
                          const void* q, const kt_paged_kv* kv, const void* reps_pool,
                          const kt_sparse_params* p, int32_t* hist_sel, int32_t* hist_cnt,
                          float* out, void* ws, size_t ws_bytes, kt_stream_t stream) {
  int32_t action = 0, slot = 0;
  kt_status s = kt_decode_layer_action(pol, token_idx, layer_idx, &action, &slot);
  if (s != KT_OK) return s;
  if (!kv || !p) return KT_ERR_INVALID_ARG;
  if (action == KT_LAYER_DENSE)
    return kt_dense_decode_attn(q, kv, p->num_q_heads, p->softmax_scale, out, ws, ws_bytes,
                                stream);
  if (!hist_sel || !hist_cnt || p->top_k < 1 || p->top_k > MAX_TOPK) return KT_ERR_INVALID_ARG;
  const int SEL = p->head_mode == KT_HEAD_SHARED ? 1 : kv->num_kv_heads;
  const size_t units = (size_t)kv->batch * SEL;
  int32_t* sel = hist_sel + (size_t)slot * units * p->top_k;
  int32_t* cnt = hist_cnt + (size_t)slot * units;
  if (action == KT_LAYER_SELECT)
    return kt_sparse_decode_step(q, kv, reps_pool, p, sel, cnt, out, ws, ws_bytes, stream);
  return kt_sparse_decode_attn(q, kv, p, sel, cnt, out, ws, ws_bytes, stream);
}

kt_status kt_append_kv(const kt_paged_kv* kv, const kt_sparse_params* p, const void* k_new,
                       const void* v_new, void* reps_pool, void* ws, size_t ws_bytes,
                       kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!k_new || !v_new || !ws || ws_bytes < 256 || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned16(ws) || (reps_pool && !aligned16(reps_pool)))
    return KT_ERR_INVALID_ARG;
  AppendLaunch a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_pool = const_cast<void*>(kv->k_pool);
  a.v_pool = const_cast<void*>(kv->v_pool);
  a.table = kv->block_table;
  a.seq_lens = const_cast<int32_t*>(kv->seq_lens);
  a.status = at<int>(ws, 0);
  a.B = kv->batch;
  a.H_kv = kv->num_kv_heads;
  a.max_blocks = kv->max_blocks_per_seq;
  a.P = kv->num_pages;
  cudaError_t e = launch_append(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return KT_ERR_CUDA;
  if (!reps_pool || p->rep == KT_REP_DYNAMIC) return KT_OK;
  // the reps of the blocks this token completed
  RepsLaunch r;
  r.k_pool = static_cast<const __half*>(kv->k_pool);
  r.table = kv->block_table;
  r.seq_lens = kv->seq_lens;
  r.reps = reps_pool;
  r.B = kv->batch;
  r.H_kv = kv->num_kv_heads;
  r.max_blocks = kv->max_blocks_per_seq;
  r.P = kv->num_pages;
  r.rep = p->rep;
  r.R = reps_rows(p);
  r.fix_stride = p->fix_stride;
  r.first_block = -1;
  r.num_blocks = 1;
  return cuda_status(launch_reps(r, (cudaStream_t)stream));
}

kt_status kt_read_device_status(void* ws, size_t ws_bytes, kt_stream_t stream,
                                int32_t* device_status) {
  if (!ws || ws_bytes < 256 || !device_status) return KT_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KT_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return KT_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(v), st) != cudaSuccess) return KT_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KT_ERR_CUDA;
  *device_status = v;
  return KT_OK;
}

kt_status kt_set_phase_stamps(void* stamps, int32_t max_ctas) {
  if (stamps && ((reinterpret_cast<uintptr_t>(stamps) & 7u) != 0 || max_ctas < 1))
    return KT_ERR_INVALID_ARG;
  stamps_buf = static_cast<unsigned long long*>(stamps);
  stamps_max_ctas = stamps ? max_ctas : 0;
  return KT_OK;
}

kt_status kt_set_max_ctas(int32_t max_ctas) {
  if (max_ctas < 0) return KT_ERR_INVALID_ARG;
  max_ctas_cap = max_ctas;
  return KT_OK;
}

kt_status kt_selftest_step_timeout(const void* q, const kt_paged_kv* kv, const void* reps_pool,
                                   const kt_sparse_params* p, int32_t* sel, int32_t* cnt,
                                   float* out, void* ws, size_t ws_bytes, int32_t skip_cta,
                                   int32_t poll_limit_us, kt_stream_t stream) {
  if (skip_cta < 0 || poll_limit_us < 1) return KT_ERR_INVALID_ARG;
  return step_impl(q, kv, reps_pool, p, nullptr, nullptr, sel, cnt, out, ws, ws_bytes, stream,
                   skip_cta + 1, (unsigned long long)poll_limit_us * 1000ull, true);
}

kt_status kt_selftest_bounded_wait(void* ws, size_t ws_bytes, int32_t spin_limit,
                                   kt_stream_t stream) {
  if (!ws || ws_bytes < 256 || spin_limit < 1) return KT_ERR_INVALID_ARG;
  return cuda_status(
      launch_selftest_wait(static_cast<int*>(ws), spin_limit, (cudaStream_t)stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of kt_sparse_decode_attn: the scratch memory lives in
// a fixed-size array of this library's device image instead of a caller
// workspace.
// ---------------------------------------------------------------------------
namespace kt {
namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(1) << 20;  // 1 MiB on every device
static __device__ __align__(256) unsigned char noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex noalloc_mu;
void* noalloc_dev_ptr[NOALLOC_MAX_DEVICES];  // device address of the array, per device

// Device address of the scratch array on the current device.  The name
// `noalloc_scratch` is only a host-side stand-in; the address has to come from
// cudaGetSymbolAddress with the device current.  Done once per device.
kt_status noalloc_scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES)
    return KT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(noalloc_mu);
  if (!noalloc_dev_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, noalloc_scratch) != cudaSuccess || !p) return KT_ERR_CUDA;
    noalloc_dev_ptr[dev] = p;
  }
  *out = noalloc_dev_ptr[dev];
  return KT_OK;
}

}  // namespace
}  // namespace kt

extern "C" kt_status kt_sparse_decode_attn_noalloc(const void* q, const kt_paged_kv* kv,
                                                   const kt_sparse_params* p, const int32_t* sel,
                                                   const int32_t* cnt, float* out,
                                                   kt_stream_t stream) {
  kt_status s = check_kv(kv);
  if (s != KT_OK) return s;
  s = check_params(kv, p);
  if (s != KT_OK) return s;
  if (!q || !sel || !cnt || !out || !aligned16(q) || !aligned16(out)) return KT_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms <= 0) return KT_ERR_CUDA;
  const int S = kv->batch * kv->num_kv_heads;
  const int G = p->num_q_heads / kv->num_kv_heads;
  const int slot_floats = ((2 * G + G * D) + 3) & ~3;
  const int base = sms < MAX_ATTN_CTAS ? sms : MAX_ATTN_CTAS;
  const int grid = base > S ? base : S;
  // status word, one ticket counter per segment, one partial per CTA
  const size_t counters_off = 256;
  const size_t parts_off = align256(counters_off + (size_t)S * 4);
  const size_t need = parts_off + (size_t)grid * slot_floats * 4;
  if (need > NOALLOC_SCRATCH_BYTES) return KT_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  s = noalloc_scratch_ptr(&scratch);
  if (s != KT_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the status word and the
  // tickets must start at zero
  if (cudaMemsetAsync(scratch, 0, parts_off, st) != cudaSuccess) return KT_ERR_CUDA;
  CUtensorMap kmap, vmap;
  if (!make_pool_map(&kmap, kv->k_pool, kv) || !make_pool_map(&vmap, kv->v_pool, kv))
    return KT_ERR_CUDA;
  AttnLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.kmap = &kmap;
  a.vmap = &vmap;
  a.q = static_cast<const __half*>(q);
  a.table = kv->block_table;
  a.seq_lens = kv->seq_lens;
  a.sel = sel;
  a.cnt = cnt;
  a.sel_pages = nullptr;
  a.out = out;
  a.status = at<int>(scratch, 0);
  a.counters = at<int>(scratch, counters_off);
  a.parts = at<float>(scratch, parts_off);
  a.B = kv->batch;
  a.H_kv = kv->num_kv_heads;
  a.G = G;
  a.max_blocks = kv->max_blocks_per_seq;
  a.P = kv->num_pages;
  a.I_b = p->initial_blocks;
  a.L_b = p->local_blocks;
  a.top_k = p->top_k;
  a.SEL = p->head_mode == KT_HEAD_SHARED ? 1 : kv->num_kv_heads;
  a.dense = 0;
  a.slot_floats = slot_floats;
  a.scale_log2 = (float)((double)p->softmax_scale * 1.4426950408889634);
  a.grid = grid;
  a.pdl = false;
  return cuda_status(launch_attention(a, st));
}

extern "C" kt_status kt_noalloc_read_status(kt_stream_t stream, int32_t* device_status) {
  if (!device_status) return KT_ERR_INVALID_ARG;
  void* scratch = nullptr;
  kt_status s = noalloc_scratch_ptr(&scratch);
  if (s != KT_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KT_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return KT_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, sizeof(v), st) != cudaSuccess) return KT_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KT_ERR_CUDA;
  *device_status = v;
  return KT_OK;
}
