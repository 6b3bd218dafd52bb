// kt_internal.cuh — constants, workspace layout and sm_103a device helpers
// shared by the libkt translation units (not part of the public ABI).
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kt.h"

namespace kt {

constexpr int D = 128;              // head_dim
constexpr int BS = 128;             // tokens per KV block
constexpr int MAX_G = 8;            // query heads per KV head
constexpr int MAX_SEGS = 2048;      // batch * num_kv_heads
constexpr int MAX_TOPK = 1024;
constexpr int MAX_ATTN_CTAS = 1024; // workspace is sized for this many attention CTAs
constexpr int SEL_TARGET_CTAS = 1024;
constexpr int SEL_MAX_CAND = 8192;  // candidates merged by the last selection CTA
constexpr int SEL_MAX_CHUNK = 4096; // context blocks scored by one selection CTA
constexpr int MAX_DYN_REPS = 32;
constexpr int ATTN_SCRATCH_BYTES = 4 * MAX_G * (D + 2) * 4;  // attention kernel scratch (smem)
constexpr int FUSED_KK_CAP = 256;  // per-CTA candidates of the fused step
constexpr int ATTN_CONSUMER_THREADS = 256;  // consumer threads of the attention kernel
constexpr int ATTN_RING_BYTES = 3 * 4 * 128 * 64 * 2;  // attention KV ring (3 stages x 64 KB)
constexpr int FUSED_GATHER_PER_THREAD = 8;  // candidate slots a merging thread holds
constexpr int FUSED_MAX_SLOTS = FUSED_GATHER_PER_THREAD * ATTN_CONSUMER_THREADS;
constexpr int FUSED_MAX_CHUNK = 8 * ATTN_CONSUMER_THREADS;  // blocks one CTA scores (keys held in registers)

// Byte offsets inside the attention kernel's scratch for the in-kernel
// selection of the fused step.  Scoring: weights (fp32), keys and page ids of
// the CTA's Context slice, and the top-k temporaries when the slice holds more
// than kk blocks.  Merge: every candidate key and page of the unit, the chosen
// indices, their block ids (padded to a multiple of 4) and the top-k
// temporaries.
// Scoring paths of the one-launch step, one kernel instantiation each (the
// kernel runs most of its code once per launch, so it carries only the path
// it uses): few fp16 blocks per CTA with 64/128/256 16-byte columns on the CUDA
// cores (COLS), few fp16 blocks otherwise (LINEAR), many fp16 blocks on the
// tensor cores (MMA), fp32 reps (F32), several reps per block (MULTI).
enum : int { SK_NONE = 0, SK_COLS = 1, SK_LINEAR = 2, SK_MMA = 3, SK_F32 = 4, SK_MULTI = 5 };
// Where the attention-only kernel reads K and V: fp16 pools in device memory
// (2-D TMA), fp16 pools in host memory the GPU reads over NVLink-C2C (16-byte
// cp.async by the producer warp), or Q8_0 pools in device memory (TMA of the
// int8 codes and bulk copies of the binary16 scales, dequantised per warp).
enum : int { KVM_F16 = 0, KVM_HOST = 1, KVM_Q8 = 2 };
// the most fp16 blocks a CTA scores on the CUDA cores in one pass
__host__ __device__ inline int fused_lin_max(int V) {
  return 8 * (ATTN_CONSUMER_THREADS / 32) / (V <= 32 ? 1 : V <= 64 ? 2 : V <= 128 ? 4 : 8);
}
// COLS also needs every slice to be its own candidate list (chunk <= top_k),
// so it carries no per-slice top-k
__host__ __device__ inline int fused_score_kind(int rep, int V, int chunk, int top_k) {
  if (rep == KT_REP_FIX || rep == KT_REP_DYNAMIC) return SK_MULTI;
  if (rep == KT_REP_MEAN) return SK_F32;
  if (chunk > fused_lin_max(V)) return SK_MMA;
  return ((V == 64 || V == 128 || V == 256) && chunk <= top_k) ? SK_COLS : SK_LINEAR;
}

struct FusedScoreLayout {
  int keys, pgs, total;
};
// A slice of more blocks than its slots finds its threshold in the scratch
// from offset 0 once its keys and pages are in registers: 2048 bins, the
// boundary bin's keys, then the slot counter.
constexpr int FUSED_KTH_BINK = 2048 * 4;
constexpr int FUSED_KTH_COUNTS = FUSED_KTH_BINK + ATTN_CONSUMER_THREADS * 8;
constexpr int FUSED_KTH_END = FUSED_KTH_COUNTS + 16;
__host__ __device__ inline FusedScoreLayout fused_score_layout(int wfl, int chunk, int kk) {
  FusedScoreLayout L;
  L.keys = (wfl * 4 + 15) & ~15;
  L.pgs = L.keys + ((chunk + 1) & ~1) * 8;  // keys padded to an even count
  L.total = L.pgs + chunk * 4;
  if (chunk > kk && L.total < FUSED_KTH_END) L.total = FUSED_KTH_END;
  return L;
}
// Pick: the 2048-bin histogram and the boundary-bin keys of the threshold
// search (the unit's keys themselves stay in registers), the chosen block ids,
// their pages, and both in ascending id order (this CTA's share is read from
// there by the producer).  Lives in the attention kernel's scratch and block-prefix
// areas, which are contiguous.
struct FusedPickLayout {
  int hist, bink, ids, pages, sorted, sorted_pages, total;
};
__host__ __device__ inline FusedPickLayout fused_pick_layout(int nslots, int kmax) {
  FusedPickLayout L;
  (void)nslots;
  const int kpad = (kmax + 3) & ~3;
  L.hist = 0;
  L.bink = 2048 * 4;
  L.ids = L.bink + ATTN_CONSUMER_THREADS * 8;
  L.pages = L.ids + kpad * 4;
  L.sorted = L.pages + kpad * 4;
  L.sorted_pages = L.sorted + kpad * 4;
  L.total = L.sorted_pages + kpad * 4;
  return L;
}
// Candidate slots of the one-launch step carry the launch's tag in their low
// 12 bits, so a reader can tell a slot written by this launch from a stale one
// without any fence: 8-byte words are written and read whole.  A slot holds
// (score bits << 32) | ((2^20 - 1 - block) << 12) | tag, which orders as the
// selection key (score, then lower block) for block ids below 2^20; an empty
// slot is the tag alone.  Beside each key slot a 4-byte page slot holds
// (page << 12) | tag, for pages below 2^20.  Tags cycle through 1..4095 (launch epoch modulo
// 4095, plus one).  Every launch writes every slot of the region once (its
// own slots with its tag, the rest with tag 0), so before a launch writes a
// slot it holds the previous launch's tag or 0, never the live one.
//
// Launch epoch: a 64-bit counter in the workspace to which the CTAs of every
// launch add shares summing to 2^FUSED_EPOCH_SHIFT (CTA c adds
// floor((c+1) 2^s / grid) - floor(c 2^s / grid), at least 1 for grids up to
// 2^s), fire-and-forget.  A CTA reading the counter during launch N sees
// N 2^s plus the shares of CTAs of launch N other than itself, less than 2^s,
// so counter >> s is N in every CTA of the launch.
constexpr int FUSED_MAX_BLOCKS = (1 << 20) - 1;
constexpr int FUSED_MAX_PAGES = (1 << 20) - 1;
constexpr uint32_t FUSED_TAG_BITS = 12;
constexpr uint32_t FUSED_TAG_CYCLE = 4095;
constexpr int FUSED_EPOCH_SHIFT = 20;
constexpr int ATTN_MERGE_BYTES = ATTN_SCRATCH_BYTES + (MAX_SEGS + 1) * 4;
constexpr uint64_t WAIT_LIMIT_NS = 100000000ull;  // 100 ms bound on any device-side wait
constexpr int KT_PHASE_STAMPS = 16;               // phase stamps per CTA (kt_set_phase_stamps)

// ---------------------------------------------------------------------------
// Selection chunking and workspace layout.  Host sizing and device addressing
// use this one description.  All regions are 256-byte aligned.
// ---------------------------------------------------------------------------
struct SelPlan {
  int SEL;      // selection units per sequence (1 or H_kv)
  int max_ctx;  // upper bound on Context blocks of a sequence
  int chunk;    // Context blocks scored by one CTA
  int nchunks;  // CTAs per unit
  int kk;       // candidates kept per chunk
};

struct WsLayout {
  size_t status;         // int32 status word, 256 B header
  size_t sel_counters;   // int32 [B*SEL]
  size_t sel_cand;       // uint64 [B*SEL*nchunks*kk]
  size_t sel_cand_pages; // int32 [B*SEL*nchunks*kk], page id of each candidate
  size_t sel_pages;      // int32 [B*SEL*top_k], page ids of the selection (step path)
  size_t f_sync;         // uint64 fused step: launch counter (epoch = counter >> FUSED_EPOCH_SHIFT)
  size_t f_cand;         // uint64 [MAX_ATTN_CTAS * min(top_k, FUSED_KK_CAP)] tagged slots
  size_t f_cand_slots;   // slots in that region
  size_t f_cpage;        // uint32, one page slot per candidate slot
  size_t attn_counters;  // int32 [S]
  size_t attn_parts;     // float [2*(MAX_ATTN_CTAS+S)][slot_floats]
  size_t dyn;            // dynamic-rep scratch
  size_t dyn_bytes;
  size_t presel_votes;   // preselection: token votes [B][H_kv][max_blocks*128] fp32
  size_t presel_bscore;  // preselection: block scores [B][SEL][max_blocks] fp32
  size_t total;
  int slot_floats;
  SelPlan sel;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int ceil_div_i(long long a, long long b) { return (int)((a + b - 1) / b); }

inline SelPlan make_sel_plan(int B, int H_kv, int max_blocks, int I, int L, int top_k,
                             int head_mode) {
  SelPlan s;
  s.SEL = head_mode == KT_HEAD_SHARED ? 1 : H_kv;
  const int mc = max_blocks - I - L;
  s.max_ctx = mc > 0 ? mc : 0;
  const long long total = (long long)B * s.SEL * (s.max_ctx > 0 ? s.max_ctx : 1);
  int ch = ceil_div_i(total, SEL_TARGET_CTAS);
  if (ch < 8) ch = 8;
  int nch = s.max_ctx > 0 ? ceil_div_i(s.max_ctx, ch) : 1;
  int kk = top_k < ch ? top_k : ch;
  if ((long long)nch * kk > SEL_MAX_CAND) {
    // larger chunks so that nchunks * top_k candidates fit the merge buffer
    ch = ceil_div_i(s.max_ctx, SEL_MAX_CAND / (top_k > 0 ? top_k : 1));
    if (ch < 8) ch = 8;
    nch = ceil_div_i(s.max_ctx, ch);
    kk = top_k < ch ? top_k : ch;
  }
  s.chunk = ch;
  s.nchunks = nch;
  s.kk = kk;
  return s;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ unsigned long long fused_slot(unsigned long long key, uint32_t tag) {
  return (key & 0xFFFFFFFF00000000ull) |
         (static_cast<unsigned long long>(static_cast<uint32_t>(key) & 0xFFFFFu) << FUSED_TAG_BITS) |
         tag;
}
__device__ __forceinline__ int fused_slot_block(unsigned long long slot) {
  return 0xFFFFF - static_cast<int>((slot >> FUSED_TAG_BITS) & 0xFFFFFull);
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_gpu_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Named barrier `id` over `nthreads` threads that also returns, to every one
// of them, whether `pred` held in all of them.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void set_status(int* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of the barrier; gives up after WAIT_LIMIT_NS of
// global time, records KT_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer() - t0 > WAIT_LIMIT_NS) {
      set_status(status, KT_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-D tiled TMA load (global -> shared), completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Untiled bulk copy (global -> shared); 16-byte aligned addresses and size.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same m16n8k16 step as a plain asm statement (registers only), which
// the compiler may schedule freely between independent accumulator chains.
__device__ __forceinline__ void mma_16816_sched(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte asynchronous copy global -> shared (L2 only), 16-byte aligned both.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrival on `bar` once every cp.async this thread issued before it has
// landed; counts as one of the barrier's expected arrivals.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Ticket counters: a CTA's writes are ordered before its ticket by a CTA
// barrier followed by one thread's acq_rel add (release is cumulative over
// what the barrier made visible to that thread); the thread that takes the
// last ticket acquires, and a CTA barrier then orders the other threads' reads.
__device__ __forceinline__ int atom_acq_rel_gpu_add(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// Shared-memory matrix descriptor of a K-major operand stored with the
// 128-byte swizzle (rows of 64 fp16, 8-row groups of 1024 bytes, as TMA
// writes a {64, rows} box): start address, stride between 8-row groups,
// descriptor version 1, swizzle mode 128B.  A K-step of 16 elements inside the
// 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;            // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024u >> 4) << 32;  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1u << 46;            // version
  d |= (uint64_t)2u << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B (both K-major), fp32
// accumulation, M x N tile.
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[sdesc a] . B[sdesc b]^T, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4) .. +31; taddr carries that lane base).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

// Order-preserving map float -> uint32 (larger float, larger key; -0 == +0).
__device__ __forceinline__ uint32_t float_key(float f) {
  if (f == 0.0f) f = 0.0f;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

#endif  // __CUDACC__

// ---------------------------------------------------------------------------
// Host: a value computed once per device (the current one) and cached; the
// launch path calls these on every step.
// ---------------------------------------------------------------------------
constexpr int KT_MAX_DEVICES = 64;
template <class F>
inline int per_device_cached(std::atomic<int> (&slot)[KT_MAX_DEVICES], F compute) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= KT_MAX_DEVICES) return compute();
  const int v = slot[dev].load(std::memory_order_relaxed);
  if (v != 0) return v - 1;
  const int r = compute();
  slot[dev].store(r + 1, std::memory_order_relaxed);
  return r;
}

// ---------------------------------------------------------------------------
// Launch entry points implemented in the kernel translation units.
// ---------------------------------------------------------------------------
struct AttnLaunch {
  const CUtensorMap* kmap;
  const CUtensorMap* vmap;
  const __half* q;
  const int32_t* table;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* cnt;        // nullable: then min(top_k, C) blocks were selected
  const int32_t* sel_pages;  // nullable: page ids of sel (skips the table lookup)
  float* out;
  int* status;
  int* counters;
  float* parts;
  int B, H_kv, G, max_blocks, P, I_b, L_b, top_k, SEL, dense, slot_floats;
  float scale_log2;
  int grid;
  bool pdl;  // launched as a programmatic dependent of the previous kernel
  bool q_mapped;  // q and out are page-locked host memory read and written over the link
  // fused step (selection inside the attention kernel, cooperative launch)
  bool fused;
  int sk;  // fused: the scoring path (SK_*)
  const void* reps;
  int rep, R;
  int ncpu;     // CTAs scoring one selection unit
  int f_chunk;  // Context blocks per scoring CTA (nominal, from max_blocks)
  int kk_f;     // candidates kept per scoring CTA
  unsigned long long* f_cand;  // tagged candidate slots [B*SEL][ncpu][kk_f]
  int f_cand_len;              // slots in the workspace region (zeroed when tags wrap)
  uint32_t* f_cpage;           // the page slot of each candidate slot
  unsigned long long* f_sync;  // launch counter (epoch = counter >> FUSED_EPOCH_SHIFT)
  int32_t* sel_out;
  int32_t* cnt_out;
  const uint32_t* presel_mask;  // nullable [B][SEL][mask_words]
  const int32_t* presel_cnt;    // with presel_mask: blocks preselected per unit
  int mask_words;
  unsigned long long* stamps;   // nullable: [grid][KT_PHASE_STAMPS] global-timer stamps
  // attention-only kernel, KV source (KVM_*): KVM_HOST reads k_src / v_src
  // (device-accessible host pools, fp16); KVM_Q8 reads the int8 codes through
  // kmap / vmap and the binary16 scales [pages][H_kv][128][4] at k_scale / v_scale
  int kvm;
  const void* k_src;
  const void* v_src;
  const void* k_scale;
  const void* v_scale;
  // one-launch step, failure-path test only: CTA skip_publish - 1 publishes
  // no candidate slots (0: every CTA publishes), and the slot and partial
  // polls give up after poll_limit_ns (0: the usual bound)
  int skip_publish;
  unsigned long long poll_limit_ns;
};
int attn_fused_max_ctas_per_sm();
cudaError_t launch_attention(const AttnLaunch& a, cudaStream_t stream);

struct SelectLaunch {
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
  int32_t* sel_pages;  // nullable
  int B, H_kv, G, max_blocks, P, I_b, L_b, top_k, rep, R, head_mode;
  SelPlan plan;
  bool trigger_dependents;
  const uint32_t* presel_mask;  // nullable: only these Context blocks compete
  int mask_words;
};
cudaError_t launch_select(const SelectLaunch& a, cudaStream_t stream);
size_t select_smem_bytes(const SelectLaunch& a);

// Q8_0 quantisation of pages [first_page, first_page + num_pages) of both pools.
struct QuantLaunch {
  const __half* k_pool;
  const __half* v_pool;
  int8_t* k_code;
  __half* k_scale;
  int8_t* v_code;
  __half* v_scale;
  int first_page, num_pages, H_kv;
};
cudaError_t launch_quant(const QuantLaunch& a, cudaStream_t stream);

struct RepsLaunch {
  const __half* k_pool;
  const int32_t* table;
  const int32_t* seq_lens;
  void* reps;
  int B, H_kv, max_blocks, P, rep, R, fix_stride, first_block, num_blocks;
};
cudaError_t launch_reps(const RepsLaunch& a, cudaStream_t stream);  // first_block < 0: completed tail blocks

struct AppendLaunch {
  const void* k_new;
  const void* v_new;
  void* k_pool;
  void* v_pool;
  const int32_t* table;
  int32_t* seq_lens;
  int* status;
  int B, H_kv, max_blocks, P;
};
cudaError_t launch_append(const AppendLaunch& a, cudaStream_t stream);

struct DynLaunch {
  const CUtensorMap* kmap;
  const __half* k_pool;
  const __half* q_local;
  const int32_t* table;
  const int32_t* seq_lens;
  void* ws;  // dynamic_ws_bytes(B, H_kv, max_blocks) bytes
  void* reps;
  float* token_scores;
  int* status;
  int B, H_kv, G, T, max_blocks, P, R, first_block, num_blocks, num_sms;
  float scale_log2;
};
cudaError_t launch_dynamic(const DynLaunch& a, cudaStream_t stream);
size_t dynamic_ws_bytes(int B, int H_kv, int max_blocks);
constexpr int MAX_DYN_ROWS = 256;  // local queries x query heads per KV head

struct PreselLaunch {
  const float* votes;  // [B][H_kv][max_blocks*128] token scores (Dynamic passes)
  const int32_t* seq_lens;
  float* bscore;       // workspace [B][SEL][max_blocks]
  uint32_t* mask;      // [B][SEL][mask_words]
  int32_t* cnt;        // [B][SEL]
  int* status;
  int B, H_kv, SEL, max_blocks, I_b, L_b, kernel, count, mask_words;
};
cudaError_t launch_preselect(const PreselLaunch& a, cudaStream_t stream);
size_t preselect_ws_bytes(int B, int H_kv, int SEL, int max_blocks);
size_t preselect_smem_bytes(int max_blocks, int mask_words);
constexpr int PRESEL_MAX_KERNEL = 65;

cudaError_t launch_selftest_wait(int* status, int spin_limit, cudaStream_t stream);

}  // namespace kt
