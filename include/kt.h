/*
 * kt.h — C ABI of libkt: block-sparse long-context decode attention on GB300.
 *
 * The method (KTransformers long-context sparse attention; article
 * "KTransformers 长上下文稀疏注意力实战：单张 24GB GPU 跑通 1M Token KVCache 的完整方案",
 * cited below as [LC §N]) keeps the whole KV cache, cut into fixed-size blocks,
 * and for each decode step attends to:
 *   - the Initial blocks at the head of the sequence          [LC §4.2]
 *   - the top-k Context blocks, ranked by representative keys [LC §4.3, §3.1]
 *   - the Local window at the tail                            [LC §4.2]
 * with exact softmax attention over that token set            [LC §4.6].
 * Parameter names follow the attention constructor and YAML keys of
 * "How to Implement Long Context Inference (Up to 139K Tokens) with
 * KTransformers" (Step 1, Step 3) and the parameter list of [LC §4.5].
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers unless a comment says otherwise.
 *     The caller owns every buffer, the workspace and the stream; the library
 *     never allocates or frees memory and never synchronises, except
 *     kt_read_device_status, kt_workspace_init (which only memsets) and the
 *     host-buffer convenience call kt_sparse_decode_step_host.
 *   - Calls are asynchronous: they validate their arguments on the host, launch
 *     on `stream` and return.  An invalid argument returns an error before any
 *     launch and has no side effect.  A failed launch returns KT_ERR_CUDA.
 *   - Device-side anomalies (a block-table entry outside the pool, a selected
 *     block outside the context range, a wait that ran out) never trap: the
 *     kernel records a kt_status code in the workspace's status word, skips the
 *     affected work and returns.  Read it with kt_read_device_status.
 *   - Element types: keys/values/queries are IEEE binary16 ("fp16"); outputs and
 *     Mean representatives are binary32.
 *   - Supported shapes: head_dim == 128, block_size == 128, num_q_heads a
 *     multiple of num_kv_heads with a group size G = num_q_heads/num_kv_heads
 *     of at most 8, batch * num_kv_heads <= 2048.  Other values return
 *     KT_ERR_UNSUPPORTED.
 *   - Alignment: every pointer must be 16-byte aligned (fp16 rows are 256 B).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 */
#ifndef KT_H_
#define KT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kt_stream_t; /* same type as cudaStream_t */

typedef enum {
  KT_OK = 0,
  KT_ERR_INVALID_ARG = 1,        /* null pointer, negative size, misaligned pointer */
  KT_ERR_UNSUPPORTED = 2,        /* valid but outside the supported shapes/methods */
  KT_ERR_WORKSPACE_TOO_SMALL = 3,
  KT_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
  KT_ERR_DEVICE_CHECK = 5,       /* device-side bounds check failed (work skipped) */
  KT_ERR_TIMEOUT = 6             /* a device-side bounded wait ran out */
} kt_status;

/* Representative-token methods [LC §4.3 table; Quest: §3.1]. */
typedef enum {
  KT_REP_MAX = 0,     /* per-channel max of the block's keys: 1 fp16 row */
  KT_REP_MEAN = 1,    /* per-channel exact mean, rounded once: 1 fp32 row */
  KT_REP_QUEST = 2,   /* per-channel min (row 0) and max (row 1): 2 fp16 rows */
  KT_REP_FIX = 3,     /* key rows at offsets 0, s, 2s, ...: 128/s fp16 rows */
  KT_REP_DYNAMIC = 4  /* key rows of the num_reps best-scored tokens, token order */
} kt_rep_method;

/* head_select_mode [LC §4.5]. */
typedef enum {
  KT_HEAD_SHARED = 0,   /* all query heads select one block set jointly */
  KT_HEAD_SEPARATE = 1  /* each KV head selects for its own query-head group */
} kt_head_mode;

/* Operations whose workspace size kt_workspace_bytes reports. */
typedef enum {
  KT_OP_SCORE_SELECT = 0,
  KT_OP_SPARSE_ATTN = 1,
  KT_OP_DENSE_ATTN = 2,
  KT_OP_SPARSE_STEP = 3,   /* score/select + sparse attention in one call */
  KT_OP_DYNAMIC_REPS = 4,
  KT_OP_PRESELECT = 5      /* kt_preselect_blocks (needs T like KT_OP_DYNAMIC_REPS) */
} kt_op;

/*
 * Paged KV cache [LC §4.3: the context is cut into fixed-size blocks].
 *   k_pool, v_pool : fp16 [num_pages][num_kv_heads][block_size][head_dim];
 *                    each (page, kv head) slab is contiguous.
 *   block_table    : int32 [batch][max_blocks_per_seq]; logical block j of
 *                    sequence b lives in page block_table[b][j].  Only entries
 *                    j < ceil(seq_lens[b] / block_size) are read.
 *   seq_lens       : int32 [batch]; tokens cached for each sequence (the decode
 *                    query attends to all of them, the current token included).
 * Pool rows past seq_lens[b] in the last page may hold any finite values.
 */
typedef struct {
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t max_blocks_per_seq;
  int32_t num_pages;
} kt_paged_kv;

/*
 * Selection parameters [LC §4.5; YAML keys of the "How to Implement..." page,
 * Step 1].
 *   num_q_heads    : query heads; head h reads KV head h / G.
 *   initial_blocks : Initial part, in blocks, always attended [LC §4.2].
 *   local_blocks   : Local window, in blocks (local_windows_len / block_size),
 *                    counted back from the last (possibly partial) block; >= 1.
 *   top_k          : second_select_num: context blocks selected per unit, 1..1024.
 *   num_reps       : anchor_num: reps per block for KT_REP_DYNAMIC (1..32).
 *   fix_stride     : token interval for KT_REP_FIX; divides block_size.
 *   rep            : kt_rep_method (anchor_type).
 *   head_mode      : kt_head_mode (head_select_mode).
 *   softmax_scale  : attention scale, normally 1/sqrt(head_dim) [LC §3.2].
 * When ceil(n/block_size) <= initial_blocks + local_blocks there is no Context
 * part and every block is attended.
 */
typedef struct {
  int32_t num_q_heads;
  int32_t initial_blocks;
  int32_t local_blocks;
  int32_t top_k;
  int32_t num_reps;
  int32_t fix_stride;
  int32_t rep;
  int32_t head_mode;
  float softmax_scale;
} kt_sparse_params;

/* Human-readable name of a status code (static string). */
const char* kt_status_string(kt_status s);

/* Representative rows per block for `p` (1, 2, block_size/fix_stride or num_reps);
 * 0 for an invalid method. */
int32_t kt_reps_per_block(const kt_sparse_params* p);

/*
 * Bytes of the representative pool for `kv`/`p`: layout
 * [num_pages][num_kv_heads][R][head_dim], fp16 (fp32 for KT_REP_MEAN).
 * Returns 0 for invalid arguments.
 */
size_t kt_reps_pool_bytes(const kt_paged_kv* kv, const kt_sparse_params* p);

/*
 * Workspace bytes needed by `op` for these shapes (host-only computation; no
 * device is touched).  T is the number of local queries for
 * KT_OP_DYNAMIC_REPS and KT_OP_PRESELECT and is ignored otherwise.  The
 * workspace holds the device status word, cross-CTA candidate lists, tickets,
 * launch counters and split-K partials.  It must be zero-filled before its
 * first use (kt_workspace_init); every call leaves it ready for the next.
 * Calls that share one workspace must not overlap on the GPU (issue them on
 * one stream).
 */
kt_status kt_workspace_bytes(kt_op op, const kt_paged_kv* kv, const kt_sparse_params* p,
                             int32_t T, size_t* bytes);

/* Zero-fills the workspace on `stream` (cudaMemsetAsync). */
kt_status kt_workspace_init(void* ws, size_t ws_bytes, kt_stream_t stream);

/*
 * Build representatives of logical blocks [first_block, first_block+num_blocks)
 * of every sequence, for rep in {MAX, MEAN, QUEST, FIX} [LC §4.3 table,
 * Quest: §3.1].  Only full blocks are built (partial tail blocks are always in
 * the Local window and never scored).  Results are written per physical page:
 * reps_pool[block_table[b][j]][kv_head][r][:].  Max/min are exact fp16 values
 * under the binary16 total order (-0 < +0); Mean is the exact per-channel mean
 * rounded once to fp32.  Reads K once (HBM-bound).  The device status word is
 * not available to this call (it takes no workspace); a block-table entry
 * outside the pool is skipped.
 */
kt_status kt_build_block_reps(const kt_paged_kv* kv, const kt_sparse_params* p,
                              int32_t first_block, int32_t num_blocks, void* reps_pool,
                              kt_stream_t stream);

/*
 * Dynamic representatives [LC §4.3 "Dynamic": accumulated attention score per
 * token, top-k tokens per block].  q_local: fp16 [batch][T][num_q_heads][128],
 * the queries of the last T positions n-T..n-1 of each sequence.  The score of
 * token t for KV head h is the sum, over those T positions and the G query heads
 * of h, of softmax(q . k * softmax_scale) where position pos sees tokens 0..pos.
 * The p->num_reps best tokens of each full block in [first_block, first_block +
 * num_blocks) (ties: lower index) become its reps, in token order.
 * token_scores (nullable): fp32 [batch][num_kv_heads][max_blocks_per_seq*128],
 * the accumulated scores (entries past seq_lens[b] are zero).
 */
kt_status kt_build_dynamic_reps(const kt_paged_kv* kv, const kt_sparse_params* p,
                                const void* q_local, int32_t T, int32_t first_block,
                                int32_t num_blocks, void* reps_pool, float* token_scores,
                                void* ws, size_t ws_bytes, kt_stream_t stream);

/*
 * Score every Context block and select the top-k per unit [LC §3.1 Quest bound,
 * §4.3 similarity to reps, §4.5 top-k and head_select_mode].
 *   q          : fp16 [batch][num_q_heads][128], the decode queries.
 *   reps_pool  : as written by kt_build_block_reps / kt_build_dynamic_reps.
 *   sel        : int32 [batch][SEL][top_k], SEL = 1 (SHARED) or num_kv_heads;
 *                the first cnt entries hold the chosen logical block ids in
 *                ascending order; the rest are left untouched.
 *   cnt        : int32 [batch][SEL] = min(top_k, number of Context blocks).
 *   sel_scores : fp32 [batch][SEL][top_k] or NULL; the unit score of each
 *                chosen block, aligned with sel.
 * Head score: Quest sum_c max(q_c kmax_c, q_c kmin_c); Max/Mean q.rep;
 * Fix/Dynamic max_r q.rep_r.  Unit score: sum of head scores over the unit's
 * query heads (all heads for SHARED, the G heads of the KV head for SEPARATE).
 * Order: score descending, then block id ascending (deterministic).
 */
kt_status kt_score_select_blocks(const void* q, const kt_paged_kv* kv, const void* reps_pool,
                                 const kt_sparse_params* p, int32_t* sel, int32_t* cnt,
                                 float* sel_scores, void* ws, size_t ws_bytes,
                                 kt_stream_t stream);

/*
 * Exact attention over Initial + selected Context + Local blocks [LC §4.2,
 * §4.6 attn(query, kvcache_after_retrieval)]: for query head h,
 * out[b][h] = softmax(q_h K_S^T * softmax_scale) V_S over the valid tokens S of
 * those blocks, fp32 accumulation.  sel/cnt as produced by
 * kt_score_select_blocks (possibly from an earlier step: the token_step /
 * layer_step reuse of [LC §4.6]); cnt is clamped to [0, min(top_k, C)].
 * out: fp32 [batch][num_q_heads][128].
 */
kt_status kt_sparse_decode_attn(const void* q, const kt_paged_kv* kv, const kt_sparse_params* p,
                                const int32_t* sel, const int32_t* cnt, float* out, void* ws,
                                size_t ws_bytes, kt_stream_t stream);

/*
 * One decode step: the selection of kt_score_select_blocks and the attention
 * of kt_sparse_decode_attn, with the same sel / cnt / out.
 * When the shape allows it (linear reps Max/Mean/Quest; at most one
 * (sequence, KV head) segment and one selection unit per SM; the per-CTA
 * selection buffers fit shared memory) the step is ONE cooperative launch:
 * every CTA streams its Initial/Local blocks while its consumer warps score a
 * slice of one unit's Context blocks, and each CTA merges its unit's
 * candidates itself before loading its share of the selected blocks.
 * Otherwise two launches: selection, then the attention as its programmatic
 * dependent.  kt_sparse_decode_step_kernels tells which.  Concurrent steps
 * need separate workspaces.  Workspace: KT_OP_SPARSE_STEP.
 */
kt_status kt_sparse_decode_step(const void* q, const kt_paged_kv* kv, const void* reps_pool,
                                const kt_sparse_params* p, int32_t* sel, int32_t* cnt,
                                float* out, void* ws, size_t ws_bytes, kt_stream_t stream);

/*
 * Kernel launches one kt_sparse_decode_step makes for this shape on the
 * current device: 1 (one cooperative launch) or 2 (selection + attention);
 * a negative kt_status value for invalid arguments.  Host only, no launch.
 */
int32_t kt_sparse_decode_step_kernels(const kt_paged_kv* kv, const kt_sparse_params* p);

/*
 * Caps the CTAs that the attention calls (kt_sparse_decode_attn,
 * kt_sparse_decode_step, kt_decode_layer, kt_dense_decode_attn) launch from
 * the calling host thread: at most max_ctas, and never fewer than one per
 * (sequence, KV head) segment; 0 restores the default of one per SM.  A
 * caller that runs other work beside the decode step can leave SMs to it.
 * The split-K partition of each segment, and in the one-launch step the
 * scoring slices, follow from the CTA count; outputs agree within rounding
 * and selections outside the near-tie zone whatever the cap.  Host only,
 * thread-local, takes effect at the next launch.  INVALID_ARG if max_ctas < 0.
 * No counterpart in the article (a launch-shape setting of this library).
 */
kt_status kt_set_max_ctas(int32_t max_ctas);

/*
 * ---- KV cache in host (Grace) memory, read over NVLink-C2C -------------------
 * The article keeps the KV cache in CPU DRAM and moves only the retrieved
 * blocks to the computation [LC §4.1; §1].  Here the K/V pools of `kv` live in
 * page-locked host memory that the GPU can address (cudaHostAlloc /
 * cudaHostRegister, mapped); the block table, lengths, queries, selection,
 * output and workspace are in device memory, and so are the representatives
 * that the selection scores (kt_score_select_blocks over the same kv reads only
 * the reps pool, never the K/V pools).  This call attends exactly as
 * kt_sparse_decode_attn (same arithmetic, same output) but fetches each
 * attended (block, KV head) — Initial, the given selection, Local — straight
 * from host memory into shared memory with 16-byte copies, so per step only
 * the attended bytes cross the link.  INVALID_ARG if either pool is not host
 * memory mapped for this device.  Workspace: KT_OP_SPARSE_ATTN.
 */
kt_status kt_sparse_decode_attn_hostkv(const void* q, const kt_paged_kv* kv,
                                       const kt_sparse_params* p, const int32_t* sel,
                                       const int32_t* cnt, float* out, void* ws, size_t ws_bytes,
                                       kt_stream_t stream);

/*
 * ---- quantised KV, Q8_0 (the kv_type FP16 / FP32 / Q4_0 / Q8_0 choice of
 * [HOWTO] Step 1) ---------------------------------------------------------------
 * Each 128-channel row of K or V is stored as 4 groups of 32 channels: one
 * binary16 scale and 32 signed 8-bit codes per group (34 bytes instead of 64).
 * With amax the group's largest |x| (binary32), dd = amax / 127 and id = 1/dd
 * (0 when dd is 0), a code is round-half-away-from-zero(x * id) in binary32
 * and the scale is dd rounded to binary16; a value is read back as
 * scale * code.
 */
typedef struct {
  const void* k_code;   /* int8 [num_pages][num_kv_heads][128][128] */
  const void* k_scale;  /* binary16 [num_pages][num_kv_heads][128][4] */
  const void* v_code;   /* int8, as k_code */
  const void* v_scale;  /* binary16, as k_scale */
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t batch, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_pages;
} kt_paged_kv_q8;

/*
 * Quantises pages [first_page, first_page + num_pages) of the fp16 pools of
 * `kv` (every KV head and token row) into the Q8_0 pools.  Codes and scales
 * are exact: they match any binary32 implementation of the definition above.
 * All pointers are device memory, 16-byte aligned.  INVALID_ARG on a page
 * range outside the pool.
 */
kt_status kt_quantize_kv_q8_0(const kt_paged_kv* kv, void* k_code, void* k_scale, void* v_code,
                              void* v_scale, int32_t first_page, int32_t num_pages,
                              kt_stream_t stream);

/*
 * kt_sparse_decode_attn over Q8_0 pools [LC §4.6 attn over the retrieved
 * blocks]: per attended (block, KV head) 34 KB are read instead of 64 KB.
 * Each consumer warp turns its token rows into fp16 (code * scale is exact in
 * binary32 and is rounded once to binary16) and the attention proceeds as for
 * fp16 pools (fp32 accumulation).  The selection is made beforehand from the
 * fp16 representatives (kt_score_select_blocks: they are built from the keys
 * as the blocks fill, before storage).  Workspace: KT_OP_SPARSE_ATTN of the
 * same shapes.
 */
kt_status kt_sparse_decode_attn_q8_0(const void* q, const kt_paged_kv_q8* kv,
                                     const kt_sparse_params* p, const int32_t* sel,
                                     const int32_t* cnt, float* out, void* ws, size_t ws_bytes,
                                     kt_stream_t stream);

/*
 * The decode step (kt_sparse_decode_step) over Q8_0 pools: the selection
 * scores the fp16 representatives `reps_pool` (built from the fp16 K before
 * quantisation, as for kt_score_select_blocks), and the attention reads the
 * chosen blocks' codes and scales as kt_sparse_decode_attn_q8_0 does.  One
 * launch when kt_sparse_decode_step_kernels says so for the same shapes,
 * else selection then attention.  Workspace: KT_OP_SPARSE_STEP.  Same errors
 * as kt_sparse_decode_step and kt_sparse_decode_attn_q8_0.
 */
kt_status kt_sparse_decode_step_q8_0(const void* q, const kt_paged_kv_q8* kv,
                                     const void* reps_pool, const kt_sparse_params* p,
                                     int32_t* sel, int32_t* cnt, float* out, void* ws,
                                     size_t ws_bytes, kt_stream_t stream);

/*
 * Phase timing of the attention launches made from the calling host thread
 * (kt_sparse_decode_attn, kt_sparse_decode_step, kt_dense_decode_attn,
 * kt_decode_layer): with a non-NULL buffer, each CTA of a launch with at most
 * max_ctas CTAs writes the device global timer (ns) at the phases below into
 * stamps[cta * 16 + phase] (uint64, device memory owned by the caller, at
 * least max_ctas * 16 entries); a phase a CTA does not reach is left as it
 * was, so clear the buffer between launches.  NULL turns it off (default).
 * Thread-local; takes effect at the next launch.  INVALID_ARG if the buffer
 * is non-NULL and misaligned or max_ctas < 1.  No counterpart in the article
 * (a measurement aid of this library).
 *   0 CTA entry                          7 first K/V block load issued
 *   1 slice block-table entries loaded   8 first selected block load issued
 *   2 slice representatives landed       9 last block attended
 *   3 slice scored                      10 partial published / output written
 *   4 slice candidates published        11 segment's partials all seen (merger)
 *   5 unit's slices all seen            12 output written (merger)
 *   6 unit's top-k picked, this CTA's pages handed to the loads
 * Phases 1-6 and 11 exist only in the one-launch step.
 */
kt_status kt_set_phase_stamps(void* stamps, int32_t max_ctas);

/*
 * Preselection [LC §4.4 "预选择 Preselect", §4.6 preselect_block()]: before
 * decoding, pick per selection unit a fixed set of Context blocks from the
 * attention of the last T prompt positions; later selections choose only
 * among them (the preselect_block / preselect_block_count keys of [HOWTO]
 * Step 1).  The vote of a Context token is its accumulated softmax probability
 * over the unit's local query rows (T positions x the query heads of each of
 * the unit's KV heads, causal), votes are average-pooled along the Context
 * tokens (window kernel_size, odd, <= 65, zero padding kernel_size/2, stride
 * 1), and the `count` blocks whose tokens rank first by pooled vote are
 * preselected, i.e. the top `count` blocks by their largest pooled vote
 * (ties: lower block).
 *   q_local     : fp16 [batch][T][num_q_heads][128] (as kt_build_dynamic_reps)
 *   presel_mask : uint32 [batch][SEL][kt_preselect_mask_words(kv)], bit j%32 of
 *                 word j/32 set when logical block j is preselected
 *   presel_cnt  : int32 [batch][SEL], min(count, C)
 * Workspace: KT_OP_PRESELECT with the same T.  T*G <= 256.
 */
int32_t kt_preselect_mask_words(const kt_paged_kv* kv);
kt_status kt_preselect_blocks(const kt_paged_kv* kv, const kt_sparse_params* p,
                              const void* q_local, int32_t T, int32_t kernel_size, int32_t count,
                              uint32_t* presel_mask, int32_t* presel_cnt, void* ws,
                              size_t ws_bytes, kt_stream_t stream);

/*
 * kt_score_select_blocks and kt_sparse_decode_step with each unit's choice
 * restricted to its preselected blocks (presel_mask / presel_cnt as written by
 * kt_preselect_blocks): the top min(top_k, presel_cnt) preselected blocks by
 * unit score.  Same workspaces as the unrestricted calls.
 */
kt_status kt_score_select_blocks_presel(const void* q, const kt_paged_kv* kv,
                                        const void* reps_pool, const kt_sparse_params* p,
                                        const uint32_t* presel_mask, int32_t* sel, int32_t* cnt,
                                        float* sel_scores, void* ws, size_t ws_bytes,
                                        kt_stream_t stream);
kt_status kt_sparse_decode_step_presel(const void* q, const kt_paged_kv* kv,
                                       const void* reps_pool, const kt_sparse_params* p,
                                       const uint32_t* presel_mask, const int32_t* presel_cnt,
                                       int32_t* sel, int32_t* cnt, float* out, void* ws,
                                       size_t ws_bytes, kt_stream_t stream);

/*
 * The same step for callers whose query and output live in HOST memory:
 * copies q_host (fp16 [batch][num_q_heads][128]) to q_dev, runs
 * kt_sparse_decode_step, copies out_dev to out_host (fp32) and synchronises
 * `stream`.  Host buffers should be pinned for asynchronous copies.
 * With q_dev and out_dev both NULL, q_host and out_host must be page-locked
 * host memory mapped for the device (16-byte aligned): the one-launch step
 * then reads the query and writes the output over the host link itself, with
 * no copies (INVALID_ARG for other host memory; UNSUPPORTED when the shapes
 * need the two-kernel path).  Either way the call returns once out_host
 * holds the output.
 */
kt_status kt_sparse_decode_step_host(const void* q_host, void* q_dev, const kt_paged_kv* kv,
                                     const void* reps_pool, const kt_sparse_params* p,
                                     int32_t* sel, int32_t* cnt, float* out_dev,
                                     float* out_host, void* ws, size_t ws_bytes,
                                     kt_stream_t stream);

/*
 * Dense decode attention over all n tokens of each sequence: the full scan
 * that [LC §1] says the sparse method avoids; kept as the sparsity reference.
 */
kt_status kt_dense_decode_attn(const void* q, const kt_paged_kv* kv, int32_t num_q_heads,
                               float softmax_scale, float* out, void* ws, size_t ws_bytes,
                               kt_stream_t stream);

/*
 * Decoding over many layers and tokens with selection reuse [LC §4.5
 * token_step / layer_step / dense_layer_num; §4.6, the decode loop of the
 * framework pseudocode].  The first dense_layer_num layers attend every
 * block.  For the other layers, with l = layer_idx - dense_layer_num (the
 * index among sparse layers), the layers l = s*layer_step .. s*layer_step +
 * layer_step - 1 share history slot s; decode step token_idx (counted from 0
 * after prefill) selects afresh at layer l, and stores that selection in slot
 * s, when token_idx % token_step == 0 and l % layer_step == 0; every other
 * sparse (token, layer) attends with the selection stored in slot s, whose
 * blocks are still Context blocks because Context only grows while decoding.
 * Counting l among the sparse layers makes the first sparse layer of every
 * slot select before the others read it.
 */
typedef struct {
  int32_t num_layers;       /* >= 1 */
  int32_t dense_layer_num;  /* 0 .. num_layers */
  int32_t layer_step;       /* >= 1 */
  int32_t token_step;       /* >= 1 */
} kt_reuse_policy;

typedef enum {
  KT_LAYER_DENSE = 0,   /* kt_dense_decode_attn */
  KT_LAYER_SELECT = 1,  /* kt_sparse_decode_step into the history slot */
  KT_LAYER_REUSE = 2    /* kt_sparse_decode_attn with the history slot */
} kt_layer_action;

/* History slots the policy needs: ceil((num_layers - dense_layer_num) /
 * layer_step); negative (a kt_status value negated) for an invalid policy. */
int32_t kt_decode_history_slots(const kt_reuse_policy* pol);

/* The action of decode step token_idx at layer layer_idx and its history
 * slot (-1 for dense layers).  Host only; no device work. */
kt_status kt_decode_layer_action(const kt_reuse_policy* pol, int32_t token_idx,
                                 int32_t layer_idx, int32_t* action, int32_t* slot);

/*
 * One layer of one decode step under the policy: the action of
 * kt_decode_layer_action on this layer's q / kv / reps.
 *   hist_sel : int32 [slots][batch][SEL][top_k], hist_cnt : int32
 *              [slots][batch][SEL], caller-owned device memory that persists
 *              across calls (slots = kt_decode_history_slots); a SELECT call
 *              writes slot s, a REUSE call reads it.
 *   ws       : a workspace of kt_workspace_bytes(KT_OP_SPARSE_STEP) bytes,
 *              which serves all three actions.
 * Errors as the call the action maps to; KT_ERR_INVALID_ARG for an invalid
 * policy or index.
 */
kt_status kt_decode_layer(const kt_reuse_policy* pol, int32_t token_idx, int32_t layer_idx,
                          const void* q, const kt_paged_kv* kv, const void* reps_pool,
                          const kt_sparse_params* p, int32_t* hist_sel, int32_t* hist_cnt,
                          float* out, void* ws, size_t ws_bytes, kt_stream_t stream);

/*
 * Appends one decoded token to every sequence: writes k_new / v_new (fp16
 * [batch][num_kv_heads][128], 16-byte aligned) as token n_b = seq_lens[b] of
 * sequence b, into row n_b % 128 of page block_table[b][n_b / 128], and
 * increments seq_lens[b] on the device.  The pools and seq_lens that kv points
 * to are written through its const pointers.  With Max, Mean, Quest or Fix
 * reps and a non-NULL reps_pool, the reps of a block that this token completes
 * are built in the same call (Dynamic reps are built by kt_build_dynamic_reps
 * when the caller chooses; reps_pool NULL skips the reps).  The caller
 * allocates the page of a new block before the call.  A sequence whose table
 * has no room, or whose page is outside the pool, records KT_ERR_DEVICE_CHECK
 * and is left unchanged.  ws: any workspace of at least 256 bytes (its status
 * word is used).  Asynchronous on `stream`.
 */
kt_status kt_append_kv(const kt_paged_kv* kv, const kt_sparse_params* p, const void* k_new,
                       const void* v_new, void* reps_pool, void* ws, size_t ws_bytes,
                       kt_stream_t stream);

/*
 * kt_sparse_decode_attn without a workspace, for callers that cannot allocate
 * device memory: for example a kernel plugged into an engine or framework
 * that hands it only its input and output buffers and owns every other byte
 * of device memory, or a latency-critical path where a cudaMalloc (which can
 * synchronise the device) is not allowed.  The article has no counterpart:
 * this is an interface variant, not part of the method.
 *
 * Same arguments, results and errors as kt_sparse_decode_attn, minus the
 * workspace.  Its scratch memory (status word, tickets, split-K partials) is a
 * fixed 1 MiB array inside this library's device image, which every GPU that
 * loads the library keeps until the process exits.  It holds one partial of
 * about G x 520 bytes per attention CTA (max(#SMs, batch*num_kv_heads) CTAs),
 * so shapes up to roughly batch*num_kv_heads = 500 at G = 4 (250 at G = 8)
 * fit; larger ones return KT_ERR_WORKSPACE_TOO_SMALL before any launch.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; each call clears the status word and tickets on
 *     `stream` before its kernel.  Calls that overlap on the GPU (different
 *     streams, or host threads without ordering) race on it.
 *   - Device-side check failures and timeouts are recorded in the shared
 *     array's status word, not returned by this call (it returns after the
 *     launch); kt_noalloc_read_status reports and clears the word.
 *   - It calls no allocator (no cudaMalloc, cudaFree or allocating library
 *     routine).
 */
kt_status kt_sparse_decode_attn_noalloc(const void* q, const kt_paged_kv* kv,
                                        const kt_sparse_params* p, const int32_t* sel,
                                        const int32_t* cnt, float* out, kt_stream_t stream);

/*
 * The device status of the last kt_sparse_decode_attn_noalloc call on the
 * current device (KT_OK, KT_ERR_DEVICE_CHECK or KT_ERR_TIMEOUT), read from the
 * library's scratch array after synchronising `stream`, then cleared.  Like
 * the call itself it allocates nothing; the article has no counterpart.
 * INVALID_ARG if device_status is NULL.
 */
kt_status kt_noalloc_read_status(kt_stream_t stream, int32_t* device_status);

/*
 * Synchronises `stream`, stores the workspace status word (a kt_status value,
 * KT_OK if no device-side anomaly was recorded since the last read) in
 * *device_status and clears it.
 */
kt_status kt_read_device_status(void* ws, size_t ws_bytes, kt_stream_t stream,
                                int32_t* device_status);

/*
 * Diagnostic: launches one CTA that waits on an mbarrier nobody completes,
 * giving up after `spin_limit` polls; the kernel then records KT_ERR_TIMEOUT in
 * the status word and returns.  Used to test the bounded-wait path.
 */
kt_status kt_selftest_bounded_wait(void* ws, size_t ws_bytes, int32_t spin_limit,
                                   kt_stream_t stream);

/*
 * Diagnostic of the one-launch step's failure path: runs kt_sparse_decode_step
 * (one-launch shapes only; UNSUPPORTED otherwise) with CTA `skip_cta`
 * publishing no candidate slots, so the polls of its selection unit never see
 * them, and with the slot and partial polls bounded by poll_limit_us.  The
 * launch records KT_ERR_TIMEOUT in the workspace status word and finishes
 * (the chosen ids and pages are range-checked, so nothing reads out of
 * bounds; sel/cnt/out of this launch are meaningless), and the workspace
 * serves the next step unchanged.  Used to test that path without a fault.
 */
kt_status kt_selftest_step_timeout(const void* q, const kt_paged_kv* kv, const void* reps_pool,
                                   const kt_sparse_params* p, int32_t* sel, int32_t* cnt,
                                   float* out, void* ws, size_t ws_bytes, int32_t skip_cta,
                                   int32_t poll_limit_us, kt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KT_H_ */
