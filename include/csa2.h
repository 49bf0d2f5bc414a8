/*
 * csa2.h -- C ABI of the CSA2 global-attention hot path (DeepSeek-V4.1-Flash) on one GB300.
 *
 * Sources (cited as page title + section):
 *   [P1] "DeepSeek-V4.1 模型结构（2）：序列维度（中），CSA2 的三种模式" (blog.javazero.top)
 *   [P2] "DeepSeek v4.1 Flash技术剖析——架构篇" (myhz0606.com)
 *   [P3] "DeepSeek-V4.1-Flash：把百万 Token 的记忆，压缩成一套分级缓存" (junki.cn)
 *   [P4] "CSA2 — l'attention creuse compressée de seconde génération" (mkdocs.reaper.mx)
 *
 * Conventions for every call:
 *   - Tensor arguments are DEVICE pointers owned by the caller; the library never
 *     allocates device memory.  Scratch comes in through (workspace, ws_bytes),
 *     sized by the matching *_workspace_size() query; workspace must be 256-byte
 *     aligned.  bf16 tensors are passed as void* (IEEE bfloat16 bits).
 *   - All tensors are dense row-major in the stated shape; every device pointer must
 *     be 16-byte aligned.  Fixed widths: entry 512 (last 64 dims RoPE), 32 indexer
 *     heads x 128, indexer-K row = 64 code bytes + 4 scale bytes.
 *   - Positions are absolute token positions, 0-based.  Query i of every sequence
 *     sits at q_pos0 + i.  Entry s of a cache covers tokens s*m .. s*m+m-1.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Arguments are validated on the host before any launch: a bad call
 *     returns CSA2_ERR_INVALID_ARG / CSA2_ERR_UNSUPPORTED / CSA2_ERR_WORKSPACE and
 *     launches nothing.  A failed launch returns CSA2_ERR_CUDA.  Conditions only
 *     the device can see (an out-of-range top-k index, an expired bounded wait)
 *     set a device error word and are reported by csa2_last_device_status().
 *   - csa2_last_error_message() gives a one-line reason for the last non-OK status
 *     returned on the calling host thread.
 *   - No call synchronises the device except csa2_last_device_status().
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad shape or table   */
  CSA2_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels cover    */
  CSA2_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small      */
  CSA2_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed            */
  CSA2_ERR_TIMEOUT = 5,       /* a bounded device-side wait expired              */
  CSA2_ERR_DEVICE_CHECK = 6   /* a device-side bounds check fired                */
};

#define CSA2_ENTRY_DIM 512
#define CSA2_ROPE_DIM 64
#define CSA2_IDX_HEADS 32
#define CSA2_IDX_DIM 128
#define CSA2_IDX_CODE_BYTES 64
#define CSA2_IDX_SCALE_BYTES 4
#define CSA2_MAX_TOPK 2048

/* Human-readable name of a status code (static storage). */
const char* csa2_status_str(int status);
/* Reason for the last non-OK status on this host thread ("" if none). */
const char* csa2_last_error_message(void);
/* Library version string. */
const char* csa2_version(void);
/* Number of GPU kernels this library has launched in this process so far (all entry
 * points, all devices; a monotone counter for instrumentation -- the difference across
 * a region is the launch count of that region).  No counterpart in the method. */
unsigned long long csa2_kernel_launches(void);

/* Synchronises `stream`, then reads and clears the device error word of the current
 * device.  Returns CSA2_OK, CSA2_ERR_DEVICE_CHECK, CSA2_ERR_TIMEOUT or CSA2_ERR_CUDA. */
int csa2_last_device_status(void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 1 -- compressor.  [P1 §压缩算子去掉了重叠和位置偏置], [P2 §Compressor]:
 * kv = x.W_kv^T and score = x.W_gate^T (float32 accumulation); entry g pools only
 * its own group of m tokens with a softmax over the group taken per channel;
 * RMSNorm(eps) times norm_w; RoPE on dims 448..511 (interleaved pairs, theta_i =
 * rope_base^(-i/32)) at the position of the group's first token.  m = 1 is the
 * gate-less special case RMSNorm(x.W_kv^T): w_gate must be NULL exactly when m == 1.
 *
 *   x       bf16 [B, T, hidden]   tokens at positions pos0 .. pos0+T-1 (pos0 % m == 0)
 *   w_kv    bf16 [512, hidden];  w_gate bf16 [512, hidden] or NULL;  norm_w f32 [512]
 *   kv_cache bf16 [B, n_cap, 512]: writes entries pos0/m .. pos0/m + T/m - 1 of every
 *           sequence (post-RoPE).  Tokens of an incomplete trailing group are ignored.
 *   kv_pre  f32 [B, T/m, 512] or NULL: the normalised entries before RoPE (input of
 *           csa2_index_k_quant).
 *   hidden must be a multiple of 64; B*T >= 1; pos0/m + T/m <= n_cap.
 * ------------------------------------------------------------------------------- */
size_t csa2_compress_workspace_size(int B, int T, int hidden, int m);
int csa2_compress(const void* x, int B, int T, int hidden, int m, int pos0,
                  const void* w_kv, const void* w_gate, const float* norm_w, float eps,
                  float rope_base, void* kv_cache, int n_cap, float* kv_pre,
                  void* workspace, size_t ws_bytes, void* stream);

/* csa2_compress with the group state carried across calls: decode one token at a time, or
 * prefill in chunks of any length.  The pages pool each group of m tokens on its own, so a
 * token that is not its group's last can only be held back until the group completes.
 * Tokens pos0 .. pos0+T-1 of every sequence (any pos0 >= 0, any T >= 1) produce exactly the
 * entries csa2_compress writes for whole groups: entries pos0/m .. (pos0+T)/m - 1 (integer
 * division), i.e. every group whose last token is in this chunk.
 *   m == 2: state f32 [B, 1024], caller-owned, 16-byte aligned.  When pos0 is odd, the group
 *           (pos0-1)/2 is completed from state (its first token, left by the call that ended
 *           at pos0-1) and this chunk's first token.  When pos0+T is odd, the chunk's last
 *           token's kv and score rows (float32, 2 x 512 per sequence) are written to state.
 *           Calls that share a state must follow one another in position order on one stream.
 *   m == 1: every token completes its entry; state must be NULL.
 *   x       bf16 [B, T, hidden];  kv_pre f32 [B, n, 512] or NULL, n = (pos0+T)/m - pos0/m.
 * Workspace: csa2_compress_workspace_size(B, T, hidden, m).  (pos0+T)/m <= n_cap.
 * Errors as csa2_compress; a state left by another position is not detected. */
int csa2_compress_chunk(const void* x, int B, int T, int hidden, int m, int pos0,
                        const void* w_kv, const void* w_gate, const float* norm_w, float eps,
                        float rope_base, float* state, void* kv_cache, int n_cap,
                        float* kv_pre, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 2 -- indexer key.  [P1 §indexer K 改由 main KV 投影]: k = W_IK . kv_pre
 * (512 -> 128) from the entry BEFORE its RoPE, then RoPE on k's dims 64..127 at the
 * entry's position, no Hadamard rotation, then FP4 E2M1 with one E4M3 scale per 32
 * dims ([P3 §六]: 68 bytes per entry).
 * Quantisation of each 32-block v (float32): s = E4M3_RNE_satfinite(amax / 6);
 * s == 0 -> all codes 0; else code = sign(u)<<3 | E2M1_RNE_satfinite(|u|), u = v / s
 * (IEEE float32 divides).  Element 2i in the low nibble of byte i.
 *
 *   kv_pre  f32 [B, G, 512]: entries entry0 .. entry0+G-1 of each sequence
 *   w_ik    bf16 [128, 512]
 *   codes   u8 [B, n_cap, 64], scales u8 [B, n_cap, 4]: rows entry0.. written
 *   k_out   f32 [B, G, 128] or NULL: the key before quantisation (debug)
 *   RoPE position of entry e is e * m.
 * ------------------------------------------------------------------------------- */
int csa2_index_k_quant(const float* kv_pre, int B, int G, int entry0, int m,
                       const void* w_ik, float rope_base, uint8_t* codes, uint8_t* scales,
                       int n_cap, float* k_out, void* stream);

/* ---------------------------------------------------------------------------------
 * FP4 main KV.  [P3 §六] (a main-KV entry takes 288 bytes) and [P3 §七 FP4 Main KV]
 * (E2M1 data, channel groups sharing an E4M3 scale, dequantised before the attention).
 * READING: groups of 16 channels, 256 B of codes + 32 scales per 512-channel entry, the
 * index keys' rounding rules applied to each stored (bf16) entry.
 *
 *   kv_cache bf16 [B, n_cap, 512]: rows entry0 .. entry0+G-1 of each sequence are read
 *   codes    u8 [B, n_cap, 256] (channel 2i in the low nibble of byte i), scales u8
 *            [B, n_cap, 32] (E4M3 bits): the same rows written, other rows untouched
 * Returns CSA2_ERR_INVALID_ARG for null or unaligned pointers and bad shapes.
 * ------------------------------------------------------------------------------- */
int csa2_main_kv_quant_fp4(const void* kv_cache, int B, int n_cap, int entry0, int G,
                           uint8_t* codes, uint8_t* scales, void* stream);

/* FP8 window KV.  [P3 §七 FP4 Main KV]: the window (SWA) KV is more sensitive to
 * quantisation and stays FP8.  READING (the pages give no format): OCP E4M3 elements with
 * one power-of-two scale per 64 channels (8 per row; the last group is the 64 RoPE dims).
 * For a group with largest magnitude amax: k = the smallest integer >= -126 with
 * amax <= 448 * 2^k, stored as the byte k + 127; code = signbit(v) << 7 | E4M3
 * nearest-even of |v| * 2^-k (an exact product, never saturating).  520 bytes per row.
 *
 *   swa_kv bf16 [B, S, 512]: rows row0 .. row0+n_rows-1 of each sequence are read
 *   codes  u8 [B, S, 512], scales u8 [B, S, 8]: the same rows written, others untouched
 * Returns CSA2_ERR_INVALID_ARG for null or unaligned pointers and bad shapes. */
int csa2_swa_kv_quant_fp8(const void* swa_kv, int B, int S, int row0, int n_rows,
                          uint8_t* codes, uint8_t* scales, void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 3 -- lightning-indexer scores and causal top-k.  [P1 §indexer K 改由 main KV
 * 投影] (scoring unchanged from V4: I[t,s] = sum_j w[t,j] * ReLU(q_hat[t,j] . k_hat[s]),
 * 32 heads x 128, top-512), [P2 §Indexer], [P2 §CSA2-ReIndex].
 *   q_hat: each head's 128 values quantised with the stage-2 FP4 rule (per 32 dims);
 *   k_hat: dequantised codes x scales.  Entry s is visible to the query at position
 *   t iff s*m + m - 1 <= t.  Top-k orders visible entries by (score desc, index asc)
 *   and returns the first min(k, visible) indices in ascending order, padded with -1.
 *
 *   q_idx   bf16 [B, Tq, 32, 128];  w  f32 [B, Tq, 32]
 *   codes/scales: cache of n_cap rows per sequence, rows 0..n_entries-1 valid
 *   cand    NULL (Full layer: all visible entries compete) or i32 [B, Tq, nb]
 *           candidate block ids (Reindex: only visible entries of these blocks of
 *           `blk` entries compete; -1 entries ignored).  Ids must be distinct and
 *           ascending, as csa2_hsi_candidates writes them; a block id >= ceil(n_entries
 *           / blk) is skipped and sets CSA2_ERR_DEVICE_CHECK.
 *   topk_out i32 [B, Tq, k], 1 <= k <= 2048
 *   blockmax_out NULL or f32 [B, Tq, ceil(n_entries/blk)]: per block of `blk`
 *           entries, the max score over its visible entries (-inf if none); Full only
 *   scores_out NULL or f32 debug: Full [B, Tq, n_entries] (entries beyond the visible
 *           range unspecified); Reindex [B, Tq, nb*blk] in candidate order (-inf for
 *           slots outside the visible pool)
 *   blk: power of two in [1, 256] when cand or blockmax_out is given.
 * ------------------------------------------------------------------------------- */
size_t csa2_indexer_workspace_size(int B, int Tq, int n_entries, int nb, int blk,
                                   int with_cand);
int csa2_indexer_score_topk(const void* q_idx, const float* w, int B, int Tq, int q_pos0,
                            const uint8_t* codes, const uint8_t* scales, int n_cap,
                            int n_entries, int m, const int32_t* cand, int nb, int blk,
                            int k, int32_t* topk_out, float* blockmax_out,
                            float* scores_out, void* workspace, size_t ws_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 3 with an explicit bound on the device waits -- a diagnostic of the library's
 * error path; the pages have no counterpart.  The same computation as
 * csa2_indexer_score_topk for a Full layer (cand, blockmax_out and scores_out NULL),
 * restricted to the calls that run the tensor-core decode scorer: 1 <= Tq < 64, and
 * entry 0 visible to the first query (n_entries >= 1, q_pos0 + 1 >= m); others return
 * CSA2_ERR_UNSUPPORTED before any launch.  Every mbarrier wait of that kernel polls at most wait_limit times
 * (0: the library's default, 2^24) before it gives up and sets CSA2_ERR_TIMEOUT in the
 * device error word (csa2_last_device_status reads and clears it).  stall != 0 (needs
 * wait_limit > 0) makes the kernel's copy thread first wait on a barrier that nothing
 * completes: no copy is issued, every other role's first wait runs out, and each CTA
 * leaves with no copy or MMA in flight; the top-k launch that follows then selects
 * from whatever the workspace's score area held.  The context stays usable.
 * ------------------------------------------------------------------------------- */
int csa2_indexer_score_topk_bounded(const void* q_idx, const float* w, int B, int Tq,
                                    int q_pos0, const uint8_t* codes, const uint8_t* scales,
                                    int n_cap, int n_entries, int m, int k, int32_t* topk_out,
                                    void* workspace, size_t ws_bytes, unsigned wait_limit,
                                    int stall, void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 3 without allocation.  The pages have no counterpart: this is a library
 * convenience.  Same computation, arguments and results as csa2_indexer_score_topk
 * (no scores_out, no workspace), for callers that cannot allocate device memory --
 * e.g. code running inside an allocator hook or under a framework that has reserved
 * all device memory, or a plain C host with no GPU allocator of its own.  The scratch
 * that csa2_indexer_score_topk takes as its workspace lives here in a fixed 16 MiB
 * array inside the library; every GPU that loads the library holds that array until
 * the process exits.  A call is accepted exactly when
 *   csa2_indexer_workspace_size(B, Tq, n_entries, nb, blk, cand != NULL)
 *       <= csa2_indexer_noalloc_max_scratch_bytes()
 * (scores of every row plus, for rows longer than 32768 entries, the chunked
 * selection's candidate lists, and 2176 bytes of FP4 query image per query row);
 * larger calls return CSA2_ERR_UNSUPPORTED before any launch.  The array's device
 * address is looked up (cudaGetSymbolAddress) on the first call in each CUDA context
 * of a device -- again after cudaDeviceReset or under another context; make that
 * first call before any stream capture.  All calls share the one array: calls that
 * overlap on the GPU (other streams, other host threads) race and must be serialised
 * by the caller.  Nothing in the array needs to start at zero: each call writes
 * every score it reads.
 * ------------------------------------------------------------------------------- */
size_t csa2_indexer_noalloc_max_scratch_bytes(void);
int csa2_indexer_score_topk_noalloc(const void* q_idx, const float* w, int B, int Tq,
                                    int q_pos0, const uint8_t* codes, const uint8_t* scales,
                                    int n_cap, int n_entries, int m, const int32_t* cand, int nb,
                                    int blk, int k, int32_t* topk_out, float* blockmax_out,
                                    void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 3b -- hierarchical candidate pool.  [P2 §CSA2-ReIndex], [P3 §五 HSI]: the
 * blocks of `blk` entries are ranked by their block max; the block that holds the
 * newest visible entry is always taken (score +inf); the top-nb blocks by (score
 * desc, block asc) are returned ascending, padded with -1.
 *   blockmax f32 [B, Tq, ceil(n_entries/blk)] (as written by csa2_indexer_score_topk)
 *   cand_out i32 [B, Tq, nb], 1 <= nb <= 2048
 * ------------------------------------------------------------------------------- */
int csa2_hsi_candidates(const float* blockmax, int B, int Tq, int q_pos0, int n_entries,
                        int m, int blk, int nb, int32_t* cand_out, void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 4 -- shared-K=V sparse attention.  [P1 §一层全局注意力算四样东西] item 4,
 * [P2 §CSA2-FULL], [P3 §四]: for every head h, over the multiset A of the selected
 * cache entries (valid top-k indices) and the window rows of positions
 * max(0, t-window+1) .. t: l_j = scale * q_h . c_j, p = softmax(l), o_h = sum_j p_j c_j
 * (the same row c_j is key and value).  Optional per-head sink adds exp(sink_h) to
 * the denominator.
 *
 *   q       bf16 [B, Tq, H, 512] (already rotated);  H in 1..128
 *   kv_cache bf16 [B, n_cap, 512], n_entries valid rows (NULL allowed iff k == 0)
 *   topk    i32 [B, Tq, k] or NULL (k == 0: window only); -1 = no entry; an index
 *           >= n_entries is skipped and sets CSA2_ERR_DEVICE_CHECK
 *   swa_kv  bf16 [B, S, 512]: row r holds position swa_pos0 + r; every query's window
 *           must lie inside [swa_pos0, swa_pos0 + S)
 *   sink    f32 [H] or NULL;  out bf16 [B, Tq, H, 512];  lse_out f32 [B, Tq, H] or NULL
 *           (natural-log sum of exp of the scaled logits, sink included)
 * ------------------------------------------------------------------------------- */
size_t csa2_sparse_attn_workspace_size(int B, int Tq, int H, int k, int window);
int csa2_sparse_attn(const void* q, int B, int Tq, int H, int q_pos0, const void* kv_cache,
                     int n_cap, int n_entries, const int32_t* topk, int k, const void* swa_kv,
                     int S, int swa_pos0, int window, const float* sink, float scale,
                     void* out, float* lse_out, void* workspace, size_t ws_bytes,
                     void* stream);

/* The same attention over FP4 main-KV entries (csa2_main_kv_quant_fp4's planes):
 *   kv_codes u8 [B, n_cap, 256], kv_scales u8 [B, n_cap, 32] in place of kv_cache; each
 *   selected entry is dequantised (code value x group scale, exact in bf16's range) into
 *   the same bf16 tile the attention reads; window rows stay bf16.  H must be 64
 *   (CSA2_ERR_UNSUPPORTED otherwise).  Other arguments and errors as csa2_sparse_attn. */
int csa2_sparse_attn_fp4kv(const void* q, int B, int Tq, int H, int q_pos0,
                           const uint8_t* kv_codes, const uint8_t* kv_scales, int n_cap,
                           int n_entries, const int32_t* topk, int k, const void* swa_kv, int S,
                           int swa_pos0, int window, const float* sink, float scale, void* out,
                           float* lse_out, void* workspace, size_t ws_bytes, void* stream);

/* The same attention with each operand in any stored format: the entries as bf16
 * (kv_cache, kv_codes = kv_scales = NULL) or FP4 (kv_codes u8 [B, n_cap, 256] + kv_scales
 * u8 [B, n_cap, 32], kv_cache = NULL); the window rows as bf16 (swa_kv, swa_codes =
 * swa_scales = NULL) or FP8 (swa_codes u8 [B, S, 512] + swa_scales u8 [B, S, 8] from
 * csa2_swa_kv_quant_fp8, swa_kv = NULL).  Quantised rows are dequantised exactly into the
 * bf16 tile the attention reads.  Any quantised operand needs H a multiple of 8 up to 64
 * (CSA2_ERR_UNSUPPORTED otherwise); giving both forms, or neither, of an operand is
 * CSA2_ERR_INVALID_ARG.  Other arguments and errors as csa2_sparse_attn. */
int csa2_sparse_attn_ex(const void* q, int B, int Tq, int H, int q_pos0, const void* kv_cache,
                        const uint8_t* kv_codes, const uint8_t* kv_scales, int n_cap,
                        int n_entries, const int32_t* topk, int k, const void* swa_kv,
                        const uint8_t* swa_codes, const uint8_t* swa_scales, int S,
                        int swa_pos0, int window, const float* sink, float scale, void* out,
                        float* lse_out, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * Stage 5 -- Full / Reindex / Reuse layer runtime.  [P1 §一层全局注意力算四样东西],
 * [P1 §共享池里有四样东西], [P1 §40 层只有 4 个 Full], [P4 §Les trois modes].
 * The layer pattern is static: kv_source_layer_ids[l] (-1 = sliding window only,
 * l = own main KV, j < l = main KV of Full layer j) and index_source_layer_ids[l]
 * (l = own top-k, r < l = top-k of index source r of the same KV).  Own KV with a
 * foreign index is rejected.  ratio[l] = m of Full layer l (1 or 2), ignored
 * elsewhere.  A Full layer whose KV some Reindex layer reads builds the HSI pool
 * (hsi_blk, hsi_nb); such Reindex layers select inside it.  The runner keeps the
 * four shared slots (compress_kv, index_k, topk_idxs, candidates) as pointers only.
 * ------------------------------------------------------------------------------- */
typedef struct csa2_runner csa2_runner;

enum { CSA2_MODE_SWA = 0, CSA2_MODE_FULL = 1, CSA2_MODE_REINDEX = 2, CSA2_MODE_REUSE = 3 };

/* Per-layer device pointers for one step.  Fields a layer's mode does not use are
 * ignored (may be NULL / 0). */
typedef struct {
  /* Full: new hidden states bf16 [B, x_tokens, hidden] at positions x_pos0..;
   * after the step the cache holds (x_pos0 + x_tokens) / m entries. */
  const void* x;
  const void* w_kv;            /* bf16 [512, hidden] */
  const void* w_gate;          /* bf16 [512, hidden], NULL iff m == 1 */
  const float* norm_w;         /* f32 [512] */
  const void* w_ik;            /* bf16 [128, 512] */
  void* kv_cache;              /* bf16 [B, n_cap, 512] */
  uint8_t* idx_codes;          /* u8 [B, n_cap, 64] */
  uint8_t* idx_scales;         /* u8 [B, n_cap, 4] */
  /* Full / Reindex */
  const void* q_idx;           /* bf16 [B, Tq, 32, 128] */
  const float* w_idx;          /* f32 [B, Tq, 32] */
  /* every layer */
  const void* q;               /* bf16 [B, Tq, H, 512] */
  const void* swa_kv;          /* bf16 [B, swa_len, 512] */
  const float* sink;           /* f32 [H] or NULL */
  void* out;                   /* bf16 [B, Tq, H, 512] */
  int32_t* topk_out;           /* optional i32 [B, Tq, k]: index sources write here */
  int32_t* cand_out;           /* optional i32 [B, Tq, hsi_nb]: pool-building Full layer */
  /* Optional stored formats ([P3 §六], [P3 §七 FP4 Main KV]).  Full: with kv_codes /
   * kv_scales (u8 [B, n_cap, 256] / [B, n_cap, 32], FP4 as csa2_main_kv_quant_fp4) the step
   * also writes the layer's new entries there, and every layer reading this KV attends over
   * the FP4 entries (kv_cache still receives the bf16 entries).  Every layer: swa_codes /
   * swa_scales (u8 [B, swa_len, 512] / [B, swa_len, 8], FP8 as csa2_swa_kv_quant_fp8) in
   * place of swa_kv (which is then NULL).  Quantised operands need H a multiple of 8 up
   * to 64. */
  uint8_t* kv_codes;
  uint8_t* kv_scales;
  const uint8_t* swa_codes;
  const uint8_t* swa_scales;
  /* Full, m == 2, optional: f32 [B, 1024] group state carried between steps (as in
   * csa2_compress_chunk), so that a step may hand over any number of new tokens, down to one
   * per sequence; without it x_pos0 must be a multiple of m and a trailing incomplete group is
   * ignored. */
  float* compress_state;
  int x_tokens;
  int x_pos0;
  int n_cap;
  int swa_len;
  int swa_pos0;
  int reserved0;
} csa2_layer_io;

typedef struct {
  int B;          /* sequences */
  int Tq;         /* queries per sequence (1 in decode) */
  int q_pos0;     /* position of query 0 */
  int H;          /* attention heads */
  int hidden;     /* hidden size of x */
  int k;          /* top-k */
  int window;     /* sliding window */
  int reserved0;
  float scale;    /* attention logit scale, e.g. 1/sqrt(512) */
  float eps;      /* RMSNorm epsilon */
  float rope_base;
  float reserved1;
} csa2_step_params;

int csa2_runner_create(int n_layers, const int32_t* kv_source_layer_ids,
                       const int32_t* index_source_layer_ids, const int32_t* ratio,
                       int hsi_blk, int hsi_nb, csa2_runner** out);
void csa2_runner_destroy(csa2_runner* r);
/* Mode of a layer (CSA2_MODE_*), or -1 for a bad layer id. */
int csa2_runner_layer_mode(const csa2_runner* r, int layer);
/* Workspace for a step of these params whose Full layers take at most max_x_tokens
 * new tokens and hold at most max_entries entries after the step. */
size_t csa2_runner_workspace_size(const csa2_runner* r, const csa2_step_params* p,
                                  int max_x_tokens, int max_entries);
/* Optional per-launch timing.  `events` holds n_events = n_layers * CSA2_STAGES * 2
 * cudaEvent_t handles (NULL entries are skipped).  Around stage s of layer l the
 * runner records events[(l * CSA2_STAGES + s) * 2 + 0] before and ... + 1] after the
 * stage's kernels, on the step's stream.  Stages: 0 compressor (projection GEMM +
 * pooling epilogue), 1 indexer key + FP4, 2 indexer scores, 3 top-k selection, 4 HSI
 * pool, 5 sparse attention.  NULL disables timing.  The runner keeps the pointer: the
 * array must stay valid for the steps that use it. */
#define CSA2_STAGES 6
int csa2_runner_set_timing(csa2_runner* r, void* const* events, int n_events);
/* Runs every layer in order on `stream`.  io[n_layers]. */
int csa2_runner_step(csa2_runner* r, const csa2_step_params* p, const csa2_layer_io* io,
                     void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
