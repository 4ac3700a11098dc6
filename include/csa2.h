/*
 * csa2.h - C ABI of the CSA2 step library (libcsa2.so): Compressed Sparse Attention 2 over an
 * FP4 main-KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The method (DeepSeek-V4.1-Flash, as described on the web pages cited below):
 *  - every attention layer is statically Full, Reindex or Reuse; Full selects fresh Top-512
 *    indices with its indexer Q against cached indexer K, Reindex rescores the same cache with
 *    its own indexer Q, Reuse takes the latest indices and skips the indexer
 *    (ai-maestro.online "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4",
 *    section "Compressed Sparse Attention 2"; wpnews.pro "DeepSeek V4.1 Flash Specs: KV Cache
 *    Compression Explained", section "What is Compressed Sparse Attention 2 CSA2?");
 *  - a Hierarchical Sparse Indexer lets the Full layer keep 2,048 blocks of eight tokens, a
 *    pool of up to 16,384 positions that later Reindex layers score instead of the whole
 *    context (same ai-maestro section; kongchang.com "DeepSeek V4.1 Flash Deep Dive",
 *    section "Compressed Absorption Attention (2nd Gen)");
 *  - main KV is stored as E2M1 codes with one E4M3 scale per 16 channels, NVFP4 without its
 *    global scale (ai-maestro section "FP4 KV, Bounded Replay, and other extensions");
 *  - every layer keeps its own main Q and a 128-token sliding-window KV (ai-maestro sections
 *    "Causal Encoder-Decoder architecture" and "Compressed Sparse Attention 2").
 * The pages give no dimensions, score formula or rounding rules.  This library fixes them:
 *   d = 512 latent channels shared as K and V, 16 main heads, indexer Q of 4 heads x 128 bf16
 *   with fp32 head weights, score s_t = sum_h w_h * relu(qI_h . KI_t) in a fixed fp32 order,
 *   Top-K ties broken by the lower position, scale byte = E4M3_RNE_satfinite(amax / 6).
 *
 * Conventions (all entry points):
 *  - Pointers are DEVICE pointers owned by the caller, unless stated otherwise.  The library
 *    never allocates device memory and never synchronises, except csa2_device_flags().
 *  - bf16 tensors are passed as uint16_t bit patterns; all arrays are contiguous, row-major,
 *    and 16-byte aligned (checked: misalignment returns CSA2_ERR_INVALID_ARG).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream).  Argument errors are reported synchronously by the return value and launch
 *    nothing.  Launch failures return CSA2_ERR_CUDA (from cudaGetLastError).
 *  - Data-dependent problems found on the device (a cache row outside [0, cap), a selected
 *    index outside the cache) are skipped, never dereferenced, and recorded as bits in a
 *    per-device flag word read by csa2_device_flags().
 *  - Scratch memory, where an entry point needs it, is the caller's `ws` buffer of at least
 *    csa2_workspace_size() bytes.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csa2_stream_t; /* cudaStream_t */
typedef struct CUevent_st* csa2_event_t;   /* cudaEvent_t  */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1, /* null/misaligned pointer, size out of range              */
  CSA2_ERR_UNSUPPORTED = 2, /* a dimension other than the fixed ones below              */
  CSA2_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed              */
  CSA2_ERR_WORKSPACE = 4,   /* ws is NULL or smaller than csa2_workspace_size()         */
  CSA2_ERR_TOO_LARGE = 5,   /* the problem needs more than the library's built-in scratch */
} csa2_status;

/* Fixed dimensions. */
#define CSA2_D 512          /* main latent channels (K = V)                      */
#define CSA2_GROUP 16       /* channels per E4M3 scale                           */
#define CSA2_CODE_BYTES 256 /* packed E2M1 bytes per cache row                   */
#define CSA2_SCALE_BYTES 32 /* E4M3 scale bytes per cache row                    */
#define CSA2_H 16           /* main heads                                        */
#define CSA2_HI 4           /* indexer heads                                     */
#define CSA2_DI 128         /* indexer width                                     */
#define CSA2_BLOCK 8        /* tokens per block of the hierarchical indexer      */
#define CSA2_MAX_K 2048     /* largest Top-K (blocks kept by the pool)           */
#define CSA2_MAX_ATTN_K 512 /* largest number of selected rows attended          */
#define CSA2_MAX_W 128      /* largest sliding window                            */
#define CSA2_MAX_LAYERS 16  /* layers per group descriptor                       */

/* Layer modes (ai-maestro "Compressed Sparse Attention 2"). */
#define CSA2_MODE_FULL 0
#define CSA2_MODE_REINDEX 1
#define CSA2_MODE_REUSE 2

/* Window row formats of csa2_group_desc.swa_format. */
#define CSA2_SWA_BF16 0
#define CSA2_SWA_E4M3 1

/* Device flag bits (csa2_device_flags). */
#define CSA2_FLAG_APPEND_OOB 1u /* an appended row fell outside [0, cap): row skipped   */
#define CSA2_FLAG_INDEX_OOB 2u  /* a selected index was >= cap: row treated as empty    */
#define CSA2_FLAG_TIMEOUT 4u    /* a kernel gave up waiting for its tensor-core work     */

/*
 * FP4 quantise-and-append.  "Main key-value cache quantises to E2M1 with one E4M3 scale per
 * 16 channels ... NVFP4 without its global scale" (ai-maestro "FP4 KV, Bounded Replay, and
 * other extensions"); quantised as it is written, without a separate pass (wpnews.pro TL;DR).
 *   x       bf16 [B][n_new][d], d must be 512.
 *   codes   uint8 [B][cap][256]: byte i of a row holds channel 2i in its low nibble and
 *           channel 2i+1 in its high nibble, E2M1 (sign, 2-bit exponent bias 1, 1 mantissa).
 *   scales  uint8 [B][cap][32]: E4M3 (FN) scale of channels 16g..16g+15.
 *   offsets int32 [B] or NULL: row r of sequence b is written to cache row offsets[b] + r
 *           (NULL: row r).  Rows outside [0, cap) are skipped (CSA2_FLAG_APPEND_OOB).
 * Per group: s8 = E4M3_RNE_satfinite(fp32(amax / 6)); code_i = E2M1_RNE_satfinite(fp32(x_i / s))
 * with s the decoded scale; s == 0 gives all-zero codes; the code's sign bit is x_i's sign.
 */
csa2_status csa2_fp4_quantize_append(const uint16_t* x, int B, int n_new, int d, uint8_t* codes,
                                     uint8_t* scales, int64_t cap, const int32_t* offsets,
                                     csa2_stream_t stream);

/*
 * 8-bit window rows (kongchang.com "DeepSeek V4.1 Flash Deep Dive", section "Compressed Absorption
 * Attention (2nd Gen)": the sliding window is kept in 8-bit precision): out[i] = E4M3FN(x[i]) for
 * n bf16 values, round-to-nearest-even, saturating to +-448, a zero result keeping x's sign; no
 * scale.  Fills the window buffers of groups with swa_format = CSA2_SWA_E4M3.  x and out 16-byte
 * aligned.  Asynchronous on `stream`.
 */
csa2_status csa2_fp8_quantize(const uint16_t* x, int64_t n, uint8_t* out, csa2_stream_t stream);

/*
 * FP4 dequantisation of `rows` cache rows: out[r][c] = E2M1(code) * E4M3(scale), exact in bf16.
 *   codes [rows][256], scales [rows][32] -> out bf16 [rows][512].  d must be 512.
 */
csa2_status csa2_fp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int d,
                                uint16_t* out, csa2_stream_t stream);

/*
 * Lightning-indexer scores of indexer Q against cached indexer K ("Full: ... projects the
 * indexer K ... selects fresh Top-512", "Reindex: ... rescores them with its own indexer Q",
 * ai-maestro "Compressed Sparse Attention 2").  s_t = sum_h w_h * relu(qI_h . KI_t), in the
 * fixed fp32 order: per head eight fused-multiply-add chains over channels 16j..16j+15 from
 * +0, combined as ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)); relu; (w0 r0 + w1 r1) + (w2 r2 + w3 r3).
 *   qI      bf16 [B][Nq][4][128];  w fp32 [B][Nq][4];  KI bf16 [B][cap][128]
 *   lens    int32 [B]: entries T_b present in sequence b's cache (clamped to cap).
 *   ratio   tokens per cache entry (>= 1); query i of sequence b sits at token position
 *           q_pos[b*Nq+i] (q_pos may be NULL: position ratio*T_b - Nq + i) and sees entry j
 *           iff ratio*j + ratio - 1 <= its position (causal mask over compressed entries).
 *   cand    NULL: row r of `scores` is [cap] and entry t holds the score of cache entry t.
 *           else int32 [B*Nq][n_cand] ascending cache positions (a pool) with cand_len[B*Nq]
 *           valid entries; entry i of the row holds the score of position cand[r][i].
 *   scores  fp32 [B*Nq][cap or n_cand]: the visible entries form a prefix of length
 *           n_valid[r] (nullable output); the rest of the row is set to -inf.
 */
csa2_status csa2_index_score(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                             int64_t cap, const int32_t* lens, const int32_t* cand,
                             const int32_t* cand_len, int64_t n_cand, int ratio,
                             const int32_t* q_pos, float* scores, int32_t* n_valid,
                             csa2_stream_t stream);

/*
 * Exact Top-K per row ("selects fresh Top-512 indices", ai-maestro "Compressed Sparse
 * Attention 2"; Top-2,048 blocks for the pool).  Larger score first, equal scores (with -0 ==
 * +0) by lower column; the selected columns are returned in ascending order, padded with -1.
 *   scores  fp32 [rows][ld]; row r uses columns [0, n_valid[r]) (n_valid NULL: [0, n)), n <= ld.
 *           Scores must not be NaN.
 *   k       1..2048.
 *   map     NULL, or int32 [rows][map_ld]: output map[r][col] instead of col (an ascending map
 *           such as a pool keeps the output ascending).
 *   idx     int32 [rows][k];  n_sel int32 [rows] (nullable): min(k, valid columns).
 *   ws      workspace of csa2_workspace_size(CSA2_OP_TOPK, ...) bytes, 16-byte aligned: for rows
 *           longer than 8192 columns the candidate lists, per-row counters, histograms and
 *           16-column group keys of the multi-CTA selection (the call clears what must start at
 *           zero); 0 bytes, and ws may be NULL, otherwise.  Rows of 8193 to 131072 columns select
 *           in one launch of a thread-block cluster per row that keeps all of this in shared
 *           memory, so only longer rows touch ws; the size asked for stays the same.
 */
csa2_status csa2_topk(const float* scores, int rows, int64_t n, int64_t ld, const int32_t* n_valid,
                      int k, const int32_t* map, int64_t map_ld, int32_t* idx, int32_t* n_sel,
                      void* ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * Block keys of the hierarchical indexer: key of block j = bf16_RNE(0.125 * sum of indexer keys
 * 8j .. 8j+7, summed in token order in fp32), for the complete blocks j < lens[b] / 8 of each
 * sequence (ai-maestro "Compressed Sparse Attention 2": "2,048 blocks of eight tokens").
 *   KI bf16 [B][cap][128] -> block_keys bf16 [B][cap/8][128].  Other rows are not written.
 */
csa2_status csa2_block_keys_build(const uint16_t* KI, int B, int64_t cap, const int32_t* lens,
                                  uint16_t* block_keys, csa2_stream_t stream);

/*
 * Hierarchical pool of the Full layer: score the visible complete blocks of each query with
 * its indexer Q (same score as csa2_index_score), keep the top min(keep, blocks) blocks (ties
 * to the lower block) and expand them into ascending token positions.
 *   block_keys bf16 [B][cap/8][128]; lens, ratio, q_pos as csa2_index_score.
 *   pool int32 [B*Nq][keep*8] (-1 padded), pool_len int32 [B*Nq].  keep in 1..2048.
 *   ws   csa2_workspace_size(CSA2_OP_BLOCK_POOL, ...) bytes.
 */
csa2_status csa2_block_pool(const uint16_t* qI, const float* w, int B, int Nq,
                            const uint16_t* block_keys, int64_t cap, const int32_t* lens, int ratio,
                            const int32_t* q_pos, int keep, int32_t* pool, int32_t* pool_len,
                            void* ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * Exact Top-k cache positions for every query of a prefill chunk, by the indexer score
 * s_t = sum_h w_h relu(qI_h . KI_t) in the canonical fp32 order (ai-maestro "Compressed Sparse
 * Attention 2"; the causal compressed positions of "Causal Encoder-Decoder architecture"), without
 * materialising the scores.  The dense [B*Nq*4 x 128] x [128 x T] product runs on the tensor cores
 * twice: first to bound each query's k-th score from below, then to mark every key whose
 * tensor-core score is within twice a rigorous error bound of that bound; the marked keys are
 * rescored canonically and selected exactly.  The result is identical to csa2_index_score followed
 * by csa2_topk (same tie rule, same visibility).
 *   qI bf16 [B][Nq][4][128], w fp32 [B][Nq][4] (16-byte aligned), KI bf16 [B][cap][128], lens,
 *   ratio, q_pos as csa2_index_score.  k in 1..2048.
 *   idx int32 [B*Nq][k] ascending, -1 padded when fewer than k positions are visible;
 *   n_sel int32 [B*Nq] (nullable): the number selected.
 *   ws csa2_workspace_size(CSA2_OP_INDEX_SELECT_PREFILL, {B, Nq, cap}) bytes.
 * Tensor-core waits are bounded; one that runs out sets CSA2_FLAG_TIMEOUT.
 */
csa2_status csa2_index_select_prefill(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                                      int64_t cap, const int32_t* lens, int ratio, const int32_t* q_pos, int k,
                                      int32_t* idx, int32_t* n_sel, void* ws, size_t ws_bytes,
                                      csa2_stream_t stream);

/*
 * Sparse attention of each query's 16 heads over its selected FP4 rows plus its sliding-window
 * rows ("Every layer retains its own main Q and sliding-window key-value cache", ai-maestro
 * "Compressed Sparse Attention 2"; 128-token window, "Causal Encoder-Decoder architecture").
 * K = V = the dequantised row; softmax over the union of the rows (a token in both sets
 * counts twice); split-KV over the rows with an online-softmax combine.
 *   q      bf16 [B][Nq][16][512]
 *   idx    int32 [B*Nq][k] cache positions (k <= 512); entries < 0, or at or past n_valid[r]
 *          (n_valid nullable), are empty.  Positions >= cap are treated as empty and flagged.
 *   swa    bf16 [B][W-1+Nq][512] or NULL (no window); query i attends rows i .. i+W-1, of which
 *          rows >= (W-1+Nq) - swa_len[b] hold tokens (swa_len int32 [B]).  W <= 128.
 *   out    bf16 [B][Nq][16][512];  lse fp32 [B][Nq][16] (nullable), natural log; a query with
 *          no rows gets out = 0 and lse = -inf.
 *   n_split  CTAs per query (0..32, 0 = chosen from the problem size).  A query's rows form
 *          64-row tiles (ceil(k/64) of selected rows, ceil(W/64) of window rows); larger splits
 *          than tiles are clamped to the tile count.  Entries of the same query are combined in split
 *          order, so results do not depend on scheduling.
 *   ws     csa2_workspace_size(CSA2_OP_SPARSE_ATTN, ...) bytes for the chosen split.
 * Tensor-core waits are bounded (about one second); one that runs out sets CSA2_FLAG_TIMEOUT.
 */
csa2_status csa2_sparse_attn_decode(const uint16_t* q, int B, int Nq, const uint8_t* codes,
                                    const uint8_t* scales, int64_t cap, const int32_t* idx,
                                    const int32_t* n_valid, int k, const uint16_t* swa,
                                    const int32_t* swa_len, int W, float softmax_scale,
                                    uint16_t* out, float* lse, int n_split, void* ws,
                                    size_t ws_bytes, csa2_stream_t stream);

/*
 * csa2_sparse_attn_decode without a workspace argument.  The pages have no counterpart: this is an
 * interface convenience.  Some callers cannot allocate device memory when they call: code running
 * inside a memory allocator's callbacks (allocating would re-enter the allocator), a service whose
 * device memory budget is reserved up front (nothing is left to allocate from), a plugin handed only
 * its input and output buffers (it owns no allocator).  This entry point takes the same arguments as
 * csa2_sparse_attn_decode minus ws / ws_bytes and allocates nothing.  Its scratch (the split
 * partials and one ticket per query) is a fixed array of csa2_sparse_attn_static_scratch_bytes()
 * (16 MiB) inside the library, which every GPU that loads the library reserves until the process
 * exits; a call whose split needs more returns CSA2_ERR_TOO_LARGE.  A split needs 32,896 B per
 * query and split plus 4 B per query: a decode batch of 64 queries at its automatic split of 2
 * (one CTA per SM on a 152-SM GB300) needs about 4.2 MB and fits, 128 queries forced to a split
 * of 5 need about 21 MB and are refused
 * (csa2_attn_auto_split gives the automatic split).  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it for the life of the process (a device
 * reset while the library is loaded is not supported), so make that first call before any stream
 * capture on the device.  Every call uses the same array and leaves its contents behind (the tickets are
 * cleared at the start of each call): calls that may overlap on the GPU, from any stream or host
 * thread, race and must be ordered by the caller.
 */
csa2_status csa2_sparse_attn_decode_static(const uint16_t* q, int B, int Nq, const uint8_t* codes,
                                           const uint8_t* scales, int64_t cap, const int32_t* idx,
                                           const int32_t* n_valid, int k, const uint16_t* swa,
                                           const int32_t* swa_len, int W, float softmax_scale,
                                           uint16_t* out, float* lse, int n_split, csa2_stream_t stream);

/* Bytes of the built-in scratch used by csa2_sparse_attn_decode_static. */
size_t csa2_sparse_attn_static_scratch_bytes(void);

/*
 * One CSA2 layer group (ai-maestro "Compressed Sparse Attention 2": Full / Reindex / Reuse,
 * groups such as 1 Full + 3 Reuse, 1 Full + 5 Reuse, Reindex + 3 Reuse).  Layers run in order:
 *   FULL     optionally appends the step's new rows first (kv_new -> FP4 cache rows and ki_new
 *            -> indexer-K rows at lens[b] - n_new .. lens[b] - 1, refreshing completed block
 *            keys when hierarchical), then scores (pool: blocks first) and selects Top-K.
 *   REINDEX  rescores with its own qI / w: the pool of the latest Full layer when hierarchical
 *            (pool / pool_len hold it, possibly from an earlier group), else all visible
 *            entries; selects Top-K.
 *   REUSE    attends with the latest layer's indices; no scoring.
 * Every layer attends with its own q and window; window rows are bf16, or one E4M3 byte per
 * channel with swa_format = CSA2_SWA_E4M3 (csa2_fp8_quantize).  The first layer must be FULL or
 * REINDEX.
 * Attention: consecutive layers that attend the same rows run in one launch; with n_split = 0 and
 * at least two CTAs per SM of (query, layer pair) work (prefill chunks), each CTA takes two layers
 * and gathers and dequantises their shared rows once.  The results stay within the same tolerance.
 * Execution: the batch is cut into `seq_chunks` groups of whole sequences (0: one group).  With
 * more than one group, the first indexer scan of group c runs on `stream` while the remaining
 * work of group c-1 runs on a library-owned, highest-priority stream of the current device
 * (created with its events on first use), which waits on an event recorded on `stream` and is
 * joined back into `stream` before the call returns.  All of the step's work is therefore ordered
 * after earlier work on `stream` and before later work on it; calls from several host threads
 * are serialised while they enqueue.
 */
typedef struct csa2_group_desc {
  int n_layers;                       /* 1 .. CSA2_MAX_LAYERS                            */
  int modes[CSA2_MAX_LAYERS];         /* CSA2_MODE_* per layer                           */
  int B, Nq;                          /* sequences, queries per sequence                 */
  int K;                              /* selected rows per query, 1..512                 */
  int W;                              /* window, 0..128                                  */
  int ratio;                          /* tokens per cache entry, >= 1                    */
  int hierarchical;                   /* 0: flat indexer, 1: block pool                  */
  int n_blocks_keep;                  /* blocks kept by the pool, 1..2048                */
  int n_split;                        /* attention split, 0 = automatic                  */
  int n_new;                          /* rows appended by the Full layer (0: none)       */
  int seq_chunks;                     /* sequence chunks pipelined over two streams, 0 = 1 */
  int swa_format;                     /* CSA2_SWA_BF16, or CSA2_SWA_E4M3: swa[l] holds one
                                         E4M3 byte per channel (rows of 512 B)           */
  int64_t cap;                        /* cache capacity (entries) per sequence           */
  const int32_t* lens;                /* [B] entries present (after the append)          */
  const int32_t* q_pos;               /* [B*Nq] query token positions, or NULL           */
  uint8_t* codes;                     /* [B][cap][256] FP4 main KV                       */
  uint8_t* scales;                    /* [B][cap][32]                                    */
  uint16_t* KI;                       /* [B][cap][128] indexer keys                      */
  uint16_t* block_keys;               /* [B][cap/8][128] (hierarchical)                  */
  const uint16_t* kv_new;             /* [B][n_new][512] bf16, or NULL                   */
  const uint16_t* ki_new;             /* [B][n_new][128] bf16, or NULL                   */
  const uint16_t* q[CSA2_MAX_LAYERS];  /* [B][Nq][16][512]                               */
  const uint16_t* qI[CSA2_MAX_LAYERS]; /* [B][Nq][4][128]  (FULL / REINDEX)              */
  const float* w[CSA2_MAX_LAYERS];     /* [B][Nq][4]       (FULL / REINDEX)              */
  const uint16_t* swa[CSA2_MAX_LAYERS];/* [B][W-1+Nq][512] or NULL                       */
  const int32_t* swa_len;             /* [B] valid window rows                           */
  uint16_t* out[CSA2_MAX_LAYERS];     /* [B][Nq][16][512]                                */
  float* lse[CSA2_MAX_LAYERS];        /* [B][Nq][16] or NULL                             */
  int32_t* idx[CSA2_MAX_LAYERS];      /* [B*Nq][K]: written by FULL / REINDEX (required),
                                         for REUSE a copy of the reused indices if non-NULL */
  int32_t* pool;                      /* [B*Nq][keep*8] (hierarchical)                   */
  int32_t* pool_len;                  /* [B*Nq]         (hierarchical)                   */
  float softmax_scale;                /* e.g. 1/sqrt(512)                                */
  csa2_event_t ev_score_begin;        /* optional: recorded on `stream` before the first  */
  csa2_event_t ev_score_end;          /*   indexer scan of the step and after the last   */
  csa2_event_t ev_attn_begin;         /* optional: recorded on the attention stream right */
  csa2_event_t ev_attn_end;           /*   before and after the step's first attention
                                         launch (a run of layers sharing their rows)     */
} csa2_group_desc;

csa2_status csa2_group_step(const csa2_group_desc* g, void* ws, size_t ws_bytes,
                            csa2_stream_t stream);

/*
 * One token's pass through a decoder stack of layer groups (ai-maestro "Compressed Sparse
 * Attention 2": Reindex layers "reuse the most recent Full layer's KV and indexer keys"; the
 * 20-layer decoder as 5 groups of 4, the first led by a Full layer, the rest by Reindex layers).
 * groups[0 .. n_groups-1] run in order, each exactly as csa2_group_step, on one workspace (the
 * largest group's csa2_workspace_size).  All groups share B, Nq, cap, lens, q_pos, ratio, the
 * cache (codes, scales, KI) and, when hierarchical, block_keys and the pool buffers (a Reindex-led
 * group rescores the pool kept by the latest Full layer of an earlier group).  Only groups[0] may
 * append (kv_new / ki_new).  Every group is checked before anything is launched: a mismatch, or
 * any check of csa2_group_step failing, returns its status with nothing enqueued.
 */
csa2_status csa2_stack_step(const csa2_group_desc* groups, int n_groups, void* ws, size_t ws_bytes,
                            csa2_stream_t stream);

/*
 * Context split of one sequence's cache over G shards (one per GPU, or G logical shards on one GPU):
 * shard g holds the cache entries [lo_g, hi_g), lo_0 = 0, hi_g = lo_{g+1}.  A query then selects in
 * two steps and attends in two (the exchanges between them are the caller's collectives):
 *   csa2_shard_topk_pairs   each shard: the local Top-k of its own scores as (score, position) pairs;
 *   csa2_merge_topk_pairs   the G x k pairs -> the exact global Top-k (the union of the local Top-k
 *                           sets contains the global one);
 *   csa2_shard_indices      each shard: the selected positions it holds, as local rows;
 *   csa2_attn_merge_shards  the shards' attention outputs and lse -> attention over the union.
 * The result equals the unsplit step: the same indices, and attention within the tolerance of the
 * extra bf16 rounding of each shard's output.  The pages motivate bounded work per query at 1M
 * context (ai-maestro "Compressed Sparse Attention 2": a pool of up to 16,384 positions); they do
 * not describe a split, and this one is the plainest exact one.
 */

/* The local Top-k of one shard as (score, global position) pairs.  scores, rows, n, ld, n_valid, k,
 * map, map_ld, ws and ws_bytes are as in csa2_topk (the workspace is csa2_workspace_size(
 * CSA2_OP_TOPK, {B = rows, Nq = 1, n})).  pos_offset is the global position of local column 0 (lo_g);
 * with a map, the map's entries are the global positions instead.
 *   pair_score fp32 [rows][k], pair_pos int32 [rows][k]: ascending positions, -1 / -inf padded;
 *   pair_n int32 [rows] (nullable): the valid pairs, min(k, visible columns). */
csa2_status csa2_shard_topk_pairs(const float* scores, int rows, int64_t n, int64_t ld, const int32_t* n_valid,
                                  int k, const int32_t* map, int64_t map_ld, int64_t pos_offset, float* pair_score,
                                  int32_t* pair_pos, int32_t* pair_n, void* ws, size_t ws_bytes,
                                  csa2_stream_t stream);

/* The exact Top-k of G shards' pairs (larger score first, equal scores by lower position), as csa2_topk
 * of the unsplit scores would select.
 *   pair_score fp32 [G][rows][k], pair_pos int32 [G][rows][k], pair_n int32 [G][rows] (nullable: all k
 *   valid): shard g's output of csa2_shard_topk_pairs; shards in ascending order of their position
 *   ranges (the caller's contract: ties are broken by position through that order).  G in 1..64.
 *   idx int32 [rows][k] ascending global positions, -1 padded; n_sel int32 [rows] (nullable).
 *   ws csa2_workspace_size(CSA2_OP_MERGE_PAIRS, {B = rows, Nq = 1, n = G, k}) bytes, 16-byte aligned. */
csa2_status csa2_merge_topk_pairs(const float* pair_score, const int32_t* pair_pos, const int32_t* pair_n, int G,
                                  int rows, int k, int32_t* idx, int32_t* n_sel, void* ws, size_t ws_bytes,
                                  csa2_stream_t stream);

/* idx_local[r][j] = idx[r][j] - lo when lo <= idx[r][j] < hi, else -1 (an empty slot for
 * csa2_sparse_attn_decode): the selected rows a shard holding [lo, hi) attends. */
csa2_status csa2_shard_indices(const int32_t* idx, int rows, int k, int64_t lo, int64_t hi, int32_t* idx_local,
                               csa2_stream_t stream);

/* Attention over the union of the shards' rows from each shard's attention over its own rows:
 * out_g bf16 [G][rows][16][512] and lse_g fp32 [G][rows][16] (csa2_sparse_attn_decode's out and lse)
 * -> out bf16 [rows][16][512] = sum_g exp(lse_g - L) out_g with L = log sum_g exp(lse_g), combined in
 * shard order in fp32; lse fp32 [rows][16] (nullable) = L.  A shard with lse = -inf weighs nothing; a
 * row no shard attended gets out = 0, lse = -inf.  out_g and out 16-byte aligned. */
csa2_status csa2_attn_merge_shards(const uint16_t* out_g, const float* lse_g, int G, int rows, uint16_t* out,
                                   float* lse, csa2_stream_t stream);

/* Workspace sizing. */
#define CSA2_OP_TOPK 1
#define CSA2_OP_BLOCK_POOL 2
#define CSA2_OP_SPARSE_ATTN 3
#define CSA2_OP_GROUP_STEP 4
#define CSA2_OP_INDEX_SELECT_PREFILL 5
#define CSA2_OP_MERGE_PAIRS 6

typedef struct csa2_dims {
  int B, Nq;
  int64_t cap;          /* cache capacity per sequence                        */
  int64_t n;            /* CSA2_OP_TOPK: columns per row; CSA2_OP_MERGE_PAIRS: shards */
  int k;                /* Top-K / selected rows                              */
  int W;                /* window                                             */
  int n_split;          /* CSA2_OP_SPARSE_ATTN / GROUP_STEP: 0 = automatic    */
  int hierarchical;     /* CSA2_OP_GROUP_STEP                                 */
  int n_blocks_keep;    /* CSA2_OP_BLOCK_POOL / GROUP_STEP                    */
} csa2_dims;

/* Bytes of workspace `op` needs for `dims` (0 if none); 0 with dims == NULL. */
size_t csa2_workspace_size(int op, const csa2_dims* dims);

/* Split-KV factor the library picks for `instances` (= B*Nq) attention queries of k rows. */
int csa2_attn_auto_split(int64_t instances, int k, int W);

/* sizeof(csa2_group_desc) as compiled into the library (lets bindings check their layout). */
size_t csa2_group_desc_size(void);

/* Static text for a status code. */
const char* csa2_status_string(csa2_status s);

/* Synchronises `stream`, returns the current device's flag word (CSA2_FLAG_*) in *flags (a
 * HOST pointer) and clears it when `clear` is nonzero. */
csa2_status csa2_device_flags(uint32_t* flags, int clear, csa2_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */
