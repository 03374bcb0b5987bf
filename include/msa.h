/*
 * msa.h -- C ABI of a single-GPU (sm_103a) library for two-stage GQA
 * block-sparse attention, the "MiniMax Sparse Attention" block.
 *
 * Source of the method: the Atlas Cloud guide "MiniMax goes sparse: decoding
 * M3's attention from a single diagram" (Portuguese, Spanish and French
 * editions), section 1:
 *   Step 1 (index branch): each GQA group has one index query; block-level
 *     scores are formed from token keys pooled per fixed-size block; a top-k
 *     keeps a short list of KV blocks per layer and per group.
 *   Step 2 (sparse branch): every query head of a group attends, with ordinary
 *     softmax attention, over the real (uncompressed) K/V of the blocks its
 *     group selected.
 * Where the guide leaves a step open, this library fixes it as a parameter:
 *   - block size 64 tokens;
 *   - block summary key = mean of the block's 64 keys of the KV head itself
 *     (scoring it equals the block mean of the token scores);
 *   - group index query = sum of the group's query heads (decode) or of the
 *     tile's 64 tokens x group heads (prefill);
 *   - the block holding the newest token (decode) or the tile's diagonal block
 *     (prefill) is always kept and never scored;
 *   - top-k ties go to the lower block index.
 *
 * Conventions for every call:
 *   - Every pointer argument is a DEVICE pointer unless marked "host".
 *   - The caller owns and allocates every buffer (inputs, outputs, workspace);
 *     the library never allocates device memory and never synchronises the
 *     stream, except msa_read_device_status.
 *   - Calls are asynchronous on `stream`. Calls that share a workspace must be
 *     ordered on one stream; distinct workspaces make calls independent.
 *   - Argument errors are found on the host before any launch and return
 *     MSA_ERR_INVALID_ARG / MSA_ERR_UNSUPPORTED / MSA_ERR_WORKSPACE with no
 *     work queued. A failed launch returns MSA_ERR_CUDA.
 *   - Data-dependent errors (a page id outside [0, num_pages), a sequence
 *     length above the cache capacity) never fault: the kernel skips the access
 *     and sets a sticky status word in the workspace, read with
 *     msa_read_device_status.
 *   - Head dimension D = 128 and block size 64 are the only supported values.
 *   - q, out, k, v and the pooled keys are moved in 16-byte pieces (vector
 *     loads and stores, asynchronous and tensor-memory-access copies): their
 *     base addresses must be 16-byte aligned (MSA_ERR_INVALID_ARG otherwise).
 *
 * Layouts (row-major, innermost last):
 *   q (decode)   [batch, num_q_heads, 128]         KV dtype
 *   q (prefill)  [n_q_tokens, num_q_heads, 128]    KV dtype
 *   KV contiguous  k, v: [batch, num_kv_heads, max_tokens, 128]
 *   KV paged       k, v: [num_pages, num_kv_heads, 64, 128], page_table
 *                  [batch, max_pages_per_seq] int32 (logical block -> page)
 *   pooled keys (same dtype as KV), per (sequence, KV head) in logical block
 *   order for both cache layouts, so a unit's candidates are one run of rows:
 *     contiguous   [batch, num_kv_heads, max_tokens/64, 128]
 *     paged        [batch, num_kv_heads, max_pages_per_seq, 128]
 *   Query head j belongs to KV head j / G, G = num_q_heads / num_kv_heads.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* msa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shapes */
  MSA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim != 128) */
  MSA_ERR_WORKSPACE = 3,     /* workspace null or smaller than msa_workspace_size */
  MSA_ERR_CUDA = 4,          /* a CUDA launch or API call failed */
  MSA_ERR_DEVICE_BOUNDS = 5, /* (device status) a page id or length was out of range */
  MSA_ERR_TIMEOUT = 6        /* (device status) a bounded wait gave up */
} msa_status;

typedef enum msa_dtype { MSA_DTYPE_F32 = 0, MSA_DTYPE_BF16 = 1 } msa_dtype;
typedef enum msa_kv_layout { MSA_KV_CONTIGUOUS = 0, MSA_KV_PAGED = 1 } msa_kv_layout;

/* The block-scoring operator of Step 1.
 * MEAN_POOLED_KEYS: q_idx . pooled[b], the summary key being the mean of the
 *   block's keys of the KV head itself -- by linearity the block mean of the
 *   token scores q_idx . k_t.
 * TOKEN_MAX: the guide's Step 1 as drawn (§1, Step 1: token-level scores
 *   against a single index-key head shared by all groups, then a block max
 *   pool): max over the block's 64 tokens of q_idx . K_idx[t], with K_idx a
 *   caller-provided index-key cache passed in place of the summaries. */
typedef enum msa_score_mode { MSA_SCORE_MEAN_POOLED_KEYS = 0, MSA_SCORE_TOKEN_MAX = 1 } msa_score_mode;

/* Description of a KV cache. All pointers are device pointers. */
typedef struct msa_kv_desc {
  int32_t layout;            /* msa_kv_layout */
  int32_t dtype;             /* msa_dtype of k, v, q, pooled keys and outputs */
  int32_t batch;             /* number of sequences */
  int32_t num_kv_heads;      /* Hkv */
  int32_t head_dim;          /* must be 128 */
  int32_t block_size;        /* must be 64 */
  const void* k;             /* keys, layout above */
  const void* v;             /* values, same layout as k */
  int64_t max_tokens;        /* contiguous: token capacity per sequence, a multiple of 64 */
  const int32_t* page_table; /* paged: [batch, max_pages_per_seq] */
  int32_t max_pages_per_seq; /* paged */
  int32_t num_pages;         /* paged: number of pages in k and v */
  const int32_t* seq_lens;   /* [batch] tokens present per sequence (device) */
} msa_kv_desc;

/* Step-1 selection parameters. */
typedef struct msa_select_cfg {
  int32_t k_scored;    /* number of scored blocks to keep per unit, >= 0 */
  int32_t force_local; /* bit 0 (1): always keep the newest / diagonal block; bit 1 (2): always keep
                          block 0, an attention sink (guide §2 names a sink among the likely
                          replacements of the sliding window). Kept blocks are not scored. */
  int32_t q_tile;      /* 1: decode (one token per sequence); 64: prefill tiles */
  int32_t mode;        /* msa_score_mode */
  int64_t q_start;     /* prefill: absolute position of the first query token (any position) */
} msa_select_cfg;

/* Operation ids for msa_workspace_size. */
typedef enum msa_op {
  MSA_OP_POOL = 0,
  MSA_OP_SELECT = 1,         /* msa_select_topk_blocks with q_tile 1 (decode) */
  MSA_OP_DECODE = 2,
  MSA_OP_PREFILL = 3,
  MSA_OP_DENSE_DECODE = 4,
  MSA_OP_DENSE_PREFILL = 5,
  MSA_OP_SELECT_PREFILL = 6, /* msa_select_topk_blocks with q_tile 64 (n_q_tokens =
                                the chunk's tokens), and
                                msa_select_topk_blocks_varlen with n_q_tokens =
                                64 * the batch's query tiles (see
                                msa_select_topk_blocks_varlen) */
  MSA_OP_DECODE_STEP = 7     /* msa_sparse_decode_step */
} msa_op;

/* Bytes of workspace `op` needs for these shapes (host call, no GPU work).
 * n_q_tokens is 1 for decode ops; k_total is the index-list length (ignored by
 * dense ops). Returns 0 when the arguments are invalid. A workspace must be
 * zero-filled once before its first use (msa_workspace_init); the library
 * leaves it ready for the next call. One workspace of the largest size serves
 * every op. */
size_t msa_workspace_size(int32_t op, const msa_kv_desc* kv /* host */, int32_t num_q_heads,
                          int32_t n_q_tokens, int32_t k_total);

/* Zero-fill `bytes` of workspace on `stream` (a memset; no allocation). */
msa_status msa_workspace_init(void* ws, size_t bytes, msa_stream_t stream);

/* Step 1a -- block summary keys (guide §1, Step 1, block pooling of the index
 * branch). For every complete block b (64 b + 63 < seq_len) of every
 * (sequence, KV head) with first_block <= b < first_block + n_blocks
 * (n_blocks = -1: all), writes pooled[b] = (1/64) * sum_{i<64} K[64 b + i]:
 * fp32 sum in row order, one multiply by 1/64, rounded to nearest even into
 * the KV dtype. Partial blocks are left untouched. Bad page ids set
 * MSA_ERR_DEVICE_BOUNDS in the status word when `ws` is given (ws may be NULL:
 * then bad pages are skipped silently); a skipped block's summary is not
 * written, the selection scores whatever that row holds, and the attention
 * reports the page again when the block is selected. */
msa_status msa_pool_block_keys(const msa_kv_desc* kv /* host */, int64_t first_block, int64_t n_blocks,
                               void* pooled, void* ws, size_t ws_bytes, msa_stream_t stream);

/* Step 1b/1c -- group index query, block scores and top-k (guide §1, Step 1:
 * one index query per GQA group, scores per block, TopK keeps the k best
 * blocks per layer and group).
 * Decode (cfg->q_tile == 1): q [batch, Hq, 128]; unit = (sequence, KV head);
 *   q_idx = sum of the group's G query heads (fp32); candidates are the
 *   complete blocks, minus the newest block nb-1 (nb = ceil(seq_len/64)) when
 *   force_local. Output idx_out [batch, Hkv, k_total].
 * Prefill (cfg->q_tile == 64, batch 1, contiguous or paged cache): q [n_q_tokens, Hq, 128] at
 *   absolute positions cfg->q_start + r (any q_start). The chunk's query
 *   tiles are its tokens grouped by the 64-token block they sit in: tile j
 *   holds the tokens whose position is in block q_start/64 + j (its diagonal
 *   block), so a chunk that starts inside a block has a shorter first tile;
 *   there are n_tiles = (q_start + n_q_tokens - 1)/64 - q_start/64 + 1 tiles.
 *   Unit = (tile j, KV head); q_idx = sum over the tile's tokens and the
 *   group's heads; candidates are the blocks before the diagonal block.
 *   Output idx_out [n_tiles, Hkv, k_total].
 * Scores are q_idx . pooled[b] in fp32 (unscaled). The top min(k_scored, n)
 * candidates by (score descending, block ascending) plus the forced block are
 * written sorted ascending, padded with -1;
 * k_total >= min(k_scored, max_blocks) + the number of kept blocks (bits of
 * force_local). With the sink bit, block 0 leads the list and the candidates
 * start at block 1.
 * scores_out (nullable): [units, max_blocks] fp32 raw scores of the candidate
 * blocks (max_blocks = max_tokens/64 or max_pages_per_seq); other entries are
 * left unspecified.
 * cfg->mode == MSA_SCORE_TOKEN_MAX (bf16, Hkv <= 8; else
 *   MSA_ERR_UNSUPPORTED): `pooled` is the index-key cache instead, one shared
 *   head laid out like one KV head of the cache -- contiguous
 *   [batch, max_tokens, 128], paged [num_pages, 64, 128] on the cache's pages
 *   -- and the score of block b is max_{t in b} q_idx . K_idx[t] (fp32), for
 *   decode and for prefill tiles alike. The index keys of a sequence are read
 *   once for all of its KV heads (decode) or once per group of 16 tiles
 *   (prefill). */
msa_status msa_select_topk_blocks(const void* q, int32_t num_q_heads, int32_t n_q_tokens,
                                  const void* pooled, const msa_kv_desc* kv /* host */,
                                  const msa_select_cfg* cfg /* host */, int32_t* idx_out, int32_t k_total,
                                  float* scores_out, void* ws, size_t ws_bytes, msa_stream_t stream);

/* Step 1b/1c for a batch of chunks (guide §1, Step 1, applied to the prefill
 * chunk of every sequence of a batch at once): sequence s (n_seqs ==
 * kv->batch, at most 64) has q_counts[s] >= 0 new tokens at absolute positions
 * q_starts[s] + r (q_starts[s] + q_counts[s] within the sequence's capacity;
 * both arrays on the host). q holds the sequences' tokens back to back:
 * [sum q_counts, Hq, 128], sequence s from row q_off[s] = q_counts[0] + ... +
 * q_counts[s-1]. Its query tiles (tokens grouped by the 64-token block they sit
 * in, as for msa_select_topk_blocks: n_s = (q_starts[s] + q_counts[s] - 1)/64 -
 * q_starts[s]/64 + 1 tiles, none for an empty chunk) are numbered globally in
 * the same order (tile_off[s] + j), and idx_out [total tiles, Hkv, k_total]
 * gets, for global tile
 * tile_off[s] + j, exactly what msa_select_topk_blocks (q_tile 64, q_start =
 * q_starts[s]) gives for tile j of sequence s alone, scored against sequence
 * s's summaries (pooled [batch, Hkv, max_blocks, 128]; in token-max mode the
 * index-key cache). cfg->q_tile must be
 * 64 (cfg->q_start is ignored); fp32 caches take one sequence only
 * (MSA_ERR_UNSUPPORTED above). A batch with no new tokens queues nothing. */
msa_status msa_select_topk_blocks_varlen(const void* q, int32_t num_q_heads, int32_t n_seqs,
                                         const int64_t* q_starts /* host */, const int32_t* q_counts /* host */,
                                         const void* pooled, const msa_kv_desc* kv /* host */,
                                         const msa_select_cfg* cfg /* host */, int32_t* idx_out, int32_t k_total,
                                         float* scores_out, void* ws, size_t ws_bytes, msa_stream_t stream);

/* Step 2, decode (guide §1, Step 2: attention over the gathered selected
 * blocks; all heads of a group share the group's list).
 * For each sequence s and query head j (KV head h = j / G):
 *   o = sum_t softmax_t(scale * q_j . K[t]) V[t]
 * over the tokens t < seq_len[s] of the blocks idx[s, h, 0..k_total) (-1
 * entries ignored; duplicates are not allowed); batch * Hkv <= 16384 units
 * (MSA_ERR_UNSUPPORTED above). out [batch, Hq, 128] in the KV
 * dtype; lse (nullable) [batch, Hq] fp32 natural-log sum of exp(scale q.k).
 * An empty selection gives out = 0 and lse = -inf. */
msa_status msa_sparse_attn_decode(const void* q, int32_t num_q_heads, const msa_kv_desc* kv /* host */,
                                  const int32_t* idx, int32_t k_total, float scale, void* out,
                                  float* lse, void* ws, size_t ws_bytes, msa_stream_t stream);

/* Step 2, chunked prefill (guide §1, Step 2, and §3: during prefill the
 * savings fall on the main attention). Batch 1, bf16, contiguous or paged
 * cache (q_start + n_q_tokens within its capacity, any q_start); query token r
 * sits at absolute position p = q_start + r and attends to the tokens t <= p
 * of the blocks idx[p / 64 - q_start / 64, h, :] (its tile's list, idx from
 * msa_select_topk_blocks with q_tile 64).
 * At most 512 entries of a list may be valid blocks (-1 padding is free); a
 * longer list is cut there and the device status records MSA_ERR_UNSUPPORTED.
 * out [n_q_tokens, Hq, 128] KV dtype; lse (nullable) [n_q_tokens, Hq] fp32. */
msa_status msa_sparse_attn_prefill(const void* q, int32_t num_q_heads, int32_t n_q_tokens, int64_t q_start,
                                   const msa_kv_desc* kv /* host */, const int32_t* idx, int32_t k_total,
                                   float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                                   msa_stream_t stream);

/* Step 2 for a batch of chunks: msa_sparse_attn_prefill for every sequence s
 * of the cache (n_seqs == kv->batch, at most 64) at once, in one launch. The
 * sequences, q, out and lse are laid out as for msa_select_topk_blocks_varlen:
 * tokens back to back (out [sum q_counts, Hq, 128], lse [sum q_counts, Hq]),
 * idx [total tiles, Hkv, k_total] with global tile numbers; token r of
 * sequence s sits at absolute position q_starts[s] + r and attends to the
 * tokens t <= that position of sequence s's listed blocks. Results equal those
 * of msa_sparse_attn_prefill on each sequence alone. */
msa_status msa_sparse_attn_prefill_varlen(const void* q, int32_t num_q_heads, int32_t n_seqs,
                                          const int64_t* q_starts /* host */, const int32_t* q_counts /* host */,
                                          const msa_kv_desc* kv /* host */, const int32_t* idx, int32_t k_total,
                                          float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                                          msa_stream_t stream);

/* One whole decode step (guide §1, Step 1 then Step 2): the index lists of
 * msa_select_topk_blocks (decode, cfg->q_tile == 1) written to idx_out, and
 * the attention of msa_sparse_attn_decode over them written to out / lse,
 * with the same results. For a bf16 cache with k_scored <= 64 it runs as one
 * kernel (for a paged cache, when the step's grid fits one wave of the
 * device): one thread-block cluster per (sequence, KV head) scores the
 * summaries, selects and attends, exchanging the lists and the partial
 * results through distributed shared memory (nothing round-trips through the
 * workspace); otherwise it launches the two kernels in turn. In token-max mode
 * (cfg->mode, pooled = the index-key cache, Hkv <= 8) the token scores are
 * written to the workspace by their own kernel first and the cluster kernel
 * selects and attends on them. ws must hold
 * msa_workspace_size(MSA_OP_DECODE_STEP, ...) bytes. */
msa_status msa_sparse_decode_step(const void* q, int32_t num_q_heads, const void* pooled,
                                  const msa_kv_desc* kv /* host */, const msa_select_cfg* cfg /* host */,
                                  int32_t* idx_out, int32_t k_total, float scale, void* out, float* lse, void* ws,
                                  size_t ws_bytes, msa_stream_t stream);

/* The decode step of a generation loop (guide, introduction: decode writes the
 * output token by token, each new token checked against everything before
 * it; the summaries of Step 1 must keep up as blocks fill). Same as
 * msa_sparse_decode_step
 * (cfg->mode must be MSA_SCORE_MEAN_POOLED_KEYS), and `pooled` is also
 * written: for every (sequence, KV head) whose seq_len is a multiple of 64 --
 * its newest block has just filled with the current token -- the summary of
 * that block is written exactly as msa_pool_block_keys would, so the next step
 * (one token longer) can score it. In the fused kernel an otherwise idle warp
 * of the unit's first CTA does this while the attention runs; otherwise one
 * small pooling launch follows the step. No other summary is touched. */
msa_status msa_sparse_decode_step_pool(const void* q, int32_t num_q_heads, void* pooled,
                                       const msa_kv_desc* kv /* host */, const msa_select_cfg* cfg /* host */,
                                       int32_t* idx_out, int32_t k_total, float scale, void* out, float* lse,
                                       void* ws, size_t ws_bytes, msa_stream_t stream);

/* Dense causal GQA decode: the full-attention comparator (guide §3 quotes
 * the sparse speed-ups against full attention). Same as msa_sparse_attn_decode
 * with every block 0..ceil(seq_len/64)-1 selected. */
msa_status msa_dense_gqa_decode(const void* q, int32_t num_q_heads, const msa_kv_desc* kv /* host */,
                                float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                                msa_stream_t stream);

/* Dense causal GQA prefill: msa_sparse_attn_prefill with every block up to the
 * diagonal selected for every tile. */
msa_status msa_dense_gqa_prefill(const void* q, int32_t num_q_heads, int32_t n_q_tokens, int64_t q_start,
                                 const msa_kv_desc* kv /* host */, float scale, void* out, float* lse,
                                 void* ws, size_t ws_bytes, msa_stream_t stream);

/* msa_sparse_attn_decode without a workspace argument, for callers that
 * cannot allocate device memory (an engine or plugin host that owns every
 * allocation, or a serving loop that must not call cudaMalloc/cudaFree once
 * running, since those can synchronise the device). The guide has no
 * counterpart to this call; it only changes where the split-K scratch lives.
 * Same arguments, layouts and results as msa_sparse_attn_decode, minus ws.
 *  - Scratch: a fixed 4 MiB device array inside this library, held by every
 *    GPU that loads it until the process exits. bf16 caches combine their
 *    splits inside a thread-block cluster and use none of it beyond a 256-byte
 *    header. fp32 caches keep split-K tickets and partial results there: an
 *    fp32 shape whose msa_workspace_size(MSA_OP_DECODE, ...) exceeds 4 MiB is
 *    rejected with MSA_ERR_WORKSPACE before any work is queued.
 *  - The first call on a device looks up the array's device address (a
 *    one-time set-up per device, cached for the life of the process); make
 *    that first call before any stream capture, and do not call this entry
 *    on a device after cudaDeviceReset (the cached address is then stale).
 *  - Every call on a device shares the one array and (fp32) clears its
 *    counters at the start (a memset on `stream`): calls whose work overlaps
 *    on the GPU race; order them on one stream.
 *  - No device memory is allocated or freed. There is no status word:
 *    data-dependent errors (bad page ids, lengths above capacity) are skipped
 *    and a bounded wait that gives up leaves its output incomplete, neither
 *    reported. Use msa_sparse_attn_decode where those must be detected. */
msa_status msa_sparse_attn_decode_noalloc(const void* q, int32_t num_q_heads, const msa_kv_desc* kv /* host */,
                                          const int32_t* idx, int32_t k_total, float scale, void* out, float* lse,
                                          msa_stream_t stream);

/* Failure-detection self test (the guide has no counterpart; it checks the
 * library's own error path): launches one warp that waits, with the same
 * bounded spin every kernel of the library uses, on a barrier that nothing
 * signals. After `limit_cycles` SM cycles (1000 .. 4e9; MSA_ERR_INVALID_ARG
 * outside) the wait gives up, the status word of `ws` gets MSA_ERR_TIMEOUT and
 * the kernel ends normally: no fault, no trap, the context stays usable.
 * ws: at least the 256-byte header (MSA_ERR_WORKSPACE otherwise). */
msa_status msa_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_cycles, msa_stream_t stream);

/* Reads (and clears) the sticky device status word of `ws`: synchronises
 * `stream`, stores an msa_status in *status_out (host). */
msa_status msa_read_device_status(const void* ws, msa_stream_t stream, int32_t* status_out /* host */);

/* Static English text for a status code. */
const char* msa_status_string(int32_t status);

/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t msa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
