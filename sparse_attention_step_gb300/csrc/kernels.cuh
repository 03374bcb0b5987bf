// Argument blocks and host launchers of the kernels, shared by the kernel
// files and the C-ABI layer.
#pragma once

#include "common.cuh"

namespace msa {

// Sequences of a (batched) chunked prefill: sequence s has q_cnt[s] new
// tokens at absolute positions q_start[s] + r, stored in rows q_off[s] + r of
// q and out. Its query tiles are its tokens grouped by the 64-token block they
// sit in: tile j holds the chunk rows r with (q_start[s] + r) / 64 ==
// q_start[s] / 64 + j (its diagonal block), so a chunk that starts inside a
// block has a shorter first tile. They are global tiles tile_off[s] ..
// tile_off[s + 1] - 1, and the prefill scorer takes them in groups of 16
// (global groups grp_off[s] .. grp_off[s + 1] - 1).
constexpr int kMaxPrefillSeqs = 64;
struct PrefillBatch {
  int n_seqs;
  int64_t q_start[kMaxPrefillSeqs];
  int32_t q_off[kMaxPrefillSeqs];
  int32_t q_cnt[kMaxPrefillSeqs];
  int32_t tile_off[kMaxPrefillSeqs + 1];
  int32_t grp_off[kMaxPrefillSeqs + 1];
  __host__ __device__ int seq_of_tile(int tile) const {
    int s = 0;
    while (s + 1 < n_seqs && tile_off[s + 1] <= tile) ++s;
    return s;
  }
  __host__ __device__ int seq_of_group(int g) const {
    int s = 0;
    while (s + 1 < n_seqs && grp_off[s + 1] <= g) ++s;
    return s;
  }
  __host__ __device__ int total_tiles() const { return tile_off[n_seqs]; }
  // Chunk row (within sequence s) of the first position of global tile
  // `tile`'s block: row tile_row0 + i sits at position 64 * diag + i. Negative
  // for the first tile of a chunk that starts inside a block; the tile's rows
  // are [max(0, tile_row0), min(q_cnt[s], tile_row0 + 64)).
  __host__ __device__ int tile_row0(int s, int tile) const {
    return (tile - tile_off[s]) * 64 - static_cast<int>(q_start[s] % 64);
  }
};
// Query tiles of a chunk of n tokens from absolute position q_start.
__host__ __device__ inline int32_t chunk_tiles(int64_t q_start, int32_t n) {
  return n <= 0 ? 0 : static_cast<int32_t>((q_start + n - 1) / 64 - q_start / 64 + 1);
}
// Fills b from host arrays; false when n_seqs is out of [1, kMaxPrefillSeqs]
// or a count is negative.
bool make_prefill_batch(int n_seqs, const int64_t* q_starts, const int32_t* q_counts, PrefillBatch* b);


// ---- Step 1a: pooling (pool.cu) ----
template <typename T>
cudaError_t launch_pool(const T* k, const KvView& kv, int batch, int64_t first_block, int64_t n_blocks, T* pooled,
                        int32_t* status, cudaStream_t stream);
template <typename T>
cudaError_t launch_pool_newest(const T* k, const KvView& kv, int batch, T* pooled, int32_t* status,
                               cudaStream_t stream);

// ---- Step 1b/1c: index query, scores, top-k (select.cu) ----
// Scratch of the fused decode selection (k_scored <= 64).
struct FusedSelect {
  float* scores_out;  // nullable
  uint64_t* cand;     // [units, n_chunks, 64]
  int32_t* tickets;   // [units]
  int num_sms;
};
template <typename T>
cudaError_t launch_select(const T* q, int hq, const PrefillBatch* pb, const T* pooled, const KvView& kv, int batch,
                          const msa_select_cfg& cfg, int32_t* idx_out, int k_total, float* scores, float* qidx_ws,
                          const FusedSelect* fused, int32_t* status, cudaStream_t stream);
void select_decode_shape(int64_t max_blocks, int64_t units, int num_sms, int* chunk, int* n_chunks);
size_t select_decode_smem(int chunk);
size_t select_decode_cand_bytes(int64_t units, int n_chunks);
cudaError_t set_select_decode_smem(size_t bytes);
cudaError_t set_topk_smem(size_t bytes);
cudaError_t set_qidx_smem();

// ---- Step 2, decode (decode.cu) ----
struct DecodeArgs {
  const void* q;
  int hq, hkv, grp;
  const int32_t* idx;   // [batch, hkv, k_total] or nullptr (dense)
  int k_total;
  int n_splits;
  int bps;              // list entries (sparse) or blocks (dense) per split
  float scale_log2;     // scale * log2(e)
  void* out;
  float* lse;
  float* partials;      // [units, n_splits, kPartFloats]
  int32_t* tickets;     // [units], zero between calls
  int32_t* status;
};
cudaError_t set_decode_smem();
size_t decode_smem_bytes();
void decode_splits(int64_t units, int64_t list_len, int num_sms, bool cluster, bool dense, int* n_splits, int* bps);
size_t decode_partials_bytes(int64_t units, int n_splits);
cudaError_t launch_decode_bf16(const CUtensorMap& tmk, const CUtensorMap& tmv, const KvView& kv, int batch,
                               const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_f32(const float* k, const float* v, const KvView& kv, int batch, const DecodeArgs& a,
                              cudaStream_t stream);

// ---- Step 2, prefill (prefill.cu) ----
struct PrefillArgs {
  const __nv_bfloat16* q;  // [total new tokens, hq, 128]
  int hq, hkv, grp;
  PrefillBatch batch;
  const int32_t* idx;  // [total tiles, hkv, k_total] or nullptr (dense)
  int k_total;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
  int num_sms;  // the device's SMs (the tcgen05 kernel's prefetch for the next wave of CTAs)
};
cudaError_t set_prefill_smem();
cudaError_t set_prefill_tc_smem();
// tcgen05 kernel: 8 query heads per KV head only
cudaError_t launch_prefill_tc(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const KvView& kv, const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_bf16(const CUtensorMap& tmk, const CUtensorMap& tmv, const KvView& kv,
                                const PrefillArgs& a, cudaStream_t stream);

// ---- fused decode step (step.cu) ----
bool step_shape(int64_t units, int64_t max_blocks, int k_scored, int k_total, int num_sms, const int* max_clusters,
                int* C, int* chunk, int* bps);
int step_max_clusters(int C);
cudaError_t set_step_smem();

// ---- token-level max-pooled scores (token_max.cu) ----
cudaError_t set_token_max_smem();
cudaError_t launch_token_max_prefill_scores(const CUtensorMap& tmi, const KvView& kv, const PrefillBatch& pb,
                                            const float* qidx, float* scores, int32_t* status, cudaStream_t stream);
cudaError_t launch_select_token_max_prefill(const CUtensorMap& tmi, const __nv_bfloat16* q, int hq,
                                            const PrefillBatch& pb, const KvView& kv, const msa_select_cfg& cfg,
                                            int32_t* idx_out, int k_total, float* scores, float* qidx_ws,
                                            int32_t* status, cudaStream_t stream);
cudaError_t launch_token_max_scores(const CUtensorMap& tmi, const KvView& kv, int batch, const __nv_bfloat16* q,
                                    int hq, int force_local, float* scores, int32_t* status, cudaStream_t stream);
cudaError_t launch_topk_scores(const float* scores, const KvView& kv, int batch, const msa_select_cfg& cfg,
                               int32_t* idx_out, int k_total, int32_t* status, cudaStream_t stream);
cudaError_t launch_decode_step(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmpool,
                               const KvView& kv, int batch, const __nv_bfloat16* q, int hq, const msa_select_cfg& cfg,
                               int k_total, int C, int chunk, int bps, float scale_log2,
                               int32_t* idx_out, __nv_bfloat16* out, float* lse, int32_t* status,
                               const __nv_bfloat16* k, __nv_bfloat16* pooled_out, const float* pre_scores,
                               cudaStream_t stream);

}  // namespace msa
