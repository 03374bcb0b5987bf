// Host side of the C ABI declared in include/msa.h: argument validation,
// workspace layout, TMA descriptors and kernel launches. No device memory is
// allocated here and no call synchronises, except msa_read_device_status.
#include <algorithm>
#include <mutex>

#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxTopkCandidates = 32768;  // shared-memory key array of the top-k kernel (2M tokens)
constexpr int64_t kTopkCandCap = 8192;         // refinement buffer of the top-k kernel

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  size_t topk_smem = 0;
  int step_clusters[5] = {0, 0, 0, 0, 0};  // co-resident fused-step clusters of 1, 2, 4, 8, 16 CTAs
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

// Per-device setup: SM count and the dynamic shared-memory opt-ins.
msa_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MSA_ERR_CUDA;
    if (set_decode_smem() != cudaSuccess) return MSA_ERR_CUDA;
    if (set_prefill_smem() != cudaSuccess) return MSA_ERR_CUDA;
    if (set_prefill_tc_smem() != cudaSuccess) return MSA_ERR_CUDA;
    if (set_step_smem() != cudaSuccess) return MSA_ERR_CUDA;
    if (set_token_max_smem() != cudaSuccess) return MSA_ERR_CUDA;
    for (int i = 0; i < 5; ++i) d.step_clusters[i] = step_max_clusters(1 << i);
    d.topk_smem = (kMaxTopkCandidates + kTopkCandCap) * sizeof(uint32_t);
    if (set_topk_smem(d.topk_smem) != cudaSuccess) return MSA_ERR_CUDA;
    if (set_qidx_smem() != cudaSuccess) return MSA_ERR_CUDA;
    if (set_select_decode_smem(select_decode_smem(4096)) != cudaSuccess) return MSA_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return MSA_OK;
}

// SM count for workspace sizing (host call without launches).
int num_sms_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D view [rows, 128] of a bf16 K or V buffer; boxes of 64 rows x 64 columns
// (128 bytes) with 128-byte swizzling.
msa_status make_kv_map(CUtensorMap* map, const void* base, int64_t rows, uint32_t box_rows = 64) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MSA_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return MSA_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MSA_OK : MSA_ERR_CUDA;
}

// 3-D view [tokens, heads, 128] of a bf16 query buffer; boxes of 16 tokens x
// 8 heads x 64 columns (128 rows of 128 bytes) with 128-byte swizzling.
msa_status make_q_map(CUtensorMap* map, const void* base, int64_t n_tokens, int hq) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MSA_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return MSA_ERR_INVALID_ARG;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(hq),
                        static_cast<cuuint64_t>(n_tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, static_cast<cuuint64_t>(hq) * kHeadDim * 2};
  cuuint32_t box[3] = {64, 8, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MSA_OK : MSA_ERR_CUDA;
}

// Queries, outputs, keys, values and pooled keys move in 16-byte pieces
// (vector loads and stores, cp.async, TMA), so their base addresses must be
// 16-byte aligned.
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

msa_status validate_kv(const msa_kv_desc* kv) {
  if (kv == nullptr) return MSA_ERR_INVALID_ARG;
  if (kv->layout != MSA_KV_CONTIGUOUS && kv->layout != MSA_KV_PAGED) return MSA_ERR_INVALID_ARG;
  if (kv->dtype != MSA_DTYPE_F32 && kv->dtype != MSA_DTYPE_BF16) return MSA_ERR_INVALID_ARG;
  if (kv->batch <= 0 || kv->num_kv_heads <= 0) return MSA_ERR_INVALID_ARG;
  if (kv->k == nullptr || kv->v == nullptr || kv->seq_lens == nullptr) return MSA_ERR_INVALID_ARG;
  if (!aligned16(kv->k) || !aligned16(kv->v)) return MSA_ERR_INVALID_ARG;
  if (kv->head_dim != kHeadDim || kv->block_size != kBlock) return MSA_ERR_UNSUPPORTED;
  if (kv->layout == MSA_KV_CONTIGUOUS) {
    if (kv->max_tokens <= 0 || kv->max_tokens % kBlock != 0) return MSA_ERR_INVALID_ARG;
  } else {
    if (kv->page_table == nullptr || kv->max_pages_per_seq <= 0 || kv->num_pages <= 0) return MSA_ERR_INVALID_ARG;
  }
  return MSA_OK;
}

int64_t kv_rows(const msa_kv_desc* kv) {
  return kv->layout == MSA_KV_CONTIGUOUS ? static_cast<int64_t>(kv->batch) * kv->num_kv_heads * kv->max_tokens
                                         : static_cast<int64_t>(kv->num_pages) * kv->num_kv_heads * kBlock;
}
int64_t kv_max_blocks(const msa_kv_desc* kv) {
  return kv->layout == MSA_KV_CONTIGUOUS ? kv->max_tokens / kBlock : kv->max_pages_per_seq;
}

KvView view_of(const msa_kv_desc* kv) {
  KvView v;
  v.layout = kv->layout;
  v.hkv = kv->num_kv_heads;
  v.max_tokens = kv->max_tokens;
  v.page_table = kv->page_table;
  v.max_pages = kv->max_pages_per_seq;
  v.num_pages = kv->num_pages;
  v.seq_lens = kv->seq_lens;
  return v;
}

int32_t* ws_status(void* ws) { return ws == nullptr ? nullptr : reinterpret_cast<int32_t*>(ws); }

// ---- workspace layouts (bytes after the header) ----
struct SelectLayout {
  size_t scores = 0, qidx = 0, cand = 0, total = 0;
};
// prefill: `tiles` query tiles (decode: ignored).
SelectLayout select_layout(const msa_kv_desc* kv, int64_t tiles, int prefill) {
  SelectLayout L;
  const int64_t units = prefill ? tiles * kv->num_kv_heads : static_cast<int64_t>(kv->batch) * kv->num_kv_heads;
  L.scores = kWsRegion;
  size_t off = kWsRegion + align_up(static_cast<size_t>(units) * kv_max_blocks(kv) * sizeof(float), 256);
  L.qidx = off;
  if (prefill) off += align_up(static_cast<size_t>(units) * kHeadDim * sizeof(float), 256);
  L.cand = off;
  if (!prefill) {
    int chunk = 0, n_chunks = 0;
    select_decode_shape(kv_max_blocks(kv), units, num_sms_current(), &chunk, &n_chunks);
    off += align_up(select_decode_cand_bytes(units, n_chunks), 256);
  }
  L.total = off;
  return L;
}

// Offsets below are from the start of the workspace.
struct DecodeLayout {
  int n_splits = 1, bps = 1;
  size_t tickets = 0, partials = 0, total = 0;
};
DecodeLayout decode_layout(const msa_kv_desc* kv, int64_t list_len, int num_sms, bool dense) {
  DecodeLayout L;
  const int64_t units = static_cast<int64_t>(kv->batch) * kv->num_kv_heads;
  decode_splits(units, list_len, num_sms > 0 ? num_sms : 1, kv->dtype == MSA_DTYPE_BF16, dense, &L.n_splits,
                &L.bps);
  L.tickets = kWsHeader;
  L.partials = kWsRegion;
  L.total = L.partials + decode_partials_bytes(units, L.n_splits);
  return L;
}
bool decode_units_fit(const msa_kv_desc* kv) {
  return static_cast<int64_t>(kv->batch) * kv->num_kv_heads <= static_cast<int64_t>(kWsMaxTicketUnits);
}

msa_status check_ws(void* ws, size_t have, size_t need) {
  if (ws == nullptr || have < need) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MSA_ERR_WORKSPACE;
  return MSA_OK;
}

msa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

// Blocks kept without scoring: the newest / diagonal one and the attention sink.
int forced_count(const msa_select_cfg* cfg) {
  return ((cfg->force_local & kForceLocal) ? 1 : 0) + ((cfg->force_local & kForceSink) ? 1 : 0);
}

msa_status check_q_heads(const msa_kv_desc* kv, int hq) {
  if (hq <= 0 || hq % kv->num_kv_heads != 0) return MSA_ERR_INVALID_ARG;
  if (hq / kv->num_kv_heads > 8) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

msa_status decode_common(const void* q, int hq, const msa_kv_desc* kv, const int32_t* idx, int k_total, float scale,
                         void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  msa_status st = validate_kv(kv);
  if (st != MSA_OK) return st;
  if ((st = check_q_heads(kv, hq)) != MSA_OK) return st;
  if (q == nullptr || out == nullptr) return MSA_ERR_INVALID_ARG;
  if (idx != nullptr && k_total <= 0) return MSA_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return MSA_ERR_INVALID_ARG;
  if (!decode_units_fit(kv)) return MSA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MSA_OK) return st;
  const int64_t list_len = idx != nullptr ? k_total : kv_max_blocks(kv);
  DecodeLayout L = decode_layout(kv, list_len, dev->num_sms, idx == nullptr);
  if ((st = check_ws(ws, ws_bytes, L.total)) != MSA_OK) return st;
  DecodeArgs a;
  a.q = q;
  a.hq = hq;
  a.hkv = kv->num_kv_heads;
  a.grp = hq / kv->num_kv_heads;
  a.idx = idx;
  a.k_total = idx != nullptr ? k_total : 0;
  a.n_splits = L.n_splits;
  a.bps = L.bps;
  a.scale_log2 = scale * kLog2e;
  a.out = out;
  a.lse = lse;
  a.tickets = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.tickets);
  a.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.partials);
  a.status = ws_status(ws);
  KvView view = view_of(kv);
  if (kv->dtype == MSA_DTYPE_BF16) {
    const int64_t rows = kv_rows(kv);
    if (rows >= (int64_t(1) << 31)) return MSA_ERR_UNSUPPORTED;
    CUtensorMap tmk, tmv;
    if ((st = make_kv_map(&tmk, kv->k, rows)) != MSA_OK) return st;
    if ((st = make_kv_map(&tmv, kv->v, rows)) != MSA_OK) return st;
    return cuda_status(launch_decode_bf16(tmk, tmv, view, kv->batch, a, stream));
  }
  return cuda_status(launch_decode_f32(static_cast<const float*>(kv->k), static_cast<const float*>(kv->v), view,
                                       kv->batch, a, stream));
}

// Host checks of a chunk batch against the cache: sequence s's new tokens
// [q_starts[s], q_starts[s] + q_counts[s]) fit in its capacity. Fills *pb;
// *n_tokens gets the rows of q and out.
msa_status build_batch(const msa_kv_desc* kv, int n_seqs, const int64_t* q_starts, const int32_t* q_counts,
                       PrefillBatch* pb, int64_t* n_tokens) {
  if (n_seqs != kv->batch || q_starts == nullptr || q_counts == nullptr) return MSA_ERR_INVALID_ARG;
  if (n_seqs > kMaxPrefillSeqs) return MSA_ERR_UNSUPPORTED;
  int64_t total = 0, tiles = 0;
  const int64_t cap = kv_max_blocks(kv) * kBlock;
  for (int s = 0; s < n_seqs; ++s) {
    if (q_counts[s] < 0 || q_starts[s] < 0) return MSA_ERR_INVALID_ARG;
    if (q_starts[s] + q_counts[s] > cap) return MSA_ERR_INVALID_ARG;
    total += q_counts[s];
    tiles += chunk_tiles(q_starts[s], q_counts[s]);
  }
  if (total >= (int64_t(1) << 31) || tiles > 65535) return MSA_ERR_UNSUPPORTED;
  if (!make_prefill_batch(n_seqs, q_starts, q_counts, pb)) return MSA_ERR_INVALID_ARG;
  *n_tokens = total;
  return MSA_OK;
}

msa_status prefill_common(const void* q, int hq, const PrefillBatch& pb, int64_t n_tokens, const msa_kv_desc* kv,
                          const int32_t* idx, int k_total, float scale, void* out, float* lse, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
  msa_status st = MSA_OK;
  if ((st = check_q_heads(kv, hq)) != MSA_OK) return st;
  if (q == nullptr || out == nullptr) return MSA_ERR_INVALID_ARG;
  if (idx != nullptr && k_total <= 0) return MSA_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return MSA_ERR_INVALID_ARG;
  if (kv->dtype != MSA_DTYPE_BF16) return MSA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out)) return MSA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MSA_OK) return st;
  if ((st = check_ws(ws, ws_bytes, kWsHeader)) != MSA_OK) return st;
  if (pb.total_tiles() == 0) return MSA_OK;  // no new tokens
  PrefillArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.hq = hq;
  a.hkv = kv->num_kv_heads;
  a.grp = hq / kv->num_kv_heads;
  a.batch = pb;
  a.idx = idx;
  a.k_total = idx != nullptr ? k_total : 0;
  a.scale_log2 = scale * kLog2e;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = ws_status(ws);
  const int64_t rows = kv_rows(kv);
  if (rows >= (int64_t(1) << 31)) return MSA_ERR_UNSUPPORTED;
  CUtensorMap tmk, tmv;
  if ((st = make_kv_map(&tmk, kv->k, rows)) != MSA_OK) return st;
  if ((st = make_kv_map(&tmv, kv->v, rows)) != MSA_OK) return st;
  if (a.grp == 8) {
    CUtensorMap tmq;
    if ((st = make_q_map(&tmq, q, n_tokens, hq)) != MSA_OK) return st;
    return cuda_status(launch_prefill_tc(tmq, tmk, tmv, view_of(kv), a, stream));
  }
  return cuda_status(launch_prefill_bf16(tmk, tmv, view_of(kv), a, stream));
}

// One sequence (kv->batch == 1) with n_q_tokens new tokens from q_start.
msa_status prefill_one(const void* q, int hq, int n_q_tokens, int64_t q_start, const msa_kv_desc* kv,
                       const int32_t* idx, int k_total, float scale, void* out, float* lse, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  msa_status st = validate_kv(kv);
  if (st != MSA_OK) return st;
  if (n_q_tokens <= 0) return MSA_ERR_INVALID_ARG;
  if (kv->batch != 1) return MSA_ERR_UNSUPPORTED;
  PrefillBatch pb;
  int64_t n_tokens = 0;
  const int32_t cnt = n_q_tokens;
  if ((st = build_batch(kv, 1, &q_start, &cnt, &pb, &n_tokens)) != MSA_OK) return st;
  return prefill_common(q, hq, pb, n_tokens, kv, idx, k_total, scale, out, lse, ws, ws_bytes, stream);
}

// Selection for decode (pb == nullptr: one query token per sequence) or for
// the 64-token tiles of a chunk batch.
msa_status select_common(const void* q, int32_t num_q_heads, int32_t n_q_tokens, const PrefillBatch* pb,
                         const void* pooled, const msa_kv_desc* kv, const msa_select_cfg* cfg, int32_t* idx_out,
                         int32_t k_total, float* scores_out, void* ws, size_t ws_bytes, msa_stream_t stream) {
  msa_status st = MSA_OK;
  const int prefill = pb != nullptr;
  if (!prefill && n_q_tokens != 1 && n_q_tokens != kv->batch) return MSA_ERR_INVALID_ARG;
  if (prefill && kv->dtype != MSA_DTYPE_BF16 && pb->n_seqs != 1) return MSA_ERR_UNSUPPORTED;
  if (kv_max_blocks(kv) > kMaxTopkCandidates) return MSA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MSA_OK) return st;
  SelectLayout L = select_layout(kv, prefill ? pb->total_tiles() : 0, prefill);
  if ((st = check_ws(ws, ws_bytes, L.total)) != MSA_OK) return st;
  if (prefill && pb->total_tiles() == 0) return MSA_OK;  // no new tokens
  float* scores = scores_out != nullptr ? scores_out : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.scores);
  float* qidx = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.qidx);
  FusedSelect fused;
  fused.scores_out = scores_out;
  fused.cand = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + L.cand);
  fused.tickets = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kWsHeader);
  fused.num_sms = dev->num_sms;
  if (!prefill && !decode_units_fit(kv)) return MSA_ERR_UNSUPPORTED;
  KvView view = view_of(kv);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->mode == MSA_SCORE_TOKEN_MAX) {
    // `pooled` holds the shared index-key head: [batch, max_tokens, 128] or [num_pages, 64, 128]
    if (kv->dtype != MSA_DTYPE_BF16 || kv->num_kv_heads > 8) return MSA_ERR_UNSUPPORTED;
    const int64_t rows = kv->layout == MSA_KV_CONTIGUOUS ? static_cast<int64_t>(kv->batch) * kv->max_tokens
                                                         : static_cast<int64_t>(kv->num_pages) * kBlock;
    if (rows >= (int64_t(1) << 31)) return MSA_ERR_UNSUPPORTED;
    CUtensorMap tmi;
    if ((st = make_kv_map(&tmi, pooled, rows)) != MSA_OK) return st;
    if (prefill)
      return cuda_status(launch_select_token_max_prefill(tmi, static_cast<const __nv_bfloat16*>(q), num_q_heads, *pb,
                                                         view, *cfg, idx_out, k_total, scores, qidx, ws_status(ws),
                                                         s));
    if ((st = cuda_status(launch_token_max_scores(tmi, view, kv->batch, static_cast<const __nv_bfloat16*>(q),
                                                  num_q_heads, cfg->force_local, scores, ws_status(ws), s))) != MSA_OK)
      return st;
    return cuda_status(launch_topk_scores(scores, view, kv->batch, *cfg, idx_out, k_total, ws_status(ws), s));
  }
  if (kv->dtype == MSA_DTYPE_BF16)
    return cuda_status(launch_select<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(q), num_q_heads, pb,
                                                    static_cast<const __nv_bfloat16*>(pooled), view, kv->batch,
                                                    *cfg, idx_out, k_total, scores, qidx, &fused, ws_status(ws), s));
  return cuda_status(launch_select<float>(static_cast<const float*>(q), num_q_heads, pb,
                                          static_cast<const float*>(pooled), view, kv->batch, *cfg, idx_out,
                                          k_total, scores, qidx, &fused, ws_status(ws), s));
}

// Checks shared by both selection entries.
msa_status check_select(const void* q, int32_t num_q_heads, const void* pooled, const msa_kv_desc* kv,
                        const msa_select_cfg* cfg, const int32_t* idx_out, int32_t k_total) {
  msa_status st = validate_kv(kv);
  if (st != MSA_OK) return st;
  if (cfg == nullptr || q == nullptr || pooled == nullptr || idx_out == nullptr) return MSA_ERR_INVALID_ARG;
  if ((st = check_q_heads(kv, num_q_heads)) != MSA_OK) return st;
  if (cfg->mode != MSA_SCORE_MEAN_POOLED_KEYS && cfg->mode != MSA_SCORE_TOKEN_MAX) return MSA_ERR_UNSUPPORTED;
  if (cfg->k_scored < 0 || k_total <= 0) return MSA_ERR_INVALID_ARG;
  if (k_total < std::min<int64_t>(cfg->k_scored, kv_max_blocks(kv)) + forced_count(cfg))
    return MSA_ERR_INVALID_ARG;
  if (cfg->force_local < 0 || cfg->force_local > (kForceLocal | kForceSink)) return MSA_ERR_INVALID_ARG;
  if (cfg->q_tile != 1 && cfg->q_tile != kBlock) return MSA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(pooled)) return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}
// The failure-detection path on the device, exercised on purpose: one warp
// waits, with a bounded spin, on a barrier that nothing will ever signal. The
// wait gives up after `limit` SM cycles and records MSA_ERR_TIMEOUT in the
// status word, as every bounded wait of the library does, and the kernel ends
// normally (no fault, no trap), so the context stays usable.
__global__ void selftest_wait_kernel(int32_t* status, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  mbar_wait_warp_limit(&bar, 0, status, kIdSelfTest, limit);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

int32_t msa_version(void) { return 0x000100; }

const char* msa_status_string(int32_t status) {
  switch (status) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_DEVICE_BOUNDS: return "device: page id, block index or length out of range";
    case MSA_ERR_TIMEOUT: return "device: bounded wait timed out";
    default: return "unknown status";
  }
}

size_t msa_workspace_size(int32_t op, const msa_kv_desc* kv, int32_t num_q_heads, int32_t n_q_tokens,
                          int32_t k_total) {
  if (validate_kv(kv) != MSA_OK) return 0;
  switch (op) {
    case MSA_OP_POOL: return kWsHeader;
    case MSA_OP_SELECT: return select_layout(kv, 0, 0).total;
    // one tile more than n_q_tokens / 64 covers a chunk of n_q_tokens tokens
    // that starts inside a block
    case MSA_OP_SELECT_PREFILL:
      return n_q_tokens > 0 ? select_layout(kv, (n_q_tokens + kBlock - 1) / kBlock + 1, 1).total : 0;
    case MSA_OP_DECODE:
      if (k_total <= 0) return 0;
      return decode_layout(kv, k_total, num_sms_current(), false).total;
    case MSA_OP_DENSE_DECODE: return decode_layout(kv, kv_max_blocks(kv), num_sms_current(), true).total;
    case MSA_OP_PREFILL:
    case MSA_OP_DENSE_PREFILL: return kWsHeader;
    case MSA_OP_DECODE_STEP:
      if (k_total <= 0) return 0;
      return std::max(select_layout(kv, 0, 0).total, decode_layout(kv, k_total, num_sms_current(), false).total);
    default: return 0;
  }
  (void)num_q_heads;
}

msa_status msa_workspace_init(void* ws, size_t bytes, msa_stream_t stream) {
  if (ws == nullptr) return MSA_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

msa_status msa_pool_block_keys(const msa_kv_desc* kv, int64_t first_block, int64_t n_blocks, void* pooled, void* ws,
                               size_t ws_bytes, msa_stream_t stream) {
  msa_status st = validate_kv(kv);
  if (st != MSA_OK) return st;
  if (pooled == nullptr || first_block < 0 || n_blocks < -1 || !aligned16(pooled)) return MSA_ERR_INVALID_ARG;
  if (ws != nullptr && ws_bytes < kWsHeader) return MSA_ERR_WORKSPACE;
  KvView view = view_of(kv);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kv->dtype == MSA_DTYPE_BF16)
    return cuda_status(launch_pool<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(kv->k), view, kv->batch,
                                                  first_block, n_blocks, static_cast<__nv_bfloat16*>(pooled),
                                                  ws_status(ws), s));
  return cuda_status(launch_pool<float>(static_cast<const float*>(kv->k), view, kv->batch, first_block, n_blocks,
                                        static_cast<float*>(pooled), ws_status(ws), s));
}

msa_status msa_select_topk_blocks(const void* q, int32_t num_q_heads, int32_t n_q_tokens, const void* pooled,
                                  const msa_kv_desc* kv, const msa_select_cfg* cfg, int32_t* idx_out,
                                  int32_t k_total, float* scores_out, void* ws, size_t ws_bytes,
                                  msa_stream_t stream) {
  msa_status st = check_select(q, num_q_heads, pooled, kv, cfg, idx_out, k_total);
  if (st != MSA_OK) return st;
  if (cfg->q_tile == 1)
    return select_common(q, num_q_heads, n_q_tokens, nullptr, pooled, kv, cfg, idx_out, k_total, scores_out, ws,
                         ws_bytes, stream);
  if (kv->batch != 1 || n_q_tokens <= 0 || cfg->q_start < 0) return MSA_ERR_INVALID_ARG;
  PrefillBatch pb;
  int64_t n_tokens = 0;
  const int64_t q_start = cfg->q_start;
  if ((st = build_batch(kv, 1, &q_start, &n_q_tokens, &pb, &n_tokens)) != MSA_OK) return st;
  return select_common(q, num_q_heads, n_q_tokens, &pb, pooled, kv, cfg, idx_out, k_total, scores_out, ws, ws_bytes,
                       stream);
}

msa_status msa_select_topk_blocks_varlen(const void* q, int32_t num_q_heads, int32_t n_seqs, const int64_t* q_starts,
                                         const int32_t* q_counts, const void* pooled, const msa_kv_desc* kv,
                                         const msa_select_cfg* cfg, int32_t* idx_out, int32_t k_total,
                                         float* scores_out, void* ws, size_t ws_bytes, msa_stream_t stream) {
  msa_status st = check_select(q, num_q_heads, pooled, kv, cfg, idx_out, k_total);
  if (st != MSA_OK) return st;
  if (cfg->q_tile != kBlock) return MSA_ERR_INVALID_ARG;
  PrefillBatch pb;
  int64_t n_tokens = 0;
  if ((st = build_batch(kv, n_seqs, q_starts, q_counts, &pb, &n_tokens)) != MSA_OK) return st;
  return select_common(q, num_q_heads, static_cast<int32_t>(n_tokens), &pb, pooled, kv, cfg, idx_out, k_total,
                       scores_out, ws, ws_bytes, stream);
}

msa_status msa_sparse_attn_decode(const void* q, int32_t num_q_heads, const msa_kv_desc* kv, const int32_t* idx,
                                  int32_t k_total, float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                                  msa_stream_t stream) {
  if (idx == nullptr) return MSA_ERR_INVALID_ARG;
  return decode_common(q, num_q_heads, kv, idx, k_total, scale, out, lse, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_dense_gqa_decode(const void* q, int32_t num_q_heads, const msa_kv_desc* kv, float scale, void* out,
                                float* lse, void* ws, size_t ws_bytes, msa_stream_t stream) {
  return decode_common(q, num_q_heads, kv, nullptr, 0, scale, out, lse, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_sparse_attn_prefill(const void* q, int32_t num_q_heads, int32_t n_q_tokens, int64_t q_start,
                                   const msa_kv_desc* kv, const int32_t* idx, int32_t k_total, float scale,
                                   void* out, float* lse, void* ws, size_t ws_bytes, msa_stream_t stream) {
  if (idx == nullptr) return MSA_ERR_INVALID_ARG;
  return prefill_one(q, num_q_heads, n_q_tokens, q_start, kv, idx, k_total, scale, out, lse, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_sparse_attn_prefill_varlen(const void* q, int32_t num_q_heads, int32_t n_seqs,
                                          const int64_t* q_starts, const int32_t* q_counts, const msa_kv_desc* kv,
                                          const int32_t* idx, int32_t k_total, float scale, void* out, float* lse,
                                          void* ws, size_t ws_bytes, msa_stream_t stream) {
  if (idx == nullptr) return MSA_ERR_INVALID_ARG;
  msa_status st = validate_kv(kv);
  if (st != MSA_OK) return st;
  PrefillBatch pb;
  int64_t n_tokens = 0;
  if ((st = build_batch(kv, n_seqs, q_starts, q_counts, &pb, &n_tokens)) != MSA_OK) return st;
  return prefill_common(q, num_q_heads, pb, n_tokens, kv, idx, k_total, scale, out, lse, ws, ws_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_dense_gqa_prefill(const void* q, int32_t num_q_heads, int32_t n_q_tokens, int64_t q_start,
                                 const msa_kv_desc* kv, float scale, void* out, float* lse, void* ws,
                                 size_t ws_bytes, msa_stream_t stream) {
  return prefill_one(q, num_q_heads, n_q_tokens, q_start, kv, nullptr, 0, scale, out, lse, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// The decode step; pooled_update (nullable, the same array as pooled) also
// gets the summary of every (sequence, head) whose newest block has just
// filled.
msa_status decode_step_common(const void* q, int32_t num_q_heads, const void* pooled, void* pooled_update,
                              const msa_kv_desc* kv, const msa_select_cfg* cfg, int32_t* idx_out, int32_t k_total,
                              float scale, void* out, float* lse, void* ws, size_t ws_bytes, msa_stream_t stream) {
  msa_status st = validate_kv(kv);
  if (st != MSA_OK) return st;
  if (cfg == nullptr || q == nullptr || pooled == nullptr || idx_out == nullptr || out == nullptr)
    return MSA_ERR_INVALID_ARG;
  if ((st = check_q_heads(kv, num_q_heads)) != MSA_OK) return st;
  if (cfg->q_tile != 1) return MSA_ERR_UNSUPPORTED;
  if (!(scale > 0.f)) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(pooled)) return MSA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MSA_OK) return st;
  int C = 0, chunk = 0, bps = 0;
  const int64_t units = static_cast<int64_t>(kv->batch) * kv->num_kv_heads;
  // A paged cache takes the fused step only when its grid is one wave (a
  // ragged batch of long and short sequences is left to the chunked selection,
  // which sizes its pieces per sequence).
  // Token-max scores (the shared index-key cache comes in place of the
  // summaries) are computed by their own kernel first; the fused step then
  // reads them in place of scoring summary rows.
  const bool token_max = cfg->mode == MSA_SCORE_TOKEN_MAX;
  const bool fused = kv->dtype == MSA_DTYPE_BF16 &&
                     (cfg->mode == MSA_SCORE_MEAN_POOLED_KEYS ||
                      (token_max && pooled_update == nullptr && kv->num_kv_heads <= 8)) &&
                     cfg->k_scored >= 0 &&
                     k_total >= std::min<int64_t>(cfg->k_scored, kv_max_blocks(kv)) + forced_count(cfg) &&
                     step_shape(units, kv_max_blocks(kv), cfg->k_scored, k_total, dev->num_sms, dev->step_clusters, &C,
                                &chunk, &bps) &&
                     (kv->layout == MSA_KV_CONTIGUOUS || units * C <= 2LL * dev->num_sms);
  if (!fused) {
    // the same step as two launches (plus the pooling of just-filled blocks)
    st = msa_select_topk_blocks(q, num_q_heads, 1, pooled, kv, cfg, idx_out, k_total, nullptr, ws, ws_bytes, stream);
    if (st != MSA_OK) return st;
    st = msa_sparse_attn_decode(q, num_q_heads, kv, idx_out, k_total, scale, out, lse, ws, ws_bytes, stream);
    if (st != MSA_OK || pooled_update == nullptr) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (kv->dtype == MSA_DTYPE_BF16)
      return cuda_status(launch_pool_newest(static_cast<const __nv_bfloat16*>(kv->k), view_of(kv), kv->batch,
                                            static_cast<__nv_bfloat16*>(pooled_update), ws_status(ws), s));
    return cuda_status(launch_pool_newest(static_cast<const float*>(kv->k), view_of(kv), kv->batch,
                                          static_cast<float*>(pooled_update), ws_status(ws), s));
  }
  const int64_t rows = kv_rows(kv);
  if (rows >= (int64_t(1) << 31)) return MSA_ERR_UNSUPPORTED;
  CUtensorMap tmk, tmv, tmp;
  if ((st = make_kv_map(&tmk, kv->k, rows)) != MSA_OK) return st;
  if ((st = make_kv_map(&tmv, kv->v, rows)) != MSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float* pre_scores = nullptr;
  if (token_max) {
    // index-key rows: [batch * max_tokens, 128] or [num_pages * 64, 128]
    const SelectLayout SL = select_layout(kv, 0, 0);
    if ((st = check_ws(ws, ws_bytes, SL.total)) != MSA_OK) return st;
    const int64_t idx_rows = kv->layout == MSA_KV_CONTIGUOUS ? static_cast<int64_t>(kv->batch) * kv->max_tokens
                                                             : static_cast<int64_t>(kv->num_pages) * kBlock;
    if (idx_rows >= (int64_t(1) << 31)) return MSA_ERR_UNSUPPORTED;
    if ((st = make_kv_map(&tmp, pooled, idx_rows)) != MSA_OK) return st;
    float* scores = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + SL.scores);
    if ((st = cuda_status(launch_token_max_scores(tmp, view_of(kv), kv->batch, static_cast<const __nv_bfloat16*>(q),
                                                  num_q_heads, cfg->force_local, scores, ws_status(ws), s))) != MSA_OK)
      return st;
    pre_scores = scores;
  } else {
    if ((st = check_ws(ws, ws_bytes, kWsHeader)) != MSA_OK) return st;
    // summary rows: [batch * hkv * max_blocks, 128], 128-row boxes
    if ((st = make_kv_map(&tmp, pooled, units * kv_max_blocks(kv), 128)) != MSA_OK) return st;
  }
  return cuda_status(launch_decode_step(tmk, tmv, tmp, view_of(kv), kv->batch, static_cast<const __nv_bfloat16*>(q),
                                        num_q_heads, *cfg, k_total, C, chunk, bps, scale * kLog2e, idx_out,
                                        static_cast<__nv_bfloat16*>(out), lse, ws_status(ws),
                                        static_cast<const __nv_bfloat16*>(kv->k),
                                        static_cast<__nv_bfloat16*>(pooled_update), pre_scores, s));
}

}  // namespace

msa_status msa_sparse_decode_step(const void* q, int32_t num_q_heads, const void* pooled, const msa_kv_desc* kv,
                                  const msa_select_cfg* cfg, int32_t* idx_out, int32_t k_total, float scale,
                                  void* out, float* lse, void* ws, size_t ws_bytes, msa_stream_t stream) {
  return decode_step_common(q, num_q_heads, pooled, nullptr, kv, cfg, idx_out, k_total, scale, out, lse, ws, ws_bytes,
                            stream);
}

msa_status msa_sparse_decode_step_pool(const void* q, int32_t num_q_heads, void* pooled, const msa_kv_desc* kv,
                                       const msa_select_cfg* cfg, int32_t* idx_out, int32_t k_total, float scale,
                                       void* out, float* lse, void* ws, size_t ws_bytes, msa_stream_t stream) {
  if (cfg != nullptr && cfg->mode != MSA_SCORE_MEAN_POOLED_KEYS) return MSA_ERR_UNSUPPORTED;
  return decode_step_common(q, num_q_heads, pooled, pooled, kv, cfg, idx_out, k_total, scale, out, lse, ws, ws_bytes,
                            stream);
}

msa_status msa_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_cycles, msa_stream_t stream) {
  if (ws == nullptr || ws_bytes < kWsHeader) return MSA_ERR_WORKSPACE;
  if (limit_cycles < 1000 || limit_cycles > kWaitCycles) return MSA_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ws_status(ws), limit_cycles);
  return cuda_status(cudaGetLastError());
}

msa_status msa_read_device_status(const void* ws, msa_stream_t stream, int32_t* status_out) {
  if (ws == nullptr || status_out == nullptr) return MSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t word[2] = {0, 0};
  if (cudaMemcpyAsync(word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MSA_ERR_CUDA;
  *status_out = word[0];
  if (word[0] != 0) {
    if (cudaMemsetAsync(const_cast<void*>(ws), 0, sizeof(word), s) != cudaSuccess) return MSA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Sparse decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory: an inference engine or plugin
// host that owns every device allocation and hands its kernels no scratch,
// or a serving loop that must not allocate once it is running, because
// cudaMalloc/cudaFree can synchronise the device and stall every stream.
// msa_sparse_attn_decode_noalloc serves them: its split-K scratch (tickets
// and partial results) lives in the fixed array below, which every GPU that
// loads this library keeps until the process exits.
// ---------------------------------------------------------------------------
namespace msa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocDevice g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current: look up the device address of
// the scratch array (its host-side name is only a stand-in, not an address a
// kernel may use).
msa_status noalloc_scratch(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MSA_ERR_CUDA;
    d.scratch = static_cast<uint8_t*>(p);
    d.ready = true;
  }
  *out = d.scratch;
  return MSA_OK;
}

}  // namespace
}  // namespace msa

extern "C" msa_status msa_sparse_attn_decode_noalloc(const void* q, int32_t num_q_heads, const msa_kv_desc* kv,
                                                     const int32_t* idx, int32_t k_total, float scale, void* out,
                                                     float* lse, msa_stream_t stream) {
  using namespace msa;
  msa_status st = validate_kv(kv);
  if (st != MSA_OK) return st;
  if ((st = check_q_heads(kv, num_q_heads)) != MSA_OK) return st;
  if (q == nullptr || out == nullptr || idx == nullptr || k_total <= 0) return MSA_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return MSA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MSA_OK) return st;
  uint8_t* ws = nullptr;
  if ((st = noalloc_scratch(&ws)) != MSA_OK) return st;
  if (!decode_units_fit(kv)) return MSA_ERR_UNSUPPORTED;
  const DecodeLayout L = decode_layout(kv, k_total, dev->num_sms, false);
  // bf16 combines its splits inside a thread-block cluster and needs no
  // scratch beyond the header; fp32 uses the tickets and the partial results
  const bool f32 = kv->dtype != MSA_DTYPE_BF16;
  const size_t need = f32 ? L.total : kWsHeader;
  if (need > kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;  // beyond the fixed scratch
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (f32) {
    // the array keeps the previous call's contents: the tickets must start at zero
    const size_t units = static_cast<size_t>(kv->batch) * kv->num_kv_heads;
    if (cudaMemsetAsync(ws + L.tickets, 0, units * sizeof(int32_t), s) != cudaSuccess) return MSA_ERR_CUDA;
  }
  DecodeArgs a;
  a.q = q;
  a.hq = num_q_heads;
  a.hkv = kv->num_kv_heads;
  a.grp = num_q_heads / kv->num_kv_heads;
  a.idx = idx;
  a.k_total = k_total;
  a.n_splits = L.n_splits;
  a.bps = L.bps;
  a.scale_log2 = scale * kLog2e;
  a.out = out;
  a.lse = lse;
  a.tickets = reinterpret_cast<int32_t*>(ws + L.tickets);
  a.partials = reinterpret_cast<float*>(ws + L.partials);
  a.status = nullptr;  // bad page ids / lengths are skipped without a report
  const KvView view = view_of(kv);
  if (kv->dtype == MSA_DTYPE_BF16) {
    const int64_t rows = kv_rows(kv);
    if (rows >= (int64_t(1) << 31)) return MSA_ERR_UNSUPPORTED;
    CUtensorMap tmk, tmv;
    if ((st = make_kv_map(&tmk, kv->k, rows)) != MSA_OK) return st;
    if ((st = make_kv_map(&tmv, kv->v, rows)) != MSA_OK) return st;
    return cuda_status(launch_decode_bf16(tmk, tmv, view, kv->batch, a, s));
  }
  return cuda_status(launch_decode_f32(static_cast<const float*>(kv->k), static_cast<const float*>(kv->v), view,
                                       kv->batch, a, s));
}
