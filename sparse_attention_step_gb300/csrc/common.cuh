// Shared device helpers: inline-PTX wrappers (mbarrier, TMA bulk tensor copies,
// ldmatrix, mma.sync, movmatrix), bf16 packing and the workspace layout.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/msa.h"

namespace msa {

constexpr int kHeadDim = 128;
constexpr int kBlock = 64;
constexpr int kMaxGroupHeads = 8;  // query heads per KV head (GQA group size) the kernels accept
// msa_select_cfg.force_local bits
constexpr int kForceLocal = 1;  // keep the newest (decode) / diagonal (prefill) block
constexpr int kForceSink = 2;   // keep block 0 (attention sink)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Workspace layout, shared by every op so one zero-filled workspace serves all:
//   [0, 256)                     header (sticky device status)
//   [256, 256 + kWsTicketBytes)  split-K ticket counters, one int32 per decode
//                                unit; zero between calls (the last CTA of a
//                                unit resets its counter) and written by
//                                nothing else
//   [kWsRegion, ...)             op-specific scratch (scores, q_idx, partials)
// ---------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;
constexpr size_t kWsMaxTicketUnits = 16384;
constexpr size_t kWsTicketBytes = kWsMaxTicketUnits * sizeof(int32_t);
constexpr size_t kWsRegion = kWsHeader + kWsTicketBytes;

struct WsHeader {
  int32_t status;  // sticky msa_status set by kernels (0 = ok)
  int32_t where;   // diagnostic: kernel id that set it
  int32_t pad[62];
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Record the first device-side error (a no-op when no workspace is given).
__device__ inline void set_status(int32_t* status, int32_t code, int32_t where) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0, code) == 0) status[1] = where;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses
// ---------------------------------------------------------------------------
__device__ inline uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// `raw` (dynamic shared memory) advanced to the next 1024-byte boundary, the
// alignment 128-byte swizzled tiles need. Offsetting the array itself, not
// rounding an integer, keeps every access through the result a
// shared-memory access (the compiler can no longer tell after an integer
// round trip, and falls back to generic loads and stores).
__device__ inline uint8_t* smem_align1024(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ inline void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ inline void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ inline void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ inline void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ inline void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ inline void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ inline bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after about
// `kWaitCycles` SM cycles (then the device status gets MSA_ERR_TIMEOUT and the
// caller must stop using the buffer the barrier guards).
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
__device__ inline bool mbar_wait_limit(uint64_t* bar, uint32_t parity, int32_t* status, int where,
                                       long long limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit_cycles) {
      set_status(status, MSA_ERR_TIMEOUT, where);
      return false;
    }
  }
}
__device__ inline bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status, int where) {
  return mbar_wait_limit(bar, parity, status, where, kWaitCycles);
}

// The whole warp waits, and leaves converged with the same result in every
// lane. Lanes leave a spin on their own, so without the vote a warp can carry
// on split in two, and every warp-collective instruction after it (shuffles,
// ldmatrix, mma.sync, tcgen05.ld) then runs once per part.
__device__ inline bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int32_t* status, int where) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, where));
}
__device__ inline bool mbar_wait_warp_limit(uint64_t* bar, uint32_t parity, int32_t* status, int where,
                                            long long limit_cycles) {
  return __all_sync(0xffffffffu, mbar_wait_limit(bar, parity, status, where, limit_cycles));
}

// Waits (bounded) until the copies of the last `stages` ring stages issued so
// far (stage i in slot i % stages, i < issued) have landed. A producer calls
// it before its CTA moves on: in a normal run the consumers have already
// waited for them all and it returns at once; after a bounded wait gave up
// somewhere it keeps copies still in flight from landing in shared memory
// that is reused or released.
__device__ inline void mbar_drain(uint64_t* full, int stages, int issued, int32_t* status, int where) {
  for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
    mbar_wait(&full[i % stages], static_cast<uint32_t>((i / stages) & 1), status, where);
}

// ---------------------------------------------------------------------------
// TMA: 2-D tiled bulk tensor copy global -> shared, completing on an mbarrier.
// x is the innermost coordinate (elements), y the row.
// ---------------------------------------------------------------------------
__device__ inline void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Untiled bulk copy global -> shared (both 16-byte aligned, size a multiple of 16).
__device__ inline void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Per-thread asynchronous 16-byte copy global -> shared (L2 only), grouped
// with commit / wait_group; a barrier after the wait publishes the data to
// the other threads.
__device__ inline void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ inline void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ inline void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Pull one 2-D tile into L2 (no shared memory, no completion to wait for).
__device__ inline void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ inline void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core fragments (m16n8k16, bf16 in, fp32 accumulate).
// Lane l: g = l >> 2 (row group), c = l & 3 (column pair).
// ---------------------------------------------------------------------------
__device__ inline void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ inline void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ inline void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ inline uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ inline uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of (row, 16-byte chunk) in a tile written by TMA with 128-byte
// swizzling: rows of 128 bytes, chunk index XOR (row mod 8).
__device__ inline uint32_t swz128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ inline float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Scores as order-preserving unsigned keys: a larger float gives a larger key.
__device__ inline uint32_t float_to_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 ranks with +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel in the stream still runs;
// pdl_wait() blocks until that kernel has completed and its writes are
// visible (call it before touching any global input), and pdl_trigger() lets
// the next kernel start launching early. Both are no-ops without the launch
// attribute.
// ---------------------------------------------------------------------------
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Thread-block clusters: rank, barrier, distributed shared memory loads.
// ---------------------------------------------------------------------------
__device__ inline uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes made
// before the barrier are visible to the cluster's loads after it.
__device__ inline void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Named barrier `id` (1..15) for the first nthreads / 32 warps of the CTA.
__device__ inline void bar_sync_warps(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Arrive at named barrier `id` without waiting (the threads that bar.sync on
// it see this thread's earlier shared-memory writes).
__device__ inline void bar_arrive_warps(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// The two halves of cluster_sync, for work that fits between them.
__device__ inline void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ inline void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Address of the same shared-memory location in the cluster's CTA `rank`.
__device__ inline uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ inline float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ inline uint64_t ld_dsmem_u64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ inline int32_t ld_dsmem_i32(uint32_t addr) {
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ inline void st_dsmem4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ inline float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// KV cache addressing shared by every kernel. Rows are 128-element (D) rows.
// ---------------------------------------------------------------------------
struct KvView {
  int32_t layout;       // MSA_KV_CONTIGUOUS / MSA_KV_PAGED
  int32_t hkv;          // KV heads
  int64_t max_tokens;   // contiguous capacity per sequence
  const int32_t* page_table;
  int32_t max_pages;    // paged: table row length
  int32_t num_pages;
  const int32_t* seq_lens;

  __device__ int64_t capacity() const {
    return layout == MSA_KV_CONTIGUOUS ? max_tokens : static_cast<int64_t>(max_pages) * kBlock;
  }
  // Length of sequence s, clamped to [0, capacity]; an out-of-range length
  // sets MSA_ERR_DEVICE_BOUNDS.
  __device__ int64_t seq_len(int s, int32_t* status, int where) const {
    int64_t n = seq_lens[s];
    int64_t cap = capacity();
    if (n < 0 || n > cap) {
      set_status(status, MSA_ERR_DEVICE_BOUNDS, where);
      n = n < 0 ? 0 : cap;
    }
    return n;
  }
  // Page holding logical block b of sequence s (paged), or -1 (status set).
  __device__ int32_t page(int s, int64_t b, int32_t* status, int where) const {
    int32_t p = page_table[static_cast<int64_t>(s) * max_pages + b];
    if (p < 0 || p >= num_pages) {
      set_status(status, MSA_ERR_DEVICE_BOUNDS, where);
      return -1;
    }
    return p;
  }
  // First K/V row of logical block b of (s, h), or -1 for a bad page.
  __device__ int64_t block_row(int s, int h, int64_t b, int32_t* status, int where) const {
    if (layout == MSA_KV_CONTIGUOUS) return (static_cast<int64_t>(s) * hkv + h) * max_tokens + b * kBlock;
    int32_t p = page(s, b, status, where);
    return p < 0 ? -1 : (static_cast<int64_t>(p) * hkv + h) * kBlock;
  }
  // Row of the pooled summary key of block b of (s, h). Summaries are kept per
  // (sequence, KV head) in logical block order for both cache layouts, so a
  // unit's candidates are one contiguous run of rows.
  __device__ int64_t pooled_row(int s, int h, int64_t b) const {
    return (static_cast<int64_t>(s) * hkv + h) * max_blocks() + b;
  }
  __host__ __device__ int64_t max_blocks() const {
    return layout == MSA_KV_CONTIGUOUS ? max_tokens / kBlock : static_cast<int64_t>(max_pages);
  }
};

// Kernel ids recorded with a device status (WsHeader::where).
enum KernelId { kIdPool = 1, kIdQidx = 2, kIdScore = 3, kIdTopk = 4, kIdDecode = 5, kIdPrefill = 6, kIdSelfTest = 7 };

}  // namespace msa
