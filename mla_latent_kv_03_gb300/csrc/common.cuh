// Internal helpers shared by the libmla kernels: constants, the workspace
// layout, device status bits, and thin inline-PTX wrappers (mbarrier, TMA,
// ldmatrix, warp mma). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "../../include/mla.h"

namespace mla {

constexpr int kDc = 512;          // kv_lora_rank
constexpr int kDr = 64;           // qk_rope_head_dim
constexpr int kDn = 128;          // qk_nope_head_dim
constexpr int kDv = 128;          // v_head_dim
constexpr int kRow = kDc + kDr;   // 576 values per cache row
constexpr int kRow8 = kDc + 2 * kDr;  // 640 bytes per FP8 cache row: 512 e4m3 codes, 64 bf16
constexpr int kTile = 64;         // kv tokens per work unit
constexpr int kHG = 16;           // heads per query tile (one m16 row block)
constexpr uint32_t kMagic = 0x4d4c4131u;  // "MLA1"

// Default bound for every spin-wait on an mbarrier (ns of %globaltimer).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// ---------------------------------------------------------------------------
// Workspace layout (device memory owned by the caller).
//   [0, 256)            WsHeader
//   counters[512]       int, CTAs done with each q-tile of the fused merge when
//                       num_q * G <= 512 (a fixed region: no layout puts
//                       anything else there, mla_workspace_init zeroes it, and
//                       the CTA that merges a q-tile resets its counter to 0)
//   row_info[num_q]     int4 {seq b, query position, tiles, first unit}
//   cta_start[C]        int4 {row n, head group g, tile k, 0}
//   lse[S][16]          float, base-2 log-sum-exp of each partial
//   opart[S][16][512]   float, normalised partial outputs
//   arrive[num_q * G]   int, the fused merge's counters when num_q * G > 512
//                       (zeroed by the plan)
// with S = C + num_q * G - 1 partial slots; slot of (CTA c, q-tile t) = c + t
// (unique because CTA shares and q-tiles are both contiguous ranges of the
// same ordered unit list).
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t status;      // MLA_DEV_* bits
  uint32_t magic;
  int32_t total_units;  // sum over rows of G * tiles(row)
  int32_t share;        // units per CTA
  int32_t num_ctas;
  int32_t groups;       // G = H / 16
  int32_t num_q;
  int32_t batch;
  int32_t mode;         // 0: units per (row, 16-head group); 1: per 128-row q-block
  int32_t qblocks;      // mode 1: number of q-blocks
  uint32_t pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct WsLayout {
  size_t row_info, cta_start, lse, opart, arrive, total;
  int64_t slots;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Query rows up to which the bf16 warp-mma decode plans its own split.
constexpr int kSelfMaxRows = 256;

// Fused-merge counters kept at a fixed place right after the header.
constexpr int kFixedCounters = 512;
constexpr size_t kFixedCountersOff = 256;
constexpr size_t kLayoutStart = kFixedCountersOff + kFixedCounters * 4;  // 2,304

__host__ __device__ inline WsLayout ws_layout(int64_t num_q, int groups, int num_ctas) {
  WsLayout L;
  L.slots = (int64_t)num_ctas + num_q * groups;  // one spare slot
  size_t off = kLayoutStart;
  L.row_info = off;   off = align_up(off + (size_t)num_q * 16, 256);
  L.cta_start = off;  off = align_up(off + (size_t)num_ctas * 16, 256);
  L.lse = off;        off = align_up(off + (size_t)L.slots * kHG * 4, 256);
  L.opart = off;      off = align_up(off + (size_t)L.slots * kHG * kDc * 4, 256);
  if (num_q * groups <= kFixedCounters) {
    L.arrive = kFixedCountersOff;
  } else {
    L.arrive = off;   off = align_up(off + (size_t)num_q * groups * 4, 256);
  }
  L.total = off;
  return L;
}

// Mode-1 workspace (the tensor-core kernel for many heads or prefill rows).
// A q-block is 8 consecutive q-tiles (128 consecutive (row, head) rows of
// q_abs) of one sequence; work units are (q-block, 64-token tile); each share
// of units is processed by two CTAs, one per 256-column half of the output.
//   [0, 256)              WsHeader (mode = 1)
//   row_info[num_q]       int4 {seq b, query position, tiles, 0}
//   seq_info[batch]       int4 {first q-tile, first q-block, end q-tile, 0}
//   qblock[QB]            int4 {seq b, first q-tile, tiles, first unit}
//   cta_start[shares]     int4 {q-block, tile, 0, 0}
//   lse[S][128]           float (base 2)
//   opart[S][128][512]    float
//   arrive[QB][2]         int (fused merge, per output half)
// with QB = ceil(num_q * G / 8) + batch and S = shares + QB; the slot of
// (share c, q-block qb) is c + qb. Rows [16 sub, 16 sub + 16) of a slot are
// q-tile (first q-tile + sub), so in units of 16-row groups the q-tile's
// partials sit at (c + qb) * 8 + sub, stride 8 between shares.
constexpr int kQBlockTiles = 8;
constexpr int kQBlockRows = kQBlockTiles * kHG;  // 128

struct WsLayoutTc {
  size_t row_info, seq_info, qblock, cta_start, lse, opart, arrive, total;
  int64_t qblocks_max, slots;
};

__host__ __device__ inline WsLayoutTc ws_layout_tc(int64_t num_q, int groups, int shares,
                                                   int batch) {
  WsLayoutTc L;
  L.qblocks_max = (num_q * groups + kQBlockTiles - 1) / kQBlockTiles + batch;
  L.slots = (int64_t)shares + L.qblocks_max;
  size_t off = kLayoutStart;  // the fixed counters belong to the 16-row layout
  L.row_info = off;  off = align_up(off + (size_t)num_q * 16, 256);
  L.seq_info = off;  off = align_up(off + (size_t)batch * 16, 256);
  L.qblock = off;    off = align_up(off + (size_t)L.qblocks_max * 16, 256);
  L.cta_start = off; off = align_up(off + (size_t)shares * 16, 256);
  L.lse = off;       off = align_up(off + (size_t)L.slots * kQBlockRows * 4, 256);
  L.opart = off;     off = align_up(off + (size_t)L.slots * kQBlockRows * kDc * 4, 256);
  L.arrive = off;    off = align_up(off + (size_t)L.qblocks_max * 2 * 4, 256);
  L.total = off;
  return L;
}

// Where the split partials of q-tile t (query row n, head group g) live, in
// units of 16-row x 512 groups of the partial buffer: `count` groups starting
// at `first`, `stride` apart. count = 0: the q-tile saw no token.
struct QtileParts {
  int64_t first;
  int stride, count;
};

__device__ __forceinline__ QtileParts locate_qtile(const uint8_t* ws, int64_t num_q, int groups,
                                                   int num_ctas, int batch, int n, int g) {
  const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
  QtileParts r{0, 1, 0};
  if (hdr->magic != kMagic || hdr->num_q != num_q || hdr->groups != groups ||
      hdr->num_ctas != num_ctas)
    return r;
  const int share = hdr->share;
  const int t = n * groups + g;
  if (hdr->mode == 0) {
    const WsLayout L = ws_layout(num_q, groups, num_ctas);
    const int4 ri = reinterpret_cast<const int4*>(ws + L.row_info)[n];
    if (ri.z <= 0) return r;
    const int U = ri.w + g * ri.z;
    const int cf = U / share, cl = (U + ri.z - 1) / share;
    r.first = (int64_t)cf + t;
    r.count = cl - cf + 1;
    return r;
  }
  const WsLayoutTc L = ws_layout_tc(num_q, groups, num_ctas / 2, batch);
  const int4 ri = reinterpret_cast<const int4*>(ws + L.row_info)[n];
  if (ri.z <= 0 || ri.x < 0 || ri.x >= batch) return r;
  const int4 si = reinterpret_cast<const int4*>(ws + L.seq_info)[ri.x];
  const int li = t - si.x;
  const int qb = si.y + li / kQBlockTiles, sub = li % kQBlockTiles;
  if (li < 0 || qb < 0 || qb >= hdr->qblocks) return r;
  const int4 bi = reinterpret_cast<const int4*>(ws + L.qblock)[qb];
  const int cf = bi.w / share, cl = (bi.w + bi.z - 1) / share;
  r.first = ((int64_t)cf + qb) * kQBlockTiles + sub;
  r.stride = kQBlockTiles;
  r.count = cl - cf + 1;
  return r;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Counting a finished split part on its q-tile's arrival counter (the fused
// split merges). Protocol, in PTX memory-model terms:
//   1. every thread that stored part of the partial (or its log-sum-exp)
//      issues fence.acq_rel.gpu (__threadfence) after its stores;
//   2. a CTA barrier orders those fences before the counting thread's atomic;
//   3. the counting thread adds with atom.acq_rel.gpu: its release half
//      publishes the CTA's stores, its acquire half -- on the CTA that counts
//      last -- makes every other part's release visible to it;
//   4. a second CTA barrier hands that to the merging threads, which read the
//      parts through L2 (ld.global.cg), never through the non-coherent path.
// The counter is reset to zero by the merging CTA after its merge; the next
// launch's atomics come after this grid has completed.
__device__ __forceinline__ int count_arrival(int* counter) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
               : "=r"(old)
               : "l"(counter)
               : "memory");
  return old;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false if it did not
// complete within timeout_ns (the caller then flags MLA_DEV_TIMEOUT and
// leaves its loop). Never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0 && globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
// x (innermost coordinate, elements) must be a multiple of 8 for 16-bit data.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read once per step (the latent cache stream): its lines
// are evicted first, so the weights and the small per-step tensors stay in L2
// from one step to the next.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled TMA load, completion counted on `bar` in bytes. x (innermost)
// must be a multiple of 8 for 16-bit data.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 4-D tiled TMA load, completion counted on `bar` in bytes. x (innermost)
// must be a multiple of 8 for 16-bit data.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// tma_load_3d with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x through the PTX approximate base-2 exponential (documented max relative
// error about 2^-22); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled
// tile whose rows are 128 bytes (the TMA SWIZZLE_128B pattern: chunk index
// XOR row mod 8; the tile base must be 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Load / store helpers for the two storage dtypes.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// RoPE inverse frequencies inv_freq_i = base^(-2i/64), i < 32, computed on
// the host in double and passed as an unevaluated float sum hi + lo.
struct RopeFreq {
  float hi[32];
  float lo[32];
};

inline RopeFreq make_rope_freq(double base) {
  RopeFreq f;
  for (int i = 0; i < 32; ++i) {
    const double v = std::pow(base, -2.0 * i / 64.0);
    f.hi[i] = (float)v;
    f.lo[i] = (float)(v - (double)f.hi[i]);
  }
  return f;
}

// cos and sin of pos * inv_freq without fp64 arithmetic (GB300's fp64 rate is
// a small fraction of fp32). The product is formed exactly as a + e + tail
// (FMA two-product, Dekker/Kahan), then reduced modulo 2*pi by Cody-Waite
// additive reduction with 2*pi split into two floats, so |r| <= pi with an
// absolute error of a few 1e-7 even at positions near 2^15; sincosf finishes.
__device__ __forceinline__ void rope_cos_sin(int pos, float hi, float lo, float* c, float* s) {
  const float p = (float)pos;                  // exact for |pos| < 2^24
  const float a = p * hi;
  const float e = fmaf(p, hi, -a);             // rounding error of p * hi, exactly
  const float tail = fmaf(p, lo, e);
  const float k = rintf(a * 0.159154943091895336f);          // a / (2 pi)
  float r = fmaf(-k, 6.28318548202514648f, a);               // 2 pi, leading float
  r = fmaf(-k, -1.74845553146951715e-07f, r);                // 2 pi - leading float
  r += tail;
  sincosf(r, s, c);
}

}  // namespace mla
