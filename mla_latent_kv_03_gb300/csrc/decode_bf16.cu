// bf16 split-KV latent attention over the paged cache: the step the decode
// time goes into. Source: "mini-infer-17: MLA Attention", sections "版本 3:
// MLAAttentionAbsorbed" (scores and output taken directly against the latent)
// and "设计取舍" (the nope and rope score parts are summed, then a
// hand-written softmax); "07. MLA / Mamba / MoE in vLLM source" 2.3 (paged
// layout and block-table indirection).
//
// One persistent CTA per SM walks its share of (query row, 16-head group,
// 64-token tile) units. Per CTA:
//   warp 4 (producer): TMA loads of 64-token cache tiles (9 boxes of 64
//     columns x block_size rows, SWIZZLE_128B) into an NST-stage ring guarded
//     by full/empty mbarriers, and of the 16x576 absorbed query (double
//     buffered). It reads the block table itself and never loads a block
//     outside [0, num_blocks).
//   warps 0-3 (math): each scores 16 of the tile's 64 tokens against all 16
//     heads (m16n8k16 warp mma over K = 576, bf16 in, fp32 accumulate), the
//     four warps agree on the running row maximum through shared memory,
//     write their bf16 probabilities in A-fragment order, then each multiplies
//     P (16 x 64) by its 128-column slice of the tile's latent part (ldmatrix
//     .trans). The output accumulator (16 x 512 fp32) lives in registers.
// Every wait is bounded; a timeout sets MLA_DEV_TIMEOUT, all math warps leave
// together, and the producer waits (bounded) for its copies in flight before
// the CTA exits.
//
// Self-planned launches (SELF): every CTA computes the split plan from
// seq_lens / query_start_loc itself (no plan kernel) and the math warps write
// it to the workspace for a later merge kernel. With early streaming the plan
// (seq_lens, query_start_loc) and the producer's first cache tiles (block
// table, cache) are read before the preceding kernel in the stream has
// finished (programmatic dependent launch); only the query copy and every
// global write wait for it.
//
// Fused merge: a (row, head group) cut into parts is merged by the CTA that
// finishes its part last. Parts are published in the math threads' fragment
// order (thread i's 16 float4 at [slot][nt][i]), so each thread of the
// merging CTA reads exactly the values it adds, coalesced, two parts per round
// trip with their log-sum-exps in the same round trip, in CTA order.
//
// FP8 cache (FP8, self-planned only): rows of 512 e4m3 codes (times kv_scale)
// and 64 bf16 rope values. The producer loads the codes as 4 boxes of 128
// codes and the rope columns as one bf16 box (40 KB stages); the math warps
// read both MMAs' latent operands straight from the codes, converting code
// pairs to f16 in registers (exact), against a query whose latent part was
// converted once per segment to f16, scaled per head by a power of two; the
// rope part stays bf16. One query buffer keeps the CTA at 106 KB, so two CTAs
// share an SM and cover each other's latencies.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"
#include "merge.cuh"
#include "sched.cuh"

namespace mla {
namespace {

constexpr int kSlabBytes = 64 * 128;         // 64 rows x 64 bf16 columns
constexpr int kStageBytes = 9 * kSlabBytes;  // one 64-token tile, 576 columns
// FP8 cache: a stage holds the tile's e4m3 codes (4 boxes of 64 rows x 128
// codes, SWIZZLE_128B; a page's rows land at their place in each box) and its
// bf16 rope slab. The math warps read their MMA operands straight from the
// codes and convert them in registers (e4m3 -> f16 is exact).
constexpr int kCodesBytes = 4 * kSlabBytes;  // 64 rows x 512 codes
constexpr int kStage8Bytes = kCodesBytes + kSlabBytes;
constexpr int kQSlabBytes = 16 * 128;        // 16 heads x 64 columns
constexpr int kQBytes = 9 * kQSlabBytes;
constexpr int kMathWarps = 4;
constexpr int kThreads = (kMathWarps + 1) * 32;
constexpr int kMathBar = 1;

template <int NST, bool SELF, bool FP8>
struct Smem {
  static constexpr int stage_bytes = FP8 ? kStage8Bytes : kStageBytes;
  // query buffers: FP8 keeps one, so that two CTAs fit on an SM
  static constexpr int qbufs = FP8 ? 1 : 2;
  static constexpr int stage = 0;
  static constexpr int q = NST * stage_bytes;
  static constexpr int pfrag = q + qbufs * kQBytes;                 // [4 warps][32 lanes] uint4
  static constexpr int smax = pfrag + kMathWarps * 32 * 16;     // [4][16] float
  static constexpr int lsum = smax + kMathWarps * 16 * 4;       // [4][16] float
  static constexpr int qsc = lsum + kMathWarps * 16 * 4;        // FP8: [2][16] float
  static constexpr int info = qsc + 2 * 16 * 4;                 // [NST] int2
  static constexpr int bars = info + NST * 8;                   // full, empty, qfull, qempty
  static constexpr int rows = (bars + (2 * NST + 4) * 8 + 15) / 16 * 16;  // SELF: plan
  static constexpr int bytes = rows + (SELF ? kSelfMaxRows * 16 + 64 : 0);
  static constexpr int alloc = bytes + 1024;                    // alignment slack
};

// D += A * B, m16n8k16, f16 inputs, fp32 accumulate (the FP8 cache's latent
// part: its e4m3 codes are exact in f16).
__device__ __forceinline__ void mma_16816_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four e4m3 codes (bytes 0..3 of x) to two f16 pairs; every e4m3 value,
// subnormals included, is exact in f16.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "barrier.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

template <int NST, bool SELF, bool FP8>
__global__ void __maxnreg__(168)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap cache_map,
                       const __grid_constant__ CUtensorMap q_map,
                       const __grid_constant__ CUtensorMap rope_map,
                       const __grid_constant__ CUtensorMap slab_map, DecodeArgs a) {
  using S = Smem<NST, SELF, FP8>;
  constexpr int QB = S::qbufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + S::bars);
  uint64_t* empty = full + NST;
  uint64_t* qfull = empty + NST;
  uint64_t* qempty = qfull + 2;
  int2* info = reinterpret_cast<int2*>(sm + S::info);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
  uint32_t* status = &reinterpret_cast<WsHeader*>(ws)->status;
  const int bs = a.block_size;
  const int bs_shift = bs == 16 ? 4 : (bs == 32 ? 5 : 6);
  const int ppt = kTile >> bs_shift;  // pages per tile

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMathWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], kMathWarps);
    }
    fence_mbar_init();
  }
  if (warp == kMathWarps && lane == 0) {
    prefetch_tensormap(&cache_map);
    prefetch_tensormap(&q_map);
    if (FP8) prefetch_tensormap(&rope_map);
    if (!FP8 && a.block_size == kTile) prefetch_tensormap(&slab_map);
  }
  __syncthreads();
  // early: only the cache stream may start before the preceding kernel ends
  const bool early = SELF && a.self_plan == 2;
  if (!early) pdl_wait();  // the plan and q_abs come from earlier kernels
  // The next kernel may launch now: its CTAs (the output projection's take
  // 36 KB of shared memory and 168 registers a thread) fit beside a decode CTA
  // and stage their weights while the decode runs.
  pdl_launch_dependents();

  SchedWalker sw;
  bool has_work;
  if constexpr (SELF) {
    int4* rows = reinterpret_cast<int4*>(sm + S::rows);
    int* scratch = reinterpret_cast<int*>(sm + S::rows + kSelfMaxRows * 16);
    const int total = self_plan<kThreads>(a.seq_lens, a.query_start_loc, a.batch, (int)a.num_q,
                                          a.groups, (int64_t)a.max_blocks_per_seq * bs, rows,
                                          scratch, status, tid);
    has_work = sw.init_rows(rows, (int)a.num_q, a.groups, total, a.num_ctas, blockIdx.x);
    if (warp < kMathWarps) {
      // the workspace and o_lat may still be read by earlier kernels
      pdl_wait();
      if (tid == 0 && has_work) {
        // the first query tile, as soon as q_abs is complete (the producer is
        // busy starting the cache stream)
        mbar_arrive_expect_tx(&qfull[0], kQBytes);
        const int qy = sw.n * a.num_heads + sw.g * kHG;
#pragma unroll 1
        for (int j = 0; j < 9; ++j)
          tma_load_2d(sm + S::q + j * kQSlabBytes, &q_map, 64 * j, qy, &qfull[0]);
      }
      // publish the plan (what plan_kernel would have written) for a later
      // mla_combine or mla_decode_planned on this workspace
      const WsLayout L = ws_layout(a.num_q, a.groups, a.num_ctas);
      int4* cta_start = reinterpret_cast<int4*>(ws + L.cta_start);
      if (tid == 0)
        cta_start[blockIdx.x] = has_work ? make_int4(sw.n, sw.g, sw.k, 0) : make_int4(-1, 0, 0, 0);
      if (blockIdx.x == 0) {
        int4* row_info = reinterpret_cast<int4*>(ws + L.row_info);
        for (int n = tid; n < (int)a.num_q; n += kMathWarps * 32) row_info[n] = rows[n];
        if (tid == 0) {
          WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
          hdr->magic = kMagic;
          hdr->mode = 0;
          hdr->qblocks = 0;
          hdr->total_units = total;
          hdr->share = sw.share;
          hdr->num_ctas = a.num_ctas;
          hdr->groups = a.groups;
          hdr->num_q = (int32_t)a.num_q;
          hdr->batch = a.batch;
        }
      }
    }
  } else {
    has_work = sw.init(ws, a.num_q, a.groups, a.num_ctas, blockIdx.x);
  }
  if (a.o_lat && warp < kMathWarps)
    zero_unvisited_rows(sw.row_info, sw.plan_ok, a.num_q, a.num_heads, a.o_lat, tid,
                        kMathWarps * 32);
  if (!has_work) return;
  Segment seg;

  if (warp == kMathWarps) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the schedule; lane 0 issues the copies. Block ids
    // come from the block table 32 at a time (lane l holds entry base + l and
    // hands it out by shuffle), so a tile never waits on a dependent load.
    const bool leader = lane == 0;
    const uint64_t policy = l2_evict_first_policy();
    int fills[NST];
#pragma unroll
    for (int i = 0; i < NST; ++i) fills[i] = 0;
    int qfills[2] = {0, 0};
    int seg_i = 0, tile_i = 0;
    bool ok_run = true;
    while (ok_run && sw.next(seg)) {
      const int qb = seg_i % QB;
      // the math warps are done with this buffer's previous query
      auto q_free = [&] {
        return seg_i < QB ||
               __all_sync(0xffffffffu, mbar_wait(&qempty[qb], ((seg_i / QB) - 1) & 1));
      };
      if (QB == 2 && !q_free()) {
        if (leader) set_status(status, MLA_DEV_TIMEOUT);
        break;
      }
      auto issue_q = [&] {
        // one buffer: the wait comes here, after this segment's first cache
        // tiles are on their way
        if (QB == 1 && !q_free()) {
          if (leader) set_status(status, MLA_DEV_TIMEOUT);
          return false;
        }
        // (self-planned: a math thread issued the first one)
        if (leader && !(SELF && seg_i == 0)) {
          if (early) pdl_wait();  // q_abs comes from the preceding kernel
          mbar_arrive_expect_tx(&qfull[qb], kQBytes);
          const int qy = seg.n * a.num_heads + seg.g * kHG;
#pragma unroll 1
          for (int j = 0; j < 9; ++j)
            tma_load_2d(sm + S::q + qb * kQBytes + j * kQSlabBytes, &q_map, 64 * j, qy, &qfull[qb]);
        }
        ++qfills[qb];
        return true;
      };
      // the first query (every query, with one buffer) goes out after the
      // segment's first NST cache tiles
      const int q_at = (seg_i == 0 || QB == 1) ? min(seg.k0 + NST, seg.k1) : seg.k0;
      auto maybe_issue_q = [&](int k) { return k != q_at || issue_q(); };
      const int visible = seg.pos + 1;
      const int32_t* bt = a.block_table + (size_t)seg.b * a.max_blocks_per_seq;
      int cache_base = -(1 << 30), cached = -1;
      for (int k = seg.k0; k < seg.k1; ++k) {
        if (!maybe_issue_q(k)) {
          ok_run = false;
          break;
        }
        const int st = tile_i % NST;
        const int tstart = k * kTile;
        const int v = min(kTile, visible - tstart);
        int blk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          blk[i] = -1;
          if (i < ppt && (i << bs_shift) < v) {  // warp-uniform
            const int bi = (tstart >> bs_shift) + i;
            if (bi < cache_base || bi - cache_base >= 32) {
              cache_base = bi;
              cached = bi + lane < a.max_blocks_per_seq ? bt[bi + lane] : -1;
            }
            blk[i] = __shfl_sync(0xffffffffu, cached, bi - cache_base);
          }
        }
        if (tile_i >= NST &&
            !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((tile_i / NST) - 1) & 1))) {
          if (leader) set_status(status, MLA_DEV_TIMEOUT);
          ok_run = false;
          break;
        }
        if (leader) {
          int okmask = 0;
          uint32_t bytes = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i < ppt && (i << bs_shift) < v) {
              if (blk[i] >= 0 && blk[i] < a.num_blocks) {
                okmask |= 1 << i;
                bytes += (FP8 ? 5u : 9u) * (uint32_t)bs * 128u;
              } else {
                set_status(status, MLA_DEV_BAD_BLOCK);
              }
            }
          }
          info[st] = make_int2(v, okmask);
          mbar_arrive_expect_tx(&full[st], bytes);
          uint8_t* dst = sm + S::stage + st * S::stage_bytes;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (okmask & (1 << i)) {
              if constexpr (FP8) {
                // 4 boxes of 128 codes, then the bf16 rope columns (element 256
                // of the row's bf16 view = byte 512) into the rope slab
#pragma unroll 1
                for (int j = 0; j < 4; ++j)
                  tma_load_2d_hint(dst + j * kSlabBytes + (i << bs_shift) * 128, &cache_map, 128 * j,
                                   blk[i] << bs_shift, &full[st], policy);
                tma_load_2d_hint(dst + kCodesBytes + (i << bs_shift) * 128, &rope_map, 256,
                                 blk[i] << bs_shift, &full[st], policy);
              } else if (ppt == 1) {
                // a 64-token page: its nine 64-column slabs in one copy (3-D view)
                tma_load_3d_hint(dst, &slab_map, 0, blk[i] << bs_shift, 0, &full[st], policy);
              } else {
#pragma unroll 1
                for (int j = 0; j < 9; ++j)
                  tma_load_2d_hint(dst + j * kSlabBytes + (i << bs_shift) * 128, &cache_map,
                                   64 * j, blk[i] << bs_shift, &full[st], policy);
              }
            }
          }
        }
        __syncwarp();
        ++fills[st];
        ++tile_i;
      }
      // a segment of fewer than NST tiles
      if (ok_run && !maybe_issue_q(seg.k1)) ok_run = false;
      ++seg_i;
    }
    if (!leader) return;
    // never leave with copies in flight
#pragma unroll
    for (int i = 0; i < NST; ++i)
      if (fills[i] > 0 && !mbar_wait(&full[i], (fills[i] - 1) & 1)) set_status(status, MLA_DEV_TIMEOUT);
    for (int i = 0; i < QB; ++i)
      if (qfills[i] > 0 && !mbar_wait(&qfull[i], (qfills[i] - 1) & 1)) set_status(status, MLA_DEV_TIMEOUT);
    return;
  }

  // -------------------------------------------------------------- math warps
  const int w = warp;
  const int g = lane >> 2, q = lane & 3;
  float* smax = reinterpret_cast<float*>(sm + S::smax);
  float* lsum = reinterpret_cast<float*>(sm + S::lsum);
  uint4* pfrag = reinterpret_cast<uint4*>(sm + S::pfrag);
  const WsLayout L = ws_layout(a.num_q, a.groups, a.num_ctas);
  float* lse_out = reinterpret_cast<float*>(ws + L.lse);
  float* o_out = reinterpret_cast<float*>(ws + L.opart);
  const float scale = a.scale_log2;

  int seg_i = 0, tile_i = 0;
  bool aborted = false;
  while (!aborted && sw.next(seg)) {
    const int qb = seg_i % QB;
    const bool qok = mbar_wait(&qfull[qb], (seg_i / QB) & 1);
    if (bar_red_or(kMathBar, kMathWarps * 32, !qok)) {
      if (lane == 0 && w == 0) set_status(status, MLA_DEV_TIMEOUT);
      break;
    }
    const uint8_t* qs = sm + S::q + qb * kQBytes;
    if constexpr (FP8) {
      // The latent part of the query becomes f16 in place, each head scaled
      // by the power of two that puts its largest magnitude in [2^14, 2^15):
      // no overflow, and every element down to 2^-28 of that maximum stays
      // exact. qsc[h] = kv_scale / that power undoes it on the scores.
      // Columns are reordered to match the key fragments: within each
      // 64-column slab, f16 column 16t + k holds query column
      // 16 ((k >> 1) & 3) + 4t + 2 (k >> 3) + (k & 1), so chunk c of a row
      // gathers the bf16 pairs at columns 16m + 2c, m = 0..3. A head's row
      // is read and written by the 8 lanes that own it, all in one warp.
      uint8_t* qw = sm + S::q + qb * kQBytes;
      const int h = tid >> 3, c = tid & 7;
      uint32_t x[8][4];
      float mx = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          x[j][m] = *reinterpret_cast<const uint32_t*>(qw + j * kQSlabBytes + sw128(h, 2 * m + (c >> 2)) +
                                                       (c & 3) * 4);
          mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(x[j][m] << 16)),
                               fabsf(__uint_as_float(x[j][m] & 0xffff0000u))));
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      const int E = (int)(__float_as_uint(mx) >> 23);
      const int e2 = E == 255 ? 0 : (E == 0 ? (mx > 0.f ? 126 : 0) : min(141 - E, 126));
      const float f = __uint_as_float((uint32_t)(e2 + 127) << 23);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t y[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          y[m] = pack_f16(__uint_as_float(x[j][m] << 16) * f, __uint_as_float(x[j][m] & 0xffff0000u) * f);
        *reinterpret_cast<uint4*>(qw + j * kQSlabBytes + sw128(h, c)) = make_uint4(y[0], y[1], y[2], y[3]);
      }
      if (c == 0)
        reinterpret_cast<float*>(sm + S::qsc)[qb * 16 + h] =
            a.kv_scale * __uint_as_float((uint32_t)(127 - e2) << 23);
      // the buffer's next TMA fill comes after these generic writes
      fence_proxy_async_smem();
    }
    float m_run0 = -INFINITY, m_run1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    for (int k = seg.k0; k < seg.k1; ++k) {
      const int st = tile_i % NST;
      const bool fok = mbar_wait(&full[st], (tile_i / NST) & 1);
      if (bar_red_or(kMathBar, kMathWarps * 32, !fok)) {
        if (lane == 0 && w == 0) set_status(status, MLA_DEV_TIMEOUT);
        aborted = true;
        break;
      }
      uint8_t* stg = sm + S::stage + st * S::stage_bytes;
      const uint8_t* rope = FP8 ? stg + kCodesBytes : stg + 8 * kSlabBytes;
      const int2 inf = info[st];
      const int v = inf.x, okmask = inf.y;
      const bool all_live = v == kTile && okmask == (1 << ppt) - 1;
      if (!FP8 && !all_live) {
        // zero the latent part of every row that is not a live token, so
        // P = 0 never meets a NaN in the product
        for (int i = tid; i < kTile * 8 * 8; i += kMathWarps * 32) {
          const int r = i >> 6, slab = (i >> 3) & 7, ch = i & 7;
          const bool live = r < v && ((okmask >> (r >> bs_shift)) & 1);
          if (!live) *reinterpret_cast<uint4*>(stg + slab * kSlabBytes + sw128(r, ch)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        named_bar_sync(kMathBar, kMathWarps * 32);
      }

      // ---- scores: S[16 heads x 16 tokens] for tokens [16w, 16w+16)
      // FP8: n index g of an n-tile is token pi(g) = g ^ 4 (g & 1) of its 8
      // (the two rows an 8-lane phase reads differ in bit 2, so the swizzled
      // 16-byte code loads never share a bank); the latent part goes to sr,
      // f16 codes against the scaled f16 query, and the head's qsc factor
      // brings it back.
      float s[2][4], sr[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        sr[i][0] = sr[i][1] = sr[i][2] = sr[i][3] = 0.f;
      }
      const int pig = FP8 ? g ^ ((g & 1) << 2) : g;
      const int qrow = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int krow = 16 * w + (FP8 ? (lane & 7) ^ ((lane & 1) << 2) : (lane & 7)) + ((lane >> 4) << 3);
      if constexpr (FP8) {
        // lane (g, q) takes codes 64j + 16q + 0..15 of its two tokens per
        // 64-column slab j: pairs 2t and 2t+1 are its B registers of k-block t
        const uint8_t* k0p = stg + (16 * w + pig) * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = (j >> 1) * kSlabBytes + (((4 * (j & 1) + q) ^ pig) << 4);
          const uint4 c0w = *reinterpret_cast<const uint4*>(k0p + off);
          const uint4 c1w = *reinterpret_cast<const uint4*>(k0p + off + 8 * 128);
          uint32_t kb[2][8];
          e4m3x4_to_f16(c0w.x, kb[0][0], kb[0][1]);
          e4m3x4_to_f16(c0w.y, kb[0][2], kb[0][3]);
          e4m3x4_to_f16(c0w.z, kb[0][4], kb[0][5]);
          e4m3x4_to_f16(c0w.w, kb[0][6], kb[0][7]);
          e4m3x4_to_f16(c1w.x, kb[1][0], kb[1][1]);
          e4m3x4_to_f16(c1w.y, kb[1][2], kb[1][3]);
          e4m3x4_to_f16(c1w.z, kb[1][4], kb[1][5]);
          e4m3x4_to_f16(c1w.w, kb[1][6], kb[1][7]);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(smem_u32(qs + j * kQSlabBytes + sw128(qrow, 2 * t + (lane >> 4))), a0, a1, a2, a3);
            mma_16816_f16(sr[0], a0, a1, a2, a3, kb[0][2 * t], kb[0][2 * t + 1]);
            mma_16816_f16(sr[1], a0, a1, a2, a3, kb[1][2 * t], kb[1][2 * t + 1]);
          }
        }
      }
#pragma unroll
      for (int kk = FP8 ? 32 : 0; kk < 36; ++kk) {
        const int j = kk >> 2, c0 = (kk & 3) * 2;
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(smem_u32(qs + j * kQSlabBytes + sw128(qrow, c0 + (lane >> 4))), a0, a1, a2, a3);
        const uint8_t* bsl = kk < 32 ? stg + j * kSlabBytes : rope;
        ldsm_x4(smem_u32(bsl + sw128(krow, c0 + ((lane >> 3) & 1))), b0, b1, b2, b3);
        mma_16816(s[0], a0, a1, a2, a3, b0, b1);
        mma_16816(s[1], a0, a1, a2, a3, b2, b3);
      }
      if constexpr (FP8) {
        const float* qsc = reinterpret_cast<const float*>(sm + S::qsc) + qb * 16;
        const float f0 = qsc[g], f1 = qsc[g + 8];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          s[nt][0] = fmaf(sr[nt][0], f0, s[nt][0]);
          s[nt][1] = fmaf(sr[nt][1], f0, s[nt][1]);
          s[nt][2] = fmaf(sr[nt][2], f1, s[nt][2]);
          s[nt][3] = fmaf(sr[nt][3], f1, s[nt][3]);
        }
      }
      // ---- mask, scale to base 2, tile row maxima
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = 2 * q + (i & 1);
          const int tok = 16 * w + nt * 8 + (FP8 ? n ^ ((n & 1) << 2) : n);
          const bool live = tok < v && ((okmask >> (tok >> bs_shift)) & 1);
          s[nt][i] = live ? s[nt][i] * scale : -INFINITY;
        }
      }
      float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      if (q == 0) {
        smax[w * 16 + g] = mx0;
        smax[w * 16 + g + 8] = mx1;
      }
      named_bar_sync(kMathBar, kMathWarps * 32);
      float t0 = smax[g], t1 = smax[g + 8];
#pragma unroll
      for (int ww = 1; ww < kMathWarps; ++ww) {
        t0 = fmaxf(t0, smax[ww * 16 + g]);
        t1 = fmaxf(t1, smax[ww * 16 + g + 8]);
      }
      const float mn0 = fmaxf(m_run0, t0), mn1 = fmaxf(m_run1, t1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(m_run0 - mu0), al1 = fast_exp2(m_run1 - mu1);
      m_run0 = mn0;
      m_run1 = mn1;
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        p[nt][0] = fast_exp2(s[nt][0] - mu0);
        p[nt][1] = fast_exp2(s[nt][1] - mu0);
        p[nt][2] = fast_exp2(s[nt][2] - mu1);
        p[nt][3] = fast_exp2(s[nt][3] - mu1);
      }
      l0 = l0 * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
      l1 = l1 * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
      if constexpr (FP8)
        pfrag[w * 32 + lane] = make_uint4(pack_f16(p[0][0], p[0][1]), pack_f16(p[0][2], p[0][3]),
                                          pack_f16(p[1][0], p[1][1]), pack_f16(p[1][2], p[1][3]));
      else
        pfrag[w * 32 + lane] = make_uint4(pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]),
                                          pack_bf16(p[1][0], p[1][1]), pack_bf16(p[1][2], p[1][3]));
      named_bar_sync(kMathBar, kMathWarps * 32);

      // ---- O[16 x 128w..128w+127] = O * alpha + P[16 x 64] V[64 x 128-slice]
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= al0; o[nt][1] *= al0;
        o[nt][2] *= al1; o[nt][3] *= al1;
      }
      if constexpr (FP8) {
        // value fragments straight from the codes. k-block ks holds tokens
        // 16ks + pi(2q + c) and 16ks + 8 + pi(2q + c), the order the
        // probabilities were written in; lane g of n-tile t in the 32-column
        // group G is column 128w + 32G + 4g + t. A lane loads one 32-bit word
        // (4 columns) from each of its 4 rows and pairs rows by byte
        // permutes. Rows that are not live tokens read as zeros, so P = 0
        // never meets garbage.
        const uint8_t* vbox = stg + w * kSlabBytes;
        const int ra = 2 * q, rb = (2 * q + 1) ^ 4;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint4 pa = pfrag[ks * 32 + lane];
          const int R0 = 16 * ks + ra, R1 = 16 * ks + rb;
          auto live_row = [&](int r) {
            return all_live || (r < v && ((okmask >> (r >> bs_shift)) & 1));
          };
          const bool l0 = live_row(R0), l1 = live_row(R1), l2 = live_row(R0 + 8), l3 = live_row(R1 + 8);
#pragma unroll
          for (int G = 0; G < 4; ++G) {
            const int cb = 2 * G + (g >> 2), bo = (g & 3) * 4;
            const uint8_t* p0 = vbox + R0 * 128 + ((cb ^ ra) << 4) + bo;
            const uint8_t* p1 = vbox + R1 * 128 + ((cb ^ rb) << 4) + bo;
            const uint32_t w0 = l0 ? *reinterpret_cast<const uint32_t*>(p0) : 0u;
            const uint32_t w1 = l1 ? *reinterpret_cast<const uint32_t*>(p1) : 0u;
            const uint32_t w2 = l2 ? *reinterpret_cast<const uint32_t*>(p0 + 8 * 128) : 0u;
            const uint32_t w3 = l3 ? *reinterpret_cast<const uint32_t*>(p1 + 8 * 128) : 0u;
            uint32_t bv[2][4];
            e4m3x4_to_f16(__byte_perm(w0, w1, 0x5140), bv[0][0], bv[0][1]);
            e4m3x4_to_f16(__byte_perm(w0, w1, 0x7362), bv[0][2], bv[0][3]);
            e4m3x4_to_f16(__byte_perm(w2, w3, 0x5140), bv[1][0], bv[1][1]);
            e4m3x4_to_f16(__byte_perm(w2, w3, 0x7362), bv[1][2], bv[1][3]);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              mma_16816_f16(o[4 * G + t], pa.x, pa.y, pa.z, pa.w, bv[0][t], bv[1][t]);
          }
        }
      } else {
        const int vrow_l = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint4 pa = pfrag[ks * 32 + lane];
          const int vrow = 16 * ks + vrow_l;
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            const int slab = 2 * w + (np >> 2);
            const int ch = (np & 3) * 2 + (lane >> 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(smem_u32(stg + slab * kSlabBytes + sw128(vrow, ch)), b0, b1, b2, b3);
            mma_16816(o[2 * np], pa.x, pa.y, pa.z, pa.w, b0, b1);
            mma_16816(o[2 * np + 1], pa.x, pa.y, pa.z, pa.w, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      ++tile_i;
    }
    if (aborted) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&qempty[qb]);

    // ---- finalise: l over all four warps' tokens, normalise, store partial
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (q == 0) {
      lsum[w * 16 + g] = l0;
      lsum[w * 16 + g + 8] = l1;
    }
    named_bar_sync(kMathBar, kMathWarps * 32);
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int ww = 0; ww < kMathWarps; ++ww) {
      L0 += lsum[ww * 16 + g];
      L1 += lsum[ww * 16 + g + 8];
    }
    // (FP8: the value rows were the codes; kv_scale restores them)
    const float vs = FP8 ? a.kv_scale : 1.f;
    const float inv0 = L0 > 0.f ? vs / L0 : 0.f, inv1 = L1 > 0.f ? vs / L1 : 0.f;
    const float lse0 = L0 > 0.f ? m_run0 + log2f(L0) : -INFINITY;
    const float lse1 = L1 > 0.f ? m_run1 + log2f(L1) : -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= inv0; o[nt][1] *= inv0;
      o[nt][2] *= inv1; o[nt][3] *= inv1;
    }
    const int t = seg.n * a.groups + seg.g;
    const int64_t slot = (int64_t)blockIdx.x + t;
    // the CTAs that share this q-tile
    const int u_first = seg.ustart + seg.g * seg.tiles;
    const int c_first = u_first / sw.share, c_last = (u_first + seg.tiles - 1) / sw.share;
    float* o_tile = a.o_lat ? a.o_lat + ((size_t)seg.n * a.num_heads + seg.g * kHG) * kDc : nullptr;
    auto store_rows = [&](float* base) {  // 16 x 512 fp32 rows, row stride kDc
      if constexpr (FP8) {
        // n-tile 4G + t, pair column n is column 128w + 32G + 4n + t: the
        // four n-tiles of a group give four consecutive columns
        float* ob = base + 128 * w + 8 * q;
#pragma unroll
        for (int G = 0; G < 4; ++G) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float* dst = ob + (size_t)(i < 2 ? g : g + 8) * kDc + 32 * G + 4 * (i & 1);
            *reinterpret_cast<float4*>(dst) =
                make_float4(o[4 * G][i], o[4 * G + 1][i], o[4 * G + 2][i], o[4 * G + 3][i]);
          }
        }
      } else {
        float* ob = base + 128 * w + 2 * q;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          *reinterpret_cast<float2*>(ob + (size_t)g * kDc + nt * 8) = make_float2(o[nt][0], o[nt][1]);
          *reinterpret_cast<float2*>(ob + (size_t)(g + 8) * kDc + nt * 8) = make_float2(o[nt][2], o[nt][3]);
        }
      }
    };
    if (o_tile == nullptr || c_first == c_last) {
      // partial for the merge kernel, or the whole q-tile straight into o_lat
      store_rows(o_tile ? o_tile : o_out + (size_t)slot * kHG * kDc);
      if (!o_tile && w == 0 && q == 0) {
        lse_out[(size_t)slot * kHG + g] = lse0;
        lse_out[(size_t)slot * kHG + g + 8] = lse1;
      }
    } else {
      // publish this part in fragment order, count it, merge if it was the last
      float4* of = reinterpret_cast<float4*>(o_out) + (size_t)slot * 16 * 128 + tid;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) of[nt * 128] = make_float4(o[nt][0], o[nt][1], o[nt][2], o[nt][3]);
      if (w == 0 && q == 0) {
        lse_out[(size_t)slot * kHG + g] = lse0;
        lse_out[(size_t)slot * kHG + g + 8] = lse1;
      }
      // every writing thread fences its stores, the barrier orders the
      // fences before the count, and one thread counts the part with an
      // acquire-release atomic (count_arrival); if it counted last, the
      // second barrier orders the merge's reads after every part's release
      int* arrive = reinterpret_cast<int*>(ws + L.arrive);
      __threadfence();
      named_bar_sync(kMathBar, kMathWarps * 32);
      int* flag = reinterpret_cast<int*>(smax);  // smax is free until the next tile
      if (tid == 0) flag[0] = count_arrival(&arrive[t]) == c_last - c_first;
      named_bar_sync(kMathBar, kMathWarps * 32);
      if (flag[0] != 0) {
        // online split-softmax merge over the parts in CTA order (the same
        // order whichever CTA merges, so repeated launches agree bit for bit):
        // running maximum M and weight sum d per row, O accumulated in o[]
        float M0 = -INFINITY, M1 = -INFINITY, d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        auto add_part = [&](const float4* v, float la, float lb) {
          const float n0 = fmaxf(M0, la), n1 = fmaxf(M1, lb);
          const float b0 = n0 == -INFINITY ? 0.f : n0, b1 = n1 == -INFINITY ? 0.f : n1;
          const float so0 = fast_exp2(M0 - b0), so1 = fast_exp2(M1 - b1);
          const float sn0 = fast_exp2(la - b0), sn1 = fast_exp2(lb - b1);
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) {
            o[nt][0] = fmaf(o[nt][0], so0, v[nt].x * sn0);
            o[nt][1] = fmaf(o[nt][1], so0, v[nt].y * sn0);
            o[nt][2] = fmaf(o[nt][2], so1, v[nt].z * sn1);
            o[nt][3] = fmaf(o[nt][3], so1, v[nt].w * sn1);
          }
          d0 = fmaf(d0, so0, sn0);
          d1 = fmaf(d1, so1, sn1);
          M0 = n0;
          M1 = n1;
        };
        const float4* op4 = reinterpret_cast<const float4*>(o_out) + tid;
        for (int c = c_first; c <= c_last; c += 2) {
          // two parts per round trip: data and log-sum-exps together
          const bool two = c + 1 <= c_last;
          const int64_t sa = (int64_t)c + t, sb = two ? sa + 1 : sa;
          float4 va[16], vb[16];
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) {
            va[nt] = __ldcg(op4 + ((size_t)sa * 16 + nt) * 128);
            vb[nt] = __ldcg(op4 + ((size_t)sb * 16 + nt) * 128);
          }
          const float la0 = __ldcg(lse_out + (size_t)sa * kHG + g);
          const float la1 = __ldcg(lse_out + (size_t)sa * kHG + g + 8);
          const float lb0 = __ldcg(lse_out + (size_t)sb * kHG + g);
          const float lb1 = __ldcg(lse_out + (size_t)sb * kHG + g + 8);
          add_part(va, la0, la1);
          if (two) add_part(vb, lb0, lb1);
        }
        const float r0 = d0 > 0.f ? 1.f / d0 : 0.f, r1 = d1 > 0.f ? 1.f / d1 : 0.f;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          o[nt][0] *= r0; o[nt][1] *= r0;
          o[nt][2] *= r1; o[nt][3] *= r1;
        }
        store_rows(o_tile);
        if (tid == 0) arrive[t] = 0;  // every part has arrived: ready for the next launch
      }
      named_bar_sync(kMathBar, kMathWarps * 32);
    }
    ++seg_i;
  }
}

}  // namespace

cudaError_t launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& cache_map,
                               const CUtensorMap& q_map, const CUtensorMap* rope_map,
                               const CUtensorMap* slab_map, cudaStream_t stream) {
  constexpr int NST = 2;
  // the maximum shared-memory carveout keeps an SM ready for a decode CTA
  // while small kernels before and after it share the SM
  auto launch = [&](auto kernel, int smem) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(a.num_ctas), dim3(kThreads), smem, stream, cache_map, q_map,
                      rope_map ? *rope_map : cache_map, slab_map ? *slab_map : cache_map, a);
  };
  if (rope_map) {
    // the FP8 cache: self-planned launches only; 40 KB stages and one query
    // buffer (106 KB in all), two CTAs to an SM
    if (!a.self_plan) return cudaErrorInvalidValue;
    return launch(decode_bf16_kernel<2, true, true>, Smem<2, true, true>::alloc);
  }
  if (a.self_plan) return launch(decode_bf16_kernel<NST, true, false>, Smem<NST, true, false>::alloc);
  return launch(decode_bf16_kernel<NST, false, false>, Smem<NST, false, false>::alloc);
}

}  // namespace mla
