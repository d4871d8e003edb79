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
#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"
#include "merge.cuh"
#include "sched.cuh"

namespace mla {
namespace {

constexpr int kSlabBytes = 64 * 128;         // 64 rows x 64 bf16 columns
constexpr int kStageBytes = 9 * kSlabBytes;  // one 64-token tile, 576 columns
constexpr int kQSlabBytes = 16 * 128;        // 16 heads x 64 columns
constexpr int kQBytes = 9 * kQSlabBytes;
constexpr int kMathWarps = 4;
constexpr int kThreads = (kMathWarps + 1) * 32;
constexpr int kMathBar = 1;

template <int NST>
struct Smem {
  static constexpr int stage = 0;
  static constexpr int q = NST * kStageBytes;
  static constexpr int pfrag = q + 2 * kQBytes;                 // [4 warps][32 lanes] uint4
  static constexpr int smax = pfrag + kMathWarps * 32 * 16;     // [4][16] float
  static constexpr int lsum = smax + kMathWarps * 16 * 4;       // [4][16] float
  static constexpr int merge = lsum + kMathWarps * 16 * 4;      // fused-merge scratch
  static constexpr int info = merge + (2 * kHG + kMergeChunk * kHG) * 4;  // [NST] int2
  static constexpr int bars = info + NST * 8;                   // full, empty, qfull, qempty
  static constexpr int bytes = bars + (2 * NST + 4) * 8;
  static constexpr int alloc = bytes + 1024;                    // alignment slack
};

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

template <int NST>
__global__ void __launch_bounds__(kThreads, 1)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap cache_map,
                       const __grid_constant__ CUtensorMap q_map, DecodeArgs a) {
  using S = Smem<NST>;
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
  }
  __syncthreads();
  // the plan and q_abs come from earlier kernels
  pdl_wait();
  pdl_launch_dependents();

  SchedWalker sw;
  const bool has_work = sw.init(ws, a.num_q, a.groups, a.num_ctas, blockIdx.x);
  if (a.o_lat && warp < kMathWarps)
    zero_unvisited_rows(sw.row_info, sw.plan_ok, a.num_q, a.num_heads, a.o_lat, tid,
                        kMathWarps * 32);
  if (!has_work) return;
  Segment seg;

  if (warp == kMathWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int fills[NST];
#pragma unroll
    for (int i = 0; i < NST; ++i) fills[i] = 0;
    int qfills[2] = {0, 0};
    int seg_i = 0, tile_i = 0;
    bool ok_run = true;
    while (ok_run && sw.next(seg)) {
      const int qb = seg_i & 1;
      if (seg_i >= 2 && !mbar_wait(&qempty[qb], ((seg_i >> 1) - 1) & 1)) {
        set_status(status, MLA_DEV_TIMEOUT);
        break;
      }
      auto issue_q = [&] {
        mbar_arrive_expect_tx(&qfull[qb], kQBytes);
        const int qy = seg.n * a.num_heads + seg.g * kHG;
#pragma unroll 1
        for (int j = 0; j < 9; ++j)
          tma_load_2d(sm + S::q + qb * kQBytes + j * kQSlabBytes, &q_map, 64 * j, qy, &qfull[qb]);
        ++qfills[qb];
      };
      // the first query goes out after the first NST cache tiles
      const int q_at = seg_i == 0 ? min(seg.k0 + NST, seg.k1) : seg.k0;
      auto maybe_issue_q = [&](int k) {
        if (k == q_at) issue_q();
      };
      const int visible = seg.pos + 1;
      const int32_t* bt = a.block_table + (size_t)seg.b * a.max_blocks_per_seq;
      for (int k = seg.k0; k < seg.k1; ++k) {
        maybe_issue_q(k);
        const int st = tile_i % NST;
        const int tstart = k * kTile;
        const int v = min(kTile, visible - tstart);
        int blk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          blk[i] = (i < ppt && (i << bs_shift) < v) ? bt[(tstart >> bs_shift) + i] : -1;
        if (tile_i >= NST && !mbar_wait(&empty[st], ((tile_i / NST) - 1) & 1)) {
          set_status(status, MLA_DEV_TIMEOUT);
          ok_run = false;
          break;
        }
        int okmask = 0;
        uint32_t bytes = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i < ppt && (i << bs_shift) < v) {
            if (blk[i] >= 0 && blk[i] < a.num_blocks) {
              okmask |= 1 << i;
              bytes += 9u * (uint32_t)bs * 128u;
            } else {
              set_status(status, MLA_DEV_BAD_BLOCK);
            }
          }
        }
        info[st] = make_int2(v, okmask);
        mbar_arrive_expect_tx(&full[st], bytes);
        uint8_t* dst = sm + S::stage + st * kStageBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (okmask & (1 << i)) {
#pragma unroll 1
            for (int j = 0; j < 9; ++j)
              tma_load_2d(dst + j * kSlabBytes + (i << bs_shift) * 128, &cache_map, 64 * j,
                          blk[i] << bs_shift, &full[st]);
          }
        }
        ++fills[st];
        ++tile_i;
      }
      if (ok_run) maybe_issue_q(seg.k1);  // a first segment of fewer than NST tiles
      ++seg_i;
    }
    // never leave with copies in flight
#pragma unroll
    for (int i = 0; i < NST; ++i)
      if (fills[i] > 0 && !mbar_wait(&full[i], (fills[i] - 1) & 1)) set_status(status, MLA_DEV_TIMEOUT);
    for (int i = 0; i < 2; ++i)
      if (qfills[i] > 0 && !mbar_wait(&qfull[i], (qfills[i] - 1) & 1)) set_status(status, MLA_DEV_TIMEOUT);
    return;
  }

  // -------------------------------------------------------------- math warps
  const int w = warp;
  const int g = lane >> 2, q = lane & 3;
  float* smax = reinterpret_cast<float*>(sm + S::smax);
  float* lsum = reinterpret_cast<float*>(sm + S::lsum);
  float* merge_scratch = reinterpret_cast<float*>(sm + S::merge);
  uint4* pfrag = reinterpret_cast<uint4*>(sm + S::pfrag);
  const WsLayout L = ws_layout(a.num_q, a.groups, a.num_ctas);
  float* lse_out = reinterpret_cast<float*>(ws + L.lse);
  float* o_out = reinterpret_cast<float*>(ws + L.opart);
  const float scale = a.scale_log2;

  int seg_i = 0, tile_i = 0;
  bool aborted = false;
  while (!aborted && sw.next(seg)) {
    const int qb = seg_i & 1;
    const bool qok = mbar_wait(&qfull[qb], (seg_i >> 1) & 1);
    if (bar_red_or(kMathBar, kMathWarps * 32, !qok)) {
      if (lane == 0 && w == 0) set_status(status, MLA_DEV_TIMEOUT);
      break;
    }
    const uint8_t* qs = sm + S::q + qb * kQBytes;
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
      uint8_t* stg = sm + S::stage + st * kStageBytes;
      const int2 inf = info[st];
      const int v = inf.x, okmask = inf.y;
      if (v < kTile || okmask != (1 << ppt) - 1) {
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
      float s[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
      const int qrow = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int krow = 16 * w + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
      for (int kk = 0; kk < 36; ++kk) {
        const int j = kk >> 2, c0 = (kk & 3) * 2;
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(smem_u32(qs + j * kQSlabBytes + sw128(qrow, c0 + (lane >> 4))), a0, a1, a2, a3);
        ldsm_x4(smem_u32(stg + j * kSlabBytes + sw128(krow, c0 + ((lane >> 3) & 1))), b0, b1, b2, b3);
        mma_16816(s[0], a0, a1, a2, a3, b0, b1);
        mma_16816(s[1], a0, a1, a2, a3, b2, b3);
      }
      // ---- mask, scale to base 2, tile row maxima
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = 16 * w + nt * 8 + 2 * q + (i & 1);
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
      pfrag[w * 32 + lane] = make_uint4(pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]),
                                        pack_bf16(p[1][0], p[1][1]), pack_bf16(p[1][2], p[1][3]));
      named_bar_sync(kMathBar, kMathWarps * 32);

      // ---- O[16 x 128w..128w+127] = O * alpha + P[16 x 64] V[64 x 128-slice]
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= al0; o[nt][1] *= al0;
        o[nt][2] *= al1; o[nt][3] *= al1;
      }
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
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    const int t = seg.n * a.groups + seg.g;
    const int64_t slot = (int64_t)blockIdx.x + t;
    // fused merge: which CTAs share this q-tile
    const int u_first = seg.ustart + seg.g * seg.tiles;
    const int c_first = u_first / sw.share, c_last = (u_first + seg.tiles - 1) / sw.share;
    const bool direct = a.o_lat != nullptr && c_first == c_last;
    float* ob = direct ? a.o_lat + ((size_t)seg.n * a.num_heads + seg.g * kHG) * kDc + 128 * w + 2 * q
                       : o_out + (size_t)slot * kHG * kDc + 128 * w + 2 * q;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      *reinterpret_cast<float2*>(ob + (size_t)g * kDc + nt * 8) = make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
      *reinterpret_cast<float2*>(ob + (size_t)(g + 8) * kDc + nt * 8) = make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
    }
    if (!direct && w == 0 && q == 0) {
      lse_out[(size_t)slot * kHG + g] = L0 > 0.f ? m_run0 + log2f(L0) : -INFINITY;
      lse_out[(size_t)slot * kHG + g + 8] = L1 > 0.f ? m_run1 + log2f(L1) : -INFINITY;
    }
    if (a.o_lat != nullptr && !direct) {
      // publish this part, count it, and merge if it was the last one
      int* arrive = reinterpret_cast<int*>(ws + L.arrive);
      __threadfence();
      named_bar_sync(kMathBar, kMathWarps * 32);
      int* flag = reinterpret_cast<int*>(smax);  // smax is free until the next tile
      if (tid == 0) flag[0] = atomicAdd(&arrive[t], 1) == c_last - c_first;
      named_bar_sync(kMathBar, kMathWarps * 32);
      const bool last = flag[0] != 0;
      if (last) {
        __threadfence();
        merge_qtile<kMathWarps * 32>(lse_out, o_out, (int64_t)c_first + t, c_last - c_first + 1, 1,
                                     a.o_lat + ((size_t)seg.n * a.num_heads + seg.g * kHG) * kDc, tid,
                                     merge_scratch, [] { named_bar_sync(kMathBar, kMathWarps * 32); });
        if (tid == 0) arrive[t] = 0;  // every part has arrived: ready for the next launch
      }
      named_bar_sync(kMathBar, kMathWarps * 32);
    }
    ++seg_i;
  }
}

}  // namespace

cudaError_t launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& cache_map,
                               const CUtensorMap& q_map, cudaStream_t stream) {
  constexpr int NST = 2;
  const int smem = Smem<NST>::alloc;
  cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel<NST>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_bf16_kernel<NST>, dim3(a.num_ctas), dim3(kThreads), smem, stream,
                    cache_map, q_map, a);
}

}  // namespace mla
