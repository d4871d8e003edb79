// The pages' two other forms of the same attention, for their three-way
// comparison ("mini-infer-17: MLA Attention", sections "版本 1:
// MLAAttentionNaive", "版本 2: MLAAttentionLatentCache" and "实验结果"):
//   version 1 caches the expanded key and value of every head:
//     row (token t, head h) = [K_nope (128) || k_rot (64) || V (128)],
//     K_nope = c_hat W_uk[h], V = c_hat W_uv[h]  (16 x 320 x 2 = 10,240 B/token)
//   version 2 caches the latent (as the absorbed form does) and re-expands
//     every cached token into those rows at every step, then attends.
//
// Kernels:
//   wt_prep_kernel      W_uk, W_uv [H, 512, 128] -> Wt [H, 256, 512] (K-major
//                       B operand of the expansion: rows 0-127 W_uk^T, 128-255 W_uv^T)
//   expand_tc_kernel    tcgen05 GEMM: 128 latent rows x 512 -> 256 columns of
//                       one head (K_nope || V) in TMEM, plus the shared k_rot,
//                       written as the rows above
//   naive_decode_kernel split-KV attention of one (query row, head) per warp
//                       over the expanded rows (HBM-bound: 640 B per token
//                       and head)
//   naive_merge_kernel  the split-softmax merge into out [num_q, H, 128]
#include "async_copy.cuh"
#include "common.cuh"
#include "rope_pairs.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kNv = 320;  // one (token, head) row of the expanded cache

// ---------------------------------------------------------------------------
// Wt[h][j][c] = W_uk[h][c][j] (j < 128), W_uv[h][c][j - 128] (j >= 128).
// 32 x 32 tiles through shared memory; grid (512 / 32, 256 / 32, H).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) wt_prep_kernel(const __nv_bfloat16* __restrict__ W_uk,
                                                      const __nv_bfloat16* __restrict__ W_uv,
                                                      __nv_bfloat16* __restrict__ Wt) {
  __shared__ __nv_bfloat16 t[32][33];
  const int c0 = blockIdx.x * 32, j0 = blockIdx.y * 32, h = blockIdx.z;
  const __nv_bfloat16* W = j0 < kDn ? W_uk : W_uv;
  const int jj0 = j0 < kDn ? j0 : j0 - kDn;
  pdl_wait();  // Wt lives in a workspace an earlier kernel may still read
  pdl_launch_dependents();
  for (int r = threadIdx.y; r < 32; r += 8)
    t[r][threadIdx.x] = W[((size_t)h * kDc + c0 + r) * kDn + jj0 + threadIdx.x];
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8)
    Wt[((size_t)h * 256 + j0 + r) * kDc + c0 + threadIdx.x] = t[threadIdx.x][r];
}

__global__ void iota_kernel(int64_t* __restrict__ out, int64_t n) {
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = i;
}

// ---------------------------------------------------------------------------
// expand_tc_kernel: a persistent tcgen05 GEMM, one CTA per SM. A unit is (128
// source rows, head h), numbered tile * H + h so that the H units of a tile
// run on neighbouring CTAs at the same time and its rows are read from DRAM
// once. D[r, j] = sum_c X[r, c] Wt[h][j][c] over the 512 latent columns in 8
// chunks of 64 columns.
//   warp 0   producer: the X chunk (128 rows, TMA boxes of box_rows rows: pages
//            of the latent cache, or slices of a dense buffer) and the Wt chunk
//            (256 rows) into a 4-stage ring, every copy of a chunk issued by one
//            warp instruction (a lane per box); a unit's box rows are looked up
//            one unit ahead
//   warp 1   MMA: 4 tcgen05.mma (M 128, N 256, K 16) per chunk into one of two
//            256-column TMEM accumulators, alternating by unit
//   warps 2-5 epilogue (TMEM lanes 32 (w % 4) ...): thread r converts row r of
//            the finished accumulator to bf16, a 64-column block at a time,
//            into the warp's staging rows in shared memory, and the warp writes
//            [K_nope || k_rot || V] of (slot, h) as whole 128-byte lines (k_rot
//            copied from the source row), while the MMAs of the next unit fill
//            the other accumulator
// Every unit goes through the pipeline; rows past a sequence's end (or with
// slot < 0) are computed from row 0 and not written.
//   mode 0: rows [128 tile, 128 tile + 128) of a dense [num_rows, 576] buffer,
//           row t written to slot dst_slots[t] (< 0: skipped).
//   mode 1: tokens [128 k, 128 k + 128) of sequence b (tile = b *
//           tiles_per_seq + k), read from and written to the same slot.
// ---------------------------------------------------------------------------
struct ExArgs {
  const int64_t* dst_slots;
  int64_t num_rows;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t max_blocks_per_seq;
  int32_t tiles_per_seq;
  int64_t num_blocks;          // latent cache blocks (mode 1)
  int32_t block_size;
  int32_t box_rows;            // rows of one source TMA box
  int32_t H;
  int32_t mode;
  int32_t total_units;         // tiles * H
  const __nv_bfloat16* src;    // the rows the source map views ([rows, 576])
  __nv_bfloat16* kv;           // [num_slots, H, 320]
  int64_t num_slots;
  uint32_t* status;
};

constexpr int kExRows = 128;
constexpr int kExA = kExRows * 128;  // 16 KB: 128 rows x 64 columns
constexpr int kExB = 256 * 128;      // 32 KB: 256 weight rows x 64 columns
constexpr int kExStages = 4;
constexpr int kExThreads = 192;   // producer, MMA, 4 epilogue warps

struct ExSmem {
  static constexpr int a = 0;                              // [stages]
  static constexpr int b = a + kExStages * kExA;           // [stages]
  static constexpr int stg = b + kExStages * kExB;         // [4 warps] 32 rows x 128 B
  static constexpr int bars = stg + 4 * 32 * 128;         // full, empty, tfull[2], tempty[2], mdone
  static constexpr int misc = bars + (2 * kExStages + 5) * 8;  // tmem base
  static constexpr int bytes = misc + 16;
  static constexpr int alloc = bytes + 1024;
};

// First source row of box `i` of unit tile (mode 1: the page's first row, or
// row 0 past the sequence's end or for a rejected block id).
__device__ __forceinline__ int ex_box_row(const ExArgs& a, int tile, int i) {
  if (a.mode == 0) return tile * kExRows + i * a.box_rows;
  const int b = tile / a.tiles_per_seq, k = tile % a.tiles_per_seq;
  const int len = a.seq_lens[b];
  if (len < 0 || (int64_t)len > (int64_t)a.max_blocks_per_seq * a.block_size) return 0;
  const int t0 = k * kExRows + i * a.box_rows;
  if (t0 >= len) return 0;
  const int page = a.block_table[(size_t)b * a.max_blocks_per_seq + t0 / a.block_size];
  return page >= 0 && page < a.num_blocks ? page * a.block_size : 0;
}

// Destination slot (-1: not written) and source row of row r of unit (tile, h);
// reports bad sequences, blocks and slots once.
__device__ __forceinline__ void ex_row(const ExArgs& a, int tile, int h, int r, int* dst,
                                       int* src) {
  *dst = -1;
  *src = 0;
  if (a.mode == 0) {
    const int64_t t = (int64_t)tile * kExRows + r;
    if (t >= a.num_rows) return;
    const int64_t slot = a.dst_slots[t];
    if (slot >= a.num_slots) {
      if (h == 0) set_status(a.status, MLA_DEV_BAD_SLOT);
    } else if (slot >= 0) {
      *dst = (int)slot;
    }
    *src = (int)t;
    return;
  }
  const int b = tile / a.tiles_per_seq, k = tile % a.tiles_per_seq;
  const int len = a.seq_lens[b];
  if (len < 0 || (int64_t)len > (int64_t)a.max_blocks_per_seq * a.block_size) {
    if (k == 0 && h == 0 && r == 0) set_status(a.status, MLA_DEV_BAD_SEQ);
    return;
  }
  const int tok = k * kExRows + r;
  if (tok >= len) return;
  const int page = a.block_table[(size_t)b * a.max_blocks_per_seq + tok / a.block_size];
  if (page >= 0 && page < a.num_blocks) {
    *dst = *src = page * a.block_size + tok % a.block_size;
  } else if (tok % a.block_size == 0 && h == 0) {
    set_status(a.status, MLA_DEV_BAD_BLOCK);
  }
}

__global__ void __launch_bounds__(kExThreads, 1) expand_tc_kernel(
    const __grid_constant__ CUtensorMap src_map, const __grid_constant__ CUtensorMap wt_map,
    ExArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + ExSmem::bars);
  uint64_t* empty = full + kExStages;
  uint64_t* tfull = empty + kExStages;   // [2] accumulator j % 2 complete
  uint64_t* tempty = tfull + 2;          // [2] accumulator j % 2 read out (4 warp arrivals)
  uint64_t* mdone = tempty + 2;          // every MMA issued so far has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + ExSmem::misc);
  const int nbox = kExRows / a.box_rows;
  const int H = a.H;

  if (tid == 0) {
    for (int i = 0; i < kExStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(mdone, 1);
    fence_mbar_init();
    prefetch_tensormap(&src_map);
    prefetch_tensormap(&wt_map);
  }
  // the source rows, Wt and the destination come from or go to earlier kernels
  pdl_wait();
  pdl_launch_dependents();
  if (warp == 0) tc::alloc(tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int c = 0;
    int last_fill[kExStages];
#pragma unroll
    for (int i = 0; i < kExStages; ++i) last_fill[i] = -1;
    bool ok = true;
    int u = blockIdx.x;
    int ycur = (u < a.total_units && lane < nbox) ? ex_box_row(a, u / H, lane) : 0;
    for (; ok && u < a.total_units; u += gridDim.x) {
      const int un = u + gridDim.x;  // look the next unit's boxes up now
      const int ynext = (un < a.total_units && lane < nbox) ? ex_box_row(a, un / H, lane) : 0;
      const int h = u % H;
#pragma unroll 1
      for (int kc = 0; kc < 8; ++kc, ++c) {
        const int st = c % kExStages;
        if (c >= kExStages &&
            !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((c / kExStages) - 1) & 1))) {
          ok = false;
          break;
        }
        // one warp instruction issues every copy of the chunk: lane i < nbox
        // the i-th box of source rows (its own looked-up row), lane nbox the
        // weight chunk
        if (lane == 0) mbar_arrive_expect_tx(&full[st], kExA + kExB);
        if (lane < nbox)
          tma_load_2d(sm + ExSmem::a + st * kExA + lane * a.box_rows * 128, &src_map, 64 * kc, ycur,
                      &full[st]);
        else if (lane == nbox)
          tma_load_2d(sm + ExSmem::b + st * kExB, &wt_map, 64 * kc, h * 256, &full[st]);
        last_fill[st] = c;
        __syncwarp();
      }
      ycur = ynext;
    }
    if (!ok && lane == 0) set_status(a.status, MLA_DEV_TIMEOUT);
    // no copy may still be in flight when the CTA ends
    if (lane == 0)
      for (int i = 0; i < kExStages; ++i)
        if (last_fill[i] >= 0) mbar_wait(&full[i], (last_fill[i] / kExStages) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t kId = tc::idesc_bf16(kExRows, 256, false, false);
    const bool leader = tc::elect_one();
    int c = 0, j = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x, ++j) {
      const int buf = j & 1;
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&tempty[buf], ((j >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t d = tmem + (uint32_t)buf * 256;
#pragma unroll 1
      for (int kc = 0; kc < 8; ++kc, ++c) {
        const int st = c % kExStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (c / kExStages) & 1))) {
          ok = false;
          break;
        }
        if (leader) {
          tc::fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ad = tc::smem_desc(smem_u32(sm + ExSmem::a + st * kExA) + 32 * ks, 16,
                                              1024, tc::kSwizzle128);
            const uint64_t bd = tc::smem_desc(smem_u32(sm + ExSmem::b + st * kExB) + 32 * ks, 16,
                                              1024, tc::kSwizzle128);
            tc::mma_bf16(d, ad, bd, kId, kc > 0 || ks > 0);
          }
          tc::commit(&empty[st]);
        }
        __syncwarp();
      }
      if (ok && leader) tc::commit(&tfull[buf]);
      __syncwarp();
    }
    if (!ok && leader) set_status(a.status, MLA_DEV_TIMEOUT);
    // every MMA must have completed before TMEM is freed
    if (leader) tc::commit(mdone);
    __syncwarp();
    mbar_wait(mdone, 0);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lane quadrant of this warp
    const int r = q * 32 + lane;     // row of the tile
    int j = 0;
    for (int u = blockIdx.x; u < a.total_units; u += gridDim.x, ++j) {
      const int buf = j & 1, tile = u / H, h = u % H;
      int dst, src;
      ex_row(a, tile, h, r, &dst, &src);   // while the MMAs run
      // the shared rope key of the row, as the source row holds it (loaded now:
      // its latency hides under the MMAs)
      uint4 kr[8];
      {
        const uint4* p = reinterpret_cast<const uint4*>(a.src + (size_t)src * kRow + kDc);
#pragma unroll
        for (int k = 0; k < 8; ++k) kr[k] = dst >= 0 ? p[k] : make_uint4(0u, 0u, 0u, 0u);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[buf], (j >> 1) & 1))) {
        if (lane == 0) set_status(a.status, MLA_DEV_TIMEOUT);
        break;
      }
      tc::fence_after_sync();
      const uint32_t trow = tmem + (uint32_t)buf * 256 + ((uint32_t)(q * 32) << 16);
      // Five 64-column blocks of the output row (K_nope 0-63, 64-127, k_rot,
      // V 0-63, 64-127): each thread puts its row's 128 bytes in the warp's
      // staging rows (16-byte chunks XOR-swizzled by row), then the warp
      // stores 4 rows per instruction as whole 128-byte lines.
      uint8_t* stg = sm + ExSmem::stg + q * 32 * 128;
#pragma unroll 1
      for (int blk = 0; blk < 5; ++blk) {
        uint4 ch[8];
        if (blk == 2) {
#pragma unroll
          for (int k = 0; k < 8; ++k) ch[k] = kr[k];
        } else {
          const uint32_t col = blk < 2 ? 64u * blk : 128u + 64u * (blk - 3);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t v[32];
            tc::ld32(trow + col + 32 * half, v);   // every lane: warp-collective
            tc::wait_ld();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              ch[4 * half + k] =
                  make_uint4(pack_bf16(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                             pack_bf16(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                             pack_bf16(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                             pack_bf16(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
          }
          if (blk == 4) {
            // the last TMEM read of this unit: the accumulator may take unit j + 2
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) = ch[k];
        __syncwarp();
        const int ocol = blk * 64;  // output columns of this block
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = 4 * i + (lane >> 3), c = lane & 7;
          const int d = __shfl_sync(0xffffffffu, dst, row);
          if (d >= 0)
            *reinterpret_cast<uint4*>(a.kv + ((size_t)d * H + h) * kNv + ocol + 8 * c) =
                *reinterpret_cast<const uint4*>(stg + row * 128 + ((c ^ (row & 7)) << 4));
        }
        __syncwarp();
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// naive_decode_kernel. Warp = (query row n, head h, split s); CTA = 8 heads of
// one (row, split). The query [q_nope || RoPE(q_pe)] sits in shared memory;
// per 32 tokens, groups of 8 lanes score 4 tokens at a time (each lane 48
// contiguous bytes of a key, partial dots summed by shuffles), the warp
// updates the online softmax, then lanes own 4 of the 128 value dimensions and
// accumulate the 32 weighted value rows (256 contiguous bytes per token). Output: the split's
// normalised partial and base-2 log-sum-exp.
// ---------------------------------------------------------------------------
struct NdArgs {
  const __nv_bfloat16* q_nope;  // [num_q, H, 128]
  const __nv_bfloat16* q_pe;    // [num_q, H, 64]
  const int32_t* q_positions;
  const __nv_bfloat16* kv;      // [num_slots, H, 320]
  int64_t num_blocks;
  const int32_t* block_table;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t batch;
  int32_t num_q;
  int32_t H;
  int32_t splits;
  int32_t split_len;  // a multiple of 32
  float scale_log2;
  RopeFreq freq;
  int32_t rope_interleaved;
  float* part_o;      // [num_q, H, splits, 128]
  float* part_lse;    // [num_q, H, splits]
  uint32_t* status;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__global__ void __launch_bounds__(256) naive_decode_kernel(NdArgs a) {
  __shared__ float sq[8][kDn + kDr];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x, s = blockIdx.y, h = blockIdx.z * 8 + w;
  pdl_wait();  // the cache and the query come from earlier kernels
  pdl_launch_dependents();

  // the sequence of row n: the last b with query_start_loc[b] <= n
  const int32_t* qsl = a.query_start_loc;
  int lo = 0, hi = a.batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (qsl[mid] <= n) lo = mid; else hi = mid;
  }
  const int b = lo, q0 = qsl[b], q1 = qsl[b + 1], len = a.seq_lens[b], ql = q1 - q0;
  const bool covered = q0 <= n && n < q1;
  const bool bad = !covered || ql > len || len < 0 ||
                   (int64_t)len > (int64_t)a.max_blocks_per_seq * a.block_size;
  if (bad && covered && s == 0 && tid == 0) set_status(a.status, MLA_DEV_BAD_SEQ);
  const int visible = bad ? 0 : len - ql + (n - q0) + 1;
  const int t0 = s * a.split_len, t1 = min(visible, t0 + a.split_len);

  // query of (n, h): nope part as given, rope part rotated to position q_positions[n]
  {
    const __nv_bfloat16* qn = a.q_nope + ((size_t)n * a.H + h) * kDn;
#pragma unroll
    for (int i = 0; i < 4; ++i) sq[w][lane + 32 * i] = __bfloat162float(qn[lane + 32 * i]);
    const __nv_bfloat16* qp = a.q_pe + ((size_t)n * a.H + h) * kDr;
    const int i1 = rope_i1(a.rope_interleaved, lane), i2 = rope_i2(a.rope_interleaved, lane);
    const float x1 = __bfloat162float(qp[i1]), x2 = __bfloat162float(qp[i2]);
    float cs, sn;
    rope_cos_sin(a.q_positions[n], a.freq.hi[lane], a.freq.lo[lane], &cs, &sn);
    sq[w][kDn + i1] = x1 * cs - x2 * sn;
    sq[w][kDn + i2] = x2 * cs + x1 * sn;
  }
  __syncwarp();

  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks_per_seq;
  const int bs = a.block_size;
  float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int tb = t0; tb < t1; tb += 32) {
    const int t = tb + lane;
    int slot = -1;
    if (t < t1) {
      const int page = bt[t / bs];
      if (page >= 0 && page < a.num_blocks) {
        slot = page * bs + t % bs;
      } else if (t % bs == 0 && w == 0) {
        set_status(a.status, MLA_DEV_BAD_BLOCK);
      }
    }
    // scores: 8 lanes share a token's 384-byte key (48 bytes each, so one
    // warp load covers 4 whole rows); partial dots summed over the 8 lanes,
    // then lane t takes token t's score
    const int g = lane >> 3, sub = lane & 7;
    float dots[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int st = __shfl_sync(0xffffffffu, slot, 4 * i + g);
      float d = 0.f;
      if (st >= 0) {
        const uint4* kr =
            reinterpret_cast<const uint4*>(a.kv + ((size_t)st * a.H + h) * kNv) + 3 * sub;
        const float* qv = &sq[w][24 * sub];
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const uint4 kk = __ldg(kr + c);
          d = fmaf(bf_lo(kk.x), qv[8 * c + 0], d);
          d = fmaf(bf_hi(kk.x), qv[8 * c + 1], d);
          d = fmaf(bf_lo(kk.y), qv[8 * c + 2], d);
          d = fmaf(bf_hi(kk.y), qv[8 * c + 3], d);
          d = fmaf(bf_lo(kk.z), qv[8 * c + 4], d);
          d = fmaf(bf_hi(kk.z), qv[8 * c + 5], d);
          d = fmaf(bf_lo(kk.w), qv[8 * c + 6], d);
          d = fmaf(bf_hi(kk.w), qv[8 * c + 7], d);
        }
      }
      dots[i] = d;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      dots[i] += __shfl_xor_sync(0xffffffffu, dots[i], 4);
      dots[i] += __shfl_xor_sync(0xffffffffu, dots[i], 2);
      dots[i] += __shfl_xor_sync(0xffffffffu, dots[i], 1);
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float v = __shfl_sync(0xffffffffu, dots[i], 8 * (lane & 3));
      if ((lane >> 2) == i) dot = v;
    }
    const float sc = slot >= 0 ? dot * a.scale_log2 : -INFINITY;
    const float mn = fmaxf(m, warp_max(sc));
    if (mn == -INFINITY) continue;  // warp-uniform: no visible token so far
    const float alpha = fast_exp2(m - mn);
    const float p = slot >= 0 ? fast_exp2(sc - mn) : 0.f;
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] *= alpha;
    m = mn;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
      const int sj = __shfl_sync(0xffffffffu, slot, j);
      const uint2 v = sj >= 0 ? __ldg(reinterpret_cast<const uint2*>(
                                    a.kv + ((size_t)sj * a.H + h) * kNv + kDn + kDr + 4 * lane))
                              : make_uint2(0u, 0u);
      acc[0] = fmaf(pj, bf_lo(v.x), acc[0]);
      acc[1] = fmaf(pj, bf_hi(v.x), acc[1]);
      acc[2] = fmaf(pj, bf_lo(v.y), acc[2]);
      acc[3] = fmaf(pj, bf_hi(v.y), acc[3]);
    }
  }
  const size_t pi = ((size_t)n * a.H + h) * a.splits + s;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  *reinterpret_cast<float4*>(a.part_o + pi * kDv + 4 * lane) =
      make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  if (lane == 0) a.part_lse[pi] = l > 0.f ? m + log2f(l) : -INFINITY;
}

// Split-softmax merge: out[n, h] = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),
// zeros for a (row, head) that saw no token. Warp = (row, head), lanes own 4
// dimensions; grid (num_q, H / 8).
__global__ void __launch_bounds__(256) naive_merge_kernel(const float* __restrict__ part_o,
                                                          const float* __restrict__ part_lse,
                                                          int splits, int H,
                                                          __nv_bfloat16* __restrict__ out) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x, h = blockIdx.y * 8 + w;
  pdl_wait();
  pdl_launch_dependents();
  const size_t base = ((size_t)n * H + h) * splits;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_lse[base + s]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float ls = part_lse[base + s];
      if (ls == -INFINITY) continue;
      const float wgt = fast_exp2(ls - M);
      const float4 o = *reinterpret_cast<const float4*>(part_o + (base + s) * kDv + 4 * lane);
      den += wgt;
      acc.x = fmaf(wgt, o.x, acc.x);
      acc.y = fmaf(wgt, o.y, acc.y);
      acc.z = fmaf(wgt, o.z, acc.z);
      acc.w = fmaf(wgt, o.w, acc.w);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint2 r;
  r.x = pack_bf16(acc.x * inv, acc.y * inv);
  r.y = pack_bf16(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(out + ((size_t)n * H + h) * kDv + 4 * lane) = r;
}

}  // namespace

namespace {

// Splits of the naive decode: about 4,096 warps over the whole batch, each
// split a multiple of 32 tokens (the same on every call with these sizes, so
// the workspace size follows from them).
struct NaiveSplit {
  int splits, split_len;
};

NaiveSplit naive_split(int64_t num_q, int H, int64_t max_len) {
  const int64_t pairs = num_q * H > 0 ? num_q * H : 1;
  const int64_t smax = max_len > 32 ? (max_len + 31) / 32 : 1;
  int64_t s = (4096 + pairs - 1) / pairs;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  int64_t len = (max_len + s - 1) / s;
  len = len < 32 ? 32 : (len + 31) / 32 * 32;
  s = max_len > 0 ? (max_len + len - 1) / len : 1;
  return {(int)s, (int)len};
}

// Workspace: [0, 256) status word and padding; Wt [H, 256, 512] bf16; then
// either (cache write) the normed rows [T, 576] bf16 and their indices [T]
// int64, or (decode) the partials [num_q, H, S, 128] f32 and log-sum-exps
// [num_q, H, S] f32.
struct NaiveWs {
  size_t wt, rows, slots, part_o, part_lse, write_end, decode_end;
};

NaiveWs naive_ws(int H, int64_t num_tokens, int64_t num_q, int splits) {
  NaiveWs L;
  L.wt = 256;
  const size_t u = align_up(L.wt + (size_t)H * 256 * kDc * 2, 256);
  L.rows = u;
  L.slots = align_up(L.rows + (size_t)num_tokens * kRow * 2, 256);
  L.write_end = align_up(L.slots + (size_t)num_tokens * 8, 256);
  L.part_o = u;
  L.part_lse = align_up(L.part_o + (size_t)num_q * H * splits * kDv * 4, 256);
  L.decode_end = align_up(L.part_lse + (size_t)num_q * H * splits * 4, 256);
  return L;
}

inline mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }
inline bool is_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

mla_status naive_common_checks(const mla_config* cfg) {
  mla_status s = validate_config(cfg);
  if (s != MLA_OK) return s;
  if (cfg->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;  // the comparison forms are bf16
  return MLA_OK;
}

// Wt (the K-major B operand of the expansion) into the workspace.
cudaError_t prep_wt(const mla_config& cfg, const void* W_uk, const void* W_uv, uint8_t* ws,
                    cudaStream_t st) {
  __nv_bfloat16* Wt = reinterpret_cast<__nv_bfloat16*>(ws + 256);
  return launch_pdl(wt_prep_kernel, dim3(kDc / 32, 256 / 32, cfg.num_heads), dim3(32, 8), 0, st,
                    (const __nv_bfloat16*)W_uk, (const __nv_bfloat16*)W_uv, Wt);
}

// The expansion of the rows `src_map` views with the workspace's Wt.
cudaError_t expand_rows(const mla_config& cfg, uint8_t* ws, const CUtensorMap& src_map,
                        const ExArgs& ea, unsigned tiles, cudaStream_t st) {
  const int H = cfg.num_heads;
  __nv_bfloat16* Wt = reinterpret_cast<__nv_bfloat16*>(ws + 256);
  cudaError_t e;
  CUtensorMap wt_map;
  if (!encode_map_2d(&wt_map, Wt, kDc, (uint64_t)H * 256, 64, 256)) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(expand_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           ExSmem::alloc);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  ExArgs args = ea;
  args.total_units = (int32_t)(tiles * (unsigned)H);
  const unsigned grid = (unsigned)args.total_units < (unsigned)sms ? (unsigned)args.total_units
                                                                    : (unsigned)sms;
  return launch_pdl(expand_tc_kernel, dim3(grid), dim3(kExThreads), ExSmem::alloc, st, src_map,
                    wt_map, args);
}

// Wt, then the expansion.
cudaError_t expand(const mla_config& cfg, const void* W_uk, const void* W_uv, uint8_t* ws,
                   const CUtensorMap& src_map, const ExArgs& ea, unsigned tiles, cudaStream_t st) {
  cudaError_t e = prep_wt(cfg, W_uk, W_uv, ws, st);
  if (e != cudaSuccess) return e;
  return expand_rows(cfg, ws, src_map, ea, tiles, st);
}

// mla_latent_expand with (W_uk, W_uv) or, when both are null, with the
// weights already prepared in the workspace.
mla_status latent_expand(const mla_config* cfg, const void* cache, int64_t num_blocks,
                         const int32_t* block_table, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, int32_t batch, const void* W_uk,
                         const void* W_uv, void* kv_cache, void* workspace, size_t ws_bytes,
                         void* stream) {
  const bool prepared = W_uk == nullptr && W_uv == nullptr;
  mla_status s = naive_common_checks(cfg);
  if (s != MLA_OK) return s;
  if (num_blocks < 0 || max_blocks_per_seq < 0 || batch < 0) return MLA_ERR_INVALID_ARGUMENT;
  if (num_blocks * cfg->block_size > ((int64_t)1 << 31) / cfg->num_heads)
    return MLA_ERR_UNSUPPORTED;
  if (!workspace || !is_aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (batch == 0 || max_blocks_per_seq == 0 || num_blocks == 0) return MLA_OK;
  if (!cache || !block_table || !seq_lens || !kv_cache || (!prepared && (!W_uk || !W_uv)))
    return MLA_ERR_INVALID_ARGUMENT;
  if (!is_aligned(cache, 16) || (!prepared && (!is_aligned(W_uk, 16) || !is_aligned(W_uv, 16))) ||
      !is_aligned(kv_cache, 16) || !is_aligned(block_table, 4) || !is_aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  const NaiveWs L = naive_ws(cfg->num_heads, 0, 0, 1);
  if (ws_bytes < L.write_end) return MLA_ERR_WORKSPACE_TOO_SMALL;
  const int bs = cfg->block_size;
  const int64_t max_len = (int64_t)max_blocks_per_seq * bs;
  const int64_t tiles = (max_len + kExRows - 1) / kExRows;
  if ((int64_t)batch * tiles * cfg->num_heads > 0x7fffffff) return MLA_ERR_UNSUPPORTED;
  CUtensorMap src_map;
  if (!encode_row_map(&src_map, cache, (uint64_t)num_blocks * bs, (uint32_t)bs)) return MLA_ERR_CUDA;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  ExArgs ea{};
  ea.block_table = block_table;
  ea.seq_lens = seq_lens;
  ea.max_blocks_per_seq = max_blocks_per_seq;
  ea.tiles_per_seq = (int32_t)tiles;
  ea.num_blocks = num_blocks;
  ea.block_size = bs;
  ea.box_rows = bs;
  ea.H = cfg->num_heads;
  ea.mode = 1;
  ea.src = reinterpret_cast<const __nv_bfloat16*>(cache);
  ea.kv = reinterpret_cast<__nv_bfloat16*>(kv_cache);
  ea.num_slots = num_blocks * bs;
  ea.status = reinterpret_cast<uint32_t*>(ws);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(prepared ? expand_rows(*cfg, ws, src_map, ea, (unsigned)(batch * tiles), st)
                              : expand(*cfg, W_uk, W_uv, ws, src_map, ea, (unsigned)(batch * tiles), st));
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_naive_workspace_size(const mla_config* cfg, int64_t num_q, int32_t max_blocks_per_seq,
                                int64_t num_tokens) {
  if (naive_common_checks(cfg) != MLA_OK || num_q < 0 || max_blocks_per_seq < 0 || num_tokens < 0)
    return 0;
  const NaiveSplit sp = naive_split(num_q, cfg->num_heads, (int64_t)max_blocks_per_seq * cfg->block_size);
  const NaiveWs L = naive_ws(cfg->num_heads, num_tokens, num_q, sp.splits);
  return L.write_end > L.decode_end ? L.write_end : L.decode_end;
}

mla_status mla_naive_cache_write(const mla_config* cfg, const void* c_kv, const void* k_pe,
                                 const int32_t* positions, const int64_t* slot_mapping,
                                 int64_t num_tokens, const void* rms_weight, const void* W_uk,
                                 const void* W_uv, void* kv_cache, int64_t num_blocks,
                                 void* workspace, size_t ws_bytes, void* stream) {
  mla_status s = naive_common_checks(cfg);
  if (s != MLA_OK) return s;
  if (num_tokens < 0 || num_blocks < 0 || num_tokens > ((int64_t)1 << 24))
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_blocks * cfg->block_size > ((int64_t)1 << 31) / cfg->num_heads)
    return MLA_ERR_UNSUPPORTED;
  if (!workspace || !is_aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return MLA_OK;
  if (!c_kv || !k_pe || !positions || !slot_mapping || !rms_weight || !W_uk || !W_uv || !kv_cache)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!is_aligned(c_kv, 16) || !is_aligned(k_pe, 16) || !is_aligned(rms_weight, 16) ||
      !is_aligned(W_uk, 16) || !is_aligned(W_uv, 16) || !is_aligned(kv_cache, 16) ||
      !is_aligned(positions, 4) || !is_aligned(slot_mapping, 8))
    return MLA_ERR_INVALID_ARGUMENT;
  const NaiveWs L = naive_ws(cfg->num_heads, num_tokens, 0, 1);
  if (ws_bytes < L.write_end) return MLA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  int64_t* rows_idx = reinterpret_cast<int64_t*>(ws + L.slots);
  void* rows = ws + L.rows;
  // 1. the normed latent and rotated key of each new token, as dense rows
  const int bs = cfg->block_size;
  cudaError_t e = launch_pdl(iota_kernel, dim3((unsigned)((num_tokens + 255) / 256 < 1024
                                                               ? (num_tokens + 255) / 256 : 1024)),
                             dim3(256), 0, st, rows_idx, num_tokens);
  if (e == cudaSuccess)
    e = launch_cache_write(*cfg, c_kv, k_pe, positions, rows_idx, num_tokens, rms_weight, rows,
                           (num_tokens + bs - 1) / bs, status, st);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  // 2. expand them into the rows of every head, at slot_mapping
  CUtensorMap src_map;
  if (!encode_row_map(&src_map, rows, (uint64_t)num_tokens, 64)) return MLA_ERR_CUDA;
  ExArgs ea{};
  ea.dst_slots = slot_mapping;
  ea.num_rows = num_tokens;
  ea.block_size = bs;
  ea.box_rows = 64;
  ea.H = cfg->num_heads;
  ea.mode = 0;
  ea.src = reinterpret_cast<const __nv_bfloat16*>(rows);
  ea.kv = reinterpret_cast<__nv_bfloat16*>(kv_cache);
  ea.num_slots = num_blocks * bs;
  ea.status = status;
  return cuda_status(expand(*cfg, W_uk, W_uv, ws, src_map, ea,
                            (unsigned)((num_tokens + kExRows - 1) / kExRows), st));
}

mla_status mla_latent_expand(const mla_config* cfg, const void* cache, int64_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t batch, const void* W_uk,
                             const void* W_uv, void* kv_cache, void* workspace, size_t ws_bytes,
                             void* stream) {
  if (!W_uk || !W_uv) return MLA_ERR_INVALID_ARGUMENT;
  return latent_expand(cfg, cache, num_blocks, block_table, max_blocks_per_seq, seq_lens, batch,
                       W_uk, W_uv, kv_cache, workspace, ws_bytes, stream);
}

mla_status mla_latent_expand_prepare(const mla_config* cfg, const void* W_uk, const void* W_uv,
                                     void* workspace, size_t ws_bytes, void* stream) {
  mla_status s = naive_common_checks(cfg);
  if (s != MLA_OK) return s;
  if (!workspace || !is_aligned(workspace, 256) || !W_uk || !W_uv || !is_aligned(W_uk, 16) ||
      !is_aligned(W_uv, 16))
    return MLA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < naive_ws(cfg->num_heads, 0, 0, 1).write_end) return MLA_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(prep_wt(*cfg, W_uk, W_uv, reinterpret_cast<uint8_t*>(workspace),
                             reinterpret_cast<cudaStream_t>(stream)));
}

mla_status mla_latent_expand_prepared(const mla_config* cfg, const void* cache, int64_t num_blocks,
                                      const int32_t* block_table, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t batch, void* kv_cache,
                                      void* workspace, size_t ws_bytes, void* stream) {
  return latent_expand(cfg, cache, num_blocks, block_table, max_blocks_per_seq, seq_lens, batch,
                       nullptr, nullptr, kv_cache, workspace, ws_bytes, stream);
}


mla_status mla_naive_decode(const mla_config* cfg, const void* q_nope, const void* q_pe,
                            const int32_t* q_positions, const void* kv_cache, int64_t num_blocks,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, const int32_t* query_start_loc,
                            int32_t batch, int64_t num_q, void* workspace, size_t ws_bytes,
                            void* out, void* stream) {
  mla_status s = naive_common_checks(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > 0x7fffffff || num_blocks * cfg->block_size > ((int64_t)1 << 31) / cfg->num_heads)
    return MLA_ERR_UNSUPPORTED;
  if (!workspace || !is_aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!q_nope || !q_pe || !q_positions || !kv_cache || !block_table || !seq_lens ||
      !query_start_loc || !out || batch == 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!is_aligned(q_nope, 16) || !is_aligned(q_pe, 16) || !is_aligned(kv_cache, 16) ||
      !is_aligned(out, 16) || !is_aligned(q_positions, 4) || !is_aligned(block_table, 4) ||
      !is_aligned(seq_lens, 4) || !is_aligned(query_start_loc, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  const int H = cfg->num_heads;
  const NaiveSplit sp = naive_split(num_q, H, (int64_t)max_blocks_per_seq * cfg->block_size);
  if (sp.splits > 65535) return MLA_ERR_UNSUPPORTED;  // grid.y
  const NaiveWs L = naive_ws(H, 0, num_q, sp.splits);
  if (ws_bytes < L.decode_end) return MLA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  NdArgs na{};
  na.q_nope = reinterpret_cast<const __nv_bfloat16*>(q_nope);
  na.q_pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  na.q_positions = q_positions;
  na.kv = reinterpret_cast<const __nv_bfloat16*>(kv_cache);
  na.num_blocks = num_blocks;
  na.block_table = block_table;
  na.max_blocks_per_seq = max_blocks_per_seq;
  na.block_size = cfg->block_size;
  na.seq_lens = seq_lens;
  na.query_start_loc = query_start_loc;
  na.batch = batch;
  na.num_q = (int32_t)num_q;
  na.H = H;
  na.splits = sp.splits;
  na.split_len = sp.split_len;
  na.scale_log2 = (float)(cfg->softmax_scale * 1.4426950408889634);
  na.freq = make_rope_freq((double)cfg->rope_base);
  na.rope_interleaved = cfg->rope_interleaved;
  na.part_o = reinterpret_cast<float*>(ws + L.part_o);
  na.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  na.status = reinterpret_cast<uint32_t*>(ws);
  cudaError_t e = launch_pdl(naive_decode_kernel, dim3((unsigned)num_q, sp.splits, H / 8),
                             dim3(256), 0, st, na);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return cuda_status(launch_pdl(naive_merge_kernel, dim3((unsigned)num_q, H / 8), dim3(256), 0,
                                st, (const float*)na.part_o, (const float*)na.part_lse,
                                sp.splits, H, reinterpret_cast<__nv_bfloat16*>(out)));
}

}  // extern "C"
