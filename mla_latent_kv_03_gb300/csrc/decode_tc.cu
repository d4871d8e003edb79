// Tensor-core (tcgen05 / TMEM) split-KV latent attention for tiles of 128
// (query row, head) rows: 128 heads of one query row, or 8 query rows x 16
// heads of a prefill chunk (any H with 8 * 16 / H rows). Sources: "mini-infer-17:
// MLA Attention", sections "版本 3: MLAAttentionAbsorbed" (scores and output
// against the latent rows) and "设计取舍" (the nope and rope score parts summed
// before a hand-written softmax); "07. MLA / Mamba / MoE in vLLM source" 2.3
// (paged layout).
//
// Work units are (q-block, 64-token tile); each equal share of the unit list
// is processed by a pair of CTAs, CTA 2c + h computing output columns
// [256h, 256h + 256) (the 128 x 512 fp32 accumulator would fill all of TMEM).
// TMEM (512 columns): O half [0, 256), two score buffers S [256, 320), two
// probability buffers P [320, 352) (bf16 pairs), query columns 256..575 of
// the q-block [352, 512) (bf16 pairs). Shared memory: query columns 0..255
// (64 KB) and a ring of four 32-token cache stages (36 KB each, SWIZZLE_128B).
// Per CTA (256 threads):
//   warp 0 (TMA producer): the q-block's shared-memory query columns and the
//     cache stages, guarded by full / empty mbarriers; every block id is
//     bounds-checked.
//   warp 1 (MMA issuer; the warp owns the TMEM allocation and issues from one
//     elected lane): S[i%2] = Q . K_i^T as 36 tcgen05.mma (M 128, N 32, K 16;
//     A from shared memory for columns < 256, from TMEM above), one stage
//     ahead of O += P[i%2] . V_i (2 tcgen05.mma, M 128, N 256, A = P in TMEM,
//     V MN-major from the stage), so the scores of stage i + 1 run while the
//     softmax of stage i does.
//   warps 4-7 (softmax): thread r owns row r: it loads the q-block's upper
//     query columns into TMEM, then per stage loads its 32 scores, masks
//     (sequence end, causal position, rejected blocks), keeps the running
//     maximum, rescales the warp's O rows in TMEM only when some row's maximum
//     grows by more than 2^8 (probabilities stay below 256), and stores bf16 P
//     to TMEM. At the end of a segment it normalises its O row into the
//     partial buffer (and, when o_lat is given, the last CTA of a q-block's
//     half merges the splits while they are in L2).
// Every wait is bounded; on a timeout the roles leave their loops, the MMA
// warp waits for its last MMAs and the producer for its copies before TMEM
// is freed.
#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"
#include "merge.cuh"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kTok = 32;                       // tokens per stage
constexpr int kSlab = kTok * 128;              // 32 rows x 64 bf16 columns
constexpr int kStage = 9 * kSlab;              // 36 KB
constexpr int kStages = 4;                     // cache stages in the ring
constexpr int kQSlab = kQBlockRows * 128;      // 128 rows x 64 columns
constexpr int kQSmemSlabs = 4;                 // query columns [0, 256) in shared memory
constexpr int kQSmemBytes = kQSmemSlabs * kQSlab;            // 64 KB
constexpr int kQTmemWords = (kRow - 64 * kQSmemSlabs) / 2;   // 160: columns [256, 576)
constexpr int kThreads = 256;
constexpr int kSoftWarp0 = 4;
constexpr int kSoftBar = 2;                    // named barrier of the softmax warps
constexpr uint32_t kOCol = 0, kSCol = 256, kPCol = 320, kQCol = 352, kTmemCols = 512;
static_assert(kQCol + kQTmemWords <= kTmemCols, "TMEM budget");
constexpr float kRescaleLog2 = 8.f;            // lazy rescale threshold (2^8)

enum {
  kFull0 = 0,
  kEmpty0 = kFull0 + kStages,
  kSFull0 = kEmpty0 + kStages,   // [2] scores of stage i in S[i % 2]
  kPFull0 = kSFull0 + 2,         // [2] probabilities of stage i in P[i % 2] (128 arrivals)
  kQFull = kPFull0 + 2,          // shared-memory query columns landed
  kQtReady,                      // TMEM query columns stored (128 arrivals)
  kQEmpty,                       // every score MMA of the segment done
  kPVDone,                       // the latest O += P . V done
  kODone,                        // every MMA of the segment done
  kOFree,                        // O read out by the epilogue (128 arrivals)
  kFinal,
  kNumBars
};

struct Smem {
  static constexpr int q = 0;
  static constexpr int stage = q + kQSmemBytes;
  static constexpr int info = stage + kStages * kStage;  // [kStages] int2
  static constexpr int bars = info + kStages * 8;
  static constexpr int misc = bars + kNumBars * 8;       // tmem base, abort flag, merge flag
  static constexpr int bytes = misc + 16;
  static constexpr int alloc = bytes + 1024;
};
static_assert(Smem::alloc <= 227 * 1024, "shared memory budget");
static_assert(Smem::bars % 8 == 0, "mbarrier alignment");

struct TcSeg {
  int qb, k0, k1, b, t_first, t_end, tiles, ustart, vis;
};

struct TcWalker {
  const int4* row_info;
  const int4* seq_info;
  const int4* qblock;
  int u, u_end, qb, k, G, share;
  bool plan_ok;

  __device__ bool init(const uint8_t* ws, int64_t num_q, int groups, int num_ctas, int batch,
                       int c) {
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    const WsLayoutTc L = ws_layout_tc(num_q, groups, num_ctas / 2, batch);
    row_info = reinterpret_cast<const int4*>(ws + L.row_info);
    seq_info = reinterpret_cast<const int4*>(ws + L.seq_info);
    qblock = reinterpret_cast<const int4*>(ws + L.qblock);
    plan_ok = hdr->magic == kMagic && hdr->mode == 1 && hdr->num_q == num_q &&
              hdr->groups == groups && hdr->num_ctas == num_ctas && hdr->batch == batch;
    if (!plan_ok) return false;
    G = groups;
    share = hdr->share;
    u = c * share;
    u_end = min(u + share, hdr->total_units);
    if (u >= u_end) return false;
    const int4 cs = reinterpret_cast<const int4*>(ws + L.cta_start)[c];
    qb = cs.x;
    k = cs.y;
    return qb >= 0;
  }

  __device__ bool next(TcSeg& s) {
    if (u >= u_end) return false;
    const int4 bi = qblock[qb];
    const int take = min(bi.z - k, u_end - u);
    s.qb = qb; s.k0 = k; s.k1 = k + take; s.b = bi.x; s.t_first = bi.y; s.tiles = bi.z;
    s.ustart = bi.w;
    s.t_end = seq_info[bi.x].z;
    const int t_last = min(bi.y + kQBlockTiles, s.t_end) - 1;
    s.vis = row_info[t_last / G].y + 1;   // tokens the block's last row sees
    u += take;
    k += take;
    if (k == bi.z) { k = 0; ++qb; }
    return true;
  }
};

// bounded wait that also gives up when another role has aborted
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
    }
  }
}

__device__ __forceinline__ bool soft_red_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "barrier.red.or.pred po, %2, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(kSoftBar)
      : "memory");
  return r != 0;
}

// Stages (32 tokens) of a segment that hold a token its last row sees: they
// form a prefix of the segment's tiles. Stage t starts at token k0 * 64 + 32 t.
__device__ __forceinline__ int seg_stages(const TcSeg& s) {
  const int span = s.vis - s.k0 * kTile;
  return span <= 0 ? 0 : min((span + kTok - 1) / kTok, 2 * (s.k1 - s.k0));
}

// Query columns [256, 576) of q-block row `qrow` into this thread's TMEM lane
// (rows past the last query row are zero). Warp-collective.
__device__ __forceinline__ void load_q_tmem(const uint16_t* q_abs, int64_t qrow, int64_t qrows,
                                            uint32_t taddr) {
  const uint4* src = reinterpret_cast<const uint4*>(q_abs + (size_t)qrow * kRow + 64 * kQSmemSlabs);
  const bool live = qrow < qrows;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 buf[20];
    if (live) {
#pragma unroll
      for (int i = 0; i < 20; ++i) buf[i] = __ldg(src + 20 * h + i);
    } else {
#pragma unroll
      for (int i = 0; i < 20; ++i) buf[i] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < 5; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[4 * k] = buf[4 * c + k].x;
        w[4 * k + 1] = buf[4 * c + k].y;
        w[4 * k + 2] = buf[4 * c + k].z;
        w[4 * k + 3] = buf[4 * c + k].w;
      }
      tc::st16(taddr + kQCol + 80 * h + 16 * c, w);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap cache_map,
                     const __grid_constant__ CUtensorMap q_map, DecodeArgs a, int batch) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::bars);
  int2* info = reinterpret_cast<int2*>(sm + Smem::info);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Smem::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Smem::misc + 4);
  int* merge_flag = reinterpret_cast<int*>(sm + Smem::misc + 8);
  uint8_t* sQ = sm + Smem::q;
  uint8_t* sStage = sm + Smem::stage;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int share_idx = blockIdx.x >> 1, half = blockIdx.x & 1;
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
  uint32_t* status = &reinterpret_cast<WsHeader*>(ws)->status;
  const int bs = a.block_size;
  const int bsr = bs < kTok ? bs : kTok;            // rows of one TMA box
  const int bsr_shift = bsr == 16 ? 4 : 5;
  const int ppst = kTok / bsr;                      // boxes (pages or half pages) per stage
  const int full_mask = (1 << ppst) - 1;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool many = i == kPFull0 || i == kPFull0 + 1 || i == kQtReady || i == kOFree;
      mbar_init(&bars[i], many ? 128 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(tmem_slot, kTmemCols);
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&cache_map);
    prefetch_tensormap(&q_map);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the plan and q_abs come from earlier kernels
  pdl_launch_dependents();

  TcWalker sw;
  const bool has_work = sw.init(ws, a.num_q, a.groups, a.num_ctas, batch, share_idx);
  if (a.o_lat && warp >= kSoftWarp0)
    zero_unvisited_rows(sw.row_info, sw.plan_ok, a.num_q, a.num_heads, a.o_lat, tid - 128, 128);
  TcSeg seg;

  if (has_work && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage_i = 0, seg_i = 0;
      bool ok = true;
      while (ok && sw.next(seg)) {
        if (seg_i > 0 && !wait_or_abort(&bars[kQEmpty], (seg_i - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars[kQFull], kQSmemBytes);
#pragma unroll 1
        for (int j = 0; j < kQSmemSlabs; ++j)
          tma_load_2d(sQ + j * kQSlab, &q_map, 64 * j, kHG * seg.t_first, &bars[kQFull]);
        ++seg_i;
        const int32_t* bt = a.block_table + (size_t)seg.b * a.max_blocks_per_seq;
        const int n = seg_stages(seg);
#pragma unroll 1
        for (int t = 0; t < n; ++t) {
          const int tstart = seg.k0 * kTile + t * kTok;
          const int v = min(kTok, seg.vis - tstart);
          const int slot = stage_i & (kStages - 1);
          int blk[2], okmask = 0, nload = 0;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            blk[i] = -1;
            if (i < ppst && (i << bsr_shift) < v) blk[i] = bt[(tstart + (i << bsr_shift)) / bs];
          }
          if (stage_i >= kStages &&
              !wait_or_abort(&bars[kEmpty0 + slot], ((stage_i / kStages) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (i < ppst && (i << bsr_shift) < v) {
              if (blk[i] >= 0 && blk[i] < a.num_blocks) {
                okmask |= 1 << i;
                ++nload;
              } else {
                set_status(status, MLA_DEV_BAD_BLOCK);
              }
            }
          }
          info[slot] = make_int2(v, okmask);
          mbar_arrive_expect_tx(&bars[kFull0 + slot], (uint32_t)nload * 9u * (uint32_t)bsr * 128u);
          uint8_t* dst = sStage + slot * kStage;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (okmask & (1 << i)) {
              const int tok = tstart + (i << bsr_shift);
              const int y = blk[i] * bs + (tok % bs);
#pragma unroll 1
              for (int j = 0; j < 9; ++j)
                tma_load_2d(dst + j * kSlab + (i << bsr_shift) * 128, &cache_map, 64 * j, y,
                            &bars[kFull0 + slot]);
            }
          }
          ++stage_i;
        }
      }
      if (!ok) {
        set_status(status, MLA_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      // never leave with copies in flight: wait for the last fill of each slot
      for (int slot = 0; slot < kStages; ++slot) {
        const int fills = stage_i > slot ? (stage_i - 1 - slot) / kStages + 1 : 0;
        if (fills > 0 && !mbar_wait(&bars[kFull0 + slot], (fills - 1) & 1))
          set_status(status, MLA_DEV_TIMEOUT);
      }
      if (seg_i > 0 && !mbar_wait(&bars[kQFull], (seg_i - 1) & 1)) set_status(status, MLA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (has_work && warp == 1) {
    // --------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdS = tc::idesc_bf16(128, kTok, false, false);
    constexpr uint32_t kIdO = tc::idesc_bf16(128, 256, false, true);
    // descriptors of the first slab; others differ only in the start address
    const uint64_t qdesc = tc::smem_desc(smem_u32(sQ), 16, 1024, tc::kSwizzle128);
    const uint64_t kdesc = tc::smem_desc(smem_u32(sStage), 16, 1024, tc::kSwizzle128);
    const uint64_t vdesc =
        tc::smem_desc(smem_u32(sStage) + 4 * half * kSlab, kSlab, 1024, tc::kSwizzle128);
    const bool leader = tc::elect_one();
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
    };
    // S[i % 2] = Q . K_i^T over the 576 columns (9 slabs x 4 k-steps)
    auto issue_score = [&](int i) {
      const int slot = i & (kStages - 1);
      const uint32_t d = tmem + kSCol + (uint32_t)(i & 1) * kTok;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 36; ++kk) {
          const int j = kk >> 2, c = kk & 3;
          const uint64_t b = kdesc + (uint64_t)((slot * kStage + j * kSlab + c * 32) >> 4);
          if (j < kQSmemSlabs)
            tc::mma_bf16(d, qdesc + (uint64_t)((j * kQSlab + c * 32) >> 4), b, kIdS, kk > 0);
          else
            tc::mma_bf16_tmem_a(d, tmem + kQCol + (uint32_t)((j - kQSmemSlabs) * 32 + c * 8), b,
                                kIdS, kk > 0);
        }
        tc::commit(&bars[kSFull0 + (i & 1)]);
      }
      __syncwarp();
    };
    // O += P[i % 2] . V_i (this CTA's 256 latent columns of the stage)
    auto issue_pv = [&](int i, bool first) {
      const int slot = i & (kStages - 1);
      if (leader) {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          tc::mma_bf16_tmem_a(tmem + kOCol, tmem + kPCol + (uint32_t)((i & 1) * 16 + ks * 8),
                              vdesc + (uint64_t)((slot * kStage + ks * 16 * 128) >> 4), kIdO,
                              !(first && ks == 0));
        tc::commit(&bars[kEmpty0 + slot]);
        tc::commit(&bars[kPVDone]);
      }
      __syncwarp();
    };
    int stage_i = 0, seg_i = 0;
    bool ok = true;
    while (ok && sw.next(seg)) {
      const int n = seg_stages(seg);
      if (!warp_wait(&bars[kQFull], seg_i & 1) || !warp_wait(&bars[kQtReady], seg_i & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (n > 0) {
        if (!warp_wait(&bars[kFull0 + (stage_i & (kStages - 1))], (stage_i / kStages) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        issue_score(stage_i);
      }
#pragma unroll 1
      for (int t = 0; t < n; ++t) {
        const int i = stage_i + t;
        if (t + 1 < n) {
          // scores of the next stage while the softmax works on this one
          if (!warp_wait(&bars[kFull0 + ((i + 1) & (kStages - 1))], ((i + 1) / kStages) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          issue_score(i + 1);
        } else {
          if (leader) tc::commit(&bars[kQEmpty]);  // the query may be replaced
          __syncwarp();
        }
        if (!warp_wait(&bars[kPFull0 + (i & 1)], (i >> 1) & 1)) {
          ok = false;
          break;
        }
        if (t == 0 && seg_i > 0 && !warp_wait(&bars[kOFree], (seg_i - 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        issue_pv(i, t == 0);
      }
      if (!ok) break;
      if (leader) {
        if (n == 0) tc::commit(&bars[kQEmpty]);
        tc::commit(&bars[kODone]);
      }
      __syncwarp();
      stage_i += n;
      ++seg_i;
    }
    if (!ok && leader) {
      set_status(status, MLA_DEV_TIMEOUT);
      *abort_flag = 1;
    }
    // every MMA issued so far must finish before TMEM is freed
    if (leader) tc::commit(&bars[kFinal]);
    __syncwarp();
    if (!mbar_wait(&bars[kFinal], 0) && leader) set_status(status, MLA_DEV_TIMEOUT);
    __syncwarp();
  } else if (has_work && warp >= kSoftWarp0) {
    // ----------------------------------------------------------- softmax
    const int r = tid - kSoftWarp0 * 32;                 // row of the q-block
    const uint32_t trow = tmem + ((uint32_t)((warp - kSoftWarp0) * 32) << 16);
    const WsLayoutTc L = ws_layout_tc(a.num_q, a.groups, a.num_ctas / 2, batch);
    float* lse_out = reinterpret_cast<float*>(ws + L.lse);
    float* o_out = reinterpret_cast<float*>(ws + L.opart);
    int* arrive = reinterpret_cast<int*>(ws + L.arrive);
    const uint16_t* q_abs = reinterpret_cast<const uint16_t*>(a.q_abs);
    const int64_t qrows = a.num_q * a.num_heads;
    const float scale = a.scale_log2;
    int stage_i = 0, seg_i = 0;
    bool aborted = false, fail = false;
    bool have = sw.next(seg);
    if (have) {
      load_q_tmem(q_abs, (int64_t)kHG * seg.t_first + r, qrows, trow);
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars[kQtReady]);
    }
    while (have) {
      const int n = seg_stages(seg);
      const int t = seg.t_first + r / kHG;
      const bool valid_row = t < seg.t_end;
      const int pos = valid_row ? sw.row_info[t / sw.G].y : -1;
      float m_used = -INFINITY, l = 0.f;
#pragma unroll 1
      for (int tt = 0; tt < n; ++tt) {
        const int i = stage_i + tt, slot = i & (kStages - 1), b = i & 1;
        bool okw = wait_or_abort(&bars[kFull0 + slot], (i / kStages) & 1, abort_flag);
        okw = okw && wait_or_abort(&bars[kSFull0 + b], (i >> 1) & 1, abort_flag);
        if (soft_red_or(!okw || fail)) { aborted = true; break; }
        tc::fence_after_sync();
        uint32_t sr[32];
        tc::ld32(trow + kSCol + (uint32_t)b * kTok, sr);
        tc::wait_ld();
        const int tstart = seg.k0 * kTile + tt * kTok;
        const int2 inf = info[slot];
        const int v = inf.x, okmask = inf.y;
        // live tokens: a prefix (sequence end, causal position) minus rejected blocks
        const int lim = min(v, pos - tstart + 1);
        float x[32];
        if (lim >= kTok && okmask == full_mask) {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(sr[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const bool live = j < lim && ((okmask >> (j >> bsr_shift)) & 1);
            x[j] = live ? __uint_as_float(sr[j]) : -INFINITY;
          }
        }
        float mx[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) mx[j] = fmaxf(x[j], x[j + 16]);
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
        const float m_cand = mx[0] * scale;   // scale > 0
        float alpha = 1.f;
        bool rescale_o = false;
        if (m_cand > m_used + kRescaleLog2 || (m_used == -INFINITY && m_cand != -INFINITY)) {
          if (m_used != -INFINITY) {
            alpha = fast_exp2(m_used - m_cand);
            rescale_o = tt > 0;
          }
          l *= alpha;
          m_used = m_cand;
        }
        if (__any_sync(0xffffffffu, rescale_o)) {
          // this warp's O rows: the previous O += P . V must have landed
          const bool okp = __all_sync(0xffffffffu, wait_or_abort(&bars[kPVDone], (i - 1) & 1, abort_flag));
          if (okp) {
            tc::fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t o[32];
              tc::ld32(trow + kOCol + 32 * c, o);
              tc::wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tc::st32(trow + kOCol + 32 * c, o);
            }
          } else {
            fail = true;
          }
        }
        const float mneg = m_used == -INFINITY ? 0.f : -m_used;
        float p[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) p[j] = fast_exp2(fmaf(x[j], scale, mneg));
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16(p[2 * j], p[2 * j + 1]);
        tc::st16(trow + kPCol + (uint32_t)b * 16, pk);
        float ps[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) ps[j] = p[j] + p[j + 16];
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) ps[j] += ps[j + w];
        l += ps[0];
        if (v < kTok || okmask != full_mask) {
          // cache rows past the sequence's last token or in a rejected block may
          // hold anything (NaN): zero this half's latent columns so P = 0 stays 0
          uint8_t* stg = sStage + slot * kStage;
          for (int e = r; e < kTok * 4 * 8; e += 128) {
            const int row = e >> 5, sl = 4 * half + ((e >> 3) & 3), ch = e & 7;
            const bool live = row < v && ((okmask >> (row >> bsr_shift)) & 1);
            if (!live) *reinterpret_cast<uint4*>(stg + sl * kSlab + sw128(row, ch)) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&bars[kPFull0 + b]);
      }
      if (aborted) break;
      stage_i += n;
      // the next segment's upper query columns, while this one's last
      // products finish (its scores are all done once QEmpty completes)
      TcSeg nxt;
      const bool more = sw.next(nxt);
      if (more) {
        const bool okq = wait_or_abort(&bars[kQEmpty], seg_i & 1, abort_flag);
        if (soft_red_or(!okq || fail)) { aborted = true; break; }
        tc::fence_after_sync();
        load_q_tmem(q_abs, (int64_t)kHG * nxt.t_first + r, qrows, trow);
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&bars[kQtReady]);
      }
      // ---- epilogue: normalise the O row half into the partial buffer
      const bool okd = wait_or_abort(&bars[kODone], seg_i & 1, abort_flag);
      if (soft_red_or(!okd || fail)) { aborted = true; break; }
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t slot = (int64_t)share_idx + seg.qb;
      float4* dst = reinterpret_cast<float4*>(o_out + ((size_t)slot * kQBlockRows + r) * kDc + 256 * half);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        tc::ld32(trow + kOCol + 32 * c, o);
        tc::wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dst[8 * c + k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                       __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
      }
      // both halves see the same scores, so both write the same lse
      lse_out[slot * kQBlockRows + r] = l > 0.f ? m_used + log2f(l) : -INFINITY;
      tc::fence_before_sync();
      mbar_arrive(&bars[kOFree]);
      if (a.o_lat != nullptr) {
        // count this part; the last part of this half merges the q-block
        const int c_first = seg.ustart / sw.share;
        const int c_last = (seg.ustart + seg.tiles - 1) / sw.share;
        __threadfence();
        named_bar_sync(kSoftBar, 128);
        if (r == 0) *merge_flag = atomicAdd(&arrive[seg.qb * 2 + half], 1) == c_last - c_first;
        named_bar_sync(kSoftBar, 128);
        if (*merge_flag) {
          __threadfence();
          if (valid_row) {
            const int ns = c_last - c_first + 1;
            const int64_t s0 = (int64_t)c_first + seg.qb;
            float M = -INFINITY;
            for (int s = 0; s < ns; ++s) M = fmaxf(M, lse_out[(s0 + s) * kQBlockRows + r]);
            float den = 0.f;
            if (M != -INFINITY)
              for (int s = 0; s < ns; ++s) den += fast_exp2(lse_out[(s0 + s) * kQBlockRows + r] - M);
            const float dinv = den > 0.f ? 1.f / den : 0.f;
            float4* orow = reinterpret_cast<float4*>(a.o_lat + ((size_t)kHG * seg.t_first + r) * kDc + 256 * half);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              float4 acc[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int s = 0; s < ns; ++s) {
                const float lv = lse_out[(s0 + s) * kQBlockRows + r];
                const float wgt = M == -INFINITY ? 0.f : fast_exp2(lv - M) * dinv;
                const float4* src = reinterpret_cast<const float4*>(
                    o_out + ((size_t)(s0 + s) * kQBlockRows + r) * kDc + 256 * half) + 8 * c;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const float4 xv = src[k];
                  acc[k].x = fmaf(wgt, xv.x, acc[k].x);
                  acc[k].y = fmaf(wgt, xv.y, acc[k].y);
                  acc[k].z = fmaf(wgt, xv.z, acc[k].z);
                  acc[k].w = fmaf(wgt, xv.w, acc[k].w);
                }
              }
#pragma unroll
              for (int k = 0; k < 8; ++k) orow[8 * c + k] = acc[k];
            }
          }
          if (r == 0) arrive[seg.qb * 2 + half] = 0;  // ready for the next launch
        }
        named_bar_sync(kSoftBar, 128);
      }
      seg = nxt;
      have = more;
      ++seg_i;
    }
    if (aborted && r == 0) {
      set_status(status, MLA_DEV_TIMEOUT);
      *abort_flag = 1;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, int32_t batch, const CUtensorMap& cache_map,
                             const CUtensorMap& q_map, cudaStream_t stream) {
  const int smem = Smem::alloc;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_tc_kernel, dim3(a.num_ctas), dim3(kThreads), smem, stream, cache_map,
                    q_map, a, (int)batch);
}

}  // namespace mla
