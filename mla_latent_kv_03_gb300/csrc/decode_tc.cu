// Tensor-core (tcgen05 / TMEM) split-KV latent attention for tiles of 128
// (query row, head) rows: 128 heads of one query row, or 8 query rows x 16
// heads of a prefill chunk (any H with 8 * 16 / H rows). Sources: "mini-infer-17:
// MLA Attention", sections "版本 3: MLAAttentionAbsorbed" (scores and output
// against the latent rows) and "设计取舍" (the nope and rope score parts summed
// before a hand-written softmax); "07. MLA / Mamba / MoE in vLLM source" 2.3
// (paged layout).
//
// Work units are (q-block, 64-token tile); each equal share of the unit list
// is processed by a cluster of two CTAs. CTA h of the pair owns cache columns
// [256h, 256h + 256 + 64h) -- 256 latent columns for h = 0, 256 latent plus
// the 64 rope columns for h = 1 -- and the same query columns:
//   S_h = Q[:, cols_h] . K[:, cols_h]^T   (partial scores, K = 256 or 320)
//   S   = S_0 + S_1                       (each CTA sends its partial to the
//                                           peer's shared memory ahead of use)
//   O_h += P . V[:, 256h : 256h + 256]    (each CTA half of the output)
// so each CTA streams only its own columns of every cache row, and both CTAs
// run the same softmax on the same sums (each partial is rounded to f16 with
// saturation before the exchange, and S_0 + S_1 == S_1 + S_0 in fp32),
// giving identical probabilities and log-sum-exps.
//
// TMEM (512 columns): O half [0, 256), two score buffers [256, 320), two
// probability buffers [320, 352) (bf16 pairs), this CTA's query columns
// [352, 512) (bf16 pairs, the A operand of the score MMAs). Shared memory: a
// ring of seven 32-token cache stages of this CTA's columns (SWIZZLE_128B slabs
// of 64 columns), four buffers of the peer's partial scores, four of this
// CTA's own (the source of the bulk copies to the peer), and merge weights.
// Per CTA (384 threads):
//   warp 0 (TMA producer): cache stages under full / empty mbarriers; every
//     block id is bounds-checked.
//   warp 1 (P.V issuer; owns the TMEM allocation): O += P . V per stage
//     (2 tcgen05.mma, M 128, N 256, K 16, A = P in TMEM, V MN-major).
//   warp 2 (score issuer): the partial scores of a stage as soon as its score
//     buffer is free (16 or 20 tcgen05.mma, M 128, N 32, K 16, A from TMEM).
//   warps 8-11 (senders): each stage's partial scores from TMEM to a staging
//     buffer and, by one bulk copy per warp (its 32 rows), into the peer's
//     shared memory, up to three stages ahead of their use.
//   warps 4-7 (softmax): thread r owns row r. Per stage it adds the peer's
//     partial scores to its own, masks (sequence end, causal position,
//     rejected blocks), keeps the running maximum, rescales the warp's O rows
//     in TMEM only when some row's maximum grows by more than 2^8
//     (probabilities stay below 256), and stores bf16 P to TMEM. At the end of
//     a segment it normalises its O row: straight into o_lat when the q-block
//     lies in this share and the merge is fused, else into the partial buffer,
//     and the last CTA of a split q-block's half merges the parts while they
//     are in L2.
// The MMA warps issue from one elected lane. Every wait is bounded; on a
// timeout the roles leave their loops, the MMA warps wait for their last
// MMAs and the producer for its copies before TMEM is freed, and the pair
// meets at a final cluster barrier so neither exits while the other may still
// write into its shared memory.
#include "async_copy.cuh"
#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"
#include "pair_math.cuh"
#include "merge.cuh"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kTok = 32;                       // tokens per stage
constexpr int kSlab = kTok * 128;              // 32 rows x 64 bf16 columns
constexpr int kMaxSlabs = 5;                   // column slabs of one CTA (64 columns each)
constexpr int kStage = kMaxSlabs * kSlab;      // 20 KB
constexpr int kStages = 7;                     // cache stages in the ring
constexpr int kXRecv = 4;                      // buffers of the peer's partial scores
constexpr int kXSend = 4;                      // buffers of this CTA's partial scores
constexpr int kThreads = 384;
constexpr int kSoftWarp0 = 4;                  // warps 4-7: softmax
constexpr int kSendWarp0 = 8;                  // warps 8-11: partial-score senders
constexpr int kSoftBar = 2;                    // named barrier of the softmax warps
constexpr uint32_t kOCol = 0, kSCol = 256, kPCol = 320, kQCol = 352, kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;            // lazy rescale threshold (2^8)
constexpr int kXRow = kTok * 2;                // one row of a stage's partial scores (f16)
constexpr int kXBytes = kQBlockRows * kXRow;   // one stage of partial scores
constexpr int kXWarpBytes = kXBytes / 4;       // the 32 rows of one sender warp
constexpr int kMergeSlots = 16;                // parts merged by the one-pass merge
static_assert(kQCol + 32 * kMaxSlabs <= kTmemCols, "TMEM budget");

enum {
  kFull0 = 0,
  kEmpty0 = kFull0 + kStages,
  kSFull0 = kEmpty0 + kStages,   // [2] partial scores of stage i in S[i % 2]
  kSFree0 = kSFull0 + 2,         // [2] S[i % 2] read out by the senders (128 arrivals)
  kXFull0 = kSFull0 + 4,         // [kXRecv] the peer's partial scores (bytes from the peer)
  kPFull0 = kXFull0 + kXRecv,    // [2] probabilities of stage i in P[i % 2] (128 arrivals)
  kPVDone0 = kPFull0 + 2,        // [2] O += P[i % 2] . V_i done
  kPeerFree0 = kPVDone0 + 2,     // [kXRecv] the peer's softmax read its buffer (1 remote arrival)
  kXsFull0 = kPeerFree0 + kXRecv,// [kXSend] own partial scores staged (128 arrivals)
  kXsFree0 = kXsFull0 + kXSend,  // [kXSend] own staged partial read by the softmax
  kQtReady = kXsFree0 + kXSend,  // query columns stored in TMEM (128 arrivals)
  kQEmpty,                       // every score MMA of the segment done
  kODone,                        // every P.V MMA of the segment done
  kOFree,                        // O read out by the epilogue (128 arrivals)
  kFinalS,                       // the score warp's last MMAs done
  kFinalP,                       // the P.V warp's last MMAs done
  kNumBars
};

struct Smem {
  static constexpr int stage = 0;
  static constexpr int x = stage + kStages * kStage;           // [kXRecv] peer partial scores
  static constexpr int xs = x + kXRecv * kXBytes;              // [kXSend] own partial scores
  static constexpr int w = xs + kXSend * kXBytes;              // merge weights [16][128]
  static constexpr int info = w + kMergeSlots * kQBlockRows * 4;  // [kStages] int2
  static constexpr int bars = info + kStages * 8;
  static constexpr int misc = bars + kNumBars * 8;             // tmem base, abort flag, merge flag
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

// Two scores (low, high) rounded to f16, saturating at +-65,504 (never inf).
__device__ __forceinline__ uint32_t pack_f16_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The fp32 sums of the low and of the high halves of two f16 pairs (each sum
// exact up to one fp32 rounding, and the same whichever pair comes first).
__device__ __forceinline__ void add_f16x2_f32(uint32_t a, uint32_t c, float& lo, float& hi) {
  asm("{\n\t.reg .b16 al, ah, cl, ch;\n\t.reg .f32 t0, t1;\n\t"
      "mov.b32 {al, ah}, %2;\n\tmov.b32 {cl, ch}, %3;\n\t"
      "cvt.f32.f16 t0, cl;\n\tcvt.f32.f16 t1, ch;\n\t"
      "add.rn.f32.f16 %0, al, t0;\n\tadd.rn.f32.f16 %1, ah, t1;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(a), "r"(c));
}

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

// Four barriers polled together (their latencies overlap); parity 2 means
// "no wait". All are waited with the default CTA-scope acquire: the peer's
// partial scores land by bulk copy with complete_tx on this CTA's own
// barrier, whose phase completion makes the copied bytes visible here.
__device__ __forceinline__ bool wait4_or_abort(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1,
                                               uint64_t* b2, uint32_t p2, uint64_t* b3, uint32_t p3,
                                               volatile int* abort_flag) {
  auto poll = [&]() {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred q0, q1, q2, q3;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
        "and.pred q0, q0, q1;\n\tand.pred q2, q2, q3;\n\tand.pred q0, q0, q2;\n\t"
        "selp.u32 %0, 1, 0, q0;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1), "r"(smem_u32(b2)), "r"(p2 & 1),
          "r"(smem_u32(b3)), "r"(p3 & 1)
        : "memory");
    return done != 0;
  };
  // a barrier that needs no wait is replaced by a copy of the second
  if (p2 > 1) b2 = b1, p2 = p1;
  if (p3 > 1) b3 = b1, p3 = p1;
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (poll()) return true;
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

// This CTA's query columns [col0, col0 + 8 * nvec) of q-block row `qrow` into
// its TMEM lane (rows past the last query row are zero). Warp-collective.
template <int NVEC>
__device__ __forceinline__ void load_q_tmem(const uint16_t* q_abs, int64_t qrow, int64_t qrows,
                                            int col0, uint32_t taddr) {
  static_assert(NVEC % 8 == 0, "whole x16 stores per batch");
  const uint4* src = reinterpret_cast<const uint4*>(q_abs + (size_t)qrow * kRow + col0);
  const bool live = qrow < qrows;
  constexpr int kHalf = NVEC / 2;   // vectors per batch (registers)
#pragma unroll
  for (int hb = 0; hb < 2; ++hb) {
    uint4 buf[kHalf];
    if (live) {
#pragma unroll
      for (int i = 0; i < kHalf; ++i) buf[i] = __ldg(src + kHalf * hb + i);
    } else {
#pragma unroll
      for (int i = 0; i < kHalf; ++i) buf[i] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < kHalf / 4; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[4 * k] = buf[4 * c + k].x;
        w[4 * k + 1] = buf[4 * c + k].y;
        w[4 * k + 2] = buf[4 * c + k].z;
        w[4 * k + 3] = buf[4 * c + k].w;
      }
      tc::st16(taddr + kQCol + 4 * kHalf * hb + 16 * c, w);
    }
  }
}

__device__ __forceinline__ void load_q_cta(int h, const uint16_t* q_abs, int64_t qrow,
                                           int64_t qrows, uint32_t trow) {
  if (h == 0)
    load_q_tmem<32>(q_abs, qrow, qrows, 0, trow);      // columns [0, 256)
  else
    load_q_tmem<40>(q_abs, qrow, qrows, 256, trow);    // columns [256, 576)
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap cache_map,
                     const __grid_constant__ CUtensorMap slab4,
                     const __grid_constant__ CUtensorMap slab5, DecodeArgs a, int batch) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::bars);
  int2* info = reinterpret_cast<int2*>(sm + Smem::info);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Smem::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Smem::misc + 4);
  int* merge_flag = reinterpret_cast<int*>(sm + Smem::misc + 8);
  uint8_t* sStage = sm + Smem::stage;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = (int)cl::rank();                    // column half of this CTA
  const int share_idx = blockIdx.x >> 1;
  const int slab0 = 4 * h, nslab = 4 + h;          // cache column slabs [slab0, slab0 + nslab)
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
  uint32_t* status = &reinterpret_cast<WsHeader*>(ws)->status;
  const int bs = a.block_size;
  const int bsr = bs < kTok ? bs : kTok;            // rows of one TMA box
  const int bsr_shift = bsr == 16 ? 4 : 5;
  const int ppst = kTok / bsr;                      // boxes (pages or half pages) per stage
  const int full_mask = (1 << ppst) - 1;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool many = (i >= kSFree0 && i < kSFree0 + 2) || (i >= kPFull0 && i < kPFull0 + 2) ||
                        (i >= kXsFull0 && i < kXsFull0 + kXSend) || i == kQtReady || i == kOFree;
      mbar_init(&bars[i], many ? 128 : 1);
    }
    // the peer's partial scores of the first kXRecv stages are expected
    for (int i = 0; i < kXRecv; ++i) mbar_arrive_expect_tx(&bars[kXFull0 + i], kXBytes);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(tmem_slot, kTmemCols);
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&cache_map);
    prefetch_tensormap(h ? &slab5 : &slab4);
  }
  tc::fence_before_sync();
  cl::sync();  // both CTAs' barriers exist before either copies into the other
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the plan and q_abs come from earlier kernels
  pdl_launch_dependents();

  TcWalker sw;
  const bool has_work = sw.init(ws, a.num_q, a.groups, a.num_ctas, batch, share_idx);
  if (a.o_lat && warp >= kSoftWarp0 && warp < kSendWarp0 && h == 0)
    zero_unvisited_rows(sw.row_info, sw.plan_ok, a.num_q, a.num_heads, a.o_lat, tid - 128, 128);
  TcSeg seg;
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
  };

  if (has_work && warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the stages; lane 0 issues the copies. Block ids
    // come from the block table 32 at a time (one per lane, handed out by
    // shuffles), so a stage never waits on a dependent global load.
    const uint64_t policy = l2_evict_first_policy();  // the cache is read once per step
    int stage_i = 0;
    bool ok = true;
    while (ok && sw.next(seg)) {
      const int32_t* bt = a.block_table + (size_t)seg.b * a.max_blocks_per_seq;
      const int n = seg_stages(seg);
      int cache_base = -(1 << 30), cached = -1;   // lane l holds bt[cache_base + l]
#pragma unroll 1
      for (int t = 0; t < n; ++t) {
        const int tstart = seg.k0 * kTile + t * kTok;
        const int v = min(kTok, seg.vis - tstart);
        const int slot = stage_i % kStages;
        int blk[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          blk[i] = -1;
          if (i < ppst && (i << bsr_shift) < v) {   // warp-uniform
            const int bi = (tstart + (i << bsr_shift)) / bs;
            if (bi - cache_base >= 32 || bi < cache_base) {
              cache_base = bi;
              cached = bi + lane < a.max_blocks_per_seq ? bt[bi + lane] : -1;
            }
            blk[i] = __shfl_sync(0xffffffffu, cached, bi - cache_base);
          }
        }
        if (stage_i >= kStages &&
            !__all_sync(0xffffffffu, wait_or_abort(&bars[kEmpty0 + slot],
                                                  ((stage_i / kStages) - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          int okmask = 0, nload = 0;
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
          mbar_arrive_expect_tx(&bars[kFull0 + slot], (uint32_t)(nload * nslab * bsr * 128));
          uint8_t* dst = sStage + slot * kStage;
          if (ppst == 1) {
            // one copy: this CTA's column slabs of the 32-row box (3-D view)
            if (okmask & 1)
              tma_load_3d_hint(dst, h ? &slab5 : &slab4, 0, blk[0] * bs + (tstart % bs), slab0,
                               &bars[kFull0 + slot], policy);
          } else {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if (okmask & (1 << i)) {
                const int tok = tstart + (i << bsr_shift);
                const int y = blk[i] * bs + (tok % bs);
#pragma unroll 1
                for (int j = 0; j < nslab; ++j)
                  tma_load_2d_hint(dst + j * kSlab + (i << bsr_shift) * 128, &cache_map,
                                   64 * (slab0 + j), y, &bars[kFull0 + slot], policy);
              }
            }
          }
        }
        __syncwarp();
        ++stage_i;
      }
    }
    if (lane == 0) {
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
    }
    __syncwarp();
  } else if (has_work && warp == 1) {
    // ------------------------------------------------------ P.V issuer
    constexpr uint32_t kIdO = tc::idesc_bf16(128, 256, false, true);
    // V: this CTA's first four slabs of the stage, MN-major
    const uint64_t vdesc = tc::smem_desc(smem_u32(sStage), kSlab, 1024, tc::kSwizzle128);
    const bool leader = tc::elect_one();
    int stage_i = 0, seg_i = 0;
    bool ok = true;
    while (ok && sw.next(seg)) {
      const int n = seg_stages(seg);
#pragma unroll 1
      for (int t = 0; t < n; ++t) {
        const int i = stage_i + t, slot = i % kStages;
        if (!warp_wait(&bars[kPFull0 + (i & 1)], (i >> 1) & 1)) { ok = false; break; }
        if (t == 0 && seg_i > 0 && !warp_wait(&bars[kOFree], (seg_i - 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            tc::mma_bf16_tmem_a(tmem + kOCol, tmem + kPCol + (uint32_t)((i & 1) * 16 + ks * 8),
                                vdesc + (uint64_t)((slot * kStage + ks * 16 * 128) >> 4), kIdO,
                                !(t == 0 && ks == 0));
          tc::commit(&bars[kEmpty0 + slot]);
          tc::commit(&bars[kPVDone0 + (i & 1)]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) tc::commit(&bars[kODone]);
      __syncwarp();
      stage_i += n;
      ++seg_i;
    }
    if (!ok && leader) {
      set_status(status, MLA_DEV_TIMEOUT);
      *abort_flag = 1;
    }
    // every MMA issued so far must finish before TMEM is freed
    if (leader) tc::commit(&bars[kFinalP]);
    __syncwarp();
    if (!mbar_wait(&bars[kFinalP], 0) && leader) set_status(status, MLA_DEV_TIMEOUT);
    __syncwarp();
  } else if (has_work && warp == 2) {
    // ----------------------------------------------------- score issuer
    constexpr uint32_t kIdS = tc::idesc_bf16(128, kTok, false, false);
    const uint64_t kdesc = tc::smem_desc(smem_u32(sStage), 16, 1024, tc::kSwizzle128);
    const bool leader = tc::elect_one();
    const int ksteps = 4 * nslab;
    int stage_i = 0, seg_i = 0;
    bool ok = true;
    while (ok && sw.next(seg)) {
      const int n = seg_stages(seg);
      if (!warp_wait(&bars[kQtReady], seg_i & 1)) { ok = false; break; }
      tc::fence_after_sync();
#pragma unroll 1
      for (int t = 0; t < n; ++t) {
        const int i = stage_i + t, slot = i % kStages;
        // S[i % 2] was read out (stage i - 2) and the stage has landed
        if (i >= 2 && !warp_wait(&bars[kSFree0 + (i & 1)], ((i - 2) >> 1) & 1)) { ok = false; break; }
        if (!warp_wait(&bars[kFull0 + slot], (i / kStages) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        if (leader) {
          const uint32_t d = tmem + kSCol + (uint32_t)(i & 1) * kTok;
#pragma unroll
          for (int kk = 0; kk < 4 * kMaxSlabs; ++kk) {
            if (kk < ksteps) {
              const int j = kk >> 2, c = kk & 3;
              tc::mma_bf16_tmem_a(d, tmem + kQCol + (uint32_t)(j * 32 + c * 8),
                                  kdesc + (uint64_t)((slot * kStage + j * kSlab + c * 32) >> 4),
                                  kIdS, kk > 0);
            }
          }
          tc::commit(&bars[kSFull0 + (i & 1)]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) tc::commit(&bars[kQEmpty]);  // the query may be replaced
      __syncwarp();
      stage_i += n;
      ++seg_i;
    }
    if (!ok && leader) {
      set_status(status, MLA_DEV_TIMEOUT);
      *abort_flag = 1;
    }
    if (leader) tc::commit(&bars[kFinalS]);
    __syncwarp();
    if (!mbar_wait(&bars[kFinalS], 0) && leader) set_status(status, MLA_DEV_TIMEOUT);
    __syncwarp();
  } else if (has_work && warp >= kSendWarp0) {
    // ------------------------------------------------------------ senders
    // Partial scores of every stage, in order: TMEM -> f16 -> own staging
    // buffer j % kXSend, which this CTA's softmax reads, and from which each
    // warp's bulk copy moves its 32 rows into the peer's buffer j % kXRecv,
    // counted on the peer's barrier. The score buffer is free as soon as the
    // senders have read it, so the next scores never wait for the softmax.
    const int r = tid - kSendWarp0 * 32;
    const int wl = warp - kSendWarp0;                  // rows [32 wl, 32 wl + 32)
    const uint32_t trow = tmem + ((uint32_t)(wl * 32) << 16);
    const uint32_t peer = (uint32_t)(h ^ 1);
    const uint32_t x_peer0 = cl::map(smem_u32(sm + Smem::x), peer) + (uint32_t)wl * kXWarpBytes;
    const uint32_t xbar_peer0 = cl::map(smem_u32(&bars[kXFull0]), peer);
    const uint32_t xs_src0 = smem_u32(sm + Smem::xs) + (uint32_t)wl * kXWarpBytes;
    const int sw4 = (r >> 1) & 3;                      // 16-byte chunk swizzle of row r
    int stage_i = 0;
    bool aborted = false;
    while (!aborted && sw.next(seg)) {
      const int n = seg_stages(seg);
#pragma unroll 1
      for (int tt = 0; tt < n; ++tt) {
        const int j = stage_i + tt, b = j & 1, xs = j % kXSend, xr = j % kXRecv;
        if (!__all_sync(0xffffffffu, wait_or_abort(&bars[kSFull0 + b], (j >> 1) & 1, abort_flag))) {
          aborted = true;
          break;
        }
        tc::fence_after_sync();
        uint32_t sv[32];
        tc::ld32(trow + kSCol + (uint32_t)b * kTok, sv);
        tc::wait_ld();
        tc::fence_before_sync();
        mbar_arrive(&bars[kSFree0 + b]);   // S[j % 2] may take stage j + 2's scores
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) pk[k] = pack_f16_sat(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]));
        // staging buffer xs: this CTA's softmax has read stage j - kXSend from
        // it, and this warp's copy of that stage has read its rows
        const bool okf = j < kXSend ||
                         wait_or_abort(&bars[kXsFree0 + xs], ((j - kXSend) / kXSend) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, okf)) { aborted = true; break; }
        if (lane == 0) cl::bulk_wait_read<kXSend - 1>();
        __syncwarp();
        uint8_t* dst = sm + Smem::xs + xs * kXBytes + r * kXRow;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(dst + ((k ^ sw4) << 4)) =
              make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        fence_proxy_async_smem();
        mbar_arrive(&bars[kXsFull0 + xs]);
        __syncwarp();
        int sent = 1;
        if (lane == 0) {
          // the peer's softmax has read its buffer for stage j - kXRecv
          if (j < kXRecv ||
              wait_or_abort(&bars[kPeerFree0 + xr], ((j - kXRecv) / kXRecv) & 1, abort_flag)) {
            cl::bulk_to_peer(x_peer0 + (uint32_t)xr * kXBytes,
                             xs_src0 + (uint32_t)xs * kXBytes, kXWarpBytes,
                             xbar_peer0 + (uint32_t)xr * 8);
            cl::bulk_commit();
          } else {
            sent = 0;
          }
        }
        if (__shfl_sync(0xffffffffu, sent, 0) == 0) { aborted = true; break; }
      }
      stage_i += n;
    }
    if (aborted && lane == 0) {
      set_status(status, MLA_DEV_TIMEOUT);
      *abort_flag = 1;
    }
    if (lane == 0) cl::bulk_wait_read<0>();   // no copy still reads the staging buffers
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
    const uint32_t peer = (uint32_t)(h ^ 1);
    const uint32_t pfree_peer0 = cl::map(smem_u32(&bars[kPeerFree0]), peer);
    float* wsm = reinterpret_cast<float*>(sm + Smem::w);
    int stage_i = 0, seg_i = 0;
    bool aborted = false, fail = false;
    // After an agreement over all 128 threads at stage i, every thread has
    // finished with stage i - 1: its receive buffer is free for the peer
    // (re-armed for stage i - 1 + kXRecv), its staging buffer for the senders.
    auto release_prev = [&](int i) {
      if (r == 0 && i >= 1) {
        const int p = i - 1;
        mbar_arrive(&bars[kXsFree0 + p % kXSend]);
        mbar_arrive_expect_tx(&bars[kXFull0 + p % kXRecv], kXBytes);
        // relaxed: the loads of stage i - 1's buffer returned long ago (their
        // sums fed that stage's softmax), and a release here would stall
        cl::arrive_remote_relaxed(pfree_peer0 + (uint32_t)(p % kXRecv) * 8);
      }
    };
    bool have = sw.next(seg);
    if (have) {
      load_q_cta(h, q_abs, (int64_t)kHG * seg.t_first + r, qrows, trow);
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
        const int i = stage_i + tt, slot = i % kStages, b = i & 1, xb = i % kXRecv, xsb = i % kXSend;
        // the peer's partial scores of stage i, this CTA's (staged by the
        // senders), the stage (for its info), and P[i % 2] free (P.V of stage i - 2)
        const bool okw = wait4_or_abort(&bars[kXFull0 + xb], (i / kXRecv) & 1,
                                        &bars[kXsFull0 + xsb], (i / kXSend) & 1,
                                        &bars[kFull0 + slot], (i / kStages) & 1,
                                        &bars[kPVDone0 + b], i >= 2 ? ((i - 2) >> 1) & 1 : 2u,
                                        abort_flag);
        if (soft_red_or(!okw || fail)) { aborted = true; break; }
        release_prev(i);
        const int tstart = seg.k0 * kTile + tt * kTok;
        const int2 inf = info[slot];
        const int v = inf.x, okmask = inf.y;
        // live tokens: a prefix (sequence end, causal position) minus rejected blocks
        const int lim = min(v, pos - tstart + 1);
        // S = own partial + the peer's partial, both as the senders rounded
        // them to f16 (so both CTAs add the same two values, in fp32), read
        // from the staging and receive buffers (16-byte chunks swizzled by
        // the row)
        float x[32];
        {
          const int sw4 = (r >> 1) & 3;
          const uint8_t* xp = sm + Smem::x + xb * kXBytes + r * kXRow;
          const uint8_t* op = sm + Smem::xs + xsb * kXBytes + r * kXRow;
          uint4 pv[4], ov[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            pv[k] = *reinterpret_cast<const uint4*>(xp + ((k ^ sw4) << 4));
            ov[k] = *reinterpret_cast<const uint4*>(op + ((k ^ sw4) << 4));
          }
          auto add2 = [&](int j, uint32_t a, uint32_t c) { add_f16x2_f32(a, c, x[j], x[j + 1]); };
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            add2(8 * k, ov[k].x, pv[k].x);
            add2(8 * k + 2, ov[k].y, pv[k].y);
            add2(8 * k + 4, ov[k].z, pv[k].z);
            add2(8 * k + 6, ov[k].w, pv[k].w);
          }
        }
        if (!(lim >= kTok && okmask == full_mask)) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const bool live = j < lim && ((okmask >> (j >> bsr_shift)) & 1);
            if (!live) x[j] = -INFINITY;
          }
        }
        // the row maximum in 16 three-input maxima (32 -> 12 -> 4 -> 2 -> 1)
        float m12[12];
#pragma unroll
        for (int j = 0; j < 10; ++j) m12[j] = fmax3(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
        m12[10] = x[30];
        m12[11] = x[31];
        const float mxr = fmaxf(fmax3(fmax3(m12[0], m12[1], m12[2]), fmax3(m12[3], m12[4], m12[5]), m12[6]),
                                fmax3(fmax3(m12[7], m12[8], m12[9]), m12[10], m12[11]));
        const float m_cand = mxr * scale;   // scale > 0
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
          const bool okp = __all_sync(
              0xffffffffu, wait_or_abort(&bars[kPVDone0 + ((i - 1) & 1)], ((i - 1) >> 1) & 1, abort_flag));
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
        // exponentials in pairs: the scale on the packed fp32 pipe, the sum as
        // packed partial sums
        float2 p[16];
        const float2 sc2 = make_float2(scale, scale), mn2 = make_float2(mneg, mneg);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 e = fma_f32x2(make_float2(x[2 * j], x[2 * j + 1]), sc2, mn2);
          p[j] = make_float2(fast_exp2(e.x), fast_exp2(e.y));
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16(p[j].x, p[j].y);
        tc::st16(trow + kPCol + (uint32_t)b * 16, pk);
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) p[j] = add_f32x2(p[j], p[j + w]);
        l += p[0].x + p[0].y;
        if (v < kTok || okmask != full_mask) {
          // cache rows past the sequence's last token or in a rejected block may
          // hold anything (NaN): zero the latent columns so P = 0 stays 0
          uint8_t* stg = sStage + slot * kStage;
          for (int e = r; e < kTok * 4 * 8; e += 128) {
            const int row = e >> 5, sl = (e >> 3) & 3, ch = e & 7;
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
      // the next segment's query columns, while this one's last products
      // finish (its scores are all done once QEmpty completes)
      TcSeg nxt;
      const bool more_seg = sw.next(nxt);
      if (more_seg) {
        const bool okq = wait_or_abort(&bars[kQEmpty], seg_i & 1, abort_flag);
        if (soft_red_or(!okq || fail)) { aborted = true; break; }
        tc::fence_after_sync();
        load_q_cta(h, q_abs, (int64_t)kHG * nxt.t_first + r, qrows, trow);
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&bars[kQtReady]);
      }
      // ---- epilogue: normalise this CTA's half of the O row
      const bool okd = wait_or_abort(&bars[kODone], seg_i & 1, abort_flag);
      if (soft_red_or(!okd || fail)) { aborted = true; break; }
      tc::fence_after_sync();
      const int c_first = seg.ustart / sw.share;
      const int c_last = (seg.ustart + seg.tiles - 1) / sw.share;
      const bool direct = a.o_lat != nullptr && c_first == c_last;   // the q-block is this share's alone
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t slot = (int64_t)share_idx + seg.qb;
      float4* dst;
      if (direct)
        dst = reinterpret_cast<float4*>(a.o_lat + ((size_t)kHG * seg.t_first + r) * kDc + 256 * h);
      else
        dst = reinterpret_cast<float4*>(o_out + ((size_t)slot * kQBlockRows + r) * kDc + 256 * h);
      const bool store = !direct || valid_row;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        tc::ld32(trow + kOCol + 32 * c, o);
        tc::wait_ld();
        if (store) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[8 * c + k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                         __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
        }
      }
      // both CTAs of the pair see the same scores and write the same lse
      if (!direct) lse_out[slot * kQBlockRows + r] = l > 0.f ? m_used + log2f(l) : -INFINITY;
      tc::fence_before_sync();
      mbar_arrive(&bars[kOFree]);
      if (a.o_lat != nullptr && !direct) {
        // count this part (fence per writing thread, barrier, acquire-release
        // count: count_arrival); the last part of this half merges the
        // q-block, reading the parts through L2 after the second barrier
        __threadfence();
        named_bar_sync(kSoftBar, 128);
        if (r == 0) *merge_flag = count_arrival(&arrive[seg.qb * 2 + h]) == c_last - c_first;
        named_bar_sync(kSoftBar, 128);
        if (*merge_flag) {
          const int ns = c_last - c_first + 1;
          const int64_t s0 = (int64_t)c_first + seg.qb;
          // row r's max lse and 1 / weight sum over its parts
          float M = -INFINITY;
          for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(lse_out + (s0 + s) * kQBlockRows + r));
          float den = 0.f;
          if (M != -INFINITY)
            for (int s = 0; s < ns; ++s) den += fast_exp2(__ldcg(lse_out + (s0 + s) * kQBlockRows + r) - M);
          const float dinv = den > 0.f ? 1.f / den : 0.f;
          const int rows_valid = min(kQBlockRows, (seg.t_end - seg.t_first) * kHG);
          const float4* op4 = reinterpret_cast<const float4*>(o_out) + 64 * h;
          float4* ol4 = reinterpret_cast<float4*>(a.o_lat + (size_t)kHG * seg.t_first * kDc) + 64 * h;
          if (ns <= kMergeSlots) {
            // weights w[s][row] to shared memory, then rows 2k + (tid / 64) with
            // float4 column tid % 64 of the half: coalesced, 16 rows per pass
            for (int s = 0; s < ns; ++s)
              wsm[s * kQBlockRows + r] =
                  M == -INFINITY ? 0.f : fast_exp2(__ldcg(lse_out + (s0 + s) * kQBlockRows + r) - M) * dinv;
            named_bar_sync(kSoftBar, 128);
            const int c4 = r & 63, rsub = r >> 6;
#pragma unroll 1
            for (int k0 = 0; k0 < kQBlockRows / 2; k0 += 16) {
              float4 acc[16];
#pragma unroll
              for (int u = 0; u < 16; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
              for (int s = 0; s < ns; ++s) {
                const float4* src = op4 + (size_t)(s0 + s) * kQBlockRows * (kDc / 4) + c4;
                float4 vv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) vv[u] = __ldcg(src + (size_t)(rsub + 2 * (k0 + u)) * (kDc / 4));
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                  const float wgt = wsm[s * kQBlockRows + rsub + 2 * (k0 + u)];
                  acc[u].x = fmaf(wgt, vv[u].x, acc[u].x);
                  acc[u].y = fmaf(wgt, vv[u].y, acc[u].y);
                  acc[u].z = fmaf(wgt, vv[u].z, acc[u].z);
                  acc[u].w = fmaf(wgt, vv[u].w, acc[u].w);
                }
              }
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const int row = rsub + 2 * (k0 + u);
                if (row < rows_valid) ol4[(size_t)row * (kDc / 4) + c4] = acc[u];
              }
            }
            named_bar_sync(kSoftBar, 128);   // the weights may be overwritten after this
          } else if (valid_row) {
            // many parts (tiny shares): row r by thread r
#pragma unroll 1
            for (int c = 0; c < 64; ++c) {
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int s = 0; s < ns; ++s) {
                const float wgt = M == -INFINITY ? 0.f : fast_exp2(__ldcg(lse_out + (s0 + s) * kQBlockRows + r) - M) * dinv;
                const float4 xv = __ldcg(op4 + ((size_t)(s0 + s) * kQBlockRows + r) * (kDc / 4) + c);
                acc.x = fmaf(wgt, xv.x, acc.x);
                acc.y = fmaf(wgt, xv.y, acc.y);
                acc.z = fmaf(wgt, xv.z, acc.z);
                acc.w = fmaf(wgt, xv.w, acc.w);
              }
              ol4[(size_t)r * (kDc / 4) + c] = acc;
            }
          }
          if (r == 0) arrive[seg.qb * 2 + h] = 0;  // ready for the next launch
        }
        named_bar_sync(kSoftBar, 128);
      }
      seg = nxt;
      have = more_seg;
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
  cl::sync();  // the peer no longer writes into this CTA's shared memory
}

}  // namespace

int decode_tc_max_clusters() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Smem::alloc) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = Smem::alloc;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &lc) != cudaSuccess) return 0;
  cached[dev] = n;
  return n;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, int32_t batch, const CUtensorMap& cache_map,
                             const CUtensorMap& slab4, const CUtensorMap& slab5,
                             cudaStream_t stream) {
  const int smem = Smem::alloc;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_tc_kernel, dim3(a.num_ctas), dim3(kThreads), smem, stream, cache_map,
                    slab4, slab5, a, (int)batch);
}

}  // namespace mla
