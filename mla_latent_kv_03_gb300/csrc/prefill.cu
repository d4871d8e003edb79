// Attention over the expanded per-head rows on tcgen05 tensor cores, for
// prefill chunks: the pages' version 1 / 2 attention (the cache rows of a head
// are [K_nope (128) | k_rot (64) | V (128)]) computed for 128 query rows of one
// sequence and one head at a time, so each key tile is read once per 128 rows
// instead of once per row. Source: "mini-infer-17: MLA Attention", sections
// "版本 1: MLAAttentionNaive" (q = [q_nope | RoPE(q_pe)], K = [k_nope | k_rot],
// softmax(q K^T * scale) V per head) and "踩坑记录" pitfall 2 (the causal mask
// of a prefill chunk); "07. MLA / Mamba / MoE in vLLM source" 2.3 (paged
// layout, block table).
//
// One CTA per (sequence, head, 128-row query tile), numbered with the tile
// fastest, so the tiles that read the same keys run side by side and share
// them in L2. TMEM (512 columns): O [0, 128) fp32; two score buffers
// S[b] [128 + 64 b, 192 + 64 b) fp32 of 64 keys; two probability buffers
// P[b] [256 + 32 b, 288 + 32 b) as bf16 pairs; the query tile [320, 416) as
// bf16 pairs (the A operand of the score MMAs). Per CTA (384 threads):
//   warp 0 (TMA producer): 64-key stages of the head's rows (per page, 5 boxes
//     of 64 columns x block_size rows: K_nope, K_nope, k_rot, V, V;
//     SWIZZLE_128B) through a 5-stage ring; every block id is bounds-checked.
//   warp 1 (score issuer; owns the TMEM allocation): S[j % 2] = Q K_j^T
//     (12 tcgen05.mma, M 128, N 64, K 16, A from TMEM) as soon as the stage
//     has landed and the buffer was read, up to two stages ahead.
//   warp 2 (product issuer): O += P[j % 2] V_j (4 tcgen05.mma, M 128, N 128,
//     K 16, A = P from TMEM, V MN-major) as soon as the probabilities are in.
//   warps 4-7 and 8-11 (softmax, two warpgroups on alternate stages): thread r
//     of either warpgroup owns query row r. Causal mask, base-2 online softmax
//     with the running maximum handed from stage to stage in shared memory
//     (published per warp on an mbarrier), O rescaled in TMEM only when a row's
//     maximum grows by more than 2^8, bf16 P to TMEM. Each warpgroup keeps its
//     own sum; the two meet at the end, and each warpgroup normalises and
//     stores half of the O columns.
// Rows of a key tile that are not live tokens (past the tile's last visible
// token, or in a rejected block) have their V zeroed in shared memory before
// the product, so P = 0 never meets garbage. Every wait is bounded; on a
// timeout the roles leave their loops, the MMA warp waits for its last MMAs
// and the producer for its copies before TMEM is freed.
#include <cuda_bf16.h>

#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"
#include "pair_math.cuh"
#include "rope_pairs.cuh"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kPtRows = 128;                       // query rows per CTA (TMEM lanes)
constexpr int kPtKeys = 64;                        // keys per stage
constexpr int kPtSlab = kPtKeys * 128;             // 64 rows x 64 bf16 = 8 KB
constexpr int kPtStageSlabs = 5;                   // K_nope x2, k_rot, V x2
constexpr int kPtStage = kPtStageSlabs * kPtSlab;  // 40 KB
constexpr int kPtStages = 5;
constexpr int kPtThreads = 384;
constexpr int kPtSoft0 = 4;                        // warps 4-7, 8-11: softmax warpgroups
constexpr int kPtBarAll = 3;                       // named barrier 3: both softmax warpgroups
constexpr uint32_t kTO = 0, kTS = 128, kTP = 256, kTQ = 320, kTCols = 512;
constexpr float kPtRescaleLog2 = 8.f;
constexpr int kNaiveRow = kDn + kDr + kDv;         // 320 values per (slot, head)

enum {
  kPtFull0 = 0,                    // [5] stage landed (TMA bytes)
  kPtEmpty0 = kPtFull0 + kPtStages,  // [5] scores and products of the stage done
  kPtSFull0 = kPtEmpty0 + kPtStages, // [2] S[b] computed
  kPtSFree0 = kPtSFull0 + 2,       // [2] S[b] read by its warpgroup (128 arrivals)
  kPtPFull0 = kPtSFree0 + 2,       // [2] P[b] stored (128 arrivals)
  kPtPVDone0 = kPtPFull0 + 2,      // [2] O += P[b] V done
  kPtQReady = kPtPVDone0 + 2,      // query tile in TMEM (256 arrivals)
  kPtODone,                        // every product done
  kPtFinal,                        // the score warp's last MMAs done
  kPtFinalP,                       // the product warp's last MMAs done
  kPtMReady0,                      // [2] stage j's row maxima published (4 warps), j % 2
  kPtNumBars = kPtMReady0 + 2
};

struct PtSmem {
  static constexpr int stage = 0;
  static constexpr int mrow = stage + kPtStages * kPtStage;   // [128] running maxima
  static constexpr int lx = mrow + kPtRows * 4;               // [2][128] sums
  static constexpr int info = lx + 2 * kPtRows * 4;           // [stages] int2
  static constexpr int bars = info + kPtStages * 8;
  static constexpr int misc = bars + kPtNumBars * 8;          // tmem base, abort flag
  static constexpr int bytes = misc + 16;
  static constexpr int alloc = bytes + 1024;
};
static_assert(PtSmem::alloc <= 227 * 1024, "shared memory budget");
static_assert(PtSmem::bars % 8 == 0, "mbarrier alignment");

struct PfArgs {
  const __nv_bfloat16* q_nope;
  const __nv_bfloat16* q_pe;
  const int32_t* q_positions;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int64_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t H;
  int32_t batch;
  float scale_log2;
  RopeFreq freq;
  int32_t rope_interleaved;
  __nv_bfloat16* out;
  uint32_t* status;
};

// OR of v over the nthreads threads that reach named barrier id.
__device__ __forceinline__ bool bar_any(int id, int nthreads, bool v) {
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

// bounded wait that also gives up when another role has aborted
__device__ __forceinline__ bool pt_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
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

__global__ void __launch_bounds__(kPtThreads, 1)
    naive_prefill_tc_kernel(const __grid_constant__ CUtensorMap kv_map,
                            const __grid_constant__ CUtensorMap slab_map, PfArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PtSmem::bars);
  int2* info = reinterpret_cast<int2*>(sm + PtSmem::info);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PtSmem::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + PtSmem::misc + 4);
  float* mrow = reinterpret_cast<float*>(sm + PtSmem::mrow);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bs = a.block_size;
  const int bs_shift = bs == 16 ? 4 : (bs == 32 ? 5 : 6);
  const int ppt = kPtKeys >> bs_shift;               // pages per stage

  if (tid == 0) {
    for (int i = 0; i < kPtNumBars; ++i) {
      const bool wg = (i >= kPtSFree0 && i < kPtSFree0 + 2) || (i >= kPtPFull0 && i < kPtPFull0 + 2);
      mbar_init(&bars[i], i == kPtQReady ? 256 : wg ? 128 : i >= kPtMReady0 ? 4 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(tmem_slot, kTCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the cache rows and the query come from earlier kernels
  pdl_launch_dependents();

  // this CTA's (sequence, head, query tile), the tile fastest
  const int32_t* qsl = a.query_start_loc;
  int b = -1, h = 0, tile = 0;
  {
    int u = blockIdx.x;
    for (int s = 0; s < a.batch; ++s) {
      const int ql = qsl[s + 1] - qsl[s];
      const int nt = ql > 0 ? (ql + kPtRows - 1) / kPtRows : 0;
      if (u < nt * a.H) {
        b = s;
        h = u / nt;
        tile = u % nt;
        break;
      }
      u -= nt * a.H;
    }
  }
  int q0 = 0, rows = 0, pos0 = 0, nk = 0;
  bool run = b >= 0;
  if (run) {
    q0 = qsl[b];
    const int ql = qsl[b + 1] - q0, len = a.seq_lens[b];
    const int r0 = tile * kPtRows;
    q0 += r0;                                       // first query row of the tile
    rows = min(kPtRows, ql - r0);                   // live rows in the tile
    const bool bad = ql > len || len < 0 || (int64_t)len > (int64_t)a.max_blocks_per_seq * bs;
    if (bad) {
      if (tid == 0) set_status(a.status, MLA_DEV_BAD_SEQ);
      for (int i = tid; i < rows * (kDv / 8); i += kPtThreads) {
        const int r = i / (kDv / 8), c = i % (kDv / 8);
        *reinterpret_cast<uint4*>(a.out + ((size_t)(q0 + r) * a.H + h) * kDv + 8 * c) =
            make_uint4(0, 0, 0, 0);
      }
      run = false;
    } else {
      // query row r of the tile sits at position pos0 + r, sees tokens 0..pos0 + r
      pos0 = len - ql + r0;
      nk = (pos0 + rows + kPtKeys - 1) / kPtKeys;
    }
  }
  const int kv_end = pos0 + rows;                   // tokens the tile's last row sees

  if (run && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      if (ppt == 1) prefetch_tensormap(&slab_map);
      const int32_t* bt = a.block_table + (size_t)b * a.max_blocks_per_seq;
      int filled = 0;
      bool ok = true;
      for (int k = 0; k < nk && ok; ++k) {
        const int st = k % kPtStages;
        if (k >= kPtStages && !pt_wait(&bars[kPtEmpty0 + st], ((k / kPtStages) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int t0 = k * kPtKeys;
        const int v = min(kPtKeys, kv_end - t0);
        int okmask = 0;
        uint32_t bytes = 0;
        int blk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          blk[i] = -1;
          if (i < ppt && (i << bs_shift) < v) {
            const int id = bt[(t0 >> bs_shift) + i];
            if (id >= 0 && id < a.num_blocks) {
              blk[i] = id;
              okmask |= 1 << i;
              bytes += kPtStageSlabs * (uint32_t)bs * 128u;
            } else {
              set_status(a.status, MLA_DEV_BAD_BLOCK);
            }
          }
        }
        info[st] = make_int2(v, okmask);
        mbar_arrive_expect_tx(&bars[kPtFull0 + st], bytes);
        uint8_t* dst = sm + PtSmem::stage + st * kPtStage;
        if (ppt == 1) {
          // a 64-token page: the head's five column slabs in one copy (4-D view)
          if (okmask & 1) tma_load_4d(dst, &slab_map, 0, blk[0] << bs_shift, 0, h, &bars[kPtFull0 + st]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (okmask & (1 << i)) {
#pragma unroll 1
              for (int c = 0; c < kPtStageSlabs; ++c)
                tma_load_3d(dst + c * kPtSlab + (i << bs_shift) * 128, &kv_map, 64 * c, h,
                            blk[i] << bs_shift, &bars[kPtFull0 + st]);
            }
          }
        }
        filled = k + 1;
      }
      if (!ok) {
        set_status(a.status, MLA_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      // never leave with copies in flight
      for (int k = filled - kPtStages < 0 ? 0 : filled - kPtStages; k < filled; ++k)
        if (!mbar_wait(&bars[kPtFull0 + k % kPtStages], (k / kPtStages) & 1))
          set_status(a.status, MLA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (run && warp == 1) {
    // ------------------------------------------------------------ score issuer
    // S[j % 2] = Q K_j^T once the stage has landed and S[j % 2] was read (up
    // to two stages ahead of the softmax)
    constexpr uint32_t kIdS = tc::idesc_bf16(128, kPtKeys, false, false);
    const uint64_t kdesc = tc::smem_desc(smem_u32(sm + PtSmem::stage), 16, 1024, tc::kSwizzle128);
    const bool leader = tc::elect_one();
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, pt_wait(bar, parity, abort_flag));
    };
    bool ok = warp_wait(&bars[kPtQReady], 0);
    for (int j = 0; ok && j < nk; ++j) {
      const int st = j % kPtStages, sb = j & 1;
      if (!warp_wait(&bars[kPtFull0 + st], (j / kPtStages) & 1)) { ok = false; break; }
      if (j >= 2 && !warp_wait(&bars[kPtSFree0 + sb], ((j - 2) >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      if (leader) {
        // descriptors advance by constant steps: 32 bytes (2 units) per K=16
        // step inside a slab, kPtSlab between slabs
        const uint64_t kd = kdesc + (uint64_t)((st * kPtStage) >> 4);
        const uint32_t d = tmem + kTS + 64 * sb;
#pragma unroll
        for (int kk = 0; kk < 12; ++kk)
          tc::mma_bf16_tmem_a(d, tmem + kTQ + 8 * kk,
                              kd + (uint64_t)((((kk >> 2) * kPtSlab) >> 4) + 2 * (kk & 3)), kIdS,
                              kk > 0);
        tc::commit(&bars[kPtSFull0 + sb]);
      }
      __syncwarp();
    }
    if (leader) {
      if (!ok) {
        set_status(a.status, MLA_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      tc::commit(&bars[kPtFinal]);   // every MMA issued so far must finish before TMEM is freed
    }
    __syncwarp();
    if (!mbar_wait(&bars[kPtFinal], 0) && leader) set_status(a.status, MLA_DEV_TIMEOUT);
    __syncwarp();
  } else if (run && warp == 2) {
    // ------------------------------------------------------------ product issuer
    // O += P[j % 2] V_j once its probabilities are stored; the stage is then
    // free (its scores completed before the softmax could read them)
    constexpr uint32_t kIdO = tc::idesc_bf16(128, kDv, false, true);
    const uint64_t vdesc = tc::smem_desc(smem_u32(sm + PtSmem::stage), kPtSlab, 1024, tc::kSwizzle128);
    const bool leader = tc::elect_one();
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      const int st = j % kPtStages, pb = j & 1;
      if (!__all_sync(0xffffffffu, pt_wait(&bars[kPtPFull0 + pb], (j >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (leader) {
#pragma unroll
        for (int ks = 0; ks < kPtKeys / 16; ++ks)
          tc::mma_bf16_tmem_a(tmem + kTO, tmem + kTP + 32 * pb + 8 * ks,
                              vdesc + (uint64_t)((st * kPtStage + 3 * kPtSlab + ks * 16 * 128) >> 4),
                              kIdO, !(j == 0 && ks == 0));
        tc::commit(&bars[kPtEmpty0 + st]);
        tc::commit(&bars[kPtPVDone0 + pb]);
      }
      __syncwarp();
    }
    if (leader) {
      if (ok) {
        tc::commit(&bars[kPtODone]);
      } else {
        set_status(a.status, MLA_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      tc::commit(&bars[kPtFinalP]);
    }
    __syncwarp();
    if (!mbar_wait(&bars[kPtFinalP], 0) && leader) set_status(a.status, MLA_DEV_TIMEOUT);
    __syncwarp();
  } else if (run && warp >= kPtSoft0) {
    // ------------------------------------------------------------ softmax
    const int wg = (warp - kPtSoft0) >> 2;            // 0: even stages, 1: odd stages
    const int wq = warp & 3;
    const int r = 32 * wq + lane;                      // query row of the tile
    const int wt = tid - (kPtSoft0 + 4 * wg) * 32;     // thread of the warpgroup
    const uint32_t trow = tmem + ((uint32_t)(32 * wq) << 16);
    const bool live_row = r < rows;
    const int n = q0 + r;                              // query row index (when live)
    const int lim = pos0 + r;                          // last token this row sees
    const float scale = a.scale_log2;
    float* lx = reinterpret_cast<float*>(sm + PtSmem::lx);
    bool aborted = false, fail = false;
    // ---- the query tile into TMEM: q_nope by warpgroup 0, RoPE(q_pe) by 1
    if (wg == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(a.q_nope + ((size_t)n * a.H + h) * kDn);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w16[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = live_row ? __ldg(src + 4 * c + k) : make_uint4(0, 0, 0, 0);
          w16[4 * k] = v.x;
          w16[4 * k + 1] = v.y;
          w16[4 * k + 2] = v.z;
          w16[4 * k + 3] = v.w;
        }
        tc::st16(trow + kTQ + 16 * c, w16);
      }
    } else {
      float y[kDr];
#pragma unroll
      for (int i = 0; i < kDr; ++i) y[i] = 0.f;
      if (live_row) {
        const __nv_bfloat16* x = a.q_pe + ((size_t)n * a.H + h) * kDr;
        const int qpos = a.q_positions[n];
#pragma unroll
        for (int p = 0; p < 32; ++p) {
          const int i1 = rope_i1(a.rope_interleaved, p), i2 = rope_i2(a.rope_interleaved, p);
          const float x1 = __bfloat162float(x[i1]), x2 = __bfloat162float(x[i2]);
          float cs, sn;
          rope_cos_sin(qpos, a.freq.hi[p], a.freq.lo[p], &cs, &sn);
          const float y1 = x1 * cs - x2 * sn, y2 = x2 * cs + x1 * sn;
          if (a.rope_interleaved) {
            y[2 * p] = y1;
            y[2 * p + 1] = y2;
          } else {
            y[p] = y1;
            y[p + 32] = y2;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w16[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) w16[k] = pack_bf16(y[32 * c + 2 * k], y[32 * c + 2 * k + 1]);
        tc::st16(trow + kTQ + 64 + 16 * c, w16);
      }
    }
    tc::wait_st();
    tc::fence_before_sync();
    mbar_arrive(&bars[kPtQReady]);

    // the maximum published for stage j (bounded wait; NaN on a timeout)
    auto wait_m = [&](int j) -> float {
      if (!pt_wait(&bars[kPtMReady0 + (j & 1)], (j >> 1) & 1, abort_flag))
        return __int_as_float(0x7fc00000);
      return mrow[r];
    };
    float m_w = -INFINITY, l = 0.f;   // this warpgroup's reference maximum and sum
#pragma unroll 1
    for (int j = wg; j < nk; j += 2) {
      const int st = j % kPtStages, sb = j & 1;
      const bool okw = pt_wait(&bars[kPtSFull0 + sb], (j >> 1) & 1, abort_flag);
      // a warp that gives up raises the abort flag; the other warps' bounded
      // waits see it and leave too, and all meet at the barrier after the loop
      if (__any_sync(0xffffffffu, !okw || fail)) {
        aborted = true;
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      float x[kPtKeys];
      {
        uint32_t s0[32], s1[32];
        tc::ld32(trow + kTS + 64 * sb, s0);
        tc::ld32(trow + kTS + 64 * sb + 32, s1);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(s0[c]);
          x[32 + c] = __uint_as_float(s1[c]);
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&bars[kPtSFree0 + sb]);            // S[j % 2] may take stage j + 2
      const int t0 = j * kPtKeys;
      const int2 inf = info[st];
      const int v = inf.x, okmask = inf.y;
      const bool full_tile = v == kPtKeys && okmask == (1 << ppt) - 1;
      // live keys of this row: a prefix (its causal position, the sequence
      // end) minus rejected blocks; rows past the tile's end see nothing
      const int vis = live_row ? min(v, lim - t0 + 1) : 0;
      if (!(full_tile && vis >= kPtKeys)) {
#pragma unroll
        for (int c = 0; c < kPtKeys; ++c) {
          const bool keep = c < vis && ((okmask >> (c >> bs_shift)) & 1);
          if (!keep) x[c] = -INFINITY;
        }
      }
      // the row maximum in 32 three-input maxima (64 -> 22 -> 8 -> 3 -> 1)
      float m22[22], m8[8];
#pragma unroll
      for (int c = 0; c < 21; ++c) m22[c] = fmax3(x[3 * c], x[3 * c + 1], x[3 * c + 2]);
      m22[21] = x[63];
#pragma unroll
      for (int c = 0; c < 7; ++c) m8[c] = fmax3(m22[3 * c], m22[3 * c + 1], m22[3 * c + 2]);
      m8[7] = m22[21];
      const float mxr = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      const float m_cand = mxr * scale;               // scale > 0
      const float m_prev = j > 0 ? wait_m(j - 1) : -INFINITY;
      if (m_prev != m_prev) fail = true;               // NaN: the wait gave up
      float m_new = m_prev, alpha = 1.f;
      bool rescale_o = false;
      if (m_cand > m_prev + kPtRescaleLog2 || (m_prev == -INFINITY && m_cand != -INFINITY)) {
        m_new = m_cand;
        if (m_prev != -INFINITY) {
          alpha = fast_exp2(m_prev - m_new);
          rescale_o = true;
        }
      }
      mrow[r] = m_new;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kPtMReady0 + (j & 1)]);
      if (m_new != m_w) {
        l *= fast_exp2(m_w - m_new);                   // 0 while m_w is -inf (l is 0 then)
        m_w = m_new;
      }
      if (__any_sync(0xffffffffu, rescale_o)) {
        // this warp's O rows: the previous O += P V must have landed
        const bool okp = __all_sync(
            0xffffffffu, pt_wait(&bars[kPtPVDone0 + ((j - 1) & 1)], ((j - 1) >> 1) & 1, abort_flag));
        if (okp) {
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < kDv / 32; ++c) {
            uint32_t o[32];
            tc::ld32(trow + kTO + 32 * c, o);
            tc::wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tc::st32(trow + kTO + 32 * c, o);
          }
        } else {
          fail = true;
        }
      }
      const float mneg = m_new == -INFINITY ? 0.f : -m_new;
      float ps = 0.f;
      {
        uint32_t pk[32];
        float2 acc = make_float2(0.f, 0.f);
        const float2 sc2 = make_float2(scale, scale), mn2 = make_float2(mneg, mneg);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 e = fma_f32x2(make_float2(x[2 * c], x[2 * c + 1]), sc2, mn2);
          const float2 p = make_float2(fast_exp2(e.x), fast_exp2(e.y));
          acc = add_f32x2(acc, p);
          pk[c] = pack_bf16(p.x, p.y);
        }
        ps = acc.x + acc.y;
        // P[j % 2] is free once the product of stage j - 2 is done
        if (j >= 2 &&
            !__all_sync(0xffffffffu, pt_wait(&bars[kPtPVDone0 + sb], ((j - 2) >> 1) & 1, abort_flag)))
          fail = true;
        tc::fence_after_sync();
        tc::st32(trow + kTP + 32 * sb, pk);
      }
      l += ps;
      if (!full_tile) {
        // key rows that are not live tokens may hold anything (NaN): zero
        // their V so that P = 0 stays 0
        uint8_t* stg = sm + PtSmem::stage + st * kPtStage;
        for (int e = wt; e < kPtKeys * 2 * 8; e += 128) {
          const int row = e >> 4, slab = 3 + ((e >> 3) & 1), ch = e & 7;
          const bool live = row < v && ((okmask >> (row >> bs_shift)) & 1);
          if (!live) *reinterpret_cast<uint4*>(stg + slab * kPtSlab + sw128(row, ch)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars[kPtPFull0 + sb]);
    }
    // ---- the row's sum over both warpgroups relative to the final maximum,
    // then half of the O row (columns [64 wg, 64 wg + 64)) normalised to bf16
    if (bar_any(kPtBarAll, 256, aborted || fail)) {
      aborted = true;
      *abort_flag = 1;
    } else {
      // (the last stage's warpgroup wrote mrow before the barrier above)
      const float m_fin = nk > 0 ? mrow[r] : -INFINITY;
      lx[wg * kPtRows + r] = m_w == -INFINITY ? 0.f : l * fast_exp2(m_w - m_fin);
      const bool okd = pt_wait(&bars[kPtODone], 0, abort_flag);
      if (bar_any(kPtBarAll, 256, !okd || fail)) {
        aborted = true;
        *abort_flag = 1;
      } else {
        tc::fence_after_sync();
        const float l_tot = lx[r] + lx[kPtRows + r];
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        uint32_t o[32];
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)n * a.H + h) * kDv + 64 * wg);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tc::ld32(trow + kTO + 64 * wg + 32 * c, o);
          tc::wait_ld();
          if (live_row) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[4 * c + k] = make_uint4(
                  pack_bf16(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                  pack_bf16(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                  pack_bf16(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                  pack_bf16(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
          }
        }
      }
    }
    if (aborted && wt == 0) set_status(a.status, MLA_DEV_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::dealloc(tmem, kTCols);
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

mla_status mla_naive_prefill(const mla_config* cfg, const void* q_nope, const void* q_pe,
                             const int32_t* q_positions, const void* kv_cache, int64_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, const int32_t* query_start_loc,
                             int32_t batch, int64_t num_q, void* workspace, size_t ws_bytes,
                             void* out, void* stream) {
  mla_status s = validate_config(cfg);
  if (s != MLA_OK) return s;
  if (cfg->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (num_q < 0 || batch < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > 0x7fffffff || num_blocks * cfg->block_size > ((int64_t)1 << 31) / cfg->num_heads)
    return MLA_ERR_UNSUPPORTED;
  auto aligned = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; };
  if (!workspace || !aligned(workspace, 256) || ws_bytes < 256) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!q_nope || !q_pe || !q_positions || !kv_cache || !block_table || !seq_lens ||
      !query_start_loc || !out || batch == 0 || num_blocks == 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
      !aligned(q_positions, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(query_start_loc, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  const int H = cfg->num_heads;
  // (sequence, head, 128-row tile) units: at most one partial tile per
  // sequence beyond num_q / 128
  const int64_t units = ((num_q + kPtRows - 1) / kPtRows + batch) * H;
  if (units > 0x7fffffff) return MLA_ERR_UNSUPPORTED;
  CUtensorMap kv_map;
  if (!encode_map_heads(&kv_map, kv_cache, kNaiveRow, (uint64_t)H,
                        (uint64_t)num_blocks * cfg->block_size, 64, (uint32_t)cfg->block_size))
    return MLA_ERR_CUDA;
  // 64-token pages: one copy per page and stage through the 4-D view
  CUtensorMap slab_map = kv_map;
  if (cfg->block_size == kPtKeys &&
      !encode_map_heads_slabs(&slab_map, kv_cache, kNaiveRow, (uint64_t)H,
                              (uint64_t)num_blocks * cfg->block_size, kPtKeys))
    return MLA_ERR_CUDA;
  PfArgs pa{};
  pa.q_nope = reinterpret_cast<const __nv_bfloat16*>(q_nope);
  pa.q_pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  pa.q_positions = q_positions;
  pa.block_table = block_table;
  pa.seq_lens = seq_lens;
  pa.query_start_loc = query_start_loc;
  pa.num_blocks = num_blocks;
  pa.max_blocks_per_seq = max_blocks_per_seq;
  pa.block_size = cfg->block_size;
  pa.H = H;
  pa.batch = batch;
  pa.scale_log2 = (float)(cfg->softmax_scale * 1.4426950408889634);
  pa.freq = make_rope_freq((double)cfg->rope_base);
  pa.rope_interleaved = cfg->rope_interleaved;
  pa.out = reinterpret_cast<__nv_bfloat16*>(out);
  pa.status = reinterpret_cast<uint32_t*>(workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaFuncSetAttribute(naive_prefill_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, PtSmem::alloc);
  if (e == cudaSuccess)
    e = launch_pdl(naive_prefill_tc_kernel, dim3((unsigned)units), dim3(kPtThreads), PtSmem::alloc,
                   st, kv_map, slab_map, pa);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
