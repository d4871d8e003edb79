// Attention over the expanded per-head rows on tensor cores, for prefill
// chunks: the pages' version 1 / 2 attention (the cache rows of a head are
// [K_nope (128) | k_rot (64) | V (128)]) computed for 64 query rows of one
// sequence and one head at a time, so each key tile is read once per 64 rows
// instead of once per row. Source: "mini-infer-17: MLA Attention", sections
// "版本 1: MLAAttentionNaive" (q = [q_nope | RoPE(q_pe)], K = [k_nope | k_rot],
// softmax(q K^T * scale) V per head) and "踩坑记录" pitfall 2 (the causal mask
// of a prefill chunk); "07. MLA / Mamba / MoE in vLLM source" 2.3 (paged
// layout, block table).
//
// One CTA per (sequence, 64-row query tile, head). Warp 4 streams 64-token key
// tiles (per page, 5 TMA boxes of 64 columns x block_size rows of the head's
// rows, SWIZZLE_128B: K_nope, K_nope, k_rot, V, V) through a 2-stage ring;
// warps 0-3 each own 16 query rows: S = Q K^T (m16n8k16 warp mma over
// K = 192), their own causal online softmax in base 2 (no exchange between
// warps), then O += P V with P taken from the score registers and V through
// ldmatrix.trans. Rows of a key tile that are not live tokens have their V
// zeroed in shared memory first, so P = 0 never meets garbage. Every wait is
// bounded. 168 registers and 105 KB of shared memory let two
// CTAs share an SM: each scheduler's register partition (16,384) then holds
// its three warps of them.
#include <cuda_bf16.h>

#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"
#include "rope_pairs.cuh"

namespace mla {
namespace {

constexpr int kPfRows = 64;              // query rows per CTA
constexpr int kPfKeys = 64;              // keys per tile
constexpr int kPfSlab = 64 * 128;        // 64 rows x 64 bf16
constexpr int kPfStageSlabs = 5;         // K_nope x2, k_rot, V x2
constexpr int kPfStages = 2;
constexpr int kPfThreads = 160;
constexpr int kPfMathBar = 1;
constexpr int kNaiveRow = kDn + kDr + kDv;  // 320 values per (slot, head)

struct PfSmem {
  static constexpr int stage = 0;
  static constexpr int q = kPfStages * kPfStageSlabs * kPfSlab;  // 3 slabs of Q
  static constexpr int info = q + 3 * kPfSlab;                   // [stages] int2
  static constexpr int bars = info + kPfStages * 8;              // full, empty
  static constexpr int bytes = bars + 2 * kPfStages * 8;
  static constexpr int alloc = bytes + 1024;
};

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

__global__ void __maxnreg__(168)
    naive_prefill_kernel(const __grid_constant__ CUtensorMap kv_map, PfArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + PfSmem::bars);
  uint64_t* empty = full + kPfStages;
  int2* info = reinterpret_cast<int2*>(sm + PfSmem::info);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int bs = a.block_size;
  const int bs_shift = bs == 16 ? 4 : (bs == 32 ? 5 : 6);
  const int ppt = kPfKeys >> bs_shift;

  if (tid == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the cache and the query come from earlier kernels
  pdl_launch_dependents();

  // this CTA's (sequence, query tile): walk the sequences' tile counts
  const int32_t* qsl = a.query_start_loc;
  int b = -1, tile = blockIdx.y;
  for (int s = 0; s < a.batch; ++s) {
    const int ql = qsl[s + 1] - qsl[s];
    const int nt = ql > 0 ? (ql + kPfRows - 1) / kPfRows : 0;
    if (tile < nt) {
      b = s;
      break;
    }
    tile -= nt;
  }
  if (b < 0) return;  // beyond the last tile
  const int q0 = qsl[b], ql = qsl[b + 1] - q0, len = a.seq_lens[b];
  const int r0 = tile * kPfRows;                      // first row of the tile in the sequence
  const int rows = min(kPfRows, ql - r0);             // live rows in the tile
  const bool bad = ql > len || len < 0 ||
                   (int64_t)len > (int64_t)a.max_blocks_per_seq * bs;
  if (bad) {
    if (tid == 0) set_status(a.status, MLA_DEV_BAD_SEQ);
    for (int i = tid; i < rows * (kDv / 8); i += kPfThreads) {
      const int r = i / (kDv / 8), c = i % (kDv / 8);
      *reinterpret_cast<uint4*>(a.out + ((size_t)(q0 + r0 + r) * a.H + h) * kDv + 8 * c) =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }
  // query row r of the tile sits at position pos0 + r and sees tokens 0..pos0 + r
  const int pos0 = len - ql + r0;
  const int kv_end = pos0 + rows;                     // tokens the tile's last row sees
  const int nk = (kv_end + kPfKeys - 1) / kPfKeys;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    prefetch_tensormap(&kv_map);
    const int32_t* bt = a.block_table + (size_t)b * a.max_blocks_per_seq;
    int filled = 0;
    for (int k = 0; k < nk; ++k) {
      const int st = k % kPfStages;
      if (k >= kPfStages && !mbar_wait(&empty[st], ((k / kPfStages) - 1) & 1)) {
        set_status(a.status, MLA_DEV_TIMEOUT);
        break;
      }
      const int t0 = k * kPfKeys;
      const int v = min(kPfKeys, kv_end - t0);
      int okmask = 0;
      uint32_t bytes = 0;
      int blk[4];
      for (int i = 0; i < ppt; ++i) {
        blk[i] = -1;
        if ((i << bs_shift) < v) {
          const int bi = (t0 >> bs_shift) + i;
          const int id = bt[bi];
          if (id >= 0 && id < a.num_blocks) {
            blk[i] = id;
            okmask |= 1 << i;
            bytes += kPfStageSlabs * (uint32_t)bs * 128u;
          } else {
            set_status(a.status, MLA_DEV_BAD_BLOCK);
          }
        }
      }
      info[st] = make_int2(v, okmask);
      mbar_arrive_expect_tx(&full[st], bytes);
      uint8_t* dst = sm + PfSmem::stage + st * kPfStageSlabs * kPfSlab;
      for (int i = 0; i < ppt; ++i) {
        if (okmask & (1 << i)) {
#pragma unroll 1
          for (int c = 0; c < kPfStageSlabs; ++c)
            tma_load_3d(dst + c * kPfSlab + (i << bs_shift) * 128, &kv_map, 64 * c, h,
                        blk[i] << bs_shift, &full[st]);
        }
      }
      filled = k + 1;
    }
    // never leave with copies in flight
    for (int k = filled - kPfStages < 0 ? 0 : filled - kPfStages; k < filled; ++k)
      if (!mbar_wait(&full[k % kPfStages], (k / kPfStages) & 1)) set_status(a.status, MLA_DEV_TIMEOUT);
    return;
  }

  // -------------------------------------------------------------- math warps
  // Q tile: [q_nope | RoPE(q_pe)] of the live rows (zeros elsewhere), three
  // 128-byte-swizzled slabs of 64 columns
  uint8_t* qs = sm + PfSmem::q;
  for (int i = tid; i < kPfRows * 16; i += 128) {
    const int r = i >> 4, ch = i & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows)
      v = *reinterpret_cast<const uint4*>(a.q_nope + ((size_t)(q0 + r0 + r) * a.H + h) * kDn + 8 * ch);
    *reinterpret_cast<uint4*>(qs + (ch >> 3) * kPfSlab + sw128(r, ch & 7)) = v;
  }
  for (int i = tid; i < kPfRows * 32; i += 128) {
    const int r = i >> 5, p = i & 31;
    float y1 = 0.f, y2 = 0.f;
    const int i1 = rope_i1(a.rope_interleaved, p), i2 = rope_i2(a.rope_interleaved, p);
    if (r < rows) {
      const int n = q0 + r0 + r;
      const __nv_bfloat16* x = a.q_pe + ((size_t)n * a.H + h) * kDr;
      const float x1 = __bfloat162float(x[i1]), x2 = __bfloat162float(x[i2]);
      float cs, sn;
      rope_cos_sin(a.q_positions[n], a.freq.hi[p], a.freq.lo[p], &cs, &sn);
      y1 = x1 * cs - x2 * sn;
      y2 = x2 * cs + x1 * sn;
    }
    uint8_t* slab = qs + 2 * kPfSlab;
    *reinterpret_cast<__nv_bfloat16*>(slab + sw128(r, i1 >> 3) + (i1 & 7) * 2) = __float2bfloat16_rn(y1);
    *reinterpret_cast<__nv_bfloat16*>(slab + sw128(r, i2 >> 3) + (i2 & 7) * 2) = __float2bfloat16_rn(y2);
  }
  named_bar_sync(kPfMathBar, 128);

  const int w = warp, g = lane >> 2, q = lane & 3;
  const int qrow = 16 * w + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int krow = (lane & 7) + ((lane >> 4) << 3);
  const int vrow_l = (lane & 7) + (((lane >> 3) & 1) << 3);
  // this lane's two rows (16w + g, 16w + g + 8): last visible token
  const int lim0 = pos0 + 16 * w + g, lim1 = lim0 + 8;
  const bool live0 = 16 * w + g < rows, live1 = 16 * w + g + 8 < rows;
  const float scale = a.scale_log2;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  // a warp whose rows are all past the tile's end still consumes the stages
  bool ok = true;
  for (int k = 0; k < nk; ++k) {
    const int st = k % kPfStages;
    // the four math warps agree (a tile may need their barrier below), so
    // on a timeout all of them leave together
    const bool fok = mbar_wait(&full[st], (k / kPfStages) & 1);
    if (bar_any(kPfMathBar, 128, !fok)) {
      if (tid == 0) set_status(a.status, MLA_DEV_TIMEOUT);
      ok = false;
      break;
    }
    uint8_t* stg = sm + PfSmem::stage + st * kPfStageSlabs * kPfSlab;
    const int2 inf = info[st];
    const int v = inf.x, okmask = inf.y;
    const int t0 = k * kPfKeys;
    if (v < kPfKeys || okmask != (1 << ppt) - 1) {
      // zero V of every row that is not a live token (its K is masked below)
      for (int i = tid; i < kPfKeys * 2 * 8; i += 128) {
        const int r = i >> 4, slab = 3 + ((i >> 3) & 1), ch = i & 7;
        const bool live = r < v && ((okmask >> (r >> bs_shift)) & 1);
        if (!live) *reinterpret_cast<uint4*>(stg + slab * kPfSlab + sw128(r, ch)) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      named_bar_sync(kPfMathBar, 128);
    }

    // ---- S[16 rows x 64 keys] = Q K^T over 192 columns
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 12; ++kk) {
      const int j = kk >> 2, c0 = (kk & 3) * 2;
      uint32_t a0, a1, a2, a3;
      ldsm_x4(smem_u32(qs + j * kPfSlab + sw128(qrow, c0 + (lane >> 4))), a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(stg + j * kPfSlab + sw128(16 * np + krow, c0 + ((lane >> 3) & 1))), b0,
                b1, b2, b3);
        mma_16816(s[2 * np], a0, a1, a2, a3, b0, b1);
        mma_16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    // ---- causal / liveness mask, base-2 scale, running maxima
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tl = 8 * nt + 2 * q + (i & 1), t = t0 + tl;
        const bool kv_ok = tl < v && ((okmask >> (tl >> bs_shift)) & 1);
        const bool vis = (i < 2) ? (live0 && t <= lim0) : (live1 && t <= lim1);
        s[nt][i] = (kv_ok && vis) ? s[nt][i] * scale : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    uint32_t pa[4][4];
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = fast_exp2(s[nt][0] - mu0), p1 = fast_exp2(s[nt][1] - mu0);
      const float p2 = fast_exp2(s[nt][2] - mu1), p3 = fast_exp2(s[nt][3] - mu1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      // n-tiles 2kb, 2kb + 1 are the A fragment of key block kb
      pa[nt >> 1][(nt & 1) * 2] = pack_bf16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= al0; o[nt][1] *= al0;
      o[nt][2] *= al1; o[nt][3] *= al1;
    }
    // ---- O[16 x 128] += P[16 x 64] V[64 x 128]
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      const int vrow = 16 * kb + vrow_l;
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const int slab = 3 + (np >> 2), ch = (np & 3) * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(stg + slab * kPfSlab + sw128(vrow, ch)), b0, b1, b2, b3);
        mma_16816(o[2 * np], pa[kb][0], pa[kb][1], pa[kb][2], pa[kb][3], b0, b1);
        mma_16816(o[2 * np + 1], pa[kb][0], pa[kb][1], pa[kb][2], pa[kb][3], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (!ok) return;
  // ---- normalise and store this warp's live rows (a row that sees no token: zeros)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int r = 16 * w + g + 8 * hf;
    if (r >= rows) continue;
    const float inv = hf ? inv1 : inv0;
    __nv_bfloat16* dst = a.out + ((size_t)(q0 + r0 + r) * a.H + h) * kDv + 2 * q;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<__nv_bfloat162*>(dst + 8 * nt) =
          __floats2bfloat162_rn(o[nt][2 * hf] * inv, o[nt][2 * hf + 1] * inv);
  }
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
  // query tiles: at most one partial tile per sequence beyond num_q / 64
  const int64_t tiles = (num_q + kPfRows - 1) / kPfRows + batch;
  if (tiles > 65535) return MLA_ERR_UNSUPPORTED;  // grid.y
  CUtensorMap kv_map;
  if (!encode_map_heads(&kv_map, kv_cache, kNaiveRow, (uint64_t)H,
                        (uint64_t)num_blocks * cfg->block_size, 64, (uint32_t)cfg->block_size))
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
  cudaError_t e = cudaFuncSetAttribute(naive_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem::alloc);
  if (e == cudaSuccess)
    e = launch_pdl(naive_prefill_kernel, dim3((unsigned)H, (unsigned)tiles), dim3(kPfThreads),
                   PfSmem::alloc, st, kv_map, pa);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
