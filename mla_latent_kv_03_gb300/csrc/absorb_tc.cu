// Query absorption on the tensor cores for many query rows (prefill chunks):
//   q_abs[n, h, 0:512]   = W_uk[h] . q_nope[n, h]      ([512, 128] . [128])
//   q_abs[n, h, 512:576] = RoPE(q_pe[n, h], pos_n)     (rotate-half)
// Sources: "mini-infer-17: MLA Attention", section "版本 3: MLAAttentionAbsorbed"
// (q_nope absorbed through W_uk into the latent space); "07. MLA / Mamba / MoE
// in vLLM source" 2.4 (decoupled RoPE on the shared rope part).
//
// CTA = 128 query rows of one head h and 256 latent columns (blockIdx.y 0 or
// 1; the CTAs of column 0 also do the RoPE part of their rows). Both operands
// arrive by TMA with the 128-byte swizzle: q_nope[rows, h, :] through a 3-D
// map (d, head, row) as 128 K-major rows of 128 dims, and W_uk[h][cols, :] as
// 256 K-major rows. One thread issues 8 tcgen05.mma (M 128, N 256, K 16) into
// a TMEM accumulator; the epilogue stages the bf16 rows in shared memory and
// writes each 512-byte row with one coalesced warp store.
// Every wait is bounded; a CTA that times out writes NaN rows.
#include "async_copy.cuh"
#include "common.cuh"
#include "rope_pairs.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kAbRows = 128;                   // query rows per CTA
constexpr int kAbCols = 256;                   // latent columns per CTA
constexpr int kAbA = kAbRows * 128;            // 16 KB: 128 rows x 64 dims (bf16)
constexpr int kAbB = kAbCols * 128;            // 32 KB: 256 rows x 64 dims
constexpr int kAbThreads = 128;
constexpr uint32_t kAbTmemCols = 256;

struct AbSmem {
  static constexpr int a = 0;                  // [2] d halves of the query rows
  static constexpr int b = a + 2 * kAbA;       // [2] d halves of the weight rows
  static constexpr int bars = b + 2 * kAbB;    // full, done
  static constexpr int misc = bars + 16;       // tmem base
  static constexpr int bytes = misc + 16;
  static constexpr int alloc = bytes + 1024;
};

__global__ void __launch_bounds__(kAbThreads) absorb_tc_kernel(
    const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap w_map,
    const __nv_bfloat16* __restrict__ q_pe, const int32_t* __restrict__ q_pos,
    __nv_bfloat16* __restrict__ q_abs, int num_q, int H, RopeFreq freq, int interleaved) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.z, row0 = blockIdx.x * kAbRows;

  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + AbSmem::bars);
  uint64_t* done = full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + AbSmem::misc);
  const int col0 = blockIdx.y * kAbCols;
  if (tid == 0) {
    mbar_init(full, 1);
    mbar_init(done, 1);
    fence_mbar_init();
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&w_map);
  }
  if (warp == 0) tc::alloc(tmem_slot, kAbTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    mbar_arrive_expect_tx(full, 2 * kAbA + 2 * kAbB);
    // the weights do not depend on earlier kernels; the query does
    for (int kh = 0; kh < 2; ++kh)
      tma_load_2d(sm + AbSmem::b + kh * kAbB, &w_map, 64 * kh, h * kDc + col0, full);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0)
    for (int kh = 0; kh < 2; ++kh) tma_load_3d(sm + AbSmem::a + kh * kAbA, &q_map, 64 * kh, h, row0, full);

  bool ok = true;
  if (warp == 0) {
    ok = __all_sync(0xffffffffu, mbar_wait(full, 0));
    if (ok && tc::elect_one()) {
      tc::fence_after_sync();
      constexpr uint32_t kId = tc::idesc_bf16(kAbRows, kAbCols, false, false);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int kh = kk >> 2, ks = kk & 3;
        const uint64_t ad = tc::smem_desc(smem_u32(sm + AbSmem::a + kh * kAbA) + 32 * ks, 16, 1024,
                                          tc::kSwizzle128);
        const uint64_t bd = tc::smem_desc(smem_u32(sm + AbSmem::b + kh * kAbB) + 32 * ks, 16, 1024,
                                          tc::kSwizzle128);
        tc::mma_bf16(tmem, ad, bd, kId, kk > 0);
      }
      tc::commit(done);
    }
    __syncwarp();
  }
  // every copy and MMA must land before TMEM is read or freed
  const bool okf = __syncthreads_and(mbar_wait(done, 0) && ok) != 0;
  if (!okf && tid == 0) mbar_wait(full, 0);
  tc::fence_after_sync();
  // TMEM row (thread) -> bf16 row r of a 128 x 512-byte staging area in the
  // operand buffers (free now), 16-byte chunks XOR-swizzled by r % 32
  const int r = tid;
  uint8_t* stg = sm;
  if (okf) {
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int cb = 0; cb < kAbCols / 32; ++cb) {
      uint32_t v[32];
      tc::ld32(trow + 32 * cb, v);
      tc::wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(stg + r * 512 + (((4 * cb + q) ^ (r & 31)) << 4)) = make_uint4(
            pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
            pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
            pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
            pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  // warp w writes rows w, w + 4, ...: one 512-byte row per store instruction
#pragma unroll 1
  for (int rr = warp; rr < kAbRows; rr += 4) {
    const int n = row0 + rr;
    if (n >= num_q) break;
    uint4* dst = reinterpret_cast<uint4*>(q_abs + ((size_t)n * H + h) * kRow + col0);
    dst[lane] = okf ? *reinterpret_cast<const uint4*>(stg + rr * 512 + ((lane ^ (rr & 31)) << 4))
                    : make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
  }
  if (blockIdx.y == 0) {
    // rotate-half RoPE of q_pe into q_abs[..., 512:576] for this CTA's rows
    // (warp w: rows w + 4 i; lane: pair p), eight rows' loads in flight at a time
    const int p = lane, i1 = rope_i1(interleaved, p), i2 = rope_i2(interleaved, p);
    const float fhi = freq.hi[p], flo = freq.lo[p];
#pragma unroll 1
    for (int rb = warp; rb < kAbRows; rb += 32) {
      float x1[8], x2[8];
      int pos[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int n = row0 + rb + 4 * u;
        const bool ok = n < num_q;
        const __nv_bfloat16* x = q_pe + ((size_t)(ok ? n : 0) * H + h) * kDr;
        x1[u] = ok ? __bfloat162float(x[i1]) : 0.f;
        x2[u] = ok ? __bfloat162float(x[i2]) : 0.f;
        pos[u] = ok ? q_pos[n] : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int n = row0 + rb + 4 * u;
        if (n >= num_q) continue;
        float cs, sn;
        rope_cos_sin(pos[u], fhi, flo, &cs, &sn);
        __nv_bfloat16* o = q_abs + ((size_t)n * H + h) * kRow + kDc;
        o[i1] = __float2bfloat16_rn(x1[u] * cs - x2[u] * sn);
        o[i2] = __float2bfloat16_rn(x2[u] * cs + x1[u] * sn);
      }
    }
  }
  tc::fence_after_sync();
  if (warp == 0) tc::dealloc(tmem, kAbTmemCols);
}

}  // namespace

cudaError_t launch_absorb_tc(const CUtensorMap& q_map, const CUtensorMap& w_map,
                             const mla_config& cfg, const void* q_pe, const int32_t* q_positions,
                             void* q_abs, int64_t num_q, cudaStream_t stream) {
  const int smem = AbSmem::alloc;
  cudaError_t e = cudaFuncSetAttribute(absorb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  const RopeFreq freq = make_rope_freq((double)cfg.rope_base);
  return launch_pdl(absorb_tc_kernel,
                    dim3((unsigned)((num_q + kAbRows - 1) / kAbRows), 2, cfg.num_heads),
                    dim3(kAbThreads), smem, stream, q_map, w_map, (const __nv_bfloat16*)q_pe,
                    q_positions, (__nv_bfloat16*)q_abs, (int)num_q, cfg.num_heads, freq,
                    cfg.rope_interleaved);
}

}  // namespace mla
