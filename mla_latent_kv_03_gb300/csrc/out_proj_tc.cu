// Output projection on the tensor cores for many query rows (prefill chunks):
//   out[n, h, :] = o_lat[n, h, :] . W_uv[h]      ([512] . [512, 128])
// Source: "mini-infer-17: MLA Attention", section "版本 3: MLAAttentionAbsorbed"
// (W_uv applied once to the latent output instead of to every cached row).
//
// CTA = 128 query rows of one head h, all 128 output columns; K = 512 in 8
// chunks of 64. Per chunk the CTA's 256 threads (two per row) read their fp32
// o_lat slices -- two chunks ahead -- round them to bf16 and store them
// K-major with the 128-byte swizzle; the W_uv chunks (64 k-rows x 128
// columns, MN-major) arrive by TMA into four stages, issued two chunks ahead.
// One elected thread issues 4 tcgen05.mma (M 128, N 128, K 16) per chunk into
// a TMEM accumulator; two A stages let the conversion of chunk c + 1 overlap
// the MMAs of chunk c. The epilogue reads the rows from TMEM and writes bf16.
// Every wait is bounded; on a timeout the CTA waits (bounded) for its last
// MMAs and writes NaN rows instead of a result, so the failure is visible.
#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kOpRows = 128;                   // query rows per CTA
constexpr int kOpKC = 64;                      // latent dims per chunk
constexpr int kOpChunks = kDc / kOpKC;         // 8
constexpr int kOpA = kOpRows * kOpKC * 2;      // 16 KB: 128 rows x 128 B (bf16)
constexpr int kOpBSlab = kOpKC * 128;          // 8 KB: 64 k-rows x 64 columns
constexpr int kOpB = 2 * kOpBSlab;             // 16 KB: 64 k-rows x 128 columns
constexpr int kOpAStages = 2, kOpBStages = 4;
constexpr int kOpThreads = 256;                // two threads per row
constexpr uint32_t kOpTmemCols = 128;

struct OpSmem {
  static constexpr int a = 0;                                  // [2] A chunks
  static constexpr int b = a + kOpAStages * kOpA;              // [4] W chunks
  static constexpr int bars = b + kOpBStages * kOpB;           // bfull[4], done[2], final
  static constexpr int misc = bars + (kOpBStages + 3) * 8;     // tmem base
  static constexpr int bytes = misc + 16;
  static constexpr int alloc = bytes + 1024;
};

__global__ void __launch_bounds__(kOpThreads) out_proj_tc_kernel(
    const __grid_constant__ CUtensorMap w_map, const float* __restrict__ o_lat,
    __nv_bfloat16* __restrict__ out, int num_q, int H) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bfull = reinterpret_cast<uint64_t*>(sm + OpSmem::bars);
  uint64_t* done = bfull + kOpBStages;
  uint64_t* fin = done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OpSmem::misc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, row0 = blockIdx.x * kOpRows;
  const int wrow = h * kDc;                    // first W_uv row of head h in the map

  if (tid == 0) {
    for (int i = 0; i < kOpBStages + 3; ++i) mbar_init(&bfull[i], 1);
    fence_mbar_init();
    prefetch_tensormap(&w_map);
  }
  if (warp == 0) tc::alloc(tmem_slot, kOpTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int w_issued = 0;              // thread 0: W chunks issued so far
  auto issue_w = [&](int c) {   // W chunk c into stage c % 4
    w_issued = c + 1;
    uint64_t* bar = &bfull[c % kOpBStages];
    mbar_arrive_expect_tx(bar, kOpB);
    for (int sl = 0; sl < 2; ++sl)
      tma_load_2d(sm + OpSmem::b + (c % kOpBStages) * kOpB + sl * kOpBSlab, &w_map, 64 * sl,
                  wrow + kOpKC * c, bar);
  };
  // the weights do not depend on earlier kernels: their first four chunks go out now
  if (tid == 0)
    for (int c = 0; c < kOpBStages; ++c) issue_w(c);
  pdl_wait();  // o_lat comes from earlier kernels
  pdl_launch_dependents();

  constexpr uint32_t kId = tc::idesc_bf16(kOpRows, 128, false, true);
  // Loads are coalesced: item u of thread t is float4 q = (256 u + t) % 16 of
  // chunk row R = (256 u + t) / 16, so 16 lanes read one row's 256 bytes.
  const int qv = tid & 15;                     // float4 within the row's chunk
  const float4* srcu[8];
  bool liveu[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int R = (256 * u + tid) >> 4;
    liveu[u] = row0 + R < num_q;
    srcu[u] = reinterpret_cast<const float4*>(o_lat + ((size_t)(row0 + R) * H + h) * kDc) + qv;
  }
  float4 pre0[8], pre1[8];                     // chunks c (even) and c + 1 in flight
  auto fetch = [&](int c, float4 (&v)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = liveu[u] ? srcu[u][16 * c] : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  // the epilogue's thread: row r of the CTA, column half hf
  const int r = (warp & 3) * 32 + lane, hf = warp >> 2;
  const bool live = row0 + r < num_q;
  fetch(0, pre0);
  fetch(1, pre1);
  bool ok = true;
  // one chunk: convert the prefetched slice, refill it two chunks ahead, MMA
  auto chunk = [&](int c, float4 (&pre)[8]) -> bool {
    const int sa = c & 1;
    float4 cur[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = pre[i];
    if (c + 2 < kOpChunks) fetch(c + 2, pre);
    // A stage sa is free once chunk c - 2's MMAs are done; so is W stage
    // (c + 2) % 4, which then takes chunk c + 2
    if (c >= 2) {
      ok = ok && mbar_wait(&done[sa], ((c - 2) >> 1) & 1);
      if (tid == 0 && ok && c + 2 < kOpChunks) {
        tc::fence_after_sync();
        issue_w(c + 2);
      }
    }
    // float4 q of row R -> bf16 at byte 8 q of the 128-byte row, 16-byte
    // chunks XOR-swizzled by the row
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int R = (256 * u + tid) >> 4;
      uint8_t* arow = sm + OpSmem::a + sa * kOpA + R * 128;
      *reinterpret_cast<uint2*>(arow + (((qv >> 1) ^ (R & 7)) << 4) + (qv & 1) * 8) =
          make_uint2(pack_bf16(cur[u].x, cur[u].y), pack_bf16(cur[u].z, cur[u].w));
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    // a failed wait anywhere ends every thread's loop at the same barrier
    if (!__syncthreads_and(ok)) return false;
    if (warp == 0) {
      const bool okb =
          __all_sync(0xffffffffu, mbar_wait(&bfull[c % kOpBStages], (c / kOpBStages) & 1));
      if (!okb) ok = false;                    // seen by all at the next barrier
      if (okb && tc::elect_one()) {
        tc::fence_after_sync();
        const uint64_t adesc = tc::smem_desc(smem_u32(sm + OpSmem::a + sa * kOpA), 16, 1024,
                                             tc::kSwizzle128);
        const uint64_t bdesc = tc::smem_desc(
            smem_u32(sm + OpSmem::b + (c % kOpBStages) * kOpB), kOpBSlab, 1024, tc::kSwizzle128);
#pragma unroll
        for (int k = 0; k < kOpKC / 16; ++k)
          tc::mma_bf16(tmem, adesc + (uint64_t)((k * 32) >> 4),
                       bdesc + (uint64_t)((k * 16 * 128) >> 4), kId, c > 0 || k > 0);
        tc::commit(&done[sa]);
      }
      __syncwarp();
    }
    return true;
  };
#pragma unroll 1
  for (int c = 0; c < kOpChunks; c += 2) {
    if (!chunk(c, pre0) || !chunk(c + 1, pre1)) { ok = false; break; }
  }
  // every MMA issued must finish before TMEM is read or freed
  if (warp == 0) {
    if (tc::elect_one()) tc::commit(fin);
    __syncwarp();
  }
  const bool okf = __syncthreads_and(mbar_wait(fin, 0) && ok);
  tc::fence_after_sync();
  uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)(row0 + r) * H + h) * kDv) + 8 * hf;
  if (okf) {
    // the TMEM loads are warp-collective: every lane loads, live rows store;
    // warps 0-3 take columns 0-63 of their rows, warps 4-7 columns 64-127
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 64 * hf;
#pragma unroll 1
    for (int cb = 0; cb < 2; ++cb) {
      uint32_t v[32];
      tc::ld32(trow + 32 * cb, v);
      tc::wait_ld();
      if (!live) continue;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[4 * cb + q] = make_uint4(
            pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
            pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
            pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
            pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
    }
  } else if (live) {
    // no result: the rows hold NaN, so the failure cannot pass for an output
    for (int q = 0; q < 8; ++q) dst[q] = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
  }
  // never leave with weight copies in flight (only after a failed wait can
  // a chunk have been issued and not consumed)
  if (tid == 0)
    for (int c = w_issued - kOpBStages > 0 ? w_issued - kOpBStages : 0; c < w_issued; ++c)
      mbar_wait(&bfull[c % kOpBStages], (c / kOpBStages) & 1);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::dealloc(tmem, kOpTmemCols);
}

}  // namespace

cudaError_t launch_out_proj_tc(const CUtensorMap& w_map, const float* o_lat, void* out,
                               int64_t num_q, int H, cudaStream_t stream) {
  const int smem = OpSmem::alloc;
  cudaError_t e = cudaFuncSetAttribute(out_proj_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(out_proj_tc_kernel, dim3((unsigned)((num_q + kOpRows - 1) / kOpRows), H),
                    dim3(kOpThreads), smem, stream, w_map, o_lat, (__nv_bfloat16*)out, (int)num_q, H);
}

}  // namespace mla
