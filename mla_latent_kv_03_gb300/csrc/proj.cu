// Per-head projections on either side of the latent attention.
//   absorb_q : q_abs[n,h,0:512]   = W_uk[h] (512x128) @ q_nope[n,h] (128)
//              q_abs[n,h,512:576] = RoPE(q_pe[n,h], pos_n)
//   out_proj : out[n,h,:]         = o_lat[n,h,:] (512) @ W_uv[h] (512x128)
// Source: "mini-infer-17: MLA Attention", section "版本 3: MLAAttentionAbsorbed"
// (_build_absorbed gives W_k_absorbed and W_v_absorbed as [H, d_c, 128]).
//
// bf16: batched-per-head GEMMs on warp mma (m16n8k16, fp32 accumulate). They
// are small and latency-bound, so each CTA issues all of its weight bytes as
// cp.async copies at once and loads its activation fragments while those are
// in flight; grids are cut into column blocks for enough CTAs.
// fp32: plain SIMT dot products in fp32 (no tensor cores: fp32 I/O is held to
// 1e-4 absolute).
#include "async_copy.cuh"
#include "common.cuh"
#include "rope_pairs.cuh"
#include "internal.h"

namespace mla {
namespace {

// ---------------------------------------------------------------------------
// absorb_q, bf16. CTA = (16*MW query rows, 128 latent columns, head h);
// MW more columns of CTAs (blockIdx.y >= 4) do the RoPE part, 16 rows each.
// The CTA's weight slice W_uk[h][col0:col0+128][0:128] (32 KB) is copied to
// shared memory with cp.async in one go (rows of 256 B, 16-byte chunks
// XOR-swizzled by row so ldmatrix is conflict-free); the query fragments of
// all 8 k-steps are loaded while the copy is in flight.
//   MW = 1: the four warps split the 128 columns (32 each).
//   MW = 4: each warp owns 16 rows and all 128 columns.
// ---------------------------------------------------------------------------
template <int MW>
__global__ void __launch_bounds__(128) absorb_bf16_kernel(
    const __nv_bfloat16* __restrict__ q_nope, const __nv_bfloat16* __restrict__ q_pe,
    const int32_t* __restrict__ q_pos, const __nv_bfloat16* __restrict__ W_uk,
    __nv_bfloat16* __restrict__ q_abs, int num_q, int H, RopeFreq freq, int interleaved) {
  constexpr int NT = MW == 1 ? 4 : 16;   // 8-column n-tiles per warp
  constexpr int ROWS = 16 * MW;
  __shared__ __align__(1024) uint8_t sB[128 * 256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int h = blockIdx.z, row0 = blockIdx.x * ROWS, col0 = blockIdx.y * 128;

  if (blockIdx.y >= 4) {
    // rotate-half RoPE of q_pe into q_abs[..., 512:576] for 16 of this row
    // block's rows; all loads of a thread are issued before any of them is used
    pdl_wait();
    pdl_launch_dependents();
    constexpr int kPer = 16 * 32 / 128;
    const int rrow0 = row0 + 16 * (blockIdx.y - 4);
    const int p = tid & 31, i1 = rope_i1(interleaved, p), i2 = rope_i2(interleaved, p);
    const float fhi = freq.hi[p], flo = freq.lo[p];
    float x1[kPer], x2[kPer];
    int pos[kPer];
#pragma unroll
    for (int it = 0; it < kPer; ++it) {
      const int r = rrow0 + (tid >> 5) + 4 * it;
      const bool ok = r < num_q;
      const __nv_bfloat16* x = q_pe + ((size_t)r * H + h) * kDr;
      x1[it] = ok ? __bfloat162float(x[i1]) : 0.f;
      x2[it] = ok ? __bfloat162float(x[i2]) : 0.f;
      pos[it] = ok ? q_pos[r] : 0;
    }
#pragma unroll
    for (int it = 0; it < kPer; ++it) {
      const int r = rrow0 + (tid >> 5) + 4 * it;
      if (r >= num_q) continue;
      float cs, sn;
      rope_cos_sin(pos[it], fhi, flo, &cs, &sn);
      __nv_bfloat16* o = q_abs + ((size_t)r * H + h) * kRow + kDc;
      o[i1] = __float2bfloat16_rn(x1[it] * cs - x2[it] * sn);
      o[i2] = __float2bfloat16_rn(x2[it] * cs + x1[it] * sn);
    }
    return;
  }

  const __nv_bfloat16* src = W_uk + ((size_t)h * kDc + col0) * kDn;
  for (int i = tid; i < 128 * 16; i += 128) {
    const int r = i >> 4, ch = i & 15;
    cp_async16(sB + r * 256 + ((ch ^ (r & 7)) << 4), src + r * kDn + ch * 8);
  }
  cp_async_commit();
  // the weights do not depend on earlier kernels; the query does
  pdl_wait();
  pdl_launch_dependents();

  const int wr = MW == 1 ? 0 : warp, wc = MW == 1 ? warp : 0;
  const int r_lo = row0 + 16 * wr + g, r_hi = r_lo + 8;
  const bool ok_lo = r_lo < num_q, ok_hi = r_hi < num_q;
  uint32_t a[8][4];
  const __nv_bfloat16* plo = q_nope + ((size_t)r_lo * H + h) * kDn + 2 * q;
  const __nv_bfloat16* phi = q_nope + ((size_t)r_hi * H + h) * kDn + 2 * q;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    a[ks][0] = ok_lo ? *reinterpret_cast<const uint32_t*>(plo + ks * 16) : 0u;
    a[ks][1] = ok_hi ? *reinterpret_cast<const uint32_t*>(phi + ks * 16) : 0u;
    a[ks][2] = ok_lo ? *reinterpret_cast<const uint32_t*>(plo + ks * 16 + 8) : 0u;
    a[ks][3] = ok_hi ? *reinterpret_cast<const uint32_t*>(phi + ks * 16 + 8) : 0u;
  }
  cp_async_wait_all();
  __syncthreads();

  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      const int n = wc * (8 * NT) + np * 16 + (lane & 7) + ((lane >> 4) << 3);
      const int ch = ks * 2 + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(smem_u32(sB + n * 256 + ((ch ^ (n & 7)) << 4)), b0, b1, b2, b3);
      mma_16816(acc[2 * np], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
      mma_16816(acc[2 * np + 1], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b2, b3);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = col0 + wc * (8 * NT) + nt * 8 + 2 * q;
    if (ok_lo)
      *reinterpret_cast<uint32_t*>(q_abs + ((size_t)r_lo * H + h) * kRow + col) =
          pack_bf16(acc[nt][0], acc[nt][1]);
    if (ok_hi)
      *reinterpret_cast<uint32_t*>(q_abs + ((size_t)r_hi * H + h) * kRow + col) =
          pack_bf16(acc[nt][2], acc[nt][3]);
  }
}

// ---------------------------------------------------------------------------
// out_proj, bf16. CTA = (16*MW query rows, 64 output columns, head h). The
// weight slice W_uv[h][0:512][col0:col0+64] (64 KB) goes to shared memory by
// cp.async in one go (128-byte rows, swizzled for ldmatrix.trans).
//   MW = 1: the four warps split K = 512 into quarters (latency: the o_lat
//           fragments of a quarter, 8 k-steps, are loaded before the wait);
//           the four partial tiles are summed through shared memory.
//   MW = 4: each warp owns 16 rows over all of K.
// o_lat is fp32 and rounded to bf16 for the mma.
// ---------------------------------------------------------------------------
template <int MW>
__global__ void __launch_bounds__(128) out_proj_bf16_kernel(const float* __restrict__ o_lat,
                                                            const __nv_bfloat16* __restrict__ W_uv,
                                                            __nv_bfloat16* __restrict__ out,
                                                            int num_q, int H) {
  extern __shared__ __align__(1024) uint8_t smem_op[];
  uint8_t* sB = smem_op;                                   // 512 x 128 B
  float* sRed = reinterpret_cast<float*>(smem_op + 512 * 128);  // [4][16][64] (MW == 1)
  constexpr int ROWS = 16 * MW;
  constexpr int KS = MW == 1 ? 8 : 32;                     // k-steps per warp
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int h = blockIdx.z, row0 = blockIdx.x * ROWS, col0 = blockIdx.y * 64;

  const __nv_bfloat16* src = W_uv + (size_t)h * kDc * kDv + col0;
  for (int i = tid; i < 512 * 8; i += 128) {
    const int r = i >> 3, ch = i & 7;
    cp_async16(sB + sw128(r, ch), src + (size_t)r * kDv + ch * 8);
  }
  cp_async_commit();
  // the weights do not depend on earlier kernels; o_lat does
  pdl_wait();
  pdl_launch_dependents();

  const int wr = MW == 1 ? 0 : warp;
  const int k0 = MW == 1 ? warp * 128 : 0;
  const int r_lo = row0 + 16 * wr + g, r_hi = r_lo + 8;
  const bool ok_lo = r_lo < num_q, ok_hi = r_hi < num_q;
  const float* plo = o_lat + ((size_t)r_lo * H + h) * kDc + k0 + 2 * q;
  const float* phi = o_lat + ((size_t)r_hi * H + h) * kDc + k0 + 2 * q;
  auto load_a = [&](int ks, uint32_t* a) {
    float2 x;
    x = ok_lo ? *reinterpret_cast<const float2*>(plo + ks * 16) : make_float2(0.f, 0.f);
    a[0] = pack_bf16(x.x, x.y);
    x = ok_hi ? *reinterpret_cast<const float2*>(phi + ks * 16) : make_float2(0.f, 0.f);
    a[1] = pack_bf16(x.x, x.y);
    x = ok_lo ? *reinterpret_cast<const float2*>(plo + ks * 16 + 8) : make_float2(0.f, 0.f);
    a[2] = pack_bf16(x.x, x.y);
    x = ok_hi ? *reinterpret_cast<const float2*>(phi + ks * 16 + 8) : make_float2(0.f, 0.f);
    a[3] = pack_bf16(x.x, x.y);
  };
  uint32_t apre[8][4];
  if (MW == 1) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) load_a(ks, apre[ks]);
  }
  cp_async_wait_all();
  __syncthreads();

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t a[4];
    if (MW == 1) {
      a[0] = apre[ks & 7][0]; a[1] = apre[ks & 7][1]; a[2] = apre[ks & 7][2]; a[3] = apre[ks & 7][3];
    } else {
      load_a(ks, a);
    }
    const int kr = k0 + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(smem_u32(sB + sw128(kr, np * 2 + (lane >> 4))), b0, b1, b2, b3);
      mma_16816(acc[2 * np], a[0], a[1], a[2], a[3], b0, b1);
      mma_16816(acc[2 * np + 1], a[0], a[1], a[2], a[3], b2, b3);
    }
  }
  if (MW == 1) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float* d = sRed + (warp * 16 + g) * 64 + nt * 8 + 2 * q;
      d[0] = acc[nt][0]; d[1] = acc[nt][1];
      d[8 * 64] = acc[nt][2]; d[8 * 64 + 1] = acc[nt][3];
    }
    __syncthreads();
    for (int i = tid; i < 16 * 32; i += 128) {
      const int r = i >> 5, c = (i & 31) * 2;
      const int row = row0 + r;
      if (row >= num_q) continue;
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        v0 += sRed[(w * 16 + r) * 64 + c];
        v1 += sRed[(w * 16 + r) * 64 + c + 1];
      }
      *reinterpret_cast<uint32_t*>(out + ((size_t)row * H + h) * kDv + col0 + c) = pack_bf16(v0, v1);
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = col0 + nt * 8 + 2 * q;
      if (ok_lo)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r_lo * H + h) * kDv + col) =
            pack_bf16(acc[nt][0], acc[nt][1]);
      if (ok_hi)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r_hi * H + h) * kDv + col) =
            pack_bf16(acc[nt][2], acc[nt][3]);
    }
  }
}

// ---------------------------------------------------------------------------
// out_proj, bf16, fewer than 256 rows. CTA = (32 query rows, 32 output
// columns, head h): the weight slice W_uv[h][0:512][col0:col0+32] is 32 KB,
// so the CTA fits on an SM beside a decode CTA. Launched as the decode's
// dependent it stages its weights while the decode still runs and then waits
// only for o_lat, which it loads in one round (all 16 k-steps of a warp's
// fragments at once). Warp w owns rows 16 (w & 1) .. +16 and K half w >> 1;
// the K halves are summed through shared memory. Slice rows are 64 bytes,
// 16-byte chunk c of row k at chunk c ^ ((k >> 1) & 3) (conflict-free
// ldmatrix.trans).
// ---------------------------------------------------------------------------
constexpr int kOpSmallSmem = 512 * 64 + 2 * 16 * 32 * 4;  // 36 KB

__device__ __forceinline__ uint32_t sw64(int row, int chunk) {
  return (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

__global__ void __launch_bounds__(128) out_proj_small_kernel(const float* __restrict__ o_lat,
                                                             const __nv_bfloat16* __restrict__ W_uv,
                                                             __nv_bfloat16* __restrict__ out,
                                                             int num_q, int H) {
  extern __shared__ __align__(128) uint8_t smem_os[];
  uint8_t* sB = smem_os;                                           // 512 x 64 B
  float* sRed = reinterpret_cast<float*>(smem_os + 512 * 64);     // [2][16][32]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int h = blockIdx.z, col0 = blockIdx.y * 32;
  const int rb = warp & 1, kh = warp >> 1;

  const __nv_bfloat16* src = W_uv + (size_t)h * kDc * kDv + col0;
  for (int i = tid; i < 512 * 4; i += 128) {
    const int r = i >> 2, ch = i & 3;
    cp_async16(sB + sw64(r, ch), src + (size_t)r * kDv + ch * 8);
  }
  cp_async_commit();
  // the weights do not depend on earlier kernels; o_lat does
  pdl_wait();
  pdl_launch_dependents();

  const int r_lo = blockIdx.x * 32 + 16 * rb + g, r_hi = r_lo + 8;
  const bool ok_lo = r_lo < num_q, ok_hi = r_hi < num_q;
  const int k0 = kh * 256;
  const float* plo = o_lat + ((size_t)r_lo * H + h) * kDc + k0 + 2 * q;
  const float* phi = o_lat + ((size_t)r_hi * H + h) * kDc + k0 + 2 * q;
  float2 x[16][4];
#pragma unroll
  for (int ks = 0; ks < 16; ++ks) {
    const float2 z = make_float2(0.f, 0.f);
    x[ks][0] = ok_lo ? *reinterpret_cast<const float2*>(plo + ks * 16) : z;
    x[ks][1] = ok_hi ? *reinterpret_cast<const float2*>(phi + ks * 16) : z;
    x[ks][2] = ok_lo ? *reinterpret_cast<const float2*>(plo + ks * 16 + 8) : z;
    x[ks][3] = ok_hi ? *reinterpret_cast<const float2*>(phi + ks * 16 + 8) : z;
  }
  cp_async_wait_all();
  __syncthreads();

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 16; ++ks) {
    const uint32_t a0 = pack_bf16(x[ks][0].x, x[ks][0].y), a1 = pack_bf16(x[ks][1].x, x[ks][1].y);
    const uint32_t a2 = pack_bf16(x[ks][2].x, x[ks][2].y), a3 = pack_bf16(x[ks][3].x, x[ks][3].y);
    const int kr = k0 + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(smem_u32(sB + sw64(kr, np * 2 + (lane >> 4))), b0, b1, b2, b3);
      mma_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
      mma_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
    }
  }
  float* red = sRed + rb * 16 * 32;
  if (kh == 1) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      *reinterpret_cast<float2*>(red + g * 32 + nt * 8 + 2 * q) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(red + (g + 8) * 32 + nt * 8 + 2 * q) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();
  if (kh == 0) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = nt * 8 + 2 * q;
      const float2 lo = *reinterpret_cast<const float2*>(red + g * 32 + c);
      const float2 hi = *reinterpret_cast<const float2*>(red + (g + 8) * 32 + c);
      if (ok_lo)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r_lo * H + h) * kDv + col0 + c) =
            pack_bf16(acc[nt][0] + lo.x, acc[nt][1] + lo.y);
      if (ok_hi)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r_hi * H + h) * kDv + col0 + c) =
            pack_bf16(acc[nt][2] + hi.x, acc[nt][3] + hi.y);
    }
  }
}

// ---------------------------------------------------------------------------
// combine + out_proj, bf16: out[n,h,:] = merge_s(partials of (n, h)) @ W_uv[h].
// Same tiling as out_proj; the A fragments are merged on the fly from the
// decode's split partials (split-softmax identity, base-2 lse) instead of
// being read from o_lat, which is never materialised. Per CTA row r the merge
// parameters (first slot, number of slots, max lse, 1 / weight sum) are
// computed once into shared memory.
// ---------------------------------------------------------------------------
struct MergeRow {
  int64_t slot0;   // first 16-row partial group
  int stride, nslots;
  float M, inv;
};

// Merge parameters of (query row n, head h): where its parts are, the max
// base-2 log-sum-exp and 1 / the weight sum. nslots = 0: a zero row.
__device__ __forceinline__ MergeRow merge_row(const uint8_t* ws, const float* lse, int64_t num_q,
                                              int groups, int num_ctas, int batch, int n, int h) {
  MergeRow mr{0, 1, 0, 0.f, 0.f};
  if (n >= num_q) return mr;
  const QtileParts qp = locate_qtile(ws, num_q, groups, num_ctas, batch, n, h / kHG);
  if (qp.count <= 0) return mr;
  const int hr = h % kHG;
  float M = -INFINITY;
  for (int s = 0; s < qp.count; ++s) M = fmaxf(M, lse[(qp.first + (int64_t)s * qp.stride) * kHG + hr]);
  float den = 0.f;
  if (M != -INFINITY)
    for (int s = 0; s < qp.count; ++s)
      den += fast_exp2(lse[(qp.first + (int64_t)s * qp.stride) * kHG + hr] - M);
  if (M == -INFINITY) return mr;
  mr.slot0 = qp.first;
  mr.stride = qp.stride;
  mr.nslots = qp.count;
  mr.M = M;
  mr.inv = den > 0.f ? 1.f / den : 0.f;
  return mr;
}

__device__ __forceinline__ void ws_parts(const uint8_t* ws, int64_t num_q, int groups, int num_ctas,
                                         int batch, const float** lse, const float** opart) {
  const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
  if (hdr->mode == 0) {
    const WsLayout L = ws_layout(num_q, groups, num_ctas);
    *lse = reinterpret_cast<const float*>(ws + L.lse);
    *opart = reinterpret_cast<const float*>(ws + L.opart);
  } else {
    const WsLayoutTc L = ws_layout_tc(num_q, groups, num_ctas / 2, batch);
    *lse = reinterpret_cast<const float*>(ws + L.lse);
    *opart = reinterpret_cast<const float*>(ws + L.opart);
  }
}

template <int MW>
__global__ void __launch_bounds__(128) combine_out_proj_bf16_kernel(
    const uint8_t* __restrict__ ws, int groups, int num_ctas, int num_q, int batch,
    const __nv_bfloat16* __restrict__ W_uv, __nv_bfloat16* __restrict__ out, int H) {
  extern __shared__ __align__(1024) uint8_t smem_cp[];
  constexpr int ROWS = 16 * MW;
  constexpr int KS = MW == 1 ? 8 : 32;
  uint8_t* sB = smem_cp;                                          // 512 x 128 B
  float* sRed = reinterpret_cast<float*>(smem_cp + 512 * 128);    // [4][16][64] (MW == 1)
  MergeRow* sRow = reinterpret_cast<MergeRow*>(smem_cp + 512 * 128 + (MW == 1 ? 4 * 16 * 64 * 4 : 0));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int h = blockIdx.z, row0 = blockIdx.x * ROWS, col0 = blockIdx.y * 64;

  const __nv_bfloat16* src = W_uv + (size_t)h * kDc * kDv + col0;
  for (int i = tid; i < 512 * 8; i += 128) {
    const int r = i >> 3, ch = i & 7;
    cp_async16(sB + sw128(r, ch), src + (size_t)r * kDv + ch * 8);
  }
  cp_async_commit();
  // the weights do not depend on earlier kernels; the partials do
  pdl_wait();
  pdl_launch_dependents();

  const float* lse;
  const float* opart;
  ws_parts(ws, num_q, groups, num_ctas, batch, &lse, &opart);
  const int hr = h % kHG;
  for (int r = tid; r < ROWS; r += 128)
    sRow[r] = merge_row(ws, lse, num_q, groups, num_ctas, batch, row0 + r, h);
  __syncthreads();

  const int wr = MW == 1 ? 0 : warp;
  const int k0 = MW == 1 ? warp * 128 : 0;
  const int rl_lo = 16 * wr + g, rl_hi = rl_lo + 8;
  const MergeRow m_lo = sRow[rl_lo], m_hi = sRow[rl_hi];
  // merged (o_lat) value pair at column k of a local row
  auto merged2 = [&](const MergeRow& m, int k) {
    float2 acc = make_float2(0.f, 0.f);
    for (int s = 0; s < m.nslots; ++s) {
      const size_t slot = (size_t)(m.slot0 + (int64_t)s * m.stride);
      const float w = fast_exp2(lse[slot * kHG + hr] - m.M) * m.inv;
      const float2 v = *reinterpret_cast<const float2*>(opart + (slot * kHG + hr) * kDc + k);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
    }
    return acc;
  };
  auto load_a = [&](int ks, uint32_t* a) {
    const int k = k0 + ks * 16 + 2 * q;
    float2 x;
    x = merged2(m_lo, k);     a[0] = pack_bf16(x.x, x.y);
    x = merged2(m_hi, k);     a[1] = pack_bf16(x.x, x.y);
    x = merged2(m_lo, k + 8); a[2] = pack_bf16(x.x, x.y);
    x = merged2(m_hi, k + 8); a[3] = pack_bf16(x.x, x.y);
  };
  uint32_t apre[8][4];
  if (MW == 1) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) load_a(ks, apre[ks]);
  }
  cp_async_wait_all();
  __syncthreads();

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t a[4];
    if (MW == 1) {
      a[0] = apre[ks & 7][0]; a[1] = apre[ks & 7][1]; a[2] = apre[ks & 7][2]; a[3] = apre[ks & 7][3];
    } else {
      load_a(ks, a);
    }
    const int kr = k0 + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(smem_u32(sB + sw128(kr, np * 2 + (lane >> 4))), b0, b1, b2, b3);
      mma_16816(acc[2 * np], a[0], a[1], a[2], a[3], b0, b1);
      mma_16816(acc[2 * np + 1], a[0], a[1], a[2], a[3], b2, b3);
    }
  }
  const int r_lo = row0 + rl_lo, r_hi = row0 + rl_hi;
  if (MW == 1) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float* d = sRed + (warp * 16 + g) * 64 + nt * 8 + 2 * q;
      d[0] = acc[nt][0]; d[1] = acc[nt][1];
      d[8 * 64] = acc[nt][2]; d[8 * 64 + 1] = acc[nt][3];
    }
    __syncthreads();
    for (int i = tid; i < 16 * 32; i += 128) {
      const int r = i >> 5, c = (i & 31) * 2;
      const int row = row0 + r;
      if (row >= num_q) continue;
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        v0 += sRed[(w * 16 + r) * 64 + c];
        v1 += sRed[(w * 16 + r) * 64 + c + 1];
      }
      *reinterpret_cast<uint32_t*>(out + ((size_t)row * H + h) * kDv + col0 + c) = pack_bf16(v0, v1);
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = col0 + nt * 8 + 2 * q;
      if (r_lo < num_q)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r_lo * H + h) * kDv + col) =
            pack_bf16(acc[nt][0], acc[nt][1]);
      if (r_hi < num_q)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r_hi * H + h) * kDv + col) =
            pack_bf16(acc[nt][2], acc[nt][3]);
    }
  }
}

// combine + out_proj, bf16, up to 16 query rows per CTA (decode batches):
// the CTA first merges its 16 latent rows of head h into shared memory as
// bf16 -- per row one warp reduces the max log-sum-exp and the weight sum over
// the parts, then 8 threads per row accumulate the weighted partial rows, one
// round trip per part -- and then projects them as out_proj does.
constexpr int kMergedStride = kDc * 2 + 16;  // bytes per merged row (padded against bank conflicts)

__global__ void __launch_bounds__(128) combine_out_proj_rows16_kernel(
    const uint8_t* __restrict__ ws, int groups, int num_ctas, int num_q, int batch,
    const __nv_bfloat16* __restrict__ W_uv, __nv_bfloat16* __restrict__ out, int H) {
  extern __shared__ __align__(1024) uint8_t smem_cr[];
  uint8_t* sB = smem_cr;                                               // 512 x 128 B
  float* sRed = reinterpret_cast<float*>(smem_cr + 512 * 128);         // [4][16][64]
  uint8_t* sA = smem_cr + 512 * 128 + 4 * 16 * 64 * 4;                 // [16] merged rows, bf16
  int64_t* sFirst = reinterpret_cast<int64_t*>(sA + 16 * kMergedStride);
  int* sStride = reinterpret_cast<int*>(sFirst + 16);
  int* sCount = sStride + 16;
  float* sM = reinterpret_cast<float*>(sCount + 16);
  float* sInv = sM + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int h = blockIdx.z, row0 = blockIdx.x * 16, col0 = blockIdx.y * 64;
  const int hr = h % kHG;

  const __nv_bfloat16* src = W_uv + (size_t)h * kDc * kDv + col0;
  for (int i = tid; i < 512 * 8; i += 128) {
    const int r = i >> 3, ch = i & 7;
    cp_async16(sB + sw128(r, ch), src + (size_t)r * kDv + ch * 8);
  }
  cp_async_commit();
  // the weights do not depend on earlier kernels; the partials do
  pdl_wait();
  pdl_launch_dependents();

  const float* lse;
  const float* opart;
  ws_parts(ws, num_q, groups, num_ctas, batch, &lse, &opart);
  if (tid < 16) {
    const int n = row0 + tid;
    QtileParts qp{0, 1, 0};
    if (n < num_q) qp = locate_qtile(ws, num_q, groups, num_ctas, batch, n, h / kHG);
    sFirst[tid] = qp.first;
    sStride[tid] = qp.stride;
    sCount[tid] = qp.count > 0 ? qp.count : 0;
  }
  __syncthreads();
  // per row: max base-2 lse and 1 / weight sum over its parts (one warp per row)
#pragma unroll 1
  for (int r = warp; r < 16; r += 4) {
    const int cnt = sCount[r];
    const int64_t f = sFirst[r];
    const int st = sStride[r];
    float M = -INFINITY;
    for (int s = lane; s < cnt; s += 32) M = fmaxf(M, lse[(f + (int64_t)s * st) * kHG + hr]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float den = 0.f;
    if (M != -INFINITY)
      for (int s = lane; s < cnt; s += 32) den += fast_exp2(lse[(f + (int64_t)s * st) * kHG + hr] - M);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane == 0) {
      sM[r] = M;
      sInv[r] = (M != -INFINITY && den > 0.f) ? 1.f / den : 0.f;
    }
  }
  __syncthreads();
  // merged rows: 8 threads per row, float4 j + 8 m of the row (m < 16)
  {
    const int r = tid >> 3, j = tid & 7;
    const int cnt = sCount[r];
    const int64_t f = sFirst[r];
    const int st = sStride[r];
    const float M = sM[r], inv = sInv[r];
    float4 acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll 1
      for (int s = 0; s < cnt; ++s) {
        const int64_t slot = f + (int64_t)s * st;
        const float4* srcp = reinterpret_cast<const float4*>(opart + (slot * kHG + hr) * kDc) + j;
        float4 v[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] = srcp[8 * m];
        const float w = fast_exp2(lse[slot * kHG + hr] - M) * inv;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          acc[m].x = fmaf(w, v[m].x, acc[m].x);
          acc[m].y = fmaf(w, v[m].y, acc[m].y);
          acc[m].z = fmaf(w, v[m].z, acc[m].z);
          acc[m].w = fmaf(w, v[m].w, acc[m].w);
        }
      }
    }
    uint8_t* dstrow = sA + r * kMergedStride;
#pragma unroll
    for (int m = 0; m < 16; ++m)
      *reinterpret_cast<uint2*>(dstrow + (j + 8 * m) * 8) =
          make_uint2(pack_bf16(acc[m].x, acc[m].y), pack_bf16(acc[m].z, acc[m].w));
  }
  cp_async_wait_all();
  __syncthreads();

  // out[16 rows x 64 cols] over this warp's quarter of K, summed through sRed
  const int k0 = warp * 128;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int k = k0 + ks * 16 + 2 * q;
    uint32_t a[4];
    a[0] = *reinterpret_cast<const uint32_t*>(sA + g * kMergedStride + k * 2);
    a[1] = *reinterpret_cast<const uint32_t*>(sA + (g + 8) * kMergedStride + k * 2);
    a[2] = *reinterpret_cast<const uint32_t*>(sA + g * kMergedStride + (k + 8) * 2);
    a[3] = *reinterpret_cast<const uint32_t*>(sA + (g + 8) * kMergedStride + (k + 8) * 2);
    const int kr = k0 + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(smem_u32(sB + sw128(kr, np * 2 + (lane >> 4))), b0, b1, b2, b3);
      mma_16816(acc[2 * np], a[0], a[1], a[2], a[3], b0, b1);
      mma_16816(acc[2 * np + 1], a[0], a[1], a[2], a[3], b2, b3);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    float* d = sRed + (warp * 16 + g) * 64 + nt * 8 + 2 * q;
    d[0] = acc[nt][0]; d[1] = acc[nt][1];
    d[8 * 64] = acc[nt][2]; d[8 * 64 + 1] = acc[nt][3];
  }
  __syncthreads();
  for (int i = tid; i < 16 * 32; i += 128) {
    const int r = i >> 5, c = (i & 31) * 2;
    const int row = row0 + r;
    if (row >= num_q) continue;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      v0 += sRed[(w * 16 + r) * 64 + c];
      v1 += sRed[(w * 16 + r) * 64 + c + 1];
    }
    *reinterpret_cast<uint32_t*>(out + ((size_t)row * H + h) * kDv + col0 + c) = pack_bf16(v0, v1);
  }
}

// combine + out_proj, fp32: one CTA per (row n, head h); the merged latent
// row goes to shared memory, then 128 threads take one output column each.
__global__ void __launch_bounds__(128) combine_out_proj_f32_kernel(
    const uint8_t* __restrict__ ws, int groups, int num_ctas, int num_q, int batch,
    const float* __restrict__ W_uv, float* __restrict__ out, int H) {
  __shared__ float so[kDc];
  __shared__ MergeRow sr;
  pdl_wait();
  pdl_launch_dependents();
  const int n = blockIdx.x, h = blockIdx.y, t0 = threadIdx.x;
  const float* lse;
  const float* opart;
  ws_parts(ws, num_q, groups, num_ctas, batch, &lse, &opart);
  const int hr = h % kHG;
  if (t0 == 0) sr = merge_row(ws, lse, num_q, groups, num_ctas, batch, n, h);
  __syncthreads();
  const MergeRow mr = sr;
  for (int c = t0; c < kDc; c += 128) {
    float acc = 0.f;
    for (int s = 0; s < mr.nslots; ++s) {
      const size_t slot = (size_t)(mr.slot0 + (int64_t)s * mr.stride);
      acc = fmaf(fast_exp2(lse[slot * kHG + hr] - mr.M) * mr.inv, opart[(slot * kHG + hr) * kDc + c], acc);
    }
    so[c] = acc;
  }
  __syncthreads();
  const float* w = W_uv + (size_t)h * kDc * kDv + t0;
  float s = 0.f;
  for (int c = 0; c < kDc; ++c) s = fmaf(so[c], w[(size_t)c * kDv], s);
  out[((size_t)n * H + h) * kDv + t0] = s;
}

// fp32 SIMT: one CTA per (row n, head h).
// absorb_q, fp32 (the fp32 configuration: a handful of rows). CTA = (head h,
// 64 latent rows c); each of its 8 warps holds 8 rows of W_uk[h] in registers
// (lane l: columns 4l..4l+3, coalesced float4 loads, all in flight at once)
// and, for every query row n, reduces the 8 dot products over its lanes. A
// ninth CTA column does the RoPE part.
constexpr int kAbsorbF32Rows = 64;

__global__ void __launch_bounds__(256) absorb_f32_kernel(
    const float* __restrict__ q_nope, const float* __restrict__ q_pe,
    const int32_t* __restrict__ q_pos, const float* __restrict__ W_uk, float* __restrict__ q_abs,
    int num_q, int H, RopeFreq freq, int interleaved) {
  const int h = blockIdx.x, chunk = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (chunk == kDc / kAbsorbF32Rows) {
    // rotate-half RoPE of q_pe into q_abs[..., 512:576]
    for (int i = tid; i < num_q * 32; i += 256) {
      const int n = i >> 5, p = i & 31;
      const float* x = q_pe + ((size_t)n * H + h) * kDr;
      float cs, sn;
      rope_cos_sin(q_pos[n], freq.hi[p], freq.lo[p], &cs, &sn);
      float* out = q_abs + ((size_t)n * H + h) * kRow + kDc;
      const int i1 = rope_i1(interleaved, p), i2 = rope_i2(interleaved, p);
      out[i1] = x[i1] * cs - x[i2] * sn;
      out[i2] = x[i2] * cs + x[i1] * sn;
    }
    return;
  }
  const int c0 = chunk * kAbsorbF32Rows + warp * 8;
  float4 w[8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
    w[r] = *reinterpret_cast<const float4*>(W_uk + ((size_t)h * kDc + c0 + r) * kDn + 4 * lane);
  for (int n = 0; n < num_q; ++n) {
    const float4 q = *reinterpret_cast<const float4*>(q_nope + ((size_t)n * H + h) * kDn + 4 * lane);
    float d[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) d[r] = fmaf(w[r].x, q.x, fmaf(w[r].y, q.y, fmaf(w[r].z, q.z, w[r].w * q.w)));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int r = 0; r < 8; ++r) d[r] += __shfl_xor_sync(0xffffffffu, d[r], o);
    if (lane < 8) {
      float v = d[0];
#pragma unroll
      for (int r = 1; r < 8; ++r) v = lane == r ? d[r] : v;
      q_abs[((size_t)n * H + h) * kRow + c0 + lane] = v;
    }
  }
}

// out_proj, fp32. CTA = (head h, 32 output columns); warp w holds rows
// [64 w, 64 w + 64) of W_uv[h] for its lane's column in registers (coalesced,
// all loads in flight at once), and for every query row n the 8 warps' partial
// sums meet in shared memory.
__global__ void __launch_bounds__(256) out_proj_f32_kernel(const float* __restrict__ o_lat,
                                                           const float* __restrict__ W_uv,
                                                           float* __restrict__ out, int num_q,
                                                           int H) {
  __shared__ float so[kDc];
  __shared__ float sred[8][32];
  const int h = blockIdx.x, v0 = blockIdx.y * 32, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  float w[64];
  const float* wp = W_uv + ((size_t)h * kDc + warp * 64) * kDv + v0 + lane;
#pragma unroll
  for (int c = 0; c < 64; ++c) w[c] = wp[(size_t)c * kDv];
  for (int n = 0; n < num_q; ++n) {
    __syncthreads();
    for (int c = tid; c < kDc; c += 256) so[c] = o_lat[((size_t)n * H + h) * kDc + c];
    __syncthreads();
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      a0 = fmaf(so[warp * 64 + c], w[c], a0);
      a1 = fmaf(so[warp * 64 + c + 1], w[c + 1], a1);
      a2 = fmaf(so[warp * 64 + c + 2], w[c + 2], a2);
      a3 = fmaf(so[warp * 64 + c + 3], w[c + 3], a3);
    }
    sred[warp][lane] = (a0 + a1) + (a2 + a3);
    __syncthreads();
    if (warp == 0) {
      float t = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) t += sred[k][lane];
      out[((size_t)n * H + h) * kDv + v0 + lane] = t;
    }
  }
}

}  // namespace

cudaError_t launch_absorb_q(const mla_config& cfg, const void* q_nope, const void* q_pe,
                            const int32_t* q_positions, const void* W_uk, void* q_abs,
                            int64_t num_q, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  const int H = cfg.num_heads;
  const RopeFreq freq = make_rope_freq((double)cfg.rope_base);
  const int inter = cfg.rope_interleaved;
  if (cfg.dtype == MLA_F32) {
    absorb_f32_kernel<<<dim3(H, kDc / kAbsorbF32Rows + 1), 256, 0, stream>>>(
        (const float*)q_nope, (const float*)q_pe, q_positions, (const float*)W_uk, (float*)q_abs,
        (int)num_q, H, freq, inter);
    return cudaGetLastError();
  }
  // More than 16 rows: 64 rows per CTA, so that a batch of up to 64 rows
  // takes one CTA per (head, column block) and each fits on an SM beside a
  // decode CTA (32 KB of shared memory; the carveout stays at its maximum).
  if (num_q > 16) {
    cudaError_t e = cudaFuncSetAttribute(absorb_bf16_kernel<4>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_pdl(absorb_bf16_kernel<4>, dim3((unsigned)((num_q + 63) / 64), 8, H), dim3(128), 0,
                      stream, (const __nv_bfloat16*)q_nope, (const __nv_bfloat16*)q_pe,
                      q_positions, (const __nv_bfloat16*)W_uk, (__nv_bfloat16*)q_abs, (int)num_q,
                      H, freq, inter);
  } else {
    cudaError_t e = cudaFuncSetAttribute(absorb_bf16_kernel<1>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_pdl(absorb_bf16_kernel<1>, dim3((unsigned)((num_q + 15) / 16), 5, H), dim3(128), 0,
                      stream, (const __nv_bfloat16*)q_nope, (const __nv_bfloat16*)q_pe,
                      q_positions, (const __nv_bfloat16*)W_uk, (__nv_bfloat16*)q_abs, (int)num_q,
                      H, freq, inter);
  }
  return cudaGetLastError();
}

cudaError_t launch_out_proj(const mla_config& cfg, const float* o_lat, const void* W_uv,
                            void* out, int64_t num_q, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  const int H = cfg.num_heads;
  if (cfg.dtype == MLA_F32) {
    out_proj_f32_kernel<<<dim3(H, kDv / 32), 256, 0, stream>>>(o_lat, (const float*)W_uv,
                                                              (float*)out, (int)num_q, H);
    return cudaGetLastError();
  }
  const bool big = num_q >= 256;
  if (!big) {
    cudaError_t e = cudaFuncSetAttribute(out_proj_small_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kOpSmallSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(out_proj_small_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_pdl(out_proj_small_kernel, dim3((unsigned)((num_q + 31) / 32), kDv / 32, H),
                      dim3(128), kOpSmallSmem, stream, o_lat, (const __nv_bfloat16*)W_uv,
                      (__nv_bfloat16*)out, (int)num_q, H);
  }
  const int smem = 512 * 128 + (big ? 0 : 4 * 16 * 64 * 4);
  cudaError_t e = big ? cudaFuncSetAttribute(out_proj_bf16_kernel<4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                      : cudaFuncSetAttribute(out_proj_bf16_kernel<1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (big) {
    return launch_pdl(out_proj_bf16_kernel<4>, dim3((unsigned)((num_q + 63) / 64), 2, H), dim3(128),
                      smem, stream, o_lat, (const __nv_bfloat16*)W_uv, (__nv_bfloat16*)out,
                      (int)num_q, H);
  } else {
    return launch_pdl(out_proj_bf16_kernel<1>, dim3((unsigned)((num_q + 15) / 16), 2, H), dim3(128),
                      smem, stream, o_lat, (const __nv_bfloat16*)W_uv, (__nv_bfloat16*)out,
                      (int)num_q, H);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine_out_proj(const mla_config& cfg, const void* workspace, int32_t groups,
                                   int32_t num_ctas, int64_t num_q, int32_t batch, const void* W_uv,
                                   void* out, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  const int H = cfg.num_heads;
  const uint8_t* ws = (const uint8_t*)workspace;
  if (cfg.dtype == MLA_F32) {
    return launch_pdl(combine_out_proj_f32_kernel, dim3((unsigned)num_q, H), dim3(128), 0, stream,
                      ws, groups, num_ctas, (int)num_q, (int)batch, (const float*)W_uv, (float*)out, H);
  }
  if (num_q >= 256) {
    const int smem = 512 * 128 + 64 * (int)sizeof(MergeRow);
    cudaError_t e = cudaFuncSetAttribute(combine_out_proj_bf16_kernel<4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(combine_out_proj_bf16_kernel<4>, dim3((unsigned)((num_q + 63) / 64), 2, H),
                      dim3(128), smem, stream, ws, groups, num_ctas, (int)num_q, (int)batch,
                      (const __nv_bfloat16*)W_uv, (__nv_bfloat16*)out, H);
  }
  const int smem = 512 * 128 + 4 * 16 * 64 * 4 + 16 * kMergedStride + 16 * (8 + 4 + 4 + 4 + 4);
  cudaError_t e = cudaFuncSetAttribute(combine_out_proj_rows16_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(combine_out_proj_rows16_kernel, dim3((unsigned)((num_q + 15) / 16), 2, H),
                    dim3(128), smem, stream, ws, groups, num_ctas, (int)num_q, (int)batch,
                    (const __nv_bfloat16*)W_uv, (__nv_bfloat16*)out, H);
}

}  // namespace mla
