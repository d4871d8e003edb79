// Per-head projections on either side of the latent attention.
//   absorb_q : q_abs[n,h,0:512]   = W_uk[h] (512x128) @ q_nope[n,h] (128)
//              q_abs[n,h,512:576] = RoPE(q_pe[n,h], pos_n)
//   out_proj : out[n,h,:]         = o_lat[n,h,:] (512) @ W_uv[h] (512x128)
// Source: "mini-infer-17: MLA Attention", section "版本 3: MLAAttentionAbsorbed"
// (_build_absorbed gives W_k_absorbed and W_v_absorbed as [H, d_c, 128]).
//
// bf16: a batched-per-head GEMM on warp mma (m16n8k16, fp32 accumulate). The
// CTA computes 16*MW query rows x 128 output columns of one head; the weight
// is staged through shared memory 64 K-values at a time (swizzled, read with
// ldmatrix), the activation fragments are loaded straight from global memory.
// fp32: plain SIMT dot products in fp32 (no tensor cores: fp32 I/O is held to
// 1e-4 absolute).
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

// B_NMAJOR = false: B stored [n][k] (k contiguous)   -- W_uk[h][c][d], k = d
// B_NMAJOR = true : B stored [k][n] (n contiguous)   -- W_uv[h][c][v], k = c
template <int MW, bool A_F32, bool B_NMAJOR, bool ROPE>
__global__ void __launch_bounds__(128) head_gemm_kernel(
    const void* __restrict__ A_, const __nv_bfloat16* __restrict__ B, __nv_bfloat16* __restrict__ C,
    int num_q, int H, int K, int a_stride_row, int c_stride_row, int b_ld,
    // rope (absorb only)
    const __nv_bfloat16* __restrict__ q_pe, const int32_t* __restrict__ q_pos, double base) {
  constexpr int NT = 4 * MW;                // n-tiles (8 cols) per warp
  constexpr int ROWS = 16 * MW;
  __shared__ __align__(1024) uint8_t sB[16384];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int h = blockIdx.z;
  const int row0 = blockIdx.x * ROWS;
  const int col0 = blockIdx.y * 128;
  const int wr = warp % MW;                 // row block of this warp
  const int wc = warp / MW;                 // column block of this warp
  const int ncol_w = 128 / (4 / MW);        // columns per warp = 8 * NT
  const int r_lo = row0 + wr * 16 + g, r_hi = r_lo + 8;
  const bool ok_lo = r_lo < num_q, ok_hi = r_hi < num_q;

  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const __nv_bfloat16* Bh = B + (size_t)h * kDc * 128;   // both weights are [H, 512, 128]
  for (int k0 = 0; k0 < K; k0 += 64) {
    __syncthreads();
    // stage 16 KB of the weight
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + i * 128;
      if (!B_NMAJOR) {  // rows = n (128), 64 k each = 8 chunks of 16 B
        const int r = idx >> 3, ch = idx & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(Bh + (size_t)(col0 + r) * b_ld + k0 + ch * 8);
        *reinterpret_cast<uint4*>(sB + sw128(r, ch)) = v;
      } else {          // rows = k (64), 128 n each = 16 chunks of 16 B
        const int r = idx >> 4, ch = idx & 15;
        const uint4 v = *reinterpret_cast<const uint4*>(Bh + (size_t)(k0 + r) * b_ld + col0 + ch * 8);
        *reinterpret_cast<uint4*>(sB + r * 256 + ((ch ^ (r & 7)) << 4)) = v;
      }
    }
    __syncthreads();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int kk = k0 + ks * 16 + 2 * q;
      uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
      if (A_F32) {
        const float* A = reinterpret_cast<const float*>(A_);
        if (ok_lo) {
          const float* p = A + (size_t)(r_lo * H + h) * a_stride_row + kk;
          const float2 x0 = *reinterpret_cast<const float2*>(p);
          const float2 x1 = *reinterpret_cast<const float2*>(p + 8);
          a0 = pack_bf16(x0.x, x0.y); a2 = pack_bf16(x1.x, x1.y);
        }
        if (ok_hi) {
          const float* p = A + (size_t)(r_hi * H + h) * a_stride_row + kk;
          const float2 x0 = *reinterpret_cast<const float2*>(p);
          const float2 x1 = *reinterpret_cast<const float2*>(p + 8);
          a1 = pack_bf16(x0.x, x0.y); a3 = pack_bf16(x1.x, x1.y);
        }
      } else {
        const __nv_bfloat16* A = reinterpret_cast<const __nv_bfloat16*>(A_);
        if (ok_lo) {
          const __nv_bfloat16* p = A + (size_t)(r_lo * H + h) * a_stride_row + kk;
          a0 = *reinterpret_cast<const uint32_t*>(p); a2 = *reinterpret_cast<const uint32_t*>(p + 8);
        }
        if (ok_hi) {
          const __nv_bfloat16* p = A + (size_t)(r_hi * H + h) * a_stride_row + kk;
          a1 = *reinterpret_cast<const uint32_t*>(p); a3 = *reinterpret_cast<const uint32_t*>(p + 8);
        }
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        const int cb = wc * ncol_w + np * 16;   // first column of the n-tile pair
        uint32_t b0, b1, b2, b3;
        if (!B_NMAJOR) {
          // matrices: (n 0-7,k 0-7) (n 0-7,k 8-15) (n 8-15,k 0-7) (n 8-15,k 8-15)
          const int n = cb + (lane & 7) + ((lane >> 4) << 3);
          const int ch = ks * 2 + ((lane >> 3) & 1);
          ldsm_x4(smem_u32(sB + sw128(n, ch)), b0, b1, b2, b3);
        } else {
          // matrices: (k 0-7,n c) (k 8-15,n c) (k 0-7,n c+1) (k 8-15,n c+1), transposed
          const int kr = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = (cb >> 3) + (lane >> 4);
          ldsm_x4_t(smem_u32(sB + kr * 256 + ((ch ^ (kr & 7)) << 4)), b0, b1, b2, b3);
        }
        mma_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  // epilogue: bf16 pairs
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = col0 + wc * ncol_w + nt * 8 + 2 * q;
    if (ok_lo)
      *reinterpret_cast<uint32_t*>(C + (size_t)(r_lo * H + h) * c_stride_row + col) =
          pack_bf16(acc[nt][0], acc[nt][1]);
    if (ok_hi)
      *reinterpret_cast<uint32_t*>(C + (size_t)(r_hi * H + h) * c_stride_row + col) =
          pack_bf16(acc[nt][2], acc[nt][3]);
  }
  if (ROPE && blockIdx.y == 0) {
    // rotate-half RoPE of q_pe into q_abs[..., 512:576] for this CTA's rows
    for (int i = tid; i < ROWS * 32; i += 128) {
      const int r = row0 + i / 32, p = i % 32;
      if (r >= num_q) continue;
      const __nv_bfloat16* x = q_pe + (size_t)(r * H + h) * kDr;
      const float x1 = __bfloat162float(x[p]), x2 = __bfloat162float(x[p + 32]);
      float cs, sn;
      rope_cos_sin(q_pos[r], p, kDr, base, &cs, &sn);
      __nv_bfloat16* o = C + (size_t)(r * H + h) * c_stride_row + kDc;
      o[p] = __float2bfloat16_rn(x1 * cs - x2 * sn);
      o[p + 32] = __float2bfloat16_rn(x2 * cs + x1 * sn);
    }
  }
}

// fp32 SIMT: one CTA per (row n, head h).
__global__ void __launch_bounds__(128) absorb_f32_kernel(
    const float* __restrict__ q_nope, const float* __restrict__ q_pe,
    const int32_t* __restrict__ q_pos, const float* __restrict__ W_uk, float* __restrict__ q_abs,
    int H, double base) {
  __shared__ float sq[kDn];
  const int n = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
  sq[t] = q_nope[((size_t)n * H + h) * kDn + t];
  __syncthreads();
  float* out = q_abs + ((size_t)n * H + h) * kRow;
  for (int c = t; c < kDc; c += 128) {
    const float* w = W_uk + ((size_t)h * kDc + c) * kDn;
    float s = 0.f;
    for (int d = 0; d < kDn; ++d) s = fmaf(w[d], sq[d], s);
    out[c] = s;
  }
  if (t < 32) {
    const float* x = q_pe + ((size_t)n * H + h) * kDr;
    float cs, sn;
    rope_cos_sin(q_pos[n], t, kDr, base, &cs, &sn);
    out[kDc + t] = x[t] * cs - x[t + 32] * sn;
    out[kDc + t + 32] = x[t + 32] * cs + x[t] * sn;
  }
}

__global__ void __launch_bounds__(128) out_proj_f32_kernel(const float* __restrict__ o_lat,
                                                           const float* __restrict__ W_uv,
                                                           float* __restrict__ out, int H) {
  __shared__ float so[kDc];
  const int n = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
  for (int c = t; c < kDc; c += 128) so[c] = o_lat[((size_t)n * H + h) * kDc + c];
  __syncthreads();
  const float* w = W_uv + (size_t)h * kDc * kDv + t;
  float s = 0.f;
  for (int c = 0; c < kDc; ++c) s = fmaf(so[c], w[(size_t)c * kDv], s);
  out[((size_t)n * H + h) * kDv + t] = s;
}

}  // namespace

cudaError_t launch_absorb_q(const mla_config& cfg, const void* q_nope, const void* q_pe,
                            const int32_t* q_positions, const void* W_uk, void* q_abs,
                            int64_t num_q, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  const int H = cfg.num_heads;
  if (cfg.dtype == MLA_F32) {
    absorb_f32_kernel<<<dim3((unsigned)num_q, H), 128, 0, stream>>>(
        (const float*)q_nope, (const float*)q_pe, q_positions, (const float*)W_uk, (float*)q_abs,
        H, (double)cfg.rope_base);
    return cudaGetLastError();
  }
  if (num_q >= 512) {
    head_gemm_kernel<4, false, false, true><<<dim3((unsigned)((num_q + 63) / 64), 4, H), 128, 0, stream>>>(
        q_nope, (const __nv_bfloat16*)W_uk, (__nv_bfloat16*)q_abs, (int)num_q, H, kDn, kDn, kRow,
        kDn, (const __nv_bfloat16*)q_pe, q_positions, (double)cfg.rope_base);
  } else {
    head_gemm_kernel<1, false, false, true><<<dim3((unsigned)((num_q + 15) / 16), 4, H), 128, 0, stream>>>(
        q_nope, (const __nv_bfloat16*)W_uk, (__nv_bfloat16*)q_abs, (int)num_q, H, kDn, kDn, kRow,
        kDn, (const __nv_bfloat16*)q_pe, q_positions, (double)cfg.rope_base);
  }
  return cudaGetLastError();
}

cudaError_t launch_out_proj(const mla_config& cfg, const float* o_lat, const void* W_uv,
                            void* out, int64_t num_q, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  const int H = cfg.num_heads;
  if (cfg.dtype == MLA_F32) {
    out_proj_f32_kernel<<<dim3((unsigned)num_q, H), 128, 0, stream>>>(o_lat, (const float*)W_uv,
                                                                   (float*)out, H);
    return cudaGetLastError();
  }
  if (num_q >= 512) {
    head_gemm_kernel<4, true, true, false><<<dim3((unsigned)((num_q + 63) / 64), 1, H), 128, 0, stream>>>(
        o_lat, (const __nv_bfloat16*)W_uv, (__nv_bfloat16*)out, (int)num_q, H, kDc, kDc, kDv, kDv,
        nullptr, nullptr, 0.0);
  } else {
    head_gemm_kernel<1, true, true, false><<<dim3((unsigned)((num_q + 15) / 16), 1, H), 128, 0, stream>>>(
        o_lat, (const __nv_bfloat16*)W_uv, (__nv_bfloat16*)out, (int)num_q, H, kDc, kDc, kDv, kDv,
        nullptr, nullptr, 0.0);
  }
  return cudaGetLastError();
}

}  // namespace mla
