// mla_cache_write: kv_a_layernorm (RMSNorm) of the compressed latent, RoPE of
// the shared key k_pe, and a scatter of [c_hat || k_hat] into the paged cache
// at slot_mapping. Sources: "07. MLA / Mamba / MoE in vLLM source" sections
// 2.2 (write c_kv by slot_mapping) and 2.3 (cache shape (n_blocks, block, 1,
// latent_d + rope_d)); "mini-infer-17: MLA Attention" sections "版本 1"
// (kv_a_layernorm before kv_b_proj), pitfall 3, and "MLA 的数学结构"
// (K_pe = x W_kr + RoPE, shared by all heads).
//
// One warp per token. Lane l holds latent values [16l, 16l+16) and the RoPE
// pair (l, l+32). HBM-bound: reads 1,152 (bf16) bytes and writes 1,152 per
// token; 8 warps per CTA, grid-stride over tokens.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) cache_write_kernel(
    const T* __restrict__ c_kv, const T* __restrict__ k_pe, const int32_t* __restrict__ positions,
    const int64_t* __restrict__ slot_mapping, int64_t num_tokens, const T* __restrict__ w,
    T* __restrict__ cache, int64_t num_slots, float eps, double base, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = warp0; t < num_tokens; t += nwarps) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (lane == 0) set_status(status, MLA_DEV_BAD_SLOT);
      continue;
    }
    // latent: 16 consecutive values per lane
    float x[16];
    const T* src = c_kv + t * kDc + lane * 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = to_f32(src[i]);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss * (1.0f / kDc) + eps);
    T* dst = cache + slot * kRow;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = lane * 16 + i;
      dst[c] = from_f32<T>(x[i] * r * to_f32(w[c]));
    }
    // rope: pair (lane, lane + 32)
    const T* kp = k_pe + t * kDr;
    const float x1 = to_f32(kp[lane]), x2 = to_f32(kp[lane + 32]);
    float cs, sn;
    rope_cos_sin(positions[t], lane, kDr, base, &cs, &sn);
    dst[kDc + lane] = from_f32<T>(x1 * cs - x2 * sn);
    dst[kDc + lane + 32] = from_f32<T>(x2 * cs + x1 * sn);
  }
}

}  // namespace

cudaError_t launch_cache_write(const mla_config& cfg, const void* c_kv, const void* k_pe,
                               const int32_t* positions, const int64_t* slot_mapping,
                               int64_t num_tokens, const void* rms_weight, void* cache,
                               int64_t num_blocks, uint32_t* dev_status, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (num_tokens + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  const int64_t num_slots = num_blocks * cfg.block_size;
  if (cfg.dtype == MLA_BF16) {
    cache_write_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, stream>>>(
        (const __nv_bfloat16*)c_kv, (const __nv_bfloat16*)k_pe, positions, slot_mapping,
        num_tokens, (const __nv_bfloat16*)rms_weight, (__nv_bfloat16*)cache, num_slots,
        cfg.rms_eps, (double)cfg.rope_base, dev_status);
  } else {
    cache_write_kernel<float><<<(unsigned)blocks, threads, 0, stream>>>(
        (const float*)c_kv, (const float*)k_pe, positions, slot_mapping, num_tokens,
        (const float*)rms_weight, (float*)cache, num_slots, cfg.rms_eps, (double)cfg.rope_base,
        dev_status);
  }
  return cudaGetLastError();
}

}  // namespace mla
