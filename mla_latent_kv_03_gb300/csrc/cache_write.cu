// mla_cache_write: kv_a_layernorm (RMSNorm) of the compressed latent, RoPE of
// the shared key k_pe, and a scatter of [c_hat || k_hat] into the paged cache
// at slot_mapping. Sources: "07. MLA / Mamba / MoE in vLLM source" sections
// 2.2 (write c_kv by slot_mapping) and 2.3 (cache shape (n_blocks, block, 1,
// latent_d + rope_d)); "mini-infer-17: MLA Attention" sections "版本 1"
// (kv_a_layernorm before kv_b_proj), pitfall 3, and "MLA 的数学结构"
// (K_pe = x W_kr + RoPE, shared by all heads).
//
// One warp per token. Lane l holds latent values [16l, 16l+16) (16-byte
// vector loads and stores) and the RoPE pair (l, l+32). HBM-bound: reads and
// writes 1,152 bytes per token (bf16); 8 warps per CTA, grid-stride.
#include <cuda_fp8.h>

#include "async_copy.cuh"
#include "common.cuh"
#include "rope_pairs.cuh"
#include "internal.h"

namespace mla {
namespace {

template <typename T>
struct Vec16;  // 16 values of T as 16-byte vectors
template <>
struct Vec16<__nv_bfloat16> {
  uint4 v[2];
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    v[0] = reinterpret_cast<const uint4*>(p)[0];
    v[1] = reinterpret_cast<const uint4*>(p)[1];
  }
  __device__ __forceinline__ float get(int i) const {
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(v);
    return __bfloat162float(e[i]);
  }
  __device__ __forceinline__ void set(int i, float x) {
    reinterpret_cast<__nv_bfloat16*>(v)[i] = __float2bfloat16_rn(x);
  }
  __device__ __forceinline__ void store(__nv_bfloat16* p) const {
    reinterpret_cast<uint4*>(p)[0] = v[0];
    reinterpret_cast<uint4*>(p)[1] = v[1];
  }
};
template <>
struct Vec16<float> {
  float4 v[4];
  __device__ __forceinline__ void load(const float* p) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = reinterpret_cast<const float4*>(p)[i];
  }
  __device__ __forceinline__ float get(int i) const { return reinterpret_cast<const float*>(v)[i]; }
  __device__ __forceinline__ void set(int i, float x) { reinterpret_cast<float*>(v)[i] = x; }
  __device__ __forceinline__ void store(float* p) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) reinterpret_cast<float4*>(p)[i] = v[i];
  }
};

template <typename T>
__global__ void __launch_bounds__(256) cache_write_kernel(
    const T* __restrict__ c_kv, const T* __restrict__ k_pe, const int32_t* __restrict__ positions,
    const int64_t* __restrict__ slot_mapping, int64_t num_tokens, const T* __restrict__ w,
    T* __restrict__ cache, int64_t num_slots, float eps, RopeFreq freq, int interleaved,
    uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  Vec16<T> wv;
  wv.load(w + lane * 16);
  const float fhi = freq.hi[lane], flo = freq.lo[lane];
  for (int64_t t = warp0; t < num_tokens; t += nwarps) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (lane == 0) set_status(status, MLA_DEV_BAD_SLOT);
      continue;
    }
    Vec16<T> x;
    x.load(c_kv + t * kDc + lane * 16);
    const T* kp = k_pe + t * kDr;
    const int i1 = rope_i1(interleaved, lane), i2 = rope_i2(interleaved, lane);
    const float x1 = to_f32(kp[i1]), x2 = to_f32(kp[i2]);
    const int pos = positions[t];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(x.get(i), x.get(i), ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss * (1.0f / kDc) + eps);
    Vec16<T> y;
#pragma unroll
    for (int i = 0; i < 16; ++i) y.set(i, x.get(i) * r * wv.get(i));
    T* dst = cache + slot * kRow;
    y.store(dst + lane * 16);
    float cs, sn;
    rope_cos_sin(pos, fhi, flo, &cs, &sn);
    dst[kDc + i1] = from_f32<T>(x1 * cs - x2 * sn);
    dst[kDc + i2] = from_f32<T>(x2 * cs + x1 * sn);
  }
}

// The FP8 cache row (640 bytes): e4m3 codes of c_hat / kv_scale (round to
// nearest even, saturating at +-448), then k_rot in bf16. Inputs bf16.
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(
    const __nv_bfloat16* __restrict__ c_kv, const __nv_bfloat16* __restrict__ k_pe,
    const int32_t* __restrict__ positions, const int64_t* __restrict__ slot_mapping,
    int64_t num_tokens, const __nv_bfloat16* __restrict__ w, uint8_t* __restrict__ cache8,
    int64_t num_slots, float eps, float inv_scale, RopeFreq freq, int interleaved,
    uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  Vec16<__nv_bfloat16> wv;
  wv.load(w + lane * 16);
  const float fhi = freq.hi[lane], flo = freq.lo[lane];
  for (int64_t t = warp0; t < num_tokens; t += nwarps) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (lane == 0) set_status(status, MLA_DEV_BAD_SLOT);
      continue;
    }
    Vec16<__nv_bfloat16> x;
    x.load(c_kv + t * kDc + lane * 16);
    const __nv_bfloat16* kp = k_pe + t * kDr;
    const int i1 = rope_i1(interleaved, lane), i2 = rope_i2(interleaved, lane);
    const float x1 = __bfloat162float(kp[i1]), x2 = __bfloat162float(kp[i2]);
    const int pos = positions[t];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(x.get(i), x.get(i), ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss * (1.0f / kDc) + eps);
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = make_float2(x.get(4 * i) * r * wv.get(4 * i) * inv_scale,
                                   x.get(4 * i + 1) * r * wv.get(4 * i + 1) * inv_scale);
      const float2 b = make_float2(x.get(4 * i + 2) * r * wv.get(4 * i + 2) * inv_scale,
                                   x.get(4 * i + 3) * r * wv.get(4 * i + 3) * inv_scale);
      q[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3) |
             ((uint32_t)__nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3) << 16);
    }
    uint8_t* dst = cache8 + slot * kRow8;
    *reinterpret_cast<uint4*>(dst + lane * 16) = make_uint4(q[0], q[1], q[2], q[3]);
    float cs, sn;
    rope_cos_sin(pos, fhi, flo, &cs, &sn);
    __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(dst + kDc);
    kr[i1] = __float2bfloat16_rn(x1 * cs - x2 * sn);
    kr[i2] = __float2bfloat16_rn(x2 * cs + x1 * sn);
  }
}

}  // namespace

cudaError_t launch_cache_write_fp8(const mla_config& cfg, const void* c_kv, const void* k_pe,
                                   const int32_t* positions, const int64_t* slot_mapping,
                                   int64_t num_tokens, const void* rms_weight, float kv_scale,
                                   void* cache8, int64_t num_blocks, uint32_t* dev_status,
                                   cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  int64_t blocks = (num_tokens + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(cache_write_fp8_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                    (const __nv_bfloat16*)c_kv, (const __nv_bfloat16*)k_pe, positions,
                    slot_mapping, num_tokens, (const __nv_bfloat16*)rms_weight, (uint8_t*)cache8,
                    num_blocks * cfg.block_size, cfg.rms_eps, 1.0f / kv_scale,
                    make_rope_freq((double)cfg.rope_base), cfg.rope_interleaved, dev_status);
}

cudaError_t launch_cache_write(const mla_config& cfg, const void* c_kv, const void* k_pe,
                               const int32_t* positions, const int64_t* slot_mapping,
                               int64_t num_tokens, const void* rms_weight, void* cache,
                               int64_t num_blocks, uint32_t* dev_status, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (num_tokens + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  const int64_t num_slots = num_blocks * cfg.block_size;
  const RopeFreq freq = make_rope_freq((double)cfg.rope_base);
  if (cfg.dtype == MLA_BF16) {
    return launch_pdl(cache_write_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(threads), 0,
                      stream, (const __nv_bfloat16*)c_kv, (const __nv_bfloat16*)k_pe, positions,
                      slot_mapping, num_tokens, (const __nv_bfloat16*)rms_weight,
                      (__nv_bfloat16*)cache, num_slots, cfg.rms_eps, freq, cfg.rope_interleaved,
                      dev_status);
  } else {
    return launch_pdl(cache_write_kernel<float>, dim3((unsigned)blocks), dim3(threads), 0, stream,
                      (const float*)c_kv, (const float*)k_pe, positions, slot_mapping, num_tokens,
                      (const float*)rms_weight, (float*)cache, num_slots, cfg.rms_eps, freq,
                      cfg.rope_interleaved, dev_status);
  }
  return cudaGetLastError();
}

}  // namespace mla
