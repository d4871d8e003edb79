// fp32 split-KV latent attention on CUDA cores (no tensor cores: fp32 inputs
// are held to 1e-4 absolute, which bf16 or tf32 operands cannot meet).
// Same partition, partial layout and online softmax as the bf16 kernel; it
// serves the fp32 configuration, whose sizes are small.
// Source: "mini-infer-17: MLA Attention", sections "版本 3" (scores and
// output against the latent rows) and "设计取舍" (nope + rope score parts
// summed, then a hand-written softmax).
#include "common.cuh"
#include "internal.h"
#include "merge.cuh"
#include "sched.cuh"

namespace mla {
namespace {

constexpr int kSub = 16;  // tokens per inner step

__global__ void __launch_bounds__(256) decode_f32_kernel(DecodeArgs a) {
  extern __shared__ float smem_f[];
  float* sQ = smem_f;                         // [16][576]
  float* sK = sQ + kHG * kRow;                // [16][577]
  float* sP = sK + kSub * (kRow + 1);         // [16][16]
  float* sA = sP + kHG * kSub;                // [16] alpha
  float* sL = sA + kHG;                       // [16] final l
  float* sM = sL + kHG;                       // [16] final m
  float* sMerge = sM + kHG;                   // fused-merge scratch
  int* sFlag = reinterpret_cast<int*>(sMerge + 2 * kHG + kMergeChunk * kHG);
  const int tid = threadIdx.x;
  const int h = tid >> 4, j = tid & 15;       // score role: head h, token j
  const int d0 = tid * 2;                     // PV role: dims d0, d0+1 for all heads
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const WsLayout L = ws_layout(a.num_q, a.groups, a.num_ctas);
  float* lse_out = reinterpret_cast<float*>(ws + L.lse);
  float* o_out = reinterpret_cast<float*>(ws + L.opart);
  const float* q_abs = reinterpret_cast<const float*>(a.q_abs);
  const float* cache = reinterpret_cast<const float*>(a.cache);

  SchedWalker sw;
  const bool has_work = sw.init(ws, a.num_q, a.groups, a.num_ctas, blockIdx.x);
  if (a.o_lat) zero_unvisited_rows(sw.row_info, sw.plan_ok, a.num_q, a.num_heads, a.o_lat, tid, 256);
  if (!has_work) return;
  Segment seg;
  while (sw.next(seg)) {
    const int t = seg.n * a.groups + seg.g;
    const int64_t slot = (int64_t)blockIdx.x + t;
    __syncthreads();
    const float* qsrc = q_abs + ((size_t)seg.n * a.num_heads + seg.g * kHG) * kRow;
    for (int i = tid; i < kHG * kRow; i += 256) sQ[i] = qsrc[i];
    float m = -INFINITY, l = 0.f;
    float o[kHG][2];
#pragma unroll
    for (int r = 0; r < kHG; ++r) o[r][0] = o[r][1] = 0.f;
    const int visible = seg.pos + 1;
    for (int k = seg.k0; k < seg.k1; ++k) {
      for (int sub = 0; sub < kTile / kSub; ++sub) {
        const int tok0 = k * kTile + sub * kSub;
        if (tok0 >= visible) break;
        __syncthreads();
        // stage 16 rows; rows that are not visible or not mapped become 0
        for (int i = tid; i < kSub * kRow; i += 256) {
          const int r = i / kRow, c = i % kRow;
          const int tok = tok0 + r;
          float v = 0.f;
          if (tok < visible) {
            const int blk = a.block_table[(size_t)seg.b * a.max_blocks_per_seq + tok / a.block_size];
            if (blk >= 0 && blk < a.num_blocks)
              v = cache[((size_t)blk * a.block_size + tok % a.block_size) * kRow + c];
          }
          sK[r * (kRow + 1) + c] = v;
        }
        __syncthreads();
        const int tok = tok0 + j;
        bool live = tok < visible;
        if (live) {
          const int blk = a.block_table[(size_t)seg.b * a.max_blocks_per_seq + tok / a.block_size];
          if (blk < 0 || blk >= a.num_blocks) {
            live = false;
            if (h == 0) set_status(&hdr->status, MLA_DEV_BAD_BLOCK);
          }
        }
        float s = 0.f;
        for (int c = 0; c < kRow; ++c) s = fmaf(sQ[h * kRow + c], sK[j * (kRow + 1) + c], s);
        s = live ? s * a.scale_log2 : -INFINITY;
        float mx = s;
#pragma unroll
        for (int o2 = 8; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float mn = fmaxf(m, mx);
        const float mu = mn == -INFINITY ? 0.f : mn;
        const float alpha = fast_exp2(m - mu);
        const float p = fast_exp2(s - mu);
        float ps = p;
#pragma unroll
        for (int o2 = 8; o2 > 0; o2 >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o2);
        l = l * alpha + ps;
        m = mn;
        sP[h * kSub + j] = p;
        if (j == 0) sA[h] = alpha;
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kHG; ++r) {
          const float al = sA[r];
          float acc0 = o[r][0] * al, acc1 = o[r][1] * al;
          for (int jj = 0; jj < kSub; ++jj) {
            const float pj = sP[r * kSub + jj];
            acc0 = fmaf(pj, sK[jj * (kRow + 1) + d0], acc0);
            acc1 = fmaf(pj, sK[jj * (kRow + 1) + d0 + 1], acc1);
          }
          o[r][0] = acc0;
          o[r][1] = acc1;
        }
      }
    }
    __syncthreads();
    if (j == 0) { sL[h] = l; sM[h] = m; }
    __syncthreads();
    const int u_first = seg.ustart + seg.g * seg.tiles;
    const int c_first = u_first / sw.share, c_last = (u_first + seg.tiles - 1) / sw.share;
    const bool direct = a.o_lat != nullptr && c_first == c_last;
    float* dst = direct ? a.o_lat + ((size_t)seg.n * a.num_heads + seg.g * kHG) * kDc
                        : o_out + (size_t)slot * kHG * kDc;
#pragma unroll
    for (int r = 0; r < kHG; ++r) {
      const float lr = sL[r];
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
      float2 v = make_float2(o[r][0] * inv, o[r][1] * inv);
      *reinterpret_cast<float2*>(dst + (size_t)r * kDc + d0) = v;
    }
    if (!direct && tid < kHG) {
      const float lr = sL[tid];
      lse_out[(size_t)slot * kHG + tid] = lr > 0.f ? sM[tid] + log2f(lr) : -INFINITY;
    }
    if (a.o_lat != nullptr && !direct) {
      int* arrive = reinterpret_cast<int*>(ws + L.arrive);
      __threadfence();
      __syncthreads();
      if (tid == 0) sFlag[0] = atomicAdd(&arrive[t], 1) == c_last - c_first;
      __syncthreads();
      if (sFlag[0]) {
        __threadfence();
        merge_qtile<256>(lse_out, o_out, (int64_t)c_first + t, c_last - c_first + 1, 1,
                         a.o_lat + ((size_t)seg.n * a.num_heads + seg.g * kHG) * kDc, tid, sMerge,
                         [] { __syncthreads(); });
        if (tid == 0) arrive[t] = 0;  // every part has arrived: ready for the next launch
      }
      __syncthreads();
    }
  }
}

}  // namespace

cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t stream) {
  const size_t smem =
      (size_t)(kHG * kRow + kSub * (kRow + 1) + kHG * kSub + 3 * kHG + 2 * kHG + kMergeChunk * kHG + 4) * 4;
  cudaError_t e = cudaFuncSetAttribute(decode_f32_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_f32_kernel<<<a.num_ctas, 256, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
