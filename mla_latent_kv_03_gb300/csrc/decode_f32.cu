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
  int64_t* sOff = reinterpret_cast<int64_t*>(sFlag + 2);   // [kSub] cache offsets (8-aligned)
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
        // stage 16 rows; rows that are not visible or not mapped become 0.
        // The rows' cache offsets are looked up once, then every float4 of
        // the 16 rows is loaded in one round trip.
        if (tid < kSub) {
          const int tok = tok0 + tid;
          int64_t off = -1;
          if (tok < visible) {
            const int blk = a.block_table[(size_t)seg.b * a.max_blocks_per_seq + tok / a.block_size];
            if (blk >= 0 && blk < a.num_blocks)
              off = ((int64_t)blk * a.block_size + tok % a.block_size) * kRow;
          }
          sOff[tid] = off;
        }
        __syncthreads();
        {
          constexpr int kVec = kSub * (kRow / 4) / 256;   // float4 per thread (9)
          float4 v[kVec];
#pragma unroll
          for (int u = 0; u < kVec; ++u) {
            const int i = tid + 256 * u, r = i / (kRow / 4), c4 = i % (kRow / 4);
            const int64_t off = sOff[r];
            v[u] = off >= 0 ? *reinterpret_cast<const float4*>(cache + off + 4 * c4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < kVec; ++u) {
            const int i = tid + 256 * u, r = i / (kRow / 4), c4 = i % (kRow / 4);
            float* d = sK + r * (kRow + 1) + 4 * c4;
            d[0] = v[u].x; d[1] = v[u].y; d[2] = v[u].z; d[3] = v[u].w;
          }
        }
        __syncthreads();
        const int tok = tok0 + j;
        bool live = tok < visible;
        if (live && sOff[j] < 0) {
          live = false;
          if (h == 0) set_status(&hdr->status, MLA_DEV_BAD_BLOCK);
        }
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        for (int c = 0; c < kRow; c += 4) {
          s0 = fmaf(sQ[h * kRow + c], sK[j * (kRow + 1) + c], s0);
          s1 = fmaf(sQ[h * kRow + c + 1], sK[j * (kRow + 1) + c + 1], s1);
          s2 = fmaf(sQ[h * kRow + c + 2], sK[j * (kRow + 1) + c + 2], s2);
          s3 = fmaf(sQ[h * kRow + c + 3], sK[j * (kRow + 1) + c + 3], s3);
        }
        float s = (s0 + s1) + (s2 + s3);
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
      __threadfence();   // publish protocol: see count_arrival
      __syncthreads();
      if (tid == 0) sFlag[0] = count_arrival(&arrive[t]) == c_last - c_first;
      __syncthreads();
      if (sFlag[0]) {
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
      (size_t)(kHG * kRow + kSub * (kRow + 1) + kHG * kSub + 3 * kHG + 2 * kHG + kMergeChunk * kHG + 2) * 4 +
      kSub * 8;
  cudaError_t e = cudaFuncSetAttribute(decode_f32_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_f32_kernel<<<a.num_ctas, 256, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
