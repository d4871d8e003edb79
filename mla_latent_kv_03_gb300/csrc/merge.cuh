// Merge of split-KV partials inside a decode kernel (the fused combine).
//
// Each CTA that finishes its part of a q-tile (query row n, 16-head group g)
// publishes its normalised partial and log-sum-exp, then counts itself in
// arrive[t] (release: __threadfence before the atomic). The CTA that brings
// the count to the number of parts merges all of them (acquire:
// __threadfence after the atomic) with the split-softmax identity
//   o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s,
// while they are still in L2. A q-tile that lies inside one CTA's share is
// written to o_lat directly and never touches the partial buffers.
#pragma once

#include "common.cuh"

namespace mla {

constexpr int kMergeChunk = 16;  // slots whose weights are staged at a time

// Scratch: 32 + kMergeChunk * 16 floats of shared memory.
// `sync` synchronises the `nthreads` participating threads (tid in [0, nthreads)).
template <int NTHREADS, typename Sync>
__device__ __forceinline__ void merge_qtile(const float* __restrict__ lse,
                                            const float* __restrict__ opart, int64_t slot0,
                                            int nslots, float* __restrict__ out, int tid,
                                            float* scratch, Sync sync) {
  constexpr int kItems = kHG * kDc / 4 / NTHREADS;  // float4 items per thread
  float* sM = scratch;
  float* sInv = scratch + kHG;
  float* sW = scratch + 2 * kHG;
  if (tid < kHG) {
    float M = -INFINITY;
    for (int s = 0; s < nslots; ++s) M = fmaxf(M, lse[(slot0 + s) * kHG + tid]);
    float den = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < nslots; ++s) den += fast_exp2(lse[(slot0 + s) * kHG + tid] - M);
    sM[tid] = M;
    sInv[tid] = den > 0.f ? 1.f / den : 0.f;
  }
  float4 acc[kItems];
#pragma unroll
  for (int j = 0; j < kItems; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* op = reinterpret_cast<const float4*>(opart);
  for (int s0 = 0; s0 < nslots; s0 += kMergeChunk) {
    const int ns = min(kMergeChunk, nslots - s0);
    sync();
    for (int i = tid; i < ns * kHG; i += NTHREADS) {
      const int r = i % kHG;
      const float M = sM[r];
      sW[i] = M == -INFINITY ? 0.f : fast_exp2(lse[(slot0 + s0 + i / kHG) * kHG + r] - M) * sInv[r];
    }
    sync();
    for (int s = 0; s < ns; ++s) {
      const float4* src = op + (slot0 + s0 + s) * (kHG * kDc / 4);
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int item = tid + j * NTHREADS;
        const float w = sW[s * kHG + item / (kDc / 4)];
        const float4 v = src[item];
        acc[j].x = fmaf(w, v.x, acc[j].x);
        acc[j].y = fmaf(w, v.y, acc[j].y);
        acc[j].z = fmaf(w, v.z, acc[j].z);
        acc[j].w = fmaf(w, v.w, acc[j].w);
      }
    }
  }
  float4* o4 = reinterpret_cast<float4*>(out);
#pragma unroll
  for (int j = 0; j < kItems; ++j) o4[tid + j * NTHREADS] = acc[j];
}

// Zero the o_lat rows that no CTA visits (query rows with no visible token),
// or every row when the workspace holds no plan for this launch. Rows are
// dealt out over CTAs; all `nthreads` threads of the CTA take part.
__device__ __forceinline__ void zero_unvisited_rows(const int4* row_info, bool plan_ok,
                                                    int64_t num_q, int heads, float* o_lat,
                                                    int tid, int nthreads) {
  for (int64_t n = blockIdx.x; n < num_q; n += gridDim.x) {
    if (plan_ok && row_info[n].z > 0) continue;
    float4* row = reinterpret_cast<float4*>(o_lat + (size_t)n * heads * kDc);
    for (int i = tid; i < heads * kDc / 4; i += nthreads) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

}  // namespace mla
