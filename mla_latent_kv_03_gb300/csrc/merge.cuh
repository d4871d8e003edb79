// Merge of split-KV partials inside a decode kernel (the fused combine).
//
// Each CTA that finishes its part of a q-tile (query row n, 16-head group g)
// publishes its normalised partial and log-sum-exp, then counts itself in
// arrive[t] (count_arrival: per-thread fences, a CTA barrier, an
// acquire-release atomic). The CTA that brings the count to the number of
// parts merges all of them with the split-softmax identity
//   o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s,
// while they are still in L2. A q-tile that lies inside one CTA's share is
// written to o_lat directly and never touches the partial buffers.
#pragma once

#include "common.cuh"

namespace mla {

constexpr int kMergeChunk = 16;  // slots whose weights are staged at a time

// The parts are 16-row groups slot0, slot0 + stride, ... of the partial buffer.
// Scratch: 32 + kMergeChunk * 16 floats of shared memory. In a fused merge
// other CTAs of the same launch wrote the parts, so they are read through L2
// (ld.global.cg) and the pointers are not declared __restrict__ (which would
// let the compiler use the non-coherent read-only path).
// `sync` synchronises the `nthreads` participating threads (tid in [0, nthreads)).
// All (slot, row) log-sum-exps of a chunk are fetched in one parallel round
// trip; the partial rows of two slots are in flight at a time.
template <int NTHREADS, typename Sync>
__device__ __forceinline__ void merge_qtile(const float* lse, const float* opart, int64_t slot0,
                                            int nslots, int stride, float* out,
                                            int tid, float* scratch, Sync sync) {
  constexpr int kItems = kHG * kDc / 4 / NTHREADS;  // float4 items per thread
  float* sM = scratch;
  float* sInv = scratch + kHG;
  float* sW = scratch + 2 * kHG;
  // pass 1: per-row maximum and weight sum over all slots (online over chunks)
  if (tid < kHG) { sM[tid] = -INFINITY; sInv[tid] = 0.f; }
  for (int s0 = 0; s0 < nslots; s0 += kMergeChunk) {
    const int ns = min(kMergeChunk, nslots - s0);
    sync();
    for (int i = tid; i < ns * kHG; i += NTHREADS)
      sW[i] = __ldcg(lse + (slot0 + (int64_t)(s0 + i / kHG) * stride) * kHG + i % kHG);
    sync();
    if (tid < kHG) {
      const float Mold = sM[tid];
      float M = Mold;
      for (int s = 0; s < ns; ++s) M = fmaxf(M, sW[s * kHG + tid]);
      float den = 0.f;
      if (M != -INFINITY) {
        den = Mold == -INFINITY ? 0.f : sInv[tid] * fast_exp2(Mold - M);
        for (int s = 0; s < ns; ++s) den += fast_exp2(sW[s * kHG + tid] - M);
      }
      sM[tid] = M;
      sInv[tid] = den;  // running sum; inverted below
    }
  }
  sync();
  if (tid < kHG) sInv[tid] = sInv[tid] > 0.f ? 1.f / sInv[tid] : 0.f;
  // pass 2: weighted sum of the partial rows
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
      sW[i] = M == -INFINITY
                  ? 0.f
                  : fast_exp2(__ldcg(lse + (slot0 + (int64_t)(s0 + i / kHG) * stride) * kHG + r) - M) * sInv[r];
    }
    sync();
    for (int s = 0; s < ns; s += 2) {
      const bool two = s + 1 < ns;
      const float4* src0 = op + (slot0 + (int64_t)(s0 + s) * stride) * (kHG * kDc / 4);
      const float4* src1 = two ? src0 + (int64_t)stride * (kHG * kDc / 4) : src0;
      float4 v0[kItems], v1[kItems];
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        v0[j] = __ldcg(src0 + tid + j * NTHREADS);
        v1[j] = __ldcg(src1 + tid + j * NTHREADS);
      }
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int row = (tid + j * NTHREADS) / (kDc / 4);
        const float w0 = sW[s * kHG + row];
        const float w1 = two ? sW[(s + 1) * kHG + row] : 0.f;
        acc[j].x = fmaf(w1, v1[j].x, fmaf(w0, v0[j].x, acc[j].x));
        acc[j].y = fmaf(w1, v1[j].y, fmaf(w0, v0[j].y, acc[j].y));
        acc[j].z = fmaf(w1, v1[j].z, fmaf(w0, v0[j].z, acc[j].z));
        acc[j].w = fmaf(w1, v1[j].w, fmaf(w0, v0[j].w, acc[j].w));
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
