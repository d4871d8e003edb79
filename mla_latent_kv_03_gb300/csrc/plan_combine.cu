// Split-KV partition (plan), the merge of split partials (combine), and the
// bounded-wait self-test.
//
// Work units. Query row n of sequence b sits at position pos_n and sees
// tiles(n) = ceil((pos_n + 1) / 64) tiles of 64 kv tokens. A q-tile is
// (row n, head group g) with 16 heads; q-tiles are ordered t = n * G + g and
// each owns tiles(n) consecutive units. The plan cuts the ordered unit list
// into num_ctas equal contiguous shares (one persistent CTA per share), so a
// ragged batch is balanced to within one unit per CTA.
//
// Combine follows the split-softmax identity (flash-decoding): for partials
// o_s (normalised) with base-2 log-sum-exp lse_s,
//   o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s.
#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  extern __shared__ int s_units[];  // num_q + 1 entries: units per row, then prefix
  __shared__ int s_warp[32];
  const int tid = threadIdx.x;
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const WsLayout L = ws_layout(a.num_q, a.groups, a.num_ctas);
  int4* row_info = reinterpret_cast<int4*>(ws + L.row_info);
  int4* cta_start = reinterpret_cast<int4*>(ws + L.cta_start);
  const int Nq = a.num_q;
  pdl_wait();
  pdl_launch_dependents();

  int* arrive = reinterpret_cast<int*>(ws + L.arrive);
  for (int n = tid; n < Nq; n += kPlanThreads) {
    row_info[n] = make_int4(-1, -1, 0, 0);
    s_units[n] = 0;
  }
  for (int i = tid; i < Nq * a.groups; i += kPlanThreads) arrive[i] = 0;
  __syncthreads();
  const int64_t max_len = (int64_t)a.max_blocks_per_seq * a.block_size;
  for (int b = tid; b < a.batch; b += kPlanThreads) {
    const int len = a.seq_lens[b];
    const int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1];
    const int ql = q1 - q0;
    if (q0 < 0 || q1 > Nq || ql < 0) {
      set_status(&hdr->status, MLA_DEV_BAD_SEQ);
      continue;
    }
    const bool bad = ql > len || len < 0 || (int64_t)len > max_len;
    if (bad && ql > 0) set_status(&hdr->status, MLA_DEV_BAD_SEQ);
    for (int j = 0; j < ql; ++j) {
      const int n = q0 + j;
      const int pos = len - ql + j;
      const int tiles = bad ? 0 : (pos + kTile) / kTile;  // ceil((pos + 1) / 64)
      row_info[n] = make_int4(b, pos, tiles, 0);
      s_units[n] = tiles * a.groups;
    }
  }
  __syncthreads();

  // exclusive scan of s_units[0..Nq) in place; s_units[Nq] = total
  const int per = (Nq + kPlanThreads - 1) / kPlanThreads;
  const int beg = min(Nq, tid * per), end = min(Nq, beg + per);
  int local = 0;
  for (int i = beg; i < end; ++i) local += s_units[i];
  // block exclusive scan of `local`
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int run = incl - local + (warp > 0 ? s_warp[warp - 1] : 0);
  const int total = s_warp[31];
  __syncthreads();
  for (int i = beg; i < end; ++i) {
    const int u = s_units[i];
    s_units[i] = run;
    run += u;
  }
  if (tid == 0) s_units[Nq] = total;
  __syncthreads();
  for (int n = tid; n < Nq; n += kPlanThreads) row_info[n].w = s_units[n];

  const int C = a.num_ctas;
  const int share = total > 0 ? (total + C - 1) / C : 1;
  if (tid == 0) {
    hdr->magic = kMagic;
    hdr->mode = 0;
    hdr->qblocks = 0;
    hdr->total_units = total;
    hdr->share = share;
    hdr->num_ctas = C;
    hdr->groups = a.groups;
    hdr->num_q = Nq;
    hdr->batch = a.batch;
  }
  for (int c = tid; c < C; c += kPlanThreads) {
    const int u0 = c * share;
    if (u0 >= total) {
      cta_start[c] = make_int4(-1, 0, 0, 0);
      continue;
    }
    // last row n with start[n] <= u0 (that row has tiles > 0)
    int lo = 0, hi = Nq;  // invariant: start[lo] <= u0 < start[hi]  (start[Nq] = total)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_units[mid] <= u0) lo = mid; else hi = mid;
    }
    const int tiles = (s_units[lo + 1] - s_units[lo]) / a.groups;
    const int off = u0 - s_units[lo];
    cta_start[c] = make_int4(lo, off / tiles, off % tiles, 0);
  }
}

// Block-wide exclusive scan of data[0..n) in place (kPlanThreads threads);
// returns the total. `scratch` holds 32 ints.
__device__ int block_exclusive_scan(int* data, int n, int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kPlanThreads - 1) / kPlanThreads;
  const int beg = min(n, tid * per), end = min(n, beg + per);
  int local = 0;
  for (int i = beg; i < end; ++i) local += data[i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  int run = incl - local + (warp > 0 ? scratch[warp - 1] : 0);
  const int total = scratch[31];
  for (int i = beg; i < end; ++i) {
    const int u = data[i];
    data[i] = run;
    run += u;
  }
  __syncthreads();
  return total;
}

// Plan for the tensor-core kernel (mode 1): q-blocks of 8 consecutive q-tiles
// of one sequence; units = (q-block, 64-token tile), a q-block owning the tiles
// its last row sees; `shares` equal contiguous shares of the unit list.
__global__ void __launch_bounds__(kPlanThreads) plan_tc_kernel(PlanArgs a) {
  extern __shared__ int s_tc[];  // [batch + 1] blocks per sequence, then [qb_max + 1] units
  __shared__ int s_scan[32];
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int shares = a.num_ctas / 2;
  const int G = a.groups, B = a.batch, Nq = a.num_q;
  const WsLayoutTc L = ws_layout_tc(Nq, G, shares, B);
  int4* row_info = reinterpret_cast<int4*>(ws + L.row_info);
  int4* seq_info = reinterpret_cast<int4*>(ws + L.seq_info);
  int4* qblock = reinterpret_cast<int4*>(ws + L.qblock);
  int4* cta_start = reinterpret_cast<int4*>(ws + L.cta_start);
  int* arrive = reinterpret_cast<int*>(ws + L.arrive);
  int* s_nb = s_tc;
  int* s_units = s_tc + B + 1;
  const int qb_max = (int)L.qblocks_max;

  for (int n = tid; n < Nq; n += kPlanThreads) row_info[n] = make_int4(-1, -1, 0, 0);
  for (int i = tid; i < qb_max * 2; i += kPlanThreads) arrive[i] = 0;
  __syncthreads();
  const int64_t max_len = (int64_t)a.max_blocks_per_seq * a.block_size;
  for (int b = tid; b < B; b += kPlanThreads) {
    const int len = a.seq_lens[b];
    const int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1];
    const int ql = q1 - q0;
    int nb = 0;
    if (q0 < 0 || q1 > Nq || ql < 0) {
      set_status(&hdr->status, MLA_DEV_BAD_SEQ);
    } else {
      const bool bad = ql > len || len < 0 || (int64_t)len > max_len;
      if (bad && ql > 0) set_status(&hdr->status, MLA_DEV_BAD_SEQ);
      if (!bad) {
        for (int j = 0; j < ql; ++j) {
          const int pos = len - ql + j;
          row_info[q0 + j] = make_int4(b, pos, (pos + kTile) / kTile, 0);
        }
        nb = (ql * G + kQBlockTiles - 1) / kQBlockTiles;
      }
    }
    s_nb[b] = nb;
  }
  __syncthreads();
  int total_blocks = block_exclusive_scan(s_nb, B, s_scan);   // s_nb[b] = first q-block of b
  if (total_blocks > qb_max) {  // overlapping query ranges: more blocks than the layout holds
    if (tid == 0) set_status(&hdr->status, MLA_DEV_BAD_SEQ);
    total_blocks = 0;
  }
  for (int b = tid; b < B && total_blocks > 0; b += kPlanThreads) {
    const int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1];
    const int nb = (b + 1 < B ? s_nb[b + 1] : total_blocks) - s_nb[b];
    const int t0 = q0 * G, t_end = q1 * G;
    seq_info[b] = make_int4(t0, s_nb[b], t_end, 0);
    for (int k = 0; k < nb; ++k) {
      const int t_first = t0 + k * kQBlockTiles;
      const int t_last = min(t_first + kQBlockTiles, t_end) - 1;
      const int tiles = row_info[t_last / G].z;   // the block's last row sees the most tokens
      qblock[s_nb[b] + k] = make_int4(b, t_first, tiles, 0);
      s_units[s_nb[b] + k] = tiles;
    }
  }
  __syncthreads();
  const int total = block_exclusive_scan(s_units, total_blocks, s_scan);
  for (int qb = tid; qb < total_blocks; qb += kPlanThreads) qblock[qb].w = s_units[qb];
  if (tid == 0) s_units[total_blocks] = total;
  __syncthreads();
  const int share = total > 0 ? (total + shares - 1) / shares : 1;
  if (tid == 0) {
    hdr->magic = kMagic;
    hdr->mode = 1;
    hdr->qblocks = total_blocks;
    hdr->total_units = total;
    hdr->share = share;
    hdr->num_ctas = a.num_ctas;
    hdr->groups = G;
    hdr->num_q = Nq;
    hdr->batch = B;
  }
  for (int c = tid; c < shares; c += kPlanThreads) {
    const int u0 = c * share;
    if (u0 >= total) {
      cta_start[c] = make_int4(-1, 0, 0, 0);
      continue;
    }
    int lo = 0, hi = total_blocks;  // start[lo] <= u0 < start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_units[mid] <= u0) lo = mid; else hi = mid;
    }
    cta_start[c] = make_int4(lo, u0 - s_units[lo], 0, 0);
  }
}

// CTA = (q-tile t = (query row n, head group g), quarter of the 512 latent
// dims): 16 head rows x 128 dims. The slots' log-sum-exps go to shared memory
// 64 slots at a time, all (slot, row) values of a chunk loaded at once; threads
// 0-15 fold each chunk into their row's running maximum and weight sum. The
// per-(slot, row) weights are then staged the same way, and each thread merges
// 4 float4 items (row, 4 dims), with the loads of 4 slots in flight together.
constexpr int kCombineThreads = 128;
constexpr int kSlotChunk = 64;
constexpr int kSlotsInFlight = 4;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const uint8_t* __restrict__ ws, int groups, int num_ctas, int64_t num_q, int batch,
    float* __restrict__ o_lat) {
  __shared__ float sM[kHG], sInv[kHG];
  __shared__ float sW[kSlotChunk][kHG];
  pdl_wait();  // everything below reads what the decode kernel wrote
  pdl_launch_dependents();
  const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
  const size_t lse_off = hdr->mode == 0 ? ws_layout(num_q, groups, num_ctas).lse
                                        : ws_layout_tc(num_q, groups, num_ctas / 2, batch).lse;
  const size_t op_off = hdr->mode == 0 ? ws_layout(num_q, groups, num_ctas).opart
                                       : ws_layout_tc(num_q, groups, num_ctas / 2, batch).opart;
  const float* lse = reinterpret_cast<const float*>(ws + lse_off);
  const float4* opart = reinterpret_cast<const float4*>(ws + op_off);
  const int t = blockIdx.x, quarter = blockIdx.y, tid = threadIdx.x;
  const int n = t / groups, g = t % groups;
  const int H = groups * kHG;
  // item j of this thread: row (tid / 32) + 4 j, float4 column (tid % 32) of this quarter
  const int c4 = quarter * 32 + (tid & 31);
  float4* out = reinterpret_cast<float4*>(o_lat + ((size_t)n * H + g * kHG) * kDc);
  const QtileParts qp = locate_qtile(ws, num_q, groups, num_ctas, batch, n, g);
  if (qp.count <= 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) out[((tid >> 5) + 4 * j) * (kDc / 4) + c4] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int nslots = qp.count;
  auto grp = [&](int s) { return qp.first + (int64_t)s * qp.stride; };
  // pass 1: per-row maximum and weight sum, online over chunks of slots
  if (tid < kHG) { sM[tid] = -INFINITY; sInv[tid] = 0.f; }
  for (int s0 = 0; s0 < nslots; s0 += kSlotChunk) {
    const int ns = min(kSlotChunk, nslots - s0);
    __syncthreads();
    for (int i = tid; i < ns * kHG; i += kCombineThreads)
      sW[i / kHG][i % kHG] = lse[grp(s0 + i / kHG) * kHG + i % kHG];
    __syncthreads();
    if (tid < kHG) {
      const float Mold = sM[tid];
      float M = Mold;
      for (int sl = 0; sl < ns; ++sl) M = fmaxf(M, sW[sl][tid]);
      float den = 0.f;
      if (M != -INFINITY) {
        den = Mold == -INFINITY ? 0.f : sInv[tid] * fast_exp2(Mold - M);
        for (int sl = 0; sl < ns; ++sl) den += fast_exp2(sW[sl][tid] - M);
      }
      sM[tid] = M;
      sInv[tid] = den;   // a running sum; inverted below
    }
  }
  __syncthreads();
  if (tid < kHG) sInv[tid] = sInv[tid] > 0.f ? 1.f / sInv[tid] : 0.f;
  // pass 2: weighted sum of the partial rows
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < nslots; s0 += kSlotChunk) {
    const int ns = min(kSlotChunk, nslots - s0);
    __syncthreads();
    for (int i = tid; i < ns * kHG; i += kCombineThreads) {
      const int sl = i / kHG, r = i % kHG;
      const float M = sM[r];
      sW[sl][r] = M == -INFINITY ? 0.f : fast_exp2(lse[grp(s0 + sl) * kHG + r] - M) * sInv[r];
    }
    __syncthreads();
    for (int sl0 = 0; sl0 < ns; sl0 += kSlotsInFlight) {
      float4 v[kSlotsInFlight][4];
#pragma unroll
      for (int u = 0; u < kSlotsInFlight; ++u) {
        if (sl0 + u < ns) {
          const float4* src = opart + grp(s0 + sl0 + u) * kHG * (kDc / 4);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[u][j] = src[((tid >> 5) + 4 * j) * (kDc / 4) + c4];
        }
      }
#pragma unroll
      for (int u = 0; u < kSlotsInFlight; ++u) {
        if (sl0 + u < ns) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float w = sW[sl0 + u][(tid >> 5) + 4 * j];
            acc[j].x = fmaf(w, v[u][j].x, acc[j].x);
            acc[j].y = fmaf(w, v[u][j].y, acc[j].y);
            acc[j].z = fmaf(w, v[u][j].z, acc[j].z);
            acc[j].w = fmaf(w, v[u][j].w, acc[j].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) out[((tid >> 5) + 4 * j) * (kDc / 4) + c4] = acc[j];
}

__global__ void wait_timeout_selftest_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Nothing arrives on `bar`: the bounded wait must give up and report.
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, timeout_ns)) set_status(status, MLA_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_plan_tc(const PlanArgs& a, cudaStream_t stream) {
  const int64_t qb_max = ws_layout_tc(a.num_q, a.groups, a.num_ctas / 2, a.batch).qblocks_max;
  const size_t smem = ((size_t)a.batch + 1 + (size_t)qb_max + 1) * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(plan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(plan_tc_kernel, dim3(1), dim3(kPlanThreads), smem, stream, a);
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
  const size_t smem = ((size_t)a.num_q + 1) * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), smem, stream, a);
}

cudaError_t launch_combine(const void* workspace, int32_t groups, int32_t num_ctas,
                           int64_t num_q, int32_t batch, float* o_lat, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  return launch_pdl(combine_kernel, dim3((unsigned)(num_q * groups), 4), dim3(kCombineThreads), 0,
                    stream, (const uint8_t*)workspace, groups, num_ctas, num_q, (int)batch, o_lat);
}

cudaError_t launch_wait_timeout_selftest(uint32_t* status, int64_t timeout_ns,
                                         cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, (uint64_t)timeout_ns);
  return cudaGetLastError();
}

}  // namespace mla
