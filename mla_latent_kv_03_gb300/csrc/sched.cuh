// Walks one CTA's share of the split-KV unit list written by the plan kernel.
// Every role in a decode CTA (TMA producer, math warps) runs its own walker
// over the same data, so they agree on the order of segments and tiles
// without talking to each other.
#pragma once

#include "common.cuh"

namespace mla {

struct Segment {
  int n;       // query row
  int g;       // head group (16 heads)
  int k0, k1;  // tiles [k0, k1) of this row's causal range
  int b;       // sequence
  int pos;     // query position: tokens 0..pos are visible
  int tiles;   // tiles of this row's causal range
  int ustart;  // first unit of the row in the ordered unit list
};

struct SchedWalker {
  const int4* row_info;
  int u, u_end, n, g, k, G, share;
  bool plan_ok;  // the workspace holds a plan for this launch

  // false if this CTA has no work (or the workspace holds no plan)
  __device__ __forceinline__ bool init(const uint8_t* ws, int64_t num_q, int groups, int num_ctas,
                                       int c) {
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    const WsLayout L = ws_layout(num_q, groups, num_ctas);
    row_info = reinterpret_cast<const int4*>(ws + L.row_info);
    // the plan must describe this launch (same rows, head groups, CTAs)
    plan_ok = hdr->magic == kMagic && hdr->mode == 0 && hdr->num_q == num_q &&
              hdr->groups == groups && hdr->num_ctas == num_ctas;
    if (!plan_ok) return false;
    const int4* cta_start = reinterpret_cast<const int4*>(ws + L.cta_start);
    share = hdr->share;
    const int total = hdr->total_units;
    G = groups;
    u = c * share;
    u_end = min(u + share, total);
    if (u >= u_end) return false;
    const int4 cs = cta_start[c];
    n = cs.x; g = cs.y; k = cs.z;
    return n >= 0;
  }

  // The same walk over a plan held in shared memory (the self-planned
  // decode): rows[n] as in row_info, `total` units cut into num_ctas shares.
  __device__ __forceinline__ bool init_rows(const int4* rows, int num_q, int groups, int total,
                                            int num_ctas, int c) {
    row_info = rows;
    plan_ok = true;
    G = groups;
    share = total > 0 ? (total + num_ctas - 1) / num_ctas : 1;
    u = c * share;
    u_end = min(u + share, total);
    if (u >= u_end) return false;
    // last row whose first unit is <= u (it owns units: the next row's first
    // unit is above u)
    int lo = 0, hi = num_q;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (rows[mid].w <= u) lo = mid; else hi = mid;
    }
    const int tiles = rows[lo].z, off = u - rows[lo].w;
    n = lo; g = off / tiles; k = off % tiles;
    return true;
  }

  // true while segments remain after the ones next() returned so far
  __device__ __forceinline__ bool more() const { return u < u_end; }

  __device__ __forceinline__ bool next(Segment& s) {
    if (u >= u_end) return false;
    int4 ri = row_info[n];
    while (ri.z <= 0) {  // rows with no visible tokens own no units
      ++n; g = 0; k = 0;
      ri = row_info[n];
    }
    const int take = min(ri.z - k, u_end - u);
    s.n = n; s.g = g; s.k0 = k; s.k1 = k + take; s.b = ri.x; s.pos = ri.y;
    s.tiles = ri.z; s.ustart = ri.w;
    u += take;
    k += take;
    if (k == ri.z) {
      k = 0;
      if (++g == G) { g = 0; ++n; }
    }
    return true;
  }
};

// ---------------------------------------------------------------------------
// The split plan computed inside a decode CTA (no plan kernel): every CTA
// derives the same partition as plan_kernel from seq_lens / query_start_loc
// into shared memory. Query rows are limited to kSelfMaxRows so the plan fits
// beside the cache ring.
// ---------------------------------------------------------------------------
// rows[n] = {sequence, query position, tiles, first unit} for n < num_q, the
// same values plan_kernel writes to row_info. All NT threads of the CTA call
// it (it uses __syncthreads); `scratch` holds NT / 32 ints. Invalid sequences
// own no tiles; only CTA 0 reports them (MLA_DEV_BAD_SEQ). Returns the total
// number of units.
template <int NT>
__device__ __forceinline__ int self_plan(const int32_t* __restrict__ seq_lens,
                                         const int32_t* __restrict__ query_start_loc, int batch,
                                         int num_q, int groups, int64_t max_len, int4* rows,
                                         int* scratch, uint32_t* status, int tid) {
  for (int n = tid; n < num_q; n += NT) rows[n] = make_int4(-1, -1, 0, 0);
  __syncthreads();
  for (int b = tid; b < batch; b += NT) {
    const int len = seq_lens[b];
    const int q0 = query_start_loc[b], q1 = query_start_loc[b + 1];
    const int ql = q1 - q0;
    if (q0 < 0 || q1 > num_q || ql < 0) {
      if (blockIdx.x == 0) set_status(status, MLA_DEV_BAD_SEQ);
      continue;
    }
    const bool bad = ql > len || len < 0 || (int64_t)len > max_len;
    if (bad && ql > 0 && blockIdx.x == 0) set_status(status, MLA_DEV_BAD_SEQ);
    for (int j = 0; j < ql; ++j) {
      const int pos = len - ql + j;
      rows[q0 + j] = make_int4(b, pos, bad ? 0 : (pos + kTile) / kTile, 0);
    }
  }
  __syncthreads();
  // exclusive scan of tiles * groups over the rows (contiguous chunk per thread)
  const int lane = tid & 31, warp = tid >> 5;
  const int per = (num_q + NT - 1) / NT;
  const int beg = min(num_q, tid * per), end = min(num_q, beg + per);
  int local = 0;
  for (int i = beg; i < end; ++i) local += rows[i].z * groups;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  int run = incl - local, total = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) run += scratch[w];
    total += scratch[w];
  }
  for (int i = beg; i < end; ++i) {
    const int u = rows[i].z * groups;
    rows[i].w = run;
    run += u;
  }
  __syncthreads();
  return total;
}

}  // namespace mla
