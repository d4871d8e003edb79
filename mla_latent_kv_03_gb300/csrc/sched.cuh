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

}  // namespace mla
