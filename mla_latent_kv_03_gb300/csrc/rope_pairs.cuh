// The RoPE pairing: pair p (p < 32, frequency inv_freq_p) rotates elements
// (p, p + 32) (rotate-half, the default) or, interleaved, (2p, 2p + 1):
// x[rope_i1] -> x1 cos - x2 sin and x[rope_i2] -> x2 cos + x1 sin. The same
// pairing applies to k_pe and q_pe, so scores depend only on the relative
// position either way.
#pragma once

namespace mla {

__device__ __forceinline__ int rope_i1(int interleaved, int p) { return interleaved ? 2 * p : p; }
__device__ __forceinline__ int rope_i2(int interleaved, int p) {
  return interleaved ? 2 * p + 1 : p + 32;
}

}  // namespace mla
