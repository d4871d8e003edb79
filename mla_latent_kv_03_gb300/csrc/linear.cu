// The projections on either side of the attention: the hidden state to the
// query (q_nope, q_pe) and to the latent and rope key (c_kv, k_pe) that the
// cache write takes, and the attention output back to the hidden size.
// Source: "mini-infer-17: MLA Attention", section "版本 1: MLAAttentionNaive"
// (q_proj viewed as [H, qk_nope + qk_rope] per head and split; the
// kv_a_proj_with_mqa output split into the kv_lora_rank latent and the rope
// key; o_proj over the heads' concatenated values); "07. MLA / Mamba / MoE in
// vLLM source" 2.2 (the same projections around the MLA attention call).
//
// Y = X W^T with X [M, K] and W [N, K] row-major bf16 (a linear layer's
// weight), fp32 accumulation, bf16 out. A CTA owns a 64 x 64 tile of Y and a
// range of K: warp 4 streams the X and W tiles (64 x 64, SWIZZLE_128B, 8 KB
// each) by TMA through a 4-stage ring; warps 0-3 each own a 32 x 32 quarter
// (m16n8k16 warp mma, ldmatrix from the swizzled tiles). The weight tiles of
// the first stages are requested before the preceding kernel has finished
// (programmatic dependent launch); X waits for it. Few rows (a decode step)
// give too few tiles for the GPU, so K is split across a grid z dimension:
// every split writes fp32 partials and a second kernel adds them in split
// order (repeated calls agree bit for bit). Column n of Y goes to one of two
// outputs: with h = n / P and d = n % P, d < Q goes to y0[m][h][d] (row length
// (N / P) Q) and the rest to y1[m][h][d - Q] (row length (N / P) (P - Q)).
#include <cuda_bf16.h>

#include "async_copy.cuh"
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kLB = 64;                  // tile rows, columns and K step
constexpr int kLStages = 4;
constexpr int kLTile = kLB * 128;        // 64 rows x 64 bf16, 8 KB
constexpr int kLThreads = 160;           // 4 math warps + 1 producer warp
constexpr int kLMaxSplits = 8;           // K splits at most
constexpr int kLSmem = kLStages * 2 * kLTile + 2 * kLStages * 8 + 1024;

struct LinArgs {
  int64_t M;
  int32_t N, K;
  int32_t k_split;     // K per split (a multiple of 64)
  int32_t P, Q;        // column map, see above
  __nv_bfloat16* y0;
  __nv_bfloat16* y1;
  float* partial;      // [splits][M][N] fp32 when K is split, else null
  uint32_t* status;    // MLA_DEV_TIMEOUT when a wait gave up
};

__device__ __forceinline__ void store_pair(const LinArgs& a, int64_t m, int n, float v0, float v1) {
  const int h = n / a.P, d = n - h * a.P;
  const int H = a.N / a.P;
  __nv_bfloat162 v = __floats2bfloat162_rn(v0, v1);
  if (d < a.Q)
    *reinterpret_cast<__nv_bfloat162*>(a.y0 + (m * H + h) * a.Q + d) = v;
  else
    *reinterpret_cast<__nv_bfloat162*>(a.y1 + (m * H + h) * (a.P - a.Q) + (d - a.Q)) = v;
}

__global__ void __launch_bounds__(kLThreads)
    linear_kernel(const __grid_constant__ CUtensorMap x_map,
                  const __grid_constant__ CUtensorMap w_map, LinArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kLStages * 2 * kLTile);
  uint64_t* empty = full + kLStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kLB;
  const int64_t m0 = (int64_t)blockIdx.y * kLB;
  const int kbeg = blockIdx.z * a.k_split, nk = a.k_split / kLB;

  if (tid == 0) {
    for (int i = 0; i < kLStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 4) {
    if (lane != 0) return;
    prefetch_tensormap(&x_map);
    prefetch_tensormap(&w_map);
    // the weight needs no earlier kernel: its first tiles go out at once
    const int pre = nk < kLStages ? nk : kLStages;
    for (int kt = 0; kt < pre; ++kt) {
      mbar_arrive_expect_tx(&full[kt], 2 * kLTile);
      tma_load_2d(sm + (2 * kt + 1) * kLTile, &w_map, kbeg + kt * kLB, n0, &full[kt]);
    }
    pdl_wait();
    for (int kt = 0; kt < pre; ++kt)
      tma_load_2d(sm + 2 * kt * kLTile, &x_map, kbeg + kt * kLB, (int)m0, &full[kt]);
    int issued = pre;
    for (int kt = pre; kt < nk; ++kt) {
      const int s = kt % kLStages;
      if (!mbar_wait(&empty[s], ((kt / kLStages) - 1) & 1)) {
        set_status(a.status, MLA_DEV_TIMEOUT);
        break;
      }
      mbar_arrive_expect_tx(&full[s], 2 * kLTile);
      tma_load_2d(sm + 2 * s * kLTile, &x_map, kbeg + kt * kLB, (int)m0, &full[s]);
      tma_load_2d(sm + (2 * s + 1) * kLTile, &w_map, kbeg + kt * kLB, n0, &full[s]);
      issued = kt + 1;
    }
    // never leave with copies in flight
    for (int kt = issued - kLStages < 0 ? 0 : issued - kLStages; kt < issued; ++kt)
      if (!mbar_wait(&full[kt % kLStages], (kt / kLStages) & 1))
        set_status(a.status, MLA_DEV_TIMEOUT);
    return;
  }

  // ------------------------------------------------------------ math warps
  const int wm = warp >> 1, wn = warp & 1;
  const int g = lane >> 2, q = lane & 3;
  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
  const int arow = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int brow = (lane & 7) + ((lane >> 4) << 3);
  bool ok = true;
  for (int kt = 0; kt < nk; ++kt) {
    const int s = kt % kLStages;
    ok = mbar_wait(&full[s], (kt / kLStages) & 1);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const uint8_t* xs = sm + 2 * s * kLTile;
    const uint8_t* ws = xs + kLTile;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t af[2][4], bf[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        ldsm_x4(smem_u32(xs + sw128(32 * wm + 16 * i + arow, 2 * kk + (lane >> 4))), af[i][0],
                af[i][1], af[i][2], af[i][3]);
#pragma unroll
      for (int j = 0; j < 2; ++j)
        ldsm_x4(smem_u32(ws + sw128(32 * wn + 16 * j + brow, 2 * kk + ((lane >> 3) & 1))),
                bf[j][0], bf[j][1], bf[j][2], bf[j][3]);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mma_16816(acc[i][2 * j], af[i][0], af[i][1], af[i][2], af[i][3], bf[j][0], bf[j][1]);
          mma_16816(acc[i][2 * j + 1], af[i][0], af[i][1], af[i][2], af[i][3], bf[j][2], bf[j][3]);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (!ok) {
    if (lane == 0) set_status(a.status, MLA_DEV_TIMEOUT);
    return;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int64_t m = m0 + 32 * wm + 16 * i + g + 8 * hf;
        const int n = n0 + 32 * wn + 8 * j + 2 * q;
        if (m >= a.M) continue;
        const float v0 = acc[i][j][2 * hf], v1 = acc[i][j][2 * hf + 1];
        if (a.partial)
          *reinterpret_cast<float2*>(a.partial + ((int64_t)blockIdx.z * a.M + m) * a.N + n) =
              make_float2(v0, v1);
        else
          store_pair(a, m, n, v0, v1);
      }
}

// Sum of the splits' partials in split order, then the column map.
__global__ void __launch_bounds__(256) linear_reduce_kernel(LinArgs a, int splits) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t pairs = a.M * (a.N / 2);
  const int64_t stride = (int64_t)a.N * a.M;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < pairs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / (a.N / 2);
    const int n = (int)(i - m * (a.N / 2)) * 2;
    const float* p = a.partial + m * a.N + n;
    // the loads go out together; the adds keep split order
    float2 t[kLMaxSplits];
#pragma unroll
    for (int z = 0; z < kLMaxSplits; ++z)
      if (z < splits) t[z] = __ldcg(reinterpret_cast<const float2*>(p + z * stride));
    float2 s = t[0];
#pragma unroll
    for (int z = 1; z < kLMaxSplits; ++z)
      if (z < splits) {
        s.x += t[z].x;
        s.y += t[z].y;
      }
    store_pair(a, m, n, s.x, s.y);
  }
}

// ---------------------------------------------------------------------------
// Many rows (prefill chunks): the same Y = X W^T on tcgen05. A CTA owns a
// 128 x NT tile of Y (NT = 256, or 192 / 128 / 64 when that does not divide
// N) and the whole of K. Thread 0 streams 64-wide K steps of X (128 rows) and
// W (NT rows) by TMA (SWIZZLE_128B) through a 4-stage ring, the weight tiles
// of the first stages before the preceding kernel has finished; one elected
// thread of warp 1 issues 4 tcgen05.mma (M 128, N NT, K 16) per step into a
// TMEM accumulator; then thread r of the four warps reads row r of the tile
// out of TMEM, rounds it to bf16 and writes it through the column map.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 128;
constexpr int kTcStages = 4;
constexpr int kTcA = kTcRows * 128;            // 128 rows x 64 bf16: 16 KB
constexpr int kTcB = 256 * 128;                // up to 256 rows x 64 bf16: 32 KB
constexpr int kTcThreads = 128;

struct LinTcSmem {
  static constexpr int a = 0;
  static constexpr int b = a + kTcStages * kTcA;
  static constexpr int bars = b + kTcStages * kTcB;   // full[4], empty[4], done
  static constexpr int misc = bars + (2 * kTcStages + 1) * 8;
  static constexpr int bytes = misc + 16;
  static constexpr int alloc = bytes + 1024;
};
static_assert(LinTcSmem::alloc <= 227 * 1024, "shared memory budget");

__global__ void __launch_bounds__(kTcThreads, 1)
    linear_tc_kernel(const __grid_constant__ CUtensorMap x_map,
                     const __grid_constant__ CUtensorMap w_map, LinArgs a, int nt) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + LinTcSmem::bars);
  uint64_t* empty = full + kTcStages;
  uint64_t* done = empty + kTcStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LinTcSmem::misc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * nt;
  const int64_t m0 = (int64_t)blockIdx.y * kTcRows;
  const int nk = a.K / kLB;
  const uint32_t stage_tx = (uint32_t)(kTcA + nt * 128);

  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    prefetch_tensormap(&x_map);
    prefetch_tensormap(&w_map);
  }
  if (warp == 1) tc::alloc(tmem_slot, 256);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  int issued = 0;
  if (tid == 0) {
    // the weight needs no earlier kernel: its first tiles go out at once
    const int pre = nk < kTcStages ? nk : kTcStages;
    for (int kt = 0; kt < pre; ++kt) {
      mbar_arrive_expect_tx(&full[kt], stage_tx);
      tma_load_2d(sm + LinTcSmem::b + kt * kTcB, &w_map, kt * kLB, n0, &full[kt]);
    }
    pdl_wait();
    for (int kt = 0; kt < pre; ++kt)
      tma_load_2d(sm + LinTcSmem::a + kt * kTcA, &x_map, kt * kLB, (int)m0, &full[kt]);
    issued = pre;
  } else {
    pdl_wait();
  }
  pdl_launch_dependents();
  if (warp == 0) {
    // ---- producer: the rest of the K steps, one stage behind the MMAs
    if (lane == 0) {
      for (int kt = issued; kt < nk; ++kt) {
        const int s = kt % kTcStages;
        if (!mbar_wait(&empty[s], ((kt / kTcStages) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], stage_tx);
        tma_load_2d(sm + LinTcSmem::b + s * kTcB, &w_map, kt * kLB, n0, &full[s]);
        tma_load_2d(sm + LinTcSmem::a + s * kTcA, &x_map, kt * kLB, (int)m0, &full[s]);
        issued = kt + 1;
      }
      if (!ok) set_status(a.status, MLA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer
    const uint32_t idesc = tc::idesc_bf16(kTcRows, nt, false, false);
    const bool leader = tc::elect_one();
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % kTcStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (kt / kTcStages) & 1))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (leader) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = tc::smem_desc(smem_u32(sm + LinTcSmem::a + s * kTcA) + 32 * ks, 16,
                                            1024, tc::kSwizzle128);
          const uint64_t bd = tc::smem_desc(smem_u32(sm + LinTcSmem::b + s * kTcB) + 32 * ks, 16,
                                            1024, tc::kSwizzle128);
          tc::mma_bf16(tmem, ad, bd, idesc, kt > 0 || ks > 0);
        }
        tc::commit(&empty[s]);
      }
      __syncwarp();
    }
    if (leader) {
      if (!ok) set_status(a.status, MLA_DEV_TIMEOUT);
      tc::commit(done);   // every MMA issued (or none) has finished when this lands
    }
    __syncwarp();
  }
  // ---- epilogue: row r of the tile from TMEM lane r, bf16, through the column map
  const bool okd = __syncthreads_and(mbar_wait(done, 0) && ok) != 0;
  if (tid == 0 && issued > 0) {
    // never leave with copies in flight
    for (int kt = issued - kTcStages < 0 ? 0 : issued - kTcStages; kt < issued; ++kt)
      if (!mbar_wait(&full[kt % kTcStages], (kt / kTcStages) & 1)) set_status(a.status, MLA_DEV_TIMEOUT);
  }
  tc::fence_after_sync();
  const int64_t m = m0 + tid;
  // okd is the same in every thread; the TMEM loads are warp-collective
  // (.sync.aligned), so every lane takes them and only the stores depend on
  // the row being one of the M rows
  if (okd) {
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const int H = a.N / a.P;
#pragma unroll 1
    for (int c = 0; c < nt / 32; ++c) {
      uint32_t v[32];
      tc::ld32(trow + 32 * c, v);
      tc::wait_ld();
      if (m >= a.M) continue;
      const int n = n0 + 32 * c, h = n / a.P, d = n - h * a.P;
      __nv_bfloat16* dst = d < a.Q ? a.y0 + (m * H + h) * a.Q + d
                                   : a.y1 + (m * H + h) * (a.P - a.Q) + (d - a.Q);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(
            pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
            pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
            pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
            pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::dealloc(tmem, 256);
}

// N tile of the tensor-core path: the largest of 256, 192, 128, 64 dividing N.
int linear_tc_tile(int N) {
  for (int t : {256, 192, 128, 64})
    if (N % t == 0) return t;
  return 0;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// Rows from which the projections run on tcgen05 (below, the split-K warp-mma
// kernel fills the GPU better).
constexpr int64_t kLinTcRows = 256;

// Workspace: the status word (bytes 0-3), then the partials.
constexpr size_t kLPartialOff = 256;

// K splits: the smallest power of two that gives two CTAs per SM, dividing
// the K steps, at most kLMaxSplits.
int linear_splits(int64_t M, int N, int K, int sms) {
  const int64_t tiles = ((M + kLB - 1) / kLB) * (N / kLB);
  const int ksteps = K / kLB;
  int s = 1;
  while (tiles * s < 2 * (int64_t)sms && ksteps % (2 * s) == 0 && s < kLMaxSplits) s *= 2;
  return s;
}

size_t linear_ws_bytes(int64_t M, int N, int K, int sms) {
  if (M >= kLinTcRows && (N % 64) == 0) return kLPartialOff;   // the tensor-core path (no splits)
  const int s = linear_splits(M, N, K, sms);
  return kLPartialOff + (s > 1 ? (size_t)s * (size_t)M * (size_t)N * 4 : 0);
}

mla_status run_linear(const void* x, const void* w, int64_t M, int N, int K, int P, int Q,
                      void* y0, void* y1, void* workspace, size_t ws_bytes, void* stream) {
  const int sms = sm_count();
  if (sms <= 0) return MLA_ERR_CUDA;
  const int nt = linear_tc_tile(N);
  if (M >= kLinTcRows && nt > 0) {
    if (ws_bytes < 256) return MLA_ERR_WORKSPACE_TOO_SMALL;
    CUtensorMap x_map, w_map;
    if (!encode_map_2d(&x_map, x, (uint64_t)K, (uint64_t)M, kLB, kTcRows) ||
        !encode_map_2d(&w_map, w, (uint64_t)K, (uint64_t)N, kLB, (uint32_t)nt))
      return MLA_ERR_CUDA;
    LinArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.k_split = K;
    a.P = P;
    a.Q = Q;
    a.y0 = reinterpret_cast<__nv_bfloat16*>(y0);
    a.y1 = reinterpret_cast<__nv_bfloat16*>(y1);
    a.partial = nullptr;
    a.status = reinterpret_cast<uint32_t*>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         LinTcSmem::alloc);
    if (e == cudaSuccess)
      e = launch_pdl(linear_tc_kernel, dim3((unsigned)(N / nt), (unsigned)((M + kTcRows - 1) / kTcRows)),
                     dim3(kTcThreads), LinTcSmem::alloc, st, x_map, w_map, a, nt);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
  }

  const int splits = linear_splits(M, N, K, sms);
  if (ws_bytes < linear_ws_bytes(M, N, K, sms)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap x_map, w_map;
  if (!encode_map_2d(&x_map, x, (uint64_t)K, (uint64_t)M, kLB, kLB) ||
      !encode_map_2d(&w_map, w, (uint64_t)K, (uint64_t)N, kLB, kLB))
    return MLA_ERR_CUDA;
  LinArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.k_split = K / splits;
  a.P = P;
  a.Q = Q;
  a.y0 = reinterpret_cast<__nv_bfloat16*>(y0);
  a.y1 = reinterpret_cast<__nv_bfloat16*>(y1);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  a.partial = splits > 1 ? reinterpret_cast<float*>(ws + kLPartialOff) : nullptr;
  a.status = reinterpret_cast<uint32_t*>(ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kLSmem);
  if (e == cudaSuccess)
    e = launch_pdl(linear_kernel, dim3((unsigned)(N / kLB), (unsigned)((M + kLB - 1) / kLB),
                                       (unsigned)splits),
                   dim3(kLThreads), kLSmem, st, x_map, w_map, a);
  if (e == cudaSuccess && splits > 1) {
    const int64_t pairs = M * (N / 2);
    const int64_t blocks = (pairs + 255) / 256;
    e = launch_pdl(linear_reduce_kernel, dim3((unsigned)(blocks < 4 * sms ? blocks : 4 * sms)),
                   dim3(256), 0, st, a, splits);
  }
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

mla_status proj_checks(const mla_config* cfg, int64_t num_tokens, int32_t hidden_size) {
  const mla_status s = validate_config(cfg);
  if (s != MLA_OK) return s;
  if (num_tokens < 0 || hidden_size <= 0) return MLA_ERR_INVALID_ARGUMENT;
  if (cfg->dtype != MLA_BF16 || hidden_size % kLB != 0 || num_tokens > ((int64_t)1 << 30))
    return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_proj_workspace_size(const mla_config* cfg, int64_t num_tokens, int32_t hidden_size) {
  if (proj_checks(cfg, num_tokens, hidden_size) != MLA_OK) return 0;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const int H = cfg->num_heads;
  size_t need = linear_ws_bytes(num_tokens, H * (kDn + kDr), hidden_size, sms);
  const size_t kv = linear_ws_bytes(num_tokens, kRow, hidden_size, sms);
  const size_t o = linear_ws_bytes(num_tokens, hidden_size, H * kDv, sms);
  if (kv > need) need = kv;
  if (o > need) need = o;
  return need;
}

mla_status mla_q_proj(const mla_config* cfg, const void* hidden, const void* W_q, void* q_nope,
                      void* q_pe, int64_t num_tokens, int32_t hidden_size, void* workspace,
                      size_t ws_bytes, void* stream) {
  mla_status s = proj_checks(cfg, num_tokens, hidden_size);
  if (s != MLA_OK) return s;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return MLA_OK;
  if (!hidden || !W_q || !q_nope || !q_pe || !aligned16(hidden) || !aligned16(W_q) ||
      !aligned16(q_nope) || !aligned16(q_pe))
    return MLA_ERR_INVALID_ARGUMENT;
  return run_linear(hidden, W_q, num_tokens, cfg->num_heads * (kDn + kDr), hidden_size, kDn + kDr,
                    kDn, q_nope, q_pe, workspace, ws_bytes, stream);
}

mla_status mla_kv_a_proj(const mla_config* cfg, const void* hidden, const void* W_kv_a,
                         void* c_kv, void* k_pe, int64_t num_tokens, int32_t hidden_size,
                         void* workspace, size_t ws_bytes, void* stream) {
  mla_status s = proj_checks(cfg, num_tokens, hidden_size);
  if (s != MLA_OK) return s;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return MLA_OK;
  if (!hidden || !W_kv_a || !c_kv || !k_pe || !aligned16(hidden) || !aligned16(W_kv_a) ||
      !aligned16(c_kv) || !aligned16(k_pe))
    return MLA_ERR_INVALID_ARGUMENT;
  return run_linear(hidden, W_kv_a, num_tokens, kRow, hidden_size, kRow, kDc, c_kv, k_pe,
                    workspace, ws_bytes, stream);
}

mla_status mla_o_proj(const mla_config* cfg, const void* attn_out, const void* W_o, void* y,
                      int64_t num_tokens, int32_t hidden_size, void* workspace, size_t ws_bytes,
                      void* stream) {
  mla_status s = proj_checks(cfg, num_tokens, hidden_size);
  if (s != MLA_OK) return s;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return MLA_OK;
  if (!attn_out || !W_o || !y || !aligned16(attn_out) || !aligned16(W_o) || !aligned16(y))
    return MLA_ERR_INVALID_ARGUMENT;
  return run_linear(attn_out, W_o, num_tokens, hidden_size, cfg->num_heads * kDv, hidden_size,
                    hidden_size, y, y, workspace, ws_bytes, stream);
}

}  // extern "C"
