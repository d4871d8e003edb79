// C ABI of libmla (declared in include/mla.h): argument validation, the
// split-KV CTA count, TMA descriptor encoding, and kernel launches. Host
// code only; every computation runs in the kernels of the other files.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

using namespace mla;

namespace {

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

mla_status check_cfg(const mla_config* cfg) {
  if (!cfg) return MLA_ERR_INVALID_ARGUMENT;
  if (cfg->kv_lora_rank != kDc || cfg->qk_rope_head_dim != kDr ||
      cfg->qk_nope_head_dim != kDn || cfg->v_head_dim != kDv)
    return MLA_ERR_UNSUPPORTED;
  const int H = cfg->num_heads;
  if (H != 16 && H != 32 && H != 64 && H != 128) return MLA_ERR_UNSUPPORTED;
  const int bs = cfg->block_size;
  if (bs != 16 && bs != 32 && bs != 64) return MLA_ERR_UNSUPPORTED;
  if (cfg->dtype != MLA_F32 && cfg->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (cfg->num_ctas < 0 || cfg->num_ctas > 65535) return MLA_ERR_INVALID_ARGUMENT;
  if (cfg->rope_interleaved != 0 && cfg->rope_interleaved != 1) return MLA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(cfg->softmax_scale) || !(cfg->rms_eps >= 0.f) ||
      !std::isfinite(cfg->rms_eps) || !(cfg->rope_base > 0.f) || !std::isfinite(cfg->rope_base))
    return MLA_ERR_INVALID_ARGUMENT;
  return MLA_OK;
}

// One CTA per SM unless the caller fixes the count. Queried on every call
// (cheap) so a change of current device is honoured.
int resolve_num_ctas(const mla_config* cfg) {
  if (cfg->num_ctas > 0) return cfg->num_ctas;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

constexpr int64_t kMaxRows = 48 * 1024;  // query rows one plan can hold in shared memory

// Tiles of 128 (row, head) rows on tcgen05 when a 16-head tile would waste
// the cache stream: many heads, or prefill chunks (several query rows per
// sequence on average). Plain decode with 16 or 32 heads uses warp mma.
bool use_tc(const mla_config* cfg, int64_t num_q, int32_t batch) {
  return cfg->dtype == MLA_BF16 && (cfg->num_heads >= 64 || num_q >= 4 * (int64_t)batch);
}

// CTA count of the decode launch: one per SM (or the caller's). In
// tensor-core mode two CTAs (a cluster) share each split, so the count is
// even, and by default it is the number of pairs the device holds at once.
int decode_ctas(const mla_config* cfg, bool tc) {
  if (tc && cfg->num_ctas <= 0) {
    const int pairs = decode_tc_max_clusters();
    if (pairs > 0) return 2 * pairs;
  }
  const int C = resolve_num_ctas(cfg);
  if (C <= 0 || !tc) return C;
  return C >= 2 ? (C & ~1) : 2;
}

// The FP8 cache's decode runs two CTAs to an SM by default.
int decode_ctas_fp8(const mla_config* cfg) {
  const int C = resolve_num_ctas(cfg);
  return (cfg->num_ctas > 0 || C <= 0) ? C : 2 * C;
}

size_t ws_bytes_needed(const mla_config* cfg, int64_t num_q, int32_t batch, bool tc, int C) {
  const int G = cfg->num_heads / kHG;
  return tc ? ws_layout_tc(num_q, G, C / 2, batch).total : ws_layout(num_q, G, C).total;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 map over rows of 576 values: box = 64 columns x box_rows rows,
// 128-byte swizzle (the layout the decode kernel's ldmatrix addressing uses).
bool make_row_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 view of rows of 576 values as (64 values, row, 64-value column
// block): the row stride (1,152 bytes) is the middle dimension and the column
// block (128 bytes) the outer one, so a box of (64, box_rows, nslab) lands in
// shared memory block-major -- nslab slabs of box_rows x 128 bytes, each laid
// out as one 2-D box of make_row_map would be -- in a single copy.
bool make_slab_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows,
                   uint32_t nslab) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(kRow / 64)};
  const cuuint64_t strides[2] = {(cuuint64_t)kRow * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, nslab};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D bf16 map over a row-major [rows, cols] matrix: box = box_cols x
// box_rows, 128-byte swizzle.
bool make_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                 uint32_t box_cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The two views of the FP8 cache's 640-byte rows: the e4m3 codes as bytes
// (boxes of 128 codes x box_rows rows, 128-byte swizzle) and the row as 320 bf16
// values for the rope columns (elements 256-319; boxes of 64 x box_rows,
// 128-byte swizzle).
bool make_fp8_maps(CUtensorMap* codes, CUtensorMap* rope, const void* base, uint64_t rows,
                   uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t stride[1] = {(cuuint64_t)kRow8};
  const cuuint32_t estr[2] = {1, 1};
  const cuuint64_t cdims[2] = {(cuuint64_t)kRow8, (cuuint64_t)rows};
  const cuuint32_t cbox[2] = {128, box_rows};
  CUresult r = fn(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), cdims, stride,
                  cbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  const cuuint64_t rdims[2] = {(cuuint64_t)kRow8 / 2, (cuuint64_t)rows};
  const cuuint32_t rbox[2] = {64, box_rows};
  r = fn(rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), rdims, stride, rbox,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 map over (d, head, row) of a [rows, heads, dims] tensor: box =
// (box_d, 1, box_rows), 128-byte swizzle.
bool make_map_heads(CUtensorMap* map, const void* base, uint64_t dims, uint64_t heads,
                    uint64_t rows, uint32_t box_d, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t gdim[3] = {(cuuint64_t)dims, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)dims * 2, (cuuint64_t)dims * heads * 2};
  const cuuint32_t box[3] = {box_d, 1, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D bf16 view of a [rows, heads, dims] tensor (dims a multiple of 64) as
// (64 values, row, 64-value column block, head): a box of (64, box_rows,
// dims / 64, 1) lands block-major -- dims / 64 slabs of box_rows x 128 bytes of
// one head -- in a single copy. 128-byte swizzle.
bool make_map_heads_slabs(CUtensorMap* map, const void* base, uint64_t dims, uint64_t heads,
                          uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t gdim[4] = {64, (cuuint64_t)rows, (cuuint64_t)(dims / 64), (cuuint64_t)heads};
  const cuuint64_t strides[3] = {(cuuint64_t)dims * heads * 2, 128, (cuuint64_t)dims * 2};
  const cuuint32_t box[4] = {64, box_rows, (cuuint32_t)(dims / 64), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gdim,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Rows from which the projections run on tcgen05 (below, the latency-bound
// warp-mma kernels are faster).
constexpr int64_t kTcProjRows = 256;

inline mla_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace

namespace mla {
mla_status validate_config(const mla_config* cfg) { return check_cfg(cfg); }

mla_status decode_paged_checks(const mla_config* cfg, const void* q_abs, const void* cache,
                               int64_t num_blocks, const int32_t* block_table,
                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* query_start_loc, int32_t batch, int64_t num_q) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (num_blocks * cfg->block_size > ((int64_t)1 << 31)) return MLA_ERR_UNSUPPORTED;
  if (num_q == 0) return MLA_OK;
  if (!q_abs || !cache || !block_table || !seq_lens || !query_start_loc || batch == 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_abs, 16) || !aligned(cache, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  return MLA_OK;
}
bool encode_row_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  return make_row_map(map, base, rows, box_rows);
}
bool encode_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows) {
  return make_map_2d(map, base, cols, rows, box_cols, box_rows);
}
bool encode_map_heads(CUtensorMap* map, const void* base, uint64_t dims, uint64_t heads,
                      uint64_t rows, uint32_t box_d, uint32_t box_rows) {
  return make_map_heads(map, base, dims, heads, rows, box_d, box_rows);
}
bool encode_map_heads_slabs(CUtensorMap* map, const void* base, uint64_t dims, uint64_t heads,
                            uint64_t rows, uint32_t box_rows) {
  return make_map_heads_slabs(map, base, dims, heads, rows, box_rows);
}
}  // namespace mla

extern "C" {

int32_t mla_version(void) { return 1; }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_TIMEOUT: return "device wait timed out";
    case MLA_ERR_BAD_BLOCK: return "block table entry out of range";
    case MLA_ERR_BAD_SEQ: return "query longer than its sequence, or sequence longer than its block table";
    case MLA_ERR_BAD_SLOT: return "slot_mapping entry out of range";
  }
  return "unknown status";
}

void mla_default_config(mla_config* cfg, int32_t num_heads, int32_t block_size, mla_dtype dtype) {
  if (!cfg) return;
  std::memset(cfg, 0, sizeof(*cfg));
  cfg->num_heads = num_heads;
  cfg->kv_lora_rank = kDc;
  cfg->qk_rope_head_dim = kDr;
  cfg->qk_nope_head_dim = kDn;
  cfg->v_head_dim = kDv;
  cfg->block_size = block_size;
  cfg->softmax_scale = 1.0f / std::sqrt((float)(kDn + kDr));
  cfg->rms_eps = 1e-6f;
  cfg->rope_base = 10000.0f;
  cfg->dtype = dtype;
  cfg->num_ctas = 0;
  cfg->rope_interleaved = 0;
}

mla_status mla_cache_write(const mla_config* cfg, const void* c_kv, const void* k_pe,
                           const int32_t* positions, const int64_t* slot_mapping,
                           int64_t num_tokens, const void* rms_weight, void* cache,
                           int64_t num_blocks, uint32_t* dev_status, void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_tokens < 0 || num_blocks < 0) return MLA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return MLA_OK;
  if (!c_kv || !k_pe || !positions || !slot_mapping || !rms_weight || !cache)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(c_kv, 16) || !aligned(k_pe, 16) || !aligned(rms_weight, 16) ||
      !aligned(cache, 16) || !aligned(positions, 4) || !aligned(slot_mapping, 8) ||
      !aligned(dev_status, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_cache_write(*cfg, c_kv, k_pe, positions, slot_mapping, num_tokens,
                                      rms_weight, cache, num_blocks, dev_status,
                                      as_stream(stream)));
}

mla_status mla_absorb_q(const mla_config* cfg, const void* q_nope, const void* q_pe,
                        const int32_t* q_positions, const void* W_uk, void* q_abs,
                        int64_t num_q, void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || num_q > (int64_t)1 << 24) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!q_nope || !q_pe || !q_positions || !W_uk || !q_abs) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(W_uk, 16) || !aligned(q_abs, 16) ||
      !aligned(q_positions, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  if (cfg->dtype == MLA_BF16 && num_q >= kTcProjRows) {
    CUtensorMap q_map, w_map;
    if (!make_map_heads(&q_map, q_nope, kDn, (uint64_t)cfg->num_heads, (uint64_t)num_q, 64, 128) ||
        !make_map_2d(&w_map, W_uk, kDn, (uint64_t)cfg->num_heads * kDc, 64, 256))
      return MLA_ERR_CUDA;
    return from_cuda(launch_absorb_tc(q_map, w_map, *cfg, q_pe, q_positions, q_abs, num_q,
                                      as_stream(stream)));
  }
  return from_cuda(launch_absorb_q(*cfg, q_nope, q_pe, q_positions, W_uk, q_abs, num_q,
                                   as_stream(stream)));
}

size_t mla_decode_workspace_size(const mla_config* cfg, int64_t num_q, int32_t batch) {
  if (check_cfg(cfg) != MLA_OK || num_q < 0 || batch < 0) return 0;
  const bool tc = use_tc(cfg, num_q, batch);
  const int C = decode_ctas(cfg, tc);
  if (C <= 0) return 0;
  return ws_bytes_needed(cfg, num_q, batch, tc, C);
}

size_t mla_decode_fp8_workspace_size(const mla_config* cfg, int64_t num_q, int32_t batch) {
  if (check_cfg(cfg) != MLA_OK || num_q < 0 || batch < 0) return 0;
  const int C = decode_ctas_fp8(cfg);
  if (C <= 0) return 0;
  return ws_bytes_needed(cfg, num_q, batch, false, C);
}

mla_status mla_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || ws_bytes < sizeof(WsHeader) || !aligned(workspace, 256))
    return MLA_ERR_INVALID_ARGUMENT;
  // the header and the fused merge's fixed counters
  const size_t n = ws_bytes < kLayoutStart ? ws_bytes : kLayoutStart;
  return from_cuda(cudaMemsetAsync(workspace, 0, n, as_stream(stream)));
}

mla_status mla_decode_plan(const mla_config* cfg, const int32_t* seq_lens,
                           const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                           int32_t max_blocks_per_seq, void* workspace, size_t ws_bytes,
                           void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0 || max_blocks_per_seq < 0) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!seq_lens || !query_start_loc || batch == 0) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(seq_lens, 4) || !aligned(query_start_loc, 4)) return MLA_ERR_INVALID_ARGUMENT;
  const bool tc = use_tc(cfg, num_q, batch);
  const int C = decode_ctas(cfg, tc);
  if (C <= 0) return MLA_ERR_CUDA;
  const int G = cfg->num_heads / kHG;
  if (ws_bytes < ws_bytes_needed(cfg, num_q, batch, tc, C)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  PlanArgs pa{seq_lens, query_start_loc, batch, (int32_t)num_q, G, C, cfg->block_size,
              max_blocks_per_seq, workspace};
  return from_cuda(tc ? launch_plan_tc(pa, as_stream(stream)) : launch_plan(pa, as_stream(stream)));
}

}  // extern "C"

namespace {

// The bf16 warp-mma kernel plans its own split for up to kSelfMaxRows rows.
bool use_self_plan(const mla_config* cfg, int64_t num_q, int32_t batch) {
  return cfg->dtype == MLA_BF16 && !use_tc(cfg, num_q, batch) && num_q <= kSelfMaxRows;
}

// self_plan: 0 = follow the plan in the workspace; 1 = plan in the kernel from
// seq_lens / query_start_loc; 2 = the same, with cache reads starting before
// the preceding kernel has finished.
mla_status decode_impl(const mla_config* cfg, const void* q_abs, const void* cache,
                       int64_t num_blocks, const int32_t* block_table, int32_t max_blocks_per_seq,
                       int32_t batch, int64_t num_q, void* workspace, size_t ws_bytes, float* o_lat,
                       void* stream, int self_plan = 0, const int32_t* seq_lens = nullptr,
                       const int32_t* query_start_loc = nullptr) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (num_blocks * cfg->block_size > ((int64_t)1 << 31)) return MLA_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!q_abs || !cache || !block_table) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_abs, 16) || !aligned(cache, 16) || !aligned(block_table, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  const bool tc = use_tc(cfg, num_q, batch);
  const int C = decode_ctas(cfg, tc);
  if (C <= 0) return MLA_ERR_CUDA;
  const int G = cfg->num_heads / kHG;
  if (ws_bytes < ws_bytes_needed(cfg, num_q, batch, tc, C)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = as_stream(stream);
  const double log2e = 1.4426950408889634;
  DecodeArgs da{q_abs, cache, num_blocks, block_table, max_blocks_per_seq, cfg->block_size,
                cfg->num_heads, G, C, num_q, (float)(cfg->softmax_scale * log2e), workspace, o_lat,
                seq_lens, query_start_loc, batch, self_plan};
  if (cfg->dtype == MLA_F32) return from_cuda(launch_decode_f32(da, st));
  // With num_blocks == 0 every block id is rejected before any copy, so the
  // map below is never used to read; it still needs a non-empty extent.
  const uint64_t map_rows = num_blocks > 0 ? (uint64_t)num_blocks * cfg->block_size
                                           : (uint64_t)cfg->block_size;
  CUtensorMap cache_map, q_map;
  if (tc) {
    // boxes: 32-token half pages (or whole pages below 32 tokens)
    const uint32_t box_rows = cfg->block_size < 32 ? (uint32_t)cfg->block_size : 32u;
    if (!make_row_map(&cache_map, cache, map_rows, box_rows)) return MLA_ERR_CUDA;
    // with 32-token boxes, one copy per stage moves a CTA's 4 or 5 column slabs
    CUtensorMap slab4 = cache_map, slab5 = cache_map;
    if (box_rows == 32 && (!make_slab_map(&slab4, cache, map_rows, 32, 4) ||
                           !make_slab_map(&slab5, cache, map_rows, 32, 5)))
      return MLA_ERR_CUDA;
    return from_cuda(launch_decode_tc(da, batch, cache_map, slab4, slab5, st));
  }
  if (!make_row_map(&cache_map, cache, map_rows, (uint32_t)cfg->block_size) ||
      !make_row_map(&q_map, q_abs, (uint64_t)num_q * cfg->num_heads, kHG))
    return MLA_ERR_CUDA;
  CUtensorMap slab9 = cache_map;
  if (cfg->block_size == kTile && !make_slab_map(&slab9, cache, map_rows, kTile, kRow / 64))
    return MLA_ERR_CUDA;
  return from_cuda(launch_decode_bf16(da, cache_map, q_map, nullptr, &slab9, st));
}

}  // namespace

extern "C" {

mla_status mla_decode_planned(const mla_config* cfg, const void* q_abs, const void* cache,
                              int64_t num_blocks, const int32_t* block_table,
                              int32_t max_blocks_per_seq, int32_t batch, int64_t num_q,
                              void* workspace, size_t ws_bytes, void* stream) {
  return decode_impl(cfg, q_abs, cache, num_blocks, block_table, max_blocks_per_seq, batch, num_q,
                     workspace, ws_bytes, nullptr, stream);
}

mla_status mla_decode_combine(const mla_config* cfg, const void* q_abs, const void* cache,
                              int64_t num_blocks, const int32_t* block_table,
                              int32_t max_blocks_per_seq, int32_t batch, int64_t num_q,
                              void* workspace, size_t ws_bytes, float* o_lat, void* stream) {
  if (num_q > 0 && (!o_lat || !aligned(o_lat, 16))) return MLA_ERR_INVALID_ARGUMENT;
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  const bool tc = use_tc(cfg, num_q, batch);
  // With few tiles per CTA (row x head group tiles of 16 rows; 128-row
  // q-blocks per CTA pair on the tensor cores) each tile is cut into many
  // splits, and one CTA merging all of them at the end of the decode is slower
  // than the merge kernel, which spreads that work over all SMs.
  const int C = decode_ctas(cfg, tc);
  const int64_t qtiles = num_q * (cfg->num_heads / kHG);
  const int64_t qblocks = num_q * cfg->num_heads / kQBlockRows;
  const bool split_heavy = tc ? qblocks < C / 2 : qtiles * 4 < C;
  if (C > 0 && split_heavy) {
    s = decode_impl(cfg, q_abs, cache, num_blocks, block_table, max_blocks_per_seq, batch, num_q,
                    workspace, ws_bytes, nullptr, stream);
    if (s != MLA_OK) return s;
    return from_cuda(launch_combine(workspace, cfg->num_heads / kHG, C, num_q, batch, o_lat,
                                    as_stream(stream)));
  }
  return decode_impl(cfg, q_abs, cache, num_blocks, block_table, max_blocks_per_seq, batch, num_q,
                     workspace, ws_bytes, o_lat, stream);
}

mla_status mla_decode_paged(const mla_config* cfg, const void* q_abs, const void* cache,
                            int64_t num_blocks, const int32_t* block_table,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                            void* workspace, size_t ws_bytes, void* stream) {
  mla_status s = mla::decode_paged_checks(cfg, q_abs, cache, num_blocks, block_table,
                                          max_blocks_per_seq, seq_lens, query_start_loc, batch,
                                          num_q);
  if (s != MLA_OK) return s;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (use_self_plan(cfg, num_q, batch)) {
    // one launch: the kernel plans and writes the plan to the workspace
    return decode_impl(cfg, q_abs, cache, num_blocks, block_table, max_blocks_per_seq, batch, num_q,
                       workspace, ws_bytes, nullptr, stream, 1, seq_lens, query_start_loc);
  }
  s = mla_decode_plan(cfg, seq_lens, query_start_loc, batch, num_q, max_blocks_per_seq, workspace,
                      ws_bytes, stream);
  if (s != MLA_OK) return s;
  return mla_decode_planned(cfg, q_abs, cache, num_blocks, block_table, max_blocks_per_seq, batch,
                            num_q, workspace, ws_bytes, stream);
}

mla_status mla_decode_paged_combine(const mla_config* cfg, const void* q_abs, const void* cache,
                                    int64_t num_blocks, const int32_t* block_table,
                                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                    const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                                    void* workspace, size_t ws_bytes, float* o_lat, void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (num_blocks * cfg->block_size > ((int64_t)1 << 31)) return MLA_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!q_abs || !cache || !block_table || !seq_lens || !query_start_loc || batch == 0 || !o_lat)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_abs, 16) || !aligned(cache, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) || !aligned(o_lat, 16))
    return MLA_ERR_INVALID_ARGUMENT;
  if (!use_self_plan(cfg, num_q, batch)) {
    s = mla_decode_plan(cfg, seq_lens, query_start_loc, batch, num_q, max_blocks_per_seq, workspace,
                        ws_bytes, stream);
    if (s != MLA_OK) return s;
    return mla_decode_combine(cfg, q_abs, cache, num_blocks, block_table, max_blocks_per_seq,
                              batch, num_q, workspace, ws_bytes, o_lat, stream);
  }
  // as in mla_decode_combine: few (row, head group) tiles per CTA are merged
  // faster by the merge kernel than by the decode CTAs
  const int C = decode_ctas(cfg, false);
  const bool split_heavy = num_q * (cfg->num_heads / kHG) * 4 < C;
  s = decode_impl(cfg, q_abs, cache, num_blocks, block_table, max_blocks_per_seq, batch, num_q,
                  workspace, ws_bytes, split_heavy ? nullptr : o_lat, stream, 2, seq_lens,
                  query_start_loc);
  if (s != MLA_OK || !split_heavy) return s;
  return from_cuda(launch_combine(workspace, cfg->num_heads / kHG, C, num_q, batch, o_lat,
                                  as_stream(stream)));
}

mla_status mla_cache_write_fp8(const mla_config* cfg, const void* c_kv, const void* k_pe,
                               const int32_t* positions, const int64_t* slot_mapping,
                               int64_t num_tokens, const void* rms_weight, float kv_scale,
                               void* cache8, int64_t num_blocks, uint32_t* dev_status,
                               void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (cfg->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_blocks < 0 || !(kv_scale > 0.f) || !std::isfinite(kv_scale))
    return MLA_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return MLA_OK;
  if (!c_kv || !k_pe || !positions || !slot_mapping || !rms_weight || !cache8)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(c_kv, 16) || !aligned(k_pe, 16) || !aligned(rms_weight, 16) ||
      !aligned(cache8, 16) || !aligned(positions, 4) || !aligned(slot_mapping, 8) ||
      !aligned(dev_status, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_cache_write_fp8(*cfg, c_kv, k_pe, positions, slot_mapping, num_tokens,
                                          rms_weight, kv_scale, cache8, num_blocks, dev_status,
                                          as_stream(stream)));
}

mla_status mla_decode_paged_combine_fp8(const mla_config* cfg, const void* q_abs,
                                        const void* cache8, int64_t num_blocks,
                                        const int32_t* block_table, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, const int32_t* query_start_loc,
                                        int32_t batch, int64_t num_q, float kv_scale,
                                        void* workspace, size_t ws_bytes, float* o_lat,
                                        void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0 || num_blocks < 0 || max_blocks_per_seq < 0 ||
      !(kv_scale > 0.f) || !std::isfinite(kv_scale))
    return MLA_ERR_INVALID_ARGUMENT;
  // the 16-head warp-mma path that plans for itself
  if (!use_self_plan(cfg, num_q, batch)) return MLA_ERR_UNSUPPORTED;
  if (num_blocks * cfg->block_size > ((int64_t)1 << 31)) return MLA_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!q_abs || !cache8 || !block_table || !seq_lens || !query_start_loc || batch == 0 || !o_lat)
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_abs, 16) || !aligned(cache8, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) || !aligned(o_lat, 16))
    return MLA_ERR_INVALID_ARGUMENT;
  const int C = decode_ctas_fp8(cfg);
  if (C <= 0) return MLA_ERR_CUDA;
  const int G = cfg->num_heads / kHG;
  if (ws_bytes < ws_bytes_needed(cfg, num_q, batch, false, C)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  const bool split_heavy = num_q * G * 4 < C;
  const double log2e = 1.4426950408889634;
  DecodeArgs da{q_abs, cache8, num_blocks, block_table, max_blocks_per_seq, cfg->block_size,
                cfg->num_heads, G, C, num_q, (float)(cfg->softmax_scale * log2e), workspace,
                split_heavy ? nullptr : o_lat, seq_lens, query_start_loc, batch, 2, kv_scale};
  const uint64_t map_rows = num_blocks > 0 ? (uint64_t)num_blocks * cfg->block_size
                                           : (uint64_t)cfg->block_size;
  CUtensorMap codes_map, rope_map, q_map;
  if (!make_fp8_maps(&codes_map, &rope_map, cache8, map_rows, (uint32_t)cfg->block_size) ||
      !make_row_map(&q_map, q_abs, (uint64_t)num_q * cfg->num_heads, kHG))
    return MLA_ERR_CUDA;
  cudaStream_t st = as_stream(stream);
  s = from_cuda(launch_decode_bf16(da, codes_map, q_map, &rope_map, nullptr, st));
  if (s != MLA_OK || !split_heavy) return s;
  return from_cuda(launch_combine(workspace, G, C, num_q, batch, o_lat, st));
}

mla_status mla_combine(const mla_config* cfg, const void* workspace, size_t ws_bytes,
                       int32_t batch, int64_t num_q, float* o_lat, void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (num_q == 0) return MLA_OK;
  if (!workspace || !o_lat || !aligned(workspace, 256) || !aligned(o_lat, 16))
    return MLA_ERR_INVALID_ARGUMENT;
  const bool tc = use_tc(cfg, num_q, batch);
  const int C = decode_ctas(cfg, tc);
  if (C <= 0) return MLA_ERR_CUDA;
  const int G = cfg->num_heads / kHG;
  if (ws_bytes < ws_bytes_needed(cfg, num_q, batch, tc, C)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(launch_combine(workspace, G, C, num_q, batch, o_lat, as_stream(stream)));
}

mla_status mla_combine_out_proj(const mla_config* cfg, const void* workspace, size_t ws_bytes,
                                int32_t batch, int64_t num_q, const void* W_uv, void* out,
                                void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || batch < 0) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if (num_q == 0) return MLA_OK;
  if (!workspace || !W_uv || !out || !aligned(workspace, 256) || !aligned(W_uv, 16) ||
      !aligned(out, 16))
    return MLA_ERR_INVALID_ARGUMENT;
  const bool tc = use_tc(cfg, num_q, batch);
  const int C = decode_ctas(cfg, tc);
  if (C <= 0) return MLA_ERR_CUDA;
  const int G = cfg->num_heads / kHG;
  if (ws_bytes < ws_bytes_needed(cfg, num_q, batch, tc, C)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(launch_combine_out_proj(*cfg, workspace, G, C, num_q, batch, W_uv, out,
                                           as_stream(stream)));
}

mla_status mla_out_proj(const mla_config* cfg, const float* o_lat, const void* W_uv, void* out,
                        int64_t num_q, void* stream) {
  mla_status s = check_cfg(cfg);
  if (s != MLA_OK) return s;
  if (num_q < 0 || num_q > (int64_t)1 << 24) return MLA_ERR_INVALID_ARGUMENT;
  if (num_q == 0) return MLA_OK;
  if (!o_lat || !W_uv || !out) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(o_lat, 16) || !aligned(W_uv, 16) || !aligned(out, 16)) return MLA_ERR_INVALID_ARGUMENT;
  if (cfg->dtype == MLA_BF16 && num_q >= kTcProjRows) {
    CUtensorMap w_map;
    if (!make_map_2d(&w_map, W_uv, kDv, (uint64_t)cfg->num_heads * kDc, 64, 64)) return MLA_ERR_CUDA;
    return from_cuda(launch_out_proj_tc(w_map, o_lat, out, num_q, cfg->num_heads, as_stream(stream)));
  }
  return from_cuda(launch_out_proj(*cfg, o_lat, W_uv, out, num_q, as_stream(stream)));
}

mla_status mla_get_device_status(const void* status_word, uint32_t* mask_out, int clear,
                                 void* stream) {
  if (!status_word || !aligned(status_word, 4)) return MLA_ERR_INVALID_ARGUMENT;
  cudaStream_t st = as_stream(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, status_word, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (clear && cudaMemsetAsync(const_cast<void*>(status_word), 0, sizeof(v), st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  if (mask_out) *mask_out = v;
  if (v & MLA_DEV_TIMEOUT) return MLA_ERR_TIMEOUT;
  if (v & MLA_DEV_BAD_BLOCK) return MLA_ERR_BAD_BLOCK;
  if (v & MLA_DEV_BAD_SEQ) return MLA_ERR_BAD_SEQ;
  if (v & MLA_DEV_BAD_SLOT) return MLA_ERR_BAD_SLOT;
  return MLA_OK;
}

mla_status mla_selftest_wait_timeout(uint32_t* status_word, int64_t timeout_ns, void* stream) {
  if (!status_word || !aligned(status_word, 4) || timeout_ns <= 0 || timeout_ns > 10000000000ll)
    return MLA_ERR_INVALID_ARGUMENT;
  return from_cuda(launch_wait_timeout_selftest(status_word, timeout_ns, as_stream(stream)));
}

}  // extern "C"
