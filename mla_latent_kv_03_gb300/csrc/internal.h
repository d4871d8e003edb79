// Host-side launchers implemented by the kernel translation units and called
// by the C ABI in libmla.cu. Arguments are validated before these are called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

struct PlanArgs {
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t batch;
  int32_t num_q;
  int32_t groups;
  int32_t num_ctas;
  int32_t block_size;
  int32_t max_blocks_per_seq;
  void* workspace;
};

struct DecodeArgs {
  const void* q_abs;
  const void* cache;
  int64_t num_blocks;
  const int32_t* block_table;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t num_heads;
  int32_t groups;
  int32_t num_ctas;
  int64_t num_q;
  float scale_log2;  // softmax_scale * log2(e)
  void* workspace;
  float* o_lat;      // non-null: merge the splits in the decode kernel (fused combine)
  // Self-planned launch (bf16 warp-mma kernel, num_q <= kSelfMaxRows): the
  // kernel derives the split plan from these itself and writes it to the
  // workspace; self_plan = 0 follows a plan already in the workspace.
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t batch;
  int32_t self_plan;  // 0: planned; 1: self-planned; 2: self-planned, cache reads
                      // start before the preceding kernel has finished
  float kv_scale;     // FP8 cache: the latent is the codes times kv_scale
};

cudaError_t launch_cache_write(const mla_config& cfg, const void* c_kv, const void* k_pe,
                               const int32_t* positions, const int64_t* slot_mapping,
                               int64_t num_tokens, const void* rms_weight, void* cache,
                               int64_t num_blocks, uint32_t* dev_status, cudaStream_t stream);

// The FP8 cache row: 512 e4m3 codes of c_hat / kv_scale, then k_rot in bf16.
cudaError_t launch_cache_write_fp8(const mla_config& cfg, const void* c_kv, const void* k_pe,
                                   const int32_t* positions, const int64_t* slot_mapping,
                                   int64_t num_tokens, const void* rms_weight, float kv_scale,
                                   void* cache8, int64_t num_blocks, uint32_t* dev_status,
                                   cudaStream_t stream);

cudaError_t launch_absorb_q(const mla_config& cfg, const void* q_nope, const void* q_pe,
                            const int32_t* q_positions, const void* W_uk, void* q_abs,
                            int64_t num_q, cudaStream_t stream);

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);
cudaError_t launch_plan_tc(const PlanArgs& a, cudaStream_t stream);

// rope_map non-null: the FP8 cache (cache_map views its rows as 640 bytes,
// rope_map as 320 bf16), self-planned launches only. slab_map (bf16 cache
// with 64-token pages): the 3-D view of make_slab_map with boxes of
// (64, 64 rows, 9 slabs), one copy per page; it must be given for that case.
cudaError_t launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& cache_map,
                               const CUtensorMap& q_map, const CUtensorMap* rope_map,
                               const CUtensorMap* slab_map, cudaStream_t stream);

cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t stream);

// Tensor-core decode (CTA pairs as clusters); num_ctas must be even. With
// 32-row boxes, slab4 / slab5 are 3-D views of the cache (make_slab_map in
// libmla.cu) whose boxes hold 4 / 5 column slabs of 32 rows: one copy per
// stage and CTA.
cudaError_t launch_decode_tc(const DecodeArgs& a, int32_t batch, const CUtensorMap& cache_map,
                             const CUtensorMap& slab4, const CUtensorMap& slab5,
                             cudaStream_t stream);

// CTA pairs of the tensor-core decode that fit on the current device at once
// (0 if the query fails).
int decode_tc_max_clusters();

cudaError_t launch_combine(const void* workspace, int32_t groups, int32_t num_ctas,
                           int64_t num_q, int32_t batch, float* o_lat, cudaStream_t stream);

cudaError_t launch_out_proj(const mla_config& cfg, const float* o_lat, const void* W_uv,
                            void* out, int64_t num_q, cudaStream_t stream);

// Query absorption on tcgen05 for bf16 and many rows; q_map views q_nope as
// (128 dims, H, num_q) with (64, 1, 128) boxes, w_map views W_uk as
// [H * 512 rows, 128 columns] with 64 x 256 boxes, both with the 128-byte swizzle.
cudaError_t launch_absorb_tc(const CUtensorMap& q_map, const CUtensorMap& w_map,
                             const mla_config& cfg, const void* q_pe, const int32_t* q_positions,
                             void* q_abs, int64_t num_q, cudaStream_t stream);

// Output projection on tcgen05 for bf16 and many rows; w_map views W_uv as
// [H * 512 rows, 128 columns] with 64 x 64 boxes and the 128-byte swizzle.
cudaError_t launch_out_proj_tc(const CUtensorMap& w_map, const float* o_lat, void* out,
                               int64_t num_q, int H, cudaStream_t stream);

cudaError_t launch_combine_out_proj(const mla_config& cfg, const void* workspace, int32_t groups,
                                   int32_t num_ctas, int64_t num_q, int32_t batch, const void* W_uv,
                                   void* out, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(uint32_t* status, int64_t timeout_ns,
                                         cudaStream_t stream);

// Shared host helpers of libmla.cu: the configuration check of every call and
// the TMA descriptors (bf16, 128-byte swizzle) of 576-value rows and of a
// row-major [rows, cols] matrix.
mla_status validate_config(const mla_config* cfg);
// Every host-side check mla_decode_paged makes on its arguments other than
// the workspace (configuration, sizes, row limit, null and misaligned
// pointers); MLA_OK for num_q == 0 once the sizes are valid.
mla_status decode_paged_checks(const mla_config* cfg, const void* q_abs, const void* cache,
                               int64_t num_blocks, const int32_t* block_table,
                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* query_start_loc, int32_t batch, int64_t num_q);
bool encode_row_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);
bool encode_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows);
// 3-D map over (d, head, row) of a [rows, heads, dims] bf16 tensor: box =
// (box_d, 1, box_rows), 128-byte swizzle.
bool encode_map_heads(CUtensorMap* map, const void* base, uint64_t dims, uint64_t heads,
                      uint64_t rows, uint32_t box_d, uint32_t box_rows);
// 4-D view of the same tensor whose box (64, box_rows, dims / 64, 1) holds
// all dims / 64 column slabs of box_rows rows of one head, block-major.
bool encode_map_heads_slabs(CUtensorMap* map, const void* base, uint64_t dims, uint64_t heads,
                            uint64_t rows, uint32_t box_rows);

}  // namespace mla
