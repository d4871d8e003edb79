/*
 * libmla -- Multi-head Latent Attention (DeepSeek-V2 style) decode over a
 * paged latent KV cache, in the matrix-absorbed form, for GB300 (sm_103a).
 *
 * Sources for the operations (web pages; section headings as printed):
 *   [MI17]  "mini-infer-17: MLA Attention -- from KV-cache compression to
 *           matrix absorption" (smarter.xin)
 *   [VLB07] "07. MLA / Mamba / MoE in vLLM source" (vLLM learning book)
 *
 * Shapes and names. H = num_heads; Dc = kv_lora_rank = 512; Dr =
 * qk_rope_head_dim = 64; Dn = qk_nope_head_dim = 128; Dv = v_head_dim = 128.
 * A cache row is [c_hat (Dc) || k_hat (Dr)] = 576 values.
 *
 * Conventions shared by every call.
 *  - Every pointer is a DEVICE pointer unless stated, 16-byte aligned, and
 *    owned by the caller. The library never allocates or frees memory.
 *  - Every array is dense, row-major, in the layout stated.
 *  - "dtype" tensors are float32 (MLA_F32) or bfloat16 (MLA_BF16) as set in
 *    mla_config.dtype. Arithmetic accumulates in fp32 in every kernel.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Every call
 *    only enqueues work: it returns before the GPU runs it.
 *  - Kernels are launched with programmatic stream serialisation: a kernel
 *    may start while the previous kernel on the stream finishes, and waits
 *    for it before reading its outputs. The weights (W_uk, W_uv, rms_weight)
 *    are read before that wait, so they must not be written by the kernel
 *    launched immediately before the call on the same stream.
 *  - Errors the host can see (bad sizes, null or misaligned pointers, an
 *    unsupported configuration, a small workspace) return at once and
 *    enqueue nothing. A failed launch returns MLA_ERR_CUDA. Errors only the
 *    GPU can see (an out-of-range block-table entry or slot, a query longer
 *    than its sequence, a wait that ran out) set bits in a device status word
 *    read by mla_get_device_status(); the offending row or token is skipped
 *    (its output is zero) and no memory outside the caller's buffers is
 *    touched.
 *  - seq_lens[b] counts every token of sequence b in the cache, including the
 *    ones written in this step. Query row j of sequence b (q_len_b rows,
 *    q_len_b = query_start_loc[b+1] - query_start_loc[b]) sits at position
 *    seq_lens[b] - q_len_b + j and attends kv positions 0..that position
 *    (causal; [MI17] pitfall 2). A decode row (q_len 1) sees every token.
 */
#ifndef LIBMLA_MLA_H_
#define LIBMLA_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARGUMENT = 1,    /* null/misaligned pointer, bad size        */
  MLA_ERR_UNSUPPORTED = 2,         /* configuration outside the supported set  */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < mla_decode_workspace_size()   */
  MLA_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed     */
  MLA_ERR_TIMEOUT = 5,             /* device: a bounded wait ran out           */
  MLA_ERR_BAD_BLOCK = 6,           /* device: block-table entry out of range   */
  MLA_ERR_BAD_SEQ = 7,             /* device: q_len > seq_len, or seq_len
                                      beyond max_blocks_per_seq * block_size   */
  MLA_ERR_BAD_SLOT = 8             /* device: slot_mapping entry out of range  */
} mla_status;

/* Bits of the device status word (a uint32_t in device memory). */
#define MLA_DEV_TIMEOUT   (1u << 0)
#define MLA_DEV_BAD_BLOCK (1u << 1)
#define MLA_DEV_BAD_SEQ   (1u << 2)
#define MLA_DEV_BAD_SLOT  (1u << 3)

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype;

/*
 * Model and launch configuration. Supported: kv_lora_rank 512,
 * qk_rope_head_dim 64, qk_nope_head_dim 128, v_head_dim 128 (DeepSeek-V2-Lite,
 * [MI17] "MLA 的数学结构"); num_heads in {16, 32, 64, 128}; block_size in
 * {16, 32, 64}; dtype MLA_F32 or MLA_BF16. num_ctas = 0 runs the decode
 * kernel with one CTA per SM; a positive value fixes the CTA count (the
 * split-KV partition), e.g. to test that results do not depend on it.
 * mla_default_config() fills the DeepSeek-V2-Lite values.
 */
typedef struct {
  int32_t num_heads;
  int32_t kv_lora_rank;
  int32_t qk_rope_head_dim;
  int32_t qk_nope_head_dim;
  int32_t v_head_dim;
  int32_t block_size;
  float softmax_scale;   /* multiplies q_abs . row; 1/sqrt(Dn + Dr) usually  */
  float rms_eps;         /* kv_a_layernorm epsilon                            */
  float rope_base;       /* RoPE base (10000 for DeepSeek-V2-Lite)            */
  int32_t dtype;         /* mla_dtype                                         */
  int32_t num_ctas;      /* 0 = one per SM                                    */
  int32_t rope_interleaved; /* RoPE pairs: 0 = (i, i + 32) (rotate-half, the
                               default), 1 = (2i, 2i + 1); the same pairing
                               for k_pe and q_pe, inv_freq_i = base^(-2i/64) */
} mla_config;

void mla_default_config(mla_config* cfg, int32_t num_heads, int32_t block_size,
                        mla_dtype dtype);

/*
 * mla_cache_write -- kv_a_layernorm + decoupled RoPE + slot scatter.
 * [VLB07] 2.2 (forward: write c_kv to the KV cache by slot_mapping) and 2.3
 * (MLA cache shape (n_blocks, block, 1, latent_d + rope_d)); [MI17] "版本 1"
 * (kv_a_layernorm before kv_b_proj), pitfall 3, and "MLA 的数学结构"
 * (K_pe = x W_kr + RoPE, one k_pe shared by all heads).
 *
 * For each token t < num_tokens with slot s = slot_mapping[t] >= 0:
 *   cache[s / block_size][s % block_size][0:512]   = RMSNorm(c_kv[t]) * rms_weight
 *   cache[s / block_size][s % block_size][512:576] = RoPE(k_pe[t], positions[t])
 * RMSNorm(x) = x / sqrt(mean(x^2) + rms_eps); RoPE rotates pairs
 * (x_i, x_{i+32}) by positions[t] * rope_base^(-2i/64) (rotate-half).
 * Statistics and rotation in fp32 (angles in fp64), one rounding to dtype.
 *   c_kv        [num_tokens, 512] dtype      k_pe [num_tokens, 64] dtype
 *   positions   [num_tokens] int32 (>= 0)    slot_mapping [num_tokens] int64
 *   rms_weight  [512] dtype                  cache [num_blocks, block_size, 576] dtype
 *   dev_status  uint32 device word or NULL; slots >= num_blocks*block_size
 *               set MLA_DEV_BAD_SLOT and are skipped. Negative slots mean
 *               "padding token" and are skipped silently.
 * Bytes of the cache other than the addressed rows are never written.
 */
mla_status mla_cache_write(const mla_config* cfg, const void* c_kv, const void* k_pe,
                           const int32_t* positions, const int64_t* slot_mapping,
                           int64_t num_tokens, const void* rms_weight, void* cache,
                           int64_t num_blocks, uint32_t* dev_status, void* stream);

/*
 * mla_absorb_q -- absorb W_uk into the query and rotate its rope part.
 * [MI17] "版本 3: MLAAttentionAbsorbed" (_build_absorbed: W_uk per head as
 * [Dc, Dn]); the DeepSeek-V2 report's absorption it cites.
 *   q_abs[n,h,0:512]   = sum_d W_uk[h][c][d] * q_nope[n,h,d]   (c < 512)
 *   q_abs[n,h,512:576] = RoPE(q_pe[n,h], q_positions[n])
 *   q_nope [num_q, H, 128] dtype   q_pe [num_q, H, 64] dtype
 *   q_positions [num_q] int32      W_uk [H, 512, 128] dtype
 *   q_abs  [num_q, H, 576] dtype (output)
 */
mla_status mla_absorb_q(const mla_config* cfg, const void* q_nope, const void* q_pe,
                        const int32_t* q_positions, const void* W_uk, void* q_abs,
                        int64_t num_q, void* stream);

/*
 * Workspace for mla_decode_paged / mla_combine: a device buffer of at least
 * mla_decode_workspace_size() bytes (it depends on the current device's SM
 * count when cfg->num_ctas is 0). Its first 4 bytes are the device status
 * word; call mla_workspace_init() once after allocating it (it zeroes the
 * status word, the plan header and the fused merge's arrival counters), and
 * again after any call that reported a device error.
 */
size_t mla_decode_workspace_size(const mla_config* cfg, int64_t num_q, int32_t batch);
mla_status mla_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_decode_paged -- split-KV attention of absorbed queries over the paged
 * latent cache, online softmax, partial results into the workspace.
 * [MI17] "版本 3" (scores and output directly against the latent) and
 * "设计取舍" (the nope and rope score parts summed before a hand-written
 * softmax); [VLB07] 2.3 (block-table indirection).
 * For each query row n, head h and every visible kv token t of its sequence:
 *   s_t = softmax_scale * (q_abs[n,h] . row_t)      (576-wide dot product)
 *   o_lat[n,h] = sum_t softmax(s)_t * row_t[0:512]
 * where row_t = cache[block_table[b][t / bs]][t % bs]. The work (row, 16-head
 * group, 64-token tile) is cut into num_ctas equal contiguous shares; each
 * CTA writes, for every (row, head group) it touches, a normalised partial
 * output and its log-sum-exp into the workspace. mla_combine() merges them.
 *   q_abs [num_q, H, 576] dtype; cache [num_blocks, block_size, 576] dtype;
 *   block_table [batch, max_blocks_per_seq] int32 (entries past a sequence's
 *   last block are never used as block ids; they may be read, within the
 *   row); seq_lens [batch] int32;
 *   query_start_loc [batch + 1] int32 (query_start_loc[batch] == num_q).
 * The same workspace must be passed, unchanged, to mla_combine().
 * Kernel choice (the same for every call given cfg, num_q and batch): with
 * bf16 and either num_heads >= 64 or num_q >= 4 * batch (prefill chunks),
 * tiles are 128 (row, head) rows on tcgen05 tensor cores with the
 * accumulator in TMEM (one query row of 128 heads, or 8 rows of 16 heads);
 * otherwise tiles are one row x 16 heads on warp mma. On that warp-mma path
 * with num_q <= 256 the call is a single kernel launch: each CTA derives the
 * split plan from seq_lens / query_start_loc itself and the kernel writes the
 * plan to the workspace; otherwise it is mla_decode_plan followed by
 * mla_decode_planned (two launches). The workspace contents are the same.
 */
mla_status mla_decode_paged(const mla_config* cfg, const void* q_abs, const void* cache,
                            int64_t num_blocks, const int32_t* block_table,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_decode_plan + mla_decode_planned -- mla_decode_paged in two calls.
 * mla_decode_paged is exactly mla_decode_plan followed by mla_decode_planned.
 * The plan (the split-KV partition for the given seq_lens/query_start_loc,
 * in the workspace) depends only on the batch layout, not on the layer, so a
 * caller decoding many layers of one step can plan once and run
 * mla_decode_planned per layer, each with its own workspace copy of the plan
 * or one workspace per layer planned once. mla_decode_planned reads no
 * seq_lens: it follows the plan; a workspace planned for another num_q, head
 * count or CTA count yields zero partials (combine then outputs zeros).
 */
mla_status mla_decode_plan(const mla_config* cfg, const int32_t* seq_lens,
                           const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                           int32_t max_blocks_per_seq, void* workspace, size_t ws_bytes,
                           void* stream);
mla_status mla_decode_planned(const mla_config* cfg, const void* q_abs, const void* cache,
                              int64_t num_blocks, const int32_t* block_table,
                              int32_t max_blocks_per_seq, int32_t batch, int64_t num_q,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_decode_combine -- mla_decode_planned and mla_combine in one kernel.
 * Same inputs as mla_decode_planned (a plan from mla_decode_plan must be in
 * the workspace) plus o_lat [num_q, H, 512] float32, the output of
 * mla_combine. The CTA that finishes a (row, 16-head group) last merges its
 * split partials while they are in L2; a (row, head group) handled by one
 * CTA is written to o_lat directly. The result equals mla_decode_planned
 * followed by mla_combine up to fp32 rounding of the merge order. When
 * there are fewer than num_ctas / 4 (row, head group) tiles, the splits of
 * each tile are many, and the call runs the decode kernel and then the merge
 * kernel of mla_combine instead (same result). The
 * workspace's arrival counters are left at zero, so the call can be repeated
 * (e.g. per layer) on one plan; after a device error, plan again.
 */
mla_status mla_decode_combine(const mla_config* cfg, const void* q_abs, const void* cache,
                              int64_t num_blocks, const int32_t* block_table,
                              int32_t max_blocks_per_seq, int32_t batch, int64_t num_q,
                              void* workspace, size_t ws_bytes, float* o_lat, void* stream);

/*
 * mla_decode_paged_combine -- mla_decode_paged and mla_combine in one call:
 * same inputs as mla_decode_paged plus o_lat [num_q, H, 512] float32, the
 * output of mla_combine. On the warp-mma path with num_q <= 256 this is one
 * kernel launch that plans, decodes and merges (the CTA that finishes a
 * (row, 16-head group) last merges its parts); with fewer than num_ctas / 4
 * (row, head group) tiles it is that kernel without the merge followed by the
 * merge kernel. Elsewhere it is mla_decode_plan + mla_decode_combine.
 * Ordering: on the one-launch path the kernel may start reading seq_lens,
 * query_start_loc, the block table and the cache before the kernel launched
 * just before it on the stream has finished (programmatic dependent launch,
 * as every libmla kernel uses); q_abs is read, and the workspace and o_lat
 * written, only after it has finished. So the kernel immediately before this
 * call must write none of those four inputs: in a layer step it is
 * mla_absorb_q, with mla_cache_write before it. (A kernel that does not use
 * programmatic launch, or a copy, finishes before this call starts.) Rows that see no token get zeros. The result
 * equals mla_decode_paged followed by mla_combine up to fp32 rounding of the
 * merge order. The arrival counters are left at zero after a successful call.
 */
mla_status mla_decode_paged_combine(const mla_config* cfg, const void* q_abs, const void* cache,
                                    int64_t num_blocks, const int32_t* block_table,
                                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                    const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                                    void* workspace, size_t ws_bytes, float* o_lat, void* stream);

/*
 * FP8 latent cache. The pages name "FP8 KV" handling of MLA only as a later
 * chapter ([MI17] "下一章"); the format is this library's reading: each row of
 * cache8 [num_blocks, block_size, 640] bytes holds the 512 OCP e4m3 codes of
 * c_hat / kv_scale (round to nearest, ties to even, saturating at +-448)
 * followed by k_rot as 64 bf16 values, i.e. 640 instead of 1,152 bytes per
 * token. kv_scale > 0 is one number for the whole cache.
 *
 * mla_cache_write_fp8 -- mla_cache_write into that layout (bf16 inputs only).
 */
mla_status mla_cache_write_fp8(const mla_config* cfg, const void* c_kv, const void* k_pe,
                               const int32_t* positions, const int64_t* slot_mapping,
                               int64_t num_tokens, const void* rms_weight, float kv_scale,
                               void* cache8, int64_t num_blocks, uint32_t* dev_status,
                               void* stream);

/*
 * mla_decode_fp8_workspace_size -- bytes of workspace mla_decode_paged_combine_fp8
 * needs for these sizes on the current device (0 for an invalid cfg).
 */
size_t mla_decode_fp8_workspace_size(const mla_config* cfg, int64_t num_q, int32_t batch);

/*
 * mla_decode_paged_combine_fp8 -- mla_decode_paged_combine over the FP8 cache:
 * the latent columns of a row are its codes times kv_scale, the rope columns
 * its bf16 values. Same inputs and ordering rules as mla_decode_paged_combine
 * plus kv_scale. Supported on the 16-head warp-mma path with num_q <= 256
 * (bf16 q_abs, 16 or 32 heads, not a prefill chunk); MLA_ERR_UNSUPPORTED
 * otherwise. The codes convert to f16 exactly and the query's latent part
 * goes to f16 scaled per head by a power of two (exact for every element down
 * to 2^-28 of the head's largest), so the result equals attention over the
 * dequantised cache up to fp32 rounding order and the f16 rounding of the
 * probabilities. The workspace must hold mla_decode_fp8_workspace_size()
 * bytes (at cfg->num_ctas = 0 this launch runs two CTAs per SM) and be
 * initialised like any decode workspace.
 */
mla_status mla_decode_paged_combine_fp8(const mla_config* cfg, const void* q_abs,
                                        const void* cache8, int64_t num_blocks,
                                        const int32_t* block_table, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, const int32_t* query_start_loc,
                                        int32_t batch, int64_t num_q, float kv_scale,
                                        void* workspace, size_t ws_bytes, float* o_lat,
                                        void* stream);

/*
 * mla_combine -- merge the split partials of mla_decode_paged.
 * For each (n, h): M = max_s lse_s, o_lat = sum_s 2^(lse_s - M) o_s /
 * sum_s 2^(lse_s - M) (the split-softmax identity; lse is kept in base 2
 * inside the workspace). Rows that see no token get zeros.
 *   o_lat [num_q, H, 512] float32 (output, always fp32).
 * cfg, batch and num_q must equal those given to mla_decode_paged.
 */
mla_status mla_combine(const mla_config* cfg, const void* workspace, size_t ws_bytes,
                       int32_t batch, int64_t num_q, float* o_lat, void* stream);

/*
 * mla_out_proj -- project the latent output back to v_head_dim.
 * [MI17] "版本 3" (W_v_absorbed [H, Dc, Dv]; attn_output = attn . (c W_v)).
 *   out[n,h,v] = sum_c o_lat[n,h,c] * W_uv[h][c][v]
 *   o_lat [num_q, H, 512] float32; W_uv [H, 512, 128] dtype;
 *   out [num_q, H, 128] dtype (output).
 */
mla_status mla_out_proj(const mla_config* cfg, const float* o_lat, const void* W_uv,
                        void* out, int64_t num_q, void* stream);

/*
 * The pages' other two forms of the same attention, for their comparison of
 * the three ([MI17] "版本 1: MLAAttentionNaive", "版本 2:
 * MLAAttentionLatentCache", "实验结果"). bf16 only (MLA_ERR_UNSUPPORTED
 * otherwise). Their cache holds, for every slot and head h, the row
 *   [K_nope (128) || k_rot (64) || V (128)],
 *   K_nope = c_hat W_uk[h], V = c_hat W_uv[h], k_rot the shared rope key,
 * in kv_cache [num_blocks, block_size, H, 320] bf16 (10,240 bytes per token
 * for 16 heads). The expansion runs on tcgen05 tensor cores (bf16 operands,
 * fp32 accumulation, one rounding to bf16).
 *
 * mla_naive_workspace_size -- bytes of the workspace these calls need for up
 * to num_q query rows, blocks of max_blocks_per_seq entries and num_tokens new
 * tokens. Its first 4 bytes are the device status word (MLA_DEV_* bits, read
 * with mla_get_device_status); zero it (mla_workspace_init) once.
 */
size_t mla_naive_workspace_size(const mla_config* cfg, int64_t num_q, int32_t max_blocks_per_seq,
                                int64_t num_tokens);

/*
 * mla_naive_cache_write -- version 1's cache write: RMSNorm and RoPE as
 * mla_cache_write, then the expansion of each new token into the rows of
 * every head at slot_mapping[t] (< 0: skipped; >= num_blocks * block_size:
 * MLA_DEV_BAD_SLOT). Same inputs as mla_cache_write plus W_uk, W_uv
 * [H, 512, 128].
 */
mla_status mla_naive_cache_write(const mla_config* cfg, const void* c_kv, const void* k_pe,
                                 const int32_t* positions, const int64_t* slot_mapping,
                                 int64_t num_tokens, const void* rms_weight, const void* W_uk,
                                 const void* W_uv, void* kv_cache, int64_t num_blocks,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_latent_expand -- version 2's per-step re-expansion: every cached token
 * of every sequence (the latent cache and block table of mla_decode_paged) is
 * expanded into kv_cache at the same slot. Followed by mla_naive_decode on
 * kv_cache, it is version 2's attention.
 */
mla_status mla_latent_expand(const mla_config* cfg, const void* cache, int64_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t batch, const void* W_uk,
                             const void* W_uv, void* kv_cache, void* workspace, size_t ws_bytes,
                             void* stream);

/*
 * mla_latent_expand in two parts, for weights that stay fixed across steps:
 * mla_latent_expand_prepare lays W_uk, W_uv [H, 512, 128] out in the
 * workspace as the expansion's operand (what every mla_latent_expand and
 * mla_naive_cache_write call does first); mla_latent_expand_prepared then
 * expands with those prepared weights and is otherwise mla_latent_expand
 * (same arguments but the weights, same checks and results, bit for bit).
 * The prepared weights stay valid until a call with other weights prepares
 * the same workspace; mla_naive_decode and mla_naive_prefill leave them. A
 * workspace never prepared gives unspecified rows (no device fault).
 */
mla_status mla_latent_expand_prepare(const mla_config* cfg, const void* W_uk, const void* W_uv,
                                     void* workspace, size_t ws_bytes, void* stream);
mla_status mla_latent_expand_prepared(const mla_config* cfg, const void* cache, int64_t num_blocks,
                                      const int32_t* block_table, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t batch, void* kv_cache,
                                      void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_naive_decode -- attention over the expanded rows:
 *   q[n,h]   = [q_nope[n,h] || RoPE(q_pe[n,h], q_positions[n])]
 *   out[n,h] = sum_t softmax_t(softmax_scale * q[n,h] . K[t,h]) V[t,h]
 * over the causal visible tokens of row n's sequence (the conventions of
 * mla_decode_paged). q_nope [num_q, H, 128], q_pe [num_q, H, 64] bf16;
 * out [num_q, H, 128] bf16 (zeros for a row that sees no token).
 */
mla_status mla_naive_decode(const mla_config* cfg, const void* q_nope, const void* q_pe,
                            const int32_t* q_positions, const void* kv_cache, int64_t num_blocks,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, const int32_t* query_start_loc,
                            int32_t batch, int64_t num_q, void* workspace, size_t ws_bytes,
                            void* out, void* stream);

/*
 * mla_naive_prefill -- mla_naive_decode's result (same arguments, same
 * conventions, zeros for a row that sees no token) on tensor cores, for
 * prefill chunks: a CTA takes 64 query rows of one sequence and one head and
 * reads each key tile of the expanded rows once for all of them (m16n8k16
 * warp mma, bf16 in, fp32 accumulation, the probabilities rounded to bf16).
 * Decode rows (one row per sequence) are better served by mla_naive_decode,
 * which splits the keys. Only the status word of the workspace is used
 * (ws_bytes >= 256).
 */
mla_status mla_naive_prefill(const mla_config* cfg, const void* q_nope, const void* q_pe,
                             const int32_t* q_positions, const void* kv_cache, int64_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, const int32_t* query_start_loc,
                             int32_t batch, int64_t num_q, void* workspace, size_t ws_bytes,
                             void* out, void* stream);

/*
 * mla_decode_paged_noalloc -- mla_decode_paged followed by mla_combine for
 * callers that cannot allocate device memory (a step callback with a fixed
 * memory budget, a real-time loop where cudaMalloc would stall or fail, a
 * plugin that must not allocate). The pages have no counterpart of this
 * call; it exists for such callers only.
 * The caller passes the same inputs as mla_decode_paged and the output
 * o_lat [num_q, H, 512] float32 of mla_combine; the workspace is instead a
 * 16 MiB array built into the library, which every GPU that loads the
 * library keeps until the process exits. With cfg->num_ctas = 0 and a
 * workspace (mla_decode_workspace_size) above 16 MiB at the default count,
 * the call uses the largest CTA count c below the SM count for which
 * mla_decode_workspace_size with num_ctas = c fits. A launch that does not
 * fit even so, or with the caller's fixed num_ctas, returns
 * MLA_ERR_WORKSPACE_TOO_SMALL. Every refusal (that one, and the argument
 * checks of mla_decode_paged, which run first and return the same codes)
 * enqueues nothing and leaves the array as it was.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. The address is kept for the life of the process: after a
 * cudaDeviceReset of a device, do not call this again on that device. Every call on a device shares the array and leaves its contents
 * for the next one: each call clears the status word and plan header itself,
 * and calls whose GPU work overlaps (other streams or host threads) race on
 * the array and must not be issued. dev_status (device word, may be NULL)
 * receives the call's device status bits (MLA_DEV_*). Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library routine is called.
 */
mla_status mla_decode_paged_noalloc(const mla_config* cfg, const void* q_abs, const void* cache,
                                    int64_t num_blocks, const int32_t* block_table,
                                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                    const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                                    float* o_lat, uint32_t* dev_status, void* stream);

/*
 * mla_combine_out_proj -- mla_combine followed by mla_out_proj without
 * writing o_lat: the split partials that mla_decode_paged / mla_decode_planned
 * left in the workspace are merged (split-softmax identity) while the mma
 * fragments of the output projection are built.
 *   out[n,h,v] = sum_c merge(n,h)[c] * W_uv[h][c][v]
 *   W_uv [H, 512, 128] dtype; out [num_q, H, 128] dtype (output).
 * cfg, batch and num_q must equal those of the decode call. Rows that see no
 * token give zeros.
 */
mla_status mla_combine_out_proj(const mla_config* cfg, const void* workspace, size_t ws_bytes,
                                int32_t batch, int64_t num_q, const void* W_uv, void* out,
                                void* stream);

/*
 * Projections on either side of the attention ([MI17] "版本 1:
 * MLAAttentionNaive": q_proj, kv_a_proj_with_mqa, o_proj; [VLB07] 2.2). bf16
 * only (MLA_ERR_UNSUPPORTED otherwise); hidden_size a positive multiple of 64,
 * num_tokens <= 2^30. Each computes Y = X W^T in fp32 with one rounding to
 * bf16, W in a linear layer's [out, in] layout, all tensors row-major and
 * 16-byte aligned:
 *
 * mla_q_proj:    hidden [T, hidden_size], W_q [H * 192, hidden_size] (rows
 *                h * 192 + 0..127 give q_nope[:, h], h * 192 + 128..191 give
 *                q_pe[:, h]); q_nope [T, H, 128], q_pe [T, H, 64] (outputs).
 * mla_kv_a_proj: hidden [T, hidden_size], W_kv_a [576, hidden_size] (rows
 *                0..511 give c_kv, 512..575 give k_pe); c_kv [T, 512],
 *                k_pe [T, 64] (outputs) -- the raw inputs of mla_cache_write,
 *                which applies the kv_a_layernorm and RoPE.
 * mla_o_proj:    attn_out [T, H * 128] (the [T, H, 128] out of mla_out_proj),
 *                W_o [hidden_size, H * 128]; y [T, hidden_size] (output).
 *
 * workspace: mla_proj_workspace_size(cfg, num_tokens, hidden_size) bytes,
 * 256-byte aligned; its first 4 bytes are a device status word (zero it with
 * mla_workspace_init once; a wait that ran out sets MLA_DEV_TIMEOUT, read it
 * with mla_get_device_status). Below 256 tokens K is split across CTAs and the
 * rest of the workspace holds their fp32 partial sums, which a second kernel
 * adds in split order; from 256 tokens one tcgen05 kernel computes each tile
 * without splitting. Results do not depend on the split beyond fp32 rounding
 * order, and repeated calls agree bit for bit. Calls that share a workspace
 * must not overlap on the GPU. The weight may be
 * read before the kernel launched just before the call on the same stream has
 * finished, so that kernel must not write it.
 */
size_t mla_proj_workspace_size(const mla_config* cfg, int64_t num_tokens, int32_t hidden_size);
mla_status mla_q_proj(const mla_config* cfg, const void* hidden, const void* W_q, void* q_nope,
                      void* q_pe, int64_t num_tokens, int32_t hidden_size, void* workspace,
                      size_t ws_bytes, void* stream);
mla_status mla_kv_a_proj(const mla_config* cfg, const void* hidden, const void* W_kv_a,
                         void* c_kv, void* k_pe, int64_t num_tokens, int32_t hidden_size,
                         void* workspace, size_t ws_bytes, void* stream);
mla_status mla_o_proj(const mla_config* cfg, const void* attn_out, const void* W_o, void* y,
                      int64_t num_tokens, int32_t hidden_size, void* workspace, size_t ws_bytes,
                      void* stream);

/*
 * mla_get_device_status -- synchronise `stream`, read the device status word
 * at `status_word` (a workspace's first word, or the dev_status buffer given
 * to mla_cache_write), optionally clear it, and map it to a status: the
 * lowest set bit wins (TIMEOUT, BAD_BLOCK, BAD_SEQ, BAD_SLOT); MLA_OK if none.
 * `mask_out` (host pointer, may be NULL) receives the raw bits.
 */
mla_status mla_get_device_status(const void* status_word, uint32_t* mask_out, int clear,
                                 void* stream);

/*
 * mla_selftest_wait_timeout -- launch one CTA that waits on a shared-memory
 * barrier nothing will ever complete, with the same bounded wait the decode
 * pipeline uses, shortened to `timeout_ns`. It sets MLA_DEV_TIMEOUT in
 * *status_word and returns; the context stays usable. Used to test the
 * timeout path without hanging the GPU.
 */
mla_status mla_selftest_wait_timeout(uint32_t* status_word, int64_t timeout_ns, void* stream);

const char* mla_status_string(mla_status s);
int32_t mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBMLA_MLA_H_ */
