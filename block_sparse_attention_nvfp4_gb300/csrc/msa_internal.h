// Host/device interface between libmsa's C ABI (msa_api.cu) and its kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/msa.h"

namespace msa {

// Fused index scan -> block max pool -> top-k (and the per-token score variant).
struct SelectParams {
  int num_reqs, num_pages, max_pages, total_rows;
  const int32_t* context_lens;
  const int32_t* q_indptr;
  const int32_t* block_table;
  const uint8_t* q_idx;
  const uint8_t* ki_scale;
  float* block_S;           // workspace [B][4][s_stride] block scores
  int s_stride;             // max_pages rounded up to a multiple of 4 (16-byte rows)
  int shard, nshards;       // scan logical blocks c with c % nshards == shard (0 of 1: all);
                            // block_S column i holds block i * nshards + shard
  uint32_t* flags;          // workspace error flags
  int32_t* block_ids;       // [B][4][16]
  float* block_scores_out;  // optional [B][4][max_pages]
  float* token_scores;      // per-token variant: [rows][4][score_stride]
  long long score_stride;
};

struct MaxpoolParams {
  int num_reqs, max_pages, total_rows;
  const int32_t* context_lens;
  const int32_t* q_indptr;
  const float* scores;
  long long score_stride;
  float* block_S;
  int s_stride;
  int32_t* block_ids;
  float* block_scores_out;
  uint32_t* flags;
};

// Sparse attention over selected blocks, split across the CTAs of a thread-block
// cluster that merges its partials through distributed shared memory.
struct AttnParams {
  int num_reqs, num_pages, max_pages, total_rows;
  const int32_t* context_lens;
  const int32_t* q_indptr;
  const int32_t* block_table;
  int32_t* block_ids;        // [B][4][16]: read, or written when block_S is set
  const float* block_S;      // set: select the ids from these block scores in the kernel
  int s_stride;              // row length of block_S ([B][4][s_stride])
  const uint8_t* q;
  const uint8_t* k_data;     // codes also read through tensor maps (launch_attn)
  const uint8_t* k_scale;
  const uint8_t* v_data;
  const uint8_t* v_scale;
  float sm_scale_log2;       // sm_scale * log2(e)
  int blocks_per_split;
  int splits;                // CTAs per (request, group) = cluster size, 1..8
  int copies;                // query-row copies down the MMA tile: 2, or 4 when rows <= 4
  int max_m;                 // 8 * max_rows_per_req
  uint32_t* flags;
  uint16_t* out;             // [rows][32][128] bf16 bits
  float* lse;                // optional [rows][32]
};

// NVFP4 insertion of new tokens (msa_kv_insert_nvfp4).
struct KvInsertParams {
  long long num_tokens;
  int num_pages;
  const int64_t* slot_mapping;
  const float* k;
  const float* v;
  const float* ki;
  uint8_t* k_data;
  uint8_t* k_scale;
  uint8_t* v_data;
  uint8_t* v_scale;
  uint8_t* ki_data;
  uint8_t* ki_scale;
  uint32_t* flags;
};

// Merge of the rank-local candidate lists of indexer decode context parallelism
// (msa_dcp_merge_topk).
struct DcpMergeParams {
  int num_reqs, max_pages, total_rows;
  const int32_t* context_lens;
  const int32_t* q_indptr;
  const uint64_t* keys;  // [world][n_groups][B][16] candidate keys
  int world, group0, n_groups;
  int32_t* block_ids;    // [B][4][16]: rows of groups group0 .. group0 + n_groups - 1 written
  uint32_t* flags;
};

// Workspace layout, offsets in bytes (each 256-aligned).
struct WsLayout {
  size_t flags, block_S, total;
};

struct Plan {
  int blocks_per_split;   // attention
  int splits;
  int copies;
};

Plan make_plan(int num_reqs, int max_rows_per_req, int sm_count);
int score_stride(int max_pages);  // block-score row length: max_pages rounded up to 4
WsLayout ws_layout(int num_reqs, int max_pages);

size_t select_smem_bytes(int num_reqs, int mode);  // mode 2: the exact-score layout
size_t attn_smem_bytes();
// grid: a fixed number of CTAs per SM over `sm_count` SMs
cudaError_t launch_select(const CUtensorMap& ki_map, const SelectParams& prm, int mode, int sm_count,
                          cudaStream_t st);
// top-k of the block scores the scan (mode 0) wrote: one CTA per request, chained
// to the scan with programmatic dependent launch
cudaError_t launch_topk(const SelectParams& prm, cudaStream_t st);
cudaError_t launch_maxpool_topk(const MaxpoolParams& prm, cudaStream_t st);
// rank-local candidate lists [4][B][16] from a sharded scan's block scores (chained to the
// scan), and their merge
cudaError_t launch_dcp_local(const SelectParams& prm, uint64_t* keys, cudaStream_t st);
cudaError_t launch_dcp_merge(const DcpMergeParams& prm, cudaStream_t st);
// kmap / vmap: tensor maps of the K and V code planes (encode_code_map over num_pages * 4 * 128 rows)
cudaError_t launch_attn(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& prm, bool pdl,
                        cudaStream_t st);
// the same step for (request, group) pairs of at most 16 query rows (R <= 2): warp-level MMAs,
// one CTA per pair; reads block_ids (never selects: block_S must be null)
size_t attn_small_smem_bytes();
cudaError_t launch_attn_small(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& prm, bool pdl,
                              cudaStream_t st);
cudaError_t launch_kv_insert(const KvInsertParams& prm, int sm_count, cudaStream_t st);
cudaError_t launch_dequant_rows(const uint8_t* codes, const uint8_t* scales, long long nrows, uint8_t* out, int path,
                                cudaStream_t st);

// Host-side helpers of the C ABI, shared by the entry points in msa_api.cu and
// msa_noalloc.cu so that both take the same checks and the same launch sequence.
// validate: every check the host can make (need_kv / need_idx: the K/V or the
// index-key operands are used). check_device: the current device is sm_103 (its SM
// count returned). encode_code_map: the TMA view of an index-key code plane.
// launch_selection: the scan (mode 0 fused, 1 per-token scores, 2 exact scores) and,
// for modes 0 and 2 with with_topk, the chained top-k, with the given flags word and
// block-score scratch ([B][4][score_stride(max_pages)] FP32). With nshards > 1 the scan
// covers the logical blocks c with c % nshards == shard (modes 0 and 2, no top-k) and, if
// dcp_keys is set, the rank-local candidate lists follow it.
msa_status validate(const msa_decode_args* a, bool need_kv, bool need_idx);
msa_status check_device(int* sm_count);
msa_status encode_code_map(CUtensorMap* map, const uint8_t* base, long long rows);
msa_status launch_selection(const msa_decode_args* args, int mode, int32_t* ids, float* scores_out, float* tok,
                            long long stride, uint32_t* flags, float* block_S, int sm_count, cudaStream_t st,
                            bool with_topk = true, int shard = 0, int nshards = 1, uint64_t* dcp_keys = nullptr);

}  // namespace msa
