/*
 * libmsa — the decode hot path of MiniMax Sparse Attention (MSA) over an NVFP4
 * paged KV cache, as CUDA kernels for NVIDIA GB300 (sm_103a).
 *
 * Sources (cited below by the tag in brackets):
 *   [vLLM-zh]  "vLLM 对 MiniMax-M3.1-Flash 的 Day-0 支持：NVFP4 MSA 内核、MegaMoE 与
 *              Agentic 基准测试" (agentlenshq.com): the vLLM day-0 blog post on
 *              MiniMax-M3.1-Flash, Chinese rewrite. Sections used: "How MiniMax
 *              sparse attention works", "Blackwell MSA kernels / dequantising NVFP4
 *              to FP8 with the CUDA 13.4 QMUL4 instruction", "NVFP4 indexer decode
 *              context parallelism", "Rubin MSA kernels".
 *   [MSA-fig]  "MiniMax goes sparse: reading the M3 attention mechanism from one
 *              diagram" (atlascloud.ai), section 1: the index branch (shared
 *              single-head K_idx, block max pool, top-k) and the sparse branch.
 *
 * What the path computes, per request b with N context tokens (including this
 * step's R query rows, which sit at positions N-R .. N-1 and see keys t <= their
 * own position):
 *   1. index scan   s[r][g][t] = q_idx[r][g] . k_idx[t]   for every context token
 *                   (one FP8 index query per GQA group against one shared NVFP4
 *                   index-key head, dequantised to FP8)           [vLLM-zh §How]
 *   2. block pool   S[g][c] = max over rows r and tokens t of block c  [vLLM-zh §How]
 *   3. top-k        16 blocks per group: the most recent block plus the 15 best
 *                   others (ties to the lower block id); all blocks if <= 16
 *                                                        [vLLM-zh §How; MSA-fig §1]
 *   4. attention    softmax((q . k) * sm_scale) V over the selected blocks' keys,
 *                   K/V dequantised from NVFP4 to FP8, every query head of the
 *                   group sharing the group's selection   [vLLM-zh §How; MSA-fig §1]
 *
 * Geometry: 4 KV heads (GQA groups) x head dim 128, 8 query heads per KV head,
 * one shared index-key head of dim 128, 128-token pages (= KV blocks), top_k 16.
 * Other values return MSA_ERR_UNSUPPORTED.
 *
 * Formats. FP8 = OCP E4M3 ("FN": no infinities, S.1111.111 = NaN, max 448).
 * NVFP4 = E2M1 element codes with one E4M3 scale per 16 consecutive elements; a
 * 128-element row is 64 code bytes (element 2i in the low nibble of byte i) plus
 * 8 scale bytes. Scale bytes of written slots must be non-negative (sign bit
 * clear), as NVFP4 scales are amax/6. The dequantised value is the E2M1 value
 * times its scale, rounded to E4M3 (nearest, ties to even, saturating) — the FP8
 * value an FP8 MMA consumes ([vLLM-zh] Blackwell and Rubin kernel sections).
 *
 * Cache layout (data and scale planes separate; P = num_pages):
 *   k_data, v_data   [P][4][128][64]   k_scale, v_scale   [P][4][128][8]
 *   ki_data          [P][128][64]      ki_scale           [P][128][8]
 * Slots of a page beyond a request's context may hold anything; they are never
 * used. Every cache pointer must be 16-byte aligned.
 *
 * Ownership and execution. Every pointer in msa_decode_args and every buffer
 * argument is a DEVICE pointer owned by the caller (unless marked host). Calls
 * enqueue work on `stream` (a cudaStream_t; NULL = legacy default stream),
 * never synchronise (except msa_get_error) and never allocate device memory.
 * Arguments are validated on the host before any launch; a failed check
 * returns an error and launches nothing. Values only the device can see (page
 * ids, context lengths, row counts) are checked by the kernels: a bad value sets
 * a flag in the workspace, the affected work is skipped, and msa_get_error
 * reports it. No call raises a device-side trap.
 *
 * Workspace. `ws` is caller-owned device memory of at least msa_workspace_size()
 * bytes, 256-byte aligned, zero-filled once before first use (msa_workspace_init).
 * The kernels leave its counters at zero when they finish, so one workspace
 * serves any number of successive calls on one stream; calls running at the
 * same time need separate workspaces.
 */
#ifndef LIBMSA_MSA_H_
#define LIBMSA_MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = -1,   /* a host-checkable argument is out of range or NULL */
  MSA_ERR_UNSUPPORTED = -2,   /* geometry other than 4 x 8 x 128, block 128, top-k 16; device not sm_103 */
  MSA_ERR_CUDA = -3,          /* a CUDA runtime call failed (launch, attribute, ...) */
  MSA_ERR_WORKSPACE = -4,     /* workspace NULL, too small or misaligned */
  MSA_ERR_BAD_TABLE = -5,     /* (msa_get_error) a page id or length seen on the device was out of range */
  MSA_ERR_TIMEOUT = -6        /* (msa_get_error) a bounded on-chip wait gave up */
} msa_status;

/* Device error flags reported by msa_get_error (bitwise OR). */
#define MSA_FLAG_BAD_PAGE    0x1u   /* block_table entry outside [0, num_pages) */
#define MSA_FLAG_BAD_LENGTH  0x2u   /* context_lens / q_indptr inconsistent with the limits */
#define MSA_FLAG_TIMEOUT     0x4u   /* an mbarrier / async-copy wait hit its time limit */
#define MSA_FLAG_BAD_IDS     0x8u   /* msa_sparse_attn_decode got a block id outside the context, or msa_dcp_merge_topk a bad candidate list */
#define MSA_FLAG_BAD_SLOT    0x10u  /* msa_kv_insert_nvfp4 got a slot on a page outside [0, num_pages) */

typedef struct {
  int32_t num_reqs;            /* B >= 0 */
  int32_t total_rows;          /* query rows this step = q_indptr[B] (host copy of the value) */
  int32_t max_rows_per_req;    /* upper bound on any request's rows, 1..8 */
  int32_t num_pages;           /* P, physical pages in each cache */
  int32_t max_pages_per_req;   /* row length of block_table; context_lens[b] <= 128 * this */
  int32_t num_kv_heads;        /* 4 */
  int32_t q_per_kv;            /* 8 */
  int32_t head_dim;            /* 128 */
  int32_t block_size;          /* 128 */
  int32_t top_k;               /* 16 */
  float sm_scale;              /* attention logit scale, usually 1/sqrt(128) */
  const int32_t* context_lens; /* [B] tokens in the cache including this step's rows */
  const int32_t* q_indptr;     /* [B+1] request b owns rows [q_indptr[b], q_indptr[b+1]) */
  const int32_t* block_table;  /* [B][max_pages_per_req] physical page of logical block c */
  const uint8_t* q;            /* [total_rows][32][128] E4M3 queries; head h uses KV head h/8 */
  const uint8_t* q_idx;        /* [total_rows][4][128] E4M3 index queries, one per group */
  const uint8_t* k_data;       /* NVFP4 caches, layouts above */
  const uint8_t* k_scale;
  const uint8_t* v_data;
  const uint8_t* v_scale;
  const uint8_t* ki_data;
  const uint8_t* ki_scale;
} msa_decode_args;

/* Static text for a status code. */
const char* msa_status_string(msa_status status);

/* Bytes of workspace the calls below need for `args` on the current device
 * (depends on num_reqs, total_rows, max_rows_per_req, max_pages_per_req and
 * the SM count). Writes *bytes; host-only, no launch. */
msa_status msa_workspace_size(const msa_decode_args* args, size_t* bytes);

/* Zero-fill a workspace (async memset on `stream`). Needed once per workspace. */
msa_status msa_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Diagnostic for the failure path: one thread on the device waits, through the same
 * bounded wait every kernel of the library uses, on a barrier phase that never
 * completes. After the wait limit (1 s of %globaltimer) it sets MSA_FLAG_TIMEOUT in
 * `ws` (at least 256 bytes, 256-byte aligned) and returns; the GPU context stays
 * usable and msa_get_error then returns MSA_ERR_TIMEOUT. Nothing else is launched,
 * no copy is in flight and no tensor memory is held while it waits. */
msa_status msa_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/* Read and clear the device error flags in `ws` (synchronises `stream`).
 * *flags (host) receives MSA_FLAG_* bits; returns MSA_OK when none is set,
 * else the matching error code. */
msa_status msa_get_error(void* ws, size_t ws_bytes, void* stream, uint32_t* flags);

/* Step 1 alone (debug / unfused path) [vLLM-zh §How; MSA-fig §1 step 1].
 * scores[(row * 4 + g) * score_stride + t] = q_idx[row][g] . k_idx(request, t)
 * for t < context length (FP32, FP8 x FP8 products summed in FP32); -inf where
 * t is after the row's position. score_stride >= max context length (elements);
 * entries at t >= context length are left unwritten. */
msa_status msa_index_scores(const msa_decode_args* args, float* scores, int64_t score_stride,
                            void* ws, size_t ws_bytes, void* stream);

/* Steps 2+3 from given token scores laid out as msa_index_scores writes them
 * [vLLM-zh §How; MSA-fig §1 "Block Max Pool", "TopK"]. Writes block_ids
 * [B][4][16] (int32, ascending, -1 padded) and, if block_scores is not NULL,
 * block_scores[B][4][max_pages_per_req] (FP32 block maxima, -inf past the
 * context). Ties between equal block scores go to the lower block id. */
msa_status msa_block_maxpool_topk(const msa_decode_args* args, const float* scores, int64_t score_stride,
                                  int32_t* block_ids, float* block_scores,
                                  void* ws, size_t ws_bytes, void* stream);

/* Steps 1+2+3: one streaming pass over the index-key cache with the block max
 * pool in its epilogue (per-token scores never reach memory; block maxima go to
 * the workspace), then a top-k kernel chained to it by programmatic dependent
 * launch. Outputs as msa_block_maxpool_topk. These are the first two kernels of
 * msa_decode. */
msa_status msa_select_blocks(const msa_decode_args* args, int32_t* block_ids, float* block_scores,
                             void* ws, size_t ws_bytes, void* stream);

/* msa_select_blocks with exact index scores (the exact-score indexer) [vLLM-zh, Rubin MSA
 * kernels: dequantising NVFP4 to FP16 keeps E2M1 x scale exact, so the scores are free of
 * the E4M3 re-rounding an FP8 MMA implies]. The index keys' values are E2M1 x E4M3 scale
 * exactly (FP16 operands, FP32 accumulation), the index queries their E4M3 values; pooling,
 * top-k and the outputs are those of msa_select_blocks. Shared memory per CTA grows with
 * num_reqs: more than about 560 requests return MSA_ERR_UNSUPPORTED. Same workspace. */
msa_status msa_select_blocks_exact(const msa_decode_args* args, int32_t* block_ids, float* block_scores,
                                   void* ws, size_t ws_bytes, void* stream);

/* Step 4 given block ids [B][4][16] (ascending or not, -1 = unused)
 * [vLLM-zh §How; MSA-fig §1 step 2]. out_bf16[row][32][128] (BF16 bits) gets
 * softmax attention over the keys of the listed blocks visible to the row; lse
 * (optional, [total_rows][32] FP32) gets log(sum(exp(logits))), natural log. */
msa_status msa_sparse_attn_decode(const msa_decode_args* args, const int32_t* block_ids,
                                  uint16_t* out_bf16, float* lse, void* ws, size_t ws_bytes, void* stream);

/* msa_sparse_attn_decode for batches whose (request, group) pairs have at most 16 query
 * rows (max_rows_per_req <= 2, else MSA_ERR_UNSUPPORTED), with warp-level MMAs instead of
 * the 128-row tensor-core tile: S = Q K^T by mma.sync m16n8k32 (E4M3 x E4M3, FP32
 * accumulation), an online softmax in FP32 per warp over 16 keys of every block, P (FP16)
 * times V (FP16, exact E4M3 values) by mma.sync m16n8k16, the 8 warps' partials merged
 * with the log-sum-exp rule. One CTA per (request, group). Same arguments, outputs, flags
 * and workspace as msa_sparse_attn_decode (a block on a page outside the cache is left out
 * and flagged). The alternative for rows that fill only a small part of a tensor-core tile
 * [vLLM-zh, Blackwell MSA kernels: tensor-core MMA once the query rows fill a tile]; on
 * GB300 it measured slower than msa_sparse_attn_decode (32.8-34.5 vs 28.7 us for 32
 * requests x 65,536 tokens x 1 row; 30.7-32.6 vs 16.1 us for 1 x 4,096 x 1), which
 * therefore serves every row count in msa_decode. */
msa_status msa_sparse_attn_decode_small_rows(const msa_decode_args* args, const int32_t* block_ids,
                                             uint16_t* out_bf16, float* lse, void* ws, size_t ws_bytes,
                                             void* stream);

/* msa_select_blocks for callers that cannot allocate device memory. The MSA
 * pages have no counterpart to this entry point; it exists for hosts that hand a
 * library only the tensors it works on and keep the allocator to themselves
 * (plugin / custom-operator interfaces), and for decode loops that must not call
 * cudaMalloc because it can synchronise the device. It runs the same host checks,
 * kernels and outputs as msa_select_blocks, but its scratch (error flags and block
 * scores: 256 + 16*B*P4 bytes, where P4 is max_pages_per_req rounded up to a
 * multiple of 4) lives in a fixed 8 MiB device buffer inside the library, which
 * every GPU that loads libmsa holds until the process exits. Batches needing more
 * return MSA_ERR_WORKSPACE before any launch. It allocates nothing: each call looks
 * the buffer's device address up (cudaGetSymbolAddress; the first lookup on a device
 * may load the library's device code there, so make the first call on each device
 * before any stream capture), clears the flags with an async memset on `stream` and
 * launches. All calls share the one buffer, so calls that overlap on the GPU (other
 * streams, other host threads) race and must be serialised by the caller. The
 * device error flags of the most recent call are read with
 * msa_select_blocks_noalloc_get_error. */
msa_status msa_select_blocks_noalloc(const msa_decode_args* args, int32_t* block_ids, float* block_scores,
                                     void* stream);

/* The device error flags (MSA_FLAG_*) left by the most recent msa_select_blocks_noalloc
 * call, read from the library's fixed buffer: synchronises `stream`, writes *flags
 * (host) and returns MSA_OK when none is set, else the matching error code
 * (MSA_ERR_TIMEOUT, MSA_ERR_BAD_TABLE), as msa_get_error does for a workspace. The
 * next msa_select_blocks_noalloc call clears them. Allocates nothing. */
msa_status msa_select_blocks_noalloc_get_error(void* stream, uint32_t* flags);

/* Indexer decode context parallelism (DCP) [vLLM-zh "NVFP4 indexer decode context
 * parallelism"]: the context's pages are spread over `world` GPUs; each scores its
 * share of every request for all four groups and sends its best blocks per group to
 * the GPU(s) that need the selection, which merge the lists into the exact top-16
 * (the same ids msa_select_blocks returns on one GPU, ties included). The two calls
 * below run on either side of that exchange; the exchange itself (an NCCL
 * all-gather of every rank's lists, or an all-to-all that sends group g's lists to
 * the rank that owns group g) is the caller's.
 *
 * Partition: logical block c of every request belongs to rank c % world (the pages
 * say only that each GPU scores its share of the context). A rank's args describe
 * the whole batch (lengths, row pointers, the replicated index queries) with its own
 * index-key cache: block_table entries are read only at the rank's own blocks and
 * name pages of that rank's ki_data/ki_scale (num_pages = its page count). Entries at
 * other ranks' blocks are never read.
 *
 * Candidate list: 16 uint64 keys per (group, request), best first: the rank's 15
 * best blocks other than the request's most recent one (which the merge always keeps),
 * zero-filled past the rank's count; slot 15 is always zero. A key is
 *   (order image of the FP32 block score) << 32 | (0xFFFFFFFF - logical block id),
 * where the order image of score bits u is u | 0x80000000 for a non-negative score
 * (-0.0 counts as +0.0) and ~u for a negative one, so a larger key is a better block
 * and equal scores rank the lower id first. 0 = no candidate. */
#define MSA_DCP_MAX_WORLD 8

/* The rank-local half: the index scan over rank `rank`'s blocks (0 <= rank < world
 * <= MSA_DCP_MAX_WORLD), then its candidate lists. cand_keys (device, 8-byte aligned):
 * [4][B][16] uint64, group-major so that group g's lists are one contiguous slice.
 * Two kernels on `stream`, the second chained to the scan by programmatic dependent
 * launch; uses the workspace's block-score scratch and flags as msa_select_blocks. */
msa_status msa_dcp_local_topk(const msa_decode_args* args, int32_t rank, int32_t world, uint64_t* cand_keys,
                              void* ws, size_t ws_bytes, void* stream);

/* The merge: all_keys (device) [world][n_groups][B][16] holds, for groups group0 ..
 * group0 + n_groups - 1, every rank's lists in rank order (an all-gather of
 * cand_keys gives group0 = 0, n_groups = 4; an all-to-all of group slices gives one
 * rank's own groups). Writes block_ids[B][4][16] rows of those groups (ascending,
 * -1 padded, as msa_select_blocks); other groups' rows are left untouched. A key
 * naming a block outside its rank's share, the recent block or a repeated block, or
 * fewer than 15 candidates for a request of more than 16 blocks, sets
 * MSA_FLAG_BAD_IDS in the workspace (msa_get_error: MSA_ERR_BAD_TABLE); such keys
 * are dropped and missing winners leave -1 at the end of the row. Only the lengths
 * and row pointers of args are read. */
msa_status msa_dcp_merge_topk(const msa_decode_args* args, int32_t world, int32_t group0, int32_t n_groups,
                              const uint64_t* all_keys, int32_t* block_ids, void* ws, size_t ws_bytes,
                              void* stream);

/* The whole decode step: the index scan with its block max pool, the top-k and the
 * sparse attention on `stream`, each kernel chained to the one before it with
 * programmatic dependent launch. The top-k runs in its own kernel (three kernels, as
 * msa_select_blocks then msa_sparse_attn_decode), or inside the attention kernel (two
 * kernels) when requests may exceed 1,025 blocks and each (request, group) is split over
 * 4 or more attention CTAs, or when every (request, group) is one attention CTA and no
 * request exceeds 1,025 blocks; the ids written are the same. */
msa_status msa_decode(const msa_decode_args* args, int32_t* block_ids, uint16_t* out_bf16, float* lse,
                      void* ws, size_t ws_bytes, void* stream);

/* The dequantisers the kernels use, exposed for checking: rows of 128 NVFP4
 * elements (codes [n][64], scales [n][8]) -> E4M3 bytes out_e4m3 [n][128], element
 * j of row i at out_e4m3[i*128 + j]. path 0 = the form of the attention
 * kernel (its K operand, and V before an exact E4M3 -> FP16 widening); path 1 =
 * the index scan's form (the same table, shifts done as multiplies). The scale
 * byte's sign bit is ignored.
 * [vLLM-zh, Blackwell kernels: NVFP4 turned into FP8 before the FP8 MMA] */
msa_status msa_dequant_rows(const uint8_t* codes, const uint8_t* scales, int64_t nrows,
                            uint8_t* out_e4m3, int32_t path, void* stream);

/* Insertion of new tokens into the NVFP4 caches, the step before the decode path
 * [vLLM-zh "QKV GEMM + norm + RoPE + KV insert fusion": the projection epilogue
 * takes the FP32 accumulators head by head, quantises K, V and the index keys to
 * NVFP4 and writes them straight into their caches]. This is that epilogue's
 * quantise-and-write half on its own.
 *
 * Token t goes to page slot_mapping[t] / 128, slot slot_mapping[t] % 128: its 4 K
 * rows (k[t][h], h = KV head), 4 V rows and its index-key row are each quantised to
 * NVFP4 and written to that slot of k_data/k_scale, v_data/v_scale and
 * ki_data/ki_scale (layouts above). NVFP4 per 16 consecutive elements: scale =
 * amax / 6 rounded to E4M3 (nearest, ties to even, saturating at 448); element code
 * = the E2M1 value nearest x / scale (ties to the even code, saturating at 6) with
 * the sign of x (so -0.0 and small negative values give code 8); a zero scale
 * gives zero codes. The kernel decides every rounding by exact comparisons, so the
 * bytes equal an exact evaluation of that rule for every finite input; inputs must
 * be finite.
 *
 * A negative slot skips the token. A NULL source (k, v or k_idx) leaves its cache
 * untouched (its cache pointers may then be NULL). Tokens whose page is outside
 * [0, num_pages) are skipped and set MSA_FLAG_BAD_SLOT in the workspace
 * (msa_get_error). Two tokens mapped to the same slot race; the caller keeps slots
 * distinct. Sources must be 16-byte aligned; ws is any workspace of at least 256
 * bytes, 256-byte aligned and zero-filled once (its first word holds the flags).
 * All pointers are device pointers owned by the caller. */
typedef struct {
  int32_t num_tokens;           /* T >= 0 */
  int32_t num_pages;            /* P, pages in each cache */
  const int64_t* slot_mapping;  /* [T] page * 128 + slot, negative = skip */
  const float* k;               /* [T][4][128] FP32, or NULL */
  const float* v;               /* [T][4][128] FP32, or NULL */
  const float* k_idx;           /* [T][128] FP32, or NULL */
  uint8_t* k_data;
  uint8_t* k_scale;
  uint8_t* v_data;
  uint8_t* v_scale;
  uint8_t* ki_data;
  uint8_t* ki_scale;
} msa_kv_insert_args;

msa_status msa_kv_insert_nvfp4(const msa_kv_insert_args* args, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LIBMSA_MSA_H_ */
