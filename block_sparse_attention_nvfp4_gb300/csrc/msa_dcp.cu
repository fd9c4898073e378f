// Indexer decode context parallelism (DCP) [vLLM-zh "NVFP4 indexer decode context
// parallelism"]: the context's pages are spread over several GPUs; each GPU scores its
// share of every request for all four groups and keeps a short local list of its best
// blocks per group; the lists go to the GPU(s) that need the selection, which merge
// them into the final top-16. The merge is exact: a block among the 15 best of the
// whole context is among the 15 best of its own rank's share.
//
// This file holds the two kernels around the exchange: the rank-local list (after a
// scan restricted to the rank's blocks) and the merge. The exchange itself (an NCCL
// all-gather or all-to-all of the lists) is the caller's.
//
// Partition (the pages do not say how the context is split): logical block c of every
// request belongs to rank c % world. Round-robin keeps each page whole on one GPU and
// gives every rank an equal share of every request, short ones included.
//
// Lists are 16 slots of 64-bit keys per (group, request): the rank's 15 best blocks
// other than the request's most recent one (every rank knows that block is kept), best
// first, zero-filled; slot 15 is always zero. Key = score order image (high 32 bits)
// and 0xFFFFFFFF - logical block id (low 32 bits), so a larger key is a better block
// and equal scores go to the lower id, the selection's tie rule.
#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr int kCand = kTopK - 1;  // 15 candidates per list
constexpr int kSlots = kTopK;     // list row: 16 keys = 128 bytes
constexpr int kDcpThreads = 32 * 4 * kGroups;  // four warps per group

// Rank-local lists, after the scan of the rank's blocks (chained to it by programmatic
// dependent launch): one CTA per request, four warps per group, warp q of group g taking
// a quarter of the group's candidates; the group's warp 0 merges the four quarter lists
// (each the exact best 15 of its quarter, so their union holds the group's best 15).
// block_S column i holds the score of logical block i * world + rank.
__global__ void __launch_bounds__(kDcpThreads) dcp_local_kernel(const SelectParams p, uint64_t* keys) {
  __shared__ uint64_t surv[kGroups][4 * 64];
  __shared__ uint64_t lists[kGroups][4 * kTopK];
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp >> 2, q = warp & 3;
  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows;
  const int nb = ok && R > 0 ? (N + kBlock - 1) / kBlock : 0;
  const int nloc = nb > p.shard ? (nb - 1 - p.shard) / p.nshards + 1 : 0;  // the rank's blocks
  // the recent block (nb - 1) is kept by the merge and is no candidate
  const int nc = nb > 0 && (nb - 1) % p.nshards == p.shard ? nloc - 1 : nloc;
  pdl_wait_primary();  // the block scores come from the scan
  uint64_t k = quad_best15(p.block_S + (static_cast<long long>(b) * kGroups + g) * p.s_stride, 0, nc > 0 ? nc : 0,
                           q, 1 + g, lists[g], surv[g]);
  if (q != 0) return;
  if (k != 0ull) {  // candidate index i -> logical block i * world + rank
    const uint32_t id = static_cast<uint32_t>(topk_id(k) * p.nshards + p.shard);
    k = (k & 0xFFFFFFFF00000000ull) | static_cast<uint64_t>(0xFFFFFFFFu - id);
  }
  if (lane < kSlots) keys[(static_cast<long long>(g) * p.num_reqs + b) * kSlots + lane] = k;
}

// The merge: one CTA per request, warp gl for group group0 + gl. Reads the lists of all
// ranks (layout [world][n_groups][B][16]), checks that each key names a block of its
// rank other than the recent one, keeps the 15 best and adds the recent block; ids
// ascending, as the single-GPU selection writes them. A list that breaks those rules
// (a corrupt or truncated exchange) sets MSA_FLAG_BAD_IDS; its bad keys are dropped.
__global__ void __launch_bounds__(32 * kGroups) dcp_merge_kernel(const DcpMergeParams p) {
  const int b = blockIdx.x, gl = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (gl >= p.n_groups) return;
  const int g = p.group0 + gl;
  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows;
  if (!ok && gl == 0 && lane == 0) set_flag(p.flags, kFlagBadLength);
  const int nb = ok && R > 0 ? (N + kBlock - 1) / kBlock : 0;
  int32_t* ids = p.block_ids + (static_cast<long long>(b) * kGroups + g) * kTopK;
  if (nb <= kTopK) {  // every block (none: an empty selection)
    if (lane < kTopK) ids[lane] = lane < nb ? lane : -1;
    return;
  }
  const int n = p.world * kSlots;  // at most 4 keys per lane (world <= 8)
  uint64_t kin[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int i = 32 * t + lane, w = i / kSlots, j = i % kSlots;
    kin[t] = i < n ? __ldcg(p.keys + ((static_cast<long long>(w) * p.n_groups + gl) * p.num_reqs + b) * kSlots + j)
                   : 0ull;
  }
  bool bad = false;
  uint64_t top = 0ull;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int i = 32 * t + lane, w = i / kSlots;
    uint64_t k = kin[t];
    if (k != 0ull) {
      const int id = topk_id(k);
      if (id < 0 || id >= nb - 1 || id % p.world != w) {
        bad = true;
        k = 0ull;
      }
    }
    top = top32_union(top, warp_sort_desc(k));
  }
  // keys are unique when every rank sent distinct blocks of its own; a repeated one is dropped
  const uint64_t prev = shfl_u64(top, lane > 0 ? lane - 1 : 0);
  if (__any_sync(0xFFFFFFFFu, lane > 0 && top != 0ull && top == prev)) {
    bad = true;
    top = warp_sort_desc(lane > 0 && top == prev ? 0ull : top);
  }
  const uint64_t win = lane < kCand ? top : 0ull;
  if (lane < kCand && win == 0ull) bad = true;  // fewer than 15 candidates arrived
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_flag(p.flags, kFlagBadIds);
  // the winners plus the recent block, ascending; -1 after them if candidates were missing
  const int my_id = lane < kCand ? (win != 0ull ? topk_id(win) : -1) : (lane == kCand ? nb - 1 : -1);
  const uint32_t valid = __ballot_sync(0xFFFFFFFFu, my_id >= 0);
  int rank = 0;
#pragma unroll
  for (int t = 0; t < kTopK; ++t) {
    const int other = __shfl_sync(0xFFFFFFFFu, my_id, t);
    rank += other >= 0 && other < my_id ? 1 : 0;
  }
  if (my_id >= 0) ids[rank] = my_id;
  const int nvalid = __popc(valid);
  if (lane >= nvalid && lane < kTopK) ids[lane] = -1;
}

}  // namespace

cudaError_t launch_dcp_local(const SelectParams& prm, uint64_t* keys, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_reqs, 1, 1);
  cfg.blockDim = dim3(kDcpThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, dcp_local_kernel, prm, keys);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dcp_merge(const DcpMergeParams& prm, cudaStream_t st) {
  dcp_merge_kernel<<<prm.num_reqs, 32 * kGroups, 0, st>>>(prm);
  return cudaGetLastError();
}

}  // namespace msa
