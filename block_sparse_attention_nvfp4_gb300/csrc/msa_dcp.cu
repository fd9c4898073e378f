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

// Descending order of a bitonic sequence held one value per lane (half-cleaners only).
__device__ __forceinline__ uint64_t warp_bitonic_merge_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = shfl_xor_u64(v, j);
    const bool lower = (lane & j) == 0;
    v = lower ? (o > v ? o : v) : (o < v ? o : v);
  }
  return v;
}

// The 32 largest of two descending lists (one value per lane), descending: the larger of
// a[i] and b[31 - i] over all i are those 32 values, and they form a bitonic sequence.
__device__ __forceinline__ uint64_t top32_union(uint64_t a, uint64_t b) {
  const int lane = threadIdx.x & 31;
  const uint64_t r = shfl_u64(b, 31 - lane);
  return warp_bitonic_merge_desc(a > r ? a : r);
}

// Keys of candidates c0 .. c1-1 of S (block scores an earlier kernel wrote: loads bypass
// L1), id field = candidate index; batch `base` gives lane l the candidates
// c0 + base + 32u + l, u < 8. All 8 loads are issued before the keys are formed.
__device__ __forceinline__ void load_keys8(const float* S, int c0, int c1, int base, uint64_t (&k)[8]) {
  const int lane = threadIdx.x & 31;
  float v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int c = c0 + base + 32 * u + lane;
    v[u] = c < c1 ? __ldcg(S + c) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int c = c0 + base + 32 * u + lane;
    k[u] = c < c1 ? topk_key(v[u], c) : 0ull;
  }
}

// Gather the keys >= T of one batch into surv (up to 64), counting all of them.
__device__ __forceinline__ void keep_survivors(const uint64_t (&k)[8], uint64_t T, uint64_t* surv, int& count) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const bool keep = k[u] != 0ull && k[u] >= T;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
    const int pos = count + __popc(bal & ((1u << lane) - 1u));
    if (keep && pos < 64) surv[pos] = k[u];
    count += __popc(bal);
  }
}

// The 15 largest keys of candidates c0 .. c1-1, descending: lane i < 15 returns the i-th
// (0 past the end). The 15th largest lane maximum T is at most the 15th largest key, so
// the keys >= T hold the answer; they are gathered (up to 64) and sorted. If more than 64
// pass, the candidates are merged 32 at a time into a running top 32 instead. Ranges of
// at most 256 candidates are read once, into registers; longer ones are streamed twice.
__device__ uint64_t warp_best15(const float* S, int c0, int c1, uint64_t* surv) {
  const int lane = threadIdx.x & 31;
  const int n = c1 - c0;
  uint64_t lmax = 0ull;
  uint64_t kr[8];
  if (n <= 256) {
    load_keys8(S, c0, c1, 0, kr);
#pragma unroll
    for (int u = 0; u < 8; ++u) lmax = kr[u] > lmax ? kr[u] : lmax;
  } else {
    for (int base = 0; base < n; base += 256) {
      uint64_t k[8];
      load_keys8(S, c0, c1, base, k);
#pragma unroll
      for (int u = 0; u < 8; ++u) lmax = k[u] > lmax ? k[u] : lmax;
    }
  }
  const uint64_t T = shfl_u64(warp_sort_desc(lmax), kCand - 1);
  int count = 0;
  if (n <= 256) {
    keep_survivors(kr, T, surv, count);
  } else {
    for (int base = 0; base < n; base += 256) {
      uint64_t k[8];
      load_keys8(S, c0, c1, base, k);
      keep_survivors(k, T, surv, count);
    }
  }
  __syncwarp();
  uint64_t top;
  if (count <= 32) {
    top = warp_sort_desc(lane < count ? surv[lane] : 0ull);
  } else if (count <= 64) {
    const uint64_t a = warp_sort_desc(surv[lane]);
    const uint64_t b = warp_sort_desc(lane + 32 < count ? surv[lane + 32] : 0ull);
    top = top32_union(a, b);
  } else {
    top = 0ull;
    for (int base = 0; base < n; base += 256) {
      uint64_t k[8];
      if (n <= 256) {
#pragma unroll
        for (int u = 0; u < 8; ++u) k[u] = kr[u];
      } else {
        load_keys8(S, c0, c1, base, k);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint64_t kk = k[u] >= T ? k[u] : 0ull;
        if (__any_sync(0xFFFFFFFFu, kk != 0ull)) top = top32_union(top, warp_sort_desc(kk));
      }
    }
  }
  __syncwarp();
  return lane < kCand ? top : 0ull;
}

// Rank-local lists, after the scan of the rank's blocks (chained to it by programmatic
// dependent launch): one CTA per request, four warps per group, warp q of group g taking
// a quarter of the group's candidates; the group's warp 0 merges the four quarter lists
// (each the exact best 15 of its quarter, so their union holds the group's best 15).
// block_S column i holds the score of logical block i * world + rank.
__global__ void __launch_bounds__(kDcpThreads) dcp_local_kernel(const SelectParams p, uint64_t* keys) {
  __shared__ uint64_t surv[kGroups][4][64];
  __shared__ uint64_t lists[kGroups][4][kSlots];
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
  const int c0 = q * nc / 4, c1 = (q + 1) * nc / 4;
  uint64_t k = 0ull;
  if (c1 > c0) k = warp_best15(p.block_S + (static_cast<long long>(b) * kGroups + g) * p.s_stride, c0, c1, surv[g][q]);
  if (lane < kSlots) lists[g][q][lane] = k;
  named_bar_sync(1 + g, 128);
  if (q != 0) return;
  uint64_t top = lane < kSlots ? lists[g][0][lane] : 0ull;
#pragma unroll
  for (int w = 1; w < 4; ++w) top = top32_union(top, lane < kSlots ? lists[g][w][lane] : 0ull);
  k = lane < kCand ? top : 0ull;
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
