// Steps 1-3 of the MSA decode path: the index scan, the block max pool and the
// top-k block selection.
//
// [vLLM-zh "How MiniMax sparse attention works"] a lightweight indexer scores
// every key in the context, one index query per GQA group against a single
// shared index-key head, max-pools the scores to one per 128-token block and
// keeps the top 16 blocks with the most recent block always kept. [MSA-fig §1]
// the index branch: K_idx has one head shared by all groups; Block Max Pool;
// TopK. The index cache is NVFP4 and is turned into FP8 in the kernel before an
// FP8 MMA [vLLM-zh, Blackwell kernels].
//
// Design (GB300, sm_103a). Decode reads the whole index-key cache every step, so
// this kernel is a stream over the cache's pages at HBM speed:
//   * One CTA = 4 "row" warps (thread = token of the current page = TMEM lane)
//     + 1 "issue" warp. A grid of 2 CTAs per SM takes equal contiguous ranges
//     of all requests' pages.
//   * The issue warp's elected lane streams pages into a ring of shared-memory
//     stages with TMA (codes: 2-D tensor copy with 64-byte swizzle, so each row
//     thread reads its 64-byte row without bank conflicts; scales: 1-D bulk copy)
//     and issues the tensor-core MMAs.
//   * Row threads dequantise their token's 128 elements into positive/negative
//     magnitude parts (byte-permute table lookups) and store them into tensor
//     memory as the A operand; the MMA computes scores = A x q_idx^T for all
//     4 x R index-query columns of the request (B = q_idx in shared memory),
//     accumulating in FP32 in tensor memory, the negative part through the
//     negate-B bit. Products of two E4M3 values are exact; only the FP32 sums
//     round.
//   * The epilogue reads each token's scores from tensor memory, applies the
//     causal mask, takes the max over the group's rows and over the block's
//     128 tokens and writes one FP32 block score per (request, group, block).
//   * The CTA that completes a request's block scores (an arrival counter, no
//     waiting) runs the top-k for that request: one warp per group.
#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr int kRowWarps = 4;
constexpr int kThreads = (kRowWarps + 1) * 32;
constexpr int kStages = 6;
constexpr uint32_t kCodeBytes = kBlock * 64;    // one page of index-key codes
constexpr uint32_t kScaleBytes = kBlock * 8;    // its scales
constexpr uint32_t kTmemCols = 256;
// TMEM columns: A buffers (positive part 32 cols + negative part 32 cols) x2,
// then D (scores, up to 32 FP32 columns) x2.
constexpr uint32_t kColA0 = 0, kColD0 = 128;

struct Smem {
  LutEntry lut[256];                        // 4 KB
  uint8_t codes[kStages][kCodeBytes];       // 1024-aligned (offset 4096)
  uint8_t qtile[32 * 128];                  // B operand: up to 32 index-query rows x 128 (SW128)
  uint8_t scales[kStages][kScaleBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t afull[2], dfull[2], dempty[2];
  int stage_bad[kStages];
  uint32_t taddr;
  int ntodo;
};

struct PageCursor {
  int b;       // request
  int c;       // logical block within the request
};

__device__ __forceinline__ void cursor_advance(PageCursor& pc, const int* nb) {
  ++pc.c;
  while (pc.c >= nb[pc.b]) {
    pc.c = 0;
    ++pc.b;
  }
}

// Locate global page index p: request b with prefix[b] <= p < prefix[b+1].
__device__ __forceinline__ PageCursor cursor_at(long long p, const long long* prefix, int B) {
  int lo = 0, hi = B;  // invariant prefix[lo] <= p < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= p) lo = mid;
    else hi = mid;
  }
  PageCursor pc;
  pc.b = lo;
  pc.c = static_cast<int>(p - prefix[lo]);
  return pc;
}

}  // namespace

// MODE 0: fused select (block scores + top-k). MODE 1: write per-token scores
// (msa_index_scores) and stop.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 2)
    select_kernel(const __grid_constant__ CUtensorMap ki_map, const SelectParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem_al = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // TMA/UMMA tiles need 1 KB
  Smem& sm = *reinterpret_cast<Smem*>(smem_al);
  long long* prefix = reinterpret_cast<long long*>(smem_al + sizeof(Smem));  // [B+1]
  int* nb = reinterpret_cast<int*>(prefix + (p.num_reqs + 1));              // [B+1] (sentinel)
  int* rows_s = nb + (p.num_reqs + 1);                                     // [B]
  int* row0_s = rows_s + p.num_reqs;                                        // [B]
  int* ctx_s = row0_s + p.num_reqs;                                         // [B]
  int* todo = ctx_s + p.num_reqs;                                           // [B]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.num_reqs;

  if (MODE == 0) pdl_launch_dependents();

  // ---- per-request geometry (validated) and the page prefix sum
  for (int b = tid; b < B; b += kThreads) {
    const int N = p.context_lens[b];
    const int r0 = p.q_indptr[b], r1 = p.q_indptr[b + 1];
    const int R = r1 - r0;
    int pages = (N + kBlock - 1) / kBlock;
    const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                    r1 <= p.total_rows;
    if (!ok) {
      if (blockIdx.x == 0) set_flag(p.flags, kFlagBadLength);
      pages = 0;
    }
    if (R == 0) pages = 0;
    nb[b] = pages;
    rows_s[b] = ok ? R : 0;
    row0_s[b] = ok ? r0 : 0;
    ctx_s[b] = ok ? N : 0;
  }
  if (tid == 0) nb[B] = 1 << 30;  // sentinel stops cursor walks
  __syncthreads();
  if (tid == 0) {  // B is at most a few thousand; a serial prefix is cheap
    long long acc = 0;
    for (int b = 0; b < B; ++b) {
      prefix[b] = acc;
      acc += nb[b];
    }
    prefix[B] = acc;
    sm.ntodo = 0;
  }
  __syncthreads();
  const long long total = prefix[B];
  const long long G = gridDim.x;
  const long long p0 = total * blockIdx.x / G, p1 = total * (blockIdx.x + 1) / G;
  const int n = static_cast<int>(p1 - p0);

  // requests with no pages get empty selections (written by CTA 0)
  if (MODE == 0 && blockIdx.x == 0) {
    for (int i = tid; i < B * kGroups * kTopK; i += kThreads) {
      const int b = i / (kGroups * kTopK);
      if (nb[b] == 0) p.block_ids[i] = -1;
    }
    if (p.block_scores_out != nullptr)
      for (long long i = tid; i < static_cast<long long>(B) * kGroups * p.max_pages; i += kThreads) {
        const int b = static_cast<int>(i / (kGroups * p.max_pages));
        if (nb[b] == 0) p.block_scores_out[i] = -INFINITY;
      }
  }
  if (n <= 0) return;

  // ---- setup: table, barriers, tensor memory
  build_lut(sm.lut);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kRowWarps);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&sm.afull[j]), kRowWarps);
      mbar_init(smem_u32(&sm.dfull[j]), 1);
      mbar_init(smem_u32(&sm.dempty[j]), kRowWarps);
    }
    mbar_fence_init();
  }
  if (warp == kRowWarps) tmem_alloc(smem_u32(&sm.taddr), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.taddr;
  bool alive = true;

  if (warp == kRowWarps) {
    // ================= issue warp: TMA producer + MMA issuer (one lane)
    if (lane == 0) {
      PageCursor ld = cursor_at(p0, prefix, B);
      PageCursor mm = ld;
      int issued = 0;
      auto issue_load = [&](int i, const PageCursor& pc) {
        const int s = i % kStages;
        const int phys = p.block_table[static_cast<long long>(pc.b) * p.max_pages + pc.c];
        const bool bad = phys < 0 || phys >= p.num_pages;
        sm.stage_bad[s] = bad ? 1 : 0;
        const uint32_t bar = smem_u32(&sm.full[s]);
        if (bad) {
          set_flag(p.flags, kFlagBadPage);
          mbar_arrive(bar);
        } else {
          mbar_arrive_expect_tx(bar, kCodeBytes + kScaleBytes);
          tma_load_2d(smem_u32(sm.codes[s]), &ki_map, 0, phys * kBlock, bar);
          bulk_load(smem_u32(sm.scales[s]), p.ki_scale + static_cast<long long>(phys) * kScaleBytes, kScaleBytes,
                    bar);
        }
      };
      for (; issued < n && issued < kStages; ++issued) {
        issue_load(issued, ld);
        cursor_advance(ld, nb);
      }
      for (int i = 0; i < n && alive; ++i) {
        const int j = i & 1;
        alive = mbar_wait(smem_u32(&sm.afull[j]), (i >> 1) & 1, p.flags);
        if (alive && i >= 2) alive = mbar_wait(smem_u32(&sm.dempty[j]), ((i - 2) >> 1) & 1, p.flags);
        if (!alive) break;
        tc_fence_after();
        const int R = rows_s[mm.b];
        const int ncols = R * kGroups;
        const int N = ncols <= 16 ? 16 : 32;
        const uint32_t id_pos = idesc_e4m3_f32(128, N, false), id_neg = idesc_e4m3_f32(128, N, true);
        const uint32_t d = tbase + kColD0 + 32 * j;
        const uint32_t a = tbase + kColA0 + 64 * j;
        const uint32_t qt = smem_u32(sm.qtile);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_f8_tmemA(d, a + 8 * k, sdesc_kmajor_sw128(qt + 32 * k), id_pos, k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_f8_tmemA(d, a + 32 + 8 * k, sdesc_kmajor_sw128(qt + 32 * k), id_neg, 1);
        mma_commit(smem_u32(&sm.dfull[j]));
        cursor_advance(mm, nb);
        if (issued < n) {
          const int s = issued % kStages;
          alive = mbar_wait(smem_u32(&sm.empty[s]), ((issued / kStages) - 1) & 1, p.flags);
          if (!alive) break;
          issue_load(issued, ld);
          cursor_advance(ld, nb);
          ++issued;
        }
      }
      if (!alive) {
        // drain: copies already issued complete on their own barriers
        for (int i = 0; i < issued; ++i) {
          const int s = i % kStages;
          if (!mbar_wait(smem_u32(&sm.full[s]), (i / kStages) & 1, p.flags)) break;
        }
      }
    }
    __syncwarp();
  } else {
    // ================= row warps: dequantise -> TMEM, epilogue
    const int r = tid;  // token slot within the page = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    PageCursor cur = cursor_at(p0, prefix, B);
    PageCursor prev = cur;
    int qtile_req = -1;
    bool cur_bad = false, prev_bad = false;  // page i / i-1 came from an out-of-range page id
    for (int i = 0; i <= n && alive; ++i) {
      uint32_t pa[32], na[32];
      if (i < n) {
        const int s = i % kStages;
        alive = mbar_wait(smem_u32(&sm.full[s]), (i / kStages) & 1, p.flags);
        if (!alive) break;
        cur_bad = sm.stage_bad[s] != 0;  // read now: the stage is refilled once released
        // this thread's row: 64 code bytes (swizzled 16-byte chunks) + 8 scale bytes
        const uint8_t* row = sm.codes[s] + r * 64;
        const int sw = (r >> 1) & 3;
        uint4 cw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) cw[c] = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
        const uint2 scw = *reinterpret_cast<const uint2*>(sm.scales[s] + r * 8);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
        const uint32_t w[16] = {cw[0].x, cw[0].y, cw[0].z, cw[0].w, cw[1].x, cw[1].y, cw[1].z, cw[1].w,
                                cw[2].x, cw[2].y, cw[2].z, cw[2].w, cw[3].x, cw[3].y, cw[3].z, cw[3].w};
#pragma unroll
        for (int gsc = 0; gsc < 8; ++gsc) {  // 16-element group gsc = code words 2gsc, 2gsc+1
          const uint32_t sb = ((gsc < 4 ? scw.x : scw.y) >> (8 * (gsc & 3))) & 0xFFu;
          const LutEntry L = sm.lut[sb];
          dq8_split(w[2 * gsc], L, pa[4 * gsc + 0], pa[4 * gsc + 1], na[4 * gsc + 0], na[4 * gsc + 1]);
          dq8_split(w[2 * gsc + 1], L, pa[4 * gsc + 2], pa[4 * gsc + 3], na[4 * gsc + 2], na[4 * gsc + 3]);
        }
      }
      // ---- epilogue of page i-1
      if (i >= 1) {
        const int jp = (i - 1) & 1;
        alive = mbar_wait(smem_u32(&sm.dfull[jp]), ((i - 1) >> 1) & 1, p.flags);
        if (!alive) break;
        tc_fence_after();
        uint32_t dv[32];
        tmem_ld32(tbase + lane_base + kColD0 + 32 * jp, dv);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.dempty[jp]));
        const int b = prev.b, c = prev.c;
        const int N = ctx_s[b], R = rows_s[b], row0 = row0_s[b];
        const int t = c * kBlock + r;
        const bool page_bad = prev_bad;
        float mg[kGroups] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int rq = 0; rq < kMaxRows; ++rq) {
          if (rq < R) {
            const bool vis = !page_bad && t <= N - R + rq;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
              const float v = vis ? __uint_as_float(dv[rq * kGroups + g]) : -INFINITY;
              mg[g] = fmaxf(mg[g], v);
              if (MODE == 1 && t < N)
                p.token_scores[(static_cast<long long>(row0 + rq) * kGroups + g) * p.score_stride + t] = v;
            }
          }
        }
        if (MODE == 0) {
          // this warp's 32 tokens; the 4 warps' partial maxima of a block sit side
          // by side and the top-k takes their max (no cross-warp barrier)
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mg[g] = fmaxf(mg[g], __shfl_xor_sync(0xFFFFFFFFu, mg[g], off));
          }
          if (lane < kGroups) {
            const float v = lane == 0 ? mg[0] : lane == 1 ? mg[1] : lane == 2 ? mg[2] : mg[3];
            p.block_S[((static_cast<long long>(b) * kGroups + lane) * p.max_pages + c) * kRowWarps + warp] = v;
          }
        }
      }
      prev = cur;
      prev_bad = cur_bad;
      if (i == n) break;
      // ---- B operand: the request's index queries, rows n = rq*4 + g (SW128 layout)
      if (cur.b != qtile_req) {
        const int R = rows_s[cur.b], row0 = row0_s[cur.b];
        const int nrows = R * kGroups <= 16 ? 16 : 32;
        for (int u = r; u < nrows * 8; u += kRowWarps * 32) {
          const int nrow = u >> 3, ch = u & 7;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (nrow < R * kGroups)
            v = *reinterpret_cast<const uint4*>(p.q_idx + (static_cast<long long>(row0) * kGroups + nrow) * kDim +
                                                ch * 16);
          *reinterpret_cast<uint4*>(sm.qtile + nrow * 128 + ((ch ^ (nrow & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        qtile_req = cur.b;
      }
      // ---- A operand into TMEM: positive part cols [0,32), negative part [32,64)
      const int j = i & 1;
      const uint32_t a = tbase + lane_base + kColA0 + 64 * j;
      uint32_t h[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) h[k] = pa[k];
      tmem_st16(a, h);
#pragma unroll
      for (int k = 0; k < 16; ++k) h[k] = pa[16 + k];
      tmem_st16(a + 16, h);
#pragma unroll
      for (int k = 0; k < 16; ++k) h[k] = na[k];
      tmem_st16(a + 32, h);
#pragma unroll
      for (int k = 0; k < 16; ++k) h[k] = na[16 + k];
      tmem_st16(a + 48, h);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.afull[j]));
      cursor_advance(cur, nb);
    }
  }

  // ---- teardown
  tc_fence_before();
  const bool all_alive = __syncthreads_and(alive ? 1 : 0) != 0;
  if (warp == kRowWarps) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  if (MODE != 0 || !all_alive) return;

  // ---- arrival: the CTA completing a request's block scores runs its top-k
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    PageCursor pc = cursor_at(p0, prefix, B);
    long long q = p0;
    while (q < p1) {
      const int b = pc.b;
      const long long end = prefix[b + 1] < p1 ? prefix[b + 1] : p1;
      const unsigned cnt = static_cast<unsigned>(end - q);
      const unsigned old = atomicAdd(p.req_cnt + b, cnt);
      if (old + cnt == static_cast<unsigned>(nb[b])) {
        p.req_cnt[b] = 0u;
        todo[sm.ntodo++] = b;
      }
      q = end;
      pc.b = b + 1;
      pc.c = 0;
      while (pc.b < B && nb[pc.b] == 0) ++pc.b;
    }
  }
  __syncthreads();
  __threadfence();
  for (int k = 0; k < sm.ntodo; ++k) {
    const int b = todo[k];
    if (warp < kGroups) {
      const float4* S = reinterpret_cast<const float4*>(p.block_S) +
                        (static_cast<long long>(b) * kGroups + warp) * p.max_pages;
      warp_topk(S, nb[b], p.block_ids + (static_cast<long long>(b) * kGroups + warp) * kTopK);
      if (p.block_scores_out != nullptr) {
        float* o = p.block_scores_out + (static_cast<long long>(b) * kGroups + warp) * p.max_pages;
        for (int c = lane; c < p.max_pages; c += 32) o[c] = c < nb[b] ? max4(S[c]) : -INFINITY;
      }
    }
  }
}

// Steps 2+3 from given per-token scores: one CTA per request, warp g pools and
// selects group g.
__global__ void __launch_bounds__(128) maxpool_topk_kernel(const MaxpoolParams p) {
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows;
  int32_t* ids = p.block_ids + (static_cast<long long>(b) * kGroups + warp) * kTopK;
  if (!ok || R == 0) {
    if (!ok && lane == 0) set_flag(p.flags, kFlagBadLength);
    if (lane < kTopK) ids[lane] = -1;
    if (p.block_scores_out != nullptr)
      for (int c = lane; c < p.max_pages; c += 32)
        p.block_scores_out[(static_cast<long long>(b) * kGroups + warp) * p.max_pages + c] = -INFINITY;
    return;
  }
  const int nb = (N + kBlock - 1) / kBlock;
  float4* S = reinterpret_cast<float4*>(p.block_S) + (static_cast<long long>(b) * kGroups + warp) * p.max_pages;
  for (int c = 0; c < nb; ++c) {
    float m = -INFINITY;
    for (int rq = 0; rq < R; ++rq) {
      const int pos = N - R + rq;
      for (int t = c * kBlock + lane; t < (c + 1) * kBlock && t < N; t += 32) {
        const float v = t <= pos ? p.scores[(static_cast<long long>(r0 + rq) * kGroups + warp) * p.score_stride + t]
                                 : -INFINITY;
        m = fmaxf(m, v);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane == 0) S[c] = make_float4(m, m, m, m);
  }
  __syncwarp();
  warp_topk(S, nb, ids);
  if (p.block_scores_out != nullptr) {
    float* o = p.block_scores_out + (static_cast<long long>(b) * kGroups + warp) * p.max_pages;
    for (int c = lane; c < p.max_pages; c += 32) o[c] = c < nb ? max4(S[c]) : -INFINITY;
  }
}

// Exposes the two dequantisers for checking.
__global__ void dequant_rows_kernel(const uint8_t* codes, const uint8_t* scales, long long nrows, uint8_t* out,
                                    int path) {
  __shared__ LutEntry lut[256];
  build_lut(lut);
  __syncthreads();
  const long long nwords = nrows * 16;
  for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < nwords;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = u >> 4;
    const int wi = static_cast<int>(u & 15);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + row * 64 + wi * 4);
    const LutEntry L = lut[scales[row * 8 + wi / 2]];
    uint32_t r0, r1;
    if (path == 0) {
      dq8_signed(w, L.p0, L.p1, r0, r1);
    } else {
      uint32_t p0, p1, n0, n1;
      dq8_split(w, L, p0, p1, n0, n1);
      // recombine: positive part where non-zero, else the negative part with its sign bit
      r0 = 0;
      r1 = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t a0 = (p0 >> (8 * k)) & 0xFFu, b0 = (n0 >> (8 * k)) & 0xFFu;
        const uint32_t a1 = (p1 >> (8 * k)) & 0xFFu, b1 = (n1 >> (8 * k)) & 0xFFu;
        r0 |= (a0 != 0 ? a0 : (b0 != 0 ? (b0 | 0x80u) : 0u)) << (8 * k);
        r1 |= (a1 != 0 ? a1 : (b1 != 0 ? (b1 | 0x80u) : 0u)) << (8 * k);
      }
    }
    *reinterpret_cast<uint32_t*>(out + row * 128 + wi * 8) = r0;
    *reinterpret_cast<uint32_t*>(out + row * 128 + wi * 8 + 4) = r1;
  }
}

size_t select_smem_bytes(int num_reqs) {
  const size_t need = sizeof(Smem) + sizeof(long long) * (num_reqs + 1) + sizeof(int) * (num_reqs + 1) +
                      4 * sizeof(int) * num_reqs + 1024;
  // at least 80 KB so no more than two CTAs share an SM's 512 tensor-memory columns
  return need > 80 * 1024 ? need : 80 * 1024;
}

cudaError_t launch_select(const CUtensorMap& ki_map, const SelectParams& prm, int mode, int grid, cudaStream_t st) {
  const size_t smem = select_smem_bytes(prm.num_reqs);
  cudaError_t e;
  if (mode == 0) {
    e = cudaFuncSetAttribute(select_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    select_kernel<0><<<grid, kThreads, smem, st>>>(ki_map, prm);
  } else {
    e = cudaFuncSetAttribute(select_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    select_kernel<1><<<grid, kThreads, smem, st>>>(ki_map, prm);
  }
  return cudaGetLastError();
}

cudaError_t launch_maxpool_topk(const MaxpoolParams& prm, cudaStream_t st) {
  maxpool_topk_kernel<<<prm.num_reqs, 128, 0, st>>>(prm);
  return cudaGetLastError();
}

cudaError_t launch_dequant_rows(const uint8_t* codes, const uint8_t* scales, long long nrows, uint8_t* out, int path,
                                cudaStream_t st) {
  long long blocks = (nrows * 16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  dequant_rows_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(codes, scales, nrows, out, path);
  return cudaGetLastError();
}

}  // namespace msa
