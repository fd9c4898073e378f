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
// this kernel is a stream over the cache's pages at HBM speed. One CTA has three
// roles, 2 CTAs per SM (256 TMEM columns each), the grid taking equal contiguous
// ranges of all requests' pages:
//   * load warp: one lane streams pages into a ring of shared-memory stages with
//     TMA (codes: 2-D tensor copy with 64-byte swizzle, so each thread reads its
//     64-byte row without bank conflicts; scales: 1-D bulk copy);
//   * MMA warp: one lane issues the tensor-core MMAs (a single issuing thread
//     sustains about one MMA per 45 cycles, so it does nothing else); the warp
//     rewrites the index-query tile (B operand) when the request changes;
//   * 4 dequant warps (thread = token of the page = TMEM lane): dequantise their
//     token's 128 elements into positive/negative magnitude parts (byte-permute
//     table lookups) and store them into a 3-deep ring of tensor-memory A
//     buffers; the MMA computes scores = A x q_idx^T for the 4 x R index-query
//     columns of the request, FP32 accumulation in tensor memory, the negative
//     part through the negate-B bit (products of two E4M3 values are exact; only
//     the FP32 sums round);
//   * 4 epilogue warps: read each page's scores from a 2-deep ring of tensor-
//     memory D buffers, mask, max-pool over the group's rows and their 32 tokens
//     and write one partial per warp and block.
// The dequant warps never wait for an MMA result, only for a free A buffer, so
// the MMA round trip hides behind the next pages' dequantisation. The CTA that
// completes a request's block scores (an arrival counter, no waiting) runs the
// top-k for that request: one warp per group.
#include <climits>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr int kRowWarps = 4;                       // dequant warps = epilogue warps
constexpr int kThreads = (2 * kRowWarps + 2) * 32;  // + the MMA warp + the TMA warp
constexpr int kIssueWarp = 2 * kRowWarps;          // MMA issue, query tile
constexpr int kLoadWarp = 2 * kRowWarps + 1;       // TMA producer
constexpr int kCtasPerSm = 2;
constexpr int kStages = 6;
constexpr int kABufs = 3, kDBufs = 2;
constexpr uint32_t kCodeBytes = kBlock * 64;    // one page of index-key codes
constexpr uint32_t kScaleBytes = kBlock * 8;    // its scales
constexpr uint32_t kTmemCols = 256;
constexpr int kCtaPages = 2048;                  // block-table entries staged per CTA
// TMEM columns: kABufs A buffers (positive part 32 cols + negative part 32 cols),
// then kDBufs D buffers (scores, up to 32 FP32 columns).
constexpr uint32_t kColA = 0, kColD = 64 * kABufs;

struct Smem {
  LutEntry lut[256];                        // 4 KB
  uint8_t codes[kStages][kCodeBytes];       // 1024-aligned (offset 4096)
  uint8_t qtile[32 * 128];                  // B operand: up to 32 index-query rows x 128 (SW128)
  uint8_t scales[kStages][kScaleBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t afull[kABufs], afree[kABufs], dfull[kDBufs], dempty[kDBufs];
  int stage_bad[kStages];
  int slot_max[4][kGroups];                 // per-page ring: ordered-int max of the epilogue warps' partials
  int slot_cnt[4];                          // epilogue warps that have contributed to the slot
  int32_t phys[kCtaPages];                  // this CTA's block-table entries (when its range fits)
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

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t* flags) {
  return mbar_try(bar, parity) || mbar_wait(bar, parity, flags);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// order-preserving int image of a float (for atomicMax), and back
__device__ __forceinline__ int ord_of(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float float_of(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7FFFFFFF)); }

__device__ __forceinline__ uint32_t bitnot_fma(uint32_t w) {  // ~w on the multiply-add pipe
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, %2;" : "=r"(r) : "r"(w), "r"(0xFFFFFFFFu));
  return r;
}

// Group maxima of a fully visible token: columns n = rq*4 + g, rq < R.
template <int R>
__device__ __forceinline__ void group_max(const uint32_t (&dv)[32], float (&mg)[kGroups]) {
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    float m = __uint_as_float(dv[g]);
#pragma unroll
    for (int rq = 1; rq < R; rq += 2) {
      const float a = __uint_as_float(dv[rq * kGroups + g]);
      const float b = rq + 1 < R ? __uint_as_float(dv[(rq + 1) * kGroups + g]) : a;
      m = fmax3(m, a, b);
    }
    mg[g] = m;
  }
}

// Dequantise 8 code words (4 groups of scale bytes sb0..sb3 = words 2k, 2k+1)
// into 16 positive-part and 16 negative-part words and store them to TMEM.
__device__ __forceinline__ void dequant_store_half(const LutEntry* lut, const uint32_t* w, uint32_t scw,
                                                   uint32_t a_pos, uint32_t a_neg) {
  uint32_t pa[16], na[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const LutEntry L = lut[(scw >> (8 * q)) & 0xFFu];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t x = w[2 * q + h];
      const uint32_t xh = x >> 16;
      pa[4 * q + 2 * h] = prmt(L.p0, L.p1, x);
      pa[4 * q + 2 * h + 1] = prmt(L.p0, L.p1, xh);
      na[4 * q + 2 * h] = prmt(L.n0, L.n1, bitnot_fma(x));
      na[4 * q + 2 * h + 1] = prmt(L.n0, L.n1, bitnot_fma(xh));
    }
  }
  tmem_st16(a_pos, pa);
  tmem_st16(a_neg, na);
}

}  // namespace

// MODE 0: fused select (block scores + top-k). MODE 1: write per-token scores
// (msa_index_scores) and stop.
template <int MODE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
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
    for (int j = 0; j < kABufs; ++j) {
      mbar_init(smem_u32(&sm.afull[j]), kRowWarps);
      mbar_init(smem_u32(&sm.afree[j]), 1);
    }
    for (int k = 0; k < kDBufs; ++k) {
      mbar_init(smem_u32(&sm.dfull[k]), 1);
      mbar_init(smem_u32(&sm.dempty[k]), kRowWarps);
    }
    mbar_fence_init();
  }
  if (tid < 4 * kGroups) sm.slot_max[tid / kGroups][tid % kGroups] = INT_MIN;
  if (tid < 4) sm.slot_cnt[tid] = 0;
  // this CTA's block-table entries, so no page waits on a dependent global load
  const bool staged = n <= kCtaPages;
  if (staged) {
    for (int i = tid; i < n; i += kThreads) {
      const PageCursor pc = cursor_at(p0 + i, prefix, B);
      sm.phys[i] = p.block_table[static_cast<long long>(pc.b) * p.max_pages + pc.c];
    }
  }
  // the first request's index queries (B operand, SW128 layout)
  const int first_req = cursor_at(p0, prefix, B).b;
  {
    const int R = rows_s[first_req], row0 = row0_s[first_req];
    const int nrows = R * kGroups <= 16 ? 16 : 32;
    for (int u = tid; u < nrows * 8; u += kThreads) {
      const int nrow = u >> 3, ch = u & 7;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (nrow < R * kGroups)
        v = *reinterpret_cast<const uint4*>(p.q_idx + (static_cast<long long>(row0) * kGroups + nrow) * kDim + ch * 16);
      *reinterpret_cast<uint4*>(sm.qtile + nrow * 128 + ((ch ^ (nrow & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
  }
  if (warp == kIssueWarp) tmem_alloc(smem_u32(&sm.taddr), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.taddr;
  bool alive = true;

  if (warp == kLoadWarp) {
    // ================= load warp: TMA producer (one lane)
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ki_map)) : "memory");
      PageCursor ld = cursor_at(p0, prefix, B);
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        if (i >= kStages) {  // the dequant warps have released this stage's previous page
          alive = wait_bar(smem_u32(&sm.empty[s]), ((i / kStages) - 1) & 1, p.flags);
          if (!alive) break;
        }
        const int phys = staged ? sm.phys[i] : p.block_table[static_cast<long long>(ld.b) * p.max_pages + ld.c];
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
        cursor_advance(ld, nb);
      }
      if (!alive) {
        // drain: copies already issued complete on their own barriers
        for (int i = 0; i < n; ++i) {
          const int s = i % kStages;
          if (!mbar_wait(smem_u32(&sm.full[s]), (i / kStages) & 1, p.flags)) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == kIssueWarp) {
    // ================= MMA warp: MMA issue (lane 0), query tile (all lanes)
    PageCursor mm = cursor_at(p0, prefix, B);
    int qtile_req = first_req;
    const uint32_t qt = smem_u32(sm.qtile);
    for (int i = 0; i < n; ++i) {
      const int j = i % kABufs, k = i % kDBufs;
      if (mm.b != qtile_req) {
        // new request: once every earlier MMA has finished reading the tile, rewrite it
        if (i >= 1) alive = wait_bar(smem_u32(&sm.dfull[(i - 1) % kDBufs]), ((i - 1) / kDBufs) & 1, p.flags);
        if (!__all_sync(0xFFFFFFFFu, alive)) {
          alive = false;
          break;
        }
        const int R = rows_s[mm.b], row0 = row0_s[mm.b];
        const int nrows = R * kGroups <= 16 ? 16 : 32;
        for (int u = lane; u < nrows * 8; u += 32) {
          const int nrow = u >> 3, ch = u & 7;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (nrow < R * kGroups)
            v = *reinterpret_cast<const uint4*>(p.q_idx + (static_cast<long long>(row0) * kGroups + nrow) * kDim +
                                                ch * 16);
          *reinterpret_cast<uint4*>(sm.qtile + nrow * 128 + ((ch ^ (nrow & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        qtile_req = mm.b;
      }
      if (lane == 0) {
        alive = wait_bar(smem_u32(&sm.afull[j]), (i / kABufs) & 1, p.flags);
        if (alive && i >= kDBufs) alive = wait_bar(smem_u32(&sm.dempty[k]), ((i / kDBufs) - 1) & 1, p.flags);
        if (alive) {
          tc_fence_after();
          const int R = rows_s[mm.b];
          const int N = R * kGroups <= 16 ? 16 : 32;
          const uint32_t id_pos = idesc_e4m3_f32(128, N, false), id_neg = idesc_e4m3_f32(128, N, true);
          const uint32_t d = tbase + kColD + 32 * k, a = tbase + kColA + 64 * j;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_tmemA(d, a + 8 * kk, sdesc_kmajor_sw128(qt + 32 * kk), id_pos, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_tmemA(d, a + 32 + 8 * kk, sdesc_kmajor_sw128(qt + 32 * kk), id_neg, 1);
          mma_commit(smem_u32(&sm.dfull[k]));
          mma_commit(smem_u32(&sm.afree[j]));
        }
      }
      cursor_advance(mm, nb);
      if (!__all_sync(0xFFFFFFFFu, alive)) {
        alive = false;
        break;
      }
    }
    __syncwarp();
  } else if (warp < kRowWarps) {
    // ================= dequant warps: page i -> TMEM A buffer i % kABufs
    const int r = tid;  // token slot within the page = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int i = 0; i < n; ++i) {
      const int s = i % kStages, j = i % kABufs;
      uint32_t w[16];
      alive = wait_bar(smem_u32(&sm.full[s]), (i / kStages) & 1, p.flags);
      if (!alive) break;
      // this thread's row: 64 code bytes (swizzled 16-byte chunks) + 8 scale bytes
      const uint8_t* row = sm.codes[s] + r * 64;
      const int sw = (r >> 1) & 3;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
      const uint2 sc = *reinterpret_cast<const uint2*>(sm.scales[s] + r * 8);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
      if (i >= kABufs) {  // the MMA that read this A buffer last time has finished
        alive = wait_bar(smem_u32(&sm.afree[j]), ((i / kABufs) - 1) & 1, p.flags);
        if (!alive) break;
        tc_fence_after();
      }
      const uint32_t a_lane = tbase + lane_base + kColA + 64 * j;
      dequant_store_half(sm.lut, w, sc.x, a_lane, a_lane + 32);
      dequant_store_half(sm.lut, w + 8, sc.y, a_lane + 16, a_lane + 48);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.afull[j]));
    }
  } else {
    // ================= epilogue warps: scores of page i from TMEM D buffer i % kDBufs
    const int ew = warp - kRowWarps;  // 0..3: TMEM lanes 32ew..32ew+31 (warp % 4 == ew)
    const int r = ew * 32 + lane;     // token slot within the page
    const uint32_t lane_base = static_cast<uint32_t>(ew * 32) << 16;
    PageCursor cur = cursor_at(p0, prefix, B);
    for (int i = 0; i < n; ++i) {
      const int k = i % kDBufs;
      alive = wait_bar(smem_u32(&sm.dfull[k]), (i / kDBufs) & 1, p.flags);
      if (!alive) break;
      tc_fence_after();
      uint32_t dv[32];
      tmem_ld32(tbase + lane_base + kColD + 32 * k, dv);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.dempty[k]));
      const int b = cur.b, c = cur.c;
      // the page's stage may already hold a later page: take the bad-id flag from the table
      const int phys = staged ? sm.phys[i] : p.block_table[static_cast<long long>(b) * p.max_pages + c];
      const bool page_bad = phys < 0 || phys >= p.num_pages;
      const int N = ctx_s[b], R = rows_s[b];
      const int t = c * kBlock + r;
      float mg[kGroups];
      if (MODE == 0 && !page_bad && c * kBlock + kBlock - 1 <= N - R) {
        // every token of the page is visible to every row
        switch (R) {
          case 1: group_max<1>(dv, mg); break;
          case 2: group_max<2>(dv, mg); break;
          case 3: group_max<3>(dv, mg); break;
          case 4: group_max<4>(dv, mg); break;
          case 5: group_max<5>(dv, mg); break;
          case 6: group_max<6>(dv, mg); break;
          case 7: group_max<7>(dv, mg); break;
          default: group_max<8>(dv, mg); break;
        }
      } else {
        const int row0 = row0_s[b];
#pragma unroll
        for (int g = 0; g < kGroups; ++g) mg[g] = -INFINITY;
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
      }
      if (MODE == 0) {
        // this warp's 32 tokens, then the 4 epilogue warps' maxima merged in a
        // shared-memory slot; the warp that completes the slot writes the block
        // score and frees the slot (epilogue warps are at most 2 pages apart, so a
        // ring of 4 slots never collides)
        const float m0 = warp_max(mg[0]), m1 = warp_max(mg[1]), m2 = warp_max(mg[2]), m3 = warp_max(mg[3]);
        const int slot = i & 3;
        if (lane < kGroups) atomicMax(&sm.slot_max[slot][lane], ord_of(lane == 0 ? m0 : lane == 1 ? m1 : lane == 2 ? m2 : m3));
        __threadfence_block();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&sm.slot_cnt[slot], 1) == kRowWarps - 1;
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        if (last) {
          __threadfence_block();
          if (lane < kGroups) {
            const int v = atomicExch(&sm.slot_max[slot][lane], INT_MIN);
            p.block_S[(static_cast<long long>(b) * kGroups + lane) * p.s_stride + c] = float_of(v);
          }
          __syncwarp();
          if (lane == 0) atomicExch(&sm.slot_cnt[slot], 0);
        }
      }
      cursor_advance(cur, nb);
    }
  }

  // ---- teardown
  tc_fence_before();
  const bool all_alive = __syncthreads_and(alive ? 1 : 0) != 0;
  if (warp == kIssueWarp) {
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
  uint64_t* tk_scratch = reinterpret_cast<uint64_t*>(sm.codes[0]) + 64 * warp;  // stages are free now
  for (int k = 0; k < sm.ntodo; ++k) {
    const int b = todo[k];
    if (warp < kGroups) {
      const float* S = p.block_S + (static_cast<long long>(b) * kGroups + warp) * p.s_stride;
      warp_topk(S, nb[b], p.block_ids + (static_cast<long long>(b) * kGroups + warp) * kTopK, tk_scratch);
      if (p.block_scores_out != nullptr) {
        float* o = p.block_scores_out + (static_cast<long long>(b) * kGroups + warp) * p.max_pages;
        for (int c = lane; c < p.max_pages; c += 32) o[c] = c < nb[b] ? S[c] : -INFINITY;
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
  float* S = p.block_S + (static_cast<long long>(b) * kGroups + warp) * p.s_stride;
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
    if (lane == 0) S[c] = m;
  }
  __syncwarp();
  __shared__ uint64_t scratch[4][64];
  warp_topk(S, nb, ids, scratch[warp]);
  if (p.block_scores_out != nullptr) {
    float* o = p.block_scores_out + (static_cast<long long>(b) * kGroups + warp) * p.max_pages;
    for (int c = lane; c < p.max_pages; c += 32) o[c] = c < nb ? S[c] : -INFINITY;
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

cudaError_t launch_select(const CUtensorMap& ki_map, const SelectParams& prm, int mode, int sm_count,
                          cudaStream_t st) {
  const size_t smem = select_smem_bytes(prm.num_reqs);
  const int grid = kCtasPerSm * sm_count;
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
