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
// this kernel is a stream over the cache's pages. One CTA per SM (896 threads, all
// 512 TMEM columns), the grid taking equal contiguous ranges of all requests' pages;
// the CTA's warps have four roles (details at the role constants below):
//   * 2 load warps (one lane each, alternate pages): stream pages into a ring of
//     shared-memory stages with TMA (codes: 2-D tensor copy with 64-byte swizzle, so
//     each thread reads its 64-byte row without bank conflicts; scales: 1-D bulk);
//   * 16 dequant warps in 4 groups taking pages round-robin (thread = token): take
//     the token's codes into registers, release the stage, dequantise its 128
//     elements to E4M3 (byte-permute table lookups for magnitudes and signs) and
//     write them as row `token` of a page tile (the MMA's B operand, K-major,
//     128-byte swizzle); MODE 2 writes the exact FP16 values instead;
//   * 2 MMA warps (alternate pages, each with its own copy of the query tile): one
//     lane issues, per page, the weight-stationary D = Q x P^T with Q the request's
//     4 x R index-query rows (M = 32) and P the page (N = 128 tokens, K = 128), FP32
//     accumulation in tensor memory (products of two E4M3 values, or of the FP16
//     forms in MODE 2, are exact; only the FP32 sums round); the warp rewrites its
//     query tile when the request changes;
//   * 8 pool warps in 2 sets taking alternate pages, one warp per TMEM lane
//     quadrant (= 32 of the page's tokens): the TMEM load's max reduction gives each
//     query row's maximum over the quadrant's tokens (masked loads where the causal
//     limit cuts the quadrant), shuffles give the group's maximum over its rows, and
//     every 4 pages a set combines its quadrants into block scores.
// The top-k runs in a second kernel (one CTA per request, four warps per group),
// launched with programmatic dependent launch so its CTAs are resident and have
// read the request geometry when the scan's last pages finish; it waits on the
// scan's completion (griddepcontrol.wait), not on any flag another CTA writes.
#include <climits>
#include <cstddef>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

// Warp roles. Warp w runs on SM sub-partition w % 4 and may read TMEM lanes
// 32 (w % 4) .. + 31. The scores of a page come from the weight-stationary MMA with
// M = 32 (the query columns), whose D puts rows 0..31 in every lane quadrant and the
// page's tokens 32q .. 32q + 31 in quadrant q (32 TMEM columns per page). Four pool
// warps, one per quadrant, reduce a page with the TMEM load's max reduction; each
// dequant group has one warp per sub-partition, so the ALU-heavy work is spread
// evenly. One thread issues an MMA only every ~45-64 cycles (measured on GB300), so
// two MMA warps take alternate pages, each with its own copy of the query tile, and
// so do two load warps. One CTA per SM: the register file holds 24 warps at up to 85
// registers.
constexpr int kLoadWarp = 0;   // TMA producer (even pages)
constexpr int kIssueWarp = 1;  // MMA issue (even pages), query tile 0, TMEM allocation
constexpr int kPoolWarp0 = 2;  // pool warps 2..9: set (w - 2) / 4 takes pages of its parity
constexpr int kPoolSets = 2;
constexpr int kDqWarp0 = kPoolWarp0 + 4 * kPoolSets;  // dequant warps 10..25: group (w - 10) / 4
constexpr int kDqGroups = 4;   // page i is dequantised by group i % kDqGroups
constexpr int kDqWarps = 4 * kDqGroups;
constexpr int kIssueWarp2 = kDqWarp0 + kDqWarps;  // MMA issue (odd pages), query tile 1
constexpr int kIssuers = 2;
constexpr int kLoadWarp2 = kIssueWarp2 + 1;       // TMA producer (odd pages)
constexpr int kLoaders = 2;
constexpr int kThreads = (kLoadWarp2 + 1) * 32;
constexpr int kPoolBatch = 4;  // a pool set's own pages per cross-quadrant combine
constexpr int kCtasPerSm = 1;
constexpr int kStages = 8, kBBufs = 4, kDBufs = 16;
// Every ring slot must have one in-order producer and one in-order consumer, or a
// parity wait could pass on a phase two uses old: a stage is filled by one load warp
// and read by one dequant group, a page tile written by one group and read by one MMA
// warp, a D buffer written by one MMA warp (and read in order by all pool warps).
static_assert(kStages % kLoaders == 0 && kStages % kDqGroups == 0, "stage ring");
static_assert(kBBufs % kIssuers == 0 && kBBufs % kDqGroups == 0, "page-tile ring");
static_assert(kDBufs % kIssuers == 0 && kDBufs % kPoolSets == 0, "D-buffer ring");
constexpr uint32_t kCodeBytes = kBlock * 64;    // one page of index-key codes
constexpr uint32_t kScaleBytes = kBlock * 8;    // its scales
constexpr uint32_t kTileBytes = kBlock * kDim;  // one dequantised page (E4M3)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCols = 32;                 // D buffer: 32 FP32 columns x 4 lane quadrants
constexpr int kCtaPages = 1024;                 // block-table entries staged per CTA
constexpr int kLutCopies = 16;                  // one per thread of a 16-thread (8-byte) wavefront
static_assert(kDBufs * kDCols <= kTmemCols, "TMEM buffers exceed the allocation");
static_assert(kDqWarp0 % 4 == 2 && kPoolWarp0 % 4 == 2, "each group of four warps covers the four lane quadrants");

// MODE 2 (exact scores) keeps the index queries and the page tiles in FP16: each 128-element
// row is two 64-element K chunks of 128 bytes, chunk c of a tile at c x (rows x 128 bytes).
template <bool kExact>
struct SmemT {
  static constexpr uint32_t kTileB = kExact ? 2 * kTileBytes : kTileBytes;  // one page tile
  static constexpr uint32_t kQB = kExact ? 2 * 32 * 128 : 32 * 128;         // one query tile
  int32_t phys[kCtaPages];                  // offset 0, 4 KB: this CTA's block-table entries (when they fit)
  uint8_t qtile[kIssuers][kQB];             // A operands, one per MMA warp: index queries (SW128)
  uint8_t codes[kStages][kCodeBytes];       // 1024-aligned
  uint8_t tile[kBBufs][kTileB];             // B operand (SW128), 1024-aligned
  uint8_t scales[kStages][kScaleBytes];
  // scaled magnitudes per scale magnitude, 16 interleaved copies (entry e of copy c
  // at 8 (16 e + c) bytes): the 16 threads of an 8-byte wavefront read 16
  // different banks whatever their scales (the FP16 form needs no table)
  uint2 lut[kExact ? 2 : 128 * kLutCopies];
  float part[kDBufs][4][kGroups];           // per D buffer: the pool warps' quadrant maxima per index group
  int2 page_bc[kDBufs];                     // per D buffer: (request, block) of its page
  uint64_t full[kStages], empty[kStages];
  uint64_t bfull[kBBufs], bfree[kBBufs], dfull[kDBufs], dempty[kDBufs];
  uint32_t taddr;
  uint32_t fma_k[4];                        // 65536, 16: constants the compiler cannot fold
};
using Smem = SmemT<false>;
static_assert(offsetof(SmemT<false>, qtile) % 1024 == 0 && offsetof(SmemT<true>, qtile) % 1024 == 0, "swizzled A tile");
static_assert(offsetof(SmemT<false>, codes) % 1024 == 0 && offsetof(SmemT<false>, tile) % 1024 == 0 &&
                  offsetof(SmemT<true>, codes) % 1024 == 0 && offsetof(SmemT<true>, tile) % 1024 == 0,
              "swizzled tiles");
static_assert(offsetof(SmemT<false>, scales) % 16 == 0 && offsetof(SmemT<true>, scales) % 16 == 0,
              "bulk copies need 16-byte alignment");

// A scan over one shard of every request's blocks (indexer decode context
// parallelism): the shard's i-th block is logical block i * nshards + shard; a whole
// scan is shard 0 of 1. Its block scores go to column i of block_S.
__device__ __forceinline__ int shard_block(const SelectParams& p, int i) { return i * p.nshards + p.shard; }

struct PageCursor {
  int b;       // request
  int c;       // logical block within the request
};

// prefix[b] = the first page of request b in the concatenation of all requests'
// pages; prefix[B + 1] is a sentinel far beyond prefix[B] that stops the walk.
__device__ __forceinline__ void cursor_advance(PageCursor& pc, const long long* prefix) {
  ++pc.c;
  while (pc.c >= prefix[pc.b + 1] - prefix[pc.b]) {
    pc.c = 0;
    ++pc.b;
  }
}

// One page forward for a walker that caches its request's page count nbc. Past the
// last request (b = B) nbc becomes INT_MAX, so the walk never reads beyond prefix[B + 1].
__device__ __forceinline__ void cursor_step(PageCursor& pc, int& nbc, const long long* prefix, int B) {
  if (++pc.c >= nbc) {
    pc.c = 0;
    do ++pc.b;
    while (pc.b < B && prefix[pc.b + 1] == prefix[pc.b]);
    nbc = pc.b < B ? static_cast<int>(prefix[pc.b + 1] - prefix[pc.b]) : INT_MAX;
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

// Maximum over the visible columns n <= lim of 32 scores starting at column n0.
__device__ __forceinline__ float max32_masked(const uint32_t (&v)[32], int n0, int lim) {
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < 32; ++u) m = fmaxf(m, n0 + u <= lim ? __uint_as_float(v[u]) : -INFINITY);
  return m;
}

// Signed dequantisation of one code word (8 elements) to two words of E4M3 bytes,
// as dq8_signed, with its two shifts on the multiply-add pipe (k16 = 65536 and
// k4 = 16 come from shared memory, so the compiler cannot turn them back into
// shifts): the byte permutes and logic already fill the integer pipe.
__device__ __forceinline__ void dq8_signed_fma(uint32_t w, uint32_t L0, uint32_t L1, uint32_t k16, uint32_t k4,
                                               uint32_t& r0, uint32_t& r1) {
  const uint32_t sel = w & 0x77777777u;
  const uint32_t m0 = prmt(L0, L1, sel);
  const uint32_t m1 = prmt(L0, L1, __umulhi(sel, k16));  // sel >> 16
  const uint32_t u = w * k4;                              // w << 4
  const uint32_t s0 = prmt(w, u, 0x1504);  // byte k's msb = sign of nibble k, k = 0..3
  const uint32_t s1 = prmt(w, u, 0x3726);  // nibbles 4..7
  r0 = m0 ^ (s0 & 0x80808080u);
  r1 = m1 ^ (s1 & 0x80808080u);
}

// Dequantise 8 code words (4 groups of 16 elements; scale byte q of scw belongs to
// words 2q, 2q+1) to 64 signed E4M3 bytes and store them as 16-byte chunks
// c0..c0+3 of a K-major SW128 row (chunk c of row r sits at chunk c ^ (r & 7)).
// lut_t: this thread's copy of the table (entry e at lut_t + 128 e).
__device__ __forceinline__ void dequant_half_to_tile(uint32_t lut_t, const uint32_t* w, uint32_t scw, uint32_t k16,
                                                     uint32_t k4, uint32_t row_addr, int r7, int c0) {
  uint32_t out[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint2 L = lds_u2(lut_t + (((scw >> (8 * q)) & 0x7Fu) << 7));
#pragma unroll
    for (int h = 0; h < 2; ++h)
      dq8_signed_fma(w[2 * q + h], L.x, L.y, k16, k4, out[4 * q + 2 * h], out[4 * q + 2 * h + 1]);
  }
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    st_shared_v4(row_addr + (static_cast<uint32_t>((c0 + cc) ^ r7) << 4), out[4 * cc], out[4 * cc + 1],
                 out[4 * cc + 2], out[4 * cc + 3]);
}

// Write the request's index-query rows (4 x R <= 32, zero rows after them) into
// the A tile: row n = q_idx[row0 + n/4][group n%4], K-major with 128-byte swizzle.
__device__ __forceinline__ void write_qtile(uint8_t* qtile, const uint8_t* q_idx, int row0, int R, int t0,
                                            int nthreads) {
  for (int u = t0; u < 32 * 8; u += nthreads) {
    const int nrow = u >> 3, ch = u & 7;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (nrow < R * kGroups)
      v = *reinterpret_cast<const uint4*>(q_idx + (static_cast<long long>(row0) * kGroups + nrow) * kDim + ch * 16);
    *reinterpret_cast<uint4*>(qtile + nrow * 128 + ((ch ^ (nrow & 7)) << 4)) = v;
  }
}

// FP16 form of write_qtile (exact-score mode): row n's 128 E4M3 values widened to FP16
// (exact) as two 64-element K chunks, chunk c at c x 4 KB, 16-byte piece p of a chunk row at
// p ^ (n & 7).
__device__ __forceinline__ void write_qtile_f16(uint8_t* qtile, const uint8_t* q_idx, int row0, int R, int t0,
                                                int nthreads) {
  for (int u = t0; u < 32 * 16; u += nthreads) {
    const int nrow = u >> 4, piece = u & 15, c = piece >> 3, pc = piece & 7;
    uint4 h = make_uint4(0u, 0u, 0u, 0u);
    if (nrow < R * kGroups) {
      const uint2 v =
          *reinterpret_cast<const uint2*>(q_idx + (static_cast<long long>(row0) * kGroups + nrow) * kDim + piece * 8);
      asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h.x) : "r"(v.x & 0xFFFFu));
      asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h.y) : "r"(v.x >> 16));
      asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h.z) : "r"(v.y & 0xFFFFu));
      asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h.w) : "r"(v.y >> 16));
    }
    *reinterpret_cast<uint4*>(qtile + c * (32 * 128) + nrow * 128 + ((pc ^ (nrow & 7)) << 4)) = h;
  }
}

// Exact-score dequantisation of one 64-element K chunk of a row: 8 code words (word i =
// elements 8i .. 8i + 7, 16-element group i / 2 scaled by byte i / 2 of scw) to FP16, E2M1
// value times the E4M3 scale, both exact in FP16 (at most 6 significant bits, |x| <= 2688),
// stored as the chunk row's 8 16-byte pieces, piece i at i ^ (r & 7).
__device__ __forceinline__ void dequant_f16_chunk(const uint32_t* w, uint32_t scw, uint32_t chunk_row, int r7) {
  uint32_t s01, s23;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(s01) : "r"(scw & 0xFFFFu));
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(s23) : "r"(scw >> 16));
  const uint32_t sq[4] = {prmt(s01, 0u, 0x1010u), prmt(s01, 0u, 0x3232u), prmt(s23, 0u, 0x1010u),
                          prmt(s23, 0u, 0x3232u)};  // each group's scale in both halves
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t h[4];
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, a; cvt.rn.f16x2.e2m1x2 %1, b; cvt.rn.f16x2.e2m1x2 %2, c; cvt.rn.f16x2.e2m1x2 %3, d; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w[i]));
#pragma unroll
    for (int k = 0; k < 4; ++k) asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h[k]) : "r"(sq[i >> 1]));
    st_shared_v4(chunk_row + (static_cast<uint32_t>(i ^ r7) << 4), h[0], h[1], h[2], h[3]);
  }
}

}  // namespace

// MODE 0: fused select (block scores + top-k). MODE 1: write per-token scores
// (msa_index_scores) and stop. MODE 2: MODE 0 with exact index scores (FP16 tiles and
// MMAs: the keys' E2M1 x scale values are not re-rounded to E4M3).
template <int MODE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    select_kernel(const __grid_constant__ CUtensorMap ki_map, const SelectParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem_al = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // TMA/UMMA tiles need 1 KB
  constexpr bool kExact = MODE == 2;
  constexpr bool kPool = MODE != 1;  // block max pool + top-k (MODE 0, 2) vs per-token scores (MODE 1)
  using Sm = SmemT<kExact>;
  Sm& sm = *reinterpret_cast<Sm*>(smem_al);
  // page prefix over requests [B + 2]: counts first, then scanned in place. Only
  // requests that passed the checks below own pages, so the geometry of a page's
  // request is read from the (validated) inputs where it is needed.
  long long* prefix = reinterpret_cast<long long*>(smem_al + sizeof(Sm));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.num_reqs;

  if (kPool) pdl_launch_dependents();

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
    prefix[b] = pages > p.shard ? (pages - 1 - p.shard) / p.nshards + 1 : 0;  // this shard's blocks
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix over requests: each lane scans a contiguous chunk
    const int per = (B + 31) / 32;
    const int b0 = min(lane * per, B), b1 = min(b0 + per, B);
    long long part = 0;
    for (int b = b0; b < b1; ++b) part += prefix[b];
    long long incl = part;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    long long acc = incl - part;
    for (int b = b0; b < b1; ++b) {
      const long long cnt = prefix[b];
      prefix[b] = acc;
      acc += cnt;
    }
    if (lane == 31) {
      prefix[B] = incl;
      prefix[B + 1] = incl + (1LL << 30);  // sentinel (a request of 2^30 pages: fits an int)
    }
  }
  __syncthreads();
  const long long total = prefix[B];
  const long long G = gridDim.x;
  const long long p0 = total * blockIdx.x / G, p1 = total * (blockIdx.x + 1) / G;
  const int n = static_cast<int>(p1 - p0);

  if (n <= 0) return;

  // ---- setup: table, barriers, tensor memory
  if (!kExact)
    for (int u = tid; u < 128 * kLutCopies; u += kThreads) sm.lut[u] = lut_magnitudes(static_cast<uint32_t>(u / kLutCopies));
  if (tid == 0) {
    sm.fma_k[0] = 65536u;
    sm.fma_k[1] = 16u;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 4);  // the 4 warps of the page's dequant group
    }
    for (int j = 0; j < kBBufs; ++j) {
      mbar_init(smem_u32(&sm.bfull[j]), 4);
      mbar_init(smem_u32(&sm.bfree[j]), 1);
    }
    for (int k = 0; k < kDBufs; ++k) {
      mbar_init(smem_u32(&sm.dfull[k]), 1);
      mbar_init(smem_u32(&sm.dempty[k]), 4);  // the 4 warps (lane quadrants) of the pooling group
    }
    mbar_fence_init();
  }
  // this CTA's block-table entries, so no page waits on a dependent global load
  const bool staged = n <= kCtaPages;
  if (staged) {
    for (int i = tid; i < n; i += kThreads) {
      const PageCursor pc = cursor_at(p0 + i, prefix, B);
      sm.phys[i] = p.block_table[static_cast<long long>(pc.b) * p.max_pages + shard_block(p, pc.c)];
    }
  }
  // the first request's index queries
  const int first_req = cursor_at(p0, prefix, B).b;
  for (int m = 0; m < kIssuers; ++m)
    if (kExact)
      write_qtile_f16(sm.qtile[m], p.q_idx, p.q_indptr[first_req], p.q_indptr[first_req + 1] - p.q_indptr[first_req],
                      tid, kThreads);
    else
      write_qtile(sm.qtile[m], p.q_idx, p.q_indptr[first_req], p.q_indptr[first_req + 1] - p.q_indptr[first_req], tid,
                  kThreads);
  fence_proxy_async_smem();
  if (warp == kIssueWarp) tmem_alloc(smem_u32(&sm.taddr), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.taddr;
  bool alive = true;

  if (warp == kLoadWarp || warp == kLoadWarp2) {
    // ================= load warps: TMA producers (one lane each), warp L takes pages L, L + 2, ...
    const int L = warp == kLoadWarp ? 0 : 1;
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ki_map)) : "memory");
      PageCursor ld = cursor_at(p0 + (L < n ? L : 0), prefix, B);
      for (int i = L; i < n; i += kLoaders) {
        const int s = i % kStages;

        if (i >= kStages) {  // the dequant group has released this stage's previous page
          alive = wait_bar(smem_u32(&sm.empty[s]), ((i / kStages) - 1) & 1, p.flags);
          if (!alive) break;
        }
        const int phys =
            staged ? sm.phys[i] : p.block_table[static_cast<long long>(ld.b) * p.max_pages + shard_block(p, ld.c)];
        const bool bad = phys < 0 || phys >= p.num_pages;
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
        cursor_advance(ld, prefix);
        cursor_advance(ld, prefix);
      }
      if (!alive) {
        // drain: copies already issued complete on their own barriers
        for (int i = L; i < n; i += kLoaders) {
          const int s = i % kStages;
          if (!mbar_wait(smem_u32(&sm.full[s]), (i / kStages) & 1, p.flags)) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == kIssueWarp || warp == kIssueWarp2) {
    // ================= MMA warps: warp m issues pages m, m + 2, ... (lane 0) and keeps
    // its own query tile (all lanes)
    const int m = warp == kIssueWarp ? 0 : 1;
    PageCursor mm = cursor_at(p0 + (m < n ? m : 0), prefix, B);
    int nbc = static_cast<int>(prefix[mm.b + 1] - prefix[mm.b]);  // pages of the cursor's request
    int qtile_req = first_req;
    // K step kk of an operand starts 32 bytes further: +2 in the start-address field
    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sm.qtile[m]));
    const uint32_t tile0 = smem_u32(sm.tile[0]);
    const uint32_t idesc = kExact ? idesc_f16_f32(32, kBlock, false) : idesc_e4m3_f32(32, kBlock, false);
    for (int i = m; i < n; i += kIssuers) {
      const int j = i % kBBufs, k = i % kDBufs;
      if (mm.b != qtile_req) {
        // new request: once this warp's earlier MMAs have finished reading its tile, rewrite it
        const int ip = i - kIssuers;
        if (ip >= 0) alive = wait_bar(smem_u32(&sm.dfull[ip % kDBufs]), (ip / kDBufs) & 1, p.flags);
        if (!__all_sync(0xFFFFFFFFu, alive)) {
          alive = false;
          break;
        }
        tc_fence_after();
        if (kExact)
          write_qtile_f16(sm.qtile[m], p.q_idx, p.q_indptr[mm.b], p.q_indptr[mm.b + 1] - p.q_indptr[mm.b], lane, 32);
        else
          write_qtile(sm.qtile[m], p.q_idx, p.q_indptr[mm.b], p.q_indptr[mm.b + 1] - p.q_indptr[mm.b], lane, 32);
        fence_proxy_async_smem();
        __syncwarp();
        qtile_req = mm.b;
      }
      if (lane == 0) {
        alive = wait_bar(smem_u32(&sm.bfull[j]), (i / kBBufs) & 1, p.flags);
        if (alive && i >= kDBufs) alive = wait_bar(smem_u32(&sm.dempty[k]), ((i / kDBufs) - 1) & 1, p.flags);
        if (alive) {
          tc_fence_after();
          const uint64_t bdesc = sdesc_kmajor_sw128(tile0 + j * Sm::kTileB);
          const uint32_t d = tbase + k * kDCols;
          if (kExact) {
            // K step kk (16 FP16 elements, 32 bytes): chunk kk / 4 (4 KB of A, 16 KB of B
            // further), +32 bytes per step inside it (start-address field in 16-byte units)
#pragma unroll
            for (int kk = 0; kk < kDim / 16; ++kk)
              mma_f16_ws(d, adesc + 256 * (kk >> 2) + 2 * (kk & 3), bdesc + 1024 * (kk >> 2) + 2 * (kk & 3), idesc,
                         kk > 0);
          } else {
#pragma unroll
            for (int kk = 0; kk < kDim / 32; ++kk) mma_f8_ws(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0);
          }
          mma_commit(smem_u32(&sm.dfull[k]));
          mma_commit(smem_u32(&sm.bfree[j]));
        }
      }
      for (int u = 0; u < kIssuers; ++u) {
        cursor_step(mm, nbc, prefix, B);
      }
      alive = __shfl_sync(0xFFFFFFFFu, alive ? 1 : 0, 0) != 0;  // lane 0 waited and issued
      if (!alive) break;
    }
    __syncwarp();
  } else if (warp < kDqWarp0) {
    // ================= pool warps: set P takes pages i = P, P + kPoolSets, ... from D
    // buffer k = i % kDBufs. The warp's lane quadrant q = warp % 4 holds the page's tokens
    // 32q .. 32q + 31 (lane m = query column rq * 4 + g). Each warp leaves its quadrant's
    // group maxima in slot k; every kPoolBatch of its pages the set's four warps meet at
    // the set's named barrier and its quadrant-0 warp combines the batch (lane = page *
    // 4 + group). A slot is rewritten only after the set's next barrier. All four run the
    // same number of steps and barriers, timeouts included, so the barrier always completes.
    static_assert(kPoolBatch * kGroups <= 32 && kDBufs >= 2 * kPoolBatch * kPoolSets, "pool slot reuse");
    const int set = (warp - kPoolWarp0) >> 2, quad = warp & 3, rq = lane >> 2, g = lane & 3;
    const uint32_t d_lane = tbase + (static_cast<uint32_t>(32 * quad) << 16);
    PageCursor pc = cursor_at(p0 + (set < n ? set : 0), prefix, B);
    int nbc = static_cast<int>(prefix[pc.b + 1] - prefix[pc.b]);  // pages of the cursor's request
    // the page's request geometry, reloaded only when the request changes
    int cur_b = -1, N = 0, row0 = 0, R = 0;
    int it = 0;
    for (int ip = set; ip < n; ip += kPoolSets, ++it) {
      const int k = ip % kDBufs;
      if (pc.b != cur_b) {
        cur_b = pc.b;
        N = p.context_lens[cur_b];
        row0 = p.q_indptr[cur_b];
        R = p.q_indptr[cur_b + 1] - row0;
      }
      if (alive) alive = wait_bar(smem_u32(&sm.dfull[k]), (ip / kDBufs) & 1, p.flags);
      alive = __all_sync(0xFFFFFFFFu, alive) != 0;
      tc_fence_after();
      const int b = pc.b, c = shard_block(p, pc.c);  // logical block of the request
      const int t0 = c * kBlock + 32 * quad;         // this quadrant's first token
      const int lim = N - R + rq - t0;        // column u is visible to this row iff u <= lim
      const uint32_t d = d_lane + static_cast<uint32_t>(k) * kDCols;
      float m = -INFINITY;
      if (alive) {
        if (kPool && N - R - t0 >= 31) {
          // every row sees the quadrant's 32 tokens (a warp-uniform test): the load's own
          // max reduction gives each row's maximum
          const float mq = tmem_ld32_max(d);
          tc_wait_ld();
          if (rq < R) m = mq;
        } else {
          uint32_t v[32];
          tmem_ld32(d, v);
          tc_wait_ld();
          if (kPool) {
            if (rq < R) m = max32_masked(v, 0, lim);
          } else if (rq < R) {
            const int phys = staged ? sm.phys[ip] : p.block_table[static_cast<long long>(b) * p.max_pages + c];
            const bool page_bad = phys < 0 || phys >= p.num_pages;
            float* out = p.token_scores + (static_cast<long long>(row0 + rq) * kGroups + g) * p.score_stride + t0;
#pragma unroll
            for (int u = 0; u < 32; ++u)
              if (t0 + u < N) out[u] = !page_bad && u <= lim ? __uint_as_float(v[u]) : -INFINITY;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.dempty[k]));
      if (kPool) {
        // the group's maximum over its rows: lanes with equal lane % 4
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
        if (lane < kGroups) sm.part[k][quad][lane] = m;
        if (quad == 0 && lane == 0) sm.page_bc[k] = make_int2(b, pc.c);  // block_S column: the shard's index
        if ((it + 1) % kPoolBatch == 0 || ip + kPoolSets >= n) {
          named_bar_sync(1 + set, 128);
          const int pg = ip - kPoolSets * (it % kPoolBatch) + kPoolSets * (lane >> 2);
          if (quad == 0 && lane < kPoolBatch * kGroups && pg <= ip) {
            const int kk = pg % kDBufs;
            const int2 bc = sm.page_bc[kk];
            // a page whose table entry is out of range scores -inf (its codes were never loaded)
            const int phys =
                staged ? sm.phys[pg] : p.block_table[static_cast<long long>(bc.x) * p.max_pages + shard_block(p, bc.y)];
            const float mm = phys < 0 || phys >= p.num_pages
                                 ? -INFINITY
                                 : fmaxf(fmax3(sm.part[kk][0][g], sm.part[kk][1][g], sm.part[kk][2][g]),
                                         sm.part[kk][3][g]);
            p.block_S[(static_cast<long long>(bc.x) * kGroups + g) * p.s_stride + bc.y] = alive ? mm : -INFINITY;
          }
        }
      }
      for (int u = 0; u < kPoolSets; ++u) {
        cursor_step(pc, nbc, prefix, B);
      }
    }
  } else {
    // ================= dequant warps: page i -> page tile i % kBBufs, by group i % kDqGroups
    const int dw = warp - kDqWarp0, grp = dw >> 2;
    const int r = (dw & 3) * 32 + lane;  // token slot within the page = row of the page tile
    const int r7 = r & 7, sw = (r >> 1) & 3;
    const uint32_t row_off = static_cast<uint32_t>(r >> 3) * 1024u + static_cast<uint32_t>(r7) * 128u;
    const uint32_t tile0 = smem_u32(sm.tile[0]);
    const uint32_t lut_t = smem_u32(sm.lut) + static_cast<uint32_t>(lane % kLutCopies) * 8u;
    const uint32_t k16 = sm.fma_k[0], k4 = sm.fma_k[1];
    for (int i = grp; i < n; i += kDqGroups) {
      const int s = i % kStages, j = i % kBBufs;
      uint32_t w[16];
      alive = wait_bar(smem_u32(&sm.full[s]), (i / kStages) & 1, p.flags);
      if (!alive) break;
      // this thread's row: 64 code bytes (swizzled 16-byte chunks) + 8 scale bytes
      const uint8_t* row = sm.codes[s] + r * 64;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((cc ^ sw) << 4));
        w[4 * cc] = v.x;
        w[4 * cc + 1] = v.y;
        w[4 * cc + 2] = v.z;
        w[4 * cc + 3] = v.w;
      }
      const uint2 sc = *reinterpret_cast<const uint2*>(sm.scales[s] + r * 8);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
      if (i >= kBBufs) {  // the MMAs that read this tile last time have finished
        alive = wait_bar(smem_u32(&sm.bfree[j]), ((i / kBBufs) - 1) & 1, p.flags);
        if (!alive) break;
        tc_fence_after();
      }
      const uint32_t row_addr = tile0 + j * Sm::kTileB + row_off;
      if (kExact) {
        dequant_f16_chunk(w, sc.x, row_addr, r7);                   // elements 0..63: K chunk 0
        dequant_f16_chunk(w + 8, sc.y, row_addr + kTileBytes, r7);  // 64..127: chunk 1, 16 KB on
      } else {
        dequant_half_to_tile(lut_t, w, sc.x, k16, k4, row_addr, r7, 0);
        dequant_half_to_tile(lut_t, w + 8, sc.y, k16, k4, row_addr, r7, 4);
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the MMA (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.bfull[j]));
    }
  }

  // ---- teardown
  tc_fence_before();
  const bool all_alive = __syncthreads_and(alive ? 1 : 0) != 0;
  if (warp == kIssueWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  (void)all_alive;
}

// The top-k of one group by its four warps q = 0..3 for requests of at most 32 * 4 * 8 + 1
// blocks, straight from the scores in global memory (read past L1): lane l of warp q holds
// candidates 256 q + 8 l .. + 7 in registers. T = the largest lane maximum with at least 15
// lane maxima at or above it, found by rank counting (no sort); the survivors (15 to 19 on
// the synthetic workloads) are ranked by counting, and the 16 ids ordered the same way. Same
// result as warp_topk; more than 32 survivors fall back to the exact insertion merge.
constexpr int kDirectMax = 32 * 4 * 8;  // candidates (blocks but the recent one)
__device__ __forceinline__ void group_topk_direct(const float* Sg, int nb, int32_t* ids_out, int q, int bar_id,
                                                  uint64_t* lm, uint64_t* tmax, uint64_t* surv, int* cnt,
                                                  int32_t* sel) {
  const int lane = threadIdx.x & 31;
  constexpr int L = kTopK - 1;
  const int nc = nb - 1;
  const int c0 = q * 256 + lane * 8;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 va = c0 < nc ? __ldcg(reinterpret_cast<const float4*>(Sg + c0)) : z;
  const float4 vb = c0 + 4 < nc ? __ldcg(reinterpret_cast<const float4*>(Sg + c0 + 4)) : z;
  const float v[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
  uint64_t k[8];
  uint64_t mx = 0ull;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    k[t] = c0 + t < nc ? topk_key(v[t], c0 + t) : 0ull;
    mx = k[t] > mx ? k[t] : mx;
  }
  lm[q * 32 + lane] = mx;
  if (q == 0 && lane == 0) *cnt = 0;
  named_bar_sync(bar_id, 128);
  int ge = 0;
#pragma unroll 8
  for (int j = 0; j < 128; ++j) ge += lm[j] >= mx ? 1 : 0;
  uint64_t T = ge >= L ? mx : 0ull;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t o = shfl_xor_u64(T, off);
    T = o > T ? o : T;
  }
  if (lane == 0) tmax[q] = T;
  named_bar_sync(bar_id, 128);
  T = tmax[0];
#pragma unroll
  for (int w = 1; w < 4; ++w) T = tmax[w] > T ? tmax[w] : T;
  // survivors: one atomic per warp reserves the warp's slots
  int mine = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) mine += (c0 + t < nc && k[t] >= T) ? 1 : 0;
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  int base = 0;
  if (lane == 31) base = atomicAdd(cnt, incl);
  base = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - mine;
#pragma unroll
  for (int t = 0; t < 8; ++t)
    if (c0 + t < nc && k[t] >= T) {
      if (base < 64) surv[base] = k[t];
      ++base;
    }
  named_bar_sync(bar_id, 128);
  if (q != 0) return;
  const int count = *cnt;
  if (count > 32) {
    topk_by_insertion<true>(Sg, nc, sel);
  } else {
    const uint64_t key = lane < count ? surv[lane] : 0ull;
    int rank = 0;
    for (int j = 0; j < count; ++j) rank += surv[j] > key ? 1 : 0;
    if (lane < count && rank < L) sel[rank] = topk_id(key);
    __syncwarp();
  }
  // the 15 winners plus the recent block, ascending
  if (lane == L) sel[L] = nb - 1;
  __syncwarp();
  if (lane < kTopK) {
    const int my_id = sel[lane];
    int rank = 0;
#pragma unroll
    for (int j = 0; j < kTopK; ++j) rank += sel[j] < my_id ? 1 : 0;
    ids_out[rank] = my_id;
  }
}

// Step 3 of the selection, after the scan: one CTA per request, four warps per group.
// A kernel of its own so it runs on SMs the scan has left; chained to the scan by
// programmatic dependent launch, it reads the request geometry before waiting.
// [vLLM-zh §How; MSA-fig §1 TopK] group g keeps its recent block and the 15 best of the
// others (score, then lower id); every block when there are at most 16. Up to 1,025 blocks
// the group's four warps rank by a threshold from their lane maxima (group_topk_direct);
// longer rows are split in quarters, one per warp (quad_best15), and the group's warp 0
// merges the quarters. Both read the scores the scan left in L2. (Measured on GB300 in the
// decode chain: the direct form ~2 us faster at 1,023 candidates, the quarters ~5 us faster
// on the ragged batch whose longest request has 2,047.)
constexpr int kTopkThreads = 128 * kGroups;
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const SelectParams p) {
  __shared__ uint64_t lists[kGroups][4 * kTopK];
  __shared__ uint64_t qsurv[kGroups][4 * 64];
  __shared__ uint64_t surv[kGroups][64];
  __shared__ uint64_t lm[kGroups][128];
  __shared__ uint64_t tmax[kGroups][4];
  __shared__ int cnt[kGroups];
  __shared__ int32_t sel[kGroups][kTopK];
  pdl_launch_dependents();
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp >> 2, q = warp & 3;
  // the request's geometry is an input (not written by the scan): read it before waiting
  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows;
  const int nbb = ok && R > 0 ? (N + kBlock - 1) / kBlock : 0;
  pdl_wait_primary();  // the block scores come from the scan kernel
  int32_t* ids = p.block_ids + (static_cast<long long>(b) * kGroups + g) * kTopK;
  const float* S = p.block_S + (static_cast<long long>(b) * kGroups + g) * p.s_stride;
  if (nbb <= kTopK) {  // every block (none: an empty selection)
    if (q == 0 && lane < kTopK) ids[lane] = lane < nbb ? lane : -1;
  } else if (nbb - 1 <= kDirectMax) {
    group_topk_direct(S, nbb, ids, q, 1 + g, lm[g], tmax[g], surv[g], &cnt[g], sel[g]);
  } else {
    const uint64_t best = quad_best15(S, 0, nbb - 1, q, 1 + g, lists[g], qsurv[g]);
    if (q == 0) write_selection(best, nbb, ids);
  }
  if (p.block_scores_out != nullptr) {
    float* sout = p.block_scores_out + (static_cast<long long>(b) * kGroups + g) * p.max_pages;
    for (int c = q * 32 + lane; c < p.max_pages; c += 128) sout[c] = c < nbb ? __ldcg(S + c) : -INFINITY;
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

// Exposes the kernels' dequantisers for checking: path 0 = dq8_signed, the
// attention kernel's form (its K operand, and V before the exact E4M3 -> FP16
// widening); path 1 = dq8_signed_fma, the index scan's form.
__global__ void dequant_rows_kernel(const uint8_t* codes, const uint8_t* scales, long long nrows, uint8_t* out,
                                    int path) {
  __shared__ uint2 lut[128];
  __shared__ uint32_t fma_k[2];
  for (int s = threadIdx.x; s < 128; s += blockDim.x) lut[s] = lut_magnitudes(static_cast<uint32_t>(s));
  if (threadIdx.x == 0) {
    fma_k[0] = 65536u;
    fma_k[1] = 16u;
  }
  __syncthreads();
  const uint32_t k16 = fma_k[0], k4 = fma_k[1];
  const long long nwords = nrows * 16;
  for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < nwords;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = u >> 4;
    const int wi = static_cast<int>(u & 15);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + row * 64 + wi * 4);
    const uint2 L = lut[scales[row * 8 + wi / 2] & 0x7Fu];
    uint32_t r0, r1;
    if (path == 0) dq8_signed(w, L.x, L.y, r0, r1);
    else dq8_signed_fma(w, L.x, L.y, k16, k4, r0, r1);
    *reinterpret_cast<uint32_t*>(out + row * 128 + wi * 8) = r0;
    *reinterpret_cast<uint32_t*>(out + row * 128 + wi * 8 + 4) = r1;
  }
}

size_t select_smem_bytes(int num_reqs, int mode) {
  const size_t need = (mode == 2 ? sizeof(SmemT<true>) : sizeof(SmemT<false>)) + sizeof(long long) * (num_reqs + 2) + 1024;
  // more than half an SM's shared memory, so one CTA holds the SM's 512 tensor-memory columns
  return need > 120 * 1024 ? need : 120 * 1024;
}

cudaError_t launch_select(const CUtensorMap& ki_map, const SelectParams& prm, int mode, int sm_count,
                          cudaStream_t st) {
  const size_t smem = select_smem_bytes(prm.num_reqs, mode);
  const int grid = kCtasPerSm * sm_count;
  cudaError_t e;
  if (mode == 0) {
    e = cudaFuncSetAttribute(select_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    select_kernel<0><<<grid, kThreads, smem, st>>>(ki_map, prm);
  } else if (mode == 2) {
    e = cudaFuncSetAttribute(select_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    select_kernel<2><<<grid, kThreads, smem, st>>>(ki_map, prm);
  } else {
    e = cudaFuncSetAttribute(select_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    select_kernel<1><<<grid, kThreads, smem, st>>>(ki_map, prm);
  }
  return cudaGetLastError();
}

cudaError_t launch_topk(const SelectParams& prm, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_reqs, 1, 1);
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, topk_kernel, prm);
  if (e != cudaSuccess) return e;
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
