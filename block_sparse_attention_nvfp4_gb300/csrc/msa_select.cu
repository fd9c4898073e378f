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
// this kernel is a stream over the cache's pages at HBM speed. 2 CTAs per SM
// (256 TMEM columns each), the grid taking equal contiguous ranges of all
// requests' pages; one CTA has four roles:
//   * load warp: one lane streams pages into a ring of shared-memory stages with
//     TMA (codes: 2-D tensor copy with 64-byte swizzle, so each thread reads its
//     64-byte row without bank conflicts; scales: 1-D bulk copy);
//   * 8 dequant warps in two groups that take alternate pages (thread = token):
//     dequantise the token's 128 elements to E4M3 (byte-permute table lookups for
//     magnitudes and signs) and write them as row `token` of a page tile in
//     shared memory (the MMA's B operand, K-major, 128-byte swizzle);
//   * MMA warp: one lane issues, per page, D = Q x P^T with Q the request's
//     4 x R index-query rows (A operand, M = 128 of which rows >= 32 are never
//     read back) and P the dequantised page (N = 128 tokens, K = 128), FP32
//     accumulation in tensor memory (products of two E4M3 values are exact; only
//     the FP32 sums round); the warp rewrites Q when the request changes;
//   * 2 epilogue warps taking alternate pages (D buffer e, TMEM lanes
//     32e..32e+31 = the 32 query columns rq*4+g): read the page's 32 x 128
//     scores, mask, take each row's maximum over the tokens and the group's
//     maximum over its rows with shuffles, and write the block score.
// Laying the scores out with the query columns on TMEM lanes puts a whole page's
// max pool in one warp (no cross-warp combine); measured on GB300, the pool was
// the costliest step when the 128 tokens were spread over four warps' lanes.
// The dequant warps never wait for an MMA result, only for a free page tile, so
// the MMA round trip hides behind the next pages' dequantisation.
//
// The top-k runs in a second kernel (one CTA per request, one warp per group),
// launched with programmatic dependent launch so its CTAs are resident and have
// read the request geometry when the scan's last pages finish; it waits on the
// scan's completion (griddepcontrol.wait), not on any flag another CTA writes.
#include <climits>
#include <cstddef>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

// Warp roles. Warp w runs on SM sub-partition w % 4 and reads TMEM lanes
// 32 (w % 4) .. + 31. D buffer e holds the 32 query columns in lanes 32e .. 32e + 31
// (its A tile starts 32 rows earlier for e = 1), so epilogue warps 0 and 1 read
// buffers 0 and 1 (pages i with i % 2 = e), and every sub-partition runs one warp of
// each dequant group plus one of: epilogue, epilogue, load, MMA (measured on GB300:
// with 3 of the 8 dequant warps on one sub-partition, those lagged the group).
constexpr int kLoadWarp = 2;   // TMA producer
constexpr int kIssueWarp = 3;  // MMA issue, query tile, TMEM allocation
constexpr int kDqWarp0 = 4;    // dequant warps 4..11: group (w - 4) / 4, one warp per sub-partition
constexpr int kDqGroups = 2;   // page i is dequantised by group i % kDqGroups
constexpr int kDqWarps = 4 * kDqGroups;
constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;
constexpr int kCtasPerSm = 2;
constexpr int kStages = 4, kBBufs = 3, kDBufs = 2;
constexpr uint32_t kCodeBytes = kBlock * 64;    // one page of index-key codes
constexpr uint32_t kScaleBytes = kBlock * 8;    // its scales
constexpr uint32_t kTileBytes = kBlock * kDim;  // one dequantised page (E4M3)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kDCols = kBlock;             // D buffer: 128 FP32 columns (tokens)
constexpr int kCtaPages = 1024;                 // block-table entries staged per CTA
constexpr int kLutCopies = 16;                  // one per thread of a 16-thread (8-byte) wavefront
static_assert(kDBufs * kDCols <= kTmemCols, "TMEM buffers exceed the allocation");

struct Smem {
  int32_t phys[kCtaPages];                  // offset 0, 4 KB: this CTA's block-table entries (when they fit)
  // A operand: the request's index queries, 32 rows of 128 bytes. The MMA reads a
  // 128-row tile starting at qtile (D buffer 0: queries in rows 0..31) or 32 rows
  // before it (D buffer 1: rows 32..63); the other rows are the staged block table
  // and the table, both written before the first MMA; their D lanes are never read.
  uint8_t qtile[32 * 128];                  // offset 4 KB
  // scaled magnitudes per scale magnitude, 16 interleaved copies (entry e of copy c
  // at 8 (16 e + c) bytes): the 16 threads of an 8-byte wavefront read 16
  // different banks whatever their scales
  uint2 lut[128 * kLutCopies];              // 16 KB
  uint8_t codes[kStages][kCodeBytes];       // offset 16 KB, 1024-aligned
  uint8_t tile[kBBufs][kTileBytes];         // B operand (SW128), 1024-aligned
  uint8_t scales[kStages][kScaleBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t bfull[kBBufs], bfree[kBBufs], dfull[kDBufs], dempty[kDBufs];
  uint32_t taddr;
  uint32_t fma_k[4];                        // 65536, 16: constants the compiler cannot fold
};
static_assert(sizeof(int32_t) * kCtaPages == 32 * 128 && sizeof(uint2) * 128 * kLutCopies >= 96 * 128,
              "both A tiles lie in the staged block table, the queries and the table");
static_assert(offsetof(Smem, codes) % 1024 == 0 && offsetof(Smem, tile) % 1024 == 0, "swizzled tiles");
static_assert(offsetof(Smem, scales) % 16 == 0, "bulk copies need 16-byte alignment");

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

// Maximum of 32 scores (one tcgen05 load): 4 independent chains.
__device__ __forceinline__ float max32(const uint32_t (&v)[32]) {
  float acc[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float a = fmax3(__uint_as_float(v[u]), __uint_as_float(v[4 + u]), __uint_as_float(v[8 + u]));
    a = fmax3(a, __uint_as_float(v[12 + u]), __uint_as_float(v[16 + u]));
    a = fmax3(a, __uint_as_float(v[20 + u]), __uint_as_float(v[24 + u]));
    acc[u] = fmaxf(a, __uint_as_float(v[28 + u]));
  }
  return fmaxf(fmax3(acc[0], acc[1], acc[2]), acc[3]);
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
  if (warp == 0) {  // exclusive prefix over requests: each lane scans a contiguous chunk
    const int per = (B + 31) / 32;
    const int b0 = min(lane * per, B), b1 = min(b0 + per, B);
    long long part = 0;
    for (int b = b0; b < b1; ++b) part += nb[b];
    long long incl = part;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    long long acc = incl - part;
    for (int b = b0; b < b1; ++b) {
      prefix[b] = acc;
      acc += nb[b];
    }
    if (lane == 31) prefix[B] = incl;
  }
  __syncthreads();
  const long long total = prefix[B];
  const long long G = gridDim.x;
  const long long p0 = total * blockIdx.x / G, p1 = total * (blockIdx.x + 1) / G;
  const int n = static_cast<int>(p1 - p0);

  if (n <= 0) return;

  // ---- setup: table, barriers, tensor memory
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
      mbar_init(smem_u32(&sm.dempty[k]), 1);
    }
    mbar_fence_init();
  }
  // this CTA's block-table entries, so no page waits on a dependent global load
  const bool staged = n <= kCtaPages;
  if (staged) {
    for (int i = tid; i < n; i += kThreads) {
      const PageCursor pc = cursor_at(p0 + i, prefix, B);
      sm.phys[i] = p.block_table[static_cast<long long>(pc.b) * p.max_pages + pc.c];
    }
  }
  // the first request's index queries
  const int first_req = cursor_at(p0, prefix, B).b;
  write_qtile(sm.qtile, p.q_idx, row0_s[first_req], rows_s[first_req], tid, kThreads);
  fence_proxy_async_smem();
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

        if (i >= kStages) {  // the dequant group has released this stage's previous page
          alive = wait_bar(smem_u32(&sm.empty[s]), ((i / kStages) - 1) & 1, p.flags);
          if (!alive) break;
        }
        const int phys = staged ? sm.phys[i] : p.block_table[static_cast<long long>(ld.b) * p.max_pages + ld.c];
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
    // K step kk of an operand starts 32 bytes further: +2 in the start-address field
    const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(sm.qtile));
    const uint64_t adesc1 = sdesc_kmajor_sw128(smem_u32(sm.qtile) - 32 * 128);
    const uint32_t tile0 = smem_u32(sm.tile[0]);
    const uint32_t idesc = idesc_e4m3_f32(128, kBlock, false);
    for (int i = 0; i < n; ++i) {
      const int j = i % kBBufs, k = i % kDBufs;
      if (mm.b != qtile_req) {
        // new request: once every earlier MMA has finished reading the tile, rewrite it
        if (i >= 1) alive = wait_bar(smem_u32(&sm.dfull[(i - 1) % kDBufs]), ((i - 1) / kDBufs) & 1, p.flags);
        if (!__all_sync(0xFFFFFFFFu, alive)) {
          alive = false;
          break;
        }
        tc_fence_after();
        write_qtile(sm.qtile, p.q_idx, row0_s[mm.b], rows_s[mm.b], lane, 32);
        fence_proxy_async_smem();
        __syncwarp();
        qtile_req = mm.b;
      }
      if (lane == 0) {
        alive = wait_bar(smem_u32(&sm.bfull[j]), (i / kBBufs) & 1, p.flags);
        if (alive && i >= kDBufs) alive = wait_bar(smem_u32(&sm.dempty[k]), ((i / kDBufs) - 1) & 1, p.flags);
        if (alive) {
          tc_fence_after();
          const uint64_t bdesc = sdesc_kmajor_sw128(tile0 + j * kTileBytes);
          const uint32_t d = tbase + k * kDCols;
          const uint64_t adesc = k == 0 ? adesc0 : adesc1;
#pragma unroll
          for (int kk = 0; kk < kDim / 32; ++kk) mma_f8_ss(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0);
          mma_commit(smem_u32(&sm.dfull[k]));
          mma_commit(smem_u32(&sm.bfree[j]));
        }
      }
      cursor_advance(mm, nb);
      if (!__all_sync(0xFFFFFFFFu, alive)) {
        alive = false;
        break;
      }
    }
    __syncwarp();
  } else if (warp >= kDqWarp0) {
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
      if (i >= kBBufs) {  // the MMAs that read this tile last time have finished
        alive = wait_bar(smem_u32(&sm.bfree[j]), ((i / kBBufs) - 1) & 1, p.flags);
        if (!alive) break;
        tc_fence_after();
      }
      const uint32_t row_addr = tile0 + j * kTileBytes + row_off;
      dequant_half_to_tile(lut_t, w, sc.x, k16, k4, row_addr, r7, 0);
      dequant_half_to_tile(lut_t, w + 8, sc.y, k16, k4, row_addr, r7, 4);
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the MMA (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.bfull[j]));
    }
  } else {
    // ================= epilogue warps 0 and 1: pages i = e, e + 2, ... (D buffer e);
    // lane m = query column rq*4 + g of D (TMEM lane 32e + m)
    const int e = warp, rq = lane >> 2, g = lane & 3;
    static_assert(kDBufs == 2, "one D buffer per epilogue warp");
    PageCursor cur = cursor_at(p0 + (e < n ? e : 0), prefix, B);
    for (int i = e; i < n; i += 2) {
      const int k = e;
      alive = wait_bar(smem_u32(&sm.dfull[k]), (i / kDBufs) & 1, p.flags);
      if (!__all_sync(0xFFFFFFFFu, alive)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const int b = cur.b, c = cur.c;
      const int phys = staged ? sm.phys[i] : p.block_table[static_cast<long long>(b) * p.max_pages + c];
      const bool page_bad = phys < 0 || phys >= p.num_pages;
      const int N = ctx_s[b], R = rows_s[b];
      const bool valid = rq < R && !page_bad;
      const int t0 = c * kBlock;
      const int lim = N - R + rq - t0;  // column n of this row is visible iff n <= lim
      const uint32_t d = tbase + (static_cast<uint32_t>(32 * e) << 16) + k * kDCols;
      float m = -INFINITY;
#pragma unroll
      for (int q = 0; q < kBlock / 32; ++q) {
        uint32_t v[32];
        tmem_ld32(d + 32 * q, v);
        tc_wait_ld();
        if (MODE == 0) {
          if (valid) m = fmaxf(m, lim >= kBlock - 1 ? max32(v) : max32_masked(v, 32 * q, lim));
        } else if (rq < R) {
          float* out = p.token_scores + (static_cast<long long>(row0_s[b] + rq) * kGroups + g) * p.score_stride + t0;
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int nn = 32 * q + u;
            if (t0 + nn < N) out[nn] = valid && nn <= lim ? __uint_as_float(v[u]) : -INFINITY;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.dempty[k]));
      if (MODE == 0) {
        // the group's maximum over its rows: lanes with equal lane % 4
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
        if (lane < kGroups) p.block_S[(static_cast<long long>(b) * kGroups + lane) * p.s_stride + c] = m;
      }
      cursor_advance(cur, nb);
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
  (void)all_alive;
}

// Step 3 of the fused selection, after the scan: one CTA per request, warp g takes
// group g's block scores (staged in shared memory when the row fits), the top 15
// plus the most recent block. A kernel of its own so it runs on SMs the scan has
// left (measured on GB300: run by the scan's last CTA per request, beside a CTA
// still scanning, it took about 15 us; here it runs on idle SMs).
__global__ void __launch_bounds__(128) topk_kernel(const SelectParams p, int stage_row) {
  extern __shared__ float tk_stage[];  // [4][stage_row] block scores (stage_row = 0: read global)
  __shared__ uint64_t scratch[kGroups][64];
  pdl_launch_dependents();
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the request's geometry is an input (not written by the scan): read it before waiting
  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  pdl_wait_primary();  // the block scores come from the scan kernel
  // stage the 4 whole score rows (16-byte padded) while the geometry loads land
  if (stage_row > 0) {
    const int row4 = stage_row / 4;
    for (int u = threadIdx.x; u < kGroups * row4; u += blockDim.x) {
      const int g = u / row4, c4 = u - g * row4;
      reinterpret_cast<float4*>(tk_stage + g * stage_row)[c4] = __ldcg(
          reinterpret_cast<const float4*>(p.block_S + (static_cast<long long>(b) * kGroups + g) * p.s_stride) + c4);
    }
  }
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows;
  const int nbb = ok && R > 0 ? (N + kBlock - 1) / kBlock : 0;
  __syncthreads();
  int32_t* ids = p.block_ids + (static_cast<long long>(b) * kGroups + warp) * kTopK;
  if (nbb == 0) {  // no pages: an empty selection
    if (lane < kTopK) ids[lane] = -1;
    if (p.block_scores_out != nullptr)
      for (int c = lane; c < p.max_pages; c += 32)
        p.block_scores_out[(static_cast<long long>(b) * kGroups + warp) * p.max_pages + c] = -INFINITY;
    return;
  }
  const float* S = stage_row > 0 ? tk_stage + warp * stage_row
                                 : p.block_S + (static_cast<long long>(b) * kGroups + warp) * p.s_stride;
  warp_topk(S, nbb, ids, scratch[warp]);
  if (p.block_scores_out != nullptr) {
    float* o = p.block_scores_out + (static_cast<long long>(b) * kGroups + warp) * p.max_pages;
    for (int c = lane; c < p.max_pages; c += 32) o[c] = c < nbb ? S[c] : -INFINITY;
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

size_t select_smem_bytes(int num_reqs) {
  const size_t need = sizeof(Smem) + sizeof(long long) * (num_reqs + 1) + sizeof(int) * (num_reqs + 1) +
                      3 * sizeof(int) * num_reqs + 1024;
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

cudaError_t launch_topk(const SelectParams& prm, cudaStream_t st) {
  // stage each group's score row in shared memory when the 4 rows fit in 160 KB
  const int stage_row = static_cast<size_t>(kGroups) * prm.s_stride * sizeof(float) <= 160 * 1024 ? prm.s_stride : 0;
  const size_t smem = static_cast<size_t>(kGroups) * stage_row * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_reqs, 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topk_kernel, prm, stage_row);
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
