// Step 4 of the MSA decode path: exact softmax attention over the selected
// blocks' NVFP4 K/V.
//
// [vLLM-zh "How MiniMax sparse attention works"] main attention runs exactly,
// but only on the 16 selected blocks, so each query uses at most 2,048 keys.
// [MSA-fig §1, sparse branch] standard GQA shapes; the blocks picked for a
// group are gathered from the real K/V and every query head of the group uses
// them. [vLLM-zh, Blackwell kernels] the K/V cache is NVFP4 and the queries FP8,
// so K/V are turned into FP8 in the kernel and the products run as FP8 MMA.
//
// Design (GB300, tcgen05). Grid = (splits, request x group), one CTA per SM; a
// CTA takes `blocks_per_split` of the group's selected blocks (flash-decoding
// split over the selection), and the splits of a (request, group) form one
// thread-block cluster that merges its partial results through distributed
// shared memory. The group's M = 8R query rows (R speculative rows x 8 heads)
// are repeated C times down the 128 rows of the MMA tile (C = 2 copies of 64
// rows, or C = 4 copies of 32 rows when R <= 4); copy c takes keys
// 128c/C .. 128(c+1)/C - 1 of every block, so the softmax of a block is spread
// over all four SM sub-partitions and a thread handles 128/C keys of its row:
//   * load warp: one lane copies each block's raw NVFP4 K and V into a 4-stage
//     shared-memory ring (codes by 2-D tensor copies with a 64-byte swizzle,
//     scales by bulk copies);
//   * 8 dequant warps in two groups taking alternate blocks, thread = one K row
//     and the same V row of the block: take the rows' codes into registers and
//     release the raw stage at once, dequantise both in one interleaved pass to
//     E4M3 (byte-permute lookups in a table of scaled magnitudes) into a
//     128-byte-swizzled K tile, and widened to FP16 into the V tile's two 64-dim
//     halves; two K tiles (free once S is computed) and three V tiles (free
//     once P V is computed), K and V ready separately;
//   * MMA warp: one lane issues S = Q K^T (FP8; A = query tile, B = K tile, both
//     shared memory, K-major) into one of two TMEM score buffers, and O += P V
//     (FP16; A = P from TMEM, B = the V tile read MN-major, so V is used in its
//     stored key-major order without a transpose) into the TMEM output; S of
//     block j+2 is issued after P V of block j;
//   * 4 softmax warps, warp q owning TMEM lanes 32q .. 32q + 31 (copy c, row m):
//     all of its keys' scores in one TMEM load, the block maximum over them, then
//     P = exp2(s c - ref) (argument by packed FP32 FMA) in packed FP16
//     (the FP16 form P takes as the next MMA's A operand in TMEM; the P columns
//     of the other copies' keys stay zero in its lane), the sum in FP32 per 32
//     keys. The exponent's reference moves only when a block's maximum exceeds
//     it by more than 2^8 (P <= 256 stays well inside FP16), and only then are the
//     lane's O columns rescaled, after the previous P V has finished; O / l does
//     not depend on the reference. The exponent argument is formed in FP32 and
//     rounded to FP16 for the packed exp2.
// P V runs in FP16: the dequantised V values (E4M3) are exact in FP16, and an
// E4M3 P (3 mantissa bits) measurably misses 2e-2 relative accuracy on rows whose
// weight sits on a few keys; FP16 P keeps 11 bits.
// At the end every lane's (O, max, sum) is a partial result of its row: the lanes
// store them into the shared memory of the cluster's CTA that finishes the row
// (each CTA finishes a share of the rows), and that CTA merges the C x splits
// partials of each of its rows with the log-sum-exp rule and writes BF16 output.
#include <cuda_bf16.h>

#include <cstddef>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr int kSoftWarps = 8;                       // warps 0..7: two sets of 4, one per TMEM lane quadrant
constexpr int kMmaWarp = 8;                         // S = Q K^T issue, TMEM allocation
constexpr int kPvWarp0 = 9;                         // warps 9, 10: O_s += P V issue for set s
constexpr int kLoadWarp = 11;                       // raw page copies
constexpr int kDqWarp0 = 12, kDqWarps = 8;          // warps 12..19: two groups of 4
constexpr int kAttnThreads = (kDqWarp0 + kDqWarps) * 32;
// raw NVFP4 page ring: two stages per dequant group (the groups take alternate blocks), so
// each stage has one consumer that takes its blocks in order; block j lands in stage
// raw_stage(j) and is that stage's (j / 4)-th block
constexpr int kAttnStages = 4;
constexpr int kKBufs = 2;                           // dequantised K tiles (free once S is computed)
constexpr int kVBufs = 3;                           // dequantised V tiles (free once P V is computed)
constexpr int kSets = 2;                            // softmax sets: set s takes blocks j = s (mod 2)
constexpr int kMaxSplits = kTopK / 2;               // CTAs per (request, group): at least 2 blocks each
constexpr uint32_t kHeadPageBytes = kBlock * 64;    // codes of one (page, KV head)
constexpr uint32_t kHeadScaleBytes = kBlock * 8;
constexpr uint32_t kTileBytes = kBlock * kDim;      // one dequantised K tile (E4M3, 128-byte rows)
constexpr uint32_t kVHalfBytes = kBlock * 128;      // one V tile half: 128 keys x 64 dims FP16 (128-byte rows)
constexpr int kLutCopies = 8;                       // interleaved copies of the magnitude table
constexpr int kLutEntryShift = 6;                   // bytes per table entry (all copies): 8 x 8 = 2^6
static_assert((8 << kLutEntryShift) / 8 == 8 * kLutCopies, "table entry stride");
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S of block j in buffer j % 2 (128 FP32, one per key), its P written over its
// first 64 columns (2 FP16 keys per column) once the scores are read; O of set s (128 FP32,
// one per dim)
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kRescaleLog2 = 8.f;  // O is rescaled only when the max grows by more than 2^8
constexpr int kMaxM = kQPerKV * kMaxRows;           // query rows of a (request, group)
static_assert(kColO + kDim * kSets <= kTmemCols && kColS + kBlock * kSets <= kColO, "TMEM buffers");
static_assert(kDqWarps * 32 == 2 * kBlock, "one dequant thread per K row and per V row");

struct AttnSmem {
  uint8_t qtile[128 * kDim];                        // A of S: C copies of the query rows
  uint8_t ktile[kKBufs][kTileBytes];                // B of S (K-major): row = key
  uint8_t vtile[kVBufs][2][kVHalfBytes];            // B of O (MN-major, FP16): [half][key][64 dims]
  uint8_t kc[kAttnStages][kHeadPageBytes];          // raw codes (tensor copies, 64-byte swizzle)
  uint8_t vc[kAttnStages][kHeadPageBytes];
  uint8_t ksc[kAttnStages][kHeadScaleBytes];        // raw scales (bulk copies)
  uint8_t vsc[kAttnStages][kHeadScaleBytes];
  uint2 lut[128 * kLutCopies];                      // scaled magnitudes per scale magnitude, interleaved
  uint64_t raw_full[kAttnStages], raw_empty[kAttnStages];
  uint64_t ktile_full[kKBufs], k_free[kKBufs], vtile_full[kVBufs], v_free[kVBufs];
  uint64_t s_full[kSets], p_full[kSets], pv_done[kSets], o_final[kSets], mma_drain[1 + kSets];
  float xm[128], xl[128];                           // set 1's reference max and sum per TMEM lane
  int stage_bad[kAttnStages];
  uint64_t tk_local[kTopK];                         // this CTA's 15 best candidates (the cluster reads them)
  int ids[kTopK];
  int phys[kTopK];                                  // block-table entries of the selected blocks
  uint32_t taddr;
  int nsel;
};
static_assert(offsetof(AttnSmem, ktile) % 1024 == 0 && offsetof(AttnSmem, vtile) % 1024 == 0 &&
                  kTileBytes % 1024 == 0 && kVHalfBytes % 1024 == 0,
              "128-byte-swizzled MMA operands");
static_assert(offsetof(AttnSmem, kc) % 1024 == 0 && offsetof(AttnSmem, vc) % 1024 == 0,
              "64-byte-swizzled tensor-copy destinations");
static_assert(offsetof(AttnSmem, ksc) % 16 == 0 && offsetof(AttnSmem, vsc) % 16 == 0 && kHeadScaleBytes % 16 == 0,
              "bulk copies need 16-byte alignment");
static_assert(offsetof(AttnSmem, raw_full) % 8 == 0, "mbarriers");
static_assert(sizeof(AttnSmem) + 1024 <= 227 * 1024, "shared memory a CTA may opt into");
// End of the main loop: the partials of the rows a CTA finishes land in its V tiles (free
// once every CTA of the cluster has finished its loop): [C S][ceil(M/S)][128] FP32 rows, then
// the rows' references and sums; at most C (M + S - 1) <= 156 rows.
static_assert(156 * (kDim + 2) * sizeof(float) <= sizeof(AttnSmem::vtile), "partials fit the V tiles");

__device__ __forceinline__ int raw_stage(int j) { return 2 * (j & 1) + ((j >> 1) & 1); }

__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
  const __nv_bfloat16 x = __float2bfloat16_rn(a), y = __float2bfloat16_rn(b);
  return static_cast<uint32_t>(__bfloat16_as_ushort(x)) | (static_cast<uint32_t>(__bfloat16_as_ushort(y)) << 16);
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t* flags) {
  return mbar_try(bar, parity) || mbar_wait(bar, parity, flags);
}

// Dequantise code chunk k of a row (16 bytes = 32 elements; scale bytes 2k and
// 2k+1 in the low 16 bits of s2) and store its 32 E4M3 bytes as chunks 2k, 2k+1
// of the row in a 128-byte-swizzled tile (chunk c of row r sits at c ^ (r & 7)).
__device__ __forceinline__ void dq_chunk(uint32_t lut_t, const uint4& v, uint32_t s2, uint32_t row_addr, int r7,
                                         int k) {
  const uint2 L0 = lds_u2(lut_t + ((s2 & 0x7Fu) << kLutEntryShift));
  const uint2 L1 = lds_u2(lut_t + (((s2 >> 8) & 0x7Fu) << kLutEntryShift));
  uint32_t o[8];
  dq8_signed(v.x, L0.x, L0.y, o[0], o[1]);
  dq8_signed(v.y, L0.x, L0.y, o[2], o[3]);
  dq8_signed(v.z, L1.x, L1.y, o[4], o[5]);
  dq8_signed(v.w, L1.x, L1.y, o[6], o[7]);
  st_shared_v4(row_addr + (static_cast<uint32_t>((2 * k) ^ r7) << 4), o[0], o[1], o[2], o[3]);
  st_shared_v4(row_addr + (static_cast<uint32_t>((2 * k + 1) ^ r7) << 4), o[4], o[5], o[6], o[7]);
}

// V row variant: the 32 E4M3 values of code chunk k widened to FP16 (exact) and
// stored as FP16 chunks 4(k & 1) .. 4(k & 1) + 3 of the row in V half k / 2.
__device__ __forceinline__ void dq_chunk_v(uint32_t lut_t, const uint4& v, uint32_t s2, uint32_t half_row0,
                                           int r7, int k) {
  const uint2 L0 = lds_u2(lut_t + ((s2 & 0x7Fu) << kLutEntryShift));
  const uint2 L1 = lds_u2(lut_t + (((s2 >> 8) & 0x7Fu) << kLutEntryShift));
  uint32_t o[8];
  dq8_signed(v.x, L0.x, L0.y, o[0], o[1]);
  dq8_signed(v.y, L0.x, L0.y, o[2], o[3]);
  dq8_signed(v.z, L1.x, L1.y, o[4], o[5]);
  dq8_signed(v.w, L1.x, L1.y, o[6], o[7]);
  uint32_t h[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h[2 * i]) : "r"(o[i] & 0xFFFFu));
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h[2 * i + 1]) : "r"(o[i] >> 16));
  }
  const uint32_t row = half_row0 + static_cast<uint32_t>(k >> 1) * kVHalfBytes;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    st_shared_v4(row + (static_cast<uint32_t>((4 * (k & 1) + cc) ^ r7) << 4), h[4 * cc], h[4 * cc + 1], h[4 * cc + 2],
                 h[4 * cc + 3]);
}

// Scratch of the fused top-k (in the first K tile, free until block 0 is dequantised).
struct TopkScratch {
  uint64_t lists[4 * kTopK];  // the four warps' lists (quad_best15)
  uint64_t surv[4 * 64];      // their survivors
};

}  // namespace

// C = copies of the query rows down the 128-row tile (2: rows < 64; 4: rows < 32).
template <int C>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const AttnParams p) {
  constexpr int kMpad = 128 / C;  // tile rows per copy = keys per thread per block
  constexpr int kDpc = kDim / C;  // output dims each copy finishes
  static_assert(kMpad % 32 == 0, "one copy per warp at least: TMEM loads take the same columns in a warp");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem_al = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // swizzled tiles: 1 KB
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_al);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.y, b = pair / kGroups, g = pair % kGroups;

  // the request's geometry is an input: checked before anything else (every CTA of the
  // cluster shares it, so they all leave here together or none does)
  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows && kQPerKV * R <= p.max_m && kQPerKV * R <= kMpad;
  if (!ok || R == 0) {
    if (!ok && tid == 0 && blockIdx.x == 0 && g == 0) set_flag(p.flags, kFlagBadLength);
    // nothing is selected for the group (when this kernel selects)
    if (p.block_S != nullptr && blockIdx.x == 0 && tid < kTopK)
      p.block_ids[(static_cast<long long>(b) * kGroups + g) * kTopK + tid] = -1;
    return;
  }
  const int nb = (N + kBlock - 1) / kBlock;
  const int M = kQPerKV * R;  // query rows of this (request, group): row m = speculative row m/8, head m%8

  for (int u = tid; u < 128 * kLutCopies; u += kAttnThreads)
    sm.lut[u] = lut_magnitudes(static_cast<uint32_t>(u / kLutCopies));
  if (tid == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(smem_u32(&sm.raw_full[s]), 1);
      mbar_init(smem_u32(&sm.raw_empty[s]), kDqWarps / 2);  // the group dequantising the block
    }
    for (int t = 0; t < kKBufs; ++t) {
      mbar_init(smem_u32(&sm.ktile_full[t]), kDqWarps / 2);  // the group dequantising the block
      mbar_init(smem_u32(&sm.k_free[t]), 1);
    }
    for (int t = 0; t < kVBufs; ++t) {
      mbar_init(smem_u32(&sm.vtile_full[t]), kDqWarps / 2);  // the group dequantising the block
      mbar_init(smem_u32(&sm.v_free[t]), 1);
    }
    for (int t = 0; t < kSets; ++t) {
      mbar_init(smem_u32(&sm.s_full[t]), 1);
      mbar_init(smem_u32(&sm.p_full[t]), kSoftWarps / kSets);
      mbar_init(smem_u32(&sm.pv_done[t]), 1);
      mbar_init(smem_u32(&sm.o_final[t]), 1);
    }
    for (int t = 0; t < 1 + kSets; ++t) mbar_init(smem_u32(&sm.mma_drain[t]), 1);
    mbar_fence_init();
  }
  // query tile: 128 rows x 128 bytes, 128-byte swizzle; row l holds query row l % kMpad
  // (zero when that is >= M)
  for (int u = tid; u < 128 * 8; u += kAttnThreads) {
    const int l = u >> 3, ch = u & 7, mq = l % kMpad;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (mq < M)
      v = *reinterpret_cast<const uint4*>(
          p.q + ((static_cast<long long>(r0 + mq / kQPerKV) * kHeads) + kQPerKV * g + mq % kQPerKV) * kDim + ch * 16);
    *reinterpret_cast<uint4*>(sm.qtile + l * 128 + ((ch ^ (l & 7)) << 4)) = v;
  }

  // the request's block-table row (an input) staged before the wait in the third V tile,
  // unused until block 2 is dequantised, so the selected pages resolve from shared memory;
  // the tensor memory too is taken before the wait (the SM's previous CTA, whose shared
  // memory this CTA needed, has exited)
  const bool bt_staged = nb <= static_cast<int>(sizeof(sm.vtile[2]) / 4);
  int32_t* bt = reinterpret_cast<int32_t*>(sm.vtile[2]);
  if (bt_staged)
    for (int c = tid; c < nb; c += kAttnThreads) bt[c] = p.block_table[static_cast<long long>(b) * p.max_pages + c];
  if (warp == kMmaWarp) tmem_alloc(smem_u32(&sm.taddr), kTmemCols);
  if (warp == kLoadWarp && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
  }
  __syncthreads();

  pdl_wait_primary();  // the block ids (or the block scores) come from the selection

  if (p.block_S == nullptr) {
    if (warp == 0) {
      // the 16 given ids in parallel; the valid ones keep their order (ballot ranks)
      const int id = lane < kTopK ? p.block_ids[(static_cast<long long>(b) * kGroups + g) * kTopK + lane] : -1;
      const bool valid = lane < kTopK && id >= 0 && id < nb;
      if (lane < kTopK && !valid && id != -1 && blockIdx.x == 0) set_flag(p.flags, kFlagBadIds);
      const unsigned vm = __ballot_sync(0xFFFFFFFFu, valid);
      if (valid) {
        const int rank = __popc(vm & ((1u << lane) - 1u));
        sm.ids[rank] = id;
        sm.phys[rank] = bt_staged ? bt[id] : p.block_table[static_cast<long long>(b) * p.max_pages + id];
      }
      if (lane == 0) sm.nsel = __popc(vm);
    }
  } else {
    // ---- the top-k of this group, fused [vLLM-zh "How MiniMax sparse attention works"; MSA-fig
    // §1 TopK]: the recent block plus the 15 best others by block score (ties to the lower
    // id); every block when there are at most 16. CTA s of the cluster ranks candidates
    // [s nc / S, (s + 1) nc / S) to its 15 best, and each CTA merges the cluster's lists: the
    // 15 best overall are among them, so the merge is exact. The split-0 CTA writes the ids.
    const int S = p.splits;
    const int rank = S > 1 ? static_cast<int>(cluster_rank()) : 0;
    int32_t* ids_out = p.block_ids + (static_cast<long long>(b) * kGroups + g) * kTopK;
    TopkScratch& tk = *reinterpret_cast<TopkScratch*>(sm.ktile[0]);
    if (nb <= kTopK) {
      if (warp == 0 && lane < kTopK) {
        if (lane < nb) {
          sm.ids[lane] = lane;
          sm.phys[lane] = bt_staged ? bt[lane] : p.block_table[static_cast<long long>(b) * p.max_pages + lane];
        }
        if (rank == 0) ids_out[lane] = lane < nb ? lane : -1;
        if (lane == 0) sm.nsel = nb;
      }
    } else {
      const int nc = nb - 1;
      const float* Sg = p.block_S + (static_cast<long long>(b) * kGroups + g) * p.s_stride;
      if (warp < 4) {
        const uint64_t best = quad_best15(Sg, rank * nc / S, (rank + 1) * nc / S, warp, 2, tk.lists, tk.surv);
        if (warp == 0 && lane < kTopK) sm.tk_local[lane] = best;  // descending, zero past the end
      }
      __syncthreads();
      if (S > 1) cluster_sync_all();  // every CTA's list is in place
      if (warp == 0) {
        // the S lists (this CTA's, or in the other CTAs' shared memory), all loads issued
        // first, merged into the 15 best; the ranges are disjoint, so the keys are distinct
        const uint32_t laddr = smem_u32(sm.tk_local) + 8u * static_cast<uint32_t>(lane & (kTopK - 1));
        uint64_t kin[kMaxSplits];
#pragma unroll
        for (int src = 0; src < kMaxSplits; ++src)
          kin[src] = (src < S && lane < kTopK)
                         ? (S > 1 ? ld_cluster_u64(cluster_map(laddr, static_cast<uint32_t>(src))) : sm.tk_local[lane])
                         : 0ull;
        uint64_t top = kin[0];
#pragma unroll
        for (int src = 1; src < kMaxSplits; ++src)
          if (src < S) top = top32_union(top, kin[src]);
        const int win = lane < kTopK - 1 ? topk_id(top) : nb - 1;  // lane 15 keeps the recent block
        // the 16 ids ascending
        int r = 0;
#pragma unroll
        for (int j = 0; j < kTopK; ++j) {
          const int other = __shfl_sync(0xFFFFFFFFu, win, j);
          r += other < win ? 1 : 0;
        }
        if (lane < kTopK) {
          sm.ids[r] = win;
          sm.phys[r] = bt_staged ? bt[win] : p.block_table[static_cast<long long>(b) * p.max_pages + win];
          if (rank == 0) ids_out[r] = win;
        }
        if (lane == 0) sm.nsel = kTopK;
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.taddr;
  const int jb0 = blockIdx.x * p.blocks_per_split;
  int nmy = sm.nsel - jb0;
  nmy = nmy < 0 ? 0 : (nmy > p.blocks_per_split ? p.blocks_per_split : nmy);

  // what a softmax lane carries past its role: its row and copy, whether its O is final,
  // its reference max (log2) and sum
  bool fin = false;
  int row_m = kMaxM, copy_c = 0;
  float ref_out = -INFINITY, sum_out = 0.f, both_w0 = 0.f, both_w1 = 0.f;

  if (warp == kLoadWarp) {
    // ================= load warp: raw K/V pages of block j into stage j % kAttnStages
    if (lane == 0) {
      auto page_bad = [&](int phys) { return phys < 0 || phys >= p.num_pages; };
      auto issue = [&](int j) {
        const int st = raw_stage(j);
        const int phys = sm.phys[jb0 + j];
        const uint32_t bar = smem_u32(&sm.raw_full[st]);
        const bool bad = page_bad(phys);
        sm.stage_bad[st] = bad ? 1 : 0;
        if (bad) {
          set_flag(p.flags, kFlagBadPage);
          mbar_arrive(bar);
          return;
        }
        const int head_row = (phys * kGroups + g) * kBlock;
        mbar_arrive_expect_tx(bar, 2 * (kHeadPageBytes + kHeadScaleBytes));
        tma_load_2d(smem_u32(sm.kc[st]), &kmap, 0, head_row, bar);
        tma_load_2d(smem_u32(sm.vc[st]), &vmap, 0, head_row, bar);
        bulk_load(smem_u32(sm.ksc[st]), p.k_scale + static_cast<long long>(head_row) * 8, kHeadScaleBytes, bar);
        bulk_load(smem_u32(sm.vsc[st]), p.v_scale + static_cast<long long>(head_row) * 8, kHeadScaleBytes, bar);
      };
      int issued = 0;
      for (; issued < nmy && issued < kAttnStages; ++issued) issue(issued);
      // (no L2 prefetch of the later blocks: with a 4-stage ring the copies keep up, and
      // asking L2 for every later block at once was measured ~1-2.6 us slower per call on
      // GB300 at 8 and 16 blocks per CTA)
      for (; issued < nmy; ++issued) {
        const int st = raw_stage(issued);
        if (!wait_bar(smem_u32(&sm.raw_empty[st]), ((issued / kAttnStages) - 1) & 1, p.flags)) break;
        issue(issued);
      }
      // no copy may still be landing when the CTA leaves: wait for the last one of each stage
      for (int j = issued - kAttnStages < 0 ? 0 : issued - kAttnStages; j < issued; ++j)
        if (!mbar_wait(smem_u32(&sm.raw_full[raw_stage(j)]), (j / kAttnStages) & 1, p.flags)) break;
    }
    __syncwarp();
  } else if (warp >= kDqWarp0) {
    // ================= dequant warps: group grp = warp-group parity takes blocks j = grp,
    // grp + 2, ... (two blocks in flight); thread = row r of that block's K and of its V, both
    // dequantised in one interleaved pass (twice the independent work per thread)
    const int t = tid - kDqWarp0 * 32;
    const int grp = t >> 7, r = t & 127;
    const int r7 = r & 7, sw = (r >> 1) & 3;   // sw: the 64-byte swizzle of the raw codes
    const uint32_t lut_t = smem_u32(sm.lut) + static_cast<uint32_t>(lane % kLutCopies) * 8u;
    for (int j = grp; j < nmy; j += 2) {
      const int st = raw_stage(j);
      // every lane takes the same branch on a wait (a lane leaving the loop alone would stall
      // its warp's next __syncwarp)
      if (!__all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.raw_full[st]), (j / kAttnStages) & 1, p.flags))) break;
      // the row's K and V codes and scales go to registers and the stage back to the load
      // warp at once, so the copy of the stage's next block overlaps this block's dequantisation
      const bool bad = sm.stage_bad[st] != 0;
      const uint32_t krow = smem_u32(sm.kc[st]) + static_cast<uint32_t>(r) * 64u;
      const uint32_t vrow = smem_u32(sm.vc[st]) + static_cast<uint32_t>(r) * 64u;
      uint4 kv[4], vv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        kv[c] = lds_u4(krow + (static_cast<uint32_t>(c ^ sw) << 4));
        vv[c] = lds_u4(vrow + (static_cast<uint32_t>(c ^ sw) << 4));
      }
      const uint2 ksc = lds_u2(smem_u32(sm.ksc[st]) + static_cast<uint32_t>(r) * 8u);
      const uint2 vsc = lds_u2(smem_u32(sm.vsc[st]) + static_cast<uint32_t>(r) * 8u);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.raw_empty[st]));
      // the tiles' previous blocks have been consumed: their S (K tiles), their P V (V tiles)
      const int kb = j % kKBufs, vb = j % kVBufs;
      if (j >= kKBufs &&
          !__all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.k_free[kb]), ((j / kKBufs) - 1) & 1, p.flags)))
        break;
      if (j >= kVBufs &&
          !__all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.v_free[vb]), ((j / kVBufs) - 1) & 1, p.flags)))
        break;
      const int pos0 = sm.ids[jb0 + j] * kBlock;
      const int nvalid = N - pos0 < kBlock ? N - pos0 : kBlock;
      const uint32_t kaddr = smem_u32(sm.ktile[kb]) + static_cast<uint32_t>(r) * 128u;
      const uint32_t vaddr = smem_u32(sm.vtile[vb][0]) + static_cast<uint32_t>(r) * 128u;
      // a bad page reads as zeros; V rows past the context are zero (their weights are 0,
      // and 0 x NaN from unwritten slots must not reach P V); K rows past it are masked
      if (bad) {
#pragma unroll
        for (int c = 0; c < 8; ++c) st_shared_v4(kaddr + (c << 4), 0u, 0u, 0u, 0u);
      }
      if (bad || r >= nvalid) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          st_shared_v4(vaddr + (c << 4), 0u, 0u, 0u, 0u);
          st_shared_v4(vaddr + kVHalfBytes + (c << 4), 0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!bad) dq_chunk(lut_t, kv[k], ((k & 2) ? ksc.y : ksc.x) >> ((k & 1) * 16), kaddr, r7, k);
        if (!bad && r < nvalid) dq_chunk_v(lut_t, vv[k], ((k & 2) ? vsc.y : vsc.x) >> ((k & 1) * 16), vaddr, r7, k);
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the MMA (async proxy)
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.ktile_full[kb]));
        mbar_arrive(smem_u32(&sm.vtile_full[vb]));
      }
    }
  } else if (warp == kMmaWarp) {
    // ================= S warp: S_j = Q K_j^T into TMEM buffer j % 2, once K_j is in its tile
    // and that buffer's previous P (block j - 2) has been consumed by its P V. One thread
    // issues an MMA only every ~70-90 cycles (measured on GB300), so the S and the two sets'
    // P V products are issued from three warps.
    if (lane == 0) {
      const uint64_t qdesc = sdesc_kmajor_sw128(smem_u32(sm.qtile));
      const uint32_t id_qk = idesc_e4m3_f32(128, kBlock, false, false);
      int nq = 0;
      for (; nq < nmy; ++nq) {
        const int tb = nq % kKBufs, sb = nq % kSets;
        if (!wait_bar(smem_u32(&sm.ktile_full[tb]), (nq / kKBufs) & 1, p.flags)) break;
        if (nq >= kSets && !wait_bar(smem_u32(&sm.pv_done[sb]), ((nq / kSets) - 1) & 1, p.flags)) break;
        tc_fence_after();
        // K step kk of an operand: +32 bytes along K-major rows (+2 in the address field)
        const uint64_t kdesc = sdesc_kmajor_sw128(smem_u32(sm.ktile[tb]));
#pragma unroll
        for (int kk = 0; kk < kDim / 32; ++kk)
          mma_f8_ss(tbase + kColS + kBlock * sb, qdesc + 2 * kk, kdesc + 2 * kk, id_qk, kk > 0);
        mma_commit(smem_u32(&sm.s_full[sb]));
        mma_commit(smem_u32(&sm.k_free[tb]));
      }
      // every MMA this thread issued has finished before the tensor memory is released
      if (nq > 0) {
        mma_commit(smem_u32(&sm.mma_drain[0]));
        mbar_wait(smem_u32(&sm.mma_drain[0]), 0, p.flags);
      }
    }
    __syncwarp();
  } else if (warp == kPvWarp0 || warp == kPvWarp0 + 1) {
    // ================= P V warp of set s: O_s += P_j V_j for the set's blocks j = s, s + 2, ...
    // once the set has written P_j (over S_j's buffer) and V_j is in its tile
    const int sb = warp - kPvWarp0;
    if (lane == 0) {
      const uint32_t id_pv = idesc_f16_f32(128, kDim, true);
      int nmine = 0;
      for (int j = sb; j < nmy; j += kSets, ++nmine) {
        const int tb = j % kVBufs;
        if (!wait_bar(smem_u32(&sm.p_full[sb]), nmine & 1, p.flags)) break;
        if (!wait_bar(smem_u32(&sm.vtile_full[tb]), (j / kVBufs) & 1, p.flags)) break;
        tc_fence_after();
        // MN-major V: 128 dims = two 128-byte swizzle atoms (the two halves, kVHalfBytes
        // apart: the leading-dimension offset), 8-key groups 1 KB apart (the stride
        // offset); K step kk = 16 keys = 2048 bytes (+128 in the field); A = P, 8 columns
        const uint64_t vdesc = sdesc_mn_sw128(smem_u32(sm.vtile[tb][0]), kVHalfBytes);
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk)
          mma_f16_tmemA(tbase + kColO + kDim * sb, tbase + kColS + kBlock * sb + 8 * kk, vdesc + 128 * kk, id_pv,
                        (nmine > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sm.pv_done[sb]));
        mma_commit(smem_u32(&sm.v_free[tb]));
        if (j + kSets >= nmy) mma_commit(smem_u32(&sm.o_final[sb]));  // single phase: O_sb complete
      }
      if (nmine > 0) {
        mma_commit(smem_u32(&sm.mma_drain[1 + sb]));
        mbar_wait(smem_u32(&sm.mma_drain[1 + sb]), 0, p.flags);
      }
    }
    __syncwarp();
  } else {
    // ================= softmax warps: set st = warp / 4 takes blocks j = st, st + 2, ...
    // with its own O accumulator; lane l = 32 (warp % 4) + lane of TMEM holds query row
    // m = l % kMpad of copy c = l / kMpad, which takes keys k0 .. k0 + kMpad - 1 of every
    // block; its O sums those keys only (the P columns of the other copies' keys are zero in
    // its lane), with its own reference max and running sum
    const int st = warp / 4, q = warp % 4;
    const int l = 32 * q + lane, m = l % kMpad, c = l / kMpad, k0 = c * kMpad;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t o_cols = tbase + lane_base + kColO + kDim * st;
    const int rq = m / kQPerKV;
    const int pos_max = N - R + rq;  // this row sees key positions <= pos_max
    const float sc = p.sm_scale_log2;
    float mref = -INFINITY, lrun = 0.f;  // reference max (log2 domain) and running sum
    bool good = true;
    int nmine = 0;  // blocks this set has processed
    for (int j = st; j < nmy; j += kSets, ++nmine) {
      const int pos0 = sm.ids[jb0 + j] * kBlock;
      const bool full_vis = pos0 + kBlock - 1 <= N - R;  // every key visible to every row
      const int lim = pos_max - pos0 - k0;                // key k0 + n visible iff n <= lim
      good = __all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.s_full[st]), nmine & 1, p.flags));
      if (!good) break;
      tc_fence_after();
      const uint32_t s_cols = tbase + lane_base + kColS + kBlock * st;
      // this thread's kMpad scores of the block, one wait for all of them
      uint32_t v[kMpad];
#pragma unroll
      for (int ch = 0; ch < kMpad / 32; ++ch)
        tmem_ld32(s_cols + k0 + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * ch));
      tc_wait_ld();
      if (!full_vis) {
#pragma unroll
        for (int u = 0; u < kMpad; ++u) v[u] = u <= lim ? v[u] : __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < kMpad; u += 2) mx = fmax3(mx, __uint_as_float(v[u]), __uint_as_float(v[u + 1]));
      // Lazy rescale: P is taken relative to a reference max mref that moves only
      // when this block's max exceeds it by more than kRescaleLog2 (P then stays
      // below 2^kRescaleLog2, well inside FP16); O / l is exact whatever mref is.
      const float bmax = mx * sc;  // sc > 0 keeps the order of the raw scores
      const bool move = bmax > mref + kRescaleLog2 || (mref == -INFINITY && bmax != -INFINITY);
      const float m_new = move ? bmax : mref;
      const float ref = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(mref - ref);  // 0 while nothing was seen yet
      const bool rescale = move && mref != -INFINITY;
      // P = exp2(s sc - ref) for this thread's keys (masked scores are -inf: P = 0), FP16
      // pairs: key n of the block in column n / 2 of the buffer (over scores already read),
      // the columns of the other copies' keys zero; summed in FP16 pairs per 32 keys, then FP32.
      // Pair u2 of a chunk is packed into v[32 ch + u2], a slot already consumed.
      float lsum = 0.f;
      const float2 sc2 = make_float2(sc, sc), nref2 = make_float2(-ref, -ref);
#pragma unroll
      for (int ch = 0; ch < kMpad / 32; ++ch) {
        uint32_t hsum = 0u;
#pragma unroll
        for (int u2 = 0; u2 < 16; ++u2) {
          const float2 d = __ffma2_rn(
              make_float2(__uint_as_float(v[32 * ch + 2 * u2]), __uint_as_float(v[32 * ch + 2 * u2 + 1])), sc2, nref2);
          uint32_t hx, hp;
          asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hx) : "f"(d.y), "f"(d.x));
          asm("ex2.approx.f16x2 %0, %1;" : "=r"(hp) : "r"(hx));
          asm("add.rn.f16x2 %0, %0, %1;" : "+r"(hsum) : "r"(hp));
          v[32 * ch + u2] = hp;
        }
        tmem_st16(s_cols + (k0 + 32 * ch) / 2, v + 32 * ch);
        float2 f;
        asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
            : "=f"(f.x), "=f"(f.y)
            : "r"(hsum));
        lsum += f.x + f.y;
      }
      // zero P columns of the other copies' keys (their scores were overwritten by S)
#pragma unroll
      for (int z = 0; z < 4; ++z)
        if (z < c * kMpad / 32 || z >= (c + 1) * kMpad / 32) tmem_zero16(s_cols + 16 * z);
      if (nmine >= 1 && __any_sync(0xFFFFFFFFu, rescale)) {
        // O must hold this set's earlier blocks before it is rescaled: the P V of its
        // previous block (phase nmine - 1 of its pv_done); P V of this block starts only after
        // the arrival below
        if (!__all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.pv_done[st]), (nmine - 1) & 1, p.flags))) {
          good = false;
          break;
        }
        tc_fence_after();
        const float a = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int qc = 0; qc < 4; ++qc) {  // one 32-column chunk live at a time
          uint32_t o[32];
          tmem_ld32(o_cols + 32 * qc, o);
          tc_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * a);
          tmem_st32(o_cols + 32 * qc, o);
        }
      }
      lrun = lrun * alpha + lsum;
      mref = m_new;
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[st]));
    }
    // ---- this set's O is final once its last P V has completed; set 1 hands its reference
    // and sum to set 0, whose lanes combine the two (same rows, same TMEM lanes)
    const bool fin_mine =
        good && nmine > 0 && __all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.o_final[st]), 0, p.flags));
    if (st == 1) {
      sm.xm[l] = fin_mine ? mref : -INFINITY;
      sm.xl[l] = fin_mine ? lrun : 0.f;
    }
    named_bar_sync(1, kSoftWarps * 32);
    if (st == 0) {
      const float m1 = sm.xm[l], l1 = sm.xl[l];
      const float m0 = fin_mine ? mref : -INFINITY, l0 = fin_mine ? lrun : 0.f;
      const float mt = fmaxf(m0, m1);
      const float rt = mt == -INFINITY ? 0.f : mt;
      const float w0 = exp2f(m0 - rt), w1 = exp2f(m1 - rt);
      fin = m0 != -INFINITY || m1 != -INFINITY;
      both_w0 = w0;
      both_w1 = w1;
      row_m = m;
      copy_c = c;
      ref_out = mt;
      sum_out = l0 * w0 + l1 * w1;
    }
  }

  // ---- every CTA of the cluster has finished its main loop, so its V tiles (where the
  // partials land) are free. Each softmax lane then sends its row's unnormalised O (128 FP32
  // from TMEM, relative to its own reference) with its (reference, sum) to the CTA that
  // finishes that row: CTA s of the cluster finishes rows [s Ro, (s + 1) Ro), Ro = ceil(M / S),
  // merging the C x S partials of each with the log-sum-exp rule. Stores into another CTA's
  // shared memory wait for nothing; the cluster barrier after them makes them visible.
  // Every thread of every CTA of the cluster reaches both barriers, on every path.
  const int S = p.splits;
  const int rank = S > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int Ro = (M + S - 1) / S;
  const int nslots = C * S;
  const uint32_t in_base = smem_u32(sm.vtile);
  const uint32_t in_m = in_base + static_cast<uint32_t>(nslots * Ro * kDim) * 4u;  // float [C S][Ro]
  const uint32_t in_l = in_m + static_cast<uint32_t>(nslots * Ro) * 4u;
  tc_fence_before();
  __syncthreads();
  if (S > 1) cluster_sync_all();
  tc_fence_after();
  if (warp < kSoftWarps / kSets) {
    // the TMEM loads are warp-wide (every lane takes part); only lanes of real rows store
    const bool real = row_m < M;
    const int owner = real ? row_m / Ro : 0, i = real ? row_m % Ro : 0, k = copy_c + C * rank;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t row_addr = in_base + static_cast<uint32_t>((k * Ro + i) * kDim) * 4u;
    auto put4 = [&](uint32_t laddr, float4 v) {
      if (S > 1) {
        const uint32_t ra = cluster_map(laddr, static_cast<uint32_t>(owner));
        asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "f"(v.x), "f"(v.y), "f"(v.z),
                     "f"(v.w)
                     : "memory");
      } else {
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(laddr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                     : "memory");
      }
    };
    auto put1 = [&](uint32_t laddr, float v) {
      if (S > 1)
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_map(laddr, static_cast<uint32_t>(owner))), "f"(v)
                     : "memory");
      else
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(laddr), "f"(v) : "memory");
    };
    // a set that processed no block has an undefined O: read it only with a nonzero weight
    const bool rd0 = __any_sync(0xFFFFFFFFu, both_w0 != 0.f), rd1 = __any_sync(0xFFFFFFFFu, both_w1 != 0.f);
#pragma unroll 1
    for (int qc = 0; qc < 4; ++qc) {
      uint32_t v[32], v1[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) v[u] = v1[u] = 0u;
      if (rd0) tmem_ld32(tbase + lane_base + kColO + 32 * qc, v);
      if (rd1) tmem_ld32(tbase + lane_base + kColO + kDim + 32 * qc, v1);
      tc_wait_ld();
#pragma unroll
      for (int u = 0; u < 32; ++u)
        v[u] = __float_as_uint((both_w0 != 0.f ? both_w0 * __uint_as_float(v[u]) : 0.f) +
                               (both_w1 != 0.f ? both_w1 * __uint_as_float(v1[u]) : 0.f));
      // 16-byte piece k4 of a row at piece (k4 + i) % 32: lanes (consecutive rows) hit
      // different banks
      if (real)
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4)
          put4(row_addr + 16u * static_cast<uint32_t>((8 * qc + u4 + i) & 31),
               make_float4(__uint_as_float(v[4 * u4]), __uint_as_float(v[4 * u4 + 1]), __uint_as_float(v[4 * u4 + 2]),
                           __uint_as_float(v[4 * u4 + 3])));
    }
    if (real) {
      put1(in_m + 4u * static_cast<uint32_t>(k * Ro + i), ref_out);
      put1(in_l + 4u * static_cast<uint32_t>(k * Ro + i), sum_out);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  if (S > 1) cluster_sync_all();  // every partial has landed

  // ---- this CTA's rows: out = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k over its C S
  // partials, BF16, and lse = log(sum) (natural log)
  const int row_lo = rank * Ro;
  const int nrows = M - row_lo < Ro ? M - row_lo : Ro;
  const int nitems = (nrows > 0 ? nrows : 0) * (kDim / 4);
  const float* fin_o = reinterpret_cast<const float*>(sm.vtile);
  const float* fin_m = fin_o + nslots * Ro * kDim;
  const float* fin_l = fin_m + nslots * Ro;
  for (int idx = tid; idx < nitems; idx += kAttnThreads) {
    const int i = idx / (kDim / 4), d4 = idx % (kDim / 4);
    float mx = -INFINITY;
    for (int k = 0; k < nslots; ++k) mx = fmaxf(mx, fin_m[k * Ro + i]);
    const float ref = mx == -INFINITY ? 0.f : mx;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    for (int k = 0; k < nslots; ++k) {
      const float mk = fin_m[k * Ro + i];
      if (mk == -INFINITY) continue;  // an empty partial (sum 0) contributes nothing
      const float wgt = exp2f(mk - ref);
      const float4 v = *reinterpret_cast<const float4*>(fin_o + (k * Ro + i) * kDim + 4 * ((d4 + i) & 31));
      acc.x += wgt * v.x;
      acc.y += wgt * v.y;
      acc.z += wgt * v.z;
      acc.w += wgt * v.w;
      den += wgt * fin_l[k * Ro + i];
    }
    const int mrow = row_lo + i;
    const long long orow = (static_cast<long long>(r0 + mrow / kQPerKV) * kHeads) + kQPerKV * g + mrow % kQPerKV;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    *reinterpret_cast<uint2*>(p.out + orow * kDim + 4 * d4) =
        make_uint2(bf16x2_bits(acc.x * inv, acc.y * inv), bf16x2_bits(acc.z * inv, acc.w * inv));
    if (d4 == 0 && p.lse != nullptr) p.lse[orow] = den > 0.f ? (ref + log2f(den)) * 0.69314718055994531f : -INFINITY;
  }
}

size_t attn_smem_bytes() { return sizeof(AttnSmem) + 1024; }

cudaError_t launch_attn(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& prm, bool pdl,
                        cudaStream_t st) {
  const size_t smem = attn_smem_bytes();
  auto kern = prm.copies == 4 ? attn_kernel<4> : attn_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.splits, prm.num_reqs * kGroups, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (prm.splits > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = prm.splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
