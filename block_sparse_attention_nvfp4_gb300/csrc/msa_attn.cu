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
// split over the selection). The group's 8R query rows (R speculative rows x 8
// heads, at most 64) are rows 0..63 of a 128-row MMA tile and again rows 64..127:
//   * load warp: one lane copies each block's raw NVFP4 K and V (codes and
//     scales) into a 2-stage shared-memory ring with bulk async copies;
//   * 8 dequant warps, thread = one K row or one V row of the block (the two
//     halves of the warps swap K and V every block, a V row costing about twice a
//     K row): take the row's codes into registers and release the raw stage at
//     once, then dequantise its 128 elements to E4M3 (byte-permute lookups in a
//     table of scaled magnitudes) into a 128-byte-swizzled tile (V rows widened to
//     FP16 into two 64-dim tiles); three tile buffers, K and V ready separately;
//   * MMA warp: one lane issues S = Q K^T (FP8; A = query tile, B = K tile, both
//     shared memory, K-major) into one of two TMEM score buffers, and O += P V
//     (FP16; A = P from TMEM, B = the V tile read MN-major, so V is used in its
//     stored key-major order without a transpose, as two 64-dim halves) into the
//     TMEM output; S of block j+2 is issued after P V of block j;
//   * 4 softmax warps, one per SM sub-partition: warp q owns TMEM lanes 32q ..
//     32q + 31 (query row 32 (q & 1) + lane) and keys 64 (q >> 1) .. + 63 of every
//     block, so each warp holds whole rows for half the keys: read its 64 scores
//     once into registers, mask, online softmax (FP32 running sum; exp2 in packed
//     FP16, two keys per instruction, which is also the FP16 form P takes as the
//     next MMA's A operand in TMEM; the P columns of the other key half stay zero
//     in its lanes). The exponent's reference point moves only when a block's max
//     exceeds it by more than 2^8 (so P <= 256 stays well inside FP16), and only
//     then are the warp's O rows in TMEM rescaled, after the previous P V has
//     finished; O / l is exact whatever the reference. The two key halves of a row
//     are combined once, at the end, with the log-sum-exp rule.
// P V runs in FP16: the dequantised V values (E4M3) are exact in FP16, and an
// E4M3 P (3 mantissa bits) measurably misses 2e-2 relative accuracy on rows whose
// weight sits on a few keys; FP16 P keeps 11 bits.
// CTAs that split the selection write (o, lse) partials and the last one to
// arrive for the (request, group) merges them with the exact log-sum-exp rule and
// writes BF16 output; finished rows go out through shared memory as coalesced
// 16-byte stores.
#include <cuda_bf16.h>

#include <cstddef>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

// Warp w may access TMEM lanes 32 (w % 4) .. + 31. Query rows are lanes 0..63 and again
// 64..127; softmax warp q owns lanes 32q .. 32q + 31 (one per SM sub-partition).
constexpr int kSoftWarps = 4;                       // warps 0..3: keys 0..63 (q < 2) or 64..127
constexpr int kMmaWarp = 4;                         // MMA issue, TMEM allocation
constexpr int kLoadWarp = 5;                        // raw page copies
constexpr int kDqWarp0 = 6, kDqWarps = 8;           // warps 6..13: K rows (0..127), V rows (128..255)
constexpr int kAttnThreads = (kDqWarp0 + kDqWarps) * 32;
constexpr int kAttnStages = 2;                      // raw NVFP4 page ring
constexpr int kTileBufs = 3;                        // dequantised K / V tiles
constexpr int kSBufs = 2;                           // TMEM score and P buffers
constexpr uint32_t kHeadPageBytes = kBlock * 64;    // codes of one (page, KV head)
constexpr uint32_t kHeadScaleBytes = kBlock * 8;
constexpr uint32_t kTileBytes = kBlock * kDim;      // one dequantised K tile (E4M3, 128-byte rows)
constexpr uint32_t kVHalfBytes = kBlock * 128;      // one V tile half: 128 keys x 64 dims FP16 (128-byte rows)
constexpr int kLutCopies = 16;                      // one per thread of a 16-thread (8-byte) wavefront
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S (2 x 128 FP32, one per key), O (128 FP32, one per dim), P (2 x 64,
// 2 FP16 keys per column)
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr float kRescaleLog2 = 8.f;  // O is rescaled only when the max grows by more than 2^8
static_assert(kColP + 64 * kSBufs <= kTmemCols, "TMEM buffers exceed the allocation");
static_assert(kDqWarps * 32 == 2 * kBlock, "one dequant thread per K row and per V row");

struct AttnSmem {
  uint8_t qtile[128 * kDim];                        // A of S: query rows 0..M-1, zero rows after
  uint8_t ktile[kTileBufs][kTileBytes];             // B of S (K-major): row = key
  uint8_t vtile[kTileBufs][2][kVHalfBytes];         // B of O (MN-major, FP16): [half][key][64 dims]
  uint8_t kc[kAttnStages][kHeadPageBytes];          // raw pages (bulk-copy destinations)
  uint8_t vc[kAttnStages][kHeadPageBytes];
  uint8_t ksc[kAttnStages][kHeadScaleBytes];
  uint8_t vsc[kAttnStages][kHeadScaleBytes];
  uint2 lut[128 * kLutCopies];                      // scaled magnitudes per scale magnitude, interleaved
  float xmax[2][64];                                // key halves' reference maxima and sums
  float xsum[2][64];
  int soft_dead;                                    // a softmax warp gave up waiting
  uint64_t raw_full[kAttnStages], raw_empty[kAttnStages];
  uint64_t ktile_full[kTileBufs], vtile_full[kTileBufs], tile_free[kTileBufs];
  uint64_t s_full[kSBufs], s_free[kSBufs], p_full[kSBufs], p_free[kSBufs], o_done, o_final;
  int stage_bad[kAttnStages];
  int ids[kTopK];
  int phys[kTopK];                                  // block-table entries of the selected blocks
  uint32_t taddr;
  int nsel;
  int last;
};
static_assert(offsetof(AttnSmem, ktile) % 1024 == 0 && offsetof(AttnSmem, vtile) % 1024 == 0 &&
                  kTileBytes % 1024 == 0 && kVHalfBytes % 1024 == 0,
              "128-byte-swizzled MMA operands");
static_assert(offsetof(AttnSmem, kc) % 16 == 0 && offsetof(AttnSmem, ksc) % 16 == 0 &&
                  offsetof(AttnSmem, vsc) % 16 == 0 && kHeadScaleBytes % 16 == 0,
              "bulk copies need 16-byte alignment");
static_assert(offsetof(AttnSmem, raw_full) % 8 == 0, "mbarriers");

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
  const uint2 L0 = lds_u2(lut_t + ((s2 & 0x7Fu) << 7)), L1 = lds_u2(lut_t + (((s2 >> 8) & 0x7Fu) << 7));
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
  const uint2 L0 = lds_u2(lut_t + ((s2 & 0x7Fu) << 7)), L1 = lds_u2(lut_t + (((s2 >> 8) & 0x7Fu) << 7));
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

}  // namespace

__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem_al = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // swizzled tiles: 1 KB
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_al);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.y, b = pair / kGroups, g = pair % kGroups;

  for (int u = tid; u < 128 * kLutCopies; u += kAttnThreads)
    sm.lut[u] = lut_magnitudes(static_cast<uint32_t>(u / kLutCopies));
  if (tid == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(smem_u32(&sm.raw_full[s]), 1);
      mbar_init(smem_u32(&sm.raw_empty[s]), kDqWarps);
    }
    for (int t = 0; t < kTileBufs; ++t) {
      mbar_init(smem_u32(&sm.ktile_full[t]), kDqWarps / 2);  // the K-row warps
      mbar_init(smem_u32(&sm.vtile_full[t]), kDqWarps / 2);  // the V-row warps
      mbar_init(smem_u32(&sm.tile_free[t]), 1);
    }
    for (int t = 0; t < kSBufs; ++t) {
      mbar_init(smem_u32(&sm.s_full[t]), 1);
      mbar_init(smem_u32(&sm.s_free[t]), kSoftWarps);
      mbar_init(smem_u32(&sm.p_full[t]), kSoftWarps);
      mbar_init(smem_u32(&sm.p_free[t]), 1);
    }
    mbar_init(smem_u32(&sm.o_done), 1);
    mbar_init(smem_u32(&sm.o_final), 1);
    mbar_fence_init();
    sm.soft_dead = 0;
  }

  // the request's geometry and query tile are inputs: read them before waiting on the
  // preceding kernel, which produces the block ids
  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows && kQPerKV * R <= p.max_m;
  if (!ok) {
    if (tid == 0 && blockIdx.x == 0 && g == 0) set_flag(p.flags, kFlagBadLength);
    return;
  }
  if (R == 0) return;
  const int nb = (N + kBlock - 1) / kBlock;
  const int M = kQPerKV * R;  // query rows of this (request, group): row m = speculative row m/8, head m%8
  // query tile: 128 rows x 128 bytes, 128-byte swizzle; row 64 + m repeats row m, and
  // rows m >= M (and 64 + m) are zero
  for (int u = tid; u < 128 * 8; u += kAttnThreads) {
    const int m = u >> 3, ch = u & 7, mq = m & 63;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (mq < M)
      v = *reinterpret_cast<const uint4*>(
          p.q + ((static_cast<long long>(r0 + mq / kQPerKV) * kHeads) + kQPerKV * g + mq % kQPerKV) * kDim + ch * 16);
    *reinterpret_cast<uint4*>(sm.qtile + m * 128 + ((ch ^ (m & 7)) << 4)) = v;
  }

  // the request's block-table row (an input) staged before the wait in the third K tile,
  // unused until block 2 is dequantised, so the selected pages resolve from shared memory;
  // the tensor memory too is taken before the wait (the SM's previous CTA, whose shared
  // memory this CTA needed, has exited)
  const bool bt_staged = nb <= static_cast<int>(kTileBytes / 4);
  int32_t* bt = reinterpret_cast<int32_t*>(sm.ktile[2]);
  if (bt_staged)
    for (int c = tid; c < nb; c += kAttnThreads) bt[c] = p.block_table[static_cast<long long>(b) * p.max_pages + c];
  if (warp == kMmaWarp) tmem_alloc(smem_u32(&sm.taddr), kTmemCols);
  __syncthreads();

  pdl_wait_primary();  // the block ids come from the selection

  if (warp == 0) {
    // the 16 ids in parallel; the valid ones keep their order (ballot ranks)
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
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.taddr;
  const int jb0 = blockIdx.x * p.blocks_per_split;
  int nmy = sm.nsel - jb0;
  nmy = nmy < 0 ? 0 : (nmy > p.blocks_per_split ? p.blocks_per_split : nmy);

  if (warp == kLoadWarp) {
    // ================= load warp: raw K/V pages of block j into stage j % kAttnStages
    if (lane == 0) {
      auto issue = [&](int j) {
        const int st = j % kAttnStages;
        const int phys = sm.phys[jb0 + j];
        const uint32_t bar = smem_u32(&sm.raw_full[st]);
        const bool bad = phys < 0 || phys >= p.num_pages;
        sm.stage_bad[st] = bad ? 1 : 0;
        if (bad) {
          set_flag(p.flags, kFlagBadPage);
          mbar_arrive(bar);
          return;
        }
        const long long head_row = (static_cast<long long>(phys) * kGroups + g) * kBlock;
        mbar_arrive_expect_tx(bar, 2 * (kHeadPageBytes + kHeadScaleBytes));
        bulk_load(smem_u32(sm.kc[st]), p.k_data + head_row * 64, kHeadPageBytes, bar);
        bulk_load(smem_u32(sm.ksc[st]), p.k_scale + head_row * 8, kHeadScaleBytes, bar);
        bulk_load(smem_u32(sm.vc[st]), p.v_data + head_row * 64, kHeadPageBytes, bar);
        bulk_load(smem_u32(sm.vsc[st]), p.v_scale + head_row * 8, kHeadScaleBytes, bar);
      };
      for (int j = 0; j < nmy && j < kAttnStages; ++j) issue(j);
      for (int j = kAttnStages; j < nmy; ++j) {
        const int st = j % kAttnStages;
        if (!wait_bar(smem_u32(&sm.raw_empty[st]), ((j / kAttnStages) - 1) & 1, p.flags)) break;
        issue(j);
      }
    }
    __syncwarp();
  } else if (warp >= kDqWarp0) {
    // ================= dequant warps: thread t = row t & 127 of K or of V. A V row costs
    // about twice a K row (its E4M3 values are widened to FP16), so the two halves of the
    // warps swap K and V every block: a half that finishes block j's K rows early goes on
    // to block j + 1's V rows
    const int t = tid - kDqWarp0 * 32;
    const int r = t & (kBlock - 1), r7 = r & 7;
    // chunk order k = c ^ h((r >> 1) & 3), h = multiplication by a generator of GF(4)
    // (0,1,2,3 -> 0,2,3,1): both h and x ^ h(x) are permutations, so the 8 rows of a
    // shared-memory wavefront hit 8 different 16-byte bank groups on the 64-byte code
    // reads (slot (r & 1) * 4 + k) and on the tile writes (slot 2k ^ (r & 7))
    const int h = (0x78 >> (2 * ((r >> 1) & 3))) & 3;
    const uint32_t lut_t = smem_u32(sm.lut) + static_cast<uint32_t>(lane % kLutCopies) * 8u;
    for (int j = 0; j < nmy; ++j) {
      const int st = j % kAttnStages, buf = j % kTileBufs;
      if (!wait_bar(smem_u32(&sm.raw_full[st]), (j / kAttnStages) & 1, p.flags)) break;
      const bool is_v = (t >= kBlock) != ((j & 1) != 0);
      // the row's codes and scales go to registers and the stage back to the load warp at
      // once, so the copy of block j + kAttnStages overlaps this block's dequantisation
      const bool bad = sm.stage_bad[st] != 0;
      const uint8_t* row = (is_v ? sm.vc[st] : sm.kc[st]) + r * 64;
      const uint2 sc = *reinterpret_cast<const uint2*>((is_v ? sm.vsc[st] : sm.ksc[st]) + r * 8);
      uint4 v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c] = *reinterpret_cast<const uint4*>(row + ((c ^ h) << 4));
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.raw_empty[st]));
      if (j >= kTileBufs && !wait_bar(smem_u32(&sm.tile_free[buf]), ((j / kTileBufs) - 1) & 1, p.flags)) break;
      const int pos0 = sm.ids[jb0 + j] * kBlock;
      const int nvalid = N - pos0 < kBlock ? N - pos0 : kBlock;
      const uint32_t row_addr = smem_u32(is_v ? sm.vtile[buf][0] : sm.ktile[buf]) + static_cast<uint32_t>(r) * 128u;
      // a bad page reads as zeros; V rows past the context are zero (their weights are
      // 0, and 0 x NaN from unwritten slots must not reach P V)
      if (bad || (is_v && r >= nvalid)) {
#pragma unroll
        for (int c = 0; c < 8; ++c) st_shared_v4(row_addr + (c << 4), 0u, 0u, 0u, 0u);
        if (is_v)
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_v4(row_addr + kVHalfBytes + (c << 4), 0u, 0u, 0u, 0u);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int k = c ^ h;
          const uint32_t s2 = ((k & 2) ? sc.y : sc.x) >> ((k & 1) * 16);
          if (is_v)
            dq_chunk_v(lut_t, v[c], s2, row_addr, r7, k);
          else
            dq_chunk(lut_t, v[c], s2, row_addr, r7, k);
        }
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the MMA (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(is_v ? &sm.vtile_full[buf] : &sm.ktile_full[buf]));
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA warp: S_j = Q K_j^T and O += P_j V_j, each issued as soon as
    // its inputs are ready (S_{j+1} does not wait behind P_j V_j or the reverse), except
    // that S_j follows P_{j-2} V_{j-2}: both wait for the same softmax arrival, and this
    // order makes S_j's completion imply that P_{j-2} V_{j-2} is done, which the softmax
    // warps' waits on o_done and on P buffer j % 2 rely on
    if (lane == 0) {
      const uint64_t qdesc = sdesc_kmajor_sw128(smem_u32(sm.qtile));
      const uint32_t id_qk = idesc_e4m3_f32(128, kBlock, false, false);
      const uint32_t id_pv = idesc_f16_f32(128, kDim, true);
      int nq = 0, np = 0;  // next block for S, next block for P V
      long long t_last = global_ns();
      while (np < nmy) {
        bool did = false;
        if (nq < nmy && np + 1 >= nq) {
          const int tb = nq % kTileBufs, sb = nq % kSBufs;
          if (mbar_test(smem_u32(&sm.ktile_full[tb]), (nq / kTileBufs) & 1) &&
              (nq < kSBufs || mbar_test(smem_u32(&sm.s_free[sb]), ((nq / kSBufs) - 1) & 1))) {
            tc_fence_after();
            // K step kk of an operand: +32 bytes along K-major rows (+2 in the address field)
            const uint64_t kdesc = sdesc_kmajor_sw128(smem_u32(sm.ktile[tb]));
#pragma unroll
            for (int kk = 0; kk < kDim / 32; ++kk)
              mma_f8_ss(tbase + kColS + kBlock * sb, qdesc + 2 * kk, kdesc + 2 * kk, id_qk, kk > 0);
            mma_commit(smem_u32(&sm.s_full[sb]));
            ++nq;
            did = true;
          }
        }
        if (np < nq) {
          const int tb = np % kTileBufs, sb = np % kSBufs;
          if (mbar_test(smem_u32(&sm.p_full[sb]), (np / kSBufs) & 1) &&
              mbar_test(smem_u32(&sm.vtile_full[tb]), (np / kTileBufs) & 1)) {
            tc_fence_after();
            // MN-major V: 128 dims = two 128-byte swizzle atoms (the two halves, kVHalfBytes
            // apart: the leading-dimension offset), 8-key groups 1 KB apart (the stride
            // offset); K step kk = 16 keys = 2048 bytes (+128 in the field); A = P, 8 columns
            const uint64_t vdesc = sdesc_mn_sw128(smem_u32(sm.vtile[tb][0]), kVHalfBytes);
#pragma unroll
            for (int kk = 0; kk < kBlock / 16; ++kk)
              mma_f16_tmemA(tbase + kColO, tbase + kColP + 64 * sb + 8 * kk, vdesc + 128 * kk, id_pv,
                            (np > 0 || kk > 0) ? 1u : 0u);
            mma_commit(smem_u32(&sm.o_done));
            mma_commit(smem_u32(&sm.tile_free[tb]));
            mma_commit(smem_u32(&sm.p_free[sb]));
            ++np;
            if (np == nmy) mma_commit(smem_u32(&sm.o_final));  // single phase: O is complete
            did = true;
          }
        }
        const long long now = global_ns();
        if (did) {
          t_last = now;
        } else if (now - t_last > kWaitLimitNs) {
          set_flag(p.flags, kFlagTimeout);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ================= softmax warps: warp q reads TMEM lanes 32q .. 32q + 31, which hold
    // query row m = 32 (q & 1) + lane, and takes keys 64 hf .. 64 hf + 63 of every block,
    // hf = q >> 1. Its lanes' O sums this key half only (the P columns of the other half
    // stay zero there), with its own reference max and running sum; the two halves of a
    // row are combined once, at the end.
    const int q = warp, hf = q >> 1;
    const int m = 32 * (q & 1) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int rq = m / kQPerKV;
    const int pos_max = N - R + rq;  // this row sees key positions <= pos_max
    const float c = p.sm_scale_log2;
    float mref = -INFINITY, lrun = 0.f;  // reference max (log2 domain) and running sum
    bool good = true;
    {
      uint32_t z[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) z[u] = 0u;
#pragma unroll
      for (int bb = 0; bb < kSBufs; ++bb) tmem_st32(tbase + lane_base + kColP + 64 * bb + 32 * (hf ^ 1), z);
      tc_wait_st();
    }
    for (int j = 0; j < nmy; ++j) {
      const int bb = j % kSBufs;
      const int pos0 = sm.ids[jb0 + j] * kBlock;
      const bool full_vis = pos0 + kBlock - 1 <= N - R;  // every key visible to every row
      const int lim = pos_max - pos0 - 64 * hf;           // key 64 hf + n visible iff n <= lim
      good = __all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.s_full[bb]), (j / kSBufs) & 1, p.flags));
      if (!good) break;
      tc_fence_after();
      float sv[64];
      {
        const uint32_t s_addr = tbase + lane_base + kColS + kBlock * bb + 64 * hf;
        uint32_t v0[32], v1[32];
        tmem_ld32(s_addr, v0);
        tmem_ld32(s_addr + 32, v1);
        tc_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          sv[u] = __uint_as_float(v0[u]);
          sv[32 + u] = __uint_as_float(v1[u]);
        }
      }
      if (!full_vis)
#pragma unroll
        for (int u = 0; u < 64; ++u) sv[u] = u <= lim ? sv[u] : -INFINITY;
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 64; u += 2) mx = fmaxf(mx, fmaxf(sv[u], sv[u + 1]));
      // Lazy rescale: P is taken relative to a reference max mref that moves only
      // when this block's max exceeds it by more than kRescaleLog2 (P then stays
      // below 2^kRescaleLog2, well inside FP16); O / l is exact whatever mref is.
      const float bmax = mx * c;  // c > 0 keeps the order of the raw scores
      const bool move = bmax > mref + kRescaleLog2 || (mref == -INFINITY && bmax != -INFINITY);
      const float m_new = move ? bmax : mref;
      const float ref = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(mref - ref);  // 0 while nothing was seen yet
      const bool rescale = move && mref != -INFINITY;
      if (j >= 1 && __any_sync(0xFFFFFFFFu, rescale)) {
        // O must hold every earlier block before it is rescaled (S_j's completion already
        // implies P_{j-2} V_{j-2}, so the phase awaited here is P_{j-1} V_{j-1}'s)
        if (!__all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.o_done), (j - 1) & 1, p.flags))) {
          good = false;
          break;
        }
        tc_fence_after();
        const float a = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int qc = 0; qc < 4; ++qc) {  // one 32-column chunk live at a time
          uint32_t v[32];
          const uint32_t o_addr = tbase + lane_base + kColO + 32 * qc;
          tmem_ld32(o_addr, v);
          tc_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) * a);
          tmem_st32(o_addr, v);
        }
      } else if (j >= kSBufs) {
        // this P buffer's previous P V (block j - 2) must have finished reading it
        if (!__all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.p_free[bb]), ((j / kSBufs) - 1) & 1, p.flags))) {
          good = false;
          break;
        }
        tc_fence_after();
      }
      // P = exp2(s c - ref) for this half's 64 keys, FP16 pairs (2 keys per TMEM column)
      uint32_t pw[32];
      uint32_t hsum = 0u;  // f16x2 partial sums
#pragma unroll
      for (int u2 = 0; u2 < 32; ++u2) {
        const float d0 = fmaf(sv[2 * u2], c, -ref), d1 = fmaf(sv[2 * u2 + 1], c, -ref);
        uint32_t hx, hp;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hx) : "f"(d1), "f"(d0));
        asm("ex2.approx.f16x2 %0, %1;" : "=r"(hp) : "r"(hx));
        asm("add.rn.f16x2 %0, %0, %1;" : "+r"(hsum) : "r"(hp));
        pw[u2] = hp;
      }
      tmem_st32(tbase + lane_base + kColP + 64 * bb + 32 * hf, pw);
      {
        float2 f;
        asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
            : "=f"(f.x), "=f"(f.y)
            : "r"(hsum));
        lrun = lrun * alpha + (f.x + f.y);
      }
      mref = m_new;
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.s_free[bb]));
        mbar_arrive(smem_u32(&sm.p_full[bb]));
      }
    }
    // ---- output: row m's two key halves (lanes m and 64 + m, warps q and q ^ 2) combined
    // with the log-sum-exp rule; warp q writes dims 64 hf .. 64 hf + 63, taking the other
    // warp's weighted O for those dims through shared memory (the K tiles, free once O is
    // complete)
    const bool fin = good && nmy > 0 &&
                     __all_sync(0xFFFFFFFFu, wait_bar(smem_u32(&sm.o_final), 0, p.flags));
    sm.xmax[hf][m] = mref;
    sm.xsum[hf][m] = lrun;
    if (!fin) sm.soft_dead = 1;
    named_bar_sync(1, kSoftWarps * 32);
    if (sm.soft_dead == 0) {
      tc_fence_after();
      const float mo = sm.xmax[hf ^ 1][m], lo = sm.xsum[hf ^ 1][m];
      const float mt = fmaxf(mref, mo);
      const float ref = mt == -INFINITY ? 0.f : mt;
      const float es = exp2f(mref - ref), eo = exp2f(mo - ref);
      const float l = lrun * es + lo * eo;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float ws = es * inv;  // weight of this half's O
      const float lse2 = l > 0.f ? ref + log2f(l) : -INFINITY;
      static_assert(kSoftWarps * 32 * 64 * sizeof(float) <= 2 * kTileBytes, "exchange fits two K tiles");
      // lane row of 64 floats, 16-byte chunk ch at slot (ch + lane) % 16: conflict-free
      float* xrow = reinterpret_cast<float*>(sm.ktile[0]) + (q * 32 + lane) * 64;
#pragma unroll
      for (int qc = 0; qc < 2; ++qc) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + kColO + 64 * (hf ^ 1) + 32 * qc, v);
        tc_wait_ld();
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4)
          *reinterpret_cast<float4*>(xrow + 4 * ((8 * qc + u4 + lane) & 15)) =
              make_float4(__uint_as_float(v[4 * u4]) * ws, __uint_as_float(v[4 * u4 + 1]) * ws,
                          __uint_as_float(v[4 * u4 + 2]) * ws, __uint_as_float(v[4 * u4 + 3]) * ws);
      }
      named_bar_sync(1, kSoftWarps * 32);
      const float* xo = reinterpret_cast<const float*>(sm.ktile[0]) + ((q ^ 2) * 32 + lane) * 64;
      const int hh = m % kQPerKV;
      // the finished O rows (FP32), staged in the V tiles (free once O is complete)
      static_assert(64 * kDim * sizeof(float) <= 2 * kVHalfBytes, "staging fits one V tile buffer");
      float* stage = reinterpret_cast<float*>(sm.vtile[0][0]);
#pragma unroll
      for (int qc = 0; qc < 2; ++qc) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + kColO + 64 * hf + 32 * qc, v);
        tc_wait_ld();
        float o[32];
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4) {
          const float4 x = *reinterpret_cast<const float4*>(xo + 4 * ((8 * qc + u4 + lane) & 15));
          o[4 * u4] = fmaf(__uint_as_float(v[4 * u4]), ws, x.x);
          o[4 * u4 + 1] = fmaf(__uint_as_float(v[4 * u4 + 1]), ws, x.y);
          o[4 * u4 + 2] = fmaf(__uint_as_float(v[4 * u4 + 2]), ws, x.z);
          o[4 * u4 + 3] = fmaf(__uint_as_float(v[4 * u4 + 3]), ws, x.w);
        }
        // combined row m, dims 64 hf + 32 qc .. + 31 (16-byte chunks 16 hf + 8 qc + u4) into the
        // staging rows; chunk c of row m sits at c ^ (m & 7), so 8 rows hit 8 bank groups
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4)
          *reinterpret_cast<float4*>(stage + m * kDim + 4 * ((16 * hf + 8 * qc + u4) ^ (m & 7))) =
              make_float4(o[4 * u4], o[4 * u4 + 1], o[4 * u4 + 2], o[4 * u4 + 3]);
      }
      named_bar_sync(1, kSoftWarps * 32);
      // coalesced copy-out by the 128 softmax threads: consecutive threads, consecutive
      // 16-byte pieces of an output row
      const int ct = q * 32 + lane;
      if (p.splits == 1) {
        for (int it = ct; it < M * (kDim / 8); it += kSoftWarps * 32) {
          const int mm = it / (kDim / 8), c8 = it % (kDim / 8);  // 8 dims: chunks 2 c8, 2 c8 + 1
          const float4 a = *reinterpret_cast<const float4*>(stage + mm * kDim + 4 * ((2 * c8) ^ (mm & 7)));
          const float4 b = *reinterpret_cast<const float4*>(stage + mm * kDim + 4 * ((2 * c8 + 1) ^ (mm & 7)));
          const long long orow = (static_cast<long long>(r0 + mm / kQPerKV) * kHeads) + kQPerKV * g + mm % kQPerKV;
          *reinterpret_cast<uint4*>(p.out + orow * kDim + 8 * c8) =
              make_uint4(bf16x2_bits(a.x, a.y), bf16x2_bits(a.z, a.w), bf16x2_bits(b.x, b.y), bf16x2_bits(b.z, b.w));
        }
      } else {
        const long long base = (static_cast<long long>(blockIdx.x) * p.num_reqs * kGroups + pair) * p.max_m;
        for (int it = ct; it < M * (kDim / 4); it += kSoftWarps * 32) {
          const int mm = it / (kDim / 4), c = it % (kDim / 4);
          *reinterpret_cast<float4*>(p.part_o + (base + mm) * kDim + 4 * c) =
              *reinterpret_cast<const float4*>(stage + mm * kDim + 4 * (c ^ (mm & 7)));
        }
      }
      if (m < M && hf == 0) {
        if (p.splits == 1) {
          if (p.lse != nullptr)
            p.lse[(static_cast<long long>(r0 + rq) * kHeads) + kQPerKV * g + hh] = lse2 * 0.69314718055994531f;
        } else {
          p.part_lse2[(static_cast<long long>(blockIdx.x) * p.num_reqs * kGroups + pair) * p.max_m + m] = lse2;
        }
      }
    }
  }

  // ---- teardown (a CTA that wrote partials makes them visible before it counts itself in)
  if (p.splits > 1) __threadfence();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }

  if (p.splits == 1) return;
  // ---- last CTA of this (request, group) merges the splits' partials
  if (tid == 0) {
    const unsigned old = atomicAdd(p.pair_cnt + pair, 1u);
    sm.last = old + 1 == static_cast<unsigned>(p.splits);
    if (sm.last) p.pair_cnt[pair] = 0u;
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  const int nsplit_used = (sm.nsel + p.blocks_per_split - 1) / p.blocks_per_split;
  const long long stride = static_cast<long long>(p.num_reqs) * kGroups * p.max_m;
  // out[row][4 dims] = sum over splits s of exp2(lse2_s - lse2) x o_s, lse2 = log2 sum_s exp2(lse2_s),
  // taken two splits at a time with a running maximum. A thread issues the loads of all its
  // items (partials and their rows' lse2) before it uses any, so a merge of up to two splits
  // is one round trip to L2.
  constexpr int kItems = 5;
  const int nitems = M * (kDim / 4);
  for (int idx0 = tid; idx0 < nitems; idx0 += kAttnThreads * kItems) {
    float4 acc[kItems];
    float mx[kItems], den[kItems];
#pragma unroll
    for (int t = 0; t < kItems; ++t) {
      acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      mx[t] = -INFINITY;
      den[t] = 0.f;
    }
    for (int s0 = 0; s0 < nsplit_used; s0 += 2) {
      float4 v[2][kItems];
      float l2[2][kItems];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < kItems; ++t) {
          const int idx = idx0 + t * kAttnThreads, s = s0 + h;
          const int mrow = idx / (kDim / 4), d4 = idx % (kDim / 4);
          const long long base = s * stride + static_cast<long long>(pair) * p.max_m + mrow;
          const bool ok = idx < nitems && s < nsplit_used;
          v[h][t] = ok ? __ldcg(reinterpret_cast<const float4*>(p.part_o + base * kDim) + d4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          l2[h][t] = ok ? __ldcg(p.part_lse2 + base) : -INFINITY;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < kItems; ++t) {
          const float nm = fmaxf(mx[t], l2[h][t]);
          const float ref = nm == -INFINITY ? 0.f : nm;
          const float a = exp2f(mx[t] - ref), w = exp2f(l2[h][t] - ref);
          acc[t].x = acc[t].x * a + w * v[h][t].x;
          acc[t].y = acc[t].y * a + w * v[h][t].y;
          acc[t].z = acc[t].z * a + w * v[h][t].z;
          acc[t].w = acc[t].w * a + w * v[h][t].w;
          den[t] = den[t] * a + w;
          mx[t] = nm;
        }
    }
#pragma unroll
    for (int t = 0; t < kItems; ++t) {
      const int idx = idx0 + t * kAttnThreads;
      if (idx < nitems) {
        const int mrow = idx / (kDim / 4), d4 = idx % (kDim / 4);
        const int rq = mrow / kQPerKV, hh = mrow % kQPerKV;
        const long long orow = (static_cast<long long>(r0 + rq) * kHeads) + kQPerKV * g + hh;
        const float inv = den[t] > 0.f ? 1.f / den[t] : 0.f;
        const uint2 packed = make_uint2(bf16x2_bits(acc[t].x * inv, acc[t].y * inv),
                                        bf16x2_bits(acc[t].z * inv, acc[t].w * inv));
        *reinterpret_cast<uint2*>(p.out + orow * kDim + 4 * d4) = packed;
        if (d4 == 0 && p.lse != nullptr)
          p.lse[orow] = den[t] > 0.f ? (mx[t] + log2f(den[t])) * 0.69314718055994531f : -INFINITY;
      }
    }
  }
}

size_t attn_smem_bytes() { return sizeof(AttnSmem) + 1024; }

cudaError_t launch_attn(const AttnParams& prm, bool pdl, cudaStream_t st) {
  const size_t smem = attn_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.splits, prm.num_reqs * kGroups, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, attn_kernel, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
