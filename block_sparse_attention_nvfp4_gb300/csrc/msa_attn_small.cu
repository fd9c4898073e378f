// Step 4 of the MSA decode path for (request, group) pairs with few query rows: exact
// softmax attention over the selected blocks' NVFP4 K/V, with warp-level MMAs.
//
// [vLLM-zh "How MiniMax sparse attention works"] main attention runs exactly on the 16
// selected blocks; [MSA-fig §1, sparse branch] every query head of a group uses the group's
// blocks; [vLLM-zh, Blackwell kernels] K/V are NVFP4, turned into FP8 in the kernel.
//
// When a group has M = 8R <= 16 query rows (R <= 2 speculative rows), a 128-row tcgen05 tile
// would be at most an eighth real, and the tile's round trips through tensor memory (S,
// softmax, P, P V) set the pace, not the arithmetic. This kernel instead keeps the group's
// rows in one 16-row warp-MMA tile:
//   * one CTA per (request, group), 8 warps; a thread of the first half
//     dequantises one K row (key) of the block to E4M3, one of the second half one V row to
//     FP16 (both exact: the E4M3 value of E2M1 x scale, rounded as the index scan does),
//     into 16-byte-chunk-swizzled tiles; the raw pages come by tensor copies (codes, 64-byte
//     swizzle) and bulk copies (scales) into a 4-stage ring, block j + 4 requested as soon
//     as block j's rows are read, every later block asked into L2 once the ids are known;
//   * warp w takes keys 16w .. 16w + 15 of every block: S = Q K^T by mma.m16n8k32 (E4M3 x
//     E4M3 -> FP32, the query fragments held in registers for the whole kernel), an online
//     softmax of its own over those keys (FP32), P in FP16 (reading 17) times V by
//     mma.m16n8k16 (FP32 accumulation) with V fragments from ldmatrix.trans;
//   * at the end the 8 warps' (O, max, sum) of each row are merged with the log-sum-exp
//     rule through shared memory and written as BF16 output and lse.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr int kSmDqWarps = 8;                           // warps 0..7: dequant, one K or V row per thread
constexpr int kSmMmWarps = 8;                           // warps 8..15: MMA and softmax, 16 keys each
constexpr int kSmThreads = 32 * (kSmDqWarps + kSmMmWarps);
constexpr int kSmStages = 4;
constexpr int kSmRows = 16;                             // query rows of the warp-MMA tile
constexpr uint32_t kSmHeadBytes = kBlock * 64;          // codes of one (page, KV head)
constexpr uint32_t kSmHeadScale = kBlock * 8;
constexpr int kSmLutCopies = 8;
constexpr int kSmLutShift = 6;                          // bytes per table entry (all copies)
static_assert(kSmMmWarps * 16 == kBlock && kSmDqWarps * 32 == 2 * kBlock, "warp roles");

struct SmallSmem {
  uint8_t kc[kSmStages][kSmHeadBytes];  // raw codes, 1024-aligned tensor-copy destinations
  uint8_t vc[kSmStages][kSmHeadBytes];
  uint8_t ktile[2][kBlock * kDim];      // K, E4M3 [key][128 B], 16-byte chunk c at c ^ (key & 7)
  uint8_t vtile[2][kBlock * kDim * 2];  // V, FP16 [key][256 B], 16-byte chunk c at c ^ (key & 7)
  uint8_t ksc[kSmStages][kSmHeadScale];
  uint8_t vsc[kSmStages][kSmHeadScale];
  uint2 lut[128 * kSmLutCopies];        // scaled magnitudes, entry e of copy c at 8 (8 e + c) bytes
  uint8_t qtile[kSmRows * kDim];        // the group's query rows (zero past M), chunk c at c ^ (row & 7)
  int32_t ids[kTopK];
  int32_t phys[kTopK];
  int nsel;
  uint64_t full[kSmStages];
  uint64_t tfull[2], tfree[2];          // tile j % 2: dequantised / consumed by the MMA warps
};
// the end-of-kernel merge reuses the raw codes and the tiles
constexpr uint32_t kMergeO = kSmMmWarps * kSmRows * kDim * 4;  // per MMA warp O [16 rows][128]
static_assert(kMergeO + 2 * kSmMmWarps * kSmRows * 4 <= offsetof(SmallSmem, ksc), "merge scratch");
static_assert(offsetof(SmallSmem, kc) % 1024 == 0 && offsetof(SmallSmem, vc) % 1024 == 0, "swizzled copies");
static_assert(offsetof(SmallSmem, ksc) % 16 == 0 && offsetof(SmallSmem, vsc) % 16 == 0, "bulk copies");

// 32 E4M3 values of code chunk k (16 bytes, groups 2k and 2k + 1 with scale bytes s2 and
// s2 >> 8) into 8 words (elements 32k .. 32k + 31 in order).
__device__ __forceinline__ void dq_chunk_regs(uint32_t lut_t, const uint4& v, uint32_t s2, uint32_t (&o)[8]) {
  const uint2 L0 = lds_u2(lut_t + ((s2 & 0x7Fu) << kSmLutShift));
  const uint2 L1 = lds_u2(lut_t + (((s2 >> 8) & 0x7Fu) << kSmLutShift));
  dq8_signed(v.x, L0.x, L0.y, o[0], o[1]);
  dq8_signed(v.y, L0.x, L0.y, o[2], o[3]);
  dq8_signed(v.z, L1.x, L1.y, o[4], o[5]);
  dq8_signed(v.w, L1.x, L1.y, o[6], o[7]);
}

__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two) {
  uint32_t h;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "r"(two));
  return h;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity, uint32_t* flags) {
  return mbar_try(bar, parity) || mbar_wait(bar, parity, flags);
}

// AND of v over the nthreads threads of named barrier id (itself a barrier).
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace

__global__ void __launch_bounds__(kSmThreads, 1)
    attn_small_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem_al = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  SmallSmem& sm = *reinterpret_cast<SmallSmem*>(smem_al);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / kGroups, g = blockIdx.x % kGroups;

  const int N = p.context_lens[b];
  const int r0 = p.q_indptr[b], R = p.q_indptr[b + 1] - r0;
  const bool ok = N >= 0 && N <= p.max_pages * kBlock && R >= 0 && R <= kMaxRows && R <= N && r0 >= 0 &&
                  r0 + R <= p.total_rows && kQPerKV * R <= kSmRows;
  if (!ok || R == 0) {
    if (!ok && tid == 0 && g == 0) set_flag(p.flags, kFlagBadLength);
    return;
  }
  const int nb = (N + kBlock - 1) / kBlock;
  const int M = kQPerKV * R;  // row m = speculative row m / 8, head m % 8 of the group

  for (int u = tid; u < 128 * kSmLutCopies; u += kSmThreads)
    sm.lut[u] = lut_magnitudes(static_cast<uint32_t>(u / kSmLutCopies));
  for (int u = tid; u < kSmRows * 8; u += kSmThreads) {
    const int row = u >> 3, c = u & 7;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < M)
      v = *reinterpret_cast<const uint4*>(
          p.q + ((static_cast<long long>(r0 + row / kQPerKV) * kHeads) + kQPerKV * g + row % kQPerKV) * kDim + 16 * c);
    *reinterpret_cast<uint4*>(sm.qtile + row * kDim + ((c ^ (row & 7)) << 4)) = v;
  }
  if (tid == 0) {
    for (int s = 0; s < kSmStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&sm.tfull[t]), kSmDqWarps);  // every dequant warp has written its rows
      mbar_init(smem_u32(&sm.tfree[t]), kSmMmWarps);  // every MMA warp is done with the tile
    }
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
  }
  __syncthreads();

  pdl_wait_primary();  // the block ids come from the selection

  if (warp == 0) {
    // the valid ids keep their order (ballot ranks); a page outside the cache is flagged and
    // its block left out
    const int id = lane < kTopK ? p.block_ids[(static_cast<long long>(b) * kGroups + g) * kTopK + lane] : -1;
    bool valid = lane < kTopK && id >= 0 && id < nb;
    if (lane < kTopK && !valid && id != -1) set_flag(p.flags, kFlagBadIds);  // outside the context
    int phys = -1;
    if (valid) {
      phys = p.block_table[static_cast<long long>(b) * p.max_pages + id];
      if (phys < 0 || phys >= p.num_pages) {
        set_flag(p.flags, kFlagBadPage);
        valid = false;
      }
    }
    const unsigned vm = __ballot_sync(0xFFFFFFFFu, valid);
    if (valid) {
      const int rank = __popc(vm & ((1u << lane) - 1u));
      sm.ids[rank] = id;
      sm.phys[rank] = phys;
    }
    if (lane == 0) sm.nsel = __popc(vm);
  }
  __syncthreads();
  const int nsel = sm.nsel;
  bool alive = true;

  if (warp < kSmDqWarps) {
    // ================= dequant warps: thread = K row tid (tid < 128) or V row tid - 128 of
    // block j, into tile j % 2; the raw ring is refilled by thread 0 once all rows are read
    auto issue = [&](int j) {
      const int st = j % kSmStages;
      const int head_row = (sm.phys[j] * kGroups + g) * kBlock;
      const uint32_t bar = smem_u32(&sm.full[st]);
      mbar_arrive_expect_tx(bar, 2 * (kSmHeadBytes + kSmHeadScale));
      tma_load_2d(smem_u32(sm.kc[st]), &kmap, 0, head_row, bar);
      tma_load_2d(smem_u32(sm.vc[st]), &vmap, 0, head_row, bar);
      bulk_load(smem_u32(sm.ksc[st]), p.k_scale + static_cast<long long>(head_row) * 8, kSmHeadScale, bar);
      bulk_load(smem_u32(sm.vsc[st]), p.v_scale + static_cast<long long>(head_row) * 8, kSmHeadScale, bar);
    };
    int issued = 0, done = 0;
    if (tid == 0) {
      for (; issued < nsel && issued < kSmStages; ++issued) issue(issued);
      // every later block into L2 now: its stage then fills from L2
      for (int j = kSmStages; j < nsel; ++j) {
        const long long head_row = (static_cast<long long>(sm.phys[j]) * kGroups + g) * kBlock;
        prefetch_l2(p.k_data + head_row * 64, kSmHeadBytes);
        prefetch_l2(p.v_data + head_row * 64, kSmHeadBytes);
        prefetch_l2(p.k_scale + head_row * 8, kSmHeadScale);
        prefetch_l2(p.v_scale + head_row * 8, kSmHeadScale);
      }
    }
    const uint32_t lut_t = smem_u32(sm.lut) + static_cast<uint32_t>(lane % kSmLutCopies) * 8u;
    const bool is_v = tid >= kBlock;
    const int r = tid & (kBlock - 1), r7 = r & 7, sw = (r >> 1) & 3;
    for (int j = 0; j < nsel; ++j) {
      const int st = j % kSmStages, tb = j % 2;
      // the block's raw pages have landed and the tile's previous block has been consumed;
      // one decision for all dequant warps (they meet at a named barrier below)
      bool okw = __all_sync(0xFFFFFFFFu, wait_full(smem_u32(&sm.full[st]), (j / kSmStages) & 1, p.flags)) != 0;
      if (okw && j >= 2)
        okw = __all_sync(0xFFFFFFFFu, wait_full(smem_u32(&sm.tfree[tb]), ((j / 2) - 1) & 1, p.flags)) != 0;
      uint4 cv[4];
      uint2 sc = make_uint2(0u, 0u);
      if (okw) {
        const uint32_t crow = smem_u32(is_v ? sm.vc[st] : sm.kc[st]) + static_cast<uint32_t>(r) * 64u;
        sc = lds_u2(smem_u32(is_v ? sm.vsc[st] : sm.ksc[st]) + static_cast<uint32_t>(r) * 8u);
#pragma unroll
        for (int c = 0; c < 4; ++c) cv[c] = lds_u4(crow + (static_cast<uint32_t>(c ^ sw) << 4));
      }
      // every dequant thread has its row's codes: the stage takes block j + kSmStages
      alive = named_bar_and(1, kSmDqWarps * 32, okw);
      if (!alive) break;
      done = j + 1;
      if (tid == 0 && issued < nsel) {
        fence_proxy_async_smem();
        issue(issued);
        ++issued;
      }
      const int pos0 = sm.ids[j] * kBlock;
      const int nvalid = N - pos0 < kBlock ? N - pos0 : kBlock;
      if (!is_v) {
        const uint32_t row = smem_u32(sm.ktile[tb]) + static_cast<uint32_t>(r) * 128u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t w8[8];
          dq_chunk_regs(lut_t, cv[k], ((k & 2) ? sc.y : sc.x) >> ((k & 1) * 16), w8);
          st_shared_v4(row + (static_cast<uint32_t>((2 * k) ^ r7) << 4), w8[0], w8[1], w8[2], w8[3]);
          st_shared_v4(row + (static_cast<uint32_t>((2 * k + 1) ^ r7) << 4), w8[4], w8[5], w8[6], w8[7]);
        }
      } else {
        // V rows past the context are zero: their weights are 0, and 0 x NaN from unwritten
        // slots must not reach P V
        const uint32_t row = smem_u32(sm.vtile[tb]) + static_cast<uint32_t>(r) * 256u;
        const bool live = r < nvalid;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t w8[8];
          dq_chunk_regs(lut_t, cv[k], ((k & 2) ? sc.y : sc.x) >> ((k & 1) * 16), w8);
          uint32_t h[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            h[2 * i] = live ? e4m3x2_to_h2(w8[i] & 0xFFFFu) : 0u;
            h[2 * i + 1] = live ? e4m3x2_to_h2(w8[i] >> 16) : 0u;
          }
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            st_shared_v4(row + (static_cast<uint32_t>((4 * k + cc) ^ r7) << 4), h[4 * cc], h[4 * cc + 1],
                         h[4 * cc + 2], h[4 * cc + 3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tfull[tb]));
    }
    // copies issued but never consumed (only after a timeout) complete before the CTA leaves
    if (tid == 0)
      for (int j = done; j < issued; ++j)
        if (!mbar_wait(smem_u32(&sm.full[j % kSmStages]), (j / kSmStages) & 1, p.flags)) break;
  }

  // ================= MMA warps: warp w takes keys 16w .. 16w + 15 of every block
  const int mw_ = warp - kSmDqWarps;
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment coordinates: row group, thread in group
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
  if (warp >= kSmDqWarps) {
    // query fragments of the m16n8k32 A operand (rows gq and gq + 8, bytes 32 ks + 4 tq .. +3 and
    // +16) are read from the query tile per K step
    const uint32_t qrow = smem_u32(sm.qtile) + static_cast<uint32_t>(gq) * kDim + 4u * tq;
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    const float c2 = p.sm_scale_log2;  // scores in log2 units
    // visibility of key position pos to rows gq and gq + 8: pos <= N - R + row / 8 (padding
    // rows m >= M see nothing)
    const int lim0 = gq < M ? N - R + gq / kQPerKV : -1;
    const int lim1 = gq + 8 < M ? N - R + (gq + 8) / kQPerKV : -1;
    for (int j = 0; j < nsel; ++j) {
      const int tb = j % 2;
      if (!__all_sync(0xFFFFFFFFu, wait_full(smem_u32(&sm.tfull[tb]), (j / 2) & 1, p.flags))) {
        alive = false;
        break;
      }
      const uint32_t ktile = smem_u32(sm.ktile[tb]), vtile = smem_u32(sm.vtile[tb]);
      const int pos0 = sm.ids[j] * kBlock;
      // ---- S = Q K^T over this warp's 16 keys
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t c0 = static_cast<uint32_t>((2 * ks) ^ (gq & 7)) << 4;
        const uint32_t c1 = static_cast<uint32_t>((2 * ks + 1) ^ (gq & 7)) << 4;
        const uint32_t qa[4] = {lds_u32(qrow + c0), lds_u32(qrow + 8 * kDim + c0), lds_u32(qrow + c1),
                                lds_u32(qrow + 8 * kDim + c1)};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int kr = 16 * mw_ + 8 * nt + gq;  // the key whose B fragment this thread holds
          const uint32_t krow = ktile + static_cast<uint32_t>(kr) * 128u + 4u * tq;
          const uint32_t b0 = lds_u32(krow + (static_cast<uint32_t>((2 * ks) ^ (kr & 7)) << 4));
          const uint32_t b1 = lds_u32(krow + (static_cast<uint32_t>((2 * ks + 1) ^ (kr & 7)) << 4));
          mma_e4m3_16832(s[nt], qa, b0, b1);
        }
      }
      // ---- mask (a select: scores of keys past the context may be NaN) and scale; block max
      float bm[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = pos0 + 16 * mw_ + 8 * nt + 2 * tq + (e & 1);
          const bool vis = pos <= ((e & 2) ? lim1 : lim0);
          s[nt][e] = vis ? s[nt][e] * c2 : -INFINITY;
          bm[e >> 1] = fmaxf(bm[e >> 1], s[nt][e]);
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        bm[h] = fmaxf(bm[h], __shfl_xor_sync(0xFFFFFFFFu, bm[h], 1));
        bm[h] = fmaxf(bm[h], __shfl_xor_sync(0xFFFFFFFFu, bm[h], 2));
      }
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float nm = fmaxf(m_run[h], bm[h]);
        alpha[h] = nm == m_run[h] ? 1.f : exp2f(m_run[h] - nm);  // m_run = -inf -> 0
        m_run[h] = nm;
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = s[nt][e] == -INFINITY ? 0.f : exp2f(s[nt][e] - m_run[e >> 1]);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        l_run[h] = l_run[h] * alpha[h] + s[0][2 * h] + s[0][2 * h + 1] + s[1][2 * h] + s[1][2 * h + 1];
      if (__any_sync(0xFFFFFFFFu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int jn = 0; jn < 16; ++jn) {
          o[jn][0] *= alpha[0];
          o[jn][1] *= alpha[0];
          o[jn][2] *= alpha[1];
          o[jn][3] *= alpha[1];
        }
      }
      // ---- O += P V over the warp's 16 keys (P in FP16, the A fragment straight from S's layout)
      const uint32_t pa[4] = {pack_h2(s[0][0], s[0][1]), pack_h2(s[0][2], s[0][3]), pack_h2(s[1][0], s[1][1]),
                              pack_h2(s[1][2], s[1][3])};
      {
        const int mat = lane >> 3, i = lane & 7;
        const int key = 16 * mw_ + 8 * (mat & 1) + i;
        const uint32_t vrow = vtile + static_cast<uint32_t>(key) * 256u;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int chunk = 2 * jj + (mat >> 1);
          uint32_t v0, v1, v2, v3;
          ldmatrix_x4_trans(vrow + (static_cast<uint32_t>(chunk ^ (key & 7)) << 4), v0, v1, v2, v3);
          mma_f16_16816(o[2 * jj], pa, v0, v1);
          mma_f16_16816(o[2 * jj + 1], pa, v2, v3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tfree[tb]));
    }
  }
  alive = __syncthreads_and(alive ? 1 : 0) != 0;  // every copy and tile is done with

  // ---- merge the 8 MMA warps' partials of each row (log-sum-exp), then BF16 output and lse
  float* ow = reinterpret_cast<float*>(smem_al);            // [warp][16 rows][128]
  float* mwv = reinterpret_cast<float*>(smem_al + kMergeO);  // [warp][16 rows]
  float* lw = mwv + kSmMmWarps * kSmRows;
  if (warp >= kSmDqWarps) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 2);
    }
    if (tq == 0) {
      mwv[mw_ * kSmRows + gq] = m_run[0];
      mwv[mw_ * kSmRows + gq + 8] = m_run[1];
      lw[mw_ * kSmRows + gq] = l_run[0];
      lw[mw_ * kSmRows + gq + 8] = l_run[1];
    }
#pragma unroll
    for (int jn = 0; jn < 16; ++jn) {
      const int d = 8 * jn + 2 * tq;
      *reinterpret_cast<float2*>(ow + (mw_ * kSmRows + gq) * kDim + d) = make_float2(o[jn][0], o[jn][1]);
      *reinterpret_cast<float2*>(ow + (mw_ * kSmRows + gq + 8) * kDim + d) = make_float2(o[jn][2], o[jn][3]);
    }
  }
  __syncthreads();
  if (!alive || warp < kSmDqWarps) return;
  const int t2 = tid - kSmDqWarps * 32;
  const int row = t2 >> 4, d0 = (t2 & 15) * 8;
  if (row >= M) return;
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kSmMmWarps; ++w) mx = fmaxf(mx, mwv[w * kSmRows + row]);
  float l = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kSmMmWarps; ++w) {
    const float mwr = mwv[w * kSmRows + row];
    const float sc = mwr == -INFINITY ? 0.f : exp2f(mwr - mx);
    l += lw[w * kSmRows + row] * sc;
    const float4 a = *reinterpret_cast<const float4*>(ow + (w * kSmRows + row) * kDim + d0);
    const float4 c = *reinterpret_cast<const float4*>(ow + (w * kSmRows + row) * kDim + d0 + 4);
    acc[0] += a.x * sc;
    acc[1] += a.y * sc;
    acc[2] += a.z * sc;
    acc[3] += a.w * sc;
    acc[4] += c.x * sc;
    acc[5] += c.y * sc;
    acc[6] += c.z * sc;
    acc[7] += c.w * sc;
  }
  const float inv = 1.f / l;
  const long long orow = static_cast<long long>(r0 + row / kQPerKV) * kHeads + kQPerKV * g + row % kQPerKV;
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    packed[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  *reinterpret_cast<uint4*>(p.out + orow * kDim + d0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  if (p.lse != nullptr && (t2 & 15) == 0) p.lse[orow] = (mx + log2f(l)) * 0.69314718055994531f;
}

size_t attn_small_smem_bytes() { return sizeof(SmallSmem) + 1024; }

cudaError_t launch_attn_small(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& prm, bool pdl,
                              cudaStream_t st) {
  const size_t smem = attn_small_smem_bytes();
  cudaError_t e =
      cudaFuncSetAttribute(attn_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_reqs * kGroups, 1, 1);
  cfg.blockDim = dim3(kSmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, attn_small_kernel, kmap, vmap, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
