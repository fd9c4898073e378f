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
// Design. Grid = (splits, request x group), one CTA per SM; a CTA takes
// `blocks_per_split` of the group's selected blocks (flash-decoding split over
// the selection), with warp roles so dequantisation and MMA overlap:
//   * 4 dequant warps: the raw NVFP4 pages arrive in a 4-stage ring by bulk async
//     copies; the warps dequantise each block's K (row-major FP8, k-step-
//     interleaved, bank-swizzled) and V (transposed: dim-major, 4 keys per word)
//     into one of two shared-memory tile buffers;
//   * 4 MMA warps, each owning 16 query rows (row = speculative row x head) and
//     a share of the block's keys: S = Q K^T with m16n8k32 FP8 MMA, FP32 online
//     softmax, P rounded to E4M3 (scaled by 256 so small weights keep precision)
//     feeding P V directly from the accumulator registers (the QK key order is
//     chosen so its output fragment is the next MMA's input fragment);
//   * MMA warps that split a block's keys merge through shared memory; CTAs that
//     split the selection write (o, lse) partials and the last one to arrive for
//     the (request, group) merges them with the exact log-sum-exp rule and
//     writes BF16 output.
// Measured on GB300, the earlier form (4 warps doing both, 2 CTAs per SM at 255
// registers) spent about 3 us dequantising and 3.5 us attending per block, one
// after the other, with each warp waiting on its own latencies.
#include <cuda_bf16.h>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr int kMathWarps = 4;   // warps 0..3: MMA + softmax
constexpr int kDqWarps = 4;     // warps 4..7: raw page copies + dequantisation
constexpr int kAttnThreads = (kMathWarps + kDqWarps) * 32;
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kAttnStages = 4;  // raw NVFP4 page ring
constexpr int kTileBufs = 2;    // dequantised K/V tiles
constexpr uint32_t kHeadPageBytes = kBlock * 64;      // codes of one (page, KV head)
constexpr uint32_t kHeadScaleBytes = kBlock * 8;

struct AttnSmem {
  uint2 lut[256];                             // magnitude bytes of E2M1 codes 0..7 per scale
  uint8_t kc[kAttnStages][kHeadPageBytes];
  uint8_t vc[kAttnStages][kHeadPageBytes];
  uint8_t ksc[kAttnStages][kHeadScaleBytes];
  uint8_t vsc[kAttnStages][kHeadScaleBytes];
  uint8_t khat[kTileBufs][kBlock * kDim];     // [key][128], k-step slots swizzled
  uint8_t vt[kTileBufs][kDim * kBlock];       // [dim][128 keys], key slots swizzled
  float comb_o[4][16][kDim];                  // key-split merge, then the split merge's weights
  float comb_ml[4][16][2];
  uint64_t full[kAttnStages], empty[kAttnStages];  // raw pages: copied / dequantised
  uint64_t tfull[kTileBufs], tempty[kTileBufs];    // tiles: dequantised / consumed
  int stage_bad[kAttnStages];
  int ids[kTopK];
  int phys[kTopK];                            // block-table entries of the selected blocks
  int nsel;
  int last;
};

__device__ __forceinline__ int khat_swz(int key) { return (key & 1) | ((key >> 1) & 2); }

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
  const __nv_bfloat16 x = __float2bfloat16_rn(a), y = __float2bfloat16_rn(b);
  return static_cast<uint32_t>(__bfloat16_as_ushort(x)) | (static_cast<uint32_t>(__bfloat16_as_ushort(y)) << 16);
}

// Dequantise block (stage st) into khat / vt. Keys at or past `nvalid` get V = 0
// (their weights are 0, and 0 * NaN from unwritten slots must not reach P V).
__device__ __forceinline__ void dequant_block(AttnSmem& sm, int st, int buf, int nvalid, bool bad) {
  const int tid = threadIdx.x - kMathWarps * 32;  // 0 .. kDqThreads-1
  // K: task = (key, 32-dim chunk) ; 8 consecutive threads read 128 contiguous bytes
  // (loops unrolled: the 4 tasks' loads and table lookups overlap)
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int u = it * kDqThreads + tid, key = u >> 2, ch = u & 3;
    uint32_t x[8];
    if (!bad) {
      const uint4 cw = *reinterpret_cast<const uint4*>(sm.kc[st] + key * 64 + ch * 16);
      const uint32_t sc = *reinterpret_cast<const uint16_t*>(sm.ksc[st] + key * 8 + 2 * ch);
      const uint2 L0 = sm.lut[sc & 0xFFu], L1 = sm.lut[sc >> 8];
      dq8_signed(cw.x, L0.x, L0.y, x[0], x[1]);
      dq8_signed(cw.y, L0.x, L0.y, x[2], x[3]);
      dq8_signed(cw.z, L1.x, L1.y, x[4], x[5]);
      dq8_signed(cw.w, L1.x, L1.y, x[6], x[7]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = 0u;
    }
    const int swz = ch ^ khat_swz(key);
    uint8_t* row = sm.khat[buf] + key * 128;
#pragma unroll
    for (int t = 0; t < 4; ++t) *reinterpret_cast<uint2*>(row + (swz * 4 + t) * 8) = make_uint2(x[t], x[t + 4]);
  }
  // V: task = (4-key quad, 8-dim code word) -> transposed words (4 keys of one dim)
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int u = it * kDqThreads + tid, q4 = u >> 4, wv = u & 15;
    uint32_t y[4][2];
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int key = 4 * q4 + k4;
      if (!bad && key < nvalid) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(sm.vc[st] + key * 64 + wv * 4);
        const uint2 L = sm.lut[sm.vsc[st][key * 8 + (wv >> 1)]];
        dq8_signed(w, L.x, L.y, y[k4][0], y[k4][1]);
      } else {
        y[k4][0] = 0u;
        y[k4][1] = 0u;
      }
    }
    const int kk = q4 >> 3, tpos = q4 & 7, t = tpos & 3, boff = (tpos >> 2) * 4;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t t0 = __byte_perm(y[0][h], y[1][h], 0x5140), t1 = __byte_perm(y[0][h], y[1][h], 0x7362);
      const uint32_t t2 = __byte_perm(y[2][h], y[3][h], 0x5140), t3 = __byte_perm(y[2][h], y[3][h], 0x7362);
      const uint32_t z[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632), __byte_perm(t1, t3, 0x5410),
                             __byte_perm(t1, t3, 0x7632)};
#pragma unroll
      for (int d4 = 0; d4 < 4; ++d4) {
        const int dim = 8 * wv + 4 * h + d4;
        *reinterpret_cast<uint32_t*>(sm.vt[buf] + dim * 128 + ((kk ^ (dim & 3)) * 4 + t) * 8 + boff) = z[d4];
      }
    }
  }
}

// Per-warp attention state for 16 query rows: A = row gq, B = row gq + 8.
struct WarpState {
  float o[16][4];
  float mA, mB, lA, lB;
};

// One block's keys [k0, k0 + 8*NT) for this warp's 16 rows.
template <int NT>
__device__ __forceinline__ void attend_keys(const uint8_t* khat, const uint8_t* vt, WarpState& ws,
                                            const uint32_t (&qa)[4][4], int k0, int blk_pos0, int posA, int posB,
                                            float scale_log2) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  float s[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
  // S = Q K^T ; n-tile j of 32-key group kg = k0/32 + j/4 holds keys chosen so the
  // accumulator layout equals the next MMA's A-operand layout
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int jl = j & 3;
    const int key = k0 + 32 * (j >> 2) + 16 * (jl >> 1) + 4 * (gq >> 1) + 2 * (jl & 1) + (gq & 1);
    const uint8_t* row = khat + key * 128;
    const int hsw = khat_swz(key);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint2 bv = *reinterpret_cast<const uint2*>(row + (((ks ^ hsw) * 4) + tq) * 8);
      mma_m16n8k32(s[j], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], bv.x, bv.y);
    }
  }
  // mask + scale, row max
  const bool need_mask = blk_pos0 + k0 + 8 * NT - 1 > (posA < posB ? posA : posB);
  float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int jl = j & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = k0 + 32 * (j >> 2) + 16 * (jl >> 1) + 4 * tq + 2 * (jl & 1) + e;
      const int pos = blk_pos0 + key;
      float a = s[j][e] * scale_log2, b = s[j][2 + e] * scale_log2;
      if (need_mask) {
        a = pos <= posA ? a : -INFINITY;
        b = pos <= posB ? b : -INFINITY;
      }
      s[j][e] = a;
      s[j][2 + e] = b;
      mxA = fmaxf(mxA, a);
      mxB = fmaxf(mxB, b);
    }
  }
  mxA = fmaxf(mxA, __shfl_xor_sync(0xFFFFFFFFu, mxA, 1));
  mxA = fmaxf(mxA, __shfl_xor_sync(0xFFFFFFFFu, mxA, 2));
  mxB = fmaxf(mxB, __shfl_xor_sync(0xFFFFFFFFu, mxB, 1));
  mxB = fmaxf(mxB, __shfl_xor_sync(0xFFFFFFFFu, mxB, 2));
  const float nA = fmaxf(ws.mA, mxA), nB = fmaxf(ws.mB, mxB);
  const float refA = nA == -INFINITY ? 0.f : nA, refB = nB == -INFINITY ? 0.f : nB;
  const float alA = exp2f(ws.mA - refA), alB = exp2f(ws.mB - refB);
  ws.mA = nA;
  ws.mB = nB;
  float sumA = 0.f, sumB = 0.f;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    s[j][0] = exp2f(s[j][0] - refA);
    s[j][1] = exp2f(s[j][1] - refA);
    s[j][2] = exp2f(s[j][2] - refB);
    s[j][3] = exp2f(s[j][3] - refB);
    sumA += s[j][0] + s[j][1];
    sumB += s[j][2] + s[j][3];
  }
  ws.lA = ws.lA * alA + sumA;
  ws.lB = ws.lB * alB + sumB;
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) {
    ws.o[nd][0] *= alA;
    ws.o[nd][1] *= alA;
    ws.o[nd][2] *= alB;
    ws.o[nd][3] *= alB;
  }
  // O += P V, P scaled by 256 and rounded to E4M3
#pragma unroll
  for (int kg = 0; kg < NT / 4; ++kg) {
    const float f = 256.f;
    const uint32_t a0 = pack_e4m3x4(s[4 * kg][0] * f, s[4 * kg][1] * f, s[4 * kg + 1][0] * f, s[4 * kg + 1][1] * f);
    const uint32_t a1 = pack_e4m3x4(s[4 * kg][2] * f, s[4 * kg][3] * f, s[4 * kg + 1][2] * f, s[4 * kg + 1][3] * f);
    const uint32_t a2 =
        pack_e4m3x4(s[4 * kg + 2][0] * f, s[4 * kg + 2][1] * f, s[4 * kg + 3][0] * f, s[4 * kg + 3][1] * f);
    const uint32_t a3 =
        pack_e4m3x4(s[4 * kg + 2][2] * f, s[4 * kg + 2][3] * f, s[4 * kg + 3][2] * f, s[4 * kg + 3][3] * f);
    const int kk = (k0 >> 5) + kg;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      const int dim = 8 * nd + gq;
      const uint2 bv = *reinterpret_cast<const uint2*>(vt + dim * 128 + ((kk ^ (dim & 3)) * 4 + tq) * 8);
      mma_m16n8k32(ws.o[nd], a0, a1, a2, a3, bv.x, bv.y);
    }
  }
}

template <int KWS>
__device__ __forceinline__ void attn_body(const AttnParams& p, AttnSmem& sm, int b, int g, int N, int r0, int R,
                                          int nmy, int jb0) {
  constexpr int MTP = kMathWarps / KWS;  // m-tiles covered by the MMA warps
  constexpr int KPW = kBlock / KWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int M = kQPerKV * R;
  const int MT = (M + 15) / 16;
  const int mt = warp % MTP, ksplit = warp / MTP;
  const bool math = warp < kMathWarps;
  const bool active = math && mt < MT;
  const int rA = 2 * mt, rB = 2 * mt + 1;  // speculative rows of this warp's two accumulator rows
  const int posA = N - R + rA, posB = N - R + rB;

  auto issue = [&](int j) {
    const int st = j % kAttnStages;
    const int phys = sm.phys[jb0 + j];
    const uint32_t bar = smem_u32(&sm.full[st]);
    const bool bad = phys < 0 || phys >= p.num_pages;
    sm.stage_bad[st] = bad ? 1 : 0;
    if (bad) {
      set_flag(p.flags, kFlagBadPage);
      mbar_arrive(bar);
      return;
    }
    const long long head_row = (static_cast<long long>(phys) * kGroups + g) * kBlock;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, 2 * (kHeadPageBytes + kHeadScaleBytes));
    bulk_load(smem_u32(sm.kc[st]), p.k_data + head_row * 64, kHeadPageBytes, bar);
    bulk_load(smem_u32(sm.ksc[st]), p.k_scale + head_row * 8, kHeadScaleBytes, bar);
    bulk_load(smem_u32(sm.vc[st]), p.v_data + head_row * 64, kHeadPageBytes, bar);
    bulk_load(smem_u32(sm.vsc[st]), p.v_scale + head_row * 8, kHeadScaleBytes, bar);
  };

  WarpState ws;
  if (!math) {
    // ================= dequant warps: raw page j (stage j % kAttnStages) -> tile j % kTileBufs
    const int dtid = tid - kMathWarps * 32;
    if (dtid == 0)
      for (int j = 0; j < nmy && j < kAttnStages; ++j) issue(j);
    for (int j = 0; j < nmy; ++j) {
      const int st = j % kAttnStages, buf = j % kTileBufs;
      if (!mbar_wait(smem_u32(&sm.full[st]), (j / kAttnStages) & 1, p.flags)) break;
      if (j >= kTileBufs && !mbar_wait(smem_u32(&sm.tempty[buf]), ((j / kTileBufs) - 1) & 1, p.flags)) break;
      const int blk = sm.ids[jb0 + j];
      const int pos0 = blk * kBlock;
      const int nvalid = N - pos0 < kBlock ? N - pos0 : kBlock;
      dequant_block(sm, st, buf, nvalid, sm.stage_bad[st] != 0);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.tfull[buf]));
        mbar_arrive(smem_u32(&sm.empty[st]));
      }
      // the stage's next page, once all 4 dequant warps have read this one
      if (dtid == 0 && j + kAttnStages < nmy) {
        if (!mbar_wait(smem_u32(&sm.empty[st]), (j / kAttnStages) & 1, p.flags)) break;
        issue(j + kAttnStages);
      }
    }
  } else {
    // ================= MMA warps
    uint32_t qa[4][4];
    {
      const uint8_t* qA = p.q + ((static_cast<long long>(r0 + rA) * kHeads) + kQPerKV * g + gq) * kDim;
      const uint8_t* qB = p.q + ((static_cast<long long>(r0 + rB) * kHeads) + kQPerKV * g + gq) * kDim;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const bool okA = active && rA < R, okB = active && rB < R;
        qa[ks][0] = okA ? *reinterpret_cast<const uint32_t*>(qA + 32 * ks + 4 * tq) : 0u;
        qa[ks][1] = okB ? *reinterpret_cast<const uint32_t*>(qB + 32 * ks + 4 * tq) : 0u;
        qa[ks][2] = okA ? *reinterpret_cast<const uint32_t*>(qA + 32 * ks + 16 + 4 * tq) : 0u;
        qa[ks][3] = okB ? *reinterpret_cast<const uint32_t*>(qB + 32 * ks + 16 + 4 * tq) : 0u;
      }
    }
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) ws.o[nd][0] = ws.o[nd][1] = ws.o[nd][2] = ws.o[nd][3] = 0.f;
    ws.mA = ws.mB = -INFINITY;
    ws.lA = ws.lB = 0.f;
    for (int j = 0; j < nmy; ++j) {
      const int buf = j % kTileBufs;
      if (!mbar_wait(smem_u32(&sm.tfull[buf]), (j / kTileBufs) & 1, p.flags)) break;
      if (active) {
        const int pos0 = sm.ids[jb0 + j] * kBlock;
        constexpr int kChunk = KPW < 64 ? KPW : 64;  // keys per online-softmax step (register budget)
#pragma unroll 1
        for (int kc = 0; kc < KPW; kc += kChunk)
          attend_keys<kChunk / 8>(sm.khat[buf], sm.vt[buf], ws, qa, ksplit * KPW + kc, pos0, posA, posB,
                                  p.sm_scale_log2);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tempty[buf]));
    }
  }
  if (!math) return;  // the dequant warps are done; the MMA warps finish
  // full row sums across the quad
  ws.lA += __shfl_xor_sync(0xFFFFFFFFu, ws.lA, 1);
  ws.lA += __shfl_xor_sync(0xFFFFFFFFu, ws.lA, 2);
  ws.lB += __shfl_xor_sync(0xFFFFFFFFu, ws.lB, 1);
  ws.lB += __shfl_xor_sync(0xFFFFFFFFu, ws.lB, 2);
  if (KWS > 1) {
    if (active && ksplit > 0) {
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        const int d = 8 * nd + 2 * tq;
        sm.comb_o[warp][gq][d] = ws.o[nd][0];
        sm.comb_o[warp][gq][d + 1] = ws.o[nd][1];
        sm.comb_o[warp][gq + 8][d] = ws.o[nd][2];
        sm.comb_o[warp][gq + 8][d + 1] = ws.o[nd][3];
      }
      if (tq == 0) {
        sm.comb_ml[warp][gq][0] = ws.mA;
        sm.comb_ml[warp][gq][1] = ws.lA;
        sm.comb_ml[warp][gq + 8][0] = ws.mB;
        sm.comb_ml[warp][gq + 8][1] = ws.lB;
      }
    }
    named_bar_sync(1, kMathWarps * 32);  // the MMA warps only
    if (active && ksplit == 0) {
      float MA = ws.mA, MB = ws.mB;
#pragma unroll
      for (int k = 1; k < KWS; ++k) {
        MA = fmaxf(MA, sm.comb_ml[warp + k * MTP][gq][0]);
        MB = fmaxf(MB, sm.comb_ml[warp + k * MTP][gq + 8][0]);
      }
      const float refA = MA == -INFINITY ? 0.f : MA, refB = MB == -INFINITY ? 0.f : MB;
      const float wA0 = exp2f(ws.mA - refA), wB0 = exp2f(ws.mB - refB);
      float lA = ws.lA * wA0, lB = ws.lB * wB0;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        ws.o[nd][0] *= wA0;
        ws.o[nd][1] *= wA0;
        ws.o[nd][2] *= wB0;
        ws.o[nd][3] *= wB0;
      }
#pragma unroll
      for (int k = 1; k < KWS; ++k) {
        const int w2 = warp + k * MTP;
        const float wA = exp2f(sm.comb_ml[w2][gq][0] - refA), wB = exp2f(sm.comb_ml[w2][gq + 8][0] - refB);
        lA += sm.comb_ml[w2][gq][1] * wA;
        lB += sm.comb_ml[w2][gq + 8][1] * wB;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
          const int d = 8 * nd + 2 * tq;
          ws.o[nd][0] += wA * sm.comb_o[w2][gq][d];
          ws.o[nd][1] += wA * sm.comb_o[w2][gq][d + 1];
          ws.o[nd][2] += wB * sm.comb_o[w2][gq + 8][d];
          ws.o[nd][3] += wB * sm.comb_o[w2][gq + 8][d + 1];
        }
      }
      ws.mA = MA;
      ws.mB = MB;
      ws.lA = lA;
      ws.lB = lB;
    }
  }

  // ---- write: final (single split) or partial for the merge
  const int pair = b * kGroups + g;
  if (active && ksplit == 0) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int rq = half ? rB : rA;
      const float m = half ? ws.mB : ws.mA, l = half ? ws.lB : ws.lA;
      if (rq >= R) continue;
      const int mrow = rq * kQPerKV + gq;  // query row within the pair
      const float inv = l > 0.f ? 1.f / (256.f * l) : 0.f;
      const float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
      if (p.splits == 1) {
        uint32_t* out = reinterpret_cast<uint32_t*>(p.out + ((static_cast<long long>(r0 + rq) * kHeads) +
                                                            kQPerKV * g + gq) * kDim);
#pragma unroll
        for (int nd = 0; nd < 16; ++nd)
          out[(8 * nd + 2 * tq) >> 1] = bf16x2_bits(ws.o[nd][2 * half] * inv, ws.o[nd][2 * half + 1] * inv);
        if (p.lse != nullptr && tq == 0)
          p.lse[(static_cast<long long>(r0 + rq) * kHeads) + kQPerKV * g + gq] = lse2 * 0.69314718055994531f;
      } else {
        const long long base =
            ((static_cast<long long>(blockIdx.x) * p.num_reqs * kGroups + pair) * p.max_m + mrow);
        float2* po = reinterpret_cast<float2*>(p.part_o + base * kDim);
#pragma unroll
        for (int nd = 0; nd < 16; ++nd)
          po[(8 * nd + 2 * tq) >> 1] = make_float2(ws.o[nd][2 * half] * inv, ws.o[nd][2 * half + 1] * inv);
        if (tq == 0) p.part_lse2[base] = lse2;
      }
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem_al = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_al);
  const int tid = threadIdx.x;
  const int pair = blockIdx.y, b = pair / kGroups, g = pair % kGroups;

  for (int s = tid; s < 256; s += kAttnThreads) {
    const uint32_t sc = e4m3_to_h2_bcast(static_cast<uint32_t>(s & 0x7F));
    sm.lut[s] = make_uint2(cvt_e2m1x2_scaled(0x10, sc) | (cvt_e2m1x2_scaled(0x32, sc) << 16),
                           cvt_e2m1x2_scaled(0x54, sc) | (cvt_e2m1x2_scaled(0x76, sc) << 16));
  }
  if (tid == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kDqWarps);
    }
    for (int t = 0; t < kTileBufs; ++t) {
      mbar_init(smem_u32(&sm.tfull[t]), kDqWarps);
      mbar_init(smem_u32(&sm.tempty[t]), kMathWarps);
    }
    mbar_fence_init();
  }

  // block ids are produced by the preceding selection kernel
  pdl_wait_primary();

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
  if (tid == 0) {
    int n = 0;
    for (int i = 0; i < kTopK; ++i) {
      const int id = p.block_ids[(static_cast<long long>(b) * kGroups + g) * kTopK + i];
      if (id >= 0 && id < nb) sm.ids[n++] = id;
      else if (id != -1 && blockIdx.x == 0) set_flag(p.flags, kFlagBadIds);
    }
    sm.nsel = n;
  }
  __syncthreads();
  // the selected blocks' page ids, read once (not on the copy-issue path)
  if (tid < sm.nsel) sm.phys[tid] = p.block_table[static_cast<long long>(b) * p.max_pages + sm.ids[tid]];
  __syncthreads();
  const int jb0 = blockIdx.x * p.blocks_per_split;
  int nmy = sm.nsel - jb0;
  nmy = nmy < 0 ? 0 : (nmy > p.blocks_per_split ? p.blocks_per_split : nmy);

  const int M = kQPerKV * R;
  const int MT = (M + 15) / 16;
  if (MT == 1) attn_body<4>(p, sm, b, g, N, r0, R, nmy, jb0);
  else if (MT == 2) attn_body<2>(p, sm, b, g, N, r0, R, nmy, jb0);
  else attn_body<1>(p, sm, b, g, N, r0, R, nmy, jb0);

  if (p.splits == 1) return;
  // ---- last CTA of this (request, group) merges the splits' partials
  __threadfence();
  __syncthreads();
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
  // 1. per query row: the splits' weights exp2(lse2_s - ref) / sum, and the row's lse
  float* wgt = &sm.comb_o[0][0][0];  // [M][kTopK], the block buffers are free now
  for (int mrow = tid; mrow < M; mrow += kAttnThreads) {
    const long long base = static_cast<long long>(pair) * p.max_m + mrow;
    float l2[kTopK];
    float mx = -INFINITY;
#pragma unroll
    for (int s = 0; s < kTopK; ++s) {
      l2[s] = s < nsplit_used ? __ldcg(p.part_lse2 + s * stride + base) : -INFINITY;
      mx = fmaxf(mx, l2[s]);
    }
    const float ref = mx == -INFINITY ? 0.f : mx;
    float den = 0.f;
#pragma unroll
    for (int s = 0; s < kTopK; ++s) {
      l2[s] = s < nsplit_used ? exp2f(l2[s] - ref) : 0.f;
      den += l2[s];
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int s = 0; s < kTopK; ++s) wgt[mrow * kTopK + s] = l2[s] * inv;
    if (p.lse != nullptr) {
      const int rq = mrow / kQPerKV, hh = mrow % kQPerKV;
      p.lse[(static_cast<long long>(r0 + rq) * kHeads) + kQPerKV * g + hh] =
          den > 0.f ? (ref + log2f(den)) * 0.69314718055994531f : -INFINITY;
    }
  }
  __syncthreads();
  // 2. out[row][4 dims] = sum over splits of weight x partial (16-byte loads, all threads)
  for (int idx = tid; idx < M * (kDim / 4); idx += kAttnThreads) {
    const int mrow = idx / (kDim / 4), d4 = idx % (kDim / 4);
    const long long base = static_cast<long long>(pair) * p.max_m + mrow;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < nsplit_used; ++s) {
      const float w = wgt[mrow * kTopK + s];
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + (s * stride + base) * kDim) + d4);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    const int rq = mrow / kQPerKV, hh = mrow % kQPerKV;
    const long long orow = (static_cast<long long>(r0 + rq) * kHeads) + kQPerKV * g + hh;
    uint2 packed = make_uint2(bf16x2_bits(acc.x, acc.y), bf16x2_bits(acc.z, acc.w));
    *reinterpret_cast<uint2*>(p.out + orow * kDim + 4 * d4) = packed;
  }
}

size_t attn_smem_bytes() { return sizeof(AttnSmem) + 128; }

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
