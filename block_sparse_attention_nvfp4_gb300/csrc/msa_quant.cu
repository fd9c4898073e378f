// NVFP4 insertion of new keys and values into the paged caches.
//
// [vLLM-zh "QKV GEMM + norm + RoPE + KV insert fusion"] the fused projection
// epilogue takes the FP32 accumulators head by head and quantises K, V and the
// index keys to NVFP4, writing them straight into their caches. This kernel is the
// quantise-and-write half of that epilogue on its own: FP32 rows in, NVFP4 rows in
// the caches' pages out (the GEMM, norm and RoPE are not part of it).
//
// NVFP4 per 16 consecutive elements: scale = amax / 6 rounded to E4M3 (nearest,
// ties to even, saturating at 448); element code = the E2M1 value nearest
// x / scale (ties to the even code, saturating at 6) with the sign of x; a zero
// scale gives zero codes.
//
// Both roundings are decided by exact FP32 comparisons, so the result equals an
// exact (real-number) evaluation for every finite input:
//  * scale: the hardware conversion of fl(amax * (1/6)) (relative error below
//    2^-22) is at most one code away from the exact rounding; it is corrected by
//    comparing amax with 6 x the midpoints to its neighbours. Two neighbouring E4M3
//    values sum to at most 5 significant bits, times 3 at most 7: exact in FP32.
//  * codes: |x| is compared with t x scale for the midpoints t of the E2M1 grid
//    (0.25 .. 5, at most 3 significant bits; the scale at most 4): exact. A
//    three-level search takes >= at the first two levels and > at the third, which
//    sends each tie to the even code.
//
// Layout: one warp per 128-element row (lane = 4 consecutive elements, 4 lanes = one
// 16-element group), rows numbered token * 9 + {0..3: K heads, 4..7: V heads,
// 8: index key}; a warp takes kRows rows per pass and issues their loads first.
#include <cstdint>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantCtasPerSm = 4;  // 32 warps x 4 rows x 512 B = 64 KB of loads in flight per SM
constexpr int kRows = 4;           // rows per warp per pass
constexpr int kRowsPerToken = 9;   // 4 K heads, 4 V heads, 1 index key

// E4M3 code 0..126 (non-negative, finite) to its FP32 value, from the bits.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;  // m 2^-9
}

// E4M3 scale code of a group whose largest magnitude is amax (finite, >= 0).
__device__ __forceinline__ uint32_t scale_code(float amax) {
  uint32_t pair;
  asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; cvt.u32.u16 %0, t; }"
      : "=r"(pair)
      : "f"(0.f), "f"(amax * (1.f / 6.f)));
  uint32_t c = pair & 0xFFu;  // the second operand lands in the low byte
  const float vc = e4m3_value(c);
  const float up = c < 126u ? 3.f * (vc + e4m3_value(c + 1u)) : __int_as_float(0x7f800000);  // 6 x midpoint
  const float dn = c > 0u ? 3.f * (e4m3_value(c - 1u) + vc) : -1.f;
  if (amax > up || (amax == up && (c & 1u))) ++c;
  else if (amax < dn || (amax == dn && (c & 1u))) --c;
  return c;
}

// E2M1 magnitude code (0..7) of |x| / sv, given the midpoint products t x sv.
struct E2m1Thresholds {
  float t025, t075, t125, t175, t25, t35, t5;
};
__device__ __forceinline__ uint32_t e2m1_code(float x, const E2m1Thresholds& t) {
  const float a = fabsf(x);
  const bool b2 = a >= t.t175;                        // codes 4..7 (tie 1.75 -> 4)
  const bool b1 = a >= (b2 ? t.t35 : t.t075);         // 6..7 | 2..3 (ties 3.5 -> 6, 0.75 -> 2)
  const float t3 = b2 ? (b1 ? t.t5 : t.t25) : (b1 ? t.t125 : t.t025);
  const bool b0 = a > t3;                             // ties 5 -> 6, 2.5 -> 4, 1.25 -> 2, 0.25 -> 0
  return (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u) | ((__float_as_uint(x) >> 28) & 8u);
}

__global__ void __launch_bounds__(kQuantThreads, kQuantCtasPerSm) kv_insert_kernel(const KvInsertParams p) {
  const int lane = threadIdx.x & 31;
  const long long nrows = p.num_tokens * kRowsPerToken;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * kQuantThreads + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * kQuantThreads) >> 5;
  for (long long r0 = warp0 * kRows; r0 < nrows; r0 += nwarps * kRows) {
    float4 x[kRows];
    uint8_t* dst_code[kRows];
    uint8_t* dst_scale[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      dst_code[i] = nullptr;
      dst_scale[i] = nullptr;
      const long long r = r0 + i;
      if (r >= nrows) continue;
      const long long t = r / kRowsPerToken;
      const int kind = static_cast<int>(r - t * kRowsPerToken);
      const long long sl = p.slot_mapping[t];
      if (sl < 0) continue;
      const long long page = sl >> 7, slot = sl & 127;
      if (page >= p.num_pages) {
        if (lane == 0 && kind == 0) set_flag(p.flags, kFlagBadSlot);
        continue;
      }
      const float* src;
      if (kind < kGroups) {
        if (p.k == nullptr) continue;
        src = p.k + (t * kGroups + kind) * kDim;
        const long long row = (page * kGroups + kind) * kBlock + slot;
        dst_code[i] = p.k_data + row * 64;
        dst_scale[i] = p.k_scale + row * 8;
      } else if (kind < 2 * kGroups) {
        if (p.v == nullptr) continue;
        src = p.v + (t * kGroups + (kind - kGroups)) * kDim;
        const long long row = (page * kGroups + (kind - kGroups)) * kBlock + slot;
        dst_code[i] = p.v_data + row * 64;
        dst_scale[i] = p.v_scale + row * 8;
      } else {
        if (p.ki == nullptr) continue;
        src = p.ki + t * kDim;
        const long long row = page * kBlock + slot;
        dst_code[i] = p.ki_data + row * 64;
        dst_scale[i] = p.ki_scale + row * 8;
      }
      x[i] = __ldcs(reinterpret_cast<const float4*>(src) + lane);  // read once: streaming
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      if (dst_code[i] == nullptr) continue;  // warp-uniform
      float amax = fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)), fmaxf(fabsf(x[i].z), fabsf(x[i].w)));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      const uint32_t sc = scale_code(amax);
      const float sv = e4m3_value(sc);
      const E2m1Thresholds th = {0.25f * sv, 0.75f * sv, 1.25f * sv, 1.75f * sv, 2.5f * sv, 3.5f * sv, 5.f * sv};
      uint32_t codes = e2m1_code(x[i].x, th) | (e2m1_code(x[i].y, th) << 4) | (e2m1_code(x[i].z, th) << 8) |
                       (e2m1_code(x[i].w, th) << 12);
      if (sv == 0.f) codes = 0u;
      reinterpret_cast<uint16_t*>(dst_code[i])[lane] = static_cast<uint16_t>(codes);
      if ((lane & 3) == 0) dst_scale[i][lane >> 2] = static_cast<uint8_t>(sc);
    }
  }
}

}  // namespace

cudaError_t launch_kv_insert(const KvInsertParams& prm, int sm_count, cudaStream_t st) {
  const long long rows = prm.num_tokens * kRowsPerToken;
  const long long warps_needed = (rows + kRows - 1) / kRows;
  const long long blocks_needed = (warps_needed + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
  const long long cap = static_cast<long long>(sm_count) * kQuantCtasPerSm;  // one full wave
  const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
  if (grid <= 0) return cudaSuccess;
  kv_insert_kernel<<<grid, kQuantThreads, 0, st>>>(prm);
  return cudaGetLastError();
}

}  // namespace msa
